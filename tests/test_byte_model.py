"""The algorithmic byte counts behind the roofline figures, pinned by brute
force: the bench's cache-byte and prefill weight-byte models against a count
of every position and every named tensor, the frame's stage program against
its structure, and (on the GPU) the library's own per-frame weight-byte count
against the tensor list of the model it loaded, BF16 and INT8."""
import os
import sys

import numpy as np
import pytest

from codebook_decode_gb300 import configs, synth

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def linear_bytes(shape, int8):
    rows, cols = shape
    return rows * cols + 4 * rows if int8 else 2 * rows * cols


def frame_weight_bytes_by_tensor(d, int8):
    """Every weight matrix one frame streams, counted from the tensor list:
    the Talker layers, the codebook-0 head and the projection once; the Code
    Predictor layers once per residual codebook (15 steps); head j once.
    Gains and embedding tables are not streamed as matrices."""
    total = 0
    for name, shape, kind in synth.tensor_specs(d):
        if kind != "weight" or name.startswith("codec_embed.") or name == "cp.proj_bias":
            continue
        if name.startswith("cp.layers."):
            total += (d.n_codebooks - 1) * linear_bytes(shape, int8)
        else:
            total += linear_bytes(shape, int8)
    return total


@pytest.mark.parametrize("d", [configs.TINY, configs.FULL])
def test_kv_bytes_per_frame_by_position(d):
    """Each Talker layer reads K and V at positions 0..kv_len and writes one
    position; each Code-Predictor layer, at its p-th of 16 positions, reads
    positions 0..p and writes one. Counted position by position."""
    kv_lens = [0, 1, 15, 16, 17, 999]
    t_elem = d.n_kv_heads * d.head_dim * 2  # one position of K (or V), bf16
    c_elem = d.cp_n_kv_heads * d.cp_head_dim * 2
    n = 0
    for L in kv_lens:
        for _ in range(d.n_layers):
            for kv in range(2):
                n += sum(t_elem for _pos in range(L + 1)) + t_elem
        for p in range(16):
            for _ in range(d.cp_layers):
                for kv in range(2):
                    n += sum(c_elem for _pos in range(p + 1)) + c_elem
    assert bench.kv_bytes_per_frame(d, kv_lens) == n


@pytest.mark.parametrize("d", [configs.TINY, configs.FULL])
@pytest.mark.parametrize("int8", [False, True])
def test_talker_pass_weight_bytes(d, int8):
    """The prefill model counts the Talker layers' projection matrices once
    per pass (per-row int8 scales left out)."""
    n = 0
    for name, shape, kind in synth.tensor_specs(d):
        if name.startswith("talker.layers.") and kind == "weight":
            n += shape[0] * shape[1] * (1 if int8 else 2)
    assert bench.talker_pass_weight_bytes(d, int8) == n


def test_full_frame_weight_bytes_closed_form():
    """Full model, by hand: a Talker layer has (16 + 2*8)*128*2048 QKV +
    2048*2048 O + 2*6144*2048 gate/up + 2048*6144 down = 50,331,648
    parameters; a Code-Predictor layer (16 + 2*8)*128*1024 + 1024*2048 +
    2*3072*1024 + 1024*3072 = 15,728,640; head 0 is 3072*2048, the projection
    1024*2048 and each of the 15 residual heads 2048*1024. A frame streams 28
    Talker layers, 15 x 5 Code-Predictor layers and all heads once."""
    params = 28 * 50_331_648 + 15 * 5 * 15_728_640 + 3072 * 2048 + 1024 * 2048 + 15 * 2048 * 1024
    rows = (28 * (32 * 128 + 2048 + 2 * 6144 + 2048) + 15 * 5 * (32 * 128 + 1024 + 2 * 3072 + 1024)
            + 3072 + 1024 + 15 * 2048)
    assert frame_weight_bytes_by_tensor(configs.FULL, False) == 2 * params == 5_257_560_064
    assert frame_weight_bytes_by_tensor(configs.FULL, True) == params + 4 * rows


@pytest.mark.parametrize("d", [configs.TINY, configs.FULL])
def test_stage_program(d):
    """begin, five stages per Talker layer, head0 + projection, sampler 0,
    then per residual codebook five stages per Code-Predictor layer, its
    head and its sampler."""
    names = bench.stage_names(d)
    assert len(names) == 1 + 5 * d.n_layers + 2 + (d.n_codebooks - 1) * (5 * d.cp_layers + 2)
    assert names[0] == "begin"
    assert names.count("talker.attn") == d.n_layers
    assert names.count("cp.attn") == (d.n_codebooks - 1) * d.cp_layers
    assert names.count("cp.sample") == d.n_codebooks - 1
    assert names[-1] == "cp.sample"
    if d is configs.FULL:
        assert len(names) == 548


def test_trace_summary_synthetic():
    """Stage times come out of the stamp layout: 8 stamps per stage (start,
    prologue end, weights end, epilogue end, ..., end), then the ring
    entries."""
    d = configs.TINY
    n = len(bench.stage_names(d))
    stamps = np.zeros(16 * n + 4 * 4096, dtype=np.int64)
    t = stamps[: 8 * n].reshape(n, 8)
    for i in range(n):
        s0 = 10_000 * i
        t[i] = [s0, s0 + 1000, s0 + 3000, s0 + 4000, 0, 0, 0, s0 + 5000]
    out = bench.trace_summary(d, stamps)
    assert out["frame_us"] == pytest.approx(((n - 1) * 10_000 + 5000) / 1e3)
    q = out["stages"]["talker.qkv"]
    assert q["n"] == d.n_layers
    assert q["body_us"] == pytest.approx(5.0)
    assert q["barrier_us"] == pytest.approx(5.0)
    assert (q["prologue_us"], q["weights_us"], q["epilogue_us"]) == pytest.approx((1.0, 2.0, 1.0))
    assert out["ring"]["uses"] == 0


@pytest.mark.gpu
@pytest.mark.parametrize("d", [configs.TINY, configs.FULL])
@pytest.mark.parametrize("int8", [False, True])
def test_library_frame_weight_bytes(d, int8):
    """qtts_frame_weight_bytes equals the tensor-list count of the model the
    library loaded."""
    import torch

    from codebook_decode_gb300 import qtts
    from codebook_decode_gb300.engine import Engine

    w = synth.make_weights(d, 1000)
    eng = Engine(d, w, max_batch=1, max_context=64, pool_pages=8, device=0, int8=int8)
    try:
        assert qtts.qtts_frame_weight_bytes(eng.m) == frame_weight_bytes_by_tensor(d, int8)
    finally:
        eng.close()
        torch.cuda.synchronize()


@pytest.mark.parametrize("d", [configs.TINY, configs.FULL])
def test_prefill_flops_brute_force(d):
    """The prefill FLOP model against a count token by token and layer by
    layer from the model's tensor list: 2 FLOPs per weight for QKV in every
    layer and for O, gate/up and down in all but the last; 4 per q dimension
    and attended position (positions 0..kv_len + t) in those layers."""
    shapes = {name: shape for name, shape, kind in synth.tensor_specs(d) if kind == "weight"}
    kv0, n_tok = [5, 17, 0], 4
    n = 0
    for n0 in kv0:
        for t in range(n_tok):
            for l in range(d.n_layers):
                pre = f"talker.layers.{l}."
                for proj in ("q_proj", "k_proj", "v_proj"):
                    n += 2 * shapes[pre + proj][0] * shapes[pre + proj][1]
                if l == d.n_layers - 1:
                    continue
                for proj in ("o_proj", "gate_proj", "up_proj", "down_proj"):
                    n += 2 * shapes[pre + proj][0] * shapes[pre + proj][1]
                n += 4 * d.n_q_heads * d.head_dim * (n0 + t + 1)
    assert bench.prefill_flops(d, kv0, n_tok) == n


def test_prefill_kv_bytes_by_hand():
    """Tiny model, one session with 10 cached positions and a 5-token prompt
    in chunks of 2: chunk reads 10, 12, 14 positions and writes 2, 2, 1; a
    position is 2 layers x K and V x 4 kv heads x 64 dims x 2 bytes."""
    t_tok = 2 * 2 * 4 * 64 * 2
    assert bench.prefill_kv_bytes(configs.TINY, [10], 5, 2) == (10 + 12 + 14 + 2 + 2 + 1) * t_tok
