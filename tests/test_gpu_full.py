"""GPU parity at the full Qwen3-TTS 1.7B-shaped sizes (28-layer 2048-wide
Talker, 5-layer 1024-wide Code Predictor), on the workloads' own batch sizes,
length mixes and shuffled paged caches, in the persistent launch the benchmark
times. The oracle checks teacher-forced windows of each workload (the first
frames, and the late windows of the B=32 workloads started from the GPU's own
cache and state), every frame's sampled codes bit for bit against the oracle's
sampler on the GPU's logits, and a free-running window."""
import numpy as np
import pytest

from codebook_decode_gb300 import configs, qtts, synth
from gpu_helpers import TOL_BF16, TOL_INT8, ParityRun, free
from oracle import orc

pytestmark = pytest.mark.gpu

FULL = configs.FULL


@pytest.fixture(scope="module")
def full_w():
    return synth.make_weights(FULL, 1001)


@pytest.fixture(scope="module")
def oracle_bf16(full_w):
    return orc.Oracle(FULL, full_w)


@pytest.fixture(scope="module")
def oracle_int8(full_w):
    return orc.Oracle(FULL, full_w, use_int8=True)


def check(run, tol, kv_layers=(0, 13, 27)):
    assert run.max_rel() < tol, run.max_rel()
    assert run.confident_agree == run.confident, (run.confident_agree, run.confident)
    run.check_state()
    run.check_kv(layers=list(kv_layers))


def test_full_b1_bf16(full_w, oracle_bf16):
    """Single stream, 128-token prefix, shuffled pages, sampling on."""
    s = synth.make_sessions(configs.WORKLOADS["full_b1"], frames=3)
    run = ParityRun(FULL, full_w, s, 3, oracle=oracle_bf16).run()
    try:
        check(run, TOL_BF16)
        print("full_b1 max rel", run.max_rel(), "confident", run.confident, "argmax", run.argmax_agree,
              run.argmax_total)
    finally:
        free(run)


def test_full_b8_bf16(full_w, oracle_bf16):
    """Lockstep B=8, prefixes uniform in [64, 512], shuffled page pool."""
    s = synth.make_sessions(configs.WORKLOADS["full_b8"], frames=2)
    run = ParityRun(FULL, full_w, s, 2, oracle=oracle_bf16).run()
    try:
        check(run, TOL_BF16)
    finally:
        free(run)


@pytest.mark.parametrize("chunk_talker,frames", [(33, 8), (8, 1)])
def test_full_b32_bf16_ragged_staggered(full_w, oracle_bf16, chunk_talker, frames):
    """Config 3's first window: B=32, prefixes uniform in [100, 1000] plus
    staggered offsets 0..200 (history pre-filled, frame counters at the
    offset), frames 0..7 with the Talker in the frame kernel (the default),
    frame 0 with it on the chunk kernels (option at 8)."""
    s = synth.make_sessions(configs.WORKLOADS["full_b32"], frames=frames)
    run = ParityRun(FULL, full_w, s, frames, oracle=oracle_bf16, chunk_talker_min_b=chunk_talker).run()
    try:
        check(run, TOL_BF16)
    finally:
        free(run)


def test_full_int8_b1_and_export(full_w, oracle_int8):
    s = synth.make_sessions(configs.WORKLOADS["int8_b1"], frames=2)
    run = ParityRun(FULL, full_w, s, 2, int8=True, oracle=oracle_int8).run()
    try:
        check(run, TOL_INT8)
        for name in ("talker.layers.0.q_proj", "talker.layers.27.k_proj", "talker.layers.5.v_proj",
                     "talker.layers.3.gate_proj", "talker.layers.3.up_proj", "talker.layers.9.down_proj",
                     "talker.codec_head", "cp.proj", "cp.layers.4.o_proj", "cp.heads.15"):
            q_ref, s_ref = oracle_int8.int8[name]
            q = np.zeros_like(q_ref)
            sc = np.zeros_like(s_ref)
            qtts.qtts_export_int8(run.eng.m, name, q, sc)
            assert np.array_equal(q, q_ref), name
            assert np.array_equal(sc.view(np.uint32), s_ref.view(np.uint32)), name
    finally:
        free(run)


def test_full_int8_b32(full_w, oracle_int8):
    """Config 4's first window at B=32: frames 0..7, INT8 weights."""
    s = synth.make_sessions(configs.WORKLOADS["int8_b32"], frames=8)
    run = ParityRun(FULL, full_w, s, 8, int8=True, oracle=oracle_int8).run()
    try:
        check(run, TOL_INT8)
    finally:
        free(run)


def test_full_b32_long_run_state(full_w):
    """64 free-running frames at B=32 in the persistent launch: no device
    error, every context advanced by 64, codes in range."""
    s = synth.make_sessions(configs.WORKLOADS["full_b32"], frames=64)
    run = ParityRun(FULL, full_w, s, 64)
    try:
        import torch
        from codebook_decode_gb300.engine import to_dev_u16
        emb = to_dev_u16(s.in_embeds(0), run.eng.dev)
        for _ in range(64):
            run.eng.step(emb, None, want_logits=False)
        assert run.eng.status() == (0, 0)
        kv = run.eng.sess.cpu().numpy()[:, 0]
        assert np.array_equal(kv, s.kv_len0 + 64)
        c = run.eng.codes.cpu().numpy()
        assert (c[:, 0] < FULL.n_codes).all() and (c[:, 1:] < FULL.cp_vocab).all() and (c >= 0).all()
        torch.cuda.synchronize()
    finally:
        free(run)


def test_full_b1_free_running(full_w, oracle_bf16):
    """Single stream, free running: the GPU commits its own sampled codes
    (Code-Predictor inputs, seen set), the oracle is forced with them; logits,
    codes (bit exact on the GPU's logits) and state agree."""
    s = synth.make_sessions(configs.WORKLOADS["full_b1"], frames=3)
    run = ParityRun(FULL, full_w, s, 3, oracle=oracle_bf16).run(free=True)
    try:
        check(run, TOL_BF16)
        assert run.codes_checked == 3 * 16
    finally:
        free(run)


def late_window(full_w, oracle, wl, n_before, n_window, int8):
    """Advance n_before free-running frames on the GPU, start the oracle from
    the GPU's cache and state, then check n_window teacher-forced frames."""
    import torch
    from codebook_decode_gb300.engine import to_dev_u16
    s = synth.make_sessions(configs.WORKLOADS[wl], frames=n_before + n_window)
    run = ParityRun(FULL, full_w, s, n_before + n_window, int8=int8, oracle=oracle)
    try:
        for f in range(n_before):
            run.eng.step(to_dev_u16(s.in_embeds(f), run.eng.dev), None, want_logits=False)
        assert run.eng.status() == (0, 0)
        assert np.array_equal(run.eng.sess.cpu().numpy()[:, 0], s.kv_len0 + n_before)
        run.sync_oracle_from_gpu()

        class Shifted:  # the window's frames draw the inputs of frames n_before, n_before + 1, ...
            B = s.B
            kv_len0 = s.kv_len0

            def in_embeds(self, f):
                return s.in_embeds(n_before + f)

            def forced_codes(self, f):
                return s.forced_codes(n_before + f)
        run.sess = Shifted()
        run.run(n_window)
        check(run, TOL_INT8 if int8 else TOL_BF16)
        torch.cuda.synchronize()
    finally:
        free(run)


def test_full_b32_late_window(full_w, oracle_bf16):
    """Config 3 (B=32, ragged and staggered contexts): frames 248..255 against
    the oracle started from the GPU's cache and state after 248 frames."""
    late_window(full_w, oracle_bf16, "full_b32", 248, 8, False)


def test_full_int8_b32_late_window(full_w, oracle_int8):
    """Config 4 (INT8 weights, B=32): frames 120..127 against the oracle
    started from the GPU's cache and state after 120 frames."""
    late_window(full_w, oracle_int8, "int8_b32", 120, 8, True)
