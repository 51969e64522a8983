"""The synthetic workloads follow their recipe: model shapes, batch sizes,
prefix-length and offset distributions, frame counts, sampling settings and
seeds; the drawn sessions stay inside their ranges, are reproducible, and
their prefix caches have the stated shape (host only)."""
import numpy as np
import pytest

from codebook_decode_gb300 import configs, synth

W = configs.WORKLOADS


def test_full_and_tiny_shapes():
    f, t = configs.FULL, configs.TINY
    assert (f.hidden, f.n_layers, f.n_q_heads, f.n_kv_heads, f.head_dim, f.ffn, f.vocab0) == \
        (2048, 28, 16, 8, 128, 6144, 3072)
    assert (f.cp_hidden, f.cp_layers, f.cp_n_q_heads, f.cp_n_kv_heads, f.cp_head_dim, f.cp_ffn, f.cp_vocab) == \
        (1024, 5, 16, 8, 128, 3072, 2048)
    assert (t.hidden, t.n_layers, t.n_q_heads, t.n_kv_heads, t.head_dim, t.ffn, t.vocab0) == \
        (512, 2, 8, 4, 64, 1536, 2049)
    assert (t.cp_hidden, t.cp_layers, t.cp_n_q_heads, t.cp_n_kv_heads, t.cp_head_dim, t.cp_ffn, t.cp_vocab) == \
        (256, 1, 4, 2, 64, 768, 2048)
    for d in (f, t):
        assert d.n_codebooks == 16 and d.eos_id == 2048 and d.n_codes == 2048
        assert d.n_q_heads % d.n_kv_heads == 0 and d.cp_n_q_heads % d.cp_n_kv_heads == 0


@pytest.mark.parametrize("name,B,prefix,offset,frames,T,k,r,shuffle,int8,seed", [
    ("tiny", 1, ("fixed", 32), ("fixed", 0), 16, 0.0, 1, 1.0, False, False, 0),
    ("full_b1", 1, ("fixed", 128), ("fixed", 0), 64, 0.9, 50, 1.05, True, False, 1),
    ("full_b8", 8, ("uniform", 64, 512), ("fixed", 0), 128, 0.9, 50, 1.05, True, False, 2),
    ("full_b32", 32, ("uniform", 100, 1000), ("uniform", 0, 200), 256, 0.9, 50, 1.05, True, False, 3),
    ("int8_b1", 1, ("uniform", 64, 512), ("fixed", 0), 128, 0.9, 50, 1.05, True, True, 4),
    ("int8_b32", 32, ("uniform", 64, 512), ("fixed", 0), 128, 0.9, 50, 1.05, True, True, 4),
])
def test_workload_recipe(name, B, prefix, offset, frames, T, k, r, shuffle, int8, seed):
    wl = W[name]
    assert wl.dims is (configs.TINY if name == "tiny" else configs.FULL)
    assert (wl.batch, wl.prefix, wl.offset, wl.frames) == (B, prefix, offset, frames)
    assert (wl.temperature, wl.top_k, wl.rep_penalty) == (T, k, r)
    assert (wl.shuffle_pages, wl.int8, wl.seed) == (shuffle, int8, seed)


def test_profiler_cases_differ_only_in_depth():
    for small, big in (("full2l_b1", "full_b1"), ("full2l_b32", "full_b32")):
        a, b = W[small], W[big]
        da, db = a.dims.as_dict(), b.dims.as_dict()
        assert da.pop("n_layers") == 2 and db.pop("n_layers") == 28
        assert da == db
        assert (a.batch, a.prefix, a.offset, a.temperature, a.top_k, a.rep_penalty, a.int8) == \
            (b.batch, b.prefix, b.offset, b.temperature, b.top_k, b.rep_penalty, b.int8)


@pytest.mark.parametrize("name", ["full_b8", "full_b32", "int8_b32"])
def test_drawn_sessions_in_range_and_reproducible(name):
    wl = W[name]
    s1, s2 = synth.make_sessions(wl), synth.make_sessions(wl)
    assert np.array_equal(s1.kv_len0, s2.kv_len0)
    lo, hi = wl.prefix[1], wl.prefix[2]
    assert (s1.prefix_lens >= lo).all() and (s1.prefix_lens <= hi).all()
    if wl.offset[0] == "uniform":
        assert (s1.offsets >= wl.offset[1]).all() and (s1.offsets <= wl.offset[2]).all()
    else:
        assert (s1.offsets == 0).all()
    assert np.array_equal(s1.kv_len0, s1.prefix_lens + s1.offsets)
    assert len(np.unique(s1.prefix_lens)) > 1  # a ragged mix, not one length


def test_prefix_cache_shape_and_seed():
    wl = W["tiny"]
    s = synth.make_sessions(wl)
    kv = s.prefix_kv(0)
    d = wl.dims
    assert kv.shape == (d.n_layers, 2, 32, d.n_kv_heads, d.head_dim) and kv.dtype == np.uint16
    assert np.array_equal(kv, synth.make_sessions(wl).prefix_kv(0))
    x = synth.bf16_to_f32(kv).astype(np.float64)
    assert abs(x.mean()) < 0.05 and 0.9 < x.std() < 1.1  # N(0, 1) prefix K/V
