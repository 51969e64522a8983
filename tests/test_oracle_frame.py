"""Frame-level pins for the oracle on the tiny model: special weights that
reduce the frame to closed forms (which embedding table, head, position and
cache slot feed what), plus batching, causality and state invariants."""
import numpy as np
import pytest

from codebook_decode_gb300 import configs, synth
from oracle import orc

D = configs.TINY
CAP = 64


def np_rms(x, g, eps=D.rms_eps):
    return x / np.sqrt(np.mean(x * x) + eps) * synth.bf16_to_f32(g).astype(np.float64)


def np_rope(v, nh, d, pos, theta):
    vv = v.reshape(nh, d)
    z = vv[:, : d // 2] + 1j * vv[:, d // 2:]
    z = z * np.exp(1j * pos * theta ** (-2.0 * np.arange(d // 2) / d))
    return np.concatenate([z.real, z.imag], axis=1).reshape(-1)


def W(w, name):
    return synth.bf16_to_f32(w[name]).astype(np.float64)


def bf16_round(L, a):
    return np.array([L.orc_from_bf16(L.orc_to_bf16(float(t))) for t in np.ravel(a)]).reshape(np.shape(a))


def zero(w, names):
    w = dict(w)
    for n in names:
        w[n] = np.zeros_like(w[n])
    return w


def run(w, sess, frame=0, forced=True, B=None, int8=False, kv_cap=CAP):
    O = orc.Oracle(D, w, use_int8=int8)
    B = B or sess.B
    rows = sess.session_array()[:B].copy()
    kv = [orc.kv_cache_from_prefix(sess.prefix_kv(b), kv_cap) for b in range(B)]
    rng = sess.rng_state()[:B].copy()
    seen = sess.seen_bitmap()[:B].copy()
    f = sess.forced_codes(frame)[:B] if forced else None
    codes, eos, lg = O.frame_step(rows, kv, kv_cap, sess.in_embeds(frame)[:B], rng, seen, forced=f)
    return dict(O=O, rows=rows, kv=kv, rng=rng, seen=seen, forced=f, codes=codes, eos=eos, logits=lg)


@pytest.fixture(scope="module")
def weights():
    return synth.make_weights(D, 1000)


def sessions(B=1, prefix=20, T=0.0, k=1):
    return synth.Sessions(D, B, [prefix + 3 * b for b in range(B)], [b for b in range(B)], 4, 2000, temperature=T,
                          top_k=k, rep_penalty=1.05)


def residual_free(w):
    names = [n for n in w if n.endswith("o_proj") or n.endswith("down_proj")]
    return zero(w, names)


@pytest.mark.parametrize("int8", [False, True])
def test_residual_passthrough_closed_form(orc_lib, weights, int8):
    """o_proj = down_proj = 0 everywhere: every layer passes x through, so
    l0 = W_h0 rms(x_in), and codebook j reads head j on P(E_{j-1}[c_{j-1}])."""
    w = residual_free(weights)
    s = sessions()
    r = run(w, s, int8=int8)
    O = r["O"]

    def lin(name, x):
        if int8:
            q, sc = O.int8[name]
            return sc.astype(np.float64) * (q.astype(np.float64) @ x)
        return W(w, name) @ x

    x = synth.bf16_to_f32(s.in_embeds(0)[0]).astype(np.float64)
    h = np_rms(x, w["talker.final_norm"])
    assert np.allclose(r["logits"][0, 0], lin("talker.codec_head", h), rtol=0, atol=1e-9)
    forced = r["forced"][0]
    for j in range(1, 16):
        e = W(w, f"codec_embed.{j - 1}")[forced[j - 1]]
        y = lin("cp.proj", e)
        ref = lin(f"cp.heads.{j}", np_rms(y, w["cp.final_norm"]))
        assert np.allclose(r["logits"][0, j, : D.cp_vocab], ref, rtol=0, atol=1e-9), j


def test_empty_prefix_attention_is_new_value(orc_lib, weights):
    """kv_len = 0 and down_proj = 0: attention sees only the new token, so each
    layer adds Wo expand(bf16(Wv rms(x))) to x."""
    w = zero(weights, [n for n in weights if n.endswith("down_proj")])
    s = sessions(prefix=0)
    s.kv_len0[:] = 0
    s.offsets[:] = 0
    r = run(w, s)
    x = synth.bf16_to_f32(s.in_embeds(0)[0]).astype(np.float64)
    grp = D.n_q_heads // D.n_kv_heads
    for l in range(D.n_layers):
        p = f"talker.layers.{l}"
        v = bf16_round(orc_lib, W(w, f"{p}.v_proj") @ np_rms(x, w[f"{p}.input_norm"])).reshape(D.n_kv_heads, -1)
        a = np.concatenate([v[h // grp] for h in range(D.n_q_heads)])
        x = x + W(w, f"{p}.o_proj") @ a
    ref = W(w, "talker.codec_head") @ np_rms(x, w["talker.final_norm"])
    assert np.allclose(r["logits"][0, 0], ref, rtol=0, atol=1e-9)


def test_kv_append_is_rotated_key_at_kv_len(orc_lib, weights):
    s = sessions(prefix=21)
    r = run(weights, s)
    pos = int(s.kv_len0[0])
    x = synth.bf16_to_f32(s.in_embeds(0)[0]).astype(np.float64)
    n = np_rms(x, weights["talker.layers.0.input_norm"])
    k = np_rope(W(weights, "talker.layers.0.k_proj") @ n, D.n_kv_heads, D.head_dim, pos, D.rope_theta)
    v = W(weights, "talker.layers.0.v_proj") @ n
    kv = r["kv"][0]
    got_k = synth.bf16_to_f32(kv[0, 0, pos].reshape(-1))
    got_v = synth.bf16_to_f32(kv[0, 1, pos].reshape(-1))
    assert np.allclose(got_k, k, rtol=2 ** -8, atol=1e-30)
    assert np.allclose(got_v, v, rtol=2 ** -8, atol=1e-30)
    # prefix untouched, nothing written past the new position
    assert np.array_equal(kv[:, :, :pos], s.prefix_kv(0))
    assert not kv[:, :, pos + 1:].any()


def test_cp_causal_extent_closed_form(orc_lib, weights):
    """Code-Predictor k_proj = 0 (flat scores) and down_proj = 0: position p
    averages the stored values of positions 0..p."""
    w = residual_free(weights)
    w["cp.layers.0.o_proj"] = weights["cp.layers.0.o_proj"]
    w["cp.layers.0.k_proj"] = np.zeros_like(weights["cp.layers.0.k_proj"])
    s = sessions()
    r = run(w, s)
    x = synth.bf16_to_f32(s.in_embeds(0)[0]).astype(np.float64)
    h = np_rms(x, w["talker.final_norm"])
    forced = r["forced"][0]
    grp = D.cp_n_q_heads // D.cp_n_kv_heads
    vs = []
    for p in range(16):
        e = h if p == 0 else W(w, f"codec_embed.{p - 1}")[forced[p - 1]]
        y = W(w, "cp.proj") @ e
        v = bf16_round(orc_lib, W(w, "cp.layers.0.v_proj") @ np_rms(y, w["cp.layers.0.input_norm"]))
        vs.append(v.reshape(D.cp_n_kv_heads, -1))
        m = np.mean(vs, axis=0)
        a = np.concatenate([m[hh // grp] for hh in range(D.cp_n_q_heads)])
        y = y + W(w, "cp.layers.0.o_proj") @ a
        if p:
            ref = W(w, f"cp.heads.{p}") @ np_rms(y, w["cp.final_norm"])
            assert np.allclose(r["logits"][0, p, : D.cp_vocab], ref, rtol=0, atol=1e-9), p


def test_batching_invariance(orc_lib, weights):
    s = sessions(B=3, T=0.9, k=50)
    together = run(weights, s, forced=False)
    for b in range(3):
        sb = synth.Sessions(D, 1, [s.prefix_lens[b]], [s.offsets[b]], 4, 2000, temperature=0.9, top_k=50,
                            rep_penalty=1.05)
        # same per-session state as row b of the batch
        O = orc.Oracle(D, weights)
        rows = s.session_array()[b:b + 1].copy()
        kv = [orc.kv_cache_from_prefix(s.prefix_kv(b), CAP)]
        rng = s.rng_state()[b:b + 1].copy()
        seen = s.seen_bitmap()[b:b + 1].copy()
        codes, eos, lg = O.frame_step(rows, kv, CAP, s.in_embeds(0)[b:b + 1], rng, seen)
        assert np.array_equal(codes[0], together["codes"][b])
        assert np.array_equal(lg[0], together["logits"][b])
        assert np.array_equal(kv[0], together["kv"][b])
        del sb


def test_future_cache_is_never_read(orc_lib, weights):
    s = sessions(prefix=12)
    O = orc.Oracle(D, weights)
    res = []
    for poison in (False, True):
        rows = s.session_array().copy()
        kv = [orc.kv_cache_from_prefix(s.prefix_kv(0), CAP)]
        if poison:
            kv[0][:, :, 13:] = 0x4480  # 1024.0 everywhere past the new position
        codes, _, lg = O.frame_step(rows, kv, CAP, s.in_embeds(0), s.rng_state(), s.seen_bitmap(),
                                    forced=s.forced_codes(0))
        res.append(lg)
    assert np.array_equal(res[0], res[1])


def test_state_advances(orc_lib, weights):
    s = sessions(B=2, T=0.9, k=50)
    r = run(weights, s)
    assert np.array_equal(r["rows"][:, 0], s.kv_len0 + 1)
    assert np.array_equal(r["rng"][:, 2], s.rng_state()[:, 2] + 1)
    for b in range(2):
        c0 = r["forced"][b, 0]
        assert (r["seen"][b, c0 >> 5] >> (c0 & 31)) & 1
        before = s.seen_bitmap()[b].copy()
        before[c0 >> 5] |= np.uint32(1 << (c0 & 31))
        assert np.array_equal(r["seen"][b], before)  # only that bit changed


def test_feedback_sum(orc_lib, weights):
    O = orc.Oracle(D, weights)
    r = np.random.default_rng(3)
    codes = r.integers(0, 2048, (2, 16)).astype(np.int32)
    text = synth.bf16_bits(r.standard_normal((2, D.hidden)).astype(np.float32))
    got = O.feedback(codes, text)
    for b in range(2):
        ref = synth.bf16_to_f32(text[b]).astype(np.float64)
        for j in range(16):
            ref = ref + W(weights, f"codec_embed.{j}")[codes[b, j]]
        assert np.allclose(got[b], ref, rtol=0, atol=1e-12)


def test_int8_frame_close_to_bf16(orc_lib, weights):
    s = sessions()
    a = run(weights, s)["logits"]
    b = run(weights, s, int8=True)["logits"]
    rel = np.abs(a[0, 0] - b[0, 0]).max() / np.abs(a[0, 0]).max()
    assert 1e-4 < rel < 5e-2


def test_mlp_only_closed_form(orc_lib, weights):
    """o_proj = 0 in the Talker (attention adds nothing): each layer adds the
    SwiGLU MLP Wd (silu(Wg n) * (Wu n)), with silu on the gate branch only."""
    w = zero(weights, [n for n in weights if n.endswith("o_proj") and n.startswith("talker.")])
    s = sessions()
    r = run(w, s)
    x = synth.bf16_to_f32(s.in_embeds(0)[0]).astype(np.float64)
    for l in range(D.n_layers):
        p = f"talker.layers.{l}"
        n = np_rms(x, w[f"{p}.post_attn_norm"])
        g = W(w, f"{p}.gate_proj") @ n
        u = W(w, f"{p}.up_proj") @ n
        x = x + W(w, f"{p}.down_proj") @ (g / (1.0 + np.exp(-g)) * u)
    ref = W(w, "talker.codec_head") @ np_rms(x, w["talker.final_norm"])
    assert np.allclose(r["logits"][0, 0], ref, rtol=0, atol=1e-9)
