"""Pins for the oracle's Talker prefill on the tiny model: with the residual
branches zeroed every layer's K/V at every prompt position reduce to a
closed form (which token, which position, which layer's weights), and the
prefill is causal and splits into consecutive chunks without change."""
import numpy as np
import pytest

from codebook_decode_gb300 import configs, synth
from oracle import orc

D = configs.TINY
CAP = 96


def W(w, name):
    return synth.bf16_to_f32(w[name]).astype(np.float64)


def np_rms(x, g, eps=D.rms_eps):
    return x / np.sqrt(np.mean(x * x) + eps) * synth.bf16_to_f32(g).astype(np.float64)


def np_rope(v, nh, d, pos, theta):
    vv = v.reshape(nh, d)
    z = vv[:, : d // 2] + 1j * vv[:, d // 2:]
    z = z * np.exp(1j * pos * theta ** (-2.0 * np.arange(d // 2) / d))
    return np.concatenate([z.real, z.imag], axis=1).reshape(-1)


@pytest.fixture(scope="module")
def weights():
    return synth.make_weights(D, 1000)


def prompt(n_tok, B, seed=7):
    """Prompt embeddings [n_tok][B][hidden] as bf16 bits, N(0, 1)."""
    x = np.random.default_rng(seed).standard_normal((n_tok, B, D.hidden)).astype(np.float32)
    return synth.bf16_bits(x)


def prefill(w, sess, embeds, int8=False):
    O = orc.Oracle(D, w, use_int8=int8)
    rows = sess.session_array().copy()
    kv = [orc.kv_cache_from_prefix(sess.prefix_kv(b), CAP) for b in range(sess.B)]
    O.talker_prefill(rows, kv, CAP, embeds)
    return rows, kv


def sessions(B, prefix):
    return synth.Sessions(D, B, [prefix + 5 * b for b in range(B)], [0] * B, 2, 2000)


def test_prefill_closed_form_without_residual_branches(orc_lib, weights):
    """o_proj and down_proj zero: the residual stream is the token's embedding
    in every layer, so layer l's K at position kv_len + t is RoPE(Wk_l rms(e_t)
    g_l, kv_len + t) and V is Wv_l rms(e_t) g_l."""
    w = dict(weights)
    for n in list(w):
        if n.endswith("o_proj") or n.endswith("down_proj"):
            w[n] = np.zeros_like(w[n])
    s = sessions(2, 9)
    e = prompt(5, 2)
    rows, kv = prefill(w, s, e)
    for b in range(2):
        p0 = int(s.kv_len0[b])
        assert rows[b, 0] == p0 + 5
        for t in range(5):
            x = synth.bf16_to_f32(e[t, b]).astype(np.float64)
            for l in range(D.n_layers):
                pre = f"talker.layers.{l}."
                n = np_rms(x, w[pre + "input_norm"])
                k = np_rope(W(w, pre + "k_proj") @ n, D.n_kv_heads, D.head_dim, p0 + t, D.rope_theta)
                v = W(w, pre + "v_proj") @ n
                got_k = synth.bf16_to_f32(kv[b][l, 0, p0 + t].reshape(-1))
                got_v = synth.bf16_to_f32(kv[b][l, 1, p0 + t].reshape(-1))
                assert np.allclose(got_k, k, rtol=2 ** -8, atol=1e-30), (b, t, l)
                assert np.allclose(got_v, v, rtol=2 ** -8, atol=1e-30), (b, t, l)
        # the prefix is untouched and nothing is written past the prompt
        assert np.array_equal(kv[b][:, :, :p0], s.prefix_kv(b))
        assert not kv[b][:, :, p0 + 5:].any()


def test_prefill_is_causal(orc_lib, weights):
    """A position's K/V depend on the prompt only up to that token."""
    s = sessions(1, 11)
    e = prompt(6, 1)
    _, kv_full = prefill(weights, s, e)
    _, kv_head = prefill(weights, s, e[:4])
    p0 = int(s.kv_len0[0])
    assert np.array_equal(kv_full[0][:, :, : p0 + 4], kv_head[0][:, :, : p0 + 4])
    e2 = e.copy()
    e2[5] = prompt(1, 1, seed=99)[0]  # change the last token only
    _, kv_alt = prefill(weights, s, e2)
    assert np.array_equal(kv_full[0][:, :, : p0 + 5], kv_alt[0][:, :, : p0 + 5])
    assert not np.array_equal(kv_full[0][:, :, p0 + 5], kv_alt[0][:, :, p0 + 5])


@pytest.mark.parametrize("int8", [False, True])
def test_prefill_chunks_compose(orc_lib, weights, int8):
    """Prefill of 7 tokens equals 3 then 4 tokens (positions continue)."""
    s = sessions(2, 4)
    e = prompt(7, 2, seed=3)
    rows1, kv1 = prefill(weights, s, e, int8=int8)
    O = orc.Oracle(D, weights, use_int8=int8)
    rows2 = s.session_array().copy()
    kv2 = [orc.kv_cache_from_prefix(s.prefix_kv(b), CAP) for b in range(2)]
    O.talker_prefill(rows2, kv2, CAP, e[:3])
    O.talker_prefill(rows2, kv2, CAP, e[3:])
    assert np.array_equal(rows1, rows2)
    for b in range(2):
        assert np.array_equal(kv1[b], kv2[b])


def test_prefill_stays_bf16_under_int8(orc_lib, weights):
    """With INT8 decode enabled the prompt pass still runs on the BF16 weights
    ("Qwen3-TTS Native v0.3.0", What changed): its K/V equal the BF16 model's
    bit for bit, while an INT8 decode frame after it differs from BF16's."""
    s = sessions(2, 4)
    e = prompt(5, 2, seed=11)
    rows_b, kv_b = prefill(weights, s, e, int8=False)
    rows_i, kv_i = prefill(weights, s, e, int8=True)
    assert np.array_equal(rows_b, rows_i)
    for b in range(2):
        assert np.array_equal(kv_b[b], kv_i[b])
    outs = []
    for int8 in (False, True):
        O = orc.Oracle(D, weights, use_int8=int8)
        rows = rows_b.copy()
        kv = [k.copy() for k in kv_b]
        rng, seen = s.rng_state().copy(), s.seen_bitmap().copy()
        O.frame_step(rows, kv, CAP, e[0], rng, seen, forced=s.forced_codes(0), want_logits=False)
        outs.append(kv)
    assert not np.array_equal(outs[0][0], outs[1][0])


def test_prefill_matches_decode_frames(orc_lib, weights):
    """The prompt pass writes the K/V the decode frame would write for the
    same inputs, one token per frame (teacher-forced, so the sampler does not
    matter)."""
    s = sessions(1, 6)
    e = prompt(3, 1, seed=5)
    rows_p, kv_p = prefill(weights, s, e)
    O = orc.Oracle(D, weights)
    rows = s.session_array().copy()
    kv = [orc.kv_cache_from_prefix(s.prefix_kv(0), CAP)]
    rng, seen = s.rng_state().copy(), s.seen_bitmap().copy()
    for t in range(3):
        O.frame_step(rows, kv, CAP, e[t], rng, seen, forced=s.forced_codes(t), want_logits=False)
    assert np.array_equal(rows[:, 0], rows_p[:, 0])
    assert np.array_equal(kv[0], kv_p[0])


def test_prefill_rejects_overflow(orc_lib, weights):
    s = sessions(1, CAP - 2)
    with pytest.raises(RuntimeError):
        prefill(weights, s, prompt(3, 1))
