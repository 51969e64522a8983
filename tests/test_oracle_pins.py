"""Pins for the CPU oracle, each against something other than the oracle itself:
published known-answer vectors, closed forms, invariants, special cases that
reduce to a library routine, and brute force on tiny inputs."""
import ctypes as C
import math
import os

import numpy as np
import pytest
from scipy.special import softmax as sp_softmax
from scipy.stats import chisquare

from codebook_decode_gb300 import configs, synth
from oracle import orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
P = lambda a: a.ctypes.data  # noqa: E731


# --------------------------------------------------------------------------
# Philox4x32-10
# --------------------------------------------------------------------------

def _philox(L, ctr, key):
    c = np.array(ctr, dtype=np.uint32)
    k = np.array(key, dtype=np.uint32)
    o = np.zeros(4, dtype=np.uint32)
    L.orc_philox4x32_10(P(c), P(k), P(o))
    return [int(x) for x in o]


def test_philox_known_answers(orc_lib):
    rows = [l.split() for l in open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")) if l.strip() and l[0] != "#"]
    assert len(rows) == 3
    for r in rows:
        v = [int(x, 16) for x in r]
        assert _philox(orc_lib, v[0:4], v[4:6]) == v[6:10]


def test_uniform_is_philox_word(orc_lib):
    key0, key1, j, f = 0x1234, 0xBEEF, 7, 99
    for v in [0, 1, 2, 3, 4, 1023, 2047, 3071]:
        u = orc_lib.orc_uniform(key0, key1, j, f, v)
        out = _philox(orc_lib, [v >> 2, j, f, 0], [key0, key1])
        assert 0.0 < u < 1.0
        # u = (bits + 0.5) * 2^-23 exactly, bits = top 23 bits of word v & 3
        assert u * 2.0 ** 23 - 0.5 == out[v & 3] >> 9


# --------------------------------------------------------------------------
# binary32 log used by the Gumbel sampler
# --------------------------------------------------------------------------

def test_logf_exact_points(orc_lib):
    assert orc_lib.orc_logf(1.0) == 0.0
    ln2 = float(np.float32(math.log(2.0)))
    for k in range(-30, 31):
        assert orc_lib.orc_logf(2.0 ** k) == float(np.float32(np.float32(k) * np.float32(ln2)))


def test_logf_accuracy(orc_lib):
    r = np.random.default_rng(5)
    xs = np.concatenate([r.uniform(1e-7, 1.0, 4000), r.uniform(1.0, 20.0, 4000),
                         np.float32(2.0) ** r.uniform(-40, 40, 2000), [5.96e-8, 1 - 2 ** -24, 16.6, 1e-40]])
    for x in xs.astype(np.float32):
        got = orc_lib.orc_logf(float(x))
        ref = math.log(float(x))
        assert abs(got - ref) <= 3e-7 * max(1.0, abs(ref)), (x, got, ref)


# --------------------------------------------------------------------------
# bf16 storage rounding
# --------------------------------------------------------------------------

def test_bf16_roundtrip_all_finite_patterns(orc_lib):
    for h in range(0, 1 << 16, 7):
        e = (h >> 7) & 0xFF
        if e == 0xFF:
            continue
        assert orc_lib.orc_to_bf16(orc_lib.orc_from_bf16(h)) == h


def test_bf16_rounding_matches_independent_rne(orc_lib):
    r = np.random.default_rng(6)
    xs = (r.standard_normal(5000) * 10.0 ** r.integers(-6, 6, 5000)).astype(np.float32)
    ref = synth.bf16_bits(xs)  # float32 bit-trick RNE, an independent implementation
    got = np.array([orc_lib.orc_to_bf16(float(x)) for x in xs], dtype=np.uint16)
    assert np.array_equal(got, ref)
    # exact ties go to even: 1 + 2^-8 sits halfway between 1 and 1 + 2^-7
    assert orc_lib.orc_to_bf16(1.0 + 2.0 ** -8) == 0x3F80
    assert orc_lib.orc_to_bf16(1.0 + 3 * 2.0 ** -8) == 0x3F82


# --------------------------------------------------------------------------
# RMSNorm, RoPE, SiLU, linear
# --------------------------------------------------------------------------

def _rms(L, x, g, eps):
    out = np.zeros_like(x)
    L.orc_rmsnorm(P(x), P(g), len(x), eps, P(out))
    return out


def test_rmsnorm_closed_forms(orc_lib):
    r = np.random.default_rng(1)
    x = r.standard_normal(512)
    ones = synth.bf16_bits(np.ones(512, np.float32))
    y = _rms(orc_lib, x, ones, 0.0)
    assert abs(np.mean(y * y) - 1.0) < 1e-12          # unit RMS
    assert np.allclose(_rms(orc_lib, 7.5 * x, ones, 0.0), y, atol=1e-12)  # scale invariant
    g = synth.bf16_bits(r.uniform(0.5, 2.0, 512).astype(np.float32))
    assert np.allclose(_rms(orc_lib, x, g, 0.0), y * synth.bf16_to_f32(g), atol=1e-12)
    # eps enters under the root: constant row c -> c / sqrt(c^2 + eps)
    c = np.full(16, 0.01)
    assert np.allclose(_rms(orc_lib, c, ones[:16], 1e-4), 0.01 / math.sqrt(1e-4 + 1e-4), atol=1e-12)


def _rope(L, v, nh, d, pos, theta):
    v = v.copy()
    L.orc_rope(P(v), nh, d, pos, theta)
    return v


def test_rope_identity_norm_and_complex_form(orc_lib):
    r = np.random.default_rng(2)
    nh, d, theta = 3, 64, 1e6
    v = r.standard_normal(nh * d)
    assert np.array_equal(_rope(orc_lib, v, nh, d, 0, theta), v)
    for pos in [1, 17, 1000]:
        w = _rope(orc_lib, v, nh, d, pos, theta)
        # rotate-half pairs (i, i + d/2) as complex numbers turned by pos * theta^(-2i/d)
        vv = v.reshape(nh, d)
        z = vv[:, : d // 2] + 1j * vv[:, d // 2:]
        ang = pos * theta ** (-2.0 * np.arange(d // 2) / d)
        zr = z * np.exp(1j * ang)
        ref = np.concatenate([zr.real, zr.imag], axis=1).reshape(-1)
        assert np.allclose(w, ref, atol=1e-12)
        assert np.allclose(np.abs(zr), np.abs(z))
    # unit vector on pair 0 at pos 1 turns by exactly 1 radian
    e = np.zeros(d)
    e[0] = 1.0
    w = _rope(orc_lib, e, 1, d, 1, theta)
    assert abs(w[0] - math.cos(1.0)) < 1e-15 and abs(w[d // 2] - math.sin(1.0)) < 1e-15


def test_rope_relative_position(orc_lib):
    r = np.random.default_rng(3)
    d = 128
    q = r.standard_normal(d)
    k = r.standard_normal(d)
    dots = [np.dot(_rope(orc_lib, q, 1, d, p + 5, 1e6), _rope(orc_lib, k, 1, d, p, 1e6)) for p in (0, 3, 40, 700)]
    assert np.allclose(dots, dots[0], atol=1e-9)


def test_silu_closed_forms(orc_lib):
    assert orc_lib.orc_silu(0.0) == 0.0
    assert abs(orc_lib.orc_silu(1.0) - 1.0 / (1.0 + math.exp(-1.0))) < 1e-15
    for x in [0.3, 2.0, 7.0]:
        assert abs(orc_lib.orc_silu(x) - orc_lib.orc_silu(-x) - x) < 1e-12  # x*s(x) + x*s(-x) = x
    assert abs(orc_lib.orc_silu(40.0) - 40.0) < 1e-12 and abs(orc_lib.orc_silu(-40.0)) < 1e-15


def _linear(L, x, w, q=None, s=None):
    N, K = (w if w is not None else q).shape
    y = np.zeros(N)
    lin = orc.Lin(None if w is None else P(w), None if q is None else P(q), None if s is None else P(s))
    L.orc_linear(P(x), lin, 1 if q is not None else 0, N, K, P(y))
    return y


def test_linear_against_matmul(orc_lib):
    r = np.random.default_rng(4)
    w = synth.bf16_bits((r.standard_normal((37, 129)) * 0.1).astype(np.float32))
    x = r.standard_normal(129)
    assert np.allclose(_linear(orc_lib, x, w), synth.bf16_to_f32(w).astype(np.float64) @ x, atol=1e-12)
    q = r.integers(-127, 128, (37, 129)).astype(np.int8)
    s = r.uniform(1e-3, 1e-2, 37).astype(np.float32)
    assert np.allclose(_linear(orc_lib, x, None, q, s), s.astype(np.float64) * (q.astype(np.float64) @ x),
                       atol=1e-12)
    # one-hot rows pick elements (catches a transposed operand)
    eye = np.zeros((5, 129), np.float32)
    for i, c in enumerate([0, 7, 64, 100, 128]):
        eye[i, c] = 1.0
    assert np.array_equal(_linear(orc_lib, x, synth.bf16_bits(eye)), x[[0, 7, 64, 100, 128]])


# --------------------------------------------------------------------------
# attention
# --------------------------------------------------------------------------

def _attn(L, q, kc, vc, n, nq, nkv, d):
    out = np.zeros(nq * d)
    L.orc_attention(P(q), P(kc), P(vc), n, nq, nkv, d, P(out))
    return out.reshape(nq, d)


def test_attention_special_cases(orc_lib):
    r = np.random.default_rng(7)
    nq, nkv, d = 4, 2, 16
    q = r.standard_normal(nq * d)
    kc = synth.bf16_bits(r.standard_normal((9, nkv, d)).astype(np.float32))
    vc = synth.bf16_bits(r.standard_normal((9, nkv, d)).astype(np.float32))
    kf, vf = synth.bf16_to_f32(kc).astype(np.float64), synth.bf16_to_f32(vc).astype(np.float64)
    # one cached position: every head returns its group's v
    o = _attn(orc_lib, q, kc, vc, 1, nq, nkv, d)
    for h in range(nq):
        assert np.allclose(o[h], vf[0, h // 2], atol=1e-12)
    # q = 0: uniform weights, output = mean of v over the positions
    o = _attn(orc_lib, np.zeros(nq * d), kc, vc, 9, nq, nkv, d)
    for h in range(nq):
        assert np.allclose(o[h], vf[:, h // 2].mean(axis=0), atol=1e-12)
    # set function: permuting positions changes nothing
    perm = r.permutation(9)
    o1 = _attn(orc_lib, q, kc, vc, 9, nq, nkv, d)
    o2 = _attn(orc_lib, q, np.ascontiguousarray(kc[perm]), np.ascontiguousarray(vc[perm]), 9, nq, nkv, d)
    assert np.allclose(o1, o2, atol=1e-12)
    # positions past n_pos are never read
    kc2, vc2 = kc.copy(), vc.copy()
    kc2[6:] = 0x7F80
    vc2[6:] = 0x7F80
    assert np.allclose(_attn(orc_lib, q, kc, vc, 6, nq, nkv, d), _attn(orc_lib, q, kc2, vc2, 6, nq, nkv, d))
    # against library softmax + matmul
    for h in range(nq):
        sc = kf[:, h // 2] @ q[h * d:(h + 1) * d] / math.sqrt(d)
        assert np.allclose(o1[h], sp_softmax(sc) @ vf[:, h // 2], atol=1e-12)
    # GQA: query heads sharing a group see the same keys; group 1 is not group 0
    qq = np.tile(q[:d], nq)
    o = _attn(orc_lib, qq, kc, vc, 9, nq, nkv, d)
    assert np.allclose(o[0], o[1]) and np.allclose(o[2], o[3]) and not np.allclose(o[0], o[2])


# --------------------------------------------------------------------------
# INT8 quantiser
# --------------------------------------------------------------------------

def _quant(L, w):
    N, K = w.shape
    q = np.zeros((N, K), np.int8)
    s = np.zeros(N, np.float32)
    L.orc_quantize_rows(P(w), N, K, P(q), P(s))
    return q, s


def test_quantizer_crafted_rows(orc_lib):
    lines = [l.strip() for l in open(os.path.join(GOLDEN, "quantize_int8_crafted.txt")) if l.strip() and l[0] != "#"]
    for i in range(0, len(lines), 3):
        w = np.array([float(t) for t in lines[i].split()[1:]], np.float32)
        qe = np.array([int(t) for t in lines[i + 1].split()[1:]], np.int8)
        se = float(lines[i + 2].split()[1])
        wb = synth.bf16_bits(w)
        assert np.array_equal(synth.bf16_to_f32(wb), w)
        q, s = _quant(orc_lib, wb[None, :])
        assert np.array_equal(q[0], qe), (q[0], qe)
        assert s[0] == np.float32(se)


def test_quantizer_matches_numpy_rule_and_error_band(orc_lib):
    r = np.random.default_rng(8)
    w = synth.bf16_bits((r.standard_normal((64, 1024)) * 0.02).astype(np.float32))
    q, s = _quant(orc_lib, w)
    wf = synth.bf16_to_f32(w)
    m = np.abs(wf).max(axis=1)
    se = (m / np.float32(127.0)).astype(np.float32)
    assert np.array_equal(s, se)
    qe = np.clip(np.rint(wf / se[:, None]), -127, 127).astype(np.int8)  # rint: half to even
    assert np.array_equal(q, qe)
    # per-channel error "on the order of 4e-3 relative" (release notes, INT8 mode)
    rel = np.linalg.norm(wf - s[:, None] * q, axis=1) / np.linalg.norm(wf, axis=1)
    assert 1e-3 < float(rel.mean()) < 1e-2


# --------------------------------------------------------------------------
# sampler
# --------------------------------------------------------------------------

def _sess(T=0.0, k=1, r=1.0, eos=0, cpT=None, cpk=None):
    return orc.Session(0, eos, T, k, r, T if cpT is None else cpT, k if cpk is None else cpk, 0)


def _sample(L, logits, cb, s, f=0, seen=None, eos_id=2048, n_codes=2048, key=(11, 22)):
    lg = np.ascontiguousarray(logits, np.float32)
    return L.orc_sample(P(lg), len(lg), cb, C.byref(s), key[0], key[1], f, None if seen is None else P(seen),
                        eos_id, n_codes)


def test_sampler_greedy_is_argmax(orc_lib):
    r = np.random.default_rng(9)
    for _ in range(20):
        lg = r.standard_normal(2048).astype(np.float32)
        assert _sample(orc_lib, lg, 3, _sess(0.0, 50)) == int(np.argmax(lg))
        assert _sample(orc_lib, lg, 3, _sess(0.9, 1)) == int(np.argmax(lg))
    lg = np.zeros(64, np.float32)
    lg[[5, 9]] = 3.0
    assert _sample(orc_lib, lg, 1, _sess()) == 5  # lowest id on ties


def test_sampler_masks_and_eos(orc_lib):
    V = 3072
    lg = np.zeros(V, np.float32)
    lg[2500] = 50.0  # special id, never sampled in codebook 0
    lg[2048] = 40.0  # eos
    lg[17] = 1.0
    seen = np.zeros(96, np.uint32)
    assert _sample(orc_lib, lg, 0, _sess(), seen=seen) == 17
    assert _sample(orc_lib, lg, 0, _sess(eos=1), seen=seen) == 2048
    for f in range(50):
        c = _sample(orc_lib, lg, 0, _sess(1.0, 0), f=f, seen=seen)
        assert c < 2048 and c != 2048


def test_sampler_repetition_penalty(orc_lib):
    seen = np.zeros(96, np.uint32)
    seen[0] |= 1
    lg = np.zeros(3072, np.float32) - 5.0
    lg[0], lg[1] = 2.0, 1.99
    assert _sample(orc_lib, lg, 0, _sess(r=1.0), seen=seen) == 0
    assert _sample(orc_lib, lg, 0, _sess(r=1.05), seen=seen) == 1  # 2/1.05 < 1.99
    lg[0], lg[1] = -1.0, -1.04
    assert _sample(orc_lib, lg, 0, _sess(r=1.0), seen=seen) == 0
    assert _sample(orc_lib, lg, 0, _sess(r=1.05), seen=seen) == 1  # -1 * 1.05 < -1.04
    # the Code-Predictor sampler has no penalty
    lg2 = lg[:2048].copy()
    assert _sample(orc_lib, lg2, 4, _sess(r=1.05), seen=seen) == 0


def test_sampler_topk_support_and_gumbel_frequencies(orc_lib):
    lg = np.array([1.0, 0.5, 0.2, -0.3, 0.9, -1.0], np.float32)
    T = 0.7
    n = 12000
    for k, keep in [(0, [0, 1, 2, 3, 4, 5]), (3, [0, 4, 1])]:
        counts = np.zeros(6)
        for f in range(n):
            counts[_sample(orc_lib, lg, 5, _sess(T, k), f=f, key=(123, 456))] += 1
        assert set(np.nonzero(counts)[0]) <= set(keep)
        p = np.zeros(6)
        z = lg[keep].astype(np.float64) / T
        p[keep] = sp_softmax(z)
        stat, pval = chisquare(counts[keep], p[keep] * n)
        assert pval > 1e-4, (k, counts, p * n)


def test_sampler_stream_depends_on_codebook_and_frame(orc_lib):
    lg = np.zeros(2048, np.float32)
    a = [_sample(orc_lib, lg, 1, _sess(1.0, 0), f=f) for f in range(40)]
    b = [_sample(orc_lib, lg, 2, _sess(1.0, 0), f=f) for f in range(40)]
    assert a != b
    assert a == [_sample(orc_lib, lg, 1, _sess(1.0, 0), f=f) for f in range(40)]  # deterministic
