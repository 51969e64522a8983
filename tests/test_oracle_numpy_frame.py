"""The oracle's whole frame against a second statement of the same steps,
written here in numpy (float64) from the method's description rather than
from the oracle's code: tiny model, general random weights, two sessions
with different prefixes and histories, three teacher-forced greedy frames.
Raw logits of all 16 codebooks, the greedy codes, the appended K/V and the
advanced state must agree, with BF16 weights and with INT8 weights
("Qwen3-TTS Native v0.3.0", What changed: per-output-channel symmetric,
quantised from BF16). The shapes of the steps (a Talker decode step
over a paged cache, the final norm and codebook-0 head, the 2048 -> 1024
style projection into the Code Predictor, 15 Code-Predictor steps each with
its own head over a cache emptied every frame) follow "Qwen3-TTS PR 5"
(Graph; What changed vs the 0.6B port) and "De grens van snelheid en kosten
verleggen voor Qwen3-TTS" (Hoe we Qwen3-TTS hebben geoptimaliseerd;
section 3)."""
import numpy as np
import pytest

from codebook_decode_gb300 import configs, synth
from oracle import orc

D = configs.TINY
CAP = 64
FRAMES = 3


def f64(a):
    return synth.bf16_to_f32(a).astype(np.float64)


def to_bf16_rne(x):
    """Round float64 values to bf16 (8 significant bits, ties to even),
    returned as float64: the storage format of the K/V caches."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                         # x = m 2^e, 0.5 <= |m| < 1
    q = np.ldexp(1.0, np.maximum(e - 8, -133))  # quantum of an 8-bit significand (bf16 subnormals: 2^-133)
    return np.where(x == 0.0, 0.0, np.round(x / q) * q)


def int8_rows(wbits):
    """Per-row symmetric INT8 in binary32: scale = max|w| / 127, q = w / scale
    rounded half to even and clamped to +-127, zero rows scale 0; returned as
    the float64 matrix scale x q the INT8 GEMM multiplies by."""
    w = synth.bf16_to_f32(wbits)
    m = np.abs(w).max(axis=1)
    scale = (m / np.float32(127.0)).astype(np.float32)
    safe = np.where(scale == 0, np.float32(1.0), scale)
    q = np.clip(np.rint((w / safe[:, None]).astype(np.float32)), -127, 127)
    q[scale == 0] = 0
    return scale.astype(np.float64)[:, None] * q.astype(np.float64)


def is_decode_linear(name):
    return name.endswith(("q_proj", "k_proj", "v_proj", "o_proj", "gate_proj", "up_proj", "down_proj")) or \
        name in ("talker.codec_head", "cp.proj") or name.startswith("cp.heads.")


class Model:
    def __init__(self, w, d, int8=False):
        self.w, self.d, self.int8 = w, d, int8

    def W(self, name):
        if self.int8 and is_decode_linear(name):
            return int8_rows(self.w[name])
        return f64(self.w[name])

    def rms(self, x, gname):
        return x / np.sqrt(np.mean(x * x) + self.d.rms_eps) * self.W(gname)

    @staticmethod
    def rope(v, nh, hd, pos, theta):
        vv = v.reshape(nh, hd)
        half = hd // 2
        ang = pos * theta ** (-2.0 * np.arange(half) / hd)
        c, s = np.cos(ang), np.sin(ang)
        a, b = vv[:, :half], vv[:, half:]
        return np.concatenate([a * c - b * s, b * c + a * s], axis=1).reshape(-1)

    def layer(self, prefix, x, pos, kc, vc, nq, nkv, hd, theta):
        """One decoder layer at position pos; kc/vc [cap][nkv][hd] float64
        caches holding bf16 values, row pos written here."""
        n = self.rms(x, prefix + "input_norm")
        q = self.rope(self.W(prefix + "q_proj") @ n, nq, hd, pos, theta)
        k = self.rope(self.W(prefix + "k_proj") @ n, nkv, hd, pos, theta)
        v = self.W(prefix + "v_proj") @ n
        kc[pos] = to_bf16_rne(k).reshape(nkv, hd)
        vc[pos] = to_bf16_rne(v).reshape(nkv, hd)
        a = np.zeros(nq * hd)
        for h in range(nq):
            g = h // (nq // nkv)
            sc = kc[: pos + 1, g] @ q[h * hd:(h + 1) * hd] / np.sqrt(hd)
            p = np.exp(sc - sc.max())
            p /= p.sum()
            a[h * hd:(h + 1) * hd] = p @ vc[: pos + 1, g]
        x = x + self.W(prefix + "o_proj") @ a
        n2 = self.rms(x, prefix + "post_attn_norm")
        gt = self.W(prefix + "gate_proj") @ n2
        up = self.W(prefix + "up_proj") @ n2
        return x + self.W(prefix + "down_proj") @ (gt / (1.0 + np.exp(-gt)) * up)


def greedy0(l0, seen, d, rep):
    """Codebook-0 greedy rule in binary32: ids >= n_codes other than EOS and
    (EOS not allowed) EOS itself never win; seen ids are penalised (positive
    divided, others multiplied); lowest id on ties."""
    l = l0.astype(np.float32)
    ids = np.arange(len(l))
    l[(ids >= d.n_codes) & (ids != d.eos_id)] = -np.inf
    l[d.eos_id] = -np.inf
    r = np.float32(rep)
    for v in np.nonzero(seen)[0]:
        l[v] = l[v] / r if l[v] > 0 else l[v] * r
    return int(np.argmax(l))


def numpy_frames(w, sess, B, int8=False):
    d = D
    M = Model(w, d, int8)
    kv_len = [int(sess.kv_len0[b]) for b in range(B)]
    caches = []
    for b in range(B):
        pre = f64(sess.prefix_kv(b))  # [L][2][n][nkv][hd]
        kc = np.zeros((d.n_layers, CAP, d.n_kv_heads, d.head_dim))
        vc = np.zeros_like(kc)
        kc[:, : pre.shape[2]] = pre[:, 0]
        vc[:, : pre.shape[2]] = pre[:, 1]
        caches.append((kc, vc))
    seen = []
    for b in range(B):
        bits = sess.seen_bitmap()[b]
        seen.append(np.array([(bits[v >> 5] >> (v & 31)) & 1 for v in range(d.vocab0)], dtype=bool))
    out = []
    for f in range(FRAMES):
        emb = sess.in_embeds(f)
        forced = sess.forced_codes(f)
        frame = []
        for b in range(B):
            kc, vc = caches[b]
            x = f64(emb[b])
            pos = kv_len[b]
            for l in range(d.n_layers):
                x = M.layer(f"talker.layers.{l}.", x, pos, kc[l], vc[l], d.n_q_heads, d.n_kv_heads, d.head_dim,
                            d.rope_theta)
            h = M.rms(x, "talker.final_norm")
            logits = [M.W("talker.codec_head") @ h]
            codes = [greedy0(logits[0], seen[b], d, sess.rep_penalty)]
            committed = [int(forced[b, 0])]
            seen[b][committed[0]] = True
            # Code Predictor: empty cache each frame; position 0 = P(h),
            # position j >= 1 = P(E_{j-1}[c_{j-1}]); codebook j from position j
            ck = np.zeros((d.cp_layers, 16, d.cp_n_kv_heads, d.cp_head_dim))
            cv = np.zeros_like(ck)
            P = M.W("cp.proj")

            def cp_pos(inp, p):
                y = inp
                for l in range(d.cp_layers):
                    y = M.layer(f"cp.layers.{l}.", y, p, ck[l], cv[l], d.cp_n_q_heads, d.cp_n_kv_heads,
                                d.cp_head_dim, d.cp_rope_theta)
                return y

            cp_pos(P @ h, 0)
            for j in range(1, 16):
                e = M.W(f"codec_embed.{j - 1}")[committed[j - 1]]
                y = cp_pos(P @ e, j)
                lj = M.W(f"cp.heads.{j}") @ M.rms(y, "cp.final_norm")
                logits.append(lj)
                codes.append(int(np.argmax(lj.astype(np.float32))))
                committed.append(int(forced[b, j]))
            kv_len[b] += 1
            frame.append((logits, codes))
        out.append(frame)
    return out, caches, kv_len


@pytest.fixture(scope="module")
def weights():
    return synth.make_weights(D, 1234)


@pytest.mark.parametrize("int8", [False, True])
def test_frames_match_numpy_restatement(orc_lib, weights, int8):
    B = 2
    sess = synth.Sessions(D, B, [20, 27], [0, 5], FRAMES + 1, 2077, temperature=0.0, top_k=1, rep_penalty=1.05)
    ref, ref_caches, ref_len = numpy_frames(weights, sess, B, int8)

    O = orc.Oracle(D, weights, use_int8=int8)
    rows = sess.session_array().copy()
    kv = [orc.kv_cache_from_prefix(sess.prefix_kv(b), CAP) for b in range(B)]
    rng, seen = sess.rng_state().copy(), sess.seen_bitmap().copy()
    for f in range(FRAMES):
        codes, _, lg = O.frame_step(rows, kv, CAP, sess.in_embeds(f), rng, seen, forced=sess.forced_codes(f))
        for b in range(B):
            logits, want = ref[f][b]
            for j in range(16):
                n = D.vocab0 if j == 0 else D.cp_vocab
                got = lg[b, j, :n]
                scale = np.abs(logits[j]).max()
                assert np.abs(got - logits[j]).max() <= 1e-10 * scale, (f, b, j)
            assert codes[b].tolist() == want, (f, b)
    for b in range(B):
        assert rows[b, 0] == ref_len[b]
        kc, vc = ref_caches[b]
        got = f64(kv[b])  # [L][2][cap][nkv][hd]
        assert np.array_equal(got[:, 0], kc) and np.array_equal(got[:, 1], vc)


def test_bf16_rounding_helper_is_rne():
    """The restatement's storage rounding against exact cases: values on the
    bf16 grid stay, halfway values go to the even neighbour."""
    assert to_bf16_rne(1.0) == 1.0
    assert to_bf16_rne(1.0 + 2.0 ** -8) == 1.0            # halfway, even neighbour below
    assert to_bf16_rne(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6  # halfway, even neighbour above
    assert to_bf16_rne(1.0 + 2.0 ** -8 + 2.0 ** -30) == 1.0 + 2.0 ** -7
    assert to_bf16_rne(-3.0) == -3.0
    x = np.random.default_rng(0).standard_normal(1000).astype(np.float32)
    assert np.array_equal(to_bf16_rne(x.astype(np.float64)), synth.bf16_to_f32(synth.bf16_bits(x)).astype(np.float64))
