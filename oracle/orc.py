"""ctypes driver for the C oracle (qtts_oracle.c).

TEST INFRASTRUCTURE (see the package docstring). The driver only marshals
arrays: all arithmetic of the frame lives in qtts_oracle.c.
"""
import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liborc.so")
_lock = threading.Lock()
_lib = None


def build_oracle(force=False):
    """Compile qtts_oracle.c with gcc (no fast-math, no FMA contraction)."""
    src = os.path.join(_HERE, "qtts_oracle.c")
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= max(
            os.path.getmtime(src), os.path.getmtime(os.path.join(_HERE, "qtts_oracle.h"))):
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-o", tmp, src, "-lm"]
    subprocess.check_call(cmd)
    os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build_oracle()
            _lib = C.CDLL(_SO)
            _declare(_lib)
    return _lib


# ---- C structs -------------------------------------------------------------

class Dims(C.Structure):
    _fields_ = [(n, C.c_int32) for n in (
        "hidden", "n_layers", "n_q_heads", "n_kv_heads", "head_dim", "ffn", "vocab0",
        "cp_hidden", "cp_layers", "cp_n_q_heads", "cp_n_kv_heads", "cp_head_dim", "cp_ffn", "cp_vocab",
        "n_codebooks", "eos_id", "n_codes", "proj_bias")] + [
        ("rms_eps", C.c_double), ("rope_theta", C.c_double), ("cp_rope_theta", C.c_double)]


class Lin(C.Structure):
    _fields_ = [("w", C.c_void_p), ("q", C.c_void_p), ("s", C.c_void_p)]


class Layer(C.Structure):
    _fields_ = [("in_norm", C.c_void_p), ("wq", Lin), ("wk", Lin), ("wv", Lin), ("wo", Lin),
                ("post_norm", C.c_void_p), ("wg", Lin), ("wu", Lin), ("wd", Lin)]


class Model(C.Structure):
    _fields_ = [("d", Dims), ("use_int8", C.c_int32), ("talker", C.POINTER(Layer)),
                ("final_norm", C.c_void_p), ("head0", Lin), ("proj", Lin), ("proj_b", C.c_void_p),
                ("cp", C.POINTER(Layer)), ("cp_final_norm", C.c_void_p), ("cp_head", Lin * 16),
                ("embed", C.c_void_p * 16)]


class Session(C.Structure):
    _fields_ = [("kv_len", C.c_int32), ("eos_allowed", C.c_int32), ("temperature", C.c_float),
                ("top_k", C.c_int32), ("rep_penalty", C.c_float), ("cp_temperature", C.c_float),
                ("cp_top_k", C.c_int32), ("reserved", C.c_int32)]


def _declare(L):
    vp, i32, f32, f64 = C.c_void_p, C.c_int, C.c_float, C.c_double
    L.orc_to_bf16.argtypes = [f64]
    L.orc_to_bf16.restype = C.c_uint16
    L.orc_from_bf16.argtypes = [C.c_uint16]
    L.orc_from_bf16.restype = f64
    L.orc_rmsnorm.argtypes = [vp, vp, i32, f64, vp]
    L.orc_rope.argtypes = [vp, i32, i32, i32, f64]
    L.orc_linear.argtypes = [vp, Lin, i32, i32, i32, vp]
    L.orc_attention.argtypes = [vp, vp, vp, i32, i32, i32, i32, vp]
    L.orc_silu.argtypes = [f64]
    L.orc_silu.restype = f64
    L.orc_quantize_rows.argtypes = [vp, i32, i32, vp, vp]
    L.orc_philox4x32_10.argtypes = [vp, vp, vp]
    L.orc_logf.argtypes = [f32]
    L.orc_logf.restype = f32
    L.orc_uniform.argtypes = [C.c_uint32, C.c_uint32, i32, C.c_uint32, i32]
    L.orc_uniform.restype = f32
    L.orc_sample.argtypes = [vp, i32, i32, C.POINTER(Session), C.c_uint32, C.c_uint32, C.c_uint32, vp, i32,
                             i32]
    L.orc_sample.restype = C.c_int32
    L.orc_frame_step.argtypes = [C.POINTER(Model), i32, vp, vp, i32, vp, vp, vp, vp, vp, vp, vp]
    L.orc_frame_step.restype = i32
    L.orc_feedback.argtypes = [C.POINTER(Model), i32, vp, vp, vp]
    L.orc_talker_prefill.argtypes = [C.POINTER(Model), i32, vp, vp, i32, vp, i32]
    L.orc_talker_prefill.restype = i32


def _p(a):
    return None if a is None else a.ctypes.data


def session_struct(row):
    """A Session from one [8] int32 descriptor row (layout of synth.Sessions.session_array)."""
    row = np.asarray(row, dtype=np.int32)
    f = row.view(np.float32)
    return Session(int(row[0]), int(row[1]), float(f[2]), int(row[3]), float(f[4]), float(f[5]), int(row[6]), 0)


class Oracle:
    """Holds a model (borrowed numpy arrays, kept alive here) for orc_frame_step."""

    def __init__(self, dims, weights, use_int8=False):
        self.L = lib()
        self.dims = dims
        self.w = weights
        self.keep = []
        self.int8 = {}
        if use_int8:
            self.int8 = {n: self.quantize(a) for n, a in weights.items() if self._is_gemm(n)}
        d = dims
        self.cd = Dims(d.hidden, d.n_layers, d.n_q_heads, d.n_kv_heads, d.head_dim, d.ffn, d.vocab0,
                       d.cp_hidden, d.cp_layers, d.cp_n_q_heads, d.cp_n_kv_heads, d.cp_head_dim, d.cp_ffn,
                       d.cp_vocab, d.n_codebooks, d.eos_id, d.n_codes, d.proj_bias, d.rms_eps, d.rope_theta,
                       d.cp_rope_theta)
        m = Model()
        m.d = self.cd
        m.use_int8 = 1 if use_int8 else 0
        talker = (Layer * d.n_layers)(*[self._layer(f"talker.layers.{l}") for l in range(d.n_layers)])
        cp = (Layer * d.cp_layers)(*[self._layer(f"cp.layers.{l}") for l in range(d.cp_layers)])
        self.keep += [talker, cp]
        m.talker = talker
        m.cp = cp
        m.final_norm = self._ptr("talker.final_norm")
        m.head0 = self._lin("talker.codec_head")
        m.proj = self._lin("cp.proj")
        m.proj_b = self._ptr("cp.proj_bias") if d.proj_bias else None
        m.cp_final_norm = self._ptr("cp.final_norm")
        for j in range(1, d.n_codebooks):
            m.cp_head[j] = self._lin(f"cp.heads.{j}")
        for j in range(d.n_codebooks):
            m.embed[j] = self._ptr(f"codec_embed.{j}")
        self.m = m

    @staticmethod
    def _is_gemm(name):
        return name.endswith("_proj") or name in ("talker.codec_head", "cp.proj") or name.startswith("cp.heads.")

    def _ptr(self, name):
        a = np.ascontiguousarray(self.w[name])
        self.keep.append(a)
        return a.ctypes.data

    def _lin(self, name):
        q, s = self.int8.get(name, (None, None))
        return Lin(self._ptr(name), _p(q), _p(s))

    def _layer(self, p):
        return Layer(self._ptr(f"{p}.input_norm"), self._lin(f"{p}.q_proj"), self._lin(f"{p}.k_proj"),
                     self._lin(f"{p}.v_proj"), self._lin(f"{p}.o_proj"), self._ptr(f"{p}.post_attn_norm"),
                     self._lin(f"{p}.gate_proj"), self._lin(f"{p}.up_proj"), self._lin(f"{p}.down_proj"))

    def quantize(self, w):
        w = np.ascontiguousarray(w, dtype=np.uint16)
        N, K = w.shape
        q = np.empty((N, K), dtype=np.int8)
        s = np.empty((N,), dtype=np.float32)
        self.L.orc_quantize_rows(_p(w), N, K, _p(q), _p(s))
        return q, s

    def frame_step(self, sess_rows, kv_list, kv_cap, in_embeds, rng, seen, forced=None, want_logits=True):
        """One frame for B sessions. sess_rows [B][8] int32 (kv_len advanced in
        place), kv_list: per-session [L][2][kv_cap][nkv][hd] uint16 arrays (new
        K/V written in place), rng [B][4] uint32 (frame counter advanced),
        seen [B][words] uint32 (updated). Returns codes [B][16], eos [B],
        logits [B][16][vocab0] float64 (or None)."""
        d = self.dims
        B = sess_rows.shape[0]
        sess = (Session * B)(*[session_struct(sess_rows[b]) for b in range(B)])
        ptrs = (C.c_void_p * B)(*[k.ctypes.data for k in kv_list])
        in_embeds = np.ascontiguousarray(in_embeds, dtype=np.uint16)
        codes = np.zeros((B, d.n_codebooks), dtype=np.int32)
        eos = np.zeros((B,), dtype=np.uint8)
        logits = np.zeros((B, d.n_codebooks, d.vocab0), dtype=np.float64) if want_logits else None
        f = None if forced is None else np.ascontiguousarray(forced, dtype=np.int32)
        rc = self.L.orc_frame_step(C.byref(self.m), B, C.addressof(sess), C.addressof(ptrs), kv_cap,
                                   _p(in_embeds), _p(rng), _p(seen), _p(f), _p(codes), _p(eos), _p(logits))
        if rc != 0:
            raise RuntimeError(f"orc_frame_step failed: {rc}")
        for b in range(B):
            sess_rows[b, 0] = sess[b].kv_len
        return codes, eos, logits

    def talker_prefill(self, sess_rows, kv_list, kv_cap, embeds):
        """Prompt tokens through the Talker layers (no head, no sampling):
        embeds [n_tok][B][hidden] bf16 bits; token t of session b at position
        kv_len_b + t, its K/V written into kv_list[b]; kv_len advanced in
        place by n_tok."""
        B = sess_rows.shape[0]
        n_tok = embeds.shape[0]
        sess = (Session * B)(*[session_struct(sess_rows[b]) for b in range(B)])
        ptrs = (C.c_void_p * B)(*[k.ctypes.data for k in kv_list])
        e = np.ascontiguousarray(embeds, dtype=np.uint16)
        rc = self.L.orc_talker_prefill(C.byref(self.m), B, C.addressof(sess), C.addressof(ptrs), kv_cap, _p(e), n_tok)
        if rc != 0:
            raise RuntimeError(f"orc_talker_prefill failed: {rc}")
        for b in range(B):
            sess_rows[b, 0] = sess[b].kv_len

    def feedback(self, codes, text):
        B = codes.shape[0]
        out = np.zeros((B, self.dims.hidden), dtype=np.float64)
        c = np.ascontiguousarray(codes, dtype=np.int32)
        t = np.ascontiguousarray(text, dtype=np.uint16)
        self.L.orc_feedback(C.byref(self.m), B, _p(c), _p(t), _p(out))
        return out


def kv_cache_from_prefix(prefix, cap):
    """Per-session oracle cache [L][2][cap][nkv][hd] with the prefix copied in."""
    L2, two, n, nkv, hd = prefix.shape
    kv = np.zeros((L2, 2, cap, nkv, hd), dtype=np.uint16)
    kv[:, :, :n] = prefix
    return kv
