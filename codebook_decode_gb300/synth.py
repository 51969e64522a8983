"""Seeded synthetic inputs shared by the tests, the oracle driver and bench.py.

This module draws random numbers and stores them as bf16 / int32; it holds
none of the frame's arithmetic. Every tensor is drawn from its own stream,
seeded by (seed, crc32(name)), so any subset can be regenerated in any order.

Recipe (no trained weights exist here, and none are needed to exercise the
arithmetic):
  * Linear weights and embedding tables: N(0, 0.02), rounded to bf16 (RNE).
  * RMSNorm gains: 1 + N(0, 0.02) (pure N(0, 0.02) gains would shrink every
    normalised activation ~50x).
  * Prefix K/V: N(0, 1) bf16, K taken as already rotated.
  * Talker input embeddings: N(0, 0.08) bf16, the spread of a sum of 16
    N(0, 0.02) code embeddings plus text.
  * Teacher-forced codes: uniform in [0, n_codes).
"""
import os
import zlib
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from .configs import Dims, PAGE_SIZE


def bf16_bits(a):
    """float32 array -> uint16 bf16 bit patterns, round to nearest even
    (finite inputs)."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    t = u >> np.uint32(16)
    t &= np.uint32(1)
    t += np.uint32(0x7FFF)
    t += u
    t >>= np.uint32(16)
    return t.astype(np.uint16)


def bf16_to_f32(h):
    """uint16 bf16 bit patterns -> float32 (exact)."""
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _rng(seed, name):
    return np.random.default_rng([int(seed), zlib.crc32(name.encode())])


def tensor_specs(d: Dims):
    """Every named tensor the model has: (name, shape, kind)."""
    out = []

    def layer(prefix, H, nq, nkv, hd, F):
        out.extend([
            (f"{prefix}.input_norm", (H,), "gain"),
            (f"{prefix}.q_proj", (nq * hd, H), "weight"),
            (f"{prefix}.k_proj", (nkv * hd, H), "weight"),
            (f"{prefix}.v_proj", (nkv * hd, H), "weight"),
            (f"{prefix}.o_proj", (H, nq * hd), "weight"),
            (f"{prefix}.post_attn_norm", (H,), "gain"),
            (f"{prefix}.gate_proj", (F, H), "weight"),
            (f"{prefix}.up_proj", (F, H), "weight"),
            (f"{prefix}.down_proj", (H, F), "weight"),
        ])

    for l in range(d.n_layers):
        layer(f"talker.layers.{l}", d.hidden, d.n_q_heads, d.n_kv_heads, d.head_dim, d.ffn)
    out.append(("talker.final_norm", (d.hidden,), "gain"))
    out.append(("talker.codec_head", (d.vocab0, d.hidden), "weight"))
    for j in range(d.n_codebooks):
        rows = d.vocab0 if j == 0 else d.cp_vocab
        out.append((f"codec_embed.{j}", (rows, d.hidden), "weight"))
    out.append(("cp.proj", (d.cp_hidden, d.hidden), "weight"))
    if d.proj_bias:
        out.append(("cp.proj_bias", (d.cp_hidden,), "weight"))
    for l in range(d.cp_layers):
        layer(f"cp.layers.{l}", d.cp_hidden, d.cp_n_q_heads, d.cp_n_kv_heads, d.cp_head_dim, d.cp_ffn)
    out.append(("cp.final_norm", (d.cp_hidden,), "gain"))
    for j in range(1, d.n_codebooks):
        out.append((f"cp.heads.{j}", (d.cp_vocab, d.cp_hidden), "weight"))
    return out


def make_tensor(seed, name, shape, kind, std=0.02):
    r = _rng(seed, name)
    a = r.standard_normal(size=shape, dtype=np.float32)
    a *= np.float32(std)
    if kind == "gain":
        a += np.float32(1.0)
    return bf16_bits(a)


def make_weights(d: Dims, seed: int, std=0.02, threads=None):
    """dict name -> uint16 bf16 array, N(0, std) weights, 1 + N(0, std) gains.
    Each tensor has its own stream, so drawing them on several threads gives
    the same values as drawing them one after another."""
    specs = tensor_specs(d)
    threads = threads or min(16, os.cpu_count() or 1)
    with ThreadPoolExecutor(max_workers=threads) as ex:
        arrs = list(ex.map(lambda t: make_tensor(seed, t[0], t[1], t[2], std), specs))
    return {t[0]: a for t, a in zip(specs, arrs)}


class Sessions:
    """Per-session synthetic state for one workload (all host numpy)."""

    def __init__(self, d: Dims, batch, prefix_lens, offsets, frames, seed,
                 temperature=0.0, top_k=1, rep_penalty=1.0, cp_temperature=None, cp_top_k=None,
                 eos_allowed=0):
        self.d = d
        self.B = batch
        self.prefix_lens = np.asarray(prefix_lens, dtype=np.int32)
        self.offsets = np.asarray(offsets, dtype=np.int32)
        # tokens cached when the run starts: the prompt prefix plus the frames
        # this session had already generated (its staggered offset)
        self.kv_len0 = self.prefix_lens + self.offsets
        self.frames = frames
        self.seed = seed
        self.temperature = float(temperature)
        self.top_k = int(top_k)
        self.rep_penalty = float(rep_penalty)
        self.cp_temperature = float(temperature if cp_temperature is None else cp_temperature)
        self.cp_top_k = int(top_k if cp_top_k is None else cp_top_k)
        self.eos_allowed = int(eos_allowed)

    # -- prefix KV: per session, per layer, K and V [len][nkv][hd] bf16
    def prefix_kv(self, b):
        d = self.d
        n = int(self.kv_len0[b])
        r = _rng(self.seed, f"prefix_kv.{b}")
        a = r.standard_normal(size=(d.n_layers, 2, n, d.n_kv_heads, d.head_dim), dtype=np.float32)
        return bf16_bits(a)

    def in_embeds(self, frame):
        d = self.d
        r = _rng(self.seed, f"in_embeds.{frame}")
        a = r.standard_normal(size=(self.B, d.hidden), dtype=np.float32) * np.float32(0.08)
        return bf16_bits(a)

    def prompt_embeds(self, n_tok, chunk=0):
        """Prompt embeddings for a Talker prefill: [n_tok][B][hidden] bf16
        bits, like the frame inputs (chunk: which prompt chunk, for distinct
        draws)."""
        d = self.d
        r = _rng(self.seed, f"prompt_embeds.{chunk}")
        a = r.standard_normal(size=(n_tok, self.B, d.hidden), dtype=np.float32) * np.float32(0.08)
        return bf16_bits(a)

    def text_embeds(self, frame):
        d = self.d
        r = _rng(self.seed, f"text_embeds.{frame}")
        a = r.standard_normal(size=(self.B, d.hidden), dtype=np.float32) * np.float32(0.02)
        return bf16_bits(a)

    def forced_codes(self, frame):
        r = _rng(self.seed, f"forced.{frame}")
        return r.integers(0, self.d.n_codes, size=(self.B, self.d.n_codebooks), dtype=np.int32)

    def rng_state(self):
        """[B][4] uint32: Philox key (seed-derived), frame counter = offset, 0."""
        out = np.zeros((self.B, 4), dtype=np.uint32)
        for b in range(self.B):
            out[b, 0] = np.uint32((3000 + self.seed) & 0xFFFFFFFF)
            out[b, 1] = np.uint32(b)
            out[b, 2] = np.uint32(self.offsets[b])
        return out

    def seen_bitmap(self):
        """[B][ceil(vocab0/32)] uint32: codes of the `offset` frames already generated."""
        d = self.d
        words = (d.vocab0 + 31) // 32
        out = np.zeros((self.B, words), dtype=np.uint32)
        for b in range(self.B):
            r = _rng(self.seed, f"history.{b}")
            hist = r.integers(0, d.n_codes, size=int(self.offsets[b]))
            for c in hist:
                out[b, c >> 5] |= np.uint32(1 << (int(c) & 31))
        return out

    def session_array(self):
        """[B][8] int32 view of the per-session descriptor (kv_len = prefix + offset)."""
        a = np.zeros((self.B, 8), dtype=np.int32)
        f = a.view(np.float32)
        for b in range(self.B):
            a[b, 0] = int(self.kv_len0[b])
            a[b, 1] = self.eos_allowed
            f[b, 2] = self.temperature
            a[b, 3] = self.top_k
            f[b, 4] = self.rep_penalty
            f[b, 5] = self.cp_temperature
            a[b, 6] = self.cp_top_k
        return a

    def page_tables(self, capacity_tokens, shuffle, pool_pages=None):
        """Block tables [B][max_pages] int32 and the pool size. Pages are
        shuffled across the pool when `shuffle` (seeded)."""
        max_pages = (capacity_tokens + PAGE_SIZE - 1) // PAGE_SIZE
        total = self.B * max_pages
        pool = pool_pages or total
        ids = np.arange(pool, dtype=np.int32)
        if shuffle:
            _rng(self.seed, "pages").shuffle(ids)
        return ids[:total].reshape(self.B, max_pages).copy(), pool


def make_sessions(wl, frames=None):
    """Sessions for a configs.Workload (prefix lengths and offsets drawn from its recipe)."""
    d = wl.dims
    seed = 2000 + wl.seed
    r = _rng(seed, "lengths")

    def draw(spec):
        if spec[0] == "fixed":
            return np.full(wl.batch, spec[1], dtype=np.int32)
        return r.integers(spec[1], spec[2] + 1, size=wl.batch).astype(np.int32)

    lens = draw(wl.prefix)
    offs = draw(wl.offset)
    return Sessions(d, wl.batch, lens, offs, frames or wl.frames, seed, temperature=wl.temperature,
                    top_k=wl.top_k, rep_penalty=wl.rep_penalty)
