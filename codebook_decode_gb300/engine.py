"""Host-side helper: set a model up from named weights and run frames through
the C ABI. Marshalling only; the arithmetic is in libqtts.so.

torch provides device memory and streams.
"""
import numpy as np
import torch

from . import qtts
from .configs import PAGE_SIZE


def make_config(d, max_batch=32, max_context=2048, pool_pages=4096):
    c = qtts.Config()
    for k in ("hidden", "n_layers", "n_q_heads", "n_kv_heads", "head_dim", "ffn", "vocab0", "cp_hidden",
              "cp_layers", "cp_n_q_heads", "cp_n_kv_heads", "cp_head_dim", "cp_ffn", "cp_vocab", "n_codebooks",
              "eos_id", "n_codes", "proj_bias"):
        setattr(c, k, int(getattr(d, k)))
    c.rms_eps = d.rms_eps
    c.rope_theta = d.rope_theta
    c.cp_rope_theta = d.cp_rope_theta
    c.page_size = PAGE_SIZE
    c.max_batch = max_batch
    c.max_context = max_context
    c.kv_pool_pages = pool_pages
    return c


def to_dev_u16(a, dev):
    """host uint16 numpy -> device int16 tensor holding the same bits."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev)


def to_dev_i32(a, dev):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int32)).to(dev)


class Engine:
    """One model on one GPU plus the device-side state of a batch of sessions."""

    def __init__(self, dims, weights, max_batch=32, max_context=2048, pool_pages=4096, device=0, int8=False):
        self.d = dims
        self.device = device
        self.m = qtts.qtts_create(make_config(dims, max_batch, max_context, pool_pages), device)
        try:
            qtts.qtts_load_weights(self.m, weights)
            if int8:
                qtts.qtts_quantize_int8(self.m)
        except Exception:
            qtts.qtts_destroy(self.m)
            self.m = None
            raise
        self.dev = torch.device("cuda", device)
        self.page_ids = None

    def close(self):
        if self.m is not None:
            qtts.qtts_destroy(self.m)
            self.m = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def setup_sessions(self, sess, capacity_tokens, shuffle=True, perm_seed=0):
        """Allocate pages for every session (shuffled across the pool when
        asked), write the synthetic prefix K/V and upload the per-session
        state. capacity_tokens: tokens each session may hold."""
        d = self.d
        B = sess.B
        per = (capacity_tokens + PAGE_SIZE - 1) // PAGE_SIZE
        ids = np.zeros(B * per, dtype=np.int32)
        qtts.qtts_kv_alloc_pages(self.m, ids)
        self.page_ids = ids.copy()
        if shuffle:
            np.random.default_rng(perm_seed).shuffle(ids)
        bt = ids.reshape(B, per).copy()
        for b in range(B):
            kv = sess.prefix_kv(b)  # [L][2][n][nkv][hd]
            n = kv.shape[2]
            for l in range(d.n_layers):
                qtts.qtts_kv_write(self.m, l, n, bt[b], np.ascontiguousarray(kv[l, 0]), np.ascontiguousarray(kv[l, 1]))
        self.B = B
        self.bt_host = bt
        self.bt_stride = per
        self.bt = torch.from_numpy(bt).to(self.dev)
        self.sess = torch.from_numpy(sess.session_array()).to(self.dev)
        self.rng = to_dev_i32(sess.rng_state(), self.dev)
        self.seen = to_dev_i32(sess.seen_bitmap(), self.dev)
        self.codes = torch.zeros(B, 16, dtype=torch.int32, device=self.dev)
        self.eos = torch.zeros(B, dtype=torch.uint8, device=self.dev)
        self.logits = torch.zeros(B, 16, d.vocab0, dtype=torch.float32, device=self.dev)

    def release_pages(self):
        if self.page_ids is not None:
            qtts.qtts_kv_free_pages(self.m, self.page_ids)
            self.page_ids = None

    def step(self, in_embeds, forced=None, want_logits=True, stream=None):
        """in_embeds: device int16 tensor [B][H] of bf16 bits; forced: device int32 [B][16] or None."""
        qtts.qtts_frame_step(self.m, self.B, self.sess, self.bt, self.bt_stride, in_embeds, self.rng, self.seen,
                             forced, self.codes, self.eos, self.logits if want_logits else None, stream)

    def prefill(self, embeds, stream=None):
        """embeds: device int16 tensor [n_tok][B][H] of bf16 bits: the prompt
        through the Talker, K/V appended, kv_len advanced."""
        qtts.qtts_talker_prefill(self.m, self.B, self.sess, self.bt, self.bt_stride, embeds, int(embeds.shape[0]),
                                 stream)

    def read_kv(self, b, layer, n_tok):
        d = self.d
        k = np.zeros((n_tok, d.n_kv_heads, d.head_dim), dtype=np.uint16)
        v = np.zeros_like(k)
        qtts.qtts_kv_read(self.m, layer, n_tok, self.bt_host[b], k, v)
        return k, v

    def status(self):
        return qtts.qtts_frame_status(self.m, raise_on_error=False)
