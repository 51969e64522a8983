"""qtts_kv_write_noalloc, the KV-cache write for callers that may not
allocate device memory (a serving loop that must not trigger cudaFree's
device-wide wait while other sessions' frames run, or code under a memory pool
it does not own). It stages through the library's static device array; here it
must leave the cache exactly as qtts_kv_write leaves it, on two calls in a
row, and refuse writes larger than that array.

This file is collected last on purpose: a run that stops at the first failure
has already run every other test."""
import dataclasses

import numpy as np
import pytest
import torch

from codebook_decode_gb300 import configs, qtts
from codebook_decode_gb300.engine import make_config

pytestmark = pytest.mark.gpu

D = dataclasses.replace(configs.FULL, n_layers=2)  # full-width K/V, two layers keep the model small
MAX_TOK = (4 << 20) // (2 * D.n_kv_heads * D.head_dim * 2)  # tokens that fit the 4 MiB staging array


def kv(rng, n):
    shape = (n, D.n_kv_heads, D.head_dim)
    return (rng.integers(0, 1 << 16, size=shape, dtype=np.uint32).astype(np.uint16),
            rng.integers(0, 1 << 16, size=shape, dtype=np.uint32).astype(np.uint16))


def test_noalloc_write_matches_kv_write_on_two_calls():
    m = qtts.qtts_create(make_config(D, 2, 2048, 300), 0)
    try:
        rng = np.random.default_rng(11)
        stream = torch.cuda.Stream()
        for layer, n_tok in ((1, MAX_TOK), (0, 37)):  # a full-size call, then a small one after it
            npg = (n_tok + 15) // 16
            ids = np.zeros(2 * npg, np.int32)
            qtts.qtts_kv_alloc_pages(m, ids)
            rng.shuffle(ids)
            pages_ref, pages_new = ids[:npg].copy(), ids[npg:].copy()
            k, v = kv(rng, n_tok)
            qtts.qtts_kv_write(m, layer, n_tok, pages_ref, k, v)
            qtts.qtts_kv_write_noalloc(m, layer, n_tok, pages_new, k, v, stream)
            stream.synchronize()
            out = []
            for pages in (pages_ref, pages_new):
                kk = np.zeros_like(k)
                vv = np.zeros_like(v)
                qtts.qtts_kv_read(m, layer, n_tok, pages, kk, vv)
                out.append((kk, vv))
            assert np.array_equal(out[0][0], out[1][0]) and np.array_equal(out[0][1], out[1][1])
            assert np.array_equal(out[1][0], k) and np.array_equal(out[1][1], v)
            qtts.qtts_kv_free_pages(m, ids)
    finally:
        qtts.qtts_destroy(m)


def test_noalloc_write_refuses_more_than_the_static_array():
    m = qtts.qtts_create(make_config(D, 2, 2048, 300), 0)
    try:
        n = MAX_TOK + 1
        ids = np.arange((n + 15) // 16, dtype=np.int32)
        k = np.zeros((n, D.n_kv_heads, D.head_dim), np.uint16)
        with pytest.raises(qtts.QttsError) as e:
            qtts.qtts_kv_write_noalloc(m, 0, n, ids, k, k)
        assert e.value.code == qtts.QTTS_E_INVALID and "static buffer" in str(e.value)
    finally:
        qtts.qtts_destroy(m)
