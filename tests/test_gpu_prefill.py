"""GPU parity of the Talker prefill (qtts_talker_prefill: chunks of up to
1,024 rows on tcgen05 GEMMs, RoPE/KV append, causal attention) against the
oracle's prompt pass: appended K/V to bf16 rounding at every layer and
position, kv_len advanced by the prompt length, and the first decode frames
after the prompt within the logit tolerance. Covers ragged prefixes across
page boundaries, chunks spanning several 128-row tiles with a ragged tail,
prompts longer than one chunk, prompts split across calls, INT8 models (whose
prefill stays BF16), full widths with several tiles, and the full model."""
import numpy as np
import pytest
import torch

from codebook_decode_gb300 import configs, qtts, synth
from codebook_decode_gb300.engine import to_dev_u16
from gpu_helpers import TOL_BF16, TOL_INT8, ParityRun, free

pytestmark = pytest.mark.gpu

TINY = configs.TINY


@pytest.fixture(scope="module")
def tiny_w():
    return synth.make_weights(TINY, 1000)


def sessions(d, B, prefixes, frames):
    return synth.Sessions(d, B, prefixes[:B], [0] * B, frames, 2100 + B, temperature=0.9, top_k=50,
                          rep_penalty=1.05)


@pytest.mark.parametrize("B,n_tok,int8", [(1, 20, False), (3, 37, False), (9, 18, False), (9, 17, True),
                                         (2, 19, True), (3, 300, False), (1, 1100, False)])
def test_prefill_matches_oracle(tiny_w, B, n_tok, int8):
    """(3, 300): 900 rows, 8 row tiles with a ragged tail; (1, 1100): two
    chunks (1,024 + 76 tokens)."""
    prefixes = [5, 16, 31, 0, 44, 9, 15, 33, 2]
    s = sessions(TINY, B, prefixes, n_tok + 3)
    run = ParityRun(TINY, tiny_w, s, n_tok + 2, shuffle=True, int8=int8)  # room for prompt + 2 frames
    try:
        e = s.prompt_embeds(n_tok)
        run.eng.prefill(to_dev_u16(e, run.eng.dev))
        rc, derr = run.eng.status()
        assert rc == 0 and derr == 0, (rc, derr)
        run.O.talker_prefill(run.rows, run.kv, run.cap, e)
        run.check_state()
        run.check_kv()
        # the frames after the prompt read its cache
        run.run(frames=2)
        assert run.max_rel() < (TOL_INT8 if int8 else TOL_BF16), run.max_rel()
        assert run.confident_agree == run.confident
        run.check_state()
        run.check_kv()
    finally:
        free(run)


@pytest.mark.parametrize("split", [None, 7, 1])
def test_prefill_in_chunks(tiny_w, split):
    """One call of 19 tokens, or calls of 7 + 12 or 1 + 18 (different pass
    sizes, so different GEMV row counts and paths), all leave the oracle's
    cache and state (the oracle pass is chunk-invariant by its pins)."""
    s = sessions(TINY, 3, [4, 17, 30], 22)
    e = s.prompt_embeds(19)
    run = ParityRun(TINY, tiny_w, s, 20, shuffle=True)
    try:
        if split is None:
            run.eng.prefill(to_dev_u16(e, run.eng.dev))
        else:
            run.eng.prefill(to_dev_u16(e[:split], run.eng.dev))
            run.eng.prefill(to_dev_u16(e[split:], run.eng.dev))
        assert run.eng.status() == (0, 0)
        run.O.talker_prefill(run.rows, run.kv, run.cap, e)
        run.check_state()
        run.check_kv()
    finally:
        free(run)


def test_prefill_refused_inside_a_split_frame(tiny_w):
    s = sessions(TINY, 1, [8], 4)
    run = ParityRun(TINY, tiny_w, s, 1, shuffle=False)
    try:
        eng = run.eng
        emb = to_dev_u16(s.in_embeds(0), eng.dev)
        qtts.qtts_frame_talker(eng.m, eng.B, eng.sess, eng.bt, eng.bt_stride, emb, eng.rng, eng.seen, None,
                               eng.codes, eng.eos, None)
        e = to_dev_u16(s.prompt_embeds(2), eng.dev)
        with pytest.raises(RuntimeError):
            eng.prefill(e)
        qtts.qtts_frame_cp(eng.m, eng.B, eng.sess, eng.bt, eng.bt_stride, emb, eng.rng, eng.seen, None, eng.codes,
                           eng.eos, None)
        torch.cuda.synchronize()
        assert eng.status() == (0, 0)
    finally:
        free(run)


def test_full_size_prefill(tiny_w):
    """Full widths and depth, B = 2, a 40-token prompt: the cache of the first
    and last layers against the oracle, then one frame's logits."""
    d = configs.FULL
    w = synth.make_weights(d, 1001)
    s = sessions(d, 2, [128, 77], 44)
    run = ParityRun(d, w, s, 42, shuffle=True)
    try:
        e = s.prompt_embeds(40)
        run.eng.prefill(to_dev_u16(e, run.eng.dev))
        assert run.eng.status() == (0, 0)
        run.O.talker_prefill(run.rows, run.kv, run.cap, e)
        run.check_state()
        run.check_kv(layers=[0, d.n_layers - 1])
        run.run(frames=1)
        assert run.max_rel() < TOL_BF16, run.max_rel()
    finally:
        free(run)


def test_full_width_prefill_several_tiles():
    """Full widths with 2 Talker layers, B = 2 x 160 tokens: 320 rows over 3
    row tiles (the last half full) and every weight tile of the full widths;
    the cache at both layers against the oracle, then one frame's logits."""
    d = configs.Dims(**{**configs.FULL.as_dict(), "n_layers": 2})
    w = synth.make_weights(d, 1002)
    s = sessions(d, 2, [100, 37], 164)
    run = ParityRun(d, w, s, 162, shuffle=True)
    try:
        e = s.prompt_embeds(160)
        run.eng.prefill(to_dev_u16(e, run.eng.dev))
        assert run.eng.status() == (0, 0)
        run.O.talker_prefill(run.rows, run.kv, run.cap, e)
        run.check_state()
        run.check_kv()
        run.run(frames=1)
        assert run.max_rel() < TOL_BF16, run.max_rel()
    finally:
        free(run)


@pytest.mark.parametrize("B,n_tok", [(3, 1), (32, 32), (32, 33), (2, 0)])
def test_prefill_edge_sizes(tiny_w, B, n_tok):
    """One prompt token (the one-row attention kernel), the largest chunk
    (32 sessions x 32 tokens = 1024 rows), one row past it (a second chunk of
    32 rows), and an empty prompt (nothing changes)."""
    prefixes = [(7 * b + 3) % 50 for b in range(B)]
    s = sessions(TINY, B, prefixes * 1, max(n_tok, 1) + 3)
    run = ParityRun(TINY, tiny_w, s, max(n_tok, 1) + 2, shuffle=True, max_batch=B)
    try:
        e = s.prompt_embeds(n_tok) if n_tok else np.zeros((0, B, TINY.hidden), dtype=np.uint16)
        sess0 = run.eng.sess.clone()
        run.eng.prefill(to_dev_u16(e, run.eng.dev))
        assert run.eng.status() == (0, 0)
        if n_tok == 0:
            assert torch.equal(run.eng.sess, sess0)
        run.O.talker_prefill(run.rows, run.kv, run.cap, e)
        run.check_state()
        if n_tok:
            run.check_kv()
        run.run(frames=1)
        assert run.max_rel() < TOL_BF16, run.max_rel()
        run.check_kv()
    finally:
        free(run)


def test_prefill_device_errors_leave_state(tiny_w):
    """A block-table entry outside the pool, or a prompt past max_context:
    the device error word says which, kv_len and every cached K/V stay as
    they were, and a valid prompt after it matches the oracle."""
    s = sessions(TINY, 2, [20, 9], 12)
    run = ParityRun(TINY, tiny_w, s, 10, shuffle=True)
    try:
        eng = run.eng
        e = s.prompt_embeds(6)
        e_d = to_dev_u16(e, eng.dev)
        sess0 = eng.sess.clone()
        kv0 = [[eng.read_kv(b, l, run.cap) for l in range(TINY.n_layers)] for b in range(2)]
        bt_bad = eng.bt.clone()
        bt_bad[0, 1] = 10 ** 6  # positions 16-31: session 0's prompt (20..25) writes there
        qtts.qtts_talker_prefill(eng.m, 2, eng.sess, bt_bad, eng.bt_stride, e_d, 6, None)
        assert eng.status() == (qtts.QTTS_E_DEVICE, qtts.QTTS_DEV_BAD_PAGE)
        assert torch.equal(eng.sess, sess0)
        too_long = eng.sess.clone()
        too_long[0, 0] = run.cap - 3  # kv_len + 6 > max_context
        qtts.qtts_talker_prefill(eng.m, 2, too_long, eng.bt, eng.bt_stride, e_d, 6, None)
        assert eng.status() == (qtts.QTTS_E_DEVICE, qtts.QTTS_DEV_BAD_SESSION)
        assert int(too_long[0, 0]) == run.cap - 3
        for b in range(2):
            for l in range(TINY.n_layers):
                k, v = eng.read_kv(b, l, run.cap)
                assert np.array_equal(k, kv0[b][l][0]) and np.array_equal(v, kv0[b][l][1]), (b, l)
        eng.prefill(e_d)
        assert eng.status() == (0, 0)
        run.O.talker_prefill(run.rows, run.kv, run.cap, e)
        run.check_state()
        run.check_kv()
    finally:
        free(run)
