"""GPU: the frame split into its Talker and Code-Predictor halves
(qtts_frame_talker + qtts_frame_cp) and the multi-frame loop with on-device
feedback (qtts_frame_steps) against the oracle (logits, sampled codes bit
exact on the GPU's logits, state, cache), and bit for bit against the
one-call frame (qtts_frame_step) and frame + qtts_feedback_embed called frame
by frame."""
import numpy as np
import pytest
import torch

from codebook_decode_gb300 import configs, qtts, synth
from codebook_decode_gb300.engine import to_dev_i32, to_dev_u16
from gpu_helpers import TOL_BF16, ParityRun, free

pytestmark = pytest.mark.gpu

TINY = configs.TINY


@pytest.fixture(scope="module")
def tiny_w():
    return synth.make_weights(TINY, 1000)


def sessions(B, frames):
    return synth.Sessions(TINY, B, [7, 20, 33, 3, 16][:B], [0] * B, frames, 2100 + B, temperature=0.9, top_k=50,
                          rep_penalty=1.05)


def snapshot(e):
    return [t.cpu().numpy().copy() for t in (e.codes, e.eos, e.logits, e.sess, e.rng, e.seen)]


@pytest.mark.parametrize("forced", [False, True])
def test_talker_then_cp_equals_frame(tiny_w, forced):
    outs = []
    for split in (False, True):
        s = sessions(4, 3)
        run = ParityRun(TINY, tiny_w, s, 3)
        e = run.eng
        try:
            res = []
            for f in range(3):
                emb = to_dev_u16(s.in_embeds(f), e.dev)
                frc = to_dev_i32(s.forced_codes(f), e.dev) if forced else None
                if split:
                    args = (e.m, e.B, e.sess, e.bt, e.bt_stride, emb, e.rng, e.seen, frc, e.codes, e.eos, e.logits)
                    qtts.qtts_frame_talker(*args)
                    qtts.qtts_frame_cp(*args)
                else:
                    e.step(emb, frc)
                assert e.status() == (0, 0)
                res.append(snapshot(e))
            outs.append(res)
        finally:
            free(run)
    for a, b in zip(outs[0], outs[1]):
        for x, y in zip(a, b):
            assert np.array_equal(x, y)


def test_cp_half_needs_talker_half(tiny_w):
    s = sessions(2, 1)
    run = ParityRun(TINY, tiny_w, s, 1)
    e = run.eng
    try:
        with pytest.raises(qtts.QttsError) as err:
            qtts.qtts_frame_cp(e.m, e.B, e.sess, e.bt, e.bt_stride, None, e.rng, e.seen, None, e.codes, e.eos)
        assert err.value.code == qtts.QTTS_E_STATE
    finally:
        free(run)


@pytest.mark.parametrize("forced", [False, True])
def test_frame_steps_equals_frame_and_feedback_loop(tiny_w, forced):
    n = 4
    outs = []
    for fused in (False, True):
        s = sessions(3, n)
        run = ParityRun(TINY, tiny_w, s, n)
        e = run.eng
        try:
            text = to_dev_u16(np.stack([s.text_embeds(f) for f in range(n)]), e.dev)
            frc = to_dev_i32(np.stack([s.forced_codes(f) for f in range(n)]), e.dev) if forced else None
            emb0 = to_dev_u16(s.in_embeds(0), e.dev)
            codes = torch.zeros(n, e.B, 16, dtype=torch.int32, device=e.dev)
            eos = torch.zeros(n, e.B, dtype=torch.uint8, device=e.dev)
            if fused:
                qtts.qtts_frame_steps(e.m, n, e.B, e.sess, e.bt, e.bt_stride, emb0, text, e.rng, e.seen, frc, codes,
                                      eos, None)
            else:
                cur = emb0
                nxt = torch.empty_like(emb0)
                for f in range(n):
                    qtts.qtts_frame_step(e.m, e.B, e.sess, e.bt, e.bt_stride, cur, e.rng, e.seen,
                                         frc[f] if forced else None, codes[f], eos[f], None)
                    qtts.qtts_feedback_embed(e.m, e.B, frc[f] if forced else codes[f], text[f], nxt)
                    cur, nxt = nxt, cur.clone()
            assert e.status() == (0, 0)
            outs.append([codes.cpu().numpy(), eos.cpu().numpy(), e.sess.cpu().numpy(), e.rng.cpu().numpy(),
                         e.seen.cpu().numpy()])
        finally:
            free(run)
    for x, y in zip(outs[0], outs[1]):
        assert np.array_equal(x, y)


@pytest.mark.parametrize("free_run", [False, True])
def test_split_halves_match_oracle(tiny_w, free_run):
    """qtts_frame_talker then qtts_frame_cp, frame by frame, against the
    oracle: logits, every sampled code, state and cache."""
    s = sessions(4, 3)
    run = ParityRun(TINY, tiny_w, s, 3).run(free=free_run, split=True)
    try:
        assert run.max_rel() < TOL_BF16, run.max_rel()
        assert run.codes_checked == 3 * 4 * 16
        run.check_state()
        run.check_kv()
    finally:
        free(run)


@pytest.mark.parametrize("forced", [False, True])
def test_frame_steps_match_oracle(tiny_w, forced):
    """qtts_frame_steps over n frames with the feedback built on the device,
    against the oracle run frame by frame on inputs text + sum_j E_j[c_j] of
    the codes each frame committed (the forced ones under teacher forcing,
    else the GPU's own): every frame's logits, its sampled codes bit exact on
    those logits, then state and cache."""
    n = 4
    s = sessions(3, n)
    run = ParityRun(TINY, tiny_w, s, n)
    e = run.eng
    try:
        text = np.stack([s.text_embeds(f) for f in range(n)])
        frc = np.stack([s.forced_codes(f) for f in range(n)]) if forced else None
        codes = torch.zeros(n, e.B, 16, dtype=torch.int32, device=e.dev)
        eos = torch.zeros(n, e.B, dtype=torch.uint8, device=e.dev)
        logits = torch.zeros(n, e.B, 16, TINY.vocab0, dtype=torch.float32, device=e.dev)
        qtts.qtts_frame_steps(e.m, n, e.B, e.sess, e.bt, e.bt_stride, to_dev_u16(s.in_embeds(0), e.dev),
                              to_dev_u16(text, e.dev), e.rng, e.seen,
                              to_dev_i32(frc, e.dev) if forced else None, codes, eos, logits)
        assert e.status() == (0, 0)
        codes, eos, logits = codes.cpu().numpy(), eos.cpu().numpy(), logits.cpu().numpy()
        emb = s.in_embeds(0)
        for f in range(n):
            committed = frc[f] if forced else codes[f]
            rng0, seen0 = run.rng.copy(), run.seen.copy()
            run.check_sampled(logits[f], codes[f], eos[f], rng0, seen0)
            _, _, ref = run.O.frame_step(run.rows, run.kv, run.cap, emb, run.rng, run.seen, forced=committed)
            run.compare_logits(f, logits[f].astype(np.float64), ref)
            emb = synth.bf16_bits(run.O.feedback(committed, text[f]).astype(np.float32))
        assert run.max_rel() < TOL_BF16, run.max_rel()
        run.check_state()
        run.check_kv()
    finally:
        free(run)
