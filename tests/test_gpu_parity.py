"""GPU parity: the CUDA frame through the C ABI against the CPU oracle on the
same seeded inputs. Gates: teacher-forced logits within 1.0% (BF16) / 1.5%
(INT8) of the logit scale per row, 100% raw-argmax agreement where the
oracle's top-2 margin exceeds 1, state (kv_len, frame counter, seen set)
exact, cache contents to bf16 rounding, INT8 weights bit exact, and the codes
each frame samples (and its EOS flags) bit exact against the oracle's sampler
fed that frame's own logits (ParityRun.check_sampled), teacher forced and
free running."""
import ctypes as C

import numpy as np
import pytest
import torch

from codebook_decode_gb300 import configs, qtts, synth
from codebook_decode_gb300.engine import Engine, to_dev_i32, to_dev_u16
from gpu_helpers import TOL_BF16, TOL_INT8, ParityRun, free
from oracle import orc

pytestmark = pytest.mark.gpu

TINY = configs.TINY


@pytest.fixture(scope="module")
def tiny_w():
    return synth.make_weights(TINY, 1000)


def tiny_sessions(B, prefix, offsets=None, T=0.0, k=1, r=1.0, frames=4, eos=0):
    return synth.Sessions(TINY, B, prefix, offsets if offsets is not None else [0] * B, frames, 2000 + B,
                          temperature=T, top_k=k, rep_penalty=r, eos_allowed=eos)


# --------------------------------------------------------------------------
# tiny model (the small workload: 2-layer Talker, 1-layer Code Predictor)
# --------------------------------------------------------------------------

def test_tiny_config_teacher_forced_16_frames(tiny_w):
    """B=1, 32-token prefix, pages in order, 16 teacher-forced greedy frames."""
    s = synth.make_sessions(configs.WORKLOADS["tiny"])
    run = ParityRun(TINY, tiny_w, s, 16, shuffle=False).run()
    try:
        assert run.max_rel() < TOL_BF16, run.max_rel()
        assert run.confident_agree == run.confident
        run.check_state()
        run.check_kv()
    finally:
        free(run)


def test_tiny_ragged_batch_shuffled_pages(tiny_w):
    """B=5, ragged prefixes across page boundaries (0, 1, 15, 16, 45 tokens),
    staggered offsets, shuffled pages, sampling parameters on."""
    s = tiny_sessions(5, [0, 1, 15, 16, 45], [0, 3, 1, 7, 2], T=0.9, k=50, r=1.05)
    run = ParityRun(TINY, tiny_w, s, 4, shuffle=True).run()
    try:
        assert run.max_rel() < TOL_BF16, run.max_rel()
        assert run.confident_agree == run.confident
        run.check_state()
        run.check_kv()
    finally:
        free(run)


def test_tiny_max_batch_long_context(tiny_w):
    """B=32 at the batch limit, contexts up to 400 tokens (several attention
    splits per session)."""
    lens = list(np.random.default_rng(3).integers(1, 400, 32))
    s = tiny_sessions(32, lens, T=0.9, k=50, r=1.05)
    run = ParityRun(TINY, tiny_w, s, 2, shuffle=True).run()
    try:
        assert run.max_rel() < TOL_BF16, run.max_rel()
        assert run.confident_agree == run.confident
        run.check_state()
        run.check_kv(layers=[0, 1])
    finally:
        free(run)


@pytest.mark.parametrize("B,tc_min,ks_min,int8", [(1, 1, 65, False), (3, 1, 1, False), (9, 65, 65, False),
                                                  (9, 8, 65, False), (9, 8, 8, False), (9, 8, 65, True),
                                                  (9, 8, 8, True), (2, 1, 1, True)])
def test_gemv_path_choice(tiny_w, B, tc_min, ks_min, int8):
    """Every GEMV path of the frame kernel matches the oracle, BF16 and INT8
    weights: tensor cores from one activation row up (tc_min 1) with one
    K-slice (ks_min 65) or K split across CTAs (ks_min <= rows), and the
    CUDA-core paths alone (tc_min 65); the Talker stays in the frame kernel
    at every batch size here."""
    s = tiny_sessions(B, [7, 33, 16, 2, 40, 1, 15, 64, 30][:B], [0, 2, 5, 1, 3, 0, 4, 6, 2][:B], T=0.9, k=50, r=1.05)
    run = ParityRun(TINY, tiny_w, s, 3, shuffle=True, int8=int8, tc_min_rows=tc_min, ksplit_min_rows=ks_min,
                    chunk_talker_min_b=33).run()
    try:
        assert run.max_rel() < (TOL_INT8 if int8 else TOL_BF16), run.max_rel()
        assert run.confident_agree == run.confident
        run.check_state()
    finally:
        free(run)


@pytest.mark.parametrize("B,free_run,split", [(8, False, False), (9, True, False), (12, False, True), (3, False, False)])
def test_chunk_kernel_talker_matches_oracle(tiny_w, B, free_run, split):
    """Frames whose Talker runs on the tensor-core chunk kernels (the option
    at 1 for B = 3, at 8 otherwise) and the rest in the frame kernel: logits,
    codes and EOS flags, K/V and state against the oracle, teacher-forced,
    free-running, and as split Talker/CP halves."""
    pre = [7, 33, 16, 2, 40, 1, 15, 64, 30, 5, 21, 48]
    off = [0, 2, 5, 1, 3, 0, 4, 6, 2, 1, 0, 3]
    s = tiny_sessions(B, pre[:B], off[:B], T=0.9, k=50, r=1.05)
    run = ParityRun(TINY, tiny_w, s, 3, shuffle=True, chunk_talker_min_b=1 if B < 8 else 8)
    try:
        run.run(free=free_run, split=split)
        assert run.max_rel() < TOL_BF16, run.max_rel()
        assert run.confident_agree == run.confident
        assert run.codes_checked == 3 * B * 16
        run.check_state()
        run.check_kv()
    finally:
        free(run)


def test_tiny_free_running_vs_oracle(tiny_w):
    """B=5 free running with sampling on: the GPU's own sampled codes feed its
    Code Predictor and seen set; the oracle, forced with those codes, agrees
    on logits and state, and each code is the oracle sampler's on the GPU's
    logits."""
    s = tiny_sessions(5, [0, 1, 15, 16, 45], [0, 3, 1, 7, 2], T=0.9, k=50, r=1.05)
    run = ParityRun(TINY, tiny_w, s, 4, shuffle=True).run(free=True)
    try:
        assert run.max_rel() < TOL_BF16, run.max_rel()
        assert run.codes_checked == 4 * 5 * 16
        run.check_state()
        run.check_kv()
    finally:
        free(run)


def test_tiny_eos_allowed(tiny_w):
    """EOS unmasked in codebook 0, temperature 1.3 without top-k (EOS is
    sampled on some frames): codes and eos_out against the oracle sampler."""
    s = tiny_sessions(6, [3, 9, 17, 30, 2, 11], T=1.3, k=0, r=1.2, eos=1)
    run = ParityRun(TINY, tiny_w, s, 6, shuffle=True).run(free=True)
    try:
        assert run.max_rel() < TOL_BF16, run.max_rel()
        run.check_state()
    finally:
        free(run)


@pytest.mark.parametrize("B,tc_min,ks_min", [(1, 65, 65), (3, 1, 1)])
def test_wait_limit_runs_out_then_recovers(tiny_w, B, tc_min, ks_min):
    """A 1 us limit on every device-side wait: the frame's waits for other
    CTAs' words run out, the frame ends with QTTS_DEV_TIMEOUT (returned as
    QTTS_E_TIMEOUT) instead of hanging, each CTA first draining its own bulk
    copies and MMAs; with the default limit back the same model runs frames
    that match the oracle. CUDA-core path (B=1) and tensor path with K split
    (B=3)."""
    s = tiny_sessions(B, [20, 7, 33][:B], T=0.9, k=50, r=1.05)
    run = ParityRun(TINY, tiny_w, s, 2, tc_min_rows=tc_min, ksplit_min_rows=ks_min)
    try:
        e = run.eng
        assert qtts.qtts_set_option(e.m, qtts.QTTS_OPT_WAIT_LIMIT_US, 1) == 0
        e.step(to_dev_u16(s.in_embeds(0), e.dev), to_dev_i32(s.forced_codes(0), e.dev))
        assert e.status() == (qtts.QTTS_E_TIMEOUT, qtts.QTTS_DEV_TIMEOUT)
        assert qtts.qtts_set_option(e.m, qtts.QTTS_OPT_WAIT_LIMIT_US, 2000000) == 0
        # the abandoned frame may have advanced part of the state: start again from the caller's copy
        e.sess.copy_(torch.from_numpy(s.session_array()).to(e.dev))
        e.rng.copy_(to_dev_i32(s.rng_state(), e.dev))
        e.seen.copy_(to_dev_i32(s.seen_bitmap(), e.dev))
        run.run(2)
        assert run.max_rel() < TOL_BF16, run.max_rel()
        run.check_state()
        run.check_kv()
    finally:
        free(run)


def test_stepwise_equals_persistent(tiny_w):
    """One launch per stage and the persistent single launch give identical bits."""
    outs = []
    for stepwise in (False, True):
        s = tiny_sessions(3, [5, 17, 33], T=0.9, k=50, r=1.05)
        run = ParityRun(TINY, tiny_w, s, 3, stepwise=stepwise)
        try:
            codes, logits = [], []
            for f in range(3):
                run.eng.step(to_dev_u16(s.in_embeds(f), run.eng.dev))  # free running
                assert run.eng.status() == (0, 0)
                codes.append(run.eng.codes.cpu().numpy().copy())
                logits.append(run.eng.logits.cpu().numpy().copy())
            outs.append((np.array(codes), np.array(logits)))
        finally:
            free(run)
    assert np.array_equal(outs[0][0], outs[1][0])
    assert np.array_equal(outs[0][1], outs[1][1])


def test_free_running_is_deterministic_and_valid(tiny_w):
    res = []
    for _ in range(2):
        s = tiny_sessions(4, [8, 9, 30, 2], T=0.9, k=50, r=1.05)
        run = ParityRun(TINY, tiny_w, s, 5)
        try:
            cs = []
            for f in range(5):
                run.eng.step(to_dev_u16(s.in_embeds(f), run.eng.dev))
                assert run.eng.status() == (0, 0)
                cs.append(run.eng.codes.cpu().numpy().copy())
            res.append(np.array(cs))
        finally:
            free(run)
    assert np.array_equal(res[0], res[1])
    c = res[0]
    assert (c >= 0).all() and (c[..., 0] < TINY.n_codes).all() and (c[..., 1:] < TINY.cp_vocab).all()


def test_int8_tiny_parity_and_export(tiny_w):
    s = tiny_sessions(3, [10, 33, 20], T=0.9, k=50, r=1.05)
    run = ParityRun(TINY, tiny_w, s, 3, int8=True).run()
    try:
        assert run.max_rel() < TOL_INT8, run.max_rel()
        assert run.confident_agree == run.confident
        run.check_state()
        for name, arr in tiny_w.items():
            if not orc.Oracle._is_gemm(name):
                continue
            q_ref, s_ref = run.O.int8[name]
            q = np.zeros_like(q_ref)
            sc = np.zeros_like(s_ref)
            qtts.qtts_export_int8(run.eng.m, name, q, sc)
            assert np.array_equal(q, q_ref), name
            assert np.array_equal(sc.view(np.uint32), s_ref.view(np.uint32)), name
    finally:
        free(run)


def test_host_buffer_entry_matches_device_entry(tiny_w):
    s = tiny_sessions(2, [12, 40], T=0.9, k=50, r=1.05)
    run = ParityRun(TINY, tiny_w, s, 1)
    try:
        sess = s.session_array().copy()
        rng = s.rng_state().copy()
        seen = s.seen_bitmap().copy()
        codes = np.zeros((2, 16), np.int32)
        eos = np.zeros(2, np.uint8)
        logits = np.zeros((2, 16, TINY.vocab0), np.float32)
        forced = s.forced_codes(0)
        qtts.qtts_frame_step_host(run.eng.m, 2, sess, run.eng.bt_host, run.eng.bt_stride, s.in_embeds(0), rng, seen,
                                  forced, codes, eos, logits)
        # the same frame through the device entry point on a second model
        run2 = ParityRun(TINY, tiny_w, s, 1)
        try:
            run2.eng.step(to_dev_u16(s.in_embeds(0), run2.eng.dev), to_dev_i32(forced, run2.eng.dev))
            assert run2.eng.status() == (0, 0)
            assert np.array_equal(codes, run2.eng.codes.cpu().numpy())
            assert np.array_equal(logits, run2.eng.logits.cpu().numpy())
            assert np.array_equal(sess, run2.eng.sess.cpu().numpy())
            assert np.array_equal(rng, run2.eng.rng.cpu().numpy().view(np.uint32))
            assert np.array_equal(seen, run2.eng.seen.cpu().numpy().view(np.uint32))
        finally:
            free(run2)
    finally:
        free(run)


def test_feedback_embedding(tiny_w):
    s = tiny_sessions(3, [4, 4, 4])
    run = ParityRun(TINY, tiny_w, s, 1)
    try:
        r = np.random.default_rng(1)
        codes = np.concatenate([r.integers(0, TINY.vocab0, (3, 1)), r.integers(0, TINY.cp_vocab, (3, 15))], 1)
        codes = codes.astype(np.int32)
        text = s.text_embeds(0)
        out = torch.zeros(3, TINY.hidden, dtype=torch.int16, device=run.eng.dev)
        qtts.qtts_feedback_embed(run.eng.m, 3, to_dev_i32(codes, run.eng.dev), to_dev_u16(text, run.eng.dev), out)
        torch.cuda.synchronize()
        got = synth.bf16_to_f32(out.cpu().numpy().view(np.uint16)).astype(np.float64)
        ref = run.O.feedback(codes, text)
        assert np.abs(got - ref).max() <= 2 ** -8 * np.abs(ref).max()
    finally:
        free(run)


# --------------------------------------------------------------------------
# sampler: bit-exact given identical logits
# --------------------------------------------------------------------------

@pytest.mark.parametrize("codebook,T,k,r,eos,V", [
    (0, 0.0, 1, 1.0, 0, 3072), (0, 0.9, 50, 1.05, 0, 3072), (0, 0.9, 50, 1.05, 1, 3072), (0, 1.3, 0, 1.2, 1, 3072),
    (3, 0.9, 50, 1.05, 0, 2048), (15, 0.7, 1, 1.0, 0, 2048), (7, 1.0, 2048, 1.0, 0, 2048), (9, 0.5, 3, 1.0, 0, 2048),
    (0, 0.9, 50, 1.05, 0, 2049),
])
def test_sampler_bit_exact_given_oracle_logits(codebook, T, k, r, eos, V):
    import dataclasses

    from codebook_decode_gb300.engine import make_config
    d = dataclasses.replace(TINY, vocab0=max(V, 2049))
    m = qtts.qtts_create(make_config(d, 32, 64, 4), 0)  # the sampler needs no weights
    try:
        L = orc.lib()
        B = 32
        dev = torch.device("cuda", 0)
        rg = np.random.default_rng(100 + codebook + V)
        logits = (rg.standard_normal((B, V)) * 2.0).astype(np.float32)
        logits[:4, :8] = 3.0                       # exact ties
        logits[4, 100:110] = np.float32(-0.0)      # signed zeros
        logits[5, :] = 0.0
        sess = np.zeros((B, 8), np.int32)
        f = sess.view(np.float32)
        sess[:, 1] = eos
        f[:, 2] = T
        sess[:, 3] = k
        f[:, 4] = r
        f[:, 5] = T
        sess[:, 6] = k
        rng = np.zeros((B, 4), np.uint32)
        rng[:, 0] = rg.integers(0, 2 ** 32, B, dtype=np.uint64).astype(np.uint32)
        rng[:, 1] = np.arange(B)
        rng[:, 2] = rg.integers(0, 1000, B).astype(np.uint32)
        words = (d.vocab0 + 31) // 32
        seen = rg.integers(0, 2 ** 32, (B, words), dtype=np.uint64).astype(np.uint32)
        if d.vocab0 % 32:
            seen[:, words - 1] &= np.uint32((1 << (d.vocab0 % 32)) - 1)
        out = torch.zeros(B, dtype=torch.int32, device=dev)
        qtts.qtts_sample(m, B, codebook, torch.from_numpy(logits).to(dev), V, to_dev_i32(sess, dev),
                         to_dev_i32(rng, dev), to_dev_i32(seen, dev) if codebook == 0 else None, out)
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        for b in range(B):
            S = orc.session_struct(sess[b])
            want = L.orc_sample(logits[b].ctypes.data, V, codebook, C.byref(S), int(rng[b, 0]), int(rng[b, 1]),
                                int(rng[b, 2]), seen[b].ctypes.data if codebook == 0 else None, d.eos_id, d.n_codes)
            assert got[b] == want, (b, got[b], want)
    finally:
        qtts.qtts_destroy(m)


# --------------------------------------------------------------------------
# device-side validation: bad inputs become an error word, never an access
# --------------------------------------------------------------------------

def test_device_side_checks_and_recovery(tiny_w):
    s = tiny_sessions(2, [20, 3], T=0.9, k=50, r=1.05)
    run = ParityRun(TINY, tiny_w, s, 1)
    try:
        eng = run.eng
        emb = to_dev_u16(s.in_embeds(0), eng.dev)
        sess0 = eng.sess.clone()
        # a block-table entry outside the pool
        bt_bad = eng.bt.clone()
        bt_bad[1, 0] = 10 ** 6
        qtts.qtts_frame_step(eng.m, 2, eng.sess, bt_bad, eng.bt_stride, emb, eng.rng, eng.seen, None, eng.codes,
                             eng.eos)
        rc, derr = eng.status()
        assert rc == qtts.QTTS_E_DEVICE and derr == qtts.QTTS_DEV_BAD_PAGE
        assert torch.equal(eng.sess, sess0)  # the frame did nothing
        # negative temperature
        bad = eng.sess.clone()
        bad.view(torch.float32)[0, 2] = -1.0
        qtts.qtts_frame_step(eng.m, 2, bad, eng.bt, eng.bt_stride, emb, eng.rng, eng.seen, None, eng.codes, eng.eos)
        assert eng.status() == (qtts.QTTS_E_DEVICE, qtts.QTTS_DEV_BAD_SAMPLING)
        # teacher-forced code outside its codebook
        forced = torch.zeros(2, 16, dtype=torch.int32, device=eng.dev)
        forced[1, 5] = TINY.cp_vocab
        qtts.qtts_frame_step(eng.m, 2, eng.sess, eng.bt, eng.bt_stride, emb, eng.rng, eng.seen, forced, eng.codes,
                             eng.eos)
        assert eng.status() == (qtts.QTTS_E_DEVICE, qtts.QTTS_DEV_BAD_CODE)
        # kv_len past the block table
        bad = eng.sess.clone()
        bad[0, 0] = eng.bt_stride * 16
        qtts.qtts_frame_step(eng.m, 2, bad, eng.bt, eng.bt_stride, emb, eng.rng, eng.seen, None, eng.codes, eng.eos)
        assert eng.status() == (qtts.QTTS_E_DEVICE, qtts.QTTS_DEV_BAD_SESSION)
        # host-side refusals
        with pytest.raises(qtts.QttsError) as e:
            qtts.qtts_frame_step(eng.m, 0, eng.sess, eng.bt, eng.bt_stride, emb, eng.rng, eng.seen, None, eng.codes,
                                 eng.eos)
        assert e.value.code == qtts.QTTS_E_BATCH
        with pytest.raises(qtts.QttsError) as e:
            qtts.qtts_frame_step(eng.m, 33, eng.sess, eng.bt, eng.bt_stride, emb, eng.rng, eng.seen, None, eng.codes,
                                 eng.eos)
        assert e.value.code == qtts.QTTS_E_BATCH
        # the model still works after the errors
        run.run(1)
        assert run.max_rel() < TOL_BF16
        run.check_state()
    finally:
        free(run)


def test_weight_coverage_checked_both_ways(tiny_w):
    from codebook_decode_gb300.engine import make_config
    for mutate, code in [(lambda w: w.pop("cp.heads.7"), qtts.QTTS_E_MISSING),
                         (lambda w: w.__setitem__("talker.layers.9.q_proj", w["talker.layers.0.q_proj"]),
                          qtts.QTTS_E_UNUSED),
                         (lambda w: w.__setitem__("cp.proj", w["cp.proj"][:, :-8].copy()), qtts.QTTS_E_SHAPE)]:
        w = dict(tiny_w)
        mutate(w)
        m = qtts.qtts_create(make_config(TINY, 2, 64, 8), 0)
        try:
            with pytest.raises(qtts.QttsError) as e:
                qtts.qtts_load_weights(m, w)
            assert e.value.code == code
        finally:
            qtts.qtts_destroy(m)


def test_kv_pool_allocator(tiny_w):
    from codebook_decode_gb300.engine import make_config
    m = qtts.qtts_create(make_config(TINY, 2, 64, 10), 0)
    try:
        ids = np.zeros(7, np.int32)
        qtts.qtts_kv_alloc_pages(m, ids)
        assert len(set(ids.tolist())) == 7 and qtts.qtts_kv_pool_free_count(m) == 3
        with pytest.raises(qtts.QttsError) as e:
            qtts.qtts_kv_alloc_pages(m, np.zeros(4, np.int32))
        assert e.value.code == qtts.QTTS_E_POOL
        qtts.qtts_kv_free_pages(m, ids[:2])
        with pytest.raises(qtts.QttsError):
            qtts.qtts_kv_free_pages(m, ids[:1])  # already free
        assert qtts.qtts_kv_pool_free_count(m) == 5
    finally:
        qtts.qtts_destroy(m)
