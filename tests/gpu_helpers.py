"""Shared driver for the GPU parity tests: run the CUDA frame (through the C
ABI) and the CPU oracle side by side on the same seeded inputs."""
import ctypes as C

import numpy as np
import torch

from codebook_decode_gb300 import qtts
from codebook_decode_gb300.configs import PAGE_SIZE
from codebook_decode_gb300.engine import Engine, to_dev_i32, to_dev_u16
from oracle import orc

# Parity gates on teacher-forced logits (max |diff| / max |logit| per row).
TOL_BF16 = 0.010
TOL_INT8 = 0.015


def rel_diff(a, b):
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-30))


class ParityRun:
    def __init__(self, dims, weights, sess, frames, shuffle=True, int8=False, max_batch=None, stepwise=False,
                 oracle=None, engine=None, tc_min_rows=None, ksplit_min_rows=None, chunk_talker_min_b=None):
        self.d = dims
        self.sess = sess
        self.frames = frames
        self.cap = int(sess.kv_len0.max()) + frames + 1
        self.cap = ((self.cap + PAGE_SIZE - 1) // PAGE_SIZE) * PAGE_SIZE
        if engine is None:
            pool = sess.B * (self.cap // PAGE_SIZE) + 8
            engine = Engine(dims, weights, max_batch=max_batch or max(sess.B, 1), max_context=max(self.cap, 64),
                            pool_pages=pool, int8=int8)
        self.eng = engine
        if stepwise:
            qtts.qtts_set_option(self.eng.m, qtts.QTTS_OPT_STEPWISE, 1)
        if tc_min_rows is not None:
            assert qtts.qtts_set_option(self.eng.m, qtts.QTTS_OPT_TC_MIN_ROWS, tc_min_rows) == 0
        if ksplit_min_rows is not None:
            assert qtts.qtts_set_option(self.eng.m, qtts.QTTS_OPT_KSPLIT_MIN_ROWS, ksplit_min_rows) == 0
        if chunk_talker_min_b is not None:
            assert qtts.qtts_set_option(self.eng.m, qtts.QTTS_OPT_CHUNK_TALKER_MIN_B, chunk_talker_min_b) == 0
        self.eng.setup_sessions(sess, self.cap, shuffle=shuffle)
        self.O = oracle or orc.Oracle(dims, weights, use_int8=int8)
        self.rows = sess.session_array().copy()
        self.kv = [orc.kv_cache_from_prefix(sess.prefix_kv(b), self.cap) for b in range(sess.B)]
        self.rng = sess.rng_state().copy()
        self.seen = sess.seen_bitmap().copy()
        self.rel = []          # (frame, session, codebook, rel diff)
        self.confident = 0
        self.confident_agree = 0
        self.argmax_agree = 0
        self.argmax_total = 0
        self.codes_checked = 0
        self.kv_synced = None

    def run(self, frames=None, check_oracle=True, free=False, split=False):
        """Run frames on the GPU and the oracle side by side. Teacher forced by
        default; free=True lets the GPU sample its own codes and forces the
        oracle with them, so both commit the same codes. split=True runs each
        frame as qtts_frame_talker + qtts_frame_cp. Every frame's own sampled
        codes and EOS flags are checked bit for bit against the oracle's
        sampler fed the GPU's logits, with the state from before the frame."""
        d = self.d
        e = self.eng
        for f in range(frames or self.frames):
            emb = self.sess.in_embeds(f)
            forced = None if free else self.sess.forced_codes(f)
            emb_d = to_dev_u16(emb, e.dev)
            frc_d = None if forced is None else to_dev_i32(forced, e.dev)
            if split:
                args = (e.m, e.B, e.sess, e.bt, e.bt_stride, emb_d, e.rng, e.seen, frc_d, e.codes, e.eos, e.logits)
                qtts.qtts_frame_talker(*args)
                qtts.qtts_frame_cp(*args)
            else:
                e.step(emb_d, frc_d)
            rc, derr = e.status()
            assert rc == 0 and derr == 0, (rc, derr, qtts.load_library().qtts_last_error(e.m))
            got32 = e.logits.cpu().numpy()
            got = got32.astype(np.float64)
            codes = e.codes.cpu().numpy()
            eos = e.eos.cpu().numpy()
            if not check_oracle:
                continue
            rng0, seen0 = self.rng.copy(), self.seen.copy()
            self.check_sampled(got32, codes, eos, rng0, seen0)
            _, _, ref = self.O.frame_step(self.rows, self.kv, self.cap, emb, self.rng, self.seen,
                                          forced=codes if free else forced)
            self.compare_logits(f, got, ref)
        return self

    def check_sampled(self, logits32, codes, eos, rng0, seen0):
        """The codes the frame sampled equal the oracle sampler's on the same
        logits rows, bit for bit (rng and seen set as they were before the
        frame); eos_out is 1 exactly where codebook 0 sampled eos_id."""
        d = self.d
        L = orc.lib()
        for b in range(self.sess.B):
            S = orc.session_struct(self.rows[b])
            for j in range(16):
                V = d.vocab0 if j == 0 else d.cp_vocab
                row = np.ascontiguousarray(logits32[b, j, :V], dtype=np.float32)
                sb = np.ascontiguousarray(seen0[b])
                want = L.orc_sample(row.ctypes.data, V, j, C.byref(S), int(rng0[b, 0]), int(rng0[b, 1]),
                                    int(rng0[b, 2]), sb.ctypes.data if j == 0 else None, d.eos_id, d.n_codes)
                assert int(codes[b, j]) == want, (b, j, int(codes[b, j]), want)
                self.codes_checked += 1
            assert int(eos[b]) == int(codes[b, 0] == d.eos_id), (b, int(eos[b]), int(codes[b, 0]))

    def compare_logits(self, f, got, ref):
        d = self.d
        for b in range(self.sess.B):
            for j in range(16):
                V = d.vocab0 if j == 0 else d.cp_vocab
                g, r = got[b, j, :V], ref[b, j, :V]
                self.rel.append((f, b, j, rel_diff(g, r)))
                top2 = np.sort(r)[-2:]
                self.argmax_total += 1
                same = int(np.argmax(g)) == int(np.argmax(r))
                self.argmax_agree += same
                if top2[1] - top2[0] > 1.0:
                    self.confident += 1
                    self.confident_agree += same

    def sync_oracle_from_gpu(self):
        """Start the oracle from the GPU's state: sessions, rng, seen set and
        every layer's cache up to kv_len, read back through the C ABI (the
        window checks of long runs)."""
        self.rows = self.eng.sess.cpu().numpy().copy()
        self.rng = self.eng.rng.cpu().numpy().view(np.uint32).copy()
        self.seen = self.eng.seen.cpu().numpy().view(np.uint32).copy()
        for b in range(self.sess.B):
            n = int(self.rows[b, 0])
            for l in range(self.d.n_layers):
                k, v = self.eng.read_kv(b, l, n)
                self.kv[b][l, 0, :n] = k
                self.kv[b][l, 1, :n] = v
        self.kv_synced = self.rows[:, 0].copy()

    def max_rel(self, codebooks=range(16)):
        return max(r for (_, _, j, r) in self.rel if j in codebooks)

    def check_state(self):
        """kv_len, frame counter and the seen set advance exactly like the oracle's."""
        sess = self.eng.sess.cpu().numpy()
        assert np.array_equal(sess[:, 0], self.rows[:, 0])
        rng = self.eng.rng.cpu().numpy().view(np.uint32)
        assert np.array_equal(rng, self.rng)
        seen = self.eng.seen.cpu().numpy().view(np.uint32)
        assert np.array_equal(seen, self.seen)

    def check_kv(self, layers=None, tol=2 ** -7):
        """Paged cache read back through the ABI against the oracle's cache:
        the prefix is untouched, appended K/V agree to bf16 rounding."""
        d = self.d
        for b in range(self.sess.B):
            n = int(self.rows[b, 0])
            n0 = int(self.sess.kv_len0[b] if self.kv_synced is None else self.kv_synced[b])
            for l in (layers if layers is not None else range(d.n_layers)):
                k, v = self.eng.read_kv(b, l, n)
                for i, got in enumerate((k, v)):
                    ref = self.kv[b][l, i, :n]
                    assert np.array_equal(got[:n0], ref[:n0])
                    gf = (got[n0:].astype(np.uint32) << 16).view(np.float32)
                    rf = (ref[n0:].astype(np.uint32) << 16).view(np.float32)
                    assert np.abs(gf - rf).max() <= tol * np.abs(rf).max(), (b, l, i)


def free(run):
    try:
        run.eng.release_pages()
        run.eng.close()
    finally:
        torch.cuda.synchronize()
