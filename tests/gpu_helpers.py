"""Shared driver for the GPU parity tests: run the CUDA frame (through the C
ABI) and the CPU oracle side by side on the same seeded inputs."""
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
                 oracle=None, engine=None, tc_min_rows=None, ksplit_min_rows=None):
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

    def run(self, frames=None, check_oracle=True):
        d = self.d
        for f in range(frames or self.frames):
            emb = self.sess.in_embeds(f)
            forced = self.sess.forced_codes(f)
            self.eng.step(to_dev_u16(emb, self.eng.dev), to_dev_i32(forced, self.eng.dev))
            rc, derr = self.eng.status()
            assert rc == 0 and derr == 0, (rc, derr, qtts.load_library().qtts_last_error(self.eng.m))
            got = self.eng.logits.cpu().numpy().astype(np.float64)
            if not check_oracle:
                continue
            _, _, ref = self.O.frame_step(self.rows, self.kv, self.cap, emb, self.rng, self.seen, forced=forced)
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
        return self

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
            n0 = int(self.sess.kv_len0[b])
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
