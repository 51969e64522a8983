"""Codec frames/s of the lockstep multi-codebook frame decode on GB300.

One step = one frame for all B sessions of the workload (the whole hot path:
Talker step, codebook-0 head and sampler, projection, 15 Code-Predictor steps
with heads and samplers) followed by the free-running feedback embedding of
the next Talker input. Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload full_b1]
  python bench.py --impl reference ...   # the CPU oracle on this host's cores

Multi-GPU: the sessions are independent, so N ranks run N replicas (one model
and B sessions each, no collective on the data path); value = all frames / the
slowest rank's time.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from codebook_decode_gb300 import configs, synth  # noqa: E402

METRIC = "codec frames/s (sessions x frames) per GB300 at B=1/8/32; % HBM roofline"
UNIT = "frames/s"


def workload_desc(wl):
    d = wl.dims
    return (f"{wl.name}: Talker {d.n_layers}L h{d.hidden} {d.n_q_heads}q/{d.n_kv_heads}kv d{d.head_dim} "
            f"ffn{d.ffn} V0 {d.vocab0}; proj {d.hidden}->{d.cp_hidden}; CP {d.cp_layers}L h{d.cp_hidden} "
            f"ffn{d.cp_ffn} 15x{d.cp_vocab}; B={wl.batch}; prefix {wl.prefix}; offsets {wl.offset}; "
            f"T {wl.temperature} top-k {wl.top_k} rep {wl.rep_penalty}; "
            f"{'INT8' if wl.int8 else 'BF16'} weights; shuffled paged KV")


def measured_peak_gbs():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def measured_peak_tflops():
    """Dense bf16 tensor peak for a kernel timed inside a longer run (the
    sustained figure), else the fallback."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        if "bf16_tflops_sustained" in j:
            return float(j["bf16_tflops_sustained"]), "measured sustained"
    return 1700.0, "fallback"


def ncu_traffic(wl):
    """DRAM bytes per frame-kernel launch from the committed ncu capture, or
    None when the kernel source changed since it was taken or the capture was
    of another workload."""
    import hashlib
    rec_path = os.path.join(ROOT, "codebook_decode_gb300", "ncu_traffic.json")
    if not os.path.exists(rec_path):
        return None
    rec = json.load(open(rec_path))
    src = open(os.path.join(ROOT, rec["source"]), "rb").read()
    if hashlib.sha256(src).hexdigest()[:16] != rec["source_sha256_prefix"] or rec["workload"] != wl.name:
        return None
    return rec["dram_bytes_per_launch"]


def kv_bytes_per_frame(d, kv_lens):
    """Algorithmic cache bytes of one frame: Talker K/V read over positions
    0..kv_len (new token included) and written at kv_len; Code-Predictor K/V
    read over positions 0..p at each of its 16 positions and written once."""
    t_tok = d.n_layers * 2 * d.n_kv_heads * d.head_dim * 2
    c_tok = d.cp_layers * 2 * d.cp_n_kv_heads * d.cp_head_dim * 2
    B = len(kv_lens)
    read = sum(int(n) + 1 for n in kv_lens) * t_tok + B * sum(p + 1 for p in range(16)) * c_tok
    write = B * (t_tok + 16 * c_tok)
    return read + write


class Clocks:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    def __init__(self, index):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        cmd = ["nvidia-smi", f"--id={index}", "--query-gpu=index,clocks.sm,clocks.max.sm,power.draw,"
               "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
               "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
               "clocks_event_reasons.sw_power_cap", "--format=csv,noheader,nounits", "-lms", "50"]
        try:
            self.p = subprocess.Popen(cmd, stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is not None:
            self.p.terminate()
            try:
                self.p.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.p.kill()
        self.f.flush()
        rows = []
        for line in open(self.f.name):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.f.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def dist_setup():
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, ws):
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cpu" if dist.get_backend() == "gloo" else "cuda"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank, seconds, ws):
    """Units all ranks processed (each rank the same count) over the slowest
    rank's time."""
    return ws * units_per_rank / max_over_ranks(seconds, ws)


# --------------------------------------------------------------------------
# our arm
# --------------------------------------------------------------------------

def stage_names(d):
    """Kind of every stage of the frame program, in order."""
    layer = ["qkv", "attn", "o", "gateup", "down"]
    names = ["begin"] + [f"talker.{n}" for _ in range(d.n_layers) for n in layer] + ["head0+proj", "sample0"]
    for _ in range(1, 16):
        names += [f"cp.{n}" for _ in range(d.cp_layers) for n in layer] + ["cp.head", "cp.sample"]
    return names


def trace_summary(d, stamps):
    """Per stage kind, in microseconds on CTA 0: the stage body (start to end),
    the wait from its end to the next stage's start (the grid barrier) and,
    for GEMV stages, the prologue / weight pass / epilogue split."""
    names = stage_names(d)
    n = len(names)
    t = stamps[: 8 * n].reshape(n, 8).astype(np.int64)
    out = {}
    for i, nm in enumerate(names):
        o = out.setdefault(nm, dict(n=0, body=0.0, barrier=0.0, pro=0.0, w=0.0, epi=0.0))
        o["n"] += 1
        o["body"] += (t[i, 7] - t[i, 0]) / 1e3
        o["barrier"] += (t[i + 1, 0] - t[i, 7]) / 1e3 if i + 1 < n else 0.0
        if t[i, 1] >= t[i, 0] and t[i, 3] <= t[i, 7] and t[i, 1] <= t[i, 2] <= t[i, 3]:
            o["pro"] += (t[i, 1] - t[i, 0]) / 1e3
            o["w"] += (t[i, 2] - t[i, 1]) / 1e3
            o["epi"] += (t[i, 3] - t[i, 2]) / 1e3
    total = (t[-1, 7] - t[0, 0]) / 1e3
    ring = stamps[16 * n: 16 * n + 4 * 4096].reshape(4096, 4)[:, :2].astype(np.int64)
    used = int((ring[:, 1] > 0).sum())
    rq = ring[:used]
    lead = (t[:, 0].min(), rq)
    return {"frame_us": total, "ring": {"uses": used, "issue_us": ((rq[:, 0] - t[0, 0]) / 1e3).tolist(),
                                          "ready_us": ((rq[:, 1] - t[0, 0]) / 1e3).tolist(),
                                          "stage_start_us": ((t[:, 0] - t[0, 0]) / 1e3).tolist()},
            "stages": {k: {"n": v["n"], "body_us": v["body"] / v["n"], "barrier_us": v["barrier"] / v["n"],
                           "prologue_us": v["pro"] / v["n"], "weights_us": v["w"] / v["n"],
                           "epilogue_us": v["epi"] / v["n"], "total_us": v["body"] + v["barrier"]}
                       for k, v in out.items()}}


def talker_pass_weight_bytes(d, int8):
    """Weight bytes one Talker pass streams (QKV, O, gate/up, down of every
    layer; int8 per-row scales are negligible)."""
    per_layer = ((d.n_q_heads + 2 * d.n_kv_heads) * d.head_dim * d.hidden + d.hidden * d.n_q_heads * d.head_dim
                 + 2 * d.ffn * d.hidden + d.hidden * d.ffn)
    return d.n_layers * per_layer * (1 if int8 else 2)


PREFILL_MAX_ROWS = 1024  # rows (sessions x prompt tokens) of one prefill chunk


def prefill_flops(d, kv_len0, n_tok):
    """Algorithmic FLOPs of a prompt pass: 2 per weight and token for every
    layer's QKV and, except the last layer (whose outputs after its K/V are
    not observable), O, gate/up and down; plus 4 x q dims per attended
    position (scores and the weighted sum of V) in those layers."""
    qkv = (d.n_q_heads + 2 * d.n_kv_heads) * d.head_dim * d.hidden
    rest = d.hidden * d.n_q_heads * d.head_dim + 3 * d.ffn * d.hidden
    toks = len(kv_len0) * n_tok
    attended = sum(int(n0) * n_tok + n_tok * (n_tok + 1) // 2 for n0 in kv_len0)
    return (2 * toks * (d.n_layers * qkv + (d.n_layers - 1) * rest)
            + 4 * d.n_q_heads * d.head_dim * attended * (d.n_layers - 1))


def prefill_kv_bytes(d, kv_len0, n_tok, per_chunk):
    """Algorithmic cache bytes of a prompt pass in chunks of per_chunk tokens
    per session: each chunk reads every position before it once (a query
    block of the chunk reuses a K/V tile for all its tokens) and writes its
    own positions once."""
    t_tok = d.n_layers * 2 * d.n_kv_heads * d.head_dim * 2  # K and V of one token, all layers
    n = 0
    for n0 in kv_len0:
        for t0 in range(0, n_tok, per_chunk):
            n += (int(n0) + t0) * t_tok + min(per_chunk, n_tok - t0) * t_tok
    return n


def run_prefill(wl, n_tok, reps, local, weights, warmup=1):
    """Talker prefill throughput: every session of the workload takes an
    n_tok-token prompt after its prefix (kv_len rewound between repetitions,
    median of reps timed with CUDA events on the launching stream)."""
    import torch

    from codebook_decode_gb300 import qtts
    from codebook_decode_gb300.engine import Engine, to_dev_u16

    d = wl.dims
    sess = synth.make_sessions(wl)
    cap = int(sess.kv_len0.max()) + n_tok + 4
    pool = wl.batch * ((cap + 15) // 16) + 8
    eng = Engine(d, weights, max_batch=wl.batch, max_context=cap, pool_pages=pool, device=local, int8=wl.int8)
    eng.setup_sessions(sess, cap, shuffle=wl.shuffle_pages)
    sess0 = eng.sess.clone()
    e = to_dev_u16(sess.prompt_embeds(n_tok), eng.dev)
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        eng.sess.copy_(sess0)
        eng.prefill(e, stream)
    times = []
    for _ in range(reps):
        eng.sess.copy_(sess0)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        eng.prefill(e, stream)
        b.record(stream)
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b))
    rc, derr = qtts.qtts_frame_status(eng.m, raise_on_error=False)
    assert rc == 0 and derr == 0, (rc, derr)
    ms = statistics.median(times)
    # a chunk takes PREFILL_MAX_ROWS // B prompt tokens of every session,
    # streams the Talker weights (BF16, also for INT8 models) once for all of
    # them, reads each session's cached K/V once and writes the chunk's
    per_chunk = max(1, PREFILL_MAX_ROWS // wl.batch)
    chunks = (n_tok + per_chunk - 1) // per_chunk
    nbytes = chunks * talker_pass_weight_bytes(d, False) + prefill_kv_bytes(d, sess.kv_len0, n_tok, per_chunk)
    flops = prefill_flops(d, sess.kv_len0, n_tok)
    eng.release_pages()
    eng.close()
    return dict(tokens_per_s=wl.batch * n_tok / (ms / 1e3), ms=ms, bytes=nbytes, achieved_gbs=nbytes / (ms / 1e3) / 1e9,
                flops=flops, achieved_tflops=flops / (ms / 1e3) / 1e12, chunks=chunks)


def run_gpu(wl, steps, warmup, local, weights, trace=False, ring_slots=None, trace_file=None, tc_min_rows=None,
            ksplit_min_rows=None, chunk_talker_min_b=None):
    import torch

    from codebook_decode_gb300 import qtts
    from codebook_decode_gb300.engine import Engine, to_dev_u16

    d = wl.dims
    sess = synth.make_sessions(wl)
    cap = min(2048, int(sess.kv_len0.max()) + steps + warmup + 4)
    limit = cap - int(sess.kv_len0.max()) - 2  # frames before the contexts are rewound
    pool = wl.batch * ((cap + 15) // 16) + 8
    torch.cuda.synchronize(local)
    free0 = torch.cuda.mem_get_info(local)[0]
    eng = Engine(d, weights, max_batch=max(wl.batch, 1), max_context=cap, pool_pages=pool, device=local, int8=wl.int8)
    eng.setup_sessions(sess, cap, shuffle=wl.shuffle_pages)
    torch.cuda.synchronize(local)
    model_bytes = free0 - torch.cuda.mem_get_info(local)[0]  # the library's allocations: weights, copies, pool, scratch
    if ring_slots is not None:
        qtts.qtts_set_option(eng.m, qtts.QTTS_OPT_RING_SLOTS, ring_slots)
    if tc_min_rows is not None:
        qtts.qtts_set_option(eng.m, qtts.QTTS_OPT_TC_MIN_ROWS, tc_min_rows)
    if ksplit_min_rows is not None:
        qtts.qtts_set_option(eng.m, qtts.QTTS_OPT_KSPLIT_MIN_ROWS, ksplit_min_rows)
    if chunk_talker_min_b is not None:
        qtts.qtts_set_option(eng.m, qtts.QTTS_OPT_CHUNK_TALKER_MIN_B, chunk_talker_min_b)
    dev = eng.dev
    stream = torch.cuda.current_stream()
    sess0 = eng.sess.clone()
    emb = to_dev_u16(sess.in_embeds(0), dev)
    text = to_dev_u16(sess.text_embeds(0), dev)
    nxt = torch.empty_like(emb)
    weight_bytes = qtts.qtts_frame_weight_bytes(eng.m)
    B = wl.batch

    def step(i, inp):
        eng.step(inp, None, want_logits=False, stream=stream)
        qtts.qtts_feedback_embed(eng.m, B, eng.codes, text, nxt, stream)
        return nxt

    cur = emb
    done = 0
    for i in range(warmup):
        cur = step(i, cur).clone()
        done += 1
    torch.cuda.synchronize()
    rc, derr = qtts.qtts_frame_status(eng.m, raise_on_error=False)
    assert rc == 0 and derr == 0, (rc, derr)
    # average context over the timed frames, for the cache bytes
    kv_start = eng.sess[:, 0].cpu().numpy().astype(np.int64)

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    kv_bytes = 0
    clocks = Clocks(local)
    torch.cuda.synchronize()
    t0.record(stream)
    kv_now = kv_start.copy()
    for i in range(steps):
        if done >= limit:  # keep every context inside the cache: rewind to the prefix
            eng.sess.copy_(sess0)
            kv_now = sess.kv_len0.astype(np.int64).copy()
            done = 0
        starts[i].record(stream)
        eng.step(cur, None, want_logits=False, stream=stream)
        ends[i].record(stream)
        qtts.qtts_feedback_embed(eng.m, B, eng.codes, text, nxt, stream)
        cur, nxt = nxt, cur
        kv_bytes += kv_bytes_per_frame(d, kv_now)
        kv_now += 1
        done += 1
    t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    rc, derr = qtts.qtts_frame_status(eng.m, raise_on_error=False)
    assert rc == 0 and derr == 0, (rc, derr)
    total_ms = t0.elapsed_time(t1)
    frame_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    avg_frame_s = statistics.mean(frame_ms) / 1e3
    bytes_per_frame = weight_bytes + kv_bytes / steps + B * 15 * d.cp_hidden * 4
    res = dict(total_ms=total_ms, frame_ms=statistics.mean(frame_ms), weight_bytes=weight_bytes,
               bytes_per_frame=bytes_per_frame, achieved_gbs=bytes_per_frame / avg_frame_s / 1e9, clocks=clk)

    # end to end through the host-buffer entry point: inputs copied in, codes
    # and advanced state copied back, every frame
    sess_h = torch.from_numpy(sess.session_array()).pin_memory().numpy()
    bt_h = torch.from_numpy(eng.bt_host).pin_memory().numpy()
    emb_h = torch.from_numpy(sess.in_embeds(0).view(np.int16)).pin_memory().numpy().view(np.uint16)
    rng_h = torch.from_numpy(sess.rng_state().view(np.int32)).pin_memory().numpy()
    seen_h = torch.from_numpy(sess.seen_bitmap().view(np.int32)).pin_memory().numpy()
    codes_h = torch.zeros(B, 16, dtype=torch.int32).pin_memory().numpy()
    eos_h = torch.zeros(B, dtype=torch.uint8).pin_memory().numpy()
    sess_init = sess_h.copy()

    def host_step():
        qtts.qtts_frame_step_host(eng.m, B, sess_h, bt_h, eng.bt_stride, emb_h, rng_h, seen_h, None, codes_h, eos_h,
                                  None, stream)

    for _ in range(warmup):
        host_step()
    sess_h[:] = sess_init
    e2e_steps = steps
    torch.cuda.synchronize()
    t = time.perf_counter()
    n_done = 0
    for _ in range(e2e_steps):
        if n_done >= limit:
            sess_h[:] = sess_init
            n_done = 0
        host_step()
        n_done += 1
    e2e_s = time.perf_counter() - t
    h2d = sess_h.nbytes + B * eng.bt_stride * 4 + emb_h.nbytes + rng_h.nbytes + seen_h.nbytes
    d2h = codes_h.nbytes + eos_h.nbytes + sess_h.nbytes + rng_h.nbytes + seen_h.nbytes
    res["e2e"] = dict(value=B * e2e_steps / e2e_s, s=e2e_s, frames=B * e2e_steps, h2d=h2d, d2h=d2h)
    res["model_device_bytes"] = model_bytes
    if trace:
        qtts.qtts_set_option(eng.m, qtts.QTTS_OPT_TRACE, 1)
        eng.sess.copy_(sess0)
        for _ in range(2):
            eng.step(emb, None, want_logits=False, stream=stream)
        stamps = np.zeros(16 * len(stage_names(d)) + 4 * 4096, dtype=np.uint64)
        qtts.qtts_frame_trace(eng.m, stamps)
        res["trace"] = trace_summary(d, stamps)
        if trace_file:  # every CTA's stage stamps, raw
            qtts.qtts_set_option(eng.m, qtts.QTTS_OPT_TRACE, 2)
            eng.sess.copy_(sess0)
            for _ in range(2):
                eng.step(emb, None, want_logits=False, stream=stream)
            G = torch.cuda.get_device_properties(local).multi_processor_count
            raw = np.zeros(8 * G * len(stage_names(d)) + 4 * 4096, dtype=np.uint64)
            qtts.qtts_frame_trace(eng.m, raw)
            np.save(trace_file, raw)
    eng.release_pages()
    eng.close()
    return res


def oracle_sample(wl, weights, frames, threads=None):
    """The CPU oracle on a bounded sample of the workload: `frames` teacher-forced
    frames of the first min(B, 2) sessions. Returns (frames/s, frames, sessions)."""
    from oracle import orc

    d = wl.dims
    sess = synth.make_sessions(wl)
    Bs = min(wl.batch, 2)
    O = orc.Oracle(d, weights, use_int8=wl.int8)
    cap = int(sess.kv_len0[:Bs].max()) + frames + 2
    rows = sess.session_array()[:Bs].copy()
    kv = [orc.kv_cache_from_prefix(sess.prefix_kv(b), cap) for b in range(Bs)]
    rng = sess.rng_state()[:Bs].copy()
    seen = sess.seen_bitmap()[:Bs].copy()
    O.frame_step(rows, kv, cap, sess.in_embeds(0)[:Bs], rng, seen, want_logits=False)  # warm-up
    t = time.perf_counter()
    for f in range(frames):
        O.frame_step(rows, kv, cap, sess.in_embeds(f)[:Bs], rng, seen, want_logits=False)
    dt = time.perf_counter() - t
    return Bs * frames / dt, frames, Bs


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="full_b1", choices=sorted(configs.WORKLOADS))
    ap.add_argument("--no-sweep", action="store_true", help="skip the B=8/B=32/INT8 side measurements")
    ap.add_argument("--oracle-frames", type=int, default=6)
    ap.add_argument("--trace", action="store_true", help="print a per-stage time breakdown to stderr")
    ap.add_argument("--trace-file", default=None, help="with --trace: save every CTA's raw stage stamps (.npy)")
    ap.add_argument("--ring-slots", type=int, default=None, help="weight-ring depth per SM (library default 8)")
    ap.add_argument("--tc-min-rows", type=int, default=None,
                    help="fewest activation rows a GEMV takes on the tensor cores (library default 8; 65: off)")
    ap.add_argument("--ksplit-min-rows", type=int, default=None,
                    help="fewest activation rows for the K-split tensor-core GEMV (library default 8; below it only the deepest GEMVs split)")
    ap.add_argument("--chunk-talker-min-b", type=int, default=None,
                    help="fewest sessions whose BF16 frames run the Talker on the chunk kernels (library default 33: off)")
    ap.add_argument("--prefill-only", type=int, default=0, metavar="TOKENS",
                    help="time only the Talker prefill of TOKENS prompt tokens per session of --workload "
                         "(--warmup untimed passes, then --steps timed ones; prints one JSON line)")
    args = ap.parse_args()
    wl = configs.WORKLOADS[args.workload]
    cores = os.cpu_count()

    if args.prefill_only > 0 and args.impl == "ours":
        w = synth.make_weights(wl.dims, 1000 + wl.seed)
        rp = run_prefill(wl, args.prefill_only, args.steps, 0, w, warmup=args.warmup)
        peak, _ = measured_peak_gbs()
        tc_peak, tc_kind = measured_peak_tflops()
        t_hbm, t_tc = rp["bytes"] / (peak * 1e9), rp["flops"] / (tc_peak * 1e12)
        tensor = t_tc > t_hbm
        line = {"metric": "Talker prefill prompt tokens/s", "value": rp["tokens_per_s"], "unit": "tokens/s",
                "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": rp["ms"],
                "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
                "config": {"workload": workload_desc(wl), "prompt_tokens": args.prefill_only,
                           "chunks": rp["chunks"]},
                "roofline": {"bound": "tensor" if tensor else "hbm",
                             "achieved": rp["achieved_tflops"] if tensor else rp["achieved_gbs"],
                             "peak": tc_peak if tensor else peak, "unit": "TFLOP/s" if tensor else "GB/s",
                             "frac": rp["achieved_tflops"] / tc_peak if tensor else rp["achieved_gbs"] / peak,
                             "flops": rp["flops"], "bytes": rp["bytes"], "peak_kind": tc_kind if tensor else "measured"}}
        print(json.dumps(line))
        return

    if args.impl == "reference":
        # the oracle on the host cores: rank 0 alone runs it (no process group
        # is needed for that); the other ranks of a multi-GPU launch exit
        if int(os.environ.get("RANK", "0")) != 0:
            return
        w = synth.make_weights(wl.dims, 1000 + wl.seed)
        t = time.perf_counter()
        for _ in range(args.warmup):
            oracle_sample(wl, w, 1)
        fps, nfr, bs = oracle_sample(wl, w, args.steps)
        ms = 1e3 * bs / fps
        line = {"metric": METRIC, "value": fps, "unit": UNIT, "impl": "reference", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": workload_desc(wl), "sessions_per_step": bs},
                "cpu_baseline": {"value": fps, "unit": UNIT, "cores": cores, "kind": "oracle",
                                 "sample": f"{nfr} teacher-forced frames x {bs} sessions of {wl.name}"},
                "e2e": {"value": fps, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
                "wall_s": time.perf_counter() - t}
        print(json.dumps(line))
        return

    ws, rank, local = dist_setup()
    import torch
    w = synth.make_weights(wl.dims, 1000 + wl.seed)
    barrier(ws)
    r = run_gpu(wl, args.steps, args.warmup, local, w, trace=args.trace, ring_slots=args.ring_slots, tc_min_rows=args.tc_min_rows,
                ksplit_min_rows=args.ksplit_min_rows, chunk_talker_min_b=args.chunk_talker_min_b,
                trace_file=args.trace_file)
    if args.trace:
        print(json.dumps(r["trace"]), file=sys.stderr)
    total_s = max_over_ranks(r["total_ms"] / 1e3, ws)
    value = ws * wl.batch * args.steps / total_s
    peak, peak_kind = measured_peak_gbs()
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "int8" if wl.int8 else "bf16",
            "data": "synthetic: seeded N(0,0.02) random-init weights and N(0,1) prefix KV, free-running sampling",
            "config": {"workload": workload_desc(wl), "global_batch": ws * wl.batch,
                       "parallelism": f"replicas x{ws}",
                       "l2": "inputs larger than L2: every frame streams the full weight set (GBs) through HBM"},
            "roofline": {"bound": "hbm", "achieved": r["achieved_gbs"], "peak": peak, "unit": "GB/s",
                         "frac": r["achieved_gbs"] / peak, "traffic": ncu_traffic(wl),
                         "peak_kind": peak_kind, "kernel": "qtts::frame_kernel",
                         "bytes_per_launch": r["bytes_per_frame"], "launch_ms": r["frame_ms"]},
            "e2e": {"value": whole_job_rate(r["e2e"]["frames"], r["e2e"]["s"], ws), "unit": UNIT,
                    "h2d_bytes_per_step": r["e2e"]["h2d"],
                    "d2h_bytes_per_step": r["e2e"]["d2h"]},
            "gpu_launches": 2 * args.steps,
            "clocks": r["clocks"],
            "model_device_bytes": r["model_device_bytes"]}
    if rank == 0:
        fps, nfr, bs = oracle_sample(wl, w, args.oracle_frames)
        line["cpu_baseline"] = {"value": fps, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": f"{nfr} teacher-forced frames x {bs} session(s) of {wl.name}"}
        if not args.no_sweep and ws == 1:
            sweep = {}
            for name in ("full_b8", "full_b32", "int8_b1", "int8_b32"):
                o = configs.WORKLOADS[name]
                rr = run_gpu(o, min(args.steps, 50), 3, local, w, ring_slots=args.ring_slots,
                             tc_min_rows=args.tc_min_rows, ksplit_min_rows=args.ksplit_min_rows,
                             chunk_talker_min_b=args.chunk_talker_min_b)  # same weights
                sweep[name] = {"frames_per_s": o.batch * min(args.steps, 50) / (rr["total_ms"] / 1e3),
                               "frame_ms": rr["frame_ms"], "achieved_gbs": rr["achieved_gbs"],
                               "frac": rr["achieved_gbs"] / peak, "bytes_per_frame": rr["bytes_per_frame"]}
            tc_peak, tc_kind = measured_peak_tflops()
            for name, n_tok in (("full_b1", 64), ("full_b1", 512), ("full_b1", 1024), ("full_b8", 64),
                                ("full_b8", 128)):
                o = configs.WORKLOADS[name]
                rp = run_prefill(o, n_tok, 3, local, w)
                t_hbm = rp["bytes"] / (peak * 1e9)
                t_tc = rp["flops"] / (tc_peak * 1e12)
                bound = "tensor" if t_tc > t_hbm else "hbm"
                sweep[f"prefill_{name}_{n_tok}tok"] = {
                    "tokens_per_s": rp["tokens_per_s"], "ms": rp["ms"], "achieved_gbs": rp["achieved_gbs"],
                    "hbm_frac": rp["achieved_gbs"] / peak, "bytes": rp["bytes"],
                    "achieved_tflops": rp["achieved_tflops"], "tensor_frac": rp["achieved_tflops"] / tc_peak,
                    "flops": rp["flops"], "bound": bound,
                    "frac": rp["achieved_tflops"] / tc_peak if bound == "tensor" else rp["achieved_gbs"] / peak,
                    "peak": {"hbm_gbs": peak, "bf16_tflops": tc_peak, "kind": tc_kind},
                    "what": f"Talker prefill of {n_tok} prompt tokens for each of {o.batch} session(s) after its "
                            f"prefix, {rp['chunks']} chunk(s) of up to {PREFILL_MAX_ROWS} rows"}
            line["sweep"] = sweep
        print(json.dumps(line))
    barrier(ws)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
