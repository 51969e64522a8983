// frame_kernel.cu -- one codec frame of the lockstep multi-codebook decode as
// a single persistent kernel: one CTA per SM walks the frame's stage program
// (Talker layers, codebook-0 head + projection, sampler, 15 Code-Predictor
// steps). Stages hand activations to one another as tagged words (value and
// frame/stage tag in one 64-bit store), so a CTA starts a stage as soon as
// the words it reads are there: no grid-wide barrier.
//
// The stage sequence follows "Qwen3-TTS Native v0.3.0", section "What
// changed" (one batched call runs the talker and the 15-step code predictor
// for every active session, each shared weight read once per frame) and
// "De grens van snelheid en kosten verleggen voor Qwen3-TTS", section 3
// (the Code Predictor's fixed 15 steps over a pre-allocated short cache).
// The pages' engines replay ~1,600 kernels per frame as a CUDA graph; here the
// whole frame is one launch.
//
// Inside a CTA, warps 0..10 compute and warp 11 is a producer: it walks the
// same stage program and streams this CTA's share of every upcoming weight
// matrix into a ring of shared-memory slots with TMA bulk copies, running
// ahead across stage boundaries (weights do not depend on activations), so
// HBM keeps streaming while the compute warps wait for their inputs.
#include <cuda_bf16.h>
#include <math.h>

#include "qtts_internal.h"
#include "device_util.cuh"

namespace qtts {

constexpr int kCWarps = kWarps - 1;          // compute warps
constexpr int kCThreads = kCWarps * 32;
constexpr int kProducerWarp = kCWarps;

// ---------------------------------------------------------------------------
// helpers
// ---------------------------------------------------------------------------

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// streaming read-only load of weights: never written while a frame runs
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}
__device__ __forceinline__ uint2 ld_stream8(const void* p) {
  uint2 v;
  asm("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

// barrier of the compute warps only (the producer warp never joins it)
__device__ __forceinline__ void cbar() { asm volatile("bar.sync 1, %0;" ::"n"(kCThreads) : "memory"); }
__device__ __forceinline__ int cbar_or(int pred) {
  int r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.s32 p, %1, 0;\n bar.red.or.pred q, 1, %2, p;\n selp.s32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"(pred), "n"(kCThreads)
      : "memory");
  return r;
}


// Time limit of every wait for another CTA's data or for weights (default
// 2 s: a frame takes milliseconds; qtts_set_option can shorten it), copied
// from Globals at kernel start. Waits for a CTA's own copies and MMAs before
// it leaves use kDrainNs instead, whatever this limit is.
__shared__ uint64_t s_wait_ns;
#define kWaitTimeoutNs s_wait_ns
constexpr uint64_t kDrainNs = 2000000000ull;

// ---- tagged words (see StageDesc): one 64-bit access carries value and tag ----

__device__ __forceinline__ uint64_t ll_word(uint32_t payload, uint32_t tag) {
  return ((uint64_t)tag << 32) | payload;
}
__device__ __forceinline__ void st_ll(uint64_t* p, float v, uint32_t tag) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(ll_word(__float_as_uint(v), tag)) : "memory");
}
__device__ __forceinline__ void st_ll_raw(uint64_t* p, uint32_t payload, uint32_t tag) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(ll_word(payload, tag)) : "memory");
}
__device__ __forceinline__ void st_ll2(uint64_t* p, float v0, float v1, uint32_t tag) {
  asm volatile("st.relaxed.gpu.global.v2.b64 [%0], {%1, %2};" ::"l"(p), "l"(ll_word(__float_as_uint(v0), tag)),
               "l"(ll_word(__float_as_uint(v1), tag))
               : "memory");
}
__device__ __forceinline__ uint64_t ld_ll(const uint64_t* p) {
  uint64_t a;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(a) : "l"(p) : "memory");
  return a;
}
// two words at a 16-byte aligned address (each word is its own atomic access)
__device__ __forceinline__ void ld_ll2(const uint64_t* p, uint64_t& a, uint64_t& b) {
  asm volatile("ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}
__device__ __forceinline__ bool ll_ok(uint64_t w, uint32_t tag) { return (uint32_t)(w >> 32) == tag; }
__device__ __forceinline__ float ll_val(uint64_t w) { return __uint_as_float((uint32_t)w); }

// Re-read the word at p until it carries `tag` and return it; after the time
// limit (sets QTTS_DEV_TIMEOUT) or once an error is set elsewhere, return 0
// (no frame's tag is 0).
__device__ __noinline__ uint64_t ll_wait(const uint64_t* p, uint32_t tag, int* err) {
  const uint64_t t0 = global_timer_ns();
  unsigned spins = 0;
  for (;;) {
    const uint64_t w = ld_ll(p);
    if (ll_ok(w, tag)) return w;
    if ((++spins & 15u) == 0u) {
      if (read_err(err) || global_timer_ns() - t0 > kWaitTimeoutNs) {
        if (!read_err(err)) set_err(err, QTTS_DEV_TIMEOUT);
        return 0;
      }
    }
  }
}
// w: the first read of the word at p; true once it carries `tag`
__device__ __forceinline__ bool ll_get(const uint64_t* p, uint32_t tag, uint64_t& w, int* err) {
  if (ll_ok(w, tag)) return true;
  w = ll_wait(p, tag, err);
  return ll_ok(w, tag);
}

// ll_settle for N pairs at base + u * stride (u < n), all with one tag.
template <int N>
__device__ __forceinline__ bool ll_settle_strided(const uint64_t* base, int stride, int n, uint32_t tag,
                                                  uint64_t (&w)[N][2], int* err) {
  bool all = true;
#pragma unroll
  for (int u = 0; u < N; ++u)
    if (u < n) all &= ll_ok(w[u][0], tag) & ll_ok(w[u][1], tag);
  if (all) return true;
  const uint64_t t0 = global_timer_ns();
  unsigned spins = 0;
  for (;;) {
    all = true;
#pragma unroll
    for (int u = 0; u < N; ++u)
      if (u < n && !(ll_ok(w[u][0], tag) & ll_ok(w[u][1], tag))) {
        ld_ll2(base + (size_t)u * stride, w[u][0], w[u][1]);
        all = false;
      }
    if (all) return true;
    if ((++spins & 15u) == 0u && (read_err(err) || global_timer_ns() - t0 > kWaitTimeoutNs)) {
      if (!read_err(err)) set_err(err, QTTS_DEV_TIMEOUT);
      return false;
    }
  }
}

// Wait until both words of every pair ps[u] (u < N, ps[u] != nullptr) carry
// tag t[u]; w holds the first reads. Every pass re-reads all pairs still
// pending at once, so a late batch costs one round trip per pass, not one per
// word. False after the time limit or once an error is set elsewhere.
template <int N>
__device__ __forceinline__ bool ll_settle(const uint64_t* const (&ps)[N], const uint32_t (&t)[N],
                                          uint64_t (&w)[N][2], int* err) {
  bool all = true;
#pragma unroll
  for (int u = 0; u < N; ++u)
    if (ps[u]) all &= ll_ok(w[u][0], t[u]) & ll_ok(w[u][1], t[u]);
  if (all) return true;
  const uint64_t t0 = global_timer_ns();
  unsigned spins = 0;
  for (;;) {
    all = true;
#pragma unroll
    for (int u = 0; u < N; ++u)
      if (ps[u] && !(ll_ok(w[u][0], t[u]) & ll_ok(w[u][1], t[u]))) {
        ld_ll2(ps[u], w[u][0], w[u][1]);
        all = false;
      }
    if (all) return true;
    if ((++spins & 15u) == 0u && (read_err(err) || global_timer_ns() - t0 > kWaitTimeoutNs)) {
      if (!read_err(err)) set_err(err, QTTS_DEV_TIMEOUT);
      return false;
    }
  }
}

// Gather-and-add of tagged words: item i (< nitems) adds the words src(i, 0..nw-1)
// (nw <= NW, in that order), each once it carries tag(i), to *dst(i); up to
// NB items per compute thread are in flight at once and every pass re-reads
// the words still pending. False after the time limit or once an error is
// set elsewhere (the sums are then incomplete).
template <int NB, int NW, typename Tag, typename Src, typename Dst>
__device__ __forceinline__ bool ll_gather_add(int nitems, int nw, const Tag& tag, const Src& src, const Dst& dst,
                                              int* err) {
  bool ok = true;
  for (int base = (int)threadIdx.x; base < nitems; base += kCThreads * NB) {
    uint64_t w[NB][NW];
#pragma unroll
    for (int u = 0; u < NB; ++u)
#pragma unroll
      for (int k = 0; k < NW; ++k) w[u][k] = (base + u * kCThreads < nitems && k < nw) ? ld_ll(src(base + u * kCThreads, k)) : 0;
    const uint64_t t0 = global_timer_ns();
    unsigned spins = 0;
    for (;;) {
      bool all = true;
#pragma unroll
      for (int u = 0; u < NB; ++u)
#pragma unroll
        for (int k = 0; k < NW; ++k)
          if (base + u * kCThreads < nitems && k < nw && !ll_ok(w[u][k], tag(base + u * kCThreads))) {
            w[u][k] = ld_ll(src(base + u * kCThreads, k));
            all = false;
          }
      if (all) break;
      if ((++spins & 15u) == 0u && (read_err(err) || global_timer_ns() - t0 > kWaitTimeoutNs)) {
        if (!read_err(err)) set_err(err, QTTS_DEV_TIMEOUT);
        return false;
      }
    }
#pragma unroll
    for (int u = 0; u < NB; ++u)
      if (base + u * kCThreads < nitems) {
        float* o = dst(base + u * kCThreads);
        float v = *o;
#pragma unroll
        for (int k = 0; k < NW; ++k)
          if (k < nw) v += ll_val(w[u][k]);
        *o = v;
      }
  }
  return ok;
}

// deterministic sum over the compute threads (fixed combination order)
__device__ float block_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum(v);
  cbar();
  if (lane == 0) red[warp] = v;
  cbar();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < kCWarps; ++w) t += red[w];
    red[kCWarps] = t;
  }
  cbar();
  return red[kCWarps];
}

// Stage trace: with tracing on, thread 0 of the traced CTAs (the first and
// the last, or all) stamps %globaltimer at up to 8 points of every stage (0
// start, 1 after the GEMV prologue, 2 after its phase 1, 3 after its phase 2,
// 7 end; ring path: 4 before warp 0's first ring wait, 5 after that unit's
// dot products, 6 after its epilogue, 3 after the dot products of warp 0's
// second unit;
// tensor path: 4 when the second activation pass starts loading, 5 when its
// first words have settled, 6 when it is staged);
// CTA 0 also stamps its weight-ring slot uses (issue, ready, and on the
// tensor path the end of the slot's MMA issue).
constexpr int kTraceMarks = 8;
constexpr int kTraceRing = 4096;
__shared__ int g_trace_stage;
__device__ __forceinline__ void trace_ring(const Globals& g, uint32_t q, int which) {
  if (g.trace && blockIdx.x == 0 && q < (uint32_t)kTraceRing)
    g.trace[(size_t)g.trace_ctas * g.n_stages * kTraceMarks + (size_t)q * 4 + which] = global_timer_ns();
}
__device__ __forceinline__ void trace_mark(const Globals& g, int which) {
  if (g.trace && threadIdx.x == 0) {
    int slot = (int)blockIdx.x;
    if (g.trace_ctas == 2) slot = blockIdx.x == 0 ? 0 : blockIdx.x == gridDim.x - 1 ? 1 : -1;
    if (slot >= 0) g.trace[((size_t)slot * g.n_stages + g_trace_stage) * kTraceMarks + which] = global_timer_ns();
  }
}

// ---- mbarriers and TMA bulk copies into shared memory ----

__device__ __forceinline__ void mbar_inval(uint64_t* bar) {
  asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
// L2 policy for data read once per frame (weights, KV): evict it first, so
// it streams through L2 without displacing the small data every stage reuses
// (activations, gains, RoPE tables, block tables, stage descriptors)
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// global -> shared bulk copy (16-byte aligned addresses, size a multiple of 16)
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                          uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_addr(dst)),
      "l"(__cvta_generic_to_global(src)), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
// generic-proxy global writes (KV appends) become visible to later bulk copies
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }
constexpr uint32_t kSuspendNs = 20000;  // recheck the error word and the time limit this often

// Wait for a copy or MMA this CTA issued itself to complete before leaving
// (its bytes must not land after the CTA is gone): up to kDrainNs, whatever
// the error word says.
__device__ void mbar_drain(uint64_t* bar, uint32_t parity) {
  if (mbar_test(bar, parity)) return;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_test_sleep(bar, parity, kSuspendNs))
    if (global_timer_ns() - t0 > kDrainNs) return;
}

// Wait for phase `parity` of `bar` to complete, at most kWaitTimeoutNs; an
// error word set elsewhere ends the wait too.
__device__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* err) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_test_sleep(bar, parity, kSuspendNs)) {
    if (read_err(err)) return false;
    if (global_timer_ns() - t0 > kWaitTimeoutNs) {
      set_err(err, QTTS_DEV_TIMEOUT);
      return false;
    }
  }
  return true;
}

// ---- 5th-generation tensor cores: the TMEM accumulator (operand
// descriptors and MMA issue: device_util.cuh) ----

constexpr uint32_t kTmemCols = 128;  // the accumulator: 128 lanes (weight rows) x up to 128 columns
// one warp
__device__ __forceinline__ void tc_alloc(uint32_t* dst) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst)),
               "n"(kTmemCols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tc_dealloc(uint32_t tmem) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTmemCols) : "memory");
}
// 16 consecutive fp32 columns of this warp's 32 TMEM lanes (one lane per thread)
__device__ __forceinline__ void tc_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}

// ---------------------------------------------------------------------------
// sampler arithmetic: Philox4x32-10 and a binary32 log written for this
// project so that any two implementations of the same steps agree bit for bit
// ---------------------------------------------------------------------------

// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): 10 rounds of two 32x32
// multiplies with a Weyl-sequence key schedule.
__device__ __forceinline__ void philox4x32_10(uint32_t c[4], uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t lo0 = 0xD2511F53u * c[0], hi0 = __umulhi(0xD2511F53u, c[0]);
    const uint32_t lo1 = 0xCD9E8D57u * c[2], hi1 = __umulhi(0xCD9E8D57u, c[2]);
    const uint32_t n0 = hi1 ^ c[1] ^ k0;
    const uint32_t n2 = hi0 ^ c[3] ^ k1;
    c[0] = n0;
    c[1] = lo1;
    c[2] = n2;
    c[3] = lo0;
  }
}

// ln(x) for finite x > 0: x = m 2^k with m in (sqrt(1/2), sqrt(2)], then
// ln m = 2 atanh(s), s = (m-1)/(m+1), atanh(s) = s (1 + s^2/3 + ... + s^10/11).
// Each step is one correctly rounded binary32 operation (no contraction).
__device__ float log_series_f32(float x) {
  uint32_t u = __float_as_uint(x);
  int k = 0;
  if (((u >> 23) & 0xFFu) == 0u) {
    x = __fmul_rn(x, 33554432.0f);  // 2^25, exact
    u = __float_as_uint(x);
    k = -25;
  }
  k += (int)((u >> 23) & 0xFFu) - 127;
  uint32_t mb = (u & 0x007FFFFFu) | 0x3F800000u;
  if (mb > 0x3FB504F3u) {
    mb = (u & 0x007FFFFFu) | 0x3F000000u;
    k += 1;
  }
  const float m = __uint_as_float(mb);
  const float s = __fdiv_rn(__fsub_rn(m, 1.0f), __fadd_rn(m, 1.0f));
  const float s2 = __fmul_rn(s, s);
  float t = 0x1.745d18p-4f;                          // 1/11
  t = __fadd_rn(__fmul_rn(t, s2), 0x1.c71c72p-4f);  // 1/9
  t = __fadd_rn(__fmul_rn(t, s2), 0x1.24924ap-3f);  // 1/7
  t = __fadd_rn(__fmul_rn(t, s2), 0x1.99999ap-3f);  // 1/5
  t = __fadd_rn(__fmul_rn(t, s2), 0x1.555556p-2f);  // 1/3
  t = __fadd_rn(__fmul_rn(t, s2), 1.0f);
  const float lm = __fmul_rn(__fadd_rn(s, s), t);
  return __fadd_rn(__fmul_rn(__int2float_rn(k), 0x1.62e430p-1f), lm);  // k ln2 + ln m
}

// Gumbel noise -ln(-ln u) for vocabulary id v of codebook j, u from word v&3
// of Philox(key, (v>>2, j, frame_ctr, 0)): u = (top 23 bits + 1/2) 2^-23.
__device__ __forceinline__ float gumbel_of_word(uint32_t w) {
  const float u = __fmul_rn(__fadd_rn(__uint2float_rn(w >> 9), 0.5f), 0x1p-23f);
  const float l1 = log_series_f32(u);
  const float l2 = log_series_f32(-l1);
  return -l2;
}
__device__ __forceinline__ float gumbel(uint32_t key0, uint32_t key1, int j, uint32_t fctr, int v) {
  uint32_t c[4] = {(uint32_t)v >> 2, (uint32_t)j, fctr, 0u};
  philox4x32_10(c, key0, key1);
  return gumbel_of_word(c[v & 3]);
}

// order-preserving map of a binary32 value to uint32 (-0 and +0 map together)
__device__ __forceinline__ uint32_t order_key(float z) {
  uint32_t u = __float_as_uint(z);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// (val, id) is better than (bv, bid): larger value, then smaller id
__device__ __forceinline__ bool better(bool have, float val, int id, bool bhave, float bv, int bid) {
  if (!have) return false;
  if (!bhave) return true;
  return val > bv || (val == bv && id < bid);
}

// Arg-best over the compute threads (have, val, id); every thread gets the winner.
__device__ int block_argbest(bool have, float val, int id, float* redv, int* redi, int* redh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, val, o);
    const int oi = __shfl_xor_sync(0xffffffffu, id, o);
    const bool oh = __shfl_xor_sync(0xffffffffu, (int)have, o) != 0;
    if (better(oh, ov, oi, have, val, id)) {
      val = ov;
      id = oi;
      have = oh;
    }
  }
  cbar();
  if (lane == 0) {
    redv[warp] = val;
    redi[warp] = id;
    redh[warp] = have;
  }
  cbar();
  if (threadIdx.x == 0) {
    bool bh = false;
    float bv = 0.f;
    int bi = 0;
    for (int w = 0; w < kCWarps; ++w)
      if (better(redh[w] != 0, redv[w], redi[w], bh, bv, bi)) {
        bh = redh[w] != 0;
        bv = redv[w];
        bi = redi[w];
      }
    redi[kCWarps] = bi;
  }
  cbar();
  return redi[kCWarps];
}

// Exclusive prefix sum of one int per compute thread (thread order).
__device__ int block_excl_scan(int v, int* wsum) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  cbar();
  if (lane == 31) wsum[warp] = incl;
  cbar();
  int base = 0;
  for (int w = 0; w < warp; ++w) base += wsum[w];
  return base + incl - v;
}

// ---------------------------------------------------------------------------
// shared sampler core: one row of raw logits -> one code
//   1. codebook 0: ids >= n_codes other than eos -> -inf; eos -> -inf unless
//      allowed; repetition penalty on the seen set ("Qwen3-TTS PR 5", "Graph":
//      group 0 sampler with repetition penalty; "Known gaps": seen tokens)
//   2. greedy (T == 0 or top_k == 1): argmax, lowest id on ties
//   3. z = l / T, keep the top_k ids by (z desc, id asc) via a radix select
//   4. Gumbel-max over the kept ids, lowest id on ties
// ---------------------------------------------------------------------------

struct SampleSmem {
  float lp[kMaxVocab];
  uint32_t key[kMaxVocab];
  float gn[kMaxVocab];  // Gumbel noise of this thread's ids, when computed ahead (gumbel_ahead)
  int hist[256];
  int wsum[kWarps];
  float redv[kWarps + 1];
  int redi[kWarps + 1];
  int redh[kWarps + 1];
  uint32_t sel_prefix;
  int sel_rem;
  int sel_whole;
};

static_assert(sizeof(SampleSmem) <= kWorkBytes, "the sampler's shared memory fits the work region");

// The noise of this thread's contiguous block of ids (the block sample_row
// gives it) into S.gn, one Philox call per 4 ids; it needs no logits, so the
// sampler stage runs it while the head stage's logits are still arriving.
__device__ void gumbel_ahead(SampleSmem& S, int V, int j, uint32_t key0, uint32_t key1, uint32_t fctr) {
  const int per = (V + kCThreads - 1) / kCThreads;
  const int v0 = min(V, (int)threadIdx.x * per), v1 = min(V, v0 + per);
  for (int q = v0 >> 2; q <= (v1 - 1) >> 2 && v0 < v1; ++q) {
    uint32_t c[4] = {(uint32_t)q, (uint32_t)j, fctr, 0u};
    philox4x32_10(c, key0, key1);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const int v = q * 4 + w;
      if (v >= v0 && v < v1) S.gn[v] = gumbel_of_word(c[w]);
    }
  }
}

// `row`: the raw logits, or nullptr when they are already in S.lp.
// noise_ahead: S.gn holds this thread's noise (gumbel_ahead ran).
__device__ int sample_row(SampleSmem& S, const float* row, int V, int j, const qtts_session& ss,
                          uint32_t key0, uint32_t key1, uint32_t fctr, const uint32_t* seen, int eos_id,
                          int n_codes, bool noise_ahead = false) {
  const int tid = threadIdx.x, lane = tid & 31;
  float T;
  int k;
  if (j == 0) {
    T = ss.temperature;
    k = ss.top_k;
  } else {
    T = ss.cp_temperature;
    k = ss.cp_top_k;
  }
  for (int v = tid; v < V; v += kCThreads) {
    float l = row ? row[v] : S.lp[v];
    if (j == 0) {
      if (v >= n_codes && v != eos_id) l = -INFINITY;
      if (v == eos_id && !ss.eos_allowed) l = -INFINITY;
      if (seen && ((seen[v >> 5] >> (v & 31)) & 1u))
        l = (l > 0.0f) ? __fdiv_rn(l, ss.rep_penalty) : __fmul_rn(l, ss.rep_penalty);
    }
    S.lp[v] = l;
  }
  cbar();

  // contiguous id block per thread, visited in ascending order
  const int per = (V + kCThreads - 1) / kCThreads;
  const int v0 = min(V, tid * per), v1 = min(V, v0 + per);

  if (T == 0.0f || k == 1) {
    bool have = false;
    float bv = 0.f;
    int bi = 0;
    for (int v = v0; v < v1; ++v)
      if (better(true, S.lp[v], v, have, bv, bi)) {
        have = true;
        bv = S.lp[v];
        bi = v;
      }
    return block_argbest(have, bv, bi, S.redv, S.redi, S.redh);
  }

  if (k <= 0 || k > V) k = V;
  for (int v = tid; v < V; v += kCThreads) {
    float z = __fdiv_rn(S.lp[v], T);
    if (z == 0.0f) z = 0.0f;
    S.lp[v] = z;
    S.key[v] = order_key(z);
  }
  cbar();

  const bool take_all = (k == V);
  uint32_t thr = 0u;
  int rem = 0;
  // whole_bin: the selection ended on a digit bin holding exactly the keys
  // still needed, so every key with the prefix thr in the bits of pmask is
  // kept (no ties to rank)
  bool whole_bin = false;
  uint32_t pmask = 0u;
  if (!take_all) {
    // MSB-first radix select of the k-th largest key, 8 bits per pass; a warp
    // adds equal digits together so hot bins see one atomic per warp
    uint32_t prefix = 0u;
    rem = k;
    for (int shift = 24; shift >= 0; shift -= 8) {
      if (tid < 256) S.hist[tid] = 0;
      cbar();
      for (int v0w = tid - lane; v0w < V; v0w += kCThreads) {
        const int v = v0w + lane;
        const uint32_t kk = v < V ? S.key[v] : 0u;
        const bool in = v < V && (kk & pmask) == prefix;
        const unsigned act = __ballot_sync(0xffffffffu, in);
        if (in) {
          const uint32_t dig = (kk >> shift) & 255u;
          const unsigned same = __match_any_sync(act, dig);
          if ((__ffs(same) - 1) == lane) atomicAdd(&S.hist[dig], __popc(same));
        }
      }
      cbar();
      if (tid < 32) {
        // lane L owns digits 255-8L .. 248-8L (descending)
        int part = 0;
        for (int i = 0; i < 8; ++i) part += S.hist[255 - 8 * tid - i];
        int incl = part;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int t = __shfl_up_sync(0xffffffffu, incl, o);
          if (tid >= o) incl += t;
        }
        const int excl = incl - part;
        const unsigned hit = __ballot_sync(0xffffffffu, incl >= rem);
        const int L = __ffs(hit) - 1;
        if (tid == L) {
          int cum = excl;
          int dsel = 255 - 8 * L - 7;
          for (int i = 0; i < 8; ++i) {
            const int dd = 255 - 8 * L - i;
            if (cum + S.hist[dd] >= rem) {
              dsel = dd;
              break;
            }
            cum += S.hist[dd];
          }
          S.sel_prefix = prefix | ((uint32_t)dsel << shift);
          S.sel_rem = rem - cum;
          S.sel_whole = S.hist[dsel] == rem - cum;
        }
      }
      cbar();
      prefix = S.sel_prefix;
      rem = S.sel_rem;
      pmask |= 255u << shift;
      if (S.sel_whole) {
        whole_bin = true;
        break;
      }
    }
    thr = prefix;  // k-th largest key (or, whole_bin, its prefix); `rem` ties with it are kept, lowest ids first
  }

  // exclusive scan of per-thread tie counts gives each tie its rank by id
  int rank = 0;
  if (!take_all && !whole_bin) {
    int ties = 0;
    for (int v = v0; v < v1; ++v) ties += (S.key[v] == thr);
    rank = block_excl_scan(ties, S.wsum);
  }

  bool have = false;
  float bv = 0.f;
  int bi = 0;
  for (int v = v0; v < v1; ++v) {
    bool cand = take_all;
    if (whole_bin) {
      cand = (S.key[v] & pmask) >= thr;
    } else if (!take_all) {
      const uint32_t kk = S.key[v];
      if (kk > thr) {
        cand = true;
      } else if (kk == thr) {
        cand = rank < rem;
        ++rank;
      }
    }
    if (cand) {
      const float val = __fadd_rn(S.lp[v], noise_ahead ? S.gn[v] : gumbel(key0, key1, j, fctr, v));
      if (better(true, val, v, have, bv, bi)) {
        have = true;
        bv = val;
        bi = v;
      }
    }
  }
  return block_argbest(have, bv, bi, S.redv, S.redi, S.redh);
}

// ---------------------------------------------------------------------------
// stage: begin -- validate every session (each CTA reaches the same verdict
// from the same data, so on bad input all CTAs leave together) and publish
// the Talker input rows
// ---------------------------------------------------------------------------

__shared__ int s_kv_len[kMaxBatch];  // each session's kv_len as this launch found it

__device__ __noinline__ bool stage_begin(const StageDesc& d, uint32_t tag, const Globals& g, const FrameArgs& fa) {
  const int tid = threadIdx.x;
  int bad = 0;
  for (int b = tid; b < fa.B; b += kCThreads) {
    const qtts_session s = fa.sess[b];
    const int kv = s_kv_len[b];
    if (kv < 0 || kv + 1 > g.max_context || kv + 1 > fa.bt_stride * kPage) bad = QTTS_DEV_BAD_SESSION;
    if (!(s.temperature >= 0.f) || !isfinite(s.temperature) || !(s.cp_temperature >= 0.f) ||
        !isfinite(s.cp_temperature) || !(s.rep_penalty > 0.f) || !isfinite(s.rep_penalty))
      bad = QTTS_DEV_BAD_SAMPLING;
  }
  for (int b = 0; b < fa.B; ++b) {
    const int kv = s_kv_len[b];
    if (kv < 0 || kv + 1 > fa.bt_stride * kPage) continue;  // reported above
    const int np = kv / kPage + 1;
    for (int p = tid; p < np; p += kCThreads) {
      const int page = fa.bt[(size_t)b * fa.bt_stride + p];
      if (page < 0 || page >= g.pool_pages) bad = QTTS_DEV_BAD_PAGE;
    }
  }
  if (fa.forced)
    for (int i = tid; i < fa.B * kCodebooks; i += kCThreads) {
      const int c = fa.forced[i];
      const int V = (i % kCodebooks) == 0 ? g.V0 : g.Vc;
      if (c < 0 || c >= V) bad = QTTS_DEV_BAD_CODE;
    }
  if (bad && blockIdx.x == 0) set_err(g.err, bad);
  if (cbar_or(bad)) return false;

  const int b = blockIdx.x;
  if (b < fa.B) {
    const uint16_t* src = fa.in_embeds + (size_t)b * g.H;
    uint64_t* dst = d.x_next + (size_t)b * g.H;
    for (int k = tid * 2; k < g.H; k += kCThreads * 2) {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(src + k);
      st_ll2(dst + k, bf_lo(w), bf_hi(w), tag);
    }
  }
  return true;
}

// ---------------------------------------------------------------------------
// stage: GEMV with a fused prologue (RMSNorm) and epilogues
//   Y[rows, N] = X[rows, K] W[N, K]^T, W streamed once for all rows.
// A segment's rows are split over the grid in contiguous row units; this
// CTA's share is cut into tasks of one unit x a 1024-wide slice of K.
// Ring path (rows small enough that the whole activation tile stays in
// shared memory): the producer warp has already copied each task's weights
// into a ring slot. Direct path (larger batches): lanes load the weights
// themselves, once per tile of activation rows.
// The RMSNorm of a row is x g / rms(x): every CTA reads the whole row anyway,
// so it computes rms itself (fixed-order sums, the same on every CTA) and
// applies 1/rms to the dot products.
// ---------------------------------------------------------------------------

constexpr int kKChunk = 1024;
constexpr int kSub = kKChunk / 256;   // 16-byte vectors per lane per row per task
constexpr int kPartFloats = 1536;
constexpr int kResidFloats = 512;
constexpr int kRingSlots = 8;
constexpr int kSlotBytes = 16384;     // whole weight rows, one bulk copy per slot
static_assert(kWorkBytes + kTailBytes + kRingSlots * kSlotBytes + kTcOverread <= kSmemBytes, "shared-memory plan");
// a K step's 128-lane A operand spans (the slice's two 8-column steps of K)
// at most 16 core-matrix rows past its start: 15 x 128 + one K step of the
// smallest (8-row) slice + 128 bytes past the slot's end
static_assert(15 * 128 + kTcRows * 16 + 128 <= kTcOverread, "tensor-path over-read guard");

// Ring-path epilogue operands, loaded in the prologue while the input words
// are polled (the ring path leaves `part` unused)
struct EpiCache {
  float cs[8][64];             // RoPE cos / sin at each tile row's position (d <= 128)
  float sn[8][64];
  int page[8];                 // Talker: KV page of each tile row's appended position
  float scale[2][128];         // int8 row scales of this CTA's share, per segment
};
constexpr int kScaleCache = 128;

struct GemvSmemTail {
  float rfac[8];               // 1/rms of the tile's rows (1 without a norm)
  float sqw[8][kWarps];        // per-warp sum-of-squares partials of the tile's rows
  union {
    float part[kPartFloats];   // direct path: phase-1 partial dot products [task][U][RT]
    EpiCache ec;               // ring path
  };
  float resid[kResidFloats];   // E_RESID operands x[row][unit] [unit][RT], read in the prologue
};
static_assert(sizeof(EpiCache) <= kPartFloats * sizeof(float), "epilogue cache");
static_assert(sizeof(GemvSmemTail) <= kTailBytes, "GEMV shared-memory tail");

// full[x]: the slot's bytes have landed (producer arms it, the bulk copy
// completes it); empty[x]: its consumer is done with it; seq[x]: which use of
// the slot (sequence index / slots in use) the producer has armed last. A
// consumer waits for seq[x] to show its use before its parity wait on
// full[x], so that wait is never for a phase two steps ahead of the barrier
// (several warps consume slots independently).
struct Ring {
  uint64_t full[kRingSlots];
  uint64_t empty[kRingSlots];
  uint32_t seq[kRingSlots];
  uint32_t done[kRingSlots];  // tasks of the slot's current use finished so far
};

__device__ __forceinline__ uint32_t ld_volatile_u32(const uint32_t* p) { return *(const volatile uint32_t*)p; }

// Wait until ring slot `slot` holds use `use` and its bytes have landed.
__device__ bool ring_wait_full(Ring* ring, int slot, uint32_t use, int* err) {
  if (ld_volatile_u32(&ring->seq[slot]) != use) {
    const uint64_t t0 = global_timer_ns();
    unsigned spins = 0;
    while (ld_volatile_u32(&ring->seq[slot]) != use) {
      __nanosleep(64);
      if ((++spins & 15u) == 0u) {
        if (read_err(err)) return false;
        if (global_timer_ns() - t0 > kWaitTimeoutNs) {
          set_err(err, QTTS_DEV_TIMEOUT);
          return false;
        }
      }
    }
  }
  return mbar_wait(&ring->full[slot], use & 1u, err);
}

// Copy a stage descriptor from global to shared memory (one warp).
__device__ __forceinline__ void fetch_desc(const StageDesc* src, StageDesc* dst) {
  constexpr int n = sizeof(StageDesc) / 16;
  static_assert(sizeof(StageDesc) % 16 == 0 && n <= 32, "descriptor copy");
  const int lane = threadIdx.x & 31;
  if (lane < n) reinterpret_cast<int4*>(dst)[lane] = __ldg(reinterpret_cast<const int4*>(src) + lane);
}

__device__ __forceinline__ unsigned char* ring_slot(unsigned char* smem, int slot) {
  return smem + kWorkBytes + kTailBytes + slot * kSlotBytes;
}

// Activation rows per tile of a GEMV stage; 0 when the stage takes the
// direct path. The producer and the compute warps evaluate the same rule.
__device__ __forceinline__ int ring_rt(const StageDesc& d, int B) {
  const int rows = B * d.rps;
  int RT = 1;
  while (RT < rows) RT *= 2;
  if (RT > 8) return 0;
  if (RT * d.K * 4 > kWorkBytes) return 0;
  for (int s = 0; s < d.nseg; ++s)  // a row unit must fit one slot
    if (d.seg[s].unit * d.K * (d.seg[s].scale ? 1 : 2) > kSlotBytes) return 0;
  return RT;
}

// How a GEMV stage runs for batch B: ring path (few rows: CUDA-core dot
// products from the weight ring), tensor path (from g.tc_min_rows up to 64
// rows, weights with a tensor-tile copy, K a multiple of 128: tcgen05 MMAs
// from the weight ring), else direct path (CUDA cores, weights loaded by the
// lanes). The producer and the compute warps evaluate the same rule.
enum GemvMode { GM_RING = 0, GM_TC = 1, GM_DIRECT = 2 };
// Whether a tensor-path segment takes its K-split partition (tc_ksplit) for
// `rows` activation rows of K: from ksplit_min_rows rows up, or when the
// activation words one CTA would stage alone (rows x K) reach kTcSplitWords
// (at B = 8 only the 6144-deep down projection: its one-slice staging costs
// more than the partial-sum exchange).
constexpr int kTcSplitWords = 8 * 6144;
__device__ __forceinline__ bool tc_split(const Seg& sg, int rows, int K, const Globals& g) {
  return sg.wtk != nullptr && (rows >= g.ksplit_min_rows || rows * K >= kTcSplitWords);
}
__device__ __forceinline__ int gemv_mode(const StageDesc& d, int B, const Globals& g) {
  const int rows = B * d.rps;
  bool tc = rows >= g.tc_min_rows && rows <= kTcMaxActRows && d.K % kTcK == 0;
  for (int s = 0; s < d.nseg; ++s) tc = tc && (tc_split(d.seg[s], rows, d.K, g) || d.seg[s].wt != nullptr);
  if (tc) return GM_TC;
  return ring_rt(d, B) > 0 ? GM_RING : GM_DIRECT;
}

// This CTA's share of a segment on the tensor path (with `split`, the K-split
// partition tc_ksplit states, else one K-slice): 16-row groups
// [g0, g0 + rows / 16) over 128-wide K chunks [kc0, kc0 + nkc); per ring
// slot, kps 16-wide K steps of the slice; `wt` the packed tiles it reads.
struct TcShare {
  int S, ks;         // K-slices of the segment, this CTA's slice
  int g0, rows;      // rows [16 g0, 16 g0 + rows) of the segment (rows = 0: nothing to do)
  int kc0, nkc;      // this CTA's K chunks
  int kstep_bytes;   // bytes of the slice per 16-wide K step
  int kps, nslot;    // K steps per ring slot, ring slots of the share
  int es;            // bytes per weight element in the tiles: 2 (bf16) or 1 (int8, widened in the slot)
  const unsigned char* wt;
  __device__ TcShare(const Seg& sg, int K, bool split) {
    S = split ? tc_ksplit(sg.N, K, (int)gridDim.x) : 1;
    wt = (const unsigned char*)(split ? sg.wtk : sg.wt);
    es = sg.scale ? 1 : 2;
    const int C = (int)gridDim.x / max(S, 1);
    ks = (int)blockIdx.x / C;
    const int c = (int)blockIdx.x - ks * C;
    const unsigned ngroups = (unsigned)((sg.N + kTcRows - 1) / kTcRows);
    g0 = (int)(ngroups * c / C);
    rows = ks < S ? ((int)(ngroups * (c + 1) / C) - g0) * kTcRows : 0;
    nkc = S ? K / kTcK / S : 0;
    kc0 = ks * nkc;
    kstep_bytes = rows * 32;  // in the slot (bf16)
    kps = rows ? kSlotBytes / kstep_bytes : 1;
    nslot = rows ? (nkc * (kTcK / 16) + kps - 1) / kps : 0;
  }
};

// This CTA's share of one segment: units [u0, u0 + nu), each cut into nkc
// K-slices (the tasks); on the ring path, slots of `upslot` whole units.
struct SegShare {
  int u0, nu, nkc, upslot, nslot;
  __device__ SegShare(const Seg& sg, int K) {
    const unsigned units = (unsigned)(sg.N / sg.unit);  // units * gridDim.x < 2^32
    u0 = (int)(units * blockIdx.x / gridDim.x);
    nu = (int)(units * (blockIdx.x + 1) / gridDim.x) - u0;
    nkc = (K + kKChunk - 1) / kKChunk;
    const int unit_bytes = sg.unit * K * (sg.scale ? 1 : 2);
    upslot = kSlotBytes / unit_bytes;
    if (upslot < 1) upslot = 1;
    nslot = (nu + upslot - 1) / upslot;
  }
};

struct RowMap {
  int rps, in_rps, in_off;
  __device__ int in_row(int r) const { return (r / rps) * in_rps + in_off + (r % rps); }
};

__device__ __forceinline__ int out_row_of(const Seg& sg, int rps, int r) {
  return (r / rps) * sg.out_rps + sg.out_off + (r % rps);
}

__device__ __forceinline__ uint16_t* talker_kv_ptr(const Globals& g, const FrameArgs& fa, int layer, int b,
                                                    int pos, int kv, int head) {
  int page = fa.bt[(size_t)b * fa.bt_stride + pos / kPage];
  if (page < 0 || page >= g.pool_pages) {  // validated in stage_begin; stay in bounds regardless
    set_err(g.err, QTTS_DEV_BAD_PAGE);
    page = 0;
  }
  return g.kv_pool +
         (((((size_t)layer * g.pool_pages + page) * 2 + kv) * g.nkv + head) * kPage + pos % kPage) * g.d;
}

// KV pool address for a page id already checked against the pool
__device__ __forceinline__ uint16_t* kv_ptr_page(const Globals& g, int layer, int page, int pos, int kv, int head) {
  return g.kv_pool +
         (((((size_t)layer * g.pool_pages + page) * 2 + kv) * g.nkv + head) * kPage + pos % kPage) * g.d;
}

// Code-Predictor cache of one layer, tagged words: [session][K|V][kv head]
// [16 positions][d/2]; K word i holds dims (i, i + d/2), V word i dims
// (2i, 2i + 1), as two bf16.
__device__ __forceinline__ uint64_t* cp_kv_word(const Globals& g, uint64_t* layer_base, int b, int pos, int kv,
                                                 int head) {
  return layer_base + ((((size_t)b * 2 + kv) * g.nkvc + head) * kCodebooks + pos) * (g.dc / 2);
}

// Epilogue for one output unit (rows n0, n0+1 when U == 2) of stage row r.
// ec: the prologue's cache of RoPE factors and pages (ring path; row r of the
// stage is row rt of the tile), or nullptr to read them from global memory.
__device__ __forceinline__ void gemv_epilogue(const StageDesc& d, const Seg& sg, const Globals& g,
                                              const FrameArgs& fa, int n0, float y0, float y1, int r, int rt,
                                              float resid, uint32_t tag, const EpiCache* ec) {
  const int b = r / d.rps, p = r % d.rps;
  const int orow = out_row_of(sg, d.rps, r);
  uint64_t* out = sg.out + (size_t)orow * sg.out_stride;
  switch (sg.epi) {
    case E_QKV_T:
    case E_QKV_CP: {
      const bool talker = sg.epi == E_QKV_T;
      const int hd = talker ? g.d : g.dc;
      const int nq = talker ? g.nq : g.nqc;
      const int nkv = talker ? g.nkv : g.nkvc;
      const int pos = talker ? s_kv_len[b] : d.pos_base + p;
      const int half = hd / 2;
      if (n0 < (nq + nkv) * hd) {
        // rows arrive as rotate-half pairs (i, i + hd/2) of one head
        const bool is_q = n0 < nq * hd;
        const int rel = is_q ? n0 : n0 - nq * hd;
        const int head = rel / hd, i = (rel % hd) / 2;
        const float c = ec ? ec->cs[rt][i] : talker ? g.rope_cos[(size_t)pos * half + i] : g.cp_rope_cos[pos * half + i];
        const float s = ec ? ec->sn[rt][i] : talker ? g.rope_sin[(size_t)pos * half + i] : g.cp_rope_sin[pos * half + i];
        const float o0 = y0 * c - y1 * s;
        const float o1 = y1 * c + y0 * s;
        if (is_q) {
          st_ll(out + head * hd + i, o0, tag);
          st_ll(out + head * hd + i + half, o1, tag);
        } else if (talker) {
          const uint16_t k0 = f2bf(o0), k1 = f2bf(o1);
          uint16_t* kp = ec ? kv_ptr_page(g, d.layer, ec->page[rt], pos, 0, head)
                            : talker_kv_ptr(g, fa, d.layer, b, pos, 0, head);
          kp[i] = k0;
          kp[i + half] = k1;
          uint64_t* kc = d.kvcur + (((size_t)b * 2 + 0) * nkv + head) * hd;
          st_ll(kc + i, bf2f(k0), tag);
          st_ll(kc + i + half, bf2f(k1), tag);
        } else {
          st_ll_raw(cp_kv_word(g, d.cp_kv, b, pos, 0, head) + i, (uint32_t)f2bf(o0) | ((uint32_t)f2bf(o1) << 16),
                    fa.tag0);
        }
      } else {
        const int rel = n0 - (nq + nkv) * hd;
        const int head = rel / hd, e = rel % hd;
        const uint16_t v0 = f2bf(y0), v1 = f2bf(y1);
        if (talker) {
          uint16_t* vp = ec ? kv_ptr_page(g, d.layer, ec->page[rt], pos, 1, head)
                            : talker_kv_ptr(g, fa, d.layer, b, pos, 1, head);
          vp[e] = v0;
          vp[e + 1] = v1;
          st_ll2(d.kvcur + (((size_t)b * 2 + 1) * nkv + head) * hd + e, bf2f(v0), bf2f(v1), tag);
        } else {
          st_ll_raw(cp_kv_word(g, d.cp_kv, b, pos, 1, head) + e / 2, (uint32_t)v0 | ((uint32_t)v1 << 16), fa.tag0);
        }
      }
      break;
    }
    case E_RESID:  // `resid`: the residual x[orow][n0], read in the prologue
      st_ll(out + n0, resid + y0, tag);
      break;
    case E_SWIGLU: {
      const float silu = y0 / (1.0f + expf(-y0));
      st_ll(out + n0 / 2, silu * y1, tag);
      break;
    }
    case E_LOGITS:
      st_ll(out + n0, y0, tag);
      if (n0 + 1 == sg.N && (sg.N & 1)) st_ll(out + n0 + 1, 0.f, tag);  // pad word: rows are read in pairs
      if (fa.logits_out) fa.logits_out[((size_t)b * kCodebooks + d.codebook) * g.V0 + n0] = y0;
      break;
    case E_CPIN: {
      float v = y0;
      if (sg.bias) v += bf2f(sg.bias[n0]);
      st_ll(out + n0, v, tag);
      break;
    }
  }
}

// The same as one out-of-line copy, for the stages that run it once per
// thread per unit (the tensor path): their code stays small.
__device__ __noinline__ void gemv_epilogue_call(const StageDesc& d, const Seg& sg, const Globals& g,
                                                const FrameArgs& fa, int n0, float y0, float y1, int r, float resid,
                                                uint32_t tag) {
  gemv_epilogue(d, sg, g, fa, n0, y0, y1, r, r, resid, tag, nullptr);
}

template <typename WT>
struct Raw8 {
  using T = uint4;  // 8 bf16
  static __device__ __forceinline__ T load(const WT* p) { return ld_stream16(p); }
  static __device__ __forceinline__ T lds(const WT* p) { return *reinterpret_cast<const uint4*>(p); }
  static __device__ __forceinline__ void unpack(const T& v, float o[8]) {
    o[0] = bf_lo(v.x); o[1] = bf_hi(v.x); o[2] = bf_lo(v.y); o[3] = bf_hi(v.y);
    o[4] = bf_lo(v.z); o[5] = bf_hi(v.z); o[6] = bf_lo(v.w); o[7] = bf_hi(v.w);
  }
};
template <>
struct Raw8<int8_t> {
  using T = uint2;  // 8 int8
  static __device__ __forceinline__ T load(const int8_t* p) { return ld_stream8(p); }
  static __device__ __forceinline__ T lds(const int8_t* p) { return *reinterpret_cast<const uint2*>(p); }
  static __device__ __forceinline__ void unpack(const T& v, float o[8]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) o[i] = (float)(int)(int8_t)((v.x >> (8 * i)) & 0xFFu);
#pragma unroll
    for (int i = 0; i < 4; ++i) o[4 + i] = (float)(int)(int8_t)((v.y >> (8 * i)) & 0xFFu);
  }
};

template <int U, int RT>
__device__ __forceinline__ void zero_acc(float (&acc)[U][RT]) {
#pragma unroll
  for (int i = 0; i < U; ++i)
#pragma unroll
    for (int r = 0; r < RT; ++r) acc[i][r] = 0.f;
}

// 1/rms of activation row r of the tile (1 without a norm), from the
// per-warp sums of squares the norm step left before its barrier.
__device__ __forceinline__ float row_rfac(const StageDesc& d, const Globals& g, const GemvSmemTail* tail, int r) {
  if (d.xsrc != X_NORM) return 1.0f;
  float sum = 0.f;
  for (int w = 0; w < kCWarps; ++w) sum += tail->sqw[r][w];
  return 1.0f / sqrtf(sum / (float)d.K + g.eps);
}

// Add one task's dot products to acc: U rows x up to 1024 of K against nr
// activation rows, from registers already holding the weight vectors.
template <typename WT, int U, int RT>
__device__ __forceinline__ void task_fma(const typename Raw8<WT>::T (&raw)[kSub][U], const float* xs, int K, int kb,
                                         int nr, float (&acc)[U][RT]) {
#pragma unroll
  for (int sb = 0; sb < kSub; ++sb) {
    const int k = kb + sb * 256;
    if (k < K) {
      float wv[U][8];
#pragma unroll
      for (int i = 0; i < U; ++i) Raw8<WT>::unpack(raw[sb][i], wv[i]);
#pragma unroll
      for (int r = 0; r < RT; ++r) {
        if (r < nr) {
          const float4 a = *reinterpret_cast<const float4*>(xs + r * K + k);
          const float4 c = *reinterpret_cast<const float4*>(xs + r * K + k + 4);
#pragma unroll
          for (int i = 0; i < U; ++i) {
            float v = acc[i][r];
            v = fmaf(wv[i][0], a.x, v);
            v = fmaf(wv[i][1], a.y, v);
            v = fmaf(wv[i][2], a.z, v);
            v = fmaf(wv[i][3], a.w, v);
            v = fmaf(wv[i][4], c.x, v);
            v = fmaf(wv[i][5], c.y, v);
            v = fmaf(wv[i][6], c.z, v);
            v = fmaf(wv[i][7], c.w, v);
            acc[i][r] = v;
          }
        }
      }
    }
  }
}

// This CTA's share of one segment for stage rows [r0, r0 + nr), in two
// phases. Phase 1 spreads (unit, K-slice) tasks over the compute warps and
// leaves one partial per task in shared memory (ring path: task t's weights
// are in the ring slot of sequence index q + t / tasks per slot; direct path:
// lanes load them). Phase 2 gives each (unit, row) to one thread, which sums
// the partials in K order, scales by 1/rms and runs the epilogue. Each phase
// is its own small function, so the code a stage runs stays in the
// instruction cache from one layer to the next.
// Ring path (few activation rows): each warp takes whole output units of the
// CTA's share, streams every K-chunk of the unit from its ring slot into
// register accumulators, reduces once across lanes and runs the epilogue
// itself (lane r for activation row r): no partials in shared memory, no
// second pass. The warp that finishes a slot's last unit frees the slot.
template <typename WT, int U, int RT>
__device__ void gemv_ring(const StageDesc& d, const Seg& sg, int si, const SegShare& sh, const Globals& g,
                          const FrameArgs& fa, const float* xs, int r0, int nr, GemvSmemTail* tail,
                          unsigned char* smem, Ring* ring, uint32_t q, uint32_t tag) {
  using R = Raw8<WT>;
  const int K = d.K;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t nsl = (uint32_t)g.ring_slots, nsl_shift = (uint32_t)(__ffs(g.ring_slots) - 1);
  const float rfac = lane < nr ? row_rfac(d, g, tail, lane) : 1.0f;  // lane r: activation row r
  for (int ul = warp; ul < sh.nu; ul += kCWarps) {
    const int sl = ul / sh.upslot;
    const int ua = sl * sh.upslot;
    const uint32_t qq = q + (uint32_t)sl;
    const int slot = (int)(qq & (nsl - 1u));
    // a failed wait (time limit or an error elsewhere) leaves zeros and the
    // warp carries on to every CTA barrier; the frame is abandoned after
    // the stage
    if (ul == 0) trace_mark(g, 4);
    const bool got = ring_wait_full(ring, slot, qq >> nsl_shift, g.err);
    if (lane == 0 && ul == ua) trace_ring(g, qq, 1);
    const WT* rowp = (const WT*)ring_slot(smem, slot) + (size_t)(ul - ua) * U * K;
    float acc[U][RT];
    zero_acc(acc);
    for (int kc = 0; kc < sh.nkc; ++kc) {
      const int kb = kc * kKChunk + lane * 8;
      typename R::T raw[kSub][U];
#pragma unroll
      for (int sb = 0; sb < kSub; ++sb)
#pragma unroll
        for (int i = 0; i < U; ++i)
          raw[sb][i] = (got && kb + sb * 256 < K) ? R::lds(rowp + (size_t)i * K + kb + sb * 256) : typename R::T{};
      task_fma<WT, U, RT>(raw, xs, K, kb, nr, acc);
    }
    __syncwarp();
    if (ul == 0) trace_mark(g, 5);
    if (ul == kCWarps) trace_mark(g, 3);
    if (lane == 0 && got) {
      const int slot_units = min(sh.nu, ua + sh.upslot) - ua;
      if (atomicAdd(&ring->done[slot], 1u) + 1u == (uint32_t)slot_units) {
        ring->done[slot] = 0u;
        mbar_arrive(&ring->empty[slot]);
      }
    }
#pragma unroll
    for (int i = 0; i < U; ++i)
#pragma unroll
      for (int r = 0; r < RT; ++r) acc[i][r] = warp_sum(acc[i][r]);
    if (lane < nr) {
      const int n0 = (sh.u0 + ul) * U;
      float y[U];
#pragma unroll
      for (int i = 0; i < U; ++i) {
        float v = acc[i][0];
#pragma unroll
        for (int r = 1; r < RT; ++r)
          if (lane == r) v = acc[i][r];
        v *= rfac;
        if (sg.scale) v *= ul * U + i < kScaleCache ? tail->ec.scale[si][ul * U + i] : sg.scale[n0 + i];
        y[i] = v;
      }
      gemv_epilogue(d, sg, g, fa, n0, y[0], y[U - 1], r0 + lane, lane, tail->resid[ul * RT + lane], tag, &tail->ec);
    }
    if (ul == 0) trace_mark(g, 6);
  }
}

template <typename WT, int U>
__device__ void gemv_ring_rt(int RT, const StageDesc& d, const Seg& sg, int si, const SegShare& sh, const Globals& g,
                             const FrameArgs& fa, const float* xs, int r0, int nr, GemvSmemTail* tail,
                             unsigned char* smem, Ring* ring, uint32_t q, uint32_t tag) {
  switch (RT) {
    case 1: gemv_ring<WT, U, 1>(d, sg, si, sh, g, fa, xs, r0, nr, tail, smem, ring, q, tag); break;
    case 2: gemv_ring<WT, U, 2>(d, sg, si, sh, g, fa, xs, r0, nr, tail, smem, ring, q, tag); break;
    case 4: gemv_ring<WT, U, 4>(d, sg, si, sh, g, fa, xs, r0, nr, tail, smem, ring, q, tag); break;
    default: gemv_ring<WT, U, 8>(d, sg, si, sh, g, fa, xs, r0, nr, tail, smem, ring, q, tag); break;
  }
}

template <typename WT, int U, int RT>
__device__ void gemv_p1_direct(const Seg& sg, int K, const float* xs, int nr, GemvSmemTail* tail) {
  using R = Raw8<WT>;
  const SegShare sh(sg, K);
  const int ntask = sh.nu * sh.nkc;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const WT* W = (const WT*)sg.w;
  for (int t = warp; t < ntask; t += kCWarps) {
    const int ul = t / sh.nkc, kc = t - ul * sh.nkc;
    const int n0 = (sh.u0 + ul) * U;
    const int kb = kc * kKChunk + lane * 8;
    typename R::T raw[kSub][U];
#pragma unroll
    for (int sb = 0; sb < kSub; ++sb) {
      const int k = kb + sb * 256;
#pragma unroll
      for (int i = 0; i < U; ++i) raw[sb][i] = (k < K) ? R::load(W + (size_t)(n0 + i) * K + k) : typename R::T{};
    }
    float acc[U][RT];
    zero_acc(acc);
    task_fma<WT, U, RT>(raw, xs, K, kb, nr, acc);
#pragma unroll
    for (int i = 0; i < U; ++i)
#pragma unroll
      for (int r = 0; r < RT; ++r) {
        const float v = warp_sum(acc[i][r]);
        if (lane == 0) tail->part[(t * U + i) * RT + r] = v;
      }
  }
}

__device__ void gemv_p2(const StageDesc& d, const Seg& sg, const Globals& g, const FrameArgs& fa,
                                     int r0, int nr, int RT, GemvSmemTail* tail, uint32_t tag) {
  const int U = sg.unit;
  const SegShare sh(sg, d.K);
  for (int idx = threadIdx.x; idx < sh.nu * nr; idx += kCThreads) {
    const int ul = idx / nr, r = idx - ul * nr;
    const int n0 = (sh.u0 + ul) * U;
    const float f = tail->rfac[r];
    float y[2] = {0.f, 0.f};
    for (int i = 0; i < U; ++i) {
      float acc = 0.f;
      for (int kc = 0; kc < sh.nkc; ++kc) acc += tail->part[((ul * sh.nkc + kc) * U + i) * RT + r];
      acc *= f;
      y[i] = sg.scale ? acc * sg.scale[n0 + i] : acc;
    }
    gemv_epilogue(d, sg, g, fa, n0, y[0], y[U - 1], r0 + r, r, tail->resid[ul * RT + r], tag, nullptr);
  }
}

// Phase 1 of one segment on the direct path: the variant for the weight
// type, unit and tile height.
__device__ void gemv_p1(const Seg& sg, int K, int RT, const float* xs, int nr, GemvSmemTail* tail) {
#define QTTS_P1_RT(WT_, U_)                                           \
  switch (RT) {                                                       \
    case 1: gemv_p1_direct<WT_, U_, 1>(sg, K, xs, nr, tail); return;  \
    case 2: gemv_p1_direct<WT_, U_, 2>(sg, K, xs, nr, tail); return;  \
    case 4: gemv_p1_direct<WT_, U_, 4>(sg, K, xs, nr, tail); return;  \
    default: gemv_p1_direct<WT_, U_, 8>(sg, K, xs, nr, tail); return; \
  }
  if (sg.scale) {
    if (sg.unit == 2) { QTTS_P1_RT(int8_t, 2) }
    else { QTTS_P1_RT(int8_t, 1) }
  } else {
    if (sg.unit == 2) { QTTS_P1_RT(uint16_t, 2) }
    else { QTTS_P1_RT(uint16_t, 1) }
  }
#undef QTTS_P1_RT
}

// One warp loads the ring-path epilogue operands of a row tile: RoPE factors
// and KV pages of the rows' positions (QKV stages) and the int8 row scales of
// the CTA's share.
__device__ void fill_epi_cache(const StageDesc& d, const Globals& g, const FrameArgs& fa, int r0, int nr, int K,
                               EpiCache* ec) {
  const int lane = threadIdx.x & 31;
  const Seg& s0 = d.seg[0];
  if (s0.epi == E_QKV_T || s0.epi == E_QKV_CP) {
    const bool talker = s0.epi == E_QKV_T;
    const int half = (talker ? g.d : g.dc) / 2;
    for (int r = 0; r < nr; ++r) {
      const int b = (r0 + r) / d.rps, p = (r0 + r) % d.rps;
      const int pos = talker ? s_kv_len[b] : d.pos_base + p;
      const float* cs = talker ? g.rope_cos + (size_t)pos * half : g.cp_rope_cos + pos * half;
      const float* sn = talker ? g.rope_sin + (size_t)pos * half : g.cp_rope_sin + pos * half;
      for (int i = lane; i < half; i += 32) {
        ec->cs[r][i] = cs[i];
        ec->sn[r][i] = sn[i];
      }
      if (talker && lane == 0) {
        int page = fa.bt[(size_t)b * fa.bt_stride + pos / kPage];
        if (page < 0 || page >= g.pool_pages) {  // validated in stage_begin; stay in bounds regardless
          set_err(g.err, QTTS_DEV_BAD_PAGE);
          page = 0;
        }
        ec->page[r] = page;
      }
    }
  }
  for (int si = 0; si < d.nseg; ++si) {
    const Seg& sg = d.seg[si];
    if (!sg.scale) continue;
    const SegShare sh(sg, K);
    const int n = min(sh.nu * sg.unit, kScaleCache);
    for (int i = lane; i < n; i += 32) ec->scale[si][i] = sg.scale[sh.u0 * sg.unit + i];
  }
}

// The int8 weight tiles a bulk copy leaves in a ring slot's upper half (nraw
// bytes) are widened to bf16 over the whole slot, element for element. Exact:
// the byte b of value v gives the float 2^23 + (v + 128) when put under the
// exponent of 2^23 (bits 0x4B000000 | (b ^ 0x80)); subtracting 2^23 + 128
// leaves v, whose float has its low 16 bits zero, so its top half is the
// bf16. Raw step c (1024 bytes) is written to bytes [2048 c, 2048 c + 2048),
// which hold raw bytes of steps 2c - 8 and 2c - 7.
__device__ __forceinline__ uint32_t widen2(uint32_t x, int i) {  // bytes i, i + 1 of x (bias-flipped) as 2 bf16
  const float a = __int_as_float((int)__byte_perm(x, 0x4B000000u, 0x7540u + i)) - 8388736.0f;
  const float b = __int_as_float((int)__byte_perm(x, 0x4B000000u, 0x7541u + i)) - 8388736.0f;
  return (__float_as_uint(a) >> 16) | (__float_as_uint(b) & 0xFFFF0000u);
}
// The whole slot by one warp, in 1024-byte steps in order (each step's reads
// precede its writes, and its output overlaps only raw bytes of steps <= c).
__device__ __forceinline__ void widen_i8_slot(unsigned char* slot, int nraw, int lane) {
  const unsigned char* raw = slot + kSlotBytes / 2;
  for (int c0 = 0; c0 < nraw; c0 += 1024) {
    uint4 v[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int o = c0 + h * 512 + lane * 16;
      v[h] = o < nraw ? *reinterpret_cast<const uint4*>(raw + o) : make_uint4(0u, 0u, 0u, 0u);
    }
    __syncwarp();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int o = c0 + h * 512 + lane * 16;
      if (o < nraw) {
        const uint32_t in[4] = {v[h].x ^ 0x80808080u, v[h].y ^ 0x80808080u, v[h].z ^ 0x80808080u,
                                v[h].w ^ 0x80808080u};
        uint32_t out[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) out[i] = widen2(in[i >> 1], (i & 1) * 2);
        *reinterpret_cast<uint4*>(slot + 2 * o) = make_uint4(out[0], out[1], out[2], out[3]);
        *reinterpret_cast<uint4*>(slot + 2 * o + 16) = make_uint4(out[4], out[5], out[6], out[7]);
      }
    }
    __syncwarp();
  }
}

// Barrier of the tensor path's stager warps only (id 5; 1 is cbar, 2.. the
// Code-Predictor attention groups).
constexpr int kStagerBarrier = 5;
// The same split over `nw` warps, one 1024-byte raw step per
// warp of `nw` warps (warp index w; raw steps <= nw): every warp reads its raw
// bytes, then, after a barrier of the nw warps, writes its widened ones (a
// step's output overlaps earlier steps' raw bytes).
__device__ __forceinline__ void widen_i8_slot_split(unsigned char* slot, int nraw, int w, int lane, int nw) {
  const unsigned char* raw = slot + kSlotBytes / 2;
  uint4 v[2];
  const int c0 = w * 1024;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int o = c0 + h * 512 + lane * 16;
    v[h] = o < nraw ? *reinterpret_cast<const uint4*>(raw + o) : make_uint4(0u, 0u, 0u, 0u);
  }
  asm volatile("bar.sync %0, %1;" ::"n"(kStagerBarrier), "r"(nw * 32) : "memory");
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int o = c0 + h * 512 + lane * 16;
    if (o < nraw) {
      const uint32_t in[4] = {v[h].x ^ 0x80808080u, v[h].y ^ 0x80808080u, v[h].z ^ 0x80808080u,
                              v[h].w ^ 0x80808080u};
      uint32_t out[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) out[i] = widen2(in[i >> 1], (i & 1) * 2);
      *reinterpret_cast<uint4*>(slot + 2 * o) = make_uint4(out[0], out[1], out[2], out[3]);
      *reinterpret_cast<uint4*>(slot + 2 * o + 16) = make_uint4(out[4], out[5], out[6], out[7]);
    }
  }
}
static_assert(kSlotBytes / 2 <= 1024 * 10, "an int8 slot's raw steps must not outnumber the stager warps");

// Tensor-path state kept across stages in shared memory.
struct TcState {
  uint64_t xfree[2];  // MMAs reading X buffer b have completed
  uint64_t done;      // every MMA of the current segment has completed
  uint64_t drain;     // leaving after an error: every MMA issued so far has completed
  uint32_t issued;    // the issuing thread has issued MMAs in this launch
  uint32_t tmem;      // TMEM base (kTmemCols columns)
  uint32_t xuse;      // X-buffer fills so far (buffer = xuse & 1)
  uint32_t nseg;      // tensor segments finished so far (phase of `done`)
};

constexpr int kTcXBytes = 32 * 1024;  // one activation buffer (a pass of 128-wide K chunks)
static_assert(2 * kTcXBytes <= kWorkBytes, "tensor-path A tiles");
static_assert(kTcMaxRows * 128 * 4 <= kWorkBytes, "tensor-path results");
constexpr int kTcIssuer = kCWarps - 1;    // the warp whose lane 0 issues the MMAs
constexpr int kTcStagers = kCWarps - 1;   // warps 0.. that stage activations
constexpr int kTcPairs = (kTcXBytes / 4 / 2 + kTcStagers * 32 - 1) / (kTcStagers * 32);  // word pairs per stager thread per pass

// Tensor path of a GEMV stage (from g.tc_min_rows up to 64 activation rows;
// bf16 weights, or int8 ones widened to bf16 in the ring slot and scaled per
// row in the epilogue): one tcgen05 MMA per 16-wide K step of this CTA's K
// range (all of K, or its K-slice, tc_ksplit), M = 128 lanes holding the activation rows
// twice, bf16 high parts (times the RMSNorm gain) in lanes 0..rows-1 and the
// bf16 low parts x - hi in lanes rows..2 rows-1, so hi + lo carries about 16
// mantissa bits of each fp32 activation (the other lanes read whatever follows
// in the activation buffers and are never used), and N = this CTA's weight
// rows (its packed slice, streamed through the ring). The accumulator stays in
// TMEM over all of K. Stager warps fill 32 KB activation tiles (several
// 128-wide K chunks per pass, two buffers) while the issuer's MMAs read the
// other buffer; a commit frees each weight slot and activation buffer when its
// MMAs are done. The epilogue adds the hi and lo lanes; with a K split, the
// CTAs of the slices exchange partial sums so that each adds up 1/S of the
// share's rows, applies 1/rms and runs their epilogues.
__device__ __noinline__ bool stage_gemv_tc(const StageDesc& d, uint32_t tag, const Globals& g, const FrameArgs& fa,
                              unsigned char* smem, Ring* ring, TcState* ts, uint32_t& q) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rows = fa.B * d.rps;
  const int K = d.K;
  const bool norm = d.xsrc == X_NORM;
  const RowMap rm{d.rps, d.in_rps, d.in_off};
  const uint32_t nsl = (uint32_t)g.ring_slots, nsl_shift = (uint32_t)(__ffs(g.ring_slots) - 1);
  // activation tile of one 128-wide K chunk: meff rows (hi and lo of each
  // activation row, rounded up to 16), lbo bytes per 8-column step of K
  const int meff = (2 * rows + 15) / 16 * 16;
  const int lbo = meff / 8 * 128;
  const int tile_bytes = meff * kTcK * 2;
  const int cpp = kTcXBytes / tile_bytes;  // K chunks per pass
  const int tpr = kTcStagers * 32 / rows;  // stager threads per activation row
  const int srow = tid / tpr, sub = tid - srow * tpr;
  const uint64_t* xrow = srow < rows ? d.x + (size_t)rm.in_row(srow) * d.x_stride : nullptr;
  const uint32_t row_tag = srow < rows ? fa.tag0 + (uint32_t)d.x_ws[srow % d.rps] : 0u;
  float* ssq = reinterpret_cast<float*>(smem + kWorkBytes);  // [kTcStagers * 32] per-thread partial sums of squares
  float* rsq = ssq + kTcStagers * 32;                         // [rows] sums of squares per activation row
  bool ok = true;
  uint32_t xuse = ts->xuse, nseg = ts->nseg;
  for (int si = 0; si < d.nseg; ++si) {
    const Seg& sg = d.seg[si];
    const TcShare sh(sg, K, tc_split(sg, rows, K, g));
    if (sh.rows == 0) continue;  // no rows of this segment on this CTA (the same on all its threads)
    // chunks, K steps and passes below count from the start of the share's K range
    const int nch = sh.nkc, nks = nch * (kTcK / 16);
    const int npass = (nch + cpp - 1) / cpp;
    float sq = 0.f;              // this thread's share of its row's sum of squares
    int slot_j = -1, slot = 0;   // issuer: the weight slot in use
    uint32_t wa = 0;
    const uint32_t idesc = tc_idesc_bf16(128, sh.rows);
    // Stager thread t takes activation row t / tpr and every tpr-th K pair of it.
    for (int pass = 0; pass < npass; ++pass, ++xuse) {
      const int b = (int)(xuse & 1u);
      unsigned char* xb = smem + b * kTcXBytes;
      const int c0 = pass * cpp, c1 = min(nch, c0 + cpp);
      if (warp < kTcStagers) {
        // the MMAs of this buffer's previous fill are done with it
        if (xuse >= 2) ok &= mbar_wait(&ts->xfree[b], ((xuse >> 1) - 1u) & 1u, g.err);
        if (pass == 1) trace_mark(g, 4);
        const int npair = (c1 - c0) * (kTcK / 2);  // pairs of this row in the pass
        for (int j0 = sub; j0 < npair && srow < rows; j0 += kTcPairs * tpr) {
          uint64_t w[kTcPairs][2];
          uint32_t gw[kTcPairs];  // RMSNorm gains of the pairs, loaded with them
          const int n = min(kTcPairs, (npair - j0 + tpr - 1) / tpr);  // this thread's pairs j0 + u tpr, u < n
          const uint64_t* base = xrow + (sh.kc0 + c0) * kTcK + 2 * j0;
          const unsigned* gbase = reinterpret_cast<const unsigned*>(d.gain + (sh.kc0 + c0) * kTcK + 2 * j0);
#pragma unroll
          for (int u = 0; u < kTcPairs; ++u) {
            w[u][0] = w[u][1] = 0;
            gw[u] = 0u;
            if (u < n) {
              ld_ll2(base + (size_t)u * 2 * tpr, w[u][0], w[u][1]);
              if (norm) gw[u] = __ldg(gbase + u * tpr);
            }
          }
          ok &= ll_settle_strided<kTcPairs>(base, 2 * tpr, n, row_tag, w, g.err);
          if (pass == 1 && j0 == sub) trace_mark(g, 5);
#pragma unroll
          for (int u = 0; u < kTcPairs; ++u) {
            if (u >= n) continue;
            const int j = j0 + u * tpr;
            const int cc = (2 * j) / kTcK, kl = (2 * j) % kTcK;  // chunk within the pass, K within the chunk
            float x0 = ll_val(w[u][0]), x1 = ll_val(w[u][1]);
            if (norm) {
              sq = fmaf(x0, x0, sq);
              sq = fmaf(x1, x1, sq);
              x0 *= bf_lo(gw[u]);
              x1 *= bf_hi(gw[u]);
            }
            const uint16_t h0 = f2bf(x0), h1 = f2bf(x1);
            const uint16_t l0 = f2bf(x0 - bf2f(h0)), l1 = f2bf(x1 - bf2f(h1));
            // element (m, k) of a chunk tile: core matrix (k/8, m/8) at (k/8) lbo + (m/8) 128, row m%8, column k%8
            unsigned char* ct = xb + cc * tile_bytes + (kl >> 3) * lbo + (kl & 7) * 2;
            *reinterpret_cast<uint32_t*>(ct + (srow >> 3) * 128 + (srow & 7) * 16) = h0 | ((uint32_t)h1 << 16);
            const int lr = rows + srow;
            *reinterpret_cast<uint32_t*>(ct + (lr >> 3) * 128 + (lr & 7) * 16) = l0 | ((uint32_t)l1 << 16);
          }
        }
        if (sh.es == 1) {
          // widen the int8 weight slots whose first K step is in this pass
          // (the issuer then only waits and issues), one raw step per stager
          // warp; at most ring_slots - 1 of them: those the producer can fill
          // before this pass's MMAs free any slot (the issuer widens the rest)
          const int s_lo = c0 * (kTcK / 16), s_hi = c1 * (kTcK / 16);
          const int jj0 = (s_lo + sh.kps - 1) / sh.kps;
          for (int jj = jj0; jj * sh.kps < s_hi && jj < jj0 + (int)nsl - 1; ++jj) {
            const uint32_t qq = q + (uint32_t)jj;
            const int sl = (int)(qq & (nsl - 1u));
            ok &= ring_wait_full(ring, sl, qq >> nsl_shift, g.err);
            widen_i8_slot_split(ring_slot(smem, sl), (min(nks, (jj + 1) * sh.kps) - jj * sh.kps) * sh.rows * 16, warp,
                                lane, kTcStagers);
          }
        }
        fence_proxy_async_smem();  // the activation tiles (and widened weights) are read by the tensor cores
      }
      cbar();
      if (pass == 0) trace_mark(g, 1);
      if (pass == 1) trace_mark(g, 6);
      if (warp == kTcIssuer) {
        tc_fence_after();
        // activation K step cs of the pass starts at xb + 2 cs lbo (a chunk tile is 16 lbo bytes)
        const int s_end = c1 * (kTcK / 16);
        for (int s = c0 * (kTcK / 16); s < s_end;) {
          const int j = s / sh.kps;
          const int slot_end = min(nks, (j + 1) * sh.kps);
          if (j != slot_j) {  // next weight slot: its first K step is in this pass
            slot_j = j;
            const uint32_t qq = q + (uint32_t)j;
            slot = (int)(qq & (nsl - 1u));
            ok &= ring_wait_full(ring, slot, qq >> nsl_shift, g.err);
            if (lane == 0) trace_ring(g, qq, 1);
            unsigned char* sp = ring_slot(smem, slot);
            // int8: the stagers widened the pass's first ring_slots - 1 new slots; the warp widens the rest
            if (sh.es == 1 && j >= (c0 * (kTcK / 16) + sh.kps - 1) / sh.kps + (int)nsl - 1) {
              widen_i8_slot(sp, (slot_end - j * sh.kps) * sh.rows * 16, lane);
              fence_proxy_async_smem();  // read by the tensor cores next
              __syncwarp();
            }
            wa = smem_addr(sp);
          }
          const int e = min(s_end, slot_end);
          if (lane == 0) {
            ts->issued = 1u;
            uint64_t da = tc_smem_desc(smem_addr(xb) + (uint32_t)((s - c0 * (kTcK / 16)) * 2 * lbo), lbo, 128);
            uint64_t db = tc_smem_desc(wa + (uint32_t)((s - j * sh.kps) * sh.kstep_bytes), sh.rows * 16, 128);
            const uint64_t da_step = (uint64_t)((2 * lbo) >> 4), db_step = (uint64_t)(sh.kstep_bytes >> 4);
            for (int t = s; t < e; ++t) {  // descriptors advance in their 16-byte address field
              tc_mma(ts->tmem, da, db, idesc, t > 0);
              da += da_step;
              db += db_step;
            }
            if (e == slot_end) {
              tc_commit(&ring->empty[slot]);  // the slot is free once these MMAs are done
              trace_ring(g, q + (uint32_t)j, 2);
            }
          }
          s = e;
        }
        if (lane == 0) {
          tc_commit(&ts->xfree[b]);
          if (pass == npass - 1) tc_commit(&ts->done);
        }
      }
      __syncwarp();
    }
    q += (uint32_t)sh.nslot;
    // all MMAs of the segment are done: read the accumulators
    ok &= mbar_wait(&ts->done, nseg & 1u, g.err);
    ++nseg;
    trace_mark(g, 2);
    tc_fence_after();
    float* res = reinterpret_cast<float*>(smem);  // [lane: hi rows, lo rows][slice row], over the activation tiles
    if (warp < 4 && 32 * warp < 2 * rows) {
      const int m = 32 * warp + lane;  // TMEM lane
      for (int cb = 0; cb < sh.rows / 16; ++cb) {
        float v[16];
        tc_ld16(ts->tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)(cb * 16), v);
        if (m < 2 * rows)
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) res[m * sh.rows + cb * 16 + jj] = v[jj];
      }
    }
    tc_fence_before();
    if (norm && warp < kTcStagers) ssq[tid] = sq;
    if (cbar_or(!ok)) return false;
    // fold the low lanes into the high ones (the low half is then free), and
    // each row's sum of squares over the share's K range, in thread order
    const int nsr = sh.rows, nres = rows * nsr;
    for (int idx = tid; idx < nres; idx += kCThreads) {
      res[idx] += res[nres + idx];
      res[nres + idx] = 0.f;
    }
    if (tid < rows) {
      float t = 0.f;
      if (norm)
        for (int i = 0; i < tpr; ++i) t += ssq[tid * tpr + i];
      rsq[tid] = t;
    }
    cbar();
    // K-split exchange area of this segment: per slice, [16 n_groups][rows]
    // partial sums then [rows] partial sums of squares. Rows [o0, o1) of the
    // share belong to this slice: it hands its partial sums of the other
    // slices' rows to them, adds theirs of its own rows and runs the
    // epilogues of its own rows (every slice takes 1/S of the share).
    const int npad = (sg.N + kTcRows - 1) / kTcRows * kTcRows;
    const size_t slice_words = (size_t)npad * rows + rows;
    const int n_base = sh.g0 * kTcRows;
    const int o0 = nsr * sh.ks / sh.S, o1 = nsr * (sh.ks + 1) / sh.S;  // whole units: nsr / S is a multiple of 4
    const int nown = (o1 - o0) * rows;
    if (sh.S > 1) {
      long long off = 0;
      for (int sp = 0; sp < si; ++sp)
        if (tc_split(d.seg[sp], rows, K, g)) off += tc_kpart_words(d.seg[sp].N, K, (int)gridDim.x, kTcMaxActRows);
      uint64_t* kp = g.kpart + (size_t)((tag - fa.tag0) & 1u) * (size_t)g.kpart_words + (size_t)off;
      uint64_t* dst = kp + (size_t)sh.ks * slice_words;
      const int nother = nres - nown;
      for (int idx = tid; idx < nother; idx += kCThreads) {
        int n = idx / rows;
        const int r = idx - n * rows;
        if (n >= o0) n += o1 - o0;  // skip the own rows
        st_ll(dst + (size_t)(n_base + n) * rows + r, res[r * nsr + n], tag);
      }
      if (tid < rows) st_ll(dst + (size_t)npad * rows + tid, rsq[tid], tag);
      cbar();  // the own sums of squares are sent before the others' are added to them
      // the other slices' partial sums of the own rows (in slice order) and their sums of squares
      const int ks = sh.ks;
      ok &= ll_gather_add<4, kTcMaxSplit - 1>(
          nown + rows, sh.S - 1, [&](int) { return tag; },
          [&](int i, int k) {
            const uint64_t* b = kp + (size_t)(k < ks ? k : k + 1) * slice_words;
            if (i >= nown) return b + (size_t)npad * rows + (i - nown);
            const int n = o0 + i / rows, r = i - (i / rows) * rows;
            return b + (size_t)(n_base + n) * rows + r;
          },
          [&](int i) {
            if (i >= nown) return rsq + (i - nown);
            const int n = o0 + i / rows, r = i - (i / rows) * rows;
            return res + r * nsr + n;
          },
          g.err);
    }
    if (sg.epi == E_RESID) {
      // the residual operands of the own rows, into the free low half
      ok &= ll_gather_add<2, 1>(
          nown, 1, [&](int i) { return fa.tag0 + (uint32_t)sg.r_ws[(i % rows) % d.rps]; },
          [&](int i, int) {
            const int n = o0 + i / rows, r = i - (i / rows) * rows;
            const int n0 = min(n_base + n, sg.N - 1);  // padding rows read a real word and never use it
            return sg.resid + (size_t)out_row_of(sg, d.rps, r) * sg.out_stride + n0;
          },
          [&](int i) {
            const int n = o0 + i / rows, r = i - (i / rows) * rows;
            return res + nres + r * nsr + n;
          },
          g.err);
    }
    if (cbar_or(!ok)) return false;
    // epilogue of the own rows: one thread per (unit, activation row)
    const int U = sg.unit;
    const int u_own0 = o0 / U, nunits = (o1 - o0) / U;
    for (int idx = tid; idx < nunits * rows; idx += kCThreads) {
      const int ul = u_own0 + idx / rows, r = idx - (idx / rows) * rows;
      const int n0 = n_base + ul * U;
      if (n0 >= sg.N) continue;  // padding rows of the last group
      const float f = norm ? 1.0f / sqrtf(rsq[r] / (float)K + g.eps) : 1.0f;
      float y[2];
      for (int i = 0; i < U; ++i) y[i] = res[r * nsr + ul * U + i] * f * (sg.scale ? __ldg(sg.scale + n0 + i) : 1.0f);
      const float resid = res[nres + r * nsr + ul * U];
      gemv_epilogue_call(d, sg, g, fa, n0, y[0], y[U - 1], r, resid, tag);
    }
    cbar();  // the results are read; the next fill may overwrite them
    trace_mark(g, 3);
  }
  if (tid == 0) {
    ts->xuse = xuse;
    ts->nseg = nseg;
  }
  return ok;
}

// q: this CTA's count of ring tasks consumed so far (advanced here).
// next / next_s: the following stage's descriptor (or nullptr) and its
// shared-memory buffer, filled by the last compute warp during phase 2.
__device__ __noinline__ bool stage_gemv(const StageDesc& d, uint32_t tag, const Globals& g, const FrameArgs& fa,
                           unsigned char* smem, Ring* ring, TcState* ts, uint32_t& q, const StageDesc* next,
                           StageDesc* next_s) {
  if (gemv_mode(d, fa.B, g) == GM_TC) {
    if (next && (threadIdx.x >> 5) == kCWarps - 2) fetch_desc(next, next_s);
    return stage_gemv_tc(d, tag, g, fa, smem, ring, ts, q);
  }
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rows = fa.B * d.rps;
  const int K = d.K;
  const bool norm = d.xsrc == X_NORM;
  float* xs = (float*)smem;
  GemvSmemTail* tail = (GemvSmemTail*)(smem + kWorkBytes);

  int RT = ring_rt(d, fa.B);
  const bool use_ring = RT > 0;
  if (!use_ring) {
    RT = kWorkBytes / (K * 4);
    RT = RT >= 8 ? 8 : RT >= 4 ? 4 : RT >= 2 ? 2 : 1;
    while (RT > 1 && RT / 2 >= rows) RT /= 2;
  }
  const Seg& s0 = d.seg[0];
  const bool has_resid = s0.epi == E_RESID;  // single-segment stage
  const SegShare sh0(s0, K);

  for (int r0 = 0; r0 < rows; r0 += RT) {
    const int nr = min(RT, rows - r0);
    if (r0) cbar();  // the previous tile is done with the activation rows (the stage loop's barrier covers the first)
    // (1) the tile's input words and this CTA's residual operands: every
    //     load is issued before the first wait, one round trip for the lot
    bool ok = true;
    const int nres = has_resid ? sh0.nu * nr : 0;  // <= kResidFloats <= 2 * kCThreads
    uint64_t rw[2] = {0, 0};
    const uint64_t* rp[2] = {nullptr, nullptr};
    // a single-row tile folds the RMSNorm into the staging: gains loaded with
    // the words, x g stored, sums of squares kept per thread
    const bool fold = norm && nr == 1;
    float sq1 = 0.f;
    {
      constexpr int NB = 4;
      const int hk = K / 2, npair = nr * hk;
      // this thread's pairs follow one another kCThreads apart: pair p of tile row r
      // (no divisions on the way to the first loads)
      int r = tid / hk, p = tid - r * hk;
      const bool two = d.rps == 2;  // rows per session: 1 or 2
      const uint32_t tag_p0 = fa.tag0 + (uint32_t)d.x_ws[0], tag_p1 = fa.tag0 + (uint32_t)d.x_ws[1];
      for (int base = tid; base < npair; base += kCThreads * NB) {
        uint64_t w[NB][2];
        const uint64_t* ps[NB];
        uint32_t tg[NB], gw[NB];
#pragma unroll
        for (int u = 0; u < NB; ++u) {
          const int i = base + u * kCThreads;
          ps[u] = nullptr;
          tg[u] = 0;
          gw[u] = 0;
          w[u][0] = w[u][1] = 0;
          if (i < npair) {
            const int rr = r0 + r;  // stage row: session rr / rps, position rr % rps
            const int in_row = two ? (rr >> 1) * d.in_rps + d.in_off + (rr & 1) : rr * d.in_rps + d.in_off;
            ps[u] = d.x + (size_t)in_row * d.x_stride + 2 * p;
            tg[u] = (two && (rr & 1)) ? tag_p1 : tag_p0;
            ld_ll2(ps[u], w[u][0], w[u][1]);
            if (fold) gw[u] = __ldg(reinterpret_cast<const unsigned*>(d.gain + 2 * p));
          }
          p += kCThreads;
          while (p >= hk) {
            p -= hk;
            ++r;
          }
        }
        if (base == tid) {
          // this CTA's residual operands, issued after the first input loads
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int idx = tid + u * kCThreads;
            if (idx < nres) {
              const int ul = idx / nr, rr = idx - ul * nr;
              rp[u] = s0.resid + (size_t)out_row_of(s0, d.rps, r0 + rr) * s0.out_stride + (sh0.u0 + ul) * s0.unit;
              rw[u] = ld_ll(rp[u]);
            }
          }
          // the epilogue operands (one warp), once its input loads are out
          if (use_ring && warp == kCWarps - 1) fill_epi_cache(d, g, fa, r0, nr, K, &tail->ec);
        }
        ok &= ll_settle<NB>(ps, tg, w, g.err);
#pragma unroll
        for (int u = 0; u < NB; ++u) {
          const int i = base + u * kCThreads;
          if (i < npair) {
            float x0 = ll_val(w[u][0]), x1 = ll_val(w[u][1]);
            if (fold) {
              sq1 = fmaf(x0, x0, sq1);
              sq1 = fmaf(x1, x1, sq1);
              x0 *= bf_lo(gw[u]);
              x1 *= bf_hi(gw[u]);
            }
            *reinterpret_cast<float2*>(xs + 2 * i) = make_float2(x0, x1);
          }
        }
      }
      if (npair <= tid) {
        // no input pair for this thread: the residual operands still go out
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int idx = tid + u * kCThreads;
          if (idx < nres) {
            const int ul = idx / nr, rr = idx - ul * nr;
            rp[u] = s0.resid + (size_t)out_row_of(s0, d.rps, r0 + rr) * s0.out_stride + (sh0.u0 + ul) * s0.unit;
            rw[u] = ld_ll(rp[u]);
          }
        }
        if (use_ring && warp == kCWarps - 1) fill_epi_cache(d, g, fa, r0, nr, K, &tail->ec);
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int idx = tid + u * kCThreads;
      if (idx < nres) {
        const int ul = idx / nr, r = idx - ul * nr;
        ok &= ll_get(rp[u], fa.tag0 + (uint32_t)s0.r_ws[(r0 + r) % d.rps], rw[u], g.err);
        tail->resid[ul * RT + r] = ll_val(rw[u]);
      }
    }
    if (fold) {
      const float t = warp_sum(sq1);
      if (lane == 0) tail->sqw[0][warp] = t;
    }
    if (cbar_or(!ok)) return false;
    // (2) RMSNorm: x <- g x in place, per-warp sums of squares of each row
    if (norm && !fold) {
      for (int r = 0; r < nr; ++r) {
        float sq = 0.f;
        for (int k = tid * 2; k < K; k += kCThreads * 2) {
          float2 v = *reinterpret_cast<float2*>(xs + r * K + k);
          sq = fmaf(v.x, v.x, sq);
          sq = fmaf(v.y, v.y, sq);
          const uint32_t gw = __ldg(reinterpret_cast<const unsigned*>(d.gain + k));
          v.x *= bf_lo(gw);
          v.y *= bf_hi(gw);
          *reinterpret_cast<float2*>(xs + r * K + k) = v;
        }
        sq = warp_sum(sq);
        if (lane == 0) tail->sqw[r][warp] = sq;
      }
      cbar();
    }
    trace_mark(g, 1);
    // 1/rms per row for phase 2 of the direct path (read after the phase-1
    // barrier); ring-path warps take it from the partials themselves
    if (!use_ring && tid < nr) tail->rfac[tid] = row_rfac(d, g, tail, tid);
    for (int s = 0; s < d.nseg; ++s) {
      const Seg& sg = d.seg[s];
      const SegShare sh = s == 0 ? sh0 : SegShare(sg, K);
      // the next descriptor is fetched once, in the last segment of the last row tile
      const bool fetch = next && s == d.nseg - 1 && r0 + RT >= rows;
      if (use_ring) {
        if (fetch && warp == kCWarps - 1) fetch_desc(next, next_s);
        if (sg.scale) {
          if (sg.unit == 2) gemv_ring_rt<int8_t, 2>(RT, d, sg, s, sh, g, fa, xs, r0, nr, tail, smem, ring, q, tag);
          else gemv_ring_rt<int8_t, 1>(RT, d, sg, s, sh, g, fa, xs, r0, nr, tail, smem, ring, q, tag);
        } else {
          if (sg.unit == 2) gemv_ring_rt<uint16_t, 2>(RT, d, sg, s, sh, g, fa, xs, r0, nr, tail, smem, ring, q, tag);
          else gemv_ring_rt<uint16_t, 1>(RT, d, sg, s, sh, g, fa, xs, r0, nr, tail, smem, ring, q, tag);
        }
        q += (uint32_t)sh.nslot;
        cbar();
        trace_mark(g, 2);
      } else {
        gemv_p1(sg, K, RT, xs, nr, tail);
        cbar();
        trace_mark(g, 2);
        if (fetch && warp == kCWarps - 1) fetch_desc(next, next_s);
        gemv_p2(d, sg, g, fa, r0, nr, RT, tail, tag);
        cbar();
        trace_mark(g, 3);
      }
    }
  }
  return true;
}

// ---------------------------------------------------------------------------
// the producer warp: stream every ring-path task's weights, in the order the
// compute warps consume them, into the ring (one elected lane issues)
// ---------------------------------------------------------------------------

__device__ void producer(const StageDesc* prog, int s0, int s1, const Globals& g, const FrameArgs& fa,
                         unsigned char* smem, Ring* ring) {
  const uint64_t policy = l2_evict_first();
  const uint32_t nsl = (uint32_t)g.ring_slots;
  uint32_t q = 0;
  bool ok = true;
  for (int s = s0; s < s1 && ok; ++s) {
    const StageDesc& d = prog[s];
    if (d.type != ST_GEMV) continue;
    const int mode = gemv_mode(d, fa.B, g);
    if (mode == GM_DIRECT) continue;
    const int K = d.K;
    if (mode == GM_TC) {
      for (int si = 0; si < d.nseg && ok; ++si) {
        const TcShare sh(d.seg[si], K, tc_split(d.seg[si], fa.B * d.rps, K, g));
        // the share's K range is contiguous in its slice of the packed tiles;
        // int8 tiles land in the slot's upper half (the compute side widens them)
        const int gstep = sh.rows * 16 * sh.es;  // tile bytes per 16-wide K step
        const unsigned char* W =
            sh.wt + ((size_t)sh.g0 * kTcRows * K + (size_t)sh.kc0 * (kTcK / 16) * sh.rows * 16) * sh.es;
        const int nks = sh.nkc * (kTcK / 16);
        const int dst_off = sh.es == 1 ? kSlotBytes / 2 : 0;
        for (int j = 0; j < sh.nslot; ++j, ++q) {
          const uint32_t bytes = (uint32_t)(min(nks, (j + 1) * sh.kps) - j * sh.kps) * gstep;
          const int slot = (int)(q % nsl);
          if (!mbar_wait(&ring->empty[slot], ((q / nsl) & 1u) ^ 1u, g.err)) {
            ok = false;
            break;
          }
          trace_ring(g, q, 0);
          *(volatile uint32_t*)&ring->seq[slot] = q / nsl;
          mbar_arrive_expect_tx(&ring->full[slot], bytes);
          bulk_load(ring_slot(smem, slot) + dst_off, W + (size_t)j * sh.kps * gstep, bytes, &ring->full[slot], policy);
        }
      }
      continue;
    }
    for (int si = 0; si < d.nseg && ok; ++si) {
      const Seg& sg = d.seg[si];
      const SegShare sh(sg, K);
      const int U = sg.unit;
      const size_t es = sg.scale ? 1 : 2;
      const unsigned char* W = (const unsigned char*)sg.w;
      const size_t unit_bytes = (size_t)U * K * es;
      for (int sl = 0; sl < sh.nslot; ++sl, ++q) {
        const int ua = sl * sh.upslot, ub = min(sh.nu, ua + sh.upslot);
        const uint32_t bytes = (uint32_t)((ub - ua) * unit_bytes);
        const int slot = (int)(q % nsl);
        if (!mbar_wait(&ring->empty[slot], ((q / nsl) & 1u) ^ 1u, g.err)) {
          ok = false;
          break;
        }
        trace_ring(g, q, 0);
        *(volatile uint32_t*)&ring->seq[slot] = q / nsl;
        mbar_arrive_expect_tx(&ring->full[slot], bytes);
        bulk_load(ring_slot(smem, slot), W + (size_t)(sh.u0 + ua) * unit_bytes, bytes, &ring->full[slot], policy);
      }
    }
  }
  // before the warp leaves, every copy it issued has landed (so none writes
  // into shared memory after the CTA is gone)
  const uint32_t first = q > nsl ? q - nsl : 0;
  for (uint32_t qq = first; qq < q; ++qq) {
    if (!mbar_test(&ring->full[qq % nsl], (qq / nsl) & 1u)) {
      const uint64_t t0 = global_timer_ns();
      while (!mbar_test_sleep(&ring->full[qq % nsl], (qq / nsl) & 1u, kSuspendNs))
        if (global_timer_ns() - t0 > kDrainNs) break;
    }
  }
}

// ---------------------------------------------------------------------------
// attention. Talker: one warp per (session, kv head, split); the split's
// 16-position tiles of K and V (one head of one page: 2 x 4 KB contiguous)
// arrive in shared memory by TMA bulk copy, the newest position (written this
// frame) from the tagged K/V rows; online softmax over the tiles.
// Code Predictor: five warps per (row, kv head), all positions from the
// tagged cache in one round trip.
// ---------------------------------------------------------------------------

constexpr int kAttnMaxHD = 128;
constexpr int kAttnMaxGrp = 2;

struct AttnTile {
  uint16_t k[kPage * kAttnMaxHD];
  uint16_t v[kPage * kAttnMaxHD];
  float q[kAttnMaxGrp * kAttnMaxHD];
  uint64_t bar;
  uint64_t pad;
};
constexpr int kAttnWarps = 8;  // warps per CTA that run Talker attention items
static_assert(kAttnWarps * sizeof(AttnTile) <= kWorkBytes, "attention tiles");
constexpr int kCpGroupWarps = 5;                      // warps per Code-Predictor attention item
constexpr int kCpGroups = kCWarps / kCpGroupWarps;    // items in flight per CTA
static_assert(kCpGroups >= 1 && kCpGroups * kCpGroupWarps <= kCWarps, "Code-Predictor attention groups");

template <int HD, int GRP>
struct AttnAcc {
  float o[GRP][HD / 32];
  float m[GRP], l[GRP];
};

template <int HD, int GRP>
__device__ __forceinline__ void attn_init(AttnAcc<HD, GRP>& A) {
#pragma unroll
  for (int j = 0; j < GRP; ++j) {
    A.m[j] = -INFINITY;
    A.l[j] = 0.f;
#pragma unroll
    for (int e = 0; e < HD / 32; ++e) A.o[j][e] = 0.f;
  }
}

// Fold positions 0..nvalid-1 of the tile into A. Scores: lane i & 15 takes
// position i, lane halves split the head dims (each lane starts at a
// different 16-byte column so the row reads do not collide in the banks).
// Values: lanes take E = HD/32 consecutive dims.
template <int HD, int GRP>
__device__ void attn_tile(const AttnTile& T, int nvalid, float scale, AttnAcc<HD, GRP>& A) {
  const int lane = threadIdx.x & 31;
  constexpr int E = HD / 32;
  constexpr int HH = HD / 2;
  const int i = lane & 15, half = lane >> 4;
  const bool valid = i < nvalid;
  float sc[GRP];
#pragma unroll
  for (int j = 0; j < GRP; ++j) sc[j] = 0.f;
  const uint16_t* krow = T.k + i * HD + half * HH;
#pragma unroll 4
  for (int tt = 0; tt < HH; tt += 8) {
    const int t = (tt + i * 8) & (HH - 1);
    const uint4 kv = *reinterpret_cast<const uint4*>(krow + t);
    const float k8[8] = {bf_lo(kv.x), bf_hi(kv.x), bf_lo(kv.y), bf_hi(kv.y),
                         bf_lo(kv.z), bf_hi(kv.z), bf_lo(kv.w), bf_hi(kv.w)};
#pragma unroll
    for (int j = 0; j < GRP; ++j) {
      const float* q = T.q + j * HD + half * HH + t;
#pragma unroll
      for (int e = 0; e < 8; ++e) sc[j] = fmaf(q[e], k8[e], sc[j]);
    }
  }
  float pj[GRP];
#pragma unroll
  for (int j = 0; j < GRP; ++j) {
    sc[j] += __shfl_xor_sync(0xffffffffu, sc[j], 16);
    const float s = valid ? sc[j] * scale : -INFINITY;
    const float mnew = fmaxf(A.m[j], warp_max(s));
    const float corr = expf(A.m[j] - mnew);
    pj[j] = valid ? expf(s - mnew) : 0.f;
    A.l[j] = A.l[j] * corr + warp_sum(half == 0 ? pj[j] : 0.f);
#pragma unroll
    for (int e = 0; e < E; ++e) A.o[j][e] *= corr;
    A.m[j] = mnew;
  }
  for (int p = 0; p < nvalid; ++p) {
    float v[E];
    const uint16_t* vr = T.v + p * HD + lane * E;
    if constexpr (E == 4) {
      const uint2 w = *reinterpret_cast<const uint2*>(vr);
      v[0] = bf_lo(w.x); v[1] = bf_hi(w.x); v[2] = bf_lo(w.y); v[3] = bf_hi(w.y);
    } else {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(vr);
      v[0] = bf_lo(w);
      v[1] = bf_hi(w);
    }
#pragma unroll
    for (int j = 0; j < GRP; ++j) {
      const float pp = __shfl_sync(0xffffffffu, pj[j], p);
#pragma unroll
      for (int e = 0; e < E; ++e) A.o[j][e] = fmaf(pp, v[e], A.o[j][e]);
    }
  }
}

// One 16-position tile by bulk copy (K then V of one head), then fold it in.
// cur_row >= 0: row cur_row of the tile is the position this frame appends;
// its K and V come from the tagged words (kw, vw: this lane's word pairs
// 2(lane + 32u), +1), not from the cache.
template <int HD, int GRP>
__device__ bool attn_fetch_fold(AttnTile& T, const uint16_t* ksrc, const uint16_t* vsrc, int nvalid, float scale,
                                uint32_t& parity, int* err, AttnAcc<HD, GRP>& A, int cur_row,
                                const uint64_t (&kw)[HD / 64][2], const uint64_t (&vw)[HD / 64][2]) {
  const int lane = threadIdx.x & 31;
  constexpr uint32_t bytes = kPage * HD * sizeof(uint16_t);
  __syncwarp();
  if (lane == 0) {
    fence_proxy_async_smem();
    const uint64_t policy = l2_evict_first();
    mbar_arrive_expect_tx(&T.bar, 2 * bytes);
    bulk_load(T.k, ksrc, bytes, &T.bar, policy);
    bulk_load(T.v, vsrc, bytes, &T.bar, policy);
  }
  const bool got = mbar_wait(&T.bar, parity, err);
  if (!got) mbar_drain(&T.bar, parity);  // never leave with the copy still landing
  const bool ok = __all_sync(0xffffffffu, got);  // one verdict per warp
  parity ^= 1u;
  if (ok) {
    if (cur_row >= 0) {
#pragma unroll
      for (int u = 0; u < HD / 64; ++u) {
        const int c = 2 * (lane + 32 * u);
        const uint32_t kk = (uint32_t)f2bf(ll_val(kw[u][0])) | ((uint32_t)f2bf(ll_val(kw[u][1])) << 16);
        const uint32_t vv = (uint32_t)f2bf(ll_val(vw[u][0])) | ((uint32_t)f2bf(ll_val(vw[u][1])) << 16);
        *reinterpret_cast<uint32_t*>(T.k + cur_row * HD + c) = kk;
        *reinterpret_cast<uint32_t*>(T.v + cur_row * HD + c) = vv;
      }
      __syncwarp();
    }
    attn_tile<HD, GRP>(T, nvalid, scale, A);
  }
  return ok;
}

template <int HD, int GRP>
__device__ __noinline__ bool stage_attn_talker(const StageDesc& d, uint32_t tag, const Globals& g, const FrameArgs& fa,
                                  unsigned char* smem) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int E = HD / 32;
  constexpr int NQ = GRP * HD / 64;  // q word pairs per lane
  constexpr int NC = HD / 64;        // current K (and V) word pairs per lane
  const int nkv = g.nkv;
  const int qstride = d.q_stride;
  if (warp >= kAttnWarps) return true;
  AttnTile& T = reinterpret_cast<AttnTile*>(smem)[warp];
  if (lane == 0) {
    mbar_init(&T.bar, 1);
    mbar_init_fence();
  }
  __syncwarp();
  uint32_t parity = 0;
  bool ok = true;
  const uint32_t tag_in = fa.tag0 + (uint32_t)d.q_ws;
  // split plan, identical on every CTA (same inputs, same arithmetic): the
  // smallest page-aligned split length whose splits (each session's rounded
  // up) number at most one per warp of the grid, so no warp runs two in turn
  const int len = lane < fa.B ? s_kv_len[lane] + 1 : 0;
  int total = len;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) total += __shfl_xor_sync(0xffffffffu, total, o);
  const int target = g.G * kAttnWarps;
  int chunk = (total * nkv + target - 1) / target;
  chunk = ((chunk + kPage - 1) / kPage) * kPage;
  if (chunk < kMinChunk) chunk = kMinChunk;
  for (;;) {  // ends by kMaxContext at the latest (one split per session)
    int cnt = (len + chunk - 1) / chunk * nkv;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    if (cnt <= target || chunk >= kMaxContext) break;
    chunk += kPage;
  }
  const int nsp = (len + chunk - 1) / chunk;
  int incl = nsp * nkv;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  const int n_items = __shfl_sync(0xffffffffu, incl, 31);
  const float scale = rsqrtf((float)HD);
  const int layer = d.layer;

  // item i goes to CTA i % G, so the splits spread over the SMs first
  for (int item = warp * g.G + blockIdx.x; item < n_items && ok; item += g.G * kAttnWarps) {
    const unsigned hit = __ballot_sync(0xffffffffu, incl > item);
    const int b = __ffs(hit) - 1;
    const int before = __shfl_sync(0xffffffffu, incl - nsp * nkv, b);
    const int nsp_b = __shfl_sync(0xffffffffu, nsp, b);
    const int len_b = __shfl_sync(0xffffffffu, len, b);
    const int rem = item - before;
    const int kvh = rem / nsp_b, sp = rem % nsp_b;
    const int p0 = sp * chunk, p1 = min(p0 + chunk, len_b);
    const int cur = len_b - 1;          // the position this frame appends
    const bool has_cur = p1 == len_b;   // ... lies in this split's last tile
    // q and the current K/V words: all loads issued, then the waits
    const uint64_t* qsrc = d.q + (size_t)b * qstride + kvh * GRP * HD;
    const uint64_t* kc = d.kvcur + (((size_t)b * 2 + 0) * nkv + kvh) * HD;
    const uint64_t* vc = d.kvcur + (((size_t)b * 2 + 1) * nkv + kvh) * HD;
    uint64_t qw[NQ][2], kw[NC][2], vw[NC][2];
    const uint64_t *pq[NQ], *pk[NC], *pv[NC];
    uint32_t tq[NQ], tk[NC];
#pragma unroll
    for (int u = 0; u < NQ; ++u) {
      pq[u] = qsrc + 2 * (lane + 32 * u);
      tq[u] = tag_in;
      ld_ll2(pq[u], qw[u][0], qw[u][1]);
    }
#pragma unroll
    for (int u = 0; u < NC; ++u) {
      kw[u][0] = kw[u][1] = vw[u][0] = vw[u][1] = 0;
      pk[u] = has_cur ? kc + 2 * (lane + 32 * u) : nullptr;
      pv[u] = has_cur ? vc + 2 * (lane + 32 * u) : nullptr;
      tk[u] = tag_in;
      if (has_cur) {
        ld_ll2(pk[u], kw[u][0], kw[u][1]);
        ld_ll2(pv[u], vw[u][0], vw[u][1]);
      }
    }
    ok &= ll_settle<NQ>(pq, tq, qw, g.err);
    ok &= ll_settle<NC>(pk, tk, kw, g.err);
    ok &= ll_settle<NC>(pv, tk, vw, g.err);
    __syncwarp();
#pragma unroll
    for (int u = 0; u < NQ; ++u) {
      const int c = 2 * (lane + 32 * u);
      T.q[c] = ll_val(qw[u][0]);
      T.q[c + 1] = ll_val(qw[u][1]);
    }
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) break;
    AttnAcc<HD, GRP> A;
    attn_init(A);
    for (int pt = p0; pt < p1 && ok; pt += kPage)
      ok = attn_fetch_fold<HD, GRP>(T, talker_kv_ptr(g, fa, layer, b, pt, 0, kvh),
                                    talker_kv_ptr(g, fa, layer, b, pt, 1, kvh), min(kPage, p1 - pt), scale, parity,
                                    g.err, A, (has_cur && cur < pt + kPage) ? cur - pt : -1, kw, vw);
    if (!ok) break;
    uint64_t* out = d.attn_out + (size_t)b * qstride + kvh * GRP * HD;
    if (nsp_b == 1) {
#pragma unroll
      for (int j = 0; j < GRP; ++j)
#pragma unroll
        for (int e = 0; e < E; ++e) st_ll(out + j * HD + lane * E + e, A.o[j][e] / A.l[j], tag);
    } else {
      // partial (m, l, o) per query head; the last split to finish combines
      float* part = g.attn_part + ((((size_t)b * nkv + kvh) * kMaxSplits + sp) * GRP) * (HD + 2);
#pragma unroll
      for (int j = 0; j < GRP; ++j) {
        float* pj = part + j * (HD + 2);
        if (lane == 0) {
          pj[0] = A.m[j];
          pj[1] = A.l[j];
        }
#pragma unroll
        for (int e = 0; e < E; ++e) pj[2 + lane * E + e] = A.o[j][e];
      }
      __threadfence();
      __syncwarp();
      unsigned old = 0;
      // arrivals wrap back to zero on the last one, ready for the next frame
      if (lane == 0) old = atomicInc(&g.attn_cnt[((size_t)layer * kMaxBatch + b) * nkv + kvh], (unsigned)(nsp_b - 1));
      old = __shfl_sync(0xffffffffu, old, 0);
      if (old == (unsigned)(nsp_b - 1)) {
        __threadfence();
        const float* base = g.attn_part + ((((size_t)b * nkv + kvh) * kMaxSplits) * GRP) * (HD + 2);
#pragma unroll
        for (int j = 0; j < GRP; ++j) {
          // lanes own splits for the max and the denominator
          float M = -INFINITY;
          float ms[kMaxSplits / 32], ls[kMaxSplits / 32];
#pragma unroll
          for (int t = 0; t < kMaxSplits / 32; ++t) {
            const int s2 = lane + 32 * t;
            ms[t] = -INFINITY;
            ls[t] = 0.f;
            if (s2 < nsp_b) {
              const float* ps = base + ((size_t)s2 * GRP + j) * (HD + 2);
              ms[t] = __ldcg(ps);
              ls[t] = __ldcg(ps + 1);
            }
          }
#pragma unroll
          for (int t = 0; t < kMaxSplits / 32; ++t) M = fmaxf(M, ms[t]);
          M = warp_max(M);
          float L = 0.f;
#pragma unroll
          for (int t = 0; t < kMaxSplits / 32; ++t)
            if (lane + 32 * t < nsp_b) L += expf(ms[t] - M) * ls[t];
          L = warp_sum(L);
          // lanes own head dimensions for the weighted sum, 4 splits per batch of loads
          float o[E];
#pragma unroll
          for (int e = 0; e < E; ++e) o[e] = 0.f;
          for (int s0 = 0; s0 < nsp_b; s0 += 4) {
            float mv[4], ov[4][E];
#pragma unroll
            for (int u = 0; u < 4; ++u)
              if (s0 + u < nsp_b) {
                const float* ps = base + ((size_t)(s0 + u) * GRP + j) * (HD + 2);
                mv[u] = __ldcg(ps);
#pragma unroll
                for (int e = 0; e < E; ++e) ov[u][e] = __ldcg(ps + 2 + lane * E + e);
              }
#pragma unroll
            for (int u = 0; u < 4; ++u)
              if (s0 + u < nsp_b) {
                const float w = expf(mv[u] - M);
#pragma unroll
                for (int e = 0; e < E; ++e) o[e] = fmaf(w, ov[u][e], o[e]);
              }
          }
#pragma unroll
          for (int e = 0; e < E; ++e) st_ll(out + j * HD + lane * E + e, o[e] / L, tag);
        }
      }
    }
  }
  __syncwarp();
  if (lane == 0) mbar_inval(&T.bar);
  return ok;
}

// named barrier of one Code-Predictor attention group (ids 2.. ; 1 is cbar)
__device__ __forceinline__ void group_bar(int grp) {
  asm volatile("bar.sync %0, %1;" ::"r"(2 + grp), "n"(kCpGroupWarps * 32) : "memory");
}

template <int HD, int GRP>
__device__ __noinline__ bool stage_attn_cp(const StageDesc& d, uint32_t tag, const Globals& g, const FrameArgs& fa,
                              unsigned char* smem) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = warp / kCpGroupWarps, gw = warp - grp * kCpGroupWarps;
  if (grp >= kCpGroups) return true;  // warps beyond the last whole group sit this stage out
  constexpr int GT = kCpGroupWarps * 32;
  const int gt = gw * 32 + lane;
  constexpr int E = HD / 32;
  constexpr int HH = HD / 2;
  // word pairs per item: q (GRP*HD words), then K and V (16 positions x HD/2 words each)
  constexpr int NQ2 = GRP * HD / 2;
  constexpr int NB = (NQ2 + 2 * kCodebooks * HD / 4 + GT - 1) / GT;
  const int nkv = g.nkvc;
  const int rows = fa.B * d.rps;
  AttnTile& T = reinterpret_cast<AttnTile*>(smem)[grp];
  const uint32_t tag_q = fa.tag0 + (uint32_t)d.q_ws, tag_kv = fa.tag0;
  const float scale = rsqrtf((float)HD);
  bool ok = true;
  // item i goes to CTA i % G, then to the CTA's next group
  for (int item = grp * g.G + blockIdx.x; item < rows * nkv; item += g.G * kCpGroups) {
    const int r = item / nkv, kvh = item % nkv;
    const int b = r / d.rps, p = r % d.rps;
    const int npos = d.pos_base + p + 1;  // positions 0..pos, all written this frame
    const int nk2 = npos * HD / 4;
    const int total = NQ2 + 2 * nk2;
    const uint64_t* qsrc = d.q + (size_t)r * d.q_stride + kvh * GRP * HD;
    const uint64_t* kb = cp_kv_word(g, d.cp_kv, b, 0, 0, kvh);
    const uint64_t* vb = cp_kv_word(g, d.cp_kv, b, 0, 1, kvh);
    uint64_t w[NB][2];
    const uint64_t* ps[NB];
    uint32_t tg[NB];
#pragma unroll
    for (int u = 0; u < NB; ++u) {
      const int i = gt + u * GT;
      ps[u] = nullptr;
      tg[u] = i < NQ2 ? tag_q : tag_kv;
      w[u][0] = w[u][1] = 0;
      if (i < total) {
        ps[u] = i < NQ2 ? qsrc + 2 * i : i < NQ2 + nk2 ? kb + 2 * (i - NQ2) : vb + 2 * (i - NQ2 - nk2);
        ld_ll2(ps[u], w[u][0], w[u][1]);
      }
    }
    ok &= ll_settle<NB>(ps, tg, w, g.err);
#pragma unroll
    for (int u = 0; u < NB; ++u) {
      const int i = gt + u * GT;
      if (i < total) {
        if (i < NQ2) {
          T.q[2 * i] = ll_val(w[u][0]);
          T.q[2 * i + 1] = ll_val(w[u][1]);
        } else if (i < NQ2 + nk2) {
          const int c = 2 * (i - NQ2), pos = c / HH, wi = c - pos * HH;  // words wi, wi + 1
          uint16_t* kr = T.k + pos * HD;
          kr[wi] = (uint16_t)w[u][0];
          kr[wi + HH] = (uint16_t)(w[u][0] >> 16);
          kr[wi + 1] = (uint16_t)w[u][1];
          kr[wi + 1 + HH] = (uint16_t)(w[u][1] >> 16);
        } else {
          const int c = 2 * (i - NQ2 - nk2), pos = c / HH, wi = c - pos * HH;
          *reinterpret_cast<uint2*>(T.v + pos * HD + 2 * wi) = make_uint2((uint32_t)w[u][0], (uint32_t)w[u][1]);
        }
      }
    }
    group_bar(grp);
    if (gw == 0) {
      AttnAcc<HD, GRP> A;
      attn_init(A);
      attn_tile<HD, GRP>(T, npos, scale, A);
      uint64_t* out = d.attn_out + (size_t)r * d.q_stride + kvh * GRP * HD;
#pragma unroll
      for (int j = 0; j < GRP; ++j)
#pragma unroll
        for (int e = 0; e < E; ++e) st_ll(out + j * HD + lane * E + e, A.o[j][e] / A.l[j], tag);
    }
    group_bar(grp);
  }
  return ok;
}

// Talker attention for few, short sessions: one CTA per (session, kv head).
// Its attention warps take the 16-position tiles round-robin (each tile by
// TMA bulk copy, the newest position from the tagged K/V rows), then the
// CTA combines the warps' partial softmax states in shared memory, in warp
// order. No cross-CTA split, so no partials in global memory, fences or
// arrival counters.
constexpr int kCtaAttnMaxTiles = 4 * kAttnWarps;  // contexts up to 512 positions take this path

template <int HD, int GRP>
__device__ __noinline__ bool stage_attn_talker_cta(const StageDesc& d, uint32_t tag, const Globals& g, const FrameArgs& fa,
                                      unsigned char* smem) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int E = HD / 32;
  constexpr int NQ = GRP * HD / 64;  // q word pairs per lane
  constexpr int NC = HD / 64;        // current K (and V) word pairs per lane
  constexpr int PS = HD + 2;         // one partial: m, l, o[HD]
  const int nkv = g.nkv;
  const int qstride = d.q_stride;
  const uint32_t tag_in = fa.tag0 + (uint32_t)d.q_ws;
  const float scale = rsqrtf((float)HD);
  AttnTile* tiles = reinterpret_cast<AttnTile*>(smem);
  float* part = reinterpret_cast<float*>(smem + kWorkBytes);  // [kAttnWarps][GRP][PS]
  static_assert(kAttnWarps * GRP * PS * sizeof(float) <= kTailBytes, "attention partials");
  if (warp < kAttnWarps && lane == 0) {
    mbar_init(&tiles[warp].bar, 1);
    mbar_init_fence();
  }
  __syncwarp();
  uint32_t parity = 0;
  bool ok = true;
  for (int item = blockIdx.x; item < fa.B * nkv; item += g.G) {  // the same trip count on every warp
    const int b = item / nkv, kvh = item - (item / nkv) * nkv;
    const int len = s_kv_len[b] + 1, cur = len - 1;
    const int ntile = (len + kPage - 1) / kPage;
    if (warp < kAttnWarps) {
      AttnTile& T = tiles[warp];
      AttnAcc<HD, GRP> A;
      attn_init(A);
      ok = __all_sync(0xffffffffu, ok);
      if (warp < ntile && ok) {
        const bool has_cur = (ntile - 1) % kAttnWarps == warp;  // this warp folds the last tile
        const uint64_t* qsrc = d.q + (size_t)b * qstride + kvh * GRP * HD;
        const uint64_t* kc = d.kvcur + (((size_t)b * 2 + 0) * nkv + kvh) * HD;
        const uint64_t* vc = d.kvcur + (((size_t)b * 2 + 1) * nkv + kvh) * HD;
        uint64_t qw[NQ][2], kw[NC][2], vw[NC][2];
        const uint64_t *pq[NQ], *pk[NC], *pv[NC];
        uint32_t tq[NQ], tk[NC];
#pragma unroll
        for (int u = 0; u < NQ; ++u) {
          pq[u] = qsrc + 2 * (lane + 32 * u);
          tq[u] = tag_in;
          ld_ll2(pq[u], qw[u][0], qw[u][1]);
        }
#pragma unroll
        for (int u = 0; u < NC; ++u) {
          kw[u][0] = kw[u][1] = vw[u][0] = vw[u][1] = 0;
          pk[u] = has_cur ? kc + 2 * (lane + 32 * u) : nullptr;
          pv[u] = has_cur ? vc + 2 * (lane + 32 * u) : nullptr;
          tk[u] = tag_in;
          if (has_cur) {
            ld_ll2(pk[u], kw[u][0], kw[u][1]);
            ld_ll2(pv[u], vw[u][0], vw[u][1]);
          }
        }
        ok &= ll_settle<NQ>(pq, tq, qw, g.err);
        ok &= ll_settle<NC>(pk, tk, kw, g.err);
        ok &= ll_settle<NC>(pv, tk, vw, g.err);
        __syncwarp();
#pragma unroll
        for (int u = 0; u < NQ; ++u) {
          const int c = 2 * (lane + 32 * u);
          T.q[c] = ll_val(qw[u][0]);
          T.q[c + 1] = ll_val(qw[u][1]);
        }
        ok = __all_sync(0xffffffffu, ok);
        for (int t = warp; t < ntile && ok; t += kAttnWarps) {
          const int pt = t * kPage;
          ok = attn_fetch_fold<HD, GRP>(T, talker_kv_ptr(g, fa, d.layer, b, pt, 0, kvh),
                                        talker_kv_ptr(g, fa, d.layer, b, pt, 1, kvh), min(kPage, len - pt), scale,
                                        parity, g.err, A, t == ntile - 1 ? cur - pt : -1, kw, vw);
        }
      }
      float* pw = part + (size_t)warp * GRP * PS;
#pragma unroll
      for (int j = 0; j < GRP; ++j) {
        if (lane == 0) {
          pw[j * PS] = A.m[j];
          pw[j * PS + 1] = A.l[j];
        }
#pragma unroll
        for (int e = 0; e < E; ++e) pw[j * PS + 2 + lane * E + e] = A.o[j][e];
      }
    }
    cbar();
    const int nw = min(ntile, kAttnWarps);
    uint64_t* out = d.attn_out + (size_t)b * qstride + kvh * GRP * HD;
    for (int idx = threadIdx.x; idx < GRP * HD; idx += kCThreads) {
      const int j = idx / HD, e = idx - j * HD;
      float M = -INFINITY;
      for (int w = 0; w < nw; ++w) M = fmaxf(M, part[(w * GRP + j) * PS]);
      float L = 0.f, o = 0.f;
      for (int w = 0; w < nw; ++w) {
        const float* pw = part + (w * GRP + j) * PS;
        const float wt = expf(pw[0] - M);
        L = fmaf(wt, pw[1], L);
        o = fmaf(wt, pw[2 + e], o);
      }
      st_ll(out + idx, o / L, tag);
    }
    cbar();  // the tiles and partials are reused by the next item
  }
  __syncwarp();
  if (warp < kAttnWarps && lane == 0) mbar_inval(&tiles[warp].bar);
  return ok;
}

// The CTA-per-head path when every (session, kv head) gets its own CTA in
// one round and the longest context fits its tiles; else the split path.
__device__ __forceinline__ bool talker_attn_by_cta(const Globals& g, const FrameArgs& fa) {
  if (fa.B * g.nkv > g.G) return false;
  int longest = 0;
  for (int b = 0; b < fa.B; ++b) longest = max(longest, s_kv_len[b] + 1);
  return (longest + kPage - 1) / kPage <= kCtaAttnMaxTiles;
}

template <bool TALKER>
__device__ bool stage_attn(const StageDesc& d, uint32_t tag, const Globals& g, const FrameArgs& fa,
                           unsigned char* smem) {
  const int hd = TALKER ? g.d : g.dc;
  const int grp = TALKER ? g.nq / g.nkv : g.nqc / g.nkvc;
  const bool by_cta = TALKER && talker_attn_by_cta(g, fa);
#define QTTS_ATTN_CASE(H_, G_)                                                                  \
  if (hd == H_ && grp == G_)                                                                    \
    return TALKER ? (by_cta ? stage_attn_talker_cta<H_, G_>(d, tag, g, fa, smem)                \
                            : stage_attn_talker<H_, G_>(d, tag, g, fa, smem))                   \
                  : stage_attn_cp<H_, G_>(d, tag, g, fa, smem);
  QTTS_ATTN_CASE(128, 2)
  QTTS_ATTN_CASE(64, 2)
  QTTS_ATTN_CASE(128, 1)
  QTTS_ATTN_CASE(64, 1)
#undef QTTS_ATTN_CASE
  return true;
}

// ---------------------------------------------------------------------------
// stage: sampler for codebook j (one CTA per session), then the next
// Code-Predictor input: the projected embedding row T_j[c] of the committed
// code
// ---------------------------------------------------------------------------

__device__ __noinline__ bool stage_sample(const StageDesc& d, uint32_t tag, const Globals& g, const FrameArgs& fa,
                             unsigned char* smem) {
  const int b = blockIdx.x;
  if (b >= fa.B) return true;
  const int tid = threadIdx.x;
  SampleSmem& S = *reinterpret_cast<SampleSmem*>(smem);
  const int j = d.codebook;
  const int V = d.V;
  const qtts_session ss = fa.sess[b];
  const qtts_rng rs = fa.rng[b];
  // the noise does not depend on the logits: compute it while they arrive
  const bool greedy = (j == 0 ? ss.temperature : ss.cp_temperature) == 0.0f || (j == 0 ? ss.top_k : ss.cp_top_k) == 1;
  if (!greedy) gumbel_ahead(S, V, j, rs.key0, rs.key1, rs.frame_ctr);
  // the session's logits, tagged by the head stage
  {
    constexpr int NB = (kMaxVocab / 2 + kCThreads - 1) / kCThreads;
    const uint32_t tl = fa.tag0 + (uint32_t)d.l_ws;
    const uint64_t* src = d.logits + (size_t)b * d.x_stride;
    const int npair = (V + 1) / 2;  // rows are padded to an even length
    bool ok = true;
    uint64_t w[NB][2];
    const uint64_t* ps[NB];
    uint32_t tg[NB];
#pragma unroll
    for (int u = 0; u < NB; ++u) {
      const int i = tid + u * kCThreads;
      w[u][0] = w[u][1] = 0;
      ps[u] = i < npair ? src + 2 * i : nullptr;
      tg[u] = tl;
      if (i < npair) ld_ll2(ps[u], w[u][0], w[u][1]);
    }
    ok &= ll_settle<NB>(ps, tg, w, g.err);
#pragma unroll
    for (int u = 0; u < NB; ++u) {
      const int i = tid + u * kCThreads;
      if (i < npair) {
        S.lp[2 * i] = ll_val(w[u][0]);
        if (2 * i + 1 < V) S.lp[2 * i + 1] = ll_val(w[u][1]);
      }
    }
    if (cbar_or(!ok)) return false;
  }
  const uint32_t* seen = (j == 0 && fa.seen) ? fa.seen + (size_t)b * g.seen_words : nullptr;
  const int code = sample_row(S, nullptr, V, j, ss, rs.key0, rs.key1, rs.frame_ctr, seen, g.eos_id, g.n_codes,
                              !greedy);
  const int committed = fa.forced ? fa.forced[(size_t)b * kCodebooks + j] : code;
  if (tid == 0) {
    fa.codes_out[(size_t)b * kCodebooks + j] = code;
    if (j == 0) {
      if (fa.seen) fa.seen[(size_t)b * g.seen_words + (committed >> 5)] |= 1u << (committed & 31);
      fa.eos_out[b] = (uint8_t)(code == g.eos_id);
      fa.sess[b].kv_len = s_kv_len[b] + 1;
    }
    if (j == kCodebooks - 1) fa.rng[b].frame_ctr = rs.frame_ctr + 1u;
  }
  if (d.table) {
    const int row = b * d.next_rps + d.next_off;
    const float* src = d.table + (size_t)committed * g.Hc;
    uint64_t* dst = d.x_next + (size_t)row * g.Hc;
    for (int k = tid * 2; k < g.Hc; k += kCThreads * 2) {
      const float2 v = *reinterpret_cast<const float2*>(src + k);
      st_ll2(dst + k, v.x, v.y, tag);
    }
  }
  return true;
}

// ---------------------------------------------------------------------------
// the persistent frame kernel
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(kThreads, 1)
    frame_kernel(const StageDesc* __restrict__ prog, int s0, int s1, Globals g_param, FrameArgs fa_param) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ int sflag;
  __shared__ Ring ring;
  // The stage functions take the frame constants by reference: keep them in
  // shared memory. (A reference to a kernel parameter would put a copy on
  // every thread's stack, and with nearly all of the SM's unified L1/shared
  // memory given to shared memory, stack reads go out to L2.)
  __shared__ Globals g;
  __shared__ FrameArgs fa;
  if (threadIdx.x == 0) {
    g = g_param;
    fa = fa_param;
    s_wait_ns = g_param.wait_ns;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    sflag = read_err(g.err);  // a device error is sticky until qtts_frame_status clears it
    for (int i = 0; i < kRingSlots; ++i) {
      mbar_init(&ring.full[i], 1);
      mbar_init(&ring.empty[i], 1);
      ring.seq[i] = 0xFFFFFFFFu;
      ring.done[i] = 0u;
    }
    mbar_init_fence();
  }
  for (int b = threadIdx.x; b < fa.B; b += kThreads) s_kv_len[b] = fa.sess[b].kv_len;
  __syncthreads();  // the last barrier of all 16 warps: from here on, producer and compute warps part
  if (sflag) return;
  if ((threadIdx.x >> 5) == kProducerWarp) {
    if ((threadIdx.x & 31) == 0) producer(prog, s0, s1, g, fa, smem, &ring);
    return;
  }
  __shared__ StageDesc sdesc[2];
  __shared__ TcState tcs;
  if ((threadIdx.x >> 5) == 0) {
    fetch_desc(&prog[s0], &sdesc[s0 & 1]);
    tc_alloc(&tcs.tmem);  // TMEM accumulators of the tensor path, released before the CTA leaves
    if (threadIdx.x == 0) {
      mbar_init(&tcs.xfree[0], 1);
      mbar_init(&tcs.xfree[1], 1);
      mbar_init(&tcs.done, 1);
      mbar_init(&tcs.drain, 1);
      mbar_init_fence();
      tcs.xuse = 0u;
      tcs.nseg = 0u;
      tcs.issued = 0u;
    }
  }
  tc_fence_before();
  cbar();
  tc_fence_after();
  uint32_t q = 0;
  bool failed = false;
  for (int s = s0; s < s1; ++s) {
    const StageDesc& d = sdesc[s & 1];
    const StageDesc* next = s + 1 < s1 ? &prog[s + 1] : nullptr;
    StageDesc* next_s = &sdesc[(s + 1) & 1];
    if (threadIdx.x == 0) g_trace_stage = s;
    trace_mark(g, 0);
    // stages other than GEMVs fetch the next descriptor up front, on a warp
    // they leave idle or finish with (Talker attention uses warps 0..7)
    if (d.type != ST_GEMV && next && (threadIdx.x >> 5) == kCWarps - 1) fetch_desc(next, next_s);
    const uint32_t tag = fa.tag0 + (uint32_t)s;
    bool ok = true;
    // each stage function is compiled on its own (not inlined): its registers
    // are allocated for it alone, so none spills to local memory, which with
    // nearly all of L1 given to shared memory would be served from L2
    switch (d.type) {
      case ST_BEGIN: ok = stage_begin(d, tag, g, fa); break;
      case ST_GEMV: ok = stage_gemv(d, tag, g, fa, smem, &ring, &tcs, q, next, next_s); break;
      case ST_ATTN_T: ok = stage_attn<true>(d, tag, g, fa, smem); break;
      case ST_ATTN_CP: ok = stage_attn<false>(d, tag, g, fa, smem); break;
      case ST_SAMPLE: ok = stage_sample(d, tag, g, fa, smem); break;
      default: break;
    }
    trace_mark(g, 7);
    // no grid barrier: the next stage waits on the tags of the words it reads
    if (cbar_or(!ok)) {
      failed = true;
      break;
    }
  }
  // A stage left after an error may have MMAs in flight: the issuing thread
  // waits until every MMA it issued has completed before TMEM is released.
  if (failed && tcs.issued && threadIdx.x == kTcIssuer * 32) {
    tc_commit(&tcs.drain);
    mbar_drain(&tcs.drain, 0u);
  }
  if (failed) cbar();
  // every TMEM read is done (each tensor stage ends at a barrier after its loads)
  if ((threadIdx.x >> 5) == 0) {
    tc_fence_after();
    tc_dealloc(tcs.tmem);
  }
}

// Sampling of caller-supplied logits [B][V] for codebook j (one CTA per
// session, the compute warps of a frame CTA): the same sampler the frame
// uses, without the next-input gather.
__global__ void __launch_bounds__(kThreads, 1)
    sample_kernel(const float* __restrict__ logits, int V, int j, Globals g, FrameArgs fa) {
  extern __shared__ __align__(128) unsigned char smem[];
  if ((threadIdx.x >> 5) >= kCWarps) return;
  const int b = blockIdx.x;
  SampleSmem& S = *reinterpret_cast<SampleSmem*>(smem);
  const qtts_session ss = fa.sess[b];
  const qtts_rng rs = fa.rng[b];
  const uint32_t* seen = (j == 0 && fa.seen) ? fa.seen + (size_t)b * g.seen_words : nullptr;
  const int code = sample_row(S, logits + (size_t)b * V, V, j, ss, rs.key0, rs.key1, rs.frame_ctr, seen, g.eos_id,
                              g.n_codes);
  if (threadIdx.x == 0) fa.codes_out[b] = code;
}

cudaError_t frame_kernel_setup() {
  cudaError_t e = cudaFuncSetAttribute(frame_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(sample_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(SampleSmem));
}

cudaError_t frame_kernel_occupancy(int* blocks_per_sm) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, frame_kernel, kThreads, kSmemBytes);
}

// Persistent mode needs every CTA resident at once (CTAs wait on one
// another's words), hence the cooperative launch; stepwise mode runs one
// stage per launch, whose inputs all come from earlier launches.
cudaError_t launch_frame(const StageDesc* prog, int s0, int s1, const Globals& g, const FrameArgs& fa, bool stepwise,
                         cudaStream_t stream) {
  if (stepwise) {
    for (int s = s0; s < s1; ++s) {
      frame_kernel<<<g.G, kThreads, kSmemBytes, stream>>>(prog, s, s + 1, g, fa);
      cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  }
  Globals gg = g;
  FrameArgs ff = fa;
  void* args[] = {(void*)&prog, (void*)&s0, (void*)&s1, (void*)&gg, (void*)&ff};
  return cudaLaunchCooperativeKernel((const void*)frame_kernel, dim3(g.G), dim3(kThreads), args, kSmemBytes, stream);
}

cudaError_t launch_sample(const float* logits, int V, int j, const Globals& g, const FrameArgs& fa,
                          cudaStream_t stream) {
  sample_kernel<<<fa.B, kThreads, sizeof(SampleSmem), stream>>>(logits, V, j, g, fa);
  return cudaGetLastError();
}

}  // namespace qtts
