// prefill.cu -- the Talker prompt pass over whole chunks of prompt tokens.
//
// "Qwen3-TTS PR 5: 1.7B CustomVoice, VoiceDesign and Base": section Graph
// (talker_prefill, the causal prompt pass through the Talker layers before
// the first frame) and section "What changed" (one packed prefill over a
// bucket of 32..1024 prompt tokens). "Qwen3-TTS Native v0.3.0", "What
// changed": prefill stays BF16 when decode runs on INT8 weights, so this pass
// always reads the BF16 weights.
//
// A chunk is M = B x P rows, row p B + b being prompt token p of session b at
// position kv_len_b + p. Per Talker layer, kernels on one stream:
//   norm     RMSNorm of the residual rows, packed as bf16 hi + lo tiles
//   gemm     QKV on the tcgen05 tensor cores, fp32 partial sums per K-slice
//   qkv      RoPE; K and V rounded to bf16 into the sessions' pages; q kept
//   attn     causal attention over each session's pages, packed hi + lo
//   gemm     O, then norm adds it to the residual and normalises
//   gemm     gate/up, then swiglu packs silu(gate) x up (or, with one
//            K-slice, the GEMM's epilogue does, into a second input buffer)
//   gemm     down, then norm adds it and applies the next layer's input norm
// The last layer stops after its K/V: nothing after them is observable.
//
// Activations enter the GEMMs as two bf16 operands, hi = bf16(a) and
// lo = bf16(a - hi), accumulated into one fp32 sum, so a product carries ~16
// mantissa bits of the fp32 activation against bf16 weights (the decode
// path's tensor stages do the same).

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "qtts_internal.h"
#include "device_util.cuh"

namespace qtts {

namespace {

// ---- device helpers of this translation unit (the shared ones: device_util.cuh) ----

// Wait for phase `parity` of `b`, at most `ns` nanoseconds.
__device__ bool bar_wait(uint64_t* b, uint32_t parity, uint64_t ns) {
  if (mbar_test_sleep(b, parity, 20000u)) return true;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_test_sleep(b, parity, 20000u))
    if (global_timer_ns() - t0 > ns) return false;
  return true;
}
// global -> shared bulk copy, completing `bytes` of the barrier's transaction
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* b) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_addr(dst)),
               "l"(__cvta_generic_to_global(src)), "r"(bytes), "r"(smem_addr(b))
               : "memory");
}

// ---- GEMM operand tiles ----
// Activations: [m tile of 128 rows][32-wide K chunk][hi | lo] images; weights
// (packed at load): [256-row tile][K chunk] images. Inside an image of R rows:
// element (r, k) at ((k / 8) * R / 8 + r / 8) * 64 + (r % 8) * 8 + k % 8.
constexpr int kBM = 128, kBN = 256, kBK = 32, kStages = 6;
// 32-wide K chunks in 6 stages keep 5 x 32 KB of copies in flight per SM
// while one stage feeds the MMAs (64-wide chunks in 3 stages, 2 x 64 KB in
// flight, measured as fast)
constexpr int kAImg = kBM * kBK;                    // elements of one hi or lo image (8 KB)
constexpr int kWImg = kBN * kBK;                    // 16 KB
constexpr int kStageBytes = (2 * kAImg + kWImg) * 2;  // 32 KB
constexpr int kGemmSmem = kStages * kStageBytes;
constexpr int kGemmThreads = 192;                   // warp 0 copies, warp 1 issues MMAs, warps 2-5 drain TMEM
constexpr uint32_t kTmemCols = 256;

__host__ __device__ __forceinline__ int core_off(int r, int k, int R) {
  return (k >> 3) * (R * 8) + (r >> 3) * 64 + (r & 7) * 8 + (k & 7);
}
__host__ __device__ __forceinline__ size_t a_off(int r, int k, int KC, int hl) {
  return ((size_t)((r / kBM) * KC + k / kBK) * 2 + hl) * kAImg + core_off(r % kBM, k % kBK, kBM);
}
__host__ __device__ __forceinline__ size_t w_off(int n, int k, int KC) {
  return (size_t)((n / kBN) * KC + k / kBK) * kWImg + core_off(n % kBN, k % kBK, kBN);
}

// hi and lo of eight consecutive activation values (k % 8 == 0) of row r
__device__ __forceinline__ void put8(uint16_t* A, int r, int k, int KC, const float (&v)[8]) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint16_t h0 = f2bf(v[2 * j]), h1 = f2bf(v[2 * j + 1]);
    const uint16_t l0 = f2bf(v[2 * j] - bf2f(h0)), l1 = f2bf(v[2 * j + 1] - bf2f(h1));
    h[j] = (uint32_t)h0 | ((uint32_t)h1 << 16);
    l[j] = (uint32_t)l0 | ((uint32_t)l1 << 16);
  }
  *reinterpret_cast<uint4*>(A + a_off(r, k, KC, 0)) = make_uint4(h[0], h[1], h[2], h[3]);
  *reinterpret_cast<uint4*>(A + a_off(r, k, KC, 1)) = make_uint4(l[0], l[1], l[2], l[3]);
}

// ---------------------------------------------------------------------------
// weights -> tiles (load time): rows past N and columns past K are zero
// ---------------------------------------------------------------------------
__global__ void pack_weights_kernel(const uint16_t* __restrict__ w, int N, int K, int Npad, int KC,
                                    uint16_t* __restrict__ dst) {
  const long long groups = (long long)Npad * KC * (kBK / 8);
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < groups;
       i += (long long)gridDim.x * blockDim.x) {
    const int n = (int)(i / (KC * (kBK / 8)));
    const int k = (int)(i % (KC * (kBK / 8))) * 8;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (n < N && k < K) v = *reinterpret_cast<const uint4*>(w + (size_t)n * K + k);
    *reinterpret_cast<uint4*>(dst + w_off(n, k, KC)) = v;
  }
}

// ---------------------------------------------------------------------------
// GEMM: out[s][m][n] = sum over K-slice s of A[m][k] W[n][k]
// Persistent: one CTA per SM walks the work units (256-row weight tile,
// 128-row activation tile, K-slice) round-robin. Warp 0 fills a 6-stage ring
// of 32-wide K chunks by bulk copies, running ahead across units; one thread
// of warp 1 issues M = 128, N = 256, K = 16 MMAs (hi, then lo, for each K
// step) into one of two 128 x 256 fp32 TMEM accumulators; warps 2-5 drain
// the other accumulator (the previous unit) meanwhile.
// ---------------------------------------------------------------------------
struct GemmArgs {
  const uint16_t* A;
  const uint16_t* W;
  float* out;  // [S][Mpad][Npad]
  int KC, S, Mpad, Npad;
  int M;       // rows with data: the epilogue stores no partial sums of rows past it
  // act != nullptr (one K-slice; columns 2j, 2j + 1 = gate j, up j): the
  // epilogue writes silu(gate) x up as the next GEMM's packed hi + lo input
  // (KCa 32-wide chunks) instead of partial sums
  uint16_t* act;
  int KCa;
  int Nt, Mt;  // tiles: units = Nt Mt S, unit u = (u % Nt, u / Nt % Mt, u / (Nt Mt))
  int* err;
  unsigned long long wait_ns;
};

constexpr int kEpiLd = 33;  // floats per row of an epilogue transpose tile (conflict-free both ways)

__global__ void __launch_bounds__(kGemmThreads, 1) gemm_kernel(GemmArgs a) {
  extern __shared__ __align__(1024) unsigned char smem[];
  __shared__ float epi[4][32 * kEpiLd];  // one 32 x 32 transpose tile per epilogue warp
  __shared__ __align__(8) uint64_t full[kStages], empty[kStages], acc_full[2], acc_empty[2];
  __shared__ uint32_t tmem_base;
  __shared__ int failed;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int units = a.Nt * a.Mt * a.S;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 4);  // one lane of each epilogue warp
    }
    failed = 0;
    mbar_init_fence();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&tmem_base)),
                 "n"(2 * kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  int consumed = 0;   // MMA thread: ring uses whose copies it waited for
  int issued_mma = 0; // MMA thread: units whose MMAs it issued
  auto unit_k = [&](int u, int& kc0, int& nk) {
    const int s = u / (a.Nt * a.Mt);
    kc0 = (int)((long long)s * a.KC / a.S);
    nk = (int)((long long)(s + 1) * a.KC / a.S) - kc0;
  };

  if (warp == 0 && lane == 0) {
    int it = 0;  // ring use counter across units
    for (int u = blockIdx.x; u < units && !*(volatile int*)&failed; u += gridDim.x) {
      const int nt = u % a.Nt, mt = (u / a.Nt) % a.Mt;
      int kc0, nk;
      unit_k(u, kc0, nk);
      for (int i = 0; i < nk; ++i, ++it) {
        const int st = it % kStages, use = it / kStages;
        if (use > 0 && !bar_wait(&empty[st], (use - 1) & 1, a.wait_ns)) {
          set_err(a.err, QTTS_DEV_TIMEOUT);
          failed = 1;
          break;
        }
        unsigned char* base = smem + st * kStageBytes;
        const int kc = kc0 + i;
        mbar_arrive_expect_tx(&full[st], kStageBytes);
        bulk_g2s(base, a.A + (size_t)(mt * a.KC + kc) * 2 * kAImg, 2 * kAImg * 2, &full[st]);
        bulk_g2s(base + 2 * kAImg * 2, a.W + (size_t)(nt * a.KC + kc) * kWImg, kWImg * 2, &full[st]);
      }
    }
  } else if (warp == 1 && lane == 0) {
    constexpr uint32_t idesc = tc_idesc_bf16(kBM, kBN);
    int it = 0, j = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++j) {
      const int buf = j & 1;
      const uint32_t acc = tmem + (uint32_t)(buf * kTmemCols);
      // the epilogue has drained this accumulator (unit j - 2)
      if (j >= 2 && !bar_wait(&acc_empty[buf], ((j >> 1) - 1) & 1, a.wait_ns)) {
        set_err(a.err, QTTS_DEV_TIMEOUT);
        failed = 1;
        break;
      }
      tc_fence_after();
      int kc0, nk;
      unit_k(u, kc0, nk);
      bool ok = true;
      for (int i = 0; i < nk; ++i, ++it) {
        const int st = it % kStages, use = it / kStages;
        if (!bar_wait(&full[st], use & 1, a.wait_ns)) {
          set_err(a.err, QTTS_DEV_TIMEOUT);
          failed = 1;
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t base = smem_addr(smem + st * kStageBytes);
#pragma unroll
        for (int ks = 0; ks < kBK / 16; ++ks) {
          const uint64_t dhi = tc_smem_desc(base + ks * 2 * (kBM * 16), kBM * 16, 128);
          const uint64_t dlo = tc_smem_desc(base + kAImg * 2 + ks * 2 * (kBM * 16), kBM * 16, 128);
          const uint64_t dw = tc_smem_desc(base + 2 * kAImg * 2 + ks * 2 * (kBN * 16), kBN * 16, 128);
          tc_mma(acc, dhi, dw, idesc, i > 0 || ks > 0);
          tc_mma(acc, dlo, dw, idesc, true);
        }
        consumed = it + 1;
        tc_commit(&empty[st]);
      }
      tc_commit(&acc_full[buf]);  // also after a failure: completes once the issued MMAs have
      issued_mma = j + 1;
      if (!ok) break;
    }
  } else if (warp >= 2) {
    const int q = warp & 3;  // this warp's TMEM lane quarter
    int j = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++j) {
      const int buf = j & 1;
      int okl = 0;
      if (lane == 0) okl = bar_wait(&acc_full[buf], (j >> 1) & 1, a.wait_ns) ? 1 : 0;
      const bool ok = __shfl_sync(0xffffffffu, okl, 0) != 0;  // one verdict per warp: the loads are warp-wide
      __syncwarp();
      if (!ok) {
        set_err(a.err, QTTS_DEV_TIMEOUT);
        failed = 1;
        break;
      }
      tc_fence_after();
      const int nt = u % a.Nt, mt = (u / a.Nt) % a.Mt, s = u / (a.Nt * a.Mt);
      const int row0 = mt * kBM + q * 32;  // this warp's 32 rows
      const uint32_t acc = tmem + (uint32_t)(buf * kTmemCols) + ((uint32_t)(q * 32) << 16);
      float* tile = epi[q];
      // 32 columns at a time: lane = row out of TMEM, through shared memory,
      // then four rows of 128 bytes per store instruction
#pragma unroll 1
      for (int c = 0; c < kBN / 32; ++c) {
        uint32_t r[32];
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
              "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
            : "r"(acc + (uint32_t)(c * 32)));
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
            : "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
              "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
              "=r"(r[30]), "=r"(r[31])
            : "r"(acc + (uint32_t)(c * 32 + 16)));
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        if (a.act) {
          // this row's 16 SwiGLU outputs, k = (n tile columns) / 2: a lane per
          // row writes 16 bytes of its core-matrix row, the warp 512 bytes
          const int k0 = (nt * kBN + c * 32) / 2;
          if (row0 + lane < a.M && k0 < a.KCa * kBK) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              float v[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const float g = __uint_as_float(r[16 * h + 2 * e]);
                v[e] = g / (1.0f + expf(-g)) * __uint_as_float(r[16 * h + 2 * e + 1]);
              }
              put8(a.act, row0 + lane, k0 + 8 * h, a.KCa, v);
            }
          }
          __syncwarp();  // converged for the next warp-wide TMEM load
          continue;
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) tile[lane * kEpiLd + j] = __uint_as_float(r[j]);
        __syncwarp();
#pragma unroll
        for (int pass = 0; pass < 8; ++pass) {
          const int rr = pass * 4 + (lane >> 3), cc = (lane & 7) * 4;
          if (row0 + rr < a.M) {
            const float* t = tile + rr * kEpiLd + cc;
            *reinterpret_cast<float4*>(a.out + ((size_t)s * a.Mpad + row0 + rr) * a.Npad + (size_t)nt * kBN + c * 32 +
                                       cc) = make_float4(t[0], t[1], t[2], t[3]);
          }
        }
        __syncwarp();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&acc_empty[buf])) : "memory");
    }
  }
  tc_fence_before();
  __syncthreads();
  if (failed) {
    // nothing may land in shared memory or TMEM after the CTA is gone: wait
    // (bounded) for copies that may still be in flight (one use past the
    // last consumed per stage) and for the issued MMAs
    if (warp == 1 && lane == 0) {
      for (int i = consumed; i < consumed + kStages; ++i)
        bar_wait(&full[i % kStages], (i / kStages) & 1, 2000000000ull);
      if (issued_mma > 0) bar_wait(&acc_full[(issued_mma - 1) & 1], ((issued_mma - 1) >> 1) & 1, 2000000000ull);
    }
    __syncthreads();
  }
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(2 * kTmemCols) : "memory");
  }
}

// ---------------------------------------------------------------------------
// row kernels (one CTA per chunk row)
// ---------------------------------------------------------------------------

constexpr int kRowThreads = 256;

// deterministic CTA sum: warps' shuffle trees, then the warps in order
__device__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = 0.f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += red[w];
  return t;
}

struct NormArgs {
  const uint16_t* emb;   // first layer: the prompt embeddings [M][H] bf16, else nullptr
  float* x;              // residual rows [M][H] fp32
  const float* part;     // added to x first (nullptr: none): [S][Mpad][Npad] partial sums
  int S, Mpad, Npad;
  const uint16_t* gain;  // RMSNorm gain [H] (nullptr: no norm, no packing)
  float eps;
  int H, KC;             // K chunks of the packed rows (H rounded up to whole chunks)
  uint16_t* A;
};

// x = emb (or x + sum of partials); then A = pack(x * rms(x)^-1 * gain).
// Each thread keeps its groups of 8 values in registers between the passes.
constexpr int kNormGroups = 5;  // groups of 8 per thread: H up to 5 x 2048
static_assert(kNormGroups * kRowThreads * 8 >= kWorkBytes / 8, "the widest accepted hidden size fits the registers");
__global__ void __launch_bounds__(kRowThreads) norm_kernel(NormArgs a) {
  __shared__ float red[kRowThreads / 32];
  const int r = blockIdx.x;
  float* x = a.x + (size_t)r * a.H;
  float v[kNormGroups][8];
  float ss = 0.f;
#pragma unroll
  for (int gi = 0; gi < kNormGroups; ++gi) {
    const int k = (threadIdx.x + gi * kRowThreads) * 8;
    if (k >= a.H) break;
    if (a.emb) {
      const uint4 e = *reinterpret_cast<const uint4*>(a.emb + (size_t)r * a.H + k);
      const uint32_t ew[4] = {e.x, e.y, e.z, e.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[gi][2 * j] = bf2f(ew[j] & 0xFFFFu);
        v[gi][2 * j + 1] = bf2f(ew[j] >> 16);
      }
    } else {
      const float4 x0 = *reinterpret_cast<const float4*>(x + k), x1 = *reinterpret_cast<const float4*>(x + k + 4);
      v[gi][0] = x0.x; v[gi][1] = x0.y; v[gi][2] = x0.z; v[gi][3] = x0.w;
      v[gi][4] = x1.x; v[gi][5] = x1.y; v[gi][6] = x1.z; v[gi][7] = x1.w;
    }
    if (a.part)
      for (int s = 0; s < a.S; ++s) {
        const float* p = a.part + ((size_t)s * a.Mpad + r) * a.Npad + k;
        const float4 p0 = *reinterpret_cast<const float4*>(p), p1 = *reinterpret_cast<const float4*>(p + 4);
        v[gi][0] += p0.x; v[gi][1] += p0.y; v[gi][2] += p0.z; v[gi][3] += p0.w;
        v[gi][4] += p1.x; v[gi][5] += p1.y; v[gi][6] += p1.z; v[gi][7] += p1.w;
      }
    *reinterpret_cast<float4*>(x + k) = make_float4(v[gi][0], v[gi][1], v[gi][2], v[gi][3]);
    *reinterpret_cast<float4*>(x + k + 4) = make_float4(v[gi][4], v[gi][5], v[gi][6], v[gi][7]);
#pragma unroll
    for (int j = 0; j < 8; ++j) ss = fmaf(v[gi][j], v[gi][j], ss);
  }
  if (!a.gain) return;
  const float tot = block_sum(ss, red);
  const float rs = 1.0f / sqrtf(tot / (float)a.H + a.eps);
#pragma unroll
  for (int gi = 0; gi < kNormGroups; ++gi) {
    const int k = (threadIdx.x + gi * kRowThreads) * 8;
    if (k >= a.H) break;
    const uint4 gw = *reinterpret_cast<const uint4*>(a.gain + k);
    const uint32_t gg[4] = {gw.x, gw.y, gw.z, gw.w};
    float o[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      o[2 * j] = v[gi][2 * j] * rs * bf2f(gg[j] & 0xFFFFu);
      o[2 * j + 1] = v[gi][2 * j + 1] * rs * bf2f(gg[j] >> 16);
    }
    put8(a.A, r, k, a.KC, o);
  }
  for (int k = a.H + threadIdx.x * 8; k < a.KC * kBK; k += kRowThreads * 8) {  // K padding
    const float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    put8(a.A, r, k, a.KC, z);
  }
}

struct QkvArgs {
  const float* part;  // [S][Mpad][Npad]
  int S, Mpad, Npad;
  int B;
  const qtts_session* sess;
  const int32_t* bt;
  int bt_stride;
  int layer, nq, nkv, d;
  uint16_t* kv_pool;
  int pool_pages;
  const float* rope_cos;  // [max_context][d/2]
  const float* rope_sin;
  float* q;               // [M][nq d]
  int* err;
};

// QKV epilogue of row r: fused rows come as rotate-half pairs (dims i and
// i + d/2 of one q or k head), then v in pairs of adjacent dims. A thread
// takes 8 columns (4 pairs) at a time: all in one head.
__global__ void __launch_bounds__(kRowThreads) qkv_kernel(QkvArgs a) {
  if (read_err(a.err)) return;  // the chunk's sessions failed validation
  const int r = blockIdx.x, b = r % a.B, p = r / a.B;
  const int pos = a.sess[b].kv_len + p;
  const int half = a.d / 2;
  const int nqk = (a.nq + a.nkv) * a.d;
  const int ncol = (a.nq + 2 * a.nkv) * a.d;
  int page = a.bt[(size_t)b * a.bt_stride + pos / kPage];
  if (page < 0 || page >= a.pool_pages) {  // checked before the chunk; stay in bounds regardless
    set_err(a.err, QTTS_DEV_BAD_PAGE);
    return;
  }
  const size_t kvrow = (size_t)(pos % kPage) * a.d;
  for (int n0 = threadIdx.x * 8; n0 < ncol; n0 += kRowThreads * 8) {
    float y[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int s = 0; s < a.S; ++s) {
      const float* src = a.part + ((size_t)s * a.Mpad + r) * a.Npad + n0;
      const float4 t0 = *reinterpret_cast<const float4*>(src), t1 = *reinterpret_cast<const float4*>(src + 4);
      y[0] += t0.x; y[1] += t0.y; y[2] += t0.z; y[3] += t0.w;
      y[4] += t1.x; y[5] += t1.y; y[6] += t1.z; y[7] += t1.w;
    }
    if (n0 < nqk) {
      const bool is_q = n0 < a.nq * a.d;
      const int rel = is_q ? n0 : n0 - a.nq * a.d;
      const int head = rel / a.d, i0 = (rel % a.d) / 2;  // pairs i0 .. i0 + 3
      const float4 c4 = *reinterpret_cast<const float4*>(a.rope_cos + (size_t)pos * half + i0);
      const float4 s4 = *reinterpret_cast<const float4*>(a.rope_sin + (size_t)pos * half + i0);
      const float cs[4] = {c4.x, c4.y, c4.z, c4.w}, sn[4] = {s4.x, s4.y, s4.z, s4.w};
      float o0[4], o1[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        o0[j] = y[2 * j] * cs[j] - y[2 * j + 1] * sn[j];
        o1[j] = y[2 * j + 1] * cs[j] + y[2 * j] * sn[j];
      }
      if (is_q) {
        float* qr = a.q + (size_t)r * a.nq * a.d + head * a.d;
        *reinterpret_cast<float4*>(qr + i0) = make_float4(o0[0], o0[1], o0[2], o0[3]);
        *reinterpret_cast<float4*>(qr + i0 + half) = make_float4(o1[0], o1[1], o1[2], o1[3]);
      } else {
        uint16_t* kp = a.kv_pool +
                       ((((size_t)a.layer * a.pool_pages + page) * 2 + 0) * a.nkv + head) * kPage * a.d + kvrow;
        *reinterpret_cast<uint2*>(kp + i0) = make_uint2((uint32_t)f2bf(o0[0]) | ((uint32_t)f2bf(o0[1]) << 16),
                                                        (uint32_t)f2bf(o0[2]) | ((uint32_t)f2bf(o0[3]) << 16));
        *reinterpret_cast<uint2*>(kp + i0 + half) =
            make_uint2((uint32_t)f2bf(o1[0]) | ((uint32_t)f2bf(o1[1]) << 16),
                       (uint32_t)f2bf(o1[2]) | ((uint32_t)f2bf(o1[3]) << 16));
      }
    } else {
      const int rel = n0 - nqk;
      const int head = rel / a.d, e = rel % a.d;
      uint16_t* vp = a.kv_pool + ((((size_t)a.layer * a.pool_pages + page) * 2 + 1) * a.nkv + head) * kPage * a.d +
                     kvrow + e;
      uint32_t w[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) w[j] = (uint32_t)f2bf(y[2 * j]) | ((uint32_t)f2bf(y[2 * j + 1]) << 16);
      *reinterpret_cast<uint4*>(vp) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

struct SwigluArgs {
  const float* part;  // [S][Mpad][Npad], columns 2j = gate j, 2j + 1 = up j
  int S, Mpad, Npad;
  int F, KC;
  uint16_t* A;
};

__global__ void __launch_bounds__(kRowThreads) swiglu_kernel(SwigluArgs a) {
  const int r = blockIdx.x;
  for (int k = threadIdx.x * 8; k < a.KC * kBK; k += kRowThreads * 8) {
    float v[8];
    if (k < a.F) {
      float y[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) y[j] = 0.f;
      for (int s = 0; s < a.S; ++s) {
        const float* p = a.part + ((size_t)s * a.Mpad + r) * a.Npad + 2 * k;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float4 t = *reinterpret_cast<const float4*>(p + 4 * j);
          y[4 * j] += t.x; y[4 * j + 1] += t.y; y[4 * j + 2] += t.z; y[4 * j + 3] += t.w;
        }
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float g = y[2 * j];
        v[j] = g / (1.0f + expf(-g)) * y[2 * j + 1];
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = 0.f;  // K padding
    }
    put8(a.A, r, k, a.KC, v);
  }
}

// ---------------------------------------------------------------------------
// causal attention on the tensor cores (mma.sync m16n8k16, bf16 operands,
// fp32 accumulation), flash style, split over the key positions: one CTA per
// (session, kv head, block of prompt tokens, chunk of kAttnChunk positions),
// each warp 16 query rows = the group's q heads of 16 / grp consecutive
// tokens; K/V tiles of 64 positions from the pages into shared memory (double
// buffered, cp.async), S = Q K^T, online softmax per row in registers (base
// 2), O += P V; the chunk's unnormalised O, running max and sum go to a
// scratch area that a second kernel combines in chunk order. Q and P enter
// as bf16 hi + lo pairs (two MMAs each), K and V are the cache's bf16 values.
// ---------------------------------------------------------------------------
constexpr int kAttnWarps = 4;
constexpr int kAttnThreads = kAttnWarps * 32;
constexpr int kAttnKT = 64;      // positions per K/V tile
constexpr int kAttnChunk = 256;  // positions per CTA (4 tiles)
__host__ __device__ constexpr int attn_ld(int HD) { return HD + 8; }  // padded row: conflict-free ldmatrix
__host__ __device__ constexpr int attn_smem(int HD) { return 2 * 2 * kAttnKT * attn_ld(HD) * 2; }

struct AttnArgs {
  const float* q;  // [M][nq d], RoPE applied
  int B, P;
  const qtts_session* sess;
  const int32_t* bt;
  int bt_stride;
  int layer, nq, nkv;
  const uint16_t* kv_pool;
  int pool_pages;
  float* po;       // partials [(row nq + head) maxc + chunk][d + 4]: O (unnormalised), max (base 2), sum, 2 pad
                   // (a multiple of 4 floats, so the rows stay 16-byte aligned)
  int maxc;
  int* err;
};

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(__cvta_generic_to_global(src)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ constexpr int h_of(int e) { return e >> 1; }  // accumulator element -> row g (0) or g + 8 (1)
// (hi, lo) bf16 pairs of two fp32 values
__device__ __forceinline__ void split2(float x, float y, uint32_t& hi, uint32_t& lo) {
  const uint16_t hx = f2bf(x), hy = f2bf(y);
  hi = (uint32_t)hx | ((uint32_t)hy << 16);
  lo = (uint32_t)f2bf(x - bf2f(hx)) | ((uint32_t)f2bf(y - bf2f(hy)) << 16);
}

template <int HD>
__global__ void __launch_bounds__(kAttnThreads) attn_kernel(AttnArgs a) {
  constexpr int LD = attn_ld(HD);
  constexpr int NKS = HD / 16;  // k steps of Q K^T; pairs of 8-wide dim tiles of P V
  constexpr int NDT = HD / 8;   // 8-wide output dim tiles
  extern __shared__ __align__(16) uint16_t kvs[];  // [2 buffers][K | V][kAttnKT][LD]
  if (read_err(a.err)) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int b = blockIdx.x / a.nkv, kvh = blockIdx.x % a.nkv;
  const int grp = a.nq / a.nkv;
  const int tw = 16 / grp;  // tokens per warp
  const int pc0 = blockIdx.y * kAttnWarps * tw;
  const int pw0 = pc0 + warp * tw;
  const int kv0 = a.sess[b].kv_len;
  const int chunk = blockIdx.z;
  // scores in base 2: q.k / sqrt(d) * log2(e)
  const float scale = 1.4426950408889634f / sqrtf((float)HD);
  // rows g and g + 8 of this lane: row i is token pw0 + i % tw, q head kvh grp + i / tw
  int tok[2], head[2], lastpos[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int i = g + 8 * h;
    tok[h] = pw0 + i % tw;
    head[h] = kvh * grp + i / tw;
    lastpos[h] = tok[h] < a.P ? kv0 + tok[h] : -1;  // -1: padding row
  }
  const int warp_last = kv0 + min(a.P, pw0 + tw) - 1;  // < kv0 when the warp has no token
  const int cta_last = kv0 + min(a.P, pc0 + kAttnWarps * tw) - 1;
  const int npos = cta_last + 1;
  if (chunk * kAttnChunk >= npos) return;  // no position of this chunk is needed by the block
  // Q fragments (A operand, row major 16 x 16 per k step), hi and lo
  uint32_t qh[NKS][4], ql[NKS][4];
#pragma unroll
  for (int ks = 0; ks < NKS; ++ks)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int h = j & 1;                       // a0a1: row g; a2a3: row g+8; then cols + 8
      const int col = 16 * ks + 2 * c + 8 * (j >> 1);
      float2 v = make_float2(0.f, 0.f);
      if (lastpos[h] >= 0)
        v = *reinterpret_cast<const float2*>(a.q + (size_t)(tok[h] * a.B + b) * a.nq * HD + head[h] * HD + col);
      split2(v.x, v.y, qh[ks][j], ql[ks][j]);
    }
  float o[NDT][4];
#pragma unroll
  for (int j = 0; j < NDT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};

  const uint32_t sbase = smem_addr(kvs);
  const int t_begin = chunk * (kAttnChunk / kAttnKT);
  const int t_end = min((npos + kAttnKT - 1) / kAttnKT, t_begin + kAttnChunk / kAttnKT);
  auto load_tile = [&](int t, int buf) {
    // K and V of positions t*KT .. t*KT + KT - 1: 16-byte pieces, zero past npos
    for (int i = threadIdx.x; i < 2 * kAttnKT * (HD / 8); i += kAttnThreads) {
      const int kv = i / (kAttnKT * (HD / 8)), rem = i % (kAttnKT * (HD / 8));
      const int j = rem / (HD / 8), e = (rem % (HD / 8)) * 8;
      const int pos = t * kAttnKT + j;
      const uint16_t* src = a.kv_pool;
      int bytes = 0;
      if (pos < npos) {
        const int page = a.bt[(size_t)b * a.bt_stride + pos / kPage];
        if (page >= 0 && page < a.pool_pages) {  // checked before the chunk
          src = a.kv_pool + ((((size_t)a.layer * a.pool_pages + page) * 2 + kv) * a.nkv + kvh) * kPage * HD +
                (size_t)(pos % kPage) * HD + e;
          bytes = 16;
        }
      }
      cp_async16(sbase + (uint32_t)((((buf * 2 + kv) * kAttnKT + j) * LD + e) * 2), src, bytes);
    }
    cp_async_commit();
  };
  load_tile(t_begin, 0);
  for (int t = t_begin; t < t_end; ++t) {
    if (t + 1 < t_end) {
      load_tile(t + 1, (t + 1 - t_begin) & 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    if (warp_last >= t * kAttnKT) {
      const int buf = (t - t_begin) & 1;
      const uint32_t kb = sbase + (uint32_t)((buf * 2 + 0) * kAttnKT * LD * 2);
      const uint32_t vb = sbase + (uint32_t)((buf * 2 + 1) * kAttnKT * LD * 2);
      const int mi = lane >> 3, mr = lane & 7;  // ldmatrix: this lane's matrix and row
      // S = Q K^T for 64 positions: 8 tiles of 8
      float sc[8][4];
#pragma unroll
      for (int j = 0; j < 8; ++j) sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < NKS; ++ks)
#pragma unroll
        for (int np = 0; np < 4; ++np) {
          uint32_t kf[4];  // positions 16np + 8 (mi / 2) + mr, dims 16ks + 8 (mi % 2)
          ldsm_x4(kf, kb + (uint32_t)(((16 * np + 8 * (mi >> 1) + mr) * LD + 16 * ks + 8 * (mi & 1)) * 2));
          mma_bf16(sc[2 * np], qh[ks], kf[0], kf[1]);
          mma_bf16(sc[2 * np], ql[ks], kf[0], kf[1]);
          mma_bf16(sc[2 * np + 1], qh[ks], kf[2], kf[3]);
          mma_bf16(sc[2 * np + 1], ql[ks], kf[2], kf[3]);
        }
      // scale, causal mask (only where the tile reaches past the warp's first
      // token: rows of padding tokens are never written, so unmasked is fine
      // for them), online softmax (rows g and g + 8; a row's values sit in the
      // 4 lanes of a group)
      float mx[2] = {-INFINITY, -INFINITY};
      if ((t + 1) * kAttnKT - 1 > kv0 + pw0) {
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int h = e >> 1;
            const int pos = t * kAttnKT + 8 * j + 2 * c + (e & 1);
            const float v = pos <= lastpos[h] ? sc[j][e] * scale : -INFINITY;
            sc[j][e] = v;
            mx[h] = fmaxf(mx[h], v);
          }
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float v = sc[j][e] * scale;
            sc[j][e] = v;
            mx[h_of(e)] = fmaxf(mx[h_of(e)], v);
          }
      }
      float corr[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
        mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
        const float mn = fmaxf(mrow[h], mx[h]);
        corr[h] = mn == -INFINITY ? 1.f : exp2f(mrow[h] - mn);  // 0 while the row had nothing yet
        mrow[h] = mn;
      }
      float rs[2] = {0.f, 0.f};
#pragma unroll
      for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int h = e >> 1;
          const float p = sc[j][e] == -INFINITY ? 0.f : exp2f(sc[j][e] - mrow[h]);
          sc[j][e] = p;
          rs[h] += p;
        }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        rs[h] += __shfl_xor_sync(0xffffffffu, rs[h], 1);
        rs[h] += __shfl_xor_sync(0xffffffffu, rs[h], 2);
        lrow[h] = lrow[h] * corr[h] + rs[h];
      }
#pragma unroll
      for (int j = 0; j < NDT; ++j) {
        o[j][0] *= corr[0];
        o[j][1] *= corr[0];
        o[j][2] *= corr[1];
        o[j][3] *= corr[1];
      }
      // O += P V: P's accumulator tiles (2kk, 2kk + 1) are the A fragment of k step kk
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        uint32_t ph[4], pl[4];
        split2(sc[2 * kk][0], sc[2 * kk][1], ph[0], pl[0]);
        split2(sc[2 * kk][2], sc[2 * kk][3], ph[1], pl[1]);
        split2(sc[2 * kk + 1][0], sc[2 * kk + 1][1], ph[2], pl[2]);
        split2(sc[2 * kk + 1][2], sc[2 * kk + 1][3], ph[3], pl[3]);
#pragma unroll
        for (int dp = 0; dp < NKS; ++dp) {
          uint32_t vf[4];  // positions 16kk + 8 (mi % 2) + mr, dims 16dp + 8 (mi / 2), transposed
          ldsm_x4_t(vf, vb + (uint32_t)(((16 * kk + 8 * (mi & 1) + mr) * LD + 16 * dp + 8 * (mi >> 1)) * 2));
          mma_bf16(o[2 * dp], ph, vf[0], vf[1]);
          mma_bf16(o[2 * dp], pl, vf[0], vf[1]);
          mma_bf16(o[2 * dp + 1], ph, vf[2], vf[3]);
          mma_bf16(o[2 * dp + 1], pl, vf[2], vf[3]);
        }
      }
    }
    __syncthreads();  // the buffer is refilled two tiles on
  }
  // the chunk's partial state of each real row: O (unnormalised), max, sum
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    if (lastpos[h] < 0) continue;
    const int r = tok[h] * a.B + b;
    float* dst = a.po + ((size_t)(r * a.nq + head[h]) * a.maxc + chunk) * (HD + 4);
#pragma unroll
    for (int j = 0; j < NDT; ++j)
      *reinterpret_cast<float2*>(dst + 8 * j + 2 * c) = make_float2(o[j][2 * h], o[j][2 * h + 1]);
    if (c == 0) {
      dst[HD] = mrow[h];
      dst[HD + 1] = lrow[h];
    }
  }
}

// ---------------------------------------------------------------------------
// attention for one query token per session (a decode step): bound by
// reading the cache, so on CUDA cores. One CTA per (session, kv head,
// kAttnChunk-position chunk), 8 warps of 32 positions: a warp stages its K
// rows in shared memory (coalesced 16-byte loads), a lane scores its
// position for the group's q heads in fp32, the warp's base-2 softmax state
// per head, then O += P V with V rows read coalesced and a lane owning HD/32
// dims; the warps' states merge in shared memory in warp order into the
// chunk's partial, the format attn_kernel writes and attn_combine_kernel
// merges.
// ---------------------------------------------------------------------------
constexpr int kDecWarps = kAttnChunk / 32;
__host__ __device__ constexpr int dec_ldk(int HD) { return HD + 8; }  // bf16 per staged K row (16-byte pad)
__host__ __device__ constexpr int dec_smem(int HD) {
  return kDecWarps * 32 * dec_ldk(HD) * 2 + 2 * HD * 4 + kDecWarps * 2 * (HD + 4) * 4;
}

template <int HD>
__global__ void __launch_bounds__(kDecWarps * 32) attn_decode_kernel(AttnArgs a) {
  constexpr int E = HD / 32;
  constexpr int LDK = dec_ldk(HD);
  extern __shared__ __align__(16) unsigned char dsm[];
  uint16_t* ks = reinterpret_cast<uint16_t*>(dsm);                                       // [warps][32][LDK]
  float* qs = reinterpret_cast<float*>(dsm + kDecWarps * 32 * LDK * 2);                 // [2][HD]
  float* st = qs + 2 * HD;                                                              // [warps][2][HD + 4]
  if (read_err(a.err)) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x / a.nkv, kvh = blockIdx.x % a.nkv;
  const int grp = a.nq / a.nkv;  // 1 or 2
  const int chunk = blockIdx.y;
  const int kv0 = a.sess[b].kv_len;
  const int npos = kv0 + 1;  // positions 0 .. kv_len: the cache and the new token
  if (chunk * kAttnChunk >= npos) return;
  const float scale = 1.4426950408889634f / sqrtf((float)HD);
  for (int i = threadIdx.x; i < grp * HD; i += kDecWarps * 32)
    qs[i] = a.q[(size_t)b * a.nq * HD + (size_t)kvh * grp * HD + i];
  // lane j resolves position p0 + j's K and V rows once (0: past the last
  // position); the warp shares them by shuffle, so no load waits on a page id
  const int p0 = chunk * kAttnChunk + warp * 32;
  const int pos = p0 + lane;
  const bool valid = pos < npos;
  unsigned long long krow = 0, vrow = 0;
  if (valid) {
    const int page = a.bt[(size_t)b * a.bt_stride + pos / kPage];
    if (page >= 0 && page < a.pool_pages) {  // checked before the step
      const size_t base = (((size_t)a.layer * a.pool_pages + page) * 2 * a.nkv + kvh) * kPage * HD + (size_t)(pos % kPage) * HD;
      krow = (unsigned long long)(a.kv_pool + base);
      vrow = (unsigned long long)(a.kv_pool + base + (size_t)a.nkv * kPage * HD);
    }
  }
  // this warp's K rows in shared memory: 32 positions x HD bf16, 16 bytes per lane step
  uint16_t* kw = ks + warp * 32 * LDK;
#pragma unroll 4
  for (int i = lane; i < 32 * (HD / 8); i += 32) {
    const int j = i / (HD / 8), e = (i % (HD / 8)) * 8;
    const unsigned long long kr = __shfl_sync(0xffffffffu, krow, j);
    uint4 v = make_uint4(0, 0, 0, 0);
    if (kr) v = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(kr) + e);
    *reinterpret_cast<uint4*>(kw + j * LDK + e) = v;
  }
  __syncthreads();
  float sc[2] = {0.f, 0.f};
#pragma unroll 4
  for (int e = 0; e < HD; e += 8) {
    const uint4 kv = *reinterpret_cast<const uint4*>(kw + lane * LDK + e);
    const uint32_t kk[4] = {kv.x, kv.y, kv.z, kv.w};
    float kf[8];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      kf[2 * u] = bf2f(kk[u] & 0xFFFFu);
      kf[2 * u + 1] = bf2f(kk[u] >> 16);
    }
#pragma unroll
    for (int h = 0; h < 2; ++h)
      if (h < grp) {
        const float4 q0 = *reinterpret_cast<const float4*>(qs + h * HD + e);
        const float4 q1 = *reinterpret_cast<const float4*>(qs + h * HD + e + 4);
        sc[h] = fmaf(q0.x, kf[0], sc[h]);
        sc[h] = fmaf(q0.y, kf[1], sc[h]);
        sc[h] = fmaf(q0.z, kf[2], sc[h]);
        sc[h] = fmaf(q0.w, kf[3], sc[h]);
        sc[h] = fmaf(q1.x, kf[4], sc[h]);
        sc[h] = fmaf(q1.y, kf[5], sc[h]);
        sc[h] = fmaf(q1.z, kf[6], sc[h]);
        sc[h] = fmaf(q1.w, kf[7], sc[h]);
      }
  }
  float m[2], l[2], p[2], o[2][E];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const float v = valid && h < grp ? sc[h] * scale : -INFINITY;
    float mx = v;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    m[h] = mx;
    p[h] = v == -INFINITY ? 0.f : exp2f(v - mx);
    float sum = p[h];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    l[h] = sum;
#pragma unroll
    for (int e = 0; e < E; ++e) o[h][e] = 0.f;
  }
  // O += P V: V row j read by the whole warp (lane: dims lane E .. lane E + E - 1)
#pragma unroll 8
  for (int j = 0; j < 32; ++j) {
    const unsigned long long vr = __shfl_sync(0xffffffffu, vrow, j);
    float vf[E];
    if (vr) {
      const uint16_t* src = reinterpret_cast<const uint16_t*>(vr) + lane * E;
      if constexpr (E == 4) {
        const uint2 w = *reinterpret_cast<const uint2*>(src);
        vf[0] = bf2f(w.x & 0xFFFFu); vf[1] = bf2f(w.x >> 16); vf[2] = bf2f(w.y & 0xFFFFu); vf[3] = bf2f(w.y >> 16);
      } else {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(src);
        vf[0] = bf2f(w & 0xFFFFu); vf[1] = bf2f(w >> 16);
      }
    } else {
#pragma unroll
      for (int e = 0; e < E; ++e) vf[e] = 0.f;
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float pb = __shfl_sync(0xffffffffu, p[h], j);
#pragma unroll
      for (int e = 0; e < E; ++e) o[h][e] = fmaf(pb, vf[e], o[h][e]);
    }
  }
  // the warps' states, then the chunk's partial per q head (warp order)
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    if (h >= grp) break;
    float* sw = st + (warp * 2 + h) * (HD + 4);
#pragma unroll
    for (int e = 0; e < E; ++e) sw[lane * E + e] = o[h][e];
    if (lane == 0) {
      sw[HD] = m[h];
      sw[HD + 1] = l[h];
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < grp * HD; i += kDecWarps * 32) {
    const int h = i / HD, e = i % HD;
    float mm = -INFINITY;
    for (int w = 0; w < kDecWarps; ++w) mm = fmaxf(mm, st[(w * 2 + h) * (HD + 4) + HD]);
    float acc = 0.f, ll = 0.f;
    for (int w = 0; w < kDecWarps; ++w) {
      const float* sw = st + (w * 2 + h) * (HD + 4);
      if (sw[HD] == -INFINITY) continue;  // no position of this warp
      const float wt = exp2f(sw[HD] - mm);
      acc = fmaf(wt, sw[e], acc);
      ll = fmaf(wt, sw[HD + 1], ll);
    }
    float* dst = a.po + ((size_t)(b * a.nq + kvh * grp + h) * a.maxc + chunk) * (HD + 4);
    dst[e] = acc;
    if (e == 0) {
      dst[HD] = mm;
      dst[HD + 1] = ll;
    }
  }
}

struct CombineArgs {
  const float* po;
  int maxc, B, nq, d, KC;
  const qtts_session* sess;
  uint16_t* A;
  int* err;
};

// O of row r and every q head: the chunks' partial states merged in chunk
// order (max of the maxima, weights 2^(m_c - m)), packed as hi + lo
__global__ void __launch_bounds__(kRowThreads) attn_combine_kernel(CombineArgs a) {
  if (read_err(a.err)) return;
  const int r = blockIdx.x, b = r % a.B, p = r / a.B;
  const int nc = (a.sess[b].kv_len + p + 1 + kAttnChunk - 1) / kAttnChunk;  // chunks holding this row's positions
  for (int u = threadIdx.x; u < a.nq * a.d / 8; u += kRowThreads) {
    const int head = (u * 8) / a.d, e = (u * 8) % a.d;
    const float* src = a.po + (size_t)(r * a.nq + head) * a.maxc * (a.d + 4);
    float m = -INFINITY;
    for (int ch = 0; ch < nc; ++ch) m = fmaxf(m, src[(size_t)ch * (a.d + 4) + a.d]);
    float l = 0.f, v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int ch = 0; ch < nc; ++ch) {
      const float* pc = src + (size_t)ch * (a.d + 4);
      const float mc = pc[a.d];
      if (mc == -INFINITY) continue;  // no position of the chunk for this row
      const float w = exp2f(mc - m);
      l += w * pc[a.d + 1];
      const float4 x0 = *reinterpret_cast<const float4*>(pc + e), x1 = *reinterpret_cast<const float4*>(pc + e + 4);
      v[0] += w * x0.x; v[1] += w * x0.y; v[2] += w * x0.z; v[3] += w * x0.w;
      v[4] += w * x1.x; v[5] += w * x1.y; v[6] += w * x1.z; v[7] += w * x1.w;
    }
    const float inv = 1.0f / l;
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] *= inv;
    put8(a.A, r, head * a.d + e, a.KC, v);
  }
}

// ---------------------------------------------------------------------------
// decode: the Talker's last residual rows as the frame kernel's tagged words
// (fp32 value in the low half, `tag` in the high half)
// ---------------------------------------------------------------------------
__global__ void publish_kernel(const float* __restrict__ x, int n, uint64_t* __restrict__ dst, uint32_t tag) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
    dst[i] = ((uint64_t)tag << 32) | __float_as_uint(x[i]);
}

// ---------------------------------------------------------------------------
// chunk validation: every session's positions kv_len .. kv_len + P - 1 fit
// the context and its block table, and every page the chunk reads or writes
// is in the pool
// ---------------------------------------------------------------------------
__global__ void check_kernel(const qtts_session* sess, const int32_t* bt, int bt_stride, int B, int P,
                             int max_context, int pool_pages, int* err) {
  for (int b = blockIdx.x; b < B; b += gridDim.x) {
    const int kv = sess[b].kv_len;
    if (kv < 0 || kv + P > max_context || kv + P > bt_stride * kPage) {
      if (threadIdx.x == 0) set_err(err, QTTS_DEV_BAD_SESSION);
      continue;
    }
    const int np = (kv + P + kPage - 1) / kPage;
    for (int i = threadIdx.x; i < np; i += blockDim.x) {
      const int page = bt[(size_t)b * bt_stride + i];
      if (page < 0 || page >= pool_pages) set_err(err, QTTS_DEV_BAD_PAGE);
    }
  }
}

}  // namespace

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

size_t pf_packed_elems(int N, int K) {
  return (size_t)((N + kBN - 1) / kBN) * kBN * ((K + kBK - 1) / kBK) * kBK;
}

size_t pf_act_elems(int rows, int maxK) {
  return (size_t)((rows + kBM - 1) / kBM) * ((maxK + kBK - 1) / kBK) * 2 * kAImg;
}

int pf_attn_chunks(int max_context) { return (max_context + kAttnChunk - 1) / kAttnChunk; }

size_t pf_attn_floats(int rows, int nq, int d, int max_context) {
  return (size_t)rows * nq * pf_attn_chunks(max_context) * (d + 4);
}

size_t pf_part_floats(int rows, int maxN) {
  return (size_t)((rows + kBM - 1) / kBM) * kBM * ((maxN + kBN - 1) / kBN) * kBN;
}

cudaError_t pf_setup() {
  cudaError_t e = cudaFuncSetAttribute(gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(attn_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, attn_smem(128));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(attn_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, attn_smem(64));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(attn_decode_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, dec_smem(128));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(attn_decode_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, dec_smem(64));
  return e;
}

cudaError_t pf_pack_weights(const uint16_t* w, int N, int K, uint16_t* dst, cudaStream_t s) {
  const int Npad = (N + kBN - 1) / kBN * kBN, KC = (K + kBK - 1) / kBK;
  const long long groups = (long long)Npad * KC * (kBK / 8);
  const int blocks = (int)std::min<long long>((groups + 255) / 256, 8192);
  pack_weights_kernel<<<blocks, 256, 0, s>>>(w, N, K, Npad, KC, dst);
  return cudaGetLastError();
}

// K-slices of a GEMM with `tiles` output tiles over KC K chunks: fewest
// (waves of the grid x K chunks a CTA runs), ties to fewer slices, within the
// partial-sum buffer
static int pf_splits(int tiles, int KC, int G, size_t cap) {
  const size_t tile_floats = (size_t)kBM * kBN;
  int best = 1;
  long long best_cost = (long long)((tiles + G - 1) / G) * KC;
  for (int S = 2; S <= 8 && S <= KC; ++S) {  // more slices measured slower (partial sums to write and re-read)
    if ((size_t)S * tiles * tile_floats > cap) break;
    const long long cost = (long long)((tiles * S + G - 1) / G) * ((KC + S - 1) / S);
    if (cost < best_cost) {
      best = S;
      best_cost = cost;
    }
  }
  return best;
}

// SwiGLU in the gate/up GEMM's epilogue (one K-slice) or a pass over the S
// slices' partial sums: the split writes S x tiles of partial sums and the
// pass re-reads them, charged here in chunk-times at ~3 MB of HBM traffic
// each (one 32-wide step of a 128 x 256 tile took ~0.46 us in the 512-row
// GEMMs, HBM moves ~6.7 TB/s). At 512 full-width rows (128 against 96 + 34)
// the single slice measured 2-3 % faster.
static bool pf_fuse_swiglu(int tiles, int KC, int G, int S) {
  const double one = (double)((tiles + G - 1) / G) * KC;
  const double split = (double)((tiles * S + G - 1) / G) * ((KC + S - 1) / S);
  return one <= split + 2.0 * S * tiles * kBM * kBN * 4 / 3.0e6;
}

// The Talker layers over B x P rows. decode: the whole last layer too, its
// output rows (the residual stream) left in c.x; else the last layer stops
// after its K/V.
static cudaError_t pf_layers(const PfCtx& c, int B, int P, const qtts_session* sess, const int32_t* bt,
                             int bt_stride, const uint16_t* embeds, bool decode, cudaStream_t s) {
  const int M = B * P;
  if (M < 1 || M > c.max_rows) return cudaErrorInvalidValue;
  const int Mt = (M + kBM - 1) / kBM, Mpad = Mt * kBM;
  const int KH = (c.H + kBK - 1) / kBK, KA = (c.nq * c.d + kBK - 1) / kBK, KF = (c.F + kBK - 1) / kBK;
  check_kernel<<<std::min(B, 32), 128, 0, s>>>(sess, bt, bt_stride, B, P, c.max_context, c.pool_pages, c.err);
  int S = 1, Npad = 0;
  auto gemm = [&](const uint16_t* W, int N, int K, const uint16_t* Ain = nullptr, uint16_t* act = nullptr,
                  int KCa = 0) {
    const int Nt = (N + kBN - 1) / kBN, KC = (K + kBK - 1) / kBK;
    S = act ? 1 : pf_splits(Nt * Mt, KC, c.G, c.part_floats);
    Npad = Nt * kBN;
    GemmArgs ga{Ain ? Ain : c.A, W, c.part, KC, S, Mpad, Npad, M, act, KCa, Nt, Mt, c.err, c.wait_ns};
    gemm_kernel<<<std::min(Nt * Mt * S, c.G), kGemmThreads, kGemmSmem, s>>>(ga);
  };
  auto norm = [&](const uint16_t* emb, bool add, const uint16_t* gain) {
    NormArgs na{emb, c.x, add ? c.part : nullptr, S, Mpad, Npad, gain, c.eps, c.H, KH, c.A};
    norm_kernel<<<M, kRowThreads, 0, s>>>(na);
  };
  norm(embeds, false, c.layers[0].in_norm);
  const int grp = c.nq / c.nkv;
  const int tpc = kAttnWarps * (16 / grp);  // prompt tokens per attention CTA
  const int maxc = pf_attn_chunks(c.max_context);
  const int gu_tiles = (2 * c.F + kBN - 1) / kBN * Mt;
  const bool fuse = pf_fuse_swiglu(gu_tiles, KH, c.G, pf_splits(gu_tiles, KH, c.G, c.part_floats));
  for (int l = 0; l < c.n_layers; ++l) {
    const PfLayer& L = c.layers[l];
    gemm(L.qkv, (c.nq + 2 * c.nkv) * c.d, c.H);
    QkvArgs qa{c.part, S, Mpad, Npad, B, sess, bt, bt_stride, l, c.nq, c.nkv, c.d, c.kv_pool, c.pool_pages,
               c.rope_cos, c.rope_sin, c.q, c.err};
    qkv_kernel<<<M, kRowThreads, 0, s>>>(qa);
    const bool last = l == c.n_layers - 1;
    if (last && !decode) break;  // the last layer's K/V are all a prompt pass leaves
    AttnArgs aa{c.q, B, P, sess, bt, bt_stride, l, c.nq, c.nkv, c.kv_pool, c.pool_pages, c.po, maxc, c.err};
    const dim3 ag(B * c.nkv, (P + tpc - 1) / tpc, maxc);
    if (P == 1) {  // one query token per session: the cache-read-bound kernel
      const dim3 dg(B * c.nkv, maxc);
      if (c.d == 128)
        attn_decode_kernel<128><<<dg, kDecWarps * 32, dec_smem(128), s>>>(aa);
      else
        attn_decode_kernel<64><<<dg, kDecWarps * 32, dec_smem(64), s>>>(aa);
    } else if (c.d == 128) {
      attn_kernel<128><<<ag, kAttnThreads, attn_smem(128), s>>>(aa);
    } else {
      attn_kernel<64><<<ag, kAttnThreads, attn_smem(64), s>>>(aa);
    }
    CombineArgs ca{c.po, maxc, B, c.nq, c.d, KA, sess, c.A, c.err};
    attn_combine_kernel<<<M, kRowThreads, 0, s>>>(ca);
    gemm(L.o, c.H, c.nq * c.d);
    norm(nullptr, true, L.post_norm);
    if (fuse) {  // silu(gate) x up straight into the second input buffer
      gemm(L.gu, 2 * c.F, c.H, nullptr, c.A2, KF);
      gemm(L.down, c.H, c.F, c.A2);
    } else {
      gemm(L.gu, 2 * c.F, c.H);
      SwigluArgs sa{c.part, S, Mpad, Npad, c.F, KF, c.A};
      swiglu_kernel<<<M, kRowThreads, 0, s>>>(sa);
      gemm(L.down, c.H, c.F);
    }
    norm(nullptr, true, last ? nullptr : c.layers[l + 1].in_norm);  // last: the residual add alone
  }
  return cudaGetLastError();
}

cudaError_t pf_chunk(const PfCtx& c, int B, int P, const qtts_session* sess, const int32_t* bt, int bt_stride,
                     const uint16_t* embeds, cudaStream_t s) {
  return pf_layers(c, B, P, sess, bt, bt_stride, embeds, false, s);
}

cudaError_t pf_talker_step(const PfCtx& c, int B, const qtts_session* sess, const int32_t* bt, int bt_stride,
                           const uint16_t* in_embeds, uint64_t* x_words, uint32_t tag, cudaStream_t s) {
  cudaError_t e = pf_layers(c, B, 1, sess, bt, bt_stride, in_embeds, true, s);
  if (e != cudaSuccess) return e;
  const int n = B * c.H;
  publish_kernel<<<(n + 255) / 256, 256, 0, s>>>(c.x, n, x_words, tag);
  return cudaGetLastError();
}

}  // namespace qtts
