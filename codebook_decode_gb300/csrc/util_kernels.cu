// util_kernels.cu -- load-time and bookkeeping kernels: weight layout gather,
// the INT8 weight-only quantiser, projected Code-Predictor input tables, KV
// page scatter/gather and the free-running feedback embedding.
#include <cuda_bf16.h>

#include "qtts_internal.h"

namespace qtts {

__device__ __forceinline__ float u16_to_f(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

// dst[r][:] = src[map[r]][:]  (rows of K bf16; K a multiple of 8)
__global__ void gather_rows_kernel(uint16_t* dst, const uint16_t* src, const int32_t* map, int n_rows, int K) {
  const int r = blockIdx.x;
  if (r >= n_rows) return;
  const int sr = map[r];
  const uint4* s = reinterpret_cast<const uint4*>(src + (size_t)sr * K);
  uint4* d = reinterpret_cast<uint4*>(dst + (size_t)r * K);
  for (int i = threadIdx.x; i < K / 8; i += blockDim.x) d[i] = s[i];
}

cudaError_t launch_gather_rows(uint16_t* dst, const uint16_t* src, const int32_t* map, int n_rows, int K,
                               cudaStream_t s) {
  gather_rows_kernel<<<n_rows, 128, 0, s>>>(dst, src, map, n_rows, K);
  return cudaGetLastError();
}

// INT8 weight-only quantiser ("Qwen3-TTS Native v0.3.0", "What changed":
// per-output-channel symmetric INT8 from the BF16 weights). One warp per row:
// m = max|w|, scale = m / 127 and q = round-half-even(w / scale), both IEEE
// binary32 divisions, q clamped to [-127, 127]; a zero row gets scale 0, q 0.
__global__ void quantize_rows_kernel(const uint16_t* w, int N, int K, int8_t* q, float* scale) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= N) return;
  const uint16_t* row = w + (size_t)warp * K;
  float m = 0.f;
  for (int k = lane; k < K; k += 32) m = fmaxf(m, fabsf(u16_to_f(row[k])));
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const float s = __fdiv_rn(m, 127.0f);
  if (lane == 0) scale[warp] = s;
  int8_t* qr = q + (size_t)warp * K;
  for (int k = lane; k < K; k += 32) {
    int v = 0;
    if (s != 0.0f) {
      v = __float2int_rn(__fdiv_rn(u16_to_f(row[k]), s));
      v = v > 127 ? 127 : (v < -127 ? -127 : v);
    }
    qr[k] = (int8_t)v;
  }
}

cudaError_t launch_quantize_rows(const uint16_t* w, int N, int K, int8_t* q, float* scale, cudaStream_t s) {
  const int warps_per_block = 8;
  quantize_rows_kernel<<<(N + warps_per_block - 1) / warps_per_block, warps_per_block * 32, 0, s>>>(w, N, K, q,
                                                                                                   scale);
  return cudaGetLastError();
}

// T[c][n] = sum_k P[n][k] E[c][k] (+ bias[n]): the small_to_mtp_projection
// applied to every row of one codebook embedding table, fp32 accumulation.
// INT8 mode: P = scale[n] * P8[n][k]. 64x64 output tiles, K in chunks of 32.
__global__ void project_table_kernel(const uint16_t* E, int rows, int H, const uint16_t* P, const int8_t* P8,
                                     const float* P8s, const uint16_t* bias, int Hc, float* T) {
  __shared__ float es[64][33];
  __shared__ float ps[64][33];
  const int c0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;  // 16 x 16 threads, 4 x 4 outputs each
  float acc[4][4] = {};
  for (int k0 = 0; k0 < H; k0 += 32) {
    for (int i = threadIdx.x; i < 64 * 32; i += 256) {
      const int r = i / 32, k = i % 32;
      const int c = c0 + r, n = n0 + r;
      es[r][k] = (c < rows && k0 + k < H) ? u16_to_f(E[(size_t)c * H + k0 + k]) : 0.f;
      float pv = 0.f;
      if (n < Hc && k0 + k < H) pv = P8 ? (float)P8[(size_t)n * H + k0 + k] : u16_to_f(P[(size_t)n * H + k0 + k]);
      ps[r][k] = pv;
    }
    __syncthreads();
#pragma unroll 8
    for (int k = 0; k < 32; ++k) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = es[ty * 4 + i][k];
#pragma unroll
      for (int i = 0; i < 4; ++i) b[i] = ps[tx * 4 + i][k];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) acc[i][jj] = fmaf(a[i], b[jj], acc[i][jj]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const int c = c0 + ty * 4 + i, n = n0 + tx * 4 + jj;
      if (c < rows && n < Hc) {
        float v = acc[i][jj];
        if (P8) v *= P8s[n];
        if (bias) v += u16_to_f(bias[n]);
        T[(size_t)c * Hc + n] = v;
      }
    }
}

cudaError_t launch_project_table(const uint16_t* E, int rows, int H, const uint16_t* P, const int8_t* P8,
                                 const float* P8s, const uint16_t* bias, int Hc, float* T, cudaStream_t s) {
  dim3 grid((Hc + 63) / 64, (rows + 63) / 64);
  project_table_kernel<<<grid, 256, 0, s>>>(E, rows, H, P, P8, P8s, bias, Hc, T);
  return cudaGetLastError();
}

// Copy n_tok tokens of one layer between a dense [n_tok][nkv][d] K/V pair and
// the paged pool [layer][page][2][nkv][16][d]. to_pool: 1 write, 0 read.
__global__ void kv_scatter_kernel(uint16_t* pool, int pool_pages, int nkv, int d, int layer, int n_tok,
                                  const int32_t* pages, uint16_t* k, uint16_t* v, int to_pool) {
  const int t = blockIdx.x;
  if (t >= n_tok) return;
  const int page = pages[t / kPage], slot = t % kPage;
  if (page < 0 || page >= pool_pages) return;  // checked on the host
  for (int i = threadIdx.x; i < 2 * nkv * d; i += blockDim.x) {
    const int kv = i / (nkv * d), rem = i % (nkv * d), h = rem / d, e = rem % d;
    uint16_t* pp = pool + (((((size_t)layer * pool_pages + page) * 2 + kv) * nkv + h) * kPage + slot) * d + e;
    uint16_t* dense = (kv == 0 ? k : v) + ((size_t)t * nkv + h) * d + e;
    if (to_pool) *pp = *dense;
    else *dense = *pp;
  }
}

cudaError_t launch_kv_scatter(uint16_t* pool, int pool_pages, int nkv, int d, int layer, int n_tok,
                              const int32_t* pages, uint16_t* k, uint16_t* v, int to_pool, cudaStream_t s) {
  if (n_tok <= 0) return cudaSuccess;
  kv_scatter_kernel<<<n_tok, 256, 0, s>>>(pool, pool_pages, nkv, d, layer, n_tok, pages, k, v, to_pool);
  return cudaGetLastError();
}

// next[b][i] = bf16(text[b][i] + sum_{j=0..15} E_j[codes[b][j]][i]), fp32 sum
// in codebook order. A code outside its table contributes nothing.
__global__ void feedback_kernel(int H, const int32_t* codes, const uint16_t* text, EmbedTables tables,
                                uint16_t* out) {
  const int b = blockIdx.x;
  for (int i = threadIdx.x; i < H; i += blockDim.x) {
    float s = u16_to_f(text[(size_t)b * H + i]);
#pragma unroll
    for (int j = 0; j < kCodebooks; ++j) {
      const int c = codes[b * kCodebooks + j];
      if (c >= 0 && c < tables.rows[j]) s += u16_to_f(tables.e[j][(size_t)c * H + i]);
    }
    out[(size_t)b * H + i] = __bfloat16_as_ushort(__float2bfloat16_rn(s));
  }
}

cudaError_t launch_feedback(int B, int H, const int32_t* codes, const uint16_t* text, EmbedTables tables,
                            uint16_t* out, cudaStream_t s) {
  feedback_kernel<<<B, 256, 0, s>>>(H, codes, text, tables, out);
  return cudaGetLastError();
}

// Row-major W [N][K] (bf16, or int8 for the weight-only INT8 path) -> the
// per-CTA tensor-core slices (layout in qtts_internal.h, by element): one
// thread per 8-element run (one core-matrix row: 16 bytes of bf16, 8 of int8).
template <typename T, typename Run>
__global__ void tile_weights_kernel(const T* w, int N, int K, int n_groups, int G, T* t) {
  const size_t runs = (size_t)n_groups * kTcRows * (K / 8);
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < runs; i += (size_t)gridDim.x * blockDim.x) {
    const int n = (int)(i / (K / 8)), k = (int)(i % (K / 8)) * 8;
    const int grp = n / kTcRows;
    // the CTA whose share holds group grp: share(c) = [n_groups c / G, n_groups (c+1) / G)
    int c = (int)((long long)grp * G / n_groups);
    while (c + 1 < G && (long long)n_groups * (c + 1) / G <= grp) ++c;
    while (c > 0 && (long long)n_groups * c / G > grp) --c;
    const int g0 = (int)((long long)n_groups * c / G), g1 = (int)((long long)n_groups * (c + 1) / G);
    const int rows_c = (g1 - g0) * kTcRows, nl = n - g0 * kTcRows;
    const size_t off = (size_t)g0 * kTcRows * K + ((size_t)(k / 8) * (rows_c / 8) + nl / 8) * 64 + (nl % 8) * 8;
    Run v{};
    if (n < N) v = *reinterpret_cast<const Run*>(w + (size_t)n * K + k);
    *reinterpret_cast<Run*>(t + off) = v;
  }
}

cudaError_t launch_tile_weights(const uint16_t* w, int N, int K, int G, uint16_t* t, cudaStream_t s) {
  const int n_groups = (N + kTcRows - 1) / kTcRows;
  tile_weights_kernel<uint16_t, uint4><<<1024, 256, 0, s>>>(w, N, K, n_groups, G, t);
  return cudaGetLastError();
}

cudaError_t launch_tile_weights_i8(const int8_t* w, int N, int K, int G, int8_t* t, cudaStream_t s) {
  const int n_groups = (N + kTcRows - 1) / kTcRows;
  tile_weights_kernel<int8_t, uint2><<<1024, 256, 0, s>>>(w, N, K, n_groups, G, t);
  return cudaGetLastError();
}

// After a prefill pass: every session's kv_len advances by the pass's prompt
// tokens, unless the pass set the device error word (then nothing was
// appended consistently).
__global__ void advance_kv_kernel(qtts_session* sess, int B, const int* err, int inc) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < B && *(const volatile int*)err == 0) sess[b].kv_len += inc;
}

cudaError_t launch_advance_kv(qtts_session* sess, int B, const int* err, int inc, cudaStream_t s) {
  advance_kv_kernel<<<1, 32, 0, s>>>(sess, B, err, inc);
  return cudaGetLastError();
}

}  // namespace qtts
