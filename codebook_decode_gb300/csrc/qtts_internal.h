// Internal declarations shared by the library's CUDA translation units.
// Nothing here is part of the C ABI (include/qtts.h).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "qtts.h"

namespace qtts {

constexpr int kThreads = 384;            // one persistent CTA per SM
constexpr int kWarps = kThreads / 32;
constexpr int kMaxBatch = 32;
constexpr int kMaxRows = 2 * kMaxBatch;  // Code-Predictor step 1 runs two positions per session
constexpr int kCodebooks = 16;
constexpr int kPage = 16;
constexpr int kMaxSplits = 128;          // split-K pieces per (session, kv head) in Talker attention
constexpr int kMinChunk = 16;            // positions per split: at least one KV page
constexpr int kMaxContext = kMaxSplits * kMinChunk;
// dynamic shared memory: a work region (GEMV activation tile, attention
// tiles, sampler), the GEMV partials, then the ring of weight slots
constexpr int kWorkBytes = 80 * 1024;
constexpr int kTailBytes = 12 * 1024;
// the last: a guard band after the ring. A tensor-path MMA reads 128 weight
// rows from its ring slot while a CTA's slice may have fewer; the extra rows
// (whose results are never used) read past the slot's data, at most
// kTcOverread bytes, which must stay inside the allocation.
constexpr int kTcOverread = 4 * 1024;
constexpr int kSmemBytes = kWorkBytes + kTailBytes + 128 * 1024 + kTcOverread;
constexpr int kMaxVocab = 4096;
constexpr int kMaxGrid = 256;            // persistent CTAs (SMs) the kernel supports
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;  // device-side wait limit: 2 s (a frame takes ms)

enum StageType { ST_BEGIN = 0, ST_GEMV = 1, ST_ATTN_T = 2, ST_ATTN_CP = 3, ST_SAMPLE = 4 };
enum XSrc { X_NORM = 0, X_PLAIN = 1 };
enum Epi { E_QKV_T = 0, E_QKV_CP = 1, E_RESID = 2, E_SWIGLU = 3, E_LOGITS = 4, E_CPIN = 5 };

// Activations pass between stages (and CTAs) as tagged 8-byte words: the
// payload in the low 32 bits, in the high 32 bits the tag of the frame and
// stage that wrote it (frame tag base + stage index). A consumer re-reads a
// word until the tag is the one it expects, so stages need no grid barrier.
// Payload: one fp32 value, except in the Code-Predictor cache (two bf16).

// One weight segment of a GEMV stage: rows [0, N) of W, split over the grid
// in units of `unit` rows, each finished by epilogue `epi`.
struct Seg {
  const void* w;          // bf16 [N][K] or int8 [N][K]
  const float* scale;     // int8 per-row scale; nullptr for bf16
  int N;
  int unit;               // 2: rows come in (RoPE pair | gate,up | v pair) pairs
  int epi;
  int out_stride;         // words per destination row
  int out_rps, out_off;   // destination row of (session b, position p) = b*out_rps + out_off + p
  int r_ws[2];            // E_RESID: stage that wrote the residual row of position p
  uint64_t* out;          // tagged destination rows
  const uint64_t* resid;  // E_RESID: residual rows, laid out like `out`
  const uint16_t* bias;   // E_CPIN: optional bf16 bias [N]
  const void* wt;         // the weights (bf16, or int8 with `scale`) as tensor-core tiles for one K-slice
                          // (see below), or nullptr
  const void* wtk;        // the same for the K-split partition (tc_ksplit > 1), or nullptr
};

// Tensor-core copy of a bf16 weight matrix, packed per CTA of one K-slice of
// the persistent grid (C CTAs per slice, see tc_ksplit): rows are split into
// 16-row groups, CTA c of C takes groups [n_groups c / C, n_groups (c+1) / C),
// i.e. rows [r0, r0 + rows_c), and its slice starts at element r0 * K and is
// one K-major canonical tile without swizzle: core matrix (k/8, row/8) of 8
// rows x 8 bf16 at element ((k/8) * rows_c/8 + row/8) * 64, row-major inside,
// so a K range of the slice is contiguous. Rows past N are zero.
constexpr int kTcRows = 16;
constexpr int kTcK = 128;
constexpr int kTcMaxRows = 128;  // rows of one CTA's slice (the MMA's N)
constexpr int kTcMaxActRows = 64;  // activation rows (sessions x rows per session) the tensor path takes

// Whether S K-slices keep every share of the grid within kTcMaxRows rows.
__host__ __device__ inline bool tc_fits(int N, int K, int G, int S) {
  const int ngroups = (N + kTcRows - 1) / kTcRows;
  const int C = G / S;
  return C >= 1 && (K / kTcK) % S == 0 && (ngroups + C - 1) / C * kTcRows <= kTcMaxRows;
}
// K-split of a tensor-path segment (N rows, K) over a grid of G CTAs: the
// grid's first S C CTAs (C = G / S) form S K-slices; CTA c of slice s takes
// the 16-row groups [n_groups c / C, n_groups (c + 1) / C) over the 128-wide
// K chunks [s K / S, (s + 1) K / S). The CTAs c of the S slices split the
// share's rows S ways: each hands its partial sums of the others' rows to
// them, adds theirs of its own rows and runs their epilogues. Among the
// powers of two S <= kTcMaxSplit that divide K / kTcK and keep a share within
// kTcMaxRows rows, S minimises the words a CTA reads per activation row: its K range
// (K / S) plus the partial sums exchanged ((S - 1) x its rows); ties
// take the smaller S. 0: none fits. A second copy of the weight tiles is
// packed for this partition (C CTAs per slice); a stage takes it from
// ksplit_min_rows activation rows up, else the one-slice copy (S = 1).
constexpr int kTcMaxSplit = 4;
__host__ __device__ inline int tc_ksplit(int N, int K, int G) {
  const int ngroups = (N + kTcRows - 1) / kTcRows;
  int best = 0, best_cost = 0;
  for (int S = 1; S <= kTcMaxSplit; S *= 2) {
    if (!tc_fits(N, K, G, S)) continue;
    const int rows = (ngroups + G / S - 1) / (G / S) * kTcRows;
    const int cost = K / S + (S - 1) * rows / S;
    if (!best || cost < best_cost) {
      best = S;
      best_cost = cost;
    }
  }
  return best;
}
// Words of the partial-sum exchange area one K-split segment needs: per
// slice, [n_groups * 16][rows] partial sums then [rows] partial sums of
// squares (each slice runs the epilogues of 1/S of the rows of its share and
// gathers the other slices' partial sums of those rows).
__host__ __device__ inline long long tc_kpart_words(int N, int K, int G, int rows) {
  const int S = tc_ksplit(N, K, G);
  const long long npad = (long long)(N + kTcRows - 1) / kTcRows * kTcRows;
  return S > 1 ? (long long)S * (npad * rows + rows) : 0;
}

struct alignas(16) StageDesc {
  int type;
  int rps;                // rows (positions) per session this stage works on
  int pos_base;           // Code-Predictor position of row p of a session: pos_base + p
  int layer;
  int codebook;           // head / sample stages
  // GEMV input X [rows][K] (tagged words)
  int K;
  int xsrc;
  int in_rps, in_off;     // input row of (b, p) = b*in_rps + in_off + p
  int x_stride;           // words per input row
  int x_ws[2];            // stage that wrote the input row of position p
  int nseg;
  const uint64_t* x;
  const uint16_t* gain;   // X_NORM gain [K]
  Seg seg[2];
  // attention: q [rows][q_stride] in, attn_out [rows][q_stride] out
  const uint64_t* q;
  uint64_t* attn_out;
  int q_stride;
  int q_ws;               // stage that wrote q (and the current K/V)
  uint64_t* kvcur;        // Talker: this frame's K and V rows [kMaxBatch][2][nkv][d]
  uint64_t* cp_kv;        // Code-Predictor cache of this layer [kMaxBatch][2][nkv][16][d/2]
  // sampler
  int V;
  int l_ws;               // stage that wrote the logits
  const uint64_t* logits; // [kMaxBatch][V] tagged
  const float* table;     // projected embedding table T_j [V_j][Hc] fp32 (nullptr for j = 15)
  uint64_t* x_next;       // begin: Talker input rows; sampler: next Code-Predictor input rows
  int next_rps, next_off;
};

// Model-constant device pointers and sizes, passed by value to the kernel.
struct Globals {
  int H, nq, nkv, d, F, V0;
  int Hc, nqc, nkvc, dc, Fc, Vc;
  int eos_id, n_codes, seen_words, max_context;
  float eps;
  int G;                  // persistent grid size (SM count)
  uint16_t* kv_pool;      // [layer][page][2][nkv][16][d]
  int pool_pages;
  const float* rope_cos;  // [max_context][d/2]
  const float* rope_sin;
  const float* cp_rope_cos;  // [16][dc/2]
  const float* cp_rope_sin;
  float* attn_part;       // [kMaxBatch][nkv][kMaxSplits][grp][d + 2]
  unsigned* attn_cnt;     // [layer][kMaxBatch][nkv] split arrivals (wrap to 0 on the last)
  int* err;               // device error word (QTTS_DEV_*)
  int n_stages;
  int ring_slots;         // weight-ring slots in use (1..8): how far the producer may run ahead
  int tc_min_rows;        // fewest activation rows (sessions x rows per session) a GEMV takes on the tensor path
  int ksplit_min_rows;    // fewest activation rows for which a tensor-path segment takes its K-split partition
  uint64_t* kpart;        // K-split partial sums: two areas of kpart_words tagged words (by stage parity)
  long long kpart_words;
  unsigned long long* trace;  // optional [trace_ctas][n_stages][8] %globaltimer stamps, then ring events
  int trace_ctas;         // 2: the first and the last CTA; G: every CTA
  unsigned long long wait_ns;  // time limit of each wait for other CTAs' data or for weights
};

struct FrameArgs {
  int B;
  uint32_t tag0;          // this frame's tag base: a word written by stage s carries tag0 + s
  qtts_session* sess;
  const int32_t* bt;
  int bt_stride;
  const uint16_t* in_embeds;
  qtts_rng* rng;
  uint32_t* seen;
  const int32_t* forced;
  int32_t* codes_out;
  uint8_t* eos_out;
  float* logits_out;
};

// frame_kernel.cu
// stages [s0, s1) of the program: one cooperative launch, or one launch per stage
cudaError_t launch_frame(const StageDesc* prog, int s0, int s1, const Globals& g, const FrameArgs& fa,
                         bool stepwise, cudaStream_t stream);
cudaError_t frame_kernel_setup();
cudaError_t frame_kernel_occupancy(int* blocks_per_sm);
cudaError_t launch_sample(const float* logits, int V, int j, const Globals& g, const FrameArgs& fa,
                          cudaStream_t stream);

// util_kernels.cu
cudaError_t launch_gather_rows(uint16_t* dst, const uint16_t* src, const int32_t* map, int n_rows, int K,
                               cudaStream_t s);
cudaError_t launch_quantize_rows(const uint16_t* w, int N, int K, int8_t* q, float* scale, cudaStream_t s);
cudaError_t launch_project_table(const uint16_t* E, int rows, int H, const uint16_t* P, const int8_t* P8,
                                 const float* P8s, const uint16_t* bias, int Hc, float* T, cudaStream_t s);
cudaError_t launch_kv_scatter(uint16_t* pool, int pool_pages, int nkv, int d, int layer, int n_tok,
                              const int32_t* pages, uint16_t* k, uint16_t* v, int to_pool, cudaStream_t s);
// Requires K % kTcK == 0; t holds ceil(N / 16) * 16 * K bf16; G: the grid the slices are cut for.
cudaError_t launch_tile_weights(const uint16_t* w, int N, int K, int G, uint16_t* t, cudaStream_t s);
cudaError_t launch_tile_weights_i8(const int8_t* w, int N, int K, int G, int8_t* t, cudaStream_t s);
cudaError_t launch_advance_kv(qtts_session* sess, int B, const int* err, int inc, cudaStream_t s);
struct EmbedTables {
  const uint16_t* e[kCodebooks];
  int rows[kCodebooks];
};
cudaError_t launch_feedback(int B, int H, const int32_t* codes, const uint16_t* text, EmbedTables tables,
                            uint16_t* out, cudaStream_t s);

// prefill.cu: the Talker prompt pass over chunks of up to kPfMaxRows rows
// (B sessions x P prompt tokens, row p B + b), on tcgen05 GEMMs
constexpr int kPfMaxRows = 1024;
struct PfLayer {
  const uint16_t *qkv, *o, *gu, *down;  // weights as prefill GEMM tiles (pf_pack_weights)
  const uint16_t *in_norm, *post_norm;  // RMSNorm gains [H] bf16
};
struct PfCtx {
  int n_layers, H, nq, nkv, d, F;
  float eps;
  int G;                    // SMs
  const PfLayer* layers;    // host array [n_layers]
  uint16_t* kv_pool;
  int pool_pages, max_context;
  const float* rope_cos;    // [max_context][d/2]
  const float* rope_sin;
  int* err;
  unsigned long long wait_ns;
  // scratch (device): residual rows, q rows, packed GEMM inputs, partial sums
  float* x;                 // [kPfMaxRows][H]
  float* q;                 // [kPfMaxRows][nq d]
  uint16_t* A;              // pf_act_elems(kPfMaxRows, max(H, nq d, F))
  uint16_t* A2;             // pf_act_elems(kPfMaxRows, F): the down GEMM's input when gate/up applies SwiGLU
  float* part;              // part_floats
  size_t part_floats;
  float* po;                // attention partials: pf_attn_floats(kPfMaxRows, nq, d, max_context)
  int max_rows;
};
size_t pf_packed_elems(int N, int K);  // bf16 elements of one weight's prefill tiles
size_t pf_act_elems(int rows, int maxK);
size_t pf_part_floats(int rows, int maxN);
int pf_attn_chunks(int max_context);
size_t pf_attn_floats(int rows, int nq, int d, int max_context);
cudaError_t pf_setup();
cudaError_t pf_pack_weights(const uint16_t* w, int N, int K, uint16_t* dst, cudaStream_t s);
// one chunk: validate, run the layers, append K/V (kv_len is not advanced here)
cudaError_t pf_chunk(const PfCtx& c, int B, int P, const qtts_session* sess, const int32_t* bt, int bt_stride,
                     const uint16_t* embeds, cudaStream_t s);
// a decode frame's Talker half on the same kernels (one row per session, the
// new token at kv_len, the whole last layer): its K/V appended, its output
// rows written as tagged words with `tag` to x_words [B][H] (the frame
// kernel's codebook-0 head stage reads them); kv_len is not advanced here
cudaError_t pf_talker_step(const PfCtx& c, int B, const qtts_session* sess, const int32_t* bt, int bt_stride,
                           const uint16_t* in_embeds, uint64_t* x_words, uint32_t tag, cudaStream_t s);

// qtts_api.cu: model internals for other translation units
struct KvLayout {
  int device;
  uint16_t* pool;
  int pool_pages, n_layers, nkv, d;
};
int model_kv_layout(qtts_model* m, KvLayout* out);
int model_fail(qtts_model* m, int code, const char* msg);

}  // namespace qtts
