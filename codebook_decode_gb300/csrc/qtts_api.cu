// qtts_api.cu -- the C ABI (include/qtts.h): model creation, weight loading
// with the two-way coverage check, INT8 quantisation, the KV page pool, the
// frame's stage program and the frame launches.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <string>
#include <vector>

#include "qtts_internal.h"

using namespace qtts;

namespace {

thread_local std::string g_create_error;

struct LinW {
  uint16_t* w = nullptr;  // bf16 [N][K], GPU row order
  uint16_t* t = nullptr;  // the same as tensor-core tiles, one K-slice (K % 128 == 0 only)
  uint16_t* tk = nullptr; // the same as tensor-core tiles for the K-split partition (tc_ksplit > 1 only)
  int8_t* tq = nullptr;   // q as tensor-core tiles, one K-slice
  int8_t* tqk = nullptr;  // q as tensor-core tiles for the K-split partition
  int8_t* q = nullptr;    // int8 [N][K]
  float* s = nullptr;     // [N]
  uint16_t* pf = nullptr; // Talker weights only: bf16 tiles of the prefill GEMMs (pf_pack_weights)
  int N = 0, K = 0;
};

struct LayerW {
  uint16_t* in_norm = nullptr;
  uint16_t* post_norm = nullptr;
  LinW qkv, o, gu, down;
};

// How one named tensor lands in device memory.
enum Kind { K_COPY, K_Q, K_K, K_V, K_GATE, K_UP };

struct Spec {
  std::string name;
  int ndim;
  int64_t shape[2];
  Kind kind;
  void* dst;  // K_COPY destination
};

// Tagged activation buffers (see StageDesc): two copies of each per-layer
// kind, used by alternate layers, so a layer never overwrites words the
// previous layer's readers may still be polling.
struct Acts {
  uint64_t* xin = nullptr;                    // Talker input rows [kMaxBatch][H]
  uint64_t *q[2] = {}, *kvcur[2] = {}, *att[2] = {}, *xmid[2] = {}, *xout[2] = {}, *act[2] = {};
  uint64_t* logits0 = nullptr;                // [kMaxBatch][V0 padded even]
  uint64_t* cpx = nullptr;                    // Code-Predictor step-1 inputs [kMaxBatch][2][Hc]
  uint64_t *qc[2] = {}, *attc[2] = {}, *xmidc[2] = {}, *xoutc[2] = {}, *actc[2] = {};
  uint64_t* logitsc[2] = {};                  // [kMaxBatch][Vc padded even]
  uint64_t* xnext[2] = {};                    // [kMaxBatch][Hc]
  uint64_t* cpkv = nullptr;                   // [cp_layers][kMaxBatch][2][nkvc][16][dc/2]
  uint64_t* base = nullptr;
  size_t words = 0;
};

}  // namespace

struct qtts_model {
  qtts_config cfg{};
  int device = 0;
  int G = 0;
  std::string err;
  std::vector<void*> allocs;

  std::vector<LayerW> tl, cl;
  uint16_t* final_norm = nullptr;
  uint16_t* cp_final_norm = nullptr;
  uint16_t* proj_b = nullptr;
  LinW head0, proj;
  LinW cp_head[kCodebooks];
  uint16_t* embed[kCodebooks] = {};
  float* T_bf[kCodebooks] = {};
  float* T_i8[kCodebooks] = {};
  bool loaded = false, quantized = false, use_int8 = false, stepwise = false;
  int chunk_talker_min_b = kMaxBatch + 1;  // BF16 frames of this many sessions or more run the Talker on the chunk kernels (off)

  uint16_t* kv_pool = nullptr;
  std::vector<int32_t> free_ids;
  std::vector<uint8_t> page_used;

  Acts acts;
  uint32_t frame_seq = 0;  // frames launched since the buffers were last cleared
  unsigned long long* trace_buf = nullptr;
  Globals g{};
  StageDesc* prog_dev[2] = {nullptr, nullptr};
  int n_stages = 0;
  int s_cp = 0;               // first Code-Predictor stage of the program
  bool cp_pending = false;    // qtts_frame_talker ran; its qtts_frame_cp has not
  uint32_t cp_tag0 = 0;       // that frame's tag base
  uint16_t* fb[2] = {nullptr, nullptr};  // qtts_frame_steps: next-frame inputs [max_batch][H]

  // prefill: per-layer weight tiles and gains, scratch (built with the weights)
  std::vector<PfLayer> pf_layers;
  PfCtx pf{};

  // staging for qtts_frame_step_host
  qtts_session* st_sess = nullptr;
  int32_t* st_bt = nullptr;
  int st_bt_cap = 0;
  uint16_t* st_in = nullptr;
  qtts_rng* st_rng = nullptr;
  uint32_t* st_seen = nullptr;
  int32_t* st_forced = nullptr;
  int32_t* st_codes = nullptr;
  uint8_t* st_eos = nullptr;
  float* st_logits = nullptr;

  cudaStream_t last_stream = nullptr;
};

namespace {

int fail(qtts_model* m, int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  if (m) m->err = buf;
  else g_create_error = buf;
  return code;
}

int cuda_fail(qtts_model* m, cudaError_t e, const char* what) {
  return fail(m, e == cudaErrorMemoryAllocation ? QTTS_E_OOM : QTTS_E_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define CK(m, call)                                          \
  do {                                                       \
    cudaError_t e_ = (call);                                 \
    if (e_ != cudaSuccess) return cuda_fail((m), e_, #call); \
  } while (0)

template <typename T>
int dalloc(qtts_model* m, T** p, size_t count) {
  void* v = nullptr;
  const size_t bytes = std::max<size_t>(count * sizeof(T), 16);
  cudaError_t e = cudaMalloc(&v, bytes);
  if (e != cudaSuccess) return cuda_fail(m, e, "cudaMalloc");
  e = cudaMemset(v, 0, bytes);
  m->allocs.push_back(v);
  if (e != cudaSuccess) return cuda_fail(m, e, "cudaMemset");
  *p = (T*)v;
  return QTTS_OK;
}

#define AL(m, p, n)                              \
  do {                                           \
    int rc_ = dalloc((m), &(p), (size_t)(n));    \
    if (rc_ != QTTS_OK) return rc_;              \
  } while (0)

bool cfg_ok(const qtts_config& c, std::string& why) {
  auto pos = [&](int v, const char* n) {
    if (v <= 0) {
      why = std::string(n) + " must be positive";
      return false;
    }
    return true;
  };
  if (!pos(c.hidden, "hidden") || !pos(c.n_layers, "n_layers") || !pos(c.n_q_heads, "n_q_heads") ||
      !pos(c.n_kv_heads, "n_kv_heads") || !pos(c.head_dim, "head_dim") || !pos(c.ffn, "ffn") ||
      !pos(c.vocab0, "vocab0") || !pos(c.cp_hidden, "cp_hidden") || !pos(c.cp_layers, "cp_layers") ||
      !pos(c.cp_n_q_heads, "cp_n_q_heads") || !pos(c.cp_n_kv_heads, "cp_n_kv_heads") ||
      !pos(c.cp_head_dim, "cp_head_dim") || !pos(c.cp_ffn, "cp_ffn") || !pos(c.cp_vocab, "cp_vocab") ||
      !pos(c.max_batch, "max_batch") || !pos(c.max_context, "max_context") || !pos(c.kv_pool_pages, "kv_pool_pages"))
    return false;
  if (c.n_codebooks != kCodebooks) return why = "n_codebooks must be 16", false;
  if (c.page_size != kPage) return why = "page_size must be 16", false;
  if (c.max_batch > kMaxBatch) return why = "max_batch must be <= 32", false;
  if (c.max_context > kMaxContext) return why = "max_context must be <= 2048", false;
  if (c.vocab0 > kMaxVocab || c.cp_vocab > kMaxVocab) return why = "vocabularies must be <= 4096", false;
  if (c.cp_vocab > c.vocab0) return why = "cp_vocab must be <= vocab0", false;
  if (c.eos_id < 0 || c.eos_id >= c.vocab0) return why = "eos_id outside vocab0", false;
  if (c.n_codes <= 0 || c.n_codes > c.cp_vocab) return why = "n_codes must be in 1..cp_vocab", false;
  for (int hd : {c.head_dim, c.cp_head_dim})
    if (hd != 64 && hd != 128) return why = "head dims must be 64 or 128", false;
  if (c.n_q_heads % c.n_kv_heads || c.cp_n_q_heads % c.cp_n_kv_heads) return why = "q heads % kv heads != 0", false;
  for (int gg : {c.n_q_heads / c.n_kv_heads, c.cp_n_q_heads / c.cp_n_kv_heads})
    if (gg != 1 && gg != 2) return why = "GQA group must be 1 or 2", false;
  if (c.n_kv_heads > 32 || c.cp_n_kv_heads > 32) return why = "at most 32 kv heads", false;
  // every GEMM K must be a multiple of 16 (16-byte weight rows in int8 for
  // the bulk copies) and one activation row plus the gains must fit the
  // GEMV's shared-memory tile
  for (int k : {c.hidden, c.ffn, c.n_q_heads * c.head_dim, c.cp_hidden, c.cp_ffn, c.cp_n_q_heads * c.cp_head_dim}) {
    if (k % 16) return why = "GEMM reduction sizes must be multiples of 16", false;
    if ((size_t)k * 8 > (size_t)kWorkBytes) return why = "a GEMM reduction size exceeds the activation tile", false;
  }
  if (!(c.rms_eps > 0.f) || !(c.rope_theta > 0.f) || !(c.cp_rope_theta > 0.f))
    return why = "eps and rope theta must be positive", false;
  return true;
}

int seen_words(const qtts_config& c) { return (c.vocab0 + 31) / 32; }

// --------------------------------------------------------------------------
// stage program
// --------------------------------------------------------------------------

Seg make_seg(const LinW& L, bool i8, int unit, int epi, uint64_t* out, int out_stride, int out_rps, int out_off,
             const uint64_t* resid, int r_ws0, int r_ws1, const uint16_t* bias) {
  Seg s{};
  s.w = i8 ? (const void*)L.q : (const void*)L.w;
  s.wt = i8 ? (const void*)L.tq : (const void*)L.t;
  s.wtk = i8 ? (const void*)L.tqk : (const void*)L.tk;
  s.scale = i8 ? L.s : nullptr;
  s.N = L.N;
  s.unit = unit;
  s.epi = epi;
  s.out = out;
  s.out_stride = out_stride;
  s.out_rps = out_rps;
  s.out_off = out_off;
  s.resid = resid;
  s.r_ws[0] = r_ws0;
  s.r_ws[1] = r_ws1;
  s.bias = bias;
  return s;
}

StageDesc gemv(int rps, int pos_base, int layer, int K, int xsrc, const uint64_t* x, int x_stride, int in_rps,
               int in_off, int x_ws0, int x_ws1, const uint16_t* gain) {
  StageDesc d{};
  d.type = ST_GEMV;
  d.rps = rps;
  d.pos_base = pos_base;
  d.layer = layer;
  d.K = K;
  d.xsrc = xsrc;
  d.x = x;
  d.x_stride = x_stride;
  d.in_rps = in_rps;
  d.in_off = in_off;
  d.x_ws[0] = x_ws0;
  d.x_ws[1] = x_ws1;
  d.gain = gain;
  d.nseg = 1;
  return d;
}

int even(int v) { return (v + 1) & ~1; }

// The frame as a sequence of stages; each reads tagged words that earlier
// stages wrote (x_ws / r_ws / q_ws / l_ws name the writing stage):
//   begin; Talker x L_T: [norm+QKV+RoPE+KV append] [attention] [O + residual]
//   [norm+gate|up+SwiGLU] [down + residual]; [final norm + codebook-0 head
//   + projection of h_t]; [sampler 0 + T_0 gather];
//   for j = 1..15: Code Predictor x L_C (the same five stages, two positions
//   per session at j = 1), [final norm + head j], [sampler j + T_j gather].
std::vector<StageDesc> build_program(qtts_model* m, bool i8) {
  const qtts_config& c = m->cfg;
  const Acts& A = m->acts;
  std::vector<StageDesc> P;
  StageDesc b{};
  b.type = ST_BEGIN;
  b.rps = 1;
  b.x_next = A.xin;
  P.push_back(b);
  // the current residual stream: buffer, row layout and writing stage per position
  struct Cur {
    const uint64_t* x;
    int rps, ws[2];
  };
  auto layer_stages = [&](const LayerW& L, bool talker, int l, int par, int rps, int pos_base, uint64_t* cp_kv,
                          Cur& cur) {
    const int H = talker ? c.hidden : c.cp_hidden;
    const int F = talker ? c.ffn : c.cp_ffn;
    const int qw = talker ? c.n_q_heads * c.head_dim : c.cp_n_q_heads * c.cp_head_dim;
    uint64_t* q = talker ? A.q[par] : A.qc[par];
    uint64_t* att = talker ? A.att[par] : A.attc[par];
    uint64_t* xmid = talker ? A.xmid[par] : A.xmidc[par];
    uint64_t* xout = talker ? A.xout[par] : A.xoutc[par];
    uint64_t* act = talker ? A.act[par] : A.actc[par];
    const int sq = (int)P.size();
    StageDesc d = gemv(rps, pos_base, l, H, X_NORM, cur.x, H, cur.rps, 0, cur.ws[0], cur.ws[1], L.in_norm);
    d.seg[0] = make_seg(L.qkv, i8, 2, talker ? E_QKV_T : E_QKV_CP, q, qw, rps, 0, nullptr, 0, 0, nullptr);
    d.kvcur = talker ? A.kvcur[par] : nullptr;
    d.cp_kv = cp_kv;
    P.push_back(d);
    StageDesc a{};
    a.type = talker ? ST_ATTN_T : ST_ATTN_CP;
    a.rps = rps;
    a.pos_base = pos_base;
    a.layer = l;
    a.q = q;
    a.q_ws = sq;
    a.attn_out = att;
    a.q_stride = qw;
    a.kvcur = d.kvcur;
    a.cp_kv = cp_kv;
    P.push_back(a);
    d = gemv(rps, pos_base, l, qw, X_PLAIN, att, qw, rps, 0, sq + 1, sq + 1, nullptr);
    d.seg[0] = make_seg(L.o, i8, 1, E_RESID, xmid, H, rps, 0, cur.x, cur.ws[0], cur.ws[1], nullptr);
    P.push_back(d);
    d = gemv(rps, pos_base, l, H, X_NORM, xmid, H, rps, 0, sq + 2, sq + 2, L.post_norm);
    d.seg[0] = make_seg(L.gu, i8, 2, E_SWIGLU, act, F, rps, 0, nullptr, 0, 0, nullptr);
    P.push_back(d);
    d = gemv(rps, pos_base, l, F, X_PLAIN, act, F, rps, 0, sq + 3, sq + 3, nullptr);
    d.seg[0] = make_seg(L.down, i8, 1, E_RESID, xout, H, rps, 0, xmid, sq + 2, sq + 2, nullptr);
    P.push_back(d);
    cur = Cur{xout, rps, {sq + 4, sq + 4}};
  };
  Cur cur{A.xin, 1, {0, 0}};
  for (int l = 0; l < c.n_layers; ++l) layer_stages(m->tl[l], true, l, l & 1, 1, 0, nullptr, cur);
  const int sh = (int)P.size();
  StageDesc h = gemv(1, 0, 0, c.hidden, X_NORM, cur.x, c.hidden, 1, 0, cur.ws[0], cur.ws[1], m->final_norm);
  h.codebook = 0;
  h.nseg = 2;
  h.seg[0] = make_seg(m->head0, i8, 1, E_LOGITS, A.logits0, even(c.vocab0), 1, 0, nullptr, 0, 0, nullptr);
  h.seg[1] = make_seg(m->proj, i8, 1, E_CPIN, A.cpx, c.cp_hidden, 2, 0, nullptr, 0, 0, m->proj_b);
  P.push_back(h);
  const int ss = (int)P.size();
  StageDesc s{};
  s.type = ST_SAMPLE;
  s.rps = 1;
  s.codebook = 0;
  s.V = c.vocab0;
  s.logits = A.logits0;
  s.l_ws = sh;
  s.x_stride = even(c.vocab0);
  s.table = i8 ? m->T_i8[0] : m->T_bf[0];
  s.x_next = A.cpx;
  s.next_rps = 2;
  s.next_off = 1;
  P.push_back(s);
  const size_t cp_layer_words = (size_t)kMaxBatch * 2 * c.cp_n_kv_heads * kCodebooks * (c.cp_head_dim / 2);
  Cur cc{A.cpx, 2, {sh, ss}};  // step 1: position 0 = P(h_t) from the head stage, 1 = T_0[c_0] from sampler 0
  for (int j = 1; j < kCodebooks; ++j) {
    const int rps = j == 1 ? 2 : 1;
    const int pos_base = j == 1 ? 0 : j;
    for (int l = 0; l < c.cp_layers; ++l)
      layer_stages(m->cl[l], false, l, ((j - 1) * c.cp_layers + l) & 1, rps, pos_base, A.cpkv + l * cp_layer_words,
                   cc);
    const int shj = (int)P.size();
    // codebook j's logits come from position j: the last row of the session
    StageDesc hd = gemv(1, 0, 0, c.cp_hidden, X_NORM, cc.x, c.cp_hidden, rps, rps - 1, cc.ws[rps - 1],
                        cc.ws[rps - 1], m->cp_final_norm);
    hd.codebook = j;
    hd.seg[0] = make_seg(m->cp_head[j], i8, 1, E_LOGITS, A.logitsc[j & 1], even(c.cp_vocab), 1, 0, nullptr, 0, 0,
                         nullptr);
    P.push_back(hd);
    const int ssj = (int)P.size();
    StageDesc sj{};
    sj.type = ST_SAMPLE;
    sj.rps = 1;
    sj.codebook = j;
    sj.V = c.cp_vocab;
    sj.logits = A.logitsc[j & 1];
    sj.l_ws = shj;
    sj.x_stride = even(c.cp_vocab);
    sj.table = (j < kCodebooks - 1) ? (i8 ? m->T_i8[j] : m->T_bf[j]) : nullptr;
    sj.x_next = A.xnext[j & 1];
    sj.next_rps = 1;
    sj.next_off = 0;
    P.push_back(sj);
    cc = Cur{A.xnext[j & 1], 1, {ssj, ssj}};
  }
  return P;
}

// The GEMV keeps one partial per (row unit, 1024-wide K slice, row) of this
// CTA's share in shared memory; check every segment's share fits.
int check_gemv_tiles(qtts_model* m, const std::vector<StageDesc>& P) {
  for (const StageDesc& d : P) {
    if (d.type != ST_GEMV) continue;
    for (int s = 0; s < d.nseg; ++s) {
      const Seg& sg = d.seg[s];
      const int units = sg.N / sg.unit;
      const int upc = (units + m->G - 1) / m->G;
      const int nkc = (d.K + 1023) / 1024;
      if ((long long)upc * nkc * sg.unit * 8 > 1536 || upc * 8 > 512)
        return fail(m, QTTS_E_INVALID, "a %d x %d GEMV share does not fit the %d-SM grid's shared memory", sg.N,
                    d.K, m->G);
    }
  }
  return QTTS_OK;
}

int upload_program(qtts_model* m, bool i8) {
  std::vector<StageDesc> P = build_program(m, i8);
  // the tensor path's MMA covers a CTA's whole row slice: at most kTcMaxRows
  // rows, for some K-split; K-split segments exchange partial sums through
  // a tagged area (two copies, by stage parity), sized for the largest stage
  long long kpart = 0;
  for (StageDesc& d : P) {
    long long need = 0;
    for (int si = 0; si < d.nseg; ++si) {
      Seg& sg = d.seg[si];
      if (sg.wt && !tc_fits(sg.N, d.K, m->G, 1)) sg.wt = nullptr;
      if (sg.wtk && tc_ksplit(sg.N, d.K, m->G) < 2) sg.wtk = nullptr;
      if (sg.wtk) need += tc_kpart_words(sg.N, d.K, m->G, kTcMaxActRows);
    }
    kpart = std::max(kpart, need);
  }
  if (kpart > m->g.kpart_words) {
    uint64_t* a = nullptr;
    AL(m, a, (size_t)(2 * kpart));
    CK(m, cudaMemset(a, 0, (size_t)(2 * kpart) * sizeof(uint64_t)));  // zero tags match no frame
    m->g.kpart = a;
    m->g.kpart_words = kpart;
  }
  int rc;
  if ((rc = check_gemv_tiles(m, P))) return rc;
  StageDesc*& dst = m->prog_dev[i8 ? 1 : 0];
  if (!dst) AL(m, dst, P.size());
  CK(m, cudaMemcpy(dst, P.data(), P.size() * sizeof(StageDesc), cudaMemcpyHostToDevice));
  m->n_stages = (int)P.size();
  m->s_cp = 1 + 5 * m->cfg.n_layers + 2;  // begin, Talker layers, head 0 + projection, sampler 0
  m->g.n_stages = m->n_stages;
  return QTTS_OK;
}

// --------------------------------------------------------------------------
// weights
// --------------------------------------------------------------------------

std::vector<Spec> specs(qtts_model* m) {
  const qtts_config& c = m->cfg;
  std::vector<Spec> v;
  auto add1 = [&](const std::string& n, int64_t a, void* dst) { v.push_back({n, 1, {a, 0}, K_COPY, dst}); };
  auto add2 = [&](const std::string& n, int64_t a, int64_t b, Kind k, void* dst) {
    v.push_back({n, 2, {a, b}, k, dst});
  };
  auto layer = [&](const std::string& p, LayerW& L, bool t) {
    const int H = t ? c.hidden : c.cp_hidden, nq = t ? c.n_q_heads : c.cp_n_q_heads;
    const int nkv = t ? c.n_kv_heads : c.cp_n_kv_heads, d = t ? c.head_dim : c.cp_head_dim, F = t ? c.ffn : c.cp_ffn;
    add1(p + ".input_norm", H, L.in_norm);
    add2(p + ".q_proj", (int64_t)nq * d, H, K_Q, nullptr);
    add2(p + ".k_proj", (int64_t)nkv * d, H, K_K, nullptr);
    add2(p + ".v_proj", (int64_t)nkv * d, H, K_V, nullptr);
    add2(p + ".o_proj", H, (int64_t)nq * d, K_COPY, L.o.w);
    add1(p + ".post_attn_norm", H, L.post_norm);
    add2(p + ".gate_proj", F, H, K_GATE, nullptr);
    add2(p + ".up_proj", F, H, K_UP, nullptr);
    add2(p + ".down_proj", H, F, K_COPY, L.down.w);
  };
  for (int l = 0; l < c.n_layers; ++l) layer("talker.layers." + std::to_string(l), m->tl[l], true);
  add1("talker.final_norm", c.hidden, m->final_norm);
  add2("talker.codec_head", c.vocab0, c.hidden, K_COPY, m->head0.w);
  for (int j = 0; j < kCodebooks; ++j)
    add2("codec_embed." + std::to_string(j), j == 0 ? c.vocab0 : c.cp_vocab, c.hidden, K_COPY, m->embed[j]);
  add2("cp.proj", c.cp_hidden, c.hidden, K_COPY, m->proj.w);
  if (c.proj_bias) add1("cp.proj_bias", c.cp_hidden, m->proj_b);
  for (int l = 0; l < c.cp_layers; ++l) layer("cp.layers." + std::to_string(l), m->cl[l], false);
  add1("cp.final_norm", c.cp_hidden, m->cp_final_norm);
  for (int j = 1; j < kCodebooks; ++j)
    add2("cp.heads." + std::to_string(j), c.cp_vocab, c.cp_hidden, K_COPY, m->cp_head[j].w);
  return v;
}

// GPU row order of the fused QKV matrix: q heads then k heads with each head's
// rows as rotate-half pairs (i, i + d/2) side by side, then v heads unchanged.
// map[fused row] = row of the stacked [q; k; v] source.
std::vector<int32_t> qkv_map(int nq, int nkv, int d) {
  std::vector<int32_t> map((size_t)(nq + 2 * nkv) * d);
  for (int r = 0; r < (nq + nkv) * d; ++r) {
    const int head = r / d, w = r % d, i = w / 2;
    map[r] = head * d + ((w % 2 == 0) ? i : i + d / 2);
  }
  for (int r = (nq + nkv) * d; r < (nq + 2 * nkv) * d; ++r) map[r] = r;
  return map;
}

// gate/up interleaved: fused row 2i = gate i, 2i + 1 = up i (source [gate; up])
std::vector<int32_t> gu_map(int F) {
  std::vector<int32_t> map(2 * (size_t)F);
  for (int i = 0; i < F; ++i) {
    map[2 * i] = i;
    map[2 * i + 1] = F + i;
  }
  return map;
}

int alloc_lin(qtts_model* m, LinW& L, int N, int K) {
  L.N = N;
  L.K = K;
  AL(m, L.w, (size_t)N * K);
  return QTTS_OK;
}

int alloc_weights(qtts_model* m) {
  const qtts_config& c = m->cfg;
  m->tl.resize(c.n_layers);
  m->cl.resize(c.cp_layers);
  auto layer = [&](LayerW& L, bool t) -> int {
    const int H = t ? c.hidden : c.cp_hidden, nq = t ? c.n_q_heads : c.cp_n_q_heads;
    const int nkv = t ? c.n_kv_heads : c.cp_n_kv_heads, d = t ? c.head_dim : c.cp_head_dim, F = t ? c.ffn : c.cp_ffn;
    AL(m, L.in_norm, H);
    AL(m, L.post_norm, H);
    int rc;
    if ((rc = alloc_lin(m, L.qkv, (nq + 2 * nkv) * d, H))) return rc;
    if ((rc = alloc_lin(m, L.o, H, nq * d))) return rc;
    if ((rc = alloc_lin(m, L.gu, 2 * F, H))) return rc;
    if ((rc = alloc_lin(m, L.down, H, F))) return rc;
    return QTTS_OK;
  };
  int rc;
  for (auto& L : m->tl)
    if ((rc = layer(L, true))) return rc;
  for (auto& L : m->cl)
    if ((rc = layer(L, false))) return rc;
  AL(m, m->final_norm, c.hidden);
  AL(m, m->cp_final_norm, c.cp_hidden);
  if (c.proj_bias) AL(m, m->proj_b, c.cp_hidden);
  if ((rc = alloc_lin(m, m->head0, c.vocab0, c.hidden))) return rc;
  if ((rc = alloc_lin(m, m->proj, c.cp_hidden, c.hidden))) return rc;
  for (int j = 1; j < kCodebooks; ++j)
    if ((rc = alloc_lin(m, m->cp_head[j], c.cp_vocab, c.cp_hidden))) return rc;
  for (int j = 0; j < kCodebooks; ++j) AL(m, m->embed[j], (size_t)(j == 0 ? c.vocab0 : c.cp_vocab) * c.hidden);
  for (int j = 0; j < kCodebooks - 1; ++j) AL(m, m->T_bf[j], (size_t)(j == 0 ? c.vocab0 : c.cp_vocab) * c.cp_hidden);
  return QTTS_OK;
}

std::vector<LinW*> all_lins(qtts_model* m) {
  std::vector<LinW*> v;
  for (auto& L : m->tl) v.insert(v.end(), {&L.qkv, &L.o, &L.gu, &L.down});
  for (auto& L : m->cl) v.insert(v.end(), {&L.qkv, &L.o, &L.gu, &L.down});
  v.push_back(&m->head0);
  v.push_back(&m->proj);
  for (int j = 1; j < kCodebooks; ++j) v.push_back(&m->cp_head[j]);
  return v;
}

// Projected Code-Predictor input tables T_j = E_j P^T (+ b), j = 0..14: the
// projection of a fixed table is itself a fixed table, so a step's input is a
// row gather instead of a GEMV over the 2048x1024 projection.
int build_tables(qtts_model* m, bool i8) {
  const qtts_config& c = m->cfg;
  for (int j = 0; j < kCodebooks - 1; ++j) {
    float* T = i8 ? m->T_i8[j] : m->T_bf[j];
    CK(m, launch_project_table(m->embed[j], j == 0 ? c.vocab0 : c.cp_vocab, c.hidden, i8 ? nullptr : m->proj.w,
                               i8 ? m->proj.q : nullptr, i8 ? m->proj.s : nullptr, m->proj_b, c.cp_hidden, T, 0));
  }
  CK(m, cudaDeviceSynchronize());
  return QTTS_OK;
}

size_t trace_words(const qtts_model* m, int ctas) { return (size_t)8 * ctas * m->n_stages + 4 * 4096; }

enum FramePart { PART_ALL = 0, PART_TALKER = 1, PART_CP = 2 };

// Launch all of a frame's stages, or its Talker half (through sampler 0) or
// its Code-Predictor half (the 15 steps), which reuses the Talker half's tag
// base: its first stages read words the Talker half wrote.
// Tag base of the next launch over the program: stage s writes tag0 + s;
// tags only grow, so no word left by an earlier launch matches. Before they
// would wrap, the tagged buffers are cleared and the count restarts.
int take_tag0(qtts_model* m, uint32_t* tag0) {
  if ((uint64_t)(m->frame_seq + 2) * (uint64_t)m->n_stages >= 0xFFFFFFFFull) {
    CK(m, cudaDeviceSynchronize());
    CK(m, cudaMemset(m->acts.base, 0, m->acts.words * sizeof(uint64_t)));
    if (m->g.kpart) CK(m, cudaMemset(m->g.kpart, 0, (size_t)(2 * m->g.kpart_words) * sizeof(uint64_t)));
    m->frame_seq = 0;
  }
  ++m->frame_seq;
  *tag0 = m->frame_seq * (uint32_t)m->n_stages;
  return QTTS_OK;
}

int frame_part(qtts_model* m, int part, int B, qtts_session* sess, const int32_t* bt, int bt_stride,
               const uint16_t* in_embeds, qtts_rng* rng, uint32_t* seen, const int32_t* forced, int32_t* codes_out,
               uint8_t* eos_out, float* logits_out, void* stream) {
  if (!m) return fail(m, QTTS_E_INVALID, "null model");
  if (!m->loaded) return fail(m, QTTS_E_STATE, "load weights first");
  if (B < 1 || B > m->cfg.max_batch) return fail(m, QTTS_E_BATCH, "B=%d outside 1..%d", B, m->cfg.max_batch);
  if (!sess || !bt || !rng || !codes_out || !eos_out || bt_stride < 1 || (part != PART_CP && !in_embeds))
    return fail(m, QTTS_E_INVALID, "null array or bad block-table stride");
  if (part == PART_CP && !m->cp_pending) return fail(m, QTTS_E_STATE, "qtts_frame_cp needs qtts_frame_talker first");
  cudaSetDevice(m->device);
  FrameArgs fa{};
  fa.B = B;
  fa.sess = sess;
  fa.bt = bt;
  fa.bt_stride = bt_stride;
  fa.in_embeds = in_embeds;
  fa.rng = rng;
  fa.seen = seen;
  fa.forced = forced;
  fa.codes_out = codes_out;
  fa.eos_out = eos_out;
  fa.logits_out = logits_out;
  cudaStream_t s = (cudaStream_t)stream;
  const bool i8 = m->use_int8;
  if (part == PART_CP) {
    fa.tag0 = m->cp_tag0;
  } else {
    int rc = take_tag0(m, &fa.tag0);
    if (rc) return rc;
  }
  const int s0 = part == PART_CP ? m->s_cp : 0;
  const int s1 = part == PART_TALKER ? m->s_cp : m->n_stages;
  const StageDesc* prog = m->prog_dev[i8 ? 1 : 0];
  cudaError_t e;
  if (part != PART_CP && !i8 && B >= m->chunk_talker_min_b) {
    // the Talker on the tensor-core chunk kernels: the begin stage validates
    // the sessions, the chunk kernels run the layers and publish the last
    // layer's rows as the words the codebook-0 head stage reads (tag of the
    // last Talker stage), then the frame kernel runs from that head stage on
    const int L = m->cfg.n_layers, s_head = 1 + 5 * L;
    e = launch_frame(prog, 0, 1, m->g, fa, m->stepwise, s);
    if (e == cudaSuccess) {
      PfCtx ctx = m->pf;
      ctx.wait_ns = m->g.wait_ns;
      e = pf_talker_step(ctx, B, sess, bt, bt_stride, in_embeds, m->acts.xout[(L - 1) & 1], fa.tag0 + (uint32_t)(s_head - 1),
                         s);
    }
    if (e == cudaSuccess) e = launch_frame(prog, s_head, s1, m->g, fa, m->stepwise, s);
  } else {
    e = launch_frame(prog, s0, s1, m->g, fa, m->stepwise, s);
  }
  m->last_stream = s;
  if (e != cudaSuccess) return cuda_fail(m, e, "frame launch");
  m->cp_pending = part == PART_TALKER;
  m->cp_tag0 = fa.tag0;
  return QTTS_OK;
}

// An abandoned frame can leave attention split counters part-way; clear them
// whenever a device error is reported.
cudaError_t reset_split_counters(qtts_model* m) {
  return cudaMemset(m->g.attn_cnt, 0, sizeof(unsigned) * m->cfg.n_layers * kMaxBatch * m->cfg.n_kv_heads);
}

// Tensor-core tile copies of every bf16 GEMM weight whose K is a multiple of
// 128 (the layout the large-batch GEMV stages stream).
// i8: tiles of the int8 weights (after qtts_quantize_int8), else of the bf16 ones.
int build_tensor_tiles(qtts_model* m, bool i8) {
  for (LinW* L : all_lins(m)) {
    if (L->K % kTcK) continue;
    const size_t nr = (size_t)(L->N + kTcRows - 1) / kTcRows * kTcRows;
    const int S = tc_ksplit(L->N, L->K, m->G);
    for (int split = 0; split < 2; ++split) {
      // one K-slice over the whole grid, then the K-split partition (G / S CTAs per slice)
      if (split ? S < 2 : !tc_fits(L->N, L->K, m->G, 1)) continue;
      const int C = split ? m->G / S : m->G;
      if (i8) {
        int8_t*& t = split ? L->tqk : L->tq;
        if (!t) AL(m, t, nr * L->K);
        CK(m, launch_tile_weights_i8(L->q, L->N, L->K, C, t, 0));
      } else {
        uint16_t*& t = split ? L->tk : L->t;
        if (!t) AL(m, t, nr * L->K);
        CK(m, launch_tile_weights(L->w, L->N, L->K, C, t, 0));
      }
    }
  }
  CK(m, cudaDeviceSynchronize());
  return QTTS_OK;
}

// Prefill GEMM tiles of every Talker weight (always the bf16 ones) and the
// prefill scratch for chunks of up to kPfMaxRows rows.
int build_prefill(qtts_model* m) {
  const qtts_config& c = m->cfg;
  m->pf_layers.resize(c.n_layers);
  for (int l = 0; l < c.n_layers; ++l) {
    LayerW& L = m->tl[l];
    for (LinW* W : {&L.qkv, &L.o, &L.gu, &L.down}) {
      AL(m, W->pf, pf_packed_elems(W->N, W->K));
      CK(m, pf_pack_weights(W->w, W->N, W->K, W->pf, 0));
    }
    m->pf_layers[l] = PfLayer{L.qkv.pf, L.o.pf, L.gu.pf, L.down.pf, L.in_norm, L.post_norm};
  }
  PfCtx& p = m->pf;
  p.n_layers = c.n_layers; p.H = c.hidden; p.nq = c.n_q_heads; p.nkv = c.n_kv_heads; p.d = c.head_dim;
  p.F = c.ffn; p.eps = c.rms_eps; p.G = m->G; p.layers = m->pf_layers.data();
  p.kv_pool = m->kv_pool; p.pool_pages = c.kv_pool_pages; p.max_context = c.max_context;
  p.rope_cos = m->g.rope_cos; p.rope_sin = m->g.rope_sin; p.err = m->g.err;
  p.max_rows = kPfMaxRows;
  const int maxK = std::max(std::max(c.hidden, c.n_q_heads * c.head_dim), c.ffn);
  const int maxN = std::max(std::max(c.hidden, (c.n_q_heads + 2 * c.n_kv_heads) * c.head_dim), 2 * c.ffn);
  p.part_floats = pf_part_floats(kPfMaxRows, maxN);
  AL(m, p.x, (size_t)kPfMaxRows * c.hidden);
  AL(m, p.q, (size_t)kPfMaxRows * c.n_q_heads * c.head_dim);
  AL(m, p.A, pf_act_elems(kPfMaxRows, maxK));
  AL(m, p.A2, pf_act_elems(kPfMaxRows, c.ffn));
  AL(m, p.part, p.part_floats);
  AL(m, p.po, pf_attn_floats(kPfMaxRows, c.n_q_heads, c.head_dim, c.max_context));
  CK(m, cudaDeviceSynchronize());
  return QTTS_OK;
}

}  // namespace

// ==========================================================================
// C ABI
// ==========================================================================

extern "C" {

int qtts_abi_version(void) { return QTTS_ABI_VERSION; }

const char* qtts_last_error(const qtts_model* m) { return m ? m->err.c_str() : g_create_error.c_str(); }

void qtts_destroy(qtts_model* m) {
  if (!m) return;
  cudaSetDevice(m->device);
  cudaDeviceSynchronize();
  for (void* p : m->allocs) cudaFree(p);
  delete m;
}

int qtts_create(const qtts_config* cfg, int device, qtts_model** out) {
  if (!cfg || !out) return fail(nullptr, QTTS_E_INVALID, "null argument");
  *out = nullptr;
  std::string why;
  if (!cfg_ok(*cfg, why)) return fail(nullptr, QTTS_E_INVALID, "bad config: %s", why.c_str());
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev)
    return fail(nullptr, QTTS_E_CUDA, "no CUDA device %d", device);
  if (cudaSetDevice(device) != cudaSuccess) return fail(nullptr, QTTS_E_CUDA, "cudaSetDevice(%d) failed", device);
  cudaError_t e = frame_kernel_setup();
  if (e == cudaSuccess) e = pf_setup();
  if (e != cudaSuccess) return fail(nullptr, QTTS_E_CUDA, "kernel setup: %s", cudaGetErrorString(e));
  int coop = 0, sms = 0;
  cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, device);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
  if (!coop) return fail(nullptr, QTTS_E_CUDA, "device %d has no cooperative launch", device);
  if (sms > kMaxGrid) return fail(nullptr, QTTS_E_CUDA, "device %d has more than %d SMs", device, kMaxGrid);
  int occ = 0;
  e = frame_kernel_occupancy(&occ);
  if (e != cudaSuccess || occ < 1)
    return fail(nullptr, QTTS_E_CUDA, "frame kernel cannot keep one CTA per SM resident (%s)", cudaGetErrorString(e));

  qtts_model* m = new qtts_model();
  m->cfg = *cfg;
  m->device = device;
  m->G = sms;
  auto bail = [&](int rc) {
    g_create_error = m->err;
    qtts_destroy(m);
    return rc;
  };
  int rc;
  if ((rc = alloc_weights(m))) return bail(rc);
  const qtts_config& c = m->cfg;
  Globals& g = m->g;
  g.H = c.hidden; g.nq = c.n_q_heads; g.nkv = c.n_kv_heads; g.d = c.head_dim; g.F = c.ffn; g.V0 = c.vocab0;
  g.Hc = c.cp_hidden; g.nqc = c.cp_n_q_heads; g.nkvc = c.cp_n_kv_heads; g.dc = c.cp_head_dim; g.Fc = c.cp_ffn;
  g.Vc = c.cp_vocab; g.eos_id = c.eos_id; g.n_codes = c.n_codes; g.seen_words = seen_words(c);
  g.max_context = c.max_context; g.eps = c.rms_eps; g.G = sms; g.pool_pages = c.kv_pool_pages;
  g.ring_slots = 8;
  g.wait_ns = kDefaultWaitNs;
  g.tc_min_rows = 8;
  g.ksplit_min_rows = 8;

  const size_t kv_elems = (size_t)c.n_layers * c.kv_pool_pages * 2 * c.n_kv_heads * kPage * c.head_dim;
  if ((rc = dalloc(m, &m->kv_pool, kv_elems))) return bail(rc);
  g.kv_pool = m->kv_pool;
  m->page_used.assign(c.kv_pool_pages, 0);
  m->free_ids.resize(c.kv_pool_pages);
  for (int i = 0; i < c.kv_pool_pages; ++i) m->free_ids[i] = c.kv_pool_pages - 1 - i;  // handed out 0, 1, 2, ...

  // RoPE tables: angles in double, stored fp32
  {
    const int half = c.head_dim / 2, chalf = c.cp_head_dim / 2;
    std::vector<float> cs((size_t)c.max_context * half), sn((size_t)c.max_context * half);
    for (int p = 0; p < c.max_context; ++p)
      for (int i = 0; i < half; ++i) {
        const double a = (double)p * std::pow((double)c.rope_theta, -2.0 * i / (double)c.head_dim);
        cs[(size_t)p * half + i] = (float)std::cos(a);
        sn[(size_t)p * half + i] = (float)std::sin(a);
      }
    std::vector<float> ccs((size_t)kCodebooks * chalf), csn((size_t)kCodebooks * chalf);
    for (int p = 0; p < kCodebooks; ++p)
      for (int i = 0; i < chalf; ++i) {
        const double a = (double)p * std::pow((double)c.cp_rope_theta, -2.0 * i / (double)c.cp_head_dim);
        ccs[(size_t)p * chalf + i] = (float)std::cos(a);
        csn[(size_t)p * chalf + i] = (float)std::sin(a);
      }
    float *a = nullptr, *b = nullptr, *cc = nullptr, *dd = nullptr;
    if ((rc = dalloc(m, &a, cs.size())) || (rc = dalloc(m, &b, sn.size())) || (rc = dalloc(m, &cc, ccs.size())) ||
        (rc = dalloc(m, &dd, csn.size())))
      return bail(rc);
    if (cudaMemcpy(a, cs.data(), cs.size() * 4, cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemcpy(b, sn.data(), sn.size() * 4, cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemcpy(cc, ccs.data(), ccs.size() * 4, cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemcpy(dd, csn.data(), csn.size() * 4, cudaMemcpyHostToDevice) != cudaSuccess)
      return bail(fail(m, QTTS_E_CUDA, "RoPE table upload failed"));
    g.rope_cos = a; g.rope_sin = b; g.cp_rope_cos = cc; g.cp_rope_sin = dd;
  }
  const int grp = c.n_q_heads / c.n_kv_heads;
  if ((rc = dalloc(m, &g.attn_part, (size_t)kMaxBatch * c.n_kv_heads * kMaxSplits * grp * (c.head_dim + 2))) ||
      (rc = dalloc(m, &g.attn_cnt, (size_t)c.n_layers * kMaxBatch * c.n_kv_heads)) || (rc = dalloc(m, &g.err, 1)))
    return bail(rc);
  // tagged activation buffers, one arena (zero tags never match a frame's)
  {
    Acts& A = m->acts;
    const size_t B = kMaxBatch, R = kMaxRows;
    const size_t qt = (size_t)c.n_q_heads * c.head_dim, qc = (size_t)c.cp_n_q_heads * c.cp_head_dim;
    std::vector<std::pair<uint64_t**, size_t>> parts = {{&A.xin, B * c.hidden},
                                                        {&A.logits0, B * even(c.vocab0)},
                                                        {&A.cpx, B * 2 * c.cp_hidden}};
    for (int i = 0; i < 2; ++i) {
      parts.push_back({&A.q[i], B * qt});
      parts.push_back({&A.kvcur[i], B * 2 * c.n_kv_heads * c.head_dim});
      parts.push_back({&A.att[i], B * qt});
      parts.push_back({&A.xmid[i], B * c.hidden});
      parts.push_back({&A.xout[i], B * c.hidden});
      parts.push_back({&A.act[i], B * c.ffn});
      parts.push_back({&A.qc[i], R * qc});
      parts.push_back({&A.attc[i], R * qc});
      parts.push_back({&A.xmidc[i], R * c.cp_hidden});
      parts.push_back({&A.xoutc[i], R * c.cp_hidden});
      parts.push_back({&A.actc[i], R * c.cp_ffn});
      parts.push_back({&A.logitsc[i], B * even(c.cp_vocab)});
      parts.push_back({&A.xnext[i], B * c.cp_hidden});
    }
    parts.push_back({&A.cpkv, (size_t)c.cp_layers * B * 2 * c.cp_n_kv_heads * kCodebooks * (c.cp_head_dim / 2)});
    size_t total = 0;
    for (auto& pr : parts) total += (pr.second + 31) & ~(size_t)31;  // 256-byte aligned pieces
    if ((rc = dalloc(m, &A.base, total))) return bail(rc);
    A.words = total;
    size_t off = 0;
    for (auto& pr : parts) {
      *pr.first = A.base + off;
      off += (pr.second + 31) & ~(size_t)31;
    }
  }
  // staging for the host-buffer frame
  m->st_bt_cap = (c.max_context + kPage - 1) / kPage;
  if ((rc = dalloc(m, &m->st_sess, kMaxBatch)) || (rc = dalloc(m, &m->st_bt, (size_t)kMaxBatch * m->st_bt_cap)) ||
      (rc = dalloc(m, &m->st_in, (size_t)kMaxBatch * c.hidden)) || (rc = dalloc(m, &m->st_rng, kMaxBatch)) ||
      (rc = dalloc(m, &m->st_seen, (size_t)kMaxBatch * seen_words(c))) ||
      (rc = dalloc(m, &m->st_forced, (size_t)kMaxBatch * kCodebooks)) ||
      (rc = dalloc(m, &m->st_codes, (size_t)kMaxBatch * kCodebooks)) || (rc = dalloc(m, &m->st_eos, kMaxBatch)) ||
      (rc = dalloc(m, &m->st_logits, (size_t)kMaxBatch * kCodebooks * c.vocab0)))
    return bail(rc);
  if (cudaDeviceSynchronize() != cudaSuccess) return bail(fail(m, QTTS_E_CUDA, "setup failed"));
  *out = m;
  return QTTS_OK;
}

int qtts_load_weights(qtts_model* m, const qtts_tensor* t, int n) {
  if (!m || (!t && n)) return fail(m, QTTS_E_INVALID, "null argument");
  if (m->loaded) return fail(m, QTTS_E_STATE, "weights already loaded");
  cudaSetDevice(m->device);
  const qtts_config& c = m->cfg;
  std::vector<Spec> sp = specs(m);
  std::map<std::string, int> idx;
  for (size_t i = 0; i < sp.size(); ++i) idx[sp[i].name] = (int)i;
  std::vector<const qtts_tensor*> got(sp.size(), nullptr);
  for (int i = 0; i < n; ++i) {
    if (!t[i].name) return fail(m, QTTS_E_INVALID, "tensor %d has no name", i);
    auto it = idx.find(t[i].name);
    if (it == idx.end()) return fail(m, QTTS_E_UNUSED, "tensor '%s' is not part of the model", t[i].name);
    if (got[it->second]) return fail(m, QTTS_E_UNUSED, "tensor '%s' supplied twice", t[i].name);
    const Spec& s = sp[it->second];
    if (t[i].dtype != QTTS_DTYPE_BF16 || t[i].ndim != s.ndim || t[i].shape[0] != s.shape[0] ||
        (s.ndim == 2 && t[i].shape[1] != s.shape[1]))
      return fail(m, QTTS_E_SHAPE, "tensor '%s': expected bf16 [%lld%s%lld]", t[i].name, (long long)s.shape[0],
                  s.ndim == 2 ? ", " : "", s.ndim == 2 ? (long long)s.shape[1] : 0LL);
    if (!t[i].data) return fail(m, QTTS_E_INVALID, "tensor '%s' has no data", t[i].name);
    got[it->second] = &t[i];
  }
  for (size_t i = 0; i < sp.size(); ++i)
    if (!got[i]) return fail(m, QTTS_E_MISSING, "tensor '%s' was not supplied", sp[i].name.c_str());

  // fused layouts go through a staging buffer and a row gather
  const size_t stage_rows = std::max<size_t>(
      std::max((size_t)(c.n_q_heads + 2 * c.n_kv_heads) * c.head_dim, (size_t)2 * c.ffn),
      std::max((size_t)(c.cp_n_q_heads + 2 * c.cp_n_kv_heads) * c.cp_head_dim, (size_t)2 * c.cp_ffn));
  const size_t stage_cols = std::max(c.hidden, c.cp_hidden);
  uint16_t* stage = nullptr;
  int32_t* dmap = nullptr;
  CK(m, cudaMalloc(&stage, stage_rows * stage_cols * 2));
  cudaError_t e = cudaMalloc(&dmap, stage_rows * 4);
  if (e != cudaSuccess) {
    cudaFree(stage);
    return cuda_fail(m, e, "cudaMalloc");
  }
  int rc = QTTS_OK;
  auto copy = [&](void* dst, const void* src, size_t bytes) {
    if (rc) return;
    cudaError_t ce = cudaMemcpy(dst, src, bytes, cudaMemcpyDefault);
    if (ce != cudaSuccess) rc = cuda_fail(m, ce, "cudaMemcpy(weights)");
  };
  auto gather = [&](uint16_t* dst, const std::vector<int32_t>& map, int K) {
    if (rc) return;
    cudaError_t ce = cudaMemcpy(dmap, map.data(), map.size() * 4, cudaMemcpyHostToDevice);
    if (ce == cudaSuccess) ce = launch_gather_rows(dst, stage, dmap, (int)map.size(), K, 0);
    if (ce == cudaSuccess) ce = cudaDeviceSynchronize();
    if (ce != cudaSuccess) rc = cuda_fail(m, ce, "weight layout gather");
  };
  for (size_t i = 0; i < sp.size() && !rc; ++i) {
    const Spec& s = sp[i];
    if (s.kind == K_COPY) copy(s.dst, got[i]->data, (size_t)s.shape[0] * (s.ndim == 2 ? s.shape[1] : 1) * 2);
  }
  auto fuse_layer = [&](const std::string& p, LayerW& L, bool tk) {
    const int H = tk ? c.hidden : c.cp_hidden, nq = tk ? c.n_q_heads : c.cp_n_q_heads;
    const int nkv = tk ? c.n_kv_heads : c.cp_n_kv_heads, d = tk ? c.head_dim : c.cp_head_dim, F = tk ? c.ffn : c.cp_ffn;
    copy(stage, got[idx[p + ".q_proj"]]->data, (size_t)nq * d * H * 2);
    copy(stage + (size_t)nq * d * H, got[idx[p + ".k_proj"]]->data, (size_t)nkv * d * H * 2);
    copy(stage + (size_t)(nq + nkv) * d * H, got[idx[p + ".v_proj"]]->data, (size_t)nkv * d * H * 2);
    gather(L.qkv.w, qkv_map(nq, nkv, d), H);
    copy(stage, got[idx[p + ".gate_proj"]]->data, (size_t)F * H * 2);
    copy(stage + (size_t)F * H, got[idx[p + ".up_proj"]]->data, (size_t)F * H * 2);
    gather(L.gu.w, gu_map(F), H);
  };
  for (int l = 0; l < c.n_layers && !rc; ++l) fuse_layer("talker.layers." + std::to_string(l), m->tl[l], true);
  for (int l = 0; l < c.cp_layers && !rc; ++l) fuse_layer("cp.layers." + std::to_string(l), m->cl[l], false);
  cudaFree(stage);
  cudaFree(dmap);
  if (rc) return rc;
  if ((rc = build_tables(m, false))) return rc;
  if ((rc = build_tensor_tiles(m, false))) return rc;
  if ((rc = build_prefill(m))) return rc;
  if ((rc = upload_program(m, false))) return rc;
  m->loaded = true;
  return QTTS_OK;
}

int qtts_quantize_int8(qtts_model* m) {
  if (!m) return fail(m, QTTS_E_INVALID, "null model");
  if (!m->loaded) return fail(m, QTTS_E_STATE, "load weights first");
  cudaSetDevice(m->device);
  if (!m->quantized) {
    const qtts_config& c = m->cfg;
    for (LinW* L : all_lins(m)) {
      AL(m, L->q, (size_t)L->N * L->K);
      AL(m, L->s, (size_t)L->N);
      CK(m, launch_quantize_rows(L->w, L->N, L->K, L->q, L->s, 0));
    }
    for (int j = 0; j < kCodebooks - 1; ++j) AL(m, m->T_i8[j], (size_t)(j == 0 ? c.vocab0 : c.cp_vocab) * c.cp_hidden);
    CK(m, cudaDeviceSynchronize());
    int rc;
    if ((rc = build_tables(m, true))) return rc;
    if ((rc = build_tensor_tiles(m, true))) return rc;
    if ((rc = upload_program(m, true))) return rc;
    m->quantized = true;
  }
  m->use_int8 = true;
  return QTTS_OK;
}

int qtts_set_int8(qtts_model* m, int enable) {
  if (!m) return fail(m, QTTS_E_INVALID, "null model");
  if (enable && !m->quantized) return fail(m, QTTS_E_STATE, "qtts_quantize_int8 has not run");
  m->use_int8 = enable != 0;
  return QTTS_OK;
}

int qtts_export_int8(qtts_model* m, const char* name, int8_t* q_host, float* scale_host) {
  if (!m || !name || !q_host || !scale_host) return fail(m, QTTS_E_INVALID, "null argument");
  if (!m->quantized) return fail(m, QTTS_E_STATE, "qtts_quantize_int8 has not run");
  cudaSetDevice(m->device);
  const qtts_config& c = m->cfg;
  const std::string n(name);
  // rows[i] = fused row that holds row i of the named tensor
  auto copy_rows = [&](const LinW& L, const std::vector<int32_t>& rows) -> int {
    std::vector<int8_t> q((size_t)L.N * L.K);
    std::vector<float> s(L.N);
    CK(m, cudaMemcpy(q.data(), L.q, q.size(), cudaMemcpyDeviceToHost));
    CK(m, cudaMemcpy(s.data(), L.s, s.size() * 4, cudaMemcpyDeviceToHost));
    for (size_t i = 0; i < rows.size(); ++i) {
      memcpy(q_host + i * L.K, q.data() + (size_t)rows[i] * L.K, L.K);
      scale_host[i] = s[rows[i]];
    }
    return QTTS_OK;
  };
  auto plain = [&](const LinW& L) {
    std::vector<int32_t> r(L.N);
    for (int i = 0; i < L.N; ++i) r[i] = i;
    return copy_rows(L, r);
  };
  const int kNoMatch = 1;
  auto layer = [&](const std::string& p, LayerW& L, bool tk) -> int {
    const int nq = tk ? c.n_q_heads : c.cp_n_q_heads, nkv = tk ? c.n_kv_heads : c.cp_n_kv_heads;
    const int d = tk ? c.head_dim : c.cp_head_dim, F = tk ? c.ffn : c.cp_ffn;
    auto inv = [&](int base, int count, bool pairs) {
      std::vector<int32_t> r(count);
      for (int i = 0; i < count; ++i) {
        if (!pairs) {
          r[i] = base + i;
          continue;
        }
        const int head = i / d, w = i % d;
        r[i] = base + head * d + (w < d / 2 ? 2 * w : 2 * (w - d / 2) + 1);
      }
      return r;
    };
    if (n == p + ".q_proj") return copy_rows(L.qkv, inv(0, nq * d, true));
    if (n == p + ".k_proj") return copy_rows(L.qkv, inv(nq * d, nkv * d, true));
    if (n == p + ".v_proj") return copy_rows(L.qkv, inv((nq + nkv) * d, nkv * d, false));
    if (n == p + ".o_proj") return plain(L.o);
    if (n == p + ".down_proj") return plain(L.down);
    if (n == p + ".gate_proj" || n == p + ".up_proj") {
      std::vector<int32_t> r(F);
      for (int i = 0; i < F; ++i) r[i] = 2 * i + (n == p + ".up_proj" ? 1 : 0);
      return copy_rows(L.gu, r);
    }
    return kNoMatch;
  };
  for (int l = 0; l < c.n_layers; ++l) {
    const int rc = layer("talker.layers." + std::to_string(l), m->tl[l], true);
    if (rc != kNoMatch) return rc;
  }
  for (int l = 0; l < c.cp_layers; ++l) {
    const int rc = layer("cp.layers." + std::to_string(l), m->cl[l], false);
    if (rc != kNoMatch) return rc;
  }
  if (n == "talker.codec_head") return plain(m->head0);
  if (n == "cp.proj") return plain(m->proj);
  for (int j = 1; j < kCodebooks; ++j)
    if (n == "cp.heads." + std::to_string(j)) return plain(m->cp_head[j]);
  return fail(m, QTTS_E_INVALID, "'%s' is not a GEMM weight", name);
}

int qtts_kv_alloc_pages(qtts_model* m, int n, int32_t* ids) {
  if (!m || n < 0 || (n && !ids)) return fail(m, QTTS_E_INVALID, "bad argument");
  if ((size_t)n > m->free_ids.size())
    return fail(m, QTTS_E_POOL, "KV pool has %zu free pages, %d requested", m->free_ids.size(), n);
  for (int i = 0; i < n; ++i) {
    ids[i] = m->free_ids.back();
    m->free_ids.pop_back();
    m->page_used[ids[i]] = 1;
  }
  return QTTS_OK;
}

int qtts_kv_free_pages(qtts_model* m, int n, const int32_t* ids) {
  if (!m || n < 0 || (n && !ids)) return fail(m, QTTS_E_INVALID, "bad argument");
  std::vector<uint8_t> seen_now(m->cfg.kv_pool_pages, 0);
  for (int i = 0; i < n; ++i) {
    if (ids[i] < 0 || ids[i] >= m->cfg.kv_pool_pages || !m->page_used[ids[i]] || seen_now[ids[i]])
      return fail(m, QTTS_E_POOL, "page %d is not allocated", ids[i]);
    seen_now[ids[i]] = 1;
  }
  for (int i = 0; i < n; ++i) {
    m->page_used[ids[i]] = 0;
    m->free_ids.push_back(ids[i]);
  }
  return QTTS_OK;
}

int qtts_kv_pool_free_count(const qtts_model* m) { return m ? (int)m->free_ids.size() : 0; }

static int kv_copy(qtts_model* m, int layer, int n_tok, const int32_t* pages, const uint16_t* k, const uint16_t* v,
                   uint16_t* k_out, uint16_t* v_out, bool write) {
  const qtts_config& c = m->cfg;
  if (layer < 0 || layer >= c.n_layers || n_tok < 0 || (n_tok && !pages)) return fail(m, QTTS_E_INVALID, "bad argument");
  if (n_tok == 0) return QTTS_OK;
  const int np = (n_tok + kPage - 1) / kPage;
  for (int i = 0; i < np; ++i)
    if (pages[i] < 0 || pages[i] >= c.kv_pool_pages) return fail(m, QTTS_E_POOL, "page id %d outside the pool", pages[i]);
  cudaSetDevice(m->device);
  const size_t elems = (size_t)n_tok * c.n_kv_heads * c.head_dim;
  uint16_t* buf = nullptr;
  int32_t* dp = nullptr;
  CK(m, cudaMalloc(&buf, elems * 4));
  cudaError_t e = cudaMalloc(&dp, np * 4);
  if (e == cudaSuccess) e = cudaMemcpy(dp, pages, np * 4, cudaMemcpyHostToDevice);
  if (e == cudaSuccess && write) e = cudaMemcpy(buf, k, elems * 2, cudaMemcpyDefault);
  if (e == cudaSuccess && write) e = cudaMemcpy(buf + elems, v, elems * 2, cudaMemcpyDefault);
  if (e == cudaSuccess)
    e = launch_kv_scatter(m->kv_pool, c.kv_pool_pages, c.n_kv_heads, c.head_dim, layer, n_tok, dp, buf, buf + elems,
                          write ? 1 : 0, 0);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e == cudaSuccess && !write) e = cudaMemcpy(k_out, buf, elems * 2, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && !write) e = cudaMemcpy(v_out, buf + elems, elems * 2, cudaMemcpyDeviceToHost);
  cudaFree(buf);
  if (dp) cudaFree(dp);
  if (e != cudaSuccess) return cuda_fail(m, e, "kv copy");
  return QTTS_OK;
}

int qtts_kv_write(qtts_model* m, int layer, int n_tok, const int32_t* pages, const uint16_t* k, const uint16_t* v) {
  if (!m) return fail(m, QTTS_E_INVALID, "null model");
  if (n_tok && (!k || !v)) return fail(m, QTTS_E_INVALID, "null argument");
  return kv_copy(m, layer, n_tok, pages, k, v, nullptr, nullptr, true);
}

int qtts_kv_read(qtts_model* m, int layer, int n_tok, const int32_t* pages, uint16_t* k, uint16_t* v) {
  if (!m) return fail(m, QTTS_E_INVALID, "null model");
  if (n_tok && (!k || !v)) return fail(m, QTTS_E_INVALID, "null argument");
  return kv_copy(m, layer, n_tok, pages, nullptr, nullptr, k, v, false);
}

int qtts_frame_step(qtts_model* m, int B, qtts_session* sess, const int32_t* bt, int bt_stride,
                    const uint16_t* in_embeds, qtts_rng* rng, uint32_t* seen, const int32_t* forced,
                    int32_t* codes_out, uint8_t* eos_out, float* logits_out, void* stream) {
  return frame_part(m, PART_ALL, B, sess, bt, bt_stride, in_embeds, rng, seen, forced, codes_out, eos_out, logits_out,
                    stream);
}

int qtts_frame_talker(qtts_model* m, int B, qtts_session* sess, const int32_t* bt, int bt_stride,
                      const uint16_t* in_embeds, qtts_rng* rng, uint32_t* seen, const int32_t* forced,
                      int32_t* codes_out, uint8_t* eos_out, float* logits_out, void* stream) {
  return frame_part(m, PART_TALKER, B, sess, bt, bt_stride, in_embeds, rng, seen, forced, codes_out, eos_out,
                    logits_out, stream);
}

int qtts_frame_cp(qtts_model* m, int B, qtts_session* sess, const int32_t* bt, int bt_stride,
                  const uint16_t* in_embeds, qtts_rng* rng, uint32_t* seen, const int32_t* forced,
                  int32_t* codes_out, uint8_t* eos_out, float* logits_out, void* stream) {
  return frame_part(m, PART_CP, B, sess, bt, bt_stride, in_embeds, rng, seen, forced, codes_out, eos_out, logits_out,
                    stream);
}

int qtts_talker_prefill(qtts_model* m, int B, qtts_session* sess, const int32_t* bt, int bt_stride,
                        const uint16_t* embeds, int n_tok, void* stream) {
  if (!m) return fail(m, QTTS_E_INVALID, "null model");
  if (!m->loaded) return fail(m, QTTS_E_STATE, "load weights first");
  if (B < 1 || B > m->cfg.max_batch) return fail(m, QTTS_E_BATCH, "B=%d outside 1..%d", B, m->cfg.max_batch);
  if (!sess || !bt || bt_stride < 1 || (n_tok > 0 && !embeds) || n_tok < 0)
    return fail(m, QTTS_E_INVALID, "null array, bad block-table stride or negative token count");
  if (m->cp_pending) return fail(m, QTTS_E_STATE, "a split frame waits for qtts_frame_cp");
  cudaSetDevice(m->device);
  cudaStream_t s = (cudaStream_t)stream;
  const int H = m->cfg.hidden;
  PfCtx ctx = m->pf;
  ctx.wait_ns = m->g.wait_ns;
  // chunks of P tokens of every session: B x P <= kPfMaxRows rows
  const int P_max = std::max(1, kPfMaxRows / B);
  for (int t0 = 0; t0 < n_tok;) {
    const int P = std::min(P_max, n_tok - t0);
    CK(m, pf_chunk(ctx, B, P, sess, bt, bt_stride, embeds + (size_t)t0 * B * H, s));
    CK(m, launch_advance_kv(sess, B, m->g.err, P, s));
    t0 += P;
  }
  m->last_stream = s;
  return QTTS_OK;
}

int qtts_frame_steps(qtts_model* m, int n_frames, int B, qtts_session* sess, const int32_t* bt, int bt_stride,
                     const uint16_t* in_embeds, const uint16_t* text_embeds, qtts_rng* rng, uint32_t* seen,
                     const int32_t* forced, int32_t* codes_out, uint8_t* eos_out, float* logits_out,
                     void* stream) {
  if (!m) return fail(m, QTTS_E_INVALID, "null model");
  if (!m->loaded) return fail(m, QTTS_E_STATE, "load weights first");
  if (n_frames < 1) return fail(m, QTTS_E_INVALID, "n_frames must be >= 1");
  if (!text_embeds || !codes_out || !eos_out) return fail(m, QTTS_E_INVALID, "null array");
  if (B < 1 || B > m->cfg.max_batch) return fail(m, QTTS_E_BATCH, "B=%d outside 1..%d", B, m->cfg.max_batch);
  cudaSetDevice(m->device);
  const int H = m->cfg.hidden;
  if (!m->fb[0]) {
    AL(m, m->fb[0], (size_t)kMaxBatch * H);
    AL(m, m->fb[1], (size_t)kMaxBatch * H);
  }
  EmbedTables t{};
  for (int j = 0; j < kCodebooks; ++j) {
    t.e[j] = m->embed[j];
    t.rows[j] = j == 0 ? m->cfg.vocab0 : m->cfg.cp_vocab;
  }
  cudaStream_t s = (cudaStream_t)stream;
  const uint16_t* in = in_embeds;
  for (int f = 0; f < n_frames; ++f) {
    int32_t* codes = codes_out + (size_t)f * B * kCodebooks;
    const int32_t* frc = forced ? forced + (size_t)f * B * kCodebooks : nullptr;
    float* lg = logits_out ? logits_out + (size_t)f * B * kCodebooks * m->cfg.vocab0 : nullptr;
    int rc = frame_part(m, PART_ALL, B, sess, bt, bt_stride, in, rng, seen, frc, codes, eos_out + (size_t)f * B, lg,
                        stream);
    if (rc) return rc;
    if (f + 1 == n_frames) break;
    // the next frame's input: text + the codes the model consumed (forced ones under teacher forcing)
    CK(m, launch_feedback(B, H, frc ? frc : codes, text_embeds + (size_t)f * B * H, t, m->fb[f & 1], s));
    in = m->fb[f & 1];
  }
  return QTTS_OK;
}

int qtts_frame_step_host(qtts_model* m, int B, qtts_session* sess, const int32_t* bt, int bt_stride,
                         const uint16_t* in_embeds, qtts_rng* rng, uint32_t* seen, const int32_t* forced,
                         int32_t* codes_out, uint8_t* eos_out, float* logits_out, void* stream) {
  if (!m) return fail(m, QTTS_E_INVALID, "null model");
  if (!m->loaded) return fail(m, QTTS_E_STATE, "load weights first");
  const qtts_config& c = m->cfg;
  if (B < 1 || B > c.max_batch) return fail(m, QTTS_E_BATCH, "B=%d outside 1..%d", B, c.max_batch);
  if (!sess || !bt || !in_embeds || !rng || !codes_out || !eos_out || bt_stride < 1)
    return fail(m, QTTS_E_INVALID, "null array or bad block-table stride");
  if (bt_stride > m->st_bt_cap) return fail(m, QTTS_E_INVALID, "bt_stride %d exceeds %d", bt_stride, m->st_bt_cap);
  for (int b = 0; b < B; ++b) {
    const qtts_session& S = sess[b];
    if (S.kv_len < 0 || S.kv_len + 1 > c.max_context || S.kv_len + 1 > bt_stride * kPage)
      return fail(m, QTTS_E_INVALID, "session %d: kv_len %d out of range", b, S.kv_len);
    for (int p = 0; p <= S.kv_len / kPage; ++p) {
      const int pg = bt[(size_t)b * bt_stride + p];
      if (pg < 0 || pg >= c.kv_pool_pages) return fail(m, QTTS_E_POOL, "session %d: page id %d outside the pool", b, pg);
    }
    if (!(S.temperature >= 0.f) || !std::isfinite(S.temperature) || !(S.cp_temperature >= 0.f) ||
        !std::isfinite(S.cp_temperature) || !(S.rep_penalty > 0.f) || !std::isfinite(S.rep_penalty))
      return fail(m, QTTS_E_INVALID, "session %d: bad sampling parameters", b);
    if (forced)
      for (int j = 0; j < kCodebooks; ++j) {
        const int cj = forced[b * kCodebooks + j];
        if (cj < 0 || cj >= (j == 0 ? c.vocab0 : c.cp_vocab))
          return fail(m, QTTS_E_INVALID, "session %d: forced code %d of codebook %d out of range", b, cj, j);
      }
  }
  cudaSetDevice(m->device);
  cudaStream_t s = (cudaStream_t)stream;
  const int sw = seen_words(c);
  CK(m, cudaMemcpyAsync(m->st_sess, sess, B * sizeof(qtts_session), cudaMemcpyHostToDevice, s));
  CK(m, cudaMemcpyAsync(m->st_bt, bt, (size_t)B * bt_stride * 4, cudaMemcpyHostToDevice, s));
  CK(m, cudaMemcpyAsync(m->st_in, in_embeds, (size_t)B * c.hidden * 2, cudaMemcpyHostToDevice, s));
  CK(m, cudaMemcpyAsync(m->st_rng, rng, B * sizeof(qtts_rng), cudaMemcpyHostToDevice, s));
  if (seen) CK(m, cudaMemcpyAsync(m->st_seen, seen, (size_t)B * sw * 4, cudaMemcpyHostToDevice, s));
  if (forced) CK(m, cudaMemcpyAsync(m->st_forced, forced, (size_t)B * kCodebooks * 4, cudaMemcpyHostToDevice, s));
  const int rc = qtts_frame_step(m, B, m->st_sess, m->st_bt, bt_stride, m->st_in, m->st_rng,
                                 seen ? m->st_seen : nullptr, forced ? m->st_forced : nullptr, m->st_codes,
                                 m->st_eos, logits_out ? m->st_logits : nullptr, stream);
  if (rc) return rc;
  CK(m, cudaMemcpyAsync(codes_out, m->st_codes, (size_t)B * kCodebooks * 4, cudaMemcpyDeviceToHost, s));
  CK(m, cudaMemcpyAsync(eos_out, m->st_eos, B, cudaMemcpyDeviceToHost, s));
  if (logits_out)
    CK(m, cudaMemcpyAsync(logits_out, m->st_logits, (size_t)B * kCodebooks * c.vocab0 * 4, cudaMemcpyDeviceToHost, s));
  CK(m, cudaMemcpyAsync(sess, m->st_sess, B * sizeof(qtts_session), cudaMemcpyDeviceToHost, s));
  CK(m, cudaMemcpyAsync(rng, m->st_rng, B * sizeof(qtts_rng), cudaMemcpyDeviceToHost, s));
  if (seen) CK(m, cudaMemcpyAsync(seen, m->st_seen, (size_t)B * sw * 4, cudaMemcpyDeviceToHost, s));
  CK(m, cudaStreamSynchronize(s));
  int derr = 0;
  CK(m, cudaMemcpy(&derr, m->g.err, 4, cudaMemcpyDeviceToHost));
  if (derr) {
    CK(m, reset_split_counters(m));
    return fail(m, derr == QTTS_DEV_TIMEOUT ? QTTS_E_TIMEOUT : QTTS_E_DEVICE, "device error %d", derr);
  }
  return QTTS_OK;
}

int qtts_frame_status(qtts_model* m, int* device_err) {
  if (!m) return fail(m, QTTS_E_INVALID, "null model");
  cudaSetDevice(m->device);
  CK(m, cudaStreamSynchronize(m->last_stream));
  int derr = 0;
  CK(m, cudaMemcpy(&derr, m->g.err, 4, cudaMemcpyDeviceToHost));
  if (derr) {
    CK(m, cudaMemset(m->g.err, 0, 4));
    CK(m, reset_split_counters(m));
  }
  if (device_err) *device_err = derr;
  if (derr) return fail(m, derr == QTTS_DEV_TIMEOUT ? QTTS_E_TIMEOUT : QTTS_E_DEVICE, "device error %d", derr);
  return QTTS_OK;
}

int qtts_feedback_embed(qtts_model* m, int B, const int32_t* codes, const uint16_t* text, uint16_t* next_out,
                        void* stream) {
  if (!m || !codes || !text || !next_out) return fail(m, QTTS_E_INVALID, "null argument");
  if (!m->loaded) return fail(m, QTTS_E_STATE, "load weights first");
  if (B < 1 || B > m->cfg.max_batch) return fail(m, QTTS_E_BATCH, "B=%d outside 1..%d", B, m->cfg.max_batch);
  cudaSetDevice(m->device);
  EmbedTables t{};
  for (int j = 0; j < kCodebooks; ++j) {
    t.e[j] = m->embed[j];
    t.rows[j] = j == 0 ? m->cfg.vocab0 : m->cfg.cp_vocab;
  }
  CK(m, launch_feedback(B, m->cfg.hidden, codes, text, t, next_out, (cudaStream_t)stream));
  m->last_stream = (cudaStream_t)stream;
  return QTTS_OK;
}

int qtts_sample(qtts_model* m, int B, int codebook, const float* logits, int V, const qtts_session* sessions,
                const qtts_rng* rng, const uint32_t* seen, int32_t* codes_out, void* stream) {
  if (!m || !logits || !sessions || !rng || !codes_out) return fail(m, QTTS_E_INVALID, "null argument");
  if (B < 1 || B > m->cfg.max_batch) return fail(m, QTTS_E_BATCH, "B=%d outside 1..%d", B, m->cfg.max_batch);
  if (codebook < 0 || codebook >= kCodebooks || V < 1 || V > kMaxVocab)
    return fail(m, QTTS_E_INVALID, "bad codebook or vocabulary size");
  if (codebook == 0 && seen && V > 32 * seen_words(m->cfg))
    return fail(m, QTTS_E_INVALID, "V exceeds the seen bitmap");
  cudaSetDevice(m->device);
  FrameArgs fa{};
  fa.B = B;
  fa.sess = (qtts_session*)sessions;
  fa.rng = (qtts_rng*)rng;
  fa.seen = (uint32_t*)seen;
  fa.codes_out = codes_out;
  CK(m, launch_sample(logits, V, codebook, m->g, fa, (cudaStream_t)stream));
  m->last_stream = (cudaStream_t)stream;
  return QTTS_OK;
}

int qtts_set_option(qtts_model* m, int option, int value) {
  if (!m) return fail(m, QTTS_E_INVALID, "null model");
  if (option == QTTS_OPT_STEPWISE) {
    m->stepwise = value != 0;
    return QTTS_OK;
  }
  if (option == QTTS_OPT_RING_SLOTS) {
    if (value != 1 && value != 2 && value != 4 && value != 8)
      return fail(m, QTTS_E_INVALID, "ring slots must be 1, 2, 4 or 8");
    m->g.ring_slots = value;
    return QTTS_OK;
  }
  if (option == QTTS_OPT_TC_MIN_ROWS) {
    if (value < 1 || value > 65) return fail(m, QTTS_E_INVALID, "tensor-path row threshold must be 1..65");
    m->g.tc_min_rows = value;
    return QTTS_OK;
  }
  if (option == QTTS_OPT_KSPLIT_MIN_ROWS) {
    if (value < 1 || value > 65) return fail(m, QTTS_E_INVALID, "K-split row threshold must be 1..65");
    m->g.ksplit_min_rows = value;
    return QTTS_OK;
  }
  if (option == QTTS_OPT_CHUNK_TALKER_MIN_B) {
    if (value < 1 || value > kMaxBatch + 1)
      return fail(m, QTTS_E_INVALID, "chunk-kernel Talker threshold must be 1..%d", kMaxBatch + 1);
    m->chunk_talker_min_b = value;
    return QTTS_OK;
  }
  if (option == QTTS_OPT_WAIT_LIMIT_US) {
    if (value < 1 || value > 2000000) return fail(m, QTTS_E_INVALID, "wait limit must be 1..2000000 us");
    m->g.wait_ns = (unsigned long long)value * 1000ull;
    return QTTS_OK;
  }
  if (option == QTTS_OPT_TRACE) {
    if (!m->loaded) return fail(m, QTTS_E_STATE, "load weights first");
    if (value < 0 || value > 2) return fail(m, QTTS_E_INVALID, "trace must be 0, 1 or 2");
    if (value && !m->trace_buf) {
      cudaSetDevice(m->device);
      AL(m, m->trace_buf, trace_words(m, m->G));
    }
    m->g.trace = value ? m->trace_buf : nullptr;
    m->g.trace_ctas = value == 2 ? m->G : 2;
    return QTTS_OK;
  }
  return fail(m, QTTS_E_INVALID, "unknown option %d", option);
}

int qtts_frame_trace(qtts_model* m, uint64_t* host, int capacity) {
  if (!m || !host || capacity < 0) return fail(m, QTTS_E_INVALID, "bad argument");
  if (!m->trace_buf) return fail(m, QTTS_E_STATE, "tracing was never enabled");
  cudaSetDevice(m->device);
  CK(m, cudaStreamSynchronize(m->last_stream));
  const int n = (int)std::min((size_t)capacity, trace_words(m, m->g.trace_ctas));
  CK(m, cudaMemcpy(host, m->trace_buf, (size_t)n * sizeof(uint64_t), cudaMemcpyDeviceToHost));
  return n;
}

int qtts_frame_weight_bytes(const qtts_model* m, int64_t* bytes) {
  if (!m || !bytes) return QTTS_E_INVALID;
  const bool i8 = m->use_int8;
  auto lb = [&](const LinW& L) -> int64_t { return i8 ? (int64_t)L.N * L.K + 4LL * L.N : 2LL * L.N * L.K; };
  int64_t t = 0;
  for (auto& L : m->tl) t += lb(L.qkv) + lb(L.o) + lb(L.gu) + lb(L.down);
  t += lb(m->head0) + lb(m->proj);
  int64_t cp = 0;
  for (auto& L : m->cl) cp += lb(L.qkv) + lb(L.o) + lb(L.gu) + lb(L.down);
  t += (int64_t)(kCodebooks - 1) * cp;
  for (int j = 1; j < kCodebooks; ++j) t += lb(m->cp_head[j]);
  *bytes = t;
  return QTTS_OK;
}

}  // extern "C"

// Accessors for translation units that do not see qtts_model's definition.
namespace qtts {

int model_kv_layout(qtts_model* m, KvLayout* out) {
  if (!m || !out) return QTTS_E_INVALID;
  out->device = m->device;
  out->pool = m->kv_pool;
  out->pool_pages = m->cfg.kv_pool_pages;
  out->n_layers = m->cfg.n_layers;
  out->nkv = m->cfg.n_kv_heads;
  out->d = m->cfg.head_dim;
  return QTTS_OK;
}

int model_fail(qtts_model* m, int code, const char* msg) { return fail(m, code, "%s", msg); }

}  // namespace qtts
