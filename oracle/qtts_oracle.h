/*
 * qtts_oracle.h -- plain, slow CPU oracle for one lockstep multi-codebook
 * codec frame of a Qwen3-TTS-style model (Talker step, 2048->1024 projection,
 * 15 Code-Predictor steps, each with its own head and sampler).
 *
 * TEST INFRASTRUCTURE. Only tests/, __graft_entry__.smoke() and bench.py's
 * cpu_baseline / reference leg may load this library. The CUDA product path
 * shares no code, header, table or constant with it.
 *
 * Sources (page title, section):
 *   "De grens van snelheid en kosten verleggen voor Qwen3-TTS" (Nari Labs),
 *     section "Hoe we Qwen3-TTS hebben geoptimaliseerd": Talker predicts
 *     codebook 0 per frame, the Code Predictor the remaining 15 codebooks;
 *     section 3: the Code Predictor always runs 15 steps per frame.
 *   "Qwen3-TTS PR 5: 1.7B CustomVoice, VoiceDesign and Base", section "Graph":
 *     Talker decode with paged KV, RoPE positions and two samplers (group 0
 *     with repetition penalty, code predictor); section "What changed vs the
 *     0.6B port": small_to_mtp_projection Talker 2048 -> predictor 1024.
 *   "Qwen3-TTS Native v0.3.0", section "What changed": lockstep batched decode,
 *     request-local KV / sampling state / histories / random states; INT8
 *     weight-only decode, per-output-channel symmetric, quantised at load from
 *     BF16.
 *
 * Precision: transformer arithmetic in double; weights are bf16 (exact in
 * double); K/V are rounded to bf16 when stored (the cache format). The INT8
 * quantiser and the sampler run in IEEE binary32, the precision the GPU path
 * takes the same integer decisions in; build with -ffp-contract=off.
 *
 * Pins: every function below is checked, without a GPU, against values fixed
 * by the pages or by the mathematics rather than by itself: Philox
 * known-answer vectors, exact points and accuracy of the log, RMSNorm / RoPE /
 * SiLU closed forms, linear and attention against library routines and
 * brute force, the quantiser on crafted ties, sampler special cases and
 * Gumbel-max frequencies, whole-frame and prefill closed forms on special
 * weights, batching invariance and causality (tests/test_oracle_*.py).
 * Parity against a trained Qwen3-TTS is unpinned: no trained weights exist
 * here, and the random-init weights exercise only the arithmetic.
 */
#ifndef QTTS_ORACLE_H
#define QTTS_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int32_t hidden, n_layers, n_q_heads, n_kv_heads, head_dim, ffn, vocab0;
  int32_t cp_hidden, cp_layers, cp_n_q_heads, cp_n_kv_heads, cp_head_dim, cp_ffn, cp_vocab;
  int32_t n_codebooks;  /* 16: codebook 0 from the Talker + 15 Code-Predictor codebooks */
  int32_t eos_id;       /* codec end-of-speech id in codebook 0 */
  int32_t n_codes;      /* ids >= n_codes other than eos_id are never sampled in codebook 0 */
  int32_t proj_bias;    /* 1: the projection has a bias vector */
  double rms_eps, rope_theta, cp_rope_theta;
} orc_dims;

/* One linear layer y = W x, W [N,K] row-major. q/s: INT8 codes + fp32 per-row
 * scale (used when the model's use_int8 flag is set). */
typedef struct { const uint16_t* w; const int8_t* q; const float* s; } orc_lin;

typedef struct {
  const uint16_t* in_norm;           /* [H] RMSNorm gain before attention */
  orc_lin wq, wk, wv, wo;            /* [nq*d,H] [nkv*d,H] [nkv*d,H] [H,nq*d] */
  const uint16_t* post_norm;         /* [H] RMSNorm gain before the MLP */
  orc_lin wg, wu, wd;                /* [F,H] [F,H] [H,F] */
} orc_layer;

typedef struct {
  orc_dims d;
  int32_t use_int8;
  const orc_layer* talker;           /* [n_layers] */
  const uint16_t* final_norm;        /* [H] */
  orc_lin head0;                     /* [vocab0,H] codebook-0 head */
  orc_lin proj;                      /* [Hc,H] small_to_mtp_projection */
  const uint16_t* proj_b;            /* [Hc] or NULL */
  const orc_layer* cp;               /* [cp_layers] */
  const uint16_t* cp_final_norm;     /* [Hc] */
  orc_lin cp_head[16];               /* entries 1..15: [cp_vocab,Hc] */
  const uint16_t* embed[16];         /* E_0 [vocab0,H], E_j [cp_vocab,H] */
} orc_model;

typedef struct {
  int32_t kv_len;          /* tokens already cached; the new token goes at this position */
  int32_t eos_allowed;     /* 0: eos_id is masked in codebook 0 */
  float temperature;       /* codebook 0; 0 => greedy */
  int32_t top_k;           /* codebook 0; 1 => greedy; <=0 or >=V => no truncation */
  float rep_penalty;       /* codebook 0 repetition penalty over the seen set */
  float cp_temperature;    /* codebooks 1..15 */
  int32_t cp_top_k;
  int32_t reserved;
} orc_session;

/* ---- per-operation entry points (pinned one by one in tests) ---- */
uint16_t orc_to_bf16(double x);
double orc_from_bf16(uint16_t h);
void orc_rmsnorm(const double* x, const uint16_t* g, int n, double eps, double* out);
void orc_rope(double* v, int n_heads, int head_dim, int pos, double theta);
void orc_linear(const double* x, orc_lin W, int use_int8, int N, int K, double* y);
void orc_attention(const double* q, const uint16_t* k_cache, const uint16_t* v_cache,
                   int n_pos, int n_q_heads, int n_kv_heads, int head_dim, double* out);
double orc_silu(double a);
void orc_quantize_rows(const uint16_t* w, int N, int K, int8_t* q, float* scale);
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);
float orc_logf(float x);
float orc_uniform(uint32_t key0, uint32_t key1, int codebook, uint32_t frame_ctr, int v);
int32_t orc_sample(const float* logits, int V, int codebook, const orc_session* s,
                   uint32_t key0, uint32_t key1, uint32_t frame_ctr, const uint32_t* seen,
                   int eos_id, int n_codes);

/* ---- one whole frame for B sessions ----
 * kv[b]: session b's Talker cache, bf16 [n_layers][2][kv_cap][n_kv][d] (K then V).
 * rng: [B][4] = {key0, key1, frame_ctr, unused}; frame_ctr advanced.
 * seen: [B][ceil(vocab0/32)] bitmap; updated with the committed codebook-0 code.
 * forced: [B][16] teacher-forced codes or NULL. codes_out: [B][16] sampled codes.
 * logits_out: [B][16][vocab0] raw logits or NULL (rows 1..15 fill cp_vocab columns). */
int orc_frame_step(const orc_model* m, int B, orc_session* sess, uint16_t* const* kv, int kv_cap,
                   const uint16_t* in_embeds, uint32_t* rng, uint32_t* seen, const int32_t* forced,
                   int32_t* codes_out, uint8_t* eos_out, double* logits_out);

/* next_in[b] = text[b] + sum_j E_j[codes[b][j]]  (free-running feedback) */
void orc_feedback(const orc_model* m, int B, const int32_t* codes, const uint16_t* text, double* out);

/* ---- Talker prefill: a prompt's tokens through the Talker layers ----
 * For each session b and prompt token t = 0..n_tok-1 (in order): the Talker
 * layers at position kv_len_b + t on input embeds[t][b] (bf16 [n_tok][B]
 * [hidden]), writing that position's K/V into kv[b] as the decode step does;
 * no head, no sampling. kv_len advanced by n_tok. -1 if a session lacks room. */
int orc_talker_prefill(const orc_model* m, int B, orc_session* sess, uint16_t* const* kv, int kv_cap,
                       const uint16_t* embeds, int n_tok);

#ifdef __cplusplus
}
#endif
#endif
