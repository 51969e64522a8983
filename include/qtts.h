/*
 * qtts.h -- C ABI of the GB300 (sm_103a) lockstep multi-codebook frame decode.
 *
 * One call, qtts_frame_step, runs one codec frame for B active sessions:
 * a Talker decode step (RMSNorm, QKV, RoPE, GQA attention over the session's
 * paged KV cache, O-proj, SwiGLU MLP, codebook-0 head and sampler), the
 * 2048->1024 small_to_mtp_projection, then 15 sequential Code-Predictor steps,
 * each with its own codebook head and sampler. Every shared weight matrix is
 * streamed from HBM once per frame for the whole batch; per-session state
 * (KV cache, sampling parameters, seen-token history, random state) stays
 * with the session.
 *
 * Sources (page title, section):
 *   [R] "Qwen3-TTS Native v0.3.0", "What changed": lockstep batched decode
 *       (one batched call runs the talker and the 15-step code predictor for
 *       every active session, shared weights read once per frame, KV caches /
 *       sampling state / histories / random states request-local); CUDA-graph
 *       frames; opt-in INT8 weight-only decode, per-output-channel symmetric,
 *       quantised at load from BF16, prefill stays BF16.
 *   [M] "Qwen3-TTS PR 5: 1.7B CustomVoice, VoiceDesign and Base", "Graph":
 *       talker decode loop with paged KV, RoPE positions and two samplers
 *       (group 0 with repetition penalty, code predictor), stop on codec EOS;
 *       "What changed vs the 0.6B port": small_to_mtp_projection 2048 -> 1024,
 *       weight loading checks coverage in both directions; "Known gaps": the
 *       per-request seen-token set of the repetition penalty.
 *   [N] "De grens van snelheid en kosten verleggen voor Qwen3-TTS", section
 *       "Hoe we Qwen3-TTS hebben geoptimaliseerd": the Talker predicts codebook
 *       0, the Code Predictor the remaining 15; section 3: a fixed 15 steps
 *       per frame over a pre-allocated short KV cache; section 5: graphs for a
 *       set of batch sizes, larger groups split over several turns.
 *
 * Conventions for every function:
 *   - Returns QTTS_OK (0) or a negative QTTS_E_* code; never throws, never
 *     aborts the process. qtts_last_error() gives a one-line message.
 *   - "device" pointers are CUDA device memory on the model's GPU; "host"
 *     pointers are ordinary (pageable or pinned) host memory.
 *   - bf16 values travel as uint16_t bit patterns.
 *   - Pointers passed in stay owned by the caller; the library copies what it
 *     keeps (weights) and owns everything it allocates (weights, KV pool,
 *     scratch), freed by qtts_destroy.
 */
#ifndef QTTS_H
#define QTTS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define QTTS_ABI_VERSION 1

#define QTTS_OK 0
#define QTTS_E_INVALID (-1)  /* bad argument: null pointer, size out of range, bad sampling value */
#define QTTS_E_CUDA (-2)     /* a CUDA runtime call failed */
#define QTTS_E_OOM (-3)      /* device allocation failed */
#define QTTS_E_MISSING (-4)  /* qtts_load_weights: a required tensor was not supplied */
#define QTTS_E_UNUSED (-5)   /* qtts_load_weights: a supplied name is not a model tensor, or is repeated */
#define QTTS_E_SHAPE (-6)    /* qtts_load_weights: a tensor has the wrong shape or dtype */
#define QTTS_E_BATCH (-7)    /* B outside 1..max_batch (the caller splits larger groups, [N] section 5) */
#define QTTS_E_STATE (-8)    /* call out of order, e.g. a frame before the weights are loaded */
#define QTTS_E_POOL (-9)     /* KV page pool exhausted, or a page id outside the pool */
#define QTTS_E_DEVICE (-10)  /* a device-side check failed (see qtts_frame_status) */
#define QTTS_E_TIMEOUT (-11) /* a device-side wait ran out its time limit */

/* device-side error word values reported by qtts_frame_status */
#define QTTS_DEV_OK 0
#define QTTS_DEV_BAD_SESSION 1  /* kv_len out of range, or not enough block-table entries */
#define QTTS_DEV_BAD_PAGE 2     /* a block-table entry outside the KV pool */
#define QTTS_DEV_BAD_SAMPLING 3 /* temperature < 0 or not finite, rep_penalty <= 0 or not finite */
#define QTTS_DEV_BAD_CODE 4     /* a teacher-forced code outside its codebook */
#define QTTS_DEV_TIMEOUT 5      /* a device-side wait (activation words, weight ring, tensor-path barriers) ran out its limit */

#define QTTS_DTYPE_BF16 0

typedef struct qtts_model qtts_model;

/* Model dimensions and run limits. Field meanings follow the names; the
 * Code-Predictor query width cp_n_q_heads * cp_head_dim may differ from
 * cp_hidden (1.7B: 16 * 128 = 2048 vs 1024). */
typedef struct {
  int32_t hidden, n_layers, n_q_heads, n_kv_heads, head_dim, ffn, vocab0;
  int32_t cp_hidden, cp_layers, cp_n_q_heads, cp_n_kv_heads, cp_head_dim, cp_ffn, cp_vocab;
  int32_t n_codebooks;   /* must be 16: codebook 0 + 15 Code-Predictor codebooks [N] */
  int32_t eos_id;        /* codec EOS id in codebook 0 [M] "Graph" */
  int32_t n_codes;       /* ids >= n_codes other than eos_id are never sampled in codebook 0 */
  int32_t proj_bias;     /* 1: tensor "cp.proj_bias" [cp_hidden] is part of the model */
  float rms_eps, rope_theta, cp_rope_theta;
  int32_t page_size;     /* KV page size in tokens; must be 16 */
  int32_t max_batch;     /* largest B per call, 1..32 */
  int32_t max_context;   /* largest kv_len + 1 a session may reach (sizes the RoPE table), <= 2048 */
  int32_t kv_pool_pages; /* pages in the library-owned Talker KV pool */
} qtts_config;

/* One named weight tensor, row-major. Names and shapes (H = hidden,
 * Hc = cp_hidden, d = head_dim, F = ffn; Code-Predictor layers use the cp_*
 * sizes):
 *   talker.layers.{l}.input_norm [H]      .q_proj [nq*d, H]   .k_proj [nkv*d, H]
 *   talker.layers.{l}.v_proj [nkv*d, H]   .o_proj [H, nq*d]   .post_attn_norm [H]
 *   talker.layers.{l}.gate_proj [F, H]    .up_proj [F, H]     .down_proj [H, F]
 *   talker.final_norm [H]                 talker.codec_head [vocab0, H]
 *   codec_embed.0 [vocab0, H]             codec_embed.{1..15} [cp_vocab, H]
 *   cp.proj [Hc, H]  (+ cp.proj_bias [Hc] when proj_bias)
 *   cp.layers.{l}.* as above              cp.final_norm [Hc]
 *   cp.heads.{1..15} [cp_vocab, Hc]
 */
typedef struct {
  const char* name;
  int32_t dtype;        /* QTTS_DTYPE_BF16 */
  int32_t ndim;         /* 1 or 2 */
  int64_t shape[2];
  const void* data;     /* host or device pointer (unified addressing); read during the call only */
} qtts_tensor;

/* Per-session descriptor, 32 bytes. Sampling follows [M] "Graph": codebook 0
 * gets the repetition penalty over the seen set, codebooks 1..15 do not.
 * temperature == 0 or top_k == 1 means greedy; top_k <= 0 or >= vocab means
 * no top-k truncation. */
typedef struct {
  int32_t kv_len;        /* tokens already cached; the new token is written at this position.
                            Advanced by one per frame. */
  int32_t eos_allowed;   /* 0: eos_id is masked in codebook 0 */
  float temperature;     /* codebook 0 */
  int32_t top_k;         /* codebook 0 */
  float rep_penalty;     /* codebook 0: positive logits divided by it, others multiplied */
  float cp_temperature;  /* codebooks 1..15 */
  int32_t cp_top_k;      /* codebooks 1..15 */
  int32_t reserved;
} qtts_session;

/* Per-session random state: Philox4x32-10 key and the frame counter. The
 * uniform for id v of codebook j is word v&3 of Philox(key, (v>>2, j,
 * frame_ctr, 0)); frame_ctr is advanced by one per frame. */
typedef struct {
  uint32_t key0, key1, frame_ctr, reserved;
} qtts_rng;

int qtts_abi_version(void);
const char* qtts_last_error(const qtts_model* m); /* m may be NULL for create errors */

/* Create a model on CUDA device `device`. Validates the dimensions, allocates
 * the KV pool, scratch and the RoPE table. */
int qtts_create(const qtts_config* cfg, int device, qtts_model** out);
void qtts_destroy(qtts_model* m);

/* Copy all weights in, in one call. The set of names must equal the model's
 * tensor list exactly ([M] "What changed vs the 0.6B port": coverage checked
 * in both directions): QTTS_E_MISSING if one is absent, QTTS_E_UNUSED for an
 * unknown or repeated name, QTTS_E_SHAPE for a wrong shape/dtype. All checks
 * run before anything is copied. Synchronous. */
int qtts_load_weights(qtts_model* m, const qtts_tensor* tensors, int n);

/* INT8 weight-only decode ([R] "What changed"): quantise every decode GEMM
 * weight per output channel, symmetric, from the loaded BF16 weights:
 * scale = max|w| / 127 (binary32), q = round-half-even(w / scale) clamped to
 * [-127, 127], zero rows get scale 0. Embeddings, norms and the KV cache stay
 * BF16. Switches frames to the INT8 path. Synchronous. */
int qtts_quantize_int8(qtts_model* m);
/* 1: frames use INT8 weights (requires qtts_quantize_int8), 0: BF16. */
int qtts_set_int8(qtts_model* m, int enable);
/* Copy the INT8 codes [N][K] and scales [N] of one named GEMM weight to host
 * memory, in the tensor's own row order. */
int qtts_export_int8(qtts_model* m, const char* name, int8_t* q_host, float* scale_host);

/* KV page pool ([M] "Graph": paged KV). A page holds page_size tokens of
 * every Talker layer's K and V. Allocation returns n page ids (not
 * necessarily contiguous) into ids_host; the caller owns the block tables. */
int qtts_kv_alloc_pages(qtts_model* m, int n, int32_t* ids_host);
int qtts_kv_free_pages(qtts_model* m, int n, const int32_t* ids_host);
int qtts_kv_pool_free_count(const qtts_model* m);
/* Write (read) n_tok tokens of K and V of Talker layer `layer`: token i goes
 * to page pages[i / page_size], slot i % page_size. k, v: [n_tok][n_kv][d]
 * bf16, host or device (read: host). pages: host array of ceil(n_tok /
 * page_size) ids. Synchronous. Places a given prompt prefix (one computed
 * from prompt embeddings is qtts_talker_prefill's) and lets tests inspect the
 * cache. */
int qtts_kv_write(qtts_model* m, int layer, int n_tok, const int32_t* pages_host, const uint16_t* k,
                  const uint16_t* v);
int qtts_kv_read(qtts_model* m, int layer, int n_tok, const int32_t* pages_host, uint16_t* k_host,
                 uint16_t* v_host);

/* qtts_kv_write for callers that must not allocate device memory. The pages
 * have no counterpart: this is a deployment variant, not part of the method.
 * qtts_kv_write stages K/V through buffers it cudaMallocs and cudaFrees on
 * every call, and cudaFree waits for the whole device; a serving loop that
 * writes a new session's prompt KV while other sessions' frames run, or code
 * living under a memory pool it does not own, cannot do that. This entry point
 * allocates nothing: it stages through one static device array of 4 MiB
 * (K then V; at most 1024 pages per call), which every GPU that loads the
 * library holds until the process exits. Larger writes are rejected with
 * QTTS_E_INVALID: split them. Same arguments and cache result as
 * qtts_kv_write, plus `stream`: the copies and the scatter are queued on it and
 * the call returns without waiting. k and v may be pageable host, pinned host
 * or device memory (pages_host is host memory): pageable host inputs are
 * copied before the call returns, while pinned host and device inputs are read
 * later, in stream order, so they must stay valid and unmodified until the
 * stream has run the copies. The first call on a device looks up the array's
 * device address (cudaGetSymbolAddress, in the device's primary context, which
 * is the context every later call uses). The caller's current device is left
 * as it was. All calls
 * share the one array, so calls whose work overlaps on the GPU (different
 * streams, no ordering between them) race. */
int qtts_kv_write_noalloc(qtts_model* m, int layer, int n_tok, const int32_t* pages_host, const uint16_t* k,
                          const uint16_t* v, void* stream);

/* One codec frame for B sessions, asynchronous on `stream` (a cudaStream_t;
 * NULL = default stream). All array pointers are device memory owned by the
 * caller, read/written in stream order:
 *   sessions      [B]                 kv_len advanced by one
 *   block_tables  [B][bt_stride]      page ids; entries 0..kv_len/page_size are read
 *   in_embeds     [B][hidden] bf16    Talker input for this frame
 *   rng           [B]                 frame_ctr advanced by one
 *   seen          [B][ceil(vocab0/32)] codebook-0 seen-token bitmap (or NULL),
 *                                      updated with the committed codebook-0 code
 *   forced_codes  [B][16] or NULL     teacher forcing: these codes, not the sampled
 *                                      ones, feed the Code Predictor and the history
 *   codes_out     [B][16]             sampled codes (codebook 0 first)
 *   eos_out       [B]                 1 if the sampled codebook-0 code is eos_id
 *   logits_out    [B][16][vocab0] or NULL   raw fp32 logits (before mask, penalty,
 *                                      temperature); rows 1..15 fill the first
 *                                      cp_vocab columns only
 * Host-side errors (B, null pointers, state) return at once. Device-side
 * checks (session, page and code ranges, sampling values, wait time-outs)
 * skip the frame's work and are reported by qtts_frame_status; a device error
 * stays set (later frames do nothing) until qtts_frame_status clears it. */
int qtts_frame_step(qtts_model* m, int B, qtts_session* sessions, const int32_t* block_tables, int bt_stride,
                    const uint16_t* in_embeds, qtts_rng* rng, uint32_t* seen, const int32_t* forced_codes,
                    int32_t* codes_out, uint8_t* eos_out, float* logits_out, void* stream);

/* The same frame with every array in HOST memory: the library validates every
 * session on the host, copies the inputs into its own device staging buffers,
 * runs the frame, copies the outputs and the advanced state (sessions, rng,
 * seen) back and waits for the stream. */
int qtts_frame_step_host(qtts_model* m, int B, qtts_session* sessions, const int32_t* block_tables,
                         int bt_stride, const uint16_t* in_embeds, qtts_rng* rng, uint32_t* seen,
                         const int32_t* forced_codes, int32_t* codes_out, uint8_t* eos_out, float* logits_out,
                         void* stream);

/* The frame in two halves, for a scheduler that interleaves Talker and
 * Code-Predictor work ("De grens van snelheid en kosten verleggen voor
 * Qwen3-TTS": the Talker step and the fixed 15-step Code Predictor as separate
 * scheduled phases). qtts_frame_talker runs the Talker step, the codebook-0
 * head, the projection of h_t and sampler 0 (codes_out[:,0], eos_out, the
 * codebook-0 logits row, kv_len and the seen bitmap advance); qtts_frame_cp
 * then runs the 15 Code-Predictor steps of that same frame (codes_out[:,1..15],
 * logits rows 1..15, rng frame_ctr advances) and must come next on the same
 * stream with the same sessions, rng, forced codes and outputs (in_embeds and
 * seen are not read; pass them or NULL). Together they give exactly
 * qtts_frame_step's results. qtts_frame_cp without a preceding
 * qtts_frame_talker returns QTTS_E_STATE. Arguments as in qtts_frame_step. */
int qtts_frame_talker(qtts_model* m, int B, qtts_session* sessions, const int32_t* block_tables, int bt_stride,
                      const uint16_t* in_embeds, qtts_rng* rng, uint32_t* seen, const int32_t* forced_codes,
                      int32_t* codes_out, uint8_t* eos_out, float* logits_out, void* stream);
int qtts_frame_cp(qtts_model* m, int B, qtts_session* sessions, const int32_t* block_tables, int bt_stride,
                  const uint16_t* in_embeds, qtts_rng* rng, uint32_t* seen, const int32_t* forced_codes,
                  int32_t* codes_out, uint8_t* eos_out, float* logits_out, void* stream);

/* n_frames consecutive frames with no host round trip in between
 * ("Qwen3-TTS PR 5", "Graph": the decode loop feeds talker_input_embeds back):
 * frame f takes in_embeds (f = 0) or text_embeds[f-1] + sum_j E_j[c_j] of
 * frame f-1's committed codes (the forced ones under teacher forcing), built
 * on the device (qtts_feedback_embed). Device arrays: text_embeds
 * [n_frames][B][hidden] bf16 (row n_frames-1 unused), forced_codes
 * [n_frames][B][16] or NULL, codes_out [n_frames][B][16], eos_out
 * [n_frames][B], logits_out [n_frames][B][16][vocab0] or NULL (each frame's
 * raw logits, laid out as in qtts_frame_step); sessions, block_tables, rng
 * and seen as in qtts_frame_step (advanced once per frame; block tables must
 * already cover kv_len + n_frames positions). Sessions that emit EOS keep
 * running: the caller compacts finished sessions between calls. Asynchronous
 * on `stream`. */
int qtts_frame_steps(qtts_model* m, int n_frames, int B, qtts_session* sessions, const int32_t* block_tables,
                     int bt_stride, const uint16_t* in_embeds, const uint16_t* text_embeds, qtts_rng* rng,
                     uint32_t* seen, const int32_t* forced_codes, int32_t* codes_out, uint8_t* eos_out,
                     float* logits_out, void* stream);

/* Talker prefill: a prompt of n_tok tokens per session through the Talker
 * layers: the causal prompt pass that runs before the first frame
 * ("Qwen3-TTS PR 5: 1.7B CustomVoice, VoiceDesign and Base", section Graph,
 * talker_prefill), packed into chunks like the page's token buckets (section
 * "What changed": 32..1024 tokens). Token t of session b sits at position
 * kv_len_b + t and its K/V are appended to the session's paged cache exactly
 * as a decode frame appends the new token's; no head, no sampling, no Code
 * Predictor. A chunk takes P = min(n_tok left, 1024 / B) tokens of every
 * session as B x P rows (row p B + b: token p of session b) and runs each
 * layer as whole-chunk kernels: RMSNorm, the QKV, O, gate/up and down
 * projections as tcgen05 tensor-core GEMMs over all rows (activations as
 * bf16 hi + lo pairs, fp32 accumulation), RoPE and the K/V append, causal
 * attention over the pages (earlier chunks and the chunk's own tokens); then
 * kv_len += P. The weights are the BF16 ones even with qtts_set_int8(m, 1):
 * prefill stays BF16 ("Qwen3-TTS Native v0.3.0", "What changed").
 * sessions, block_tables, bt_stride: as for qtts_frame_step (kv_len advanced
 * by n_tok in place; the block tables must cover kv_len + n_tok, which must
 * not exceed max_context). embeds: device [n_tok][B][hidden] bf16 (caller
 * owns). Asynchronous on `stream`; device-side errors (bad session or page,
 * found before a chunk writes anything) stop that chunk and every later one
 * and are read with qtts_frame_status. Not allowed between
 * qtts_frame_talker and qtts_frame_cp (QTTS_E_STATE). */
int qtts_talker_prefill(qtts_model* m, int B, qtts_session* sessions, const int32_t* block_tables, int bt_stride,
                        const uint16_t* embeds, int n_tok, void* stream);

/* Synchronise the model's last stream and read, then clear, the device error
 * word (QTTS_DEV_*). Returns QTTS_E_DEVICE / QTTS_E_TIMEOUT when it was set. */
int qtts_frame_status(qtts_model* m, int* device_err);

/* Free-running feedback for the next Talker input ([M] "Graph": the decode
 * loop feeds talker_input_embeds back):
 * next[b] = text[b] + sum_{j=0..15} E_j[codes[b][j]], bf16 out. Device
 * pointers, asynchronous on `stream`. */
int qtts_feedback_embed(qtts_model* m, int B, const int32_t* codes, const uint16_t* text, uint16_t* next_out,
                        void* stream);

/* The frame's sampler alone, on caller logits: one code per session for
 * codebook `codebook` (0: masks, EOS rule and repetition penalty over `seen`
 * apply; 1..15: none, [M] "Graph": two samplers). logits: device [B][V] fp32
 * with V <= 4096; sessions, rng: device [B] (read only, nothing advanced);
 * seen: device [B][ceil(vocab0/32)] or NULL; codes_out: device [B].
 * Asynchronous on `stream`. */
int qtts_sample(qtts_model* m, int B, int codebook, const float* logits, int V, const qtts_session* sessions,
                const qtts_rng* rng, const uint32_t* seen, int32_t* codes_out, void* stream);

/* Execution options (the same frame within the parity tolerance whatever their
 * values; STEPWISE and TRACE bit for bit):
 *   QTTS_OPT_STEPWISE  1: one launch per stage instead of one persistent
 *                      launch per frame (debugging aid). Default 0.
 *   QTTS_OPT_TRACE     1: record %globaltimer stamps inside every stage on
 *                      the first and last CTA (qtts_frame_trace); 2: on
 *                      every CTA. 0 (default): off.
 *   QTTS_OPT_RING_SLOTS 1, 2, 4 or 8: 16 KB weight slots per SM the producer
 *                      warp may fill ahead of the compute warps. Default 8.
 *   QTTS_OPT_TC_MIN_ROWS 1..65: a GEMV stage whose activation rows (sessions
 *                      x rows per session) number at least this and at most
 *                      64 runs on the tensor cores (BF16 weights, or INT8
 *                      widened to bf16 in shared memory; K a multiple of
 *                      128); 65 turns the tensor path off.
 *                      Default 8.
 *   QTTS_OPT_KSPLIT_MIN_ROWS 1..65: from this many activation rows up, a
 *                      tensor-path GEMV splits K across groups of CTAs
 *                      whose partial sums one CTA per group adds (fewer
 *                      activation words per CTA, one more exchange); below
 *                      it only GEMVs of at least 8 x 6144 activation values
 *                      (rows x K) split. Default 8.
 *   QTTS_OPT_WAIT_LIMIT_US 1..2000000: the limit, in microseconds, of every
 *                      device-side wait for another CTA's data or for
 *                      weights; a wait that runs it out sets
 *                      QTTS_DEV_TIMEOUT and the frame is abandoned (its
 *                      work partly done: re-run it from the caller's copy of
 *                      the state). Default 2000000 (2 s). A short limit is a
 *                      test of the time-out path, which otherwise a working
 *                      GPU never takes.
 *   QTTS_OPT_CHUNK_TALKER_MIN_B 1..33: a BF16 frame (or Talker half) of at
 *                      least this many sessions runs the Talker layers on
 *                      the prefill's tensor-core chunk kernels, one row per
 *                      session (whole-matrix GEMMs over all sessions, then
 *                      RoPE/KV append and attention kernels), and the frame
 *                      kernel from the codebook-0 head on; INT8 frames and
 *                      smaller batches keep the Talker in the frame kernel.
 *                      The prompt pass and such frames share the chunk
 *                      kernels' scratch: run them on one stream. 33 turns
 *                      it off. Default 33 (off: at B = 8 and 32 it runs no
 *                      faster than the frame kernel's Talker). */
#define QTTS_OPT_STEPWISE 1
#define QTTS_OPT_TRACE 3
#define QTTS_OPT_RING_SLOTS 4
#define QTTS_OPT_TC_MIN_ROWS 5
#define QTTS_OPT_KSPLIT_MIN_ROWS 6
#define QTTS_OPT_WAIT_LIMIT_US 7
#define QTTS_OPT_CHUNK_TALKER_MIN_B 8
int qtts_set_option(qtts_model* m, int option, int value);

/* Stage timestamps of the last frame run with QTTS_OPT_TRACE on: 8 values
 * per stage for CTA 0 (every stage in order), then the same for the last CTA
 * (trace 1) or for CTAs 1, 2, ... in order (trace 2) (nanoseconds,
 * %globaltimer; 0 = stage start, 1 after the GEMV prologue (tensor path:
 * its first activation pass), 2 after its weight pass, 3 after its
 * epilogues, 7 = stage end; 4-6 ring path: before warp 0's first ring wait,
 * after that unit's dot products, after its epilogue, and 3 then marks warp
 * 0's second unit's dot products; 4-6 tensor path: the second activation
 * pass starts loading, its first words settle, it is staged; unused marks
 * keep older values); then, for CTA 0, 4096 quadruples (issue, ready, MMAs
 * issued on the tensor path, unused) of the weight ring's slot uses in
 * order. Synchronises the model's last stream. Returns the number of values
 * written (<= capacity) or a negative error. */
int qtts_frame_trace(qtts_model* m, uint64_t* host, int capacity);

/* Bytes of weights one frame streams (the roofline's numerator, without KV):
 * every GEMM weight once per pass that uses it, in the current precision. */
int qtts_frame_weight_bytes(const qtts_model* m, int64_t* bytes);

#ifdef __cplusplus
}
#endif
#endif
