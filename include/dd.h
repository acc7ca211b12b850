/*
 * dd.h -- block-wise masked-diffusion decoding on one B300 (sm_103a).
 *
 * The library runs the denoising step of a TwoTower-style block diffusion
 * decoder: a block of S [MASK]-initialised positions per sequence attends
 * bidirectionally within the block and, by cross-attention, to a fixed
 * context KV cache (the frozen context tower's state); a dense SwiGLU MLP and
 * an LM head follow; every masked position whose softmax confidence reaches
 * gamma is committed (the single most confident one if none does), and the
 * step repeats until the block is full.
 *
 * Sources (web pages on the method):
 *  - poko-everyday.com, "Nemotron-TwoTower" article, section "技術/ビジネス面":
 *    frozen causal context tower; denoising tower with bidirectional block
 *    attention and cross-attention to the context.
 *  - prednext.com, "拡散言語モデル" explainer, section "拡散言語モデルで推論するには":
 *    steps 1-5 of decoding (feed [MASK]s, adopt positions whose output passes
 *    a threshold, return the others to [MASK], repeat until none is left).
 *  - dzen.guru, Nemotron TwoTower news, "Что нового" and "Как попробовать?":
 *    block size 16, confidence threshold gamma = 0.8, the mock-AR mode.
 *
 * Conventions for every entry point:
 *  - Device memory is owned by the caller.  The library allocates no device
 *    memory: `dd_create` receives a caller-allocated workspace (size from
 *    `dd_workspace_size`), and weights are borrowed device pointers that must
 *    stay valid until `dd_destroy`.
 *  - bf16 = IEEE bfloat16 stored as 2 bytes; all matrices are row-major and
 *    linear weights are stored [out_features][in_features].
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *    asynchronous on `stream` unless stated otherwise.
 *  - Return value: DD_OK, or an error code; `dd_last_error()` then gives a
 *    one-line message (thread-local).  Argument errors are detected on the
 *    host before anything is enqueued.
 *  - A dd_ctx is not thread-safe; one context serves one host thread at a time.
 *  - The [MASK] input id is V (vocab size).  The LM head has V outputs, so
 *    [MASK] is never predicted.
 */
#ifndef DD_H
#define DD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct dd_ctx dd_ctx;

typedef enum dd_status {
  DD_OK = 0,
  DD_ERR_INVALID_ARG = 1,    /* null pointer, bad size or unsupported shape */
  DD_ERR_CUDA = 2,           /* a CUDA runtime/driver call failed */
  DD_ERR_NOT_READY = 3,      /* weights not set */
  DD_ERR_STEP_LIMIT = 4,     /* dd_decode_block hit max_steps with positions still masked */
  DD_ERR_DEVICE_TIMEOUT = 5, /* a bounded device-side wait expired, or a device-side consistency check
                                failed (dd_last_error() says which); results are invalid */
  DD_ERR_UNSUPPORTED = 6     /* shape outside what the kernels implement */
} dd_status;

/* Commit modes (the `mode` argument of the step and decode calls).  Top-k and
 * fixed steps carry a parameter in bits 8 and up: DD_MODE_PARAM(DD_MODE_TOPK, k)
 * or DD_MODE_PARAM(DD_MODE_STEPS, N), 1 <= k, N <= 65535; gamma is ignored by
 * mock-AR, top-k and fixed steps. */
enum {
  DD_MODE_THRESHOLD = 0, /* commit masked positions with confidence >= gamma (fallback: the most confident one) */
  DD_MODE_MOCK_AR = 1,   /* commit the leftmost masked position each step (one token per step) */
  DD_MODE_TOPK = 2,      /* commit the k most confident masked positions (the explainer's "adopt the top few"
                          * alternative, prednext.com "拡散言語モデルで推論するには" step 3); ties: lower position */
  DD_MODE_STEPS = 3      /* fixed-steps schedule: with r positions masked after t steps, commit the
                          * ceil(r / (N - t)) most confident, so a block fills in N steps (N <= block);
                          * t is recovered from r by replaying the schedule from the full block */
};
#define DD_MODE_PARAM(mode, param) ((int32_t)((mode) | ((param) << 8)))

/* Model and batch shape.  Supported: 1 <= block <= 32 with batch*block a
 * multiple of 16; head_dim 64 or 128; (n_q_heads/n_kv_heads)*block a multiple
 * of 16 and at most 128; hidden a multiple of 256 and at most 2048, or 4096
 * (the row kernels give each row hidden/8 threads, whole warps); mlp and
 * (n_q_heads+2*n_kv_heads)*head_dim multiples of 128; n_q_heads*head_dim a
 * multiple of 64; vocab a multiple of 256; max_ctx >= 0.  Other shapes are
 * refused with DD_ERR_UNSUPPORTED (or DD_ERR_INVALID_ARG). */
typedef struct dd_config {
  int32_t batch;      /* B: sequences decoded together */
  int32_t block;      /* S: positions per block */
  int32_t hidden;     /* H */
  int32_t n_q_heads;  /* Hq */
  int32_t n_kv_heads; /* Hkv, divides Hq; query head h reads kv head h / (Hq/Hkv) */
  int32_t head_dim;   /* D */
  int32_t n_layers;   /* L >= 1 */
  int32_t mlp;        /* F: SwiGLU width */
  int32_t vocab;      /* V */
  int32_t max_ctx;    /* capacity of the context KV cache, in positions */
  float rms_eps;      /* RMSNorm epsilon (1e-5 in the synthetic workloads) */
  float rope_theta;   /* 0: in-block positions from the learned table only.  > 0: also rotary
                       * positions on the block's queries and keys: block position i sits at
                       * T + i (T = context length) and the pair (2j, 2j+1) of every query and
                       * key head turns by (T + i) * rope_theta^(-2j/D) radians; the context
                       * keys are taken as already positioned (the pages are silent on
                       * positions; rotary positions are an optional alternative to the
                       * learned in-block table alone) */
} dd_config;

/* Borrowed device pointers to bf16 weights (stacked over layers). */
typedef struct dd_weights {
  const void* embed;   /* [V+1][H]; row V is the [MASK] embedding */
  const void* pos;     /* [S][H]; in-block position embedding added to every token */
  const void* wqkv;    /* [L][(Hq+2*Hkv)*D][H]: q rows (head-major), then k rows, then v rows */
  const void* wo;      /* [L][H][Hq*D] */
  const void* wgu;     /* [L][2*F][H]: gate rows 0..F-1, then up rows */
  const void* wd;      /* [L][H][F] */
  const void* g_attn;  /* [L][H] RMSNorm gain before attention */
  const void* g_mlp;   /* [L][H] RMSNorm gain before the MLP */
  const void* g_final; /* [H] final RMSNorm gain */
  const void* lm_head; /* [V][H] */
} dd_weights;

/* ---------------------------------------------------------------- context */

/* Bytes of device workspace `dd_create` needs for `cfg` (KV cache included:
 * 2 * L*B*Hkv*max_ctx*D bf16).  Fails with DD_ERR_INVALID_ARG/UNSUPPORTED on
 * a shape the kernels do not implement. */
dd_status dd_workspace_size(const dd_config* cfg, size_t* bytes);

/* Create a context over a caller-allocated device workspace of at least
 * dd_workspace_size() bytes, 256-byte aligned, on the current device.  The
 * workspace must outlive the context.  The KV cache is zero-filled and the
 * context length is 0.  Synchronous. */
dd_status dd_create(const dd_config* cfg, void* workspace, size_t workspace_bytes, dd_ctx** out);

/* Destroy a context (host state only; the workspace stays the caller's). */
void dd_destroy(dd_ctx* ctx);

/* Set the weights (borrowed; see dd_weights).  Every pointer must be non-null
 * and 16-byte aligned.  The decoder weights follow the pre-norm dense
 * transformer reading of the TwoTower denoising tower (attention, then
 * SwiGLU MLP, per layer; final RMSNorm; untied LM head).  Synchronous on the
 * host; enqueues nothing.  May be called again with other weights: the calls
 * after it use the new ones (the step and decode-loop graphs are captured
 * anew); work already enqueued still reads the previous weights, which must
 * stay valid until it completes. */
dd_status dd_init_weights(dd_ctx* ctx, const dd_weights* w);

/* Write context K/V for positions [t0, t0+n) of every layer and sequence and
 * set the context length to t0+n (positions >= t0+n are no longer attended).
 * k, v: bf16 [L][B][Hkv][n][D], device or host memory (copied on `stream`).
 * n = 0 only sets the length.  Requires 0 <= t0, t0+n <= max_ctx.  This is the
 * frozen context tower's output (TwoTower article, "技術/ビジネス面"); the
 * library takes it as given. */
dd_status dd_set_context_kv(dd_ctx* ctx, const void* k, const void* v, int32_t t0, int32_t n,
                            void* stream);

/* Weights of a synthetic context tower.  The pages' tower is a frozen, trained
 * causal model that encodes the committed tokens (TwoTower article,
 * "技術/ビジネス面"); it is out of scope, and this stand-in is one causal
 * self-attention layer over each committed block followed by the K/V
 * projections of every denoiser layer:
 *   e_i = embed[t_i], y_i = RMSNorm(e_i) * g, q|k|v_i = y_i wqkv^T (n_kv_heads
 *   heads of head_dim each), a_i = softmax over j <= i of q_i.k_j / sqrt(D)
 *   applied to v_j, h_i = e_i + a_i wo^T, z_i = RMSNorm(h_i) * g2, and per
 *   denoiser layer l the K rows then the V rows z_i wkv[l]^T.
 * Position i of an appended block depends on the committed tokens at
 * positions <= i only.  Borrowed bf16 device pointers, 16-byte aligned:
 * embed [V][H], g [H], wqkv [3*Hkv*D][H] (q rows, then k, then v),
 * wo [H][Hkv*D], g2 [H], wkv [L][2*Hkv*D][H]. */
typedef struct dd_context_tower {
  const void* embed;
  const void* g;
  const void* wqkv;
  const void* wo;
  const void* g2;
  const void* wkv;
} dd_context_tower;

/* Register (or replace) the context tower.  Synchronous on the host; enqueues
 * nothing. */
dd_status dd_set_context_tower(dd_ctx* ctx, const dd_context_tower* tower);

/* Encode a committed block with the context tower and append it to the
 * context on the device: the K/V of every layer at positions [T, T+S) (T =
 * the current context length, then T += S), with no host round trip.
 * Requires n_layers*2*n_kv_heads*head_dim and 3*n_kv_heads*head_dim to be
 * multiples of 128 (checked by dd_set_context_tower).
 * tokens: int32 [B][S] device memory (ids in [0, V); others read id 0).
 * Requires T + S <= max_ctx.  Asynchronous on `stream`. */
dd_status dd_append_block(dd_ctx* ctx, const int32_t* tokens, void* stream);

/* ------------------------------------------------------------------ decode */

/* One denoising step (explainer steps 2-4).  tokens: int32 [B][S], mask:
 * uint32 [B] (bit i set = position i is [MASK]); both device or host memory,
 * read and updated in place.  Masked positions are fed as [MASK] whatever
 * their id.  For each sequence it commits every masked position with softmax
 * confidence >= gamma, or, if none qualifies, the single most confident one
 * (lowest position on ties); DD_MODE_MOCK_AR commits the leftmost masked
 * position.  A committed position gets the argmax id (lowest id on ties) and
 * its mask bit cleared; committed positions never change.  n_committed:
 * int32 [B] (device or host, may be NULL) receives the count per sequence.
 * Asynchronous on `stream` (host pointers make the copies synchronous). */
dd_status dd_denoise_step(dd_ctx* ctx, int32_t* tokens, uint32_t* mask, float gamma, int32_t mode,
                          int32_t* n_committed, void* stream);

/* Decode one block (explainer step 5): set every position to [MASK] and run
 * denoising steps until no position is masked.  tokens: int32 [B][S], device
 * or host memory, receives the committed ids.  max_steps <= 0 means 4*S.
 * The steps run as one CUDA graph whose conditional while node repeats the
 * step on the device until no position is masked (or a kernel timed out, or
 * max_steps is reached), so the call synchronises `stream` once, at the end;
 * where the driver refuses that graph the loop runs on the host, one
 * synchronisation per step.  steps_out (host, may be NULL) receives the step
 * count.  Returns
 * DD_ERR_STEP_LIMIT if positions are still masked after max_steps and
 * DD_ERR_DEVICE_TIMEOUT if a kernel's bounded wait expired. */
dd_status dd_decode_block(dd_ctx* ctx, int32_t* tokens, float gamma, int32_t mode, int32_t max_steps,
                          int32_t* steps_out, void* stream);

/* Synchronise `stream` and return DD_ERR_DEVICE_TIMEOUT if any kernel of this
 * context recorded an expired wait (or a failed device-side check, such as a
 * pair of GEMM CTAs given different tensor memory) since the last call (the
 * flag is then cleared), else DD_OK. */
dd_status dd_device_status(dd_ctx* ctx, void* stream);

const char* dd_status_string(dd_status s);
const char* dd_last_error(void);

/* ------------------------------------------------------ step probes (tests) */

/* Optional device outputs of one step, for parity checks.  Any pointer may be
 * NULL.  Activations are kept as a bf16 head plus a bf16 remainder (their sum
 * carries the fp32 value to ~2^-17), so the two bf16 outputs hold heads in
 * rows [0, B*S) and remainders in rows [B*S, 2*B*S).
 * attn_out: bf16 [L][2*B*S][Hq*D], the attention output of every layer
 * (before the O projection); hidden: bf16 [2*B*S][H], the final RMSNorm output;
 * logits: fp32 [B*S][V], computed by the same tensor-core LM-head mainloop with
 * a plain store instead of the fused select; conf: fp32 [B*S]; arg: int32 [B*S].
 * With DD_OPT_COMPACT_SEQUENCES (the default) attn_out, hidden and logits hold
 * the active sequences' rows first, compacted (see that option), and conf/arg
 * are valid for the active sequences' rows only. */
typedef struct dd_probe {
  void* attn_out;
  void* hidden;
  float* logits;
  float* conf;
  int32_t* arg;
} dd_probe;

/* dd_denoise_step, and also fill `probe`.  Runs eagerly (not from the cached
 * CUDA graph).  tokens/mask/n_committed must be device memory here. */
dd_status dd_denoise_step_probe(dd_ctx* ctx, int32_t* tokens, uint32_t* mask, float gamma, int32_t mode,
                                int32_t* n_committed, const dd_probe* probe, void* stream);

/* Kernel launches one denoising step enqueues (embedding through commit,
 * plus the loop-control kernel when dd_decode_block runs the device-side
 * loop). */
dd_status dd_step_launch_count(dd_ctx* ctx, int32_t* n);

/* Context options.
 *   DD_OPT_COMPACT_SEQUENCES (set/get, 0 or 1, default 1): with 1 each
 *     denoising step runs only the rows of the sequences that still have a
 *     masked position (explainer step 5: a block stops once no [MASK] is
 *     left, and sequences are independent, so a finished sequence needs no
 *     further computation): the first kernel of the step lists the active
 *     sequences and every later kernel works on their rows, compacted to the
 *     front, and skips the rest (linear-layer tiles past the active rows,
 *     attention work items of finished sequences).  Results are those of the
 *     uncompacted step; with 0 every step runs all B*S rows.  Not combined
 *     with DD_OPT_FUSED_REDUCE (which runs all rows).  Activations reported by
 *     dd_denoise_step_probe (attention outputs, final hidden state, logits)
 *     are then in compacted row order: rows k*S .. k*S+S-1 belong to the k-th
 *     sequence (in order) that had a masked position before the step; conf
 *     and arg stay in the original order, valid for those sequences' rows.
 *     Switching drops the captured graphs.
 *   DD_OPT_FUSED_REDUCE (set/get, 0 or 1): with 1 the linear layers of the
 *     step (QKV, O, gate|up and every down projection but the last) sum
 *     their split-K partials inside the GEMM: the CTAs that split one
 *     128-feature tile's K form a group (the whole grid resident at once),
 *     exchange fp32 partial tiles through an L2-resident scratch and a
 *     per-group counter, and apply the layer's epilogue there (rotary
 *     positions, SwiGLU, residual add); the RMSNorms before attention and
 *     before the MLP are then deferred into the consuming GEMM (the layer is
 *     linear in its input, so only the rounding order changes).  With 0
 *     every linear layer writes fp32 partials and a separate kernel reduces
 *     them.  1 is available where batch * block <= 128; elsewhere setting it
 *     returns DD_ERR_UNSUPPORTED.  Switching drops the captured graphs.
 *   DD_OPT_FUSED_SPLITS_* / DD_OPT_FUSED_GRID_* (get only): the K splits
 *     (group size) and grid of each fused layer (0 when unavailable).
 */
enum {
  DD_OPT_FUSED_REDUCE = 1,
  DD_OPT_COMPACT_SEQUENCES = 10,
  DD_OPT_FUSED_SPLITS_QKV = 2, DD_OPT_FUSED_SPLITS_O, DD_OPT_FUSED_SPLITS_GATE_UP, DD_OPT_FUSED_SPLITS_DOWN,
  DD_OPT_FUSED_GRID_QKV = 6, DD_OPT_FUSED_GRID_O, DD_OPT_FUSED_GRID_GATE_UP, DD_OPT_FUSED_GRID_DOWN
};
dd_status dd_set_option(dd_ctx* ctx, int32_t option, int32_t value);
dd_status dd_get_option(dd_ctx* ctx, int32_t option, int32_t* value);

/* Launch kinds reported by dd_profile_step.  DD_KIND_ATTENTION is the context
 * attention (all of it on the mma.sync path); DD_KIND_ATTN_COMBINE merges the
 * split partials and, on the tcgen05 path, attends to the in-block keys. */
enum {
  DD_KIND_EMBED = 0, DD_KIND_GEMM_QKV, DD_KIND_REDUCE_QKV, DD_KIND_ATTENTION, DD_KIND_ATTN_COMBINE, DD_KIND_GEMM_O,
  DD_KIND_NORM_O, DD_KIND_GEMM_GATE_UP, DD_KIND_SWIGLU, DD_KIND_GEMM_DOWN, DD_KIND_NORM_DOWN, DD_KIND_LM_SELECT,
  DD_KIND_SELECT_COMBINE, DD_KIND_COMMIT
};

/* One denoising step, as dd_denoise_step, but launched eagerly with a CUDA
 * event recorded after every kernel on `stream`; synchronises, then writes
 * the duration of each launch (ms, event to event) to times_ms and its
 * DD_KIND_* to kinds (capacity `cap`) and the number written to *n.
 * tokens/mask: device or host, updated in place. */
dd_status dd_profile_step(dd_ctx* ctx, int32_t* tokens, uint32_t* mask, float gamma, int32_t mode, float* times_ms,
                          int32_t* kinds, int32_t cap, int32_t* n, void* stream);

/* ------------------------------------------- single-kernel entry points */

/* Block attention for one layer (TwoTower article, "技術/ビジネス面"): for
 * every sequence b, query head h and block position i, one softmax over the
 * ctx_len context keys and the S block keys of kv head h/(Hq/Hkv), scale
 * 1/sqrt(D), no mask.
 *   qkv:   bf16 [B*S][(Hq+2*Hkv)*D], row b*S+i holds q (Hq heads), k, v of position i
 *   k_ctx, v_ctx: bf16 [B][Hkv][ctx_stride][D] (positions >= ctx_len are
 *          never used: they may hold anything, NaN included)
 *   out:   bf16 [B*S][Hq*D]
 *   workspace: device scratch of dd_block_attention_workspace_size() bytes
 *          (split-context partials), 256-byte aligned.  Its first 4 bytes are
 *          the call's status word (int32): the call clears it, and a kernel
 *          whose bounded wait expires sets it non-zero, in which case `out`
 *          is not valid.  Read it once the stream has completed the call.
 * All pointers device memory, 16-byte aligned.  Asynchronous on `stream`. */
typedef struct dd_attn_problem {
  int32_t batch, block, n_q_heads, n_kv_heads, head_dim;
  int32_t ctx_len, ctx_stride;
  const void* qkv;
  const void* k_ctx;
  const void* v_ctx;
  void* out;
  void* workspace;
  size_t workspace_bytes;
} dd_attn_problem;

dd_status dd_block_attention_workspace_size(const dd_attn_problem* p, size_t* bytes);
dd_status dd_block_attention(const dd_attn_problem* p, void* stream);

/* LM head fused with the confidence select: logits = x W^T (fp32 accumulate on
 * the tensor cores, never written to memory), then per row conf = 1/sum_v
 * exp(l_v - max) and arg = the lowest id of the maximum logit.
 *   x: bf16 [rows][hidden], w: bf16 [vocab][hidden], conf: fp32 [rows], arg: int32 [rows]
 *   workspace: dd_lmhead_select_workspace_size() bytes (per-tile partials),
 *   256-byte aligned; its first 4 bytes are the call's status word (int32),
 *   cleared by the call and set non-zero by a kernel whose bounded wait
 *   expires, in which case conf and arg are not valid (read it once the
 *   stream has completed the call).
 * hidden a multiple of 64, vocab a multiple of 256, rows >= 1.  Device
 * memory; asynchronous on `stream`. */
dd_status dd_lmhead_select_workspace_size(int32_t rows, int32_t hidden, int32_t vocab, size_t* bytes);
dd_status dd_lmhead_select(int32_t rows, int32_t hidden, int32_t vocab, const void* x, const void* w,
                           float* conf, int32_t* arg, void* workspace, size_t workspace_bytes, void* stream);

/* The same LM head + confidence select as dd_lmhead_select, for callers that
 * cannot allocate device memory: code running under a host framework's memory
 * pool or a fixed device-memory budget it must not bypass, or latency-critical
 * loops that cannot afford the device synchronisation an allocation may
 * cause.  The web pages on the method have no counterpart of this call; it
 * is a deployment convenience.  It takes no workspace: the per-tile scratch
 * lives in an 8 MiB array inside the library, held on every device that loads
 * the library until the process exits, which limits rows * (vocab/256) to
 * at most 698944 (larger requests fail with DD_ERR_INVALID_ARG before
 * anything is launched).  It calls no allocating routine.  The first call on
 * each device is a warm-up: it looks up that array's device address (with the
 * device current), and under lazy module loading (CUDA's default) that
 * lookup loads the module and creates the array, so it may allocate and
 * synchronise; make it before any stream capture and outside any region that
 * must not allocate.  The address is cached, so a device reset after the
 * first call is not supported.  All calls share the array and it keeps the
 * last call's contents, so calls that overlap on the GPU race.  If a bounded
 * wait inside the kernel expires, every output of the call is overwritten
 * with conf = NaN and arg = -1 (the call itself has already returned DD_OK,
 * being asynchronous).
 * x: bf16 [rows][hidden], w: bf16 [vocab][hidden], conf: fp32 [rows],
 * arg: int32 [rows], all device memory; asynchronous on `stream`. */
dd_status dd_lmhead_select_noalloc(int32_t rows, int32_t hidden, int32_t vocab, const void* x, const void* w,
                                   float* conf, int32_t* arg, void* stream);

/* Plain tensor-core GEMM y = x w^T with fp32 output, through the same kernel
 * the linear layers use.  x: bf16 [rows][k], w: bf16 [n][k], y: fp32 [rows][n].
 * n a multiple of 128, k a multiple of 64, rows a multiple of 16.  workspace:
 * dd_gemm_workspace_size() bytes (split-K partials), 256-byte aligned; its
 * first 4 bytes are the call's status word (int32), cleared by the call and
 * set non-zero by a kernel whose bounded wait expires, in which case y is not
 * valid (read it once the stream has completed the call).  Device memory;
 * asynchronous on `stream`. */
dd_status dd_gemm_workspace_size(int32_t rows, int32_t n, int32_t k, size_t* bytes);
dd_status dd_gemm(int32_t rows, int32_t n, int32_t k, const void* x, const void* w, float* y,
                  void* workspace, size_t workspace_bytes, void* stream);

/* The plan the tensor-core GEMM takes for a linear layer of `rows` activation
 * rows (split_act != 0: bf16 head + remainder rows, as in the denoising step),
 * n outputs and k inputs (rows % 16 == 0, n % 128 == 0, k % 64 == 0).  Host
 * only: no device is touched.  Writes up to n_out of, in order: grid (CTAs),
 * cluster (1, or 2 for CTA pairs), cg (2: one MMA of M = 256 per pair),
 * bk (K elements per block), BN (activation rows per tile), m_tiles, n_tiles,
 * kb_total (K blocks per tile), splits (partial slots), kb_per_split,
 * sk_units (> 0: stream-K, K blocks per worker), sk_total, stages, smem_bytes.
 * For tests and tuning. */
enum { DD_GEMM_PLAN_FIELDS = 14 };
dd_status dd_gemm_plan_query(int32_t rows, int32_t n, int32_t k, int32_t split_act, int32_t* out, int32_t n_out);

/* The commit rule alone (explainer steps 3-4) on given confidences and ids.
 * conf: fp32 [B][S], arg: int32 [B][S], tokens: int32 [B][S] (updated),
 * mask: uint32 [B] (updated), n_committed: int32 [B], remaining: int32 [1]
 * (masked positions left over all sequences).  Device memory. */
dd_status dd_commit(int32_t batch, int32_t block, const float* conf, const int32_t* arg, int32_t* tokens,
                    uint32_t* mask, float gamma, int32_t mode, int32_t* n_committed, int32_t* remaining,
                    void* stream);

/* Launch a kernel that waits on a barrier nothing will ever complete, with a
 * wait limit of `timeout_us` microseconds (1..1e7), and report what it
 * recorded: DD_ERR_DEVICE_TIMEOUT when the bounded wait expired as designed.
 * status: one device int32 used as the kernel's status word.  For testing the
 * timeout path; synchronous. */
dd_status dd_test_wait_timeout(int32_t timeout_us, int32_t* status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DD_H */
