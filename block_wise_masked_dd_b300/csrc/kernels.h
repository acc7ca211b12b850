// Host-side launch interfaces of the CUDA kernels (internal to libdd).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dd {

// Values of the device status word (0: ok), set by kernels and read by the host.
enum : int { kStatusOk = 0, kStatusTimeout = 1, kStatusPairTmem = 2 };

// Launch `kernel` on `st` with programmatic dependent launch allowed: the
// kernel may start while its predecessor drains and must call pdl_wait()
// before touching the predecessor's outputs (every kernel of this library
// does).

template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                     Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// launch_k with thread-block clusters of `cluster_x` CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_k_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                             int cluster_x, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster_x;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

constexpr int kNumSMs = 148;
constexpr int kMaxSplits = 16;  // split-K partials of one linear layer, at most
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;  // 2 s per bounded wait

// ------------------------------------------------------------ tcgen05 GEMM

enum GemmEpi : int {
  kEpiPartial = 0,   // D = W_tile * X_tile^T (features on lanes), fp32 partial [split][row][feature]
  kEpiSelect = 1,    // D = X_tile * W_tile^T (rows on lanes), per-row (max, sumexp, argmax) per vocab tile
  kEpiStore = 2,     // D = X_tile * W_tile^T, fp32 store [row][col] (logit probe)
};

struct GemmPlan {
  int epi;
  int m_tiles, n_tiles, splits;   // tile grid (M = 128 per tile)
  int kb_total, kb_per_split;     // K blocks of bk
  int bk;                         // K elements per block: 64 (128-byte swizzle) or 32 (64-byte swizzle)
  int BN;                         // MMA N (multiple of 16, <= 256)
  int stages;
  int tiles_total;
  int grid;
  int smem_bytes;
  uint32_t tmem_half;             // TMEM columns per accumulator buffer (power of two >= BN)
  int split_act;                  // activation operand = bf16 head rows [0,R) + remainder rows [R,2R)
  int split_rows;                 // R
  int fused_op;                   // fused plans (plan_gemm_fused): the epilogue op; splits = group size
  int sk_units, sk_total;         // stream-K (> 0): (tile, K block) units per CTA and in all; splits = slots
  int cluster;                    // 2: CTA pairs on adjacent weight tiles (cluster of 2)
  int cg;                         // 2: the pair runs one MMA of M = 256 (cta_group::2)
  int box_rows_b;                 // rows of the activation operand's TMA box (BN / cluster)
};

// Which partial slots of a linear layer's output hold data: with a uniform
// K split every tile fills `splits` slots; with stream-K a tile fills one
// slot per piece it was cut into (its run of K blocks over the workers).
struct SlotPlan {
  int splits;    // slots of the partial buffer
  int sk_units;  // > 0: stream-K, K blocks per worker
  int kb_total;  // K blocks per tile
  int n_tiles;   // activation-row tiles
  int BN;        // activation rows per tile
  int cluster;   // weight tiles per schedule unit (CTA pairs: 2)
};

// The slots holding data at (activation row, output feature).
__host__ __device__ inline int slots_of(const SlotPlan& p, int row, int feature) {
  if (p.sk_units <= 0) return p.splits;
  const long long t = (long long)(feature / 128 / p.cluster) * p.n_tiles + row / p.BN;
  const long long first = t * p.kb_total / p.sk_units;
  const long long last = ((t + 1) * p.kb_total - 1) / p.sk_units;
  return (int)(last - first + 1);
}

struct GemmOut {
  float* partial;          // kEpiPartial: [splits][rows][ld]; kEpiStore: [rows][ld]
  long long split_stride;  // elements between splits
  int ld;
  int rows_valid;          // rows of the activation operand
  float* sel_m;            // kEpiSelect: [n_tiles][rows_valid]
  float* sel_s;
  int* sel_a;
  const int* rows_dev;     // device count of valid activation rows (compacted), or nullptr: tiles whose
                           // first activation row is at or past it are skipped (except a CTA's first)
};

// Plan a GEMM over activations [rows][K] and weights [N][K].  With
// split_act the activation map covers [2*rows][K]: bf16 heads then remainders.
// allow_pairs = 0: no CTA pairs (every activation map then has BN-row boxes).
GemmPlan plan_gemm(int epi, int rows, int N, int K, int split_act = 0, int allow_pairs = 1);
inline SlotPlan slot_plan(const GemmPlan& p) {
  return SlotPlan{p.splits, p.sk_units, p.kb_total, p.n_tiles, p.BN, p.cluster};
}
// Enqueue.  map_w / map_x: 2D bf16 tensor maps with 128-byte swizzle, box
// {64, 128} for the operand on the MMA M side and {64, BN} for the other.
cudaError_t launch_gemm(const GemmPlan& p, const CUtensorMap& map_a, const CUtensorMap& map_b, const GemmOut& out,
                        int* status, uint64_t timeout_ns, cudaStream_t st);

// ------------------------------------------- fused split-K linear layers
//
// A linear layer of the step whose K splits run as one group of CTAs (all
// CTAs of the grid resident at once): the members each take a K range of the
// same 128-feature tile, write their fp32 partial tile to a scratch slot that
// stays in L2, and once the group's counter shows all of them, each sums a
// share of the tile's rows and applies the layer's epilogue, so no reduce
// kernel runs.  Activations are split (bf16 head + remainder rows) and at
// most 128 rows long.
//
// Deferred RMSNorm: a residual epilogue writes y' = x * g (not normalised)
// and, per 128-feature tile, the sum of x^2 of each row; the consuming GEMM
// scales row r of its result by rsqrt(sum over tiles / hidden + eps), which
// equals normalising first since the layer is linear in its input.

enum FusedOp : int {
  kOpQkv = 0,       // q|k|v = rs * sum, rotary on q and k heads, bf16 head + remainder
  kOpSwiglu = 1,    // tile = 64 gate + 64 up features: h = silu(rs g) * (rs u), head + remainder
  kOpResidual = 2,  // x += sum; y' = x * g as head + remainder; per-tile row sums of x^2
};

struct FusedOut {
  void* out;            // bf16 [2*rows][ld]: heads, then remainders
  int ld;               // features of `out` (qkv width, F, or hidden)
  float* x;             // kOpResidual: fp32 [rows][ld], updated in place
  const void* g;        // kOpResidual: bf16 gain [ld]
  float* sq_out;        // kOpResidual: [ld/128][rows] sums of x^2 per feature tile
  const float* sq_in;   // kOpQkv, kOpSwiglu: [n_sq][rows] sums of squares of the input rows
  int n_sq;
  int hidden;
  float eps;
  int S, D, qk_cols;    // kOpQkv rotary: block length, head dim, columns of the q and k heads
  const int* ctx_len;
  float theta;          // 0: no rotary
  float* xpart;         // scratch of fused_scratch_bytes(rows)
  unsigned* cnt;        // fused_counter_bytes() of zeros; left zero by every launch
};

// rows <= 128 and a multiple of 16; N = features (2F for kOpSwiglu).  Returns
// a plan with fused_op = -1 for shapes it does not take; splits = group size.
GemmPlan plan_gemm_fused(int op, int rows, int N, int K);
size_t fused_scratch_bytes(int rows);
size_t fused_counter_bytes();
// map_w: the weights, box {64, 128} (kOpSwiglu: box {64, 64}; the up rows
// start at row F = N / 2); map_x: the split activations, box {64, rows}.
cudaError_t launch_gemm_fused(const GemmPlan& p, const CUtensorMap& map_w, const CUtensorMap& map_x,
                              const FusedOut& out, int* status, uint64_t timeout_ns, cudaStream_t st);
cudaError_t prepare_gemm_fused_kernels();

// ------------------------------------------------------------- attention

struct AttnPlan {
  int D, rows, warps_c, n_splits, stages, smem_bytes;
  // tcgen05 context path (D = 128, 64 query rows): the context splits write
  // partial slots 0..n_ctx-1 (n_splits = n_ctx); the merge kernel adds the
  // block keys and combines.
  int use_tc, n_ctx;
};

struct AttnArgs {
  const void* qkv;     // bf16 [B*S][ld_qkv] (with split: [2*B*S][ld_qkv], heads then remainders)
  int ld_qkv;
  int split;           // q and block k/v carry bf16 remainders; the output is written as head + remainder
  int B, S, Hq, Hkv, G;
  const int* ctx_len;  // device int (context length)
  int z0;              // tensor-map z offset of (b=0, kvh=0) for this layer
  void* out;           // bf16 [B*S][ld_out]
  int ld_out;
  float* part_o;       // [B][Hkv][n_splits][rows][D]
  float2* part_ml;     // [B][Hkv][n_splits][rows]
  float scale_log2;
  int* status;
  uint64_t timeout_ns;
  // Active-sequence compaction record (see launch_embed_norm) or nullptr: the
  // rows of qkv/out and the partials are those of the cmp[1] active
  // sequences, compacted; the context cache of compacted sequence k is that
  // of sequence cmp[2 + k]; (sequence, kv head) pairs past the active ones do
  // nothing.  With it the tcgen05 path also chooses its context splits on the
  // device, per launch, for the active pairs (attn_ctx_splits), within the
  // partial slots the workspace holds (max_pair_splits = pairs x splits).
  const int* cmp;
  int max_pair_splits;
};

// Context splits for `pairs` (sequence, kv head) pairs over `ntiles` 128-key
// tiles: persistent CTAs (one per SM) walk pairs x splits items; the busiest
// takes ceil(items / SMs) items of ceil(tiles / splits) tiles each, plus about
// one tile's worth per item for its partial write.  At most max_splits (and
// 32, and one tile per split).
__host__ __device__ inline int attn_ctx_splits(int pairs, int ntiles, int max_splits) {
  if (ntiles <= 0 || pairs <= 0) return 1;
  int lim = ntiles < 32 ? ntiles : 32;
  if (max_splits < lim) lim = max_splits < 1 ? 1 : max_splits;
  int best = 1;
  long long best_cost = -1;
  for (int s = 1; s <= lim; ++s) {
    const long long per_cta = ((long long)pairs * s + kNumSMs - 1) / kNumSMs;
    const long long cost = per_cta * ((ntiles + s - 1) / s + 1) * 64 + s;
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = s;
    }
  }
  return best;
}

// The context splits a tcgen05-path launch uses: the plan's, or with the
// compaction record the device-side choice for the active pairs.
__host__ __device__ inline int attn_launch_splits(const AttnArgs& a, int n_ctx_plan, int T) {
  if (!a.cmp) return n_ctx_plan;
#ifdef __CUDA_ARCH__
  const int pairs = __ldcg(a.cmp + 1) * a.Hkv;  // L2: the record may be read before the launch's wait
#else
  const int pairs = a.cmp[1] * a.Hkv;
#endif
  return attn_ctx_splits(pairs, (T + 127) / 128, pairs > 0 ? a.max_pair_splits / pairs : 1);
}

AttnPlan plan_attention(int B, int S, int Hq, int Hkv, int D, int max_ctx, int allow_tc = 1);
size_t attention_partial_bytes(const AttnPlan& p, int B, int Hkv);
// map_k/map_v: context cache maps with 64-row boxes; map_k128/map_v128: the
// same caches with 128-row boxes, and map_q the query rows (make_map_q), for
// the tcgen05 path.
// map_q2 (optional): the stacked query map (make_map_q_stacked) for split
// activations; with it the context kernel runs its stacked form.
cudaError_t launch_attention(const AttnPlan& p, const AttnArgs& a, const CUtensorMap& map_k, const CUtensorMap& map_v,
                             const CUtensorMap& map_k128, const CUtensorMap& map_v128, const CUtensorMap& map_q,
                             cudaStream_t st, const CUtensorMap* map_q2 = nullptr);
// tcgen05 context attention (attention_tc.cu)
bool attention_tc_supported(int D, int rows);
int attention_tc_splits(int B, int Hkv, int max_ctx);
bool attention_tc_stacked_supported(int G, int S);
cudaError_t launch_attention_tc(const AttnArgs& a, int n_ctx, const CUtensorMap& map_k128,
                                const CUtensorMap& map_v128, const CUtensorMap& map_q, cudaStream_t st,
                                const CUtensorMap* map_q2 = nullptr);
cudaError_t prepare_attention_tc_kernels();
// Merge the split partials (no-op for the mma.sync path with one split); on
// the tcgen05 path this also attends to the block keys.
cudaError_t launch_attention_combine(const AttnPlan& p, const AttnArgs& a, cudaStream_t st);

// --------------------------------------------------- elementwise / small

// Activation outputs named "split" below are written as bf16 heads in rows
// [0, rows) and bf16 remainders (value - head, rounded) in rows [rows, 2*rows).
// With sq != nullptr the norm is deferred: y = x * g (not normalised) and
// sq[r] = sum of x[r]^2 (the consumer scales by rsqrt(sq / H + eps)).
//
// Active-sequence compaction: with cmp != nullptr the step runs on the rows
// of the sequences that still have a masked position only, compacted to the
// front (row k*S + i = position i of the k-th active sequence).  The embedding
// kernel writes the compaction record, int32 [2 + B + B*S]:
//   cmp[0] active rows, cmp[1] active sequences, cmp[2 + k] the k-th active
//   sequence, cmp[2 + B + r] the original row b*S + i of compacted row r;
// every later kernel of the step reads it (&cmp[0] is the dynamic row count
// of the linear layers and their reduces).
constexpr int cmp_words(int B, int S) { return 2 + B + B * S; }
// With rope_cs (theta > 0) the embedding kernel also writes the step's rotary
// table: rope_cs[i * D/2 + j] = (cos, sin) of (*ctx_len + i) * theta^(-2j/D),
// the angle in double reduced modulo 2 pi, for block positions i < S.
cudaError_t launch_embed_norm(const int32_t* tokens, const uint32_t* mask, const void* embed, const void* pos,
                              const void* g, float* x, void* y_split, int B, int S, int H, int V, float eps,
                              cudaStream_t st, float* sq = nullptr, int* cmp = nullptr, float2* rope_cs = nullptr,
                              float theta = 0.f, int D = 0, const int* ctx_len = nullptr);
// q|k|v of the step: the split-K sum written as bf16 head + remainder; with
// theta > 0 the query and key heads (columns < qk_cols) of row r are rotated
// to position *ctx_len + r % S (see dd_config.rope_theta).
// With rows_dev only the first *rows_dev rows (the active ones) are written;
// with rope_cs the rotation reads the step's table instead of recomputing it.
cudaError_t launch_reduce_qkv(const float* part, const SlotPlan& sp, long long split_stride, int rows, int N, void* out, int S,
                              int D, int qk_cols, const int* ctx_len, float theta, cudaStream_t st,
                              const int* rows_dev = nullptr, const float2* rope_cs = nullptr);
// Context tower (dd_append_block): e = embed[token] (fp32, to x) and
// y = RMSNorm(e) * g as bf16 head + remainder; its causal self-attention over
// each committed block (fp32 q|k|v [rows][3 * heads * D] -> head + remainder
// [2 * rows][heads * D]); then, after the residual and second RMSNorm, the
// split-K sum of y W_kv^T scattered as bf16 into the K/V cache
// [L][B][Hkv][alloc_ctx][D] at positions *ctx_len + i, after which *ctx_len
// grows by S.
cudaError_t launch_tower_embed_norm(const int32_t* tokens, const void* embed, const void* g, float* x, void* y_split,
                                    int rows, int H, int V, float eps, cudaStream_t st);
cudaError_t launch_tower_attention(const float* qkv, void* out_split, int rows, int S, int heads, int D,
                                   cudaStream_t st);
// `done` is a zeroed counter the kernel leaves zeroed again.
cudaError_t launch_reduce_kv_append(const float* part, const SlotPlan& sp, long long split_stride, int rows, int N, int S,
                                    int B, int Hkv, int D, int alloc_ctx, int* ctx_len, unsigned int* done, void* kc,
                                    void* vc, cudaStream_t st);
cudaError_t launch_reduce_f32(const float* part, const SlotPlan& sp, long long split_stride, int rows, int N, float* out,
                              cudaStream_t st);
// With mask != nullptr the rows still masked are also written, compacted, to
// y_c (head rows [0, count), remainders [rows, rows + count)), with
// row_index[k] = the original row (b*S + i) of compacted row k and *count
// their number.  With cmp (active-sequence compaction) rows at or past cmp[0]
// do nothing and row r belongs to sequence cmp[2 + r/S].
cudaError_t launch_reduce_residual_norm(const float* part, const SlotPlan& sp, long long split_stride, float* x,
                                        const void* g, void* y_split, int rows, int H, float eps, cudaStream_t st,
                                        const uint32_t* mask = nullptr, int S = 1, void* y_c = nullptr,
                                        int* row_index = nullptr, int* count = nullptr, const int* cmp = nullptr);
cudaError_t launch_reduce_swiglu(const float* part, const SlotPlan& sp, long long split_stride, void* h_split, int rows,
                                 int F, cudaStream_t st, const int* rows_dev = nullptr);
// With count/row_index (compacted rows): rows r < *count, written to row_index[r].
cudaError_t launch_select_combine(const float* sel_m, const float* sel_s, const int* sel_a, int n_tiles, int rows,
                                  float* conf, int* arg, cudaStream_t st, const int* count = nullptr,
                                  const int* row_index = nullptr);
// params: device float[2] {gamma, mode-as-float}, read at run time so one
// captured graph serves every gamma; when NULL, `gamma` and `mode` are used.
cudaError_t launch_commit(const float* conf, const int* arg, int32_t* tokens, uint32_t* mask, const float* params,
                          float gamma, int mode, int32_t* n_committed, int32_t* remaining, int B, int S,
                          cudaStream_t st);
// Set the dynamic shared-memory limits of every pipelined kernel (once per process).
cudaError_t prepare_kernels();
cudaError_t prepare_gemm_kernels();
cudaError_t prepare_attention_kernels();
cudaError_t prepare_small_kernels();
cudaError_t launch_set_params(float* params, float gamma, int mode, cudaStream_t st);
cudaError_t launch_set_int(int* dst, int value, cudaStream_t st);
// Device-side decode loop: reset the step counter and set the limit; count
// a step and set the while-loop condition (see small_kernels.cu).
cudaError_t launch_loop_init(int32_t* small, int max_steps, cudaStream_t st);
cudaError_t launch_loop_control(int32_t* small, cudaGraphConditionalHandle handle, cudaStream_t st);
cudaError_t launch_init_block(int32_t* tokens, uint32_t* mask, int B, int S, int V, cudaStream_t st);
cudaError_t launch_wait_forever_bounded(int* status, uint64_t timeout_ns, cudaStream_t st);

// Set the thread-local message dd_last_error() returns.
void set_error_message(const char* msg);

// ------------------------------------------------------------ tensor maps

// 2D bf16 map over a row-major [rows][cols] matrix, box {box_cols, box_rows}:
// box_cols 64 with the 128-byte swizzle, 32 with the 64-byte swizzle (a GEMM
// plan's bk).
bool make_map_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                 uint32_t box_cols = 64);
// 3D bf16 map over [planes][rows][cols] (cols = head dim), box {64, box_rows, 1};
// planes lie stride_rows rows apart and rows >= `rows` read as zero.
bool make_map_3d(CUtensorMap* m, const void* base, uint64_t planes, uint64_t rows, uint64_t stride_rows, uint64_t cols,
                 uint32_t box_rows);
// The query heads of a q|k|v buffer [rows][ld] (query head h at columns
// h*D..h*D+D-1) as a 3D bf16 map {D, Hq, rows}, box {64, G, S}: one box is the
// G query heads of a kv head at S consecutive rows, in row order i * G + g.
bool make_map_q(CUtensorMap* m, const void* qkv, uint64_t rows, uint64_t ld, int Hq, int D, int G, int S);
// The query heads of a split q|k|v buffer (bf16 heads in rows [0, rows),
// remainders in rows [rows, 2 rows)) as a 5D map {D, Hq, 8/G positions,
// 2 parts, rows/(8/G)}, box {64, G, 8/G, 2, S*G/8}: one box holds, for S
// consecutive rows, the G query heads of a kv head as 16-row groups of 8
// queries (order i * G + g) -- their 8 head rows, then their 8 remainder rows.
// G must divide 8.
bool make_map_q_stacked(CUtensorMap* m, const void* qkv, uint64_t rows, uint64_t ld, int Hq, int D, int G, int S);

}  // namespace dd
