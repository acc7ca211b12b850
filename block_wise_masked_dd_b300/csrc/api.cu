// C-ABI of libdd: context and workspace management, tensor maps, the
// per-step launch sequence (captured once into a CUDA graph), the decode
// loop, and the single-kernel entry points.  See include/dd.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <string>
#include <vector>

#include "../../include/dd.h"
#include "kernels.h"

namespace {

thread_local std::string g_last_error;

dd_status fail(dd_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

#define DD_CUDA(call)                                                                                   \
  do {                                                                                                  \
    cudaError_t e_ = (call);                                                                            \
    if (e_ != cudaSuccess) return fail(DD_ERR_CUDA, "%s failed: %s", #call, cudaGetErrorString(e_));   \
  } while (0)

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

}  // namespace

namespace dd {

void set_error_message(const char* msg) { g_last_error = msg; }

bool make_map_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                 uint32_t box_cols) {
  auto fn = encode_fn();
  if (!fn || (box_cols != 64 && box_cols != 32)) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, box_cols == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// planes x rows x cols bf16 with planes `stride_rows` rows apart; rows at or
// beyond `rows` read as zero (TMA out-of-bounds fill).
bool make_map_3d(CUtensorMap* m, const void* base, uint64_t planes, uint64_t rows, uint64_t stride_rows, uint64_t cols,
                 uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {cols, rows, planes};
  cuuint64_t strides[2] = {cols * 2, stride_rows * cols * 2};
  cuuint32_t box[3] = {64, box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_q(CUtensorMap* m, const void* qkv, uint64_t rows, uint64_t ld, int Hq, int D, int G, int S) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Hq, rows};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, ld * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)S};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(qkv), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_q_stacked(CUtensorMap* m, const void* qkv, uint64_t rows, uint64_t ld, int Hq, int D, int G, int S) {
  auto fn = encode_fn();
  if (!fn || G < 1 || 8 % G || rows % (8 / G) || S % (8 / G)) return false;
  const uint64_t q8 = 8 / G;  // block positions per 8-query group
  cuuint64_t dims[5] = {(cuuint64_t)D, (cuuint64_t)Hq, q8, 2, rows / q8};
  cuuint64_t strides[4] = {(cuuint64_t)D * 2, ld * 2, rows * ld * 2, q8 * ld * 2};
  cuuint32_t box[5] = {64, (cuuint32_t)G, (cuuint32_t)q8, 2, (cuuint32_t)(S / q8)};
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(qkv), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace dd

// ---------------------------------------------------------------------------
// Context
// ---------------------------------------------------------------------------

struct Layout {
  size_t kc, vc, x, y, yc, row_index, qkv, attn, hmid, part, attn_part, sel_m, sel_s, sel_a, conf, arg, tok, mask,
      ncommit, small, params, sq_a, sq_b, xpart, fcnt, cmp, rope_cs, total;
  size_t part_elems;
  int alloc_ctx;
  dd::GemmPlan p_qkv, p_o, p_gu, p_d, p_lm, p_store, p_tower, p_tqkv, p_to;
  dd::AttnPlan p_attn;
};

struct dd_ctx {
  dd_config cfg;
  int R, G, qkvw, HqD;
  Layout L;
  uint8_t* ws;
  int ctx_len;
  bool have_weights;
  dd_weights w;
  std::vector<CUtensorMap> m_wqkv, m_wo, m_wgu, m_wd;
  std::vector<CUtensorMap> m_wgu64;  // gate|up weights with 64-row boxes (the fused SwiGLU tiles)
  // Linear layers with the split-K reduction and epilogue inside the GEMM
  // (groups of CTAs); fused_ok: planned for this shape.
  dd::GemmPlan f_qkv, f_o, f_gu, f_d;
  bool fused_ok, fused_on;
  // Active-sequence compaction: each step runs only the rows of sequences
  // that still have a masked position (not with the fused linear layers).
  bool compact_on;
  dd_context_tower tower;  // borrowed; tower.wkv == nullptr until dd_set_context_tower
  CUtensorMap m_tower, m_tower_qkv, m_tower_o, m_tower_a;
  CUtensorMap m_lm, m_y_b, m_attn_b, m_h_b, m_y_a, m_yc_a, m_kc, m_vc, m_kc128, m_vc128, m_q;
  CUtensorMap m_q2;  // stacked query map (head and remainder rows), when the stacked context kernel applies
  bool have_q2;
  cudaStream_t cap_stream;
  cudaGraphExec_t exec;       // one denoising step
  cudaGraphExec_t loop_exec;  // while (masked left): step  -- the device-side decode loop
  bool loop_tried;
  int32_t* hpin;  // pinned host: [0] remaining, [1] status, [2] ctx_len, [3] steps, [4] step limit
  uint64_t timeout_ns;
  int device;
  int step_launches;  // kernels one denoising step launches
};

namespace {

template <typename T>
T* at(uint8_t* ws, size_t off) {
  return reinterpret_cast<T*>(ws + off);
}

// Commit mode: threshold or mock-AR with no parameter; top-k or fixed steps
// with a parameter (k or N) in [1, 65535] in bits 8 and up.
bool valid_mode(int32_t mode) {
  const int base = mode & 0xFF, param = (int)((uint32_t)mode >> 8);
  if (base == DD_MODE_THRESHOLD || base == DD_MODE_MOCK_AR) return param == 0;
  if (base == DD_MODE_TOPK || base == DD_MODE_STEPS) return param >= 1 && param <= 65535;
  return false;
}

dd_status check_config(const dd_config* c) {
  if (!c) return fail(DD_ERR_INVALID_ARG, "config is NULL");
  if (c->batch < 1 || c->block < 1 || c->block > 32)
    return fail(DD_ERR_INVALID_ARG, "batch must be >= 1 and block in [1, 32] (got %d, %d)", c->batch, c->block);
  if ((c->batch * c->block) % 16)
    return fail(DD_ERR_UNSUPPORTED, "batch*block must be a multiple of 16 (got %d)", c->batch * c->block);
  if (c->head_dim != 64 && c->head_dim != 128)
    return fail(DD_ERR_UNSUPPORTED, "head_dim must be 64 or 128 (got %d)", c->head_dim);
  if (c->n_q_heads < 1 || c->n_kv_heads < 1 || c->n_q_heads % c->n_kv_heads)
    return fail(DD_ERR_INVALID_ARG, "n_kv_heads must divide n_q_heads (got %d, %d)", c->n_q_heads, c->n_kv_heads);
  const int G = c->n_q_heads / c->n_kv_heads;
  if ((G * c->block) % 16 || G * c->block > 128)
    return fail(DD_ERR_UNSUPPORTED, "(n_q_heads/n_kv_heads)*block must be a multiple of 16 and <= 128 (got %d)",
                G * c->block);
  // The row kernels (embedding, norms) give a row hidden/8 threads, which
  // must be whole warps for their warp-wide reductions.
  if (c->hidden < 256 || c->hidden % 256)
    return fail(DD_ERR_UNSUPPORTED, "hidden must be a multiple of 256 (got %d)", c->hidden);
  if (c->hidden > 4096 || (c->hidden > 2048 && c->hidden % 2048))
    return fail(DD_ERR_UNSUPPORTED, "hidden must be <= 2048, or 4096 (got %d)", c->hidden);
  if (c->mlp < 128 || c->mlp % 128) return fail(DD_ERR_UNSUPPORTED, "mlp must be a multiple of 128 (got %d)", c->mlp);
  if (((c->n_q_heads + 2 * c->n_kv_heads) * c->head_dim) % 128)
    return fail(DD_ERR_UNSUPPORTED, "(n_q_heads+2*n_kv_heads)*head_dim must be a multiple of 128");
  if ((c->n_q_heads * c->head_dim) % 64) return fail(DD_ERR_UNSUPPORTED, "n_q_heads*head_dim must be a multiple of 64");
  if (c->vocab < 256 || c->vocab % 256)
    return fail(DD_ERR_UNSUPPORTED, "vocab must be a multiple of 256 (got %d)", c->vocab);
  if (c->n_layers < 1) return fail(DD_ERR_INVALID_ARG, "n_layers must be >= 1");
  if (c->max_ctx < 0) return fail(DD_ERR_INVALID_ARG, "max_ctx must be >= 0");
  if (!(c->rms_eps >= 0.f)) return fail(DD_ERR_INVALID_ARG, "rms_eps must be >= 0");
  if (!(c->rope_theta >= 0.f) || c->rope_theta > 1e30f) return fail(DD_ERR_INVALID_ARG, "rope_theta must be >= 0 and finite");
  return DD_OK;
}

Layout make_layout(const dd_config& c) {
  Layout L{};
  const int R = c.batch * c.block;
  const int qkvw = (c.n_q_heads + 2 * c.n_kv_heads) * c.head_dim;
  const int HqD = c.n_q_heads * c.head_dim;
  L.alloc_ctx = c.max_ctx < 128 ? 128 : c.max_ctx;  // at least one 128-position TMA box
  // Every activation operand of the step is split (bf16 head + remainder).
  // The linear layers share activation maps, so they share one choice of CTA
  // pairs: when one of them has an odd number of weight tiles none pairs.
  for (int allow_pairs = 1; allow_pairs >= 0; --allow_pairs) {
    L.p_qkv = dd::plan_gemm(dd::kEpiPartial, R, qkvw, c.hidden, 1, allow_pairs);
    L.p_o = dd::plan_gemm(dd::kEpiPartial, R, c.hidden, HqD, 1, allow_pairs);
    L.p_gu = dd::plan_gemm(dd::kEpiPartial, R, 2 * c.mlp, c.hidden, 1, allow_pairs);
    L.p_d = dd::plan_gemm(dd::kEpiPartial, R, c.hidden, c.mlp, 1, allow_pairs);
    L.p_tower = dd::plan_gemm(dd::kEpiPartial, R, c.n_layers * 2 * c.n_kv_heads * c.head_dim, c.hidden, 1,
                              allow_pairs);
    // context tower's attention layer: q|k|v projection and output projection
    L.p_tqkv = dd::plan_gemm(dd::kEpiPartial, R, 3 * c.n_kv_heads * c.head_dim, c.hidden, 1, allow_pairs);
    L.p_to = dd::plan_gemm(dd::kEpiPartial, R, c.hidden, c.n_kv_heads * c.head_dim, 1, allow_pairs);
    const dd::GemmPlan* ps[] = {&L.p_qkv, &L.p_o, &L.p_gu, &L.p_d, &L.p_tower, &L.p_tqkv, &L.p_to};
    bool same = true;
    for (const dd::GemmPlan* q : ps) same = same && q->cluster == L.p_qkv.cluster;
    if (same) break;
  }
  L.p_lm = dd::plan_gemm(dd::kEpiSelect, R, c.vocab, c.hidden, 1);
  L.p_store = dd::plan_gemm(dd::kEpiStore, R, c.vocab, c.hidden, 1);
  L.p_attn = dd::plan_attention(c.batch, c.block, c.n_q_heads, c.n_kv_heads, c.head_dim, c.max_ctx);
  size_t pe = 0;
  auto upd = [&](const dd::GemmPlan& p, int N) {
    size_t e = (size_t)p.splits * R * N;
    if (e > pe) pe = e;
  };
  upd(L.p_qkv, qkvw);
  upd(L.p_o, c.hidden);
  upd(L.p_gu, 2 * c.mlp);
  upd(L.p_d, c.hidden);
  upd(L.p_tower, c.n_layers * 2 * c.n_kv_heads * c.head_dim);
  upd(L.p_tqkv, 3 * c.n_kv_heads * c.head_dim);
  upd(L.p_to, c.hidden);
  L.part_elems = pe;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  const size_t kv = (size_t)c.n_layers * c.batch * c.n_kv_heads * L.alloc_ctx * c.head_dim * 2;
  L.kc = take(kv);
  L.vc = take(kv);
  L.x = take((size_t)R * c.hidden * 4);
  // bf16 activations: heads in rows [0, R), remainders in rows [R, 2R)
  L.y = take((size_t)2 * R * c.hidden * 2);
  // the final norm's rows still masked, compacted (LM-head input), and their rows
  L.yc = take((size_t)2 * R * c.hidden * 2);
  L.row_index = take((size_t)R * 4);
  L.qkv = take((size_t)2 * R * qkvw * 2);
  L.attn = take((size_t)2 * R * HqD * 2);
  L.hmid = take((size_t)2 * R * c.mlp * 2);
  L.part = take(pe * 4);
  L.attn_part = take(dd::attention_partial_bytes(L.p_attn, c.batch, c.n_kv_heads));
  const size_t sel = (size_t)L.p_lm.n_tiles * R * 4;
  L.sel_m = take(sel);
  L.sel_s = take(sel);
  L.sel_a = take(sel);
  L.conf = take((size_t)R * 4);
  L.arg = take((size_t)R * 4);
  L.tok = take((size_t)R * 4);
  L.mask = take((size_t)c.batch * 4);
  L.ncommit = take((size_t)c.batch * 4);
  L.small = take(32);   // [0] remaining, [1] status, [2] ctx_len, [3] steps, [4] step limit, [5] append counter,
                        // [6] rows still masked (the LM head's compacted rows)
  L.params = take(8);   // gamma, mode
  // per-128-feature-tile row sums of squares of the deferred RMSNorms (fused
  // linear layers): before attention and before the MLP
  L.sq_a = take((size_t)(c.hidden / 128) * R * 4);
  L.sq_b = take((size_t)(c.hidden / 128) * R * 4);
  // fused linear layers: partial-tile scratch and group counters (zeroed here,
  // left zero by every launch)
  const bool fusable = R <= 128;
  L.xpart = take(fusable ? dd::fused_scratch_bytes(R) : 0);
  L.fcnt = take(fusable ? dd::fused_counter_bytes() : 0);
  // active-sequence compaction record (written by the embedding kernel each step)
  L.cmp = take((size_t)dd::cmp_words(c.batch, c.block) * 4);
  // rotary (cos, sin) table of the step's block positions (written by the embedding kernel)
  L.rope_cs = take((size_t)c.block * (c.head_dim / 2) * 8);
  L.total = off;
  return L;
}

int32_t* small_ptr(dd_ctx* c) { return at<int32_t>(c->ws, c->L.small); }

// The stacked form of the tcgen05 context-attention kernel (head and
// remainder rows of one M = 128 operand) for split activations.
constexpr bool kStackedContextKernel = true;

// Kinds of launches in one step (for the per-kernel profile).
enum LaunchKind : int {
  kKEmbed = 0, kKGemmQkv, kKReduceQkv, kKAttention, kKAttnCombine, kKGemmO, kKNormO, kKGemmGu, kKSwiglu,
  kKGemmDown, kKNormDown, kKLmSelect, kKSelectCombine, kKCommit, kKNumKinds
};

// Records an event after each launch when profiling; counts launches always.
struct Marker {
  cudaStream_t st;
  cudaEvent_t* ev = nullptr;
  int32_t* kinds = nullptr;
  int cap = 0;
  int n = 0;
  cudaError_t err = cudaSuccess;
  void operator()(int kind) {
    if (ev && n < cap) {
      kinds[n] = kind;
      cudaError_t e = cudaEventRecord(ev[n + 1], st);
      if (e != cudaSuccess) err = e;
    }
    ++n;
  }
};

dd_status enqueue_step(dd_ctx* c, cudaStream_t st, const dd_probe* probe, Marker* mk_in = nullptr) {
  Marker local{st};
  Marker& mk = mk_in ? *mk_in : local;
  const dd_config& cf = c->cfg;
  const Layout& L = c->L;
  uint8_t* ws = c->ws;
  const int R = c->R, H = cf.hidden, F = cf.mlp;
  float* x = at<float>(ws, L.x);
  void* y = ws + L.y;
  float* part = at<float>(ws, L.part);
  int* status = small_ptr(c) + 1;
  const uint8_t* g_attn = static_cast<const uint8_t*>(c->w.g_attn);
  const uint8_t* g_mlp = static_cast<const uint8_t*>(c->w.g_mlp);
  const bool lm_compact = !probe && L.p_lm.m_tiles > 1;
  // Active-sequence compaction record (nullptr: every sequence's rows run).
  int* cmp = (c->compact_on && !c->fused_on) ? at<int>(ws, L.cmp) : nullptr;
  // Fused linear layers: the norms before attention and before the MLP are
  // deferred (y = x * g, sums of squares in sq_a / sq_b) and applied by the
  // consuming GEMM; the last layer's down projection keeps the separate
  // residual + RMSNorm kernel (final norm, LM-head row compaction).
  const bool fz = c->fused_on;
  float* sq_a = at<float>(ws, L.sq_a);
  float* sq_b = at<float>(ws, L.sq_b);
  dd::FusedOut fo{};
  fo.hidden = H;
  fo.eps = cf.rms_eps;
  fo.S = cf.block;
  fo.D = cf.head_dim;
  fo.qk_cols = (cf.n_q_heads + cf.n_kv_heads) * cf.head_dim;
  fo.ctx_len = small_ptr(c) + 2;
  fo.theta = cf.rope_theta;
  fo.xpart = at<float>(ws, L.xpart);
  fo.cnt = at<unsigned>(ws, L.fcnt);

  float2* rope_cs = cf.rope_theta > 0.f ? at<float2>(ws, L.rope_cs) : nullptr;
  DD_CUDA(dd::launch_embed_norm(at<int32_t>(ws, L.tok), at<uint32_t>(ws, L.mask), c->w.embed, c->w.pos, g_attn,
                                x, y, cf.batch, cf.block, H, cf.vocab, cf.rms_eps, st, fz ? sq_a : nullptr, cmp,
                                rope_cs, cf.rope_theta, cf.head_dim, small_ptr(c) + 2));
  mk(kKEmbed);
  for (int l = 0; l < cf.n_layers; ++l) {
    dd::GemmOut o{};
    o.partial = part;
    o.rows_valid = R;
    o.rows_dev = cmp;  // active rows (cmp[0]); N tiles past them are skipped
    // q|k|v = y Wqkv^T
    if (fz) {
      fo.out = ws + L.qkv;
      fo.ld = c->qkvw;
      fo.sq_in = sq_a;
      fo.n_sq = l == 0 ? 1 : H / 128;  // the embedding's norm sums a whole row in one slot
      DD_CUDA(dd::launch_gemm_fused(c->f_qkv, c->m_wqkv[l], c->m_y_b, fo, status, c->timeout_ns, st));
      mk(kKGemmQkv);
    } else {
      o.ld = c->qkvw;
      o.split_stride = (long long)R * c->qkvw;
      DD_CUDA(dd::launch_gemm(L.p_qkv, c->m_wqkv[l], c->m_y_b, o, status, c->timeout_ns, st));
      mk(kKGemmQkv);
      DD_CUDA(dd::launch_reduce_qkv(part, dd::slot_plan(L.p_qkv), o.split_stride, R, c->qkvw, ws + L.qkv, cf.block,
                                    cf.head_dim, fo.qk_cols, small_ptr(c) + 2, cf.rope_theta, st, cmp, rope_cs));
      mk(kKReduceQkv);
    }
    // block attention
    dd::AttnArgs a{};
    a.qkv = ws + L.qkv;
    a.ld_qkv = c->qkvw;
    a.split = 1;
    a.B = cf.batch;
    a.S = cf.block;
    a.Hq = cf.n_q_heads;
    a.Hkv = cf.n_kv_heads;
    a.G = c->G;
    a.ctx_len = small_ptr(c) + 2;
    a.z0 = l * cf.batch * cf.n_kv_heads;
    a.out = ws + L.attn;
    a.ld_out = c->HqD;
    a.part_o = at<float>(ws, L.attn_part);
    a.part_ml = reinterpret_cast<float2*>(
        ws + L.attn_part +
        align_up((size_t)cf.batch * cf.n_kv_heads * L.p_attn.n_splits * L.p_attn.rows * cf.head_dim * 4, 16));
    a.scale_log2 = 1.4426950408889634f / sqrtf((float)cf.head_dim);
    a.status = status;
    a.timeout_ns = c->timeout_ns;
    a.cmp = cmp;
    a.max_pair_splits = cf.batch * cf.n_kv_heads * L.p_attn.n_splits;
    DD_CUDA(dd::launch_attention(L.p_attn, a, c->m_kc, c->m_vc, c->m_kc128, c->m_vc128, c->m_q, st,
                                 c->have_q2 ? &c->m_q2 : nullptr));
    mk(kKAttention);
    if (L.p_attn.use_tc || L.p_attn.n_splits > 1) {
      DD_CUDA(dd::launch_attention_combine(L.p_attn, a, st));
      mk(kKAttnCombine);
    }
    if (probe && probe->attn_out)
      DD_CUDA(cudaMemcpyAsync(static_cast<uint8_t*>(probe->attn_out) + (size_t)l * 2 * R * c->HqD * 2, ws + L.attn,
                              (size_t)2 * R * c->HqD * 2, cudaMemcpyDeviceToDevice, st));
    if (fz) {
      // x += attn Wo^T ; y = x g_mlp (deferred norm) ; then h = silu(y Wg^T) * (y Wu^T)
      fo.out = y;
      fo.ld = H;
      fo.x = x;
      fo.g = g_mlp + (size_t)l * H * 2;
      fo.sq_out = sq_b;
      DD_CUDA(dd::launch_gemm_fused(c->f_o, c->m_wo[l], c->m_attn_b, fo, status, c->timeout_ns, st));
      mk(kKGemmO);
      fo.out = ws + L.hmid;
      fo.ld = F;
      fo.sq_in = sq_b;
      fo.n_sq = H / 128;
      DD_CUDA(dd::launch_gemm_fused(c->f_gu, c->m_wgu64[l], c->m_y_b, fo, status, c->timeout_ns, st));
      mk(kKGemmGu);
    } else {
      // x += attn Wo^T ; y = norm(x) g_mlp
      o.ld = H;
      o.split_stride = (long long)R * H;
      DD_CUDA(dd::launch_gemm(L.p_o, c->m_wo[l], c->m_attn_b, o, status, c->timeout_ns, st));
      mk(kKGemmO);
      DD_CUDA(dd::launch_reduce_residual_norm(part, dd::slot_plan(L.p_o), o.split_stride, x, g_mlp + (size_t)l * H * 2, y, R,
                                              H, cf.rms_eps, st, nullptr, cf.block, nullptr, nullptr, nullptr, cmp));
      mk(kKNormO);
      // h = silu(y Wg^T) * (y Wu^T)
      o.ld = 2 * F;
      o.split_stride = (long long)R * 2 * F;
      DD_CUDA(dd::launch_gemm(L.p_gu, c->m_wgu[l], c->m_y_b, o, status, c->timeout_ns, st));
      mk(kKGemmGu);
      DD_CUDA(dd::launch_reduce_swiglu(part, dd::slot_plan(L.p_gu), o.split_stride, ws + L.hmid, R, F, st, cmp));
      mk(kKSwiglu);
    }
    const void* gn = (l + 1 < cf.n_layers) ? (const void*)(g_attn + (size_t)(l + 1) * H * 2) : c->w.g_final;
    if (fz && l + 1 < cf.n_layers) {
      // x += h Wd^T ; y = x g_attn[l + 1] (deferred norm)
      fo.out = y;
      fo.ld = H;
      fo.x = x;
      fo.g = gn;
      fo.sq_out = sq_a;
      DD_CUDA(dd::launch_gemm_fused(c->f_d, c->m_wd[l], c->m_h_b, fo, status, c->timeout_ns, st));
      mk(kKGemmDown);
      continue;
    }
    // x += h Wd^T ; y = norm(x) g (next layer's attention norm, or the final norm)
    o.ld = H;
    o.split_stride = (long long)R * H;
    DD_CUDA(dd::launch_gemm(L.p_d, c->m_wd[l], c->m_h_b, o, status, c->timeout_ns, st));
    mk(kKGemmDown);
    // The final norm also compacts the rows still masked for the LM head
    // (except on the probe path, which reports every row, and when the LM
    // head has one row tile, which no compaction can skip).
    const bool compact = lm_compact && l + 1 == cf.n_layers;
    DD_CUDA(dd::launch_reduce_residual_norm(part, dd::slot_plan(L.p_d), o.split_stride, x, gn, y, R, H, cf.rms_eps, st,
                                            compact ? at<uint32_t>(ws, L.mask) : nullptr, cf.block, ws + L.yc,
                                            at<int>(ws, L.row_index), small_ptr(c) + 6, cmp));
    mk(kKNormDown);
  }
  // LM head + fused select, over the compacted masked rows (all rows when not
  // compacting them; with active-sequence compaction those rows are in
  // compacted order, and the select scatters them back to their own rows)
  dd::GemmOut so{};
  so.rows_valid = R;
  so.sel_m = at<float>(ws, L.sel_m);
  so.sel_s = at<float>(ws, L.sel_s);
  so.sel_a = at<int>(ws, L.sel_a);
  so.rows_dev = lm_compact ? small_ptr(c) + 6 : cmp;
  DD_CUDA(dd::launch_gemm(L.p_lm, lm_compact ? c->m_yc_a : c->m_y_a, c->m_lm, so, status, c->timeout_ns, st));
  mk(kKLmSelect);
  const int* sel_index = lm_compact ? at<int>(ws, L.row_index) : (cmp ? cmp + 2 + cf.batch : nullptr);
  DD_CUDA(dd::launch_select_combine(so.sel_m, so.sel_s, so.sel_a, L.p_lm.n_tiles, R, at<float>(ws, L.conf),
                                    at<int>(ws, L.arg), st, so.rows_dev, sel_index));
  mk(kKSelectCombine);
  if (probe) {
    if (probe->hidden)
      DD_CUDA(cudaMemcpyAsync(probe->hidden, y, (size_t)2 * R * H * 2, cudaMemcpyDeviceToDevice, st));
    if (probe->conf) DD_CUDA(cudaMemcpyAsync(probe->conf, ws + L.conf, (size_t)R * 4, cudaMemcpyDeviceToDevice, st));
    if (probe->arg) DD_CUDA(cudaMemcpyAsync(probe->arg, ws + L.arg, (size_t)R * 4, cudaMemcpyDeviceToDevice, st));
    if (probe->logits) {
      dd::GemmOut lo{};
      lo.partial = probe->logits;
      lo.ld = cf.vocab;
      lo.rows_valid = R;
      DD_CUDA(dd::launch_gemm(L.p_store, c->m_y_a, c->m_lm, lo, status, c->timeout_ns, st));
    }
  }
  DD_CUDA(dd::launch_commit(at<float>(ws, L.conf), at<int>(ws, L.arg), at<int32_t>(ws, L.tok),
                            at<uint32_t>(ws, L.mask), at<float>(ws, L.params), 0.f, 0,
                            at<int32_t>(ws, L.ncommit), small_ptr(c), cf.batch, cf.block, st));
  mk(kKCommit);
  if (mk.err != cudaSuccess) return fail(DD_ERR_CUDA, "event record failed: %s", cudaGetErrorString(mk.err));
  return DD_OK;
}

dd_status ensure_graph(dd_ctx* c) {
  if (c->exec) return DD_OK;
  cudaGraph_t g = nullptr;
  Marker counter{c->cap_stream};
  DD_CUDA(cudaStreamBeginCapture(c->cap_stream, cudaStreamCaptureModeThreadLocal));
  dd_status s = enqueue_step(c, c->cap_stream, nullptr, &counter);
  c->step_launches = counter.n;
  cudaError_t e = cudaStreamEndCapture(c->cap_stream, &g);
  if (s != DD_OK) {
    if (g) cudaGraphDestroy(g);
    return s;
  }
  if (e != cudaSuccess) return fail(DD_ERR_CUDA, "graph capture failed: %s", cudaGetErrorString(e));
  e = cudaGraphInstantiate(&c->exec, g, 0);
  cudaGraphDestroy(g);
  if (e != cudaSuccess) {
    c->exec = nullptr;
    return fail(DD_ERR_CUDA, "graph instantiate failed: %s", cudaGetErrorString(e));
  }
  return DD_OK;
}

// The decode loop as one graph: a conditional while node whose body is the
// step followed by k_loop_control, which sets the condition on the device.
// Returns false (and leaves loop_exec unset) where the driver refuses the
// graph; dd_decode_block then loops on the host.
bool ensure_loop_graph(dd_ctx* c) {
  if (c->loop_exec) return true;
  if (c->loop_tried) return false;
  c->loop_tried = true;
  cudaGraph_t g = nullptr;
  if (cudaGraphCreate(&g, 0) != cudaSuccess) return false;
  cudaGraphConditionalHandle h = 0;
  cudaGraphNodeParams np = {};
  cudaGraphNode_t node = nullptr;
  bool ok = cudaGraphConditionalHandleCreate(&h, g, 1, cudaGraphCondAssignDefault) == cudaSuccess;
  if (ok) {
    np.type = cudaGraphNodeTypeConditional;
    np.conditional.handle = h;
    np.conditional.type = cudaGraphCondTypeWhile;
    np.conditional.size = 1;
    ok = cudaGraphAddNode(&node, g, nullptr, nullptr, 0, &np) == cudaSuccess;
  }
  if (ok) {
    cudaGraph_t body = np.conditional.phGraph_out[0];
    ok = cudaStreamBeginCaptureToGraph(c->cap_stream, body, nullptr, nullptr, 0, cudaStreamCaptureModeThreadLocal) ==
         cudaSuccess;
    if (ok) {
      dd_status s = enqueue_step(c, c->cap_stream, nullptr, nullptr);
      const bool launched = s == DD_OK && dd::launch_loop_control(small_ptr(c), h, c->cap_stream) == cudaSuccess;
      cudaGraph_t captured = nullptr;
      ok = cudaStreamEndCapture(c->cap_stream, &captured) == cudaSuccess && launched;
    }
  }
  if (ok) ok = cudaGraphInstantiate(&c->loop_exec, g, 0) == cudaSuccess;
  if (!ok) {
    c->loop_exec = nullptr;
    cudaGetLastError();  // clear a refused capture or instantiation
  }
  cudaGraphDestroy(g);
  return ok;
}

// Drop the captured graphs (the step's and the decode loop's): they hold the
// weights' tensor maps and pointers and the options' kernel choices by value.
// An executable graph still in flight is freed once it completes.
void drop_graphs(dd_ctx* c) {
  if (c->exec) cudaGraphExecDestroy(c->exec);
  if (c->loop_exec) cudaGraphExecDestroy(c->loop_exec);
  c->exec = nullptr;
  c->loop_exec = nullptr;
  c->loop_tried = false;
}

dd_status check_ctx(dd_ctx* c) {
  if (!c) return fail(DD_ERR_INVALID_ARG, "ctx is NULL");
  if (!c->have_weights) return fail(DD_ERR_NOT_READY, "weights not set (call dd_init_weights)");
  int dev = -1;
  DD_CUDA(cudaGetDevice(&dev));
  if (dev != c->device) return fail(DD_ERR_INVALID_ARG, "current device %d is not the context's device %d", dev, c->device);
  return DD_OK;
}

}  // namespace

extern "C" {

const char* dd_status_string(dd_status s) {
  switch (s) {
    case DD_OK: return "ok";
    case DD_ERR_INVALID_ARG: return "invalid argument";
    case DD_ERR_CUDA: return "CUDA error";
    case DD_ERR_NOT_READY: return "not ready";
    case DD_ERR_STEP_LIMIT: return "step limit reached";
    case DD_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case DD_ERR_UNSUPPORTED: return "unsupported shape";
  }
  return "unknown status";
}

const char* dd_last_error(void) { return g_last_error.c_str(); }

dd_status dd_workspace_size(const dd_config* cfg, size_t* bytes) {
  dd_status s = check_config(cfg);
  if (s != DD_OK) return s;
  if (!bytes) return fail(DD_ERR_INVALID_ARG, "bytes is NULL");
  *bytes = make_layout(*cfg).total;
  return DD_OK;
}

dd_status dd_create(const dd_config* cfg, void* workspace, size_t workspace_bytes, dd_ctx** out) {
  dd_status s = check_config(cfg);
  if (s != DD_OK) return s;
  if (!out) return fail(DD_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (!workspace) return fail(DD_ERR_INVALID_ARG, "workspace is NULL");
  if (reinterpret_cast<uintptr_t>(workspace) % 256) return fail(DD_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  Layout L = make_layout(*cfg);
  if (workspace_bytes < L.total)
    return fail(DD_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes", workspace_bytes, L.total);
  if (!encode_fn()) return fail(DD_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  dd_ctx* c = new dd_ctx();
  c->cfg = *cfg;
  c->R = cfg->batch * cfg->block;
  c->G = cfg->n_q_heads / cfg->n_kv_heads;
  c->qkvw = (cfg->n_q_heads + 2 * cfg->n_kv_heads) * cfg->head_dim;
  c->HqD = cfg->n_q_heads * cfg->head_dim;
  c->L = L;
  c->ws = static_cast<uint8_t*>(workspace);
  c->timeout_ns = dd::kDefaultTimeoutNs;
  cudaError_t e = cudaGetDevice(&c->device);
  if (e == cudaSuccess) e = dd::prepare_kernels();
  if (e == cudaSuccess) e = cudaMemset(workspace, 0, L.total);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&c->cap_stream, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaHostAlloc(reinterpret_cast<void**>(&c->hpin), 32, cudaHostAllocDefault);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    dd_destroy(c);
    return fail(DD_ERR_CUDA, "dd_create: %s", cudaGetErrorString(e));
  }
  const dd_config& cf = *cfg;
  const uint64_t planes = (uint64_t)cf.n_layers * cf.batch * cf.n_kv_heads;
  bool ok = dd::make_map_3d(&c->m_kc, c->ws + L.kc, planes, L.alloc_ctx, L.alloc_ctx, cf.head_dim, 64) &&
            dd::make_map_3d(&c->m_vc, c->ws + L.vc, planes, L.alloc_ctx, L.alloc_ctx, cf.head_dim, 64) &&
            dd::make_map_3d(&c->m_kc128, c->ws + L.kc, planes, L.alloc_ctx, L.alloc_ctx, cf.head_dim, 128) &&
            dd::make_map_3d(&c->m_vc128, c->ws + L.vc, planes, L.alloc_ctx, L.alloc_ctx, cf.head_dim, 128) &&
            dd::make_map_2d(&c->m_y_b, c->ws + L.y, 2 * c->R, cf.hidden, L.p_qkv.box_rows_b, L.p_qkv.bk) &&
            dd::make_map_2d(&c->m_attn_b, c->ws + L.attn, 2 * c->R, c->HqD, L.p_o.box_rows_b, L.p_o.bk) &&
            dd::make_map_2d(&c->m_h_b, c->ws + L.hmid, 2 * c->R, cf.mlp, L.p_d.box_rows_b, L.p_d.bk) &&
            dd::make_map_2d(&c->m_y_a, c->ws + L.y, 2 * c->R, cf.hidden, 128) &&
            dd::make_map_2d(&c->m_yc_a, c->ws + L.yc, 2 * c->R, cf.hidden, 128) &&
            dd::make_map_q(&c->m_q, c->ws + L.qkv, 2 * c->R, c->qkvw, cf.n_q_heads, cf.head_dim, c->G, cf.block);
  if (!ok) {
    dd_destroy(c);
    return fail(DD_ERR_CUDA, "tensor map encoding failed for the workspace buffers");
  }
  // stacked query rows for the tcgen05 context kernel (head and remainder as
  // two rows of one M = 128 operand)
  if (kStackedContextKernel && L.p_attn.use_tc && dd::attention_tc_stacked_supported(c->G, cf.block)) {
    if (!dd::make_map_q_stacked(&c->m_q2, c->ws + L.qkv, c->R, c->qkvw, cf.n_q_heads, cf.head_dim, c->G, cf.block)) {
      dd_destroy(c);
      return fail(DD_ERR_CUDA, "tensor map encoding failed for the stacked query rows");
    }
    c->have_q2 = true;
  }
  // Fused linear layers (at most 128 activation rows, which the activation
  // maps above then hold in one box).
  if (c->R <= 128) {
    c->f_qkv = dd::plan_gemm_fused(dd::kOpQkv, c->R, c->qkvw, cf.hidden);
    c->f_o = dd::plan_gemm_fused(dd::kOpResidual, c->R, cf.hidden, c->HqD);
    c->f_gu = dd::plan_gemm_fused(dd::kOpSwiglu, c->R, 2 * cf.mlp, cf.hidden);
    c->f_d = dd::plan_gemm_fused(dd::kOpResidual, c->R, cf.hidden, cf.mlp);
    c->fused_ok = c->f_qkv.fused_op >= 0 && c->f_o.fused_op >= 0 && c->f_gu.fused_op >= 0 &&
                  c->f_d.fused_op >= 0 && L.p_qkv.BN == c->R && L.p_o.BN == c->R && L.p_d.BN == c->R &&
                  L.p_qkv.bk == 64 && L.p_qkv.cluster == 1;  // 64-wide K blocks, BN-row activation boxes
  }
  // Measured on the small decode workload the fused layers lose to the
  // separate reduce kernels inside the step graph, so they are opt-in.
  c->fused_on = false;
  c->compact_on = true;
  *out = c;
  return DD_OK;
}

void dd_destroy(dd_ctx* c) {
  if (!c) return;
  if (c->exec) cudaGraphExecDestroy(c->exec);
  if (c->loop_exec) cudaGraphExecDestroy(c->loop_exec);
  if (c->cap_stream) cudaStreamDestroy(c->cap_stream);
  if (c->hpin) cudaFreeHost(c->hpin);
  delete c;
}

dd_status dd_init_weights(dd_ctx* c, const dd_weights* w) {
  if (!c) return fail(DD_ERR_INVALID_ARG, "ctx is NULL");
  if (!w) return fail(DD_ERR_INVALID_ARG, "weights is NULL");
  const void* ptrs[] = {w->embed, w->pos, w->wqkv, w->wo, w->wgu, w->wd, w->g_attn, w->g_mlp, w->g_final, w->lm_head};
  const char* names[] = {"embed", "pos", "wqkv", "wo", "wgu", "wd", "g_attn", "g_mlp", "g_final", "lm_head"};
  for (int i = 0; i < 10; ++i) {
    if (!ptrs[i]) return fail(DD_ERR_INVALID_ARG, "weight '%s' is NULL", names[i]);
    if (reinterpret_cast<uintptr_t>(ptrs[i]) % 16) return fail(DD_ERR_INVALID_ARG, "weight '%s' is not 16-byte aligned", names[i]);
  }
  const dd_config& cf = c->cfg;
  const int H = cf.hidden, F = cf.mlp;
  c->m_wqkv.assign(cf.n_layers, CUtensorMap{});
  c->m_wo.assign(cf.n_layers, CUtensorMap{});
  c->m_wgu.assign(cf.n_layers, CUtensorMap{});
  c->m_wd.assign(cf.n_layers, CUtensorMap{});
  c->m_wgu64.assign(cf.n_layers, CUtensorMap{});
  bool ok = true;
  for (int l = 0; l < cf.n_layers && ok; ++l) {
    ok = dd::make_map_2d(&c->m_wqkv[l], (const uint8_t*)w->wqkv + (size_t)l * c->qkvw * H * 2, c->qkvw, H, 128, c->L.p_qkv.bk) &&
         dd::make_map_2d(&c->m_wo[l], (const uint8_t*)w->wo + (size_t)l * H * c->HqD * 2, H, c->HqD, 128, c->L.p_o.bk) &&
         dd::make_map_2d(&c->m_wgu[l], (const uint8_t*)w->wgu + (size_t)l * 2 * F * H * 2, 2 * F, H, 128, c->L.p_gu.bk) &&
         dd::make_map_2d(&c->m_wgu64[l], (const uint8_t*)w->wgu + (size_t)l * 2 * F * H * 2, 2 * F, H, 64) &&
         dd::make_map_2d(&c->m_wd[l], (const uint8_t*)w->wd + (size_t)l * H * F * 2, H, F, 128, c->L.p_d.bk);
  }
  ok = ok && dd::make_map_2d(&c->m_lm, w->lm_head, cf.vocab, H, c->L.p_lm.BN);
  if (!ok) return fail(DD_ERR_CUDA, "tensor map encoding failed for the weights");
  c->w = *w;
  c->have_weights = true;
  drop_graphs(c);  // both graphs captured the previous weights
  return DD_OK;
}

dd_status dd_set_context_kv(dd_ctx* c, const void* k, const void* v, int32_t t0, int32_t n, void* stream) {
  if (!c) return fail(DD_ERR_INVALID_ARG, "ctx is NULL");
  const dd_config& cf = c->cfg;
  if (t0 < 0 || n < 0 || (long long)t0 + n > cf.max_ctx)
    return fail(DD_ERR_INVALID_ARG, "need 0 <= t0, 0 <= n, t0+n <= max_ctx (t0=%d n=%d max_ctx=%d)", t0, n, cf.max_ctx);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (n > 0) {
    if (!k || !v) return fail(DD_ERR_INVALID_ARG, "k/v is NULL");
    const size_t row = (size_t)cf.head_dim * 2;
    const size_t planes = (size_t)cf.n_layers * cf.batch * cf.n_kv_heads;
    DD_CUDA(cudaMemcpy2DAsync(c->ws + c->L.kc + (size_t)t0 * row, (size_t)c->L.alloc_ctx * row, k, (size_t)n * row,
                              (size_t)n * row, planes, cudaMemcpyDefault, st));
    DD_CUDA(cudaMemcpy2DAsync(c->ws + c->L.vc + (size_t)t0 * row, (size_t)c->L.alloc_ctx * row, v, (size_t)n * row,
                              (size_t)n * row, planes, cudaMemcpyDefault, st));
  }
  DD_CUDA(dd::launch_set_int(small_ptr(c) + 2, t0 + n, st));
  c->ctx_len = t0 + n;
  return DD_OK;
}

dd_status dd_set_context_tower(dd_ctx* c, const dd_context_tower* t) {
  if (!c) return fail(DD_ERR_INVALID_ARG, "ctx is NULL");
  if (!t || !t->embed || !t->g || !t->wqkv || !t->wo || !t->g2 || !t->wkv)
    return fail(DD_ERR_INVALID_ARG, "context tower weights are NULL");
  const dd_config& cf = c->cfg;
  for (const void* ptr : {t->embed, t->g, t->wqkv, t->wo, t->g2, t->wkv})
    if (reinterpret_cast<uintptr_t>(ptr) % 16) return fail(DD_ERR_INVALID_ARG, "context tower weights must be 16-byte aligned");
  if (!encode_fn()) return fail(DD_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  const uint64_t W = (uint64_t)cf.n_kv_heads * cf.head_dim;
  const uint64_t n = (uint64_t)cf.n_layers * 2 * W;
  if (n % 128 || (3 * W) % 128)
    return fail(DD_ERR_UNSUPPORTED, "n_layers*2*n_kv_heads*head_dim and 3*n_kv_heads*head_dim must be multiples of 128");
  if (!dd::make_map_2d(&c->m_tower, t->wkv, n, cf.hidden, 128, c->L.p_tower.bk) ||
      !dd::make_map_2d(&c->m_tower_qkv, t->wqkv, 3 * W, cf.hidden, 128, c->L.p_tqkv.bk) ||
      !dd::make_map_2d(&c->m_tower_o, t->wo, cf.hidden, W, 128, c->L.p_to.bk) ||
      !dd::make_map_2d(&c->m_tower_a, c->ws + c->L.attn, 2 * c->R, W, c->L.p_to.box_rows_b, c->L.p_to.bk))
    return fail(DD_ERR_CUDA, "tensor map encoding failed for the context tower");
  c->tower = *t;
  return DD_OK;
}

dd_status dd_append_block(dd_ctx* c, const int32_t* tokens, void* stream) {
  dd_status s = check_ctx(c);
  if (s != DD_OK) return s;
  if (!c->tower.wkv) return fail(DD_ERR_NOT_READY, "no context tower (call dd_set_context_tower)");
  if (!tokens) return fail(DD_ERR_INVALID_ARG, "tokens is NULL");
  const dd_config& cf = c->cfg;
  if (c->ctx_len + cf.block > cf.max_ctx)
    return fail(DD_ERR_INVALID_ARG, "context %d + block %d exceeds max_ctx %d", c->ctx_len, cf.block, cf.max_ctx);
  DD_CUDA(dd::prepare_kernels());
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = c->ws;
  const Layout& L = c->L;
  const int R = c->R, H = cf.hidden, W = cf.n_kv_heads * cf.head_dim, N = cf.n_layers * 2 * W;
  int* small = small_ptr(c);
  float* x = at<float>(ws, L.x);
  float* part = at<float>(ws, L.part);
  // e = E_ctx[token] (x), y = RMSNorm(e) g
  DD_CUDA(dd::launch_tower_embed_norm(tokens, c->tower.embed, c->tower.g, x, ws + L.y, R, H, cf.vocab, cf.rms_eps,
                                      st));
  // q|k|v = y Wqkv^T (fp32, in the q|k|v activation buffer, which is large enough)
  dd::GemmOut o{};
  o.partial = part;
  o.rows_valid = R;
  o.ld = 3 * W;
  o.split_stride = (long long)R * 3 * W;
  float* tqkv = at<float>(ws, L.qkv);
  DD_CUDA(dd::launch_gemm(L.p_tqkv, c->m_tower_qkv, c->m_y_b, o, small + 1, c->timeout_ns, st));
  DD_CUDA(dd::launch_reduce_f32(part, dd::slot_plan(L.p_tqkv), o.split_stride, R, 3 * W, tqkv, st));
  // causal self-attention over each committed block -> a (head + remainder)
  DD_CUDA(dd::launch_tower_attention(tqkv, ws + L.attn, R, cf.block, cf.n_kv_heads, cf.head_dim, st));
  // x = e + a Wo^T ; y = RMSNorm(x) g2
  o.ld = H;
  o.split_stride = (long long)R * H;
  DD_CUDA(dd::launch_gemm(L.p_to, c->m_tower_o, c->m_tower_a, o, small + 1, c->timeout_ns, st));
  DD_CUDA(dd::launch_reduce_residual_norm(part, dd::slot_plan(L.p_to), o.split_stride, x, c->tower.g2, ws + L.y, R, H,
                                          cf.rms_eps, st));
  // K/V of every denoiser layer = y W_kv^T, appended at positions [T, T + S)
  o.ld = N;
  o.split_stride = (long long)R * N;
  DD_CUDA(dd::launch_gemm(L.p_tower, c->m_tower, c->m_y_b, o, small + 1, c->timeout_ns, st));
  DD_CUDA(dd::launch_reduce_kv_append(o.partial, dd::slot_plan(L.p_tower), o.split_stride, R, N, cf.block, cf.batch,
                                      cf.n_kv_heads, cf.head_dim, L.alloc_ctx, small + 2,
                                      reinterpret_cast<unsigned int*>(small + 5), ws + L.kc, ws + L.vc, st));
  c->ctx_len += cf.block;
  return DD_OK;
}

dd_status dd_denoise_step(dd_ctx* c, int32_t* tokens, uint32_t* mask, float gamma, int32_t mode,
                          int32_t* n_committed, void* stream) {
  dd_status s = check_ctx(c);
  if (s != DD_OK) return s;
  if (!tokens || !mask) return fail(DD_ERR_INVALID_ARG, "tokens/mask is NULL");
  if (!valid_mode(mode)) return fail(DD_ERR_INVALID_ARG, "bad mode %d", mode);
  if (!(gamma == gamma)) return fail(DD_ERR_INVALID_ARG, "gamma is NaN");
  s = ensure_graph(c);
  if (s != DD_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const dd_config& cf = c->cfg;
  uint8_t* ws = c->ws;
  DD_CUDA(cudaMemcpyAsync(ws + c->L.tok, tokens, (size_t)c->R * 4, cudaMemcpyDefault, st));
  DD_CUDA(cudaMemcpyAsync(ws + c->L.mask, mask, (size_t)cf.batch * 4, cudaMemcpyDefault, st));
  DD_CUDA(dd::launch_set_params(at<float>(ws, c->L.params), gamma, mode, st));
  DD_CUDA(cudaGraphLaunch(c->exec, st));
  DD_CUDA(cudaMemcpyAsync(tokens, ws + c->L.tok, (size_t)c->R * 4, cudaMemcpyDefault, st));
  DD_CUDA(cudaMemcpyAsync(mask, ws + c->L.mask, (size_t)cf.batch * 4, cudaMemcpyDefault, st));
  if (n_committed)
    DD_CUDA(cudaMemcpyAsync(n_committed, ws + c->L.ncommit, (size_t)cf.batch * 4, cudaMemcpyDefault, st));
  return DD_OK;
}

dd_status dd_denoise_step_probe(dd_ctx* c, int32_t* tokens, uint32_t* mask, float gamma, int32_t mode,
                                int32_t* n_committed, const dd_probe* probe, void* stream) {
  dd_status s = check_ctx(c);
  if (s != DD_OK) return s;
  if (!tokens || !mask) return fail(DD_ERR_INVALID_ARG, "tokens/mask is NULL");
  if (!valid_mode(mode)) return fail(DD_ERR_INVALID_ARG, "bad mode %d", mode);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const dd_config& cf = c->cfg;
  uint8_t* ws = c->ws;
  DD_CUDA(cudaMemcpyAsync(ws + c->L.tok, tokens, (size_t)c->R * 4, cudaMemcpyDeviceToDevice, st));
  DD_CUDA(cudaMemcpyAsync(ws + c->L.mask, mask, (size_t)cf.batch * 4, cudaMemcpyDeviceToDevice, st));
  DD_CUDA(dd::launch_set_params(at<float>(ws, c->L.params), gamma, mode, st));
  s = enqueue_step(c, st, probe);
  if (s != DD_OK) return s;
  DD_CUDA(cudaMemcpyAsync(tokens, ws + c->L.tok, (size_t)c->R * 4, cudaMemcpyDeviceToDevice, st));
  DD_CUDA(cudaMemcpyAsync(mask, ws + c->L.mask, (size_t)cf.batch * 4, cudaMemcpyDeviceToDevice, st));
  if (n_committed)
    DD_CUDA(cudaMemcpyAsync(n_committed, ws + c->L.ncommit, (size_t)cf.batch * 4, cudaMemcpyDeviceToDevice, st));
  return DD_OK;
}

// What a non-zero device status word means (ptx.cuh kStatus*).
const char* device_status_text(int v) {
  return v == dd::kStatusPairTmem ? "a pair of GEMM CTAs was given different tensor memory columns"
                                  : "a kernel's bounded wait expired";
}

dd_status dd_decode_block(dd_ctx* c, int32_t* tokens, float gamma, int32_t mode, int32_t max_steps,
                          int32_t* steps_out, void* stream) {
  dd_status s = check_ctx(c);
  if (s != DD_OK) return s;
  if (!tokens) return fail(DD_ERR_INVALID_ARG, "tokens is NULL");
  if (!valid_mode(mode)) return fail(DD_ERR_INVALID_ARG, "bad mode %d", mode);
  if (!(gamma == gamma)) return fail(DD_ERR_INVALID_ARG, "gamma is NaN");
  s = ensure_graph(c);
  if (s != DD_OK) return s;
  const dd_config& cf = c->cfg;
  if (max_steps <= 0) max_steps = 4 * cf.block;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = c->ws;
  DD_CUDA(dd::launch_init_block(at<int32_t>(ws, c->L.tok), at<uint32_t>(ws, c->L.mask), cf.batch, cf.block, cf.vocab, st));
  DD_CUDA(dd::launch_set_params(at<float>(ws, c->L.params), gamma, mode, st));
  DD_CUDA(dd::launch_loop_init(small_ptr(c), max_steps, st));
  int steps = 0;
  bool done = false;
  if (ensure_loop_graph(c)) {
    // device-side loop: one graph launch and one read-back per block
    DD_CUDA(cudaGraphLaunch(c->loop_exec, st));
    DD_CUDA(cudaMemcpyAsync(c->hpin, small_ptr(c), 20, cudaMemcpyDeviceToHost, st));
    DD_CUDA(cudaMemcpyAsync(tokens, ws + c->L.tok, (size_t)c->R * 4, cudaMemcpyDefault, st));
    DD_CUDA(cudaStreamSynchronize(st));
    steps = c->hpin[3];
    if (steps_out) *steps_out = steps;
    if (c->hpin[1] != 0) return fail(DD_ERR_DEVICE_TIMEOUT, "%s during step %d", device_status_text(c->hpin[1]), steps);
    if (c->hpin[0] != 0) return fail(DD_ERR_STEP_LIMIT, "%d steps without filling the block", max_steps);
    return DD_OK;
  }
  while (steps < max_steps) {
    DD_CUDA(cudaGraphLaunch(c->exec, st));
    ++steps;
    DD_CUDA(cudaMemcpyAsync(c->hpin, small_ptr(c), 8, cudaMemcpyDeviceToHost, st));
    DD_CUDA(cudaStreamSynchronize(st));
    if (c->hpin[1] != 0) {
      if (steps_out) *steps_out = steps;
      return fail(DD_ERR_DEVICE_TIMEOUT, "%s during step %d", device_status_text(c->hpin[1]), steps);
    }
    if (c->hpin[0] == 0) {
      done = true;
      break;
    }
  }
  DD_CUDA(cudaMemcpyAsync(tokens, ws + c->L.tok, (size_t)c->R * 4, cudaMemcpyDefault, st));
  DD_CUDA(cudaStreamSynchronize(st));  // host `tokens` hold the ids on return, as on the graph path
  if (steps_out) *steps_out = steps;
  if (!done) return fail(DD_ERR_STEP_LIMIT, "%d steps without filling the block", max_steps);
  return DD_OK;
}

dd_status dd_device_status(dd_ctx* c, void* stream) {
  if (!c) return fail(DD_ERR_INVALID_ARG, "ctx is NULL");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  DD_CUDA(cudaMemcpyAsync(c->hpin, small_ptr(c), 8, cudaMemcpyDeviceToHost, st));
  DD_CUDA(cudaStreamSynchronize(st));
  if (c->hpin[1] != 0) {
    const int v = c->hpin[1];
    DD_CUDA(cudaMemsetAsync(small_ptr(c) + 1, 0, 4, st));
    DD_CUDA(cudaStreamSynchronize(st));
    return fail(DD_ERR_DEVICE_TIMEOUT, "%s", device_status_text(v));
  }
  return DD_OK;
}

dd_status dd_step_launch_count(dd_ctx* c, int32_t* n) {
  dd_status s = check_ctx(c);
  if (s != DD_OK) return s;
  if (!n) return fail(DD_ERR_INVALID_ARG, "n is NULL");
  s = ensure_graph(c);
  if (s != DD_OK) return s;
  *n = c->step_launches + (ensure_loop_graph(c) ? 1 : 0);
  return DD_OK;
}

dd_status dd_set_option(dd_ctx* c, int32_t option, int32_t value) {
  if (!c) return fail(DD_ERR_INVALID_ARG, "ctx is NULL");
  if (option != DD_OPT_FUSED_REDUCE && option != DD_OPT_COMPACT_SEQUENCES)
    return fail(DD_ERR_INVALID_ARG, "option %d cannot be set", option);
  if (value != 0 && value != 1) return fail(DD_ERR_INVALID_ARG, "option %d takes 0 or 1 (got %d)", option, value);
  if (option == DD_OPT_FUSED_REDUCE && value && !c->fused_ok)
    return fail(DD_ERR_UNSUPPORTED, "the fused linear layers are not available for this shape or device");
  bool& flag = option == DD_OPT_FUSED_REDUCE ? c->fused_on : c->compact_on;
  if ((value != 0) != flag) {
    // the captured graphs hold the other path
    DD_CUDA(cudaDeviceSynchronize());
    drop_graphs(c);
    flag = value != 0;
  }
  return DD_OK;
}

dd_status dd_get_option(dd_ctx* c, int32_t option, int32_t* value) {
  if (!c) return fail(DD_ERR_INVALID_ARG, "ctx is NULL");
  if (!value) return fail(DD_ERR_INVALID_ARG, "value is NULL");
  const dd::GemmPlan* fp[] = {&c->f_qkv, &c->f_o, &c->f_gu, &c->f_d};
  switch (option) {
    case DD_OPT_FUSED_REDUCE: *value = c->fused_on ? 1 : 0; return DD_OK;
    case DD_OPT_COMPACT_SEQUENCES: *value = c->compact_on ? 1 : 0; return DD_OK;
    case DD_OPT_FUSED_SPLITS_QKV:
    case DD_OPT_FUSED_SPLITS_O:
    case DD_OPT_FUSED_SPLITS_GATE_UP:
    case DD_OPT_FUSED_SPLITS_DOWN: {
      const dd::GemmPlan& p = *fp[option - DD_OPT_FUSED_SPLITS_QKV];
      *value = c->fused_ok ? p.splits : 0;
      return DD_OK;
    }
    case DD_OPT_FUSED_GRID_QKV:
    case DD_OPT_FUSED_GRID_O:
    case DD_OPT_FUSED_GRID_GATE_UP:
    case DD_OPT_FUSED_GRID_DOWN: {
      const dd::GemmPlan& p = *fp[option - DD_OPT_FUSED_GRID_QKV];
      *value = c->fused_ok ? p.grid : 0;
      return DD_OK;
    }
  }
  return fail(DD_ERR_INVALID_ARG, "unknown option %d", option);
}

dd_status dd_profile_step(dd_ctx* c, int32_t* tokens, uint32_t* mask, float gamma, int32_t mode, float* times_ms,
                          int32_t* kinds, int32_t cap, int32_t* n, void* stream) {
  dd_status s = check_ctx(c);
  if (s != DD_OK) return s;
  if (!tokens || !mask || !times_ms || !kinds || !n || cap < 1) return fail(DD_ERR_INVALID_ARG, "bad profile arguments");
  if (!valid_mode(mode)) return fail(DD_ERR_INVALID_ARG, "bad mode %d", mode);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const dd_config& cf = c->cfg;
  uint8_t* ws = c->ws;
  std::vector<cudaEvent_t> ev(cap + 1);
  for (auto& e : ev) DD_CUDA(cudaEventCreate(&e));
  DD_CUDA(cudaMemcpyAsync(ws + c->L.tok, tokens, (size_t)c->R * 4, cudaMemcpyDefault, st));
  DD_CUDA(cudaMemcpyAsync(ws + c->L.mask, mask, (size_t)cf.batch * 4, cudaMemcpyDefault, st));
  DD_CUDA(dd::launch_set_params(at<float>(ws, c->L.params), gamma, mode, st));
  Marker mk{st, ev.data(), kinds, cap};
  DD_CUDA(cudaEventRecord(ev[0], st));
  s = enqueue_step(c, st, nullptr, &mk);
  if (s == DD_OK) {
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) s = fail(DD_ERR_CUDA, "profile step: %s", cudaGetErrorString(e));
  }
  const int m = mk.n < cap ? mk.n : cap;
  for (int i = 0; s == DD_OK && i < m; ++i) {
    cudaError_t e = cudaEventElapsedTime(&times_ms[i], ev[i], ev[i + 1]);
    if (e != cudaSuccess) s = fail(DD_ERR_CUDA, "event timing: %s", cudaGetErrorString(e));
  }
  for (auto& e : ev) cudaEventDestroy(e);
  if (s != DD_OK) return s;
  *n = m;
  DD_CUDA(cudaMemcpyAsync(tokens, ws + c->L.tok, (size_t)c->R * 4, cudaMemcpyDefault, st));
  DD_CUDA(cudaMemcpyAsync(mask, ws + c->L.mask, (size_t)cf.batch * 4, cudaMemcpyDefault, st));
  return DD_OK;
}

// ----------------------------------------------------------- single kernels

static dd_status attn_check(const dd_attn_problem* p) {
  if (!p) return fail(DD_ERR_INVALID_ARG, "problem is NULL");
  if (p->batch < 1 || p->block < 1 || p->block > 32) return fail(DD_ERR_INVALID_ARG, "bad batch/block");
  if (p->head_dim != 64 && p->head_dim != 128) return fail(DD_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  if (p->n_q_heads < 1 || p->n_kv_heads < 1 || p->n_q_heads % p->n_kv_heads)
    return fail(DD_ERR_INVALID_ARG, "n_kv_heads must divide n_q_heads");
  const int G = p->n_q_heads / p->n_kv_heads;
  if ((G * p->block) % 16 || G * p->block > 128)
    return fail(DD_ERR_UNSUPPORTED, "(n_q_heads/n_kv_heads)*block must be a multiple of 16 and <= 128");
  if (p->ctx_len < 0 || p->ctx_stride < p->ctx_len || p->ctx_stride < 1)
    return fail(DD_ERR_INVALID_ARG, "need 0 <= ctx_len <= ctx_stride, ctx_stride >= 1");
  return DD_OK;
}

static size_t attn_ws_bytes(const dd_attn_problem* p, dd::AttnPlan* plan) {
  // the tcgen05 path streams 128-position boxes: it needs ctx_stride >= 128
  *plan = dd::plan_attention(p->batch, p->block, p->n_q_heads, p->n_kv_heads, p->head_dim, p->ctx_len,
                             p->ctx_stride >= 128);
  return 256 + dd::attention_partial_bytes(*plan, p->batch, p->n_kv_heads);
}

dd_status dd_block_attention_workspace_size(const dd_attn_problem* p, size_t* bytes) {
  dd_status s = attn_check(p);
  if (s != DD_OK) return s;
  if (!bytes) return fail(DD_ERR_INVALID_ARG, "bytes is NULL");
  dd::AttnPlan plan;
  *bytes = attn_ws_bytes(p, &plan);
  return DD_OK;
}

dd_status dd_block_attention(const dd_attn_problem* p, void* stream) {
  dd_status s = attn_check(p);
  if (s != DD_OK) return s;
  if (!p->qkv || !p->k_ctx || !p->v_ctx || !p->out || !p->workspace)
    return fail(DD_ERR_INVALID_ARG, "null pointer in attention problem");
  dd::AttnPlan plan;
  const size_t need = attn_ws_bytes(p, &plan);
  if (p->workspace_bytes < need) return fail(DD_ERR_INVALID_ARG, "workspace too small: %zu < %zu", p->workspace_bytes, need);
  if (reinterpret_cast<uintptr_t>(p->workspace) % 256) return fail(DD_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  if (!encode_fn()) return fail(DD_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  DD_CUDA(dd::prepare_kernels());
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(p->workspace);
  CUtensorMap mk, mv, mk128, mv128;
  const uint64_t planes = (uint64_t)p->batch * p->n_kv_heads;
  // rows beyond ctx_len read as zero, whatever the caller's buffer holds there
  const uint64_t ext = p->ctx_len > 0 ? (uint64_t)p->ctx_len : 1;
  if (!dd::make_map_3d(&mk, p->k_ctx, planes, ext, p->ctx_stride, p->head_dim, 64) ||
      !dd::make_map_3d(&mv, p->v_ctx, planes, ext, p->ctx_stride, p->head_dim, 64) ||
      !dd::make_map_3d(&mk128, p->k_ctx, planes, ext, p->ctx_stride, p->head_dim, 128) ||
      !dd::make_map_3d(&mv128, p->v_ctx, planes, ext, p->ctx_stride, p->head_dim, 128))
    return fail(DD_ERR_CUDA, "tensor map encoding failed for k_ctx/v_ctx");
  int* small = reinterpret_cast<int*>(ws);  // [0] status (the caller may read it), [1] ctx_len
  DD_CUDA(cudaMemsetAsync(small, 0, 4, st));
  DD_CUDA(dd::launch_set_int(small + 1, p->ctx_len, st));
  dd::AttnArgs a{};
  a.qkv = p->qkv;
  a.ld_qkv = (p->n_q_heads + 2 * p->n_kv_heads) * p->head_dim;
  a.B = p->batch;
  a.S = p->block;
  a.Hq = p->n_q_heads;
  a.Hkv = p->n_kv_heads;
  a.G = p->n_q_heads / p->n_kv_heads;
  a.ctx_len = small + 1;
  a.z0 = 0;
  a.out = p->out;
  a.ld_out = p->n_q_heads * p->head_dim;
  a.part_o = reinterpret_cast<float*>(ws + 256);
  a.part_ml = reinterpret_cast<float2*>(
      ws + 256 + align_up((size_t)p->batch * p->n_kv_heads * plan.n_splits * plan.rows * p->head_dim * 4, 16));
  a.scale_log2 = 1.4426950408889634f / sqrtf((float)p->head_dim);
  a.status = small;
  a.timeout_ns = dd::kDefaultTimeoutNs;
  a.max_pair_splits = p->batch * p->n_kv_heads * plan.n_splits;
  CUtensorMap mq;
  if (!dd::make_map_q(&mq, p->qkv, (uint64_t)p->batch * p->block, a.ld_qkv, p->n_q_heads, p->head_dim, a.G, p->block))
    return fail(DD_ERR_CUDA, "tensor map encoding failed for qkv");
  DD_CUDA(dd::launch_attention(plan, a, mk, mv, mk128, mv128, mq, st));
  DD_CUDA(dd::launch_attention_combine(plan, a, st));
  return DD_OK;
}

dd_status dd_lmhead_select_workspace_size(int32_t rows, int32_t hidden, int32_t vocab, size_t* bytes) {
  if (rows < 1 || hidden < 64 || hidden % 64 || vocab < 256 || vocab % 256)
    return fail(DD_ERR_UNSUPPORTED, "need rows >= 1, hidden %% 64 == 0, vocab %% 256 == 0");
  if (!bytes) return fail(DD_ERR_INVALID_ARG, "bytes is NULL");
  const size_t n = (size_t)(vocab / 256) * rows * 4;
  *bytes = 256 + 3 * align_up(n, 256);
  return DD_OK;
}

dd_status dd_lmhead_select(int32_t rows, int32_t hidden, int32_t vocab, const void* x, const void* w, float* conf,
                           int32_t* arg, void* workspace, size_t workspace_bytes, void* stream) {
  size_t need = 0;
  dd_status s = dd_lmhead_select_workspace_size(rows, hidden, vocab, &need);
  if (s != DD_OK) return s;
  if (!x || !w || !conf || !arg || !workspace) return fail(DD_ERR_INVALID_ARG, "null pointer");
  if (workspace_bytes < need) return fail(DD_ERR_INVALID_ARG, "workspace too small: %zu < %zu", workspace_bytes, need);
  if (reinterpret_cast<uintptr_t>(workspace) % 256) return fail(DD_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  if (!encode_fn()) return fail(DD_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  DD_CUDA(dd::prepare_kernels());
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  dd::GemmPlan p = dd::plan_gemm(dd::kEpiSelect, rows, vocab, hidden);
  CUtensorMap mx, mw;
  if (!dd::make_map_2d(&mx, x, rows, hidden, 128) || !dd::make_map_2d(&mw, w, vocab, hidden, p.BN))
    return fail(DD_ERR_CUDA, "tensor map encoding failed");
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t n = align_up((size_t)p.n_tiles * rows * 4, 256);
  dd::GemmOut o{};
  o.rows_valid = rows;
  o.sel_m = reinterpret_cast<float*>(ws + 256);
  o.sel_s = reinterpret_cast<float*>(ws + 256 + n);
  o.sel_a = reinterpret_cast<int*>(ws + 256 + 2 * n);
  DD_CUDA(cudaMemsetAsync(ws, 0, 4, st));  // the call's status word
  DD_CUDA(dd::launch_gemm(p, mx, mw, o, reinterpret_cast<int*>(ws), dd::kDefaultTimeoutNs, st));
  DD_CUDA(dd::launch_select_combine(o.sel_m, o.sel_s, o.sel_a, p.n_tiles, rows, conf, arg, st));
  return DD_OK;
}

dd_status dd_gemm_workspace_size(int32_t rows, int32_t n, int32_t k, size_t* bytes) {
  if (rows < 16 || rows % 16 || n < 128 || n % 128 || k < 64 || k % 64)
    return fail(DD_ERR_UNSUPPORTED, "need rows %% 16 == 0, n %% 128 == 0, k %% 64 == 0");
  if (!bytes) return fail(DD_ERR_INVALID_ARG, "bytes is NULL");
  dd::GemmPlan p = dd::plan_gemm(dd::kEpiPartial, rows, n, k);
  *bytes = 256 + (size_t)p.splits * rows * n * 4;
  return DD_OK;
}

dd_status dd_gemm_plan_query(int32_t rows, int32_t n, int32_t k, int32_t split_act, int32_t* out, int32_t n_out) {
  if (rows < 16 || rows % 16 || n < 128 || n % 128 || k < 64 || k % 64)
    return fail(DD_ERR_UNSUPPORTED, "need rows %% 16 == 0, n %% 128 == 0, k %% 64 == 0");
  if (!out || n_out < 0) return fail(DD_ERR_INVALID_ARG, "out is NULL or n_out < 0");
  const dd::GemmPlan p = dd::plan_gemm(dd::kEpiPartial, rows, n, k, split_act ? 1 : 0);
  const int32_t v[DD_GEMM_PLAN_FIELDS] = {p.grid,     p.cluster,  p.cg,           p.bk,       p.BN,
                                          p.m_tiles,  p.n_tiles,  p.kb_total,     p.splits,   p.kb_per_split,
                                          p.sk_units, p.sk_total, p.stages,       p.smem_bytes};
  for (int i = 0; i < n_out && i < DD_GEMM_PLAN_FIELDS; ++i) out[i] = v[i];
  return DD_OK;
}

dd_status dd_gemm(int32_t rows, int32_t n, int32_t k, const void* x, const void* w, float* y, void* workspace,
                  size_t workspace_bytes, void* stream) {
  size_t need = 0;
  dd_status s = dd_gemm_workspace_size(rows, n, k, &need);
  if (s != DD_OK) return s;
  if (!x || !w || !y || !workspace) return fail(DD_ERR_INVALID_ARG, "null pointer");
  if (workspace_bytes < need) return fail(DD_ERR_INVALID_ARG, "workspace too small: %zu < %zu", workspace_bytes, need);
  if (reinterpret_cast<uintptr_t>(workspace) % 256) return fail(DD_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  if (!encode_fn()) return fail(DD_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  DD_CUDA(dd::prepare_kernels());
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  dd::GemmPlan p = dd::plan_gemm(dd::kEpiPartial, rows, n, k);
  CUtensorMap mw, mx;
  if (!dd::make_map_2d(&mw, w, n, k, 128, p.bk) || !dd::make_map_2d(&mx, x, rows, k, p.box_rows_b, p.bk))
    return fail(DD_ERR_CUDA, "tensor map encoding failed");
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  dd::GemmOut o{};
  o.partial = reinterpret_cast<float*>(ws + 256);
  o.split_stride = (long long)rows * n;
  o.ld = n;
  o.rows_valid = rows;
  DD_CUDA(cudaMemsetAsync(ws, 0, 4, st));  // the call's status word
  DD_CUDA(dd::launch_gemm(p, mw, mx, o, reinterpret_cast<int*>(ws), dd::kDefaultTimeoutNs, st));
  DD_CUDA(dd::launch_reduce_f32(o.partial, dd::slot_plan(p), o.split_stride, rows, n, y, st));
  return DD_OK;
}

dd_status dd_commit(int32_t batch, int32_t block, const float* conf, const int32_t* arg, int32_t* tokens,
                    uint32_t* mask, float gamma, int32_t mode, int32_t* n_committed, int32_t* remaining,
                    void* stream) {
  if (batch < 1 || block < 1 || block > 32) return fail(DD_ERR_INVALID_ARG, "bad batch/block");
  if (!conf || !arg || !tokens || !mask || !remaining) return fail(DD_ERR_INVALID_ARG, "null pointer");
  if (!valid_mode(mode)) return fail(DD_ERR_INVALID_ARG, "bad mode %d", mode);
  DD_CUDA(dd::launch_commit(conf, arg, tokens, mask, nullptr, gamma, mode, n_committed, remaining, batch, block,
                            static_cast<cudaStream_t>(stream)));
  return DD_OK;
}

dd_status dd_test_wait_timeout(int32_t timeout_us, int32_t* status, void* stream) {
  if (timeout_us < 1 || timeout_us > 10000000) return fail(DD_ERR_INVALID_ARG, "timeout_us must be in [1, 1e7]");
  if (!status) return fail(DD_ERR_INVALID_ARG, "status is NULL");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  DD_CUDA(cudaMemsetAsync(status, 0, 4, st));
  DD_CUDA(dd::launch_wait_forever_bounded(status, (uint64_t)timeout_us * 1000ull, st));
  int h = 0;
  DD_CUDA(cudaMemcpyAsync(&h, status, 4, cudaMemcpyDeviceToHost, st));
  DD_CUDA(cudaStreamSynchronize(st));
  if (h != 0) return fail(DD_ERR_DEVICE_TIMEOUT, "bounded wait expired after %d us", timeout_us);
  return DD_OK;
}

}  // extern "C"
