// Context part of the block attention on the tcgen05 tensor cores (head dim
// 128, 64 query rows per (sequence, kv head)).  Each split writes a partial
// (o, m, l); the merge kernel adds the block keys and combines them all
// (TwoTower article, "技術/ビジネス面": one softmax over the context and the
// block).
//
// Per 128-key tile:
//   S[64 q][128 keys] = Q[64][128] . K_tile[128][128]^T     (M=64, K-major A and B)
//   O[64 q][128 d]    = P[64][128 keys] . V_tile[128][128]    (M=64, K-major A, MN-major B)
// With M = 64 the accumulator rows 16w..16w+15 live in TMEM lanes 32w..32w+15,
// and the 16x256b load shape hands them to warp w in the m16n8 fragment
// layout (row = 16w + lane/4 (+8), column = 8*rep + 2*(lane%4) (+1)).  So each
// softmax warp owns 16 query rows: row maxima and sums are in-thread plus two
// quad shuffles, and P (a bf16 head and a bf16 remainder) goes to shared
// memory with stmatrix in the swizzled K-major layout the PV MMA reads.
// O accumulates in TMEM over all tiles of a work item (two buffers, taken by
// the non-empty items in turn).  P is taken against a reference maximum per
// query that moves only when a tile's maximum exceeds it by more than 2^8;
// then the softmax warp rescales its O rows in TMEM between the previous PV
// and the next (the scheme published with FlashAttention-4), and otherwise
// P <= 2^8.  Each item's O is read out once.
//
// Roles (192 threads): warp 0 streams Q (double-buffered, one per work item)
// and the K and V tiles with TMA (two slots each; K released after QK^T, V
// after PV), warp 1 owns TMEM and issues the MMAs, warps 2-5 run the softmax
// and write each item's partial.  Every mbarrier wait is bounded.
#include <math.h>

#include "kernels.h"
#include "ptx.cuh"

namespace dd {

namespace {

constexpr int kKT = 128;                 // keys per tile (MMA N of QK^T, K of PV)
constexpr int kNQ = 64;                  // query rows (MMA M)
constexpr int kD = 128;                  // head dim
constexpr int kBox = kKT * 128;          // one [128 keys][64 d] TMA box: 16 KB
constexpr int kKV = 2 * kBox;            // K or V tile: 32 KB
constexpr float kRescaleLog2 = 8.f;      // O rescaled in TMEM when a row maximum grows by more than 2^8
constexpr int kRowBox = kNQ * 128;       // one [64 rows][64 cols] box: 8 KB
constexpr int kQ = 2 * kRowBox;          // Q head or remainder: 16 KB
constexpr int kP = 2 * kRowBox;          // P head or remainder [64][128 keys]: 16 KB
constexpr int kThreads = 192;
constexpr int kOffK = 0;                 // 2 K slots
constexpr int kOffV = 2 * kKV;           // 2 V slots
constexpr int kOffQ = 4 * kKV;           // 2 Q buffers, each a head then a remainder
constexpr int kOffPh = kOffQ + 4 * kQ;
constexpr int kOffPl = kOffPh + kP;
constexpr int kOffBar = kOffPl + kP;
constexpr int kNumBars = 23;
constexpr int kSmemBytes = 1024 + kOffBar + kNumBars * 8 + 16;
constexpr uint32_t kTmemCols = 512;      // S x2 (128 cols each), O x2 (128 cols each)

__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Offset of element (row, col) of a [rows][...] tile stored as 64-column
// boxes of `rows` x 128 bytes with the 128-byte swizzle.
__device__ __forceinline__ uint32_t swz(int rows, int r, int col) {
  return (col >> 6) * rows * 128 + r * 128 + ((((col & 63) >> 3) ^ (r & 7)) << 4) + (col & 7) * 2;
}

// 64 fp32 values of this warp's 16 accumulator rows (M = 64 layout), columns
// [col, col + 128): register i holds row lane/4 + 8*((i%4)/2), column
// 8*(i/4) + 2*(lane%4) + (i%2).
__device__ __forceinline__ void tmem_ld_frag(uint32_t taddr, float (&v)[64]) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]),
        "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]),
        "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]),
        "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]),
        "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

// The inverse of tmem_ld_frag: write the 64 values back to the same 16 rows x
// 128 columns (same register order), then wait for the stores.
__device__ __forceinline__ void tmem_st_frag(uint32_t taddr, const float (&v)[64]) {
  uint32_t r[64];
#pragma unroll
  for (int i = 0; i < 64; ++i) r[i] = __float_as_uint(v[i]);
  asm volatile(
      "tcgen05.st.sync.aligned.16x256b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(r[0]),"r"(r[1]),"r"(r[2]),"r"(r[3]),"r"(r[4]),"r"(r[5]),"r"(r[6]),"r"(r[7]),"r"(r[8]),"r"(r[9]),"r"(r[10]),"r"(r[11]),"r"(r[12]),"r"(r[13]),"r"(r[14]),"r"(r[15]),"r"(r[16]),"r"(r[17]),"r"(r[18]),"r"(r[19]),"r"(r[20]),"r"(r[21]),"r"(r[22]),"r"(r[23]),"r"(r[24]),"r"(r[25]),"r"(r[26]),"r"(r[27]),"r"(r[28]),"r"(r[29]),"r"(r[30]),"r"(r[31]),"r"(r[32]),"r"(r[33]),"r"(r[34]),"r"(r[35]),"r"(r[36]),"r"(r[37]),"r"(r[38]),"r"(r[39]),"r"(r[40]),"r"(r[41]),"r"(r[42]),"r"(r[43]),"r"(r[44]),"r"(r[45]),"r"(r[46]),"r"(r[47]),"r"(r[48]),"r"(r[49]),"r"(r[50]),"r"(r[51]),"r"(r[52]),"r"(r[53]),"r"(r[54]),"r"(r[55]),"r"(r[56]),"r"(r[57]),"r"(r[58]),"r"(r[59]),"r"(r[60]),"r"(r[61]),"r"(r[62]),"r"(r[63])
      : "memory");
}

__device__ __forceinline__ void stmatrix_x4(uint32_t saddr, uint32_t r0, uint32_t r1, uint32_t r2, uint32_t r3) {
  asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1, %2, %3, %4};" ::"r"(saddr), "r"(r0), "r"(r1),
               "r"(r2), "r"(r3)
               : "memory");
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Persistent: CTA c takes the work items c, c + gridDim.x, ... where item w
// is context split w % n_ctx of the (sequence, kv head) pair w / n_ctx.  The
// producer streams the next item's Q and K/V tiles while the softmax warps
// still fold and write the previous item, so an SM pays the pipeline fill
// once rather than once per item.  Q arrives by TMA from the q|k|v rows with
// the box {64 dims, G heads, S positions}, i.e. in row order i * G + g; the
// partials are written in the order g * S + i that the merge kernels read.
template <bool SPLITQ>
__global__ void __launch_bounds__(kThreads, 1)
    k_attn_ctx_tc(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                  const __grid_constant__ CUtensorMap map_q, const AttnArgs a, int n_ctx_plan, int n_items_max) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* kfull = bars + 0;
  uint64_t* kempty = bars + 2;
  uint64_t* vfull = bars + 4;
  uint64_t* vempty = bars + 6;
  uint64_t* sfull = bars + 8;
  uint64_t* sfree = bars + 10;
  uint64_t* pfull = bars + 12;
  uint64_t* pfree = bars + 13;
  uint64_t* ofull = bars + 14;
  uint64_t* ofree = bars + 16;
  uint64_t* drain = bars + 18;
  uint64_t* qfull = bars + 19;
  uint64_t* qempty = bars + 21;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = warp_id(), lane = lane_id();
  const int T = *a.ctx_len;
  // With active-sequence compaction the pairs are those of the active
  // sequences; the record was written by the step's first kernel, at least
  // three launches upstream, so it is complete before this kernel starts
  // (read through L2, since this happens before the launch's wait).
  const int n_ctx = attn_launch_splits(a, n_ctx_plan, T);
  const int n_items = a.cmp ? __ldcg(a.cmp + 1) * a.Hkv * n_ctx : n_items_max;
  const int ntiles_all = (T + kKT - 1) / kKT;
  const int per = (ntiles_all + n_ctx - 1) / n_ctx;
  const int R = a.B * a.S;
  // item w -> (split, kv head, sequence (compacted), first tile, tile count)
  auto item = [&](int w, int& split, int& kvh, int& b, int& tile0, int& nt) {
    split = w % n_ctx;
    const int pair = w / n_ctx;
    kvh = pair % a.Hkv;
    b = pair / a.Hkv;
    tile0 = split * per;
    nt = max(0, min(ntiles_all, tile0 + per) - tile0);
  };

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&kfull[i], 1);
      mbar_init(&kempty[i], 1);
      mbar_init(&vfull[i], 1);
      mbar_init(&vempty[i], 1);
      mbar_init(&sfull[i], 1);
      mbar_init(&sfree[i], 4);
      mbar_init(&ofull[i], 1);
      mbar_init(&ofree[i], 4);
      mbar_init(&qfull[i], 1);
      mbar_init(&qempty[i], 1);
    }
    mbar_init(pfull, 4);
    mbar_init(pfree, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&map_k);
    tma_prefetch_desc(&map_v);
    tma_prefetch_desc(&map_q);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t t_s = tmem;             // S buffers at columns 0 and 128
  const uint32_t t_o = tmem + 256;       // O buffers at columns 256 and 384

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      auto load_kv = [&](int g, int key0, int z) {
        const int s = g & 1;
        const uint32_t ph = (g >> 1) & 1;
        if (!mbar_wait_bounded(&kempty[s], ph ^ 1, a.timeout_ns, abort_flag, a.status)) return false;
        mbar_arrive_expect_tx(&kfull[s], kKV);
        tma_load_3d(smem + kOffK + s * kKV, &map_k, &kfull[s], 0, key0, z);
        tma_load_3d(smem + kOffK + s * kKV + kBox, &map_k, &kfull[s], 64, key0, z);
        if (!mbar_wait_bounded(&vempty[s], ph ^ 1, a.timeout_ns, abort_flag, a.status)) return false;
        mbar_arrive_expect_tx(&vfull[s], kKV);
        tma_load_3d(smem + kOffV + s * kKV, &map_v, &vfull[s], 0, key0, z);
        tma_load_3d(smem + kOffV + s * kKV + kBox, &map_v, &vfull[s], 64, key0, z);
        return true;
      };
      // The context K/V do not depend on the preceding kernel: the first
      // item's first two tiles go out before waiting for it (programmatic
      // dependent launch); q does, so its load waits.
      // the context cache plane of (compacted sequence b, kv head)
      auto plane = [&](int b, int kvh) { return a.z0 + (a.cmp ? __ldcg(a.cmp + 2 + b) : b) * a.Hkv + kvh; };
      int split, kvh, b, tile0, nt;
      int pre = 0;
      bool ok = true;
      if ((int)blockIdx.x < n_items) {
        item(blockIdx.x, split, kvh, b, tile0, nt);
        const int z = plane(b, kvh);
        for (; pre < min(nt, 2) && ok; ++pre) ok = load_kv(pre, (tile0 + pre) * kKT, z);
      }
      pdl_wait();
      pdl_launch_dependents();
      int g = 0;
      for (int w = blockIdx.x, it = 0; w < n_items && ok; w += gridDim.x, ++it) {
        item(w, split, kvh, b, tile0, nt);
        const int qb = it & 1;
        if (!mbar_wait_bounded(&qempty[qb], ((it >> 1) & 1) ^ 1, a.timeout_ns, abort_flag, a.status)) break;
        uint8_t* q = smem + kOffQ + qb * 2 * kQ;
        mbar_arrive_expect_tx(&qfull[qb], (SPLITQ ? 2 : 1) * kQ);
        tma_load_3d(q, &map_q, &qfull[qb], 0, kvh * a.G, b * a.S);
        tma_load_3d(q + kRowBox, &map_q, &qfull[qb], 64, kvh * a.G, b * a.S);
        if (SPLITQ) {
          tma_load_3d(q + kQ, &map_q, &qfull[qb], 0, kvh * a.G, R + b * a.S);
          tma_load_3d(q + kQ + kRowBox, &map_q, &qfull[qb], 64, kvh * a.G, R + b * a.S);
        }
        const int z = plane(b, kvh);
        for (int t = 0; t < nt && ok; ++t, ++g)
          if (g >= pre) ok = load_kv(g, (tile0 + t) * kKT, z);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      const uint32_t idesc_qk = idesc_bf16_f32(kNQ, kKT);
      const uint32_t idesc_pv = idesc_bf16_f32(kNQ, kD) | (1u << 16);  // B (V) MN-major
      const uint32_t p_h = smem_u32(smem + kOffPh), p_l = smem_u32(smem + kOffPl);
      bool ok = true;
      // O of an item accumulates over its tiles in one of two TMEM buffers
      // (the non-empty items alternate); PV of tile u (global tile index) of
      // the item with non-empty index oi, first/last: its place in the item.
      auto issue_pv = [&](int u, int oi, bool first, bool last) {
        const int s = u & 1;
        const uint32_t ph = (u >> 1) & 1;
        const int ob = oi & 1;
        if (!mbar_wait_bounded(&vfull[s], ph, a.timeout_ns, abort_flag, a.status)) return false;
        if (!mbar_wait_bounded(pfull, u & 1, a.timeout_ns, abort_flag, a.status)) return false;
        // the buffer's previous item has been read out
        if (first && !mbar_wait_bounded(&ofree[ob], ((oi >> 1) & 1) ^ 1, a.timeout_ns, abort_flag, a.status))
          return false;
        tc_fence_after();
        const uint32_t vb = smem_u32(smem + kOffV + s * kKV);
#pragma unroll
        for (int j = 0; j < kKT / 16; ++j) {
          const uint32_t aoff = (j >> 2) * kRowBox + (j & 3) * 32;
          tc_mma_bf16(t_o + ob * kD, desc_sw128(p_h + aoff, 0, 1024), desc_sw128(vb + j * 2048, kBox, 1024),
                      idesc_pv, (j > 0 || !first) ? 1u : 0u);
        }
#pragma unroll
        for (int j = 0; j < kKT / 16; ++j) {
          const uint32_t aoff = (j >> 2) * kRowBox + (j & 3) * 32;
          tc_mma_bf16(t_o + ob * kD, desc_sw128(p_l + aoff, 0, 1024), desc_sw128(vb + j * 2048, kBox, 1024),
                      idesc_pv, 1u);
        }
        if (last) tc_commit(&ofull[ob]);
        tc_commit(&vempty[s]);
        tc_commit(pfree);
        return true;
      };
      int g = 0;
      int oi = -1;                                       // non-empty items so far, minus one
      int p_oi = 0;                                      // the pending PV's item and place in it
      bool p_first = false, p_last = false;
      for (int w = blockIdx.x, it = 0; w < n_items && ok; w += gridDim.x, ++it) {
        int split, kvh, b, tile0, nt;
        item(w, split, kvh, b, tile0, nt);
        if (nt >= 1) ++oi;
        const int qb = it & 1;
        if (!mbar_wait_bounded(&qfull[qb], (it >> 1) & 1, a.timeout_ns, abort_flag, a.status)) { ok = false; break; }
        const uint32_t qh = smem_u32(smem + kOffQ + qb * 2 * kQ), ql = qh + kQ;
        for (int t = 0; t < nt; ++t, ++g) {
          const int s = g & 1;
          const uint32_t ph = (g >> 1) & 1;
          if (!mbar_wait_bounded(&kfull[s], ph, a.timeout_ns, abort_flag, a.status)) { ok = false; break; }
          if (!mbar_wait_bounded(&sfree[s], ph ^ 1, a.timeout_ns, abort_flag, a.status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t kb = smem_u32(smem + kOffK + s * kKV);
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk) {
            const uint32_t off = (kk & 3) * 32;
            tc_mma_bf16(t_s + s * kKT, desc_sw128(qh + (kk >> 2) * kRowBox + off, 0, 1024),
                        desc_sw128(kb + (kk >> 2) * kBox + off, 0, 1024), idesc_qk, kk > 0 ? 1u : 0u);
          }
          if (SPLITQ) {
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk) {
              const uint32_t off = (kk & 3) * 32;
              tc_mma_bf16(t_s + s * kKT, desc_sw128(ql + (kk >> 2) * kRowBox + off, 0, 1024),
                          desc_sw128(kb + (kk >> 2) * kBox + off, 0, 1024), idesc_qk, 1u);
            }
          }
          tc_commit(&sfull[s]);
          tc_commit(&kempty[s]);
          if (g >= 1 && !issue_pv(g - 1, p_oi, p_first, p_last)) { ok = false; break; }
          p_oi = oi;
          p_first = t == 0;
          p_last = t == nt - 1;
        }
        tc_commit(&qempty[qb]);  // this item's QK^T products are all issued
      }
      if (ok && g >= 1) issue_pv(g - 1, p_oi, p_first, p_last);
      tc_commit(drain);
      volatile int no_abort = 0;
      mbar_wait_bounded(drain, 0, a.timeout_ns, &no_abort, a.status);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------- softmax
    const int q4 = warp & 3;                        // TMEM lane quarter -> rows 16*q4 .. 16*q4+15
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const int r0 = 16 * q4 + (lane >> 2);           // the two rows this thread holds (order i * G + g)
    const int r1 = r0 + 8;
    const int cq = 2 * (lane & 3);                  // column offset inside each 8-column block
    const float c = a.scale_log2;
    // stmatrix row address of this lane: matrix mi = lane/8 covers rows
    // 16*q4 + 8*(mi&1) + lane%8 and columns +8*(mi>>1) of each 16-key group
    const int st_row = 16 * q4 + 8 * ((lane >> 3) & 1) + (lane & 7);
    const int st_colh = 8 * (lane >> 4);
    // partial rows in the order g * S + i
    const int pr0 = (r0 % a.G) * a.S + r0 / a.G;
    const int pr1 = (r1 % a.G) * a.S + r1 / a.G;
    bool ok = true;
    int g = 0;
    int oi = -1;  // non-empty items so far, minus one (their O buffers alternate)
    for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x) {
      int split, kvh, b, tile0, nt;
      item(w, split, kvh, b, tile0, nt);
      if (nt >= 1) ++oi;
      const int ob = oi & 1;
      // O accumulates in TMEM over the item's tiles against a reference
      // maximum per query that moves only when a tile's maximum exceeds it by
      // more than kRescaleLog2 (then the warp rescales its O rows in TMEM once
      // the previous PV has completed); read out once per item.
      float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
      for (int t = 0; t < nt; ++t, ++g) {
        const int s = g & 1;
        bool wt = true;
        if (lane == 0) wt = mbar_wait_bounded(&sfull[s], (g >> 1) & 1, a.timeout_ns, abort_flag, a.status);
        wt = __shfl_sync(0xffffffffu, wt ? 1 : 0, 0) != 0;
        if (!wt) { ok = false; break; }
        tc_fence_after();
        float v[64];
        tmem_ld_frag(t_s + s * kKT + lane_off, v);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sfree[s]);
        const int kbase = (tile0 + t) * kKT;
        if (kbase + kKT > T) {  // tail tile: keys >= T do not exist
#pragma unroll
          for (int j = 0; j < 64; ++j) {
            const int key = kbase + 8 * (j >> 2) + cq + (j & 1);
            if (key >= T) v[j] = -INFINITY;
          }
        }
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int j = 0; j < 64; j += 4) {
          mx0 = fmaxf(mx0, fmaxf(v[j], v[j + 1]));
          mx1 = fmaxf(mx1, fmaxf(v[j + 2], v[j + 3]));
        }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        // move the reference (the first tile sets it; O then starts afresh)
        float a0 = 1.f, a1 = 1.f;
        if (mx0 * c > m0 + kRescaleLog2) {
          a0 = m0 == -INFINITY ? 0.f : ex2(m0 - mx0 * c);
          m0 = mx0 * c;
        }
        if (mx1 * c > m1 + kRescaleLog2) {
          a1 = m1 == -INFINITY ? 0.f : ex2(m1 - mx1 * c);
          m1 = mx1 * c;
        }
        const bool rescale = t > 0 && __any_sync(0xffffffffu, a0 != 1.f || a1 != 1.f);
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int j = 0; j < 64; j += 4) {
          v[j] = ex2(fmaf(v[j], c, -m0));
          v[j + 1] = ex2(fmaf(v[j + 1], c, -m0));
          v[j + 2] = ex2(fmaf(v[j + 2], c, -m1));
          v[j + 3] = ex2(fmaf(v[j + 3], c, -m1));
          s0 += v[j] + v[j + 1];
          s1 += v[j + 2] + v[j + 3];
        }
        s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
        s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
        s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
        s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
        l0 = l0 * a0 + s0;
        l1 = l1 * a1 + s1;
        // P (head, remainder) -> shared memory, once the previous PV is done;
        // with a moved reference, O is rescaled first
        if (g >= 1) {
          bool pw = true;
          if (lane == 0) pw = mbar_wait_bounded(pfree, (g - 1) & 1, a.timeout_ns, abort_flag, a.status);
          pw = __shfl_sync(0xffffffffu, pw ? 1 : 0, 0) != 0;
          if (!pw) { ok = false; break; }
        }
        if (rescale) {
          tc_fence_after();
          float h[64];
          tmem_ld_frag(t_o + ob * kD + lane_off, h);
#pragma unroll
          for (int j = 0; j < 64; ++j) h[j] *= (j & 2) ? a1 : a0;
          tmem_st_frag(t_o + ob * kD + lane_off, h);
          tc_fence_before();
        }
#pragma unroll
        for (int gg = 0; gg < kKT / 16; ++gg) {
          // 16-key group gg: fragment reps 2gg (keys 16gg..16gg+7) and 2gg+1 (16gg+8..)
          uint32_t h0, l0p, h1, l1p, h2, l2p, h3, l3p;
          split_bf16(v[8 * gg + 0], v[8 * gg + 1], h0, l0p);   // rows 0-7,  keys 16gg + cq
          split_bf16(v[8 * gg + 2], v[8 * gg + 3], h1, l1p);   // rows 8-15, keys 16gg + cq
          split_bf16(v[8 * gg + 4], v[8 * gg + 5], h2, l2p);   // rows 0-7,  keys 16gg + 8 + cq
          split_bf16(v[8 * gg + 6], v[8 * gg + 7], h3, l3p);   // rows 8-15, keys 16gg + 8 + cq
          const uint32_t off = swz(kNQ, st_row, 16 * gg + st_colh);
          stmatrix_x4(smem_u32(smem + kOffPh) + off, h0, h1, h2, h3);
          stmatrix_x4(smem_u32(smem + kOffPl) + off, l0p, l1p, l2p, l3p);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(pfull);
      }
      // the item's O once its last PV has completed
      float o[64];                                  // O rows r0/r1 in fragment order
#pragma unroll
      for (int j = 0; j < 64; ++j) o[j] = 0.f;
      if (ok && nt >= 1) {
        bool wt = true;
        if (lane == 0) wt = mbar_wait_bounded(&ofull[ob], (oi >> 1) & 1, a.timeout_ns, abort_flag, a.status);
        wt = __shfl_sync(0xffffffffu, wt ? 1 : 0, 0) != 0;
        if (!wt) { ok = false; }
        else {
          tc_fence_after();
          tmem_ld_frag(t_o + ob * kD + lane_off, o);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&ofree[ob]);
        }
      }
      // partial slot `split`: o (unnormalised, [q][d]), (m, l) per q
      const long long prow = ((long long)(b * a.Hkv + kvh) * n_ctx + split) * kNQ;
#pragma unroll
      for (int rep = 0; rep < 16; ++rep) {
        const int d = 8 * rep + cq;
        *reinterpret_cast<float2*>(a.part_o + (prow + pr0) * kD + d) = make_float2(o[4 * rep], o[4 * rep + 1]);
        *reinterpret_cast<float2*>(a.part_o + (prow + pr1) * kD + d) = make_float2(o[4 * rep + 2], o[4 * rep + 3]);
      }
      if ((lane & 3) == 0) {
        a.part_ml[prow + pr0] = make_float2(m0, l0);
        a.part_ml[prow + pr1] = make_float2(m1, l1);
      }
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Stacked form, for split activations (q as a bf16 head plus a bf16
// remainder).  An M = 64 MMA occupies the tensor core as long as an M = 128
// one, so instead of two M = 64 products per K step (head and remainder) the
// head and the remainder rows of the 64 queries form one M = 128 operand and
// their product rows are added afterwards:
//   S'[128][128 keys] = Q'[128][128] . K_tile^T      O'[128][128 d] = P'[128][128 keys] . V_tile
// Row order: 16-row groups, each holding 8 consecutive queries (query order
// i * G + g) as 8 head rows then the same queries' 8 remainder rows, so row
// 16k + j is the head and 16k + 8 + j the remainder of query 8k + j.  Q'
// comes from the q|k|v rows as one 5D TMA box {64 dims, G heads, 8/G
// positions, 2 parts, S*G/8 position pairs} (the part dimension strides from
// the head rows to the remainder rows); P' is written in the same order.
// The 16x256b TMEM load hands a thread the rows r and r + 8 of its lane
// group, i.e. the head and the remainder of one query, so the sum is one
// in-thread add, and after it every register holds what the M = 64 form's
// load would: rows q and q + 8 of the query order, 32 columns each.  Per
// 128-key tile this is 16 MMAs instead of 32.
template <int G>
__global__ void __launch_bounds__(kThreads, 1)
    k_attn_ctx_stk(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                   const __grid_constant__ CUtensorMap map_q2, const AttnArgs a, int n_ctx_plan, int n_items_max) {
  static_assert(G == 2 || G == 4 || G == 8, "G must be 2, 4 or 8");
  constexpr int Q8 = 8 / G;         // block positions per 8-query group
  constexpr int kAtom = 128 * 128;  // [128 rows][64 cols] bf16, 128-byte swizzle: 16 KB
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* kfull = bars + 0;
  uint64_t* kempty = bars + 2;
  uint64_t* vfull = bars + 4;
  uint64_t* vempty = bars + 6;
  uint64_t* sfull = bars + 8;
  uint64_t* sfree = bars + 10;
  uint64_t* pfull = bars + 12;
  uint64_t* pfree = bars + 13;
  uint64_t* ofull = bars + 14;
  uint64_t* ofree = bars + 16;
  uint64_t* drain = bars + 18;
  uint64_t* qfull = bars + 19;
  uint64_t* qempty = bars + 21;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = warp_id(), lane = lane_id();
  const int S = a.S;  // S * G == 64
  const int T = *a.ctx_len;
  // the active sequences' record is written by the step's first kernel, at
  // least three launches upstream, so it is complete before this kernel starts
  // (read through L2, since this happens before the launch's wait)
  const int n_ctx = attn_launch_splits(a, n_ctx_plan, T);
  const int n_items = a.cmp ? __ldcg(a.cmp + 1) * a.Hkv * n_ctx : n_items_max;
  const int ntiles_all = (T + kKT - 1) / kKT;
  const int per = (ntiles_all + n_ctx - 1) / n_ctx;
  auto item = [&](int w, int& split, int& kvh, int& b, int& tile0, int& nt) {
    split = w % n_ctx;
    const int pair = w / n_ctx;
    kvh = pair % a.Hkv;
    b = pair / a.Hkv;
    tile0 = split * per;
    nt = max(0, min(ntiles_all, tile0 + per) - tile0);
  };

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&kfull[i], 1);
      mbar_init(&kempty[i], 1);
      mbar_init(&vfull[i], 1);
      mbar_init(&vempty[i], 1);
      mbar_init(&sfull[i], 1);
      mbar_init(&sfree[i], 4);
      mbar_init(&ofull[i], 1);
      mbar_init(&ofree[i], 4);
      mbar_init(&qfull[i], 1);
      mbar_init(&qempty[i], 1);
    }
    mbar_init(pfull, 4);
    mbar_init(pfree, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&map_k);
    tma_prefetch_desc(&map_v);
    tma_prefetch_desc(&map_q2);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t t_s = tmem;        // S' buffers at columns 0 and 128
  const uint32_t t_o = tmem + 256;  // O' buffers at columns 256 and 384

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      auto load_kv = [&](int g, int key0, int z) {
        const int s = g & 1;
        const uint32_t ph = (g >> 1) & 1;
        if (!mbar_wait_bounded(&kempty[s], ph ^ 1, a.timeout_ns, abort_flag, a.status)) return false;
        mbar_arrive_expect_tx(&kfull[s], kKV);
        tma_load_3d(smem + kOffK + s * kKV, &map_k, &kfull[s], 0, key0, z);
        tma_load_3d(smem + kOffK + s * kKV + kBox, &map_k, &kfull[s], 64, key0, z);
        if (!mbar_wait_bounded(&vempty[s], ph ^ 1, a.timeout_ns, abort_flag, a.status)) return false;
        mbar_arrive_expect_tx(&vfull[s], kKV);
        tma_load_3d(smem + kOffV + s * kKV, &map_v, &vfull[s], 0, key0, z);
        tma_load_3d(smem + kOffV + s * kKV + kBox, &map_v, &vfull[s], 64, key0, z);
        return true;
      };
      auto plane = [&](int b, int kvh) { return a.z0 + (a.cmp ? __ldcg(a.cmp + 2 + b) : b) * a.Hkv + kvh; };
      int split, kvh, b, tile0, nt;
      int pre = 0;
      bool ok = true;
      // context K/V do not depend on the preceding kernel: the first item's
      // first two tiles go out before waiting for it; q does, so it waits
      if ((int)blockIdx.x < n_items) {
        item(blockIdx.x, split, kvh, b, tile0, nt);
        const int z = plane(b, kvh);
        for (; pre < min(nt, 2) && ok; ++pre) ok = load_kv(pre, (tile0 + pre) * kKT, z);
      }
      pdl_wait();
      pdl_launch_dependents();
      int g = 0;
      for (int w = blockIdx.x, it = 0; w < n_items && ok; w += gridDim.x, ++it) {
        item(w, split, kvh, b, tile0, nt);
        const int qb = it & 1;
        if (!mbar_wait_bounded(&qempty[qb], ((it >> 1) & 1) ^ 1, a.timeout_ns, abort_flag, a.status)) break;
        uint8_t* q = smem + kOffQ + qb * 2 * kAtom;
        mbar_arrive_expect_tx(&qfull[qb], 2 * kAtom);
        tma_load_5d(q, &map_q2, &qfull[qb], 0, kvh * G, 0, 0, b * S / Q8);
        tma_load_5d(q + kAtom, &map_q2, &qfull[qb], 64, kvh * G, 0, 0, b * S / Q8);
        const int z = plane(b, kvh);
        for (int t = 0; t < nt && ok; ++t, ++g)
          if (g >= pre) ok = load_kv(g, (tile0 + t) * kKT, z);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      const uint32_t idesc_qk = idesc_bf16_f32(128, kKT);
      const uint32_t idesc_pv = idesc_bf16_f32(128, kD) | (1u << 16);  // B (V) MN-major
      const uint32_t p_base = smem_u32(smem + kOffPh);                  // P' [128 rows][128 keys]
      bool ok = true;
      // O' of an item accumulates over its tiles in one of two TMEM buffers
      // (the non-empty items alternate); PV of tile u (global tile index) of
      // the item with non-empty index oi, first/last: its place in the item.
      auto issue_pv = [&](int u, int oi, bool first, bool last) {
        const int s = u & 1;
        const uint32_t ph = (u >> 1) & 1;
        const int ob = oi & 1;
        if (!mbar_wait_bounded(&vfull[s], ph, a.timeout_ns, abort_flag, a.status)) return false;
        if (!mbar_wait_bounded(pfull, u & 1, a.timeout_ns, abort_flag, a.status)) return false;
        // the buffer's previous item has been read out
        if (first && !mbar_wait_bounded(&ofree[ob], ((oi >> 1) & 1) ^ 1, a.timeout_ns, abort_flag, a.status))
          return false;
        tc_fence_after();
        const uint32_t vb = smem_u32(smem + kOffV + s * kKV);
#pragma unroll
        for (int j = 0; j < kKT / 16; ++j) {
          const uint32_t aoff = (j >> 2) * kAtom + (j & 3) * 32;
          tc_mma_bf16(t_o + ob * kD, desc_sw128(p_base + aoff, 0, 1024), desc_sw128(vb + j * 2048, kBox, 1024),
                      idesc_pv, (j > 0 || !first) ? 1u : 0u);
        }
        if (last) tc_commit(&ofull[ob]);
        tc_commit(&vempty[s]);
        tc_commit(pfree);
        return true;
      };
      int g = 0;
      int oi = -1;                                       // non-empty items so far, minus one
      int p_oi = 0;                                      // the pending PV's item and place in it
      bool p_first = false, p_last = false;
      for (int w = blockIdx.x, it = 0; w < n_items && ok; w += gridDim.x, ++it) {
        int split, kvh, b, tile0, nt;
        item(w, split, kvh, b, tile0, nt);
        if (nt >= 1) ++oi;
        const int qb = it & 1;
        if (!mbar_wait_bounded(&qfull[qb], (it >> 1) & 1, a.timeout_ns, abort_flag, a.status)) { ok = false; break; }
        const uint32_t qa = smem_u32(smem + kOffQ + qb * 2 * kAtom);
        for (int t = 0; t < nt; ++t, ++g) {
          const int s = g & 1;
          const uint32_t ph = (g >> 1) & 1;
          if (!mbar_wait_bounded(&kfull[s], ph, a.timeout_ns, abort_flag, a.status)) { ok = false; break; }
          if (!mbar_wait_bounded(&sfree[s], ph ^ 1, a.timeout_ns, abort_flag, a.status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t kb = smem_u32(smem + kOffK + s * kKV);
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk) {
            const uint32_t off = (kk & 3) * 32;
            tc_mma_bf16(t_s + s * kKT, desc_sw128(qa + (kk >> 2) * kAtom + off, 0, 1024),
                        desc_sw128(kb + (kk >> 2) * kBox + off, 0, 1024), idesc_qk, kk > 0 ? 1u : 0u);
          }
          tc_commit(&sfull[s]);
          tc_commit(&kempty[s]);
          if (g >= 1 && !issue_pv(g - 1, p_oi, p_first, p_last)) { ok = false; break; }
          p_oi = oi;
          p_first = t == 0;
          p_last = t == nt - 1;
        }
        tc_commit(&qempty[qb]);  // this item's QK^T products are all issued
      }
      if (ok && g >= 1) issue_pv(g - 1, p_oi, p_first, p_last);
      tc_commit(drain);
      volatile int no_abort = 0;
      mbar_wait_bounded(drain, 0, a.timeout_ns, &no_abort, a.status);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------- softmax
    const int q4 = warp & 3;                         // TMEM lane quarter: rows 32*q4 .. 32*q4 + 31
    const uint32_t lane_a = (uint32_t)(q4 * 32) << 16;        // 16-row group 2*q4
    const uint32_t lane_b = (uint32_t)(q4 * 32 + 16) << 16;   // 16-row group 2*q4 + 1
    // the two queries (order i * G + g) whose rows this thread holds, as in
    // the M = 64 form: r0 from group 2*q4, r1 = r0 + 8 from group 2*q4 + 1
    const int r0 = 16 * q4 + (lane >> 2);
    const int r1 = r0 + 8;
    const int cq = 2 * (lane & 3);                   // column offset inside each 8-column block
    const float c = a.scale_log2;
    // stmatrix row addresses of P': matrix mi = lane/8 holds rows 32*q4 + 16*(mi&1) + lane%8 (heads;
    // the remainders 8 rows further) and columns +8*(mi>>1) of each 16-key group
    const int st_row = 32 * q4 + 16 * ((lane >> 3) & 1) + (lane & 7);
    const int st_colh = 8 * (lane >> 4);
    const int pr0 = (r0 % G) * S + r0 / G;           // partial rows in the order g * S + i
    const int pr1 = (r1 % G) * S + r1 / G;
    // the head + remainder sums of a 128-column TMEM block in the M = 64
    // fragment order: register 4k + e holds row r0 (e < 2) or r1 (e >= 2),
    // column 8k + cq + (e & 1)
    auto load_sum = [&](uint32_t taddr, float (&v)[64]) {
      float h[64];
      tmem_ld_frag(taddr + lane_a, h);  // rows: group 2q4 head (e < 2) and remainder (e >= 2)
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        v[4 * k] = h[4 * k] + h[4 * k + 2];
        v[4 * k + 1] = h[4 * k + 1] + h[4 * k + 3];
      }
      tmem_ld_frag(taddr + lane_b, h);  // group 2q4 + 1
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        v[4 * k + 2] = h[4 * k] + h[4 * k + 2];
        v[4 * k + 3] = h[4 * k + 1] + h[4 * k + 3];
      }
    };
    bool ok = true;
    int g = 0;
    int oi = -1;  // non-empty items so far, minus one (their O' buffers alternate)
    for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x) {
      int split, kvh, b, tile0, nt;
      item(w, split, kvh, b, tile0, nt);
      if (nt >= 1) ++oi;
      const int ob = oi & 1;
      // O' accumulates in TMEM over the item's tiles.  P is taken against a
      // reference maximum per query (base-2 units) that moves only when a
      // tile's maximum exceeds it by more than kRescaleLog2: then, once the
      // previous PV has completed, the warp rescales its O' rows in TMEM.
      // Otherwise P <= 2^kRescaleLog2, well inside fp32 and the split P.
      float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
      for (int t = 0; t < nt; ++t, ++g) {
        const int s = g & 1;
        bool wt = true;
        if (lane == 0) wt = mbar_wait_bounded(&sfull[s], (g >> 1) & 1, a.timeout_ns, abort_flag, a.status);
        wt = __shfl_sync(0xffffffffu, wt ? 1 : 0, 0) != 0;
        if (!wt) { ok = false; break; }
        tc_fence_after();
        float v[64];
        load_sum(t_s + s * kKT, v);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sfree[s]);
        const int kbase = (tile0 + t) * kKT;
        if (kbase + kKT > T) {  // tail tile: keys >= T do not exist
#pragma unroll
          for (int j = 0; j < 64; ++j) {
            const int key = kbase + 8 * (j >> 2) + cq + (j & 1);
            if (key >= T) v[j] = -INFINITY;
          }
        }
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int j = 0; j < 64; j += 4) {
          mx0 = fmaxf(mx0, fmaxf(v[j], v[j + 1]));
          mx1 = fmaxf(mx1, fmaxf(v[j + 2], v[j + 3]));
        }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        // move the reference (the first tile sets it; O' then starts afresh)
        float a0 = 1.f, a1 = 1.f;
        if (mx0 * c > m0 + kRescaleLog2) {
          a0 = m0 == -INFINITY ? 0.f : ex2(m0 - mx0 * c);
          m0 = mx0 * c;
        }
        if (mx1 * c > m1 + kRescaleLog2) {
          a1 = m1 == -INFINITY ? 0.f : ex2(m1 - mx1 * c);
          m1 = mx1 * c;
        }
        const bool rescale = t > 0 && __any_sync(0xffffffffu, a0 != 1.f || a1 != 1.f);
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int j = 0; j < 64; j += 4) {
          v[j] = ex2(fmaf(v[j], c, -m0));
          v[j + 1] = ex2(fmaf(v[j + 1], c, -m0));
          v[j + 2] = ex2(fmaf(v[j + 2], c, -m1));
          v[j + 3] = ex2(fmaf(v[j + 3], c, -m1));
          s0 += v[j] + v[j + 1];
          s1 += v[j + 2] + v[j + 3];
        }
        s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
        s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
        s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
        s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
        l0 = l0 * a0 + s0;
        l1 = l1 * a1 + s1;
        // P' (heads, and remainders 8 rows further) once the previous PV is
        // done; with a moved reference, O' is rescaled first
        if (g >= 1) {
          bool pw = true;
          if (lane == 0) pw = mbar_wait_bounded(pfree, (g - 1) & 1, a.timeout_ns, abort_flag, a.status);
          pw = __shfl_sync(0xffffffffu, pw ? 1 : 0, 0) != 0;
          if (!pw) { ok = false; break; }
        }
        if (rescale) {
          tc_fence_after();
          float h[64];
          const uint32_t to = t_o + ob * kD;
          tmem_ld_frag(to + lane_a, h);  // head and remainder rows of query r0
#pragma unroll
          for (int j = 0; j < 64; ++j) h[j] *= a0;
          tmem_st_frag(to + lane_a, h);
          tmem_ld_frag(to + lane_b, h);  // ... of query r1
#pragma unroll
          for (int j = 0; j < 64; ++j) h[j] *= a1;
          tmem_st_frag(to + lane_b, h);
          tc_fence_before();
        }
        const uint32_t pbase = smem_u32(smem + kOffPh);
#pragma unroll
        for (int gg = 0; gg < kKT / 16; ++gg) {
          // 16-key group gg: fragment reps 2gg (keys 16gg..16gg+7) and 2gg+1 (16gg+8..)
          uint32_t h0, l0p, h1, l1p, h2, l2p, h3, l3p;
          split_bf16(v[8 * gg + 0], v[8 * gg + 1], h0, l0p);   // query r0, keys 16gg + cq
          split_bf16(v[8 * gg + 2], v[8 * gg + 3], h1, l1p);   // query r1, keys 16gg + cq
          split_bf16(v[8 * gg + 4], v[8 * gg + 5], h2, l2p);   // query r0, keys 16gg + 8 + cq
          split_bf16(v[8 * gg + 6], v[8 * gg + 7], h3, l3p);   // query r1, keys 16gg + 8 + cq
          stmatrix_x4(pbase + swz(128, st_row, 16 * gg + st_colh), h0, h1, h2, h3);
          stmatrix_x4(pbase + swz(128, st_row + 8, 16 * gg + st_colh), l0p, l1p, l2p, l3p);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(pfull);
      }
      // the item's O' once its last PV has completed
      float o[64];                                  // O rows r0/r1 in fragment order
#pragma unroll
      for (int j = 0; j < 64; ++j) o[j] = 0.f;
      if (ok && nt >= 1) {
        bool wt = true;
        if (lane == 0) wt = mbar_wait_bounded(&ofull[ob], (oi >> 1) & 1, a.timeout_ns, abort_flag, a.status);
        wt = __shfl_sync(0xffffffffu, wt ? 1 : 0, 0) != 0;
        if (!wt) { ok = false; }
        else {
          tc_fence_after();
          load_sum(t_o + ob * kD, o);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&ofree[ob]);
        }
      }
      // partial slot `split`: o (unnormalised, [q][d]), (m, l) per q
      const long long prow = ((long long)(b * a.Hkv + kvh) * n_ctx + split) * kNQ;
#pragma unroll
      for (int rep = 0; rep < 16; ++rep) {
        const int d = 8 * rep + cq;
        *reinterpret_cast<float2*>(a.part_o + (prow + pr0) * kD + d) = make_float2(o[4 * rep], o[4 * rep + 1]);
        *reinterpret_cast<float2*>(a.part_o + (prow + pr1) * kD + d) = make_float2(o[4 * rep + 2], o[4 * rep + 3]);
      }
      if ((lane & 3) == 0) {
        a.part_ml[prow + pr0] = make_float2(m0, l0);
        a.part_ml[prow + pr1] = make_float2(m1, l1);
      }
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

bool attention_tc_supported(int D, int rows) { return D == kD && rows == kNQ; }

int attention_tc_splits(int B, int Hkv, int max_ctx) {
  return attn_ctx_splits(B * Hkv, (max_ctx + kKT - 1) / kKT, 32);
}


bool attention_tc_stacked_supported(int G, int S) { return (G == 2 || G == 4 || G == 8) && G * S == kNQ; }

cudaError_t launch_attention_tc(const AttnArgs& a, int n_ctx, const CUtensorMap& map_k128,
                                const CUtensorMap& map_v128, const CUtensorMap& map_q, cudaStream_t st,
                                const CUtensorMap* map_q2) {
  const int items = a.B * a.Hkv * n_ctx;
  const int grid = items < kNumSMs ? items : kNumSMs;
  if (a.split && map_q2 && attention_tc_stacked_supported(a.G, a.S)) {
    switch (a.G) {
      case 2: return launch_k(k_attn_ctx_stk<2>, grid, kThreads, kSmemBytes, st, map_k128, map_v128, *map_q2, a, n_ctx, items);
      case 4: return launch_k(k_attn_ctx_stk<4>, grid, kThreads, kSmemBytes, st, map_k128, map_v128, *map_q2, a, n_ctx, items);
      default: return launch_k(k_attn_ctx_stk<8>, grid, kThreads, kSmemBytes, st, map_k128, map_v128, *map_q2, a, n_ctx, items);
    }
  }
  if (a.split)
    return launch_k(k_attn_ctx_tc<true>, grid, kThreads, kSmemBytes, st, map_k128, map_v128, map_q, a, n_ctx, items);
  return launch_k(k_attn_ctx_tc<false>, grid, kThreads, kSmemBytes, st, map_k128, map_v128, map_q, a, n_ctx, items);
}

cudaError_t prepare_attention_tc_kernels() {
  const void* fns[] = {(const void*)k_attn_ctx_tc<true>, (const void*)k_attn_ctx_tc<false>,
                       (const void*)k_attn_ctx_stk<2>,   (const void*)k_attn_ctx_stk<4>,
                       (const void*)k_attn_ctx_stk<8>};
  cudaError_t e = cudaSuccess;
  for (const void* f : fns)
    if (e == cudaSuccess) e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  return e;
}

}  // namespace dd
