// Block attention of the denoising tower (TwoTower article, "技術/ビジネス面":
// bidirectional attention inside the block plus cross-attention to the frozen
// context tower's state), as one softmax per query over
// [ctx_len context keys | S block keys], scale 1/sqrt(D), no mask.
//
// One CTA serves one (sequence, kv head, context split): all G query heads
// that share the kv head (G*S query rows, 16 per compute warp) read each
// context K/V tile once.  A producer warp streams the tiles from HBM with
// TMA (3D tensor map over the [planes][positions][D] cache, 128-byte
// swizzle) into a ring of shared-memory stages; the compute warps run
// QK^T and PV on the tensor cores (mma.sync m16n8k16, bf16 in, fp32 out)
// with an online softmax in base 2 (quad shuffles for the row max/sum).
// The S block keys/values come from the packed q|k|v activation rows and
// are staged once, by split 0.  With several splits per (sequence, kv head)
// each CTA writes an unnormalised partial (o, m, l) and a combine kernel
// merges them.
//
// Precision: P is multiplied as a bf16 head plus a bf16 remainder.  With
// SPLIT, the activations (q and the block k/v) also arrive as head +
// remainder rows and the remainder products are added (q_lo K, q K_blk_lo,
// P V_blk_lo), and the output is written as head + remainder rows, so the
// result tracks an fp32 computation to ~1e-5 relative.
#include <math.h>

#include "kernels.h"
#include "ptx.cuh"

namespace dd {

namespace {

constexpr int kKT = 64;      // context keys per tile
constexpr int kKTB = 32;     // block-key tile (S <= 32)

// Byte offset of element (row, col) in a tile of `rows` rows x D columns
// stored as D/64 boxes of [rows][128 B] with the TMA 128-byte swizzle
// (16-byte chunk c of row r lives at chunk c ^ (r & 7)).
__device__ __forceinline__ uint32_t swz_off(int rows, int r, int col) {
  const int box = col >> 6;
  const int chunk = (col & 63) >> 3;
  return box * rows * 128 + r * 128 + ((chunk ^ (r & 7)) << 4) + (col & 7) * 2;
}

// Process one tile of NK keys (NK = 64 context keys, or 32 block keys).
// QLO: add q_lo K^T.  KVLO: the tile has remainder K/V (block keys) to add.
template <int D, int NK, bool QLO, bool KVLO>
__device__ __forceinline__ void attend_tile(uint32_t k_base, uint32_t v_base, uint32_t k_lo, uint32_t v_lo,
                                            int n_valid, const uint32_t (&qh)[D / 16][4],
                                            const uint32_t (&ql)[D / 16][4], float (&o)[D / 8][4], float& m0,
                                            float& m1, float& l0, float& l1, float scale_log2, int lane) {
  // S = Q K^T : 16 rows x NK keys
  float s[NK / 8][4];
#pragma unroll
  for (int j = 0; j < NK / 8; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
  for (int j = 0; j < NK / 8; ++j) {
    const int key = j * 8 + (lane & 7);
#pragma unroll
    for (int kk = 0; kk < D / 16; kk += 2) {
      const int col = kk * 16 + (lane >> 3) * 8;
      uint32_t b0, b1, b2, b3;
      ldmatrix_x4(k_base + swz_off(NK, key, col), b0, b1, b2, b3);
      mma_bf16_16816(s[j], qh[kk], b0, b1);
      mma_bf16_16816(s[j], qh[kk + 1], b2, b3);
      if (QLO) {
        mma_bf16_16816(s[j], ql[kk], b0, b1);
        mma_bf16_16816(s[j], ql[kk + 1], b2, b3);
      }
      if (KVLO) {
        ldmatrix_x4(k_lo + swz_off(NK, key, col), b0, b1, b2, b3);
        mma_bf16_16816(s[j], qh[kk], b0, b1);
        mma_bf16_16816(s[j], qh[kk + 1], b2, b3);
      }
    }
  }
  // scale to base-2 units and mask keys beyond n_valid
  float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
  for (int j = 0; j < NK / 8; ++j) {
    const int key = j * 8 + (lane & 3) * 2;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const bool valid = (key + e) < n_valid;
      s[j][e] = valid ? s[j][e] * scale_log2 : -INFINITY;
      s[j][2 + e] = valid ? s[j][2 + e] * scale_log2 : -INFINITY;
      mx0 = fmaxf(mx0, s[j][e]);
      mx1 = fmaxf(mx1, s[j][2 + e]);
    }
  }
  mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
  mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
  mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
  mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
  const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
  const float base0 = mn0 == -INFINITY ? 0.f : mn0;
  const float base1 = mn1 == -INFINITY ? 0.f : mn1;
  const float alpha0 = exp2f(m0 - base0), alpha1 = exp2f(m1 - base1);
  m0 = mn0;
  m1 = mn1;
  float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
  for (int j = 0; j < NK / 8; ++j) {
    s[j][0] = exp2f(s[j][0] - base0);
    s[j][1] = exp2f(s[j][1] - base0);
    s[j][2] = exp2f(s[j][2] - base1);
    s[j][3] = exp2f(s[j][3] - base1);
    ps0 += s[j][0] + s[j][1];
    ps1 += s[j][2] + s[j][3];
  }
  l0 = l0 * alpha0 + ps0;
  l1 = l1 * alpha1 + ps1;
#pragma unroll
  for (int n = 0; n < D / 8; ++n) {
    o[n][0] *= alpha0;
    o[n][1] *= alpha0;
    o[n][2] *= alpha1;
    o[n][3] *= alpha1;
  }
  // O += P V.  P is split into a bf16 head and a bf16 remainder
  // (p = hi + lo to ~2^-17 relative) and both are multiplied by the same V
  // fragment: a bf16-rounded P alone perturbs the output by ~2^-9 relative,
  // which the residual stream and RMSNorm amplify into visible logit error.
#pragma unroll
  for (int kk = 0; kk < NK / 16; ++kk) {
    uint32_t ph[4], pl[4];
    split_bf16(s[2 * kk][0], s[2 * kk][1], ph[0], pl[0]);
    split_bf16(s[2 * kk][2], s[2 * kk][3], ph[1], pl[1]);
    split_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1], ph[2], pl[2]);
    split_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3], ph[3], pl[3]);
    const int mi = lane >> 3;
    const int key = kk * 16 + (lane & 7) + (mi & 1) * 8;
#pragma unroll
    for (int jj = 0; jj < D / 16; ++jj) {
      const int col = jj * 16 + (mi >> 1) * 8;
      uint32_t b0, b1, b2, b3;
      ldmatrix_x4_trans(v_base + swz_off(NK, key, col), b0, b1, b2, b3);
      mma_bf16_16816(o[2 * jj], ph, b0, b1);
      mma_bf16_16816(o[2 * jj + 1], ph, b2, b3);
      mma_bf16_16816(o[2 * jj], pl, b0, b1);
      mma_bf16_16816(o[2 * jj + 1], pl, b2, b3);
      if (KVLO) {
        ldmatrix_x4_trans(v_lo + swz_off(NK, key, col), b0, b1, b2, b3);
        mma_bf16_16816(o[2 * jj], ph, b0, b1);
        mma_bf16_16816(o[2 * jj + 1], ph, b2, b3);
      }
    }
  }
}

template <int D>
__host__ __device__ constexpr int attn_stages() {
  return D == 128 ? 3 : 4;
}

template <int D, bool SPLIT>
__host__ __device__ constexpr int attn_smem_bytes() {
  return 1024 + attn_stages<D>() * 2 * kKT * D * 2 + (SPLIT ? 4 : 2) * kKTB * D * 2 + 2 * attn_stages<D>() * 8 + 16;
}

// MAXW: most compute warps a launch may use (register budget follows it).
template <int D, bool SPLIT, int MAXW>
__global__ void __launch_bounds__((MAXW + 1) * 32, 1) k_block_attn(const __grid_constant__ CUtensorMap map_k,
                                                    const __grid_constant__ CUtensorMap map_v, const AttnArgs a,
                                                    int n_splits, int warps_c) {
  constexpr int STAGES = attn_stages<D>();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int kTileB = kKT * D * 2;
  constexpr int kBlkB = kKTB * D * 2;
  uint8_t* kv_stages = smem;                      // STAGES x (K tile, V tile)
  uint8_t* blk = smem + STAGES * 2 * kTileB;       // block K, V (then K_lo, V_lo with SPLIT)
  uint64_t* full = reinterpret_cast<uint64_t*>(blk + (SPLIT ? 4 : 2) * kBlkB);
  uint64_t* empty = full + STAGES;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + STAGES);

  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;  // b: compacted sequence
  const int warp = warp_id(), lane = lane_id();
  pdl_wait();  // q|k|v come from the preceding kernel
  pdl_launch_dependents();
  if (a.cmp && b >= a.cmp[1]) return;  // not an active sequence
  const int T = *a.ctx_len;
  const int ntiles = (T + kKT - 1) / kKT;
  const int per = (ntiles + n_splits - 1) / n_splits;
  const int tile0 = split * per;
  const int tile1 = min(ntiles, tile0 + per);
  const int z = a.z0 + (a.cmp ? a.cmp[2 + b] : b) * a.Hkv + kvh;
  const int R = a.B * a.S;
  const __nv_bfloat16* qkv = reinterpret_cast<const __nv_bfloat16*>(a.qkv);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], warps_c);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (split == 0) {
    // Stage the block keys/values of this kv head (rows >= S zero-filled):
    // tiles k, v, and with SPLIT k_lo, v_lo.
    // Loads are issued in batches of 8 per thread before their stores, so
    // their latencies overlap.
    const int chunks = kKTB * (D / 8);
    const int ntile = SPLIT ? 4 : 2;
    for (int c0 = 0; c0 < ntile * chunks; c0 += 8 * blockDim.x) {
      uint4 val[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int c = c0 + threadIdx.x + j * blockDim.x;
        val[j] = make_uint4(0, 0, 0, 0);
        if (c < ntile * chunks) {
          const int which = c / chunks;  // 0 = k, 1 = v, 2 = k_lo, 3 = v_lo
          const int cc = c % chunks;
          const int r = cc / (D / 8), col = (cc % (D / 8)) * 8;
          if (r < a.S) {
            const long long row = (long long)(which >= 2 ? R : 0) + b * a.S + r;
            const long long off = row * a.ld_qkv + (a.Hq + (which & 1) * a.Hkv + kvh) * D + col;
            val[j] = *reinterpret_cast<const uint4*>(qkv + off);
          }
        }
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int c = c0 + threadIdx.x + j * blockDim.x;
        if (c < ntile * chunks) {
          const int which = c / chunks;
          const int cc = c % chunks;
          const int r = cc / (D / 8), col = (cc % (D / 8)) * 8;
          *reinterpret_cast<uint4*>(blk + which * kBlkB + swz_off(kKTB, r, col)) = val[j];
        }
      }
    }
  }
  __syncthreads();

  if (warp == warps_c) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      int s = 0;
      uint32_t phase = 0;
      for (int t = tile0; t < tile1; ++t) {
        if (!mbar_wait_bounded(&empty[s], phase ^ 1, a.timeout_ns, abort_flag, a.status)) break;
        uint8_t* kd = kv_stages + s * 2 * kTileB;
        uint8_t* vd = kd + kTileB;
        mbar_arrive_expect_tx(&full[s], 2 * kTileB);
#pragma unroll
        for (int box = 0; box < D / 64; ++box) {
          tma_load_3d(kd + box * kKT * 128, &map_k, &full[s], box * 64, t * kKT, z);
          tma_load_3d(vd + box * kKT * 128, &map_v, &full[s], box * 64, t * kKT, z);
        }
        if (++s == STAGES) { s = 0; phase ^= 1; }
      }
    }
    __syncwarp();
    return;
  }

  // ------------------------------------------------------------ compute
  // Rows of this warp: r = warp*16 + lane/4 (+8); row r = (g, i) with
  // g = r / S (query head within the group) and i = r % S (block position).
  const int r0 = warp * 16 + (lane >> 2);
  const int r1 = r0 + 8;
  const int g0 = r0 / a.S, i0 = r0 % a.S;
  const int g1 = r1 / a.S, i1 = r1 % a.S;
  const int h0 = kvh * a.G + g0, h1 = kvh * a.G + g1;
  uint32_t qh[D / 16][4], ql[D / 16][4];
#pragma unroll
  for (int half = 0; half < (SPLIT ? 2 : 1); ++half) {
    const long long ro = half ? R : 0;
    const __nv_bfloat16* q0 = qkv + (ro + b * a.S + i0) * a.ld_qkv + h0 * D + (lane & 3) * 2;
    const __nv_bfloat16* q1 = qkv + (ro + b * a.S + i1) * a.ld_qkv + h1 * D + (lane & 3) * 2;
    uint32_t(&qf)[D / 16][4] = half ? ql : qh;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      qf[kk][0] = *reinterpret_cast<const uint32_t*>(q0 + kk * 16);
      qf[kk][1] = *reinterpret_cast<const uint32_t*>(q1 + kk * 16);
      qf[kk][2] = *reinterpret_cast<const uint32_t*>(q0 + kk * 16 + 8);
      qf[kk][3] = *reinterpret_cast<const uint32_t*>(q1 + kk * 16 + 8);
    }
  }
  float o[D / 8][4];
#pragma unroll
  for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

  if (split == 0) {
    const uint32_t bk = smem_u32(blk);
    attend_tile<D, kKTB, SPLIT, SPLIT>(bk, bk + kBlkB, bk + 2 * kBlkB, bk + 3 * kBlkB, a.S, qh, ql, o, m0, m1, l0,
                                       l1, a.scale_log2, lane);
  }
  {
    int s = 0;
    uint32_t phase = 0;
    for (int t = tile0; t < tile1; ++t) {
      bool ok = true;
      if (lane == 0) ok = mbar_wait_bounded(&full[s], phase, a.timeout_ns, abort_flag, a.status);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      const uint32_t kb = smem_u32(kv_stages + s * 2 * kTileB);
      attend_tile<D, kKT, SPLIT, false>(kb, kb + kTileB, 0, 0, min(kKT, T - t * kKT), qh, ql, o, m0, m1, l0, l1,
                                        a.scale_log2, lane);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      if (++s == STAGES) { s = 0; phase ^= 1; }
    }
  }
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

  if (n_splits == 1) {
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.out);
    const float inv0 = 1.f / l0, inv1 = 1.f / l1;
    const long long lo_off = (long long)R * a.ld_out;
    __nv_bfloat16* d0 = out + (long long)(b * a.S + i0) * a.ld_out + h0 * D + (lane & 3) * 2;
    __nv_bfloat16* d1 = out + (long long)(b * a.S + i1) * a.ld_out + h1 * D + (lane & 3) * 2;
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      uint32_t hi, lo;
      split_bf16(o[n][0] * inv0, o[n][1] * inv0, hi, lo);
      *reinterpret_cast<uint32_t*>(d0 + n * 8) = hi;
      if (SPLIT) *reinterpret_cast<uint32_t*>(d0 + lo_off + n * 8) = lo;
      split_bf16(o[n][2] * inv1, o[n][3] * inv1, hi, lo);
      *reinterpret_cast<uint32_t*>(d1 + n * 8) = hi;
      if (SPLIT) *reinterpret_cast<uint32_t*>(d1 + lo_off + n * 8) = lo;
    }
  } else {
    const long long prow = ((long long)(b * a.Hkv + kvh) * n_splits + split) * (a.G * a.S);
    float* p0 = a.part_o + (prow + r0) * D + (lane & 3) * 2;
    float* p1 = a.part_o + (prow + r1) * D + (lane & 3) * 2;
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      *reinterpret_cast<float2*>(p0 + n * 8) = make_float2(o[n][0], o[n][1]);
      *reinterpret_cast<float2*>(p1 + n * 8) = make_float2(o[n][2], o[n][3]);
    }
    if ((lane & 3) == 0) {
      a.part_ml[prow + r0] = make_float2(m0, l0);
      a.part_ml[prow + r1] = make_float2(m1, l1);
    }
  }
}

// Merge split partials: o = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s.
// One warp per (sequence, kv head, row).
template <int D>
__global__ void k_attn_combine(const AttnArgs a, int n_splits) {
  pdl_wait();
  pdl_launch_dependents();
  const int rows = a.G * a.S;
  const long long gw = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const long long total = (long long)a.B * a.Hkv * rows;
  if (gw >= total) return;
  const int lane = threadIdx.x & 31;
  const int r = (int)(gw % rows);
  const long long bk = gw / rows;  // b * Hkv + kvh
  const int kvh = (int)(bk % a.Hkv), b = (int)(bk / a.Hkv);
  if (a.cmp && b >= a.cmp[1]) return;  // not an active sequence
  float M = -INFINITY;
  for (int s = 0; s < n_splits; ++s) M = fmaxf(M, a.part_ml[(bk * n_splits + s) * rows + r].x);
  float L = 0.f;
  float acc[D / 32];
#pragma unroll
  for (int k = 0; k < D / 32; ++k) acc[k] = 0.f;
  for (int s = 0; s < n_splits; ++s) {
    const float2 ml = a.part_ml[(bk * n_splits + s) * rows + r];
    const float w = ml.x == -INFINITY ? 0.f : exp2f(ml.x - M);
    L += w * ml.y;
    const float* po = a.part_o + ((bk * n_splits + s) * rows + r) * D;
#pragma unroll
    for (int k = 0; k < D / 32; ++k) acc[k] += w * po[lane + 32 * k];
  }
  const int g = r / a.S, i = r % a.S;
  const long long R = (long long)a.B * a.S;
  __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.out) + (long long)(b * a.S + i) * a.ld_out +
                       (kvh * a.G + g) * D;
  const float inv = 1.f / L;
#pragma unroll
  for (int k = 0; k < D / 32; ++k) {
    const float v = acc[k] * inv;
    const __nv_bfloat16 h = __float2bfloat16_rn(v);
    out[lane + 32 * k] = h;
    if (a.split) out[R * a.ld_out + lane + 32 * k] = __float2bfloat16_rn(v - __bfloat162float(h));
  }
}

// tcgen05 path, after the context kernel: the S in-block keys of one
// (sequence, kv head) on the mma.sync tensor cores (q, k, v and p as bf16
// head + remainder, as in the context kernels), then the log-sum-exp merge
// with the n_ctx context partials:
// o = (2^(m_b - M) o_b + sum_s 2^(m_s - M) o_s) / (2^(m_b - M) l_b + sum_s 2^(m_s - M) l_s).
// One CTA per (sequence, kv head); warp w takes query rows 16w .. 16w + 15
// (row r = g * S + i) and keeps them in the m16n8 fragment layout throughout.
// The block's q|k|v were written by the kernel before the context kernel,
// which lets this kernel launch only after its own wait on that kernel: the
// block keys are staged (through L2) and attended before waiting for the
// context partials.
template <int D, bool SPLIT>
__global__ void __launch_bounds__(128) k_attn_merge_block(const AttnArgs a, int n_ctx_plan) {
  constexpr int kBlkB = kKTB * D * 2;
  __shared__ __align__(128) uint8_t blk[(SPLIT ? 4 : 2) * kBlkB];  // k, v (, k_lo, v_lo)
  const int kvh = blockIdx.x % a.Hkv, b = blockIdx.x / a.Hkv;
  if (a.cmp && b >= __ldcg(a.cmp + 1)) {  // not an active sequence
    pdl_wait();
    pdl_launch_dependents();
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rows = a.G * a.S;
  const int R = a.B * a.S;
  const __nv_bfloat16* qkv = reinterpret_cast<const __nv_bfloat16*>(a.qkv);

  // block K and V (rows >= S zero) -> swizzled tiles; all of a thread's
  // loads are issued before its stores
  {
    constexpr int kChunks = kKTB * (D / 8);
    constexpr int kTiles = SPLIT ? 4 : 2;
    constexpr int kPer = (kTiles * kChunks + 127) / 128;
    uint4 val[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int c = threadIdx.x + j * 128;
      const int which = c / kChunks;  // 0 = k, 1 = v, 2 = k_lo, 3 = v_lo
      const int cc = c % kChunks;
      const int r = cc / (D / 8), col = (cc % (D / 8)) * 8;
      val[j] = make_uint4(0, 0, 0, 0);
      if (c < kTiles * kChunks && r < a.S) {
        const long long row = (long long)(which >= 2 ? R : 0) + b * a.S + r;
        val[j] = __ldcg(reinterpret_cast<const uint4*>(qkv + row * a.ld_qkv + (a.Hq + (which & 1) * a.Hkv + kvh) * D +
                                                       col));
      }
    }
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int c = threadIdx.x + j * 128;
      if (c < kTiles * kChunks) {
        const int which = c / kChunks;
        const int cc = c % kChunks;
        const int r = cc / (D / 8), col = (cc % (D / 8)) * 8;
        *reinterpret_cast<uint4*>(blk + which * kBlkB + swz_off(kKTB, r, col)) = val[j];
      }
    }
  }
  // q fragments of this warp's rows (r0 = 16w + lane/4, r1 = r0 + 8)
  const int r0 = warp * 16 + (lane >> 2);
  const int r1 = r0 + 8;
  const int g0 = r0 / a.S, i0 = r0 % a.S;
  const int g1 = r1 / a.S, i1 = r1 % a.S;
  const int h0 = kvh * a.G + g0, h1 = kvh * a.G + g1;
  uint32_t qh[D / 16][4], ql[D / 16][4];
#pragma unroll
  for (int half = 0; half < (SPLIT ? 2 : 1); ++half) {
    const long long ro = half ? R : 0;
    const __nv_bfloat16* q0 = qkv + (ro + b * a.S + i0) * a.ld_qkv + h0 * D + (lane & 3) * 2;
    const __nv_bfloat16* q1 = qkv + (ro + b * a.S + i1) * a.ld_qkv + h1 * D + (lane & 3) * 2;
    uint32_t(&qf)[D / 16][4] = half ? ql : qh;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      qf[kk][0] = __ldcg(reinterpret_cast<const unsigned int*>(q0 + kk * 16));
      qf[kk][1] = __ldcg(reinterpret_cast<const unsigned int*>(q1 + kk * 16));
      qf[kk][2] = __ldcg(reinterpret_cast<const unsigned int*>(q0 + kk * 16 + 8));
      qf[kk][3] = __ldcg(reinterpret_cast<const unsigned int*>(q1 + kk * 16 + 8));
    }
  }
  __syncthreads();
  const bool active = warp * 16 < rows;
  float o[D / 8][4];
#pragma unroll
  for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  if (active) {
    const uint32_t bk = smem_u32(blk);
    attend_tile<D, kKTB, SPLIT, SPLIT>(bk, bk + kBlkB, bk + 2 * kBlkB, bk + 3 * kBlkB, a.S, qh, ql, o, m0, m1, l0,
                                       l1, a.scale_log2, lane);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  }
  pdl_wait();  // the context partials come from the preceding kernel
  pdl_launch_dependents();
  if (!active) return;
  const int n_ctx = attn_launch_splits(a, n_ctx_plan, *a.ctx_len);  // as the context kernel chose

  // fold in the context partials, one slot per round trip
  const long long pbase = (long long)(b * a.Hkv + kvh) * n_ctx * rows;
  for (int sl = 0; sl < n_ctx; ++sl) {
    const long long pr = pbase + (long long)sl * rows;
    const float2 ml0 = a.part_ml[pr + r0], ml1 = a.part_ml[pr + r1];
    const float* p0 = a.part_o + (pr + r0) * D + (lane & 3) * 2;
    const float* p1 = a.part_o + (pr + r1) * D + (lane & 3) * 2;
    float2 v0[D / 8], v1[D / 8];
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      v0[n] = *reinterpret_cast<const float2*>(p0 + n * 8);
      v1[n] = *reinterpret_cast<const float2*>(p1 + n * 8);
    }
    const float mn0 = fmaxf(m0, ml0.x), mn1 = fmaxf(m1, ml1.x);
    const float wa0 = exp2f(m0 - mn0), wb0 = ml0.x == -INFINITY ? 0.f : exp2f(ml0.x - mn0);
    const float wa1 = exp2f(m1 - mn1), wb1 = ml1.x == -INFINITY ? 0.f : exp2f(ml1.x - mn1);
    l0 = l0 * wa0 + ml0.y * wb0;
    l1 = l1 * wa1 + ml1.y * wb1;
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      o[n][0] = o[n][0] * wa0 + v0[n].x * wb0;
      o[n][1] = o[n][1] * wa0 + v0[n].y * wb0;
      o[n][2] = o[n][2] * wa1 + v1[n].x * wb1;
      o[n][3] = o[n][3] * wa1 + v1[n].y * wb1;
    }
    m0 = mn0;
    m1 = mn1;
  }

  __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.out);
  const float inv0 = 1.f / l0, inv1 = 1.f / l1;
  const long long lo_off = (long long)R * a.ld_out;
  __nv_bfloat16* d0 = out + (long long)(b * a.S + i0) * a.ld_out + h0 * D + (lane & 3) * 2;
  __nv_bfloat16* d1 = out + (long long)(b * a.S + i1) * a.ld_out + h1 * D + (lane & 3) * 2;
#pragma unroll
  for (int n = 0; n < D / 8; ++n) {
    uint32_t hi, lo;
    split_bf16(o[n][0] * inv0, o[n][1] * inv0, hi, lo);
    *reinterpret_cast<uint32_t*>(d0 + n * 8) = hi;
    if (SPLIT) *reinterpret_cast<uint32_t*>(d0 + lo_off + n * 8) = lo;
    split_bf16(o[n][2] * inv1, o[n][3] * inv1, hi, lo);
    *reinterpret_cast<uint32_t*>(d1 + n * 8) = hi;
    if (SPLIT) *reinterpret_cast<uint32_t*>(d1 + lo_off + n * 8) = lo;
  }
}

// The same merge for shapes with few (sequence, kv head) pairs, where one
// CTA per pair would leave most SMs idle: one warp per query row, 8 rows per
// CTA, the block keys in fp32 on the CUDA cores (q, k, v rebuilt from head +
// remainder).  Scores: lane = (key j = lane / 2, half of the head dim), so
// each dot product is split over two lanes; the output: lane owns dims
// lane + 32 k.  The block keys are staged and attended while the context
// kernel still runs; only the fold of its partials waits for it.
constexpr int kMergeBatch = 4;  // context partials per row held in registers

template <int D>
__global__ void __launch_bounds__(256) k_attn_merge_rows(const AttnArgs a, int n_ctx_plan) {
  constexpr int P = D / 32;      // output dims per lane
  constexpr int H2 = D / 2;      // dims per half dot product
  constexpr int KS = D + 8;      // padded row stride of the staged K (floats)
  __shared__ __align__(16) float ks[kKTB * KS];
  __shared__ __align__(16) float vs[kKTB * D];
  __shared__ __align__(16) float qs[8 * D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = a.S, rows = a.G * S;
  const int ctas_per_bk = (rows + 7) / 8;
  const int bk = blockIdx.x / ctas_per_bk;  // b * Hkv + kvh
  const int r0 = (blockIdx.x % ctas_per_bk) * 8;
  const int nq = min(8, rows - r0);
  const int kvh = bk % a.Hkv, b = bk / a.Hkv;
  const long long R = (long long)a.B * S;
  const long long lo = a.split ? R * a.ld_qkv : 0;
  const __nv_bfloat16* qkv = reinterpret_cast<const __nv_bfloat16*>(a.qkv);
  const int r = r0 + warp;
  const bool active = warp < nq;
  // The block's q|k|v were written by the kernel before the context kernel,
  // which lets this kernel launch only after its own wait on that kernel:
  // they are complete here, so the block keys are staged (through L2) and
  // attended before waiting for the context partials.
  const bool seq_on = !a.cmp || b < __ldcg(a.cmp + 1);  // an active sequence
  float acc[P];
  float M = -INFINITY, L = 0.f;
  if (seq_on) {
    // q rows of this CTA, block K and block V -> shared memory (fp32, head +
    // remainder); every load of this thread is issued before its first store
    constexpr int CPR = D / 8;                                // 16-byte chunks per row
    constexpr int kPer = ((8 + 2 * kKTB) * CPR + 255) / 256;  // chunks per thread, at most
    const int total = (nq + 2 * S) * CPR;
    uint4 hv[kPer], lv[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int c = threadIdx.x + u * 256;
      if (c < total) {
        const int row = c / CPR, col = (c % CPR) * 8;
        long long off;
        if (row < nq) {
          const int rr = r0 + row;
          off = (long long)(b * S + rr % S) * a.ld_qkv + (kvh * a.G + rr / S) * D + col;
        } else {
          const int kv = row - nq, which = kv >= S ? 1 : 0, j = kv - which * S;
          off = (long long)(b * S + j) * a.ld_qkv + (a.Hq + which * a.Hkv + kvh) * D + col;
        }
        hv[u] = __ldcg(reinterpret_cast<const uint4*>(qkv + off));
        lv[u] = a.split ? __ldcg(reinterpret_cast<const uint4*>(qkv + lo + off)) : make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int c = threadIdx.x + u * 256;
      if (c < total) {
        const int row = c / CPR, col = (c % CPR) * 8;
        float* dst;
        if (row < nq) {
          dst = qs + row * D + col;
        } else {
          const int kv = row - nq, which = kv >= S ? 1 : 0, j = kv - which * S;
          dst = which ? vs + j * D + col : ks + j * KS + col;
        }
        const uint32_t hw[4] = {hv[u].x, hv[u].y, hv[u].z, hv[u].w};
        const uint32_t lw[4] = {lv[u].x, lv[u].y, lv[u].z, lv[u].w};
        float v[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          v[2 * e] = __uint_as_float(hw[e] << 16) + __uint_as_float(lw[e] << 16);
          v[2 * e + 1] = __uint_as_float(hw[e] & 0xffff0000u) + __uint_as_float(lw[e] & 0xffff0000u);
        }
        reinterpret_cast<float4*>(dst)[0] = make_float4(v[0], v[1], v[2], v[3]);
        reinterpret_cast<float4*>(dst)[1] = make_float4(v[4], v[5], v[6], v[7]);
      }
    }
    __syncthreads();
    if (active) {
      // scores of keys j = lane / 2 + 16 u (u = 0, 1; S <= 32), in base-2 units
      const int half = lane & 1;
      float sj[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int j = (lane >> 1) + 16 * u;
        float t0 = 0.f, t1 = 0.f, t2 = 0.f, t3 = 0.f;
        if (j < S) {
          const float4* kr = reinterpret_cast<const float4*>(ks + j * KS);
          const float4* qr = reinterpret_cast<const float4*>(qs + warp * D);
#pragma unroll
          for (int m = 0; m < H2 / 4; ++m) {
            // interleaved 16-byte chunks: this half takes chunk 2m + half
            const float4 kv = kr[2 * m + half], qv = qr[2 * m + half];
            t0 = fmaf(qv.x, kv.x, t0);
            t1 = fmaf(qv.y, kv.y, t1);
            t2 = fmaf(qv.z, kv.z, t2);
            t3 = fmaf(qv.w, kv.w, t3);
          }
        }
        float t = (t0 + t1) + (t2 + t3);
        t += __shfl_xor_sync(0xffffffffu, t, 1);
        sj[u] = j < S ? t * a.scale_log2 : -INFINITY;
      }
      float mb = fmaxf(sj[0], sj[1]);
#pragma unroll
      for (int o = 2; o < 32; o <<= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, o));
      float pj[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) pj[u] = sj[u] == -INFINITY ? 0.f : exp2f(sj[u] - mb);
      float lb = half ? 0.f : pj[0] + pj[1];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) lb += __shfl_xor_sync(0xffffffffu, lb, o);
#pragma unroll
      for (int k = 0; k < P; ++k) acc[k] = 0.f;
      for (int jj = 0; jj < S; ++jj) {
        const float p = __shfl_sync(0xffffffffu, jj < 16 ? pj[0] : pj[1], 2 * (jj & 15));
#pragma unroll
        for (int k = 0; k < P; ++k) acc[k] = fmaf(p, vs[jj * D + lane + 32 * k], acc[k]);
      }
      M = mb;
      L = lb;
    }
  }
  pdl_wait();  // the context partials come from the preceding kernel
  pdl_launch_dependents();
  if (!seq_on || !active) return;
  const int n_ctx = attn_launch_splits(a, n_ctx_plan, *a.ctx_len);  // as the context kernel chose

  // merge with the context partials of this warp's row, kMergeBatch slots
  // per round trip
  const long long pbase = (long long)bk * n_ctx * rows + r;
  for (int s0 = 0; s0 < n_ctx; s0 += kMergeBatch) {
    float2 ml[kMergeBatch];
    float po[kMergeBatch][P];
#pragma unroll
    for (int t = 0; t < kMergeBatch; ++t) {
      if (s0 + t < n_ctx) {
        const long long pr = pbase + (long long)(s0 + t) * rows;
        ml[t] = a.part_ml[pr];
#pragma unroll
        for (int k = 0; k < P; ++k) po[t][k] = a.part_o[pr * D + lane + 32 * k];
      }
    }
#pragma unroll
    for (int t = 0; t < kMergeBatch; ++t) {
      if (s0 + t < n_ctx && ml[t].x != -INFINITY) {
        const float Mn = fmaxf(M, ml[t].x);
        const float wa = exp2f(M - Mn), wb = exp2f(ml[t].x - Mn);
        L = L * wa + ml[t].y * wb;
#pragma unroll
        for (int k = 0; k < P; ++k) acc[k] = acc[k] * wa + po[t][k] * wb;
        M = Mn;
      }
    }
  }
  const int g = r / S, i = r % S;
  __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.out) + (long long)(b * S + i) * a.ld_out +
                       (kvh * a.G + g) * D + lane;
  const float inv = 1.f / L;
#pragma unroll
  for (int k = 0; k < P; ++k) {
    const float v = acc[k] * inv;
    const __nv_bfloat16 h = __float2bfloat16_rn(v);
    out[32 * k] = h;
    if (a.split) out[R * a.ld_out + 32 * k] = __float2bfloat16_rn(v - __bfloat162float(h));
  }
}

template <int D, bool SPLIT>
void launch_attn_kernel(const AttnPlan& p, const AttnArgs& a, int grid_x, const CUtensorMap& mk,
                        const CUtensorMap& mv, cudaStream_t st) {
  dim3 grid(grid_x, a.Hkv, a.B);
  const int threads = (p.warps_c + 1) * 32;
  if (p.warps_c <= 4)
    launch_k(k_block_attn<D, SPLIT, 4>, grid, threads, attn_smem_bytes<D, SPLIT>(), st, mk, mv, a, p.n_splits,
             p.warps_c);
  else
    launch_k(k_block_attn<D, SPLIT, 8>, grid, threads, attn_smem_bytes<D, SPLIT>(), st, mk, mv, a, p.n_splits,
             p.warps_c);
}

}  // namespace

AttnPlan plan_attention(int B, int S, int Hq, int Hkv, int D, int max_ctx, int allow_tc) {
  AttnPlan p{};
  p.D = D;
  p.rows = (Hq / Hkv) * S;
  p.warps_c = p.rows / 16;
  p.stages = D == 128 ? attn_stages<128>() : attn_stages<64>();
  p.smem_bytes = D == 128 ? attn_smem_bytes<128, true>() : attn_smem_bytes<64, true>();
  if (allow_tc && attention_tc_supported(D, p.rows) && max_ctx > 0) {
    p.use_tc = 1;
    p.n_ctx = attention_tc_splits(B, Hkv, max_ctx);
    p.n_splits = p.n_ctx;  // partial slots: the context splits (block keys are merged in-line)
    return p;
  }
  const int pairs = B * Hkv;
  const int ntiles = (max_ctx + kKT - 1) / kKT;
  // Enough CTAs for ~4 resident waves (2 CTAs per SM), at least 4 tiles per split.
  const int want = (4 * 2 * kNumSMs + pairs - 1) / pairs;
  int max_splits = (ntiles + 3) / 4;
  if (max_splits < 1) max_splits = 1;
  p.n_splits = want < max_splits ? want : max_splits;
  if (p.n_splits < 1) p.n_splits = 1;
  return p;
}

size_t attention_partial_bytes(const AttnPlan& p, int B, int Hkv) {
  if (p.n_splits <= 1 && !p.use_tc) return 0;
  const size_t n = (size_t)B * Hkv * p.n_splits * p.rows;
  return n * p.D * sizeof(float) + n * sizeof(float2) + 256;
}

cudaError_t launch_attention(const AttnPlan& p, const AttnArgs& a_in, const CUtensorMap& map_k, const CUtensorMap& map_v,
                             const CUtensorMap& map_k128, const CUtensorMap& map_v128, const CUtensorMap& map_q,
                             cudaStream_t st, const CUtensorMap* map_q2) {
  AttnArgs a = a_in;
  // tcgen05 path: context splits only; the block keys join in the merge
  if (p.use_tc) return launch_attention_tc(a, p.n_ctx, map_k128, map_v128, map_q, st, map_q2);
  if (p.D == 128) {
    if (a.split) launch_attn_kernel<128, true>(p, a, p.n_splits, map_k, map_v, st);
    else launch_attn_kernel<128, false>(p, a, p.n_splits, map_k, map_v, st);
  } else {
    if (a.split) launch_attn_kernel<64, true>(p, a, p.n_splits, map_k, map_v, st);
    else launch_attn_kernel<64, false>(p, a, p.n_splits, map_k, map_v, st);
  }
  return cudaGetLastError();
}

cudaError_t launch_attention_combine(const AttnPlan& p, const AttnArgs& a, cudaStream_t st) {
  if (p.use_tc) {
    const int bk = a.B * a.Hkv;
    if (bk < kNumSMs) {
      // few pairs: one warp per row, 8 rows per CTA
      const int blocks = bk * ((p.rows + 7) / 8);
      if (p.D == 128) return launch_k(k_attn_merge_rows<128>, blocks, 256, 0, st, a, p.n_ctx);
      return launch_k(k_attn_merge_rows<64>, blocks, 256, 0, st, a, p.n_ctx);
    }
    // one CTA per (sequence, kv head), one warp per 16 query rows
    const int blocks = bk, threads = ((p.rows + 15) / 16) * 32;
    if (p.D == 128) {
      if (a.split) return launch_k(k_attn_merge_block<128, true>, blocks, threads, 0, st, a, p.n_ctx);
      return launch_k(k_attn_merge_block<128, false>, blocks, threads, 0, st, a, p.n_ctx);
    }
    if (a.split) return launch_k(k_attn_merge_block<64, true>, blocks, threads, 0, st, a, p.n_ctx);
    return launch_k(k_attn_merge_block<64, false>, blocks, threads, 0, st, a, p.n_ctx);
  }
  if (p.n_splits == 1) return cudaSuccess;
  const long long warps = (long long)a.B * a.Hkv * p.rows;
  const int blocks = (int)((warps + 7) / 8);
  if (p.D == 128) return launch_k(k_attn_combine<128>, blocks, 256, 0, st, a, p.n_splits);
  else return launch_k(k_attn_combine<64>, blocks, 256, 0, st, a, p.n_splits);
  return cudaGetLastError();
}

cudaError_t prepare_attention_kernels() {
  const int lim = 227 * 1024;
  const void* fns[] = {(const void*)k_block_attn<128, true, 4>,  (const void*)k_block_attn<128, false, 4>,
                       (const void*)k_block_attn<64, true, 4>,   (const void*)k_block_attn<64, false, 4>,
                       (const void*)k_block_attn<128, true, 8>,  (const void*)k_block_attn<128, false, 8>,
                       (const void*)k_block_attn<64, true, 8>,   (const void*)k_block_attn<64, false, 8>};
  cudaError_t e = cudaSuccess;
  for (const void* f : fns) {
    if (e == cudaSuccess) e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  }
  const void* comb[] = {(const void*)k_attn_combine<128>,          (const void*)k_attn_combine<64>,
                        (const void*)k_attn_merge_block<128, true>, (const void*)k_attn_merge_block<128, false>,
                        (const void*)k_attn_merge_block<64, true>,  (const void*)k_attn_merge_block<64, false>,
                        (const void*)k_attn_merge_rows<128>,        (const void*)k_attn_merge_rows<64>};
  for (const void* f : comb) {
    if (e == cudaSuccess) e = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  }
  return e;
}

}  // namespace dd
