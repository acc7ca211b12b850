// Tensor-core GEMM for sm_103a: TMA -> shared memory (128-byte swizzle) ->
// tcgen05.mma (bf16 in, fp32 accumulate in TMEM) -> epilogue warps reading
// TMEM with tcgen05.ld.
//
// One warp-specialised kernel serves every dense contraction of the
// denoising step:
//   * linear layers (QKV, O, gate|up, down): the weight tile sits on the MMA
//     M side (128 output features per tile) and the B*S activation rows on
//     the N side, so a 128-row decode batch still fills the 128-lane
//     accumulator; K may be split across CTAs, each writing an fp32 partial
//     that a reduce kernel sums and post-processes (bf16 store, residual +
//     RMSNorm, SwiGLU);
//   * the LM head: activation rows on the M side (one TMEM lane per row) and
//     256 vocab entries per tile on the N side; the epilogue folds each
//     row's 256 logits into a running (max, sum of exp, first argmax) so the
//     logits never reach global memory.
//
// Split activations: an activation operand may be stored as a bf16 head
// (rows [0, R)) and a bf16 remainder (rows [R, 2R)) of the same tensor map;
// both tiles are loaded per K block and both products accumulate into the
// same fp32 accumulator, so the GEMM sees the activation to ~2^-17.
//
// Roles (192 threads): warp 0 issues TMA loads, warp 1 owns TMEM and issues
// MMAs, warps 2-5 run the epilogue (TMEM lane quarter = warp % 4).  Two
// accumulator buffers let the epilogue of one tile overlap the MMAs of the
// next.  Every mbarrier wait is bounded; on expiry the kernel records a
// timeout in the status word and unwinds.
//
// Linear layers whose activation tile is wider than 128 rows run as CTA
// pairs (clusters of two on weight tiles 2p and 2p + 1) sharing one MMA of
// M = 256 (tcgen05 cta_group::2): each CTA stages its own weight tile and half
// of the activation rows, rank 0 waits for both CTAs' bytes on its barrier
// and issues the MMAs, and each CTA's tensor memory receives its own weight
// tile's accumulator rows for all activation rows.
#include <math.h>

#include "kernels.h"
#include "ptx.cuh"

namespace dd {

namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;  // K elements per block, 128-byte swizzle (32: 64-byte swizzle)
constexpr int kThreads = 192;
constexpr float kLog2e = 1.4426950408889634f;

struct KArgs {
  int m_tiles, n_tiles, splits, kb_total, kb_per_split, BN, stages, tiles_total;
  int sk_units;    // > 0: stream-K, each CTA takes this many consecutive (tile, K block) units
  int sk_total;    // units of the whole GEMM (tiles x K blocks)
  int split_rows;  // row offset of the remainder half in the activation map
  int cluster;     // 1, or 2: CTA pairs (ranks 0, 1) on weight tiles 2p, 2p + 1, one MMA of M = 256 (CG 2)
  uint32_t tmem_half;
  GemmOut out;
  int* status;
  uint64_t timeout_ns;
};

// Bytes of one pipeline stage: A tile, B tile, and the activation remainder.
__host__ __device__ inline int stage_bytes_of(int epi, int BN, int split, int bk) {
  const int a = kBM * bk * 2;
  const int b = BN * bk * 2;
  const int act = (epi == kEpiPartial) ? b : a;
  return a + b + (split ? act : 0);
}

// Shared-memory descriptor of a K-major tile as TMA wrote it for K blocks of BK.
template <int BK>
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr) {
  static_assert(BK == 64 || BK == 32, "K blocks of 64 or 32");
  return BK == 64 ? smem_desc_sw128(saddr) : smem_desc_sw64(saddr);
}

// One piece of work of a CTA: K blocks [kb0, kb1) of tile (mt, nt), whose
// fp32 result goes to partial slot `slot`.  Uniform split-K: the CTA takes
// items blockIdx.x, blockIdx.x + gridDim.x, ... of tiles x splits.  Stream-K
// (linear layers, sk_units > 0): the CTA takes units [c*L, (c+1)*L) of the
// (tile, K block) sequence, tile by tile, so every CTA does the same number of
// K blocks; a tile cut between CTAs gets one slot per piece (slot = the CTA's
// place among the tile's CTAs); the reduce reads a tile's pieces only
// (slots_of).
struct Seg {
  int mt, nt, kb0, kb1, slot;
  bool first;                             // the CTA's first piece (never skipped)
};

//
// With CTA pairs (cluster 2) both CTAs of a pair take the same pieces of the
// same pair tile (weight tiles 2p and 2p + 1, one activation tile): the pair
// is the unit of the schedule, and the CTA's rank picks its weight tile.
__device__ __forceinline__ bool seg_of(const KArgs& a, int epi, int i, Seg& g) {
  const int rank = a.cluster == 2 ? (int)(blockIdx.x & 1) : 0;
  const int cid = a.cluster == 2 ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;  // the schedule's worker
  const int workers = a.cluster == 2 ? (int)(gridDim.x >> 1) : (int)gridDim.x;
  const int m_tiles = a.m_tiles / a.cluster;
  const int per_split = m_tiles * a.n_tiles;
  int tile;
  if (a.sk_units > 0) {
    const int u0 = cid * a.sk_units;
    const int u1 = min(u0 + a.sk_units, a.sk_total);
    const int start = i == 0 ? u0 : (u0 / a.kb_total + i) * a.kb_total;
    if (start >= u1) return false;
    tile = start / a.kb_total;
    g.kb0 = start - tile * a.kb_total;
    g.kb1 = min(a.kb_total, u1 - tile * a.kb_total);
    g.slot = cid - tile * a.kb_total / a.sk_units;  // this piece's place among the tile's workers
  } else {
    const int t = cid + i * workers;
    if (t >= a.tiles_total) return false;
    const int split = t / per_split;
    tile = t % per_split;
    g.kb0 = split * a.kb_per_split;
    g.kb1 = min(a.kb_total, g.kb0 + a.kb_per_split);
    g.slot = split;
  }
  if (epi == kEpiPartial) { g.nt = tile % a.n_tiles; g.mt = (tile / a.n_tiles) * a.cluster + rank; }
  else { g.mt = tile % m_tiles; g.nt = tile / m_tiles; }
  g.first = i == 0;
  return true;
}

// SPLIT is a template parameter: a run-time test inside the MMA issue loop
// slowed the LM head by a sixth.  BK: K elements per block and stage (the
// tensor maps' box width).  CG = 2: the CTA pairs of a cluster run one MMA of
// M = 256 (cta_group::2): each CTA stages its own weight tile and its half of
// the activation rows (head and remainder), rank 0 issues the MMAs, and each
// CTA's tensor memory holds its own weight tile's accumulator rows.
template <int EPI, int SPLIT, int BK, int CG = 1>
__global__ void __launch_bounds__(kThreads, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b, const KArgs args) {
  static_assert(CG == 1 || (CG == 2 && EPI == kEpiPartial), "cta_group::2 for the linear layers only");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int kA = kBM * BK * 2;  // bytes of a 128-row tile of one K block
  const int stage_b = args.BN / CG * BK * 2;  // this CTA's activation rows of one K block
  const int stage_bytes = stage_bytes_of(EPI, args.BN / CG, SPLIT, BK);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + args.stages * stage_bytes);
  uint64_t* empty = full + args.stages;
  uint64_t* acc_full = empty + args.stages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint64_t* ready = drain + 1;  // the producer has read the activation row count
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ready + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* rows_smem = abort_flag + 1;
  uint32_t* tmem_slot2 = reinterpret_cast<uint32_t*>(const_cast<int*>(rows_smem + 1));  // CG 2: second buffer
  // Compacted activation rows (the LM head's masked rows, or the active
  // sequences' rows of a linear layer): the valid row count is known on the
  // device only.  A CTA never skips its first tile (its weights were
  // requested before the count existed); a later tile is skipped when its
  // first activation row is at or beyond the count.  (A shorter MMA for a
  // partly filled tile does not pay: tcgen05 M = 64 takes as long as M = 128.)
  const bool dyn = EPI != kEpiStore && args.out.rows_dev != nullptr;
  auto first_row = [&](int mt, int nt) { return EPI == kEpiPartial ? nt * args.BN : mt * kBM; };

  const int warp = warp_id();
  const int lane = lane_id();

  if (threadIdx.x == 0) {
    for (int s = 0; s < args.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);  // released by this CTA's MMAs (CG 2: rank 0's, to both CTAs)
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 4 * CG);  // CG 2: rank 0's, released by both CTAs' epilogue warps
    }
    mbar_init(drain, 1);
    mbar_init(ready, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&map_a);
    tma_prefetch_desc(&map_b);
  }
  const int rank = args.cluster == 2 ? (int)(blockIdx.x & 1) : 0;
  uint32_t tbuf[2];    // the two accumulator buffers
  int tmem_held = 0;   // CG 2: buffers allocated
  bool pair_ok = true;
  if constexpr (CG == 1) {
    if (warp == 1) {
      tmem_alloc(tmem_slot, 2 * args.tmem_half);
      tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    tbuf[0] = *tmem_slot;
    tbuf[1] = tbuf[0] + args.tmem_half;
  } else {
    // Each buffer is allocated for the pair in its own round of tmem_half
    // (<= 256) columns, and the two CTAs compare the addresses they got: two
    // rounds can never wait on each other, and a mismatch stops the kernel
    // with kStatusPairTmem instead of running MMAs into foreign columns.
    uint32_t* slots[2] = {tmem_slot, tmem_slot2};
    for (int round = 0; round < 2 && pair_ok; ++round) {
      if (warp == 1) {
        tmem_alloc_pair(slots[round], args.tmem_half);
        tc_fence_before();
      }
      __syncthreads();
      tc_fence_after();
      cluster_sync_all();  // (the first one also publishes both CTAs' barriers)
      tbuf[round] = *slots[round];
      tmem_held = round + 1;
      pair_ok = tbuf[round] == ld_cluster_u32(cluster_addr(slots[round], rank ^ 1));
    }
    if (!pair_ok && threadIdx.x == 0) {
      *abort_flag = 1;
      atomicExch(args.status, kStatusPairTmem);
    }
    __syncthreads();
  }

  if (!pair_ok) {
    // the pair's tensor memory did not match: no work (status recorded); the
    // grid still completes only after its predecessor, as every kernel does
    if (threadIdx.x == 0) {
      pdl_wait();
      pdl_launch_dependents();
    }
  } else if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      // CG 2: both CTAs' loads are counted on rank 0's stage barriers
      const uint32_t full_c = CG == 2 ? cluster_addr(&full[0], 0) : 0u;
      // Weight tiles do not depend on the preceding kernel: the first stages'
      // weight loads go out before waiting for it (programmatic dependent
      // launch), the activation loads of those stages right after the wait.
      auto load_w = [&](uint8_t* sa, int s, int kb, int mt, int nt) {
        if constexpr (CG == 2) tma_load_2d_pair(sa, &map_a, full_c + 8u * s, kb * BK, mt * kBM);
        else if (EPI == kEpiPartial) tma_load_2d(sa, &map_a, &full[s], kb * BK, mt * kBM);
        else tma_load_2d(sa + kA, &map_b, &full[s], kb * BK, nt * args.BN);
      };
      auto load_x = [&](uint8_t* sa, int s, int kb, int mt, int nt) {
        if constexpr (CG == 2) {
          // this CTA's half of the activation rows (the MMA's B reads both)
          const int half = args.BN / 2;
          tma_load_2d_pair(sa + kA, &map_b, full_c + 8u * s, kb * BK, nt * args.BN + rank * half);
          if (SPLIT)
            tma_load_2d_pair(sa + kA + stage_b, &map_b, full_c + 8u * s, kb * BK,
                             args.split_rows + nt * args.BN + rank * half);
        } else if (EPI == kEpiPartial) {
          tma_load_2d(sa + kA, &map_b, &full[s], kb * BK, nt * args.BN);
          if (SPLIT)
            tma_load_2d(sa + kA + stage_b, &map_b, &full[s], kb * BK, args.split_rows + nt * args.BN);
        } else {
          tma_load_2d(sa, &map_a, &full[s], kb * BK, mt * kBM);
          if (SPLIT)
            tma_load_2d(sa + kA + stage_b, &map_a, &full[s], kb * BK, args.split_rows + mt * kBM);
        }
      };
      auto publish_rows = [&]() {
        *rows_smem = dyn ? *args.out.rows_dev : args.out.rows_valid;
        mbar_arrive(ready);
      };
      int s = 0;
      uint32_t phase = 0;
      bool ok = true, waited = false;
      int pend_s[8], pend_kb[8], pend_n = 0;
      Seg sg;
      for (int si = 0; ok && seg_of(args, EPI, si, sg); ++si) {
        const int mt = sg.mt, nt = sg.nt;
        if (dyn && !sg.first && first_row(mt, nt) >= *rows_smem) continue;
        const int kb0 = sg.kb0, kb1 = sg.kb1;
        const int count = kb1 - kb0;
        for (int i = 0; i < count; ++i) {
          const int kb = kb0 + i;
          if (!mbar_wait_bounded(&empty[s], phase ^ 1, args.timeout_ns, abort_flag, args.status)) { ok = false; break; }
          uint8_t* sa = smem + s * stage_bytes;
          if (CG == 1) mbar_arrive_expect_tx(&full[s], stage_bytes);
          else if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * stage_bytes);  // both CTAs' bytes
          load_w(sa, s, kb, mt, nt);
          if (waited) {
            load_x(sa, s, kb, mt, nt);
          } else {
            pend_s[pend_n] = s;
            pend_kb[pend_n] = kb;
            ++pend_n;
            if (pend_n == args.stages || pend_n == 8 || i == count - 1) {
              pdl_wait();
              pdl_launch_dependents();
              waited = true;
              publish_rows();
              for (int i = 0; i < pend_n; ++i) load_x(smem + pend_s[i] * stage_bytes, pend_s[i], pend_kb[i], mt, nt);
            }
          }
          if (++s == args.stages) { s = 0; phase ^= 1; }
        }
      }
      if (!waited) {
        pdl_wait();
        pdl_launch_dependents();
        publish_rows();
      }
      // A pair: wait until both CTAs have released every stage, so no stage
      // release of the peer is still on its way to this CTA when it leaves.
      for (int i = 0; ok && args.cluster == 2 && i < args.stages; ++i) {
        ok = mbar_wait_bounded(&empty[s], phase ^ 1, args.timeout_ns, abort_flag, args.status);
        if (++s == args.stages) { s = 0; phase ^= 1; }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA
    if (lane == 0 && CG == 2 && rank == 1) {
      // rank 0 issues the pair's MMAs: wait until they have all completed
      // (they write this CTA's tensor memory) before it is released
      mbar_wait_bounded(drain, 0, args.timeout_ns, abort_flag, args.status);
    } else if (lane == 0) {
      bool ok = true;
      int rows = -1;  // read when the first skippable tile comes up
      int s = 0;
      uint32_t phase = 0;
      int it = 0;
      Seg sg;
      for (int si = 0; ok && seg_of(args, EPI, si, sg); ++si) {
        const int mt = sg.mt, nt = sg.nt;
        if (dyn && !sg.first) {
          if (rows < 0) {
            if (!mbar_wait_bounded(ready, 0, args.timeout_ns, abort_flag, args.status)) break;
            rows = *rows_smem;
          }
          if (first_row(mt, nt) >= rows) continue;
        }
        const uint32_t idesc = idesc_bf16_f32(kBM * CG, args.BN);
        const int kb0 = sg.kb0, kb1 = sg.kb1;
        const int ab = it & 1;
        const uint32_t aphase = (it >> 1) & 1;
        if (!mbar_wait_bounded(&acc_empty[ab], aphase ^ 1, args.timeout_ns, abort_flag, args.status)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tbuf[ab];
        for (int kb = kb0; kb < kb1; ++kb) {  // stage order; the producer picks which K block fills it
          if (!mbar_wait_bounded(&full[s], phase, args.timeout_ns, abort_flag, args.status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + s * stage_bytes);
          const uint32_t b_addr = a_addr + kA;
          const uint32_t lo_addr = b_addr + stage_b;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            if constexpr (CG == 2) {
              tc_mma_bf16_pair(d_tmem, smem_desc<BK>(a_addr + k * 32), smem_desc<BK>(b_addr + k * 32), idesc,
                               (kb > kb0 || k > 0) ? 1u : 0u);
              if (SPLIT)
                tc_mma_bf16_pair(d_tmem, smem_desc<BK>(a_addr + k * 32), smem_desc<BK>(lo_addr + k * 32), idesc, 1u);
            } else {
              tc_mma_bf16(d_tmem, smem_desc<BK>(a_addr + k * 32), smem_desc<BK>(b_addr + k * 32), idesc,
                          (kb > kb0 || k > 0) ? 1u : 0u);
              if (SPLIT) {
                if (EPI == kEpiPartial)
                  tc_mma_bf16(d_tmem, smem_desc<BK>(a_addr + k * 32), smem_desc<BK>(lo_addr + k * 32), idesc, 1u);
                else
                  tc_mma_bf16(d_tmem, smem_desc<BK>(lo_addr + k * 32), smem_desc<BK>(b_addr + k * 32), idesc, 1u);
              }
            }
          }
          if constexpr (CG == 2) tc_commit_pair_mc(&empty[s], 0x3);
          else tc_commit(&empty[s]);
          if (++s == args.stages) { s = 0; phase ^= 1; }
        }
        if (ok) {
          if constexpr (CG == 2) tc_commit_pair_mc(&acc_full[ab], 0x3);
          else tc_commit(&acc_full[ab]);
        }
        ++it;
      }
      // Drain: wait until every MMA issued by this thread has completed, so
      // TMEM can be released safely on every exit path.
      if constexpr (CG == 2) tc_commit_pair_mc(drain, 0x3);
      else tc_commit(drain);
      mbar_wait_bounded(drain, 0, args.timeout_ns, abort_flag, args.status);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    bool rows_ok = true;
    if (dyn) {
      if (lane == 0) rows_ok = mbar_wait_bounded(ready, 0, args.timeout_ns, abort_flag, args.status);
      rows_ok = __shfl_sync(0xffffffffu, rows_ok ? 1 : 0, 0) != 0;
    }
    const int rows = dyn ? *rows_smem : args.out.rows_valid;
    int it = 0;
    Seg sg;
    for (int si = 0; rows_ok && seg_of(args, EPI, si, sg); ++si) {
      const int mt = sg.mt, nt = sg.nt;
      if (dyn && !sg.first && first_row(mt, nt) >= rows) continue;
      const int ab = it & 1;
      const uint32_t aphase = (it >> 1) & 1;
      ++it;
      bool ok = true;
      if (lane == 0) ok = mbar_wait_bounded(&acc_full[ab], aphase, args.timeout_ns, abort_flag, args.status);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      tc_fence_after();
      const uint32_t tbase = tbuf[ab] + ((uint32_t)(q * 32) << 16);
      const int lrow = mt * kBM + q * 32 + lane;  // accumulator row owned by this thread

      if (EPI == kEpiPartial) {
        // lrow = output feature, columns = activation rows.  TMEM is read 64
        // columns per wait (16 for a ragged tail).
        float* dst = args.out.partial + (long long)sg.slot * args.out.split_stride + lrow;
        int c = 0;
        for (; c + 64 <= args.BN; c += 64) {
          float v[64];
          tmem_ld64(tbase + c, v);
          const int row0 = nt * args.BN + c;
#pragma unroll
          for (int j = 0; j < 64; ++j) {
            if (row0 + j < args.out.rows_valid) dst[(long long)(row0 + j) * args.out.ld] = v[j];
          }
        }
        for (; c < args.BN; c += 16) {
          float v[16];
          tmem_ld16(tbase + c, v);
          const int row0 = nt * args.BN + c;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (row0 + j < args.out.rows_valid) dst[(long long)(row0 + j) * args.out.ld] = v[j];
          }
        }
      } else if (EPI == kEpiSelect) {
        // lrow = activation row, columns = vocab ids nt*BN + c.
        float m = -INFINITY, ssum = 0.f;
        int arg = 0;
        for (int c = 0; c < args.BN; c += 64) {  // BN is 256
          float v[64];
          tmem_ld64(tbase + c, v);
          float cm = v[0];
          int ci = 0;
#pragma unroll
          for (int j = 1; j < 64; ++j) {
            if (v[j] > cm) { cm = v[j]; ci = j; }
          }
          if (cm > m) {
            ssum *= exp2f((m - cm) * kLog2e);
            m = cm;
            arg = nt * args.BN + c + ci;
          }
          const float mb = m * kLog2e;
#pragma unroll
          for (int j = 0; j < 64; ++j) ssum += exp2f(fmaf(v[j], kLog2e, -mb));
        }
        if (lrow < (dyn ? rows : args.out.rows_valid)) {
          const long long o = (long long)nt * args.out.rows_valid + lrow;
          args.out.sel_m[o] = m;
          args.out.sel_s[o] = ssum;
          args.out.sel_a[o] = arg;
        }
      } else {
        // Plain fp32 store of the tile: row lrow, columns nt*BN + c.
        float* dst = args.out.partial + (long long)lrow * args.out.ld + nt * args.BN;
        for (int c = 0; c < args.BN; c += 16) {
          float v[16];
          tmem_ld16(tbase + c, v);
          if (lrow < args.out.rows_valid) {
#pragma unroll
            for (int j = 0; j < 16; j += 4)
              *reinterpret_cast<float4*>(dst + c + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (CG == 2) mbar_arrive_cluster(cluster_addr(&acc_empty[ab], 0));  // rank 0 issues the MMAs
        else mbar_arrive(&acc_empty[ab]);
      }
    }
  }

  __syncthreads();
  // The peer's last stage releases arrive on this CTA's barriers: neither CTA
  // of a pair leaves before both are done.
  if (args.cluster == 2) cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (CG == 2) {
      for (int r = 0; r < tmem_held; ++r) tmem_dealloc_pair(tbuf[r], args.tmem_half);
    } else {
      tmem_dealloc(tbuf[0], 2 * args.tmem_half);
    }
  }
}

uint32_t pow2_at_least(uint32_t v, uint32_t lo) {
  uint32_t p = lo;
  while (p < v) p <<= 1;
  return p;
}

}  // namespace

GemmPlan plan_gemm(int epi, int rows, int N, int K, int split_act, int allow_pairs) {
  GemmPlan p{};
  p.epi = epi;
  p.split_act = split_act;
  p.split_rows = rows;
  p.bk = kBK;
  p.cluster = 1;
  p.cg = 1;
  if (epi == kEpiPartial) {
    // features on M, activation rows on N
    p.m_tiles = N / kBM;
    p.BN = rows <= 256 ? ((rows + 15) / 16) * 16 : 256;
    p.n_tiles = (rows + p.BN - 1) / p.BN;
    // Wider activation tiles: a 256-row split stage of 64-wide K blocks is
    // 80 KB, only two fit and the MMAs wait on every refill.  CTA pairs on
    // adjacent weight tiles run one MMA of M = 256 (cta_group::2): each CTA
    // stages its weight tile and half of the activation rows, a 48 KB stage,
    // four in flight, with 128-byte TMA rows.  (Both halves of a stage's
    // activation tile start on a 1024-byte boundary: BN a multiple of 32.)
    // Shapes that cannot pair take K blocks of 32: 40 KB stages, five in
    // flight, at twice the TMA requests per byte.
    if (p.BN > 128) {
      if (allow_pairs && p.m_tiles % 2 == 0 && p.BN % 32 == 0) {
        p.cluster = 2;
        p.cg = 2;
      } else {
        p.bk = 32;
      }
    }
  } else {
    // activation rows on M, vocab on N (256 per tile)
    p.m_tiles = (rows + kBM - 1) / kBM;
    p.BN = 256;
    p.n_tiles = N / p.BN;
  }
  p.kb_total = K / p.bk;
  const int stage_bytes = stage_bytes_of(epi, p.BN / p.cg, split_act, p.bk);
  p.stages = (200 * 1024) / stage_bytes;
  if (p.stages > 8) p.stages = 8;
  if (p.stages < 2) p.stages = 2;
  p.smem_bytes = 1024 + p.stages * stage_bytes + 256;
  p.tmem_half = pow2_at_least(p.BN, 32);
  p.box_rows_b = p.BN / p.cluster;

  // The schedule's workers: CTAs, or CTA pairs each taking a pair of weight
  // tiles (both CTAs of a pair do the same K blocks of their own tile).
  const int workers = kNumSMs / p.cluster;
  const int base = (p.m_tiles / p.cluster) * p.n_tiles;
  if (epi == kEpiPartial) {
    // Persistent CTAs (at most one per SM) walk the tiles; split K so that
    // the busiest SM's K blocks are few, charging each split for the fp32
    // partial it writes and the reduce kernel reads back (in units of one
    // K block of weights per SM, bk wide).
    int best_s = 1;
    double best_cost = -1.0;
    const int max_s = p.kb_total < kMaxSplits ? p.kb_total : kMaxSplits;
    const double partial_kb = 0.5 * (double)rows * N * 8.0 / ((double)kNumSMs * kBM * p.bk * 2);
    for (int s = 1; s <= max_s; ++s) {
      const int kbps = (p.kb_total + s - 1) / s;
      const int real_s = (p.kb_total + kbps - 1) / kbps;
      if (real_s != s) continue;
      const long long tiles = (long long)base * s;
      const long long per_sm = (tiles + workers - 1) / workers;
      const double cost = (double)(per_sm * kbps) + partial_kb * s + 0.01 * s;
      if (best_cost < 0 || cost < best_cost) { best_cost = cost; best_s = s; }
    }
    p.kb_per_split = (p.kb_total + best_s - 1) / best_s;
    p.splits = best_s;
    p.tiles_total = base * p.splits;
    p.grid = (p.tiles_total < workers ? p.tiles_total : workers) * p.cluster;
    // Stream-K for the wide activation shapes (more than 128 rows): every CTA
    // an equal run of (tile, K block) units, a tile cut between CTAs reduced
    // through one slot per piece.  Taken when its estimate (the run, the
    // slots' partial traffic, one more epilogue) beats the uniform split by
    // 5 %.  (At 128 rows the extra epilogue of a cut tile sits on the
    // critical path of a latency-bound kernel, and it measured slower.)
    if (rows > 128) {
      const long long total = (long long)base * p.kb_total;
      const int L = (int)((total + workers - 1) / workers);
      int max_seg = 1;
      for (int t = 0; t < base; ++t) {
        const long long first = (long long)t * p.kb_total / L, last = ((long long)(t + 1) * p.kb_total - 1) / L;
        if (last - first + 1 > max_seg) max_seg = (int)(last - first + 1);
      }
      const double cost_sk = L + partial_kb * max_seg + 2.0 * kBK / p.bk;
      if (max_seg <= kMaxSplits && cost_sk < 0.95 * best_cost) {
        p.sk_units = L;
        p.sk_total = (int)total;
        p.splits = max_seg;
        p.grid = (int)((total + L - 1) / L) * p.cluster;
      }
    }
  } else {
    p.splits = 1;
    p.kb_per_split = p.kb_total;
    p.tiles_total = base;
    p.grid = p.tiles_total < kNumSMs ? p.tiles_total : kNumSMs;
  }
  return p;
}

cudaError_t launch_gemm(const GemmPlan& p, const CUtensorMap& map_a, const CUtensorMap& map_b, const GemmOut& out,
                        int* status, uint64_t timeout_ns, cudaStream_t st) {
  KArgs a;
  a.m_tiles = p.m_tiles;
  a.n_tiles = p.n_tiles;
  a.splits = p.splits;
  a.kb_total = p.kb_total;
  a.kb_per_split = p.kb_per_split;
  a.BN = p.BN;
  a.stages = p.stages;
  a.tiles_total = p.tiles_total;
  a.sk_units = p.sk_units;
  a.sk_total = p.sk_total;
  a.split_rows = p.split_rows;
  a.cluster = p.cluster;
  a.tmem_half = p.tmem_half;
  a.out = out;
  a.status = status;
  a.timeout_ns = timeout_ns;
  void (*k)(const CUtensorMap, const CUtensorMap, const KArgs) = nullptr;
  switch (p.epi) {
    case kEpiPartial:
      if (p.cg == 2) k = p.split_act ? k_gemm_tc<kEpiPartial, 1, 64, 2> : k_gemm_tc<kEpiPartial, 0, 64, 2>;
      else if (p.bk == 32) k = p.split_act ? k_gemm_tc<kEpiPartial, 1, 32> : k_gemm_tc<kEpiPartial, 0, 32>;
      else k = p.split_act ? k_gemm_tc<kEpiPartial, 1, 64> : k_gemm_tc<kEpiPartial, 0, 64>;
      break;
    case kEpiSelect: k = p.split_act ? k_gemm_tc<kEpiSelect, 1, 64> : k_gemm_tc<kEpiSelect, 0, 64>; break;
    default: k = p.split_act ? k_gemm_tc<kEpiStore, 1, 64> : k_gemm_tc<kEpiStore, 0, 64>; break;
  }
  if (p.cluster > 1) return launch_k_cluster(k, p.grid, kThreads, p.smem_bytes, st, p.cluster, map_a, map_b, a);
  return launch_k(k, p.grid, kThreads, p.smem_bytes, st, map_a, map_b, a);
}

cudaError_t prepare_gemm_kernels() {
  const int lim = 227 * 1024;
  const void* ks[10] = {(const void*)k_gemm_tc<kEpiPartial, 0, 64>,    (const void*)k_gemm_tc<kEpiPartial, 1, 64>,
                        (const void*)k_gemm_tc<kEpiPartial, 0, 32>,    (const void*)k_gemm_tc<kEpiPartial, 1, 32>,
                        (const void*)k_gemm_tc<kEpiPartial, 0, 64, 2>, (const void*)k_gemm_tc<kEpiPartial, 1, 64, 2>,
                        (const void*)k_gemm_tc<kEpiSelect, 0, 64>,     (const void*)k_gemm_tc<kEpiSelect, 1, 64>,
                        (const void*)k_gemm_tc<kEpiStore, 0, 64>,      (const void*)k_gemm_tc<kEpiStore, 1, 64>};
  cudaError_t e = cudaSuccess;
  for (int i = 0; i < 10 && e == cudaSuccess; ++i)
    e = cudaFuncSetAttribute(ks[i], cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
  for (int i = 0; i < 10 && e == cudaSuccess; ++i)
    e = cudaFuncSetAttribute(ks[i], cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  return e;
}

cudaError_t prepare_kernels() {
  static cudaError_t done = cudaErrorNotReady;
  if (done == cudaSuccess) return done;
  cudaError_t e = prepare_gemm_kernels();
  if (e == cudaSuccess) e = prepare_gemm_fused_kernels();
  if (e == cudaSuccess) e = prepare_attention_kernels();
  if (e == cudaSuccess) e = prepare_attention_tc_kernels();
  if (e == cudaSuccess) e = prepare_small_kernels();
  done = e;
  return e;
}

}  // namespace dd
