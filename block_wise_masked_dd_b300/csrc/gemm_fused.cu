// Linear layers of the denoising step with their split-K reduction and
// elementwise epilogue inside the GEMM (tcgen05 + TMA), so a layer is one
// launch instead of a GEMM plus a reduce kernel.
//
// Work split: the grid is G groups of gs CTAs, at most one CTA per SM and at
// most one CTA per SM's worth of grid, so every CTA is resident at once.  A
// group owns one 128-feature weight tile at a time (groups walk the tiles);
// CTA rank r of the group multiplies K blocks [r*kbps, (r+1)*kbps) of the tile
// against every activation row, so the gs CTAs stream disjoint weight bytes.
// Each CTA writes its fp32 accumulator tile ([row][feature], from TMEM) to a
// double-buffered scratch slot in global memory (it stays in L2), then
// raises the group's arrival counter; once the counter shows all gs partials
// of the tile, CTA r sums rows r, r+gs, r+2gs, ... over them (always in rank
// order) and applies the layer's epilogue.  A group waits only on its own
// members, all resident, so the waits always end; they are bounded all the
// same.  The last member to finish resets the group's counters for the next
// launch.  The accumulator is double-buffered in TMEM, so the MMAs of a
// group's next tile run during this epilogue.
//
// Epilogues (see FusedOp): q|k|v with rotary positions, SwiGLU over a tile
// made of 64 gate and the matching 64 up rows of the weight, and the residual
// update whose RMSNorm is deferred to the consuming GEMM (x * g is stored and
// the consumer scales each row by rsqrt(mean x^2 + eps), summing per-tile
// squares this epilogue writes).  The normalisation is the RMSNorm of the
// TwoTower article's dense stand-in block; deferring it changes only the
// rounding order.
//
// Inside the step graph of the small decode workload (128 rows) this path
// measured slower than plain GEMMs followed by reduce kernels (20.2k against
// 24.8k committed tokens/s): under programmatic dependent launch a reduce
// kernel overlaps the GEMM's drain and the next GEMM's first weight loads,
// while a reduction at the end of the GEMM is wholly on the critical path.
// The step runs it only when DD_OPT_FUSED_REDUCE asks for it.
//
// Roles (192 threads) as in the plain GEMM: warp 0 issues TMA loads, warp 1
// owns TMEM and issues the MMAs, warps 2-5 run the epilogue.  Every wait is
// bounded; a decision that ends the epilogue loop is taken jointly by its four
// warps (bar.red), so no named barrier is ever left short.
#include <math.h>

#include "kernels.h"
#include "ptx.cuh"

namespace dd {

namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;
constexpr int kEpiBar = 1;              // named barrier of the epilogue warps (0 is __syncthreads)
constexpr int kStageA = kBM * kBK * 2;  // 16 KB weight tile per K block
constexpr int kMaxGroup = 8;     // CTAs that split one tile's K, at most
constexpr int kRB = 4;           // rows an epilogue warp reduces per batch (their loads issued together)

struct FArgs {
  int m_tiles, kb_total, kb_per_split, BN, stages, rows, F;
  int gs;  // group size (K splits of a tile)
  uint32_t tmem_half;
  FusedOut o;
  int* status;
  uint64_t timeout_ns;
};

// One pipeline stage: the weight tile, then the activation heads and remainders.
__host__ __device__ inline int fused_stage_bytes(int BN) { return kStageA + 2 * BN * kBK * 2; }
// One fp32 partial tile [BN rows][128 features] in the global scratch.
__host__ __device__ inline int fused_partial_elems(int BN) { return BN * kBM; }
// Alignment slack, stages, mbarriers, the rotary frequency table (64
// doubles), the per-row norm scales (128 floats), the TMEM address and the
// abort flag.
__host__ inline int fused_smem_bytes(int BN, int stages) {
  return 1024 + stages * fused_stage_bytes(BN) + (2 * stages + 5) * 8 + 64 * 8 + 128 * 4 + 16;
}

// Spin until *p >= target (acquire, GPU scope), bounded like the mbarrier waits.
__device__ __forceinline__ bool wait_count_bounded(const unsigned* p, unsigned target, uint64_t limit_ns,
                                                   volatile int* abort, int* status) {
  auto load = [&]() {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
  };
  if (load() >= target) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (load() >= target) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      *abort = 1;
      if (status) atomicExch(status, kStatusTimeout);
      return false;
    }
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ void store4_split(__nv_bfloat16* hi, __nv_bfloat16* lo, float a, float b, float c,
                                             float d) {
  uint2 h, r;
  split_bf16(a, b, h.x, r.x);
  split_bf16(c, d, h.y, r.y);
  *reinterpret_cast<uint2*>(hi) = h;
  *reinterpret_cast<uint2*>(lo) = r;
}

// The epilogue of activation row j for this lane's four features of tile t:
// v = the group's sum over K of those four outputs; rs = the row's deferred
// norm scale (kOpQkv, kOpSwiglu); xv = x at those features and gv the gains
// (kOpResidual).
template <int OP>
__device__ __forceinline__ void epilogue_row(const FArgs& args, int t, int j, int lane, float4 v, float rs,
                                             float4 xv, float4 gv, const double* freq, int T) {
  const FusedOut& o = args.o;
  const int R = args.rows;
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(o.out);
  if (OP == kOpResidual) {
    const int f = t * kBM + 4 * lane;
    xv.x += v.x;
    xv.y += v.y;
    xv.z += v.z;
    xv.w += v.w;
    *reinterpret_cast<float4*>(o.x + (long long)j * o.ld + f) = xv;
    store4_split(out + (long long)j * o.ld + f, out + (long long)(R + j) * o.ld + f, xv.x * gv.x, xv.y * gv.y,
                 xv.z * gv.z, xv.w * gv.w);
    const float ss = warp_sum(xv.x * xv.x + xv.y * xv.y + xv.z * xv.z + xv.w * xv.w);
    if (lane == 0) o.sq_out[(long long)t * R + j] = ss;
    return;
  }
  v.x *= rs;
  v.y *= rs;
  v.z *= rs;
  v.w *= rs;
  if (OP == kOpQkv) {
    const int f = t * kBM + 4 * lane;
    if (o.theta > 0.f && f < o.qk_cols) {
      const int d0 = f % o.D;
      const double pos = (double)(T + j % o.S);
      rope_pair(v.x, v.y, pos, freq[d0 >> 1]);
      rope_pair(v.z, v.w, pos, freq[(d0 >> 1) + 1]);
    }
    store4_split(out + (long long)j * o.ld + f, out + (long long)(R + j) * o.ld + f, v.x, v.y, v.z, v.w);
  } else {
    // lanes 0-15 hold gate features 4*lane.., lanes 16-31 the matching up features
    const float u0 = __shfl_down_sync(0xffffffffu, v.x, 16);
    const float u1 = __shfl_down_sync(0xffffffffu, v.y, 16);
    const float u2 = __shfl_down_sync(0xffffffffu, v.z, 16);
    const float u3 = __shfl_down_sync(0xffffffffu, v.w, 16);
    if (lane < 16) {
      const int f = t * 64 + 4 * lane;
      store4_split(out + (long long)j * o.ld + f, out + (long long)(R + j) * o.ld + f,
                   v.x / (1.f + expf(-v.x)) * u0, v.y / (1.f + expf(-v.y)) * u1, v.z / (1.f + expf(-v.z)) * u2,
                   v.w / (1.f + expf(-v.w)) * u3);
    }
  }
}

template <int OP>
__global__ void __launch_bounds__(kThreads, 1)
    k_gemm_fused(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_x,
                 const FArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int BN = args.BN;
  const int stage_b = BN * kBK * 2;
  const int stage_bytes = fused_stage_bytes(BN);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + args.stages * stage_bytes);
  uint64_t* empty = full + args.stages;
  uint64_t* acc_full = empty + args.stages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  double* freq = reinterpret_cast<double*>(drain + 1);
  float* rs_s = reinterpret_cast<float*>(freq + 64);  // deferred norm scale of each activation row
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(rs_s + 128);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int cs = args.gs;
  const int rank = (int)blockIdx.x % cs;
  const int cid = (int)blockIdx.x / cs;  // group
  const int ncl = (int)gridDim.x / cs;   // groups
  const int warp = warp_id();
  const int lane = lane_id();
  const int kb0 = rank * args.kb_per_split;
  const int kb1 = min(args.kb_total, kb0 + args.kb_per_split);

  if (threadIdx.x == 0) {
    for (int s = 0; s < args.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&map_w);
    tma_prefetch_desc(&map_x);
  }
  if (OP == kOpQkv && threadIdx.x < 64)
    freq[threadIdx.x] = (args.o.theta > 0.f && (int)threadIdx.x < args.o.D / 2)
                            ? pow((double)args.o.theta, -2.0 * threadIdx.x / args.o.D)
                            : 0.0;
  if (warp == 1) {
    tmem_alloc(tmem_slot, 2 * args.tmem_half);
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      // Weight loads of the first stages go out before the wait on the
      // preceding kernel, the activation loads of those stages right after.
      auto load_w = [&](uint8_t* sa, int s, int kb, int t) {
        if (OP == kOpSwiglu) {
          tma_load_2d(sa, &map_w, &full[s], kb * kBK, t * 64);
          tma_load_2d(sa + kStageA / 2, &map_w, &full[s], kb * kBK, args.F + t * 64);
        } else {
          tma_load_2d(sa, &map_w, &full[s], kb * kBK, t * kBM);
        }
      };
      auto load_x = [&](uint8_t* sa, int s, int kb) {
        tma_load_2d(sa + kStageA, &map_x, &full[s], kb * kBK, 0);
        tma_load_2d(sa + kStageA + stage_b, &map_x, &full[s], kb * kBK, args.rows);
      };
      int s = 0;
      uint32_t phase = 0;
      bool ok = true, waited = false;
      int pend_s[8], pend_kb[8], pend_n = 0;
      for (int t = cid; t < args.m_tiles && ok; t += ncl) {
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait_bounded(&empty[s], phase ^ 1, args.timeout_ns, abort_flag, args.status)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + s * stage_bytes;
          mbar_arrive_expect_tx(&full[s], stage_bytes);
          load_w(sa, s, kb, t);
          if (waited) {
            load_x(sa, s, kb);
          } else {
            pend_s[pend_n] = s;
            pend_kb[pend_n] = kb;
            ++pend_n;
            if (pend_n == args.stages || pend_n == 8 || kb == kb1 - 1) {
              pdl_wait();
              pdl_launch_dependents();
              waited = true;
              for (int i = 0; i < pend_n; ++i) load_x(smem + pend_s[i] * stage_bytes, pend_s[i], pend_kb[i]);
            }
          }
          if (++s == args.stages) {
            s = 0;
            phase ^= 1;
          }
        }
      }
      if (!waited) {
        pdl_wait();
        pdl_launch_dependents();
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA
    if (lane == 0) {
      bool ok = true;
      int s = 0;
      uint32_t phase = 0;
      int it = 0;
      const uint32_t idesc = idesc_bf16_f32(kBM, BN);
      for (int t = cid; t < args.m_tiles && ok; t += ncl, ++it) {
        const int ab = it & 1;
        const uint32_t aphase = (it >> 1) & 1;
        if (!mbar_wait_bounded(&acc_empty[ab], aphase ^ 1, args.timeout_ns, abort_flag, args.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + ab * args.tmem_half;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait_bounded(&full[s], phase, args.timeout_ns, abort_flag, args.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + s * stage_bytes);
          const uint32_t b_addr = a_addr + kStageA;
          const uint32_t lo_addr = b_addr + stage_b;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            tc_mma_bf16(d_tmem, smem_desc_sw128(a_addr + k * 32), smem_desc_sw128(b_addr + k * 32), idesc,
                        (kb > kb0 || k > 0) ? 1u : 0u);
            tc_mma_bf16(d_tmem, smem_desc_sw128(a_addr + k * 32), smem_desc_sw128(lo_addr + k * 32), idesc, 1u);
          }
          tc_commit(&empty[s]);
          if (++s == args.stages) {
            s = 0;
            phase ^= 1;
          }
        }
        if (ok) tc_commit(&acc_full[ab]);
      }
      // every MMA issued here completes before TMEM is released
      tc_commit(drain);
      volatile int no_abort = 0;
      mbar_wait_bounded(drain, 0, args.timeout_ns, &no_abort, args.status);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lane quarter of this warp
    const int et = threadIdx.x - 64;
    pdl_wait();  // x, the squares and the context length come from preceding kernels
    const int T = (OP == kOpQkv && args.o.theta > 0.f) ? *args.o.ctx_len : 0;
    if (OP != kOpResidual && et < BN) {
      // the row scales do not depend on the tile: once, during the first mainloop
      const float* sq = args.o.sq_in + et;
      float ss = 0.f;
      int k = 0;
      for (; k + 8 <= args.o.n_sq; k += 8) {
        float a[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) a[u] = sq[(long long)(k + u) * args.rows];
#pragma unroll
        for (int u = 0; u < 8; ++u) ss += a[u];
      }
      for (; k < args.o.n_sq; ++k) ss += sq[(long long)k * args.rows];
      rs_s[et] = rsqrtf(ss / args.o.hidden + args.o.eps);
    }
    // this CTA's rows: rank, rank + cs, ... (owned of them)
    const int owned = BN > rank ? (BN - rank + cs - 1) / cs : 0;
    unsigned* arrivals = args.o.cnt + 2 * cid;  // [0] partials written, [1] members finished
    auto slot = [&](int member, int buf) {
      return args.o.xpart + ((long long)(cid * cs + member) * 2 + buf) * fused_partial_elems(BN);
    };
    int it = 0;
    for (int t = cid; t < args.m_tiles; t += ncl, ++it) {
      const int ab = it & 1;
      const uint32_t aphase = (it >> 1) & 1;
      const int buf = it & 1;
      bool w = true;
      if (et == 0) w = mbar_wait_bounded(&acc_full[ab], aphase, args.timeout_ns, abort_flag, args.status);
      if (!bar_and(kEpiBar, kEpiThreads, w)) break;
      tc_fence_after();
      // accumulator (TMEM lane = feature, column = activation row) -> this
      // member's scratch slot [row][feature].  The slot of two tiles back is
      // free: every member passed the previous tile's count, which it raised
      // only after reading that tile's partials.
      const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + ab * args.tmem_half;
      const int lf = q * 32 + lane;
      float* mine = slot(rank, buf);
      int c = 0;
      for (; c + 64 <= BN; c += 64) {
        float v[64];
        tmem_ld64(tbase + c, v);
#pragma unroll
        for (int j = 0; j < 64; ++j) mine[(c + j) * kBM + lf] = v[j];
      }
      for (; c < BN; c += 16) {
        float v[16];
        tmem_ld16(tbase + c, v);
#pragma unroll
        for (int j = 0; j < 16; ++j) mine[(c + j) * kBM + lf] = v[j];
      }
      tc_fence_before();
      __threadfence();
      bar_and(kEpiBar, kEpiThreads, true);  // the whole partial is written and the TMEM buffer read
      w = true;
      if (et == 0) {
        mbar_arrive(&acc_empty[ab]);
        atomicAdd(&arrivals[0], 1u);
        w = wait_count_bounded(&arrivals[0], (unsigned)(cs * (it + 1)), args.timeout_ns, abort_flag, args.status);
        __threadfence();
      }
      if (!bar_and(kEpiBar, kEpiThreads, w)) break;
      // Owned rows in batches of kRB consecutive ones, batch b to the warp of
      // quarter b % 4; a batch's loads (staged partials of every rank, and x)
      // all go out before the first sum.
      float4 gv = make_float4(0.f, 0.f, 0.f, 0.f);
      if (OP == kOpResidual) {
        const uint2 gr =
            *reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(args.o.g) + t * kBM + 4 * lane);
        gv = make_float4(__uint_as_float(gr.x << 16), __uint_as_float(gr.x & 0xffff0000u),
                         __uint_as_float(gr.y << 16), __uint_as_float(gr.y & 0xffff0000u));
      }
      for (int k0 = q * kRB; k0 < owned; k0 += 4 * kRB) {
        float4 xv[kRB];
        float4 v[kRB][kMaxGroup];
#pragma unroll
        for (int b = 0; b < kRB; ++b) {
          const int j = rank + cs * (k0 + b);
          xv[b] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (OP == kOpResidual && k0 + b < owned)
            xv[b] = *reinterpret_cast<const float4*>(args.o.x + (long long)j * args.o.ld + t * kBM + 4 * lane);
        }
#pragma unroll
        for (int b = 0; b < kRB; ++b) {
          // member p's slot lies p * 2 partial tiles after member 0's
          const float* pb = slot(0, buf) + (rank + cs * (k0 + b)) * kBM + 4 * lane;
#pragma unroll
          for (int p = 0; p < kMaxGroup; ++p)
            if (k0 + b < owned && p < cs)
              v[b][p] = __ldcg(reinterpret_cast<const float4*>(pb + (long long)p * 2 * fused_partial_elems(BN)));
        }
#pragma unroll
        for (int b = 0; b < kRB; ++b) {
          if (k0 + b >= owned) break;
          const int j = rank + cs * (k0 + b);
          float4 acc = v[b][0];
#pragma unroll
          for (int p = 1; p < kMaxGroup; ++p) {
            if (p < cs) {
              acc.x += v[b][p].x;
              acc.y += v[b][p].y;
              acc.z += v[b][p].z;
              acc.w += v[b][p].w;
            }
          }
          epilogue_row<OP>(args, t, j, lane, acc, OP == kOpResidual ? 1.f : rs_s[j], xv[b], gv, freq, T);
        }
      }
    }
    // The last member to finish resets the group's counters: every member
    // has passed its last wait on them.
    bar_and(kEpiBar, kEpiThreads, true);
    if (et == 0) {
      __threadfence();
      if (atomicAdd(&arrivals[1], 1u) == (unsigned)(cs - 1)) {
        atomicExch(&arrivals[0], 0u);
        atomicExch(&arrivals[1], 0u);
      }
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 2 * args.tmem_half);
  }
}

using FusedKernel = void (*)(const CUtensorMap, const CUtensorMap, const FArgs);

FusedKernel fused_kernel(int op) {
  switch (op) {
    case kOpQkv: return k_gemm_fused<kOpQkv>;
    case kOpSwiglu: return k_gemm_fused<kOpSwiglu>;
    default: return k_gemm_fused<kOpResidual>;
  }
}

uint32_t pow2_cols(uint32_t v) {
  uint32_t p = 32;
  while (p < v) p <<= 1;
  return p;
}

}  // namespace

GemmPlan plan_gemm_fused(int op, int rows, int N, int K) {
  GemmPlan p{};
  p.epi = kEpiPartial;
  p.fused_op = -1;
  p.split_act = 1;
  p.split_rows = rows;
  if (rows < 16 || rows > 128 || rows % 16 || N < kBM || N % kBM || K < kBK || K % kBK) return p;
  p.BN = rows;
  p.m_tiles = N / kBM;
  p.n_tiles = 1;
  p.kb_total = K / kBK;
  int stages = (227 * 1024 - fused_smem_bytes(rows, 0)) / (fused_stage_bytes(rows) + 16);
  if (stages > 8) stages = 8;
  if (stages < 2) return p;
  p.stages = stages;
  p.smem_bytes = fused_smem_bytes(rows, stages);
  p.tmem_half = pow2_cols(rows);
  // One CTA per SM (shared memory), at most kNumSMs CTAs: all resident at
  // once.  Cost in microseconds: the busiest CTA's weight bytes at about the
  // fair share of HBM per SM (48 GB/s) against the whole weight at 6.4 TB/s,
  // plus an exchange per tile round and a small charge per group member.
  const double weight_us = (double)N * K * 2 / 6.4e6;
  double best = -1.0;
  for (int gs = 1; gs <= kMaxGroup && gs <= p.kb_total; ++gs) {
    const int kbps = (p.kb_total + gs - 1) / gs;
    if ((p.kb_total + kbps - 1) / kbps != gs) continue;  // every member gets at least one K block
    const int groups = kNumSMs / gs < p.m_tiles ? kNumSMs / gs : p.m_tiles;
    if (groups < 1) continue;
    const int rounds = (p.m_tiles + groups - 1) / groups;
    const double sm_us = (double)rounds * kbps * kStageA / 48e3;
    const double cost = (sm_us > weight_us ? sm_us : weight_us) + 0.3 * rounds + 0.05 * gs;
    if (best < 0 || cost < best) {
      best = cost;
      p.splits = gs;
      p.kb_per_split = kbps;
      p.grid = groups * gs;
    }
  }
  if (best < 0) return p;
  p.tiles_total = p.m_tiles;
  p.fused_op = op;
  return p;
}

size_t fused_scratch_bytes(int rows) { return (size_t)kNumSMs * 2 * fused_partial_elems(rows) * 4; }
size_t fused_counter_bytes() { return (size_t)kNumSMs * 2 * 4; }

cudaError_t launch_gemm_fused(const GemmPlan& p, const CUtensorMap& map_w, const CUtensorMap& map_x,
                              const FusedOut& out, int* status, uint64_t timeout_ns, cudaStream_t st) {
  if (p.fused_op < 0 || p.splits < 1 || p.grid % p.splits || p.grid > kNumSMs || !out.xpart || !out.cnt)
    return cudaErrorInvalidValue;
  FArgs a;
  a.m_tiles = p.m_tiles;
  a.kb_total = p.kb_total;
  a.kb_per_split = p.kb_per_split;
  a.BN = p.BN;
  a.stages = p.stages;
  a.rows = p.split_rows;
  a.F = p.fused_op == kOpSwiglu ? p.m_tiles * 64 : 0;  // the up rows follow the F gate rows
  a.gs = p.splits;
  a.tmem_half = p.tmem_half;
  a.o = out;
  a.status = status;
  a.timeout_ns = timeout_ns;
  return launch_k(fused_kernel(p.fused_op), p.grid, kThreads, p.smem_bytes, st, map_w, map_x, a);
}

cudaError_t prepare_gemm_fused_kernels() {
  cudaError_t e = cudaSuccess;
  for (int op = 0; op < 3 && e == cudaSuccess; ++op) {
    const void* k = (const void*)fused_kernel(op);
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  }
  return e;
}

}  // namespace dd
