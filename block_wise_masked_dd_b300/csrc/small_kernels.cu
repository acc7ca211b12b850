// Bandwidth-trivial kernels of the denoising step: embedding + RMSNorm, the
// split-K reduce epilogues of the linear layers (bf16 store, residual +
// RMSNorm, SwiGLU), the vocab-tile merge of the LM-head select, and the
// commit rule.
#include <math.h>

#include "kernels.h"
#include "ptx.cuh"

namespace dd {

namespace {

constexpr int kNormThreads = 256;

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  float t = 0.f;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) t += red[i];
  return t;
}

__device__ __forceinline__ float bf(const __nv_bfloat16* p, long long i) { return __bfloat162float(p[i]); }

// Store v as a bf16 head at hi[0] and the bf16-rounded remainder at lo[0].
__device__ __forceinline__ void store_split(__nv_bfloat16* hi, __nv_bfloat16* lo, float v) {
  const __nv_bfloat16 h = __float2bfloat16_rn(v);
  *hi = h;
  *lo = __float2bfloat16_rn(v - __bfloat162float(h));
}

// x[r] = E[id] + Pos[i] with id = V ([MASK]) for masked positions;
// y[r] = x / sqrt(mean(x^2) + eps) * g, split into head (row r) and
// remainder (row R + r).  One CTA per row.
__global__ void k_embed_norm(const int32_t* tokens, const uint32_t* mask, const __nv_bfloat16* embed,
                             const __nv_bfloat16* pos, const __nv_bfloat16* g, float* x, __nv_bfloat16* y, int S,
                             int H, int V, float eps) {
  const long long lo_off = (long long)gridDim.x * H;
  __shared__ float red[32];
  extern __shared__ float xs[];
  const int r = blockIdx.x, b = r / S, i = r % S;
  const bool masked = (mask[b] >> i) & 1u;
  // Ids outside [0, V] (never produced by the commit rule) read the [MASK] row.
  const int t = tokens[r];
  const int id = (masked || t < 0 || t > V) ? V : t;
  float ss = 0.f;
  for (int c = threadIdx.x; c < H; c += blockDim.x) {
    const float v = bf(embed, (long long)id * H + c) + bf(pos, (long long)i * H + c);
    xs[c] = v;
    ss += v * v;
  }
  ss = block_sum(ss, red);
  const float rs = rsqrtf(ss / H + eps);
  for (int c = threadIdx.x; c < H; c += blockDim.x) {
    x[(long long)r * H + c] = xs[c];
    store_split(y + (long long)r * H + c, y + lo_off + (long long)r * H + c, xs[c] * rs * bf(g, c));
  }
}

// out[r][n] = sum over splits of part[s][r][n]; bf16 output optionally split
// (remainder at out + total).
template <typename OutT>
__global__ void k_reduce(const float* part, int splits, long long split_stride, long long total, OutT* out,
                         int split) {
  for (long long e = ((long long)blockIdx.x * blockDim.x + threadIdx.x) * 4; e < total;
       e += (long long)gridDim.x * blockDim.x * 4) {
    float4 acc = *reinterpret_cast<const float4*>(part + e);
    for (int s = 1; s < splits; ++s) {
      const float4 v = *reinterpret_cast<const float4*>(part + s * split_stride + e);
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    if constexpr (sizeof(OutT) == 2) {
      __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(out);
      uint2 hi, lo;
      split_bf16(acc.x, acc.y, hi.x, lo.x);
      split_bf16(acc.z, acc.w, hi.y, lo.y);
      *reinterpret_cast<uint2*>(o + e) = hi;
      if (split) *reinterpret_cast<uint2*>(o + total + e) = lo;
    } else {
      *reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + e) = acc;
    }
  }
}

// x[r] += sum_s part[s][r]; y[r] = rmsnorm(x[r]) * g, split into head (row r)
// and remainder (row R + r).  One CTA per row.
__global__ void k_reduce_residual_norm(const float* part, int splits, long long split_stride, float* x,
                                       const __nv_bfloat16* g, __nv_bfloat16* y, int H, float eps) {
  __shared__ float red[32];
  extern __shared__ float xs[];
  const int r = blockIdx.x;
  const long long lo_off = (long long)gridDim.x * H;
  float ss = 0.f;
  for (int c = threadIdx.x; c < H; c += blockDim.x) {
    float v = x[(long long)r * H + c];
    for (int s = 0; s < splits; ++s) v += part[s * split_stride + (long long)r * H + c];
    xs[c] = v;
    ss += v * v;
  }
  ss = block_sum(ss, red);
  const float rs = rsqrtf(ss / H + eps);
  for (int c = threadIdx.x; c < H; c += blockDim.x) {
    x[(long long)r * H + c] = xs[c];
    store_split(y + (long long)r * H + c, y + lo_off + (long long)r * H + c, xs[c] * rs * bf(g, c));
  }
}

// h[r][f] = silu(gate) * up, gate = column f, up = column F + f of the
// summed partials [rows][2F]; split into head and remainder (at h + rows*F).
__global__ void k_reduce_swiglu(const float* part, int splits, long long split_stride, __nv_bfloat16* h, int rows,
                                int F) {
  const long long total = (long long)rows * F;
  for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < total;
       e += (long long)gridDim.x * blockDim.x) {
    const long long r = e / F;
    const int f = (int)(e % F);
    const long long gi = r * 2 * F + f;
    float gt = 0.f, up = 0.f;
    for (int s = 0; s < splits; ++s) {
      gt += part[s * split_stride + gi];
      up += part[s * split_stride + gi + F];
    }
    const float si = gt / (1.f + expf(-gt));
    store_split(h + e, h + total + e, si * up);
  }
}

// Merge per-vocab-tile (max, sumexp, argmax) into conf = 1/sum exp(l - max)
// and the lowest argmax.  One warp per row.
__global__ void k_select_combine(const float* sel_m, const float* sel_s, const int* sel_a, int n_tiles, int rows,
                                 float* conf, int* arg) {
  const int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  float m = -INFINITY, s = 0.f;
  int t_best = 0x7fffffff;
  for (int t = lane; t < n_tiles; t += 32) {
    const float mt = sel_m[(long long)t * rows + r];
    const float st = sel_s[(long long)t * rows + r];
    if (mt > m) {
      s = s * expf(m - mt) + st;
      m = mt;
      t_best = t;
    } else {
      s += st * expf(mt - m);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float mo = __shfl_xor_sync(0xffffffffu, m, o);
    const float so = __shfl_xor_sync(0xffffffffu, s, o);
    const int to = __shfl_xor_sync(0xffffffffu, t_best, o);
    const float mn = fmaxf(m, mo);
    const float a = (m == -INFINITY) ? 0.f : s * expf(m - mn);
    const float c = (mo == -INFINITY) ? 0.f : so * expf(mo - mn);
    int tn;
    if (m > mo) tn = t_best;
    else if (mo > m) tn = to;
    else tn = min(t_best, to);
    m = mn;
    s = a + c;
    t_best = tn;
  }
  if (lane == 0) {
    conf[r] = 1.f / s;
    arg[r] = sel_a[(long long)t_best * rows + r];
  }
}

// Commit rule, one warp per sequence, lane i = block position i (S <= 32).
// Threshold mode: every masked position with conf >= gamma; if none, the
// masked position of highest confidence (lowest position on ties).
// Mock-AR mode: the lowest masked position.  Writes the remaining masked
// count over all sequences to remaining[0].
__global__ void k_commit(const float* conf, const int* arg, int32_t* tokens, uint32_t* mask, const float* params,
                         float gamma_arg, int mode_arg, int32_t* n_committed, int32_t* remaining, int B, int S) {
  __shared__ int left[32];
  const float gamma = params ? params[0] : gamma_arg;
  const int mode = params ? (int)params[1] : mode_arg;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nw = blockDim.x >> 5;
  int my_left = 0;
  for (int b = w; b < B; b += nw) {
    const uint32_t mk = mask[b];
    const bool masked = lane < S && ((mk >> lane) & 1u);
    const float c = lane < S ? conf[b * S + lane] : 0.f;
    uint32_t chosen = 0;
    if (mk != 0) {
      if (mode == 1) {
        chosen = mk & (~mk + 1u);  // lowest set bit
      } else {
        chosen = __ballot_sync(0xffffffffu, masked && c >= gamma);
        if (chosen == 0) {
          float bc = masked ? c : -INFINITY;
          int bi = masked ? lane : 0x7fffffff;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            const float oc = __shfl_xor_sync(0xffffffffu, bc, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (oc > bc || (oc == bc && oi < bi)) { bc = oc; bi = oi; }
          }
          chosen = 1u << bi;
        }
      }
    }
    if (lane < S && ((chosen >> lane) & 1u)) tokens[b * S + lane] = arg[b * S + lane];
    __syncwarp();
    if (lane == 0) {
      const uint32_t nm = mk & ~chosen;
      mask[b] = nm;
      if (n_committed) n_committed[b] = __popc(chosen);
      my_left += __popc(nm);
    }
  }
  if (lane == 0) left[w] = my_left;
  __syncthreads();
  if (threadIdx.x == 0) {
    int t = 0;
    for (int i = 0; i < nw; ++i) t += left[i];
    remaining[0] = t;
  }
}

__global__ void k_set_params(float* params, float gamma, int mode) {
  params[0] = gamma;
  params[1] = (float)mode;
}

__global__ void k_set_int(int* dst, int v) { *dst = v; }

__global__ void k_init_block(int32_t* tokens, uint32_t* mask, int B, int S, int V) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e < B * S) tokens[e] = V;
  if (e < B) mask[e] = S == 32 ? 0xffffffffu : ((1u << S) - 1u);
}

__global__ void k_copy_i32(int32_t* dst, const int32_t* src, int n) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e < n) dst[e] = src[e];
}

// Waits on a barrier that nothing completes, bounded by timeout_ns: the
// timeout path of every pipelined kernel, in isolation.
__global__ void k_wait_forever_bounded(int* status, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait_bounded(&bar, 0, timeout_ns, &abort_flag, status);
}

int grid_for(long long work, int threads) {
  long long b = (work + threads - 1) / threads;
  if (b > 8 * kNumSMs) b = 8 * kNumSMs;
  if (b < 1) b = 1;
  return (int)b;
}

}  // namespace

cudaError_t launch_embed_norm(const int32_t* tokens, const uint32_t* mask, const void* embed, const void* pos,
                              const void* g, float* x, void* y, int B, int S, int H, int V, float eps,
                              cudaStream_t st) {
  k_embed_norm<<<B * S, kNormThreads, H * sizeof(float), st>>>(
      tokens, mask, (const __nv_bfloat16*)embed, (const __nv_bfloat16*)pos, (const __nv_bfloat16*)g, x,
      (__nv_bfloat16*)y, S, H, V, eps);
  return cudaGetLastError();
}

cudaError_t launch_reduce_bf16(const float* part, int splits, long long split_stride, int rows, int N, void* out,
                               int split, cudaStream_t st) {
  const long long total = (long long)rows * N;
  k_reduce<__nv_bfloat16><<<grid_for(total / 4, 256), 256, 0, st>>>(part, splits, split_stride, total,
                                                                    (__nv_bfloat16*)out, split);
  return cudaGetLastError();
}

cudaError_t launch_reduce_f32(const float* part, int splits, long long split_stride, int rows, int N, float* out,
                              cudaStream_t st) {
  const long long total = (long long)rows * N;
  k_reduce<float><<<grid_for(total / 4, 256), 256, 0, st>>>(part, splits, split_stride, total, out, 0);
  return cudaGetLastError();
}

cudaError_t launch_reduce_residual_norm(const float* part, int splits, long long split_stride, float* x,
                                        const void* g, void* y, int rows, int H, float eps, cudaStream_t st) {
  k_reduce_residual_norm<<<rows, kNormThreads, H * sizeof(float), st>>>(part, splits, split_stride, x,
                                                                        (const __nv_bfloat16*)g,
                                                                        (__nv_bfloat16*)y, H, eps);
  return cudaGetLastError();
}

cudaError_t launch_reduce_swiglu(const float* part, int splits, long long split_stride, void* h, int rows, int F,
                                 cudaStream_t st) {
  k_reduce_swiglu<<<grid_for((long long)rows * F, 256), 256, 0, st>>>(part, splits, split_stride,
                                                                      (__nv_bfloat16*)h, rows, F);
  return cudaGetLastError();
}

cudaError_t launch_select_combine(const float* sel_m, const float* sel_s, const int* sel_a, int n_tiles, int rows,
                                  float* conf, int* arg, cudaStream_t st) {
  k_select_combine<<<(rows + 7) / 8, 256, 0, st>>>(sel_m, sel_s, sel_a, n_tiles, rows, conf, arg);
  return cudaGetLastError();
}

cudaError_t launch_commit(const float* conf, const int* arg, int32_t* tokens, uint32_t* mask, const float* params,
                          float gamma, int mode, int32_t* n_committed, int32_t* remaining, int B, int S,
                          cudaStream_t st) {
  int warps = B < 32 ? B : 32;
  if (warps < 1) warps = 1;
  k_commit<<<1, warps * 32, 0, st>>>(conf, arg, tokens, mask, params, gamma, mode, n_committed, remaining, B, S);
  return cudaGetLastError();
}

cudaError_t launch_set_params(float* params, float gamma, int mode, cudaStream_t st) {
  k_set_params<<<1, 1, 0, st>>>(params, gamma, mode);
  return cudaGetLastError();
}

cudaError_t launch_set_int(int* dst, int value, cudaStream_t st) {
  k_set_int<<<1, 1, 0, st>>>(dst, value);
  return cudaGetLastError();
}

cudaError_t launch_init_block(int32_t* tokens, uint32_t* mask, int B, int S, int V, cudaStream_t st) {
  const int n = B * S > B ? B * S : B;
  k_init_block<<<(n + 255) / 256, 256, 0, st>>>(tokens, mask, B, S, V);
  return cudaGetLastError();
}

cudaError_t launch_copy_i32(int32_t* dst, const int32_t* src, int n, cudaStream_t st) {
  k_copy_i32<<<(n + 255) / 256, 256, 0, st>>>(dst, src, n);
  return cudaGetLastError();
}

cudaError_t launch_wait_forever_bounded(int* status, uint64_t timeout_ns, cudaStream_t st) {
  k_wait_forever_bounded<<<1, 32, 0, st>>>(status, timeout_ns);
  return cudaGetLastError();
}

}  // namespace dd
