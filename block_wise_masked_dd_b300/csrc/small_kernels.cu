// Bandwidth-trivial kernels of the denoising step: embedding + RMSNorm, the
// split-K reduce epilogues of the linear layers (bf16 store, residual +
// RMSNorm, SwiGLU), the vocab-tile merge of the LM-head select, and the
// commit rule.  Each kernel waits for its predecessor (programmatic dependent
// launch) before reading its outputs, then lets its successor start.
#include <math.h>

#include "kernels.h"
#include "ptx.cuh"

namespace dd {

namespace {

constexpr int kMaxRowPasses = 2;  // rows up to 2 * 256 * 8 = 4096 wide

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

// 8 bf16 (one 16-byte load) -> fp32
__device__ __forceinline__ void load8_bf16(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

__device__ __forceinline__ void load8_f32(const float* p, float (&v)[8]) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

__device__ __forceinline__ void store8_f32(float* p, const float (&v)[8]) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  *reinterpret_cast<float4*>(p + 4) = make_float4(v[4], v[5], v[6], v[7]);
}

// Store 8 values as bf16 heads at hi and bf16 remainders at lo (16 B each).
__device__ __forceinline__ void store8_split(__nv_bfloat16* hi, __nv_bfloat16* lo, const float (&v)[8]) {
  uint4 h, l;
  split_bf16(v[0], v[1], h.x, l.x);
  split_bf16(v[2], v[3], h.y, l.y);
  split_bf16(v[4], v[5], h.z, l.z);
  split_bf16(v[6], v[7], h.w, l.w);
  *reinterpret_cast<uint4*>(hi) = h;
  *reinterpret_cast<uint4*>(lo) = l;
}

// acc += p[s * stride .. + 8] for s = s0, s0 + 1, ..., s1 - 1 in that order.
// The loads of up to MAXS partials are issued together before the first add,
// so a reduce costs about one round trip per MAXS splits.  The reduce kernels
// are compiled for MAXS = 2, 4 and 8 and launched with the smallest that
// covers the layer's splits: registers held for unused slots would only cap
// the resident warps, and with them the partial bytes in flight.
template <int MAXS>
__device__ __forceinline__ void add_partials(const float* p, int s0, int s1, long long stride, float (&acc)[8]) {
  for (int b = s0; b < s1; b += MAXS) {
    float v[MAXS][8];
#pragma unroll
    for (int j = 0; j < MAXS; ++j)
      if (b + j < s1) load8_f32(p + (long long)(b + j) * stride, v[j]);
#pragma unroll
    for (int j = 0; j < MAXS; ++j) {
      if (b + j < s1) {
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[k] += v[j][k];
      }
    }
  }
}

// y[r] = x[r] * rsqrt(mean(x[r]^2) + eps) * g, written as head (row r) and
// remainder (row R + r); x held in registers (passes of 8 per thread).
// With sq != nullptr the norm is deferred: rs = 1 and sq[r] = sum of x^2.
__device__ __forceinline__ void norm_store(const float (&xv)[kMaxRowPasses][8], int passes, int r, int H, int R,
                                           const float (&gv)[kMaxRowPasses][8], __nv_bfloat16* y, float eps,
                                           float* red, __nv_bfloat16* y2 = nullptr, int r2 = -1,
                                           float* sq = nullptr) {
  float ss = 0.f;
#pragma unroll
  for (int p = 0; p < kMaxRowPasses; ++p) {
    if (p >= passes) break;
#pragma unroll
    for (int i = 0; i < 8; ++i) ss += xv[p][i] * xv[p][i];
  }
  ss = block_sum(ss, red);
  if (sq && threadIdx.x == 0) sq[r] = ss;
  const float rs = sq ? 1.f : rsqrtf(ss / H + eps);
#pragma unroll
  for (int p = 0; p < kMaxRowPasses; ++p) {
    if (p >= passes) break;
    const int c = (p * blockDim.x + threadIdx.x) * 8;
    float yv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) yv[i] = xv[p][i] * rs * gv[p][i];
    store8_split(y + (long long)r * H + c, y + ((long long)R + r) * H + c, yv);
    if (r2 >= 0) store8_split(y2 + (long long)r2 * H + c, y2 + ((long long)R + r2) * H + c, yv);
  }
}

// The gains of this thread's columns (weights: read before the wait on the
// preceding kernel).
__device__ __forceinline__ void load_gains(const __nv_bfloat16* g, int passes, float (&gv)[kMaxRowPasses][8]) {
#pragma unroll
  for (int p = 0; p < kMaxRowPasses; ++p)
    if (p < passes) load8_bf16(g + (p * blockDim.x + threadIdx.x) * 8, gv[p]);
}

// The k-th sequence (in order) whose mask word is non-zero, and the number
// of such sequences, for the calling lanes of warp 0 (lanes < min(32,
// blockDim.x); every one gets both; seq = -1 if there is no k-th).
__device__ __forceinline__ void kth_active(const uint32_t* mask, int B, int k, int& seq, int& n_act) {
  const int lane = threadIdx.x & 31;
  const int nl = blockDim.x < 32 ? (int)blockDim.x : 32;
  const unsigned lanes = nl == 32 ? 0xffffffffu : ((1u << nl) - 1u);
  seq = -1;
  n_act = 0;
  for (int base = 0; base < B; base += nl) {
    const unsigned bal = __ballot_sync(lanes, base + lane < B && mask[base + lane] != 0u);
    const int cnt = __popc(bal);
    if (seq < 0 && k >= n_act && k < n_act + cnt) {
      unsigned m = bal;
      for (int j = 0; j < k - n_act; ++j) m &= m - 1u;
      seq = base + __ffs(m) - 1;
    }
    n_act += cnt;
  }
}

// x[r] = E[id] + Pos[i] with id = V ([MASK]) for masked positions;
// y[r] = RMSNorm(x[r]) * g as head + remainder.  One CTA per row.
//
// With cmp != nullptr the rows are those of the active sequences (any
// position still masked), compacted: row r = k*S + i is position i of the
// k-th active sequence, and rows past the active ones do nothing.  The
// kernel also writes the compaction record the rest of the step reads:
// cmp[0] = active rows, cmp[1] = active sequences, cmp[2 + k] = the k-th
// active sequence, cmp[2 + B + r] = the original row (b*S + i) of row r.
__global__ void k_embed_norm(const int32_t* tokens, const uint32_t* mask, const __nv_bfloat16* embed,
                             const __nv_bfloat16* pos, const __nv_bfloat16* g, float* x, __nv_bfloat16* y, int S,
                             int H, int V, float eps, float* sq, int* cmp, float2* rope_cs, float theta, int D,
                             const int* ctx_len) {
  __shared__ float red[32];
  __shared__ int s_seq;
  const int r = blockIdx.x, i = r % S, R = gridDim.x, B = R / S;
  const int passes = H / (8 * blockDim.x);
  float gv[kMaxRowPasses][8], pv[kMaxRowPasses][8];
  load_gains(g, passes, gv);
#pragma unroll
  for (int p = 0; p < kMaxRowPasses; ++p)
    if (p < passes) load8_bf16(pos + (long long)i * H + (p * blockDim.x + threadIdx.x) * 8, pv[p]);
  pdl_wait();
  pdl_launch_dependents();
  // rotary table of the step: CTA i < S writes block position i's row
  if (rope_cs && r < S) {
    const double p = (double)(*ctx_len + r);
    for (int j = threadIdx.x; j < D / 2; j += blockDim.x)
      rope_cs[r * (D / 2) + j] = rope_cos_sin(p, pow((double)theta, -2.0 * j / D));
  }
  int b = r / S;
  if (cmp) {
    if (threadIdx.x < 32) {  // warp 0 (the whole CTA when it is narrower)
      int seq, n_act;
      kth_active(mask, B, r / S, seq, n_act);
      if (threadIdx.x == 0) {
        s_seq = seq;
        if (r == 0) {
          cmp[0] = n_act * S;
          cmp[1] = n_act;
        }
        if (seq >= 0) {
          cmp[2 + B + r] = seq * S + i;
          if (i == 0) cmp[2 + r / S] = seq;
        }
      }
    }
    __syncthreads();
    if (s_seq < 0) return;
    b = s_seq;
  }
  const bool masked = (mask[b] >> i) & 1u;
  // Ids outside [0, V] (never produced by the commit rule) read the [MASK] row.
  const int t = tokens[b * S + i];
  const int id = (masked || t < 0 || t > V) ? V : t;
  float xv[kMaxRowPasses][8];
#pragma unroll
  for (int p = 0; p < kMaxRowPasses; ++p) {
    if (p >= passes) break;
    const int c = (p * blockDim.x + threadIdx.x) * 8;
    float e[8];
    load8_bf16(embed + (long long)id * H + c, e);
#pragma unroll
    for (int k = 0; k < 8; ++k) xv[p][k] = e[k] + pv[p][k];
    store8_f32(x + (long long)r * H + c, xv[p]);
  }
  norm_store(xv, passes, r, H, R, gv, y, eps, red, nullptr, -1, sq);
}

// x[r] += sum_s part[s][r]; y[r] = RMSNorm(x[r]) * g as head + remainder.
// One CTA per row; the split partial loads of each pass are independent.
// With cmp (the compaction record of k_embed_norm) rows past the active ones
// do nothing, and row r belongs to sequence cmp[2 + r / S].
// (With two slots, four 256-thread CTAs fit an SM: the large decode's 512
// rows run in one wave.  Forcing four slots into the same registers spilled
// and measured no faster.)
template <int MAXS>
__global__ void __launch_bounds__(256, MAXS == 2 ? 4 : 2)
    k_reduce_residual_norm(const float* part, const SlotPlan sp, long long split_stride, float* x,
                                       const __nv_bfloat16* g, __nv_bfloat16* y, int H, float eps,
                                       const uint32_t* mask, int S, __nv_bfloat16* y_c, int* row_index, int* count,
                                       const int* cmp) {
  __shared__ float red[32];
  __shared__ int cpos;
  const int r = blockIdx.x, R = gridDim.x, B = R / S;
  const int passes = H / (8 * blockDim.x);
  float gv[kMaxRowPasses][8];
  load_gains(g, passes, gv);
  pdl_wait();
  pdl_launch_dependents();
  const int n_act = cmp ? cmp[1] : B;
  if (cmp && r >= cmp[0]) {
    if (r == 0 && mask && threadIdx.x == 0) *count = 0;  // no sequence active
    return;
  }
  float xv[kMaxRowPasses][8];
#pragma unroll
  for (int p = 0; p < kMaxRowPasses; ++p) {
    if (p >= passes) break;
    const long long e = (long long)r * H + (p * blockDim.x + threadIdx.x) * 8;
    load8_f32(x + e, xv[p]);
    add_partials<MAXS>(part + e, 0, slots_of(sp, r, (p * blockDim.x + threadIdx.x) * 8), split_stride, xv[p]);
    store8_f32(x + e, xv[p]);
  }
  // With `mask`: the rows still masked are also written, in order, to y_c
  // (rows [0, count) and their remainders at [R, R + count)) for the LM head,
  // with row_index[k] = the original row (b*S + i) of compacted row k.
  int r2 = -1;
  if (mask) {
    // masked rows before this one: the sequences before this row's (their
    // mask words read in parallel, one block sum) plus the positions before i
    const int k = r / S, i = r % S;
    int before = 0, all = 0;
    for (int kk = threadIdx.x; kk < n_act; kk += blockDim.x) {
      const int n = __popc(mask[cmp ? cmp[2 + kk] : kk]);
      before += kk < k ? n : 0;
      all += n;
    }
    before = (int)block_sum((float)before, red);
    if (r == 0) all = (int)block_sum((float)all, red);
    if (threadIdx.x == 0) {
      const int b = cmp ? cmp[2 + k] : k;
      const uint32_t mb = mask[b];
      const bool masked = (mb >> i) & 1u;
      const int pos = before + __popc(mb & ((1u << i) - 1u));
      cpos = masked ? pos : -1;
      if (masked) row_index[pos] = b * S + i;
      if (r == 0) *count = all;
    }
    __syncthreads();
    r2 = cpos;
  }
  norm_store(xv, passes, r, H, R, gv, y, eps, red, y_c, r2);
}

// out[r][n] = sum over splits of part[s][r][n] (fp32; the standalone GEMM).
template <int MAXS>
__global__ void k_reduce(const float* part, const SlotPlan sp, long long split_stride, long long total, int N,
                         float* out) {
  pdl_wait();
  pdl_launch_dependents();
  for (long long e = ((long long)blockIdx.x * blockDim.x + threadIdx.x) * 8; e < total;
       e += (long long)gridDim.x * blockDim.x * 8) {
    float acc[8];
    load8_f32(part + e, acc);
    add_partials<MAXS>(part + e, 1, slots_of(sp, (int)(e / N), (int)(e % N)), split_stride, acc);
    store8_f32(out + e, acc);
  }
}

// q|k|v = the sum of the split-K partials, written as bf16 head (rows
// [0, rows)) + remainder (rows [rows, 2 rows)); with rows_dev only the first
// *rows_dev rows (the active ones).  With theta > 0 the pairs
// (2j, 2j+1) of every query and key head (columns < qk_cols) of row r turn by
// (T + r % S) * theta^(-2j/D) radians, T = *ctx_len: the frequencies and the
// angle in double, the angle reduced modulo 2 pi in double before an fp32
// sine and cosine, the rotation in fp32.  With rope_cs (the step's table of
// those cosines and sines, [S][D/2], written by the embedding kernel) the
// rotation reads them instead of recomputing them per element.
template <int MAXS>
__global__ void k_reduce_qkv(const float* part, const SlotPlan sp, long long split_stride, int rows, int N,
                             __nv_bfloat16* out, int S, int D, int qk_cols, const int* ctx_len, float theta,
                             const int* rows_dev, const float2* rope_cs) {
  __shared__ double freq[64];  // theta^(-2j/D), j < D/2 (D <= 128)
  if (theta > 0.f && !rope_cs && threadIdx.x < D / 2) freq[threadIdx.x] = pow((double)theta, -2.0 * threadIdx.x / D);
  __syncthreads();
  pdl_wait();
  pdl_launch_dependents();
  const long long total = (long long)rows * N;  // remainders start here
  const long long used = rows_dev ? (long long)*rows_dev * N : total;
  const int T = theta > 0.f ? *ctx_len : 0;
  for (long long e = ((long long)blockIdx.x * blockDim.x + threadIdx.x) * 8; e < used;
       e += (long long)gridDim.x * blockDim.x * 8) {
    float acc[8];
    load8_f32(part + e, acc);
    add_partials<MAXS>(part + e, 1, slots_of(sp, (int)(e / N), (int)(e % N)), split_stride, acc);
    const int n = (int)(e % N);
    if (theta > 0.f && n < qk_cols) {
      const int d0 = n % D;
      const int i = (int)(e / N) % S;
      if (rope_cs) {
#pragma unroll
        for (int p = 0; p < 4; ++p) rope_rotate(acc[2 * p], acc[2 * p + 1], rope_cs[i * (D / 2) + (d0 >> 1) + p]);
      } else {
        const double pos = (double)(T + i);
#pragma unroll
        for (int p = 0; p < 4; ++p) rope_pair(acc[2 * p], acc[2 * p + 1], pos, freq[(d0 >> 1) + p]);
      }
    }
    store8_split(out + e, out + total + e, acc);
  }
}

// Context tower, first step: e[r] = embed[tokens[r]] (fp32, the residual
// stream of its attention layer) and y[r] = RMSNorm(e[r]) * g as head +
// remainder (ids outside [0, V) read row 0).  One CTA per row.
__global__ void k_tower_embed_norm(const int32_t* tokens, const __nv_bfloat16* embed, const __nv_bfloat16* g,
                                   float* x, __nv_bfloat16* y, int H, int V, float eps) {
  __shared__ float red[32];
  const int r = blockIdx.x, R = gridDim.x;
  const int passes = H / (8 * blockDim.x);
  float gv[kMaxRowPasses][8];
  load_gains(g, passes, gv);
  pdl_wait();
  pdl_launch_dependents();
  const int t = tokens[r];
  const int id = (t < 0 || t >= V) ? 0 : t;
  float xv[kMaxRowPasses][8];
#pragma unroll
  for (int p = 0; p < kMaxRowPasses; ++p) {
    if (p >= passes) break;
    const int c = (p * blockDim.x + threadIdx.x) * 8;
    load8_bf16(embed + (long long)id * H + c, xv[p]);
    store8_f32(x + (long long)r * H + c, xv[p]);
  }
  norm_store(xv, passes, r, H, R, gv, y, eps, red);
}

// Context tower, causal self-attention inside each committed block: query
// position i of sequence b, head h attends to positions j <= i of the same
// block, softmax(q.k / sqrt(D)) in fp32.  qkv: fp32 [rows][3 * heads * D]
// (q heads, then k, then v); out: bf16 head + remainder [2 * rows][heads * D].
// One CTA per (sequence, head), one warp per query position; lane l holds
// dims l, l + 32, ...
template <int D>
__global__ void k_tower_attention(const float* qkv, __nv_bfloat16* out, int rows, int S, int heads, float scale) {
  constexpr int P = D / 32;
  pdl_wait();
  pdl_launch_dependents();
  const int b = blockIdx.x / heads, h = blockIdx.x % heads;
  const int i = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (i >= S) return;
  const int W = heads * D;
  const float* qrow = qkv + (long long)(b * S + i) * 3 * W + h * D;
  float q[P], acc[P];
#pragma unroll
  for (int k = 0; k < P; ++k) {
    q[k] = qrow[lane + 32 * k];
    acc[k] = 0.f;
  }
  // running max and sum over the keys j <= i (online softmax, one key at a time)
  float m = -INFINITY, l = 0.f;
  for (int j = 0; j <= i; ++j) {
    const float* krow = qkv + (long long)(b * S + j) * 3 * W + W + h * D;
    float d = 0.f;
#pragma unroll
    for (int k = 0; k < P; ++k) d = fmaf(q[k], krow[lane + 32 * k], d);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
    const float s = d * scale;
    const float mn = fmaxf(m, s);
    const float a = expf(m - mn), e = expf(s - mn);
    l = l * a + e;
    const float* vrow = krow + W;
#pragma unroll
    for (int k = 0; k < P; ++k) acc[k] = fmaf(acc[k], a, e * vrow[lane + 32 * k]);
    m = mn;
  }
  const float inv = 1.f / l;
  __nv_bfloat16* o_hi = out + (long long)(b * S + i) * W + h * D;
  __nv_bfloat16* o_lo = o_hi + (long long)rows * W;
#pragma unroll
  for (int k = 0; k < P; ++k) {
    const float v = acc[k] * inv;
    const __nv_bfloat16 hv = __float2bfloat16_rn(v);
    o_hi[lane + 32 * k] = hv;
    o_lo[lane + 32 * k] = __float2bfloat16_rn(v - __bfloat162float(hv));
  }
}

// Context tower, second half: the split-K sum of y W_kv^T (column n of row
// r = b*S + i is layer n / (2 Hkv D), K or V, kv head, dim) rounded to bf16
// and stored at cache position T + i, T = *ctx_len; the last CTA to finish
// then advances *ctx_len by S.
template <int MAXS>
__global__ void k_reduce_kv_append(const float* part, const SlotPlan sp, long long split_stride, int rows, int N, int S,
                                   int B, int Hkv, int D, int alloc_ctx, int* ctx_len, __nv_bfloat16* kc,
                                   __nv_bfloat16* vc, unsigned int* done) {
  pdl_wait();
  pdl_launch_dependents();
  const int T = *ctx_len;
  const long long total = (long long)rows * N;
  const int kvw = Hkv * D;
  for (long long e = ((long long)blockIdx.x * blockDim.x + threadIdx.x) * 8; e < total;
       e += (long long)gridDim.x * blockDim.x * 8) {
    float acc[8];
    load8_f32(part + e, acc);
    add_partials<MAXS>(part + e, 1, slots_of(sp, (int)(e / N), (int)(e % N)), split_stride, acc);
    const int r = (int)(e / N), n = (int)(e % N);
    const int l = n / (2 * kvw), rem = n % (2 * kvw);
    const int h = (rem % kvw) / D, d = rem % D;
    const int b = r / S, i = r % S;
    __nv_bfloat16* dst = (rem < kvw ? kc : vc) + ((((long long)l * B + b) * Hkv + h) * alloc_ctx + T + i) * D + d;
    uint4 o, unused;
    split_bf16(acc[0], acc[1], o.x, unused.x);
    split_bf16(acc[2], acc[3], o.y, unused.y);
    split_bf16(acc[4], acc[5], o.z, unused.z);
    split_bf16(acc[6], acc[7], o.w, unused.w);
    *reinterpret_cast<uint4*>(dst) = o;
  }
  // every CTA has read *ctx_len; the last one to get here moves it on
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(done, 1u) == gridDim.x - 1) {
      *ctx_len = T + S;
      *done = 0;
    }
  }
}

// h[r][f] = silu(gate) * up, gate = column f, up = column F + f of the
// summed partials [rows][2F]; head + remainder (remainder at h + rows*F);
// with rows_dev only the first *rows_dev rows.
template <int MAXS>
__global__ void k_reduce_swiglu(const float* part, const SlotPlan sp, long long split_stride, __nv_bfloat16* h, int rows,
                                int F, const int* rows_dev) {
  pdl_wait();
  pdl_launch_dependents();
  const long long total = (long long)rows * F;  // remainders start here
  const long long used = rows_dev ? (long long)*rows_dev * F : total;
  for (long long e = ((long long)blockIdx.x * blockDim.x + threadIdx.x) * 8; e < used;
       e += (long long)gridDim.x * blockDim.x * 8) {
    const long long r = e / F;
    const int f = (int)(e % F);
    const long long gi = r * 2 * F + f;
    float gt[8], up[8];
    load8_f32(part + gi, gt);
    load8_f32(part + gi + F, up);
    add_partials<MAXS>(part + gi, 1, slots_of(sp, (int)r, f), split_stride, gt);
    add_partials<MAXS>(part + gi + F, 1, slots_of(sp, (int)r, F + f), split_stride, up);
    float hv[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) hv[k] = gt[k] / (1.f + expf(-gt[k])) * up[k];
    store8_split(h + e, h + total + e, hv);
  }
}

// Merge per-vocab-tile (max, sumexp, argmax) into conf = 1/sum exp(l - max)
// and the lowest argmax.  One warp per row.
__global__ void k_select_combine(const float* sel_m, const float* sel_s, const int* sel_a, int n_tiles, int rows,
                                 float* conf, int* arg, const int* count, const int* row_index) {
  pdl_wait();
  pdl_launch_dependents();
  const int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows || (count && r >= *count)) return;
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
    const int dst = row_index ? row_index[r] : r;  // compacted rows go back to their positions
    conf[dst] = 1.f / s;
    arg[dst] = sel_a[(long long)t_best * rows + r];
  }
}

// Positions the fixed-steps schedule commits when `left` of a block of S are
// masked: the schedule commits ceil(left_t / (N - t)) at its step t, so the
// block fills in N steps; t is the first step whose count is at most `left`.
__device__ int steps_schedule_k(int S, int N, int left) {
  int rem = S, t = 0;
  while (rem > left && t < N) {
    rem -= (rem + (N - t) - 1) / (N - t);
    ++t;
  }
  const int steps_left = N - t;
  return steps_left <= 0 ? left : (left + steps_left - 1) / steps_left;
}

// Commit rule, one warp per sequence, lane i = block position i (S <= 32).
// The mode's low byte selects the rule and its upper bits carry k or N.
// Threshold: every masked position with conf >= gamma; if none, the masked
// position of highest confidence (lowest position on ties).  Mock-AR: the
// lowest masked position.  Top-k: the k most confident masked positions.
// Fixed steps: top-k with k from steps_schedule_k.  Writes the remaining masked
// count over all sequences to remaining[0].
__global__ void k_commit(const float* conf, const int* arg, int32_t* tokens, uint32_t* mask, const float* params,
                         float gamma_arg, int mode_arg, int32_t* n_committed, int32_t* remaining, int B, int S) {
  __shared__ int left[32];
  pdl_wait();
  pdl_launch_dependents();
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
    const int base = mode & 0xFF, param = mode >> 8;
    if (mk != 0) {
      if (base == 2 || base == 3) {
        // top-k: the k most confident masked positions (ties: lower position)
        const int k = base == 2 ? param : steps_schedule_k(S, param, __popc(mk));
        int rank = 0;
        for (int j = 0; j < S; ++j) {
          const float cj = __shfl_sync(0xffffffffu, c, j);
          rank += (((mk >> j) & 1u) && (cj > c || (cj == c && j < lane))) ? 1 : 0;
        }
        chosen = __ballot_sync(0xffffffffu, masked && rank < k);
      } else if (base == 1) {
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

// Device-side decode loop.  small: [0] masked positions left, [1] status,
// [3] steps taken in this block, [4] step limit.
__global__ void k_loop_init(int32_t* small, int max_steps) {
  small[3] = 0;
  small[4] = max_steps;
}

// Last kernel of each step in the while-loop graph: count the step and keep
// looping while a position is masked, no kernel timed out and the limit is
// not reached.
__global__ void k_loop_control(int32_t* small, cudaGraphConditionalHandle handle) {
  pdl_wait();  // the commit's remaining count
  const int steps = small[3] + 1;
  small[3] = steps;
  const bool more = small[0] > 0 && small[1] == 0 && steps < small[4];
  cudaGraphSetConditional(handle, more ? 1u : 0u);
}

__global__ void k_init_block(int32_t* tokens, uint32_t* mask, int B, int S, int V) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e < B * S) tokens[e] = V;
  if (e < B) mask[e] = S == 32 ? 0xffffffffu : ((1u << S) - 1u);
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

// The reduce kernels' slot batch for `n` partial slots after the first.
int slot_batch(int n) { return n <= 2 ? 2 : (n <= 4 ? 4 : 8); }

// The instantiation of a reduce kernel for `n` partial slots after the first.
template <typename K>
K pick_batch(int n, K k2, K k4, K k8) {
  const int b = slot_batch(n);
  return b == 2 ? k2 : (b == 4 ? k4 : k8);
}

// threads per row for the row kernels: 8 elements per thread per pass
int row_threads(int H) {
  int t = H / 8;
  if (t > 256) t = 256;
  return t;
}

}  // namespace

// Every kernel of the step runs with the largest shared-memory carveout, the
// one the tensor-core kernels need: an SM then never has to drain to change
// its L1 / shared split before the next kernel's CTAs can join it.
cudaError_t prepare_small_kernels() {
  const void* fns[] = {(const void*)k_embed_norm,              (const void*)k_select_combine,
                       (const void*)k_reduce_residual_norm<2>,  (const void*)k_reduce_residual_norm<4>,
                       (const void*)k_reduce_residual_norm<8>,  (const void*)k_reduce<2>,
                       (const void*)k_reduce<4>,                (const void*)k_reduce<8>,
                       (const void*)k_reduce_swiglu<2>,         (const void*)k_reduce_swiglu<4>,
                       (const void*)k_reduce_swiglu<8>,         (const void*)k_reduce_qkv<2>,
                       (const void*)k_reduce_qkv<4>,            (const void*)k_reduce_qkv<8>,
                       (const void*)k_reduce_kv_append<2>,      (const void*)k_reduce_kv_append<4>,
                       (const void*)k_reduce_kv_append<8>,      (const void*)k_tower_embed_norm,
                       (const void*)k_tower_attention<64>,      (const void*)k_tower_attention<128>,
                       (const void*)k_commit};
  cudaError_t e = cudaSuccess;
  for (const void* f : fns) {
    if (e == cudaSuccess) e = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  }
  return e;
}

cudaError_t launch_embed_norm(const int32_t* tokens, const uint32_t* mask, const void* embed, const void* pos,
                              const void* g, float* x, void* y, int B, int S, int H, int V, float eps,
                              cudaStream_t st, float* sq, int* cmp, float2* rope_cs, float theta, int D,
                              const int* ctx_len) {
  return launch_k(k_embed_norm, B * S, row_threads(H), 0, st, tokens, mask, (const __nv_bfloat16*)embed,
                  (const __nv_bfloat16*)pos, (const __nv_bfloat16*)g, x, (__nv_bfloat16*)y, S, H, V, eps, sq, cmp,
                  rope_cs, theta, D, ctx_len);
}

cudaError_t launch_reduce_qkv(const float* part, const SlotPlan& sp, long long split_stride, int rows, int N, void* out, int S,
                              int D, int qk_cols, const int* ctx_len, float theta, cudaStream_t st,
                              const int* rows_dev, const float2* rope_cs) {
  return launch_k(pick_batch(sp.splits - 1, k_reduce_qkv<2>, k_reduce_qkv<4>, k_reduce_qkv<8>),
                  grid_for((long long)rows * N / 8, 256), 256, 0, st, part, sp, split_stride, rows, N,
                  (__nv_bfloat16*)out, S, D, qk_cols, ctx_len, theta, rows_dev, rope_cs);
}

cudaError_t launch_tower_embed_norm(const int32_t* tokens, const void* embed, const void* g, float* x, void* y,
                                    int rows, int H, int V, float eps, cudaStream_t st) {
  return launch_k(k_tower_embed_norm, rows, row_threads(H), 0, st, tokens, (const __nv_bfloat16*)embed,
                  (const __nv_bfloat16*)g, x, (__nv_bfloat16*)y, H, V, eps);
}

cudaError_t launch_tower_attention(const float* qkv, void* out, int rows, int S, int heads, int D, cudaStream_t st) {
  const float scale = 1.f / sqrtf((float)D);
  const int blocks = (rows / S) * heads;
  if (D == 128)
    return launch_k(k_tower_attention<128>, blocks, S * 32, 0, st, qkv, (__nv_bfloat16*)out, rows, S, heads, scale);
  return launch_k(k_tower_attention<64>, blocks, S * 32, 0, st, qkv, (__nv_bfloat16*)out, rows, S, heads, scale);
}

cudaError_t launch_reduce_kv_append(const float* part, const SlotPlan& sp, long long split_stride, int rows, int N, int S,
                                    int B, int Hkv, int D, int alloc_ctx, int* ctx_len, unsigned int* done, void* kc,
                                    void* vc, cudaStream_t st) {
  return launch_k(pick_batch(sp.splits - 1, k_reduce_kv_append<2>, k_reduce_kv_append<4>, k_reduce_kv_append<8>),
                  grid_for((long long)rows * N / 8, 256), 256, 0, st, part, sp, split_stride, rows, N, S, B, Hkv,
                  D, alloc_ctx, ctx_len, (__nv_bfloat16*)kc, (__nv_bfloat16*)vc, done);
}

cudaError_t launch_reduce_f32(const float* part, const SlotPlan& sp, long long split_stride, int rows, int N, float* out,
                              cudaStream_t st) {
  const long long total = (long long)rows * N;
  return launch_k(pick_batch(sp.splits - 1, k_reduce<2>, k_reduce<4>, k_reduce<8>), grid_for(total / 8, 256), 256, 0,
                  st, part, sp, split_stride, total, N, out);
}

cudaError_t launch_reduce_residual_norm(const float* part, const SlotPlan& sp, long long split_stride, float* x,
                                        const void* g, void* y, int rows, int H, float eps, cudaStream_t st,
                                        const uint32_t* mask, int S, void* y_c, int* row_index, int* count,
                                        const int* cmp) {
  // (its partial loads start at slot 0)
  return launch_k(pick_batch(sp.splits, k_reduce_residual_norm<2>, k_reduce_residual_norm<4>, k_reduce_residual_norm<8>),
                  rows, row_threads(H), 0, st, part, sp, split_stride, x, (const __nv_bfloat16*)g,
                  (__nv_bfloat16*)y, H, eps, mask, S, (__nv_bfloat16*)y_c, row_index, count, cmp);
}

cudaError_t launch_reduce_swiglu(const float* part, const SlotPlan& sp, long long split_stride, void* h, int rows, int F,
                                 cudaStream_t st, const int* rows_dev) {
  return launch_k(pick_batch(sp.splits - 1, k_reduce_swiglu<2>, k_reduce_swiglu<4>, k_reduce_swiglu<8>),
                  grid_for((long long)rows * F / 8, 256), 256, 0, st, part, sp, split_stride, (__nv_bfloat16*)h,
                  rows, F, rows_dev);
}

cudaError_t launch_select_combine(const float* sel_m, const float* sel_s, const int* sel_a, int n_tiles, int rows,
                                  float* conf, int* arg, cudaStream_t st, const int* count, const int* row_index) {
  return launch_k(k_select_combine, (rows + 7) / 8, 256, 0, st, sel_m, sel_s, sel_a, n_tiles, rows, conf, arg, count,
                  row_index);
}

cudaError_t launch_commit(const float* conf, const int* arg, int32_t* tokens, uint32_t* mask, const float* params,
                          float gamma, int mode, int32_t* n_committed, int32_t* remaining, int B, int S,
                          cudaStream_t st) {
  int warps = B < 32 ? B : 32;
  if (warps < 1) warps = 1;
  return launch_k(k_commit, 1, warps * 32, 0, st, conf, arg, tokens, mask, params, gamma, mode, n_committed,
                  remaining, B, S);
}

cudaError_t launch_set_params(float* params, float gamma, int mode, cudaStream_t st) {
  k_set_params<<<1, 1, 0, st>>>(params, gamma, mode);
  return cudaGetLastError();
}

cudaError_t launch_set_int(int* dst, int value, cudaStream_t st) {
  k_set_int<<<1, 1, 0, st>>>(dst, value);
  return cudaGetLastError();
}

cudaError_t launch_loop_init(int32_t* small, int max_steps, cudaStream_t st) {
  k_loop_init<<<1, 1, 0, st>>>(small, max_steps);
  return cudaGetLastError();
}

cudaError_t launch_loop_control(int32_t* small, cudaGraphConditionalHandle handle, cudaStream_t st) {
  return launch_k(k_loop_control, 1, 1, 0, st, small, handle);
}

cudaError_t launch_init_block(int32_t* tokens, uint32_t* mask, int B, int S, int V, cudaStream_t st) {
  const int n = B * S > B ? B * S : B;
  k_init_block<<<(n + 255) / 256, 256, 0, st>>>(tokens, mask, B, S, V);
  return cudaGetLastError();
}

cudaError_t launch_wait_forever_bounded(int* status, uint64_t timeout_ns, cudaStream_t st) {
  k_wait_forever_bounded<<<1, 32, 0, st>>>(status, timeout_ns);
  return cudaGetLastError();
}

}  // namespace dd
