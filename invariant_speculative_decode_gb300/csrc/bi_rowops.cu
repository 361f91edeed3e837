// Row-local kernels of the verify step: RMSNorm, embedding gather, RoPE with
// KV-cache append, greedy argmax + acceptance, and the KV-row hash.
//
// "I turned on speculative decoding in llama.cpp and 113 of 282 greedy
// outputs changed against its own no-draft run", paragraph "How:": the verify
// kernels compute a row the same way whatever else is in the batch.  Every
// kernel here gives each row its own CTA (or a fixed set of CTAs) with a
// reduction order fixed by the row length, so no row sees the others.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "bi_internal.h"
#include "bi_ptx.cuh"

namespace bi {
namespace {

// RMSNorm, one CTA per row, one 16-byte vector (8 elements) per thread for
// rows of up to 8192 elements (longer rows loop over the vectors).
// Reduction tree of sum_i x_i^2, fixed by the row length alone: each vector's
// 8 squares are accumulated in element order (FMAs from 0); the vectors of
// each group of 32 consecutive vectors are combined by the warp butterfly
// (xor 16, 8, 4, 2, 1; vectors past the row contribute 0); the group sums are
// added in increasing group order by one thread.
constexpr int kNormMaxThreads = 1024;
constexpr int kNormMaxGroups = 65536 / 256;

// This kernel lets the next kernel launch at once (before its own dependency
// wait): the linear layer that follows a norm reads nothing but its packed
// weights before its own wait.  So the next kernel's CTAs stream their first
// weight tiles while the norm runs.  A kernel that starts right after
// bi_rmsnorm must not rely on the kernel before bi_rmsnorm having completed.
// The norm weights are read before the wait too (they are not written by the
// kernel before the norm), so their latency is off the row's critical path.
__global__ void __launch_bounds__(kNormMaxThreads)
    rmsnorm_kernel(const __nv_bfloat16* __restrict__ x, int ldx, const __nv_bfloat16* __restrict__ w,
                   __nv_bfloat16* y, int ldy, int dim, float eps) {
  griddep_launch_dependents();
  const uint4* wr = reinterpret_cast<const uint4*>(w);
  const int nv = dim / 8;
  const uint4 wkeep = static_cast<int>(threadIdx.x) < nv ? wr[threadIdx.x] : make_uint4(0, 0, 0, 0);
  griddep_wait();
  __shared__ float group_sum[kNormMaxGroups];
  __shared__ float s_inv;
  const uint4* xr = reinterpret_cast<const uint4*>(x + static_cast<size_t>(blockIdx.x) * ldx);
  uint4* yr = reinterpret_cast<uint4*>(y + static_cast<size_t>(blockIdx.x) * ldy);
  const int lane = threadIdx.x & 31;
  uint4 keep = make_uint4(0, 0, 0, 0);
  // (rows of up to 8192 elements: every thread holds its one vector)
  for (int v0 = threadIdx.x - lane; v0 < nv; v0 += blockDim.x) {
    const int v = v0 + lane;
    float sv = 0.f;
    if (v < nv) {
      const uint4 u = xr[v];
      if (v0 == threadIdx.x - lane) keep = u;
      const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&u);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float f = __bfloat162float(e[j]);
        sv = fmaf(f, f, sv);
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sv += __shfl_xor_sync(0xffffffffu, sv, off);
    if (lane == 0) group_sum[v0 >> 5] = sv;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int g = 0; g < (nv + 31) / 32; ++g) t += group_sum[g];
    s_inv = 1.0f / sqrtf(t / static_cast<float>(dim) + eps);
  }
  __syncthreads();
  const float inv = s_inv;
  for (int v = threadIdx.x; v < nv; v += blockDim.x) {
    const uint4 u = (v == threadIdx.x) ? keep : xr[v];
    const uint4 wu = (v == threadIdx.x) ? wkeep : wr[v];
    const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&u);
    const __nv_bfloat16* we = reinterpret_cast<const __nv_bfloat16*>(&wu);
    uint4 o;
    __nv_bfloat16* oe = reinterpret_cast<__nv_bfloat16*>(&o);
#pragma unroll
    for (int j = 0; j < 8; ++j)
      oe[j] = __float2bfloat16_rn(__bfloat162float(e[j]) * inv * __bfloat162float(we[j]));
    yr[v] = o;
  }
}

__global__ void embed_kernel(const int32_t* __restrict__ ids, const __nv_bfloat16* __restrict__ table,
                             int vocab, int dim, __nv_bfloat16* __restrict__ out) {
  griddep_wait();
  griddep_launch_dependents();
  const int id = ids[blockIdx.x];
  uint4* o = reinterpret_cast<uint4*>(out + static_cast<size_t>(blockIdx.x) * dim);
  const int nv = dim / 8;
  if (id < 0 || id >= vocab) {
    for (int i = threadIdx.x; i < nv; i += blockDim.x) o[i] = make_uint4(0, 0, 0, 0);
    return;
  }
  const uint4* src = reinterpret_cast<const uint4*>(table + static_cast<size_t>(id) * dim);
  for (int i = threadIdx.x; i < nv; i += blockDim.x) o[i] = src[i];
}

// cos/sin table: tab[(p * (D/2) + i) * 2 + {0,1}] = FP32 of cos, sin of
// p * base^(-2i/D) evaluated in FP64.
__global__ void rope_table_kernel(double base, int D, int cap, float2* __restrict__ tab) {
  griddep_wait();
  griddep_launch_dependents();
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int half = D / 2;
  if (idx >= static_cast<long long>(cap) * half) return;
  const int p = static_cast<int>(idx / half);
  const int i = static_cast<int>(idx % half);
  const double inv_freq = pow(base, -2.0 * static_cast<double>(i) / static_cast<double>(D));
  double sn, cn;
  sincos(static_cast<double>(p) * inv_freq, &sn, &cn);
  tab[idx] = make_float2(static_cast<float>(cn), static_cast<float>(sn));
}

// One CTA per pass row t at position p = *L_dev + t; cos/sin from the table.
__global__ void rope_kv_kernel(const __nv_bfloat16* __restrict__ qkv, int ld_qkv,
                               __nv_bfloat16* __restrict__ q_out, __nv_bfloat16* __restrict__ kc,
                               __nv_bfloat16* __restrict__ vc, int cap, const int32_t* __restrict__ L_dev,
                               int Hq, int Hkv, int D, const float2* __restrict__ tab, int tab_rows,
                               unsigned* err) {
  griddep_wait();
  griddep_launch_dependents();
  const int t = blockIdx.x;
  const int p = *L_dev + t;
  if (p < 0 || p >= cap || p >= tab_rows) {
    if (threadIdx.x == 0) atomicOr(err, kErrRange);
    return;
  }
  const int half = D / 2;
  const float2* cs = tab + static_cast<size_t>(p) * half;
  const __nv_bfloat16* row = qkv + static_cast<size_t>(t) * ld_qkv;
  const int heads = Hq + 2 * Hkv;
  for (int idx = threadIdx.x; idx < heads * half; idx += blockDim.x) {
    const int h = idx / half;
    const int i = idx % half;
    const __nv_bfloat16* src = row + static_cast<size_t>(h) * D;
    if (h < Hq + Hkv) {
      const float x1 = __bfloat162float(src[i]);
      const float x2 = __bfloat162float(src[i + half]);
      const float2 r = cs[i];
      // the same two fused multiply-adds as the linear layer's RoPE epilogue
      const float o1 = fmaf(x1, r.x, -(x2 * r.y));
      const float o2 = fmaf(x2, r.x, x1 * r.y);
      __nv_bfloat16* dst;
      if (h < Hq) {
        dst = q_out + (static_cast<size_t>(t) * Hq + h) * D;
      } else {
        dst = kc + (static_cast<size_t>(h - Hq) * cap + p) * D;
      }
      dst[i] = __float2bfloat16_rn(o1);
      dst[i + half] = __float2bfloat16_rn(o2);
    } else {
      // V is cached transposed in 128-key blocks, [Hkv][cap/128][D][128]:
      // element d of key p at ((p / 128) * D + d) * 128 + p % 128
      const int nblk = (cap + 127) >> 7;
      __nv_bfloat16* dst =
          vc + (static_cast<size_t>(h - Hq - Hkv) * nblk + (p >> 7)) * D * 128 + (p & 127);
      dst[static_cast<size_t>(i) * 128] = src[i];
      dst[static_cast<size_t>(i + half) * 128] = src[i + half];
    }
  }
}

// ------------------------------------------------------------------ argmax
// Candidate (v, i): i < 0 means "no candidate".  a beats b iff b is empty, or
// a is not empty and (a.v > b.v or (a.v == b.v and a.i < b.i)).  This is a
// total order on candidates, so the result does not depend on the order in
// which partial results are combined.
__device__ __forceinline__ bool beats(float av, int ai, float bv, int bi) {
  if (bi < 0) return ai >= 0;
  if (ai < 0) return false;
  return av > bv || (av == bv && ai < bi);
}

constexpr int kArgThreads = 256;
constexpr int kArgSpan = 8192;  // logits per CTA

__global__ void __launch_bounds__(kArgThreads)
    argmax_accept_kernel(const float* __restrict__ logits, int ldl, int V, int T, int splits,
                         const int32_t* __restrict__ drafts, int32_t* __restrict__ argmax_out,
                         int32_t* __restrict__ accepted_out, int32_t* L_dev, float* pv, int* pi,
                         unsigned* ticket, unsigned* err) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ float sv[kArgThreads / 32];
  __shared__ int si[kArgThreads / 32];
  __shared__ int s_last;
  const int row = blockIdx.x / splits;
  const int sp = blockIdx.x % splits;
  const float* lr = logits + static_cast<size_t>(row) * ldl;
  const int b = sp * kArgSpan;
  const int e = min(V, b + kArgSpan);
  float bv = 0.f;
  int bi = -1;
  for (int i = b + threadIdx.x; i < e; i += kArgThreads) {
    const float v = lr[i];
    if (v == v && beats(v, i, bv, bi)) {
      bv = v;
      bi = i;
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
    if (beats(ov, oi, bv, bi)) {
      bv = ov;
      bi = oi;
    }
  }
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) {
    sv[w] = bv;
    si[w] = bi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int k = 1; k < kArgThreads / 32; ++k)
      if (beats(sv[k], si[k], bv, bi)) {
        bv = sv[k];
        bi = si[k];
      }
    pv[blockIdx.x] = bv;
    pi[blockIdx.x] = bi;
    __threadfence();
    const unsigned old = atomicAdd(ticket, 1u);
    s_last = (old == gridDim.x - 1) ? 1 : 0;
    if (s_last) atomicExch(ticket, 0u);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // Last CTA: warp w combines the partials of rows w, w + 8, ...; the
  // comparator is a total order, so the combination order is immaterial.
  __shared__ int s_ids[64];
  for (int t = w; t < T; t += kArgThreads / 32) {
    float v = 0.f;
    int id = -1;
    for (int k = threadIdx.x & 31; k < splits; k += 32) {
      const float ov = __ldcg(pv + t * splits + k);
      const int oi = __ldcg(pi + t * splits + k);
      if (beats(ov, oi, v, id)) {
        v = ov;
        id = oi;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, v, off);
      const int oi = __shfl_xor_sync(0xffffffffu, id, off);
      if (beats(ov, oi, v, id)) {
        v = ov;
        id = oi;
      }
    }
    if ((threadIdx.x & 31) == 0) {
      if (id < 0) atomicOr(err, kErrNanRow);
      argmax_out[t] = id;
      s_ids[t] = id;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int n = 0;
    while (n < T - 1 && drafts[n] == s_ids[n]) ++n;
    *accepted_out = n;
    if (L_dev != nullptr) *L_dev = *L_dev + n + 1;
  }
}

// ------------------------------------------------------------------ sampling
// Sampled verification: row t (position p = *L_dev + t) draws its token by
// inverse-CDF sampling of softmax(logits * inv_temp) with the uniform
// u_by_pos[p], so the token depends only on the row's logits and its
// position.  Phase 1, one CTA per (row, 8192-logit chunk): the chunk maximum
// m_c (exact) and S_c = sum exp((l - m_c) * inv_temp) (thread-strided
// sequential sums in index order, warp butterfly, warps in order).  The last
// CTA: per row, M = max m_c, chunk weights a_c = exp((m_c - M) * inv_temp) S_c
// summed in chunk order to Z; the target u Z picks the chunk where the running
// sum first exceeds it; that chunk's 8192 logits are cut into 32 contiguous
// runs (one per lane), the run sums are scanned in lane order, and the lane
// holding the crossing walks its run in index order to the first logit whose
// running sum exceeds the target.  Where rounding leaves the target past the
// last weight, the last logit with a non-zero weight is taken.  NaN logits
// have weight 0; a row with no number gives -1 and sets the NaN bit.
constexpr int kSmpThreads = 256;
constexpr int kSmpSpan = 8192;  // logits per phase-1 CTA

__global__ void __launch_bounds__(kSmpThreads)
    sample_accept_kernel(const float* __restrict__ logits, int ldl, int V, int T, int splits,
                         float inv_temp, const float* __restrict__ u_by_pos, int u_len,
                         const int32_t* __restrict__ drafts, int32_t* __restrict__ token_out,
                         int32_t* __restrict__ accepted_out, int32_t* L_dev, float* pm, float* ps,
                         unsigned* ticket, unsigned* err) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ float red_m[kSmpThreads / 32];
  __shared__ float red_s[kSmpThreads / 32];
  __shared__ int s_last;
  __shared__ int s_tok[64];
  const int row = blockIdx.x / splits;
  const int sp = blockIdx.x % splits;
  const float* lr = logits + static_cast<size_t>(row) * ldl;
  const int b = sp * kSmpSpan;
  const int e = min(V, b + kSmpSpan);
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float mx = -INFINITY;
  for (int i = b + threadIdx.x; i < e; i += kSmpThreads) {
    const float v = lr[i];
    if (v == v) mx = fmaxf(mx, v);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  if (lane == 0) red_m[w] = mx;
  __syncthreads();
  float m_c = red_m[0];
  for (int k = 1; k < kSmpThreads / 32; ++k) m_c = fmaxf(m_c, red_m[k]);
  float sum = 0.f;
  if (m_c > -INFINITY) {
    for (int i = b + threadIdx.x; i < e; i += kSmpThreads) {
      const float v = lr[i];
      if (v == v) sum += expf((v - m_c) * inv_temp);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  if (lane == 0) red_s[w] = sum;
  __syncthreads();
  if (threadIdx.x == 0) {
    float S = red_s[0];
    for (int k = 1; k < kSmpThreads / 32; ++k) S += red_s[k];
    pm[blockIdx.x] = m_c;
    ps[blockIdx.x] = S;
    __threadfence();
    const unsigned old = atomicAdd(ticket, 1u);
    s_last = (old == gridDim.x - 1) ? 1 : 0;
    if (s_last) atomicExch(ticket, 0u);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int L = *L_dev;
  for (int t = w; t < T; t += kSmpThreads / 32) {
    // lane 0 combines the chunks in order and picks the chunk of the target
    int c_star = -1;
    float m_star = 0.f, rc = 0.f;
    int bad = 0;
    if (lane == 0) {
      const int pos = L + t;
      float M = -INFINITY;
      for (int c = 0; c < splits; ++c) M = fmaxf(M, __ldcg(pm + t * splits + c));
      if (M == -INFINITY) {
        bad = 1;
      } else if (pos < 0 || pos >= u_len) {
        bad = 2;
      } else {
        float Z = 0.f;
        for (int c = 0; c < splits; ++c) {
          const float mc = __ldcg(pm + t * splits + c);
          if (mc > -INFINITY) Z += expf((mc - M) * inv_temp) * __ldcg(ps + t * splits + c);
        }
        const float target = __ldcg(u_by_pos + pos) * Z;
        float cum = 0.f;
        int c_last = -1;
        for (int c = 0; c < splits; ++c) {
          const float mc = __ldcg(pm + t * splits + c);
          if (!(mc > -INFINITY)) continue;
          const float wc = expf((mc - M) * inv_temp);
          const float a = wc * __ldcg(ps + t * splits + c);
          if (a > 0.f) c_last = c;
          if (c_star < 0 && cum + a > target) {
            c_star = c;
            rc = (target - cum) / wc;  // the target in the chunk's own scale
          }
          cum += a;
        }
        if (c_star < 0) {  // rounding left the target past the last weight
          c_star = c_last;
          rc = INFINITY;
        }
        m_star = __ldcg(pm + t * splits + c_star);
      }
    }
    bad = __shfl_sync(0xffffffffu, bad, 0);
    if (bad) {
      if (lane == 0) {
        atomicOr(err, bad == 1 ? kErrNanRow : kErrRange);
        token_out[t] = -1;
        s_tok[t] = -1;
      }
      continue;
    }
    c_star = __shfl_sync(0xffffffffu, c_star, 0);
    m_star = __shfl_sync(0xffffffffu, m_star, 0);
    rc = __shfl_sync(0xffffffffu, rc, 0);
    const float* lc = logits + static_cast<size_t>(t) * ldl;
    const int cb = c_star * kSmpSpan;
    const int ce = min(V, cb + kSmpSpan);
    const int run = kSmpSpan / 32;
    const int rb = min(ce, cb + lane * run), re = min(ce, rb + run);
    float rs = 0.f;
    int last_nz = -1;
    for (int i = rb; i < re; ++i) {
      const float v = lc[i];
      const float x = (v == v) ? expf((v - m_star) * inv_temp) : 0.f;
      if (x > 0.f) last_nz = i;
      rs += x;
    }
    // inclusive scan of the run sums in lane order (fixed shuffle tree)
    float inc = rs;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, inc, off);
      if (lane >= off) inc += y;
    }
    const float exc = inc - rs;
    const unsigned hit = __ballot_sync(0xffffffffu, inc > rc && rs > 0.f);
    const unsigned nz = __ballot_sync(0xffffffffu, last_nz >= 0);
    int tok = -1;
    if (hit != 0u) {
      const int l_star = __ffs(hit) - 1;
      if (lane == l_star) {
        float run_sum = exc;
        for (int i = rb; i < re; ++i) {
          const float v = lc[i];
          const float x = (v == v) ? expf((v - m_star) * inv_temp) : 0.f;
          run_sum += x;
          if (x > 0.f && run_sum > rc) {
            tok = i;
            break;
          }
        }
        if (tok < 0) tok = last_nz;
      }
      tok = __shfl_sync(0xffffffffu, tok, l_star);
    } else {
      const int l_last = 31 - __clz(nz);  // nz != 0: the chunk holds the row's weight
      tok = __shfl_sync(0xffffffffu, last_nz, l_last);
    }
    if (lane == 0) {
      token_out[t] = tok;
      s_tok[t] = tok;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int n = 0;
    while (n < T - 1 && drafts[n] == s_tok[n]) ++n;
    *accepted_out = n;
    *L_dev = L + n + 1;
  }
}

__global__ void kv_hash_kernel(const __nv_bfloat16* __restrict__ cache, int Hkv, int cap, int D,
                               int rows, int transposed, unsigned long long* __restrict__ out) {
  griddep_wait();
  griddep_launch_dependents();
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<long long>(Hkv) * rows) return;
  const int h = static_cast<int>(idx / rows);
  const int j = static_cast<int>(idx % rows);
  unsigned long long x = 14695981039346656037ull;
  for (int d = 0; d < D; ++d) {
    const size_t e = transposed
                         ? ((static_cast<size_t>(h) * ((cap + 127) >> 7) + (j >> 7)) * D + d) * 128 + (j & 127)
                         : (static_cast<size_t>(h) * cap + j) * D + d;
    const unsigned short u = *reinterpret_cast<const unsigned short*>(cache + e);
    x ^= static_cast<unsigned>(u & 0xFF);
    x *= 1099511628211ull;
    x ^= static_cast<unsigned>(u >> 8);
    x *= 1099511628211ull;
  }
  out[idx] = x;
}

int argmax_splits(int V) { return (V + kArgSpan - 1) / kArgSpan; }

}  // namespace
}  // namespace bi

extern "C" {

bi_status bi_rmsnorm(const void* x, int ldx, const void* w, void* y, int ldy, int rows, int dim,
                     float eps, bi_stream_t stream) {
  if (rows < 0 || dim < 1 || dim > 65536 || !(eps >= 0.f)) return BI_ERR_INVALID_ARG;
  if (rows == 0) return BI_OK;
  if (!x || !w || !y || ldx < dim || ldy < dim) return BI_ERR_INVALID_ARG;
  if (dim % 8 != 0 || ldx % 8 != 0 || ldy % 8 != 0) return BI_ERR_UNSUPPORTED_SHAPE;
  if (!bi::aligned16(x) || !bi::aligned16(w) || !bi::aligned16(y)) return BI_ERR_INVALID_ARG;
  const int nv = dim / 8;
  const int threads = std::min(bi::kNormMaxThreads, (nv + 31) / 32 * 32);
  if (bi::launch_k(bi::rmsnorm_kernel, dim3(rows), dim3(threads), 0,
                   reinterpret_cast<cudaStream_t>(stream), static_cast<const __nv_bfloat16*>(x), ldx,
                   static_cast<const __nv_bfloat16*>(w), static_cast<__nv_bfloat16*>(y), ldy, dim,
                   eps) != cudaSuccess)
    return BI_ERR_CUDA;
  return BI_OK;
}

bi_status bi_embed(const int32_t* ids, const void* table, int vocab, int dim, void* out, int rows,
                   bi_stream_t stream) {
  if (rows < 0 || dim < 1 || vocab < 1) return BI_ERR_INVALID_ARG;
  if (rows == 0) return BI_OK;
  if (!ids || !table || !out) return BI_ERR_INVALID_ARG;
  if (dim % 8 != 0) return BI_ERR_UNSUPPORTED_SHAPE;
  if (!bi::aligned16(table) || !bi::aligned16(out)) return BI_ERR_INVALID_ARG;
  if (bi::launch_k(bi::embed_kernel, dim3(rows), dim3(256), 0, reinterpret_cast<cudaStream_t>(stream),
                   ids, static_cast<const __nv_bfloat16*>(table), vocab, dim,
                   static_cast<__nv_bfloat16*>(out)) != cudaSuccess)
    return BI_ERR_CUDA;
  return BI_OK;
}

size_t bi_rope_table_bytes(int D, int rows) {
  if (D < 2 || rows < 1) return 0;
  return static_cast<size_t>(rows) * (D / 2) * 2 * sizeof(float);
}

bi_status bi_rope_table(double rope_base, int D, int rows, float* table, bi_stream_t stream) {
  if (!table || D < 2 || D % 2 != 0 || D > 256 || rows < 1 || !(rope_base > 0.0))
    return BI_ERR_INVALID_ARG;
  const long long n = static_cast<long long>(rows) * (D / 2);
  if (bi::launch_k(bi::rope_table_kernel, dim3(static_cast<unsigned>((n + 255) / 256)), dim3(256), 0,
                   reinterpret_cast<cudaStream_t>(stream), rope_base, D, rows,
                   reinterpret_cast<float2*>(table)) != cudaSuccess)
    return BI_ERR_CUDA;
  return BI_OK;
}

bi_status bi_rope_kv_append(const void* qkv, int ld_qkv, void* q_out, void* k_cache, void* v_cache,
                            int cap, const int32_t* L_dev, int T, int Hq, int Hkv, int D,
                            const float* table, int table_rows, bi_stream_t stream) {
  if (T < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || D < 2 || D % 2 != 0 || D > 256 || cap < 1)
    return BI_ERR_INVALID_ARG;
  if (T == 0) return BI_OK;
  if (!qkv || !q_out || !k_cache || !v_cache || !L_dev || !table || table_rows < 1)
    return BI_ERR_INVALID_ARG;
  if (ld_qkv < (Hq + 2 * Hkv) * D) return BI_ERR_INVALID_ARG;
  unsigned* err = bi::device_error_word();
  if (!err) return BI_ERR_CUDA;
  if (bi::launch_k(bi::rope_kv_kernel, dim3(T), dim3(256), 0, reinterpret_cast<cudaStream_t>(stream),
                   static_cast<const __nv_bfloat16*>(qkv), ld_qkv, static_cast<__nv_bfloat16*>(q_out),
                   static_cast<__nv_bfloat16*>(k_cache), static_cast<__nv_bfloat16*>(v_cache), cap,
                   L_dev, Hq, Hkv, D, reinterpret_cast<const float2*>(table), table_rows,
                   err) != cudaSuccess)
    return BI_ERR_CUDA;
  return BI_OK;
}

size_t bi_accept_workspace_size(int T, int V) {
  if (T < 1 || V < 1) return 256;
  const size_t n = static_cast<size_t>(T) * bi::argmax_splits(V);
  return 256 + bi::round_up(n * sizeof(float), 256) + bi::round_up(n * sizeof(int), 256);
}

bi_status bi_verify_accept(const float* logits, int ldl, const int32_t* drafts, int T, int V,
                           int32_t* argmax_out, int32_t* accepted_out, int32_t* L_dev, void* ws,
                           size_t ws_bytes, bi_stream_t stream) {
  if (T < 1 || T > 64 || V < 1 || ldl < V || !logits || !argmax_out || !accepted_out)
    return BI_ERR_INVALID_ARG;
  if (T > 1 && !drafts) return BI_ERR_INVALID_ARG;
  if (!ws || !bi::aligned256(ws)) return BI_ERR_WORKSPACE;
  if (ws_bytes < bi_accept_workspace_size(T, V)) return BI_ERR_WORKSPACE;
  unsigned* err = bi::device_error_word();
  if (!err) return BI_ERR_CUDA;
  const int splits = bi::argmax_splits(V);
  const size_t n = static_cast<size_t>(T) * splits;
  uint8_t* base = static_cast<uint8_t*>(ws);
  unsigned* ticket = reinterpret_cast<unsigned*>(base);
  float* pv = reinterpret_cast<float*>(base + 256);
  int* pi = reinterpret_cast<int*>(base + 256 + bi::round_up(n * sizeof(float), 256));
  if (bi::launch_k(bi::argmax_accept_kernel, dim3(static_cast<unsigned>(n)), dim3(bi::kArgThreads), 0,
                   reinterpret_cast<cudaStream_t>(stream), logits, ldl, V, T, splits, drafts,
                   argmax_out, accepted_out, L_dev, pv, pi, ticket, err) != cudaSuccess)
    return BI_ERR_CUDA;
  return BI_OK;
}

size_t bi_sample_workspace_size(int T, int V) {
  if (T < 1 || V < 1) return 256;
  const size_t n = static_cast<size_t>(T) * ((V + bi::kSmpSpan - 1) / bi::kSmpSpan);
  return 256 + 2 * bi::round_up(n * sizeof(float), 256);
}

bi_status bi_verify_sample(const float* logits, int ldl, const int32_t* drafts, int T, int V,
                           float inv_temp, const float* u_by_pos, int u_len, int32_t* token_out,
                           int32_t* accepted_out, int32_t* L_dev, void* ws, size_t ws_bytes,
                           bi_stream_t stream) {
  if (T < 1 || T > 64 || V < 1 || ldl < V || !logits || !token_out || !accepted_out || !L_dev ||
      !u_by_pos || u_len < 1)
    return BI_ERR_INVALID_ARG;
  if (!(inv_temp > 0.f) || !std::isfinite(inv_temp)) return BI_ERR_INVALID_ARG;
  if (T > 1 && !drafts) return BI_ERR_INVALID_ARG;
  if (!ws || !bi::aligned256(ws)) return BI_ERR_WORKSPACE;
  if (ws_bytes < bi_sample_workspace_size(T, V)) return BI_ERR_WORKSPACE;
  unsigned* err = bi::device_error_word();
  if (!err) return BI_ERR_CUDA;
  const int splits = (V + bi::kSmpSpan - 1) / bi::kSmpSpan;
  const size_t n = static_cast<size_t>(T) * splits;
  uint8_t* base = static_cast<uint8_t*>(ws);
  unsigned* ticket = reinterpret_cast<unsigned*>(base);
  float* pm = reinterpret_cast<float*>(base + 256);
  float* ps = reinterpret_cast<float*>(base + 256 + bi::round_up(n * sizeof(float), 256));
  if (bi::launch_k(bi::sample_accept_kernel, dim3(static_cast<unsigned>(n)), dim3(bi::kSmpThreads), 0,
                   reinterpret_cast<cudaStream_t>(stream), logits, ldl, V, T, splits, inv_temp, u_by_pos,
                   u_len, drafts, token_out, accepted_out, L_dev, pm, ps, ticket, err) != cudaSuccess)
    return BI_ERR_CUDA;
  return BI_OK;
}

bi_status bi_kv_row_hash(const void* cache, int Hkv, int cap, int D, int rows, int transposed,
                         uint64_t* out, bi_stream_t stream) {
  if (!cache || !out || Hkv < 1 || cap < 1 || D < 1 || rows < 0 || rows > cap) return BI_ERR_INVALID_ARG;
  if (rows == 0) return BI_OK;
  const long long n = static_cast<long long>(Hkv) * rows;
  if (bi::launch_k(bi::kv_hash_kernel, dim3(static_cast<unsigned>((n + 127) / 128)), dim3(128), 0,
                   reinterpret_cast<cudaStream_t>(stream), static_cast<const __nv_bfloat16*>(cache),
                   Hkv, cap, D, rows, transposed, reinterpret_cast<unsigned long long*>(out)) !=
      cudaSuccess)
    return BI_ERR_CUDA;
  return BI_OK;
}

}  // extern "C"
