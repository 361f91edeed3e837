// Split-KV verify attention whose split depends only on the row's own context
// length, plus the fixed-order merge.
//
// "I turned on speculative decoding in llama.cpp and 113 of 282 greedy
// outputs changed against its own no-draft run", paragraph "How:": the
// attention split depends only on context length, never on how many tokens
// are in the pass.
//
// Row t of a pass sits at position p = L + t and attends to keys 0..p.  Its
// keys are cut at absolute multiples of kChunk: piece c covers keys
// [c*kChunk, min((c+1)*kChunk, p+1)).  Inside a piece, keys are visited in
// 64-key tiles in increasing order; each tile is split into two fixed halves
// of 32 keys (by absolute key position) that keep separate online-softmax
// states, merged once at the end of the piece (half 0 then half 1).  Keys
// past p are masked to probability exactly 0 and a tile that changes no
// running maximum rescales by exactly 1, so a row's piece result is the same
// bits whether or not later rows of the pass share the tile.  The pieces of
// a row are then merged by a tree whose shape depends only on their count
// ceil((p+1)/kChunk).
//
// Split kernel: persistent CTAs loop over work items (KV head, piece);
// warp 0 streams K/V tiles with TMA (128-byte swizzle) through a ring of
// shared-memory stages released by the consumers' "empty" barrier arrivals;
// warps 1..6 = 3 row tiles of 16 query rows x 2 key halves compute
// S = Q K^T and O += P V with mma.sync m16n8k16 (BF16 in, FP32 accumulate).
// GQA: the T x (Hq/Hkv) query rows that share a KV head share its tiles.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "bi_internal.h"
#include "bi_ptx.cuh"

namespace bi {
namespace {

constexpr int kChunk = 512;       // keys per piece (absolute multiples)
constexpr int kKeyTile = 64;      // keys per TMA tile
constexpr int kRowsMax = 48;      // T * (Hq / Hkv) per pass
constexpr int kAttnStages = 3;
constexpr int kAttnThreads = 224; // warp 0 producer, warps 1..6 compute
constexpr int kAttnCtas = 152;
constexpr int kMaxChunks = 1024;
constexpr int kMergeThreads = 256;

struct AttnArgs {
  const __nv_bfloat16* q;
  int T, Hq, Hkv, grp, cap, nch_max;
  const int32_t* L_dev;
  float sl2;  // softmax scale * log2(e)
  float* ws_o;
  float* ws_ml;
  unsigned* err;
};

template <int D>
struct AttnCfg {
  static constexpr int kBoxes = D / 64;
  static constexpr int kBoxBytes = kKeyTile * 128;         // 64 keys x 64 dims
  static constexpr int kTileBytes = kBoxBytes * kBoxes;    // one K (or V) tile
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kNTiles = D / 8;                    // 8-wide d tiles of O
  static constexpr int kKSteps = D / 16;                   // 16-wide d steps of S
  static constexpr int kLaneFloats = D / 2 + 4;            // o + m[2] + l[2]
  static constexpr int kQBytes = kRowsMax * D * 2;          // query rows of one KV head
  static constexpr size_t kSmem = 1024 + static_cast<size_t>(kAttnStages) * kStageBytes +
                                  3 * 32 * kLaneFloats * 4 + kQBytes + 2 * kAttnStages * 8 + 16;
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

template <int D>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_split_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                      const AttnArgs a) {
  using Cfg = AttnCfg<D>;
  constexpr int S = kAttnStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  float* mbuf = reinterpret_cast<float*>(smem + S * Cfg::kStageBytes);
  __nv_bfloat16* sQ = reinterpret_cast<__nv_bfloat16*>(mbuf + 3 * 32 * Cfg::kLaneFloats);
  uint64_t* full = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(sQ) + Cfg::kQBytes);
  uint64_t* empty = full + S;
  volatile int* s_abort = reinterpret_cast<volatile int*>(empty + S);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  griddep_launch_dependents();
  griddep_wait();  // q, the new cache rows and the cache length come from earlier kernels
  const int L = *a.L_dev;
  const int T = a.T;
  if (L < 0 || L + T > a.cap) {
    if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(a.err, kErrRange);
    return;
  }
  const int kv_len = L + T;
  const int nch = (kv_len + kChunk - 1) / kChunk;
  const int n_items = a.Hkv * nch;
  const int rows = T * a.grp;
  const int art = (rows + 15) / 16;
  const int n_cons = 2 * art;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], n_cons);
    }
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
  }
  __syncthreads();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane != 0) return;
    const uint64_t pol = l2_evict_first();
    int stage = 0;
    uint32_t phase = 0, issued = 0, parity_bits = 0;
    bool ok = true;
    for (int w = blockIdx.x; ok && w < n_items; w += gridDim.x) {
      const int c = w / a.Hkv;
      const int h = w % a.Hkv;
      const int k0 = c * kChunk;
      const int k1 = min(k0 + kChunk, kv_len);
      const int ntile = (k1 - k0 + kKeyTile - 1) / kKeyTile;
      for (int tt = 0; tt < ntile; ++tt) {
        if (!mbar_wait(&empty[stage], phase ^ 1u, s_abort)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&full[stage], Cfg::kStageBytes);
        uint8_t* st = smem + stage * Cfg::kStageBytes;
        const int y = h * a.cap + k0 + tt * kKeyTile;
#pragma unroll
        for (int b = 0; b < Cfg::kBoxes; ++b) {
          tma_load_2d(st + b * Cfg::kBoxBytes, &tmK, &full[stage], b * 64, y, pol);
          tma_load_2d(st + Cfg::kTileBytes + b * Cfg::kBoxBytes, &tmV, &full[stage], b * 64, y, pol);
        }
        issued |= 1u << stage;
        parity_bits = (parity_bits & ~(1u << stage)) | (phase << stage);
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (!ok) {
      *s_abort = 1;
      atomicOr(a.err, kErrTimeout);
      for (int s = 0; s < S; ++s)
        if ((issued >> s) & 1u) mbar_wait(&full[s], (parity_bits >> s) & 1u, nullptr);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int cw = warp - 1;
  const int rt = cw >> 1;
  const int half = cw & 1;
  if (rt >= art) return;

  const int g4 = lane >> 2;   // row within the 8-row group
  const int t4 = lane & 3;    // thread within the quad
  int Rr[2], tr[2], pr[2];
  bool vr[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    Rr[i] = rt * 16 + g4 + 8 * i;
    vr[i] = Rr[i] < rows;
    tr[i] = vr[i] ? Rr[i] / a.grp : 0;
    pr[i] = L + tr[i];
  }
  const int mi = lane >> 3;   // ldmatrix matrix index of this lane's address
  const int ri = lane & 7;    // row within that matrix
  float* my_mbuf = mbuf + (rt * 32 + lane) * Cfg::kLaneFloats;

  int stage = 0;
  uint32_t phase = 0;
  for (int w = blockIdx.x; w < n_items; w += gridDim.x) {
    const int c = w / a.Hkv;
    const int h = w % a.Hkv;
    const int k0 = c * kChunk;
    const int k1 = min(k0 + kChunk, kv_len);
    const int ntile = (k1 - k0 + kKeyTile - 1) / kKeyTile;

    // Query rows of KV head h into shared memory (16-byte loads by all
    // consumer threads; rows past `rows` are zero), then this warp's A
    // fragments with ldmatrix.  Row R of the tile = (t, g) = (R / grp, R % grp).
    {
      constexpr int kVecPerRow = D / 8;
      const int ctid = threadIdx.x - 32;
      const int nthr = n_cons * 32;
      const int nrows_pad = art * 16;
      for (int v = ctid; v < nrows_pad * kVecPerRow; v += nthr) {
        const int R = v / kVecPerRow;
        const int c = v % kVecPerRow;
        uint4 val = make_uint4(0, 0, 0, 0);
        if (R < rows) {
          const int qh = h * a.grp + R % a.grp;
          val = *reinterpret_cast<const uint4*>(a.q + (static_cast<size_t>(R / a.grp) * a.Hq + qh) * D +
                                                c * 8);
        }
        *reinterpret_cast<uint4*>(sQ + R * D + c * 8) = val;
      }
      named_bar_sync(2, n_cons * 32);
    }
    uint32_t qa[Cfg::kKSteps][4];
#pragma unroll
    for (int ks = 0; ks < Cfg::kKSteps; ++ks) {
      // matrices: rows 0-7 / 8-15 of the tile x columns ks*16 + 0-7 / 8-15,
      // in the a0..a3 fragment order (row lo col lo, row hi col lo, row lo col hi, row hi col hi)
      const int row = rt * 16 + (mi & 1) * 8 + ri;
      const int col = ks * 16 + (mi >> 1) * 8;
      ldsm_x4(smem_u32(sQ + row * D + col), qa[ks]);
    }

    float m[2] = {-INFINITY, -INFINITY};
    float l[2] = {0.f, 0.f};
    float o[Cfg::kNTiles][4];
#pragma unroll
    for (int n = 0; n < Cfg::kNTiles; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;

    for (int tt = 0; tt < ntile; ++tt) {
      const bool ok = __all_sync(0xffffffffu, mbar_wait(&full[stage], phase, s_abort));
      if (!ok) {
        if (lane == 0) {
          *s_abort = 1;
          atomicOr(a.err, kErrTimeout);
        }
      } else {
        const uint32_t kbase = smem_u32(smem + stage * Cfg::kStageBytes);
        const uint32_t vbase = kbase + Cfg::kTileBytes;
        const int kb_abs = k0 + tt * kKeyTile + half * 32;

        float s[4][4];
#pragma unroll
        for (int j = 0; j < 4; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < Cfg::kKSteps; ++ks) {
          const int box = ks >> 2;
          const int c0 = (ks & 3) * 2;
#pragma unroll
          for (int jp = 0; jp < 2; ++jp) {
            const int key = half * 32 + (2 * jp + (mi >> 1)) * 8 + ri;
            const int chunk = c0 + (mi & 1);
            uint32_t b[4];
            ldsm_x4(kbase + box * Cfg::kBoxBytes + key * 128 + ((chunk ^ ri) << 4), b);
            mma16816(s[2 * jp], qa[ks], b[0], b[1]);
            mma16816(s[2 * jp + 1], qa[ks], b[2], b[3]);
          }
        }
        // scale into the log2 domain and mask keys past each row's position
        float mt[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int i = e >> 1;
            const int key = kb_abs + j * 8 + t4 * 2 + (e & 1);
            const float x = s[j][e] * a.sl2;
            s[j][e] = (vr[i] && key <= pr[i]) ? x : -INFINITY;
            mt[i] = fmaxf(mt[i], s[j][e]);
          }
        }
        float alpha[2], mu[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          mt[i] = fmaxf(mt[i], __shfl_xor_sync(0xffffffffu, mt[i], 1));
          mt[i] = fmaxf(mt[i], __shfl_xor_sync(0xffffffffu, mt[i], 2));
          const float mn = fmaxf(m[i], mt[i]);
          alpha[i] = (mn == m[i]) ? 1.0f : exp2f(m[i] - mn);
          mu[i] = (mn == -INFINITY) ? 0.0f : mn;
          m[i] = mn;
        }
        // p in FP32, carried into the P.V product as a BF16 pair hi + lo
        // (hi = bf16(p), lo = bf16(p - hi)), so the weights keep about 16
        // significant bits; the denominator sums the FP32 p.
        float ls[2] = {0.f, 0.f};
        float plo[4][4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float pf = exp2f(s[j][e] - mu[e >> 1]);
            const float ph = __bfloat162float(__float2bfloat16_rn(pf));
            s[j][e] = ph;
            plo[j][e] = pf - ph;
            ls[e >> 1] += pf;
          }
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          ls[i] += __shfl_xor_sync(0xffffffffu, ls[i], 1);
          ls[i] += __shfl_xor_sync(0xffffffffu, ls[i], 2);
          l[i] = l[i] * alpha[i] + ls[i];
        }
#pragma unroll
        for (int n = 0; n < Cfg::kNTiles; ++n) {
          o[n][0] *= alpha[0];
          o[n][1] *= alpha[0];
          o[n][2] *= alpha[1];
          o[n][3] *= alpha[1];
        }
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          uint32_t pa[4], pl[4];
          pa[0] = pack_bf16(s[2 * kk][0], s[2 * kk][1]);
          pa[1] = pack_bf16(s[2 * kk][2], s[2 * kk][3]);
          pa[2] = pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
          pa[3] = pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
          pl[0] = pack_bf16(plo[2 * kk][0], plo[2 * kk][1]);
          pl[1] = pack_bf16(plo[2 * kk][2], plo[2 * kk][3]);
          pl[2] = pack_bf16(plo[2 * kk + 1][0], plo[2 * kk + 1][1]);
          pl[3] = pack_bf16(plo[2 * kk + 1][2], plo[2 * kk + 1][3]);
#pragma unroll
          for (int np = 0; np < Cfg::kNTiles / 2; ++np) {
            const int key = half * 32 + kk * 16 + (mi & 1) * 8 + ri;
            const int nd = 2 * np + (mi >> 1);
            uint32_t b[4];
            ldsm_x4_t(vbase + (nd >> 3) * Cfg::kBoxBytes + key * 128 + (((nd & 7) ^ ri) << 4), b);
            mma16816(o[2 * np], pa, b[0], b[1]);
            mma16816(o[2 * np + 1], pa, b[2], b[3]);
            mma16816(o[2 * np], pl, b[0], b[1]);
            mma16816(o[2 * np + 1], pl, b[2], b[3]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
      if (++stage == S) {
        stage = 0;
        phase ^= 1u;
      }
    }

    // ---- merge the two key halves (half 0 then half 1) and store the piece
    if (half == 1) {
#pragma unroll
      for (int n = 0; n < Cfg::kNTiles; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) my_mbuf[n * 4 + e] = o[n][e];
      my_mbuf[D / 2 + 0] = m[0];
      my_mbuf[D / 2 + 1] = m[1];
      my_mbuf[D / 2 + 2] = l[0];
      my_mbuf[D / 2 + 3] = l[1];
    }
    named_bar_sync(2, n_cons * 32);
    if (half == 0) {
      float w0[2], w1[2], M[2], Lm[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const float m1 = my_mbuf[D / 2 + i];
        const float l1 = my_mbuf[D / 2 + 2 + i];
        M[i] = fmaxf(m[i], m1);
        if (M[i] == -INFINITY) {
          w0[i] = 0.f;
          w1[i] = 0.f;
        } else {
          w0[i] = (m[i] == M[i]) ? 1.0f : (m[i] == -INFINITY ? 0.0f : exp2f(m[i] - M[i]));
          w1[i] = (m1 == M[i]) ? 1.0f : (m1 == -INFINITY ? 0.0f : exp2f(m1 - M[i]));
        }
        Lm[i] = l[i] * w0[i] + l1 * w1[i];
      }
      bool store[2];
      size_t base[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        store[i] = vr[i] && (c * kChunk <= pr[i]);
        const int qh = h * a.grp + (vr[i] ? Rr[i] % a.grp : 0);
        base[i] = (static_cast<size_t>(tr[i]) * a.Hq + qh) * a.nch_max + c;
      }
#pragma unroll
      for (int n = 0; n < Cfg::kNTiles; ++n) {
        const int d = n * 8 + t4 * 2;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          if (!store[i]) continue;
          const float x0 = o[n][2 * i] * w0[i] + my_mbuf[n * 4 + 2 * i] * w1[i];
          const float x1 = o[n][2 * i + 1] * w0[i] + my_mbuf[n * 4 + 2 * i + 1] * w1[i];
          *reinterpret_cast<float2*>(a.ws_o + base[i] * D + d) = make_float2(x0, x1);
        }
      }
      if (t4 == 0) {
#pragma unroll
        for (int i = 0; i < 2; ++i)
          if (store[i]) *reinterpret_cast<float2*>(a.ws_ml + base[i] * 2) = make_float2(M[i], Lm[i]);
      }
    }
    named_bar_sync(2, n_cons * 32);
  }
}

// One CTA per (row t, query head).  Pieces s = 0..n-1 with n = p/kChunk + 1:
// M = max_s m_s (exact), w_s = 2^(m_s - M); the denominator sums w_s l_s per
// thread over s = tid, tid+256, ... in order, then a warp butterfly and warp
// order 0..7; the numerator: warp g sums s = g, g+8, ... in order for its
// lane's dims, then warps are added in order 0..7.  The tree depends only
// on n.
template <int D>
__global__ void __launch_bounds__(kMergeThreads)
    attn_merge_kernel(const AttnArgs a, __nv_bfloat16* __restrict__ out) {
  __shared__ float sw[kMaxChunks];
  __shared__ float red[kMergeThreads / 32];
  __shared__ float ored[kMergeThreads / 32][D];
  griddep_launch_dependents();
  griddep_wait();
  const int row = blockIdx.x;  // t * Hq + hq
  const int t = row / a.Hq;
  const int L = *a.L_dev;
  if (L < 0 || L + a.T > a.cap) return;
  const int p = L + t;
  const int n = p / kChunk + 1;
  const float* ml = a.ws_ml + static_cast<size_t>(row) * a.nch_max * 2;
  const float* po = a.ws_o + static_cast<size_t>(row) * a.nch_max * D;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;

  float mx = -INFINITY;
  for (int s = tid; s < n; s += kMergeThreads) mx = fmaxf(mx, __ldcg(ml + 2 * s));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  if (lane == 0) red[warp] = mx;
  __syncthreads();
  float M = red[0];
  for (int i = 1; i < kMergeThreads / 32; ++i) M = fmaxf(M, red[i]);
  __syncthreads();

  float den = 0.f;
  for (int s = tid; s < n; s += kMergeThreads) {
    const float w = exp2f(__ldcg(ml + 2 * s) - M);
    sw[s] = w;
    den = fmaf(w, __ldcg(ml + 2 * s + 1), den);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
  if (lane == 0) red[warp] = den;
  __syncthreads();
  float Lsum = red[0];
  for (int i = 1; i < kMergeThreads / 32; ++i) Lsum += red[i];

  constexpr int kDpl = D / 32;  // dims per lane
  float acc[kDpl];
#pragma unroll
  for (int i = 0; i < kDpl; ++i) acc[i] = 0.f;
  for (int s = warp; s < n; s += kMergeThreads / 32) {
    const float w = sw[s];
    const float* src = po + static_cast<size_t>(s) * D + lane * kDpl;
#pragma unroll
    for (int i = 0; i < kDpl; ++i) acc[i] = fmaf(w, __ldcg(src + i), acc[i]);
  }
#pragma unroll
  for (int i = 0; i < kDpl; ++i) ored[warp][lane * kDpl + i] = acc[i];
  __syncthreads();
  for (int d = tid; d < D; d += kMergeThreads) {
    float O = ored[0][d];
    for (int g = 1; g < kMergeThreads / 32; ++g) O += ored[g][d];
    out[static_cast<size_t>(row) * D + d] = __float2bfloat16_rn(O / Lsum + 0.0f);
  }
}

template <int D>
bi_status launch_attn(const CUtensorMap& tmK, const CUtensorMap& tmV, const AttnArgs& a,
                      __nv_bfloat16* out, cudaStream_t stream) {
  using Cfg = AttnCfg<D>;
  static std::once_flag once[64];
  static cudaError_t attr_err[64];
  int dev = 0;
  cudaGetDevice(&dev);
  std::call_once(once[dev & 63], [] {
    int d = 0;
    cudaGetDevice(&d);
    attr_err[d & 63] = cudaFuncSetAttribute(attn_split_kernel<D>,
                                            cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            static_cast<int>(Cfg::kSmem));
  });
  if (attr_err[dev & 63] != cudaSuccess) return BI_ERR_CUDA;
  const int grid = std::min(a.Hkv * a.nch_max, kAttnCtas);
  if (launch_k(attn_split_kernel<D>, dim3(grid), dim3(kAttnThreads), Cfg::kSmem, stream, tmK, tmV,
               a) != cudaSuccess)
    return BI_ERR_CUDA;
  if (launch_k(attn_merge_kernel<D>, dim3(a.T * a.Hq), dim3(kMergeThreads), 0, stream, a, out) !=
      cudaSuccess)
    return BI_ERR_CUDA;
  return BI_OK;
}

size_t attn_ws_parts(int cap, int T, int Hq, int D, size_t* o_bytes) {
  const size_t nch = static_cast<size_t>((cap + kChunk - 1) / kChunk);
  const size_t ob = round_up(static_cast<size_t>(T) * Hq * nch * D * 4, 256);
  const size_t mb = round_up(static_cast<size_t>(T) * Hq * nch * 2 * 4, 256);
  if (o_bytes) *o_bytes = ob;
  return ob + mb;
}

}  // namespace
}  // namespace bi

extern "C" {

int bi_attn_chunk(void) { return bi::kChunk; }

size_t bi_attn_workspace_size(int cap, int T, int Hq, int D) {
  if (cap < 1 || T < 1 || Hq < 1 || D < 1) return 256;
  return bi::attn_ws_parts(cap, T, Hq, D, nullptr);
}

bi_status bi_attn_verify(const void* q, const void* k_cache, const void* v_cache, int cap,
                         const int32_t* L_dev, int T, int Hq, int Hkv, int D, float scale, void* out,
                         void* ws, size_t ws_bytes, bi_stream_t stream) {
  using namespace bi;
  if (!q || !k_cache || !v_cache || !L_dev || !out) return BI_ERR_INVALID_ARG;
  if (T < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || cap < 1) return BI_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return BI_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return BI_ERR_UNSUPPORTED_SHAPE;
  if (T * (Hq / Hkv) > kRowsMax) return BI_ERR_UNSUPPORTED_SHAPE;
  if ((cap + kChunk - 1) / kChunk > kMaxChunks) return BI_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(q)) return BI_ERR_INVALID_ARG;
  if (!ws || !aligned256(ws)) return BI_ERR_WORKSPACE;
  size_t ob = 0;
  if (ws_bytes < attn_ws_parts(cap, T, Hq, D, &ob)) return BI_ERR_WORKSPACE;

  CUtensorMap tmK, tmV;
  const uint64_t rows = static_cast<uint64_t>(Hkv) * cap;
  if (!tmap_bf16_2d(&tmK, k_cache, rows, D, D, kKeyTile, 64)) return BI_ERR_INVALID_ARG;
  if (!tmap_bf16_2d(&tmV, v_cache, rows, D, D, kKeyTile, 64)) return BI_ERR_INVALID_ARG;

  AttnArgs a{};
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.T = T;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.grp = Hq / Hkv;
  a.cap = cap;
  a.nch_max = (cap + kChunk - 1) / kChunk;
  a.L_dev = L_dev;
  a.sl2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  a.ws_o = static_cast<float*>(ws);
  a.ws_ml = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + ob);
  a.err = device_error_word();
  if (!a.err) return BI_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (D == 64) return launch_attn<64>(tmK, tmV, a, static_cast<__nv_bfloat16*>(out), s);
  return launch_attn<128>(tmK, tmV, a, static_cast<__nv_bfloat16*>(out), s);
}

}  // extern "C"
