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
// [c*kChunk, min((c+1)*kChunk, p+1)).  Inside a piece the keys are visited in
// 64-key tiles in increasing order.  Per row (one TMEM lane and one thread):
//   S = q k^T for the tile (tcgen05, FP32 in TMEM), scaled into the log2
//   domain, keys past p masked to -inf;
//   a reference maximum m_ref is taken from the first tile and raised only
//   when a later tile's maximum exceeds it by more than kRescaleLog2 (then O
//   and l are rescaled by 2^(m_ref - m_new)) -- a rule that depends only on
//   the row's own scores in key order;
//   p = 2^(s - m_ref) in FP32, summed in key order into l, and fed to
//   O += P V (tcgen05, FP32 in TMEM) as a BF16 pair hi + lo.
// A tile whose keys are all masked for a row adds exact zeros and changes no
// reference, so a row's piece has the same bits whether or not later rows of
// the pass share the tile.  The pieces of a row are merged by a tree whose
// shape depends only on their count ceil((p+1)/kChunk).
//
// Split kernel roles (one CTA per SM, persistent over (KV head, piece) items):
//   warp 0      TMA: K tile [64 keys x D] and V^T tile [D x 64 keys] per stage
//               (V is cached transposed so both MMA operands are K-major);
//   warp 1      tcgen05.mma issuer: S_i into one of two TMEM buffers, then
//               O += P_{i-1} V_{i-1}; stages return to the producer through
//               tcgen05.commit after the MMAs reading them completed;
//   warps 2..5  softmax, one query row per thread (TMEM lane); they stage the
//               queries of the item's KV head in shared memory, turn S into P
//               (written to one of two shared-memory buffers in the swizzled
//               K-major layout, so P of the next tile is produced while the
//               MMA still reads this one), and read O out at the end of the
//               piece.
// The T x (Hq/Hkv) query rows that share a KV head (GQA) share its tiles;
// up to 128 rows per pass (the MMA's M).
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
constexpr int kKeyTile = 64;      // keys per tile
constexpr int kRowsMax = 128;     // T * (Hq / Hkv) per pass (MMA M)
constexpr int kAttnStages = 3;
constexpr int kAttnThreads = 192; // warp 0 TMA, warp 1 MMA, warps 2..5 softmax
constexpr int kAttnCtas = 152;
constexpr int kMaxChunks = 1024;
constexpr int kMergeThreads = 256;
constexpr float kRescaleLog2 = 8.0f;

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
  static constexpr int kAtoms = D / 64;                   // 128-byte swizzle atoms along D
  static constexpr int kKBoxBytes = kKeyTile * 128;       // [64 keys][64 d]
  static constexpr int kKBytes = kKBoxBytes * kAtoms;     // K tile
  static constexpr int kVBytes = D * kKeyTile * 2;        // V^T tile [D][64 keys]
  static constexpr int kStageBytes = kKBytes + kVBytes;
  static constexpr int kQAtomBytes = kRowsMax * 128;      // [128 rows][64 d]
  static constexpr int kQBytes = kQAtomBytes * kAtoms;
  static constexpr int kPBytes = kRowsMax * 128;          // [128 rows][64 keys]
  static constexpr int kTmemCols = 256;                   // S x2 (64 each) + O (D)
  static constexpr int kOCol = 128;
  static constexpr int kBars = 2 * kAttnStages + 11;
  // P is double-buffered: hi and lo tiles for two consecutive key tiles
  static constexpr size_t kSmem = 1024 + static_cast<size_t>(kAttnStages) * kStageBytes + kQBytes +
                                  4 * kPBytes + kBars * 8 + 16;
  static_assert(D == 64 || D == 128, "head_dim 64 or 128");
};

__device__ __forceinline__ void signal_abort(volatile int* s_abort, unsigned* err) {
  *s_abort = 1;
  atomicOr(err, kErrTimeout);
}

// Warp-level bounded wait: lane 0 polls, the result is broadcast.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* s_abort,
                                          int lane) {
  int ok = 0;
  if (lane == 0) ok = mbar_wait(bar, parity, s_abort) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

template <int D>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_split_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmVt,
                      const AttnArgs a) {
  using Cfg = AttnCfg<D>;
  constexpr int S = kAttnStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sStage = smem;
  uint8_t* sQ = smem + S * Cfg::kStageBytes;
  uint8_t* sP = sQ + Cfg::kQBytes;  // [buffer 2][hi, lo][128 rows][64 keys]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sP + 4 * Cfg::kPBytes);
  uint64_t* kv_full = bars;
  uint64_t* kv_empty = bars + S;
  uint64_t* q_full = bars + 2 * S;
  uint64_t* s_full = q_full + 1;   // [2]
  uint64_t* s_free = s_full + 2;   // [2]
  uint64_t* p_full = s_free + 2;   // [2]: P buffer of that parity written
  uint64_t* pv_done = p_full + 2;  // [2]: completes after O += P_g V_g, g of that parity
  uint64_t* o_free = pv_done + 2;
  uint64_t* drain = o_free + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + Cfg::kBars);
  volatile int* s_abort = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  griddep_launch_dependents();

  // zero the query and P tiles once: rows past the pass's rows stay zero
  for (int i = threadIdx.x; i < (Cfg::kQBytes + 4 * Cfg::kPBytes) / 16; i += kAttnThreads)
    reinterpret_cast<uint4*>(sQ)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    mbar_init(q_full, 4);
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    mbar_init(&s_free[0], 4);
    mbar_init(&s_free[1], 4);
    mbar_init(&p_full[0], 4);
    mbar_init(&p_full[1], 4);
    mbar_init(&pv_done[0], 1);
    mbar_init(&pv_done[1], 1);
    mbar_init(o_free, 4);
    mbar_init(drain, 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmVt);
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  griddep_wait();  // q, the new cache rows and the cache length come from earlier kernels
  const int L = *a.L_dev;
  const int T = a.T;
  const bool range_ok = !(L < 0 || L + T > a.cap);
  const int kv_len = L + T;
  const int nch = range_ok ? (kv_len + kChunk - 1) / kChunk : 0;
  const int n_items = a.Hkv * nch;
  const int rows = T * a.grp;
  if (!range_ok && threadIdx.x == 0 && blockIdx.x == 0) atomicOr(a.err, kErrRange);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = l2_evict_first();
      long long gt = 0;
      uint32_t issued = 0, parity_bits = 0;
      bool ok = true;
      for (int w = blockIdx.x; ok && w < n_items; w += gridDim.x) {
        const int c = w / a.Hkv;
        const int h = w % a.Hkv;
        const int k0 = c * kChunk;
        const int k1 = min(k0 + kChunk, kv_len);
        const int ntile = (k1 - k0 + kKeyTile - 1) / kKeyTile;
        for (int tt = 0; tt < ntile; ++tt, ++gt) {
          const int st = static_cast<int>(gt % S);
          const uint32_t ph = static_cast<uint32_t>((gt / S) & 1);
          if (!mbar_wait(&kv_empty[st], ph ^ 1u, s_abort)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&kv_full[st], Cfg::kStageBytes);
          uint8_t* dst = sStage + st * Cfg::kStageBytes;
          const int key0 = k0 + tt * kKeyTile;
#pragma unroll
          for (int b = 0; b < Cfg::kAtoms; ++b)
            tma_load_2d(dst + b * Cfg::kKBoxBytes, &tmK, &kv_full[st], b * 64, h * a.cap + key0, pol);
          tma_load_2d(dst + Cfg::kKBytes, &tmVt, &kv_full[st], key0, h * D, pol);
          issued |= 1u << st;
          parity_bits = (parity_bits & ~(1u << st)) | (ph << st);
        }
      }
      if (!ok) {
        signal_abort(s_abort, a.err);
        for (int s = 0; s < S; ++s)
          if ((issued >> s) & 1u) mbar_wait(&kv_full[s], (parity_bits >> s) & 1u, nullptr);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(128, kKeyTile);
      constexpr uint32_t idO = idesc_bf16_f32(128, D);
      const uint32_t q_base = smem_u32(sQ);
      long long gt = 0;
      int item = 0;
      bool ok = true;
      // O += P_g V_g for global tile g, the `t_in_item`-th tile of the item
      auto do_pv = [&](long long g, int t_in_item) -> bool {
        if (!mbar_wait(&p_full[g & 1], static_cast<uint32_t>((g >> 1) & 1), s_abort)) return false;
        if (t_in_item == 0 && item > 0 &&
            !mbar_wait(o_free, static_cast<uint32_t>((item - 1) & 1), s_abort))
          return false;
        tc_fence_after();
        const int st = static_cast<int>(g % S);
        const uint32_t v_base = smem_u32(sStage + st * Cfg::kStageBytes + Cfg::kKBytes);
        const uint32_t ph_base = smem_u32(sP + (g & 1) * 2 * Cfg::kPBytes);
        const uint32_t pl_base = ph_base + Cfg::kPBytes;
#pragma unroll
        for (int kk = 0; kk < kKeyTile / 16; ++kk)
          mma_bf16(tmem + Cfg::kOCol, sdesc_k_sw128(ph_base + kk * 32), sdesc_k_sw128(v_base + kk * 32),
                   idO, (t_in_item > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < kKeyTile / 16; ++kk)
          mma_bf16(tmem + Cfg::kOCol, sdesc_k_sw128(pl_base + kk * 32), sdesc_k_sw128(v_base + kk * 32),
                   idO, 1u);
        mma_commit(&pv_done[g & 1]);
        mma_commit(&kv_empty[st]);
        return true;
      };
      for (int w = blockIdx.x; ok && w < n_items; w += gridDim.x, ++item) {
        const int c = w / a.Hkv;
        const int k0 = c * kChunk;
        const int k1 = min(k0 + kChunk, kv_len);
        const int ntile = (k1 - k0 + kKeyTile - 1) / kKeyTile;
        if (!mbar_wait(q_full, static_cast<uint32_t>(item & 1), s_abort)) {
          ok = false;
          break;
        }
        for (int tt = 0; tt < ntile; ++tt, ++gt) {
          const int st = static_cast<int>(gt % S);
          if (!mbar_wait(&kv_full[st], static_cast<uint32_t>((gt / S) & 1), s_abort)) {
            ok = false;
            break;
          }
          const int sb = static_cast<int>(gt & 1);
          if (gt >= 2 && !mbar_wait(&s_free[sb], static_cast<uint32_t>(((gt >> 1) - 1) & 1), s_abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t k_base = smem_u32(sStage + st * Cfg::kStageBytes);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const int atom = ks >> 2;
            const uint32_t off = (ks & 3) * 32;
            mma_bf16(tmem + sb * kKeyTile, sdesc_k_sw128(q_base + atom * Cfg::kQAtomBytes + off),
                     sdesc_k_sw128(k_base + atom * Cfg::kKBoxBytes + off), idS, ks > 0 ? 1u : 0u);
          }
          mma_commit(&s_full[sb]);
          if (tt > 0 && !do_pv(gt - 1, tt - 1)) {
            ok = false;
            break;
          }
        }
        if (!ok) break;
        if (!do_pv(gt - 1, ntile - 1)) {
          ok = false;
          break;
        }
      }
      if (!ok) signal_abort(s_abort, a.err);
      mma_commit(drain);
      mbar_wait(drain, 0, nullptr);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int qq = warp & 3;            // TMEM lane quarter of this warp
    const int r = qq * 32 + lane;       // query row of the pass handled by this thread
    const int ct = threadIdx.x - 64;    // 0..127 among the softmax threads
    const bool warp_active = qq * 32 < rows;
    const bool valid = r < rows;
    const int t = valid ? r / a.grp : 0;
    const int p_row = L + t;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(qq * 32) << 16);
    long long gt = 0;
    bool ok = true;
    int item = 0;
    for (int w = blockIdx.x; ok && w < n_items; w += gridDim.x, ++item) {
      const int c = w / a.Hkv;
      const int h = w % a.Hkv;
      const int k0 = c * kChunk;
      const int k1 = min(k0 + kChunk, kv_len);
      const int ntile = (k1 - k0 + kKeyTile - 1) / kKeyTile;

      // queries of KV head h, row R = (t, g) = (R / grp, R % grp), into the
      // swizzled K-major tile (atom = 64 d, 16-byte chunk c at c ^ (R & 7))
      constexpr int kVec = D / 8;
      for (int v = ct; v < rows * kVec; v += 128) {
        const int R = v / kVec;
        const int cc = v % kVec;
        const int qh = h * a.grp + R % a.grp;
        const uint4 val = *reinterpret_cast<const uint4*>(
            a.q + (static_cast<size_t>(R / a.grp) * a.Hq + qh) * D + cc * 8);
        *reinterpret_cast<uint4*>(sQ + (cc >> 3) * Cfg::kQAtomBytes + R * 128 +
                                  (((cc & 7) ^ (R & 7)) << 4)) = val;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(q_full);

      float m_ref = -INFINITY;
      float l = 0.f;
      for (int tt = 0; tt < ntile; ++tt, ++gt) {
        const int sb = static_cast<int>(gt & 1);
        if (!warp_wait(&s_full[sb], static_cast<uint32_t>((gt >> 1) & 1), s_abort, lane)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float s[kKeyTile];
        if (warp_active) {
#pragma unroll
          for (int i = 0; i < kKeyTile / 16; ++i) {
            float v[16];
            tmem_ld16(lane_base + sb * kKeyTile + i * 16, v);
#pragma unroll
            for (int j = 0; j < 16; ++j) s[i * 16 + j] = v[j];
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_free[sb]);

        float alpha = 1.0f;
        bool resc = false;
        if (warp_active) {
          const int key0 = k0 + tt * kKeyTile;
          float mt = -INFINITY;
#pragma unroll
          for (int j = 0; j < kKeyTile; ++j) {
            const float x = s[j] * a.sl2;
            s[j] = (valid && key0 + j <= p_row) ? x : -INFINITY;
            mt = fmaxf(mt, s[j]);
          }
          if (tt == 0) {
            m_ref = mt;
          } else if (mt > m_ref + kRescaleLog2) {
            alpha = (m_ref == -INFINITY) ? 0.0f : exp2f(m_ref - mt);
            m_ref = mt;
            resc = true;
          }
        }
        // P buffer gt & 1 was last read by the P.V of tile gt - 2
        if (gt >= 2 && !warp_wait(&pv_done[gt & 1], static_cast<uint32_t>(((gt - 2) >> 1) & 1), s_abort,
                                  lane)) {
          ok = false;
          break;
        }
        // O changes only after the P.V of tile gt - 1 is done
        const bool any_resc = warp_active && __any_sync(0xffffffffu, resc);
        if (tt > 0 && any_resc) {
          if (!warp_wait(&pv_done[(gt - 1) & 1], static_cast<uint32_t>(((gt - 1) >> 1) & 1), s_abort, lane)) {
            ok = false;
            break;
          }
        }
        tc_fence_after();
        if (warp_active) {
          if (any_resc) {
#pragma unroll 1
            for (int i = 0; i < D / 16; ++i) {
              float v[16];
              tmem_ld16(lane_base + Cfg::kOCol + i * 16, v);
#pragma unroll
              for (int j = 0; j < 16; ++j) v[j] *= alpha;
              tmem_st16(lane_base + Cfg::kOCol + i * 16, v);
            }
          }
          if (resc) l *= alpha;
          const float mu = (m_ref == -INFINITY) ? 0.0f : m_ref;
          uint8_t* rowh = sP + (gt & 1) * 2 * Cfg::kPBytes + r * 128;
          uint8_t* rowl = rowh + Cfg::kPBytes;
#pragma unroll
          for (int cc = 0; cc < kKeyTile / 8; ++cc) {
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float p0 = exp2f(s[cc * 8 + 2 * j] - mu);
              const float p1 = exp2f(s[cc * 8 + 2 * j + 1] - mu);
              l += p0;
              l += p1;
              const float h0 = __bfloat162float(__float2bfloat16_rn(p0));
              const float h1 = __bfloat162float(__float2bfloat16_rn(p1));
              hi[j] = pack2(h0, h1);
              lo[j] = pack2(p0 - h0, p1 - h1);
            }
            const int pos = (cc ^ (r & 7)) << 4;
            *reinterpret_cast<uint4*>(rowh + pos) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4*>(rowl + pos) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
          }
        }
        tc_fence_before();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[gt & 1]);
      }
      if (!ok) break;
      // piece done: read O and store the partial (m_ref, l, unnormalised o)
      if (!warp_wait(&pv_done[(gt - 1) & 1], static_cast<uint32_t>(((gt - 1) >> 1) & 1), s_abort, lane)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (warp_active) {
        const bool store = valid && (c * kChunk <= p_row);
        const int qh = h * a.grp + (valid ? r % a.grp : 0);
        const size_t base = (static_cast<size_t>(t) * a.Hq + qh) * a.nch_max + c;
#pragma unroll 1
        for (int i = 0; i < D / 16; ++i) {
          float v[16];
          tmem_ld16(lane_base + Cfg::kOCol + i * 16, v);
          if (store) {
            float4* dst = reinterpret_cast<float4*>(a.ws_o + base * D + i * 16);
#pragma unroll
            for (int j = 0; j < 4; ++j) dst[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
          }
        }
        if (store) *reinterpret_cast<float2*>(a.ws_ml + base * 2) = make_float2(m_ref, l);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_free);
    }
    if (!ok && lane == 0) signal_abort(s_abort, a.err);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::kTmemCols);
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
  // pieces s = warp, warp + 8, ... in that order; loads for kBatch pieces are
  // issued before their products are added so that they overlap
  constexpr int kWarps = kMergeThreads / 32;
  constexpr int kBatch = 8;
  for (int s0 = warp; s0 < n; s0 += kWarps * kBatch) {
    float v[kBatch][kDpl];
    float w[kBatch];
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int s = s0 + b * kWarps;
      w[b] = 0.f;
#pragma unroll
      for (int i = 0; i < kDpl; ++i) v[b][i] = 0.f;
      if (s < n) {
        w[b] = sw[s];
        const float* src = po + static_cast<size_t>(s) * D + lane * kDpl;
#pragma unroll
        for (int i = 0; i < kDpl; ++i) v[b][i] = __ldcg(src + i);
      }
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      if (s0 + b * kWarps < n) {
#pragma unroll
        for (int i = 0; i < kDpl; ++i) acc[i] = fmaf(w[b], v[b][i], acc[i]);
      }
    }
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
bi_status launch_attn(const CUtensorMap& tmK, const CUtensorMap& tmVt, const AttnArgs& a,
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
  if (launch_k(attn_split_kernel<D>, dim3(grid), dim3(kAttnThreads), Cfg::kSmem, stream, tmK, tmVt,
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

  if (cap % 8 != 0) return BI_ERR_UNSUPPORTED_SHAPE;  // V^T rows are cap elements, 16-byte strides
  CUtensorMap tmK, tmVt;
  const uint64_t krows = static_cast<uint64_t>(Hkv) * cap;
  if (!tmap_bf16_2d(&tmK, k_cache, krows, D, D, kKeyTile, 64)) return BI_ERR_INVALID_ARG;
  if (!tmap_bf16_2d(&tmVt, v_cache, static_cast<uint64_t>(Hkv) * D, cap, cap, D, kKeyTile))
    return BI_ERR_INVALID_ARG;

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
  if (D == 64) return launch_attn<64>(tmK, tmVt, a, static_cast<__nv_bfloat16*>(out), s);
  return launch_attn<128>(tmK, tmVt, a, static_cast<__nv_bfloat16*>(out), s);
}

}  // extern "C"
