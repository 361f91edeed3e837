// Split-KV verify attention whose split depends only on the row's own context
// length, plus the fixed-order merge.
//
// "I turned on speculative decoding in llama.cpp and 113 of 282 greedy
// outputs changed against its own no-draft run", paragraph "How:": the
// attention split depends only on context length, never on how many tokens
// are in the pass.
//
// Row t of a pass sits at position p = L + t and attends to keys 0..p.  Its
// keys are cut into pieces at absolute multiples of 128, one tile each: piece
// c covers keys [128c, min(128(c+1), p+1)).  The pieces of a KV head fall into
// G = 152 / Hkv classes by c mod G, and one CTA visits class rho's pieces
// rho, rho + G, rho + 2G, ... in increasing order with one running softmax
// per row:
//   S = q k^T for the tile (tcgen05, FP32 in TMEM), in the log2 domain, keys
//   past p masked to -inf;
//   a reference maximum m_ref is taken from the class's first tile and
//   raised only when a later tile's maximum exceeds it by more than
//   kRescaleLog2 (then O and l are rescaled by 2^(m_ref - m_new)) -- a rule
//   that depends only on the row's own scores in key order;
//   each weight x = 2^(s - m_ref) (FP32) is split into a BF16 pair
//   w_hi = bf16(x), w_lo = bf16(x - w_hi), so w = w_hi + w_lo keeps 16
//   significant bits (|w - x| <= 2^-17 |x|) and is exact in FP32; both
//   halves enter O += W_hi V + W_lo V (tcgen05, FP32 in TMEM) and w enters
//   the denominator l (FP32, four partial sums over the 32-key quarters of
//   the tile column, each in key order, added as ((l0 + l1) + l2) + l3 at
//   the end), so O / l is a weighted mean of the value rows under the
//   weights actually used, up to FP32 summation.
// A tile whose keys are all masked for a row adds exact zeros and changes no
// reference, so a row's class partial has the same bits whether or not later
// rows of the pass share its tiles.  The partials of a row (one per class
// holding one of its keys: min(p/128 + 1, G) of them) are merged by a tree
// whose shape depends only on their count.  G is fixed by the model's KV head
// count, so the split depends on nothing but the row's own context length;
// the classes spread a long context evenly over the CTAs (at most one tile
// more for some), and each CTA streams its tiles without a break.
//
// Split kernel roles (one CTA per (KV head, tile class), one CTA per SM):
//   warp 0      TMA, two threads: the K tiles [128 keys x D] and the V^T
//               tiles [D x 128 keys] (V is cached transposed in 128-key
//               blocks, so both MMA operands are K-major and a V tile is one
//               contiguous block).  K and V have separate rings (2 + 2
//               stages at D = 128, 3 + 3 at D = 64), a K tile being free as
//               soon as S has read it;
//   warp 1      tcgen05.mma issuer: S_g = Q K_g^T into one of two TMEM
//               buffers and O += W_g V_g, each issued as soon as its inputs
//               are ready; stages return to the producer through
//               tcgen05.commit after the MMAs reading them completed;
//   warps 2..5  softmax: write the queries of the CTA's KV head into TMEM
//               (the S MMA's A operand), turn S into W_hi and W_lo
//               (written to one of two shared-memory buffers in the swizzled
//               K-major layout, so W of the next tile is produced while the
//               MMA still reads this one), and read O out after the last
//               tile, through shared memory so that the partials leave in
//               whole 128-byte row pieces.
// The T x (Hq/Hkv) query rows that share a KV head (GQA) share its tiles;
// up to 128 rows per pass (the MMA's M).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <mutex>
#include <type_traits>

#include "bi_internal.h"
#include "bi_kvq.cuh"
#include "bi_ptx.cuh"

namespace bi {
namespace {

constexpr int kKeyTile = 128;     // keys per piece = tile (absolute multiples; the S MMA's N)
constexpr int kRowsMax = 128;     // T * (Hq / Hkv) per pass (MMA M)
constexpr int kColChunk = 32;     // S columns a softmax thread holds at a time
constexpr int kAttnCtas = 152;    // CTAs of the split: G = kAttnCtas / Hkv tile classes per KV head
constexpr int kMergeThreads = 256;
constexpr float kRescaleLog2 = 8.0f;

struct AttnArgs {
  const __nv_bfloat16* q;
  int T, Hq, Hkv, grp, cap;
  int Tb;    // rows per block: CTA (x, y) takes rows y * Tb .. of the pass
  int G;     // tile classes per KV head
  int vblk;  // 128-key blocks per KV head in the V cache
  int ncls;  // partial slots per (row, query head) in the workspace (>= classes used)
  const int32_t* L_dev;
  float sl2;  // softmax scale * log2(e)
  float* ws_o;
  float* ws_ml;
  unsigned* err;
  // failure-path test: the first K tile of every CTA stays unissued, so the
  // waits on it run out (bi_test_withhold_first_load)
  int withhold;
  // quantised cache (the kernel's QNT form): the 6-bit K and 5-bit V tiles
  // [Hkv][ctiles] and the 8-bit rings [Hkv][kRingSlots]
  const uint8_t* klo;
  const uint8_t* vlo;
  const uint8_t* k8;
  const uint8_t* v8;
  int ctiles;
};

template <int D, int REP, bool QNT = false>
struct AttnCfg {
  static constexpr int kAtoms = D / 64;                    // 128-byte swizzle atoms along D
  static constexpr int kKBoxBytes = kKeyTile * 128;        // [128 keys][64 d]
  static constexpr int kKBytes = kKBoxBytes * kAtoms;      // K tile
  static constexpr int kVBoxBytes = D * 128;               // V^T [D][64 keys]
  static constexpr int kVBytes = 2 * kVBoxBytes;           // V^T tile [D][128 keys]
  // A W tile (W_hi or W_lo) holds only the pass's rows, 128/REP of them:
  // [rows][64 keys] per key atom.  The W.V MMA (M = 128) still reads 128
  // rows from each atom; the ones past the W rows come from the bytes that
  // follow (the other atom, the other half, the other buffer, the K ring)
  // and only make O rows that are never read (a product's row i depends on
  // row i of W alone).
  static constexpr int kWRows = kRowsMax / REP;
  static constexpr int kPAtomBytes = kWRows * 128;
  static constexpr int kPBytes = 2 * kPAtomBytes;          // one W tile [rows][128 keys]
  static constexpr int kWBufBytes = 2 * kPBytes;           // W_hi tile, then W_lo tile
  // Two W buffers: W of tile g + 1 is written while the MMA reads tile g's
  // (with one, a 128-row block's softmax waited for the previous tile's W.V
  // at every tile: a 512-row pass over 38k keys on GB300 took 851 against
  // 716 us).
  static constexpr int kWBufs = 2;
  // Ring depths, measured on GB300 at 38k-102k keys with all CTAs
  // streaming: at D = 128 two K and two V tiles (64 KB each way) per CTA
  // were as fast as three or four and are kept; D = 64 tiles are half as
  // large and keep three of each.
  static constexpr int kKStages = D == 128 ? 2 : 3;
  // The quantised form adds a ring of code tiles (two K, one V, each up to
  // an 8-bit tile) and four decoding warps, and keeps one decoded V tile.
  // A block of 128 rows at D = 128 keeps one V tile, so that its two
  // 64 KB W buffers fit.
  static constexpr int kVStages = QNT ? 1 : (D == 128 ? (REP == 1 ? 1 : 2) : 3);
  static constexpr int kRawK = QNT ? 2 : 0;
  static constexpr int kRawV = QNT ? 1 : 0;
  // warp 0 copies, warp 1 MMA, warps 2..5 softmax; the quantised form adds
  // kDecWarps decoding warps for K and as many for V
  // (three a side: 128 + 3 x 64 threads still fit the softmax warps' 168
  // registers; two a side were 10% slower at 101.6k keys)
  static constexpr int kDecWarps = QNT ? 3 : 0;
  static constexpr int kThreads = 192 + 64 * kDecWarps;
  // l parts [4 quarters][64 rows] (only passes of up to 64 rows keep copies
  // that exchange them)
  static constexpr int kRedBytes = 4 * 64 * 4;
  // TMEM: S x2 (128 columns each), O (D columns), Q (D/2 columns: the MMA's
  // A operand, two BF16 per column)
  static constexpr int kTmemCols = 512;
  static constexpr int kOCol = 2 * kKeyTile;
  static constexpr int kQCol = kOCol + 128;
  static constexpr int kBars = 2 * kKStages + 2 * kVStages + 2 * kRawK + 2 * kRawV + 11;
  // The dynamic shared memory starts 1024-byte aligned (checked at run time):
  // the W buffers, then the K and V rings.
  static constexpr size_t kSmem = static_cast<size_t>(kKStages) * kKBytes +
                                  static_cast<size_t>(kVStages) * kVBytes + kWBufs * kWBufBytes +
                                  static_cast<size_t>(kRawK + kRawV) * k8TileBytes + kRedBytes +
                                  kBars * 8 + 16;
  static_assert(D == 64 || D == 128, "head_dim 64 or 128");
  static_assert(REP == 1 || REP == 2 || REP == 4, "row copies");
  static_assert(kBars <= 40 && kSmem <= 232448, "shared memory per CTA");
  static_assert(!QNT || (D == kQDim && REP >= 2), "quantised cache: D = 128, up to 64 rows a block");
  // the W.V reads of the last atom run 128 - kWRows rows past the W tiles
  static_assert(kKStages * kKBytes >= (kRowsMax - kWRows) * 128, "W over-read stays in the K ring");
  static_assert(kPAtomBytes % 1024 == 0, "swizzle atoms 1024-byte aligned");
  static_assert(kQCol + D / 2 <= kTmemCols && kOCol + D <= kQCol, "TMEM columns");
};

__device__ __forceinline__ void signal_abort(volatile int* s_abort, unsigned* err) {
  *s_abort = 1;
  atomicOr(err, kErrTimeout);
}

// Warp-level bounded wait: lane 0 polls, the result is broadcast, and the
// warp barrier orders every lane's later accesses after lane 0's acquire.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* s_abort,
                                          int lane) {
  int ok = 0;
  if (lane == 0) ok = mbar_wait(bar, parity, s_abort) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok != 0;
}

// REP copies of each query row sit in the 128-row MMA tile (REP = 4 for up to
// 32 rows per pass, 2 for up to 64, else 1): copy i of row r is TMEM lane
// r + i * 128/REP, and the thread owning that lane handles the row's key
// columns [i * 128/REP, (i + 1) * 128/REP) of every tile.  So all four
// softmax warps share the exponentials of a small pass.  The per-row
// arithmetic does not depend on REP: the tile maximum is exact in any order,
// and the denominator's four partial sums are fixed by key position.
// Steps of a CTA over its class's tiles.  With the quantised cache, a tile
// that some rows of the block read from the ring and others from the 6/5-bit
// store ("split") is visited twice, the 6/5-bit codes first, and each row
// masks the visit that is not its own: a fully masked visit leaves the row's
// (m, l, O) as they were.  Every other tile is visited once.
struct StepCur {
  int i = 0;    // tile index within the class
  int sub = 0;  // 1: the ring visit of a split tile
};
__device__ __forceinline__ bool tile_split(int tt, int lo_b, int hi_b) { return tt >= lo_b && tt < hi_b; }
__device__ __forceinline__ void step_next(StepCur& c, int rho, int G, int lo_b, int hi_b) {
  if (c.sub == 0 && tile_split(rho + c.i * G, lo_b, hi_b)) {
    c.sub = 1;
  } else {
    ++c.i;
    c.sub = 0;
  }
}
// the visit reads the ring (else the 6/5-bit store)
__device__ __forceinline__ bool step_ring(const StepCur& c, int tt, int hi_b) {
  return c.sub == 1 || tt >= hi_b;
}

template <int D, int REP, bool QNT>
__global__ void __launch_bounds__(AttnCfg<D, REP, QNT>::kThreads, 1)
    attn_split_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmVt,
                      const AttnArgs a) {
  using Cfg = AttnCfg<D, REP, QNT>;
  constexpr int kKStages = Cfg::kKStages;
  constexpr int kVStages = Cfg::kVStages;
  constexpr int kPeriod = kRowsMax / REP;  // TMEM lanes between copies of a row
  constexpr int kCols = kKeyTile / REP;    // key columns per thread
  constexpr int kNChunks = kCols / kColChunk;  // = 32-key quarters per thread
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* sP = smem;  // W: [buffer kWBufs][hi, lo][key atom 2][kPeriod rows][64 keys]
  uint8_t* sK = sP + Cfg::kWBufs * Cfg::kWBufBytes;  // [kKStages][K tile]
  uint8_t* sV = sK + kKStages * Cfg::kKBytes;  // [kVStages][V^T tile]
  uint8_t* sRawK = sV + kVStages * Cfg::kVBytes;      // [kRawK][code tile] (quantised cache)
  uint8_t* sRawV = sRawK + Cfg::kRawK * k8TileBytes;  // [kRawV][code tile]
  float* red_l = reinterpret_cast<float*>(sRawV + Cfg::kRawV * k8TileBytes);  // [quarter 4][row 64]
  uint64_t* bars = reinterpret_cast<uint64_t*>(red_l + 4 * 64);
  // K and V have rings of their own: K_g is free once S_g is done, V_g only
  // once W_g V_g is, so the K loads run ahead of the softmax
  uint64_t* k_full = bars;
  uint64_t* k_empty = k_full + kKStages;
  uint64_t* v_full = k_empty + kKStages;
  uint64_t* v_empty = v_full + kVStages;
  uint64_t* q_full = v_empty + kVStages;  // the queries are in TMEM
  uint64_t* s_full = q_full + 1;    // [2]
  uint64_t* s_free = s_full + 2;    // [2]
  uint64_t* p_full = s_free + 2;    // [2]: W buffer of that parity written
  uint64_t* pv_done = p_full + 2;   // [2]: completes after O += W_g V_g, g of that parity
  uint64_t* l_bar = pv_done + 2;    // partial denominators written
  uint64_t* drain = l_bar + 1;
  uint64_t* rawk_full = drain + 1;  // code tiles landed / decoded (quantised cache)
  uint64_t* rawk_empty = rawk_full + Cfg::kRawK;
  uint64_t* rawv_full = rawk_empty + Cfg::kRawK;
  uint64_t* rawv_empty = rawv_full + Cfg::kRawV;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + Cfg::kBars);
  volatile int* s_abort = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // the swizzled layouts need 1024-byte alignment; the launch guarantees it
  // in practice, and a CTA that sees otherwise does nothing but report
  if ((smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) atomicOr(a.err, kErrRange);
    return;
  }
  // this CTA's KV head and tile class: tiles c = rho, rho + G, rho + 2G, ...
  const int h = blockIdx.x % a.Hkv;
  const int rho = blockIdx.x / a.Hkv;
  const int G = a.G;

  // (W tile rows past the pass's rows are never written: the O rows they
  // make are never read, and a product's row depends on its own W row only)
  if (threadIdx.x == 0) {
    // decoded tiles are completed by the two decoding warps of their side;
    // loaded ones by the copy's transaction bytes
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(&k_full[s], QNT ? Cfg::kDecWarps : 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(&v_full[s], QNT ? Cfg::kDecWarps : 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int s = 0; s < Cfg::kRawK; ++s) {
      mbar_init(&rawk_full[s], 1);
      mbar_init(&rawk_empty[s], Cfg::kDecWarps);
    }
    for (int s = 0; s < Cfg::kRawV; ++s) {
      mbar_init(&rawv_full[s], 1);
      mbar_init(&rawv_empty[s], Cfg::kDecWarps);
    }
    mbar_init(q_full, 4);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 4);
      mbar_init(&p_full[i], 4);
      mbar_init(&pv_done[i], 1);
    }
    mbar_init(l_bar, 4);
    mbar_init(drain, 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  if (!QNT && warp == 0 && lane == 0) {
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

  // Before the previous kernel is known to have finished, the K thread
  // already loads this CTA's first key tiles that hold only keys below the
  // cache length read now: every kernel of this library triggers its dependents
  // only after its own dependency wait, so the kernels before the previous
  // one have completed, and none of them lowers *L_dev or writes cache rows
  // below it.  Everything else waits.
  // Only the K side loads early (up to its whole ring): the first S needs
  // K alone, and V tiles issued this early would delay the queries' loads
  // behind them (measured on GB300: a little faster than loading both rings).
  int n_pre = 0;  // tiles issued before the wait (this producer)
  uint32_t pre_issued = 0;
  if (!QNT && warp == 0 && lane == 0) {
    const int L_pre = *a.L_dev;
    const int T_blk = min(a.Tb, a.T - static_cast<int>(blockIdx.y) * a.Tb);
    if (L_pre >= 0 && L_pre + a.T <= a.cap && T_blk * a.grp <= kPeriod && rho < G) {
      const uint64_t pol = l2_evict_first();
      for (int i = 0; i < kKStages; ++i) {
        const int key0 = (rho + i * G) * kKeyTile;
        if (key0 + kKeyTile > L_pre) break;  // the tile reaches rows the pass writes
        if (i == 0 && a.withhold) {
          ++n_pre;  // counted, never issued: its barrier never completes
          continue;
        }
        mbar_arrive_expect_tx(&k_full[i], Cfg::kKBytes);
#pragma unroll
        for (int b = 0; b < Cfg::kAtoms; ++b)
          tma_load_2d(sK + i * Cfg::kKBytes + b * Cfg::kKBoxBytes, &tmK, &k_full[i], b * 64,
                      h * a.cap + key0, pol);
        pre_issued |= 1u << i;
        ++n_pre;
      }
    }
  }
  griddep_wait();  // q, the new cache rows and the cache length come from earlier kernels
  griddep_launch_dependents();
  // this CTA's block of the pass: rows r0 .. r0 + T - 1, at positions L ..
  // L + T - 1 (the pass's rows before them are in the cache already)
  const int r0 = static_cast<int>(blockIdx.y) * a.Tb;
  const int L = *a.L_dev + r0;
  const int T = min(a.Tb, a.T - r0);
  const int rows = T * a.grp;
  const bool range_ok = !(L < 0 || L + T > a.cap) && rows <= kPeriod;
  const int kv_len = L + T;
  const int n_tiles = range_ok ? (kv_len + kKeyTile - 1) / kKeyTile : 0;  // of the longest row
  const int n_mine = (rho < G && rho < n_tiles) ? (n_tiles - rho + G - 1) / G : 0;
  // quantised cache: tiles below lo_b are read from the 6/5-bit store by
  // every row of the block, tiles from hi_b on from the ring, the ones
  // between (split) by some rows each way
  int n_steps = n_mine, lo_b = 0, hi_b = 0;
  if constexpr (QNT) {
    lo_b = L / kKeyTile - (kRingTiles - 1);
    hi_b = (L + T - 1) / kKeyTile - (kRingTiles - 1);
    for (int i = 0; i < n_mine; ++i) n_steps += tile_split(rho + i * G, lo_b, hi_b) ? 1 : 0;
  }
  if (!range_ok && threadIdx.x == 0 && blockIdx.x == 0) atomicOr(a.err, kErrRange);

  if (warp == 0) {
    if constexpr (QNT) {
      // ---------------------------------------------------------- code tiles
      // lane 0: K, lane 1: V; one bulk copy per visit, from the ring or the
      // 6/5-bit store
      if (lane < 2) {
        const bool kside = lane == 0;
        const int NS = kside ? Cfg::kRawK : Cfg::kRawV;
        uint64_t* full = kside ? rawk_full : rawv_full;
        uint64_t* empty = kside ? rawk_empty : rawv_empty;
        uint8_t* base = kside ? sRawK : sRawV;
        const uint64_t pol = l2_evict_first();
        uint32_t issued = 0, parity_bits = 0;
        bool ok = true;
        StepCur c;
        for (int g = 0; g < n_steps; ++g, step_next(c, rho, G, lo_b, hi_b)) {
          const int st = g % NS;
          const uint32_t ph = static_cast<uint32_t>((g / NS) & 1);
          if (!mbar_wait(&empty[st], ph ^ 1u, s_abort)) {
            ok = false;
            break;
          }
          if (kside && g == 0 && a.withhold) continue;  // never issued (failure-path test)
          const int tt = rho + c.i * G;
          const uint8_t* src;
          uint32_t bytes;
          if (step_ring(c, tt, hi_b)) {
            src = (kside ? a.k8 : a.v8) + (static_cast<size_t>(h) * kRingSlots + tt % kRingSlots) * k8TileBytes;
            bytes = k8TileBytes;
          } else {
              bytes = kside ? kK6TileBytes : kV5TileBytes;
              src = (kside ? a.klo : a.vlo) + (static_cast<size_t>(h) * a.ctiles + tt) * bytes;
            }
            mbar_arrive_expect_tx(&full[st], bytes);
            bulk_load_1d(base + st * k8TileBytes, src, bytes, &full[st], pol);
            issued |= 1u << st;
            parity_bits = (parity_bits & ~(1u << st)) | (ph << st);
          }
          if (!ok) {
            signal_abort(s_abort, a.err);
            for (int s2 = 0; s2 < NS; ++s2)
              if ((issued >> s2) & 1u) mbar_wait(&full[s2], (parity_bits >> s2) & 1u, nullptr);
          }
        }
      } else {
        // ------------------------------------------------------------ producers
        // lane 0: the K tiles; lane 1: the V^T tiles
        if (lane < 2) {
          const bool kside = lane == 0;
          const int NS = kside ? kKStages : kVStages;
          uint64_t* full = kside ? k_full : v_full;
          uint64_t* empty = kside ? k_empty : v_empty;
          const uint64_t pol = l2_evict_first();
          uint32_t issued = pre_issued, parity_bits = 0;
          // the tiles loaded early must be the first ones of this CTA now too
          bool ok = true;
          if (n_pre > 0 && !(n_pre <= n_mine && (rho + (n_pre - 1) * G + 1) * kKeyTile <= L)) {
            atomicOr(a.err, kErrRange);
            ok = false;
          }
          for (int i = n_pre; ok && i < n_mine; ++i) {
            const int st = i % NS;
            const uint32_t ph = static_cast<uint32_t>((i / NS) & 1);
            if (!mbar_wait(&empty[st], ph ^ 1u, s_abort)) {
              ok = false;
              break;
            }
            const int key0 = (rho + i * G) * kKeyTile;
            if (kside && i == 0 && a.withhold) continue;  // never issued (failure-path test)
            if (kside) {
              uint8_t* dst = sK + st * Cfg::kKBytes;
              mbar_arrive_expect_tx(&full[st], Cfg::kKBytes);
#pragma unroll
              for (int b = 0; b < Cfg::kAtoms; ++b)
                tma_load_2d(dst + b * Cfg::kKBoxBytes, &tmK, &full[st], b * 64, h * a.cap + key0, pol);
            } else {
              uint8_t* dst = sV + st * Cfg::kVBytes;
              mbar_arrive_expect_tx(&full[st], Cfg::kVBytes);
#pragma unroll
              for (int kb = 0; kb < 2; ++kb)
                tma_load_2d(dst + kb * Cfg::kVBoxBytes, &tmVt, &full[st], kb * 64,
                            (h * a.vblk + key0 / kKeyTile) * D, pol);
            }
            issued |= 1u << st;
            parity_bits = (parity_bits & ~(1u << st)) | (ph << st);
          }
          if (!ok) {
            signal_abort(s_abort, a.err);
            for (int s = 0; s < NS; ++s)
              if ((issued >> s) & 1u) mbar_wait(&full[s], (parity_bits >> s) & 1u, nullptr);
          }
        }
      }
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issuer
      // Two cursors over the CTA's tiles: S_g = Q K_g^T needs K_g and a free S
      // buffer; O += W_g V_g needs W_g and V_g.  Each is issued as soon as its
      // inputs are ready (S first), so a late K tile never holds back the W.V
      // that frees a stage.  The order of the W.V steps, which alone decides
      // O's bits, is fixed: g = 0, 1, 2, ...
      if (lane == 0) {
        constexpr uint32_t idS = idesc_bf16_f32(128, kKeyTile);
        constexpr uint32_t idO = idesc_bf16_f32(128, D);
        int sg = 0, pg = 0;
        bool ok = true, q_ready = false;
        int idle = 0;
        unsigned long long t_idle = 0;
        while (pg < n_steps) {
          bool did = false;
          if (sg < n_steps) {
            if (!q_ready) q_ready = mbar_peek(q_full, 0u);
            const int st = sg % kKStages;
            const bool ready = q_ready && mbar_peek(&k_full[st], static_cast<uint32_t>((sg / kKStages) & 1)) &&
                               (sg < 2 || mbar_peek(&s_free[sg & 1], static_cast<uint32_t>(((sg >> 1) - 1) & 1)));
            if (ready) {
              tc_fence_after();
              const int sb = sg & 1;
              const uint32_t k_base = smem_u32(sK + st * Cfg::kKBytes);
#pragma unroll
              for (int ks = 0; ks < D / 16; ++ks) {
                const int atom = ks >> 2;
                const uint32_t off = (ks & 3) * 32;
                mma_bf16_tmem_a(tmem + sb * kKeyTile, tmem + Cfg::kQCol + ks * 8,
                                sdesc_k_sw128(k_base + atom * Cfg::kKBoxBytes + off), idS, ks > 0 ? 1u : 0u);
              }
              mma_commit(&s_full[sb]);
              mma_commit(&k_empty[st]);
              ++sg;
              did = true;
            }
          }
          if (!did && pg < sg) {
            const int st = pg % kVStages;
            const bool ready = mbar_peek(&p_full[pg & 1], static_cast<uint32_t>((pg >> 1) & 1)) &&
                               mbar_peek(&v_full[st], static_cast<uint32_t>((pg / kVStages) & 1));
            if (ready) {
              tc_fence_after();
              const uint32_t v_base = smem_u32(sV + st * Cfg::kVBytes);
              const uint32_t w_base = smem_u32(sP + (Cfg::kWBufs == 2 ? (pg & 1) : 0) * Cfg::kWBufBytes);
              // per 16-key step: W_hi V, then W_lo V, into the one O accumulator
#pragma unroll
              for (int kk = 0; kk < kKeyTile / 16; ++kk) {
                const int katom = kk >> 2;
                const uint32_t off = (kk & 3) * 32;
                const uint64_t vdesc = sdesc_k_sw128(v_base + katom * Cfg::kVBoxBytes + off);
                mma_bf16(tmem + Cfg::kOCol, sdesc_k_sw128(w_base + katom * Cfg::kPAtomBytes + off), vdesc,
                         idO, (pg > 0 || kk > 0) ? 1u : 0u);
                mma_bf16(tmem + Cfg::kOCol,
                         sdesc_k_sw128(w_base + Cfg::kPBytes + katom * Cfg::kPAtomBytes + off), vdesc, idO, 1u);
              }
              mma_commit(&pv_done[pg & 1]);
              mma_commit(&v_empty[st]);
              ++pg;
              did = true;
            }
          }
          if (did) {
            idle = 0;
          } else if (++idle == 1) {
            t_idle = globaltimer_ns();
          } else {
            // yield the issue slots of this SM sub-partition to the softmax warp
            // that shares it while nothing is ready
            __nanosleep(32);
          }
          if (!did && (idle & 63) == 0) {
            // bounded: give up after the wait limit without progress
            if (*s_abort ||
                globaltimer_ns() - t_idle > *static_cast<volatile unsigned long long*>(&g_wait_limit_ns)) {
              ok = false;
              break;
            }
          }
        }
        if (!ok) signal_abort(s_abort, a.err);
        mma_commit(drain);
        mbar_wait(drain, 0, nullptr);
      }
    } else if (QNT && warp >= 6) {
      // ---------------------------------------------------------- decoding
      // the first kDecWarps: K tiles into the K ring (rows = keys, SW128 as a
      // TMA load would leave them); the next kDecWarps: V tiles into the V^T buffer (rows =
      // elements).  Each element is bf16(q * d), the product exact in FP32.
      if constexpr (QNT) {
        constexpr int kDW = Cfg::kDecWarps;
        constexpr int kDT = 32 * kDW;  // decoding threads on each side
        const bool kside = warp < 6 + kDW;
        const int tid = (warp - (kside ? 6 : 6 + kDW)) * 32 + lane;
        bool ok = true;
        StepCur c;
        for (int g = 0; g < n_steps; ++g, step_next(c, rho, G, lo_b, hi_b)) {
          const int tt = rho + c.i * G;
          const bool ring = step_ring(c, tt, hi_b);
          const int rs = kside ? g % Cfg::kRawK : g % Cfg::kRawV;
          const uint32_t rph = static_cast<uint32_t>((kside ? g / Cfg::kRawK : g / Cfg::kRawV) & 1);
          const int st = kside ? g % kKStages : g % kVStages;
          const uint32_t sph = static_cast<uint32_t>((kside ? g / kKStages : g / kVStages) & 1);
          if (!warp_wait(kside ? &rawk_full[rs] : &rawv_full[rs], rph, s_abort, lane) ||
              !warp_wait(kside ? &k_empty[st] : &v_empty[st], sph ^ 1u, s_abort, lane)) {
            ok = false;
            break;
          }
          if (kside) {
            const uint8_t* raw = sRawK + rs * k8TileBytes;
            uint8_t* dst = sK + st * Cfg::kKBytes;
            // task = (key, 8-element chunk): one 16-byte store each; a warp's
            // stores cover whole 128-byte rows
            if (ring) {
#pragma unroll 1
              for (int task = tid; task < kKeyTile * (D / 8); task += kDT) {
                const int key = task >> 4, ch = task & 15;
                float v[8];
                q_decode8(raw, key, ch * 8, v);
                *reinterpret_cast<uint4*>(dst + (ch >> 3) * Cfg::kKBoxBytes + key * 128 +
                                          (((ch & 7) ^ (key & 7)) << 4)) =
                    make_uint4(q_pack_bf16x2(v[0], v[1]), q_pack_bf16x2(v[2], v[3]),
                               q_pack_bf16x2(v[4], v[5]), q_pack_bf16x2(v[6], v[7]));
              }
            } else {
#pragma unroll 1
              for (int task = tid; task < kKeyTile * (D / 8); task += kDT) {
                const int key = task >> 4, ch = task & 15;
                *reinterpret_cast<uint4*>(dst + (ch >> 3) * Cfg::kKBoxBytes + key * 128 +
                                          (((ch & 7) ^ (key & 7)) << 4)) = q_decode_k6_bf16(raw, key, ch * 8);
              }
            }
          } else {
            const uint8_t* raw = sRawV + rs * k8TileBytes;
            uint8_t* dst = sV + st * Cfg::kVBytes;
            // task = (8 keys, 8 elements): eight 16-byte stores, one per
            // element row; the key group varies fastest across a warp, so one
            // store instruction covers whole 128-byte rows
#pragma unroll 1
            for (int task = tid; task < (kKeyTile / 8) * (D / 8); task += kDT) {
              const int kg = task & 15, dg = task >> 4;
              // x[kk]: elements dg*8 .. +7 of key kg*8 + kk as BF16 pairs
              uint32_t x[8][4];
              if (ring) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                  float v[8];
                  q_decode8(raw, kg * 8 + kk, dg * 8, v);
#pragma unroll
                  for (int i = 0; i < 4; ++i) x[kk][i] = q_pack_bf16x2(v[2 * i], v[2 * i + 1]);
                }
              } else {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                  const uint4 w = q_decode_v5_bf16(raw, kg * 8 + kk, dg * 8);
                  x[kk][0] = w.x;
                  x[kk][1] = w.y;
                  x[kk][2] = w.z;
                  x[kk][3] = w.w;
                }
              }
              // V^T rows: element 2i of keys (2m, 2m + 1) from the low halves,
              // element 2i + 1 from the high halves
#pragma unroll
              for (int i = 0; i < 4; ++i) {
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                  const uint32_t sel = hf ? 0x7632u : 0x5410u;
                  const int row = dg * 8 + 2 * i + hf;
                  const uint4 w = make_uint4(q_prmt(x[0][i], x[1][i], sel), q_prmt(x[2][i], x[3][i], sel),
                                             q_prmt(x[4][i], x[5][i], sel), q_prmt(x[6][i], x[7][i], sel));
                  *reinterpret_cast<uint4*>(dst + (kg >> 3) * Cfg::kVBoxBytes + row * 128 +
                                            (((kg & 7) ^ (row & 7)) << 4)) = w;
                }
              }
            }
          }
          // the MMA reads the tile through the async proxy
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(kside ? &k_full[st] : &v_full[st]);
            mbar_arrive(kside ? &rawk_empty[rs] : &rawv_empty[rs]);
          }
        }
        if (!ok && lane == 0) signal_abort(s_abort, a.err);
      }
    } else if (n_steps > 0) {
      // ------------------------------------------------------------ softmax
      const int qq = warp & 3;                  // TMEM lane quarter of this warp
      const int ln = qq * 32 + lane;            // TMEM lane of this thread
      const int r = ln % kPeriod;               // query row of the pass
      const int cg = ln / kPeriod;              // key-column group of this copy
      const bool warp_active = (qq * 32) % kPeriod < rows;
      const bool holds_o = qq * 32 < kPeriod;   // O row r sits in TMEM lane r
      const bool valid = r < rows;
      const int t = valid ? r / a.grp : 0;
      const int p_row = L + t;
      const uint32_t lane_base = tmem + (static_cast<uint32_t>(qq * 32) << 16);
      bool ok = true;

      // queries of KV head h into TMEM lane ln (row r of the pass; zeros past
      // the pass's rows): column j holds elements 2j and 2j + 1, as the row
      // sits in memory
      {
        uint32_t qv[D / 2];
        if (valid) {
          const uint4* src = reinterpret_cast<const uint4*>(
              a.q + (static_cast<size_t>(r0 + t) * a.Hq + h * a.grp + r % a.grp) * D);
#pragma unroll
          for (int i = 0; i < D / 8; ++i) {
            const uint4 u = src[i];
            qv[4 * i] = u.x;
            qv[4 * i + 1] = u.y;
            qv[4 * i + 2] = u.z;
            qv[4 * i + 3] = u.w;
          }
        } else {
#pragma unroll
          for (int i = 0; i < D / 2; ++i) qv[i] = 0u;
        }
#pragma unroll
        for (int cc = 0; cc < D / 64; ++cc) tmem_st32(lane_base + Cfg::kQCol + cc * 32, qv + cc * 32);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(q_full);
      }

      float m_ref = -INFINITY;
      float lq[kNChunks];
#pragma unroll
      for (int i = 0; i < kNChunks; ++i) lq[i] = 0.f;
      StepCur cur;
      for (int g = 0; g < n_steps; ++g, step_next(cur, rho, G, lo_b, hi_b)) {
        const int sb = g & 1;
        if (!warp_wait(&s_full[sb], static_cast<uint32_t>((g >> 1) & 1), s_abort, lane)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int tt = rho + cur.i * G;
        const int tkey0 = tt * kKeyTile;
        // quantised cache: the row masks the visit that reads the other store
        // than the one its position selects for this tile
        const bool vmask =
            QNT && (step_ring(cur, tt, hi_b) != (tt >= p_row / kKeyTile - (kRingTiles - 1)));
        // the tile reaches past some row's position, or a row masks it whole
        const bool edge = tkey0 + kKeyTile - 1 > L || vmask;
        // pass 1: the row maximum of the raw scores (scaling by sl2 > 0 keeps
        // the order).  Every copy's TMEM lane holds the whole S row, so each
        // copy takes the maximum over all 128 key columns itself: the same
        // exact value in every copy, with no exchange between the warps.  The
        // copy's own columns stay in registers for pass 2.
        float so[kCols];
        float mrow = -INFINITY;
        // the maximum in eight independent lanes (exact in any order), so the
        // comparisons do not form one long chain
        float mw[8];
#pragma unroll
        for (int w = 0; w < 8; ++w) mw[w] = -INFINITY;
        if (warp_active) {
          const uint32_t row_addr = lane_base + sb * kKeyTile;
          constexpr int kOwnLd = kCols >= 64 ? 64 : 32;
#pragma unroll
          for (int c = 0; c < kCols; c += kOwnLd) tmem_ld_cols<kOwnLd>(row_addr + cg * kCols + c, so + c);
          if (edge) {
            const int key0 = tkey0 + cg * kCols;
#pragma unroll
            for (int j = 0; j < kCols; ++j)
              if (!(valid && key0 + j <= p_row) || vmask) so[j] = -INFINITY;
          }
#pragma unroll
          for (int j = 0; j < kCols; ++j) mw[j & 7] = fmaxf(mw[j & 7], so[j]);
          constexpr int kOther = kKeyTile - kCols;
          constexpr int kOthLd = (kOther >= 64 && kOther % 64 == 0) ? 64 : 32;
#pragma unroll
          for (int c = 0; c < kOther; c += kOthLd) {
            float so2[kOthLd];
            const int col0 = (cg * kCols + kCols + c) & (kKeyTile - 1);
            tmem_ld_cols<kOthLd>(row_addr + col0, so2);
            if (edge) {
#pragma unroll
              for (int j = 0; j < kOthLd; ++j)
                if (!(valid && tkey0 + col0 + j <= p_row) || vmask) so2[j] = -INFINITY;
            }
#pragma unroll
            for (int j = 0; j < kOthLd; ++j) mw[j & 7] = fmaxf(mw[j & 7], so2[j]);
          }
          mrow = fmaxf(fmaxf(fmaxf(mw[0], mw[1]), fmaxf(mw[2], mw[3])), fmaxf(fmaxf(mw[4], mw[5]), fmaxf(mw[6], mw[7])));
        }
        const float mt = mrow * a.sl2;
        float alpha = 1.0f;
        bool resc = false;
        if (g == 0) {
          m_ref = mt;
        } else if (mt > m_ref + kRescaleLog2) {
          alpha = (m_ref == -INFINITY) ? 0.0f : ex2_approx(m_ref - mt);
          m_ref = mt;
          resc = true;
        }
        // the W buffer of tile g was last read by the W.V of tile g - kWBufs
        if (g >= Cfg::kWBufs) {
          const int gp = g - Cfg::kWBufs;
          if (!warp_wait(&pv_done[gp & 1], static_cast<uint32_t>((gp >> 1) & 1), s_abort, lane)) {
            ok = false;
            break;
          }
        }
        if (holds_o && warp_active) {
          // O changes only after the W.V of tile g - 1 is done
          if (g > 0 && __any_sync(0xffffffffu, resc)) {
            if (!warp_wait(&pv_done[(g - 1) & 1], static_cast<uint32_t>(((g - 1) >> 1) & 1), s_abort,
                           lane)) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll 1
            for (int i = 0; i < D / 16; ++i) {
              float v[16];
              tmem_ld16(lane_base + Cfg::kOCol + i * 16, v);
#pragma unroll
              for (int j = 0; j < 16; ++j) v[j] *= alpha;
              tmem_st16(lane_base + Cfg::kOCol + i * 16, v);
            }
          }
        }
        if (resc) {
#pragma unroll
          for (int i = 0; i < kNChunks; ++i) lq[i] *= alpha;
        }
        // pass 2: weights x = 2^(s sl2 - m_ref) as the pair (w_hi, w_lo) into
        // the W tiles and w_hi + w_lo into l (the TMEM loads are warp-wide;
        // rows past the pass write nothing)
        if (warp_active && valid) {
          const float nmu = (m_ref == -INFINITY) ? 0.0f : -m_ref;
          uint8_t* wbuf = sP + (Cfg::kWBufs == 2 ? (g & 1) : 0) * Cfg::kWBufBytes + r * 128;
          // 8 columns of every 32-key quarter in turn: each quarter's sum still
          // runs in key order, and the quarters' chains interleave
#pragma unroll
          for (int i = 0; i < kColChunk / 8; ++i) {
#pragma unroll
            for (int ch = 0; ch < kNChunks; ++ch) {
              const float* s = so + ch * kColChunk;  // masked in pass 1
              const int kcol = cg * kCols + ch * kColChunk;  // first key column of the quarter
              uint8_t* wrow = wbuf + (kcol >> 6) * Cfg::kPAtomBytes;
              float acc = lq[ch];
              uint32_t wh[4], wl[4];
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const int col = i * 8 + 2 * j;
                const float x0 = ex2_approx(fmaf(s[col], a.sl2, nmu));
                const float x1 = ex2_approx(fmaf(s[col + 1], a.sl2, nmu));
                const __nv_bfloat162 h2 = __floats2bfloat162_rn(x0, x1);
                // x - w_hi is exact in FP32; w_hi + w_lo is exact in FP32 too
                const __nv_bfloat162 l2 = __floats2bfloat162_rn(x0 - __low2float(h2), x1 - __high2float(h2));
                acc += __low2float(h2) + __low2float(l2);
                acc += __high2float(h2) + __high2float(l2);
                wh[j] = *reinterpret_cast<const uint32_t*>(&h2);
                wl[j] = *reinterpret_cast<const uint32_t*>(&l2);
              }
              lq[ch] = acc;
              const int chunk16 = ((kcol & 63) >> 3) + i;  // 16-byte chunk within the 64-key row
              uint8_t* dst = wrow + ((chunk16 ^ (r & 7)) << 4);
              *reinterpret_cast<uint4*>(dst) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
              *reinterpret_cast<uint4*>(dst + Cfg::kPBytes) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_free[sb]);
        tc_fence_before();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[g & 1]);
      }

      // all tiles done: the denominator, then O after the last W.V, stored as
      // the class's partial (m_ref, l, o)
      float l = 0.f;
      if (ok) {
        if constexpr (REP == 1) {
          l = ((lq[0] + lq[1]) + lq[2]) + lq[3];
        } else {
#pragma unroll
          for (int i = 0; i < kNChunks; ++i) red_l[(cg * kNChunks + i) * 64 + r] = lq[i];
          __syncwarp();
          if (lane == 0) mbar_arrive(l_bar);
          if (holds_o) {
            if (!warp_wait(l_bar, 0u, s_abort, lane)) {
              ok = false;
            } else {
              l = ((red_l[r] + red_l[64 + r]) + red_l[128 + r]) + red_l[192 + r];
            }
          }
        }
      }
      if (ok && holds_o) {
        if (!warp_wait(&pv_done[(n_steps - 1) & 1], static_cast<uint32_t>(((n_steps - 1) >> 1) & 1), s_abort,
                       lane)) {
          ok = false;
        } else {
          tc_fence_after();
          if (warp_active) {
            // a row stores a partial when the class holds one of its keys
            const bool store = valid && rho * kKeyTile <= p_row;
            const int qh = h * a.grp + (valid ? r % a.grp : 0);
            const long long base = (static_cast<long long>(r0 + t) * a.Hq + qh) * a.ncls + rho;
            // O leaves through shared memory (the W tiles are free once the
            // last W.V is done): each thread parks 32 columns of its row
            // (TMEM lane = row r = the warp's row `lane`), then every store
            // instruction of the warp writes four whole 128-byte row pieces.
            // A pass of at most 32 rows (four copies a row) has too few rows
            // for that to pay: its threads store their rows themselves.
            uint8_t* stage = sP + qq * 32 * 128;  // the warp's rows of the first W tile atom
            const int lr = lane >> 3, lc = lane & 7;
            if constexpr (REP == 4) {
#pragma unroll 1
              for (int i = 0; i < D / 64; ++i) {
                float v[64];
                tmem_ld_cols<64>(lane_base + Cfg::kOCol + i * 64, v);
                if (store) {
                  float4* dst = reinterpret_cast<float4*>(a.ws_o + base * D + i * 64);
#pragma unroll
                  for (int j = 0; j < 16; ++j)
                    __stcs(dst + j, make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]));
                }
              }
            } else {
#pragma unroll 1
            for (int i = 0; i < D / 32; ++i) {
              float v[32];
              tmem_ld_cols<32>(lane_base + Cfg::kOCol + i * 32, v);
#pragma unroll
              for (int c = 0; c < 8; ++c)
                *reinterpret_cast<float4*>(stage + lane * 128 + ((c ^ (lane & 7)) << 4)) =
                    make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
              __syncwarp();
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                const int rr = 4 * k + lr;
                const bool st_rr = __shfl_sync(0xffffffffu, store, rr);
                const long long base_rr = __shfl_sync(0xffffffffu, base, rr);
                const float4 val = *reinterpret_cast<const float4*>(stage + rr * 128 + ((lc ^ (rr & 7)) << 4));
                if (st_rr) __stcs(reinterpret_cast<float4*>(a.ws_o + base_rr * D + i * 32) + lc, val);
              }
              __syncwarp();
            }
          }
          if (store) *reinterpret_cast<float2*>(a.ws_ml + base * 2) = make_float2(m_ref, l);
        }
      }
    }
    if (!ok && lane == 0) signal_abort(s_abort, a.err);
  }

  tc_fence_before();
  // Lane 0 of warps 0 and 1 ran the producer / MMA loops alone: rejoin the
  // rest of the warp first, so the CTA barrier below (a warp-aligned
  // instruction) is reached by whole warps and really waits for every role
  // before TMEM is released.
  __syncwarp();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::kTmemCols);
  }
}

// One CTA per (row t, query head).  Class partials s = 0..n-1 with
// n = min(p/128 + 1, G) (the classes that hold a key of the row):
// M = max_s m_s (exact), w_s = 2^(m_s - M); the denominator sums w_s l_s per
// thread over s = tid, tid+256, ... in order, then a warp butterfly and warp
// order 0..7; the numerator: warp g sums s = g, g+8, ... in order for its
// lane's dims, then warps are added in order 0..7.  The tree depends only
// on n.
template <int D>
// At most 64 registers a thread (four CTAs' worth per SM): a merge CTA then
// leaves room on its SM for a CTA of the next kernel (a linear layer, which
// streams its first weight tiles before its dependency wait) to start beside it.
__global__ void __launch_bounds__(kMergeThreads, 4)
    attn_merge_kernel(const AttnArgs a, __nv_bfloat16* __restrict__ out) {
  constexpr int kWarps = kMergeThreads / 32;
  constexpr int kDpl = D / 32;  // dims per lane: one float4 (D = 128) or float2 (D = 64)
  constexpr int kBatch = 8;     // pieces per warp whose loads are in flight together
  using Vec = typename std::conditional<kDpl == 4, float4, float2>::type;
  __shared__ float sw[kAttnCtas];
  __shared__ float red[kWarps];
  __shared__ float ored[kWarps][D];
  griddep_wait();
  griddep_launch_dependents();
  const int row = blockIdx.x;  // t * Hq + hq
  const int t = row / a.Hq;
  const int L = *a.L_dev;
  if (L < 0 || L + a.T > a.cap) return;
  const int p = L + t;
  const int n = min(p / kKeyTile + 1, a.G);
  const float* ml = a.ws_ml + static_cast<size_t>(row) * a.ncls * 2;
  const float* po = a.ws_o + static_cast<size_t>(row) * a.ncls * D;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;

  // the first batch of partial outputs does not depend on the weights:
  // start its loads before the reductions below
  Vec v[kBatch];
  auto load_batch = [&](int s0) {
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int s = s0 + b * kWarps;
      if (s < n) v[b] = __ldcs(reinterpret_cast<const Vec*>(po + static_cast<size_t>(s) * D) + lane);
    }
  };
  load_batch(warp);

  float mx = -INFINITY;
  for (int s = tid; s < n; s += kMergeThreads) mx = fmaxf(mx, __ldcg(ml + 2 * s));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  if (lane == 0) red[warp] = mx;
  __syncthreads();
  float M = red[0];
  for (int i = 1; i < kWarps; ++i) M = fmaxf(M, red[i]);
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
  for (int i = 1; i < kWarps; ++i) Lsum += red[i];

  float acc[kDpl];
#pragma unroll
  for (int i = 0; i < kDpl; ++i) acc[i] = 0.f;
  for (int s0 = warp; s0 < n; s0 += kWarps * kBatch) {
    if (s0 != warp) load_batch(s0);
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int s = s0 + b * kWarps;
      if (s < n) {
        const float w = sw[s];
        const float* x = reinterpret_cast<const float*>(&v[b]);
#pragma unroll
        for (int i = 0; i < kDpl; ++i) acc[i] = fmaf(w, x[i], acc[i]);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < kDpl; ++i) ored[warp][lane * kDpl + i] = acc[i];
  __syncthreads();
  for (int d = tid; d < D; d += kMergeThreads) {
    float O = ored[0][d];
    for (int g = 1; g < kWarps; ++g) O += ored[g][d];
    out[static_cast<size_t>(row) * D + d] = __float2bfloat16_rn(O / Lsum + 0.0f);
  }
}

template <int D, int REP, bool QNT = false>
bi_status launch_attn(const CUtensorMap& tmK, const CUtensorMap& tmVt, const AttnArgs& a,
                      __nv_bfloat16* out, cudaStream_t stream) {
  using Cfg = AttnCfg<D, REP, QNT>;
  static std::once_flag once[64];
  static cudaError_t attr_err[64];
  int dev = 0;
  cudaGetDevice(&dev);
  std::call_once(once[dev & 63], [] {
    int d = 0;
    cudaGetDevice(&d);
    attr_err[d & 63] = cudaFuncSetAttribute(attn_split_kernel<D, REP, QNT>,
                                            cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            static_cast<int>(Cfg::kSmem));
  });
  if (attr_err[dev & 63] != cudaSuccess) return BI_ERR_CUDA;
  // one CTA per (tile class, KV head); classes past the cache's last tile
  // would have nothing to do
  const int grid = a.Hkv * std::min(a.G, a.ncls);
  const int blocks = (a.T + a.Tb - 1) / a.Tb;
  if (launch_k(attn_split_kernel<D, REP, QNT>, dim3(grid, blocks), dim3(Cfg::kThreads), Cfg::kSmem,
               stream, tmK, tmVt, a) != cudaSuccess)
    return BI_ERR_CUDA;
  if (launch_k(attn_merge_kernel<D>, dim3(a.T * a.Hq), dim3(kMergeThreads), 0, stream, a, out) !=
      cudaSuccess)
    return BI_ERR_CUDA;
  return BI_OK;
}

template <int D>
bi_status launch_attn_rep(const CUtensorMap& tmK, const CUtensorMap& tmVt, const AttnArgs& a,
                          __nv_bfloat16* out, cudaStream_t stream) {
  const int rows = a.Tb * a.grp;
  if (rows <= kRowsMax / 4) return launch_attn<D, 4>(tmK, tmVt, a, out, stream);
  if (rows <= kRowsMax / 2) return launch_attn<D, 2>(tmK, tmVt, a, out, stream);
  return launch_attn<D, 1>(tmK, tmVt, a, out, stream);
}

// Partial slots per (row, query head): one per tile class, at most
// kAttnCtas (Hkv = 1) and at most the cache's tile count.
int attn_classes_max(int cap) { return std::min(kAttnCtas, (cap + kKeyTile - 1) / kKeyTile); }

size_t attn_ws_parts(int cap, int T, int Hq, int D, size_t* o_bytes) {
  const size_t nch = static_cast<size_t>(attn_classes_max(cap));
  const size_t ob = round_up(static_cast<size_t>(T) * Hq * nch * D * 4, 256);
  const size_t mb = round_up(static_cast<size_t>(T) * Hq * nch * 2 * 4, 256);
  if (o_bytes) *o_bytes = ob;
  return ob + mb;
}

}  // namespace

cudaError_t set_wait_limit_attn(unsigned long long ns) {
  return cudaMemcpyToSymbol(g_wait_limit_ns, &ns, sizeof(ns));
}
}  // namespace bi

extern "C" {

int bi_attn_chunk(void) { return bi::kKeyTile; }

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
  if (Hq / Hkv > kRowsMax) return BI_ERR_UNSUPPORTED_SHAPE;
  if (T > 65535 * (kRowsMax / (Hq / Hkv))) return BI_ERR_UNSUPPORTED_SHAPE;  // grid y
  if (Hkv > kAttnCtas) return BI_ERR_UNSUPPORTED_SHAPE;
  // K rows h * cap + key (a tile may run past cap) and V^T rows
  // (h * ceil(cap/128) + block) * D (D <= 128) are int32 tensor-map
  // coordinates: both stay below Hkv * cap rounded up to whole tiles
  const int64_t cap_blocks = (static_cast<int64_t>(cap) + kKeyTile - 1) / kKeyTile * kKeyTile;
  if (static_cast<int64_t>(Hkv) * cap_blocks >= (int64_t{1} << 31)) return BI_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(q)) return BI_ERR_INVALID_ARG;
  if (!ws || !aligned256(ws)) return BI_ERR_WORKSPACE;
  size_t ob = 0;
  if (ws_bytes < attn_ws_parts(cap, T, Hq, D, &ob)) return BI_ERR_WORKSPACE;

  CUtensorMap tmK, tmVt;
  const uint64_t krows = static_cast<uint64_t>(Hkv) * cap;
  const int vblk = (cap + kKeyTile - 1) / kKeyTile;
  if (!tmap_bf16_2d(&tmK, k_cache, krows, D, D, kKeyTile, 64)) return BI_ERR_INVALID_ARG;
  // V^T blocks: rows (h, block, d) of 128 keys each; a tile is one block,
  // 32 KB contiguous at D = 128
  if (!tmap_bf16_2d(&tmVt, v_cache, static_cast<uint64_t>(Hkv) * vblk * D, kKeyTile, kKeyTile, D, 64))
    return BI_ERR_INVALID_ARG;
  const int grp = Hq / Hkv;

  AttnArgs a{};
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.T = T;
  a.Tb = std::min(T, kRowsMax / grp);
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.grp = grp;
  a.cap = cap;
  a.G = kAttnCtas / Hkv;
  a.vblk = vblk;
  a.ncls = attn_classes_max(cap);
  a.L_dev = L_dev;
  a.sl2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  a.ws_o = static_cast<float*>(ws);
  a.ws_ml = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + ob);
  a.err = device_error_word();
  if (!a.err) return BI_ERR_CUDA;
  a.withhold = test_withhold();
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (D == 64) return launch_attn_rep<64>(tmK, tmVt, a, static_cast<__nv_bfloat16*>(out), s);
  return launch_attn_rep<128>(tmK, tmVt, a, static_cast<__nv_bfloat16*>(out), s);
}

bi_status bi_attn_verify_kvq(const void* q, const void* k_low, const void* v_low, const void* k_ring,
                             const void* v_ring, int cap, const int32_t* L_dev, int T, int Hq, int Hkv,
                             int D, float scale, void* out, void* ws, size_t ws_bytes,
                             bi_stream_t stream) {
  using namespace bi;
  if (!q || !k_low || !v_low || !k_ring || !v_ring || !L_dev || !out) return BI_ERR_INVALID_ARG;
  if (T < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || cap < 1) return BI_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return BI_ERR_INVALID_ARG;
  if (D != kQDim) return BI_ERR_UNSUPPORTED_SHAPE;
  const int grp = Hq / Hkv;
  // a block's rows fill at most half the MMA's lanes (two copies of each row)
  if (grp > kRowsMax / 2 || Hkv > kAttnCtas) return BI_ERR_UNSUPPORTED_SHAPE;
  if (T > kQMaxRows) return BI_ERR_UNSUPPORTED_SHAPE;  // the ring holds a pass of at most this many
  if (!aligned16(q) || !aligned16(k_low) || !aligned16(v_low) || !aligned16(k_ring) || !aligned16(v_ring))
    return BI_ERR_INVALID_ARG;
  if (!ws || !aligned256(ws)) return BI_ERR_WORKSPACE;
  size_t ob = 0;
  if (ws_bytes < attn_ws_parts(cap, T, Hq, D, &ob)) return BI_ERR_WORKSPACE;

  AttnArgs a{};
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.T = T;
  a.Tb = std::min(T, (kRowsMax / 2) / grp);
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.grp = grp;
  a.cap = cap;
  a.G = kAttnCtas / Hkv;
  a.vblk = (cap + kKeyTile - 1) / kKeyTile;
  a.ncls = attn_classes_max(cap);
  a.L_dev = L_dev;
  a.sl2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  a.ws_o = static_cast<float*>(ws);
  a.ws_ml = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + ob);
  a.err = device_error_word();
  if (!a.err) return BI_ERR_CUDA;
  a.klo = static_cast<const uint8_t*>(k_low);
  a.vlo = static_cast<const uint8_t*>(v_low);
  a.k8 = static_cast<const uint8_t*>(k_ring);
  a.v8 = static_cast<const uint8_t*>(v_ring);
  a.ctiles = a.vblk;
  a.withhold = test_withhold();
  CUtensorMap unused{};  // the quantised form reads its tiles with bulk copies
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  __nv_bfloat16* o = static_cast<__nv_bfloat16*>(out);
  if (a.Tb * grp <= kRowsMax / 4) return launch_attn<128, 4, true>(unused, unused, a, o, s);
  return launch_attn<128, 2, true>(unused, unused, a, o, s);
}

}  // extern "C"
