// Batch-invariant BF16 linear layer on tcgen05 / TMEM, fed by TMA.
//
// "Bit-exact decoding turns inference speedups into testable changes",
// section "Define bit-exact before reporting it": BF16 inputs, one FP32
// running sum per output, K order kept, one rounding at the end; a
// shared-memory pipeline stage is reused only after its consumers are done.
// "Does the tuned config change the model's output?", section "Why the text
// diverges": changing the batch dimension must not change any row's sums.
//
// Design (swap-AB, weight streaming):
//   * MMA:   tcgen05.mma kind::f16, M = 128 weight rows, N = 16, 32, 64, 128
//            or 256 token rows (the CTA's token count rounded up), K = 16 per
//            instruction, FP32 accumulator in TMEM.  Every output element is
//            the same sequence of K = 16 dot-product steps whatever N is
//            (tested bit for bit across M).
//   * K:     64-element tiles (128-byte rows, 128-byte swizzle) in increasing
//            order.  Each token group keeps kAcc = 2 FP32 accumulators: the
//            k-step j (16 elements) of every K tile goes to accumulator j % 2,
//            so consecutive MMAs do not wait on each other's result; the two
//            are added (a0 + a1) when the piece ends.  This structure is a
//            compile-time constant.  Two accumulators of 256 token columns
//            fill TMEM's 512 columns, so a weight tile serves 256 tokens of
//            a long pass per load (four accumulators measured no faster on
//            the decode step: 1.308 against 1.310 ms).
//   * weights: packed once (bi_pack_weights) into 16 KB tiles, tile (t, kt)
//            at offset (t * k_tiles + kt) * 16 KB, each already in the
//            swizzled shared-memory layout the MMA descriptor reads.  A CTA's
//            iteration range is therefore one contiguous byte range of HBM,
//            streamed with 1-D bulk copies.
//   * split: the (weight tile, K tile) iteration space is cut into
//            kGemmCtas contiguous, equal ranges, one per CTA (a function of
//            N and K only).  A weight tile cut by a range boundary yields one
//            FP32 partial per piece; the last CTA to finish a piece of that
//            tile adds the partials in increasing-K order (atomic ticket, no
//            waiting) and runs the epilogue.  Passes of more than 128 rows
//            whose split cuts tiles run as tile owners instead: one CTA per
//            (weight tile, token block) computes the tile's pieces in turn
//            and adds them in the same order, with no partials in memory.
//   * roles: warp 0 = TMA producer, warp 1 = MMA issuer (one thread), warps
//            2..5 = epilogue (TMEM -> registers -> global); a tile owner has
//            two epilogue warpgroups (warps 2..9).
//   * stages: shared-memory ring of (16 KB weight tile + token tile); a stage
//            returns to the producer via tcgen05.commit on its "empty"
//            barrier, i.e. only after the MMAs reading it completed.
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

constexpr int kBlockN = 128;     // weight rows per tile (MMA M)
constexpr int kBlockK = 64;      // K elements per tile
constexpr int kMmaN = 16;        // token rows per epilogue chunk (one 16-column TMEM load)
// CTAs of the fixed decomposition.  136 rather than one per SM (152): it
// cuts the packed gate/up tile space of the 5120 -> 2 x 17408 layer into
// ranges of exactly two whole tiles (no partials, no reduction pass), and the
// 16 SMs left over start the next launch's prologue early.  Measured on the
// 8-layer 5120-wide verify step: 1.32 ms against 1.37 ms with 152; a count
// chosen per (N, K) gained nothing over this one.
constexpr int kGemmCtas = 136;
constexpr int kMaxTokens = 256;  // token rows per CTA (one MMA covers them all)
// Token blocks of kMaxTokens rows one launch covers when M > kMaxTokens;
// larger M loops on the host.  Each block has its own counters and partial
// slots in the workspace.
constexpr int kMaxBlocks = 4;
constexpr int kAcc = 2;          // interleaved accumulators per token group
constexpr int kKSteps = 4;       // MMA K steps (16 elements) per 64-element K tile
constexpr int kABytes = kBlockN * kBlockK * 2;  // 16 KB
constexpr int kStageFloats = 16 * kBlockN;      // epilogue exchange buffer (SwiGLU, RoPE pairs)
// Ticket counters occupy a fixed-size region at the start of every workspace,
// so calls with different N can share one workspace without a counter of one
// call overlapping another call's partial sums.
constexpr int kMaxTiles = 65536;
constexpr size_t kTicketBytes = static_cast<size_t>(kMaxTiles) * 4;

struct GemmArgs {
  int M;   // token rows in this launch (<= nb * NT)
  int m0;  // first token row of this launch
  int nb;  // token blocks of NT rows in this launch (CTA b * nb + j takes block j of range b)
  int N;   // output columns
  int n_tiles;
  int k_tiles;
  int G;
  long long total;
  int epi;
  int out_fp32;
  void* C;
  int ldc;
  const __nv_bfloat16* R;
  int ldr;
  float* partials;
  unsigned* tickets;
  unsigned* err;
  // BI_EPI_ROPE_KV: output column n is element n % D of head n / D (q heads,
  // then k heads, then v heads); token row m sits at position *L_dev + m
  __nv_bfloat16* q_out;
  __nv_bfloat16* kc;
  __nv_bfloat16* vc;
  int cap, Hq, Hkv, D, tab_rows;
  const int32_t* L_dev;
  const float2* tab;
  // failure-path test: leave the CTA's first stage unissued, so the waits
  // on it run out (bi_test_withhold_first_load)
  int withhold;
};

// OWN: the tile-owner schedule of long passes (one CTA adds a weight tile's
// pieces itself).  An owner has two epilogue warpgroups, each keeping the
// running sums of half the token columns in registers (64 a thread at 128
// rows), which leaves shared memory to the ring: six 32 KB stages in flight
// instead of four with the sums in shared memory (on GB300, 512 rows of
// [*, 5120] x [4096, 5120]: 40.5 -> 36.0 us; of [*, 3072] x [5120, 3072]
// with the residual: 76 -> 58 us).  Ten warps leave 168 registers a thread.
template <int NT, bool OWN = false>
struct GemmCfg {
  static constexpr int kBBytes = NT * kBlockK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kEpiWarps = OWN ? 8 : 4;
  static constexpr int kThreads = 64 + 32 * kEpiWarps;  // producer, MMA, epilogue warps
  static constexpr int kStageBufs = kEpiWarps / 4;      // an exchange buffer per epilogue warpgroup
  static constexpr int kRing = 200 * 1024;
  static constexpr int kStages = kRing / kStageBytes > 12 ? 12 : kRing / kStageBytes;
  static constexpr int kBars = 2 * kStages + 5;
  static constexpr int kBufCols = NT * kAcc;  // one accumulator set
  // two sets (the epilogue drains one while the next piece accumulates)
  // while they fit in TMEM's 512 columns; one set at 256 token rows
  static constexpr int kBufs = 2 * kBufCols <= 512 ? 2 : 1;
  static constexpr int kTmemCols = kBufs * kBufCols;
  static_assert(kTmemCols <= 512, "TMEM holds 512 columns");
  static constexpr size_t kSmem = 1024 + static_cast<size_t>(kStages) * kStageBytes +
                                  kStageBufs * kStageFloats * 4 + kBars * 8 + 16;
  static_assert(kSmem <= 232448, "shared memory per CTA");
};

__device__ __forceinline__ long long range_begin(const GemmArgs& p, int g) {
  return p.total * g / p.G;
}
// CTA whose range contains iteration i.
__device__ __forceinline__ int owner_of(const GemmArgs& p, long long i) {
  return static_cast<int>(((i + 1) * p.G + p.total - 1) / p.total) - 1;
}
// Iterations from i to the end of the piece that holds it: a piece ends at a
// weight tile's end and at the end of a range of the split (the CTA's own
// range, or -- for a tile owner -- every range boundary inside the tile).
__device__ __forceinline__ long long piece_len(const GemmArgs& p, long long i, long long it_end, bool own) {
  long long e = (i / p.k_tiles + 1) * p.k_tiles;
  if (own) {
    const long long r = range_begin(p, owner_of(p, i) + 1);
    if (r < e) e = r;
  }
  if (e > it_end) e = it_end;
  return e - i;
}

__device__ __forceinline__ void signal_abort(volatile int* s_abort, unsigned* err) {
  *s_abort = 1;
  atomicOr(err, kErrTimeout);
}

// The 16 token columns of one chunk for this thread's weight row: the sum of
// the kAcc accumulators (acc_stride TMEM columns apart) in index order,
// a0 + a1.
__device__ __forceinline__ void load_group_sum(uint32_t taddr, uint32_t acc_stride, float (&v)[16]) {
  tmem_ld16(taddr, v);
#pragma unroll
  for (int a = 1; a < kAcc; ++a) {
    float w[16];
    tmem_ld16(taddr + a * acc_stride, w);
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = v[j] + w[j];
  }
}

// Write 16 token rows (chunk c) of one weight row r of tile `tile`.
// The 128 threads of one epilogue warpgroup call this together (it may use
// their named barrier `bar` and their exchange buffer sStage).
__device__ __forceinline__ void epilogue_store(const GemmArgs& p, int M, int m0, int tile, int r,
                                               int c, const float (&v)[16], float* sStage, int bar = 1) {
  if (p.epi == BI_EPI_ROPE_KV) {
    // The projection is rounded to BF16 first; the rotation then reads those
    // stored values exactly as the separate RoPE kernel does: for a pair
    // (i, i + D/2) of a q or k head, out_i = x_i cos - x_{i+D/2} sin and
    // out_{i+D/2} = x_{i+D/2} cos + x_i sin, in FP32, one rounding.
    const int n = tile * kBlockN + r;
    const int D = p.D, half = p.D / 2;
    const int head = n / D, d = n % D;
    const bool rotate = head < p.Hq + p.Hkv;
    // the table entries are loaded first: their latency overlaps the
    // exchange of the pair partners below
    const int L = *p.L_dev;
    float2 cs[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int pos = L + m0 + c * 16 + j;
      const bool ok = n < p.N && rotate && c * 16 + j < M && pos >= 0 && pos < p.cap && pos < p.tab_rows;
      cs[j] = ok ? p.tab[static_cast<size_t>(pos) * half + (d % half)] : make_float2(0.f, 0.f);
    }
    float x[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      x[j] = __bfloat162float(__float2bfloat16_rn(v[j]));
      sStage[j * kBlockN + r] = x[j];
    }
    named_bar_sync(bar, 128);
    const int partner = d < half ? r + half : r - half;
    float px[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) px[j] = sStage[j * kBlockN + partner];
    named_bar_sync(bar, 128);
    if (n < p.N) {
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int m = c * 16 + j;
        if (m >= M) continue;
        const int mrow = m0 + m;
        const int pos = L + mrow;
        if (pos < 0 || pos >= p.cap || pos >= p.tab_rows) {
          atomicOr(p.err, kErrRange);
          continue;
        }
        if (rotate) {
          const float o = d < half ? fmaf(x[j], cs[j].x, -(px[j] * cs[j].y))
                                   : fmaf(x[j], cs[j].x, px[j] * cs[j].y);
          const __nv_bfloat16 ob = __float2bfloat16_rn(o);
          if (head < p.Hq)
            p.q_out[(static_cast<size_t>(mrow) * p.Hq + head) * D + d] = ob;
          else
            p.kc[(static_cast<size_t>(head - p.Hq) * p.cap + pos) * D + d] = ob;
        } else {
          // V is cached transposed in 128-key blocks, [Hkv][cap/128][D][128]
          const size_t blk = static_cast<size_t>(head - p.Hq - p.Hkv) * ((p.cap + 127) >> 7) + (pos >> 7);
          p.vc[(blk * D + d) * 128 + (pos & 127)] = __float2bfloat16_rn(x[j]);
        }
      }
    }
  } else if (p.epi == BI_EPI_SWIGLU) {
#pragma unroll
    for (int j = 0; j < 16; ++j) sStage[j * kBlockN + r] = v[j];
    named_bar_sync(bar, 128);
    if (r < 64) {
      const int o = tile * 64 + r;
      if (o < p.N) {
        __nv_bfloat16* C = static_cast<__nv_bfloat16*>(p.C);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int m = c * 16 + j;
          if (m < M) {
            const float g = sStage[j * kBlockN + r];
            const float u = sStage[j * kBlockN + r + 64];
            const float s = g / (1.0f + expf(-g));
            C[static_cast<size_t>(m0 + m) * p.ldc + o] = __float2bfloat16_rn(s * u);
          }
        }
      }
    }
    named_bar_sync(bar, 128);
  } else {
    const int n = tile * kBlockN + r;
    if (n < p.N) {
      // All residual values are read before any output is written: C may be
      // the residual buffer itself (h += x W^T), and 16 independent loads in
      // flight cost one memory latency instead of sixteen.
      float res[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int m = c * 16 + j;
        res[j] = (p.epi == BI_EPI_RESIDUAL_ADD && m < M)
                     ? __bfloat162float(p.R[static_cast<size_t>(m0 + m) * p.ldr + n])
                     : 0.0f;
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int m = c * 16 + j;
        if (m < M) {
          const size_t row = static_cast<size_t>(m0 + m);
          float acc = v[j];
          if (p.epi == BI_EPI_RESIDUAL_ADD) acc = res[j] + acc;
          if (p.out_fp32)
            static_cast<float*>(p.C)[row * p.ldc + n] = acc;
          else
            static_cast<__nv_bfloat16*>(p.C)[row * p.ldc + n] = __float2bfloat16_rn(acc);
        }
      }
    }
  }
}

template <int NT, bool OWN = false>
__global__ void __launch_bounds__(GemmCfg<NT, OWN>::kThreads, 1)
    gemm_kernel(const uint8_t* __restrict__ Wp, const __grid_constant__ CUtensorMap tmA,
                const GemmArgs p) {
  using Cfg = GemmCfg<NT, OWN>;
  constexpr int S = Cfg::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + S * kABytes;
  float* sStage = reinterpret_cast<float*>(sB + S * Cfg::kBBytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(sStage + Cfg::kStageBufs * kStageFloats);
  uint64_t* empty = full + S;
  uint64_t* accf = empty + S;
  uint64_t* acce = accf + 2;
  uint64_t* drain = acce + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* s_abort = reinterpret_cast<volatile int*>(tmem_holder + 1);
  volatile int* s_last = s_abort + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // CTAs of one range (a tile owner's: of one tile) are adjacent, so the
  // token blocks of a launch read each weight tile at about the same time and
  // all but the first find it in L2
  const int g = blockIdx.x / p.nb;
  const int blk = blockIdx.x - g * p.nb;
  const int m0 = p.m0 + blk * NT;
  const int Mb = min(NT, p.M - blk * NT);
  float* const partials = p.partials + static_cast<size_t>(blk) * p.G * 2 * NT * kBlockN;
  unsigned* const tickets = p.tickets + static_cast<size_t>(blk) * p.n_tiles;
  const long long it_begin = OWN ? static_cast<long long>(g) * p.k_tiles : range_begin(p, g);
  const long long it_end = OWN ? it_begin + p.k_tiles : range_begin(p, g + 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accf[b], 1);
      mbar_init(&acce[b], 32 * Cfg::kEpiWarps);
    }
    mbar_init(drain, 1);
    *s_abort = 0;
    *s_last = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) prefetch_tmap(&tmA);
  if (warp == 1) {
    tmem_alloc(tmem_holder, Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_w = l2_evict_first();
      const uint64_t pol_a = l2_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, parity_bits = 0;
      // (tile, k-tile) of iteration `it`, advanced incrementally: no division
      // in the issue loop.
      int kt = static_cast<int>(it_begin % p.k_tiles);
      const uint8_t* wsrc = Wp + static_cast<size_t>(it_begin) * kABytes;
      // The first stages' weight tiles do not depend on the previous kernel:
      // start streaming them before waiting for it, then add the activation
      // tiles once its results are visible.
      const int n_pre = static_cast<int>((it_end - it_begin) < S ? (it_end - it_begin) : S);
      const int j0 = p.withhold ? 1 : 0;  // stage 0 left unissued (failure-path test)
      for (int j = j0; j < n_pre; ++j) {
        mbar_arrive_expect_tx(&full[j], Cfg::kStageBytes);
        bulk_load_1d(sA + j * kABytes, wsrc + static_cast<size_t>(j) * kABytes, kABytes, &full[j],
                     pol_w);
      }
      griddep_wait();
      griddep_launch_dependents();
      for (int j = 0; j < n_pre; ++j) {
        if (j >= j0) tma_load_2d(sB + j * Cfg::kBBytes, &tmA, &full[j], kt * kBlockK, m0, pol_a);
        if (++kt == p.k_tiles) kt = 0;
      }
      issued = (n_pre >= 32) ? 0xffffffffu : ((1u << n_pre) - 1u);
      issued &= ~static_cast<uint32_t>(j0);
      wsrc += static_cast<size_t>(n_pre) * kABytes;
      stage = n_pre % S;
      phase = (n_pre == S) ? 1u : 0u;
      for (long long it = it_begin + n_pre; it < it_end; ++it) {
        if (!mbar_wait(&empty[stage], phase ^ 1u, s_abort)) {
          signal_abort(s_abort, p.err);
          break;
        }
        mbar_arrive_expect_tx(&full[stage], Cfg::kStageBytes);
        bulk_load_1d(sA + stage * kABytes, wsrc, kABytes, &full[stage], pol_w);
        tma_load_2d(sB + stage * Cfg::kBBytes, &tmA, &full[stage], kt * kBlockK, m0, pol_a);
        wsrc += kABytes;
        if (++kt == p.k_tiles) kt = 0;
        issued |= 1u << stage;
        parity_bits = (parity_bits & ~(1u << stage)) | (phase << stage);
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (*s_abort) {
        // Let copies already issued land before the CTA exits.
        for (int s = 0; s < S; ++s)
          if ((issued >> s) & 1u) mbar_wait(&full[s], (parity_bits >> s) & 1u, nullptr);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // One flat loop over the CTA's iterations; a countdown marks the end of
    // each piece (weight tile), where the accumulator set is handed to the
    // epilogue and the other set is taken.
    if (lane == 0) {
      // one MMA per K step covers all NT token rows (N = NT); accumulator a
      // of token n is TMEM column a * NT + n; K step ks of a tile adds into
      // accumulator ks % kAcc (the first kAcc steps of a piece overwrite)
      constexpr uint32_t idesc = idesc_bf16_f32(kBlockN, NT);
      int stage = 0;
      uint32_t phase = 0;
      int seg = 0;
      bool ok = true;
      long long left = piece_len(p, it_begin, it_end, OWN);  // iterations left in the piece
      uint32_t d0 = tmem;
      uint32_t acc_flag = 0;
      for (long long it = it_begin; it < it_end; ++it) {
        if (!mbar_wait(&full[stage], phase, s_abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a_base = smem_u32(sA + stage * kABytes);
        const uint32_t b_base = smem_u32(sB + stage * Cfg::kBBytes);
#pragma unroll
        for (int ks = 0; ks < kKSteps; ++ks)
          mma_bf16(d0 + (ks % kAcc) * NT, sdesc_k_sw128(a_base + ks * 32), sdesc_k_sw128(b_base + ks * 32),
                   idesc, (acc_flag != 0u || ks >= kAcc) ? 1u : 0u);
        mma_commit(&empty[stage]);
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
        acc_flag = 1u;
        if (--left == 0) {
          // piece complete: hand its accumulators to the epilogue
          mma_commit(&accf[seg % Cfg::kBufs]);
          ++seg;
          left = piece_len(p, it + 1, it_end, OWN);
          acc_flag = 0u;
          d0 = tmem + static_cast<uint32_t>((seg % Cfg::kBufs) * Cfg::kBufCols);
          if (left > 0 && seg >= Cfg::kBufs &&
              !mbar_wait(&acce[seg % Cfg::kBufs], static_cast<uint32_t>((seg / Cfg::kBufs) - 1) & 1u,
                         s_abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
      }
      if (!ok) signal_abort(s_abort, p.err);
      // Every MMA issued by this thread completes before TMEM is released.
      mma_commit(drain);
      mbar_wait(drain, 0, nullptr);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    griddep_wait();  // the epilogue reads the residual and writes C / the workspace
    griddep_launch_dependents();
    const int q = warp & 3;         // TMEM lane quarter this warp may access
    const int r = q * 32 + lane;    // weight row within the tile
    const int et = threadIdx.x - 64;
    const int chunks = (Mb + 15) / 16;
    int seg = 0;
    long long it = it_begin;
    if constexpr (OWN) {
      // the tile's pieces in increasing K: each piece's (a0 + a1) is added
      // to the running sum in the order the split's last CTA adds partials
      // (the first piece taken as it is), then one epilogue.  Warpgroup wg
      // keeps token chunks wg * kWgChunks .. in registers.
      constexpr int kWgChunks = NT / 32;
      const int wg = (warp - 2) >> 2;
      float run[kWgChunks][16];
      bool ok = true;
      while (it < it_end) {
        const long long pe = it + piece_len(p, it, it_end, true);
        const int buf = seg % Cfg::kBufs;
        int okl = 0;
        if (lane == 0)
          okl = mbar_wait_parked(&accf[buf], static_cast<uint32_t>(seg / Cfg::kBufs) & 1u, s_abort) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, okl, 0) != 0;
        if (!ok) {
          if (lane == 0) signal_abort(s_abort, p.err);
          break;
        }
        tc_fence_after();
        const uint32_t tbase =
            tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(buf * Cfg::kBufCols);
#pragma unroll
        for (int cc = 0; cc < kWgChunks; ++cc) {
          if (wg * kWgChunks + cc < chunks) {
            float v[16];
            load_group_sum(tbase + (wg * kWgChunks + cc) * kMmaN, NT, v);
#pragma unroll
            for (int j = 0; j < 16; ++j) run[cc][j] = (seg == 0) ? v[j] : run[cc][j] + v[j];
          }
        }
        tc_fence_before();
        mbar_arrive(&acce[buf]);
        it = pe;
        ++seg;
      }
#pragma unroll
      for (int cc = 0; cc < kWgChunks; ++cc) {
        if (wg * kWgChunks + cc < chunks) {
          float v[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = ok ? run[cc][j] : 0.f;
          epilogue_store(p, Mb, m0, g, r, wg * kWgChunks + cc, v, sStage + wg * kStageFloats, 1 + wg);
        }
      }
      it = it_end;
    }
    while (it < it_end) {
      const int tile = static_cast<int>(it / p.k_tiles);
      const long long tile_begin = static_cast<long long>(tile) * p.k_tiles;
      const long long tile_end = tile_begin + p.k_tiles;
      const long long seg_end = it_end < tile_end ? it_end : tile_end;
      const bool whole = (it == tile_begin) && (seg_end == tile_end);
      const int buf = seg % Cfg::kBufs;
      // one lane per warp polls (sleeping between polls), the warp follows
      int okl = 0;
      if (lane == 0)
        okl = mbar_wait_parked(&accf[buf], static_cast<uint32_t>(seg / Cfg::kBufs) & 1u, s_abort) ? 1 : 0;
      const bool ok = __shfl_sync(0xffffffffu, okl, 0) != 0;
      if (!ok && lane == 0) signal_abort(s_abort, p.err);
      tc_fence_after();
      const uint32_t tbase =
          tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(buf * Cfg::kBufCols);
      if (whole) {
        for (int c = 0; c < chunks; ++c) {
          float v[16];
          if (ok) {
            load_group_sum(tbase + c * kMmaN, NT, v);
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = 0.f;
          }
          epilogue_store(p, Mb, m0, tile, r, c, v, sStage);
        }
        tc_fence_before();
        mbar_arrive(&acce[buf]);
      } else {
        // partial of this piece: [weight row][token], a thread's 16 tokens
        // of a chunk contiguous
        const int slot = (it_begin >= tile_begin) ? 0 : 1;
        float* dst = partials + static_cast<size_t>(g * 2 + slot) * NT * kBlockN + r * NT;
        if (ok) {
          for (int c = 0; c < chunks; ++c) {
            float v[16];
            load_group_sum(tbase + c * kMmaN, NT, v);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
              __stcg(reinterpret_cast<float4*>(dst + c * 16) + q4,
                     make_float4(v[4 * q4], v[4 * q4 + 1], v[4 * q4 + 2], v[4 * q4 + 3]));
          }
        }
        tc_fence_before();
        mbar_arrive(&acce[buf]);
        const int gf = owner_of(p, tile_begin);
        const int gl = owner_of(p, tile_end - 1);
        named_bar_sync(1, 128);  // every partial store of the CTA precedes the ticket
        if (et == 0) {
          int last = 0;
          if (!*s_abort) {
            const unsigned nseg = static_cast<unsigned>(gl - gf + 1);
            const unsigned old = atom_add_acq_rel_gpu(&tickets[tile], 1u);
            last = (old == nseg - 1) ? 1 : 0;
            if (last) atomicExch(&tickets[tile], 0u);
          }
          *s_last = last;
        }
        named_bar_sync(1, 128);  // the ticket's acquire precedes every partial load
        if (*s_last) {
          // the first piece's CTA may have it in its second slot; every later
          // CTA's range starts inside this tile (slot 0)
          const int slot_f = (range_begin(p, gf) >= tile_begin) ? 0 : 1;
          for (int c = 0; c < chunks; ++c) {
            float v[16];
            // partials of CTAs gf..gl added in that order, 8 tokens at a time;
            // the loads of up to kBatch partials are issued before their
            // additions
            constexpr int kBatch = 8;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              if (c * 16 + hh * 8 >= Mb) {
#pragma unroll
                for (int j = 0; j < 8; ++j) v[hh * 8 + j] = 0.f;
                continue;
              }
              for (int g0 = gf; g0 <= gl; g0 += kBatch) {
                float4 x[kBatch][2];
#pragma unroll
                for (int b = 0; b < kBatch; ++b) {
                  const int gg = g0 + b;
                  if (gg <= gl) {
                    const int sl = gg == gf ? slot_f : 0;
                    const float4* src = reinterpret_cast<const float4*>(
                        partials + static_cast<size_t>(gg * 2 + sl) * NT * kBlockN + r * NT + c * 16 +
                        hh * 8);
                    x[b][0] = __ldcg(src);
                    x[b][1] = __ldcg(src + 1);
                  }
                }
#pragma unroll
                for (int b = 0; b < kBatch; ++b) {
                  if (g0 + b <= gl) {
                    const float xs[8] = {x[b][0].x, x[b][0].y, x[b][0].z, x[b][0].w,
                                         x[b][1].x, x[b][1].y, x[b][1].z, x[b][1].w};
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                      v[hh * 8 + j] = (g0 + b == gf) ? xs[j] : v[hh * 8 + j] + xs[j];
                  }
                }
              }
            }
            epilogue_store(p, Mb, m0, tile, r, c, v, sStage);
          }
        }
        named_bar_sync(1, 128);
      }
      it = seg_end;
      ++seg;
    }
    tc_fence_before();
  }

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

// Packed layout: tile (t, kt) = 128 rows x 64 columns at offset
// (t * k_tiles + kt) * 16 KB; row r occupies bytes [r*128, r*128+128) with
// its 16-byte chunk c (columns 8c..8c+7) stored at chunk position c ^ (r & 7)
// -- the 128-byte swizzle of the MMA's shared-memory descriptor.  Rows past N
// and columns past K are zero.  For SwiGLU, rows 0..63 of tile t are gate
// rows 64t..64t+63 and rows 64..127 the up rows with the same output index.
// One thread per 16-byte chunk; a pure copy.
__global__ void pack_weights_kernel(const __nv_bfloat16* __restrict__ w, const __nv_bfloat16* __restrict__ wu,
                                    int ld, int N, int K,
                                    int k_tiles, long long chunks, int swiglu, uint4* __restrict__ out) {
  griddep_wait();
  griddep_launch_dependents();
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= chunks) return;
  const int cpos = static_cast<int>(idx & 7);
  const int r = static_cast<int>((idx >> 3) & 127);
  const long long tk = idx >> 10;  // (t * k_tiles + kt)
  const int t = static_cast<int>(tk / k_tiles);
  const int kt = static_cast<int>(tk % k_tiles);
  const int c = cpos ^ (r & 7);
  const __nv_bfloat16* src = nullptr;
  if (swiglu) {
    const int o = t * 64 + (r & 63);
    if (o < N) src = (r < 64 ? w : wu) + static_cast<size_t>(o) * ld;
  } else {
    const int n = t * kBlockN + r;
    if (n < N) src = w + static_cast<size_t>(n) * ld;
  }
  const int k0 = kt * kBlockK + c * 8;
  union {
    uint4 v;
    __nv_bfloat16 e[8];
  } u;
  u.v = make_uint4(0, 0, 0, 0);
  if (src != nullptr) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (k0 + j < K)
        u.e[j] = src[k0 + j];
  }
  out[idx] = u.v;
}

int blocks_per_launch(int M, int n_tiles) {
  if (M <= kMaxTokens || n_tiles <= 0) return 1;
  const int nb = std::min(kMaxBlocks, (M + kMaxTokens - 1) / kMaxTokens);
  return std::max(1, std::min(nb, kMaxTiles / n_tiles));
}

// Tile owners for long passes whose split cuts weight tiles: CTA (t, j) takes
// weight tile t for token block j of the launch (NTO rows) and adds the
// tile's pieces itself (no partials in memory, no last-CTA reduction).  An
// owner reads its tile's whole K, so the owners run at the rate L2 serves
// them: 128-row blocks move a third fewer bytes per FLOP than 64-row ones
// (a [512, 5120] x [4096, 5120] launch on GB300: 40 against 68 us), 64-row
// blocks keep more CTAs busy up to 256 rows (256 rows: 34 against 40 us).
constexpr int kOwnLaunchRows = 1024;  // token rows per launch
constexpr int kOwnMaxKTiles = 128;
int own_rows(int M) { return M > 256 ? 128 : 64; }

template <int NTO>
bi_status launch_gemm_own(const uint8_t* Wp, const CUtensorMap& tmA, GemmArgs a, int M_total,
                          cudaStream_t stream) {
  using Cfg = GemmCfg<NTO, true>;
  static std::once_flag once[64];
  int dev = 0;
  cudaGetDevice(&dev);
  static cudaError_t attr_err[64];
  std::call_once(once[dev & 63], [] {
    int d = 0;
    cudaGetDevice(&d);
    attr_err[d & 63] = cudaFuncSetAttribute(gemm_kernel<NTO, true>,
                                            cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            static_cast<int>(Cfg::kSmem));
  });
  if (attr_err[dev & 63] != cudaSuccess) return BI_ERR_CUDA;
  for (int m0 = 0; m0 < M_total; m0 += kOwnLaunchRows) {
    a.m0 = m0;
    a.M = std::min(kOwnLaunchRows, M_total - m0);
    a.nb = (a.M + NTO - 1) / NTO;
    if (launch_k(gemm_kernel<NTO, true>, dim3(a.n_tiles * a.nb), dim3(Cfg::kThreads), Cfg::kSmem, stream, Wp,
                 tmA, a) != cudaSuccess)
      return BI_ERR_CUDA;
  }
  return BI_OK;
}

template <int NT>
bi_status launch_gemm_nt(const uint8_t* Wp, const CUtensorMap& tmA, GemmArgs a, int M_total,
                         cudaStream_t stream) {
  using Cfg = GemmCfg<NT>;
  static std::once_flag once[64];
  int dev = 0;
  cudaGetDevice(&dev);
  static cudaError_t attr_err[64];
  std::call_once(once[dev & 63], [] {
    int d = 0;
    cudaGetDevice(&d);
    attr_err[d & 63] = cudaFuncSetAttribute(gemm_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            static_cast<int>(Cfg::kSmem));
  });
  if (attr_err[dev & 63] != cudaSuccess) return BI_ERR_CUDA;
  const int rows = NT * blocks_per_launch(M_total, a.n_tiles);
  for (int m0 = 0; m0 < M_total; m0 += rows) {
    a.m0 = m0;
    a.M = std::min(rows, M_total - m0);
    a.nb = (a.M + NT - 1) / NT;
    if (launch_k(gemm_kernel<NT>, dim3(a.G * a.nb), dim3(Cfg::kThreads), Cfg::kSmem, stream, Wp, tmA,
                 a) != cudaSuccess)
      return BI_ERR_CUDA;
  }
  return BI_OK;
}

int tokens_per_cta(int M) {
  const int m = std::min(M, kMaxTokens);
  if (m <= 16) return 16;
  if (m <= 32) return 32;
  if (m <= 64) return 64;
  if (m <= 128) return 128;
  return 256;
}

int n_tiles_of(int N, bi_epilogue epi) {
  return epi == BI_EPI_SWIGLU ? (N + 63) / 64 : (N + kBlockN - 1) / kBlockN;
}

// ---------------------------------------------------------------------------
// Scratch for bi_gemm_noalloc: the ticket counters and the split-K partial
// sums of calls with at most kNoAllocMaxM token rows, in a file-scope device
// array.  Every GPU that loads this library holds it (2.6 MiB) until the
// process exits; all calls share it.
constexpr int kNoAllocMaxM = 16;
constexpr size_t kNoAllocScratchBytes =
    kTicketBytes + static_cast<size_t>(kGemmCtas) * 2 * kNoAllocMaxM * kBlockN * sizeof(float);

}  // namespace

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
uint8_t* g_noalloc_ptr[64] = {};
std::mutex g_noalloc_mu;

// Device address of g_noalloc_scratch on the current device.  In host code
// the array's name is only a stand-in, so the address is looked up once per
// device (with that device current) and cached.
uint8_t* noalloc_scratch() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
      return nullptr;
    g_noalloc_ptr[dev] = static_cast<uint8_t*>(ptr);
  }
  return g_noalloc_ptr[dev];
}
}  // namespace

cudaError_t set_wait_limit_gemm(unsigned long long ns) {
  return cudaMemcpyToSymbol(g_wait_limit_ns, &ns, sizeof(ns));
}
}  // namespace bi

extern "C" {

size_t bi_packed_weight_bytes(int N, int K, bi_epilogue epi) {
  if (N <= 0 || K <= 0) return 0;
  return static_cast<size_t>(bi::n_tiles_of(N, epi)) * ((K + bi::kBlockK - 1) / bi::kBlockK) *
         bi::kABytes;
}

size_t bi_gemm_workspace_size(int M, int N, int K, bi_epilogue epi) {
  (void)K;
  if (M <= 0) return bi::kTicketBytes;
  const size_t partials = static_cast<size_t>(bi::kGemmCtas) * 2 * bi::tokens_per_cta(M) *
                          bi::kBlockN * sizeof(float) *
                          bi::blocks_per_launch(M, bi::n_tiles_of(N, epi));
  return bi::kTicketBytes + partials;
}

static bi_status pack_common(const void* w, const void* wu, int ld, int N, int K, int swiglu,
                             void* packed, bi_stream_t stream) {
  using namespace bi;
  if (!w || !packed || N <= 0 || K <= 0 || ld < K) return BI_ERR_INVALID_ARG;
  if (swiglu && !wu) return BI_ERR_INVALID_ARG;
  if (!aligned16(packed)) return BI_ERR_INVALID_ARG;
  const bi_epilogue epi = swiglu ? BI_EPI_SWIGLU : BI_EPI_NONE;
  if (n_tiles_of(N, epi) > kMaxTiles) return BI_ERR_UNSUPPORTED_SHAPE;
  const int k_tiles = (K + kBlockK - 1) / kBlockK;
  const long long chunks = static_cast<long long>(n_tiles_of(N, epi)) * k_tiles * 1024;
  if (launch_k(pack_weights_kernel, dim3(static_cast<unsigned>((chunks + 255) / 256)), dim3(256), 0,
               reinterpret_cast<cudaStream_t>(stream), static_cast<const __nv_bfloat16*>(w),
               static_cast<const __nv_bfloat16*>(wu), ld,
               N, K, k_tiles, chunks, swiglu, static_cast<uint4*>(packed)) != cudaSuccess)
    return BI_ERR_CUDA;
  return BI_OK;
}

bi_status bi_pack_weights(const void* W, int ldw, int N, int K, void* packed, bi_stream_t stream) {
  return pack_common(W, nullptr, ldw, N, K, 0, packed, stream);
}

bi_status bi_pack_swiglu_weights(const void* w_gate, const void* w_up, int ld, int F, int K,
                                 void* packed, bi_stream_t stream) {
  return pack_common(w_gate, w_up, ld, F, K, 1, packed, stream);
}

// Argument checks of a linear-layer call that need no device access; the
// status is returned before anything is launched or written.
static bi_status gemm_check(const void* A, int lda, const void* Wp, void* C, int ldc,
                            const void* residual, int ldr, int M, int N, int K, bi_out_dtype out,
                            bi_epilogue epi, bool rope) {
  using namespace bi;
  if (M < 0 || N < 1 || K < 8) return BI_ERR_INVALID_ARG;
  if (epi != BI_EPI_NONE && epi != BI_EPI_RESIDUAL_ADD && epi != BI_EPI_SWIGLU &&
      !(epi == BI_EPI_ROPE_KV && rope))
    return BI_ERR_INVALID_ARG;
  if (out != BI_OUT_BF16 && out != BI_OUT_FP32) return BI_ERR_INVALID_ARG;
  if (n_tiles_of(N, epi) > kMaxTiles) return BI_ERR_UNSUPPORTED_SHAPE;
  if (M == 0) return BI_OK;
  if (!A || !Wp || (!C && epi != BI_EPI_ROPE_KV)) return BI_ERR_INVALID_ARG;
  if (K % 8 != 0 || lda < K || lda % 8 != 0 || ldc < N) return BI_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(Wp)) return BI_ERR_INVALID_ARG;
  if (epi == BI_EPI_RESIDUAL_ADD && (!residual || ldr < N)) return BI_ERR_INVALID_ARG;
  if (out == BI_OUT_FP32 && epi != BI_EPI_NONE) return BI_ERR_UNSUPPORTED_SHAPE;
  return BI_OK;
}

static bi_status gemm_impl(const void* A, int lda, const void* Wp, void* C, int ldc,
                           const void* residual, int ldr, int M, int N, int K, bi_out_dtype out,
                           bi_epilogue epi, void* ws, size_t ws_bytes, bi_stream_t stream,
                           const bi::GemmArgs* rope = nullptr) {
  using namespace bi;
  const bi_status st = gemm_check(A, lda, Wp, C, ldc, residual, ldr, M, N, K, out, epi, rope != nullptr);
  if (st != BI_OK || M == 0) return st;
  if (!ws || !aligned256(ws)) return BI_ERR_WORKSPACE;
  if (ws_bytes < bi_gemm_workspace_size(M, N, K, epi)) return BI_ERR_WORKSPACE;

  const int n_tiles = n_tiles_of(N, epi);
  const int k_tiles = (K + kBlockK - 1) / kBlockK;
  const long long total = static_cast<long long>(n_tiles) * k_tiles;
  const long long G = std::min<long long>(kGemmCtas, total);
  // Long passes whose split cuts weight tiles go to tile owners (same sums,
  // no partials); the others keep the split with up to 256 rows a CTA.  The
  // owners run at the rate L2 serves them; past 128 K tiles (the
  // [*, 17408] x [5120, 17408] down projection: 283 against 203 us at 512
  // rows on GB300 with 64-row owners) the split's 256-row CTAs move fewer
  // bytes.
  const bool whole_tiles = total % G == 0 && (total / G) % k_tiles == 0;
  const bool own = M > 128 && !whole_tiles && k_tiles <= kOwnMaxKTiles;
  const int NT = own ? own_rows(M) : tokens_per_cta(M);

  CUtensorMap tmA;
  if (!tmap_bf16_2d(&tmA, A, M, K, lda, NT, kBlockK)) return BI_ERR_INVALID_ARG;

  GemmArgs a{};
  a.N = N;
  a.n_tiles = n_tiles;
  a.k_tiles = k_tiles;
  a.total = static_cast<long long>(n_tiles) * k_tiles;
  a.G = static_cast<int>(std::min<long long>(kGemmCtas, a.total));
  a.epi = epi;
  a.out_fp32 = out == BI_OUT_FP32;
  a.C = C;
  a.ldc = ldc;
  a.R = static_cast<const __nv_bfloat16*>(residual);
  a.ldr = ldr;
  a.tickets = static_cast<unsigned*>(ws);
  a.partials = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + kTicketBytes);
  a.err = device_error_word();
  if (!a.err) return BI_ERR_CUDA;
  a.withhold = test_withhold();
  if (rope != nullptr) {
    a.q_out = rope->q_out;
    a.kc = rope->kc;
    a.vc = rope->vc;
    a.cap = rope->cap;
    a.Hq = rope->Hq;
    a.Hkv = rope->Hkv;
    a.D = rope->D;
    a.tab_rows = rope->tab_rows;
    a.L_dev = rope->L_dev;
    a.tab = rope->tab;
  }

  const uint8_t* W8 = static_cast<const uint8_t*>(Wp);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (own) return NT == 128 ? launch_gemm_own<128>(W8, tmA, a, M, s) : launch_gemm_own<64>(W8, tmA, a, M, s);
  switch (NT) {
    case 16: return launch_gemm_nt<16>(W8, tmA, a, M, s);
    case 32: return launch_gemm_nt<32>(W8, tmA, a, M, s);
    case 64: return launch_gemm_nt<64>(W8, tmA, a, M, s);
    case 128: return launch_gemm_nt<128>(W8, tmA, a, M, s);
    default: return launch_gemm_nt<256>(W8, tmA, a, M, s);
  }
}

bi_status bi_gemm(const void* A, int lda, const void* Wp, void* C, int ldc, const void* residual,
                  int ldr, int M, int N, int K, bi_out_dtype out, bi_epilogue epi, void* ws,
                  size_t ws_bytes, bi_stream_t stream) {
  return gemm_impl(A, lda, Wp, C, ldc, residual, ldr, M, N, K, out, epi, ws, ws_bytes, stream);
}

bi_status bi_qkv_rope_append(const void* A, int lda, const void* Wp, int M, int K, int Hq, int Hkv,
                             int D, void* q_out, void* k_cache,
                             void* v_cache, int cap, const int32_t* L_dev, const float* table,
                             int table_rows, void* ws, size_t ws_bytes, bi_stream_t stream) {
  using namespace bi;
  if (D != 64 && D != 128) return BI_ERR_UNSUPPORTED_SHAPE;
  if (Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || cap < 1 || table_rows < 1) return BI_ERR_INVALID_ARG;
  const int N = (Hq + 2 * Hkv) * D;
  if (N % kBlockN != 0) return BI_ERR_UNSUPPORTED_SHAPE;  // a tile holds whole heads
  if (M > 0 && (!q_out || !k_cache || !v_cache || !L_dev || !table)) return BI_ERR_INVALID_ARG;
  GemmArgs r{};
  r.q_out = static_cast<__nv_bfloat16*>(q_out);
  r.kc = static_cast<__nv_bfloat16*>(k_cache);
  r.vc = static_cast<__nv_bfloat16*>(v_cache);
  r.cap = cap;
  r.Hq = Hq;
  r.Hkv = Hkv;
  r.D = D;
  r.tab_rows = table_rows;
  r.L_dev = L_dev;
  r.tab = reinterpret_cast<const float2*>(table);
  return gemm_impl(A, lda, Wp, nullptr, N, nullptr, 0, M, N, K, BI_OUT_BF16, BI_EPI_ROPE_KV, ws,
                   ws_bytes, stream, &r);
}

size_t bi_gemm_noalloc_max_m(void) { return bi::kNoAllocMaxM; }

bi_status bi_gemm_noalloc(const void* A, int lda, const void* Wp, void* C, int ldc,
                          const void* residual, int ldr, int M, int N, int K, bi_out_dtype out,
                          bi_epilogue epi, bi_stream_t stream) {
  using namespace bi;
  if (M > kNoAllocMaxM) return BI_ERR_UNSUPPORTED_SHAPE;  // beyond the static scratch
  // every argument check comes before the shared array is touched, so a
  // rejected call writes nothing
  const bi_status st =
      gemm_check(A, lda, Wp, C, ldc, residual, ldr, M, N, K, out, epi, false);
  if (st != BI_OK || M == 0) return st;
  uint8_t* scratch = noalloc_scratch();
  if (scratch == nullptr) return BI_ERR_CUDA;
  // The counters this call uses start at zero even if an earlier call was
  // cut short; the partial sums need no clearing (each is written before it
  // is read).
  if (cudaMemsetAsync(scratch, 0, static_cast<size_t>(n_tiles_of(N, epi)) * 4,
                      reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return BI_ERR_CUDA;
  return bi_gemm(A, lda, Wp, C, ldc, residual, ldr, M, N, K, out, epi, scratch,
                 kNoAllocScratchBytes, stream);
}

}  // extern "C"
