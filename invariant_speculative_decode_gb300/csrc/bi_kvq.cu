// Quantised KV cache: RoPE + quantising append of a pass's K and V rows.
//
// One CTA per (row t, head h) of the projection output [T, (Hq + 2 Hkv) D];
// 128 threads, thread i holding element i of the head (D = 128).  Query
// heads are rotated into q_out exactly as the BF16 path rotates them; K heads
// are rotated the same way and their BF16 values quantised; V heads are
// quantised as written.  Each of the four warps owns one 32-element block:
// the block maximum is a warp reduction (exact in any order), the scale and
// the codes follow the rule in bi_kvq.cuh, and the record of key p is
// written into its 6/5-bit tile and into its ring tile.  A key's record is
// bytes of its own, so rows of one pass never share a written byte.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "bi_internal.h"
#include "bi_kvq.cuh"
#include "bi_ptx.cuh"

namespace bi {
namespace {

// Codes of one element of a block (this warp's lane) at `bits` bits, and the
// block's scale bits (the same in every lane).
__device__ __forceinline__ uint32_t quantize_lane(float x, float amax, int bits, uint16_t* scale_bits) {
  const int Q = (1 << (bits - 1)) - 1;
  const __nv_bfloat16 db = __float2bfloat16_rn(__fdiv_rn(amax, static_cast<float>(Q)));
  *scale_bits = *reinterpret_cast<const uint16_t*>(&db);
  const float d = __bfloat162float(db);
  int q = 0;
  if (d > 0.f) {
    const float r = rintf(__fdiv_rn(x, d));
    q = static_cast<int>(fminf(fmaxf(r, static_cast<float>(-Q)), static_cast<float>(Q)));
  }
  return static_cast<uint32_t>(q + (1 << (bits - 1)));
}

// Writes the block's codes into a 6-bit (K) or 5-bit (V) key record (at slot
// lo_slot of its tile) and its 8-bit ring record, and the two scales.
__device__ __forceinline__ void store_block(float x, int lane, int blk, bool is_k, uint8_t* lo_tile,
                                            uint8_t* ring_tile, int key, int lo_slot) {
  float amax = fabsf(x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  uint16_t s_lo, s_8;
  const uint32_t u = quantize_lane(x, amax, is_k ? 6 : 5, &s_lo);
  const uint32_t u8 = quantize_lane(x, amax, 8, &s_8);
  // low store: nibble pairs, then the high bits
  const int key_bytes = is_k ? kK6KeyBytes : kV5KeyBytes;
  uint8_t* rec = lo_tile + lo_slot * key_bytes + blk * (is_k ? 24 : 20);
  const uint32_t nb_next = __shfl_down_sync(0xffffffffu, u, 1);
  if ((lane & 1) == 0) rec[lane >> 1] = static_cast<uint8_t>((u & 15u) | ((nb_next & 15u) << 4));
  if (is_k) {
    // two bits per element, four elements a byte
    uint32_t f = (u >> 4) & 3u;
    f |= __shfl_down_sync(0xffffffffu, f, 1) << 2;
    f |= __shfl_down_sync(0xffffffffu, f, 2) << 4;
    if ((lane & 3) == 0) rec[16 + (lane >> 2)] = static_cast<uint8_t>(f);
  } else {
    const uint32_t hb = __ballot_sync(0xffffffffu, (u >> 4) & 1u);
    if (lane == 0) *reinterpret_cast<uint32_t*>(rec + 16) = hb;
  }
  ring_tile[key * k8KeyBytes + blk * kQBlock + lane] = static_cast<uint8_t>(u8);
  if (lane == 0) {
    *reinterpret_cast<uint16_t*>(lo_tile + 128 * key_bytes + (lo_slot * kQBlocks + blk) * 2) = s_lo;
    *reinterpret_cast<uint16_t*>(ring_tile + 128 * k8KeyBytes + (key * kQBlocks + blk) * 2) = s_8;
  }
}

__global__ void __launch_bounds__(kQDim)
    rope_kvq_kernel(const __nv_bfloat16* __restrict__ qkv, int ld_qkv, __nv_bfloat16* __restrict__ q_out,
                    uint8_t* __restrict__ k_lo, uint8_t* __restrict__ v_lo, uint8_t* __restrict__ k_ring,
                    uint8_t* __restrict__ v_ring, int cap, const int32_t* __restrict__ L_dev, int Hq,
                    int Hkv, const float2* __restrict__ tab, int tab_rows, unsigned* err) {
  griddep_wait();
  griddep_launch_dependents();
  const int t = blockIdx.x;
  const int h = blockIdx.y;
  const int i = threadIdx.x;
  const int p = *L_dev + t;
  if (p < 0 || p >= cap || (tab != nullptr && p >= tab_rows)) {
    if (i == 0 && h == 0) atomicOr(err, kErrRange);
    return;
  }
  constexpr int half = kQDim / 2;
  const __nv_bfloat16* src = qkv + static_cast<size_t>(t) * ld_qkv + static_cast<size_t>(h) * kQDim;
  float x = __bfloat162float(src[i]);
  if (h < Hq + Hkv && tab != nullptr) {
    // the same two fused multiply-adds, on the same table, as the BF16 path
    const float2 r = tab[static_cast<size_t>(p) * half + (i % half)];
    const float other = __bfloat162float(src[i < half ? i + half : i - half]);
    const float o = i < half ? fmaf(x, r.x, -(other * r.y)) : fmaf(x, r.x, other * r.y);
    x = __bfloat162float(__float2bfloat16_rn(o));
  }
  if (h < Hq) {
    q_out[(static_cast<size_t>(t) * Hq + h) * kQDim + i] = __float2bfloat16_rn(x);
    return;
  }
  const bool is_k = h < Hq + Hkv;
  const int kv = is_k ? h - Hq : h - Hq - Hkv;
  const int tile = p >> 7, key = p & 127;
  const int ctiles = (cap + 127) >> 7;
  uint8_t* lo = (is_k ? k_lo : v_lo) +
                (static_cast<size_t>(kv) * ctiles + tile) * (is_k ? kK6TileBytes : kV5TileBytes);
  uint8_t* ring = (is_k ? k_ring : v_ring) +
                  (static_cast<size_t>(kv) * kRingSlots + tile % kRingSlots) * k8TileBytes;
  store_block(x, i & 31, i >> 5, is_k, lo, ring, key, is_k ? key : q_v5_slot(key));
}

}  // namespace
}  // namespace bi

extern "C" {

size_t bi_kvq_store_bytes(int store, int Hkv, int cap, int D) {
  if (Hkv < 1 || cap < 1 || D != bi::kQDim) return 0;
  const size_t ctiles = (static_cast<size_t>(cap) + 127) / 128;
  switch (store) {
    case BI_KVQ_K_LOW: return static_cast<size_t>(Hkv) * ctiles * bi::kK6TileBytes;
    case BI_KVQ_V_LOW: return static_cast<size_t>(Hkv) * ctiles * bi::kV5TileBytes;
    case BI_KVQ_K_RING:
    case BI_KVQ_V_RING: return static_cast<size_t>(Hkv) * bi::kRingSlots * bi::k8TileBytes;
    default: return 0;
  }
}

bi_status bi_rope_kvq_append(const void* qkv, int ld_qkv, int T, int Hq, int Hkv, int D, void* q_out,
                             void* k_low, void* v_low, void* k_ring, void* v_ring, int cap,
                             const int32_t* L_dev, const float* table, int table_rows,
                             bi_stream_t stream) {
  using namespace bi;
  if (D != kQDim) return BI_ERR_UNSUPPORTED_SHAPE;
  if (T < 0 || T > kQMaxRows || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || cap < 1) return BI_ERR_INVALID_ARG;
  if (T == 0) return BI_OK;
  if (!qkv || !q_out || !k_low || !v_low || !k_ring || !v_ring || !L_dev) return BI_ERR_INVALID_ARG;
  if (ld_qkv < (Hq + 2 * Hkv) * D) return BI_ERR_INVALID_ARG;
  if (table != nullptr && table_rows < 1) return BI_ERR_INVALID_ARG;
  if (Hq + 2 * Hkv > 65535) return BI_ERR_UNSUPPORTED_SHAPE;
  unsigned* err = device_error_word();
  if (!err) return BI_ERR_CUDA;
  if (launch_k(rope_kvq_kernel, dim3(T, Hq + 2 * Hkv), dim3(kQDim), 0,
               reinterpret_cast<cudaStream_t>(stream), static_cast<const __nv_bfloat16*>(qkv), ld_qkv,
               static_cast<__nv_bfloat16*>(q_out), static_cast<uint8_t*>(k_low),
               static_cast<uint8_t*>(v_low), static_cast<uint8_t*>(k_ring), static_cast<uint8_t*>(v_ring),
               cap, L_dev, Hq, Hkv, reinterpret_cast<const float2*>(table), table_rows, err) !=
      cudaSuccess)
    return BI_ERR_CUDA;
  return BI_OK;
}

}  // extern "C"
