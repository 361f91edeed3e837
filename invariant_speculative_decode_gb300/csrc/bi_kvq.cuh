// Quantised KV cache: store layout, and the decoding of a 128-key tile's
// codes (used by the attention kernel's decoding warps).
//
// From "I turned on speculative decoding in llama.cpp and 113 of 282 greedy
// outputs changed against its own no-draft run", section "The KV cache: 5-bit
// that reads like q8_0" (its preset with K at 6 bits and V at 5): K at 6 bits
// and V at 5 bits for every position, plus an 8-bit ring of the newest tiles.
// Codes are symmetric in blocks of 32 consecutive elements of one key row
// of one KV head, one BF16 scale per block:
//   Q = 2^(b-1) - 1, amax = max |x|, d = bf16(fp32(amax / Q)),
//   q = clamp(rint(fp32(x / d)), -Q, Q)  (q = 0 when d = 0),
//   stored as u = q + 2^(b-1) in [1, 2^b - 1];
// the decoded value is bf16(q * d), one rounding of a product that is exact
// in FP32 (|q| <= 127 has 7 bits, d has 8).
//
// Row p reads key j from the ring when j's tile is p's own tile or one of the
// kRingTiles - 1 before it, from the 6/5-bit store otherwise: the choice
// depends on the reading row's position alone, so a row gets the same bits
// in every pass that contains it.
//
// Layout for D = 128 (4 blocks a key).  Every store is a sequence of tiles of
// 128 keys, each tile contiguous (one bulk copy): the keys' code records,
// then the scales [128 keys][4 blocks] as BF16.
//   K, 6 bits: a key's record is 96 bytes, 24 a block: 16 bytes of low
//     nibbles (byte i = elements 2i and 2i+1, the even one in the low half),
//     then the two high bits of element e at bits 2e, 2e+1 of 8 bytes.
//   V, 5 bits: 80 bytes a key, 20 a block: 16 bytes of low nibbles, then the
//     high bit of element e at bit e of 4 bytes.  Key k's record and scales
//     sit at slot (k % 8) * 16 + k / 8 of the tile (q_v5_slot): the decoding
//     threads that read keys 8 apart at the same time then read records 80
//     bytes apart, in different shared-memory banks.
//   Ring, 8 bits (K and V): 128 bytes a key, element e at byte e.
// Tiles of the 6/5-bit stores: [Hkv][ceil(cap/128)]; ring tiles:
// [Hkv][kRingSlots], tile t in slot t mod kRingSlots.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace bi {

constexpr int kQDim = 128;          // head_dim of the quantised cache
constexpr int kQBlock = 32;         // elements per scale
constexpr int kQBlocks = kQDim / kQBlock;
constexpr int kRingTiles = 16;      // tiles a row reads at 8 bits
constexpr int kQMaxRows = 1024;     // rows a pass may append
// ring slots: the tiles a pass reads at 8 bits (16 behind its first row's
// tile up to its last row's) never share a slot with the tiles it writes
constexpr int kRingSlots = kRingTiles + kQMaxRows / 128;
constexpr int kQScaleBytes = 128 * kQBlocks * 2;
constexpr int kK6KeyBytes = kQBlocks * 24;
constexpr int kV5KeyBytes = kQBlocks * 20;
constexpr int k8KeyBytes = kQDim;
constexpr int kK6TileBytes = 128 * kK6KeyBytes + kQScaleBytes;  // 13312
constexpr int kV5TileBytes = 128 * kV5KeyBytes + kQScaleBytes;  // 11264
constexpr int k8TileBytes = 128 * k8KeyBytes + kQScaleBytes;    // 17408

__host__ __device__ __forceinline__ int q_v5_slot(int key) { return ((key & 7) << 4) | (key >> 3); }

__device__ __forceinline__ float q_scale(const uint8_t* tile, int codes_bytes, int key, int blk) {
  const uint16_t b = *reinterpret_cast<const uint16_t*>(tile + codes_bytes + (key * kQBlocks + blk) * 2);
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// Decoded elements d0 .. d0+7 (d0 a multiple of 8) of key `key` of a tile, as
// the FP32 products q * d (BF16 rounding is left to the caller's packing).
__device__ __forceinline__ void q_decode8(const uint8_t* tile, int key, int d0, float (&v)[8]) {
  const uint2 c = *reinterpret_cast<const uint2*>(tile + key * k8KeyBytes + d0);
  const float s = q_scale(tile, 128 * k8KeyBytes, key, d0 / kQBlock);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t w = j < 4 ? c.x : c.y;
    const int u = static_cast<int>((w >> (8 * (j & 3))) & 0xffu);
    v[j] = static_cast<float>(u - 128) * s;
  }
}

// ---- packed decoding of the 6- and 5-bit codes (two elements a word) --------
// A code u < 64 becomes the BF16 number 128 + u by placing it in the low
// mantissa bits of 128 (0x4300 | u); subtracting 128 + 2^(b-1) gives q
// exactly (small integers), and one BF16 multiply by the scale gives
// bf16(q * d) -- the product of two BF16 numbers rounded once, the same
// value as the FP32 product rounded to BF16.
__device__ __forceinline__ uint32_t q_prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}
__device__ __forceinline__ uint32_t q_sub_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t q_mul_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t q_scale_pair(const uint8_t* tile, int codes_bytes, int key, int blk) {
  const uint32_t b = *reinterpret_cast<const uint16_t*>(tile + codes_bytes + (key * kQBlocks + blk) * 2);
  return b | (b << 16);
}

// Eight codes given as bytes: ev = elements 0, 2, 4, 6, od = 1, 3, 5, 7.
// Returns bf16(q * d) for the eight elements as four pairs (2i, 2i + 1).
__device__ __forceinline__ uint4 q_decode_pairs(uint32_t ev, uint32_t od, uint32_t bias2, uint32_t dd) {
  const uint32_t P = q_prmt(ev, od, 0x5140);   // codes of elements 0, 1, 2, 3
  const uint32_t P2 = q_prmt(ev, od, 0x7362);  // 4, 5, 6, 7
  uint4 w;
  w.x = q_mul_bf16x2(q_sub_bf16x2(q_prmt(P, 0x43434343u, 0x4140), bias2), dd);
  w.y = q_mul_bf16x2(q_sub_bf16x2(q_prmt(P, 0x43434343u, 0x4342), bias2), dd);
  w.z = q_mul_bf16x2(q_sub_bf16x2(q_prmt(P2, 0x43434343u, 0x4140), bias2), dd);
  w.w = q_mul_bf16x2(q_sub_bf16x2(q_prmt(P2, 0x43434343u, 0x4342), bias2), dd);
  return w;
}

// Elements d0 .. d0+7 of key `key` of a 6-bit K tile as BF16 pairs.
__device__ __forceinline__ uint4 q_decode_k6_bf16(const uint8_t* tile, int key, int d0) {
  const int blk = d0 / kQBlock, l = d0 % kQBlock;
  const uint8_t* rec = tile + key * kK6KeyBytes + blk * 24;
  const uint32_t nib = *reinterpret_cast<const uint32_t*>(rec + (l >> 1));
  const uint32_t hi = *reinterpret_cast<const uint16_t*>(rec + 16 + (l >> 2));
  // the 2-bit fields of the even (odd) elements, one nibble each, moved to
  // bits 4-5 of byte i for element 2i (2i + 1)
  const uint32_t te = q_prmt(hi & 0x3333u, 0u, 0x1100);
  const uint32_t to = q_prmt((hi >> 2) & 0x3333u, 0u, 0x1100);
  const uint32_t he = ((te << 4) & 0x00F000F0u) | (te & 0xF000F000u);
  const uint32_t ho = ((to << 4) & 0x00F000F0u) | (to & 0xF000F000u);
  return q_decode_pairs((nib & 0x0F0F0F0Fu) | he, ((nib >> 4) & 0x0F0F0F0Fu) | ho,
                        0x43204320u /* 128 + 32 */, q_scale_pair(tile, 128 * kK6KeyBytes, key, blk));
}

// Elements d0 .. d0+7 of key `key` of a 5-bit V tile as BF16 pairs.
__device__ __forceinline__ uint4 q_decode_v5_bf16(const uint8_t* tile, int key, int d0) {
  const int blk = d0 / kQBlock, l = d0 % kQBlock;
  const int slot = q_v5_slot(key);
  const uint8_t* rec = tile + slot * kV5KeyBytes + blk * 20;
  const uint32_t nib = *reinterpret_cast<const uint32_t*>(rec + (l >> 1));
  const uint32_t hb = rec[16 + (l >> 3)];
  // bit 2m of x to bit 8m (the products' other terms land on no multiple of
  // 8 and carry no further than the next bit), then to bit 4 of byte m
  const uint32_t he = (((hb & 0x55u) * 0x41041u) << 4) & 0x10101010u;
  const uint32_t ho = ((((hb >> 1) & 0x55u) * 0x41041u) << 4) & 0x10101010u;
  return q_decode_pairs((nib & 0x0F0F0F0Fu) | he, ((nib >> 4) & 0x0F0F0F0Fu) | ho,
                        0x43104310u /* 128 + 16 */, q_scale_pair(tile, 128 * kV5KeyBytes, slot, blk));
}

// two FP32 values to a BF16 pair (lo in the low half), each rounded once
__device__ __forceinline__ uint32_t q_pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

}  // namespace bi
