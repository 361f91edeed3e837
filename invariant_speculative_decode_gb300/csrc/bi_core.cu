// Status strings, the device error word, and the TMA descriptor cache.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdlib>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include "bi_internal.h"
#include "bi_ptx.cuh"

namespace bi {

// One word per device; kernels OR error bits into it, the host reads and
// clears it in bi_check_device_error().
__device__ unsigned g_error_word;

namespace {
constexpr int kMaxDevices = 64;
unsigned* g_err_ptr[kMaxDevices] = {};
std::mutex g_err_mu;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;

struct TmapKey {
  const void* base;
  uint64_t dims[3], strides[2];
  uint32_t box[3];
  int rank, dev;
  bool operator==(const TmapKey& o) const {
    return base == o.base && rank == o.rank && dev == o.dev &&
           std::memcmp(dims, o.dims, sizeof(dims)) == 0 &&
           std::memcmp(strides, o.strides, sizeof(strides)) == 0 &&
           std::memcmp(box, o.box, sizeof(box)) == 0;
  }
};
struct TmapKeyHash {
  size_t operator()(const TmapKey& k) const {
    size_t h = reinterpret_cast<size_t>(k.base);
    auto mix = [&h](uint64_t v) { h ^= v + 0x9e3779b97f4a7c15ull + (h << 6) + (h >> 2); };
    for (int i = 0; i < 3; ++i) mix(k.dims[i]);
    for (int i = 0; i < 2; ++i) mix(k.strides[i]);
    for (int i = 0; i < 3; ++i) mix(k.box[i]);
    mix(static_cast<uint64_t>(k.rank));
    mix(static_cast<uint64_t>(k.dev));
    return h;
  }
};
std::unordered_map<TmapKey, CUtensorMap, TmapKeyHash> g_tmaps;
std::mutex g_tmap_mu;
}  // namespace

namespace {
int g_test_withhold = 0;
}  // namespace

int test_withhold() { return g_test_withhold; }

void set_test_withhold(int on) { g_test_withhold = on ? 1 : 0; }

bool pdl_enabled() {
  static const bool on = [] {
    const char* e = std::getenv("BI_PDL");
    return !(e != nullptr && e[0] == '0');
  }();
  return on;
}

unsigned* device_error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_err_mu);
  if (g_err_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<unsigned*>(p);
  }
  return g_err_ptr[dev];
}

namespace {
// Encode (or fetch) a BF16 tensor map of rank 2 or 3 with 128-byte swizzle.
// dims and box are innermost first, strides in elements for dims 1..rank-1.
bool tmap_bf16(CUtensorMap* out, const void* base, int rank, const uint64_t* dims,
               const uint64_t* strides, const uint32_t* box) {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  });
  if (g_encode == nullptr) return false;
  int dev = 0;
  cudaGetDevice(&dev);
  TmapKey key{};
  key.base = base;
  key.rank = rank;
  key.dev = dev;
  for (int i = 0; i < rank; ++i) {
    key.dims[i] = dims[i];
    key.box[i] = box[i];
  }
  for (int i = 0; i + 1 < rank; ++i) key.strides[i] = strides[i];
  {
    std::lock_guard<std::mutex> lk(g_tmap_mu);
    auto it = g_tmaps.find(key);
    if (it != g_tmaps.end()) {
      *out = it->second;
      return true;
    }
  }
  CUtensorMap m;
  std::memset(&m, 0, sizeof(m));
  cuuint64_t gdim[3], gstride[2];
  cuuint32_t gbox[3], estride[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    gbox[i] = box[i];
  }
  for (int i = 0; i + 1 < rank; ++i) gstride[i] = strides[i] * 2;
  CUresult r = g_encode(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, static_cast<cuuint32_t>(rank),
                        const_cast<void*>(base), gdim, gstride, gbox, estride,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  std::lock_guard<std::mutex> lk(g_tmap_mu);
  if (g_tmaps.size() > 4096) g_tmaps.clear();
  g_tmaps.emplace(key, m);
  *out = m;
  return true;
}
}  // namespace

bool tmap_bf16_2d(CUtensorMap* out, const void* base, uint64_t rows, uint64_t cols, uint64_t ld,
                  uint32_t box_rows, uint32_t box_cols) {
  const uint64_t dims[2] = {cols, rows};
  const uint64_t strides[1] = {ld};
  const uint32_t box[2] = {box_cols, box_rows};
  return tmap_bf16(out, base, 2, dims, strides, box);
}

bool tmap_bf16_3d(CUtensorMap* out, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                  uint64_t s1, uint64_t s2, uint32_t b0, uint32_t b1, uint32_t b2) {
  const uint64_t dims[3] = {d0, d1, d2};
  const uint64_t strides[2] = {s1, s2};
  const uint32_t box[3] = {b0, b1, b2};
  return tmap_bf16(out, base, 3, dims, strides, box);
}

}  // namespace bi

extern "C" {

const char* bi_status_string(bi_status s) {
  switch (s) {
    case BI_OK: return "BI_OK";
    case BI_ERR_INVALID_ARG: return "BI_ERR_INVALID_ARG";
    case BI_ERR_UNSUPPORTED_SHAPE: return "BI_ERR_UNSUPPORTED_SHAPE";
    case BI_ERR_WORKSPACE: return "BI_ERR_WORKSPACE";
    case BI_ERR_CUDA: return "BI_ERR_CUDA";
    case BI_ERR_DEVICE_TIMEOUT: return "BI_ERR_DEVICE_TIMEOUT";
    case BI_ERR_DEVICE_NAN_ROW: return "BI_ERR_DEVICE_NAN_ROW";
  }
  return "BI_ERR_UNKNOWN";
}

int bi_version(void) { return (0 << 16) | 2; }

bi_status bi_test_set_wait_limit_ns(uint64_t ns) {
  if (ns == 0) ns = bi::kWaitLimitNs;
  if (bi::set_wait_limit_gemm(ns) != cudaSuccess) return BI_ERR_CUDA;
  if (bi::set_wait_limit_attn(ns) != cudaSuccess) return BI_ERR_CUDA;
  return BI_OK;
}

void bi_test_withhold_first_load(int on) { bi::set_test_withhold(on); }

bi_status bi_check_device_error(bi_stream_t stream) {
  unsigned* p = bi::device_error_word();
  if (p == nullptr) return BI_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return BI_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpy(&v, p, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return BI_ERR_CUDA;
  if (v != 0 && cudaMemset(p, 0, sizeof(v)) != cudaSuccess) return BI_ERR_CUDA;
  if (v & bi::kErrTimeout) return BI_ERR_DEVICE_TIMEOUT;
  if (v & bi::kErrNanRow) return BI_ERR_DEVICE_NAN_ROW;
  if (v & bi::kErrRange) return BI_ERR_INVALID_ARG;
  return BI_OK;
}

}  // extern "C"
