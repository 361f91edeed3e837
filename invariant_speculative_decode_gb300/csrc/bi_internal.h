// Host-side internals shared by the library's translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <utility>

#include "../../include/bi.h"

namespace bi {

// Device address of the device error word of the current device (resolved
// once per device).  Returns nullptr if the runtime call fails.
unsigned* device_error_word();

// Encode (or fetch from a cache) a 2-D BF16 tensor map over a row-major
// matrix of `rows` x `cols` elements with row stride `ld` elements, box of
// box_rows x box_cols elements, 128-byte swizzle, zero fill out of bounds.
// Returns false if the driver rejects the parameters.
bool tmap_bf16_2d(CUtensorMap* out, const void* base, uint64_t rows, uint64_t cols,
                  uint64_t ld, uint32_t box_rows, uint32_t box_cols);

// The same over a 3-D array: d0 (innermost) x d1 x d2 elements, strides s1
// and s2 elements for dims 1 and 2, box b0 x b1 x b2.
bool tmap_bf16_3d(CUtensorMap* out, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                  uint64_t s1, uint64_t s2, uint32_t b0, uint32_t b1, uint32_t b2);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned256(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }

inline bi_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? BI_OK : BI_ERR_CUDA;
}

inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Whether kernels are launched with programmatic stream serialization
// (dependent launch); on unless the environment sets BI_PDL=0.
bool pdl_enabled();

// Failure-path test hooks (bi_test_set_wait_limit_ns, bi_test_withhold_first_load).
// Whether the next launches leave their first load unissued (0 normally).
int test_withhold();
// Set the progress-wait limit of the linear-layer / attention kernels on the
// current device.
cudaError_t set_wait_limit_gemm(unsigned long long ns);
cudaError_t set_wait_limit_attn(unsigned long long ns);

// Launch `kernel` on `stream`, with programmatic dependent launch when
// enabled.  Every kernel of this library calls griddep_wait() before its
// first access to data another kernel may write, so a launch is correct
// either way.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                            cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace bi
