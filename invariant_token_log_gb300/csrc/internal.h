// Host functions shared by the library's translation units.  They are not
// part of the C ABI (hidden visibility: the shared library does not export
// them).
#pragma once

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>  // header-only NVTX v3: ranges cost a pointer test unless a profiler is attached
#include <stdint.h>

#define BIL_INTERNAL __attribute__((visibility("hidden")))

namespace bil_internal {

// Check active targets on the host: copies them in chunks through a stack
// buffer (synchronises the stream).  BIL_E_TARGET_RANGE if an active target
// lies outside [0, vocab).
BIL_INTERNAL int check_targets_host(const int64_t* targets, int64_t n, int64_t ignore_index, int64_t vocab,
                                    cudaStream_t stream);

// rcp = 1/temperature rounded once to float32; BIL_E_INVALID_ARG unless the
// temperature is finite and > 0 and its reciprocal is finite.
BIL_INTERNAL int temperature_rcp(float temperature, float* rcp);

// Streaming multiprocessors and opt-in shared memory per block of the current
// device (cached per device).
BIL_INTERNAL int device_limits(int* sms, int* max_smem_optin);

// Bytes of one element of a BIL_* type (0 for an unknown type).
BIL_INTERNAL int elem_bytes(int dtype);

// num_tiles = ceil(vocab / tile_v) after checking tile_v (a positive multiple
// of 8 of at most BIL_MAX_TILE_BYTES bytes) and the element type.
BIL_INTERNAL int check_tile(int dtype, int64_t vocab, int32_t tile_v, int64_t* num_tiles);

// rows x pitch x eb within BIL_MAX_EXTENT_BYTES (rows <= 0: nothing spanned).
// pitch and eb are positive.
BIL_INTERNAL bool extent_ok(int64_t rows, int64_t pitch, int64_t eb);

// A named NVTX range over the rest of the enclosing scope.  Every C-ABI entry
// point that queues work opens one named after itself, so that a profiler's
// timeline attributes host time and the kernels launched inside it to the call.
class BIL_INTERNAL NvtxRange {
 public:
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// The LM-head kernels' watchdog word of the current device (see
// bil_watchdog_status); cleared when `clear` is non-zero.
BIL_INTERNAL int linear_watchdog(unsigned int* flags, int clear);

}  // namespace bil_internal
