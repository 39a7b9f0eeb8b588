// Device-side helpers shared by libtpa's kernels: launch checks, the
// per-translation-unit status word, and small integer utilities.
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

#include "tpa.h"

// Codes written into a translation unit's device status word.
enum : unsigned int {
  TPA_DEV_OK = 0,
  TPA_DEV_TIMEOUT = 1,    // a bounded mbarrier wait ran out; the kernel returned early
  TPA_DEV_BAD_INPUT = 4,  // an input was outside its range (e.g. a label id >= vocab); it was skipped
};

// Debug builds (TPA_DEBUG=1, libtpa_debug.so) check every metadata index a
// kernel reads from a tree view before using it as an address: a bad one is
// recorded in the translation unit's status word (TPA_DEV_BAD_INPUT, which
// tpa_sync_status reports as TPA_ERR_INVALID_ARG) and its access is skipped.
// Release builds compile the checks away (dbg_ok is always true there).
#ifndef TPA_DEBUG
#define TPA_DEBUG 0
#endif

__device__ __forceinline__ bool dbg_ok(bool ok, unsigned int* status) {
#if TPA_DEBUG
  if (!ok) {
    atomicOr(status, TPA_DEV_BAD_INPUT);
    return false;
  }
#else
  (void)ok;
  (void)status;
#endif
  return true;
}

#define TPA_CUDA_TRY(expr)                        \
  do {                                            \
    if ((expr) != cudaSuccess) {                  \
      (void)cudaGetLastError();                   \
      return TPA_ERR_CUDA;                        \
    }                                             \
  } while (0)

// Reads and optionally clears a device status word.  Must run after the
// stream that may have written it has been synchronised.
#define TPA_DEFINE_STATUS_READER(fn_name, symbol)                                  \
  int fn_name(bool clear) {                                                        \
    unsigned int v = 0;                                                            \
    if (cudaMemcpyFromSymbol(&v, symbol, sizeof(v)) != cudaSuccess) {              \
      (void)cudaGetLastError();                                                    \
      return TPA_ERR_CUDA;                                                         \
    }                                                                              \
    if (clear && v != 0) {                                                         \
      const unsigned int z = 0;                                                    \
      if (cudaMemcpyToSymbol(symbol, &z, sizeof(z)) != cudaSuccess) {              \
        (void)cudaGetLastError();                                                  \
        return TPA_ERR_CUDA;                                                       \
      }                                                                            \
    }                                                                              \
    if (v & TPA_DEV_BAD_INPUT) return TPA_ERR_INVALID_ARG;                         \
    return v == 0 ? TPA_OK : TPA_ERR_DEVICE_TIMEOUT;                               \
  }

__device__ __forceinline__ int warp_sum(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
