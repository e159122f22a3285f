// Shared device helpers of the gated delta-rule library (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

// Chunk length of the chunked forward (sglang fla/chunk_fwd.py: BT = 64).
constexpr int BT = 64;
// Longest key dimension the chunk kernels take.
constexpr int KMAX = 128;
// Largest grid y / z dimension of a launch: heads and sequences index them.
constexpr int MAX_GRID_YZ = 65535;
// Most segments per sequence of the segment-parallel state pass.
constexpr int MAX_SEGMENTS = 64;

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// Record the first device-side error in the library's error word.
__device__ __forceinline__ void record_error(int *err, int code) {
  if (err) atomicCAS(err, 0, code);
}

// Checked builds (-DGDN_CHECKED): before a CTA touches memory it compares the
// index ranges it derived with the extents of the tensors they index; on a
// violation it records GDN_ERR_BOUNDS and returns, uniformly over the CTA and
// before any barrier.  `cond` must be uniform over the CTA.  Release builds
// compile the check away.
#ifdef GDN_CHECKED
constexpr bool kChecked = true;
#else
constexpr bool kChecked = false;
#endif
__device__ __forceinline__ bool bounds_ok(bool cond, int *err) {
  if (kChecked && !cond) {
    if (threadIdx.x == 0) record_error(err, GDN_ERR_BOUNDS);
    return false;
  }
  return true;
}

// Host: device address of the error word of the current device.
int *device_error_word();

}  // namespace gdn
