// gdn_self_test_wait: runs the library's bounded mbarrier wait on a barrier
// that nothing arrives on (or that the kernel has completed itself), so that
// the timeout path -- the wait giving up after its poll limit and recording
// GDN_ERR_TIMEOUT in the device error word -- can be exercised on a GPU
// without any copy or tensor-core work in flight.  gdn_self_test_bounds runs
// the bounds check of a checked build (GDN_ERR_BOUNDS) the same way.
#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "ptx.cuh"

namespace gdn {
namespace {

constexpr uint32_t MAX_SELF_TEST_POLLS = 1u << 22;  // the kernels' own default limit

__global__ void self_test_wait_kernel(int arrive, uint32_t max_polls, int *err) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  ptx::mbar_init(&bar, 1);
  ptx::fence_mbar_init();
  if (arrive) ptx::mbar_arrive(&bar);  // completes phase 0
  if (!ptx::mbar_wait_bounded(&bar, 0, max_polls)) record_error(err, GDN_ERR_TIMEOUT);
}

// One CTA: the check every kernel of a checked build makes at its start.
__global__ void self_test_bounds_kernel(int index, int extent, int *err) {
  if (!bounds_ok(index >= 0 && index < extent, err)) return;
}

}  // namespace
}  // namespace gdn

extern "C" gdn_status_t gdn_self_test_wait(int32_t arrive, int32_t max_polls, gdn_stream_t stream) {
  using namespace gdn;
  if ((arrive != 0 && arrive != 1) || max_polls < 1 || (uint32_t)max_polls > MAX_SELF_TEST_POLLS)
    return set_host_error(GDN_ERR_INVALID_ARG, "arrive must be 0 or 1 and max_polls in [1, 2^22]");
  int *err = device_error_word();
  if (err == nullptr) {
    (void)cudaGetLastError();
    return set_host_error(GDN_ERR_CUDA, "device error word");
  }
  self_test_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      arrive, (uint32_t)max_polls, err);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_host_error(GDN_ERR_CUDA, cudaGetErrorString(e));
  return GDN_OK;
}

extern "C" gdn_status_t gdn_self_test_bounds(int32_t index, int32_t extent, int32_t *checked_build,
                                             gdn_stream_t stream) {
  using namespace gdn;
  if (checked_build) *checked_build = kChecked ? 1 : 0;
  int *err = device_error_word();
  if (err == nullptr) {
    (void)cudaGetLastError();
    return set_host_error(GDN_ERR_CUDA, "device error word");
  }
  self_test_bounds_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(index, extent, err);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_host_error(GDN_ERR_CUDA, cudaGetErrorString(e));
  return GDN_OK;
}
