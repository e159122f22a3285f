// gdn_chunk_fwd_noalloc: the GDN chunked forward for callers that cannot hand
// the library a workspace.
//
// The tensor-core path of gdn_chunk_fwd needs scratch memory (per chunk and
// head operand blocks written by the intra-chunk kernel and read by the
// sequential state kernel).  Normally the caller allocates it.  Some callers
// cannot: a host runtime that owns a fixed device-memory budget and forbids
// plugins from calling cudaMalloc, a serving loop that must not hit
// cudaMalloc's implicit device synchronisation on its latency path, or code
// that runs where no allocator is available to it.  This entry point uses a
// file-scope device array instead, so it allocates nothing at all.
//
// The array is NOALLOC_SCRATCH_BYTES (32 MiB) and lives on every GPU that
// loads this library until the process exits.  Problems whose workspace
// (gdn_chunk_workspace_size) exceeds it are rejected with GDN_ERR_WORKSPACE.
// Nothing in the scratch has to start at zero: every byte the kernels read
// in a call is written earlier in the same call.  All calls on a device share
// the one array, so calls that overlap on the GPU (different streams, or
// devices' work not ordered by the caller) race on it; order them.
//
// The first call on each device looks up the array's device address with
// cudaGetSymbolAddress while that device is current (the host-side symbol is
// not a device address); that first call should therefore come before any
// stream capture.
#include "gdn.h"

#include <cuda_runtime.h>

#include <atomic>

#include "gdn_internal.h"

namespace {

constexpr size_t NOALLOC_SCRATCH_BYTES = size_t(32) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

constexpr int MAX_DEVICES = 64;
// Per-device address of the array, resolved once per device.  Host threads
// may make their first call on a device at the same time: the slot is an
// atomic, so concurrent first calls at worst both resolve the (same) address.
std::atomic<void *> g_scratch_ptr[MAX_DEVICES];

// Device address of the scratch array on the current device (set up once).
void *scratch_address(gdn_status_t *st) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) {
    (void)cudaGetLastError();
    *st = GDN_ERR_CUDA;
    return nullptr;
  }
  void *p = g_scratch_ptr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      (void)cudaGetLastError();
      *st = GDN_ERR_CUDA;
      return nullptr;
    }
    g_scratch_ptr[dev].store(p, std::memory_order_release);
  }
  *st = GDN_OK;
  return p;
}

}  // namespace

extern "C" size_t gdn_noalloc_scratch_bytes(void) { return NOALLOC_SCRATCH_BYTES; }

extern "C" gdn_status_t gdn_chunk_fwd_noalloc(const gdn_chunk_args *args, gdn_stream_t stream) {
  if (args == nullptr) return gdn::set_host_error(GDN_ERR_INVALID_ARG, "args is NULL");
  size_t need = 0;
  gdn_status_t st = gdn_chunk_workspace_size(args, &need);
  if (st != GDN_OK) return st;
  if (need > NOALLOC_SCRATCH_BYTES)
    return gdn::set_host_error(GDN_ERR_WORKSPACE,
                               "problem needs more scratch than the 32 MiB fixed array holds");
  gdn_chunk_args a = *args;
  a.workspace = nullptr;
  a.workspace_bytes = 0;
  if (need > 0) {
    a.workspace = scratch_address(&st);
    if (st != GDN_OK) return gdn::set_host_error(st, "cannot resolve the scratch array's address");
    a.workspace_bytes = NOALLOC_SCRATCH_BYTES;
  }
  return gdn_chunk_fwd(&a, stream);
}
