// C entry points: argument checks on the host, then one launch per call.
// Nothing here allocates device memory.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {

// The device error word (one int per device that loads the library).
__device__ int g_error_word = 0;

int *device_error_word() {
  void *p = nullptr;
  if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
  return static_cast<int *>(p);
}

namespace {

thread_local char g_msg[256] = "";

gdn_status_t fail(gdn_status_t st, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return st;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

#define REQUIRE(cond, st, ...)            \
  do {                                    \
    if (!(cond)) return fail(st, __VA_ARGS__); \
  } while (0)

#define REQUIRE_PTR(ptr, name)                                                       \
  do {                                                                               \
    if ((ptr) == nullptr) return fail(GDN_ERR_INVALID_ARG, "%s must not be NULL", name); \
    if (!aligned16(ptr)) return fail(GDN_ERR_MISALIGNED, "%s is not 16-byte aligned", name); \
  } while (0)

#define REQUIRE_OPT_PTR(ptr, name)                                                   \
  do {                                                                               \
    if ((ptr) != nullptr && !aligned16(ptr))                                         \
      return fail(GDN_ERR_MISALIGNED, "%s is not 16-byte aligned", name);            \
  } while (0)

// Checks shared by the two chunked forwards.  Hk = key heads, Hv = value heads.
gdn_status_t check_chunk(int32_t dtype, const void *q, const void *k, const void *v,
                         const float *g, const float *beta, const float *h0, const float *ht,
                         const void *o, const int32_t *cu, int B, int T, int Hk, int Hv, int K,
                         int V, int N, int chunk_size, int g_is_cumsum, int v_first,
                         int o_f32, int segments, float scale, const char *hk_name,
                         bool sizes_only = false) {
  REQUIRE(dtype == GDN_F32 || dtype == GDN_BF16, GDN_ERR_INVALID_ARG, "dtype %d is not GDN_F32/GDN_BF16", dtype);
  REQUIRE(B >= 1 && T >= 0 && Hk >= 1 && Hv >= 1 && K >= 1 && V >= 1 && N >= 1,
          GDN_ERR_INVALID_ARG, "sizes must be positive (B=%d T=%d heads=%d/%d K=%d V=%d N=%d)", B,
          T, Hk, Hv, K, V, N);
  REQUIRE(Hv % Hk == 0, GDN_ERR_UNSUPPORTED, "value heads (%d) must be a multiple of %s (%d)", Hv,
          hk_name, Hk);
  REQUIRE(N <= MAX_GRID_YZ && Hv <= MAX_GRID_YZ, GDN_ERR_UNSUPPORTED,
          "N (%d) and the value heads (%d) must be at most %d", N, Hv, MAX_GRID_YZ);
  REQUIRE(K <= KMAX, GDN_ERR_UNSUPPORTED, "K=%d exceeds %d", K, KMAX);
  REQUIRE(chunk_size == BT, GDN_ERR_UNSUPPORTED, "chunk_size must be %d (got %d)", BT, chunk_size);
  REQUIRE(g_is_cumsum == 0 || g_is_cumsum == 1, GDN_ERR_INVALID_ARG, "g_is_cumsum must be 0 or 1");
  REQUIRE(v_first == 0 || v_first == 1, GDN_ERR_INVALID_ARG, "state_v_first must be 0 or 1");
  REQUIRE(o_f32 == 0 || o_f32 == 1, GDN_ERR_INVALID_ARG, "o_fp32 must be 0 or 1");
  REQUIRE(segments >= 0, GDN_ERR_INVALID_ARG, "segments must not be negative");
  REQUIRE(segments <= MAX_SEGMENTS && (long long)N * (segments > 0 ? segments : 1) <= MAX_GRID_YZ,
          GDN_ERR_UNSUPPORTED, "segments (%d) must be at most %d and N * segments at most %d",
          segments, MAX_SEGMENTS, MAX_GRID_YZ);
  REQUIRE(isfinite(scale), GDN_ERR_INVALID_ARG, "scale must be finite");
  if (cu == nullptr) {
    REQUIRE(N == B, GDN_ERR_INVALID_ARG, "without cu_seqlens N (%d) must equal B (%d)", N, B);
  } else {
    REQUIRE(B == 1, GDN_ERR_INVALID_ARG, "with cu_seqlens B must be 1 (got %d)", B);
  }
  if (sizes_only) return GDN_OK;
  if (T > 0) {
    REQUIRE_PTR(q, "q");
    REQUIRE_PTR(k, "k");
    REQUIRE_PTR(v, "v");
    REQUIRE_PTR(g, "g");
    REQUIRE_PTR(beta, "beta");
    REQUIRE_PTR(o, "o");
  } else {  // no token is read or written: the per-token arrays may be NULL
    REQUIRE_OPT_PTR(q, "q");
    REQUIRE_OPT_PTR(k, "k");
    REQUIRE_OPT_PTR(v, "v");
    REQUIRE_OPT_PTR(g, "g");
    REQUIRE_OPT_PTR(beta, "beta");
    REQUIRE_OPT_PTR(o, "o");
  }
  REQUIRE_OPT_PTR(h0, "h0");
  REQUIRE_OPT_PTR(ht, "ht");
  REQUIRE_OPT_PTR(cu, "cu_seqlens");
  (void)T;
  return GDN_OK;
}

gdn_status_t cuda_status(cudaError_t e, const char *what) {
  if (e == cudaSuccess) return GDN_OK;
  // The status carries the error; take it out of the runtime's last-error
  // slot so that the caller's next, unrelated CUDA call does not report it
  // (a sticky error stays in the context whatever this does).
  (void)cudaGetLastError();
  return fail(GDN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

ChunkParams gdn_params(const gdn_chunk_args &a) {
  ChunkParams p{};
  p.q = a.q; p.k = a.k; p.v = a.v; p.g = a.g; p.beta = a.beta; p.h0 = a.h0; p.ht = a.ht;
  p.o = a.o; p.cu_seqlens = a.cu_seqlens;
  p.B = a.B; p.T = a.T; p.H = a.H; p.Hk = a.Hg; p.K = a.K; p.V = a.V; p.N = a.N;
  p.g_is_cumsum = a.g_is_cumsum;
  p.v_first = a.state_v_first;
  p.o_f32 = a.o_fp32 || a.dtype == GDN_F32;
  p.segments = a.segments;
  p.scale = a.scale > 0.f ? a.scale : 1.0f / sqrtf((float)(a.K > 0 ? a.K : 1));
  return p;
}

ChunkParams kda_params(const kda_chunk_args &a) {
  ChunkParams p{};
  p.q = a.q; p.k = a.k; p.v = a.v; p.g = a.g; p.beta = a.beta; p.h0 = a.h0; p.ht = a.ht;
  p.o = a.o; p.cu_seqlens = a.cu_seqlens;
  p.B = a.B; p.T = a.T; p.H = a.HV; p.Hk = a.H; p.K = a.K; p.V = a.V; p.N = a.N;
  p.g_is_cumsum = a.g_is_cumsum;
  p.v_first = a.state_v_first;
  p.o_f32 = a.o_fp32 || a.dtype == GDN_F32;
  p.segments = a.segments;
  p.scale = a.scale > 0.f ? a.scale : 1.0f / sqrtf((float)(a.K > 0 ? a.K : 1));
  return p;
}

// Launch either path: the tensor-core kernels when they serve the arguments,
// else the exact fp32 CUDA-core kernel.
gdn_status_t run_chunk(ChunkParams &p, bool bf16, bool kda, void *ws, size_t ws_bytes,
                       cudaStream_t s) {
  const bool tc = chunk_tc_supported(p, bf16);
  if (tc) {
    const size_t need = chunk_tc_workspace(p, kda);
    if (ws == nullptr || ws_bytes < need)
      return fail(GDN_ERR_WORKSPACE, "workspace of %zu bytes needed (got %zu)", need, ws_bytes);
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
      return fail(GDN_ERR_MISALIGNED, "workspace is not 256-byte aligned");
  }
  p.err = device_error_word();
  if (p.err == nullptr) return cuda_status(cudaGetLastError(), "device error word");
  if (tc) return cuda_status(launch_chunk_tc(p, kda, ws, s), "tensor-core chunk launch");
  return cuda_status(launch_chunk_simt(p, bf16, kda, s), "chunk launch");
}

}  // namespace

gdn_status_t check_gdn_chunk_sizes(const gdn_chunk_args &a) {
  g_msg[0] = '\0';
  return check_chunk(a.dtype, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                     nullptr, a.cu_seqlens, a.B, a.T, a.Hg, a.H, a.K, a.V,
                     a.N, a.chunk_size, a.g_is_cumsum, a.state_v_first, a.o_fp32, a.segments,
                     a.scale, "Hg", true);
}

gdn_status_t set_host_error(gdn_status_t st, const char *msg) { return fail(st, "%s", msg); }

}  // namespace gdn

using namespace gdn;

extern "C" {

const char *gdn_status_string(gdn_status_t s) {
  switch (s) {
    case GDN_OK: return "GDN_OK";
    case GDN_ERR_INVALID_ARG: return "GDN_ERR_INVALID_ARG";
    case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED";
    case GDN_ERR_MISALIGNED: return "GDN_ERR_MISALIGNED";
    case GDN_ERR_WORKSPACE: return "GDN_ERR_WORKSPACE";
    case GDN_ERR_CUDA: return "GDN_ERR_CUDA";
    case GDN_ERR_TIMEOUT: return "GDN_ERR_TIMEOUT";
    case GDN_ERR_BAD_SEQLENS: return "GDN_ERR_BAD_SEQLENS";
    case GDN_ERR_BAD_SLOT: return "GDN_ERR_BAD_SLOT";
    case GDN_ERR_BOUNDS: return "GDN_ERR_BOUNDS";
  }
  return "GDN_ERR_UNKNOWN";
}

const char *gdn_last_error_message(void) { return g_msg; }

gdn_status_t gdn_chunk_workspace_size(const gdn_chunk_args *a, size_t *bytes) {
  if (a == nullptr || bytes == nullptr) return fail(GDN_ERR_INVALID_ARG, "NULL argument");
  *bytes = 0;
  ChunkParams p = gdn_params(*a);
  if (chunk_tc_supported(p, a->dtype == GDN_BF16)) *bytes = chunk_tc_workspace(p, false);
  return GDN_OK;
}

gdn_status_t gdn_chunk_segment_count(const gdn_chunk_args *a, int32_t *segments) {
  if (a == nullptr || segments == nullptr) return fail(GDN_ERR_INVALID_ARG, "NULL argument");
  *segments = 1;
  gdn_status_t st = check_gdn_chunk_sizes(*a);
  if (st != GDN_OK) return st;
  ChunkParams p = gdn_params(*a);
  if (chunk_tc_supported(p, a->dtype == GDN_BF16)) *segments = chunk_tc_segments(p);
  return GDN_OK;
}

gdn_status_t kda_chunk_workspace_size(const kda_chunk_args *a, size_t *bytes) {
  if (a == nullptr || bytes == nullptr) return fail(GDN_ERR_INVALID_ARG, "NULL argument");
  *bytes = 0;
  ChunkParams p = kda_params(*a);
  if (chunk_tc_supported(p, a->dtype == GDN_BF16)) *bytes = chunk_tc_workspace(p, true);
  return GDN_OK;
}

gdn_status_t gdn_chunk_fwd(const gdn_chunk_args *a, gdn_stream_t stream) {
  g_msg[0] = '\0';
  if (a == nullptr) return fail(GDN_ERR_INVALID_ARG, "args is NULL");
  gdn_status_t st = check_chunk(a->dtype, a->q, a->k, a->v, a->g, a->beta, a->h0, a->ht, a->o,
                                a->cu_seqlens, a->B, a->T, a->Hg, a->H, a->K, a->V, a->N,
                                a->chunk_size, a->g_is_cumsum, a->state_v_first, a->o_fp32,
                                a->segments, a->scale, "Hg");
  if (st != GDN_OK) return st;
  ChunkParams p = gdn_params(*a);
  return run_chunk(p, a->dtype == GDN_BF16, false, a->workspace, a->workspace_bytes,
                   reinterpret_cast<cudaStream_t>(stream));
}

gdn_status_t kda_chunk_fwd(const kda_chunk_args *a, gdn_stream_t stream) {
  g_msg[0] = '\0';
  if (a == nullptr) return fail(GDN_ERR_INVALID_ARG, "args is NULL");
  gdn_status_t st = check_chunk(a->dtype, a->q, a->k, a->v, a->g, a->beta, a->h0, a->ht, a->o,
                                a->cu_seqlens, a->B, a->T, a->H, a->HV, a->K, a->V, a->N,
                                a->chunk_size, a->g_is_cumsum, a->state_v_first, a->o_fp32,
                                a->segments, a->scale, "H");
  if (st != GDN_OK) return st;
  ChunkParams p = kda_params(*a);
  return run_chunk(p, a->dtype == GDN_BF16, true, a->workspace, a->workspace_bytes,
                   reinterpret_cast<cudaStream_t>(stream));
}

gdn_status_t gdn_chunk_state_fwd(const gdn_state_args *a, gdn_stream_t stream) {
  g_msg[0] = '\0';
  if (a == nullptr) return fail(GDN_ERR_INVALID_ARG, "args is NULL");
  REQUIRE(a->dtype == GDN_F32 || a->dtype == GDN_BF16, GDN_ERR_INVALID_ARG,
          "dtype %d is not GDN_F32/GDN_BF16", a->dtype);
  REQUIRE(a->gate >= GDN_GATE_NONE && a->gate <= GDN_GATE_GV, GDN_ERR_INVALID_ARG,
          "gate %d is not a gdn_gate_kind_t", a->gate);
  REQUIRE(a->B >= 1 && a->T >= 0 && a->H >= 1 && a->K >= 1 && a->V >= 1 && a->N >= 1,
          GDN_ERR_INVALID_ARG, "sizes must be positive (B=%d T=%d H=%d K=%d V=%d N=%d)", a->B,
          a->T, a->H, a->K, a->V, a->N);
  REQUIRE(a->H <= MAX_GRID_YZ, GDN_ERR_UNSUPPORTED, "H (%d) must be at most %d", a->H,
          MAX_GRID_YZ);
  REQUIRE(a->K <= KMAX, GDN_ERR_UNSUPPORTED, "K=%d exceeds %d", a->K, KMAX);
  REQUIRE(a->K % 8 == 0 && a->V % 8 == 0, GDN_ERR_UNSUPPORTED,
          "K (%d) and V (%d) must be multiples of 8", a->K, a->V);
  REQUIRE(a->N <= MAX_GRID_YZ, GDN_ERR_UNSUPPORTED, "N (%d) must be at most %d", a->N,
          MAX_GRID_YZ);
  REQUIRE(a->chunk_size == BT, GDN_ERR_UNSUPPORTED, "chunk_size must be %d (got %d)", BT,
          a->chunk_size);
  REQUIRE(a->split_size >= 0 && a->split_size % BT == 0, GDN_ERR_INVALID_ARG,
          "split_size (%d) must be 0 or a positive multiple of %d", a->split_size, BT);
  const int split = a->split_size > 0 ? a->split_size / BT : 1;
  REQUIRE(a->state_v_first == 0 || a->state_v_first == 1, GDN_ERR_INVALID_ARG,
          "state_v_first must be 0 or 1");
  if (a->cu_seqlens == nullptr) {
    REQUIRE(a->N == a->B, GDN_ERR_INVALID_ARG, "without cu_seqlens N (%d) must equal B (%d)",
            a->N, a->B);
  } else {
    REQUIRE(a->B == 1, GDN_ERR_INVALID_ARG, "with cu_seqlens B must be 1 (got %d)", a->B);
  }
  if (a->T > 0) {
    REQUIRE_PTR(a->k, "k");
    REQUIRE_PTR(a->v, "v");
  }
  if (a->gate == GDN_GATE_NONE) {
    REQUIRE(a->gate_values == nullptr, GDN_ERR_INVALID_ARG, "gate_values given without a gate");
  } else if (a->T > 0 || a->gate == GDN_GATE_G_GAMMA) {
    REQUIRE_PTR(a->gate_values, "gate_values");
  }
  REQUIRE_OPT_PTR(a->h0, "h0");
  REQUIRE_OPT_PTR(a->ht, "ht");
  REQUIRE_OPT_PTR(a->cu_seqlens, "cu_seqlens");
  if (a->hs != nullptr) {
    REQUIRE_PTR(a->hs, "hs");
    REQUIRE(a->hs_dtype == GDN_F32 || a->hs_dtype == GDN_BF16, GDN_ERR_INVALID_ARG,
            "hs_dtype %d is not GDN_F32/GDN_BF16", a->hs_dtype);
    if (a->cu_seqlens == nullptr) {
      const long long split_tokens = (long long)BT * split;
      const long long need = (long long)a->B * ((a->T + split_tokens - 1) / split_tokens);
      REQUIRE(a->num_chunks >= need, GDN_ERR_INVALID_ARG,
              "hs holds %lld chunks, %lld needed", (long long)a->num_chunks, need);
    }
  }
  StateParams p{};
  p.k = a->k; p.v = a->v; p.gate = a->gate; p.gate_values = a->gate_values;
  p.h0 = a->h0; p.ht = a->ht; p.hs = a->hs; p.hs_bf16 = a->hs_dtype == GDN_BF16;
  p.cu_seqlens = a->cu_seqlens;
  p.B = a->B; p.T = a->T; p.H = a->H; p.K = a->K; p.V = a->V; p.N = a->N;
  p.HG = a->H;
  p.num_chunks = a->hs ? a->num_chunks : 0;
  p.reverse = 0;
  p.scale = 1.f;
  p.split = split;
  p.v_first = a->state_v_first;
  p.err = device_error_word();
  if (p.err == nullptr) return cuda_status(cudaGetLastError(), "device error word");
  return cuda_status(launch_state_pass(p, a->dtype == GDN_BF16,
                                       reinterpret_cast<cudaStream_t>(stream)),
                     "state pass launch");
}

gdn_status_t gdn_chunk_state_bwd(const gdn_state_bwd_args *a, gdn_stream_t stream) {
  g_msg[0] = '\0';
  if (a == nullptr) return fail(GDN_ERR_INVALID_ARG, "args is NULL");
  REQUIRE(a->dtype == GDN_F32 || a->dtype == GDN_BF16, GDN_ERR_INVALID_ARG,
          "dtype %d is not GDN_F32/GDN_BF16", a->dtype);
  REQUIRE(a->gate >= GDN_GATE_NONE && a->gate <= GDN_GATE_GV, GDN_ERR_INVALID_ARG,
          "gate %d is not a gdn_gate_kind_t", a->gate);
  REQUIRE(a->B >= 1 && a->T >= 0 && a->HQ >= 1 && a->H >= 1 && a->K >= 1 && a->V >= 1 &&
              a->N >= 1,
          GDN_ERR_INVALID_ARG, "sizes must be positive (B=%d T=%d HQ=%d H=%d K=%d V=%d N=%d)",
          a->B, a->T, a->HQ, a->H, a->K, a->V, a->N);
  REQUIRE(a->HQ % a->H == 0, GDN_ERR_UNSUPPORTED, "HQ (%d) must be a multiple of H (%d)", a->HQ,
          a->H);
  REQUIRE(a->HQ <= MAX_GRID_YZ, GDN_ERR_UNSUPPORTED, "HQ (%d) must be at most %d", a->HQ,
          MAX_GRID_YZ);
  REQUIRE(a->K <= KMAX, GDN_ERR_UNSUPPORTED, "K=%d exceeds %d", a->K, KMAX);
  REQUIRE(a->K % 8 == 0 && a->V % 8 == 0, GDN_ERR_UNSUPPORTED,
          "K (%d) and V (%d) must be multiples of 8", a->K, a->V);
  REQUIRE(a->N <= MAX_GRID_YZ, GDN_ERR_UNSUPPORTED, "N (%d) must be at most %d", a->N,
          MAX_GRID_YZ);
  REQUIRE(a->chunk_size == BT, GDN_ERR_UNSUPPORTED, "chunk_size must be %d (got %d)", BT,
          a->chunk_size);
  REQUIRE(a->split_size >= 0 && a->split_size % BT == 0, GDN_ERR_INVALID_ARG,
          "split_size (%d) must be 0 or a positive multiple of %d", a->split_size, BT);
  const int split = a->split_size > 0 ? a->split_size / BT : 1;
  REQUIRE(a->state_v_first == 0 || a->state_v_first == 1, GDN_ERR_INVALID_ARG,
          "state_v_first must be 0 or 1");
  REQUIRE(isfinite(a->scale), GDN_ERR_INVALID_ARG, "scale must be finite");
  if (a->cu_seqlens == nullptr) {
    REQUIRE(a->N == a->B, GDN_ERR_INVALID_ARG, "without cu_seqlens N (%d) must equal B (%d)",
            a->N, a->B);
  } else {
    REQUIRE(a->B == 1, GDN_ERR_INVALID_ARG, "with cu_seqlens B must be 1 (got %d)", a->B);
  }
  if (a->T > 0) {
    REQUIRE_PTR(a->q, "q");
    REQUIRE_PTR(a->do_, "do");
  }
  if (a->gate == GDN_GATE_NONE) {
    REQUIRE(a->gate_values == nullptr, GDN_ERR_INVALID_ARG, "gate_values given without a gate");
  } else if (a->T > 0 || a->gate == GDN_GATE_G_GAMMA) {
    REQUIRE_PTR(a->gate_values, "gate_values");
  }
  REQUIRE_OPT_PTR(a->dht, "dht");
  REQUIRE_OPT_PTR(a->dh0, "dh0");
  REQUIRE_OPT_PTR(a->cu_seqlens, "cu_seqlens");
  if (a->dh != nullptr) {
    REQUIRE_PTR(a->dh, "dh");
    REQUIRE(a->dh_dtype == GDN_F32 || a->dh_dtype == GDN_BF16, GDN_ERR_INVALID_ARG,
            "dh_dtype %d is not GDN_F32/GDN_BF16", a->dh_dtype);
    if (a->cu_seqlens == nullptr) {
      const long long split_tokens = (long long)BT * split;
      const long long need = (long long)a->B * ((a->T + split_tokens - 1) / split_tokens);
      REQUIRE(a->num_chunks >= need, GDN_ERR_INVALID_ARG,
              "dh holds %lld chunks, %lld needed", (long long)a->num_chunks, need);
    }
  }
  StateParams p{};
  p.k = a->q; p.v = a->do_; p.gate = a->gate; p.gate_values = a->gate_values;
  p.h0 = a->dht; p.ht = a->dh0; p.hs = a->dh; p.hs_bf16 = a->dh_dtype == GDN_BF16;
  p.cu_seqlens = a->cu_seqlens;
  p.B = a->B; p.T = a->T; p.H = a->HQ; p.K = a->K; p.V = a->V; p.N = a->N;
  p.HG = a->H;
  p.num_chunks = a->dh ? a->num_chunks : 0;
  p.reverse = 1;
  p.scale = a->scale > 0.f ? a->scale : 1.0f / sqrtf((float)a->K);
  p.split = split;
  p.v_first = a->state_v_first;
  p.err = device_error_word();
  if (p.err == nullptr) return cuda_status(cudaGetLastError(), "device error word");
  return cuda_status(launch_state_pass(p, a->dtype == GDN_BF16,
                                       reinterpret_cast<cudaStream_t>(stream)),
                     "state backward launch");
}

gdn_status_t gdn_decode(const gdn_decode_args *a, gdn_stream_t stream) {
  g_msg[0] = '\0';
  if (a == nullptr) return fail(GDN_ERR_INVALID_ARG, "args is NULL");
  REQUIRE(a->B >= 1 && a->H >= 1 && a->HV >= 1 && a->pool >= 1, GDN_ERR_INVALID_ARG,
          "sizes must be positive (B=%d H=%d HV=%d pool=%d)", a->B, a->H, a->HV, a->pool);
  REQUIRE(a->T >= 1 && a->T <= 4, GDN_ERR_UNSUPPORTED, "T must be 1..4 (got %d)", a->T);
  REQUIRE(a->K == 128 && a->V == 128, GDN_ERR_UNSUPPORTED, "decode needs K = V = 128 (got %d, %d)",
          a->K, a->V);
  REQUIRE(a->HV % a->H == 0, GDN_ERR_UNSUPPORTED, "HV (%d) must be a multiple of H (%d)", a->HV, a->H);
  REQUIRE(a->slot_indices != nullptr || a->pool >= a->B, GDN_ERR_INVALID_ARG,
          "identity slots need pool (%d) >= B (%d)", a->pool, a->B);
  REQUIRE(a->use_qk_l2norm == 0 || a->use_qk_l2norm == 1, GDN_ERR_INVALID_ARG,
          "use_qk_l2norm must be 0 or 1");
  REQUIRE(a->o_fp32 == 0 || a->o_fp32 == 1, GDN_ERR_INVALID_ARG, "o_fp32 must be 0 or 1");
  REQUIRE(isfinite(a->scale) && isfinite(a->softplus_beta) && isfinite(a->softplus_threshold) &&
              isfinite(a->eps),
          GDN_ERR_INVALID_ARG, "scalar arguments must be finite");
  REQUIRE_PTR(a->q, "q");
  REQUIRE_PTR(a->k, "k");
  REQUIRE_PTR(a->v, "v");
  REQUIRE_PTR(a->a, "a");
  REQUIRE_PTR(a->b, "b");
  REQUIRE_PTR(a->A_log, "A_log");
  REQUIRE_PTR(a->dt_bias, "dt_bias");
  REQUIRE_PTR(a->state, "state");
  REQUIRE_PTR(a->o, "o");
  REQUIRE_OPT_PTR(a->slot_indices, "slot_indices");
  REQUIRE_OPT_PTR(a->new_state_f32, "new_state_f32");
  DecodeParams p{};
  p.q = a->q; p.k = a->k; p.v = a->v; p.a = a->a; p.b = a->b;
  p.A_log = a->A_log; p.dt_bias = a->dt_bias; p.state = a->state;
  p.slot_indices = a->slot_indices; p.o = a->o; p.state_f32 = a->new_state_f32;
  p.o_f32 = a->o_fp32;
  p.B = a->B; p.T = a->T; p.H = a->H; p.HV = a->HV; p.K = a->K; p.V = a->V; p.pool = a->pool;
  p.use_qk_l2norm = a->use_qk_l2norm;
  p.scale = a->scale > 0.f ? a->scale : 1.0f / sqrtf((float)a->K);
  p.softplus_beta = a->softplus_beta > 0.f ? a->softplus_beta : 1.0f;
  p.softplus_threshold = a->softplus_threshold;
  p.eps = a->eps >= 0.f ? a->eps : 1e-6f;
  p.err = device_error_word();
  if (p.err == nullptr) return cuda_status(cudaGetLastError(), "device error word");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return cuda_status(launch_decode(p, s), "decode launch");
}

gdn_status_t gdn_check_device_error(gdn_stream_t stream, int32_t *code) {
  g_msg[0] = '\0';
  if (code == nullptr) return fail(GDN_ERR_INVALID_ARG, "code is NULL");
  *code = GDN_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  gdn_status_t st = cuda_status(cudaStreamSynchronize(s), "stream synchronize");
  if (st != GDN_OK) return st;
  int host = 0;
  const int zero = 0;
  st = cuda_status(cudaMemcpyFromSymbol(&host, g_error_word, sizeof(int)), "read error word");
  if (st != GDN_OK) return st;
  st = cuda_status(cudaMemcpyToSymbol(g_error_word, &zero, sizeof(int)), "clear error word");
  if (st != GDN_OK) return st;
  *code = host;
  return GDN_OK;
}

}  // extern "C"
