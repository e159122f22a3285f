// Internal launch interface between the C entry points (gdn_abi.cu) and the
// kernel translation units.  Plain host types only.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

// One chunked-forward problem, already validated.  `H` counts value heads and
// `Hk` key/query heads for both gate kinds.
struct ChunkParams {
  const void *q, *k, *v;
  const float *g, *beta, *h0;
  float *ht;
  void *o;
  const int32_t *cu_seqlens;
  int *err;
  int B, T, H, Hk, K, V, N;
  int g_is_cumsum;
  int v_first;                // h0, ht as [V, K] instead of [K, V]
  int o_f32;                  // o written as float32 (else in the input dtype)
  int segments;               // state pass segments: 0 = choose, 1 = none, >= 2
  float scale;
};

struct DecodeParams {
  const void *q, *k, *v, *a, *b;
  const float *A_log, *dt_bias;
  void *state;
  const int32_t *slot_indices;
  void *o;
  float *state_f32;           // updated states in fp32 [B, HV, V, K] or NULL
  int *err;
  int B, T, H, HV, K, V, pool;
  int use_qk_l2norm;
  int o_f32;                  // o written as float32 (else bf16)
  float scale, softplus_beta, softplus_threshold, eps;
};

// One chunk-state-pass problem (gated linear attention), already validated.
struct StateParams {
  const void *k, *v;
  int gate;                   // gdn_gate_kind_t
  const float *gate_values;
  const float *h0;
  float *ht;
  void *hs;                   // chunk-start states or NULL
  int hs_bf16;
  const int32_t *cu_seqlens;
  int *err;
  int B, T, H, K, V, N;
  int HG;                     // gate heads (H % HG == 0; head h uses gate head h / (H / HG))
  long long num_chunks;       // capacity of hs in chunks
  // Backward (dh) pass: chunks from last to first, k = q scaled by `scale`,
  // v = do, gate factors taken from the chunk start instead of its end,
  // h0 = dht, ht = dh0, hs = dh (the gradient at the end of every chunk).
  int reverse;
  float scale;
  int split;                  // chunks per stored state (>= 1): hs holds chunks 0, split, ..
  int v_first;                // h0, ht, hs as [V, K] instead of [K, V]
};

// Each launcher enqueues its kernel(s) and returns the launch status.
cudaError_t launch_chunk_simt(const ChunkParams &p, bool bf16, bool per_channel_gate,
                              cudaStream_t stream);
cudaError_t launch_decode(const DecodeParams &p, cudaStream_t stream);
cudaError_t launch_state_pass(const StateParams &p, bool bf16, cudaStream_t stream);
// The state pass on tcgen05 + TMA (bf16, K = 128, V % 32 == 0, gates whose
// chunk factors ride on the value side): whether it serves p, and its launch.
bool state_pass_tc5_supported(const StateParams &p, bool bf16);
cudaError_t launch_state_pass_tc5(const StateParams &p, cudaStream_t stream);
// The decode step on the warp-level tensor cores (K = V = 128).
cudaError_t launch_decode_tc(const DecodeParams &p, cudaStream_t stream);

// Tensor-core chunked forward (bf16, K = 128, V % 32 == 0): whether it serves
// these arguments, the workspace it needs, and the launch.
bool chunk_tc_supported(const ChunkParams &p, bool bf16);
size_t chunk_tc_workspace(const ChunkParams &p, bool per_channel_gate);
cudaError_t launch_chunk_tc(const ChunkParams &p, bool per_channel_gate, void *workspace,
                            cudaStream_t stream);
// Segments per sequence the tensor-core state pass uses for these arguments.
int chunk_tc_segments(const ChunkParams &p);

// The checks of gdn_chunk_fwd that read only sizes, dtype and flags (no
// pointer is dereferenced; cu_seqlens only counts as given or NULL).
gdn_status_t check_gdn_chunk_sizes(const gdn_chunk_args &a);

// Record `msg` as the calling thread's last host-side error; returns `st`.
gdn_status_t set_host_error(gdn_status_t st, const char *msg);

}  // namespace gdn
