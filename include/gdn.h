/*
 * gdn.h - C interface of the GB300 (sm_103a) gated delta-rule library.
 *
 * The method: a linear-attention state S (V x K per value head) evolves per
 * token t as
 *     S_t = S_{t-1} * D_t * (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
 *     o_t = scale * S_t q_t,
 * with D_t = exp(g_t) * I (GDN, one log-gate per token and head) or
 * D_t = diag(exp(g_t[0..K))) (KDA, one log-gate per token, head and key
 * channel).  The token form (decay, pred = S k, delta = beta (v - pred),
 * S += delta k^T, o = S q) is the one of the FlashInfer page
 * gdn_decode_bf16_state.py (per-token helpers); the chunked form with BT = 64
 * token chunks follows the sglang page fla/chunk_fwd.py (fused KK^T + solve
 * kernel, Steps 1-5, and chunk_gated_delta_rule_fwd_intra), the KDA page
 * _fla/ops/common/chunk_h.py (chunk_fwd_kernel_h, chunk_fwd_h) and the vLLM
 * kimi_k3 kda/chunk_intra page (chunk_kda_fwd_kernel_inter_solve_fused).
 *
 * Conventions shared by every entry point
 *  - Memory: every tensor pointer is a DEVICE pointer owned by the caller.
 *    The library never allocates, frees or retains device memory; outputs are
 *    written in place.  Tensors are dense, row-major, last index fastest, in
 *    the layouts given per argument.  Every tensor pointer must be 16-byte
 *    aligned (GDN_ERR_MISALIGNED otherwise).
 *  - Streams: work is enqueued on the caller's stream (NULL = the legacy
 *    default stream) and the call returns without waiting for it.
 *  - Errors: every call returns a gdn_status_t and never throws, exits or
 *    prints.  Argument errors are found on the host before anything is
 *    enqueued (nothing is written then).  Errors that only the device can see
 *    (bad cu_seqlens, bad slot index, a bounded wait that ran out) are
 *    recorded in a device-side error word, which gdn_check_device_error()
 *    reads and clears.  gdn_last_error_message() describes the last host-side
 *    failure of the calling thread.
 *  - Log-gates are natural logarithms (exp, not exp2).
 */
#ifndef GDN_GB300_H
#define GDN_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream. */
typedef struct CUstream_st *gdn_stream_t;

typedef enum gdn_status {
  GDN_OK = 0,
  GDN_ERR_INVALID_ARG = 1,  /* NULL required pointer, bad size or flag    */
  GDN_ERR_UNSUPPORTED = 2,  /* valid request this library does not serve */
  GDN_ERR_MISALIGNED = 3,   /* a tensor pointer is not 16-byte aligned    */
  GDN_ERR_WORKSPACE = 4,    /* workspace smaller than *_workspace_size     */
  GDN_ERR_CUDA = 5,         /* a CUDA runtime call failed                  */
  GDN_ERR_TIMEOUT = 6,      /* device: a bounded wait gave up              */
  GDN_ERR_BAD_SEQLENS = 7,  /* device: cu_seqlens not rising from 0 to T   */
  GDN_ERR_BAD_SLOT = 8,     /* device: a slot index outside [0, pool)      */
  GDN_ERR_BOUNDS = 9        /* device, checked builds only: an index range a
                               kernel derived falls outside its tensor; the
                               CTA skips its work                          */
} gdn_status_t;

typedef enum gdn_dtype {
  GDN_F32 = 0,   /* float32 q, k, v, o  */
  GDN_BF16 = 1   /* bfloat16 q, k, v, o */
} gdn_dtype_t;

/*
 * Chunked forward with one scalar log-gate per token and value head (GDN).
 * Shapes follow chunk_gated_delta_rule_fwd_intra (sglang fla/chunk_fwd.py)
 * and chunk_fwd_h (KDA _fla/ops/common/chunk_h.py):
 *   q, k   [B, T, Hg, K]  dtype       key/query heads; value head h reads
 *                                     key head h / (H / Hg)
 *   v, o   [B, T, H, V]   dtype       o is written, in float32 instead
 *                                     when o_fp32 = 1 (the same result
 *                                     before its rounding to dtype: with
 *                                     o_fp32 = 0 and bf16, o is exactly the
 *                                     round-to-nearest-even of that value)
 *   g      [B, T, H]      float32     natural-log gate per token; with
 *                                     g_is_cumsum = 1 it is instead the
 *                                     inclusive cumulative sum inside each
 *                                     64-token chunk (chunks counted from
 *                                     each sequence's first token)
 *   beta   [B, T, H]      float32
 *   h0     [N, H, K, V]   float32     initial state h = S^T, NULL = zeros
 *   ht     [N, H, K, V]   float32     final state, NULL = not returned
 *   state_v_first = 1     h0 and ht hold every state transposed,
 *                                     [N, H, V, K] (S itself; the chunk_h
 *                                     page's state_v_first); 0 = [K, V]
 *   cu_seqlens [N + 1]    int32       NULL: N = B sequences of T tokens.
 *                                     Else B must be 1 and sequence n is
 *                                     tokens cu_seqlens[n] .. cu_seqlens[n+1]
 *                                     (0 = cu_seqlens[0] <= ... <= cu_seqlens[N]
 *                                     = T, checked on the device)
 * Limits: 1 <= K <= 128, V >= 1, chunk_size == 64, H % Hg == 0, N and H at
 * most 65535 (GDN_ERR_UNSUPPORTED otherwise).  With T == 0
 * nothing per token is read or written, so q, k, v, g, beta and o may be NULL
 * (ht = h0, or zeros).
 * scale <= 0 selects 1/sqrt(K).
 * Workspace: bf16 inputs with K == 128 and V a multiple of 32 up to 128 run on
 * the tensor cores and need `workspace` (device, 256-byte aligned,
 * caller-owned, contents irrelevant before and after the call) of at least
 * gdn_chunk_workspace_size() bytes, else GDN_ERR_WORKSPACE.  Every other
 * shape runs the exact fp32 CUDA-core kernel and needs none.
 * Segment-parallel state pass (tensor-core path; `segments`): the chunk
 * recurrence h <- M_c h + B_c is affine in h, so with S >= 2 every sequence
 * is cut into S runs of ceil(chunks / S) chunks that are all processed at
 * once -- each from a zero state and on the identity, which gives the run's
 * map (M, B) -- then combined in order (start of run s + 1 = M start_s + B)
 * and run again from their true starts, writing o.  The sequential part
 * shrinks from `chunks` to about 2 chunks / S steps, at about three times
 * the work; it pays when the sequences' own chains (V / 32 per head and
 * sequence) leave most SMs idle.  0 lets the library choose (1 unless that
 * holds); the fp32 CUDA-core kernel ignores it.  1 <= segments <= 64 and
 * N * segments <= 65535, else GDN_ERR_UNSUPPORTED.
 */
typedef struct gdn_chunk_args {
  int32_t dtype;               /* gdn_dtype_t of q, k, v, o */
  const void *q, *k, *v;
  const float *g, *beta;
  const float *h0;
  float *ht;
  void *o;
  const int32_t *cu_seqlens;
  int32_t B, T, H, Hg, K, V, N;
  int32_t chunk_size;
  int32_t g_is_cumsum;
  int32_t state_v_first;       /* 1: h0, ht are [N, H, V, K] instead of [N, H, K, V] */
  int32_t o_fp32;              /* 1: o is float32 whatever dtype is; 0: o has dtype */
  int32_t segments;            /* state pass: 0 = library's choice, 1 = one chain per
                                  sequence, 2..64 = segment-parallel (see above) */
  float scale;
  void *workspace;
  size_t workspace_bytes;
} gdn_chunk_args;

/* Bytes of workspace gdn_chunk_fwd needs for these arguments (0 when the
 * CUDA-core kernel serves them).  Reads only sizes, dtype and whether
 * cu_seqlens is NULL. */
gdn_status_t gdn_chunk_workspace_size(const gdn_chunk_args *args, size_t *bytes);

/* The segment count gdn_chunk_fwd would use for the state pass with these
 * arguments (args->segments, or the library's choice when it is 0; 1 when
 * the exact fp32 CUDA-core kernel serves them).  Reads only sizes, dtype,
 * segments and whether cu_seqlens is NULL. */
gdn_status_t gdn_chunk_segment_count(const gdn_chunk_args *args, int32_t *segments);

/* Enqueue the GDN chunked forward (gate cumsum, intra-chunk (I+A)^-1 with the
 * WY vectors w, u, the sequential inter-chunk state pass and the output) on
 * `stream`.  Writes o and, if given, ht. */
gdn_status_t gdn_chunk_fwd(const gdn_chunk_args *args, gdn_stream_t stream);

/*
 * The same forward end to end from HOST memory: q, k, v, g, beta, h0,
 * cu_seqlens are read from and o, ht written to host buffers (pinned memory
 * lets the copies run asynchronously and at full speed; pageable memory is
 * accepted).  Shapes, limits and NULL rules are those of gdn_chunk_fwd.
 * `workspace` is a DEVICE buffer on the current device, 256-byte aligned,
 * caller-owned, of at least gdn_chunk_host_workspace_size() bytes: it takes
 * device copies of the inputs and outputs and the kernels' scratch.
 * The call enqueues everything behind the work already on `stream` and
 * returns; o and ht are complete in host memory when `stream` has completed
 * (e.g. cudaStreamSynchronize).  Host buffers must stay valid and unchanged
 * until then.  Inside, the problem is cut into pieces of whole 64-token
 * chunks along time (sequences of more than 704 tokens; the pieces shrink
 * towards the end) or into ranges of whole sequences, and each piece's host->device copies, kernels
 * and device->host copies run on an internal copy-in stream, `stream` and an
 * internal copy-out stream, so the copies of one piece overlap the kernels of
 * its neighbours.  The state pass runs one chain per sequence (`segments`
 * is ignored), and the results equal gdn_chunk_fwd's with segments = 1 bit
 * for bit: a time cut hands the fp32 state of the chunkwise recurrence (Gated
 * Delta Networks, section 3) from one piece to the next exactly as the
 * kernels carry it between chunks.
 * Errors: argument errors as gdn_chunk_fwd, plus GDN_ERR_INVALID_ARG when an
 * input or output pointer is device memory, GDN_ERR_WORKSPACE when the
 * workspace is missing, too small or not device memory, GDN_ERR_BAD_SEQLENS
 * (returned by the call itself) when cu_seqlens does not rise from 0 to T.
 * With cu_seqlens the call copies offsets rebased per piece from pageable
 * memory, so it cannot be captured into a CUDA graph; without, it can.
 * Calls from several host threads are serialised inside the library.
 */
gdn_status_t gdn_chunk_fwd_host(const gdn_chunk_args *args, gdn_stream_t stream);

/*
 * Chunk state pass of gated linear attention (KDA _fla/ops/common/chunk_h.py:
 * chunk_fwd_kernel_h / chunk_fwd_h, "h += k^T v" with an optional decay).
 * For every sequence n and head h the state h [K, V] starts at h0 (or zeros)
 * and takes, token by token,
 *     h <- Dk_t h Dv_t + k_t v_t^T
 * where the decay depends on `gate` (natural-log gates):
 *   GDN_GATE_NONE      Dk = Dv = I                       gate_values NULL
 *   GDN_GATE_G         Dk = e^{r_t} I                    gate_values [B,T,H]
 *   GDN_GATE_G_GAMMA   Dk = e^{gamma_h} I, every token   gate_values [H]
 *   GDN_GATE_GK        Dk = diag(e^{r_t[:]}) (keys)      gate_values [B,T,H,K]
 *   GDN_GATE_GV        Dv = diag(e^{r_t[:]}) (values)    gate_values [B,T,H,V]
 * The per-token gates are given as the page's kernel takes them: inclusive
 * cumulative sums of r_t inside each 64-token chunk (chunks counted from each
 * sequence's first token); g_gamma is the per-token rate itself.
 *   k [B,T,H,K], v [B,T,H,V]   dtype (GDN_F32 or GDN_BF16)
 *   h0, ht [N,H,K,V]           float32, NULL = zeros / not returned
 *   hs [C,H,K,V]               hs_dtype (GDN_F32 or GDN_BF16): the state at the
 *                              start of every split (split_size tokens, a
 *                              multiple of 64; 0 = 64: every chunk), sequence
 *                              after sequence (sequence n contributes
 *                              ceil(len_n / split_size) entries; B equal
 *                              sequences: [B, ceil(T/split_size), ...]);
 *                              NULL = not returned; num_chunks = C, its capacity
 *   cu_seqlens [N + 1] int32   as gdn_chunk_fwd (device memory; checked on the
 *                              device, GDN_ERR_BAD_SEQLENS also when the chunks
 *                              do not fit num_chunks)
 *   state_v_first = 1          every state tensor (h0, ht, hs) holds each
 *                              state transposed, [V, K] (the page's
 *                              state_v_first); the arithmetic is unchanged
 * Limits: 1 <= K <= 128, K and V multiples of 8, chunk_size == 64, N and H at
 * most 65535.
 * Arithmetic in fp32 (bf16 inputs are widened).  Nothing is allocated; no
 * workspace.
 */
typedef enum gdn_gate_kind {
  GDN_GATE_NONE = 0,
  GDN_GATE_G = 1,
  GDN_GATE_G_GAMMA = 2,
  GDN_GATE_GK = 3,
  GDN_GATE_GV = 4
} gdn_gate_kind_t;

typedef struct gdn_state_args {
  int32_t dtype;               /* gdn_dtype_t of k, v */
  const void *k, *v;
  int32_t gate;                /* gdn_gate_kind_t */
  const float *gate_values;
  const float *h0;
  float *ht;
  void *hs;
  int32_t hs_dtype;            /* gdn_dtype_t of hs */
  const int32_t *cu_seqlens;
  int32_t B, T, H, K, V, N;
  int32_t chunk_size;
  int64_t num_chunks;
  int32_t split_size;          /* tokens between stored states; 0 = chunk_size */
  int32_t state_v_first;       /* 1: h0, ht, hs are [.., V, K] instead of [.., K, V] */
} gdn_state_args;

/* Enqueue the chunk state pass on `stream`. */
gdn_status_t gdn_chunk_state_fwd(const gdn_state_args *args, gdn_stream_t stream);

/*
 * Backward state pass (KDA _fla/ops/common/chunk_h.py: chunk_bwd_kernel_dh /
 * chunk_bwd_dh): for the recurrence of gdn_chunk_state_fwd with outputs
 * o_t = scale S_t^T q_t (S_t the state after token t), the gradient
 * G = dL/dS of a loss with dL/do_t = do_t, going from the last token back:
 *     G <- G + scale q_t do_t^T,   then   G <- decay_t^T(G)
 * starting from dht (or zeros).  Per query head hq (gate head hq / (HQ / H)):
 *   q [B,T,HQ,K], do [B,T,HQ,V]  dtype (GDN_F32 or GDN_BF16)
 *   gate, gate_values            as gdn_chunk_state_fwd, with H heads
 *   dht, dh0 [N,HQ,K,V]          float32, NULL = zeros / not returned
 *   dh [C,HQ,K,V]                dh_dtype: the gradient with respect to the
 *                                state at the end of the first chunk of every
 *                                split (before that chunk's tokens are folded
 *                                in; split_size as gdn_chunk_state_fwd, 0 = every
 *                                chunk), sequence after sequence; NULL = not
 *                                returned; num_chunks = C
 *   scale                        <= 0 selects 1/sqrt(K)
 * Limits, errors and the rest as gdn_chunk_state_fwd; HQ % H == 0.
 */
typedef struct gdn_state_bwd_args {
  int32_t dtype;               /* gdn_dtype_t of q, do */
  const void *q, *do_;
  int32_t gate;                /* gdn_gate_kind_t */
  const float *gate_values;
  const float *dht;
  float *dh0;
  void *dh;
  int32_t dh_dtype;            /* gdn_dtype_t of dh */
  const int32_t *cu_seqlens;
  int32_t B, T, HQ, H, K, V, N;
  int32_t chunk_size;
  int64_t num_chunks;
  float scale;
  int32_t split_size;          /* tokens between stored gradients; 0 = chunk_size */
  int32_t state_v_first;       /* 1: dht, dh0, dh are [.., V, K] instead of [.., K, V] */
} gdn_state_bwd_args;

/* Enqueue the backward state pass on `stream`. */
gdn_status_t gdn_chunk_state_bwd(const gdn_state_bwd_args *args, gdn_stream_t stream);

/* Bytes of device workspace gdn_chunk_fwd_host needs for these arguments.
 * Reads sizes, dtype and, when given, the host array cu_seqlens. */
gdn_status_t gdn_chunk_host_workspace_size(const gdn_chunk_args *args, size_t *bytes);

/*
 * Chunked forward with one log-gate per token, value head and key channel
 * (KDA).  Shapes follow chunk_kda_fwd_kernel_inter_solve_fused (vLLM kimi_k3
 * kda/chunk_intra page):
 *   q, k   [B, T, H, K]   dtype       value head hv reads key head hv / (HV / H)
 *   v, o   [B, T, HV, V]  dtype       (o float32 with o_fp32 = 1, as for GDN)
 *   g      [B, T, HV, K]  float32     chunk-local inclusive cumulative sum of
 *                                     the per-channel log-gates when
 *                                     g_is_cumsum = 1 (as that kernel takes
 *                                     it), raw per-token log-gates when 0
 *   beta   [B, T, HV]     float32
 *   h0, ht [N, HV, K, V]  float32     as for GDN ([N, HV, V, K] with
 *                                     state_v_first = 1)
 *   cu_seqlens            as for GDN
 * Limits: 1 <= K <= 128, V >= 1, chunk_size == 64, HV % H == 0, N and HV at
 * most 65535.  With T == 0
 * q, k, v, g, beta and o may be NULL (ht = h0, or zeros).
 * Workspace: as for GDN (tensor cores for bf16, K == 128, V % 32 == 0,
 * V <= 128; kda_chunk_workspace_size() bytes).
 */
typedef struct kda_chunk_args {
  int32_t dtype;
  const void *q, *k, *v;
  const float *g, *beta;
  const float *h0;
  float *ht;
  void *o;
  const int32_t *cu_seqlens;
  int32_t B, T, H, HV, K, V, N;
  int32_t chunk_size;
  int32_t g_is_cumsum;
  int32_t state_v_first;       /* 1: h0, ht are [N, HV, V, K] instead of [N, HV, K, V] */
  int32_t o_fp32;              /* 1: o is float32 whatever dtype is; 0: o has dtype */
  int32_t segments;            /* as gdn_chunk_args.segments */
  float scale;
  void *workspace;
  size_t workspace_bytes;
} kda_chunk_args;

gdn_status_t kda_chunk_workspace_size(const kda_chunk_args *args, size_t *bytes);
gdn_status_t kda_chunk_fwd(const kda_chunk_args *args, gdn_stream_t stream);

/*
 * Decode step for T = 1..4 new tokens per batch entry against a pooled
 * bfloat16 state, updated in place (FlashInfer gdn_decode_bf16_state.py,
 * public gated_delta_rule and compute_single_gate):
 *   q, k     [B, T, H, K]     bf16
 *   v        [B, T, HV, V]    bf16      value head hv reads key head hv/(HV/H)
 *   a, b     [B, T, HV]       bf16      gate inputs
 *   A_log    [HV]             float32
 *   dt_bias  [HV]             float32
 *   state    [pool, HV, V, K] bf16      K fastest; slot slot_indices[b] is
 *                                       read, advanced by the T tokens in
 *                                       float32 and written back once
 *                                       (round to nearest even)
 *   slot_indices [B]          int32     NULL = identity (needs pool >= B).
 *                                       Slots must be distinct; a slot
 *                                       outside [0, pool) records
 *                                       GDN_ERR_BAD_SLOT and that entry's o
 *                                       is written as zeros.
 *   o        [B, T, HV, V]    bf16      (float32 when o_fp32 = 1: the same
 *                                       value before its rounding to bf16)
 *   new_state_f32 [B, HV, V, K] float32 or NULL: when given, entry b's
 *                                       updated state in float32, the value
 *                                       whose round-to-nearest-even the pool
 *                                       receives (NULL = not written)
 * Per token: g = -exp(A_log) * softplus(a + dt_bias) with
 *   softplus(x) = log(1 + exp(beta_sp x)) / beta_sp if beta_sp x <= threshold
 *   else x; beta = sigmoid(b); if use_qk_l2norm, q and k are divided by
 *   sqrt(sum(x^2) + eps); q is multiplied by scale.
 * Limits: K == V == 128, 1 <= T <= 4, HV % H == 0.  scale <= 0 selects
 * 1/sqrt(K); softplus_beta <= 0 selects 1; eps < 0 selects 1e-6.
 */
typedef struct gdn_decode_args {
  const void *q, *k, *v;
  const void *a, *b;
  const float *A_log, *dt_bias;
  void *state;
  const int32_t *slot_indices;
  void *o;
  float *new_state_f32;
  int32_t B, T, H, HV, K, V, pool;
  int32_t use_qk_l2norm;
  int32_t o_fp32;
  float scale, softplus_beta, softplus_threshold, eps;
} gdn_decode_args;

gdn_status_t gdn_decode(const gdn_decode_args *args, gdn_stream_t stream);

/*
 * GDN chunked forward without a workspace, for callers that cannot allocate
 * device memory (a host runtime that owns a fixed device-memory budget and
 * forbids cudaMalloc from plugins, or a latency-critical loop that must not
 * hit cudaMalloc's implicit synchronisation).  The pages have no counterpart
 * to this entry point; it is a convenience of this library.
 * Same arguments and results as gdn_chunk_fwd; `workspace` and
 * `workspace_bytes` are ignored.  Scratch comes from a fixed device array of
 * gdn_noalloc_scratch_bytes() bytes (32 MiB) that every GPU loading the
 * library holds until the process exits; a problem whose
 * gdn_chunk_workspace_size exceeds it returns GDN_ERR_WORKSPACE and enqueues
 * nothing.  All calls on a device share that array: calls that may overlap
 * on the GPU (e.g. on different streams) race and must be ordered by the
 * caller.  The first call on each device resolves the array's device address
 * (with that device current), so make it before any stream capture.
 */
gdn_status_t gdn_chunk_fwd_noalloc(const gdn_chunk_args *args, gdn_stream_t stream);

/* Size in bytes of the fixed scratch array used by gdn_chunk_fwd_noalloc. */
size_t gdn_noalloc_scratch_bytes(void);

/*
 * Self-test of the failure path shared by every kernel that waits on an
 * asynchronous copy or tensor-core operation: each such wait polls an
 * mbarrier a bounded number of times and, if the phase has not completed by
 * then, records GDN_ERR_TIMEOUT in the device error word and lets the kernel
 * finish instead of hanging.  This call runs that same wait once, in a
 * one-thread kernel, on a barrier of its own: with arrive = 0 nothing ever
 * arrives, so the wait gives up after max_polls polls (1 .. 2^22; the kernels
 * use 2^22) and GDN_ERR_TIMEOUT is recorded; with arrive = 1 the kernel
 * completes the phase itself first and nothing is recorded.  No copy or
 * tensor-core operation is in flight, so giving up leaves nothing behind.
 * Read the outcome with gdn_check_device_error().  GDN_ERR_INVALID_ARG for
 * arguments outside those ranges.
 */
gdn_status_t gdn_self_test_wait(int32_t arrive, int32_t max_polls, gdn_stream_t stream);

/*
 * Self-test of the bounds checks of a checked build (the library compiled
 * with -DGDN_CHECKED; the release build compiles them away).  Before a CTA of
 * any kernel touches memory, a checked build compares the index ranges the
 * CTA derived (chunk slots, token rows, heads, value columns, state slots)
 * with the extents of the tensors they index; when one falls outside, the CTA
 * records GDN_ERR_BOUNDS in the device error word and returns, uniformly and
 * before any barrier, so that nothing waits on it.  This call runs that check
 * in a one-CTA kernel on the index `index` against the extent `extent`: a
 * checked build records GDN_ERR_BOUNDS unless 0 <= index < extent, a release
 * build never does.  Read the outcome with gdn_check_device_error();
 * *checked_build is set to 1 in a checked build, else 0 (it may be NULL).
 */
gdn_status_t gdn_self_test_bounds(int32_t index, int32_t extent, int32_t *checked_build,
                                  gdn_stream_t stream);

/* Wait for `stream`, then read and clear the device error word of the current
 * device into *code (a gdn_status_t value, GDN_OK if nothing was recorded).
 * The word is shared by every stream of the device: the first error recorded
 * since the last clear is kept. */
gdn_status_t gdn_check_device_error(gdn_stream_t stream, int32_t *code);

/* Static, NUL-terminated name of a status. */
const char *gdn_status_string(gdn_status_t status);

/* Description of the calling thread's last host-side failure ("" if none). */
const char *gdn_last_error_message(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_GB300_H */
