// Chunk state pass of gated linear attention (KDA _fla/ops/common/chunk_h.py,
// chunk_fwd_kernel_h and chunk_fwd_h): for every sequence and head, the state
// h [K, V] at the start of every 64-token chunk and the final state of
//   h <- Dk_t h Dv_t + k_t v_t^T
// with one of the gate kinds of gdn.h.  In chunk form, with gamma the gate's
// inclusive cumulative sum inside the chunk and L its last valid row:
//   h_{c+1} = e^{g_L} diag(e^{gk_L}) h_c diag(e^{gv_L}) + sum_i k~_i v~_i^T,
//   k~_i = k_i e^{gk_L - gk_i},   v~_i = v_i e^{g_L - g_i} e^{gv_L - gv_i}
// (each factor present only for its gate kind; the per-head rate g_gamma has
// g_i = g_gamma (i + 1)).
//
// Exact fp32 CUDA-core kernel: one CTA per (32-column tile of V, head,
// sequence); each of its 256 threads keeps 16 state values (one key row, 16
// columns) in registers across the chunks, and each chunk's gated k~ and v~
// are staged in shared memory first.
#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int SP_THREADS = 256, SP_VT = 32;

template <typename T>
__global__ void __launch_bounds__(SP_THREADS) state_pass_kernel(StateParams p) {
  __shared__ float ks[BT][KMAX];      // k~ of the chunk, token-major
  __shared__ __align__(16) float vs[BT][SP_VT];  // v~ of the chunk's column tile
  __shared__ float gam[BT];           // per-token cumulative gate (g, g_gamma)
  __shared__ float gkl[KMAX];         // per-key cumulative gate of the last row (gk)
  __shared__ float gvl[SP_VT];        // per-column cumulative gate of the last row (gv)
  __shared__ long long seq_info[2];   // first chunk of this sequence, ok flag

  const int tid = threadIdx.x;
  const int v0 = blockIdx.x * SP_VT, h = blockIdx.y, n = blockIdx.z;
  const int H = p.H, K = p.K, V = p.V;
  const int r = tid >> 1, c0 = (tid & 1) * 16;  // this thread's key row and columns
  const bool row_ok = r < K;
  const T *k = static_cast<const T *>(p.k);
  const T *v = static_cast<const T *>(p.v);

  // ---- sequence bounds and the index of its first chunk in hs
  int bos = 0, eos = p.T, b = n;
  if (p.cu_seqlens) {
    b = 0;
    bos = p.cu_seqlens[n];
    eos = p.cu_seqlens[n + 1];
    if (tid == 0) {
      bool ok = bos >= 0 && eos >= bos && eos <= p.T && p.cu_seqlens[0] == 0 &&
                p.cu_seqlens[p.N] == p.T;
      long long first = 0;
      for (int m = 0; m < n && ok; ++m) {
        const int len = p.cu_seqlens[m + 1] - p.cu_seqlens[m];
        if (len < 0) ok = false;
        first += (len + BT - 1) / BT;
      }
      seq_info[0] = first;
      seq_info[1] = ok ? 1 : 0;
      if (!ok) record_error(p.err, GDN_ERR_BAD_SEQLENS);
    }
    __syncthreads();
    if (seq_info[1] == 0) bos = eos = 0;  // nothing read, no chunk written
  } else if (tid == 0) {
    seq_info[0] = (long long)n * ((p.T + BT - 1) / BT);
    seq_info[1] = 1;
  }
  __syncthreads();
  const int nch = (eos - bos + BT - 1) / BT;
  const long long first = seq_info[0];
  const bool write_hs = p.hs && seq_info[1] && first + nch <= p.num_chunks;
  if (p.hs && seq_info[1] && !write_hs && tid == 0) record_error(p.err, GDN_ERR_BAD_SEQLENS);

  // ---- the state tile: row r, columns v0 + c0 .. v0 + c0 + 15
  float hv[16];
  const size_t sbase = (((size_t)n * H + h) * K + r) * V;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int col = v0 + c0 + j;
    hv[j] = (p.h0 && row_ok && col < V) ? p.h0[sbase + col] : 0.f;
  }

#pragma unroll 1
  for (int c = 0; c < nch; ++c) {
    const int t0 = bos + c * BT;
    const int L = min(BT, eos - t0);
    const size_t row0 = (size_t)b * p.T + t0;  // global token row of the chunk's first token

    // chunk-start state
    if (write_hs && row_ok) {
      const size_t o = (((size_t)(first + c) * H + h) * K + r) * V;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int col = v0 + c0 + j;
        if (col < V) {
          if (p.hs_bf16)
            static_cast<__nv_bfloat16 *>(p.hs)[o + col] = __float2bfloat16_rn(hv[j]);
          else
            static_cast<float *>(p.hs)[o + col] = hv[j];
        }
      }
    }

    // gates of the chunk
    if (p.gate == GDN_GATE_G || p.gate == GDN_GATE_G_GAMMA) {
      if (tid < BT) {
        float x = 0.f;
        if (tid < L)
          x = p.gate == GDN_GATE_G ? p.gate_values[(row0 + tid) * H + h]
                                   : p.gate_values[h] * (float)(tid + 1);
        gam[tid] = x;
      }
    } else if (p.gate == GDN_GATE_GK) {
      if (tid < K) gkl[tid] = p.gate_values[((row0 + L - 1) * H + h) * K + tid];
    } else if (p.gate == GDN_GATE_GV) {
      if (tid < SP_VT) {
        const int col = v0 + tid;
        gvl[tid] = col < V ? p.gate_values[((row0 + L - 1) * H + h) * V + col] : 0.f;
      }
    }
    __syncthreads();
    const bool scalar_gate = p.gate == GDN_GATE_G || p.gate == GDN_GATE_G_GAMMA;
    const float gL = scalar_gate ? gam[L - 1] : 0.f;

    // stage k~ (per-key gate applied) and v~ (scalar and per-column gates)
    for (int idx = tid; idx < BT * K; idx += SP_THREADS) {
      const int i = idx / K, kk = idx % K;
      float x = 0.f;
      if (i < L) {
        x = to_f32(k[(row0 + i) * H * K + (size_t)h * K + kk]);
        if (p.gate == GDN_GATE_GK)
          x *= expf(gkl[kk] - p.gate_values[((row0 + i) * H + h) * K + kk]);
      }
      ks[i][kk] = x;
    }
    for (int idx = tid; idx < BT * SP_VT; idx += SP_THREADS) {
      const int i = idx / SP_VT, cc = idx % SP_VT, col = v0 + cc;
      float x = 0.f;
      if (i < L && col < V) {
        x = to_f32(v[(row0 + i) * H * V + (size_t)h * V + col]);
        if (scalar_gate) x *= expf(gL - gam[i]);
        if (p.gate == GDN_GATE_GV)
          x *= expf(gvl[cc] - p.gate_values[((row0 + i) * H + h) * V + col]);
      }
      vs[i][cc] = x;
    }
    __syncthreads();

    // h <- decay(h) + k~^T v~
    float dk = 1.f;
    if (scalar_gate) dk = expf(gL);
    if (p.gate == GDN_GATE_GK && row_ok) dk = expf(gkl[r]);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float dv = p.gate == GDN_GATE_GV ? expf(gvl[c0 + j]) : 1.f;
      hv[j] *= dk * dv;
    }
    if (row_ok) {
#pragma unroll 4
      for (int i = 0; i < L; ++i) {
        const float a = ks[i][r];
        const float4 *vr = reinterpret_cast<const float4 *>(&vs[i][c0]);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 w = vr[q];
          hv[4 * q] = fmaf(a, w.x, hv[4 * q]);
          hv[4 * q + 1] = fmaf(a, w.y, hv[4 * q + 1]);
          hv[4 * q + 2] = fmaf(a, w.z, hv[4 * q + 2]);
          hv[4 * q + 3] = fmaf(a, w.w, hv[4 * q + 3]);
        }
      }
    }
    __syncthreads();  // the next chunk restages ks, vs and the gates
  }

  if (p.ht && row_ok) {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int col = v0 + c0 + j;
      if (col < V) p.ht[sbase + col] = hv[j];
    }
  }
}

}  // namespace

cudaError_t launch_state_pass(const StateParams &p, bool bf16, cudaStream_t stream) {
  const dim3 grid((unsigned)((p.V + SP_VT - 1) / SP_VT), (unsigned)p.H, (unsigned)p.N);
  if (bf16)
    state_pass_kernel<__nv_bfloat16><<<grid, SP_THREADS, 0, stream>>>(p);
  else
    state_pass_kernel<float><<<grid, SP_THREADS, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace gdn
