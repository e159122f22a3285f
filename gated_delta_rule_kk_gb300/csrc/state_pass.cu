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
// columns) in registers across the chunks.  A chunk's k, v and gates are
// loaded into registers (16-byte loads; K and V are multiples of 8) while the
// previous chunk is computed, then written to shared memory with the gate
// factors applied.
#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int SP_THREADS = 256, SP_VT = 32;

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {  // RNE, a in the low half
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t *>(&v);
}

// 8 consecutive elements (16-byte aligned) widened to fp32; zeros if !ok.
__device__ __forceinline__ void load8(const float *src, bool ok, float *out) {
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
  if (ok) {
    a = reinterpret_cast<const float4 *>(src)[0];
    b = reinterpret_cast<const float4 *>(src)[1];
  }
  out[0] = a.x; out[1] = a.y; out[2] = a.z; out[3] = a.w;
  out[4] = b.x; out[5] = b.y; out[6] = b.z; out[7] = b.w;
}
__device__ __forceinline__ void load8(const __nv_bfloat16 *src, bool ok, float *out) {
  uint4 u = make_uint4(0u, 0u, 0u, 0u);
  if (ok) u = *reinterpret_cast<const uint4 *>(src);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    out[2 * q] = __uint_as_float(w[q] << 16);
    out[2 * q + 1] = __uint_as_float(w[q] & 0xffff0000u);
  }
}

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

  // Each thread's share of a chunk's inputs, loaded into registers one chunk
  // ahead (16-byte loads, all independent, so their latency overlaps the
  // current chunk's arithmetic): 8 consecutive keys of rows (tid >> 4) + 16 p,
  // p = 0..3, of the [64, K] k tile (keys 8 (tid & 15) ..), and 8 consecutive
  // columns of row tid >> 2 of the [64, 32] v tile (columns 8 (tid & 3) ..),
  // with the matching gates.
  float kx[4][8], gkx[4][8], vx[8], gvx[8];
  float gtok = 0.f, glast = 0.f;
  const bool gk = p.gate == GDN_GATE_GK, gvg = p.gate == GDN_GATE_GV;
  const bool scalar_gate = p.gate == GDN_GATE_G || p.gate == GDN_GATE_G_GAMMA;
  const int kq = (tid & 15) * 8, vi = tid >> 2, vq = (tid & 3) * 8;
  const bool kq_ok = kq < K, vq_ok = v0 + vq < V;
  auto load = [&](int c) {
    const int t0 = bos + c * BT;
    const int L = min(BT, eos - t0);
    const size_t row0 = (size_t)b * p.T + t0;
#pragma unroll
    for (int pp = 0; pp < 4; ++pp) {
      const int i = (tid >> 4) + 16 * pp;
      const bool ok = i < L && kq_ok;
      const size_t e = (row0 + i) * H * K + (size_t)h * K + kq;
      load8(k + e, ok, kx[pp]);
      load8(p.gate_values + e, ok && gk, gkx[pp]);
    }
    {
      const bool ok = vi < L && vq_ok;
      const size_t e = (row0 + vi) * H * V + (size_t)h * V + v0 + vq;
      load8(v + e, ok, vx);
      load8(p.gate_values + e, ok && gvg, gvx);
    }
    gtok = 0.f;
    if (p.gate == GDN_GATE_G && tid < L) gtok = p.gate_values[(row0 + tid) * H + h];
    if (p.gate == GDN_GATE_G_GAMMA && tid < L) gtok = p.gate_values[h] * (float)(tid + 1);
    glast = 0.f;
    if (gk && tid < K) glast = p.gate_values[((row0 + L - 1) * H + h) * K + tid];
    if (gvg && tid < SP_VT && v0 + tid < V)
      glast = p.gate_values[((row0 + L - 1) * H + h) * V + v0 + tid];
  };

  if (nch > 0) load(0);
#pragma unroll 1
  for (int c = 0; c < nch; ++c) {
    const int L = min(BT, eos - (bos + c * BT));

    // chunk-start state, 8 columns (16 or 32 bytes) per store
    if (write_hs && row_ok) {
      const size_t o = (((size_t)(first + c) * H + h) * K + r) * V + v0 + c0;
#pragma unroll
      for (int g8 = 0; g8 < 2; ++g8) {
        if (v0 + c0 + 8 * g8 >= V) continue;  // V is a multiple of 8
        const float *x = hv + 8 * g8;
        if (p.hs_bf16) {
          __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(p.hs) + o + 8 * g8;
          uint4 w;
          w.x = pack_bf16x2(x[0], x[1]); w.y = pack_bf16x2(x[2], x[3]);
          w.z = pack_bf16x2(x[4], x[5]); w.w = pack_bf16x2(x[6], x[7]);
          *reinterpret_cast<uint4 *>(dst) = w;
        } else {
          float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.hs) + o + 8 * g8);
          dst[0] = make_float4(x[0], x[1], x[2], x[3]);
          dst[1] = make_float4(x[4], x[5], x[6], x[7]);
        }
      }
    }

    // this chunk's gates, then k~ and v~, from the registers (rows past the
    // chunk's last one hold zeros and take no factor)
    if (scalar_gate && tid < BT) gam[tid] = gtok;
    if (gk && tid < K) gkl[tid] = glast;
    if (gvg && tid < SP_VT) gvl[tid] = glast;
    __syncthreads();
    const float gL = scalar_gate ? gam[L - 1] : 0.f;
    if (kq_ok) {
#pragma unroll
      for (int pp = 0; pp < 4; ++pp) {
        const int i = (tid >> 4) + 16 * pp;
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
          x[e] = (gk && i < L) ? kx[pp][e] * expf(gkl[kq + e] - gkx[pp][e]) : kx[pp][e];
        float4 *dst = reinterpret_cast<float4 *>(&ks[i][kq]);
        dst[0] = make_float4(x[0], x[1], x[2], x[3]);
        dst[1] = make_float4(x[4], x[5], x[6], x[7]);
      }
    }
    {
      float x[8];
      const float sf = (scalar_gate && vi < L) ? expf(gL - gam[vi]) : 1.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        x[e] = vx[e] * sf;
        if (gvg && vi < L) x[e] *= expf(gvl[vq + e] - gvx[e]);
      }
      float4 *dst = reinterpret_cast<float4 *>(&vs[vi][vq]);
      dst[0] = make_float4(x[0], x[1], x[2], x[3]);
      dst[1] = make_float4(x[4], x[5], x[6], x[7]);
    }
    __syncthreads();
    if (c + 1 < nch) load(c + 1);  // in flight during the update below

    // h <- decay(h) + k~^T v~
    float dk = 1.f;
    if (scalar_gate) dk = expf(gL);
    if (gk && row_ok) dk = expf(gkl[r]);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float dv = gvg ? expf(gvl[c0 + j]) : 1.f;
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
