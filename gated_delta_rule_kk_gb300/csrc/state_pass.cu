// Chunk state pass of gated linear attention (KDA _fla/ops/common/chunk_h.py,
// chunk_fwd_kernel_h and chunk_fwd_h): for every sequence and head, the state
// h [K, V] at the start of every 64-token chunk and the final state of
//   h <- Dk_t h Dv_t + k_t v_t^T
// with one of the gate kinds of gdn.h.  In chunk form, with gamma the gate's
// inclusive cumulative sum inside the chunk and L its last valid row:
//   h_{c+1} = e^{g_L} diag(e^{gk_L}) h_c diag(e^{gv_L}) + sum_i k~_i v~_i^T,
//   k~_i = k_i e^{gk_L - gk_i},   v~_i = v_i e^{g_L - g_i} e^{gv_L - gv_i}
// (each factor present only for its gate kind; the per-head rate g_gamma has
// g_i = g_gamma (i + 1)).  The backward pass (chunk_bwd_kernel_dh) runs the
// same steps from the last chunk to the first with q (scaled) for k, do for v
// and the factors e^{gamma_i} measured from the chunk's start:
//   dh_{c} = e^{g_L} diag(e^{gk_L}) dh_{c+1} diag(e^{gv_L}) + sum_i q~_i do~_i^T.
//
// Two kernels, one CTA per (32-column tile of V, head, sequence), 256 threads,
// the fp32 state in registers across the chunks.  A chunk's k, v and gates are
// loaded into registers (16-byte loads; K and V are multiples of 8) while the
// previous chunk is computed, then staged in shared memory with the gate
// factors applied.
//   state_pass_kernel     exact fp32 FMAs; every thread holds one key row x
//                         16 columns (any K <= 128, fp32 or bf16 inputs)
//   state_pass_tc_kernel  bf16 inputs with K = 128: warp w holds key rows
//                         16 w .. 16 w + 15 as m16n8k16 accumulators and adds
//                         k~^T v~ on the tensor cores from bf16 hi/lo pairs of
//                         k~ and v~ (hi.hi + hi.lo + lo.hi: fp32-grade products)
#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "ptx.cuh"

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

// Bounds of sequence n and the index of its first chunk in hs (every thread
// calls it; it synchronises the block).  A bad cu_seqlens is recorded and
// leaves the sequence empty.
struct SeqInfo {
  int bos, eos, b, nch;
  long long first;
  bool write_hs;
};
__device__ SeqInfo sequence_of(const StateParams &p, int n, int tid, long long *shared_info) {
  SeqInfo s;
  s.bos = 0; s.eos = p.T; s.b = n;
  if (p.cu_seqlens) {
    s.b = 0;
    s.bos = p.cu_seqlens[n];
    s.eos = p.cu_seqlens[n + 1];
    if (tid == 0) {
      bool ok = s.bos >= 0 && s.eos >= s.bos && s.eos <= p.T && p.cu_seqlens[0] == 0 &&
                p.cu_seqlens[p.N] == p.T;
      long long first = 0;
      for (int m = 0; m < n && ok; ++m) {
        const int len = p.cu_seqlens[m + 1] - p.cu_seqlens[m];
        if (len < 0) ok = false;
        first += (len + BT - 1) / BT;
      }
      shared_info[0] = first;
      shared_info[1] = ok ? 1 : 0;
      if (!ok) record_error(p.err, GDN_ERR_BAD_SEQLENS);
    }
    __syncthreads();
    if (shared_info[1] == 0) s.bos = s.eos = 0;  // nothing read, no chunk written
  } else if (tid == 0) {
    shared_info[0] = (long long)n * ((p.T + BT - 1) / BT);
    shared_info[1] = 1;
  }
  __syncthreads();
  s.nch = (s.eos - s.bos + BT - 1) / BT;
  s.first = shared_info[0];
  s.write_hs = p.hs && shared_info[1] && s.first + s.nch <= p.num_chunks;
  if (p.hs && shared_info[1] && !s.write_hs && tid == 0) record_error(p.err, GDN_ERR_BAD_SEQLENS);
  return s;
}

// One thread's share of a chunk's inputs, held in registers until staged:
// 8 consecutive keys (kq = 8 (tid & 15) ..) of rows (tid >> 4) + 16 pp,
// pp = 0..3, of the [64, K] k tile, and 8 consecutive columns (vq = 8 (tid & 3)
// ..) of row tid >> 2 of the [64, 32] v tile, with the matching gates.
struct ChunkRegs {
  float kx[4][8], gkx[4][8], vx[8], gvx[8];
  float gtok, glast;
};

template <typename T>
__device__ __forceinline__ void load_chunk(const StateParams &p, const SeqInfo &sq, int c, int h,
                                           int v0, int tid, ChunkRegs &R) {
  const int H = p.H, K = p.K, V = p.V, HG = p.HG, hg = h / (H / HG);
  const T *k = static_cast<const T *>(p.k);
  const T *v = static_cast<const T *>(p.v);
  const bool gk = p.gate == GDN_GATE_GK, gvg = p.gate == GDN_GATE_GV;
  const int kq = (tid & 15) * 8, vi = tid >> 2, vq = (tid & 3) * 8;
  const int t0 = sq.bos + c * BT;
  const int L = min(BT, sq.eos - t0);
  const size_t row0 = (size_t)sq.b * p.T + t0;
#pragma unroll
  for (int pp = 0; pp < 4; ++pp) {
    const int i = (tid >> 4) + 16 * pp;
    const bool ok = i < L && kq < K;
    const size_t e = (row0 + i) * H * K + (size_t)h * K + kq;
    load8(k + e, ok, R.kx[pp]);
    load8(p.gate_values + ((row0 + i) * HG + hg) * K + kq, ok && gk, R.gkx[pp]);
  }
  {
    const bool ok = vi < L && v0 + vq < V;
    const size_t e = (row0 + vi) * H * V + (size_t)h * V + v0 + vq;
    load8(v + e, ok, R.vx);
    load8(p.gate_values + ((row0 + vi) * HG + hg) * V + v0 + vq, ok && gvg, R.gvx);
  }
  R.gtok = 0.f;
  if (p.gate == GDN_GATE_G && tid < L) R.gtok = p.gate_values[(row0 + tid) * HG + hg];
  if (p.gate == GDN_GATE_G_GAMMA && tid < L) R.gtok = p.gate_values[hg] * (float)(tid + 1);
  R.glast = 0.f;
  if (gk && tid < K) R.glast = p.gate_values[((row0 + L - 1) * HG + hg) * K + tid];
  if (gvg && tid < SP_VT && v0 + tid < V)
    R.glast = p.gate_values[((row0 + L - 1) * HG + hg) * V + v0 + tid];
}

// The gated k~ (8 values of row (tid >> 4) + 16 pp) and v~ (8 values of row
// tid >> 2) of a chunk, once its gate vectors are in shared memory.  Forward:
// factors e^{gamma_L - gamma_i} (from token i to the chunk's end); backward:
// e^{gamma_i} (from the chunk's start to token i) and the scale on q.  Rows
// past the chunk's last one hold zeros and take no factor.
__device__ __forceinline__ void gated_k(const StateParams &p, const ChunkRegs &R, int pp, int tid,
                                        int L, const float *gkl, float *x) {
  const int i = (tid >> 4) + 16 * pp, kq = (tid & 15) * 8;
  const bool apply = p.gate == GDN_GATE_GK && i < L;
  const float s = p.reverse ? p.scale : 1.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const float f = p.reverse ? R.gkx[pp][e] : gkl[kq + e] - R.gkx[pp][e];
    x[e] = s * (apply ? R.kx[pp][e] * expf(f) : R.kx[pp][e]);
  }
}
__device__ __forceinline__ void gated_v(const StateParams &p, const ChunkRegs &R, int tid, int L,
                                        float gL, const float *gam, const float *gvl, float *x) {
  const int vi = tid >> 2, vq = (tid & 3) * 8;
  const bool scalar_gate = p.gate == GDN_GATE_G || p.gate == GDN_GATE_G_GAMMA;
  float sf = 1.f;
  if (scalar_gate && vi < L) sf = expf(p.reverse ? gam[vi] : gL - gam[vi]);
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    x[e] = R.vx[e] * sf;
    if (p.gate == GDN_GATE_GV && vi < L)
      x[e] *= expf(p.reverse ? R.gvx[e] : gvl[vq + e] - R.gvx[e]);
  }
}

// 8 fp32 values -> bf16 hi and lo halves (hi = RNE(x), lo = RNE(x - hi)).
__device__ __forceinline__ void split8_bf16(const float *x, uint4 &hi, uint4 &lo) {
  uint32_t hw[4], lw[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    hw[q] = pack_bf16x2(x[2 * q], x[2 * q + 1]);
    lw[q] = pack_bf16x2(x[2 * q] - __uint_as_float(hw[q] << 16),
                        x[2 * q + 1] - __uint_as_float(hw[q] & 0xffff0000u));
  }
  hi = make_uint4(hw[0], hw[1], hw[2], hw[3]);
  lo = make_uint4(lw[0], lw[1], lw[2], lw[3]);
}

// ---------------------------------------------------------------------------
// exact fp32 kernel

template <typename T>
__global__ void __launch_bounds__(SP_THREADS) state_pass_kernel(StateParams p) {
  __shared__ float ks[BT][KMAX];                 // k~ of the chunk, token-major
  __shared__ __align__(16) float vs[BT][SP_VT];  // v~ of the chunk's column tile
  __shared__ float gam[BT];                      // per-token cumulative gate (g, g_gamma)
  __shared__ float gkl[KMAX];                    // per-key cumulative gate of the last row (gk)
  __shared__ float gvl[SP_VT];                   // per-column one of the last row (gv)
  __shared__ long long seq_info[2];

  const int tid = threadIdx.x;
  const int v0 = blockIdx.x * SP_VT, h = blockIdx.y, n = blockIdx.z;
  const int H = p.H, K = p.K, V = p.V;
  const int r = tid >> 1, c0 = (tid & 1) * 16;  // this thread's key row and columns
  const bool row_ok = r < K;
  const bool gk = p.gate == GDN_GATE_GK, gvg = p.gate == GDN_GATE_GV;
  const bool scalar_gate = p.gate == GDN_GATE_G || p.gate == GDN_GATE_G_GAMMA;
  const SeqInfo sq = sequence_of(p, n, tid, seq_info);

  float hv[16];
  const size_t sbase = (((size_t)n * H + h) * K + r) * V;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int col = v0 + c0 + j;
    hv[j] = (p.h0 && row_ok && col < V) ? p.h0[sbase + col] : 0.f;
  }

  // chunk of the it-th step: forward from the first, backward from the last
  auto chunk_at = [&](int it) { return p.reverse ? sq.nch - 1 - it : it; };
  ChunkRegs R;
  if (sq.nch > 0) load_chunk<T>(p, sq, chunk_at(0), h, v0, tid, R);
#pragma unroll 1
  for (int it = 0; it < sq.nch; ++it) {
    const int c = chunk_at(it);
    const int L = min(BT, sq.eos - (sq.bos + c * BT));

    // chunk-start state, 8 columns (16 or 32 bytes) per store
    if (sq.write_hs && row_ok) {
      const size_t o = (((size_t)(sq.first + c) * H + h) * K + r) * V + v0 + c0;
#pragma unroll
      for (int g8 = 0; g8 < 2; ++g8) {
        if (v0 + c0 + 8 * g8 >= V) continue;  // V is a multiple of 8
        const float *x = hv + 8 * g8;
        if (p.hs_bf16) {
          uint4 w;
          w.x = pack_bf16x2(x[0], x[1]); w.y = pack_bf16x2(x[2], x[3]);
          w.z = pack_bf16x2(x[4], x[5]); w.w = pack_bf16x2(x[6], x[7]);
          *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.hs) + o + 8 * g8) = w;
        } else {
          float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.hs) + o + 8 * g8);
          dst[0] = make_float4(x[0], x[1], x[2], x[3]);
          dst[1] = make_float4(x[4], x[5], x[6], x[7]);
        }
      }
    }

    // this chunk's gates, then k~ and v~, from the registers
    if (scalar_gate && tid < BT) gam[tid] = R.gtok;
    if (gk && tid < K) gkl[tid] = R.glast;
    if (gvg && tid < SP_VT) gvl[tid] = R.glast;
    __syncthreads();
    const float gL = scalar_gate ? gam[L - 1] : 0.f;
    const int kq = (tid & 15) * 8;
    if (kq < K) {
#pragma unroll
      for (int pp = 0; pp < 4; ++pp) {
        float x[8];
        gated_k(p, R, pp, tid, L, gkl, x);
        float4 *dst = reinterpret_cast<float4 *>(&ks[(tid >> 4) + 16 * pp][kq]);
        dst[0] = make_float4(x[0], x[1], x[2], x[3]);
        dst[1] = make_float4(x[4], x[5], x[6], x[7]);
      }
    }
    {
      float x[8];
      gated_v(p, R, tid, L, gL, gam, gvl, x);
      float4 *dst = reinterpret_cast<float4 *>(&vs[tid >> 2][(tid & 3) * 8]);
      dst[0] = make_float4(x[0], x[1], x[2], x[3]);
      dst[1] = make_float4(x[4], x[5], x[6], x[7]);
    }
    __syncthreads();
    if (it + 1 < sq.nch) load_chunk<T>(p, sq, chunk_at(it + 1), h, v0, tid, R);  // in flight below

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

// ---------------------------------------------------------------------------
// tensor-core kernel (bf16 inputs, K = 128)

// Row pitches of the staged operands (bf16): 272 B and 80 B, so the eight
// 16-byte rows an ldmatrix reads fall in eight different bank quads.
constexpr int TC_KP = 136;
constexpr int TC_VP = 40;

__global__ void __launch_bounds__(SP_THREADS) state_pass_tc_kernel(StateParams p) {
  __shared__ __align__(16) __nv_bfloat16 ksh[BT][TC_KP], ksl[BT][TC_KP];  // k~ hi, lo
  __shared__ __align__(16) __nv_bfloat16 vsh[BT][TC_VP], vsl[BT][TC_VP];  // v~ hi, lo
  __shared__ float gam[BT], gkl[KMAX], gvl[SP_VT];
  __shared__ long long seq_info[2];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, tig = lane & 3;
  const int v0 = blockIdx.x * SP_VT, h = blockIdx.y, n = blockIdx.z;
  const int H = p.H, V = p.V;
  constexpr int K = KMAX;
  const bool gk = p.gate == GDN_GATE_GK, gvg = p.gate == GDN_GATE_GV;
  const bool scalar_gate = p.gate == GDN_GATE_G || p.gate == GDN_GATE_G_GAMMA;
  const SeqInfo sq = sequence_of(p, n, tid, seq_info);

  // accumulator rows rA = 16 warp + g and rA + 8, columns v0 + 8 nt + 2 tig (+ 1)
  const int rA = 16 * warp + g;
  float C[4][4];
  const size_t sA = (((size_t)n * H + h) * K + rA) * V, sB = sA + (size_t)8 * V;
#pragma unroll
  for (int nt = 0; nt < 4; ++nt) {
    const int col = v0 + 8 * nt + 2 * tig;
    const bool ok = p.h0 && col < V;  // V is a multiple of 8, so col + 1 < V too
    C[nt][0] = ok ? p.h0[sA + col] : 0.f;
    C[nt][1] = ok ? p.h0[sA + col + 1] : 0.f;
    C[nt][2] = ok ? p.h0[sB + col] : 0.f;
    C[nt][3] = ok ? p.h0[sB + col + 1] : 0.f;
  }

  auto chunk_at = [&](int it) { return p.reverse ? sq.nch - 1 - it : it; };
  ChunkRegs R;
  if (sq.nch > 0) load_chunk<__nv_bfloat16>(p, sq, chunk_at(0), h, v0, tid, R);
#pragma unroll 1
  for (int it = 0; it < sq.nch; ++it) {
    const int c = chunk_at(it);
    const int L = min(BT, sq.eos - (sq.bos + c * BT));

    // chunk-start state: two columns per 8-column tile and row
    if (sq.write_hs) {
      const size_t oA = (((size_t)(sq.first + c) * H + h) * K + rA) * V, oB = oA + (size_t)8 * V;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const int col = v0 + 8 * nt + 2 * tig;
        if (col >= V) continue;
        if (p.hs_bf16) {
          __nv_bfloat16 *hb = static_cast<__nv_bfloat16 *>(p.hs);
          *reinterpret_cast<uint32_t *>(hb + oA + col) = pack_bf16x2(C[nt][0], C[nt][1]);
          *reinterpret_cast<uint32_t *>(hb + oB + col) = pack_bf16x2(C[nt][2], C[nt][3]);
        } else {
          float *hf = static_cast<float *>(p.hs);
          *reinterpret_cast<float2 *>(hf + oA + col) = make_float2(C[nt][0], C[nt][1]);
          *reinterpret_cast<float2 *>(hf + oB + col) = make_float2(C[nt][2], C[nt][3]);
        }
      }
    }

    // stage k~ and v~ as bf16 hi/lo pairs
    if (scalar_gate && tid < BT) gam[tid] = R.gtok;
    if (gk && tid < K) gkl[tid] = R.glast;
    if (gvg && tid < SP_VT) gvl[tid] = R.glast;
    __syncthreads();
    const float gL = scalar_gate ? gam[L - 1] : 0.f;
#pragma unroll
    for (int pp = 0; pp < 4; ++pp) {
      float x[8];
      gated_k(p, R, pp, tid, L, gkl, x);
      uint4 hi, lo;
      split8_bf16(x, hi, lo);
      const int i = (tid >> 4) + 16 * pp, kq = (tid & 15) * 8;
      *reinterpret_cast<uint4 *>(&ksh[i][kq]) = hi;
      *reinterpret_cast<uint4 *>(&ksl[i][kq]) = lo;
    }
    {
      float x[8];
      gated_v(p, R, tid, L, gL, gam, gvl, x);
      uint4 hi, lo;
      split8_bf16(x, hi, lo);
      const int vi = tid >> 2, vq = (tid & 3) * 8;
      *reinterpret_cast<uint4 *>(&vsh[vi][vq]) = hi;
      *reinterpret_cast<uint4 *>(&vsl[vi][vq]) = lo;
    }
    __syncthreads();
    if (it + 1 < sq.nch) load_chunk<__nv_bfloat16>(p, sq, chunk_at(it + 1), h, v0, tid, R);

    // decay: rows by e^{g_L} e^{gk_L[row]}, columns by e^{gv_L[col]}
    float dA = 1.f, dB = 1.f;
    if (scalar_gate) dA = dB = expf(gL);
    if (gk) {
      dA = expf(gkl[rA]);
      dB = expf(gkl[rA + 8]);
    }
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      float d0 = 1.f, d1 = 1.f;
      if (gvg) {
        d0 = expf(gvl[8 * nt + 2 * tig]);
        d1 = expf(gvl[8 * nt + 2 * tig + 1]);
      }
      C[nt][0] *= dA * d0;
      C[nt][1] *= dA * d1;
      C[nt][2] *= dB * d0;
      C[nt][3] *= dB * d1;
    }

    // C += k~^T v~ over the chunk's tokens, 16 at a time.  A = k~^T (this
    // warp's 16 keys x 16 tokens) and B = v~ (16 tokens x 16 columns) come
    // from the token-major tiles by transposing ldmatrix.
#pragma unroll
    for (int kt = 0; kt < 4; ++kt) {
      if (16 * kt >= L) break;
      uint32_t ah[4], al[4];
      {
        const int row = 16 * kt + (lane & 7) + ((lane >> 4) << 3);
        const int key = 16 * warp + ((lane >> 3) & 1) * 8;
        ptx::ldmatrix_x4_trans(&ksh[row][key], ah[0], ah[1], ah[2], ah[3]);
        ptx::ldmatrix_x4_trans(&ksl[row][key], al[0], al[1], al[2], al[3]);
      }
#pragma unroll
      for (int np = 0; np < 2; ++np) {
        uint32_t bh[4], bl[4];
        const int row = 16 * kt + (lane & 7) + (((lane >> 3) & 1) << 3);
        const int col = 16 * np + ((lane >> 4) << 3);
        ptx::ldmatrix_x4_trans(&vsh[row][col], bh[0], bh[1], bh[2], bh[3]);
        ptx::ldmatrix_x4_trans(&vsl[row][col], bl[0], bl[1], bl[2], bl[3]);
        ptx::mma_16816_bf16(C[2 * np], ah, bh[0], bh[1]);
        ptx::mma_16816_bf16(C[2 * np], ah, bl[0], bl[1]);
        ptx::mma_16816_bf16(C[2 * np], al, bh[0], bh[1]);
        ptx::mma_16816_bf16(C[2 * np + 1], ah, bh[2], bh[3]);
        ptx::mma_16816_bf16(C[2 * np + 1], ah, bl[2], bl[3]);
        ptx::mma_16816_bf16(C[2 * np + 1], al, bh[2], bh[3]);
      }
    }
    __syncthreads();  // the next chunk restages the operands and the gates
  }

  if (p.ht) {
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const int col = v0 + 8 * nt + 2 * tig;
      if (col >= V) continue;
      p.ht[sA + col] = C[nt][0];
      p.ht[sA + col + 1] = C[nt][1];
      p.ht[sB + col] = C[nt][2];
      p.ht[sB + col + 1] = C[nt][3];
    }
  }
}

}  // namespace

cudaError_t launch_state_pass(const StateParams &p, bool bf16, cudaStream_t stream) {
  const dim3 grid((unsigned)((p.V + SP_VT - 1) / SP_VT), (unsigned)p.H, (unsigned)p.N);
  if (bf16 && p.K == KMAX)
    state_pass_tc_kernel<<<grid, SP_THREADS, 0, stream>>>(p);
  else if (bf16)
    state_pass_kernel<__nv_bfloat16><<<grid, SP_THREADS, 0, stream>>>(p);
  else
    state_pass_kernel<float><<<grid, SP_THREADS, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace gdn
