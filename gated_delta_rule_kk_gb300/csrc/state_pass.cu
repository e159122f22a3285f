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
// The state (or gradient) is stored at chunks c = 0, S, 2 S, .. of each
// sequence for a split of S chunks (the page's split_size / chunk_size).
//
// Two kernels, one CTA per (32-column tile of V, head, sequence), the fp32
// state in registers across the chunks (K and V are multiples of 8, so every
// row piece is a 16-byte load or copy).
//   state_pass_kernel     256 threads, exact fp32 FMAs; every thread holds one
//                         key row x 16 columns (any K <= 128, fp32 or bf16
//                         inputs); a chunk's k, v and gates are loaded into
//                         registers while the previous chunk is computed, then
//                         staged in shared memory with the gate factors applied
//   state_pass_tc_kernel  bf16 inputs with K = 128, 512 threads: each warp
//                         holds 16 key rows x 16 columns as m16n8k16
//                         accumulators; raw chunks stream into a shared-memory
//                         ring by cp.async several steps ahead, v~ (and with
//                         the per-key gate k~) is staged as a bf16 hi/lo pair
//                         into double-buffered operands, and the tensor-core
//                         update takes fp32-grade products (below)
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

// Bounds of sequence n and the index of its first stored state in hs (one
// per split of p.split chunks; every thread calls it; it synchronises the
// block).  A bad cu_seqlens is recorded and leaves the sequence empty.
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
        first += (len + BT * p.split - 1) / (BT * p.split);
      }
      shared_info[0] = first;
      shared_info[1] = ok ? 1 : 0;
      if (!ok) record_error(p.err, GDN_ERR_BAD_SEQLENS);
    }
    __syncthreads();
    if (shared_info[1] == 0) s.bos = s.eos = 0;  // nothing read, no chunk written
  } else if (tid == 0) {
    shared_info[0] = (long long)n * ((p.T + BT * p.split - 1) / (BT * p.split));
    shared_info[1] = 1;
  }
  __syncthreads();
  s.nch = (s.eos - s.bos + BT - 1) / BT;
  s.first = shared_info[0];
  s.write_hs =
      p.hs && shared_info[1] && s.first + (s.nch + p.split - 1) / p.split <= p.num_chunks;
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
__global__ void __launch_bounds__(SP_THREADS, 1) state_pass_kernel(StateParams p) {
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
  if (!bounds_ok(n < p.N && h < p.H && v0 < p.V && sq.bos >= 0 && sq.bos <= sq.eos && sq.eos <= p.T,
                 p.err))
    return;

  float hv[16];
  // element (key r, column col) of a [K, V] state (or [V, K] with v_first)
  const size_t hbase = ((size_t)n * H + h) * K * V;
  auto at = [&](int col) { return p.v_first ? (size_t)col * K + r : (size_t)r * V + col; };
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int col = v0 + c0 + j;
    hv[j] = (p.h0 && row_ok && col < V) ? p.h0[hbase + at(col)] : 0.f;
  }

  // chunk of the it-th step: forward from the first, backward from the last
  auto chunk_at = [&](int it) { return p.reverse ? sq.nch - 1 - it : it; };
  // stored chunks 0, split, 2 split, ..; the reverse pass meets them last first
  int store_i = p.reverse && sq.nch > 0 ? (sq.nch - 1) / p.split : 0;
  int store_c = store_i * p.split;
  ChunkRegs R;
  if (sq.nch > 0) load_chunk<T>(p, sq, chunk_at(0), h, v0, tid, R);
#pragma unroll 1
  for (int it = 0; it < sq.nch; ++it) {
    const int c = chunk_at(it);
    const int L = min(BT, sq.eos - (sq.bos + c * BT));
    const bool store = c == store_c;
    const long long slot = sq.first + store_i;
    if (store) {
      store_c += p.reverse ? -p.split : p.split;
      store_i += p.reverse ? -1 : 1;
    }

    // chunk-start state, 8 columns (16 or 32 bytes) per store; one element
    // at a time in the [V, K] layout
    if (sq.write_hs && row_ok && store && p.v_first) {
      const size_t sb = ((size_t)slot * H + h) * K * V;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int col = v0 + c0 + j;
        if (col >= V) continue;
        if (p.hs_bf16)
          static_cast<__nv_bfloat16 *>(p.hs)[sb + at(col)] = __float2bfloat16_rn(hv[j]);
        else
          static_cast<float *>(p.hs)[sb + at(col)] = hv[j];
      }
    } else if (sq.write_hs && row_ok && store) {
      const size_t o = (((size_t)slot * H + h) * K + r) * V + v0 + c0;
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
      if (col < V) p.ht[hbase + at(col)] = hv[j];
    }
  }
}

// ---------------------------------------------------------------------------
// tensor-core kernel (bf16 inputs, K = 128)
//
// 512 threads.  Warp w holds key rows 16 (w & 7) .. + 15 and columns
// 16 (w >> 3) .. + 15 of the 32-column tile as two m16n8k16 accumulators.
// Raw chunks (k, v and the gate rows) stream into a ring of RING slots by
// asynchronous copies issued several steps ahead.  In the step of chunk c
// every thread stages chunk c+1 from the ring into the other operand buffer,
// refills a free ring slot, then runs the MMAs of chunk c, so staging and
// tensor-core work of different warps overlap and a step needs one barrier.
//
// The token-dependent gate factors and the backward scale go on v~ (staged
// as a bf16 hi/lo pair).  k then stays exact in bf16 and is read by the MMAs
// straight from the ring (C += k^T (v~hi + v~lo)), except with the per-key
// gate (KSTAGE), whose factor e^{gk_L - gk_i} depends on key and token: there
// k~ is staged as a hi/lo pair too (C += k~hi^T v~hi + k~hi^T v~lo + k~lo^T v~hi).

constexpr int TC_THREADS = 512;
// Row pitches of the operands (bf16): 272 B and 80 B, so the eight 16-byte
// rows an ldmatrix reads fall in eight different bank quads.
constexpr int TC_KP = 136;
constexpr int TC_VP = 40;
constexpr uint32_t TC_KS = BT * TC_KP * 2, TC_VS = BT * TC_VP * 2;  // one tile, bytes
// Operand buffer: [k~ hi, k~ lo] (KSTAGE only), then v~ hi, v~ lo.
__host__ __device__ constexpr uint32_t tc_buf_bytes(bool kstage) {
  return (kstage ? 2 * TC_KS : 0) + 2 * TC_VS;
}
// A ring slot: raw k [64][TC_KP] bf16 (rows padded like the operands), raw v
// [64][32] bf16, then the gate rows (g: [64] fp32, gk: [64][128] fp32,
// gv: [64][32] fp32; none for g_gamma).
constexpr uint32_t RS_K = 0, RS_V = TC_KS, RS_G = RS_V + BT * SP_VT * 2;
__host__ __device__ constexpr uint32_t ring_slot_bytes(int gate) {
  return RS_G + (gate == GDN_GATE_G    ? BT * 4
                 : gate == GDN_GATE_GK ? BT * KMAX * 4
                 : gate == GDN_GATE_GV ? BT * SP_VT * 4
                                       : 0);
}

// Issue the copies of chunk c into a ring slot (rows past the chunk's end and
// columns past V are zero-filled).
__device__ __forceinline__ void tc_fetch(const StateParams &p, const SeqInfo &sq, int c, int h,
                                         int v0, int tid, unsigned char *slot) {
  const int H = p.H, V = p.V, HG = p.HG, hg = h / (H / HG);
  constexpr int K = KMAX;
  const __nv_bfloat16 *k = static_cast<const __nv_bfloat16 *>(p.k);
  const __nv_bfloat16 *v = static_cast<const __nv_bfloat16 *>(p.v);
  const float *gvals = p.gate_values;
  const int t0 = sq.bos + c * BT;
  const int L = min(BT, sq.eos - t0);
  const size_t row0 = (size_t)sq.b * p.T + t0;
#pragma unroll
  for (int j = 0; j < 2; ++j) {  // k: 64 rows x 16 pieces
    const int piece = tid + TC_THREADS * j, i = piece >> 4, q = piece & 15;
    const bool ok = i < L;
    ptx::cp_async16(slot + RS_K + (i * TC_KP + 8 * q) * 2,
                    k + ((row0 + (ok ? i : 0)) * H + h) * K + 8 * q, ok);
  }
  if (tid < 4 * BT) {  // v: 64 rows x 4 pieces
    const int i = tid >> 2, q = tid & 3;
    const bool ok = i < L && v0 + 8 * q < V;
    ptx::cp_async16(slot + RS_V + (i * SP_VT + 8 * q) * 2,
                    v + ((row0 + (ok ? i : 0)) * H + h) * V + (ok ? v0 + 8 * q : 0), ok);
  }
  if (p.gate == GDN_GATE_G) {
    if (tid < BT) {
      const bool ok = tid < L;
      ptx::cp_async4(slot + RS_G + tid * 4, gvals + (row0 + (ok ? tid : 0)) * HG + hg, ok);
    }
  } else if (p.gate == GDN_GATE_GK) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {  // 64 rows x 32 pieces
      const int piece = tid + TC_THREADS * j, i = piece >> 5, q = piece & 31;
      const bool ok = i < L;
      ptx::cp_async16(slot + RS_G + (i * K + 4 * q) * 4,
                      gvals + ((row0 + (ok ? i : 0)) * HG + hg) * K + 4 * q, ok);
    }
  } else if (p.gate == GDN_GATE_GV) {  // 64 rows x 8 pieces
    const int i = tid >> 3, q = tid & 7;
    const bool ok = i < L && v0 + 4 * q < V;  // V, v0 multiples of 8: the piece is whole
    ptx::cp_async16(slot + RS_G + (i * SP_VT + 4 * q) * 4,
                    gvals + ((row0 + (ok ? i : 0)) * HG + hg) * V + (ok ? v0 + 4 * q : 0), ok);
  }
}

// Decay of the accumulators over one chunk (rows rA, rA + 8; columns of the
// two n-tiles, two each).
struct TcDecay {
  float r[2], c[4];
};

__device__ __forceinline__ void unpack8_bf16(const uint4 &u, float *out) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    out[2 * q] = __uint_as_float(w[q] << 16);
    out[2 * q + 1] = __uint_as_float(w[q] & 0xffff0000u);
  }
}
__device__ __forceinline__ void ld8_shared(const float *src, float *out) {
  const float4 a = reinterpret_cast<const float4 *>(src)[0];
  const float4 b = reinterpret_cast<const float4 *>(src)[1];
  out[0] = a.x; out[1] = a.y; out[2] = a.z; out[3] = a.w;
  out[4] = b.x; out[5] = b.y; out[6] = b.z; out[7] = b.w;
}

// Stage a chunk (L valid rows) from a ring slot into an operand buffer and
// return its accumulator decay.  Forward: v~ = v e^{g_L - g_i} e^{gv_L - gv_i}
// (and k~ = k e^{gk_L - gk_i}); backward: v~ = scale do e^{g_i} e^{gv_i} (and
// k~ = q e^{gk_i}).  Rows past the chunk's end are zeros and take no factor.
template <bool KSTAGE>
__device__ __forceinline__ void tc_stage(const StateParams &p, const unsigned char *slot, int L,
                                         float gamma, unsigned char *buf, int tid, int rA, int cl,
                                         TcDecay &d) {
  constexpr int K = KMAX;
  const bool gvg = p.gate == GDN_GATE_GV;
  const bool scalar_gate = p.gate == GDN_GATE_G || p.gate == GDN_GATE_G_GAMMA;
  const float *gr = reinterpret_cast<const float *>(slot + RS_G);
  if (KSTAGE) {  // per-key gate
    const int kq = (tid & 15) * 8;
    __nv_bfloat16(*ksh)[TC_KP] = reinterpret_cast<__nv_bfloat16(*)[TC_KP]>(buf);
    __nv_bfloat16(*ksl)[TC_KP] = reinterpret_cast<__nv_bfloat16(*)[TC_KP]>(buf + TC_KS);
    float gkl[8];
    if (!p.reverse) ld8_shared(gr + (L - 1) * K + kq, gkl);
#pragma unroll
    for (int pp = 0; pp < 2; ++pp) {
      const int i = (tid >> 4) + 32 * pp;
      float x[8];
      unpack8_bf16(*reinterpret_cast<const uint4 *>(slot + RS_K + (i * TC_KP + kq) * 2), x);
      if (i < L) {
        float gi[8];
        ld8_shared(gr + i * K + kq, gi);
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] *= expf(p.reverse ? gi[e] : gkl[e] - gi[e]);
      }
      uint4 hi, lo;
      split8_bf16(x, hi, lo);
      *reinterpret_cast<uint4 *>(&ksh[i][kq]) = hi;
      *reinterpret_cast<uint4 *>(&ksl[i][kq]) = lo;
    }
  }
  float glast = 0.f;
  if (p.gate == GDN_GATE_G) glast = gr[L - 1];
  if (p.gate == GDN_GATE_G_GAMMA) glast = gamma * (float)L;
  if (tid < 4 * BT) {
    const int vi = tid >> 2, vq = (tid & 3) * 8;
    unsigned char *vb = buf + (KSTAGE ? 2 * TC_KS : 0);
    __nv_bfloat16(*vsh)[TC_VP] = reinterpret_cast<__nv_bfloat16(*)[TC_VP]>(vb);
    __nv_bfloat16(*vsl)[TC_VP] = reinterpret_cast<__nv_bfloat16(*)[TC_VP]>(vb + TC_VS);
    float x[8];
    unpack8_bf16(*reinterpret_cast<const uint4 *>(slot + RS_V + (vi * SP_VT + vq) * 2), x);
    float sf = p.reverse ? p.scale : 1.f;
    if (scalar_gate && vi < L) {
      const float gi = p.gate == GDN_GATE_G ? gr[vi] : gamma * (float)(vi + 1);
      sf *= expf(p.reverse ? gi : glast - gi);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] *= sf;
    if (gvg && vi < L) {
      float gi[8], gl[8];
      ld8_shared(gr + vi * SP_VT + vq, gi);
      ld8_shared(gr + (L - 1) * SP_VT + vq, gl);
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] *= expf(p.reverse ? gi[e] : gl[e] - gi[e]);
    }
    uint4 hi, lo;
    split8_bf16(x, hi, lo);
    *reinterpret_cast<uint4 *>(&vsh[vi][vq]) = hi;
    *reinterpret_cast<uint4 *>(&vsl[vi][vq]) = lo;
  }
  d.r[0] = d.r[1] = scalar_gate ? expf(glast) : 1.f;
  if (KSTAGE) {
    d.r[0] = expf(gr[(L - 1) * K + rA]);
    d.r[1] = expf(gr[(L - 1) * K + rA + 8]);
  }
#pragma unroll
  for (int j = 0; j < 4; ++j)
    d.c[j] = gvg ? expf(gr[(L - 1) * SP_VT + cl + 8 * (j >> 1) + (j & 1)]) : 1.f;
}

// RING slots; KSTAGE: the per-key gate (k~ staged; RING = 2 for its 32 KB gate
// rows); VF: states in the [V, K] layout; SPLIT: a state stored every p.split
// > 1 chunks (else every chunk).  Without KSTAGE the MMAs of a step
// read k from its ring slot, so a slot is refilled one step later (LAG = 1)
// than when only staging reads it.
template <int RING, bool KSTAGE, bool VF, bool SPLIT>
__global__ void __launch_bounds__(TC_THREADS, 1) state_pass_tc_kernel(StateParams p) {
  constexpr int LAG = KSTAGE ? 0 : 1;
  static_assert(RING >= 2 + LAG, "the ring must hold the staged, the computed and a refilled slot");
  extern __shared__ __align__(16) unsigned char tc_smem[];
  __shared__ long long seq_info[2];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, tig = lane & 3;
  const int kb = warp & 7, ch = warp >> 3;  // key block, column half
  const int v0 = blockIdx.x * SP_VT, h = blockIdx.y, n = blockIdx.z;
  const int H = p.H, V = p.V;
  constexpr int K = KMAX;
  constexpr uint32_t BUF = tc_buf_bytes(KSTAGE);
  // g_gamma: the block's per-head rate (gamma_i = rate (i + 1))
  const float gamma = p.gate == GDN_GATE_G_GAMMA ? p.gate_values[h / (H / p.HG)] : 0.f;
  const SeqInfo sq = sequence_of(p, n, tid, seq_info);
  if (!bounds_ok(n < p.N && h < p.H && v0 < p.V && sq.bos >= 0 && sq.bos <= sq.eos && sq.eos <= p.T,
                 p.err))
    return;
  unsigned char *ring = tc_smem + 2 * BUF;
  const uint32_t slot_bytes = ring_slot_bytes(p.gate);
  auto slot_of = [&](int it) { return ring + (uint32_t)(it % RING) * slot_bytes; };

  // accumulator rows rA = 16 kb + g and rA + 8, columns v0 + cl + 8 nt (+ 1)
  const int rA = 16 * kb + g, cl = 16 * ch + 2 * tig, cB = v0 + cl;
  float C[2][4];
  // element (key, column) of a [K, V] state (or [V, K] with v_first); the
  // accumulator element e of n-tile nt is (rA + 8 (e >> 1), cB + 8 nt + (e & 1))
  const size_t hbase = ((size_t)n * H + h) * K * V;
  auto at = [&](int key, int col) { return VF ? (size_t)col * K + key : (size_t)key * V + col; };
  const size_t sA = hbase + (size_t)rA * V, sB = sA + (size_t)8 * V;  // [K, V] rows rA, rA + 8
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    const int col = cB + 8 * nt;
    const bool ok = p.h0 && col < V;  // V is a multiple of 8, so col + 1 < V too
    if (VF) {
#pragma unroll
      for (int e = 0; e < 4; ++e)
        C[nt][e] = ok ? p.h0[hbase + at(rA + 8 * (e >> 1), col + (e & 1))] : 0.f;
    } else {
      C[nt][0] = ok ? p.h0[sA + col] : 0.f;
      C[nt][1] = ok ? p.h0[sA + col + 1] : 0.f;
      C[nt][2] = ok ? p.h0[sB + col] : 0.f;
      C[nt][3] = ok ? p.h0[sB + col + 1] : 0.f;
    }
  }

  // chunk of the it-th step: forward from the first, backward from the last
  auto chunk_at = [&](int it) { return p.reverse ? sq.nch - 1 - it : it; };
  auto rows_of = [&](int it) { return min(BT, sq.eos - (sq.bos + chunk_at(it) * BT)); };
  // The ring starts with steps 0 .. RING-1, one copy group each (empty past
  // the end); step it commits one more group, holding step it - LAG + RING.
#pragma unroll
  for (int j = 0; j < RING; ++j) {
    if (j < sq.nch) tc_fetch(p, sq, chunk_at(j), h, v0, tid, slot_of(j));
    ptx::cp_async_commit();
  }
  // stored chunks 0, split, 2 split, ..; the reverse pass meets them last first
  int store_i = SPLIT && p.reverse && sq.nch > 0 ? (sq.nch - 1) / p.split : 0;
  int store_c = store_i * p.split;
  TcDecay dec;
  if (sq.nch > 0) {
    ptx::cp_async_wait<RING - 2>();  // steps 0 and 1 have landed
    __syncthreads();
    tc_stage<KSTAGE>(p, slot_of(0), rows_of(0), gamma, tc_smem, tid, rA, cl, dec);
  }
  __syncthreads();
#pragma unroll 1
  for (int it = 0; it < sq.nch; ++it) {
    const int c = chunk_at(it);
    bool store = true;
    long long slot = sq.first + c;
    if (SPLIT) {
      store = c == store_c;
      slot = sq.first + store_i;
      if (store) {
        store_c += p.reverse ? -p.split : p.split;
        store_i += p.reverse ? -1 : 1;
      }
    }

    // chunk-start state: two columns per 8-column tile and row; one element
    // at a time in the [V, K] layout
    if (VF && sq.write_hs && store) {
      const size_t sb = ((size_t)slot * H + h) * K * V;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int col = cB + 8 * nt;
        if (col >= V) continue;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const size_t o = sb + at(rA + 8 * (e >> 1), col + (e & 1));
          if (p.hs_bf16)
            static_cast<__nv_bfloat16 *>(p.hs)[o] = __float2bfloat16_rn(C[nt][e]);
          else
            static_cast<float *>(p.hs)[o] = C[nt][e];
        }
      }
    } else if (!VF && sq.write_hs && store) {
      const size_t oA = (((size_t)slot * H + h) * K + rA) * V, oB = oA + (size_t)8 * V;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int col = cB + 8 * nt;
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

    // decay: rows by e^{g_L} e^{gk_L[row]}, columns by e^{gv_L[col]}
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      C[nt][0] *= dec.r[0] * dec.c[2 * nt];
      C[nt][1] *= dec.r[0] * dec.c[2 * nt + 1];
      C[nt][2] *= dec.r[1] * dec.c[2 * nt];
      C[nt][3] *= dec.r[1] * dec.c[2 * nt + 1];
    }

    // the next step's operands into the other buffer; the slot of step
    // it - LAG (read out before the last barrier) takes step it - LAG + RING
    if (it + 1 < sq.nch)
      tc_stage<KSTAGE>(p, slot_of(it + 1), rows_of(it + 1), gamma,
                       tc_smem + ((it + 1) & 1) * BUF, tid, rA, cl, dec);
    if (it >= LAG && it - LAG + RING < sq.nch)
      tc_fetch(p, sq, chunk_at(it - LAG + RING), h, v0, tid, slot_of(it - LAG));
    ptx::cp_async_commit();

    // C += k~^T v~ over the chunk's 64 rows, 16 at a time (rows past its end
    // are zeros).  A = k~^T (16 keys x 16 tokens) and B = v~ (16 tokens x 16
    // columns) come from token-major tiles by transposing ldmatrix.
    const unsigned char *buf = tc_smem + (it & 1) * BUF;
    const __nv_bfloat16(*ksh)[TC_KP] = reinterpret_cast<const __nv_bfloat16(*)[TC_KP]>(
        KSTAGE ? buf : slot_of(it) + RS_K);
    const __nv_bfloat16(*ksl)[TC_KP] = reinterpret_cast<const __nv_bfloat16(*)[TC_KP]>(buf + TC_KS);
    const unsigned char *vb = buf + (KSTAGE ? 2 * TC_KS : 0);
    const __nv_bfloat16(*vsh)[TC_VP] = reinterpret_cast<const __nv_bfloat16(*)[TC_VP]>(vb);
    const __nv_bfloat16(*vsl)[TC_VP] = reinterpret_cast<const __nv_bfloat16(*)[TC_VP]>(vb + TC_VS);
#pragma unroll
    for (int kt = 0; kt < 4; ++kt) {
      uint32_t ah[4], al[4], bh[4], bl[4];
      const int arow = 16 * kt + (lane & 7) + ((lane >> 4) << 3);
      const int key = 16 * kb + ((lane >> 3) & 1) * 8;
      ptx::ldmatrix_x4_trans(&ksh[arow][key], ah[0], ah[1], ah[2], ah[3]);
      if (KSTAGE) ptx::ldmatrix_x4_trans(&ksl[arow][key], al[0], al[1], al[2], al[3]);
      const int brow = 16 * kt + (lane & 7) + (((lane >> 3) & 1) << 3);
      const int col = 16 * ch + ((lane >> 4) << 3);
      ptx::ldmatrix_x4_trans(&vsh[brow][col], bh[0], bh[1], bh[2], bh[3]);
      ptx::ldmatrix_x4_trans(&vsl[brow][col], bl[0], bl[1], bl[2], bl[3]);
      ptx::mma_16816_bf16(C[0], ah, bh[0], bh[1]);
      ptx::mma_16816_bf16(C[1], ah, bh[2], bh[3]);
      ptx::mma_16816_bf16(C[0], ah, bl[0], bl[1]);
      ptx::mma_16816_bf16(C[1], ah, bl[2], bl[3]);
      if (KSTAGE) {
        ptx::mma_16816_bf16(C[0], al, bh[0], bh[1]);
        ptx::mma_16816_bf16(C[1], al, bh[2], bh[3]);
      }
    }
    // step it + 2's copies have landed (this thread's); the barrier makes them
    // and the staged buffer visible and frees this step's buffer and slot
    ptx::cp_async_wait<RING - 2 - LAG>();
    __syncthreads();
  }
  ptx::cp_async_wait<0>();  // no copy outlives the block

  if (p.ht) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int col = cB + 8 * nt;
      if (col >= V) continue;
      if (VF) {
#pragma unroll
        for (int e = 0; e < 4; ++e) p.ht[hbase + at(rA + 8 * (e >> 1), col + (e & 1))] = C[nt][e];
      } else {
        p.ht[sA + col] = C[nt][0];
        p.ht[sA + col + 1] = C[nt][1];
        p.ht[sB + col] = C[nt][2];
        p.ht[sB + col + 1] = C[nt][3];
      }
    }
  }
}

}  // namespace

cudaError_t launch_state_pass(const StateParams &p, bool bf16, cudaStream_t stream) {
  if (state_pass_tc5_supported(p, bf16)) return launch_state_pass_tc5(p, stream);
  const dim3 grid((unsigned)((p.V + SP_VT - 1) / SP_VT), (unsigned)p.H, (unsigned)p.N);
  if (bf16 && p.K == KMAX) {
    // per-key gate: k~ staged, two ring slots (its gate rows are 32 KB a
    // chunk); otherwise six slots, four steps of copies in flight
    const bool kstage = p.gate == GDN_GATE_GK;
    const int ring = kstage ? 2 : 6;
    const int smem = (int)(2 * tc_buf_bytes(kstage) + ring * ring_slot_bytes(p.gate));
    const bool split = p.split > 1;
    auto pick = [&](auto k00, auto k01, auto k10, auto k11) {
      return p.v_first ? (split ? k11 : k10) : (split ? k01 : k00);
    };
    auto kern = kstage ? pick(state_pass_tc_kernel<2, true, false, false>,
                              state_pass_tc_kernel<2, true, false, true>,
                              state_pass_tc_kernel<2, true, true, false>,
                              state_pass_tc_kernel<2, true, true, true>)
                       : pick(state_pass_tc_kernel<6, false, false, false>,
                              state_pass_tc_kernel<6, false, false, true>,
                              state_pass_tc_kernel<6, false, true, false>,
                              state_pass_tc_kernel<6, false, true, true>);
    const cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, TC_THREADS, smem, stream>>>(p);
  } else if (bf16) {
    state_pass_kernel<__nv_bfloat16><<<grid, SP_THREADS, 0, stream>>>(p);
  } else {
    state_pass_kernel<float><<<grid, SP_THREADS, 0, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace gdn
