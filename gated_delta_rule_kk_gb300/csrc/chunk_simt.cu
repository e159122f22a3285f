// Chunked forward on the CUDA cores (fp32 FFMA), both gate kinds.
//
// One CTA owns one (sequence, value head, 32-wide V tile) chain and walks its
// 64-token chunks in order, keeping the fp32 state tile h[K, 32] in shared
// memory for the whole sequence.  Per chunk it computes, without touching
// HBM for anything but the inputs and the output:
//   gamma   chunk-local inclusive cumsum of the log-gates
//   A, Aqk  beta_i k_i.k_j exp(gamma_i - gamma_j) (i > j) and
//           scale q_i.k_j exp(gamma_i - gamma_j) (i >= j)
//           (sglang fla/chunk_fwd.py, fused KK^T + solve kernel, Steps 1-2;
//            per-channel factors as in vLLM kimi_k3 kda/chunk_intra,
//            chunk_kda_fwd_kernel_inter_solve_fused)
//   T       (I + A)^-1 by forward substitution in fp32 (Step 3 of the same
//           kernel, done over the whole 64x64 block column by column)
//   w, u    T diag(beta) (k exp(gamma)), T diag(beta) v      (WY vectors)
//   v_new   u - w h;  o = (scale q exp(gamma)) h + Aqk v_new
//   h       diag(exp(gamma_L)) h + (k exp(gamma_L - gamma))^T v_new
//           (KDA _fla/ops/common/chunk_h.py, chunk_fwd_kernel_h: decay by
//            the last row's gate, keys scaled by exp(g_last - g))
// This is the exact-fp32 path (fp32 inputs, and any K <= 128, V).  bf16
// inputs are widened on load.
#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int THREADS = 256;
constexpr int VT = 32;      // V columns per CTA
constexpr int LDA = BT + 1; // row stride of the 64x64 matrices

__host__ __device__ inline size_t smem_floats(int K, bool kda) {
  const int KS = K + 1, VS = VT + 1;
  size_t n = 3 * (size_t)BT * KS;            // q, k, w
  if (kda) n += (size_t)BT * KS;             // gamma / beta k exp(gamma)
  n += 3 * (size_t)BT * LDA;                 // A, Aqk, T
  n += 2 * (size_t)BT * VS;                  // v tile, u / v_new
  n += (size_t)K * VS;                       // state tile
  n += 3 * BT + KMAX;                        // gamma, beta, d, gamma_L
  return n;
}

template <typename T, bool KDA>
__global__ void __launch_bounds__(THREADS, 1) chunk_fwd_simt_kernel(ChunkParams p) {
  extern __shared__ float smem[];
  const int tid = threadIdx.x;
  const int v0 = blockIdx.x * VT;
  const int h = blockIdx.y;
  const int n = blockIdx.z;
  const int hk = h / (p.H / p.Hk);
  const int K = p.K, V = p.V, H = p.H, Hk = p.Hk;
  const int KS = K + 1, VS = VT + 1;

  int b, bos, eos;
  if (p.cu_seqlens) {
    b = 0;
    bos = p.cu_seqlens[n];
    eos = p.cu_seqlens[n + 1];
    const bool bad = bos < 0 || eos < bos || eos > p.T || (n == 0 && bos != 0) ||
                     (n == p.N - 1 && eos != p.T);
    if (bad) {
      if (tid == 0) record_error(p.err, GDN_ERR_BAD_SEQLENS);
      return;
    }
  } else {
    b = n;
    bos = 0;
    eos = p.T;
  }
  if (!bounds_ok(n < p.N && b >= 0 && b < p.B && h < H && hk < Hk && v0 < V && bos >= 0 &&
                     bos <= eos && eos <= p.T,
                 p.err))
    return;

  const T *q = static_cast<const T *>(p.q);
  const T *k = static_cast<const T *>(p.k);
  const T *v = static_cast<const T *>(p.v);
  T *o = static_cast<T *>(p.o);

  float *qS = smem;
  float *kS = qS + BT * KS;
  float *wS = kS + BT * KS;
  float *xS = wS + BT * KS;                   // KDA only
  float *AS = xS + (KDA ? BT * KS : 0);
  float *QS = AS + BT * LDA;
  float *TS = QS + BT * LDA;
  float *vS = TS + BT * LDA;
  float *uS = vS + BT * VS;
  float *hS = uS + BT * VS;
  float *gam = hS + K * VS;
  float *bet = gam + BT;
  float *dS = bet + BT;
  float *gL = dS + BT;

  // initial state tile
  for (int idx = tid; idx < K * VT; idx += THREADS) {
    const int c = idx / VT, j = idx % VT;
    float x = 0.f;
    if (p.h0 && v0 + j < V)
      x = p.v_first ? p.h0[(((size_t)n * H + h) * V + v0 + j) * K + c]
                    : p.h0[(((size_t)n * H + h) * K + c) * V + v0 + j];
    hS[c * VS + j] = x;
  }

  for (int s = bos; s < eos; s += BT) {
    const int L = min(BT, eos - s);
    const size_t row0 = (size_t)b * p.T + s;

    // ---- load the chunk (rows >= L are zero)
    for (int idx = tid; idx < BT * K; idx += THREADS) {
      const int i = idx / K, c = idx % K;
      float qv = 0.f, kv = 0.f, gv = 0.f;
      if (i < L) {
        const size_t off = ((row0 + i) * Hk + hk) * K + c;
        qv = to_f32(q[off]);
        kv = to_f32(k[off]);
        if (KDA) gv = p.g[((row0 + i) * H + h) * K + c];
      }
      qS[i * KS + c] = qv;
      kS[i * KS + c] = kv;
      if (KDA) xS[i * KS + c] = gv;
    }
    for (int idx = tid; idx < BT * VT; idx += THREADS) {
      const int i = idx / VT, j = idx % VT;
      float x = 0.f;
      if (i < L && v0 + j < V) x = to_f32(v[((row0 + i) * H + h) * V + v0 + j]);
      vS[i * VS + j] = x;
    }
    if (tid < BT) {
      bet[tid] = tid < L ? p.beta[(row0 + tid) * H + h] : 0.f;
      if (!KDA) gam[tid] = tid < L ? p.g[(row0 + tid) * H + h] : 0.f;
    }
    __syncthreads();

    // ---- chunk-local inclusive cumsum of the gates; padded rows repeat row L-1
    if (!KDA) {
      if (tid < 32) {
        float a0 = gam[2 * tid], a1 = gam[2 * tid + 1];
        if (p.g_is_cumsum) {
          // already cumulative: only flatten the padding
          const float last = gam[L - 1];
          if (2 * tid >= L) a0 = last;
          if (2 * tid + 1 >= L) a1 = last;
          gam[2 * tid] = a0;
          gam[2 * tid + 1] = a1;
        } else {
          const float pair = a0 + a1;
          float incl = pair;
#pragma unroll
          for (int off = 1; off < 32; off <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, incl, off);
            if (tid >= off) incl += y;
          }
          const float excl = incl - pair;
          gam[2 * tid] = excl + a0;
          gam[2 * tid + 1] = excl + a0 + a1;
        }
      }
    } else {
      for (int c = tid; c < K; c += THREADS) {
        if (p.g_is_cumsum) {
          const float last = xS[(L - 1) * KS + c];
          for (int i = L; i < BT; ++i) xS[i * KS + c] = last;
        } else {
          float acc = 0.f;
          for (int i = 0; i < BT; ++i) {
            acc += xS[i * KS + c];
            xS[i * KS + c] = acc;
          }
        }
      }
    }
    __syncthreads();
    if (KDA) {
      for (int c = tid; c < K; c += THREADS) gL[c] = xS[(L - 1) * KS + c];
    }

    // ---- A (strictly lower, times beta) and Aqk (lower, times scale)
    for (int idx = tid; idx < BT * BT; idx += THREADS) {
      const int i = idx >> 6, j = idx & 63;
      float a = 0.f, aq = 0.f;
      if (i < L && j <= i) {
        float dkk = 0.f, dqk = 0.f;
        if (!KDA) {
          for (int c = 0; c < K; ++c) {
            const float kj = kS[j * KS + c];
            dkk = fmaf(kS[i * KS + c], kj, dkk);
            dqk = fmaf(qS[i * KS + c], kj, dqk);
          }
          const float f = expf(gam[i] - gam[j]);
          a = (j < i) ? bet[i] * f * dkk : 0.f;
          aq = p.scale * f * dqk;
        } else {
          for (int c = 0; c < K; ++c) {
            const float e = expf(xS[i * KS + c] - xS[j * KS + c]);
            const float kj = kS[j * KS + c] * e;
            dkk = fmaf(kS[i * KS + c], kj, dkk);
            dqk = fmaf(qS[i * KS + c], kj, dqk);
          }
          a = (j < i) ? bet[i] * dkk : 0.f;
          aq = p.scale * dqk;
        }
      }
      AS[i * LDA + j] = a;
      QS[i * LDA + j] = aq;
    }
    __syncthreads();

    // ---- T = (I + A)^-1: thread j forward-substitutes column j
    if (tid < BT) {
      const int j = tid;
      for (int i = 0; i < BT; ++i) {
        float x = (i == j) ? 1.f : 0.f;
        if (i > j) {
          for (int m = j; m < i; ++m) x = fmaf(-AS[i * LDA + m], TS[m * LDA + j], x);
        }
        TS[i * LDA + j] = x;
      }
    } else if (!KDA && tid < 2 * BT) {
      const int j = tid - BT;
      dS[j] = bet[j] * expf(gam[j]);
    }
    __syncthreads();

    // ---- WY vectors: w = T diag(beta) (k exp(gamma)), u = T diag(beta) v;
    //      then the operands of the state pass are rescaled in place.
    if (KDA) {
      for (int idx = tid; idx < BT * K; idx += THREADS) {
        const int i = idx / K, c = idx % K;
        const float g_ic = xS[i * KS + c];
        const float kv = kS[i * KS + c];
        xS[i * KS + c] = bet[i] * kv * expf(g_ic);
        kS[i * KS + c] = kv * expf(gL[c] - g_ic);
        qS[i * KS + c] = p.scale * qS[i * KS + c] * expf(g_ic);
      }
      __syncthreads();
      for (int idx = tid; idx < BT * K; idx += THREADS) {
        const int i = idx / K, c = idx % K;
        float acc = 0.f;
        for (int j = 0; j <= i; ++j) acc = fmaf(TS[i * LDA + j], xS[j * KS + c], acc);
        wS[i * KS + c] = acc;
      }
    } else {
      for (int idx = tid; idx < BT * K; idx += THREADS) {
        const int i = idx / K, c = idx % K;
        float acc = 0.f;
        for (int j = 0; j <= i; ++j) acc = fmaf(TS[i * LDA + j] * dS[j], kS[j * KS + c], acc);
        wS[i * KS + c] = acc;
      }
    }
    for (int idx = tid; idx < BT * VT; idx += THREADS) {
      const int i = idx / VT, j = idx % VT;
      float acc = 0.f;
      for (int m = 0; m <= i; ++m) acc = fmaf(TS[i * LDA + m] * bet[m], vS[m * VS + j], acc);
      uS[i * VS + j] = acc;
    }
    __syncthreads();
    if (!KDA) {
      const float gl = gam[L - 1];
      for (int idx = tid; idx < BT * K; idx += THREADS) {
        const int i = idx / K, c = idx % K;
        kS[i * KS + c] *= expf(gl - gam[i]);
        qS[i * KS + c] *= p.scale * expf(gam[i]);
      }
    }
    // (the w/u loops above only read kS and qS; their rescaling is safe
    //  after the barrier below and before the state pass reads them)
    __syncthreads();

    // ---- v_new = u - w h
    for (int idx = tid; idx < BT * VT; idx += THREADS) {
      const int i = idx / VT, j = idx % VT;
      float acc = uS[i * VS + j];
      for (int c = 0; c < K; ++c) acc = fmaf(-wS[i * KS + c], hS[c * VS + j], acc);
      uS[i * VS + j] = acc;
    }
    __syncthreads();

    // ---- o = q~ h + Aqk v_new ; h' = decay h + k~^T v_new
    for (int idx = tid; idx < BT * VT; idx += THREADS) {
      const int i = idx / VT, j = idx % VT;
      if (i < L && v0 + j < V) {
        float acc = 0.f;
        for (int c = 0; c < K; ++c) acc = fmaf(qS[i * KS + c], hS[c * VS + j], acc);
        for (int m = 0; m <= i; ++m) acc = fmaf(QS[i * LDA + m], uS[m * VS + j], acc);
        const size_t oi = ((row0 + i) * H + h) * V + v0 + j;
        if (p.o_f32)
          static_cast<float *>(p.o)[oi] = acc;
        else
          o[oi] = from_f32<T>(acc);
      }
    }
    float hn[(KMAX * VT) / THREADS];
#pragma unroll
    for (int r = 0; r < (KMAX * VT) / THREADS; ++r) {
      const int idx = tid + r * THREADS;
      if (idx < K * VT) {
        const int c = idx / VT, j = idx % VT;
        const float decay = KDA ? expf(gL[c]) : expf(gam[L - 1]);
        float acc = decay * hS[c * VS + j];
        for (int m = 0; m < L; ++m) acc = fmaf(kS[m * KS + c], uS[m * VS + j], acc);
        hn[r] = acc;
      }
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < (KMAX * VT) / THREADS; ++r) {
      const int idx = tid + r * THREADS;
      if (idx < K * VT) hS[(idx / VT) * VS + idx % VT] = hn[r];
    }
    __syncthreads();
  }

  if (p.ht) {
    for (int idx = tid; idx < K * VT; idx += THREADS) {
      const int c = idx / VT, j = idx % VT;
      if (v0 + j >= V) continue;
      const size_t at = p.v_first ? (((size_t)n * H + h) * V + v0 + j) * K + c
                                  : (((size_t)n * H + h) * K + c) * V + v0 + j;
      p.ht[at] = hS[c * VS + j];
    }
  }
}

template <typename T, bool KDA>
cudaError_t launch_typed(const ChunkParams &p, cudaStream_t stream) {
  const size_t bytes = smem_floats(p.K, KDA) * sizeof(float);
  auto kern = chunk_fwd_simt_kernel<T, KDA>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)bytes);
  if (e != cudaSuccess) return e;
  dim3 grid((p.V + VT - 1) / VT, p.H, p.N);
  kern<<<grid, THREADS, bytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_chunk_simt(const ChunkParams &p, bool bf16, bool kda, cudaStream_t stream) {
  if (bf16) {
    return kda ? launch_typed<__nv_bfloat16, true>(p, stream)
               : launch_typed<__nv_bfloat16, false>(p, stream);
  }
  return kda ? launch_typed<float, true>(p, stream) : launch_typed<float, false>(p, stream);
}

}  // namespace gdn
