// Decode step (T = 1..4 tokens) against a pooled bf16 state, HBM-streaming.
//
// FlashInfer gdn_decode_bf16_state.py (compute_single_gate,
// normalize_and_store_qk_to_smem, the per-token helpers and the public
// gated_delta_rule) gives the arithmetic: per token
//   g = -exp(A_log) softplus(a + dt_bias), beta = sigmoid(b),
//   q^ = scale q / sqrt(|q|^2 + eps), k^ = k / sqrt(|k|^2 + eps),
//   S <- e^g S;  delta = beta (v - S k^);  S <- S + delta k^T;  o = S q^.
//
// Design (ours): a persistent kernel, two CTAs of 256 threads per SM.  Each
// CTA walks (batch entry, value head) items; for every item one thread issues
// bulk (TMA) copies of the 32 KB state slot and of the q/k/v rows into a
// shared-memory stage, NSTAGE items ahead, so the HBM stream never waits on
// arithmetic.  Thread t owns rows {t/8 + 32 i : i < 4} of the [V, K] state and
// the 16 columns {8 (t%8) + j, 64 + 8 (t%8) + j : j < 8}: every quarter-warp
// reads (and later writes) 128 contiguous bytes, bank-conflict free, and row
// sums need three butterfly shuffles.  All T tokens run on fp32 registers
// and the slot is written back once, rounded to bf16 (round to nearest even).
// Per token the two dot products are taken in one pass over the undecayed
// state and the decay is folded in afterwards:
//   pred = e^g (S k^),   (S q^) after the update = e^g (S q^) + delta (k^ . q^).
#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "ptx.cuh"

namespace gdn {
namespace {

constexpr int DK = 128, DV = 128, DTHREADS = 256, DTMAX = 4;
constexpr uint32_t SLOT_BYTES = DK * DV * 2;    // 32 KB bf16 state slot
constexpr uint32_t ROW_BYTES = DK * 2;          // one q/k/v row (256 B)
constexpr int ROWS_PER_THREAD = 4;

template <int T>
struct DecodeSmem {
  static constexpr uint32_t STAGE_BYTES = SLOT_BYTES + 3 * T * ROW_BYTES;
  static constexpr int NSTAGE = T <= 2 ? 3 : 2;
  static constexpr size_t BYTES = (size_t)NSTAGE * STAGE_BYTES + 3 * DTMAX * DK * 4 + 256;
};

__device__ __forceinline__ float softplus_f(float x, float beta, float thr) {
  const float bx = beta * x;
  return bx <= thr ? log1pf(expf(bx)) / beta : x;
}

template <int T>
__global__ void __launch_bounds__(DTHREADS, 2) decode_kernel(DecodeParams p) {
  using L = DecodeSmem<T>;
  constexpr int NSTAGE = L::NSTAGE;
  extern __shared__ __align__(128) unsigned char smem[];
  // stage s: [state 32 KB][q rows][k rows][v rows]
  float *qs = reinterpret_cast<float *>(smem + (size_t)NSTAGE * L::STAGE_BYTES);
  float *ks = qs + DTMAX * DK;
  float *vs = ks + DTMAX * DK;
  uint64_t *full = reinterpret_cast<uint64_t *>(vs + DTMAX * DK);
  int *slot_s = reinterpret_cast<int *>(full + NSTAGE);
  float *gexp_s = reinterpret_cast<float *>(slot_s + NSTAGE);
  float *beta_s = gexp_s + DTMAX;
  float *kq_s = beta_s + DTMAX;

  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int rg = tid >> 3;   // row group: rows rg + 32 i
  const int cs = tid & 7;    // column slice: pieces cs and cs + 8
  const int HV = p.HV;
  const int nitems = p.B * HV;

  const __nv_bfloat16 *q = static_cast<const __nv_bfloat16 *>(p.q);
  const __nv_bfloat16 *k = static_cast<const __nv_bfloat16 *>(p.k);
  const __nv_bfloat16 *v = static_cast<const __nv_bfloat16 *>(p.v);
  const __nv_bfloat16 *ga = static_cast<const __nv_bfloat16 *>(p.a);
  const __nv_bfloat16 *gb = static_cast<const __nv_bfloat16 *>(p.b);
  __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(p.o);
  __nv_bfloat16 *state = static_cast<__nv_bfloat16 *>(p.state);

  // Producer: fill stage s with item `item` (thread 0 only).
  auto issue = [&](int item, int s) {
    const int bi = item / HV, hv = item % HV, hk = hv / (HV / p.H);
    const int slot = p.slot_indices ? p.slot_indices[bi] : bi;
    unsigned char *st = smem + (size_t)s * L::STAGE_BYTES;
    if (slot < 0 || slot >= p.pool) {
      slot_s[s] = -1;
      ptx::mbar_arrive(&full[s]);
      return;
    }
    slot_s[s] = slot;
    ptx::mbar_arrive_expect_tx(&full[s], L::STAGE_BYTES);
    ptx::bulk_g2s(st, state + ((size_t)slot * HV + hv) * DV * DK, SLOT_BYTES, &full[s]);
#pragma unroll
    for (int t = 0; t < T; ++t) {
      const size_t qk_off = (((size_t)bi * T + t) * p.H + hk) * DK;
      const size_t v_off = (((size_t)bi * T + t) * HV + hv) * DV;
      ptx::bulk_g2s(st + SLOT_BYTES + t * ROW_BYTES, q + qk_off, ROW_BYTES, &full[s]);
      ptx::bulk_g2s(st + SLOT_BYTES + (T + t) * ROW_BYTES, k + qk_off, ROW_BYTES, &full[s]);
      ptx::bulk_g2s(st + SLOT_BYTES + (2 * T + t) * ROW_BYTES, v + v_off, ROW_BYTES, &full[s]);
    }
  };

  if (tid == 0) {
    for (int s = 0; s < NSTAGE; ++s) ptx::mbar_init(&full[s], 1);
    ptx::fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      const int item = blockIdx.x + s * gridDim.x;
      if (item < nitems) issue(item, s);
    }
  }

  for (int it = 0;; ++it) {
    const int item = blockIdx.x + it * gridDim.x;
    if (item >= nitems) break;
    const int s = it % NSTAGE;
    const uint32_t parity = (uint32_t)((it / NSTAGE) & 1);
    const int bi = item / HV, hv = item % HV;
    const bool arrived = ptx::mbar_wait_bounded(&full[s], parity);
    if (!__syncthreads_and(arrived)) {
      if (tid == 0) record_error(p.err, GDN_ERR_TIMEOUT);
      return;
    }
    const unsigned char *st = smem + (size_t)s * L::STAGE_BYTES;
    const int slot = slot_s[s];
    if (slot < 0) {
      if (tid == 0) record_error(p.err, GDN_ERR_BAD_SLOT);
      for (int idx = tid; idx < T * DV; idx += DTHREADS)
        o[(((size_t)bi * T + idx / DV) * HV + hv) * DV + idx % DV] = __float2bfloat16_rn(0.f);
      __syncthreads();
      if (tid == 0 && item + NSTAGE * (int)gridDim.x < nitems)
        issue(item + NSTAGE * gridDim.x, s);
      continue;
    }

    // ---- gates, normalised q/k, v: stage -> fp32 shared arrays
    if (tid < T) {
      const size_t gi = ((size_t)bi * T + tid) * HV + hv;
      const float x = __bfloat162float(ga[gi]) + p.dt_bias[hv];
      const float g = -expf(p.A_log[hv]) * softplus_f(x, p.softplus_beta, p.softplus_threshold);
      gexp_s[tid] = expf(g);
      beta_s[tid] = 1.f / (1.f + expf(-__bfloat162float(gb[gi])));
    }
    const __nv_bfloat16 *sq = reinterpret_cast<const __nv_bfloat16 *>(st + SLOT_BYTES);
    if (warp < 2 * T) {
      const int t = warp >> 1;
      const bool is_k = warp & 1;
      const __nv_bfloat16 *src = sq + (is_k ? T + t : t) * DK;
      float x[DK / 32];
      float ss = 0.f;
#pragma unroll
      for (int i = 0; i < DK / 32; ++i) {
        x[i] = __bfloat162float(src[lane + 32 * i]);
        ss = fmaf(x[i], x[i], ss);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
      float f = p.use_qk_l2norm ? rsqrtf(ss + p.eps) : 1.f;
      if (!is_k) f *= p.scale;
      float *dst = is_k ? ks + t * DK : qs + t * DK;
#pragma unroll
      for (int i = 0; i < DK / 32; ++i) dst[lane + 32 * i] = x[i] * f;
    }
    for (int idx = tid; idx < T * DV; idx += DTHREADS)
      vs[idx] = __bfloat162float(sq[2 * T * DK + idx]);

    // ---- state slice: stage -> fp32 registers
    float S[ROWS_PER_THREAD][16];
    const __nv_bfloat16 *ss_ = reinterpret_cast<const __nv_bfloat16 *>(st);
#pragma unroll
    for (int i = 0; i < ROWS_PER_THREAD; ++i) {
      const int row = rg + 32 * i;
#pragma unroll
      for (int pc = 0; pc < 2; ++pc) {
        const uint4 raw = *reinterpret_cast<const uint4 *>(ss_ + row * DK + (cs + 8 * pc) * 8);
        const __nv_bfloat162 *h2 = reinterpret_cast<const __nv_bfloat162 *>(&raw);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f2 = __bfloat1622float2(h2[e]);
          S[i][pc * 8 + 2 * e] = f2.x;
          S[i][pc * 8 + 2 * e + 1] = f2.y;
        }
      }
    }
    __syncthreads();  // stage s fully consumed; q/k/v/gates published
    if (tid == 0 && item + NSTAGE * (int)gridDim.x < nitems) {
      ptx::fence_proxy_async_smem();
      issue(item + NSTAGE * gridDim.x, s);
    }
    if (warp < T) {
      float d = 0.f;
#pragma unroll
      for (int i = 0; i < DK / 32; ++i)
        d = fmaf(ks[warp * DK + lane + 32 * i], qs[warp * DK + lane + 32 * i], d);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
      if (lane == 0) kq_s[warp] = d;
    }
    __syncthreads();

#pragma unroll
    for (int t = 0; t < T; ++t) {
      const float ge = gexp_s[t], be = beta_s[t], kq = kq_s[t];
      float pk[ROWS_PER_THREAD], pq[ROWS_PER_THREAD];
#pragma unroll
      for (int i = 0; i < ROWS_PER_THREAD; ++i) pk[i] = pq[i] = 0.f;
#pragma unroll
      for (int pc = 0; pc < 2; ++pc) {
        const float4 *kp = reinterpret_cast<const float4 *>(ks + t * DK + (cs + 8 * pc) * 8);
        const float4 *qp = reinterpret_cast<const float4 *>(qs + t * DK + (cs + 8 * pc) * 8);
        const float4 k0 = kp[0], k1 = kp[1], q0 = qp[0], q1 = qp[1];
        const float kr[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
        const float qr[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
        for (int i = 0; i < ROWS_PER_THREAD; ++i)
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            pk[i] = fmaf(S[i][pc * 8 + e], kr[e], pk[i]);
            pq[i] = fmaf(S[i][pc * 8 + e], qr[e], pq[i]);
          }
      }
#pragma unroll
      for (int off = 1; off < 8; off <<= 1)
#pragma unroll
        for (int i = 0; i < ROWS_PER_THREAD; ++i) {
          pk[i] += __shfl_xor_sync(0xffffffffu, pk[i], off);
          pq[i] += __shfl_xor_sync(0xffffffffu, pq[i], off);
        }
      float delta[ROWS_PER_THREAD];
#pragma unroll
      for (int i = 0; i < ROWS_PER_THREAD; ++i)
        delta[i] = be * (vs[t * DV + rg + 32 * i] - ge * pk[i]);
#pragma unroll
      for (int pc = 0; pc < 2; ++pc) {
        const float4 *kp = reinterpret_cast<const float4 *>(ks + t * DK + (cs + 8 * pc) * 8);
        const float4 k0 = kp[0], k1 = kp[1];
        const float kr[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
#pragma unroll
        for (int i = 0; i < ROWS_PER_THREAD; ++i)
#pragma unroll
          for (int e = 0; e < 8; ++e)
            S[i][pc * 8 + e] = fmaf(ge, S[i][pc * 8 + e], delta[i] * kr[e]);
      }
      // lane cs == i writes row rg + 32 i of this token's output
#pragma unroll
      for (int i = 0; i < ROWS_PER_THREAD; ++i)
        if (cs == i)
          o[(((size_t)bi * T + t) * HV + hv) * DV + rg + 32 * i] =
              __float2bfloat16_rn(fmaf(delta[i], kq, ge * pq[i]));
    }

    // ---- write the slot back once
    __nv_bfloat16 *dst = state + ((size_t)slot * HV + hv) * DV * DK;
#pragma unroll
    for (int i = 0; i < ROWS_PER_THREAD; ++i) {
      const int row = rg + 32 * i;
#pragma unroll
      for (int pc = 0; pc < 2; ++pc) {
        uint4 w;
        __nv_bfloat162 *h2 = reinterpret_cast<__nv_bfloat162 *>(&w);
#pragma unroll
        for (int e = 0; e < 4; ++e)
          h2[e] = __floats2bfloat162_rn(S[i][pc * 8 + 2 * e], S[i][pc * 8 + 2 * e + 1]);
        *reinterpret_cast<uint4 *>(dst + row * DK + (cs + 8 * pc) * 8) = w;
      }
    }
    __syncthreads();  // q/k/v/gate arrays are rewritten by the next item
  }
}

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

template <int T>
cudaError_t launch_t(const DecodeParams &p, cudaStream_t stream) {
  const size_t bytes = DecodeSmem<T>::BYTES;
  cudaError_t e = cudaFuncSetAttribute(decode_kernel<T>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  const int items = p.B * p.HV;
  const int grid = items < 2 * sm_count() ? items : 2 * sm_count();
  decode_kernel<T><<<grid, DTHREADS, bytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeParams &p, cudaStream_t stream) {
  switch (p.T) {
    case 1: return launch_t<1>(p, stream);
    case 2: return launch_t<2>(p, stream);
    case 3: return launch_t<3>(p, stream);
    case 4: return launch_t<4>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gdn
