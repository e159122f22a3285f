// Decode step (T = 1..4 tokens) against a pooled bf16 state, HBM-streaming.
//
// FlashInfer gdn_decode_bf16_state.py (compute_single_gate,
// normalize_and_store_qk_to_smem, the per-token helpers and the public
// gated_delta_rule) gives the arithmetic: per token
//   g = -exp(A_log) softplus(a + dt_bias), beta = sigmoid(b),
//   q^ = scale q / sqrt(|q|^2 + eps), k^ = k / sqrt(|k|^2 + eps),
//   S <- e^g S;  delta = beta (v - S k^);  S <- S + delta k^T;  o = S q^.
//
// Design (ours): a persistent kernel, two CTAs of eight warps per SM, with no
// block-wide barrier inside the item loop.  Each CTA walks (batch entry,
// value head) items through a ring of NSTAGE shared-memory stages; a stage
// holds the 32 KB state slot, the q/k/v rows and a small header (the slot
// index), filled by bulk (TMA) copies NSTAGE items ahead.  Thread t owns rows
// {t/8 + 32 i : i < 4} of the [V, K] state and the 16 columns
// {8 (t%8) + j, 64 + 8 (t%8) + j : j < 8}: every quarter-warp touches 128
// contiguous bytes (bank-conflict free), and the eight column slices of a row
// group sit in one warp, so the L2 norms, k^.q^ and the row sums are
// three-step butterfly shuffles.  Warps run independently: each counts
// itself out of a stage with one shared-memory atomic, and the last warp out
// issues the refill.  Gate inputs are prefetched into registers one item
// ahead and the gates are computed warp-locally.  q and k enter raw: the four
// row groups of a warp split the tokens' norms and k.q, and the L2 factors are
// applied to row sums.  All T tokens run on fp32 registers with packed
// two-lane FMAs, holding S / c for a running decay scale c (the product of
// the gates so far), so a token costs three FMAs per state element:
//   y_k = (S/c) k,  y_q = (S/c) q,
//   delta = beta (v - c e^g fk y_k),  o = c e^g fq y_q + delta (k^ . q^),
//   S/c' += (delta fk / c') k  with c' = c e^g;
// when c' would fall below 2^-40 the scale is folded back into the registers.
// Row sums are a reduce-scatter over the eight column lanes.  The slot is
// written back once, times c, rounded to bf16 (round to nearest even).
#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "ptx.cuh"

namespace gdn {
namespace {

constexpr int DK = 128, DV = 128;
constexpr int NWARPS = 8, DTHREADS = NWARPS * 32;
constexpr uint32_t SLOT_BYTES = DK * DV * 2;  // 32 KB bf16 state slot
constexpr uint32_t ROW_BYTES = DK * 2;        // one q/k/v row (256 B)
constexpr int ROWS_PER_THREAD = 4;

template <int T>
struct DecodeSmem {
  // stage: [state 32 KB][q rows][k rows][v rows][header: slot index]
  static constexpr uint32_t HDR = SLOT_BYTES + 3 * T * ROW_BYTES;
  static constexpr uint32_t STAGE_BYTES = HDR + 16;
  static constexpr uint32_t TX = SLOT_BYTES + 3 * T * ROW_BYTES;
  static constexpr int NSTAGE = 3;
  // after the stages: full barriers, then the per-stage done counters
  static constexpr size_t BYTES = (size_t)NSTAGE * STAGE_BYTES + NSTAGE * 8 + NSTAGE * 4;
};

__device__ __forceinline__ float softplus_f(float x, float beta, float thr) {
  const float bx = beta * x;
  return bx <= thr ? log1pf(expf(bx)) / beta : x;
}

// two fp32 FMAs in one instruction (each rounded to nearest)
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 r;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return r;
}

// eight bf16 -> four fp32 pairs
__device__ __forceinline__ void unpack8(uint4 u, float2 *f) {
  const __nv_bfloat162 *h2 = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
  for (int e = 0; e < 4; ++e) f[e] = __bfloat1622float2(h2[e]);
}

// sum over the eight column-slice lanes of a row group (lane bits 0..2)
__device__ __forceinline__ float sum8(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 1);
  x += __shfl_xor_sync(0xffffffffu, x, 2);
  x += __shfl_xor_sync(0xffffffffu, x, 4);
  return x;
}

// Reduce-scatter over the eight column-slice lanes of a row group: v[0..3]
// are this lane's partial S k of rows 0..3, v[4..7] its partial S q.  Lane
// cs returns the full sum of v[4 (cs >> 2) + (cs & 3)]: lanes 0-3 hold S k of
// row cs, lanes 4-7 S q of row cs - 4.
__device__ __forceinline__ float reduce_scatter8(const float *v, int cs) {
  const bool b2 = cs & 4, b1 = cs & 2, b0 = cs & 1;
  float w[4], x[2];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float keep = b2 ? v[4 + j] : v[j], send = b2 ? v[j] : v[4 + j];
    w[j] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
  }
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const float keep = b1 ? w[2 + j] : w[j], send = b1 ? w[j] : w[2 + j];
    x[j] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
  }
  const float keep = b0 ? x[1] : x[0], send = b0 ? x[0] : x[1];
  return keep + __shfl_xor_sync(0xffffffffu, send, 1);
}

__device__ __forceinline__ int slot_of(const DecodeParams &p, int item) {
  const int bi = item / p.HV;
  return p.slot_indices ? p.slot_indices[bi] : bi;
}

// Fill stage `st` with item `item` (one thread).  An out-of-range slot is
// marked in the header and the barrier completes with no copies.
template <int T>
__device__ __forceinline__ void issue(const DecodeParams &p, unsigned char *st, uint64_t *full,
                                      int item, int slot) {
  using L = DecodeSmem<T>;
  const int HV = p.HV;
  const int bi = item / HV, hv = item % HV, hk = hv / (HV / p.H);
  int *hdr = reinterpret_cast<int *>(st + L::HDR);
  if (slot < 0 || slot >= p.pool) {
    *hdr = -1;
    ptx::mbar_arrive(full);
    return;
  }
  *hdr = slot;
  ptx::fence_proxy_async_smem();
  ptx::mbar_arrive_expect_tx(full, L::TX);
  const __nv_bfloat16 *state = static_cast<const __nv_bfloat16 *>(p.state);
  ptx::bulk_g2s(st, state + ((size_t)slot * HV + hv) * DV * DK, SLOT_BYTES, full);
  const __nv_bfloat16 *q = static_cast<const __nv_bfloat16 *>(p.q);
  const __nv_bfloat16 *k = static_cast<const __nv_bfloat16 *>(p.k);
  const __nv_bfloat16 *v = static_cast<const __nv_bfloat16 *>(p.v);
#pragma unroll
  for (int t = 0; t < T; ++t) {
    const size_t qk_off = (((size_t)bi * T + t) * p.H + hk) * DK;
    const size_t v_off = (((size_t)bi * T + t) * HV + hv) * DV;
    ptx::bulk_g2s(st + SLOT_BYTES + t * ROW_BYTES, q + qk_off, ROW_BYTES, full);
    ptx::bulk_g2s(st + SLOT_BYTES + (T + t) * ROW_BYTES, k + qk_off, ROW_BYTES, full);
    ptx::bulk_g2s(st + SLOT_BYTES + (2 * T + t) * ROW_BYTES, v + v_off, ROW_BYTES, full);
  }
}

// Raw gate inputs of one item, held by lane t < T for token t.
struct GateIn {
  float a, b, A_log, dt_bias;
};

__device__ __forceinline__ GateIn load_gate_in(const DecodeParams &p, int item, int lane, int T) {
  GateIn g{0.f, 0.f, 0.f, 0.f};
  if (lane < T) {
    const int bi = item / p.HV, hv = item % p.HV;
    const size_t gi = ((size_t)bi * T + lane) * p.HV + hv;
    g.a = __bfloat162float(static_cast<const __nv_bfloat16 *>(p.a)[gi]);
    g.b = __bfloat162float(static_cast<const __nv_bfloat16 *>(p.b)[gi]);
    g.A_log = p.A_log[hv];
    g.dt_bias = p.dt_bias[hv];
  }
  return g;
}

template <int T>
__global__ void __launch_bounds__(DTHREADS, 2) decode_kernel(DecodeParams p) {
  using L = DecodeSmem<T>;
  constexpr int NSTAGE = L::NSTAGE;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)NSTAGE * L::STAGE_BYTES);
  int *done = reinterpret_cast<int *>(full + NSTAGE);

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int rg = tid >> 3;   // row group: rows rg + 32 i
  const int cs = tid & 7;    // column slice: pieces cs and cs + 8
  const int HV = p.HV;
  const int nitems = p.B * HV;
  const int stride = gridDim.x;
  __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(p.o);
  __nv_bfloat16 *state = static_cast<__nv_bfloat16 *>(p.state);

  if (tid == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      ptx::mbar_init(&full[s], 1);
      done[s] = 0;
    }
    ptx::fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      const int item = blockIdx.x + s * stride;
      if (item < nitems) issue<T>(p, smem + (size_t)s * L::STAGE_BYTES, &full[s], item, slot_of(p, item));
    }
  }

  GateIn gin = load_gate_in(p, blockIdx.x < nitems ? blockIdx.x : 0, lane, T);
#pragma unroll 1
  for (int it = 0;; ++it) {
    const int item = blockIdx.x + it * stride;
    if (item >= nitems) break;
    const int s = it % NSTAGE;
    const uint32_t parity = (uint32_t)((it / NSTAGE) & 1);
    const int bi = item / HV, hv = item % HV;
    const int refill = item + NSTAGE * stride;
    // prefetch: the slot of the item this stage takes next, the next item's gates
    const int next_slot = (lane == 0 && refill < nitems) ? slot_of(p, refill) : 0;
    const GateIn gnext = load_gate_in(p, item + stride < nitems ? item + stride : item, lane, T);
    // this item's gates, lane t for token t
    float gexp_l = 0.f, beta_l = 0.f;
    if (lane < T) {
      gexp_l = expf(-expf(gin.A_log) *
                    softplus_f(gin.a + gin.dt_bias, p.softplus_beta, p.softplus_threshold));
      beta_l = 1.f / (1.f + expf(-gin.b));
    }
    gin = gnext;

    if (!ptx::mbar_wait_bounded(&full[s], parity)) record_error(p.err, GDN_ERR_TIMEOUT);
    const unsigned char *st = smem + (size_t)s * L::STAGE_BYTES;
    const int slot = *reinterpret_cast<const int *>(st + L::HDR);

    float2 S[ROWS_PER_THREAD][8];
    float c = 1.f;  // the true state is c * S (running decay scale)
    if (slot >= 0) {
      const __nv_bfloat16 *ss = reinterpret_cast<const __nv_bfloat16 *>(st);
#pragma unroll
      for (int i = 0; i < ROWS_PER_THREAD; ++i) {
        const int row = rg + 32 * i;
#pragma unroll
        for (int pc = 0; pc < 2; ++pc)
          unpack8(*reinterpret_cast<const uint4 *>(ss + row * DK + (cs + 8 * pc) * 8),
                  &S[i][pc * 4]);
      }
      const __nv_bfloat16 *sq = reinterpret_cast<const __nv_bfloat16 *>(st + SLOT_BYTES);

      // Norms: the four row groups of a warp take tokens grp % T; lane 8 t
      // then holds token t's factors.
      float fk, fq, kqh;
      {
        const int tn = ((lane >> 3) & 3) % T;
        float2 kr[8], qr[8];
        unpack8(*reinterpret_cast<const uint4 *>(sq + (T + tn) * DK + cs * 8), &kr[0]);
        unpack8(*reinterpret_cast<const uint4 *>(sq + (T + tn) * DK + 64 + cs * 8), &kr[4]);
        unpack8(*reinterpret_cast<const uint4 *>(sq + tn * DK + cs * 8), &qr[0]);
        unpack8(*reinterpret_cast<const uint4 *>(sq + tn * DK + 64 + cs * 8), &qr[4]);
        float2 akk = make_float2(0.f, 0.f), aqq = akk, akq = akk;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          akk = ffma2(kr[j], kr[j], akk);
          aqq = ffma2(qr[j], qr[j], aqq);
          akq = ffma2(kr[j], qr[j], akq);
        }
        const float ssk = sum8(akk.x + akk.y), ssq = sum8(aqq.x + aqq.y);
        const float kqr = sum8(akq.x + akq.y);
        fk = p.use_qk_l2norm ? rsqrtf(ssk + p.eps) : 1.f;
        fq = (p.use_qk_l2norm ? rsqrtf(ssq + p.eps) : 1.f) * p.scale;
        kqh = fk * fq * kqr;
      }

      const bool qlane = cs >= 4;  // after the reduction: lanes 0-3 hold S k, lanes 4-7 S q
      const int rsel = cs & 3;     // ... of row rg + 32 rsel
#pragma unroll
      for (int t = 0; t < T; ++t) {
        const float fk_t = __shfl_sync(0xffffffffu, fk, 8 * t);
        const float fq_t = __shfl_sync(0xffffffffu, fq, 8 * t);
        const float kq_t = __shfl_sync(0xffffffffu, kqh, 8 * t);
        const float ge = __shfl_sync(0xffffffffu, gexp_l, t);
        const float be = __shfl_sync(0xffffffffu, beta_l, t);
        float2 kr[8], qr[8];
        unpack8(*reinterpret_cast<const uint4 *>(sq + (T + t) * DK + cs * 8), &kr[0]);
        unpack8(*reinterpret_cast<const uint4 *>(sq + (T + t) * DK + 64 + cs * 8), &kr[4]);
        unpack8(*reinterpret_cast<const uint4 *>(sq + t * DK + cs * 8), &qr[0]);
        unpack8(*reinterpret_cast<const uint4 *>(sq + t * DK + 64 + cs * 8), &qr[4]);

        // raw row dots S k and S q, partial over this lane's 16 columns
        float vals[2 * ROWS_PER_THREAD];
#pragma unroll
        for (int i = 0; i < ROWS_PER_THREAD; ++i) {
          float2 ak = make_float2(0.f, 0.f), aq = ak;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            ak = ffma2(S[i][j], kr[j], ak);
            aq = ffma2(S[i][j], qr[j], aq);
          }
          vals[i] = ak.x + ak.y;
          vals[ROWS_PER_THREAD + i] = aq.x + aq.y;
        }
        const float y = reduce_scatter8(vals, cs);

        const float cg = c * ge;  // decay of the true state through token t
        const float vv = __bfloat162float(sq[(2 * T + t) * DK + rg + 32 * rsel]);
        const float delta = be * (vv - cg * fk_t * y);      // valid on lanes 0-3
        const float dq = __shfl_xor_sync(0xffffffffu, delta, 4);
        if (qlane)
          o[(((size_t)bi * T + t) * HV + hv) * DV + rg + 32 * rsel] =
              __float2bfloat16_rn(fmaf(cg * fq_t, y, dq * kq_t));
        float d[ROWS_PER_THREAD];
#pragma unroll
        for (int i = 0; i < ROWS_PER_THREAD; ++i) d[i] = __shfl_sync(0xffffffffu, delta, i, 8);

        if (cg >= 0x1p-40f) {
          // S <- S + (delta fk / cg) k_raw, and the scale takes the decay
          const float f = fk_t / cg;
#pragma unroll
          for (int i = 0; i < ROWS_PER_THREAD; ++i) {
            const float2 d2 = make_float2(d[i] * f, d[i] * f);
#pragma unroll
            for (int j = 0; j < 8; ++j) S[i][j] = ffma2(d2, kr[j], S[i][j]);
          }
          c = cg;
        } else {
          // the scale would underflow: fold it into S
          const float2 g2 = make_float2(cg, cg), z2 = make_float2(0.f, 0.f);
#pragma unroll
          for (int i = 0; i < ROWS_PER_THREAD; ++i) {
            const float2 d2 = make_float2(d[i] * fk_t, d[i] * fk_t);
#pragma unroll
            for (int j = 0; j < 8; ++j) S[i][j] = ffma2(g2, S[i][j], ffma2(d2, kr[j], z2));
          }
          c = 1.f;
        }
      }
    }

    // This warp has read all of stage s; the last warp out refills it.
    __syncwarp();
    if (lane == 0) {
      __threadfence_block();
      if (atomicAdd(&done[s], 1) == NWARPS - 1) {
        done[s] = 0;
        __threadfence_block();
        if (refill < nitems)
          issue<T>(p, smem + (size_t)s * L::STAGE_BYTES, &full[s], refill, next_slot);
      }
    }
    __syncwarp();

    if (slot < 0) {
      if (tid == 0) record_error(p.err, GDN_ERR_BAD_SLOT);
      for (int idx = tid; idx < T * DV; idx += DTHREADS)
        o[(((size_t)bi * T + idx / DV) * HV + hv) * DV + idx % DV] = __float2bfloat16_rn(0.f);
      continue;
    }
    // write the slot back once
    __nv_bfloat16 *dst = state + ((size_t)slot * HV + hv) * DV * DK;
#pragma unroll
    for (int i = 0; i < ROWS_PER_THREAD; ++i) {
      const int row = rg + 32 * i;
#pragma unroll
      for (int pc = 0; pc < 2; ++pc) {
        uint4 w;
        __nv_bfloat162 *h2 = reinterpret_cast<__nv_bfloat162 *>(&w);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 x = S[i][pc * 4 + e];
          h2[e] = __float22bfloat162_rn(make_float2(c * x.x, c * x.y));
        }
        *reinterpret_cast<uint4 *>(dst + row * DK + (cs + 8 * pc) * 8) = w;
      }
    }
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
