// Decode step against a pooled bf16 state, HBM-streaming: the kernel for
// T = 1, 2 tokens (T = 3, 4 run on the warp-level tensor cores, decode_tc.cu).
//
// FlashInfer gdn_decode_bf16_state.py (compute_single_gate,
// normalize_and_store_qk_to_smem, the per-token helpers and the public
// gated_delta_rule) gives the arithmetic: per token t
//   g_t = -exp(A_log) softplus(a_t + dt_bias),  beta_t = sigmoid(b_t),
//   q^ = scale q / sqrt(|q|^2 + eps),  k^ = k / sqrt(|k|^2 + eps),
//   S <- e^g S;  delta = beta (v - S k^);  S <- S + delta k^T;  o = S q^.
//
// Design (ours).  The T tokens of one (batch entry, value head) item are
// taken together in the chunk (WY) form of that recurrence.  With
// G_t = e^{g_0 + ... + g_t}, R_ts = e^{g_{s+1} + ... + g_t} (R_tt = 1) and the
// initial state S0:
//   y_t = S0 k^_t,  z_t = S0 q^_t                         (2T dot products)
//   delta_t = beta_t v_t - beta_t G_t y_t - sum_{s<t} beta_t R_ts (k^_s.k^_t) delta_s
//   o_t = G_t z_t + sum_{s<=t} R_ts (k^_s.q^_t) delta_s
//   S_T = G_{T-1} S0 + sum_s R_{T-1,s} delta_s k^_s^T   (one rank-T update)
// so the state is read, dotted with 2T vectors at once and updated once,
// with no dependent per-token chain over the [V, K] tile.
//
// Kernel: persistent, two CTAs of eight warps per SM, no block-wide barrier
// in the item loop.  Each CTA walks its items through NSTAGE shared-memory
// stages filled by bulk (TMA) copies of the 32 KB state slot and the q/k/v
// rows.  Per item one warp prepares the stage: it turns q and k into
// normalised fp32 vectors (in place, in a lane-friendly permuted order) and
// writes the gates and the scalar coefficients above into the stage header.
// The first warp to finish item i prepares item i + PREP_AHEAD and the last
// warp to finish item i issues the copies of item i + NSTAGE, so warps wait
// on one another only through those per-stage events.  Thread t owns rows
// {t/8 + 32 i : i < 4} of the state and the 16 columns
// {8 (t%8) + j, 64 + 8 (t%8) + j : j < 8}; row sums are reduce-scatters over
// the eight column lanes of a row group.  State arithmetic is fp32 on
// registers with packed two-lane FMAs; the slot is written back once, rounded
// to bf16 (round to nearest even).
#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "ptx.cuh"

#include <type_traits>

namespace gdn {
namespace {

constexpr int DK = 128, DV = 128;
constexpr int NWARPS = 8, DTHREADS = NWARPS * 32;
constexpr uint32_t SLOT_BYTES = DK * DV * 2;  // 32 KB bf16 state slot
constexpr uint32_t ROW_BYTES = DK * 2;        // one bf16 q/k/v row
constexpr uint32_t VEC_BYTES = DK * 4;        // one fp32 q/k vector slot
constexpr int ROWS_PER_THREAD = 4;
// Stages per CTA: three (prepared two items ahead) for T = 2; two (prepared
// one ahead) for T = 1, whose item is shortest (88.1 against 92.2 us at
// B = 256, HV = 32; two stages made T = 2 slower, 100.4 against 94.2 us).
template <int T>
struct Ring {
  static constexpr int NSTAGE = T == 1 ? 2 : 3;
  static constexpr int PREP_AHEAD = NSTAGE - 1;  // the first warp out of item i prepares i + this
};

// Stage header (32-bit words): slot index, G_{T-1}, beta_t G_t, beta_t, G_t,
// R_{T-1,t}, beta_t R_ts (k^_s.k^_t) [t][s], R_ts (k^_s.q^_t) [t][s].
constexpr int H_SLOT = 0, H_GT = 1, H_BG = 4, H_BE = 8, H_GAM = 12, H_C = 16, H_A = 20,
              H_B = 36;

template <int T>
struct DecodeSmem {
  // stage: [state 32 KB][2T vector slots: k_0..k_{T-1}, q_0..q_{T-1}][v rows][header]
  // A vector slot receives the bf16 row in its first half; the preparing warp
  // rewrites it as the fp32 normalised vector.
  static constexpr uint32_t VEC = SLOT_BYTES;
  static constexpr uint32_t VROWS = VEC + 2 * T * VEC_BYTES;
  static constexpr uint32_t HDR = VROWS + T * ROW_BYTES;
  static constexpr uint32_t STAGE_BYTES = HDR + 256;
  static constexpr uint32_t TX = SLOT_BYTES + 3 * T * ROW_BYTES;
  // after the stages: full and prepared barriers, then the per-stage done counters
  static constexpr int NSTAGE = Ring<T>::NSTAGE;
  static constexpr size_t BYTES = (size_t)NSTAGE * STAGE_BYTES + NSTAGE * 16 + NSTAGE * 4;
};

__device__ __forceinline__ float softplus_f(float x, float beta, float thr) {
  const float bx = beta * x;
  return bx <= thr ? log1pf(expf(bx)) / beta : x;
}

// Packed fp32 pairs (each half rounded to nearest).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 r;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return r;
}

__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  float2 r;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}

// eight bf16 -> four fp32 pairs
__device__ __forceinline__ void unpack8(uint4 u, float2 *f) {
  const __nv_bfloat162 *h2 = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
  for (int e = 0; e < 4; ++e) f[e] = __bfloat1622float2(h2[e]);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

__device__ __forceinline__ float pick(bool hi, float a_lo, float a_hi) { return hi ? a_hi : a_lo; }

// Row sums over the eight column lanes of a row group, for one or two
// tokens.  v[t][i] is this lane's partial sum for token t and row i; on
// return y[t] holds the full sum of row cs & 3 (the same on lanes cs and
// cs ^ 4).
template <int T>
__device__ __forceinline__ void row_sums(const float (&v)[T][ROWS_PER_THREAD], int cs,
                                         float (&y)[T]) {
  const bool b2 = cs & 4, b1 = cs & 2, b0 = cs & 1;
  static_assert(T == 1 || T == 2, "row sums are taken one or two tokens at a time");
  if constexpr (T == 2) {
    // token b2 stays on this lane
    float x[4], w[2];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      x[i] = pick(b2, v[0][i], v[1][i]) +
             __shfl_xor_sync(0xffffffffu, pick(b2, v[1][i], v[0][i]), 4);
#pragma unroll
    for (int ii = 0; ii < 2; ++ii)
      w[ii] = pick(b1, x[ii], x[2 + ii]) +
              __shfl_xor_sync(0xffffffffu, pick(b1, x[2 + ii], x[ii]), 2);
    const float u = pick(b0, w[0], w[1]) + __shfl_xor_sync(0xffffffffu, pick(b0, w[1], w[0]), 1);
    const float other = __shfl_xor_sync(0xffffffffu, u, 4);
    y[0] = pick(b2, u, other);
    y[1] = pick(b2, other, u);
  } else {
    float x[4], w[2];
#pragma unroll
    for (int i = 0; i < 4; ++i) x[i] = v[0][i] + __shfl_xor_sync(0xffffffffu, v[0][i], 4);
#pragma unroll
    for (int ii = 0; ii < 2; ++ii)
      w[ii] = pick(b1, x[ii], x[2 + ii]) +
              __shfl_xor_sync(0xffffffffu, pick(b1, x[2 + ii], x[ii]), 2);
    y[0] = pick(b0, w[0], w[1]) + __shfl_xor_sync(0xffffffffu, pick(b0, w[1], w[0]), 1);
  }
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
  // checked builds: an item whose batch entry or key head falls outside its
  // tensor is skipped like a bad slot
  const bool in_range = !kChecked || (bi < p.B && hk < p.H);
  if (!in_range) record_error(p.err, GDN_ERR_BOUNDS);
  if (!in_range || slot < 0 || slot >= p.pool) {
    hdr[H_SLOT] = -1;
    ptx::mbar_arrive(full);
    return;
  }
  hdr[H_SLOT] = slot;
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
    ptx::bulk_g2s(st + L::VEC + t * VEC_BYTES, k + qk_off, ROW_BYTES, full);
    ptx::bulk_g2s(st + L::VEC + (T + t) * VEC_BYTES, q + qk_off, ROW_BYTES, full);
    ptx::bulk_g2s(st + L::VROWS + t * ROW_BYTES, v + v_off, ROW_BYTES, full);
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

// Prepare a landed stage (one warp): normalised fp32 q/k vectors in place,
// gates and coefficients in the header; then every lane arrives on `prep`.
// Lane l handles the four vector entries that consumer lane cs = l % 8 reads
// as its float4 number l / 8, so both sides touch contiguous bytes.
template <int T>
__device__ __noinline__ void prepare(const DecodeParams &p, unsigned char *st, uint64_t *full,
                                     uint64_t *prep, uint32_t parity, GateIn gin, int lane) {
  using L = DecodeSmem<T>;
  if (!ptx::mbar_wait_bounded(full, parity)) record_error(p.err, GDN_ERR_TIMEOUT);
  float *hdr = reinterpret_cast<float *>(st + L::HDR);
  if (*reinterpret_cast<const int *>(hdr) >= 0) {
    const int j = lane >> 3, csl = lane & 7;
    const int c0 = (j >> 1) * 64 + csl * 8 + (j & 1) * 4;
    float x[2 * T][4];
#pragma unroll
    for (int n = 0; n < 2 * T; ++n) {
      const uint2 raw = *reinterpret_cast<const uint2 *>(st + L::VEC + n * VEC_BYTES + c0 * 2);
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&raw.x));
      const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&raw.y));
      x[n][0] = a.x;
      x[n][1] = a.y;
      x[n][2] = b.x;
      x[n][3] = b.y;
    }
    // L2 norms (q also takes the output scale)
#pragma unroll
    for (int n = 0; n < 2 * T; ++n) {
      float ss = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) ss = fmaf(x[n][e], x[n][e], ss);
      ss = warp_sum(ss);
      float f = p.use_qk_l2norm ? rsqrtf(ss + p.eps) : 1.f;
      if (n >= T) f *= p.scale;
#pragma unroll
      for (int e = 0; e < 4; ++e) x[n][e] *= f;
    }
    // Gram scalars: gk[t][s] = k^_s . k^_t (s < t), gq[t][s] = k^_s . q^_t (s <= t)
    float gk[T][T], gq[T][T];
#pragma unroll
    for (int t = 0; t < T; ++t)
#pragma unroll
      for (int s = 0; s < T; ++s) {
        float dk = 0.f, dq = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          dk = fmaf(x[s][e], x[t][e], dk);
          dq = fmaf(x[s][e], x[T + t][e], dq);
        }
        gk[t][s] = s < t ? warp_sum(dk) : 0.f;
        gq[t][s] = s <= t ? warp_sum(dq) : 0.f;
      }
    __syncwarp();  // every raw row has been read before it is overwritten
#pragma unroll
    for (int n = 0; n < 2 * T; ++n)
      *reinterpret_cast<float4 *>(st + L::VEC + n * VEC_BYTES + lane * 16) =
          make_float4(x[n][0], x[n][1], x[n][2], x[n][3]);

    // gates (lane t for token t), then the coefficients (uniform over lanes)
    float gl = 1.f, bl = 0.f;
    if (lane < T) {
      gl = expf(-expf(gin.A_log) *
                softplus_f(gin.a + gin.dt_bias, p.softplus_beta, p.softplus_threshold));
      bl = 1.f / (1.f + expf(-gin.b));
    }
    float gam[T], be[T];
#pragma unroll
    for (int t = 0; t < T; ++t) {
      gam[t] = __shfl_sync(0xffffffffu, gl, t);
      be[t] = __shfl_sync(0xffffffffu, bl, t);
    }
    float G[T], R[T][T];
#pragma unroll
    for (int t = 0; t < T; ++t) {
      G[t] = t == 0 ? gam[0] : G[t - 1] * gam[t];
      R[t][t] = 1.f;
#pragma unroll
      for (int s = t - 1; s >= 0; --s) R[t][s] = R[t][s + 1] * gam[s + 1];
    }
    if (lane == 0) {
      hdr[H_GT] = G[T - 1];
#pragma unroll
      for (int t = 0; t < T; ++t) {
        hdr[H_BG + t] = be[t] * G[t];
        hdr[H_BE + t] = be[t];
        hdr[H_GAM + t] = G[t];
        hdr[H_C + t] = R[T - 1][t];
#pragma unroll
        for (int s = 0; s < T; ++s) {
          hdr[H_A + 4 * t + s] = s < t ? be[t] * R[t][s] * gk[t][s] : 0.f;
          hdr[H_B + 4 * t + s] = s <= t ? R[t][s] * gq[t][s] : 0.f;
        }
      }
    }
  }
  ptx::mbar_arrive(prep);  // each lane releases its own writes
}

// F32: the variant that writes o in fp32 (p.o_f32) and/or the fp32 updated
// states (p.state_f32); the default variant is compiled without either.
template <int T, bool F32>
__global__ void __launch_bounds__(DTHREADS, 2) decode_kernel(DecodeParams p) {
  using L = DecodeSmem<T>;
  constexpr int NSTAGE = L::NSTAGE, PREP_AHEAD = Ring<T>::PREP_AHEAD;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)NSTAGE * L::STAGE_BYTES);
  uint64_t *prep = full + NSTAGE;
  int *done = reinterpret_cast<int *>(prep + NSTAGE);

  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int rg = tid >> 3;   // row group: rows rg + 32 i
  const int cs = tid & 7;    // column slice: pieces cs and cs + 8
  const int rsel = cs & 3;   // after row_sums: this lane holds row rg + 32 rsel
  const int HV = p.HV;
  const int nitems = p.B * HV;
  const int stride = gridDim.x;
  const int zmask = p.B >> 31;  // zero (B > 0), opaque to the compiler
  __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(p.o);
  __nv_bfloat16 *state = static_cast<__nv_bfloat16 *>(p.state);

  if (tid == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&prep[s], 32);
      done[s] = 0;
    }
    ptx::fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      const int item = blockIdx.x + s * stride;
      if (item < nitems)
        issue<T>(p, smem + (size_t)s * L::STAGE_BYTES, &full[s], item, slot_of(p, item));
    }
  }
  // the first PREP_AHEAD items are prepared by warps 0 .. PREP_AHEAD-1
  if (warp < PREP_AHEAD) {
    const int item = blockIdx.x + warp * stride;
    if (item < nitems)
      prepare<T>(p, smem + (size_t)warp * L::STAGE_BYTES, &full[warp], &prep[warp], 0u,
                 load_gate_in(p, item, lane, T), lane);
  }

#pragma unroll 1
  for (int it = 0;; ++it) {
    const int item = blockIdx.x + it * stride;
    if (item >= nitems) break;
    const int s = it % NSTAGE;
    const uint32_t parity = (uint32_t)((it / NSTAGE) & 1);
    const int bi = item / HV, hv = item % HV;
    const int refill = item + NSTAGE * stride;
    const int ahead = item + PREP_AHEAD * stride;

    if (!ptx::mbar_wait_bounded(&full[s], parity)) record_error(p.err, GDN_ERR_TIMEOUT);
    unsigned char *st = smem + (size_t)s * L::STAGE_BYTES;
    const float *hdr = reinterpret_cast<const float *>(st + L::HDR);
    const int slot = *reinterpret_cast<const int *>(hdr);

    float2 S[ROWS_PER_THREAD][8];
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
      if (!ptx::mbar_wait_bounded(&prep[s], parity)) record_error(p.err, GDN_ERR_TIMEOUT);

      // y_t = S0 k^_t and z_t = S0 q^_t of row rg + 32 rsel
      float y[T], z[T];
      auto dots = [&](auto n0_c, auto nt_c, float *out) {
        constexpr int N0 = decltype(n0_c)::value, NT = decltype(nt_c)::value;
        float part[NT][ROWS_PER_THREAD];
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const float4 *vp =
              reinterpret_cast<const float4 *>(st + L::VEC + (N0 + t) * VEC_BYTES) + cs;
          float2 xv[8];
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const float4 f = vp[8 * jj];
            xv[2 * jj] = make_float2(f.x, f.y);
            xv[2 * jj + 1] = make_float2(f.z, f.w);
          }
#pragma unroll
          for (int i = 0; i < ROWS_PER_THREAD; ++i) {
            float2 acc = fmul2(S[i][0], xv[0]);
#pragma unroll
            for (int m = 1; m < 8; ++m) acc = ffma2(S[i][m], xv[m], acc);
            part[t][i] = acc.x + acc.y;
          }
        }
        float r[NT];
        row_sums<NT>(part, cs, r);
#pragma unroll
        for (int t = 0; t < NT; ++t) out[t] = r[t];
      };
      using C0 = std::integral_constant<int, 0>;
      using CT = std::integral_constant<int, T>;
      dots(C0{}, CT{}, y);
      dots(CT{}, CT{}, z);

      // deltas and outputs of row rg + 32 rsel (the same on lanes cs and cs ^ 4)
      float dl[T];
#pragma unroll
      for (int t = 0; t < T; ++t) {
        const float vv = __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(
            st + L::VROWS + t * ROW_BYTES)[rg + 32 * rsel]);
        float d = fmaf(hdr[H_BE + t], vv, -hdr[H_BG + t] * y[t]);
#pragma unroll
        for (int s2 = 0; s2 < t; ++s2) d = fmaf(-hdr[H_A + 4 * t + s2], dl[s2], d);
        dl[t] = d;
      }
      if (cs < 4) {
#pragma unroll
        for (int t = 0; t < T; ++t) {
          float ov = hdr[H_GAM + t] * z[t];
#pragma unroll
          for (int s2 = 0; s2 <= t; ++s2) ov = fmaf(hdr[H_B + 4 * t + s2], dl[s2], ov);
          const size_t oi = (((size_t)bi * T + t) * HV + hv) * DV + rg + 32 * rsel;
          if (F32 && p.o_f32)
            static_cast<float *>(p.o)[oi] = ov;
          else
            o[oi] = __float2bfloat16_rn(ov);
        }
      }

      // S <- G_{T-1} S + sum_t R_{T-1,t} delta_t k^_t^T
      const float gt = hdr[H_GT];
#pragma unroll
      for (int i = 0; i < ROWS_PER_THREAD; ++i)
#pragma unroll
        for (int m = 0; m < 8; ++m) S[i][m] = fmul2(make_float2(gt, gt), S[i][m]);
      // Token t's vector loads take a (zero) offset computed from token t-1's
      // first result, so the compiler cannot hoist all T vectors at once.
      int chain = 0;
#pragma unroll
      for (int t = 0; t < T; ++t) {
        const float4 *vp =
            reinterpret_cast<const float4 *>(st + L::VEC + t * VEC_BYTES + chain) + cs;
        float2 kv[8];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const float4 f = vp[8 * jj];
          kv[2 * jj] = make_float2(f.x, f.y);
          kv[2 * jj + 1] = make_float2(f.z, f.w);
        }
        const float ct = hdr[H_C + t];
#pragma unroll
        for (int i = 0; i < ROWS_PER_THREAD; ++i) {
          const float cf = ct * __shfl_sync(0xffffffffu, dl[t], i, 8);
          const float2 c2 = make_float2(cf, cf);
#pragma unroll
          for (int m = 0; m < 8; ++m) S[i][m] = ffma2(c2, kv[m], S[i][m]);
        }
        chain = __float_as_int(S[0][0].x) & zmask;
      }
    }

    // This warp has read all of stage s.  The last warp out refills it; the
    // first warp out prepares the item PREP_AHEAD ahead after its write-back.
    __syncwarp();
    int order = 0;
    if (lane == 0) {
      __threadfence_block();
      order = atomicAdd(&done[s], 1);
      if (order == NWARPS - 1) {
        done[s] = 0;
        __threadfence_block();
        if (refill < nitems) issue<T>(p, st, &full[s], refill, slot_of(p, refill));
      }
    }
    order = __shfl_sync(0xffffffffu, order, 0);

    if (slot < 0) {
      if (tid == 0) record_error(p.err, GDN_ERR_BAD_SLOT);
      for (int idx = tid; idx < T * DV; idx += DTHREADS) {
        const size_t oi = (((size_t)bi * T + idx / DV) * HV + hv) * DV + idx % DV;
        if (F32 && p.o_f32)
          static_cast<float *>(p.o)[oi] = 0.f;
        else
          o[oi] = __float2bfloat16_rn(0.f);
      }
    } else {
      __nv_bfloat16 *dst = state + ((size_t)slot * HV + hv) * DV * DK;
      if (F32 && p.state_f32) {
        // the fp32 values the bf16 write-back rounds (entry bi, not its slot)
        float *d32 = p.state_f32 + ((size_t)bi * HV + hv) * DV * DK;
#pragma unroll
        for (int i = 0; i < ROWS_PER_THREAD; ++i) {
          const int row = rg + 32 * i;
#pragma unroll
          for (int pc = 0; pc < 2; ++pc) {
            float4 *q4 = reinterpret_cast<float4 *>(d32 + row * DK + (cs + 8 * pc) * 8);
            q4[0] = make_float4(S[i][pc * 4].x, S[i][pc * 4].y, S[i][pc * 4 + 1].x,
                                S[i][pc * 4 + 1].y);
            q4[1] = make_float4(S[i][pc * 4 + 2].x, S[i][pc * 4 + 2].y, S[i][pc * 4 + 3].x,
                                S[i][pc * 4 + 3].y);
          }
        }
      }
#pragma unroll
      for (int i = 0; i < ROWS_PER_THREAD; ++i) {
        const int row = rg + 32 * i;
#pragma unroll
        for (int pc = 0; pc < 2; ++pc) {
          uint4 w;
          __nv_bfloat162 *h2 = reinterpret_cast<__nv_bfloat162 *>(&w);
#pragma unroll
          for (int e = 0; e < 4; ++e) h2[e] = __float22bfloat162_rn(S[i][pc * 4 + e]);
          *reinterpret_cast<uint4 *>(dst + row * DK + (cs + 8 * pc) * 8) = w;
        }
      }
    }
    if (order == 0 && ahead < nitems) {
      const int sa = (it + PREP_AHEAD) % NSTAGE;
      prepare<T>(p, smem + (size_t)sa * L::STAGE_BYTES, &full[sa], &prep[sa],
                 (uint32_t)(((it + PREP_AHEAD) / NSTAGE) & 1), load_gate_in(p, ahead, lane, T),
                 lane);
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

template <int T, bool F32>
cudaError_t launch_tf(const DecodeParams &p, cudaStream_t stream) {
  const size_t bytes = DecodeSmem<T>::BYTES;
  cudaError_t e = cudaFuncSetAttribute(decode_kernel<T, F32>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  // persistent grid: as many CTAs as are resident at once (two per SM)
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_kernel<T, F32>, DTHREADS,
                                                    bytes);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  const int items = p.B * p.HV;
  const int cap = per_sm * sm_count();
  const int grid = items < cap ? items : cap;
  decode_kernel<T, F32><<<grid, DTHREADS, bytes, stream>>>(p);
  return cudaGetLastError();
}

template <int T>
cudaError_t launch_t(const DecodeParams &p, cudaStream_t stream) {
  return (p.o_f32 || p.state_f32) ? launch_tf<T, true>(p, stream) : launch_tf<T, false>(p, stream);
}

}  // namespace

// T <= 2 is HBM-bound on this kernel; from T = 3 the packed-FMA work per item
// outgrows the state stream and the tensor-core kernel is faster (at B = 256,
// HV = 32: T = 3 107 against 112.6 us, T = 4 117 against 137 us).
cudaError_t launch_decode(const DecodeParams &p, cudaStream_t stream) {
  if (p.T >= 3) return launch_decode_tc(p, stream);
  switch (p.T) {
    case 1: return launch_t<1>(p, stream);
    case 2: return launch_t<2>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gdn
