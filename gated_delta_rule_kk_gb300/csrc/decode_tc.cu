// Decode step for T = 3, 4 tokens on the warp-level tensor cores (mma.sync
// m16n8k16, bf16 in, fp32 accumulate): same arithmetic and item schedule as
// decode.cu.  (The kernel is written for any T <= 4; at T <= 2 decode.cu is
// HBM-bound and faster, so it serves those.)
//
// FlashInfer gdn_decode_bf16_state.py (compute_single_gate,
// normalize_and_store_qk_to_smem, the per-token helpers and gated_delta_rule)
// defines the step; the T tokens of an item are taken in the chunk (WY) form
// (G_t cumulative decay, R_ts = G_t / G_s):
//   y_t = S0 k^_t,  z_t = S0 q^_t
//   delta_t = beta_t v_t - beta_t G_t y_t - sum_{s<t} beta_t R_ts (k^_s.k^_t) delta_s
//   o_t = G_t z_t + sum_{s<=t} R_ts (k^_s.q^_t) delta_s
//   S_T = G_{T-1} S0 + sum_s R_{T-1,s} delta_s k^_s^T
//
// Warp w owns rows 16 w .. 16 w + 15 of the [V, K] state of the item.  The
// state slot arrives by TMA in the 128-byte-swizzled layout; ldmatrix gives
// each warp its rows as bf16 A fragments.  The 2T dot products are one
// M16 x N(8 or 16) x K128 product with B = [k^_0 hi, k^_0 lo, k^_1 hi, ...]
// (bf16 pairs, so the vectors keep fp32-grade accuracy).  The A fragments
// stay in registers as bf16 for the update, which streams over 16-column
// blocks: a block's fragments, converted and scaled by G_{T-1}, are exactly
// the fp32 accumulator fragments (lossless: the state is bf16) of one K = 16
// product per 8 columns with A = [c delta hi | c delta lo | c delta hi] and
// B = [k^ hi; k^ hi; k^ lo]; the block goes back into the slot by stmatrix.
// No fp32 copy of the whole tile is held in registers.  One TMA store per warp
// writes its rows back.  Per item the first warp to finish item i - 2 prepares it
// (normalised q/k as the bf16 operand images, gates, coefficients); the last
// warp out of a ring entry refills it; no block-wide barrier in the item loop.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "ptx.cuh"

namespace gdn {
namespace {

constexpr int DK = 128, DV = 128;
constexpr int NWARPS = 8, NTHREADS = NWARPS * 32;
// Two rings per CTA (two CTAs per SM): the 32 KB state slots (NSW deep,
// each slot two 64-column halves of 128 rows x 128 B, swizzled, 1024-aligned)
// and small per-item entries (NAUX deep) holding
//   RAW  [0, 3072)       q, k, v rows as copied (T <= 4)
//   BD   [3072, 7424)    dot operand: 16 rows (k^_t hi/lo, then q^_t hi/lo) x 128
//   BU   [7424, 13568)   update operand: 128 rows (state columns) x 16 (pitch 48 B)
//   HDR  [13568, 13824)  slot index and coefficients
// The per-item ring is deeper, so an item is prepared two items ahead of its
// use, off the critical path.
constexpr int NSW = 2, NAUX = 3, PREP_AHEAD = 2;
constexpr uint32_t SLOT_BYTES = DK * DV * 2;  // 32 KB bf16 state slot
constexpr uint32_t ROW_BYTES = DK * 2;        // one bf16 q/k/v row
constexpr uint32_t BD_PITCH = 272, BU_PITCH = 48;
constexpr uint32_t A_RAW = 0, A_BD = 3072, A_BU = 7424, A_HDR = 13568, AUX_BYTES = 13824;
constexpr uint32_t O_AUX = NSW * SLOT_BYTES, O_BARS = O_AUX + NAUX * AUX_BYTES;
constexpr size_t SMEM_BYTES = O_BARS + (NSW + 2 * NAUX) * 8 + (NSW + NAUX) * 4 + 1024;

// header words
constexpr int H_SLOT = 0, H_GT = 1, H_BG = 4, H_BE = 8, H_GAM = 12, H_C = 16, H_A = 20, H_B = 36;

__device__ __forceinline__ float softplus_f(float x, float beta, float thr) {
  const float bx = beta * x;
  return bx <= thr ? log1pf(expf(bx)) / beta : x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ float2 unpack2(uint32_t u) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u));
}
__device__ __forceinline__ float bf16_round(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}

// Address of the 16-byte row piece lane `lane` supplies to ldmatrix/stmatrix
// for the 16 x 16 block (rows r0 .. r0 + 15, columns 16 j .. 16 j + 15) of a
// swizzled state tile.
__device__ __forceinline__ unsigned char *sw_addr(unsigned char *sw, int r0, int j, int lane) {
  const int r = r0 + (lane & 15);
  const int c = (j & 3) * 2 + (lane >> 4);  // 16-byte chunk within the 128-byte row
  return sw + (j >> 2) * 16384 + r * 128 + ((c ^ (r & 7)) << 4);
}

__device__ __forceinline__ int slot_of(const DecodeParams &p, int item) {
  const int bi = item / p.HV;
  return p.slot_indices ? p.slot_indices[bi] : bi;
}

// Checked builds: whether an item's batch entry and key head fall inside their
// tensors (both issuers skip an item that does not, like a bad slot).
__device__ __forceinline__ bool item_in_range(const DecodeParams &p, int item) {
  const int bi = item / p.HV, hk = (item % p.HV) / (p.HV / p.H);
  return !kChecked || (bi < p.B && hk < p.H);
}

// Fill a state-slot stage (one thread); an out-of-range slot completes the
// barrier with no copies.
__device__ __forceinline__ void issue_sw(const DecodeParams &p, const CUtensorMap *tm_ld,
                                         unsigned char *sw, uint64_t *full, int item, int slot) {
  if (!item_in_range(p, item) || slot < 0 || slot >= p.pool) {
    ptx::mbar_arrive(full);
    return;
  }
  ptx::fence_proxy_async_smem();
  ptx::mbar_arrive_expect_tx(full, SLOT_BYTES);
  const int row0 = (slot * p.HV + item % p.HV) * DV;
  ptx::tma_load_2d(sw, tm_ld, 0, row0, full);
  ptx::tma_load_2d(sw + 16384, tm_ld, 64, row0, full);
}

// Fill a per-item entry with the item's q, k, v rows and its slot index.
template <int T>
__device__ __forceinline__ void issue_aux(const DecodeParams &p, unsigned char *aux,
                                          uint64_t *full, int item, int slot) {
  const int HV = p.HV;
  const int bi = item / HV, hv = item % HV, hk = hv / (HV / p.H);
  int *hdr = reinterpret_cast<int *>(aux + A_HDR);
  const bool in_range = item_in_range(p, item);
  if (!in_range) record_error(p.err, GDN_ERR_BOUNDS);
  if (!in_range || slot < 0 || slot >= p.pool) {
    hdr[H_SLOT] = -1;
    ptx::mbar_arrive(full);
    return;
  }
  hdr[H_SLOT] = slot;
  ptx::fence_proxy_async_smem();
  ptx::mbar_arrive_expect_tx(full, 3 * T * ROW_BYTES);
  const __nv_bfloat16 *q = static_cast<const __nv_bfloat16 *>(p.q);
  const __nv_bfloat16 *k = static_cast<const __nv_bfloat16 *>(p.k);
  const __nv_bfloat16 *v = static_cast<const __nv_bfloat16 *>(p.v);
#pragma unroll
  for (int t = 0; t < T; ++t) {
    const size_t qk_off = (((size_t)bi * T + t) * p.H + hk) * DK;
    const size_t v_off = (((size_t)bi * T + t) * HV + hv) * DV;
    ptx::bulk_g2s(aux + A_RAW + t * ROW_BYTES, k + qk_off, ROW_BYTES, full);
    ptx::bulk_g2s(aux + A_RAW + (T + t) * ROW_BYTES, q + qk_off, ROW_BYTES, full);
    ptx::bulk_g2s(aux + A_RAW + (2 * T + t) * ROW_BYTES, v + v_off, ROW_BYTES, full);
  }
}

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

// Prepare a landed per-item entry (one warp): operand images of the
// normalised q/k, gates and coefficients; every lane then arrives on `prep`.
// Lane l handles columns 4 l .. 4 l + 3 of every vector.
template <int T>
__device__ __noinline__ void prepare(const DecodeParams &p, unsigned char *st, uint64_t *full,
                                     uint64_t *prep, uint32_t parity, GateIn gin, int lane) {
  if (!ptx::mbar_wait_bounded(full, parity)) record_error(p.err, GDN_ERR_TIMEOUT);
  float *hdr = reinterpret_cast<float *>(st + A_HDR);
  if (*reinterpret_cast<const int *>(hdr) >= 0) {
    float x[2 * T][4];
#pragma unroll
    for (int n = 0; n < 2 * T; ++n) {
      const uint2 raw = *reinterpret_cast<const uint2 *>(st + A_RAW + n * ROW_BYTES + lane * 8);
      const float2 a = unpack2(raw.x), b = unpack2(raw.y);
      x[n][0] = a.x; x[n][1] = a.y; x[n][2] = b.x; x[n][3] = b.y;
    }
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
    // BD: row 2 n = hi, row 2 n + 1 = lo of vector n (k^_0.., then q^_0..)
    unsigned char *bd = st + A_BD;
    float hi[2 * T][4], lo[2 * T][4];
#pragma unroll
    for (int n = 0; n < 2 * T; ++n) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        hi[n][e] = bf16_round(x[n][e]);
        lo[n][e] = x[n][e] - hi[n][e];
      }
      *reinterpret_cast<uint2 *>(bd + (2 * n) * BD_PITCH + lane * 8) =
          make_uint2(pack2(hi[n][0], hi[n][1]), pack2(hi[n][2], hi[n][3]));
      *reinterpret_cast<uint2 *>(bd + (2 * n + 1) * BD_PITCH + lane * 8) =
          make_uint2(pack2(lo[n][0], lo[n][1]), pack2(lo[n][2], lo[n][3]));
    }
    // BU: row = state column c, k index t: k^_t hi, T + t: k^_t hi, 2T + t: k^_t lo
    unsigned char *bu = st + A_BU;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float row[16];
#pragma unroll
      for (int kk = 0; kk < 16; ++kk) row[kk] = 0.f;
#pragma unroll
      for (int t = 0; t < T; ++t) {
        row[t] = hi[t][e];
        row[T + t] = hi[t][e];
        row[2 * T + t] = lo[t][e];
      }
      uint4 w0, w1;
      w0.x = pack2(row[0], row[1]); w0.y = pack2(row[2], row[3]);
      w0.z = pack2(row[4], row[5]); w0.w = pack2(row[6], row[7]);
      w1.x = pack2(row[8], row[9]); w1.y = pack2(row[10], row[11]);
      w1.z = pack2(row[12], row[13]); w1.w = pack2(row[14], row[15]);
      *reinterpret_cast<uint4 *>(bu + (4 * lane + e) * BU_PITCH) = w0;
      *reinterpret_cast<uint4 *>(bu + (4 * lane + e) * BU_PITCH + 16) = w1;
    }
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
__global__ void __launch_bounds__(NTHREADS, 2)
decode_tc_kernel(const __grid_constant__ CUtensorMap tm_ld, const __grid_constant__ CUtensorMap tm_st,
                 DecodeParams p) {
  extern __shared__ unsigned char smem_raw[];
  // slots on a 1024-byte boundary (the 128-byte swizzle repeats every 1 KB)
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t *sw_full = reinterpret_cast<uint64_t *>(smem + O_BARS);
  uint64_t *aux_full = sw_full + NSW, *prep = aux_full + NAUX;
  int *sw_done = reinterpret_cast<int *>(prep + NAUX), *aux_done = sw_done + NSW;
  auto sw_at = [&](int s) { return smem + s * SLOT_BYTES; };
  auto aux_at = [&](int a) { return smem + O_AUX + a * AUX_BYTES; };
  constexpr int NT_DOT = (2 * T + 3) / 4;  // 8-column tiles of the dot product

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, tig = lane & 3;
  const int HV = p.HV, nitems = p.B * HV, stride = gridDim.x;
  __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(p.o);

  if (tid == 0) {
    for (int s = 0; s < NSW; ++s) {
      ptx::mbar_init(&sw_full[s], 1);
      sw_done[s] = 0;
    }
    for (int a = 0; a < NAUX; ++a) {
      ptx::mbar_init(&aux_full[a], 1);
      ptx::mbar_init(&prep[a], 32);
      aux_done[a] = 0;
    }
    ptx::fence_mbar_init();
  }
  // BD rows past the 2T vectors stay zero
  for (int a = 0; a < NAUX; ++a)
    for (int i = tid; i < (16 - 4 * T) * (int)BD_PITCH / 16; i += NTHREADS)
      reinterpret_cast<uint4 *>(aux_at(a) + A_BD + 4 * T * BD_PITCH)[i] = make_uint4(0, 0, 0, 0);
  __syncthreads();
  if (tid == 0) {
    ptx::prefetch_tmap(&tm_ld);
    ptx::prefetch_tmap(&tm_st);
    for (int s = 0; s < NSW; ++s) {
      const int item = blockIdx.x + s * stride;
      if (item < nitems) issue_sw(p, &tm_ld, sw_at(s), &sw_full[s], item, slot_of(p, item));
    }
    for (int a = 0; a < NAUX; ++a) {
      const int item = blockIdx.x + a * stride;
      if (item < nitems) issue_aux<T>(p, aux_at(a), &aux_full[a], item, slot_of(p, item));
    }
  }
  if (warp < PREP_AHEAD) {
    const int item = blockIdx.x + warp * stride;
    if (item < nitems)
      prepare<T>(p, aux_at(warp), &aux_full[warp], &prep[warp], 0u, load_gate_in(p, item, lane, T),
                 lane);
  }

#pragma unroll 1
  for (int it = 0;; ++it) {
    const int item = blockIdx.x + it * stride;
    if (item >= nitems) break;
    const int s = it % NSW, a = it % NAUX;
    const uint32_t sp = (uint32_t)((it / NSW) & 1), ap = (uint32_t)((it / NAUX) & 1);
    const int bi = item / HV, hv = item % HV;
    unsigned char *sw = sw_at(s);
    unsigned char *aux = aux_at(a);
    const float *hdr = reinterpret_cast<const float *>(aux + A_HDR);
    const int r0 = 16 * warp;  // this warp's first state row

    if (!ptx::mbar_wait_bounded(&prep[a], ap)) record_error(p.err, GDN_ERR_TIMEOUT);
    const int slot = *reinterpret_cast<const int *>(hdr);
    uint32_t S0f[8][4];  // this warp's rows of S0 as bf16 A fragments, block j = columns 16 j ..
    if (slot >= 0) {
      if (!ptx::mbar_wait_bounded(&sw_full[s], sp)) record_error(p.err, GDN_ERR_TIMEOUT);
      // ---- dot products: S0 rows as A fragments
      float D[NT_DOT][4];
#pragma unroll
      for (int n = 0; n < NT_DOT; ++n) D[n][0] = D[n][1] = D[n][2] = D[n][3] = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        uint32_t *af = S0f[j];
        ptx::ldmatrix_x4(sw_addr(sw, r0, j, lane), af[0], af[1], af[2], af[3]);
        // dot products: B rows n (vectors' hi/lo), k = 16 j .. 16 j + 15
        uint32_t b[4];
        const int n = (lane & 7) + ((lane >> 4) << 3);
        ptx::ldmatrix_x4(aux + A_BD + n * BD_PITCH + (16 * j + 8 * ((lane >> 3) & 1)) * 2, b[0],
                         b[1], b[2], b[3]);
        ptx::mma_16816_bf16(D[0], af, b[0], b[1]);
        if (NT_DOT > 1) ptx::mma_16816_bf16(D[NT_DOT - 1], af, b[2], b[3]);
      }
      // vector 4 nt + tig on this lane: rows g (hi + lo) and g + 8
      float vg[NT_DOT], vg8[NT_DOT];
#pragma unroll
      for (int n = 0; n < NT_DOT; ++n) {
        vg[n] = D[n][0] + D[n][1];
        vg8[n] = D[n][2] + D[n][3];
      }
      // all 2T values of rows g and g + 8 on every lane of the quad
      float y[2][T], z[2][T];
#pragma unroll
      for (int jv = 0; jv < 2 * T; ++jv) {
        const int src = (lane & ~3) | (jv & 3);
        const float a0 = __shfl_sync(0xffffffffu, vg[jv >> 2], src);
        const float a1 = __shfl_sync(0xffffffffu, vg8[jv >> 2], src);
        if (jv < T) {
          y[0][jv] = a0;
          y[1][jv] = a1;
        } else {
          z[0][jv - T] = a0;
          z[1][jv - T] = a1;
        }
      }
      // ---- deltas and outputs of rows r0 + g and r0 + g + 8
      const __nv_bfloat16 *vraw =
          reinterpret_cast<const __nv_bfloat16 *>(aux + A_RAW + 2 * T * ROW_BYTES);
      // the coefficients, read as float4 groups (one broadcast load each)
      const float4 *h4 = reinterpret_cast<const float4 *>(hdr);
      auto el = [](const float4 &v, int i) { return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w; };
      const float4 be4 = h4[H_BE / 4], bg4 = h4[H_BG / 4], gam4 = h4[H_GAM / 4], c4 = h4[H_C / 4];
      float4 a4[T], b4[T];
#pragma unroll
      for (int t = 0; t < T; ++t) {
        a4[t] = h4[H_A / 4 + t];
        b4[t] = h4[H_B / 4 + t];
      }
      float dl[2][T];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int row = r0 + g + 8 * h;
#pragma unroll
        for (int t = 0; t < T; ++t) {
          const float vv = __bfloat162float(vraw[t * DV + row]);
          float d = fmaf(el(be4, t), vv, -el(bg4, t) * y[h][t]);
#pragma unroll
          for (int s2 = 0; s2 < t; ++s2) d = fmaf(-el(a4[t], s2), dl[h][s2], d);
          dl[h][t] = d;
        }
        if (tig < T) {
          // lane tig writes token tig
#pragma unroll
          for (int t = 0; t < T; ++t) {
            if (t != tig) continue;
            float ov = el(gam4, t) * z[h][t];
#pragma unroll
            for (int s2 = 0; s2 <= t; ++s2) ov = fmaf(el(b4[t], s2), dl[h][s2], ov);
            const size_t oi = (((size_t)bi * T + t) * HV + hv) * DV + row;
            if (F32 && p.o_f32)
              static_cast<float *>(p.o)[oi] = ov;
            else
              o[oi] = __float2bfloat16_rn(ov);
          }
        }
      }
      // ---- update: C = G_{T-1} S0 + A B with A = [c d hi | c d lo | c d hi]
      const float gt = hdr[H_GT];
      uint32_t ua[4];
      {
        float dh[2][T], dlo[2][T];
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int t = 0; t < T; ++t) {
            const float d = el(c4, t) * dl[h][t];
            dh[h][t] = bf16_round(d);
            dlo[h][t] = d - dh[h][t];
          }
        auto kval = [&](int h, int kk) {
          float r = 0.f;
#pragma unroll
          for (int t = 0; t < T; ++t) {
            if (kk == t) r = dh[h][t];
            if (kk == T + t) r = dlo[h][t];
            if (kk == 2 * T + t) r = dh[h][t];
          }
          return r;
        };
        ua[0] = pack2(kval(0, 2 * tig), kval(0, 2 * tig + 1));
        ua[1] = pack2(kval(1, 2 * tig), kval(1, 2 * tig + 1));
        ua[2] = pack2(kval(0, 2 * tig + 8), kval(0, 2 * tig + 9));
        ua[3] = pack2(kval(1, 2 * tig + 8), kval(1, 2 * tig + 9));
      }
      float *d32 = F32 && p.state_f32 ? p.state_f32 + ((size_t)bi * HV + hv) * DV * DK : nullptr;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        // block j of S0: af[0] / af[1] rows g / g + 8, columns 16 j + 2 tig (+1);
        // af[2] / af[3] the same rows, columns + 8
        unsigned char *blk = sw_addr(sw, r0, j, lane);
        const uint32_t *af = S0f[j];
        float C[2][4];
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const float2 rg = unpack2(af[2 * hf]), rg8 = unpack2(af[2 * hf + 1]);
          C[hf][0] = gt * rg.x; C[hf][1] = gt * rg.y; C[hf][2] = gt * rg8.x; C[hf][3] = gt * rg8.y;
        }
        uint32_t b[4];
        const int n = 16 * j + (lane & 7) + ((lane >> 4) << 3);
        ptx::ldmatrix_x4(aux + A_BU + n * BU_PITCH + ((lane >> 3) & 1) * 16, b[0], b[1], b[2], b[3]);
        ptx::mma_16816_bf16(C[0], ua, b[0], b[1]);
        ptx::mma_16816_bf16(C[1], ua, b[2], b[3]);
        if (F32 && d32) {
          // the fp32 values the bf16 write-back rounds (entry bi, not its slot)
          const int col = 16 * j + 2 * tig;
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            *reinterpret_cast<float2 *>(d32 + (r0 + g) * DK + col + 8 * hf) =
                make_float2(C[hf][0], C[hf][1]);
            *reinterpret_cast<float2 *>(d32 + (r0 + g + 8) * DK + col + 8 * hf) =
                make_float2(C[hf][2], C[hf][3]);
          }
        }
        ptx::stmatrix_x4(blk, pack2(C[0][0], C[0][1]), pack2(C[0][2], C[0][3]),
                         pack2(C[1][0], C[1][1]), pack2(C[1][2], C[1][3]));
      }
    }

    // Done with the per-item entry: the last warp out refills it with the
    // item NAUX ahead; the first prepares the item PREP_AHEAD ahead (below).
    __syncwarp();
    int order = 0;
    if (lane == 0) {
      __threadfence_block();
      order = atomicAdd(&aux_done[a], 1);
      if (order == NWARPS - 1) {
        aux_done[a] = 0;
        __threadfence_block();
        const int refill = item + NAUX * stride;
        if (refill < nitems) issue_aux<T>(p, aux, &aux_full[a], refill, slot_of(p, refill));
      }
    }
    order = __shfl_sync(0xffffffffu, order, 0);

    if (slot >= 0) {
      // ---- write back: this warp's updated rows of the slot -> TMA store
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        const int grow = (slot * HV + hv) * DV + r0;
        ptx::tma_store_2d(&tm_st, 0, grow, sw + r0 * 128);
        ptx::tma_store_2d(&tm_st, 64, grow, sw + 16384 + r0 * 128);
        ptx::bulk_commit();
        ptx::bulk_wait_read<0>();  // the slot may be refilled only after this
      }
    } else {
      if (tid == 0) record_error(p.err, GDN_ERR_BAD_SLOT);
      for (int idx = tid; idx < T * DV; idx += NTHREADS) {
        const size_t oi = (((size_t)bi * T + idx / DV) * HV + hv) * DV + idx % DV;
        if (F32 && p.o_f32)
          static_cast<float *>(p.o)[oi] = 0.f;
        else
          o[oi] = __float2bfloat16_rn(0.f);
      }
    }
    // done with the state slot: the last warp out refills it
    __syncwarp();
    if (lane == 0) {
      __threadfence_block();
      if (atomicAdd(&sw_done[s], 1) == NWARPS - 1) {
        sw_done[s] = 0;
        __threadfence_block();
        const int refill = item + NSW * stride;
        if (refill < nitems) issue_sw(p, &tm_ld, sw, &sw_full[s], refill, slot_of(p, refill));
      }
    }
    const int ahead = item + PREP_AHEAD * stride;
    if (order == 0 && ahead < nitems) {
      const int pa = (it + PREP_AHEAD) % NAUX;
      prepare<T>(p, aux_at(pa), &aux_full[pa], &prep[pa], (uint32_t)(((it + PREP_AHEAD) / NAUX) & 1),
                 load_gate_in(p, ahead, lane, T), lane);
    }
  }
  // the last stores must have left shared memory before the block exits
  if (lane == 0) ptx::bulk_wait<0>();
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// The pool as a 2-D bf16 tensor [pool * HV * V rows][K], boxes of 64 columns x
// `rows` rows, 128-byte swizzle.
bool make_state_map(CUtensorMap *m, void *base, long long rows, int box_rows) {
  auto fn = encoder();
  if (!fn) return false;
  cuuint64_t gdim[2] = {(cuuint64_t)DK, (cuuint64_t)rows};
  cuuint64_t gstride[1] = {(cuuint64_t)DK * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, gdim, gstride, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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
  CUtensorMap ld, stm;
  const long long rows = (long long)p.pool * p.HV * DV;
  if (!make_state_map(&ld, p.state, rows, 128) || !make_state_map(&stm, p.state, rows, 16))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel<T, F32>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_tc_kernel<T, F32>, NTHREADS,
                                                    SMEM_BYTES);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  const int items = p.B * p.HV;
  const int cap = per_sm * sm_count();
  const int grid = items < cap ? items : cap;
  decode_tc_kernel<T, F32><<<grid, NTHREADS, SMEM_BYTES, stream>>>(ld, stm, p);
  return cudaGetLastError();
}

template <int T>
cudaError_t launch_t(const DecodeParams &p, cudaStream_t stream) {
  return (p.o_f32 || p.state_f32) ? launch_tf<T, true>(p, stream) : launch_tf<T, false>(p, stream);
}

}  // namespace

cudaError_t launch_decode_tc(const DecodeParams &p, cudaStream_t stream) {
  switch (p.T) {
    case 3: return launch_t<3>(p, stream);
    case 4: return launch_t<4>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gdn
