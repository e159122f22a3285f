// Chunked forward on the 5th-generation tensor cores (tcgen05, TMEM
// accumulators, TMA/bulk copies), bf16 inputs, K = 128, V a multiple of 32.
//
// Two kernels per call (plus a tiny chunk-table kernel for packed sequences):
//
// 1. intra (one CTA per (chunk, value head), all chunks in parallel).  With
//    gamma the chunk-local cumulative gate and S = [k; q] k^T (one M=128
//    tcgen05 GEMM):
//      A   = beta_i S_kk[i,j] exp(gamma_i - gamma_j), i > j      (sglang
//      Aqk = scale S_qk[i,j] exp(gamma_i - gamma_j),  i >= j     fla/chunk_fwd.py,
//      T   = (I + A)^-1  (fp32: 16x16 diagonal blocks by forward  fused kernel
//            substitution, then the block merge; Steps 3-4)       Steps 1-4)
//      Tw  = T diag(beta exp(gamma)),  Tu = T diag(beta)
//      [w; Aqk w] = [Tw; Aqk Tw] k          (WY recompute, tcgen05)
//    and stores per (chunk, head) a block that holds everything the
//    sequential pass needs as ready-made tcgen05 operand images:
//      WQ = [-w ; scale exp(gamma) q - Aqk w]   (128 x 128, K-major)
//      TU = [Tu ; Aqk Tu]                       (128 x 64,  K-major)
//      KT = k exp(gamma_L - gamma)              (64 x 128, as keys x tokens)
//      exp(gamma_L) per key row
//    For the per-channel gate (KDA, vLLM kimi_k3 kda/chunk_intra) the
//    exponentials move into the operands: S = [k e^g; q e^g] (k e^-g)^T with
//    the chunk start as reference row, w = T diag(beta) (k e^g), and
//    KT = k exp(gamma_L - gamma) per channel.
//
// 2. chain (one CTA per (32-wide V tile, value head, sequence)), the
//    sequential inter-chunk pass with the fp32 state tile h[128, 32] held in
//    registers (one key row per thread) for the whole sequence:
//      D  = TU v_tile                  ([u; Aqk u])
//      D += WQ bf16(h)                 (rows 0..63: v_new = u - w h,
//                                       rows 64..127: o = q~ h + Aqk v_new)
//      h  = exp(gamma_L) h + KT^T v_new
//    (KDA _fla/ops/common/chunk_h.py, chunk_fwd_kernel_h, gives the state
//    recurrence this delta form extends; o is fused into the same GEMM.)
//
// Shared-memory operand images use the canonical no-swizzle layout: element
// (r, c) of an image with column-group stride `cs` sits at
// (c / 8) * cs + r * 16 + (c % 8) * 2 bytes, i.e. every group of 8 columns is
// a contiguous run of 16-byte rows.  Read with rows as M/N (K-major) the
// descriptor has LBO = cs, SBO = 128; read with rows as K (MN-major) it has
// LBO = 128, SBO = cs.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "ptx.cuh"

namespace gdn {
namespace tc {

constexpr int KD = 128;
constexpr int VTILE = 32;
constexpr uint32_t WQ_BYTES = 32768, TU_BYTES = 16384, KT_BYTES = 16384, GATE_BYTES = 512;
constexpr uint32_t OFF_WQ = 0, OFF_TU = WQ_BYTES, OFF_KT = OFF_TU + TU_BYTES,
                   OFF_GATE = OFF_KT + KT_BYTES;
constexpr uint32_t BLOCK_BYTES = OFF_GATE + GATE_BYTES;  // 66048
constexpr uint32_t VT_BYTES = 64 * VTILE * 2;            // 4096
constexpr uint32_t STAGE_BYTES = BLOCK_BYTES + VT_BYTES;
constexpr float GATE_FACTOR_LIMIT = 80.f;  // |gamma| bound for split exponentials

__device__ __forceinline__ uint32_t img_off(int r, int c, uint32_t cs) {
  return (uint32_t)(c >> 3) * cs + (uint32_t)r * 16u + (uint32_t)(c & 7) * 2u;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ void unpack8(uint4 u, float *f) {
  const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 x = __bfloat1622float2(h[e]);
    f[2 * e] = x.x;
    f[2 * e + 1] = x.y;
  }
}

__device__ __forceinline__ uint4 pack8(const float *f) {
  uint4 u;
  u.x = pack_bf16x2(f[0], f[1]);
  u.y = pack_bf16x2(f[2], f[3]);
  u.z = pack_bf16x2(f[4], f[5]);
  u.w = pack_bf16x2(f[6], f[7]);
  return u;
}

struct TcParams {
  const float *g, *beta, *h0;
  float *ht;
  __nv_bfloat16 *o;
  const int32_t *cu_seqlens;
  int32_t *table;          // [N + 1] chunk offsets (packed sequences)
  unsigned char *blocks;   // per (chunk, head) operand blocks
  const void *kraw, *qraw;  // KDA exact fallback reads raw k/q
  int *err;
  int B, T, H, Hk, V, N, NT;  // NT: chunks per sequence without cu_seqlens
  int g_is_cumsum;
  float scale;
};

// Bounded wait shared by all threads; false means it gave up.
__device__ __forceinline__ bool wait_all(uint64_t *bar, uint32_t parity) {
  return ptx::mbar_wait_bounded(bar, parity);
}

// ---------------------------------------------------------------------------
// chunk table for packed sequences: table[n] = sum_{m<n} ceil(len_m / 64)
__global__ void chunk_table_kernel(const int32_t *cu, int N, int T, int32_t *table, int *err) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  bool ok = cu[0] == 0 && cu[N] == T;
  for (int n = 0; n < N && ok; ++n) ok = cu[n + 1] >= cu[n];
  if (!ok) record_error(err, GDN_ERR_BAD_SEQLENS);
  int acc = 0;
  for (int n = 0; n < N; ++n) {
    table[n] = acc;
    if (ok) acc += (cu[n + 1] - cu[n] + BT - 1) / BT;
  }
  table[N] = acc;
}

// Map a global chunk id to (sequence, chunk-in-sequence, token bounds).
struct ChunkPos {
  int n, c, bos, eos, b;
};

__device__ __forceinline__ bool locate_chunk(const TcParams &p, int id, ChunkPos &cp) {
  if (p.cu_seqlens) {
    const int total = p.table[p.N];
    if (id >= total) return false;
    int lo = 0, hi = p.N - 1;  // largest n with table[n] <= id
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.table[mid] <= id) lo = mid; else hi = mid - 1;
    }
    cp.n = lo;
    cp.c = id - p.table[lo];
    cp.bos = p.cu_seqlens[lo];
    cp.eos = p.cu_seqlens[lo + 1];
    cp.b = 0;
  } else {
    if (id >= p.B * p.NT) return false;
    cp.n = id / p.NT;
    cp.c = id % p.NT;
    cp.bos = 0;
    cp.eos = p.T;
    cp.b = cp.n;
  }
  return cp.bos + cp.c * BT < cp.eos;
}

// ---------------------------------------------------------------------------
// (I + A)^-1 for strictly lower-triangular 64x64 A (fp32, row stride 65) by
// 16x16 diagonal-block forward substitution and a three-level block merge
// (T_ij = -T_ii sum_{j<=m<i} A_im T_mj).  128 threads; X is scratch for
// 3 x 16 x 17 floats.  Only the lower block triangle of T is written.
__device__ void unit_lower_inverse_64(const float *A, float *Tm, float *X, int tid) {
  constexpr int LD = 65, XLD = 17;
  if (tid < 64) {
    const int o = (tid >> 4) * 16, j = tid & 15;
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float acc = (i == j) ? 1.f : 0.f;
#pragma unroll
      for (int m = 0; m < i; ++m) acc = fmaf(-A[(o + i) * LD + o + m], x[m], acc);
      x[i] = acc;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) Tm[(o + i) * LD + o + j] = x[i];
  }
  __syncthreads();
  // level d: blocks (b + d, b) for b = 0 .. 3 - d
  for (int d = 1; d <= 3; ++d) {
    const int nblk = 4 - d;
    // X_b = sum_{m = b .. b+d-1} A_{b+d, m} T_{m, b}
    for (int e = tid; e < nblk * 256; e += 128) {
      const int b = e >> 8, r = (e >> 4) & 15, cc = e & 15;
      const int ro = (b + d) * 16 + r;
      float acc = 0.f;
      for (int mb = b; mb < b + d; ++mb)
#pragma unroll
        for (int m = 0; m < 16; ++m)
          acc = fmaf(A[ro * LD + mb * 16 + m], Tm[(mb * 16 + m) * LD + b * 16 + cc], acc);
      X[(b * 16 + r) * XLD + cc] = acc;
    }
    __syncthreads();
    // T_{b+d, b} = -T_{b+d, b+d} X_b
    for (int e = tid; e < nblk * 256; e += 128) {
      const int b = e >> 8, r = (e >> 4) & 15, cc = e & 15;
      const int o = (b + d) * 16;
      float acc = 0.f;
#pragma unroll
      for (int m = 0; m < 16; ++m) acc = fmaf(Tm[(o + r) * LD + o + m], X[(b * 16 + m) * XLD + cc], acc);
      Tm[(o + r) * LD + b * 16 + cc] = -acc;
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// intra kernel
//
// shared memory (bytes):
//   KQ   [0, 32768)        k rows 0..63 / q rows 64..127 (x 128 keys), cs 2048
//   TA   [32768, 65536)    [Tw | Tu ; Aqk Tw | Aqk Tu] (128 x 128), cs 2048;
//                          during the solve its start holds the merge scratch,
//                          after the WY GEMM its first half holds KT (cs 1024)
//   R1   [65536, 98816)    A, T fp32 (64 x 65 each); later WQ (cs 2048)
//   AQK  [98816, 107008)   Aqk bf16 (64 x 64), cs 1024; KDA: also k e^-g
//                          (64 x 128, cs 1024) in [98816, 115200)
//   small                  gamma, factors, gate, barriers
constexpr uint32_t I_KQ = 0, I_TA = 32768, I_R1 = 65536, I_AQK = 98816;
constexpr uint32_t I_KB = I_AQK + 8192;     // KDA: k e^{-gamma} image (16 KB)
constexpr uint32_t I_KT = I_KB + 16384;     // KDA: KT image (16 KB)
template <bool KDA>
struct IntraLayout {
  static constexpr uint32_t SMALL = KDA ? I_KT + 16384 : I_AQK + 8192 + 1024;
  static constexpr uint32_t SMEM = SMALL + 4096;
};

template <bool KDA>
__global__ void __launch_bounds__(128, 1)
intra_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
             TcParams p) {
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char *KQ = smem + I_KQ;
  unsigned char *TA = smem + I_TA;
  float *Asm = reinterpret_cast<float *>(smem + I_R1);
  float *Tsm = Asm + 64 * 65;
  unsigned char *WQ = smem + I_R1;
  unsigned char *AQK = smem + I_AQK;
  unsigned char *KB = smem + I_KB;
  unsigned char *KTs = KDA ? smem + I_KT : TA;  // GDN: KT reuses TA's first half
  float *Xs = reinterpret_cast<float *>(smem + I_TA);
  float *gam = reinterpret_cast<float *>(smem + IntraLayout<KDA>::SMALL);  // [64]
  float *bet = gam + 64;                                   // [64]
  float *eg = bet + 64;                                    // [64] e^{gamma}
  float *eng = eg + 64;                                    // [64] e^{-gamma}
  float *gate = eng + 64;                                  // [128] e^{gamma_L}
  float *gl = gate + 128;                                  // [128] KDA gamma_L
  uint64_t *bars = reinterpret_cast<uint64_t *>(gl + 128); // tma, mma
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2);
  int *flags = reinterpret_cast<int *>(tmem_slot + 1);     // [0]: split exps ok

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.y;
  ChunkPos cp;
  if (!locate_chunk(p, blockIdx.x, cp)) return;
  const int hk = h / (p.H / p.Hk);
  const int s0 = cp.bos + cp.c * BT;
  const int L = min(BT, cp.eos - s0);
  const int row0 = cp.b * p.T + s0;  // token row in the [B*T] flattening
  const int chunk_id = blockIdx.x;
  unsigned char *blk = p.blocks + ((size_t)chunk_id * p.H + h) * BLOCK_BYTES;

  if (tid == 0) {
    ptx::mbar_init(&bars[0], 1);
    ptx::mbar_init(&bars[1], 1);
    ptx::fence_mbar_init();
    flags[0] = 1;
  }
  if (warp == 0) ptx::tmem_alloc<128>(tmem_slot);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (tid == 0) {
    ptx::mbar_arrive_expect_tx(&bars[0], 32768);
#pragma unroll 1
    for (int j = 0; j < 16; ++j) {
      ptx::tma_load_3d(KQ + j * 2048, &tm_k, 8 * j, hk, row0, &bars[0]);
      ptx::tma_load_3d(KQ + j * 2048 + 1024, &tm_q, 8 * j, hk, row0, &bars[0]);
    }
  }

  // ---- gates: gamma (chunk-local inclusive cumsum), beta
  if (tid < 64) bet[tid] = tid < L ? p.beta[(size_t)(row0 + tid) * p.H + h] : 0.f;
  bool gate_ok = true;
  if (!KDA) {
    if (warp == 0) {
      float a0 = 2 * lane < L ? p.g[(size_t)(row0 + 2 * lane) * p.H + h] : 0.f;
      float a1 = 2 * lane + 1 < L ? p.g[(size_t)(row0 + 2 * lane + 1) * p.H + h] : 0.f;
      float c0, c1;
      if (p.g_is_cumsum) {
        c0 = a0;
        c1 = a1;
        const float last = __shfl_sync(0xffffffffu, ((L - 1) & 1) ? a1 : a0, (L - 1) >> 1);
        if (2 * lane >= L) c0 = last;
        if (2 * lane + 1 >= L) c1 = last;
      } else {
        const float pair = a0 + a1;
        float incl = pair;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, incl, off);
          if (lane >= off) incl += y;
        }
        c0 = incl - pair + a0;
        c1 = c0 + a1;
      }
      gam[2 * lane] = c0;
      gam[2 * lane + 1] = c1;
      const bool ok = fabsf(c0) <= GATE_FACTOR_LIMIT && fabsf(c1) <= GATE_FACTOR_LIMIT;
      if (!__all_sync(0xffffffffu, ok) && lane == 0) flags[0] = 0;
    }
    __syncthreads();
    if (tid < 64) {
      eg[tid] = __expf(gam[tid]);
      eng[tid] = __expf(-gam[tid]);
    }
    if (tid < KD) gate[tid] = __expf(gam[L - 1]);
  } else {
    // thread c owns key channel c: running cumsum down the 64 rows into R1
    // (fp32 [64][128]); gamma of padded rows repeats row L - 1
    float *G = Asm;  // R1 is free until the solve
    const int c = tid;
    float acc = 0.f, mn = 0.f, mx = 0.f;
    for (int i = 0; i < 64; ++i) {
      float gv;
      if (i < L) {
        const float raw = p.g[((size_t)(row0 + i) * p.H + h) * KD + c];
        acc = p.g_is_cumsum ? raw : acc + raw;
        gv = acc;
      } else {
        gv = acc;
      }
      G[i * KD + c] = gv;
      mn = fminf(mn, gv);
      mx = fmaxf(mx, gv);
    }
    gl[c] = acc;
    gate[c] = __expf(acc);
    gate_ok = mn >= -GATE_FACTOR_LIMIT && mx <= GATE_FACTOR_LIMIT;
    if (!__syncthreads_and(gate_ok) && tid == 0) flags[0] = 0;
  }
  __syncthreads();

  const bool ok_tma = wait_all(&bars[0], 0);
  if (!__syncthreads_and(ok_tma)) {
    if (tid == 0) record_error(p.err, GDN_ERR_TIMEOUT);
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) ptx::tmem_dealloc<128>(tmem);
    return;
  }
  const bool split = flags[0] != 0;

  if (KDA) {
    // KQ <- [k e^g ; q e^g] (never overflows: gamma <= 80),
    // KB <- k e^-g (split path only), KT <- k e^{gamma_L - g} (exact)
    const float *G = Asm;
    for (int pc = tid; pc < 64 * 16; pc += 128) {
      const int i = pc & 63, cg = pc >> 6;
      uint4 *kp = reinterpret_cast<uint4 *>(KQ + img_off(i, 8 * cg, 2048));
      uint4 *qp = reinterpret_cast<uint4 *>(KQ + img_off(64 + i, 8 * cg, 2048));
      float kf[8], qf[8], a[8], b[8], c[8], t[8];
      unpack8(*kp, kf);
      unpack8(*qp, qf);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float gv = G[i * KD + 8 * cg + e];
        const float ep = __expf(gv);
        a[e] = kf[e] * ep;
        b[e] = qf[e] * ep;
        c[e] = split ? kf[e] * __expf(-gv) : 0.f;
        t[e] = i < L ? kf[e] * __expf(gl[8 * cg + e] - gv) : 0.f;
      }
      *kp = pack8(a);
      *qp = pack8(b);
      *reinterpret_cast<uint4 *>(KB + img_off(i, 8 * cg, 1024)) = pack8(c);
      *reinterpret_cast<uint4 *>(KTs + img_off(i, 8 * cg, 1024)) = pack8(t);
    }
    ptx::fence_proxy_async_smem();
    __syncthreads();
  } else {
    ptx::fence_proxy_async_smem();
  }

  // ---- S = [k; q] k^T  (M = 128, N = 64, K = 128)
  const uint32_t dS = tmem;  // columns [0, 64)
  uint32_t mma_phase = 0;
  if (tid == 0) {
    ptx::tc_fence_after();
    const uint32_t id = ptx::idesc_bf16(128, 64, 0, 0);
    const unsigned char *Bop = KDA ? KB : KQ;
    const uint32_t b_cs = KDA ? 1024u : 2048u;
#pragma unroll 1
    for (int ks = 0; ks < 8; ++ks) {
      const uint64_t a = ptx::sdesc(KQ + ks * 2 * 2048, 2048, 128);
      const uint64_t b = ptx::sdesc(Bop + ks * 2 * b_cs, b_cs, 128);
      ptx::mma_bf16(dS, a, b, id, ks > 0);
    }
    ptx::mma_commit(&bars[1]);
  }
  const bool ok1 = wait_all(&bars[1], mma_phase);
  mma_phase ^= 1;
  ptx::tc_fence_after();

  // ---- gating: thread r holds row r of S (r < 64: kk, r >= 64: qk)
  {
    float srow[64];
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    ptx::tmem_ld32(dS + lane_base, srow);
    ptx::tmem_ld32(dS + lane_base + 32, srow + 32);
    const int i = tid & 63;
    const bool is_q = tid >= 64;
    if (KDA && !split) {
      // exact per-element exponentials (only when |gamma| leaves the split
      // range): raw k/q from global memory, gamma from R1
      const float *G = Asm;
      const __nv_bfloat16 *kg = static_cast<const __nv_bfloat16 *>(p.kraw);
      const __nv_bfloat16 *qg = static_cast<const __nv_bfloat16 *>(p.qraw);
      const __nv_bfloat16 *xg = is_q ? qg : kg;
      for (int j = 0; j < 64; ++j) {
        float acc = 0.f;
        if (i < L && j <= i) {
          const size_t oi = ((size_t)(row0 + i) * p.Hk + hk) * KD;
          const size_t oj = ((size_t)(row0 + j) * p.Hk + hk) * KD;
          for (int c = 0; c < KD; ++c)
            acc = fmaf(__bfloat162float(xg[oi + c]) * __bfloat162float(kg[oj + c]),
                       __expf(G[i * KD + c] - G[j * KD + c]), acc);
        }
        srow[j] = acc;
      }
      __syncthreads();  // everyone done reading gamma before A overwrites R1
    }
    if (!is_q) {
      // A (fp32, row stride 65) for the solve: beta_i S_kk e^{g_i - g_j}, j < i < L
      const float bi = bet[i];
#pragma unroll
      for (int j = 0; j < 64; ++j) {
        float f;
        if (KDA) f = 1.f;
        else f = split ? eg[i] * eng[j] : __expf(gam[i] - gam[j]);
        Asm[i * 65 + j] = (j < i && i < L) ? bi * f * srow[j] : 0.f;
      }
    } else {
      // Aqk (bf16 image, cs 1024): scale S_qk e^{g_i - g_j}, j <= i < L
#pragma unroll
      for (int cg = 0; cg < 8; ++cg) {
        float v8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int j = cg * 8 + e;
          float f;
          if (KDA) f = 1.f;
          else f = split ? eg[i] * eng[j] : __expf(gam[i] - gam[j]);
          v8[e] = (j <= i && i < L) ? p.scale * f * srow[j] : 0.f;
        }
        *reinterpret_cast<uint4 *>(AQK + img_off(i, 8 * cg, 1024)) = pack8(v8);
      }
    }
  }
  ptx::tc_fence_before();
  __syncthreads();

  // ---- T = (I + A)^-1 (fp32)
  unit_lower_inverse_64(Asm, Tsm, Xs, tid);

  // ---- TA rows 0..63: Tw = T diag(dw), Tu = T diag(beta)  (lower triangle)
  for (int pc = tid; pc < 64 * 16; pc += 128) {
    const int i = pc & 63, cg = pc >> 6;
    const bool is_u = cg >= 8;
    const int j0 = (cg & 7) * 8;
    float v8[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int j = j0 + e;
      const float t = (j <= i) ? Tsm[i * 65 + j] : 0.f;
      const float d = is_u ? bet[j] : (KDA ? bet[j] : bet[j] * eg[j]);
      v8[e] = t * d;
    }
    *reinterpret_cast<uint4 *>(TA + img_off(i, 8 * cg, 2048)) = pack8(v8);
  }
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before();
  __syncthreads();

  // ---- P = Aqk [Tw | Tu]  (M = 64, N = 128, K = 64)
  const uint32_t dP = tmem;
  if (tid == 0) {
    ptx::tc_fence_after();
    const uint32_t id = ptx::idesc_bf16(64, 128, 0, 1);
#pragma unroll 1
    for (int ks = 0; ks < 4; ++ks) {
      const uint64_t a = ptx::sdesc(AQK + ks * 2 * 1024, 1024, 128);
      const uint64_t b = ptx::sdesc(TA + ks * 256, 128, 2048);
      ptx::mma_bf16(dP, a, b, id, ks > 0);
    }
    ptx::mma_commit(&bars[1]);
  }
  const bool ok2 = wait_all(&bars[1], mma_phase);
  mma_phase ^= 1;
  ptx::tc_fence_after();
  {
    // M = 64 layout: row 16 w + l lives in lane 32 w + l (l < 16)
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const int i = warp * 16 + (lane & 15);
#pragma unroll 1
    for (int half = 0; half < 4; ++half) {
      float v[32];
      ptx::tmem_ld32(dP + lane_base + half * 32, v);
      if (lane < 16) {
#pragma unroll
        for (int q8 = 0; q8 < 4; ++q8)
          *reinterpret_cast<uint4 *>(TA + img_off(64 + i, half * 32 + q8 * 8, 2048)) =
              pack8(v + q8 * 8);
      }
    }
  }
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before();
  __syncthreads();

  // ---- [w; Aqk w] = [Tw; Aqk Tw] k  (M = 128, N = 128 keys, K = 64 tokens);
  //      meanwhile TU (second half of TA) streams out to the block
  const uint32_t dW = tmem;
  if (tid == 0) {
    ptx::tc_fence_after();
    const uint32_t id = ptx::idesc_bf16(128, 128, 0, 1);
#pragma unroll 1
    for (int ks = 0; ks < 4; ++ks) {
      const uint64_t a = ptx::sdesc(TA + ks * 2 * 2048, 2048, 128);
      const uint64_t b = ptx::sdesc(KQ + ks * 256, 128, 2048);
      ptx::mma_bf16(dW, a, b, id, ks > 0);
    }
    ptx::mma_commit(&bars[1]);
    ptx::bulk_s2g(blk + OFF_TU, TA + 16384, TU_BYTES);
    ptx::bulk_commit();
  }
  const bool ok3 = wait_all(&bars[1], mma_phase);
  mma_phase ^= 1;
  ptx::tc_fence_after();

  // ---- WQ, KT
  {
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const int r = tid;
    const int i = r & 63;
    const bool is_q = r >= 64;
    const float gli = KDA ? 0.f : gam[L - 1];
    const float fq = KDA ? p.scale : p.scale * eg[i];
    const float fk = KDA ? 0.f : (split ? gate[0] * eng[i] : __expf(gli - gam[i]));
#pragma unroll 1
    for (int q4 = 0; q4 < 4; ++q4) {
      float v[32];
      ptx::tmem_ld32(dW + lane_base + q4 * 32, v);
#pragma unroll
      for (int q8 = 0; q8 < 4; ++q8) {
        const int c0 = q4 * 32 + q8 * 8;
        float out[8];
        if (!is_q) {
#pragma unroll
          for (int e = 0; e < 8; ++e) out[e] = -v[q8 * 8 + e];
        } else {
          float qf[8];
          unpack8(*reinterpret_cast<const uint4 *>(KQ + img_off(64 + i, c0, 2048)), qf);
#pragma unroll
          for (int e = 0; e < 8; ++e) out[e] = fq * qf[e] - v[q8 * 8 + e];
        }
        *reinterpret_cast<uint4 *>(WQ + img_off(r, c0, 2048)) = pack8(out);
      }
    }
    if (!KDA && !is_q) {
      // KT row i: k e^{gamma_L - gamma_i} (zero beyond the chunk)
#pragma unroll 1
      for (int cg = 0; cg < 16; ++cg) {
        float kr[8], kt[8];
        unpack8(*reinterpret_cast<const uint4 *>(KQ + img_off(i, 8 * cg, 2048)), kr);
#pragma unroll
        for (int e = 0; e < 8; ++e) kt[e] = (i < L) ? kr[e] * fk : 0.f;
        *reinterpret_cast<uint4 *>(KTs + img_off(i, 8 * cg, 1024)) = pack8(kt);
      }
    }
  }
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before();
  __syncthreads();
  if (tid == 0) {
    ptx::bulk_s2g(blk + OFF_WQ, WQ, WQ_BYTES);
    ptx::bulk_s2g(blk + OFF_KT, KTs, KT_BYTES);
    ptx::bulk_s2g(blk + OFF_GATE, gate, GATE_BYTES);
    ptx::bulk_commit();
    ptx::bulk_wait<0>();
  }
  if (!(ok1 && ok2 && ok3) && tid == 0) record_error(p.err, GDN_ERR_TIMEOUT);
  __syncthreads();
  if (warp == 0) ptx::tmem_dealloc<128>(tmem);
}

// ---------------------------------------------------------------------------
// chain kernel
//
// shared memory: two stages of [operand block (66048 B) | v tile (4096 B)],
// then the bf16 state image H (128 keys x 32, cs 2048) and v_new image VN
// (64 tokens x 32, cs 1024).
constexpr uint32_t C_STAGE0 = 0, C_H = 2 * STAGE_BYTES, C_VN = C_H + 8192,
                   C_SMALL = C_VN + 4096, C_SMEM = C_SMALL + 256;

__global__ void __launch_bounds__(128, 1)
chain_kernel(const __grid_constant__ CUtensorMap tm_v, TcParams p) {
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char *Himg = smem + C_H;
  unsigned char *VN = smem + C_VN;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C_SMALL);  // full0, full1, mma
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 3);

  const int tid = threadIdx.x, warp = tid >> 5;
  const int v0 = blockIdx.x * VTILE;
  const int h = blockIdx.y;
  const int n = blockIdx.z;
  int bos, eos, b, base;
  if (p.cu_seqlens) {
    bos = p.cu_seqlens[n];
    eos = p.cu_seqlens[n + 1];
    b = 0;
    base = p.table[n];
    if (p.table[p.N] == 0 || eos < bos) eos = bos;  // invalid table: no chunks
  } else {
    bos = 0;
    eos = p.T;
    b = n;
    base = n * p.NT;
  }
  const int nch = (eos - bos + BT - 1) / BT;

  if (tid == 0) {
    ptx::mbar_init(&bars[0], 1);
    ptx::mbar_init(&bars[1], 1);
    ptx::mbar_init(&bars[2], 1);
    ptx::fence_mbar_init();
  }
  if (warp == 0) ptx::tmem_alloc<128>(tmem_slot);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;

  auto issue = [&](int c) {
    const int s = c & 1;
    unsigned char *st = smem + C_STAGE0 + s * STAGE_BYTES;
    ptx::mbar_arrive_expect_tx(&bars[s], STAGE_BYTES);
    ptx::bulk_g2s(st, p.blocks + ((size_t)(base + c) * p.H + h) * BLOCK_BYTES, BLOCK_BYTES,
                  &bars[s]);
    const int trow = b * p.T + bos + c * BT;
#pragma unroll
    for (int vg = 0; vg < 4; ++vg)
      ptx::tma_load_3d(st + BLOCK_BYTES + vg * 1024, &tm_v, v0 + 8 * vg, h, trow, &bars[s]);
  };
  if (tid == 0) {
    if (nch > 0) issue(0);
    if (nch > 1) issue(1);
  }

  // initial state: thread c owns key row c of the tile
  float hs[VTILE];
  {
    const int c = tid;
    if (p.h0) {
      const float4 *src =
          reinterpret_cast<const float4 *>(p.h0 + (((size_t)n * p.H + h) * KD + c) * p.V + v0);
#pragma unroll
      for (int q = 0; q < VTILE / 4; ++q) {
        const float4 x = src[q];
        hs[4 * q] = x.x; hs[4 * q + 1] = x.y; hs[4 * q + 2] = x.z; hs[4 * q + 3] = x.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < VTILE; ++j) hs[j] = 0.f;
    }
#pragma unroll
    for (int vg = 0; vg < 4; ++vg)
      *reinterpret_cast<uint4 *>(Himg + img_off(c, 8 * vg, 2048)) = pack8(hs + 8 * vg);
  }
  ptx::fence_proxy_async_smem();
  __syncthreads();

  uint32_t mma_phase = 0;
  bool ok = true;
  const uint32_t id_u = ptx::idesc_bf16(128, VTILE, 0, 1);
  const uint32_t id_c3 = ptx::idesc_bf16(128, VTILE, 1, 1);
#pragma unroll 1
  for (int c = 0; c < nch; ++c) {
    const int s = c & 1;
    unsigned char *st = smem + C_STAGE0 + s * STAGE_BYTES;
    const uint32_t dU = tmem + s * 32;
    const uint32_t dH = tmem + 64;
    const int L = min(BT, eos - bos - c * BT);
    ok = wait_all(&bars[s], (uint32_t)((c >> 1) & 1)) && ok;
    if (tid == 0) {
      ptx::tc_fence_after();
      // D = TU v_tile
#pragma unroll 1
      for (int ks = 0; ks < 4; ++ks) {
        const uint64_t a = ptx::sdesc(st + OFF_TU + ks * 2 * 2048, 2048, 128);
        const uint64_t bb = ptx::sdesc(st + BLOCK_BYTES + ks * 256, 128, 1024);
        ptx::mma_bf16(dU, a, bb, id_u, ks > 0);
      }
      // D += WQ h
#pragma unroll 1
      for (int ks = 0; ks < 8; ++ks) {
        const uint64_t a = ptx::sdesc(st + OFF_WQ + ks * 2 * 2048, 2048, 128);
        const uint64_t bb = ptx::sdesc(Himg + ks * 256, 128, 2048);
        ptx::mma_bf16(dU, a, bb, id_u, 1);
      }
      ptx::mma_commit(&bars[2]);
    }
    const float decay = reinterpret_cast<const float *>(st + OFF_GATE)[tid];
    ok = wait_all(&bars[2], mma_phase) && ok;
    mma_phase ^= 1;
    ptx::tc_fence_after();
    {
      float d[32];
      ptx::tmem_ld32(dU + lane_base, d);
      if (tid < 64) {
#pragma unroll
        for (int vg = 0; vg < 4; ++vg)
          *reinterpret_cast<uint4 *>(VN + img_off(tid, 8 * vg, 1024)) = pack8(d + 8 * vg);
      } else {
        const int i = tid - 64;
        if (i < L) {
          uint4 *dst = reinterpret_cast<uint4 *>(
              p.o + ((size_t)(b * p.T + bos + c * BT + i) * p.H + h) * p.V + v0);
#pragma unroll
          for (int vg = 0; vg < 4; ++vg) dst[vg] = pack8(d + 8 * vg);
        }
      }
    }
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      ptx::tc_fence_after();
      // D_H = KT^T v_new  (M = 128 keys, K = 64 tokens)
#pragma unroll 1
      for (int ks = 0; ks < 4; ++ks) {
        const uint64_t a = ptx::sdesc(st + OFF_KT + ks * 256, 128, 1024);
        const uint64_t bb = ptx::sdesc(VN + ks * 256, 128, 1024);
        ptx::mma_bf16(dH, a, bb, id_c3, ks > 0);
      }
      ptx::mma_commit(&bars[2]);
    }
    ok = wait_all(&bars[2], mma_phase) && ok;
    mma_phase ^= 1;
    ptx::tc_fence_after();
    {
      float d[32];
      ptx::tmem_ld32(dH + lane_base, d);
#pragma unroll
      for (int j = 0; j < VTILE; ++j) hs[j] = fmaf(decay, hs[j], d[j]);
#pragma unroll
      for (int vg = 0; vg < 4; ++vg)
        *reinterpret_cast<uint4 *>(Himg + img_off(tid, 8 * vg, 2048)) = pack8(hs + 8 * vg);
    }
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_before();
    if (!__syncthreads_and(ok)) break;
    if (tid == 0 && c + 2 < nch) {
      ptx::fence_proxy_async_smem();  // generic reads of stage s precede the refill
      issue(c + 2);
    }
  }
  if (!ok) {
    if (tid == 0) record_error(p.err, GDN_ERR_TIMEOUT);
  } else if (p.ht) {
    float4 *dst =
        reinterpret_cast<float4 *>(p.ht + (((size_t)n * p.H + h) * KD + tid) * p.V + v0);
#pragma unroll
    for (int q = 0; q < VTILE / 4; ++q)
      dst[q] = make_float4(hs[4 * q], hs[4 * q + 1], hs[4 * q + 2], hs[4 * q + 3]);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) ptx::tmem_dealloc<128>(tmem);
}

// ---------------------------------------------------------------------------
// host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// [rows][heads][dim] bf16 tensor, boxes of 8 x 1 x 64 (16-byte rows).
bool make_map(CUtensorMap *m, const void *base, int dim, int heads, long long rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t gdim[3] = {(cuuint64_t)dim, (cuuint64_t)heads, (cuuint64_t)rows};
  cuuint64_t gstride[2] = {(cuuint64_t)dim * 2, (cuuint64_t)heads * dim * 2};
  cuuint32_t box[3] = {8, 1, 64};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), gdim, gstride, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t table_bytes(int N) { return (((size_t)N + 1) * 4 + 255) / 256 * 256; }

size_t max_chunks(int B, int T, int N, bool varlen) {
  const size_t nt = ((size_t)T + BT - 1) / BT;
  return varlen ? nt + (size_t)N : (size_t)B * nt;
}

}  // namespace tc

bool chunk_tc_supported(const ChunkParams &p, bool bf16) {
  return bf16 && p.K == tc::KD && p.V % tc::VTILE == 0 && p.T > 0;
}

size_t chunk_tc_workspace(const ChunkParams &p) {
  const bool varlen = p.cu_seqlens != nullptr;
  return tc::table_bytes(p.N) + tc::max_chunks(p.B, p.T, p.N, varlen) * (size_t)p.H * tc::BLOCK_BYTES;
}

cudaError_t launch_chunk_tc(const ChunkParams &cp, bool kda, void *ws, cudaStream_t stream) {
  using namespace tc;
  const bool varlen = cp.cu_seqlens != nullptr;
  CUtensorMap mk, mq, mv;
  const long long rows = (long long)cp.B * cp.T;
  if (!make_map(&mk, cp.k, KD, cp.Hk, rows) || !make_map(&mq, cp.q, KD, cp.Hk, rows) ||
      !make_map(&mv, cp.v, cp.V, cp.H, rows))
    return cudaErrorInvalidValue;
  TcParams p{};
  p.g = cp.g; p.beta = cp.beta; p.h0 = cp.h0; p.ht = cp.ht;
  p.kraw = cp.k; p.qraw = cp.q;
  p.o = static_cast<__nv_bfloat16 *>(cp.o);
  p.cu_seqlens = cp.cu_seqlens;
  p.table = static_cast<int32_t *>(ws);
  p.blocks = static_cast<unsigned char *>(ws) + table_bytes(cp.N);
  p.err = cp.err;
  p.B = cp.B; p.T = cp.T; p.H = cp.H; p.Hk = cp.Hk; p.V = cp.V; p.N = cp.N;
  p.NT = (cp.T + BT - 1) / BT;
  p.g_is_cumsum = cp.g_is_cumsum;
  p.scale = cp.scale;
  if (varlen) {
    chunk_table_kernel<<<1, 32, 0, stream>>>(cp.cu_seqlens, cp.N, cp.T, p.table, cp.err);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const size_t nchunks = max_chunks(cp.B, cp.T, cp.N, varlen);
  auto ik = kda ? intra_kernel<true> : intra_kernel<false>;
  const uint32_t ismem = kda ? IntraLayout<true>::SMEM : IntraLayout<false>::SMEM;
  cudaError_t e = cudaFuncSetAttribute(ik, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ismem);
  if (e != cudaSuccess) return e;
  ik<<<dim3((unsigned)nchunks, cp.H), 128, ismem, stream>>>(mk, mq, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C_SMEM);
  if (e != cudaSuccess) return e;
  chain_kernel<<<dim3(cp.V / VTILE, cp.H, cp.N), 128, C_SMEM, stream>>>(mv, p);
  return cudaGetLastError();
}

}  // namespace gdn
