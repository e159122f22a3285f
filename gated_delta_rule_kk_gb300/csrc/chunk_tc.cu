// Chunked forward on the 5th-generation tensor cores (tcgen05, TMEM
// accumulators, TMA and bulk copies), bf16 inputs, K = 128, V in {32..128}
// a multiple of 32.
//
// Two kernels per call (plus a small chunk-table kernel for packed
// sequences):
//
// 1. intra: one CTA per (chunk, value head) -- for the scalar gate per (chunk,
//    key head), taking the key head's value heads in turn -- all chunks in
//    parallel.  With
//    gamma the chunk-local cumulative gate and S = [k; q] k^T (one M = 128
//    tcgen05 GEMM; sglang fla/chunk_fwd.py, fused KK^T + solve kernel):
//      A   = beta_i S_kk[i,j] exp(gamma_i - gamma_j), i > j       (Steps 1-2)
//      Aqk = scale S_qk[i,j] exp(gamma_i - gamma_j),  i >= j
//      T   = (I + A)^-1: 16 x 16 diagonal blocks by forward substitution
//            (fp32), then the block merge on the warp-level tensor
//            cores (bf16 hi/lo operands, fp32 accumulation)     (Steps 3-4)
//      w   = T diag(beta e^gamma) k,  u = T diag(beta) v         (WY recompute)
//    T enters the two WY GEMMs as a hi + lo pair of bf16 matrices, so w and u
//    carry fp32-grade accuracy.  Per (chunk, head) the kernel stores a block
//    of ready-made operand images the sequential pass consumes directly:
//      AW  [-w ; q] (bf16)                U   u (fp32, per 32-wide V tile)
//      KT  [k~_hi ; k~_lo] (bf16 pair,    SC  exp(gamma_L) per key row,
//          k~ = k e^{gamma_L - gamma};        exp(gamma_L - gamma_i) and
//          per-channel gate only)             scale exp(gamma_i) per token
//      AQ  [Aqk_lo ; Aqk_hi] (bf16 pair)
//    For the per-channel gate (KDA, vLLM kimi_k3 kda/chunk_intra,
//    chunk_kda_fwd_kernel_inter_solve_fused) the exponentials move into the
//    operands: S = [k e^g; q e^g] (k e^-g)^T with the chunk start as the
//    reference row, w = T diag(beta) (k e^g), AW holds q e^g and KT holds
//    k e^{gamma_L - g}.
//
// 2. chain: one CTA per (32-wide V tile, value head, sequence), the
//    sequential inter-chunk pass, warp-specialised: warp 16 streams the
//    chunk's operand block in (five bulk copies), warp 17 issues the tcgen05
//    GEMMs, warps 0-15 run the epilogues (warps w, w + 4, w + 8, w + 12 share
//    TMEM lane quarter w % 4 and split its 32 columns; each thread keeps 8
//    columns of one key row of the fp32 state tile h[128, 32] in registers for
//    the whole sequence).  Per chunk
//      D1  = [-w ; q~] [h_hi | h_lo]      rows 0..63: -w h, rows 64..127: q h
//      v_new = u + D1[0..63]             (fp32; split into a hi + lo bf16 pair)
//      DH  = k~^T v_new                  (scalar gate: k^T (e^{gamma_L - gamma} v_new),
//                                         the factor on v_new's hi + lo pair and k
//                                         read raw from the input by TMA, exact in
//                                         bf16; per-channel gate: k~ = k
//                                         e^{gamma_L - g} as a hi + lo pair from
//                                         KT; either way the state update keeps
//                                         fp32-grade accuracy over long memories)
//      D5  = [Aqk_lo ; Aqk_hi] v_new
//      h   = exp(gamma_L) h + DH
//      o   = scale e^gamma (q h) + Aqk v_new
//    (KDA _fla/ops/common/chunk_h.py, chunk_fwd_kernel_h, is the gated state
//    recurrence that this delta form extends; the output is fused into it.)
//
// Shared-memory operand images are rows of 128 bytes in the 128-byte swizzle
// (the layout TMA writes): the 16-byte piece j of row r sits at piece
// j ^ (r & 7) of the row, and wider images keep their 64-column halves a
// fixed stride apart (swz_off, swz_row, sw128_kmajor below); v arrives in the
// 64-byte swizzle.  Only KT keeps the canonical no-swizzle layout: element
// (r, c) of an image with column-group stride `cs` sits at
// (c / 8) * cs + r * 16 + (c % 8) * 2 bytes, every group of 8 columns a
// contiguous run of 16-byte rows; read with rows as K (MN-major) its
// descriptor has LBO = 128, SBO = cs.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cmath>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "ptx.cuh"

namespace gdn {
namespace tc {

constexpr int KD = 128;
constexpr int VTILE = 32;
constexpr int VMAX = 128;
constexpr float GATE_FACTOR_LIMIT = 80.f;  // |gamma| bound for split exponentials

// per (chunk, head) block in the workspace: the chain's operand images
//   AW  [-w ; q~] (128 x 128 bf16, 128-byte swizzled rows, 64-column halves 16 KB apart)
//   KT  [k~_hi ; k~_lo] (128 token rows x 128 keys bf16, cs 2048)
//   AQ  [Aqk_lo ; Aqk_hi] (128 x 64, 128-byte swizzled rows) SC  decay[128], rs[64], qs[64]
//   U   u, fp32 [V / 32 tiles][64][32], 16-byte group q of row i at q ^ (i & 7)
constexpr uint32_t OFF_AW = 0, OFF_KT = 32768, OFF_AQ = 65536, OFF_SC = 81920, OFF_U = 82944;
__host__ __device__ constexpr uint32_t block_bytes(int V, bool) {
  return OFF_U + (uint32_t)V * 256u;
}

__device__ __forceinline__ uint32_t img_off(int r, int c, uint32_t cs) {
  return (uint32_t)(c >> 3) * cs + (uint32_t)r * 16u + (uint32_t)(c & 7) * 2u;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&v);
}

// hi = RNE(x), lo = RNE(x - hi), two values each (x0 in the low halves)
__device__ __forceinline__ void split_bf16x2(float x0, float x1, uint32_t &hi, uint32_t &lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  const float2 hf = __bfloat1622float2(h);
  hi = *reinterpret_cast<const uint32_t *>(&h);
  lo = pack_bf16x2(x0 - hf.x, x1 - hf.y);
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

// Packed fp32 pairs (sm_100: two lanes per instruction, each rounded to
// nearest, so the results equal the scalar operations').
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
  float2 r;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "sub.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  float2 r;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}

// x = hi + lo with hi = bf16(x), lo = bf16(x - hi): 16 significant bits.
__device__ __forceinline__ void split8(const float *f, uint4 &hi, uint4 &lo) {
  float r[8];
  hi = pack8(f);
  unpack8(hi, r);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 d = sub2(make_float2(f[2 * e], f[2 * e + 1]), make_float2(r[2 * e], r[2 * e + 1]));
    r[2 * e] = d.x;
    r[2 * e + 1] = d.y;
  }
  lo = pack8(r);
}

struct TcParams {
  const float *g, *beta, *h0;
  float *ht;
  void *o;                 // bf16, or fp32 with o_f32
  const int32_t *cu_seqlens;
  int32_t *table;          // [N + 1] chunk offsets, then [N] chain order (packed sequences)
  unsigned char *blocks;   // per (chunk, head) operand blocks
  const void *kraw, *qraw;  // KDA exact fallback reads raw k/q
  int *err;
  int B, T, H, Hk, V, N, NT;  // NT: chunks per sequence without cu_seqlens
  int g_is_cumsum;
  int v_first;             // h0, ht stored [V, K] per (sequence, head) instead of [K, V]
  int o_f32;               // o written as fp32 instead of bf16
  float scale;
  uint32_t block;          // bytes per (chunk, head) block
  int nblk;                // chunk slots in `blocks` (blocks holds nblk * H blocks)
  // segment-parallel state pass (seg_count >= 2; see chain_kernel)
  int seg_count;           // segments per sequence
  int seg_phase;           // 0: whole sequences; 1: every segment from zero / identity;
                           // 2: segments 1 .. seg_count-1 again from their true start
  float *seg_state;        // [N][seg_count][H][K][K + V]: phase-1 ends, [M_s | B_s]
  float *seg_start;        // [N][seg_count][H][K][V]: combined start states (s >= 1)
};

// ---------------------------------------------------------------------------
// Chunk table for packed sequences: table[n] = sum_{m<n} ceil(len_m / 64)
// for n = 0..N, then the order in which the chain kernel takes the sequences:
// by decreasing chunk count (ties by index) when N <= ORDER_MAX, else by
// index.  The chain CTAs are dispatched in that order, so the longest chains,
// which set the call's length, start first.
constexpr int TABLE_THREADS = 512, ORDER_MAX = 1024;
__global__ void __launch_bounds__(TABLE_THREADS)
    chunk_table_kernel(const int32_t *cu, int N, int T, int32_t *table, int *err) {
  __shared__ int cnt[ORDER_MAX];
  __shared__ int valid;
  const int tid = threadIdx.x;
  int32_t *order = table + N + 1;
  if (tid == 0) {
    bool ok = cu[0] == 0 && cu[N] == T;
    for (int n = 0; n < N && ok; ++n) ok = cu[n + 1] >= cu[n];
    if (!ok) record_error(err, GDN_ERR_BAD_SEQLENS);
    int acc = 0;
    for (int n = 0; n < N; ++n) {
      table[n] = acc;
      if (ok) acc += (cu[n + 1] - cu[n] + BT - 1) / BT;
    }
    table[N] = acc;
    valid = ok ? 1 : 0;
  }
  __syncthreads();
  if (!valid || N > ORDER_MAX) {
    for (int n = tid; n < N; n += TABLE_THREADS) order[n] = n;
    return;
  }
  for (int n = tid; n < N; n += TABLE_THREADS) cnt[n] = (cu[n + 1] - cu[n] + BT - 1) / BT;
  __syncthreads();
  for (int n = tid; n < N; n += TABLE_THREADS) {
    const int c = cnt[n];
    int rank = 0;  // position of n under (count descending, index ascending)
    for (int m = 0; m < N; ++m) rank += (cnt[m] > c) || (cnt[m] == c && m < n);
    order[rank] = n;
  }
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
// (I + A)^-1 for strictly lower-triangular 64x64 A (fp32, row stride SLD, rows
// 16-byte aligned) by 16x16 diagonal-block forward substitution (fp32, CUDA
// cores) and a three-level block merge T_ij = -T_ii sum_{j<=m<i} A_im T_mj
// (warp-level tensor cores).  NT threads; only the lower block triangle of T
// is written.
constexpr int SLD = 68, XLD = 18;  // XLD: the small region keeps 3 x 16 x XLD floats free
template <int NT>
__device__ void unit_lower_inverse_64(const float *A, float *Tm, int tid) {
  static_assert(NT >= 96, "the merge takes warps 0..2");
  if (tid < 64) {
    // thread (o, j): column j of diagonal block o
    const int o = (tid >> 4) * 16, j = tid & 15;
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float a[16];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (4 * q < i) {
          const float4 v = *reinterpret_cast<const float4 *>(A + (o + i) * SLD + o + 4 * q);
          a[4 * q] = v.x; a[4 * q + 1] = v.y; a[4 * q + 2] = v.z; a[4 * q + 3] = v.w;
        }
      }
      float acc0 = (i == j) ? 1.f : 0.f, acc1 = 0.f;
#pragma unroll
      for (int m = 0; m < i; ++m) {
        if (m & 1) acc1 = fmaf(-a[m], x[m], acc1);
        else acc0 = fmaf(-a[m], x[m], acc0);
      }
      x[i] = acc0 + acc1;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) Tm[(o + i) * SLD + o + j] = x[i];
  }
  __syncthreads();
  // level d: blocks (b + d, b) for b = 0 .. 3 - d, warp b each, on the tensor
  // cores (m16n8k16 with bf16 hi/lo operands: hi.hi + hi.lo + lo.hi, fp32
  // accumulation).  The warp forms X^T = sum_m T_{m,b}^T A_{b+d,m}^T, then
  // T_{b+d,b}^T = -X^T T_{b+d,b+d}^T with X^T's accumulators serving directly
  // as the second product's A fragments.
  const int warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
#pragma unroll 1
  for (int d = 1; d <= 3; ++d) {
    if (warp <= 3 - d) {
      const int b = warp, r = (b + d) * 16, c = b * 16;
      float xt[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll 1
      for (int m = b; m < b + d; ++m) {
        // A = T_{m,b}^T: element (i, k) = T[16 m + k][c + i]
        const float *Tb = Tm + (16 * m) * SLD + c;
        uint32_t ah[4], al[4];
        split_bf16x2(Tb[(2 * t) * SLD + g], Tb[(2 * t + 1) * SLD + g], ah[0], al[0]);
        split_bf16x2(Tb[(2 * t) * SLD + g + 8], Tb[(2 * t + 1) * SLD + g + 8], ah[1], al[1]);
        split_bf16x2(Tb[(2 * t + 8) * SLD + g], Tb[(2 * t + 9) * SLD + g], ah[2], al[2]);
        split_bf16x2(Tb[(2 * t + 8) * SLD + g + 8], Tb[(2 * t + 9) * SLD + g + 8], ah[3], al[3]);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          // B = A_{b+d,m}^T: element (k, n) = A[r + 8 nt + n][16 m + k]
          const float *Ar = A + (r + 8 * nt + g) * SLD + 16 * m;
          const float2 p0 = *reinterpret_cast<const float2 *>(Ar + 2 * t);
          const float2 p1 = *reinterpret_cast<const float2 *>(Ar + 2 * t + 8);
          uint32_t bh0, bl0, bh1, bl1;
          split_bf16x2(p0.x, p0.y, bh0, bl0);
          split_bf16x2(p1.x, p1.y, bh1, bl1);
          ptx::mma_16816_bf16(xt[nt], ah, bh0, bh1);
          ptx::mma_16816_bf16(xt[nt], ah, bl0, bl1);
          ptx::mma_16816_bf16(xt[nt], al, bh0, bh1);
        }
      }
      uint32_t xh[4], xl[4];
      split_bf16x2(xt[0][0], xt[0][1], xh[0], xl[0]);
      split_bf16x2(xt[0][2], xt[0][3], xh[1], xl[1]);
      split_bf16x2(xt[1][0], xt[1][1], xh[2], xl[2]);
      split_bf16x2(xt[1][2], xt[1][3], xh[3], xl[3]);
      float *Tw = Tm + r * SLD + c;  // T_{b+d,b}
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        // B = T_{b+d,b+d}^T: element (k, n) = T[r + 8 nt + n][r + k]
        const float *Tr = Tm + (r + 8 * nt + g) * SLD + r;
        const float2 p0 = *reinterpret_cast<const float2 *>(Tr + 2 * t);
        const float2 p1 = *reinterpret_cast<const float2 *>(Tr + 2 * t + 8);
        uint32_t bh0, bl0, bh1, bl1;
        split_bf16x2(p0.x, p0.y, bh0, bl0);
        split_bf16x2(p1.x, p1.y, bh1, bl1);
        float o[4] = {0.f, 0.f, 0.f, 0.f};
        ptx::mma_16816_bf16(o, xh, bh0, bh1);
        ptx::mma_16816_bf16(o, xh, bl0, bl1);
        ptx::mma_16816_bf16(o, xl, bh0, bh1);
        // o: T_{b+d,b}^T rows g, g + 8 and columns 8 nt + 2 t (+ 1)
        Tw[(8 * nt + 2 * t) * SLD + g] = -o[0];
        Tw[(8 * nt + 2 * t + 1) * SLD + g] = -o[1];
        Tw[(8 * nt + 2 * t) * SLD + g + 8] = -o[2];
        Tw[(8 * nt + 2 * t + 1) * SLD + g + 8] = -o[3];
      }
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// intra kernel (256 threads; warps w and w + 4 share TMEM lane quarter w % 4
// and split the columns of every accumulator row)
//
// shared memory (bytes):
//   KQ   [0, 32768)        k rows 0..63 / q rows 64..127 (x 128 keys) as TMA
//                          lands them: 128-byte swizzle, 64-key halves 16 KB
//                          apart (swz_off); at the end [-w ; q], the chain's A
//                          operand, in the same layout
//   VS   [32768, 49152)    v (64 tokens x V) as TMA lands it: 64-byte swizzle,
//                          32-column tiles 4 KB apart (the u GEMM's MN-major B)
//                          (KDA: first k e^-g, the B operand of S, 128-byte
//                          swizzle, halves 8 KB apart; v is loaded once S is
//                          done)
//   R1   [49152, 83968)    KDA gamma (fp32 64 x 128, swizzled: gidx); then A | T
//                          (fp32, 64 x 68 each); after the solve [Tw ; Tu] hi
//                          (128 x 64, 128-byte swizzled rows) over A; last, the
//                          fp32 u tile for the block store
//   AQ   [83968, 100352)   [Aqk_lo ; Aqk_hi] (128 x 64, 128-byte swizzled rows);
//                          once stored, [Tw ; Tu] lo
//   small                  scales, gamma, factors, merge scratch, barriers
// k, q and v land where the tensor cores read them, so there is no staging
// copy; the KDA gating pass rewrites k and q in place.  Both fit two CTAs per
// SM.
constexpr uint32_t I_KQ = 0, I_VS = 32768, I_R1 = 49152, I_AQ = 83968, I_SMALL = 100352;
constexpr int INTRA_THREADS = 256;

// KDA gate tile in R1: four TMA boxes of 32 channels x 64 rows (128-byte rows,
// 128-byte swizzle), so that a warp reading one channel group of 32
// consecutive rows, or one row of 32 channels, touches every bank once.
// Index (in floats) of token row i, channel c.
__device__ __forceinline__ int gidx(int i, int c) {
  return (c >> 5) * 2048 + i * 32 + ((((c >> 2) & 7) ^ (i & 7)) << 2) + (c & 3);
}

// K-major image with a 128-byte swizzle (the layout TMA writes with 128-byte
// rows): rows of 64 keys (128 bytes), the two 64-key halves `half` bytes
// apart; the 16-byte piece cg (keys 8 cg ..) of row r sits at piece
// (cg & 7) ^ (r & 7) of its row.  Offset of that piece:
__device__ __forceinline__ uint32_t swz_off(int r, int cg, uint32_t half) {
  return (uint32_t)(cg >> 3) * half + (uint32_t)r * 128u + ((uint32_t)((cg & 7) ^ (r & 7)) << 4);
}
// Offset of 16-byte piece j of row r of a one-half image (64 columns).
__device__ __forceinline__ uint32_t swz_row(int r, int j) {
  return (uint32_t)r * 128u + ((uint32_t)(j ^ (r & 7)) << 4);
}
// Descriptor of such an image as a K-major operand at key step ks (16 keys):
// 32 bytes into the row inside a half, 8-row groups 1 KB apart.
__device__ __forceinline__ uint64_t sw128_kmajor(const unsigned char *img, int ks, uint32_t half) {
  return ptx::sdesc(img + (ks >> 2) * half + (ks & 3) * 32, 16, 1024) | (2ull << 61);
}
template <bool KDA>
struct IntraLayout {
  static constexpr uint32_t SMALL = I_SMALL;
  static constexpr uint32_t SMEM = SMALL + 8192 + 1024;  // + up to 1 KB to align the base
};

template <bool KDA>
__global__ void __launch_bounds__(INTRA_THREADS, 2)
intra_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
             const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g,
             TcParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // the 128-byte swizzle of the KDA k / q tiles follows address bits 4-9
  unsigned char *smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
  unsigned char *KQ = smem + I_KQ;
  unsigned char *VS = smem + I_VS;
  float *Asm = reinterpret_cast<float *>(smem + I_R1);
  float *Tsm = Asm + 64 * SLD;
  unsigned char *TH = smem + I_R1;   // [Tw ; Tu] hi (after the solve, 128 x 64, swizzled rows)
  unsigned char *AQ = smem + I_AQ;   // Aqk pair, later [Tw ; Tu] lo
  unsigned char *KB = VS;  // KDA: k e^-g, until the S GEMM is done
  float *sc = reinterpret_cast<float *>(smem + IntraLayout<KDA>::SMALL);  // decay, rs, qs
  float *gam = sc + 256;                                   // [64]
  float *bet = gam + 64;                                   // [64]
  float *eg = bet + 64;                                    // [64] e^{gamma}
  float *eng = eg + 64;                                    // [64] e^{-gamma}
  float *gl = eng + 64;                                    // [128] KDA gamma_L
  uint64_t *bars = reinterpret_cast<uint64_t *>(gl + 128 + 3 * 16 * XLD + 4);  // tma, mma
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2);
  int *flags = reinterpret_cast<int *>(tmem_slot + 1);     // [0]: split exps ok

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qd = warp & 3, hf = warp >> 2;  // TMEM lane quarter, column half
  // KDA: one head per CTA.  Scalar gate: one key head per CTA, whose R value
  // heads share k, q and the S product; the CTA takes them in turn, loading
  // k and q once and each head's v while the previous head finishes.
  const int R = KDA ? 1 : p.H / p.Hk;
  const int hk = KDA ? blockIdx.y / (p.H / p.Hk) : blockIdx.y;
  int h = KDA ? blockIdx.y : blockIdx.y * R;
  ChunkPos cp;
  // packed sequences: launched as a programmatic dependent of the chunk-table
  // kernel, so the table is read once that kernel is done
  if (p.cu_seqlens) ptx::griddep_wait();
  if (!locate_chunk(p, blockIdx.x, cp)) return;
  const int V = p.V;
  const int s0 = cp.bos + cp.c * BT;
  const int L = min(BT, cp.eos - s0);
  const int row0 = cp.b * p.T + s0;  // token row in the [B*T] flattening
  if (!bounds_ok((int)blockIdx.x < p.nblk && h >= 0 && h + R <= p.H && hk < p.Hk && cp.b >= 0 &&
                     cp.b < p.B && s0 >= 0 && s0 < cp.eos && cp.eos <= p.T,
                 p.err))
    return;
  unsigned char *blk = p.blocks + ((size_t)blockIdx.x * p.H + h) * p.block;

  // Loads first: the gate inputs into registers (warp 3: g, warps 4-5: beta)
  // and the TMA of k, q, v, so their latency overlaps the set-up below.
  float ga0 = 0.f, ga1 = 0.f, gbe = 0.f;
  auto load_gates = [&](int hh) {
    if (!KDA && warp == 3) {
      ga0 = 2 * lane < L ? p.g[(size_t)(row0 + 2 * lane) * p.H + hh] : 0.f;
      ga1 = 2 * lane + 1 < L ? p.g[(size_t)(row0 + 2 * lane + 1) * p.H + hh] : 0.f;
    }
    if (warp == 4 || warp == 5) {
      const int i = tid - 128;
      gbe = i < L ? p.beta[(size_t)(row0 + i) * p.H + hh] : 0.f;
    }
  };
  load_gates(h);
  if (tid == 0) {
    ptx::mbar_init(&bars[0], 1);
    ptx::mbar_init(&bars[1], 1);
    ptx::fence_mbar_init();
    // KDA: k, q and the gate tile now, v after the S GEMM (second phase)
    ptx::mbar_arrive_expect_tx(&bars[0], KDA ? 65536u : 32768u + (uint32_t)V * 128);
    flags[0] = 1;
  }
  // three issuing threads, one per tensor, once warp 0 has set the barrier up
  if (warp < 3) asm volatile("bar.sync 1, 96;" ::: "memory");
  // k, q and v arrive in 128-byte (v: 64-byte) swizzled rows, few large
  // requests, straight into the operand images
  if (lane == 0 && warp == 0) {
    // k rows 0..63 of each 64-key half of KQ
    ptx::tma_load_3d(KQ, &tm_k, 0, hk, row0, &bars[0]);
    ptx::tma_load_3d(KQ + 16384, &tm_k, 64, hk, row0, &bars[0]);
  }
  if (lane == 0 && warp == 1) {
    // q rows 64..127
    ptx::tma_load_3d(KQ + 8192, &tm_q, 0, hk, row0, &bars[0]);
    ptx::tma_load_3d(KQ + 24576, &tm_q, 64, hk, row0, &bars[0]);
  }
  if (lane == 0 && warp == 2) {
    if (KDA) {
      // the fp32 gate tile (64 tokens x 128 channels) into R1, four boxes
#pragma unroll 1
      for (int j = 0; j < 4; ++j) ptx::tma_load_3d(Asm + j * 2048, &tm_g, 32 * j, h, row0, &bars[0]);
    } else {
#pragma unroll 1
      for (int j = 0; j < V / 32; ++j) ptx::tma_load_3d(VS + j * 4096, &tm_v, 32 * j, h, row0, &bars[0]);
    }
  }
  if (warp == 0) ptx::tmem_alloc<256>(tmem_slot);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  uint32_t mma_phase = 0;

#pragma unroll 1
  for (int r = 0;; ++r) {
  // ---- gates: gamma (chunk-local inclusive cumsum), beta, scales
  if (warp == 4 || warp == 5) bet[tid - 128] = gbe;
  if (!KDA) {
    if (warp == 3) {
      const float a0 = ga0, a1 = ga1;
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
    const float gL = gam[L - 1];
    if (tid < 64) {
      eg[tid] = __expf(gam[tid]);
      eng[tid] = __expf(-gam[tid]);
      sc[128 + tid] = tid < L ? __expf(gL - gam[tid]) : 0.f;  // rs: e^{gamma_L - gamma_i}
      sc[192 + tid] = p.scale * __expf(gam[tid]);              // qs: scale e^{gamma_i}
    } else if (tid < 192) {
      sc[tid - 64] = __expf(gL);                               // decay per key row
    }
  } else {
    if (tid >= KD && tid < KD + 64) {
      const int i = tid - KD;
      sc[128 + i] = i < L ? 1.f : 0.f;
      sc[192 + i] = p.scale;
    }
  }
  __syncthreads();

  const bool ok_tma = ptx::mbar_wait_bounded(&bars[0], (uint32_t)(r & 1));
  if (!__syncthreads_and(ok_tma)) {
    if (tid == 0) record_error(p.err, GDN_ERR_TIMEOUT);
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) ptx::tmem_dealloc<256>(tmem);
    return;
  }
  ptx::fence_proxy_async_smem();  // the images feed the tensor cores
  __syncthreads();
  if (!KDA && tid == 0) {
    // the q rows of [-w ; q] are the raw input: they leave now
    ptx::bulk_s2g(blk + OFF_AW + 8192, KQ + 8192, 8192);
    ptx::bulk_s2g(blk + OFF_AW + 24576, KQ + 24576, 8192);
    ptx::bulk_commit();
  }
  if (KDA) {
    // thread c < 128 owns key channel c: running cumsum down the TMA-loaded
    // gate tile in place (rows >= L repeat row L - 1)
    float *G = Asm;
    float mn = 0.f, mx = 0.f;
    if (p.g_is_cumsum) {
      // already the cumulative gate: thread (c, half) checks the range of 32
      // rows of channel c and repeats row L - 1 over the padding rows
      const int c = tid & (KD - 1), r0 = (tid >> 7) * 32;
      const float last = G[gidx(L - 1, c)];
#pragma unroll 8
      for (int i = r0; i < r0 + 32; ++i) {
        float x = last;
        if (i < L) x = G[gidx(i, c)]; else G[gidx(i, c)] = last;
        mn = fminf(mn, x);
        mx = fmaxf(mx, x);
      }
      if (tid < KD) {
        gl[c] = last;
        sc[c] = __expf(last);
      }
    } else if (tid < KD) {
      const int c = tid;
      float acc = 0.f;
#pragma unroll 8
      for (int i = 0; i < 64; ++i) {
        if (i < L) acc += G[gidx(i, c)];
        G[gidx(i, c)] = acc;
        mn = fminf(mn, acc);
        mx = fmaxf(mx, acc);
      }
      gl[c] = acc;
      sc[c] = __expf(acc);
    }
    const bool ok = mn >= -GATE_FACTOR_LIMIT && mx <= GATE_FACTOR_LIMIT;
    if (!__syncthreads_and(ok) && tid == 0) flags[0] = 0;
    __syncthreads();
  }
  const bool split = flags[0] != 0;

  // KDA, split range: the lo halves of the gated operands, for the S GEMM's
  // hi.lo and lo.hi passes (KQ_lo where the gate tile was, KB_lo in the AQ
  // staging area, both dead until the gating)
  unsigned char *KQL = smem + I_R1;
  unsigned char *KBL = AQ;
  if (KDA) {
    // KQ <- [k e^g ; q e^g] (bounded by |k|, |q| for gates <= 0),
    // KB <- k e^-g (split path only), KT <- k e^{gamma_L - g} (to the block);
    // each a hi + lo pair in the split path (the per-channel gate sits inside
    // the products, so its operands carry the rounding)
    const float *G = Asm;
    uint4 klo[4], qlo[4];
#pragma unroll
    for (int it = 0; it < 4; ++it) {
      const int pc = tid + it * INTRA_THREADS;
      const int i = pc & 63, cg = pc >> 6;
      // rewritten in place: each piece is read and written by its own thread
      uint4 *kp = reinterpret_cast<uint4 *>(KQ + swz_off(i, cg, 16384));
      uint4 *qp = reinterpret_cast<uint4 *>(KQ + swz_off(64 + i, cg, 16384));
      float kf[8], qf[8], a[8], b[8], c[8], t[8];
      unpack8(*kp, kf);
      unpack8(*qp, qf);
      const float4 ga = *reinterpret_cast<const float4 *>(G + gidx(i, 8 * cg));
      const float4 gb = *reinterpret_cast<const float4 *>(G + gidx(i, 8 * cg + 4));
      const float gr[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
      // (fp32 pairs: two products per instruction)
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        const float2 ep = make_float2(__expf(gr[e]), __expf(gr[e + 1]));
        const float2 kk = make_float2(kf[e], kf[e + 1]), qq = make_float2(qf[e], qf[e + 1]);
        const float2 ka = mul2(kk, ep), qb = mul2(qq, ep);
        a[e] = ka.x; a[e + 1] = ka.y;
        b[e] = qb.x; b[e + 1] = qb.y;
        // split range (|gamma| bounded): e^{gamma_L - g} = e^{gamma_L} e^{-g}
        const float2 en = split ? make_float2(__expf(-gr[e]), __expf(-gr[e + 1])) : make_float2(0.f, 0.f);
        const float2 kc = mul2(kk, en);
        c[e] = kc.x; c[e + 1] = kc.y;
        const float2 fl = split ? mul2(make_float2(sc[8 * cg + e], sc[8 * cg + e + 1]), en)
                                : make_float2(__expf(gl[8 * cg + e] - gr[e]),
                                              __expf(gl[8 * cg + e + 1] - gr[e + 1]));
        const float2 kt = mul2(kk, fl);
        t[e] = i < L ? kt.x : 0.f;
        t[e + 1] = i < L ? kt.y : 0.f;
      }
      uint4 hi, lo;
      split8(a, hi, klo[it]);
      *kp = hi;
      split8(b, hi, qlo[it]);
      *qp = hi;
      split8(c, hi, lo);
      *reinterpret_cast<uint4 *>(KB + swz_off(i, cg, 8192)) = hi;
      if (split) *reinterpret_cast<uint4 *>(KBL + swz_off(i, cg, 8192)) = lo;
      split8(t, hi, lo);
      *reinterpret_cast<uint4 *>(blk + OFF_KT + img_off(i, 8 * cg, 2048)) = hi;
      *reinterpret_cast<uint4 *>(blk + OFF_KT + img_off(64 + i, 8 * cg, 2048)) = lo;
    }
    if (split) {
      __syncthreads();  // every thread is done reading the gate tile
#pragma unroll
      for (int it = 0; it < 4; ++it) {
        const int pc = tid + it * INTRA_THREADS;
        const int i = pc & 63, cg = pc >> 6;
        *reinterpret_cast<uint4 *>(KQL + swz_off(i, cg, 16384)) = klo[it];
        *reinterpret_cast<uint4 *>(KQL + swz_off(64 + i, cg, 16384)) = qlo[it];
      }
    }
    ptx::fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      // the q rows of [-w ; q e^g] are final: they leave now
      ptx::bulk_s2g(blk + OFF_AW + 8192, KQ + 8192, 8192);
      ptx::bulk_s2g(blk + OFF_AW + 24576, KQ + 24576, 8192);
      ptx::bulk_commit();
    }
  } else {
    ptx::fence_proxy_async_smem();
  }

  // ---- S = [k; q] k^T  (M = 128, N = 64, K = 128); KDA split range: three
  //      passes hi.hi + hi.lo + lo.hi of the gated operands
  if (tid == 0) {
    ptx::tc_fence_after();
    const uint32_t id = ptx::idesc_bf16(128, 64, 0, 0);
    // (B: the k rows of KQ; KDA: KB, 64 rows a half)
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const uint64_t a = sw128_kmajor(KQ, ks, 16384);
      const uint64_t b = KDA ? sw128_kmajor(KB, ks, 8192) : a;
      ptx::mma_bf16(tmem, a, b, id, ks > 0);
    }
    if (KDA && split) {
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        ptx::mma_bf16(tmem, sw128_kmajor(KQ, ks, 16384), sw128_kmajor(KBL, ks, 8192), id, 1);
        ptx::mma_bf16(tmem, sw128_kmajor(KQL, ks, 16384), sw128_kmajor(KB, ks, 8192), id, 1);
      }
    }
    ptx::mma_commit(&bars[1]);
  }
  // (scalar gate: no KT -- the chain reads k raw and puts e^{gamma_L - gamma_i}
  // on v_new)
  const bool ok1 = ptx::mbar_wait_bounded(&bars[1], mma_phase);
  mma_phase ^= 1;
  ptx::tc_fence_after();
  if (KDA && tid == 0) {
    // S is done with KB: v into VS, counted on the second phase of bars[0]
    ptx::mbar_arrive_expect_tx(&bars[0], (uint32_t)V * 128);
    for (int j = 0; j < V / 32; ++j) ptx::tma_load_3d(VS + j * 4096, &tm_v, 32 * j, h, row0, &bars[0]);
  }

  // ---- gating: thread (qd, hf, lane) holds row r = 32 qd + lane of S,
  //      columns 32 hf .. 32 hf + 31 (r < 64: kk, r >= 64: qk)
  {
    const int r = qd * 32 + lane;
    const int i = r & 63;
    const bool is_q = r >= 64;
    const int j0 = hf * 32;
    float srow[32];
    ptx::tmem_ld32(tmem + ((uint32_t)(qd * 32) << 16) + j0, srow);
    if (KDA && !split) {
      // exact per-element exponentials (only when |gamma| leaves the split
      // range): raw k/q from global memory, gamma from R1
      const float *G = Asm;
      const __nv_bfloat16 *kg = static_cast<const __nv_bfloat16 *>(p.kraw);
      const __nv_bfloat16 *xg = static_cast<const __nv_bfloat16 *>(is_q ? p.qraw : p.kraw);
#pragma unroll
      for (int jj = 0; jj < 32; ++jj) {  // unrolled: srow stays in registers
        const int j = j0 + jj;
        float acc = 0.f;
        if (i < L && j <= i) {
          const size_t oi = ((size_t)(row0 + i) * p.Hk + hk) * KD;
          const size_t oj = ((size_t)(row0 + j) * p.Hk + hk) * KD;
          for (int c = 0; c < KD; ++c)
            acc = fmaf(__bfloat162float(xg[oi + c]) * __bfloat162float(kg[oj + c]),
                       __expf(G[gidx(i, c)] - G[gidx(j, c)]), acc);
        }
        srow[jj] = acc;
      }
      __syncthreads();  // everyone done reading gamma before A overwrites R1
    }
    if (!is_q) {
      // A (fp32, row stride SLD) for the solve: beta_i S_kk e^{g_i - g_j}, j < i < L
      const float bi = bet[i];
#pragma unroll
      for (int j4 = 0; j4 < 32; j4 += 4) {
        float a4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = j0 + j4 + e;
          float f = 1.f;
          if (!KDA) f = split ? eg[i] * eng[j] : __expf(gam[i] - gam[j]);
          a4[e] = (j < i && i < L) ? bi * f * srow[j4 + e] : 0.f;
        }
        *reinterpret_cast<float4 *>(Asm + i * SLD + j0 + j4) = make_float4(a4[0], a4[1], a4[2], a4[3]);
      }
    } else {
      // Aqk = scale S_qk e^{g_i - g_j} (j <= i < L) as a bf16 pair:
      // hi in rows 64.., lo in rows 0.. of the AQ image
#pragma unroll
      for (int cg = 0; cg < 4; ++cg) {
        float v8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int j = j0 + cg * 8 + e;
          float f = 1.f;
          if (!KDA) f = split ? eg[i] * eng[j] : __expf(gam[i] - gam[j]);
          v8[e] = (j <= i && i < L) ? p.scale * f * srow[cg * 8 + e] : 0.f;
        }
        uint4 hi, lo;
        split8(v8, hi, lo);
        *reinterpret_cast<uint4 *>(AQ + swz_row(64 + i, (j0 >> 3) + cg)) = hi;
        *reinterpret_cast<uint4 *>(AQ + swz_row(i, (j0 >> 3) + cg)) = lo;
      }
    }
  }
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before();
  __syncthreads();
  if (tid == 0) {
    ptx::bulk_s2g(blk + OFF_AQ, AQ, 16384);
    ptx::bulk_commit();
  }

  // ---- T = (I + A)^-1 (fp32)
  unit_lower_inverse_64<INTRA_THREADS>(Asm, Tsm, tid);
  if (tid == 0) ptx::bulk_wait_read<0>();
  __syncthreads();  // AQ and the k rows may be overwritten now

  // ---- Tw = T diag(beta e^g) (GDN) / T diag(beta) (KDA) in rows 0..63 and
  //      Tu = T diag(beta) in rows 64..127 of one 128 x 64 image per bf16 half
  //      (hi in TH, lo in the AQ region; 128-byte swizzled rows), so that one M = 128 GEMM per
  //      operand puts w and u in all four TMEM lane quarters
  for (int pc = tid; pc < 64 * 16; pc += INTRA_THREADS) {
    const int i = pc & 63, cg = pc >> 6;
    const bool is_u = cg >= 8;
    const int j0 = (cg & 7) * 8;
    float v8[8], t8[8];
    {
      const float4 x0 = *reinterpret_cast<const float4 *>(Tsm + i * SLD + j0);
      const float4 x1 = *reinterpret_cast<const float4 *>(Tsm + i * SLD + j0 + 4);
      t8[0] = x0.x; t8[1] = x0.y; t8[2] = x0.z; t8[3] = x0.w;
      t8[4] = x1.x; t8[5] = x1.y; t8[6] = x1.z; t8[7] = x1.w;
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int j = j0 + e;
      const float t = (j <= i) ? t8[e] : 0.f;
      const float d = (is_u || KDA) ? bet[j] : bet[j] * eg[j];
      v8[e] = t * d;
    }
    uint4 hi, lo;
    split8(v8, hi, lo);
    const int row = is_u ? 64 + i : i;
    *reinterpret_cast<uint4 *>(TH + swz_row(row, j0 >> 3)) = hi;
    *reinterpret_cast<uint4 *>(AQ + swz_row(row, j0 >> 3)) = lo;
  }
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before();
  __syncthreads();

  // ---- [Tw ; Tu] k (N = 128 keys) and [Tw ; Tu] v (N = V), M = 128, K = 64
  //      tokens, hi + lo passes accumulating in TMEM: w = rows 0..63 of the
  //      first, u = rows 64..127 of the second (the other halves are unused)
  const uint32_t dW = tmem, dU = tmem + 128;
  bool ok_v = true;
  if (tid == 0) {
    if (KDA) ok_v = ptx::mbar_wait_bounded(&bars[0], 1);  // v has landed
    ptx::tc_fence_after();
    const uint32_t idw = ptx::idesc_bf16(128, 128, 0, 1);
    const uint32_t idu = ptx::idesc_bf16(128, V, 0, 1);
#pragma unroll
    for (int part = 0; part < 2; ++part) {
      unsigned char *img = part ? AQ : TH;
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        const uint64_t a = sw128_kmajor(img, ks, 0);  // K = 64 tokens: one half
        // k rows of KQ, MN-major: 64-key halves 16 KB apart, 8-token groups 1 KB
        const uint64_t b = ptx::sdesc(KQ + ks * 2048, 16384, 1024) | (2ull << 61);
        ptx::mma_bf16(dW, a, b, idw, part > 0 || ks > 0);
        // v, MN-major with a 64-byte swizzle: 32-column tiles 4 KB apart,
        // 8-token groups 512 bytes
        const uint64_t bv = ptx::sdesc(VS + ks * 1024, 4096, 512) | (4ull << 61);
        ptx::mma_bf16(dU, a, bv, idu, part > 0 || ks > 0);
      }
    }
    ptx::mma_commit(&bars[1]);
    ptx::bulk_s2g(blk + OFF_SC, sc, 1024);
    ptx::bulk_commit();
  }
  const bool ok2 = ptx::mbar_wait_bounded(&bars[1], mma_phase);
  mma_phase ^= 1;
  ptx::tc_fence_after();
  if (r + 1 < R) {
    // the next value head: its v into VS (the WY GEMM is done with it) and its
    // gate inputs into registers, landing while this head finishes
    if (tid == 0) {
      ptx::mbar_arrive_expect_tx(&bars[0], (uint32_t)V * 128);
#pragma unroll 1
      for (int j = 0; j < V / 32; ++j)
        ptx::tma_load_3d(VS + j * 4096, &tm_v, 32 * j, h + 1, row0, &bars[0]);
    }
    load_gates(h + 1);
  }
  const bool last = r + 1 == R;
  // -w replaces k in KQ, which is then the chain's A operand [-w ; q]; while
  // another value head follows, k stays and -w goes to the AQ region (the WY
  // GEMM is done with it) with the key halves 8 KB apart
  unsigned char *wimg = last ? KQ : AQ;
  const uint32_t whalf = last ? 16384u : 8192u;
  {
    // M = 128 layout: row r lives in TMEM lane r.  Lane quarters 0-1 hold the
    // w rows (keys split between the two warps of a quarter), quarters 2-3
    // the u rows (value tiles split likewise).
    const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
    if (qd < 2) {
      const int i = qd * 32 + lane;
#pragma unroll 1
      for (int q4 = 2 * hf; q4 < 2 * hf + 2; ++q4) {
        float v[32];
        ptx::tmem_ld32(dW + lane_base + q4 * 32, v);
#pragma unroll
        for (int q8 = 0; q8 < 4; ++q8) {
          float out[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) out[e] = -v[q8 * 8 + e];
          *reinterpret_cast<uint4 *>(wimg + swz_off(i, q4 * 4 + q8, whalf)) = pack8(out);
        }
      }
      // this warp's 32 rows of key half hf (4 KB) leave at once
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        ptx::bulk_s2g(blk + OFF_AW + hf * 16384 + qd * 4096, wimg + hf * whalf + qd * 4096, 4096);
        ptx::bulk_commit();
        ptx::bulk_wait_read<0>();
      }
      __syncwarp();
    } else {
      const int i = (qd - 2) * 32 + lane;
#pragma unroll 1
      for (int t = hf; t < V / 32; t += 2) {
        float v[32];
        ptx::tmem_ld32(dU + lane_base + t * 32, v);
        // 16-byte group q of row i sits at group q ^ (i & 7), so that the
        // chain's per-row loads (one row per lane) hit eight different groups
        // in every quarter warp: no shared-memory bank conflicts.  The tile is
        // staged in R1 (free once the WY GEMM is done) in the block's layout.
        float4 *dst = reinterpret_cast<float4 *>(smem + I_R1 + t * 8192 + i * 128);
#pragma unroll
        for (int q = 0; q < 8; ++q)
          dst[q ^ (i & 7)] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        // this warp's 32 rows of the tile (4 KB) leave at once, while the
        // other warps still form -w
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          const uint32_t off = t * 8192 + (qd - 2) * 32 * 128;
          ptx::bulk_s2g(blk + OFF_U + off, smem + I_R1 + off, 4096);
          ptx::bulk_commit();
        }
      }
      // the tile's rows must be read out before the buffers are reused
      if (lane == 0) ptx::bulk_wait_read<0>();
      __syncwarp();
    }
  }
  // Every part of the block has left in pieces as soon as it was final (the
  // q rows of [-w ; q] once the inputs landed or the gating pass ended, each
  // warp's -w and u rows from the epilogue).  After the last head the tensor
  // memory is no longer read: free it before the last wait, so that the next
  // CTA on this SM can allocate it while this one drains.
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before();
  __syncthreads();
  if (last && warp == 0) ptx::tmem_dealloc<256>(tmem);
  if (tid == 0) ptx::bulk_wait_read<0>();  // shared memory read out; the writes land on their own
  if (!(ok1 && ok2 && ok_v) && tid == 0) record_error(p.err, GDN_ERR_TIMEOUT);
  if (last) break;
  // next value head: the stores above have read AQ, R1 and the scales
  ++h;
  blk = p.blocks + ((size_t)blockIdx.x * p.H + h) * p.block;
  if (tid == 0) flags[0] = 1;
  __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// chain kernel (576 threads: warps 0-15 epilogue, warp 16 producer, warp 17 MMA)
//
// shared memory: two stages holding one operand block each
//   AW  [0, 32768)       [-w ; q~] (128 x 128, 128-byte swizzle, halves 16 KB apart)
//   KT  [32768, 65536)   [k~_hi ; k~_lo] (128 token rows x 128 keys, cs 2048);
//                        scalar gate: raw k of the chunk by TMA, two 8 KB halves
//                        of 64 keys x 64 token rows (128-byte swizzle)
//   AQ  [65536, 81920)   [Aqk_lo ; Aqk_hi] (128 x 64, 128-byte swizzled rows)
//   SC  [81920, 82944)   decay[128], rs[64], qs[64]
//   U   [82944, 91136)   u tile, fp32 64 x 32 (row-swizzled 16-byte groups)
// then H = [h_hi | h_lo] (128 keys x 64), VN = [vn_hi | vn_lo]
// (64 tokens x 64; both in 128-byte swizzled rows; scalar gate: e^{gamma_L - gamma_i} v_new, the
// state update's operand, with v_new itself for the output GEMM in VN2) and
// the fp32 exchange X.  A stage is filled and
// released in two halves: AW, SC and U are free once D1 has run and v_new is
// formed, KT and AQ only after the output GEMM, so the first half of the next
// block but one streams in half a step earlier.
// Every bf16 pair rides in the N dimension of one GEMM (N = 64), so the
// split costs no extra tcgen05 instructions; each accumulator holds the two
// halves side by side and the epilogue adds them.
constexpr uint32_t S_AW = 0, S_KT = 32768, S_AQ = 65536, S_SC = 81920, S_U = 82944,
                   STAGE_BYTES = 91136;
constexpr uint32_t C_H = 2 * STAGE_BYTES, C_VN = C_H + 16384, C_VN2 = C_VN + 8192,
                   C_X = C_VN2 + 8192, C_BAR = C_X + 64 * 33 * 4,
                   C_SMEM = C_BAR + 256 + 1024;  // + up to 1 KB to align the base
constexpr int EPI_WARPS = 16;               // four per TMEM lane quarter
constexpr int EC = 32 / (EPI_WARPS / 4);    // state columns per epilogue thread (8)
constexpr int CHAIN_THREADS = 32 * (EPI_WARPS + 2);
// Named barriers of the chain kernel (1 is the epilogue warps' own).  The
// epilogue warps arrive (without waiting) once h, or v_new, is in shared
// memory; the MMA warp waits on them.  Each phase's arrivals depend on MMAs
// the MMA warp issues only after it passed the previous phase, so phases
// never overlap; every role runs every chunk, so every phase completes.
constexpr int BAR_HREADY = 2, BAR_HREADY_THREADS = 32 * (EPI_WARPS + 1);
// v_new comes from the epilogue warps of lane quarters 0-1 (rows 0..63), half of them
constexpr int BAR_VNREADY = 3, BAR_VNREADY_THREADS = 32 * (EPI_WARPS / 2 + 1);
constexpr int BAR_VN2READY = 4;  // (scalar gate) v_new for the output GEMM, same threads

__device__ __forceinline__ void bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}
__device__ __forceinline__ void bar_arrive(int id, int threads) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// start-address field of a shared-memory descriptor advanced by `bytes`
__device__ __forceinline__ uint64_t adv(uint64_t desc, uint32_t bytes) {
  return desc + (uint64_t)(bytes >> 4);
}

// columns [c0, c0 + 8) of a 64-column accumulator holding the hi product in
// columns 0..31 and the lo product in 32..63, summed; both loads are in flight
// before the one wait, which takes the registers so that nothing reads them
// earlier
__device__ __forceinline__ void tmem_ld_pair8(uint32_t taddr, int c0, float *v) {
  uint32_t h[8], l[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3]), "=r"(h[4]), "=r"(h[5]),
                 "=r"(h[6]), "=r"(h[7])
               : "r"(taddr + c0)
               : "memory");
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(l[0]), "=r"(l[1]), "=r"(l[2]), "=r"(l[3]), "=r"(l[4]), "=r"(l[5]),
                 "=r"(l[6]), "=r"(l[7])
               : "r"(taddr + 32 + c0)
               : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(h[0]), "+r"(h[1]), "+r"(h[2]), "+r"(h[3]), "+r"(h[4]), "+r"(h[5]),
                 "+r"(h[6]), "+r"(h[7]), "+r"(l[0]), "+r"(l[1]), "+r"(l[2]), "+r"(l[3]),
                 "+r"(l[4]), "+r"(l[5]), "+r"(l[6]), "+r"(l[7])
               :
               : "memory");
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] = __uint_as_float(h[j]) + __uint_as_float(l[j]);
}

// 8 values -> hi/lo bf16 halves of row r of a 64-column image with 128-byte
// rows in the 128-byte swizzle (hi in columns c0 .. c0 + 7, lo in columns
// 32 + c0 ..; 16-byte piece j of row r at piece j ^ (r & 7))
__device__ __forceinline__ void store_pair8(unsigned char *img, int r, int c0, const float *v) {
  uint4 hi, lo;
  split8(v, hi, lo);
  const int jh = c0 >> 3, jl = 4 + (c0 >> 3);
  *reinterpret_cast<uint4 *>(img + r * 128 + ((jh ^ (r & 7)) << 4)) = hi;
  *reinterpret_cast<uint4 *>(img + r * 128 + ((jl ^ (r & 7)) << 4)) = lo;
}

__device__ __forceinline__ void tma_load_4d(void *dst, const void *tmap, int c0, int c1, int c2,
                                            int c3, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(ptx::smem_u32(dst)),
      "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(ptx::smem_u32(bar))
      : "memory");
}

// RAWK (scalar gate): the state update reads k raw (tm_k: 4-D map of k as
// (64 keys, rows, 2 halves, key heads), 128-byte swizzle) and the token
// factors ride on v_new; otherwise (per-channel gate) it reads KT.
template <bool RAWK>
__global__ void __launch_bounds__(CHAIN_THREADS, 1)
chain_kernel(const __grid_constant__ CUtensorMap tm_k, TcParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // the 128-byte swizzle follows address bits 4-9: the stages start on 1 KB
  unsigned char *smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
  unsigned char *Himg = smem + C_H;
  unsigned char *VN = smem + C_VN;
  unsigned char *VN2 = RAWK ? smem + C_VN2 : VN;
  float *X = reinterpret_cast<float *>(smem + C_X);
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + C_BAR);
  // each stage has two halves with their own barriers: A = AW, SC, U (read
  // by D1 and the v_new epilogue), B = KT, AQ (read by DH and D5), so that A
  // is refilled as soon as v_new is formed, half a step before B
  uint64_t *fullA = bar, *emptyA = bar + 2, *fullB = bar + 4, *emptyB = bar + 6;
  uint64_t *d1 = bar + 8, *d3 = bar + 9, *d5 = bar + 10;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar + 11);
  volatile int *abort_flag = reinterpret_cast<int *>(bar + 12);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // The CTA's chain.  Phase 0: value tile blockIdx.x of sequence blockIdx.z,
  // all its chunks.  Segment-parallel pass (every sequence cut into
  // seg_count segments of equal chunk counts): phase 1 runs every segment
  // at once, grid x over K / 32 transition tiles then V / 32 value tiles --
  // a transition tile starts from 32 columns of the identity with u = 0, so
  // it ends on those columns of the segment's linear map M_s; a value tile
  // starts from zero (segment 0: from h0, writing o), ending on B_s -- both
  // stored to seg_state; phase 2 reruns segments 1.. from the start states
  // the combine kernel formed (start_{s+1} = M_s start_s + B_s), writing o
  // and, for the last segment, ht.
  constexpr int KTILES = KD / VTILE;
  int zz = blockIdx.z, seg = 0;
  if (p.seg_phase == 1) {
    seg = zz % p.seg_count;
    zz /= p.seg_count;
  } else if (p.seg_phase == 2) {
    seg = zz % (p.seg_count - 1) + 1;
    zz /= p.seg_count - 1;
  }
  bool trans = false;  // transition tile (phase 1)
  int vt = blockIdx.x;
  if (p.seg_phase == 1) {
    if (vt < KTILES) {
      if (seg == 0) return;  // segment 0 starts from h0: no map needed
      trans = true;
    } else {
      vt -= KTILES;
    }
  }
  const int v0 = vt * VTILE;
  const int h = blockIdx.y;
  const int n = p.cu_seqlens ? p.table[p.N + 1 + zz] : zz;
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
  int cfirst = 0, nch = (eos - bos + BT - 1) / BT;
  if (p.seg_phase != 0) {
    const int per = (nch + p.seg_count - 1) / p.seg_count;
    cfirst = min(seg * per, nch);
    nch = min(per, nch - cfirst);
  }
  const bool write_o = p.seg_phase != 1 || seg == 0;
  if (!bounds_ok(n >= 0 && n < p.N && b >= 0 && b < p.B && bos >= 0 && bos <= eos && eos <= p.T &&
                     base >= 0 && base + cfirst + nch <= p.nblk && h < p.H &&
                     v0 + VTILE <= (trans ? KD : p.V) && (p.seg_phase == 0 || seg < p.seg_count),
                 p.err))
    return;

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&fullA[i], 1);
      ptx::mbar_init(&emptyA[i], 1 + EPI_WARPS);
      ptx::mbar_init(&fullB[i], 1);
      ptx::mbar_init(&emptyB[i], 1);
    }
    ptx::mbar_init(d1, 1);
    ptx::mbar_init(d3, 1);
    ptx::mbar_init(d5, 1);
    ptx::fence_mbar_init();
    *abort_flag = 0;
  }
  if (warp == 0) ptx::tmem_alloc<256>(tmem_slot);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t dD1 = tmem, dDH = tmem + 64, dD5 = tmem + 128;
  // launched as a programmatic dependent of the intra kernel: the operand
  // blocks are read only once it has completed and its writes are visible
  ptx::griddep_wait();

  if (warp == EPI_WARPS) {
    // ---------------- producer: one operand block per chunk, in two halves.
    // Half A of chunk c + 1 is released (v_new of chunk c - 1) before half B
    // of chunk c (output GEMM of chunk c - 2), so waiting in the order
    // A(c), B(c), A(c + 1), ... never holds a release back.
    // Each copy has its own lane: the copies one thread issues complete one
    // after another, those of different threads overlap.
    if (lane == 0 && RAWK) ptx::prefetch_tmap(&tm_k);
    const int hk = h / (p.H / p.Hk);
    // a transition tile's u is zero: its U tile is not loaded
    const uint32_t A_BYTES = 32768 + 1024 + (trans ? 0 : 8192), B_BYTES = RAWK ? 32768 : 49152;
#pragma unroll 1
    for (int c = 0; c < nch; ++c) {
      const int s = c & 1, k = c >> 1;
      unsigned char *st = smem + s * STAGE_BYTES;
      const unsigned char *src = p.blocks + ((size_t)(base + cfirst + c) * p.H + h) * p.block;
      if (k > 0 && !ptx::mbar_wait_bounded(&emptyA[s], (uint32_t)((k - 1) & 1)) && lane == 0) {
        record_error(p.err, GDN_ERR_TIMEOUT);  // keep going: no role may stall the others
        *abort_flag = 1;
      }
      if (lane == 0) ptx::mbar_arrive_expect_tx(&fullA[s], A_BYTES);
      __syncwarp();
      if (lane == 0) ptx::bulk_g2s(st + S_AW, src + OFF_AW, 32768, &fullA[s]);
      if (lane == 1) ptx::bulk_g2s(st + S_SC, src + OFF_SC, 1024, &fullA[s]);
      if (lane == 2 && !trans) ptx::bulk_g2s(st + S_U, src + OFF_U + vt * 8192, 8192, &fullA[s]);
      if (k > 0 && !ptx::mbar_wait_bounded(&emptyB[s], (uint32_t)((k - 1) & 1)) && lane == 0) {
        record_error(p.err, GDN_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      if (lane == 0) ptx::mbar_arrive_expect_tx(&fullB[s], B_BYTES);
      __syncwarp();
      if (RAWK) {
        // k rows of the chunk (rows past the tensor read as zero; rows past
        // the sequence meet zero factors on v_new)
        if (lane == 3)
          tma_load_4d(st + S_KT, &tm_k, 0, b * p.T + bos + (cfirst + c) * BT, 0, hk, &fullB[s]);
        if (lane == 4) ptx::bulk_g2s(st + S_AQ, src + OFF_AQ, 16384, &fullB[s]);
      } else {
        if (lane == 3) ptx::bulk_g2s(st + S_KT, src + OFF_KT, 32768, &fullB[s]);
        if (lane == 4) ptx::bulk_g2s(st + S_AQ, src + OFF_AQ, 16384, &fullB[s]);
      }
    }
  } else if (warp == EPI_WARPS + 1) {
    // ---------------- MMA issuer (lane 0 issues; the whole warp takes part in
    // the named barriers that hand over h and v_new)
    const uint32_t id_kmn = ptx::idesc_bf16(128, 2 * VTILE, 0, 1);   // A K-major, B MN-major
    const uint32_t id_mnmn = ptx::idesc_bf16(128, 2 * VTILE, 1, 1);  // both MN-major
    // H (128 key rows) and VN / VN2 (64 token rows) as MN-major B operands:
    // 64 columns of 128-byte swizzled rows, 8-row groups 1 KB apart
    const uint64_t dH0 = ptx::sdesc(Himg, 16384, 1024) | (2ull << 61);
    const uint64_t dVN0 = ptx::sdesc(VN, 8192, 1024) | (2ull << 61);
    bool ok = true;
#pragma unroll 1
    for (int c = 0; c < nch; ++c) {
      const int s = c & 1, k = c >> 1;
      unsigned char *st = smem + s * STAGE_BYTES;
      const uint64_t kt = ptx::sdesc(st + S_KT, 128, 2048);
      ok = ptx::mbar_wait_bounded(&fullA[s], (uint32_t)(k & 1)) && ok;
      __syncwarp();
      bar_sync(BAR_HREADY, BAR_HREADY_THREADS);  // h of this chunk is in H
      ptx::tc_fence_after();
      if (lane == 0) {
        // D1 = [-w ; q~] [h_hi | h_lo] (AW K-major, 128-byte swizzle: swz_off)
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          ptx::mma_bf16(dD1, sw128_kmajor(st + S_AW, ks, 16384), adv(dH0, ks * 2048), id_kmn, ks > 0);
        ptx::mma_commit(d1);
        ptx::mma_commit(&emptyA[s]);  // D1 no longer reads AW
      }
      ok = ptx::mbar_wait_bounded(&fullB[s], (uint32_t)(k & 1)) && ok;
      __syncwarp();
      bar_sync(BAR_VNREADY, BAR_VNREADY_THREADS);  // v_new is in VN
      ptx::tc_fence_after();
      if (lane == 0) {
        if (RAWK) {
          // DH = k^T [v~_hi | v~_lo] (K = 64 tokens; k MN-major, 128-byte
          // swizzle: 64-key halves 8 KB apart, 8-token groups 1 KB apart)
          const uint64_t kr = ptx::sdesc(st + S_KT, 8192, 1024) | (2ull << 61);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            ptx::mma_bf16(dDH, adv(kr, ks * 2048), adv(dVN0, ks * 2048), id_mnmn, ks > 0);
        } else {
          // DH = [k~_hi ; k~_lo]^T [vn_hi | vn_lo ; vn_hi | vn_lo] (K = 128:
          // the token rows once with each half of k~; critical path)
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            ptx::mma_bf16(dDH, adv(kt, ks * 256), adv(dVN0, (ks & 3) * 2048), id_mnmn, ks > 0);
        }
        ptx::mma_commit(d3);
      }
      if (RAWK) {
        __syncwarp();
        bar_sync(BAR_VN2READY, BAR_VNREADY_THREADS);  // v_new itself is in VN2
        ptx::tc_fence_after();
      }
      if (lane == 0) {
        // D5 = AQ [vn_hi | vn_lo]
        const uint64_t dVN2 = ptx::sdesc(VN2, 8192, 1024) | (2ull << 61);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          ptx::mma_bf16(dD5, sw128_kmajor(st + S_AQ, ks, 0), adv(dVN2, ks * 2048), id_kmn, ks > 0);
        ptx::mma_commit(d5);
        ptx::mma_commit(&emptyB[s]);
      }
      __syncwarp();
    }
    if (!ok && lane == 0) {
      record_error(p.err, GDN_ERR_TIMEOUT);
      *abort_flag = 1;
    }
  } else {
    // ---------------- epilogue warps: row r = TMEM lane, columns c0 .. c0 + EC - 1
    const int qd = warp & 3;
    const int c0 = (warp >> 2) * EC;
    const int r = qd * 32 + lane;
    const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
    float hs[EC];
    const bool from_h0 = p.seg_phase == 0 || (p.seg_phase == 1 && seg == 0);
    if (trans) {
      // columns v0 + c0 .. of the identity (key index = column)
#pragma unroll
      for (int j = 0; j < EC; ++j) hs[j] = (r == v0 + c0 + j) ? 1.f : 0.f;
    } else if (p.seg_phase == 2) {
      const float4 *src = reinterpret_cast<const float4 *>(
          p.seg_start + ((((size_t)n * p.seg_count + seg) * p.H + h) * KD + r) * p.V + v0 + c0);
#pragma unroll
      for (int q = 0; q < EC / 4; ++q) {
        const float4 x = src[q];
        hs[4 * q] = x.x; hs[4 * q + 1] = x.y; hs[4 * q + 2] = x.z; hs[4 * q + 3] = x.w;
      }
    } else if (!from_h0) {
#pragma unroll
      for (int j = 0; j < EC; ++j) hs[j] = 0.f;
    } else if (p.h0 && p.v_first) {
      // [V, K]: the lanes of a warp read 32 consecutive keys of one value row
      const float *src = p.h0 + ((size_t)n * p.H + h) * KD * p.V + (size_t)(v0 + c0) * KD + r;
#pragma unroll
      for (int j = 0; j < EC; ++j) hs[j] = src[(size_t)j * KD];
    } else if (p.h0) {
      const float4 *src = reinterpret_cast<const float4 *>(
          p.h0 + (((size_t)n * p.H + h) * KD + r) * p.V + v0 + c0);
#pragma unroll
      for (int q = 0; q < EC / 4; ++q) {
        const float4 x = src[q];
        hs[4 * q] = x.x; hs[4 * q + 1] = x.y; hs[4 * q + 2] = x.z; hs[4 * q + 3] = x.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < EC; ++j) hs[j] = 0.f;
    }
    store_pair8(Himg, r, c0, hs);
    ptx::fence_proxy_async_smem();
    __syncwarp();
    bar_arrive(BAR_HREADY, BAR_HREADY_THREADS);

    bool ok = true;
#pragma unroll 1
    for (int c = 0; c < nch; ++c) {
      const int s = c & 1, k = c >> 1;
      const unsigned char *st = smem + s * STAGE_BYTES;
      const int L = min(BT, eos - bos - (cfirst + c) * BT);
      ok = ptx::mbar_wait_bounded(&fullA[s], (uint32_t)(k & 1)) && ok;
      const float *scs = reinterpret_cast<const float *>(st + S_SC);
      const float decay = scs[r];
      const float qs = r >= 64 ? scs[192 + r - 64] : 0.f;
      ok = ptx::mbar_wait_bounded(d1, (uint32_t)(c & 1)) && ok;
      ptx::tc_fence_after();
      float qh[EC];
      {
        float d[EC];
        tmem_ld_pair8(dD1 + lane_base, c0, d);
        if (r < 64) {
          const float4 *u4 = reinterpret_cast<const float4 *>(st + S_U + r * 128);
          float vn[EC];
#pragma unroll
          for (int q = 0; q < EC / 4; ++q) {
            const float4 u = trans ? make_float4(0.f, 0.f, 0.f, 0.f)
                                   : u4[((c0 >> 2) + q) ^ (r & 7)];  // row-swizzled groups
            vn[4 * q] = u.x + d[4 * q];
            vn[4 * q + 1] = u.y + d[4 * q + 1];
            vn[4 * q + 2] = u.z + d[4 * q + 2];
            vn[4 * q + 3] = u.w + d[4 * q + 3];
          }
          if (RAWK) {
            // the state update's operand: e^{gamma_L - gamma_r} v_new (zero
            // on padding rows), then v_new itself for the output GEMM
            const float f = scs[128 + r];
            float vt[EC];
#pragma unroll
            for (int j = 0; j < EC; ++j) vt[j] = f * vn[j];
            store_pair8(VN, r, c0, vt);
          } else {
            store_pair8(VN, r, c0, vn);
          }
          ptx::fence_proxy_async_smem();
          ptx::tc_fence_before();
          __syncwarp();
          bar_arrive(BAR_VNREADY, BAR_VNREADY_THREADS);
          if (RAWK) {
            store_pair8(VN2, r, c0, vn);
            ptx::fence_proxy_async_smem();
            __syncwarp();
            bar_arrive(BAR_VN2READY, BAR_VNREADY_THREADS);
          }
        } else {
#pragma unroll
          for (int j = 0; j < EC; ++j) qh[j] = d[j];
        }
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&emptyA[s]);  // this warp no longer reads SC, U
      ok = ptx::mbar_wait_bounded(d3, (uint32_t)(c & 1)) && ok;
      ptx::tc_fence_after();
      {
        float d[EC];
        tmem_ld_pair8(dDH + lane_base, c0, d);
#pragma unroll
        for (int j = 0; j < EC; ++j) hs[j] = fmaf(decay, hs[j], d[j]);
        store_pair8(Himg, r, c0, hs);
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        __syncwarp();
        bar_arrive(BAR_HREADY, BAR_HREADY_THREADS);
      }
      ok = ptx::mbar_wait_bounded(d5, (uint32_t)(c & 1)) && ok;
      ptx::tc_fence_after();
      float d5v[EC];
      tmem_ld_pair8(dD5 + lane_base, c0, d5v);
      ptx::tc_fence_before();
      if (r < 64) {
#pragma unroll
        for (int j = 0; j < EC; ++j) X[r * 33 + c0 + j] = d5v[j];
      }
      asm volatile("bar.sync 1, %0;" ::"n"(32 * EPI_WARPS) : "memory");
      if (r >= 64 && write_o) {
        const int i = r - 64;
        if (i < L) {
          float ov[EC];
#pragma unroll
          for (int j = 0; j < EC; ++j) ov[j] = fmaf(qs, qh[j], d5v[j] + X[i * 33 + c0 + j]);
          const size_t oi =
              ((size_t)(b * p.T + bos + (cfirst + c) * BT + i) * p.H + h) * p.V + v0 + c0;
          if (p.o_f32) {
            float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.o) + oi);
#pragma unroll
            for (int q = 0; q < EC / 4; ++q)
              dst[q] = make_float4(ov[4 * q], ov[4 * q + 1], ov[4 * q + 2], ov[4 * q + 3]);
          } else {
            uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.o) + oi);
#pragma unroll
            for (int q = 0; q < EC / 8; ++q) dst[q] = pack8(ov + 8 * q);
          }
        }
      }
      asm volatile("bar.sync 1, %0;" ::"n"(32 * EPI_WARPS) : "memory");
    }
    if (!ok) {
      if (lane == 0) record_error(p.err, GDN_ERR_TIMEOUT);
    } else if (p.seg_phase == 1 && *abort_flag == 0) {
      // row r of [M_s | B_s]: transition tiles fill columns 0 .. K - 1,
      // value tiles columns K + v0 ..
      const int W = KD + p.V, col = (trans ? v0 : KD + v0) + c0;
      float4 *dst = reinterpret_cast<float4 *>(
          p.seg_state + ((((size_t)n * p.seg_count + seg) * p.H + h) * KD + r) * W + col);
#pragma unroll
      for (int q = 0; q < EC / 4; ++q)
        dst[q] = make_float4(hs[4 * q], hs[4 * q + 1], hs[4 * q + 2], hs[4 * q + 3]);
    } else if (p.seg_phase == 2 && seg != p.seg_count - 1) {
      // an inner segment's end is the next one's start: already formed
    } else if (p.ht && *abort_flag == 0 && p.v_first) {
      float *dst = p.ht + ((size_t)n * p.H + h) * KD * p.V + (size_t)(v0 + c0) * KD + r;
#pragma unroll
      for (int j = 0; j < EC; ++j) dst[(size_t)j * KD] = hs[j];
    } else if (p.ht && *abort_flag == 0) {
      float4 *dst = reinterpret_cast<float4 *>(p.ht + (((size_t)n * p.H + h) * KD + r) * p.V + v0 + c0);
#pragma unroll
      for (int q = 0; q < EC / 4; ++q)
        dst[q] = make_float4(hs[4 * q], hs[4 * q + 1], hs[4 * q + 2], hs[4 * q + 3]);
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) ptx::tmem_dealloc<256>(tmem);
}

// ---------------------------------------------------------------------------
// Segment combine (between the two phases of the segment-parallel pass): the
// affine map of segment s takes its start state to M_s start + B_s, so
//   start_1 = B_0 (segment 0's end, run from h0),
//   start_{s+1} = M_s start_s + B_s          for s = 1 .. seg_count - 2,
// in fp32 on the CUDA cores.  Every M_s and B_s is known when the kernel
// starts, so only the running state is sequential: one CTA per (8-column
// value tile, head, sequence), thread t holding row t / 2, columns
// 4 (t % 2) .. + 3 of it; M_{s+1} streams into the other of two shared-memory
// buffers (cp.async) while step s computes.
constexpr int COMB_THREADS = 256, COMB_COLS = 8, COMB_LDM = KD + 4;
constexpr uint32_t COMB_SMEM = (2 * KD * COMB_LDM + KD * COMB_COLS) * 4;
__global__ void __launch_bounds__(COMB_THREADS) segment_combine_kernel(TcParams p) {
  extern __shared__ __align__(16) float csm[];
  ptx::griddep_wait();  // a programmatic dependent of the phase-1 chain grid
  float *X = csm + 2 * KD * COMB_LDM;  // the running state's tile, [KD][COMB_COLS]
  const int h = blockIdx.y, n = blockIdx.z;
  const int S = p.seg_count, W = KD + p.V, tid = threadIdx.x;
  if (!bounds_ok(n < p.N && h < p.H && (int)(blockIdx.x + 1) * COMB_COLS <= p.V, p.err)) return;
  const int r = tid >> 1, cq = (tid & 1) * 4, col = blockIdx.x * COMB_COLS + cq;
  auto state = [&](int sg) {
    return p.seg_state + (((size_t)n * S + sg) * p.H + h) * KD * W;
  };
  auto stage_m = [&](int sg) {  // M_sg into buffer sg & 1
    const float *Ms = state(sg);
    float *dst = csm + (sg & 1) * KD * COMB_LDM;
    for (int idx = tid; idx < KD * KD / 4; idx += COMB_THREADS) {
      const int rr = idx >> 5, c4 = idx & 31;
      ptx::cp_async16(dst + rr * COMB_LDM + 4 * c4, Ms + (size_t)rr * W + 4 * c4, true);
    }
    ptx::cp_async_commit();
  };
  float4 acc = *reinterpret_cast<const float4 *>(state(0) + (size_t)r * W + KD + col);
  float4 bnext = make_float4(0.f, 0.f, 0.f, 0.f);
  if (S > 2) {
    stage_m(1);
    bnext = *reinterpret_cast<const float4 *>(state(1) + (size_t)r * W + KD + col);
  }
#pragma unroll 1
  for (int sg = 1; sg < S; ++sg) {
    *reinterpret_cast<float4 *>(
        p.seg_start + ((((size_t)n * S + sg) * p.H + h) * KD + r) * p.V + col) = acc;
    if (sg == S - 1) break;
    const float4 b = bnext;
    __syncthreads();  // the previous step is done with X and with the buffer refilled next
    *reinterpret_cast<float4 *>(X + r * COMB_COLS + cq) = acc;
    if (sg + 1 < S - 1) {
      stage_m(sg + 1);
      bnext = *reinterpret_cast<const float4 *>(state(sg + 1) + (size_t)r * W + KD + col);
      ptx::cp_async_wait<1>();  // M_sg has landed
    } else {
      ptx::cp_async_wait<0>();
    }
    __syncthreads();
    const float *mrow = csm + (sg & 1) * KD * COMB_LDM + r * COMB_LDM;
    // four partial sums per output (k = m mod 4) keep sixteen FMA chains in flight
    float part[4][4] = {{b.x, b.y, b.z, b.w}};
#pragma unroll 2
    for (int m = 0; m < KD; m += 4) {
      const float4 mv = *reinterpret_cast<const float4 *>(mrow + m);
      const float mm[4] = {mv.x, mv.y, mv.z, mv.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float4 x = *reinterpret_cast<const float4 *>(X + (m + e) * COMB_COLS + cq);
        part[e][0] = fmaf(mm[e], x.x, part[e][0]);
        part[e][1] = fmaf(mm[e], x.y, part[e][1]);
        part[e][2] = fmaf(mm[e], x.z, part[e][2]);
        part[e][3] = fmaf(mm[e], x.w, part[e][3]);
      }
    }
    acc = make_float4((part[0][0] + part[1][0]) + (part[2][0] + part[3][0]),
                      (part[0][1] + part[1][1]) + (part[2][1] + part[3][1]),
                      (part[0][2] + part[1][2]) + (part[2][2] + part[3][2]),
                      (part[0][3] + part[1][3]) + (part[2][3] + part[3][3]));
  }
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

// [rows][heads][128] fp32 gate tensor, boxes of 32 x 1 x 64 (a quarter tile:
// 64 rows of 128 bytes, 128-byte swizzle).
bool make_gate_map(CUtensorMap *m, const float *base, int heads, long long rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t gdim[3] = {(cuuint64_t)KD, (cuuint64_t)heads, (cuuint64_t)rows};
  cuuint64_t gstride[2] = {(cuuint64_t)KD * 4, (cuuint64_t)heads * KD * 4};
  cuuint32_t box[3] = {32, 1, 64};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(base), gdim, gstride, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [rows][heads][dim] bf16 tensor, boxes of `width` x 1 x 64 (64 rows of
// `width` contiguous elements each, in the given swizzle: 128-byte rows with
// the 128-byte swizzle, 64-byte rows with the 64-byte one).
bool make_map(CUtensorMap *m, const void *base, int dim, int heads, long long rows, int width,
              CUtensorMapSwizzle swz) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t gdim[3] = {(cuuint64_t)dim, (cuuint64_t)heads, (cuuint64_t)rows};
  cuuint64_t gstride[2] = {(cuuint64_t)dim * 2, (cuuint64_t)heads * dim * 2};
  cuuint32_t box[3] = {(cuuint32_t)width, 1, 64};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), gdim, gstride, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// k ([rows][heads][128] bf16) seen as (64 keys, rows, 2 halves, heads): one
// box of (64, 64 rows, 2, 1) lands as two 8 KB halves of 64 rows x 128 bytes,
// 128-byte swizzle (the MN-major operand the state update reads).
bool make_k_sw128_map(CUtensorMap *m, const void *base, int heads, long long rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t gdim[4] = {64, (cuuint64_t)rows, 2, (cuuint64_t)heads};
  cuuint64_t gstride[3] = {(cuuint64_t)heads * KD * 2, 128, KD * 2};
  cuuint32_t box[4] = {64, 64, 2, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), gdim, gstride, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t table_bytes(int N) { return ((2 * (size_t)N + 1) * 4 + 255) / 256 * 256; }

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    (void)cudaGetLastError();
    return 148;
  }
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
      (void)cudaGetLastError();
      n = 148;
    }
    cached[dev] = n;
  }
  return cached[dev];
}

// Segments per sequence for the state pass: `requested` if given (>= 1),
// else the count that shortens the sequential chain most while the first
// phase's CTAs (one per SM) still fit on the GPU at once.  Cost in chain
// steps: 2 ceil(nc / S) for the two phases, about half a step per combine
// step and four for the two extra launches; taken only when it beats nc, so
// never when the sequences' own chains already fill half the SMs.
int segment_count(const ChunkParams &cp, bool varlen) {
  if (cp.segments >= 1) return cp.segments;
  const long long vtiles = cp.V / VTILE, ktiles = KD / VTILE;
  const long long chains = vtiles * cp.H * cp.N;
  const double nc = varlen ? (double)cp.T / cp.N / BT : (double)((cp.T + BT - 1) / BT);
  const long long sms = sm_count();
  if (2 * chains > sms || nc < 16.0) return 1;
  int best = 1;
  double best_cost = nc;
  for (int S = 2; S <= 16; ++S) {
    if ((long long)cp.H * cp.N * (vtiles + (S - 1) * (ktiles + vtiles)) > sms) break;
    const double cost = 2.0 * std::ceil(nc / S) + 0.5 * (S - 2) + 4.0;
    if (cost < best_cost) {
      best = S;
      best_cost = cost;
    }
  }
  return best;
}

size_t segment_bytes(const ChunkParams &cp, int S) {
  if (S <= 1) return 0;
  const size_t per = (size_t)cp.N * S * cp.H * KD;
  return (per * (KD + cp.V) * 4 + 255) / 256 * 256 + (per * cp.V * 4 + 255) / 256 * 256;
}

size_t max_chunks(int B, int T, int N, bool varlen) {
  const size_t nt = ((size_t)T + BT - 1) / BT;
  return varlen ? nt + (size_t)N : (size_t)B * nt;
}

}  // namespace tc

bool chunk_tc_supported(const ChunkParams &p, bool bf16) {
  return bf16 && p.K == tc::KD && p.V % tc::VTILE == 0 && p.V <= tc::VMAX && p.T > 0;
}

int chunk_tc_segments(const ChunkParams &p) {
  return tc::segment_count(p, p.cu_seqlens != nullptr);
}

size_t chunk_tc_workspace(const ChunkParams &p, bool kda) {
  const bool varlen = p.cu_seqlens != nullptr;
  return tc::table_bytes(p.N) +
         tc::max_chunks(p.B, p.T, p.N, varlen) * (size_t)p.H * tc::block_bytes(p.V, kda) +
         tc::segment_bytes(p, tc::segment_count(p, varlen));
}

cudaError_t launch_chunk_tc(const ChunkParams &cp, bool kda, void *ws, cudaStream_t stream) {
  using namespace tc;
  const bool varlen = cp.cu_seqlens != nullptr;
  CUtensorMap mk, mq, mv, mg;
  const long long rows = (long long)cp.B * cp.T;
  // k, q: 64-key tiles, 128-byte swizzle; v: 32-column tiles, 64-byte swizzle
  if (!make_map(&mk, cp.k, KD, cp.Hk, rows, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&mq, cp.q, KD, cp.Hk, rows, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&mv, cp.v, cp.V, cp.H, rows, 32, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  if (kda) {
    if (!make_gate_map(&mg, cp.g, cp.H, rows)) return cudaErrorInvalidValue;
  } else {
    mg = mk;  // unused by the scalar-gate kernel
  }
  TcParams p{};
  p.g = cp.g; p.beta = cp.beta; p.h0 = cp.h0; p.ht = cp.ht;
  p.kraw = cp.k; p.qraw = cp.q;
  p.o = cp.o;
  p.o_f32 = cp.o_f32;
  p.cu_seqlens = cp.cu_seqlens;
  p.table = static_cast<int32_t *>(ws);
  p.blocks = static_cast<unsigned char *>(ws) + table_bytes(cp.N);
  p.err = cp.err;
  p.B = cp.B; p.T = cp.T; p.H = cp.H; p.Hk = cp.Hk; p.V = cp.V; p.N = cp.N;
  p.NT = (cp.T + BT - 1) / BT;
  p.g_is_cumsum = cp.g_is_cumsum;
  p.v_first = cp.v_first;
  p.scale = cp.scale;
  p.block = block_bytes(cp.V, kda);
  p.nblk = (int)max_chunks(cp.B, cp.T, cp.N, varlen);
  const int S = segment_count(cp, varlen);
  p.seg_count = S;
  p.seg_phase = 0;
  if (S > 1) {
    const size_t nchunks_all = max_chunks(cp.B, cp.T, cp.N, varlen);
    unsigned char *seg = p.blocks + nchunks_all * (size_t)cp.H * p.block;
    const size_t per = (size_t)cp.N * S * cp.H * KD;
    p.seg_state = reinterpret_cast<float *>(seg);
    p.seg_start = reinterpret_cast<float *>(seg + (per * (KD + cp.V) * 4 + 255) / 256 * 256);
  }
  if (varlen) {
    chunk_table_kernel<<<1, TABLE_THREADS, 0, stream>>>(cp.cu_seqlens, cp.N, cp.T, p.table, cp.err);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const size_t nchunks = max_chunks(cp.B, cp.T, cp.N, varlen);
  auto ik = kda ? intra_kernel<true> : intra_kernel<false>;
  const uint32_t ismem = kda ? IntraLayout<true>::SMEM : IntraLayout<false>::SMEM;
  cudaError_t e = cudaFuncSetAttribute(ik, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ismem);
  if (e != cudaSuccess) return e;
  // Every kernel after the first is a programmatic dependent launch: its CTAs
  // start as the previous grid's CTAs exit and wait (griddepcontrol.wait)
  // for its results before reading them, which hides the launch gap (few long
  // chains with segments: 82.9 -> 78 us).  The intra kernel is one only behind
  // the chunk-table kernel: as the first kernel of a call it was 0.9 us slower.
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t icfg = {};
  icfg.gridDim = dim3((unsigned)nchunks, kda ? cp.H : cp.Hk);  // scalar gate: one key head a CTA
  icfg.blockDim = dim3(INTRA_THREADS);
  icfg.dynamicSmemBytes = ismem;
  icfg.stream = stream;
  icfg.attrs = pdl;
  icfg.numAttrs = varlen ? 1 : 0;
  if ((e = cudaLaunchKernelEx(&icfg, ik, mk, mq, mv, mg, p)) != cudaSuccess) return e;
  CUtensorMap mkr;
  if (kda) {
    mkr = mk;  // unused: the per-channel chain reads KT
  } else if (!make_k_sw128_map(&mkr, cp.k, cp.Hk, rows)) {
    return cudaErrorInvalidValue;
  }
  auto chain = kda ? chain_kernel<false> : chain_kernel<true>;
  e = cudaFuncSetAttribute(chain, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C_SMEM);
  if (e != cudaSuccess) return e;
  // The chain kernel runs its set-up before it waits for the intra kernel's
  // results (GDN 170.2 -> 166.9 us).  An explicit early trigger in the intra
  // kernel, which lets the chain grid be scheduled during the intra kernel's
  // last wave, was slower (176.1 us).
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(CHAIN_THREADS);
  cfg.dynamicSmemBytes = C_SMEM;
  cfg.stream = stream;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  if (S <= 1) {
    cfg.gridDim = dim3(cp.V / VTILE, cp.H, cp.N);
    return cudaLaunchKernelEx(&cfg, chain, mkr, p);
  }
  // segment-parallel: every segment at once (transition and value tiles),
  // the combine, then segments 1.. again from their true start states
  p.seg_phase = 1;
  cfg.gridDim = dim3(KD / VTILE + cp.V / VTILE, cp.H, cp.N * S);
  if ((e = cudaLaunchKernelEx(&cfg, chain, mkr, p)) != cudaSuccess) return e;
  e = cudaFuncSetAttribute(segment_combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)COMB_SMEM);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t ccfg = cfg;
  ccfg.gridDim = dim3(cp.V / COMB_COLS, cp.H, cp.N);
  ccfg.blockDim = dim3(COMB_THREADS);
  ccfg.dynamicSmemBytes = COMB_SMEM;
  if ((e = cudaLaunchKernelEx(&ccfg, segment_combine_kernel, p)) != cudaSuccess) return e;
  p.seg_phase = 2;
  cfg.gridDim = dim3(cp.V / VTILE, cp.H, cp.N * (S - 1));
  return cudaLaunchKernelEx(&cfg, chain, mkr, p);
}

}  // namespace gdn
