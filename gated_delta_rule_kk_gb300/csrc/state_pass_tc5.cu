// Chunk state pass on the 5th-generation tensor cores (tcgen05 + TMA), bf16
// inputs with K = 128, V a multiple of 32, every gate kind.  The recurrence is
// that of state_pass.cu (KDA _fla/ops/common/chunk_h.py, chunk_fwd_kernel_h and
// chunk_bwd_kernel_dh):
//   h_{c+1} = decay_c o h_c + Delta_c,   Delta_c = k~_c^T v~_c,
// where decay_c is e^{g_L} (per column e^{gv_L}, per key row e^{gk_L}).  For
// the value-side gates (none, g, g_gamma, gv) v~ carries every token factor
// (forward e^{g_L - g_i} e^{gv_L - gv_i}, backward scale e^{g_i} e^{gv_i}) and
// k~ = k; for the per-key gate gk, k~ = k e^{gk_L - gk_i} (backward q e^{gk_i})
// and v~ = v (backward the scale on the product).  Delta_c does not depend on
// h, so the tensor core computes it for chunks ahead of the state: only the
// element-wise update is sequential.
//
// One CTA per (32-column V tile, head, sequence); warps 0-3 state, then the
// stagers (4, or 8 for gk), the producer, the MMA issuer and the store warp:
//   producer    one TMA each (from lanes 0, 1, 2..) for the chunk's k tile, its
//               v tile and, for gv / gk, its gate tile, into a ring of NS
//               slots, all with swizzled rows of 64 or 128 bytes (a TMA moves
//               a box row by row, so narrow rows cost requests): k lands as two
//               128-byte swizzled MN-major atoms columns (keys 0-63 and 64-127)
//               that the MMA reads directly; the per-token gate g by cp.async
//               from every lane (counted on the slot's barrier), so no consumer
//               ever waits on a global load
//   stagers     value-side gates: thread (i, half) forms row i, 16 columns, of
//               v~ = v x factor as a bf16 hi/lo pair (zero past the chunk's
//               end) into one of two operand images; gk: thread (i, part)
//               forms k~ for row i, 32 keys, as a bf16 hi/lo pair in the raw k
//               image's layout (hi over the raw k in its slot, lo into one of
//               two images)
//   MMA         Delta_c = k^T [v~_hi | v~_lo] (M = 128 keys, N = 64, K = 64
//               tokens; gk: k~_hi^T v + k~_lo^T v at N = 32, v raw from its
//               64-byte-swizzled tile) into one of two TMEM accumulators
//   store       one TMA store per stored chunk state, from a ring of NB
//               staging tiles the state warps fill (so the stores leave in
//               whole rows and their issue and completion stay off the
//               state's sequential path)
//   state       thread r holds key row r, 32 columns, of the fp32 state; per
//               chunk it writes the chunk-start state (when that chunk is
//               stored) and applies h = decay o h + Delta, the scalar or
//               per-key decay from a load issued one chunk ahead, gv's from
//               the chunk's ring slot
// Every wait is bounded (GDN_ERR_TIMEOUT, then every role still runs every
// chunk so no barrier is left short of arrivals).
#include <cuda.h>
#include <cudaTypedefs.h>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "ptx.cuh"

namespace gdn {
namespace {

constexpr int T5_VT = 32, T5_KD = 128, T5_NB = 2;
// ring depth: the loads take ~2-3 K cycles under load, so the ring is as deep
// as shared memory allows (a slot holds a chunk from its TMA issue until the
// stagers and the MMA, and for gv the state warps, are done with it)
// gate modes: 0 = value-side scalar gates (g, g_gamma, none), 1 = gv, 2 = gk
constexpr int t5_ns(int gm) { return gm == 1 ? 6 : gm == 2 ? 3 : 8; }
// warps 0-3 state, then the stagers (8 for gk, whose k~ takes an exponential
// per element, else 4), the producer, the MMA issuer and the store warp
constexpr int t5_stagers(int gm) { return gm == 2 ? 8 : 4; }
constexpr int t5_threads(int gm) { return 32 * (7 + t5_stagers(gm)); }
// ring slot: k image (two 8 KB halves of 64 keys: 64 token rows of 128 bytes,
// 128-byte swizzle), v tile (64 token rows of 32 bf16, 64-byte swizzle),
// gate: g per token (64 fp32), the gv tile (64 token rows of 32 fp32) or the
// gk tile (four 8 KB boxes of 32 keys x 64 token rows fp32), 128-byte swizzle,
// all inside the slot
constexpr uint32_t T5_RK = 0, T5_RV = 16384, T5_RG = 20480;
// (1024-byte multiples, so every slot's k image stays 1024-aligned)
constexpr uint32_t t5_slot_bytes(int gm) { return gm == 1 ? 28672u : gm == 2 ? 53248u : 21504u; }
// NB staging tiles of one chunk state, 128 x 32 fp32 (16 KB): [key row][32
// columns] in 128-byte (fp32) or 64-byte (bf16) swizzled rows, or [column]
// [128 keys] unswizzled for states stored as [V, K]
constexpr uint32_t T5_TILE = 16384, T5_STAGE = T5_NB * T5_TILE;
// v~ image: 64 token rows x 64 columns (hi 0..31, lo 32..63), group stride 1024
constexpr uint32_t T5_VTB = 8192;
// operand images the stagers write, two buffers: v~ (8 KB each) or, for gk,
// the lo half of k~ = k e^(gk_L - gk) in the raw k image's layout (16 KB
// each; the hi half replaces the raw k image in its ring slot, which only
// the stagers read)
constexpr uint32_t t5_img_bytes(int gm) { return gm == 2 ? 2u * 16384u : 2u * T5_VTB; }

struct T5Seq {
  int bos, eos, b, nch;
  long long first;
  bool write_hs;
};

// Sequence n's token range and first stored-state index (one thread reads the
// offsets; bad cu_seqlens or too small a num_chunks are recorded).
__device__ T5Seq t5_sequence(const StateParams &p, int n, int tid, long long *sh) {
  T5Seq s;
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
      sh[0] = first;
      sh[1] = ok ? 1 : 0;
      if (!ok) record_error(p.err, GDN_ERR_BAD_SEQLENS);
    }
    __syncthreads();
    if (sh[1] == 0) s.bos = s.eos = 0;
  } else if (tid == 0) {
    sh[0] = (long long)n * ((p.T + BT * p.split - 1) / (BT * p.split));
    sh[1] = 1;
  }
  __syncthreads();
  s.nch = (s.eos - s.bos + BT - 1) / BT;
  s.first = sh[0];
  s.write_hs = p.hs && sh[1] && s.first + (s.nch + p.split - 1) / p.split <= p.num_chunks;
  if (p.hs && sh[1] && !s.write_hs && tid == 0) record_error(p.err, GDN_ERR_BAD_SEQLENS);
  return s;
}

// Packed fp32 pairs (sm_100: two lanes per instruction, each rounded to
// nearest).
__device__ __forceinline__ float2 t5_sub2(float2 a, float2 b) {
  float2 r;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "sub.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}
__device__ __forceinline__ float2 t5_mul2(float2 a, float2 b) {
  float2 r;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}

__device__ __forceinline__ void t5_split8(const float *f, uint4 &hi, uint4 &lo) {
  __nv_bfloat162 h2[4];
  float r[8];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    h2[e] = __floats2bfloat162_rn(f[2 * e], f[2 * e + 1]);
    const float2 d = t5_sub2(make_float2(f[2 * e], f[2 * e + 1]), __bfloat1622float2(h2[e]));
    r[2 * e] = d.x;
    r[2 * e + 1] = d.y;
  }
  hi = *reinterpret_cast<const uint4 *>(h2);
  __nv_bfloat162 l2[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) l2[e] = __floats2bfloat162_rn(r[2 * e], r[2 * e + 1]);
  lo = *reinterpret_cast<const uint4 *>(l2);
}

// The stored-state index of each chunk in processing order: every chunk, or
// with `split` > 1 every split-th one (chunk 0, split, ..), numbered from the
// sequence's first stored state; next() returns -1 for a chunk not stored.
struct T5Stores {
  long long first;
  int split, step, store_i, store_c;
  __device__ T5Stores(const StateParams &p, long long first_, int nch) : first(first_) {
    split = p.split;
    step = p.reverse ? -1 : 1;
    store_i = split > 1 && p.reverse && nch > 0 ? (nch - 1) / split : 0;
    store_c = store_i * split;
  }
  template <bool SPLIT>
  __device__ long long next(int c) {
    if (!SPLIT) return first + c;
    if (c != store_c) return -1;
    const long long slot = first + store_i;
    store_c += step * split;
    store_i += step;
    return slot;
  }
};

__device__ __forceinline__ void t5_tma_load_4d(void *dst, const void *tmap, int c0, int c1, int c2,
                                               int c3, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(ptx::smem_u32(dst)),
      "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(ptx::smem_u32(bar))
      : "memory");
}

// Shared-memory matrix descriptor for a 128-byte-swizzled operand (layout
// field 2); lbo / sbo as for the MN-major swizzled layouts: the distance
// between 64-element atoms columns along M or N, and between 8-row groups
// along K.
__device__ __forceinline__ uint64_t t5_sdesc_sw128(const void *smem, uint32_t lbo, uint32_t sbo) {
  return ptx::sdesc(smem, lbo, sbo) | (2ull << 61);
}

template <int GM, bool VF, bool SPLIT>
__global__ void __launch_bounds__(t5_threads(GM), 1)
state_pass_tc5_kernel(const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_g,
                      const __grid_constant__ CUtensorMap tm_hs, StateParams p) {
  extern __shared__ __align__(1024) unsigned char sm5_raw[];
  constexpr bool GV = GM == 1, GK = GM == 2;
  constexpr int T5_STAGERS = t5_stagers(GM), T5_WPROD = 4 + T5_STAGERS, T5_WMMA = T5_WPROD + 1,
                T5_WSTORE = T5_WPROD + 2;
  constexpr int K = T5_KD;
  constexpr uint32_t SLOT = t5_slot_bytes(GM);
  // the swizzle patterns follow address bits 4-9: slots start on 1024 bytes
  unsigned char *sm5 = sm5_raw + ((1024u - (ptx::smem_u32(sm5_raw) & 1023u)) & 1023u);
  unsigned char *ring = sm5;
  constexpr int T5_NS = t5_ns(GM);
  unsigned char *vimg = sm5 + T5_NS * SLOT;       // two operand images (v~, or k~ pairs)
  unsigned char *stage = vimg + t5_img_bytes(GM);  // NB state staging tiles
  uint64_t *bars = reinterpret_cast<uint64_t *>(stage + T5_STAGE);
  uint64_t *full = bars, *empty = bars + T5_NS;
  uint64_t *vready = bars + 2 * T5_NS, *vfree = vready + 2, *afull = vfree + 2, *afree = afull + 2;
  uint64_t *staged = afree + 2, *stfree = staged + T5_NB;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(stfree + T5_NB);
  __shared__ long long seq_sh[2];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int v0 = blockIdx.x * T5_VT, h = blockIdx.y, n = blockIdx.z;
  const int H = p.H, V = p.V, HG = p.HG, hg = h / (H / HG);
  const bool scalar_gate = p.gate == GDN_GATE_G || p.gate == GDN_GATE_G_GAMMA;
  const float gamma = p.gate == GDN_GATE_G_GAMMA ? p.gate_values[hg] : 0.f;
  const T5Seq sq = t5_sequence(p, n, tid, seq_sh);
  if (!bounds_ok(n < p.N && h < H && hg < HG && v0 + T5_VT <= V && sq.bos >= 0 &&
                     sq.bos <= sq.eos && sq.eos <= p.T,
                 p.err))
    return;
  auto chunk_at = [&](int it) { return p.reverse ? sq.nch - 1 - it : it; };

  if (tid == 0) {
    for (int s = 0; s < T5_NS; ++s) {
      // the producer's expect-tx arrival + one cp.async arrival per lane
      ptx::mbar_init(&full[s], 1 + 32);
      // the stager warps + the MMA's commit (+ for gv the four state warps,
      // which read the chunk's last gate row there)
      ptx::mbar_init(&empty[s], T5_STAGERS + 1 + (GV ? 4 : 0));
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&vready[b], T5_STAGERS);
      ptx::mbar_init(&vfree[b], 1);
      ptx::mbar_init(&afull[b], 1);
      ptx::mbar_init(&afree[b], 4);
    }
    for (int b = 0; b < T5_NB; ++b) {
      ptx::mbar_init(&staged[b], 4);  // the four state warps
      ptx::mbar_init(&stfree[b], 1);  // the store warp
    }
    ptx::fence_mbar_init();
  }
  if (warp == 0) ptx::tmem_alloc<128>(tmem_slot);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;

  if (warp == T5_WPROD) {
    // ---------------- producer
    if (lane == 0) {
      ptx::prefetch_tmap(&tm_k);
      ptx::prefetch_tmap(&tm_v);
      if (GV) ptx::prefetch_tmap(&tm_g);
    }
    const uint32_t bytes = 16384u + 4096u + (GV ? 8192u : 0u) + (GK ? 32768u : 0u);
    const long long rows = (long long)p.B * p.T;
#pragma unroll 1
    for (int it = 0; it < sq.nch; ++it) {
      const int s = it % T5_NS;
      if (it >= T5_NS)
        ok = ptx::mbar_wait_bounded(&empty[s], (uint32_t)((it / T5_NS - 1) & 1)) && ok;
      __syncwarp();
      unsigned char *slot = ring + s * SLOT;
      const int row0 = sq.b * p.T + sq.bos + chunk_at(it) * BT;
      // one copy per lane: the copies one thread issues complete one after
      // another, those of different threads overlap
      if (lane == 0) ptx::mbar_arrive_expect_tx(&full[s], bytes);
      __syncwarp();
      if (lane == 0) t5_tma_load_4d(slot + T5_RK, &tm_k, 0, row0, 0, h, &full[s]);
      if (lane == 1) ptx::tma_load_3d(slot + T5_RV, &tm_v, v0, h, row0, &full[s]);
      if (GV && lane == 2) ptx::tma_load_3d(slot + T5_RG, &tm_g, v0, hg, row0, &full[s]);
      if (GK && lane >= 2 && lane < 6)
        ptx::tma_load_3d(slot + T5_RG + (lane - 2) * 8192, &tm_g, 32 * (lane - 2), hg, row0, &full[s]);
      if (p.gate == GDN_GATE_G) {
        // g of the chunk's 64 rows (rows past the tensor read as zero)
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const long long r = (long long)row0 + lane + 32 * q;
          const bool in = r < rows;
          ptx::cp_async4(slot + T5_RG + (lane + 32 * q) * 4,
                         p.gate_values + (in ? r : 0) * HG + hg, in);
        }
      }
      ptx::cp_async_mbar_arrive(&full[s]);
    }
  } else if (GK && warp >= 4 && warp < 4 + T5_STAGERS) {
    // ---------------- gk stagers: thread (i, part) = token row i, keys 32 part ..
    // k~ = k e^(gk_L - gk_i) (backward: q e^(gk_i)), zero past the chunk's
    // end, as a bf16 hi/lo pair in the raw k image's layout (hi in place)
    constexpr int CPT = 8 * 4 / T5_STAGERS;  // 16-byte chunks (8 keys) per thread
    const int i = (tid - 128) & 63, part = (tid - 128) >> 6;
    const int half = part * CPT / 8, c0 = part * CPT % 8;
    auto len_of = [&](int it) { return min(BT, sq.eos - (sq.bos + chunk_at(it) * BT)); };
#pragma unroll 1
    for (int it = 0; it < sq.nch; ++it) {
      const int s = it % T5_NS, b = it & 1;
      const int L = len_of(it);
      ok = ptx::mbar_wait_bounded(&full[s], (uint32_t)((it / T5_NS) & 1)) && ok;
      if (it >= 2) ok = ptx::mbar_wait_bounded(&vfree[b], (uint32_t)(((it >> 1) - 1) & 1)) && ok;
      unsigned char *slot = ring + s * SLOT;
      // k~_hi over the raw k it is formed from (each thread reads and writes
      // the same 16-byte chunks), k~_lo into its own image
      unsigned char *khi = slot + T5_RK + half * 8192;
      unsigned char *klo = vimg + b * 16384 + half * 8192;
      const unsigned char *kin = khi;
#pragma unroll
      for (int cc = 0; cc < CPT; ++cc) {
        const int c = c0 + cc;
        // keys 64 half + 8 c .. + 7: 16-byte chunk c of row i (chunk c ^ (i & 7));
        // in the gk tile, box 2 half + c / 4, chunks 2 (c % 4), + 1 of row i
        const int cs = (c ^ (i & 7)) << 4;
        float kf[8];
        {
          const uint4 u = *reinterpret_cast<const uint4 *>(kin + i * 128 + cs);
          const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            kf[2 * e] = __uint_as_float(w[e] << 16);
            kf[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
          }
        }
        const unsigned char *gb = slot + T5_RG + (2 * half + (c >> 2)) * 8192;
        const int g0 = 2 * (c & 3);
        float x[8];
        if (i < L) {
          const float4 a0 = *reinterpret_cast<const float4 *>(gb + i * 128 + ((g0 ^ (i & 7)) << 4));
          const float4 a1 = *reinterpret_cast<const float4 *>(gb + i * 128 + (((g0 + 1) ^ (i & 7)) << 4));
          float2 gi[4] = {make_float2(a0.x, a0.y), make_float2(a0.z, a0.w), make_float2(a1.x, a1.y),
                          make_float2(a1.z, a1.w)};
          if (!p.reverse) {
            const int l = L - 1;
            const float4 b0 = *reinterpret_cast<const float4 *>(gb + l * 128 + ((g0 ^ (l & 7)) << 4));
            const float4 b1 = *reinterpret_cast<const float4 *>(gb + l * 128 + (((g0 + 1) ^ (l & 7)) << 4));
            gi[0] = t5_sub2(make_float2(b0.x, b0.y), gi[0]);
            gi[1] = t5_sub2(make_float2(b0.z, b0.w), gi[1]);
            gi[2] = t5_sub2(make_float2(b1.x, b1.y), gi[2]);
            gi[3] = t5_sub2(make_float2(b1.z, b1.w), gi[3]);
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 y = t5_mul2(make_float2(kf[2 * e], kf[2 * e + 1]),
                                     make_float2(__expf(gi[e].x), __expf(gi[e].y)));
            x[2 * e] = y.x;
            x[2 * e + 1] = y.y;
          }
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] = 0.f;
        }
        uint4 hi, lo;
        t5_split8(x, hi, lo);
        *reinterpret_cast<uint4 *>(khi + i * 128 + cs) = hi;
        *reinterpret_cast<uint4 *>(klo + i * 128 + cs) = lo;
      }
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        ptx::mbar_arrive(&vready[b]);
        ptx::mbar_arrive(&empty[s]);  // this warp has read the slot's k and gate tile
      }
    }
  } else if (!GK && warp >= 4 && warp < 4 + T5_STAGERS) {
    // ---------------- stagers: thread (i, half) = token row i, columns 16 half ..
    const int i = (tid - 128) & 63, half = (tid - 128) >> 6;
    auto len_of = [&](int it) { return min(BT, sq.eos - (sq.bos + chunk_at(it) * BT)); };
#pragma unroll 1
    for (int it = 0; it < sq.nch; ++it) {
      const int s = it % T5_NS, b = it & 1;
      const int L = len_of(it);
      ok = ptx::mbar_wait_bounded(&full[s], (uint32_t)((it / T5_NS) & 1)) && ok;
      const unsigned char *slot = ring + s * SLOT;
      const float *gslot = reinterpret_cast<const float *>(slot + T5_RG);
      float f = 0.f;
      if (i < L) {
        f = p.reverse ? p.scale : 1.f;
        if (scalar_gate) {
          const float g_i = p.gate == GDN_GATE_G ? gslot[i] : gamma * (float)(i + 1);
          const float g_l = p.gate == GDN_GATE_G ? gslot[L - 1] : gamma * (float)L;
          f *= expf(p.reverse ? g_i : g_l - g_i);
        }
      }
      // the thread's two 16-byte chunks of v row i (64-byte swizzle: chunk c
      // of row i sits at chunk c ^ ((i >> 1) & 3))
      float x[16];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int c = (2 * half + q) ^ ((i >> 1) & 3);
        const uint4 u = *reinterpret_cast<const uint4 *>(slot + T5_RV + i * 64 + c * 16);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          x[8 * q + 2 * e] = __uint_as_float(w[e] << 16) * f;
          x[8 * q + 2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u) * f;
        }
      }
      if (GV && i < L) {
        // gv rows of 128 bytes, 128-byte swizzle (chunk c of row r at chunk
        // c ^ (r & 7)): this thread's 16 columns are chunks 4 half .. 4 half + 3
        const unsigned char *gt = slot + T5_RG;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int c = 4 * half + q;
          const float4 gi4 = *reinterpret_cast<const float4 *>(gt + i * 128 + (c ^ (i & 7)) * 16);
          const float4 gl4 = *reinterpret_cast<const float4 *>(gt + (L - 1) * 128 +
                                                               (c ^ ((L - 1) & 7)) * 16);
          const float gi[4] = {gi4.x, gi4.y, gi4.z, gi4.w}, gl[4] = {gl4.x, gl4.y, gl4.z, gl4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) x[4 * q + e] *= expf(p.reverse ? gi[e] : gl[e] - gi[e]);
        }
      }
      if (it >= 2) ok = ptx::mbar_wait_bounded(&vfree[b], (uint32_t)(((it >> 1) - 1) & 1)) && ok;
      unsigned char *img = vimg + b * T5_VTB;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        uint4 hi, lo;
        t5_split8(x + 8 * q, hi, lo);
        *reinterpret_cast<uint4 *>(img + (2 * half + q) * 1024 + i * 16) = hi;
        *reinterpret_cast<uint4 *>(img + (4 + 2 * half + q) * 1024 + i * 16) = lo;
      }
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        ptx::mbar_arrive(&vready[b]);
        ptx::mbar_arrive(&empty[s]);  // this warp has read the slot's v (and gate) tile
      }
    }
  } else if (warp == T5_WMMA) {
    // ---------------- MMA issuer
    // A and B MN-major; gk: N = 32 (v raw), otherwise N = 64 (v~ hi | lo)
    const uint32_t id = ptx::idesc_bf16(128, GK ? T5_VT : 2 * T5_VT, 1, 1);
#pragma unroll 1
    for (int it = 0; it < sq.nch; ++it) {
      const int s = it % T5_NS, b = it & 1;
      ok = ptx::mbar_wait_bounded(&full[s], (uint32_t)((it / T5_NS) & 1)) && ok;
      ok = ptx::mbar_wait_bounded(&vready[b], (uint32_t)((it >> 1) & 1)) && ok;
      if (it >= 2) ok = ptx::mbar_wait_bounded(&afree[b], (uint32_t)(((it >> 1) - 1) & 1)) && ok;
      __syncwarp();
      ptx::tc_fence_after();
      if (lane == 0) {
        // A: MN-major, 128-byte swizzle, 64-key atoms columns 8 KB apart, 8-token
        // groups 1 KB apart; a K step of 16 tokens is two groups (2 KB)
        if (GK) {
          // D = k~_hi^T v + k~_lo^T v; B = the raw v tile, MN-major with
          // 64-byte swizzle (one 32-column atom, 8-token groups 512 bytes
          // apart; a K step is 1 KB)
          const uint64_t ah = t5_sdesc_sw128(ring + s * SLOT + T5_RK, 8192, 1024);
          const uint64_t al = t5_sdesc_sw128(vimg + b * 16384, 8192, 1024);
          const uint64_t bv = ptx::sdesc(ring + s * SLOT + T5_RV, 512, 512) | (4ull << 61);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            ptx::mma_bf16(tmem + 64 * b, ah + (uint64_t)(ks * 2048 >> 4),
                          bv + (uint64_t)(ks * 1024 >> 4), id, ks > 0);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            ptx::mma_bf16(tmem + 64 * b, al + (uint64_t)(ks * 2048 >> 4),
                          bv + (uint64_t)(ks * 1024 >> 4), id, 1);
        } else {
          const uint64_t a = t5_sdesc_sw128(ring + s * SLOT + T5_RK, 8192, 1024);
          const uint64_t bv = ptx::sdesc(vimg + b * T5_VTB, 128, 1024);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            ptx::mma_bf16(tmem + 64 * b, a + (uint64_t)(ks * 2048 >> 4),
                          bv + (uint64_t)(ks * 256 >> 4), id, ks > 0);
        }
        ptx::mma_commit(&afull[b]);
        ptx::mma_commit(&vfree[b]);
        ptx::mma_commit(&empty[s]);
      }
      __syncwarp();
    }
  } else if (warp == T5_WSTORE) {
    // ---------------- store: one TMA store per staged chunk state
    if (lane == 0 && sq.write_hs) {
      ptx::prefetch_tmap(&tm_hs);
      T5Stores stores(p, sq.first, sq.nch);
      int nst = 0;
#pragma unroll 1
      for (int it = 0; it < sq.nch; ++it) {
        const long long slot = stores.next<SPLIT>(chunk_at(it));
        if (slot < 0) continue;
        const int sb = nst % T5_NB;
        ok = ptx::mbar_wait_bounded(&staged[sb], (uint32_t)((nst / T5_NB) & 1)) && ok;
        // hs seen as 2-D: [stored state, head, K or V rows][V or K columns]
        const long long row0 = (slot * H + h) * (VF ? V : K) + (VF ? v0 : 0);
        ptx::tma_store_2d(&tm_hs, VF ? 0 : v0, (int)row0, stage + sb * T5_TILE);
        ptx::bulk_commit();
        if (nst > 0) {  // the previous tile has been read: hand it back
          ptx::bulk_wait_read<1>();
          ptx::mbar_arrive(&stfree[(nst - 1) % T5_NB]);
        }
        ++nst;
      }
      ptx::bulk_wait<0>();  // every chunk state is written
    }
  } else {
    // ---------------- state warps 0-3: key row r, columns v0 .. v0 + 31
    const int r = warp * 32 + lane;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const size_t hbase = ((size_t)n * H + h) * K * V;
    auto at = [&](int col) { return VF ? (size_t)(v0 + col) * K + r : (size_t)r * V + v0 + col; };
    float hs[T5_VT];
    if (p.h0) {
      if (VF) {
#pragma unroll
        for (int j = 0; j < T5_VT; ++j) hs[j] = p.h0[hbase + at(j)];
      } else {
        const float4 *src = reinterpret_cast<const float4 *>(p.h0 + hbase + at(0));
#pragma unroll
        for (int q = 0; q < T5_VT / 4; ++q) {
          const float4 x = src[q];
          hs[4 * q] = x.x; hs[4 * q + 1] = x.y; hs[4 * q + 2] = x.z; hs[4 * q + 3] = x.w;
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < T5_VT; ++j) hs[j] = 0.f;
    }
    auto len_of = [&](int it) { return min(BT, sq.eos - (sq.bos + chunk_at(it) * BT)); };
    int nst = 0;  // chunk states written to the staging ring
    T5Stores stores(p, sq.first, sq.nch);
    // gate g at the chunk's last row (chunk-local cumulative sum)
    // (gk: this thread's key row r of the per-key gate there)
    auto g_end = [&](int it) {
      const long long row = (long long)sq.b * p.T + sq.bos + chunk_at(it) * BT + len_of(it) - 1;
      return GK ? p.gate_values[(row * HG + hg) * K + r] : p.gate_values[row * HG + hg];
    };
    const bool row_gate = p.gate == GDN_GATE_G || GK;
    float g_next = row_gate && sq.nch > 0 ? g_end(0) : 0.f;
#pragma unroll 1
    for (int it = 0; it < sq.nch; ++it) {
      const int b = it & 1, s = it % T5_NS;
      const long long slot = stores.next<SPLIT>(chunk_at(it));
      if (sq.write_hs && slot >= 0) {
        const int sb = nst % T5_NB;
        unsigned char *stg = stage + sb * T5_TILE;
        if (nst >= T5_NB)  // the store warp has read the tile's previous state
          ok = ptx::mbar_wait_bounded(&stfree[sb], (uint32_t)((nst / T5_NB - 1) & 1)) && ok;
        if (VF) {
#pragma unroll
          for (int j = 0; j < T5_VT; ++j) {
            if (p.hs_bf16)
              reinterpret_cast<__nv_bfloat16 *>(stg)[j * K + r] = __float2bfloat16_rn(hs[j]);
            else
              reinterpret_cast<float *>(stg)[j * K + r] = hs[j];
          }
        } else if (p.hs_bf16) {
#pragma unroll
          for (int q = 0; q < T5_VT / 8; ++q) {
            __nv_bfloat162 w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) w[e] = __floats2bfloat162_rn(hs[8 * q + 2 * e], hs[8 * q + 2 * e + 1]);
            *reinterpret_cast<uint4 *>(stg + r * 64 + ((q ^ ((r >> 1) & 3)) << 4)) =
                *reinterpret_cast<const uint4 *>(w);
          }
        } else {
#pragma unroll
          for (int q = 0; q < T5_VT / 4; ++q)
            *reinterpret_cast<float4 *>(stg + r * 128 + ((q ^ (r & 7)) << 4)) =
                make_float4(hs[4 * q], hs[4 * q + 1], hs[4 * q + 2], hs[4 * q + 3]);
        }
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&staged[sb]);
        ++nst;
      }
      // the chunk's decay: for gv from its ring slot, for g from the gate
      // value loaded one chunk ahead
      const float g_cur = g_next;
      if (row_gate && it + 1 < sq.nch) g_next = g_end(it + 1);
      float dv[T5_VT];
      if (GV) {
        ok = ptx::mbar_wait_bounded(&full[s], (uint32_t)((it / T5_NS) & 1)) && ok;
        const int L = len_of(it);
        const float *gslot = reinterpret_cast<const float *>(ring + s * SLOT + T5_RG);
#pragma unroll
        for (int j = 0; j < T5_VT; ++j)  // gv row L - 1, 128-byte swizzle
          dv[j] = expf(gslot[(L - 1) * 32 + (((j >> 2) ^ ((L - 1) & 7)) << 2) + (j & 3)]);
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&empty[s]);  // this warp is done with the slot
      } else {
        float ds = 1.f;
        if (p.gate == GDN_GATE_G || GK) ds = expf(g_cur);
        if (p.gate == GDN_GATE_G_GAMMA) ds = expf(gamma * (float)len_of(it));
#pragma unroll
        for (int j = 0; j < T5_VT; ++j) dv[j] = ds;
      }
      ok = ptx::mbar_wait_bounded(&afull[b], (uint32_t)((it >> 1) & 1)) && ok;
      ptx::tc_fence_after();
      float dh[T5_VT], dl[T5_VT];
      ptx::tmem_ld32(tmem + 64 * b + lane_base, dh);
      if (GK) {
        // one product (v raw); backward: times the scale, which v~ carries
        // for the other gates
        const float sc = p.reverse ? p.scale : 1.f;
#pragma unroll
        for (int j = 0; j < T5_VT; ++j) hs[j] = fmaf(dv[j], hs[j], sc * dh[j]);
      } else {
        ptx::tmem_ld32(tmem + 64 * b + 32 + lane_base, dl);
#pragma unroll
        for (int j = 0; j < T5_VT; ++j) hs[j] = fmaf(dv[j], hs[j], dh[j] + dl[j]);
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&afree[b]);
    }
    if (p.ht && ok) {
      if (VF) {
#pragma unroll
        for (int j = 0; j < T5_VT; ++j) p.ht[hbase + at(j)] = hs[j];
      } else {
        float4 *dst = reinterpret_cast<float4 *>(p.ht + hbase + at(0));
#pragma unroll
        for (int q = 0; q < T5_VT / 4; ++q)
          dst[q] = make_float4(hs[4 * q], hs[4 * q + 1], hs[4 * q + 2], hs[4 * q + 3]);
      }
    }
  }
  if (!ok && lane == 0) record_error(p.err, GDN_ERR_TIMEOUT);
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) ptx::tmem_dealloc<128>(tmem);
}

PFN_cuTensorMapEncodeTiled_v12000 t5_encoder() {
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

// A [rows][heads][dim] tensor of `elt`-byte elements, boxes of width x 1 x 64
// rows with the given swizzle (width x elt = the swizzle span).
bool t5_map3(CUtensorMap *m, const void *base, CUtensorMapDataType type, int elt, int dim,
             int heads, long long rows, int width, CUtensorMapSwizzle sw) {
  auto fn = t5_encoder();
  if (!fn) return false;
  cuuint64_t gdim[3] = {(cuuint64_t)dim, (cuuint64_t)heads, (cuuint64_t)rows};
  cuuint64_t gstride[2] = {(cuuint64_t)dim * elt, (cuuint64_t)heads * dim * elt};
  cuuint32_t box[3] = {(cuuint32_t)width, 1, 64};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, type, 3, const_cast<void *>(base), gdim, gstride, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A [rows][cols] tensor of `elt`-byte elements, boxes of bw x bh with the
// given swizzle (for the stored states).
bool t5_map2(CUtensorMap *m, void *base, CUtensorMapDataType type, int elt, int cols,
             long long rows, int bw, int bh, CUtensorMapSwizzle sw) {
  auto fn = t5_encoder();
  if (!fn) return false;
  cuuint64_t gdim[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t gstride[1] = {(cuuint64_t)cols * elt};
  cuuint32_t box[2] = {(cuuint32_t)bw, (cuuint32_t)bh};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, type, 2, base, gdim, gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// k ([rows][heads][128] bf16) seen as (64 keys, rows, 2 halves, heads): one
// box of (64, 64 rows, 2, 1) lands as two 8 KB halves of 64 rows x 128 bytes,
// 128-byte swizzle.
bool t5_map_k(CUtensorMap *m, const void *base, int heads, long long rows) {
  auto fn = t5_encoder();
  if (!fn) return false;
  cuuint64_t gdim[4] = {64, (cuuint64_t)rows, 2, (cuuint64_t)heads};
  cuuint64_t gstride[3] = {(cuuint64_t)heads * T5_KD * 2, 128, T5_KD * 2};
  cuuint32_t box[4] = {64, 64, 2, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), gdim, gstride, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool state_pass_tc5_supported(const StateParams &p, bool bf16) {
  const uintptr_t al = (uintptr_t)p.k | (uintptr_t)p.v | (uintptr_t)p.hs |
                       (p.gate == GDN_GATE_GV || p.gate == GDN_GATE_GK ? (uintptr_t)p.gate_values : 0);
  // (row coordinates of the stored states are 32-bit)
  return bf16 && p.K == T5_KD && p.V % T5_VT == 0 && p.T > 0 && al % 16 == 0 &&
         (!p.hs || p.num_chunks * p.H * (long long)(p.K > p.V ? p.K : p.V) < (1ll << 31)) &&
         (p.gate == GDN_GATE_NONE || p.gate == GDN_GATE_G || p.gate == GDN_GATE_G_GAMMA ||
          p.gate == GDN_GATE_GV || p.gate == GDN_GATE_GK);
}

cudaError_t launch_state_pass_tc5(const StateParams &p, cudaStream_t stream) {
  const int gm = p.gate == GDN_GATE_GV ? 1 : p.gate == GDN_GATE_GK ? 2 : 0;
  CUtensorMap mk, mv, mg;
  const long long rows = (long long)p.B * p.T;
  if (!t5_map_k(&mk, p.k, p.H, rows) ||
      !t5_map3(&mv, p.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.V, p.H, rows, T5_VT,
               CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  if (gm != 0) {
    // gv: [rows][HG][V], boxes of 32 values; gk: [rows][HG][K], boxes of 32 keys
    if (!t5_map3(&mg, p.gate_values, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, gm == 1 ? p.V : T5_KD,
                 p.HG, rows, 32, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  } else {
    mg = mv;  // unused
  }
  CUtensorMap mh = mv;  // unused without hs
  if (p.hs) {
    const int elt = p.hs_bf16 ? 2 : 4;
    const int cols = p.v_first ? p.K : p.V, rws = p.v_first ? p.V : p.K;
    const CUtensorMapSwizzle sw = p.v_first ? CU_TENSOR_MAP_SWIZZLE_NONE
                                  : p.hs_bf16 ? CU_TENSOR_MAP_SWIZZLE_64B
                                              : CU_TENSOR_MAP_SWIZZLE_128B;
    if (!t5_map2(&mh, p.hs, p.hs_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                      : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                 elt, cols, (long long)p.num_chunks * p.H * rws, p.v_first ? T5_KD : T5_VT,
                 p.v_first ? T5_VT : T5_KD, sw))
      return cudaErrorInvalidValue;
  }
  // + state staging, barriers, TMEM slot, and up to 1 KB to align the ring
  const size_t smem = t5_ns(gm) * t5_slot_bytes(gm) + t5_img_bytes(gm) + T5_STAGE + 256 + 1024;
  const bool split = p.split > 1, vf = p.v_first != 0;
  using KernT = decltype(&state_pass_tc5_kernel<0, false, false>);
  const KernT kernels[3][2][2] = {
      {{state_pass_tc5_kernel<0, false, false>, state_pass_tc5_kernel<0, false, true>},
       {state_pass_tc5_kernel<0, true, false>, state_pass_tc5_kernel<0, true, true>}},
      {{state_pass_tc5_kernel<1, false, false>, state_pass_tc5_kernel<1, false, true>},
       {state_pass_tc5_kernel<1, true, false>, state_pass_tc5_kernel<1, true, true>}},
      {{state_pass_tc5_kernel<2, false, false>, state_pass_tc5_kernel<2, false, true>},
       {state_pass_tc5_kernel<2, true, false>, state_pass_tc5_kernel<2, true, true>}}};
  const KernT kern = kernels[gm][vf][split];
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)(p.V / T5_VT), (unsigned)p.H, (unsigned)p.N);
  kern<<<grid, t5_threads(gm), smem, stream>>>(mk, mv, mg, mh, p);
  return cudaGetLastError();
}

}  // namespace gdn
