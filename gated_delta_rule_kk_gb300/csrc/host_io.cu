// gdn_chunk_fwd_host: the GDN chunked forward from and to host memory.
//
// The caller passes host buffers for every input and output and one device
// buffer (the workspace) that receives device copies of them and the scratch
// of the tensor-core kernels.  The problem is cut into pieces:
//   * time pieces (fixed-length batches of sequences of more than 11
//     64-token chunks): piece j holds tokens t0_j .. t1_j of every sequence,
//     t0_j a multiple of 64, and the pieces shrink geometrically towards the
//     end (see time_pieces);
//   * sequence pieces (shorter fixed-length sequences, or cu_seqlens): piece
//     j holds whole sequences n0_j .. n1_j, cut so that the pieces carry
//     about the same number of tokens.
// On the caller's stream each piece waits for its host->device copies (issued
// on an internal copy-in stream), runs gdn_chunk_fwd on its device copy, and
// hands its output to an internal copy-out stream.  So the copy-in of piece
// j+1 and the copy-out of piece j-1 overlap the kernels of piece j, and the
// two copy directions overlap each other.
//
// Results equal one gdn_chunk_fwd over the whole problem bit for bit: the
// chunk grid is the same (time cuts fall on chunk boundaries counted from
// each sequence's first token), sequences are independent, and a time cut
// hands the state h from one piece to the next as the same fp32 values the
// kernels carry from chunk to chunk inside one call (ht of piece j is h0 of
// piece j+1).  This is the recurrence of the gated delta rule: the state
// after a chunk depends on the tokens before it only through the state
// entering it (Gated Delta Networks, section 3, chunkwise form).
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <mutex>
#include <vector>

#include <cuda_runtime.h>

#include "gdn.h"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int MAX_PIECES = 8;
constexpr int MIN_PIECE_CHUNKS = 4;       // the last (shortest) time piece, in chunks
constexpr double PIECE_GROWTH = 2.0;      // each time piece is this much longer than the next
constexpr int64_t PIECE_TOKENS = 2048;    // sequence piece: >= 2048 tokens
constexpr int CHUNK = 64;
constexpr int MAX_DEVICES = 64;

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct Piece {
  int n0, n1;          // sequences (batch rows, or cu_seqlens entries) n0 .. n1-1
  int64_t t0, t1;      // tokens t0 .. t1-1 of each sequence (varlen: packed rows)
  int cu_off;          // varlen: first int of this piece's rebased offsets
};

struct Plan {
  bool varlen = false;  // pieces are ranges of packed sequences
  bool time_cut = false;
  int P = 0;
  Piece pc[MAX_PIECES];
  int64_t rows_per_seq = 0;                           // T (fixed-length batches)
  size_t rq = 0, rv = 0, ro = 0, rg = 0, state_seq = 0;  // bytes per row / sequence state
  size_t q[MAX_PIECES], v[MAX_PIECES], o[MAX_PIECES], g[MAX_PIECES];  // piece offsets
  size_t s[MAX_PIECES];                               // sequence pieces: state slice offset
  size_t reg_q = 0, reg_v = 0, reg_o = 0, reg_g = 0, reg_s = 0, reg_cu = 0;
  size_t off_q = 0, off_k = 0, off_v = 0, off_g = 0, off_beta = 0, off_o = 0;
  size_t off_s0 = 0, off_s1 = 0, off_cu = 0, off_ws = 0, ws_bytes = 0, total = 0;
  std::vector<int32_t> cu;                            // varlen: rebased offsets, all pieces
};

int64_t piece_rows(const Plan &L, const Piece &p) {
  return L.varlen ? (p.t1 - p.t0) : int64_t(p.n1 - p.n0) * (p.t1 - p.t0);
}

// Arguments of gdn_chunk_fwd for piece j; device pointers relative to `base`
// (nullptr while planning, when only sizes matter).
gdn_chunk_args piece_args(const gdn_chunk_args &a, const Plan &L, int j, unsigned char *base) {
  const Piece &p = L.pc[j];
  gdn_chunk_args d = a;
  // the pieces' state passes run one chain per sequence, as gdn_chunk_fwd
  // with segments = 1 does: a time cut hands the state on exactly as a chunk
  // boundary inside one chain does
  d.segments = 1;
  d.B = L.varlen ? 1 : p.n1 - p.n0;
  d.T = (int32_t)(p.t1 - p.t0);
  d.N = p.n1 - p.n0;
  d.cu_seqlens = L.varlen ? reinterpret_cast<const int32_t *>(base + L.off_cu) + p.cu_off
                          : nullptr;
  d.q = base + L.off_q + L.q[j];
  d.k = base + L.off_k + L.q[j];
  d.v = base + L.off_v + L.v[j];
  d.o = base + L.off_o + L.o[j];
  d.g = reinterpret_cast<const float *>(base + L.off_g + L.g[j]);
  d.beta = reinterpret_cast<const float *>(base + L.off_beta + L.g[j]);
  float *s0 = reinterpret_cast<float *>(base + L.off_s0);
  float *s1 = reinterpret_cast<float *>(base + L.off_s1);
  if (L.time_cut) {
    float *st[2] = {s0, s1};
    d.h0 = j == 0 ? (a.h0 ? s0 : nullptr) : st[j & 1];
    d.ht = (j + 1 < L.P || a.ht) ? st[(j + 1) & 1] : nullptr;
  } else {
    d.h0 = a.h0 ? reinterpret_cast<float *>(base + L.off_s0 + L.s[j]) : nullptr;
    d.ht = a.ht ? reinterpret_cast<float *>(base + L.off_s1 + L.s[j]) : nullptr;
  }
  d.workspace = base + L.off_ws;
  d.workspace_bytes = L.ws_bytes;
  return d;
}

// Chunk boundaries c[0..P] of the time pieces of a sequence of nc chunks.
// What is left once the last copy-in has landed (the last piece's kernels and
// its copy-out) is short because the last piece is short; earlier pieces grow
// by PIECE_GROWTH each, so that every piece's kernels finish while the next,
// shorter piece is still being copied in.  P is the largest count whose
// smallest piece still holds MIN_PIECE_CHUNKS chunks; 1 = no time cut.
int time_pieces(int nc, int *c) {
  int P = 0;
  double sum = 0.0, w = MIN_PIECE_CHUNKS;
  while (P < MAX_PIECES && sum + w <= nc) {
    sum += w;
    w *= PIECE_GROWTH;
    ++P;
  }
  if (P < 2) return 1;
  double W = 0.0;
  for (int j = 0; j < P; ++j) W += std::pow(PIECE_GROWTH, j);
  double acc = 0.0;
  c[0] = 0;
  for (int j = 0; j < P; ++j) {
    acc += std::pow(PIECE_GROWTH, P - 1 - j);
    c[j + 1] = (int)std::llround(nc * acc / W);
  }
  c[P] = nc;
  return P;
}

gdn_status_t make_plan(const gdn_chunk_args &a, Plan *L) {
  gdn_status_t st = check_gdn_chunk_sizes(a);
  if (st != GDN_OK) return st;
  const size_t elt = a.dtype == GDN_BF16 ? 2 : 4;
  L->rq = size_t(a.Hg) * a.K * elt;
  L->rv = size_t(a.H) * a.V * elt;
  L->ro = size_t(a.H) * a.V * (a.o_fp32 ? 4 : elt);
  L->rg = size_t(a.H) * 4;
  L->state_seq = size_t(a.H) * a.K * a.V * 4;
  L->varlen = a.cu_seqlens != nullptr;
  L->cu.clear();

  if (L->varlen) {
    const int32_t *cu = a.cu_seqlens;  // host memory
    if (cu[0] != 0 || cu[a.N] != a.T)
      return set_host_error(GDN_ERR_BAD_SEQLENS, "cu_seqlens must start at 0 and end at T");
    for (int n = 0; n < a.N; ++n)
      if (cu[n + 1] < cu[n])
        return set_host_error(GDN_ERR_BAD_SEQLENS, "cu_seqlens must not decrease");
    // cut at sequence ends into pieces of about T / P tokens
    int P = (int)std::min<int64_t>({(int64_t)MAX_PIECES, (int64_t)a.N, a.T / PIECE_TOKENS});
    P = std::max(P, 1);
    L->P = 0;
    int n0 = 0;
    for (int j = 0; j < P && n0 < a.N; ++j) {
      int n1 = a.N;
      if (j + 1 < P) {
        const int64_t goal = (int64_t)a.T * (j + 1) / P;
        n1 = n0 + 1;
        while (n1 < a.N && cu[n1] < goal) ++n1;
        if (a.N - n1 < 1) n1 = a.N;
      }
      Piece &p = L->pc[L->P++];
      p.n0 = n0; p.n1 = n1; p.t0 = cu[n0]; p.t1 = cu[n1];
      p.cu_off = (int)L->cu.size();
      for (int n = n0; n <= n1; ++n) L->cu.push_back(cu[n] - cu[n0]);
      while (L->cu.size() % 4) L->cu.push_back(0);  // 16-byte aligned next piece
      n0 = n1;
    }
  } else {
    L->rows_per_seq = a.T;
    const int nc = (a.T + CHUNK - 1) / CHUNK;
    int cb[MAX_PIECES + 1];
    const int Pt = time_pieces(nc, cb);
    if (Pt >= 2) {
      L->time_cut = true;
      L->P = Pt;
      for (int j = 0; j < Pt; ++j) {
        Piece &p = L->pc[j];
        p.n0 = 0; p.n1 = a.B; p.cu_off = 0;
        p.t0 = std::min<int64_t>((int64_t)CHUNK * cb[j], a.T);
        p.t1 = std::min<int64_t>((int64_t)CHUNK * cb[j + 1], a.T);
      }
    } else {
      const int64_t tokens = (int64_t)a.B * a.T;
      int P = (int)std::min<int64_t>({(int64_t)MAX_PIECES, (int64_t)a.B, tokens / PIECE_TOKENS});
      P = std::max(P, 1);
      L->P = P;
      for (int j = 0; j < P; ++j) {
        Piece &p = L->pc[j];
        p.n0 = (int)((int64_t)a.B * j / P);
        p.n1 = (int)((int64_t)a.B * (j + 1) / P);
        p.t0 = 0; p.t1 = a.T; p.cu_off = 0;
      }
    }
  }

  // regions: each piece's slice starts on a 256-byte boundary
  L->reg_q = L->reg_v = L->reg_o = L->reg_g = L->reg_s = 0;
  for (int j = 0; j < L->P; ++j) {
    const int64_t rows = piece_rows(*L, L->pc[j]);
    L->q[j] = L->reg_q; L->reg_q += align256(rows * L->rq);
    L->v[j] = L->reg_v; L->reg_v += align256(rows * L->rv);
    L->o[j] = L->reg_o; L->reg_o += align256(rows * L->ro);
    L->g[j] = L->reg_g; L->reg_g += align256(rows * L->rg);
    L->s[j] = L->reg_s; L->reg_s += align256(size_t(L->pc[j].n1 - L->pc[j].n0) * L->state_seq);
  }
  if (L->time_cut) L->reg_s = align256(size_t(a.N) * L->state_seq);
  L->reg_cu = align256(L->cu.size() * sizeof(int32_t));
  size_t off = 0;
  L->off_q = off; off += L->reg_q;
  L->off_k = off; off += L->reg_q;
  L->off_v = off; off += L->reg_v;
  L->off_o = off; off += L->reg_o;
  L->off_g = off; off += L->reg_g;
  L->off_beta = off; off += L->reg_g;
  L->off_s0 = off; off += L->reg_s;
  L->off_s1 = off; off += L->reg_s;
  L->off_cu = off; off += L->reg_cu;
  L->off_ws = off;
  L->ws_bytes = 0;
  for (int j = 0; j < L->P; ++j) {
    gdn_chunk_args d = piece_args(a, *L, j, nullptr);
    if (L->varlen) d.cu_seqlens = reinterpret_cast<const int32_t *>(a.cu_seqlens);  // non-NULL
    size_t need = 0;
    st = gdn_chunk_workspace_size(&d, &need);
    if (st != GDN_OK) return st;
    L->ws_bytes = std::max(L->ws_bytes, align256(need));
  }
  L->total = L->off_ws + L->ws_bytes;
  return GDN_OK;
}

// Internal copy streams and events of one device, made on first use and kept
// for the life of the process.
struct DeviceQueues {
  bool ready = false;
  int max_pitch = 0;
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, in_end = nullptr, out_end = nullptr;
  cudaEvent_t loaded[MAX_PIECES] = {}, computed[MAX_PIECES] = {};
};

std::mutex g_mu;
DeviceQueues g_q[MAX_DEVICES];

cudaError_t device_queues(DeviceQueues **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= MAX_DEVICES) return cudaErrorInvalidDevice;
  DeviceQueues &q = g_q[dev];
  if (!q.ready) {
    const unsigned fl = cudaEventDisableTiming;
    if ((e = cudaDeviceGetAttribute(&q.max_pitch, cudaDevAttrMaxPitch, dev)) != cudaSuccess ||
        (e = cudaStreamCreateWithFlags(&q.in, cudaStreamNonBlocking)) != cudaSuccess ||
        (e = cudaStreamCreateWithFlags(&q.out, cudaStreamNonBlocking)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&q.start, fl)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&q.in_end, fl)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&q.out_end, fl)) != cudaSuccess)
      return e;
    for (int j = 0; j < MAX_PIECES; ++j) {
      if ((e = cudaEventCreateWithFlags(&q.loaded[j], fl)) != cudaSuccess ||
          (e = cudaEventCreateWithFlags(&q.computed[j], fl)) != cudaSuccess)
        return e;
    }
    q.ready = true;
  }
  *out = &q;
  return cudaSuccess;
}

// `height` rows of `width` bytes, source rows `spitch` and destination rows
// `dpitch` bytes apart.
cudaError_t copy_rows(void *dst, size_t dpitch, const void *src, size_t spitch, size_t width,
                      size_t height, cudaMemcpyKind kind, cudaStream_t s, int max_pitch) {
  if (width == 0 || height == 0) return cudaSuccess;
  if (height == 1 || (dpitch == width && spitch == width))
    return cudaMemcpyAsync(dst, src, width * height, kind, s);
  if (dpitch <= (size_t)max_pitch && spitch <= (size_t)max_pitch)
    return cudaMemcpy2DAsync(dst, dpitch, src, spitch, width, height, kind, s);
  for (size_t r = 0; r < height; ++r) {
    cudaError_t e = cudaMemcpyAsync(static_cast<char *>(dst) + r * dpitch,
                                    static_cast<const char *>(src) + r * spitch, width, kind, s);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

bool is_device_memory(const void *p) {
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeDevice;
}

gdn_status_t cuda_fail(cudaError_t e, const char *what) {
  (void)cudaGetLastError();  // reported here, not by the caller's next CUDA call
  char msg[200];
  snprintf(msg, sizeof(msg), "%s: %s", what, cudaGetErrorString(e));
  return set_host_error(GDN_ERR_CUDA, msg);
}

}  // namespace
}  // namespace gdn

using namespace gdn;

extern "C" gdn_status_t gdn_chunk_host_workspace_size(const gdn_chunk_args *a, size_t *bytes) {
  if (a == nullptr || bytes == nullptr) return set_host_error(GDN_ERR_INVALID_ARG, "NULL argument");
  *bytes = 0;
  Plan L;
  gdn_status_t st = make_plan(*a, &L);
  if (st != GDN_OK) return st;
  *bytes = L.total;
  return GDN_OK;
}

extern "C" gdn_status_t gdn_chunk_fwd_host(const gdn_chunk_args *a, gdn_stream_t stream) {
  if (a == nullptr) return set_host_error(GDN_ERR_INVALID_ARG, "args is NULL");
  const struct { const void *p; const char *name; bool required; } host[] = {
      {a->q, "q", true}, {a->k, "k", true}, {a->v, "v", true}, {a->g, "g", true},
      {a->beta, "beta", true}, {a->o, "o", true}, {a->h0, "h0", false}, {a->ht, "ht", false},
      {a->cu_seqlens, "cu_seqlens", false}};
  char msg[96];
  for (const auto &h : host) {
    if (h.p == nullptr && h.required && a->T > 0) {  // T = 0: no token array is touched
      snprintf(msg, sizeof(msg), "%s must not be NULL", h.name);
      return set_host_error(GDN_ERR_INVALID_ARG, msg);
    }
  }
  Plan L;
  gdn_status_t st = make_plan(*a, &L);
  if (st != GDN_OK) return st;
  if (a->workspace == nullptr) return set_host_error(GDN_ERR_WORKSPACE, "workspace is NULL");
  if ((reinterpret_cast<uintptr_t>(a->workspace) & 255u) != 0)
    return set_host_error(GDN_ERR_MISALIGNED, "workspace is not 256-byte aligned");
  if (a->workspace_bytes < L.total) {
    snprintf(msg, sizeof(msg), "workspace of %zu bytes needed (got %zu)", L.total,
             a->workspace_bytes);
    return set_host_error(GDN_ERR_WORKSPACE, msg);
  }
  // first CUDA calls: where each pointer lives
  for (const auto &h : host) {
    if (h.p != nullptr && is_device_memory(h.p)) {
      snprintf(msg, sizeof(msg), "%s must be host memory", h.name);
      return set_host_error(GDN_ERR_INVALID_ARG, msg);
    }
  }
  if (!is_device_memory(a->workspace))
    return set_host_error(GDN_ERR_WORKSPACE, "workspace must be device memory");

  std::lock_guard<std::mutex> lock(g_mu);
  DeviceQueues *dq = nullptr;
  cudaError_t e = device_queues(&dq);
  if (e != cudaSuccess) return cuda_fail(e, "copy streams");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  unsigned char *base = static_cast<unsigned char *>(a->workspace);
  const char *hq = static_cast<const char *>(a->q), *hk = static_cast<const char *>(a->k);
  const char *hv = static_cast<const char *>(a->v);
  const char *hg = reinterpret_cast<const char *>(a->g);
  const char *hb = reinterpret_cast<const char *>(a->beta);
  char *ho = static_cast<char *>(a->o);
  const cudaMemcpyKind H2D = cudaMemcpyHostToDevice, D2H = cudaMemcpyDeviceToHost;
  const int mp = dq->max_pitch;

  // The copies wait for the work already on `stream` (it may still use the workspace).
  if ((e = cudaEventRecord(dq->start, s)) != cudaSuccess) return cuda_fail(e, "event record");
  if ((e = cudaStreamWaitEvent(dq->in, dq->start, 0)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(dq->out, dq->start, 0)) != cudaSuccess)
    return cuda_fail(e, "stream wait");

  gdn_status_t result = GDN_OK;
  const char *what = nullptr;
  auto ok = [&](cudaError_t err, const char *w) {
    if (err != cudaSuccess && e == cudaSuccess) { e = err; what = w; }
    return e == cudaSuccess && result == GDN_OK;
  };
  // The rebased offsets come from a pageable vector: cudaMemcpyAsync has
  // staged pageable host->device data by the time it returns.
  if (L.varlen)
    ok(cudaMemcpyAsync(base + L.off_cu, L.cu.data(), L.cu.size() * sizeof(int32_t), H2D, dq->in),
       "cu_seqlens copy");
  if (L.time_cut && a->h0)
    ok(cudaMemcpyAsync(base + L.off_s0, a->h0, size_t(a->N) * L.state_seq, H2D, dq->in),
       "h0 copy");

  const size_t T = (size_t)L.rows_per_seq;
  for (int j = 0; j < L.P && ok(cudaSuccess, nullptr); ++j) {
    const Piece &p = L.pc[j];
    const size_t height = L.varlen ? 1 : size_t(p.n1 - p.n0);
    const size_t first = L.varlen ? size_t(p.t0) : size_t(p.n0) * T + size_t(p.t0);
    const size_t len = size_t(p.t1 - p.t0);
    ok(copy_rows(base + L.off_q + L.q[j], len * L.rq, hq + first * L.rq, T * L.rq, len * L.rq,
                 height, H2D, dq->in, mp), "q copy");
    ok(copy_rows(base + L.off_k + L.q[j], len * L.rq, hk + first * L.rq, T * L.rq, len * L.rq,
                 height, H2D, dq->in, mp), "k copy");
    ok(copy_rows(base + L.off_v + L.v[j], len * L.rv, hv + first * L.rv, T * L.rv, len * L.rv,
                 height, H2D, dq->in, mp), "v copy");
    ok(copy_rows(base + L.off_g + L.g[j], len * L.rg, hg + first * L.rg, T * L.rg, len * L.rg,
                 height, H2D, dq->in, mp), "g copy");
    ok(copy_rows(base + L.off_beta + L.g[j], len * L.rg, hb + first * L.rg, T * L.rg,
                 len * L.rg, height, H2D, dq->in, mp), "beta copy");
    if (!L.time_cut && a->h0)
      ok(cudaMemcpyAsync(base + L.off_s0 + L.s[j],
                         reinterpret_cast<const char *>(a->h0) + size_t(p.n0) * L.state_seq,
                         size_t(p.n1 - p.n0) * L.state_seq, H2D, dq->in), "h0 copy");
    ok(cudaEventRecord(dq->loaded[j], dq->in), "event record");
    if (!ok(cudaStreamWaitEvent(s, dq->loaded[j], 0), "stream wait")) break;

    gdn_chunk_args d = piece_args(*a, L, j, base);
    result = gdn_chunk_fwd(&d, stream);
    if (result != GDN_OK) break;

    ok(cudaEventRecord(dq->computed[j], s), "event record");
    ok(cudaStreamWaitEvent(dq->out, dq->computed[j], 0), "stream wait");
    ok(copy_rows(ho + first * L.ro, T * L.ro, base + L.off_o + L.o[j], len * L.ro, len * L.ro,
                 height, D2H, dq->out, mp), "o copy");
    if (!L.time_cut && a->ht)
      ok(cudaMemcpyAsync(reinterpret_cast<char *>(a->ht) + size_t(p.n0) * L.state_seq,
                         base + L.off_s1 + L.s[j], size_t(p.n1 - p.n0) * L.state_seq, D2H,
                         dq->out), "ht copy");
  }
  if (L.time_cut && a->ht && ok(cudaSuccess, nullptr))
    ok(cudaMemcpyAsync(a->ht, base + ((L.P & 1) ? L.off_s1 : L.off_s0),
                       size_t(a->N) * L.state_seq, D2H, dq->out), "ht copy");

  // Join both copy streams back into `stream`, also after a failure, so that
  // nothing of this call is left running unordered.
  cudaError_t j1 = cudaEventRecord(dq->in_end, dq->in);
  cudaError_t j2 = cudaEventRecord(dq->out_end, dq->out);
  cudaError_t j3 = j1 == cudaSuccess ? cudaStreamWaitEvent(s, dq->in_end, 0) : j1;
  cudaError_t j4 = j2 == cudaSuccess ? cudaStreamWaitEvent(s, dq->out_end, 0) : j2;
  if (result != GDN_OK) return result;
  if (e != cudaSuccess) return cuda_fail(e, what ? what : "copy");
  if (j3 != cudaSuccess) return cuda_fail(j3, "join copy-in stream");
  if (j4 != cudaSuccess) return cuda_fail(j4, "join copy-out stream");
  return GDN_OK;
}
