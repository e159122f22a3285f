/*
 * A plain C caller of the library, with no Python or PyTorch in the process:
 * the chunked GDN forward through gdn_chunk_fwd (device buffers the program
 * allocates itself) and through gdn_chunk_fwd_host (host buffers).
 *
 * usage: c_abi_program <in.bin> <out_device.bin> <out_host.bin>
 *   in.bin:  int32 B, T, H, Hg, K, V; float32 scale; then q, k [B,T,Hg,K] and
 *            v [B,T,H,V] as bf16 bit patterns (uint16), g, beta [B,T,H] and
 *            h0 [B,H,K,V] as float32
 *   out_*:   o [B,T,H,V] as bf16 bit patterns, then ht [B,H,K,V] as float32
 * Exit status 0 when every call returned GDN_OK and the device error word is
 * clear; otherwise a message on stderr and status 1.
 */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "gdn.h"

static int fail(const char *what, const char *detail) {
  fprintf(stderr, "c_abi_program: %s: %s\n", what, detail ? detail : "");
  return 1;
}

#define CUDA_OK(call)                                              \
  do {                                                             \
    cudaError_t e_ = (call);                                       \
    if (e_ != cudaSuccess) return fail(#call, cudaGetErrorString(e_)); \
  } while (0)

#define GDN_OK_OR_FAIL(call)                                       \
  do {                                                             \
    gdn_status_t s_ = (call);                                      \
    if (s_ != GDN_OK) return fail(#call, gdn_last_error_message()); \
  } while (0)

static void *read_exact(FILE *f, size_t bytes) {
  void *p = malloc(bytes ? bytes : 1);
  if (p && fread(p, 1, bytes, f) != bytes) {
    free(p);
    return NULL;
  }
  return p;
}

static int write_out(const char *path, const void *o, size_t o_bytes, const void *ht,
                     size_t ht_bytes) {
  FILE *f = fopen(path, "wb");
  if (!f) return fail("open output", path);
  int bad = fwrite(o, 1, o_bytes, f) != o_bytes || fwrite(ht, 1, ht_bytes, f) != ht_bytes;
  if (fclose(f) != 0 || bad) return fail("write output", path);
  return 0;
}

int main(int argc, char **argv) {
  if (argc != 4) return fail("usage", "c_abi_program <in.bin> <out_device.bin> <out_host.bin>");
  FILE *f = fopen(argv[1], "rb");
  if (!f) return fail("open input", argv[1]);
  int32_t dims[6];
  float scale;
  if (fread(dims, sizeof(int32_t), 6, f) != 6 || fread(&scale, sizeof(float), 1, f) != 1)
    return fail("read input", "header");
  const size_t B = dims[0], T = dims[1], H = dims[2], Hg = dims[3], K = dims[4], V = dims[5];
  const size_t n_qk = B * T * Hg * K, n_v = B * T * H * V, n_g = B * T * H, n_s = B * H * K * V;
  uint16_t *q = read_exact(f, n_qk * 2), *k = read_exact(f, n_qk * 2), *v = read_exact(f, n_v * 2);
  float *g = read_exact(f, n_g * 4), *beta = read_exact(f, n_g * 4), *h0 = read_exact(f, n_s * 4);
  fclose(f);
  if (!q || !k || !v || !g || !beta || !h0) return fail("read input", "arrays");
  uint16_t *o = malloc(n_v * 2);
  float *ht = malloc(n_s * 4);
  if (!o || !ht) return fail("malloc", "outputs");

  /* 1. device buffers, gdn_chunk_fwd */
  void *dq, *dk, *dv, *dg, *db, *dh0, *dht, *dout, *ws = NULL;
  CUDA_OK(cudaMalloc(&dq, n_qk * 2));
  CUDA_OK(cudaMalloc(&dk, n_qk * 2));
  CUDA_OK(cudaMalloc(&dv, n_v * 2));
  CUDA_OK(cudaMalloc(&dg, n_g * 4));
  CUDA_OK(cudaMalloc(&db, n_g * 4));
  CUDA_OK(cudaMalloc(&dh0, n_s * 4));
  CUDA_OK(cudaMalloc(&dht, n_s * 4));
  CUDA_OK(cudaMalloc(&dout, n_v * 2));
  CUDA_OK(cudaMemcpy(dq, q, n_qk * 2, cudaMemcpyHostToDevice));
  CUDA_OK(cudaMemcpy(dk, k, n_qk * 2, cudaMemcpyHostToDevice));
  CUDA_OK(cudaMemcpy(dv, v, n_v * 2, cudaMemcpyHostToDevice));
  CUDA_OK(cudaMemcpy(dg, g, n_g * 4, cudaMemcpyHostToDevice));
  CUDA_OK(cudaMemcpy(db, beta, n_g * 4, cudaMemcpyHostToDevice));
  CUDA_OK(cudaMemcpy(dh0, h0, n_s * 4, cudaMemcpyHostToDevice));

  gdn_chunk_args a;
  memset(&a, 0, sizeof(a));
  a.dtype = GDN_BF16;
  a.q = dq; a.k = dk; a.v = dv; a.g = dg; a.beta = db; a.h0 = dh0; a.ht = dht; a.o = dout;
  a.cu_seqlens = NULL;
  a.B = (int32_t)B; a.T = (int32_t)T; a.H = (int32_t)H; a.Hg = (int32_t)Hg;
  a.K = (int32_t)K; a.V = (int32_t)V; a.N = (int32_t)B;
  a.chunk_size = 64;
  a.g_is_cumsum = 0;
  a.scale = scale;
  a.segments = 1; /* one chain per sequence, as the host entry point runs it */
  size_t ws_bytes = 0;
  GDN_OK_OR_FAIL(gdn_chunk_workspace_size(&a, &ws_bytes));
  if (ws_bytes) CUDA_OK(cudaMalloc(&ws, ws_bytes));
  a.workspace = ws;
  a.workspace_bytes = ws_bytes;
  GDN_OK_OR_FAIL(gdn_chunk_fwd(&a, NULL));
  CUDA_OK(cudaDeviceSynchronize());
  int32_t code = -1;
  GDN_OK_OR_FAIL(gdn_check_device_error(NULL, &code));
  if (code != GDN_OK) return fail("device error word", gdn_status_string((gdn_status_t)code));
  CUDA_OK(cudaMemcpy(o, dout, n_v * 2, cudaMemcpyDeviceToHost));
  CUDA_OK(cudaMemcpy(ht, dht, n_s * 4, cudaMemcpyDeviceToHost));
  if (write_out(argv[2], o, n_v * 2, ht, n_s * 4)) return 1;

  /* 2. host buffers (pageable), gdn_chunk_fwd_host */
  memset(o, 0, n_v * 2);
  memset(ht, 0, n_s * 4);
  gdn_chunk_args h = a;
  h.q = q; h.k = k; h.v = v; h.g = g; h.beta = beta; h.h0 = h0; h.ht = ht; h.o = o;
  h.workspace = NULL;
  h.workspace_bytes = 0;
  size_t hws_bytes = 0;
  void *hws = NULL;
  GDN_OK_OR_FAIL(gdn_chunk_host_workspace_size(&h, &hws_bytes));
  CUDA_OK(cudaMalloc(&hws, hws_bytes));
  h.workspace = hws;
  h.workspace_bytes = hws_bytes;
  GDN_OK_OR_FAIL(gdn_chunk_fwd_host(&h, NULL));
  CUDA_OK(cudaDeviceSynchronize());
  GDN_OK_OR_FAIL(gdn_check_device_error(NULL, &code));
  if (code != GDN_OK) return fail("device error word", gdn_status_string((gdn_status_t)code));
  if (write_out(argv[3], o, n_v * 2, ht, n_s * 4)) return 1;

  cudaFree(dq); cudaFree(dk); cudaFree(dv); cudaFree(dg); cudaFree(db);
  cudaFree(dh0); cudaFree(dht); cudaFree(dout); cudaFree(ws); cudaFree(hws);
  free(q); free(k); free(v); free(g); free(beta); free(h0); free(o); free(ht);
  return 0;
}
