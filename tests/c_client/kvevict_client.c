/* A plain C client of the kvevict C ABI (no Python): one handle driven through
 * the device-buffer path (prefill + decode + read_state), a second through the
 * host-buffer path (run_host) from malloc'd (pageable) memory and a third from
 * cudaMallocHost (page-locked) memory, on the same synthetic keys. Checks:
 *   - every call returns KVEVICT_OK and the error word stays clear;
 *   - each row keeps min(position, budget) rows, its sinks (positions
 *     0..n_sink-1) in place, positions strictly increasing;
 *   - scores are finite and non-negative, and the kept rows' scores sum to at
 *     most the number of tokens the row has seen (each step adds one softmax,
 *     of mass 1; evicted rows take theirs with them);
 *   - both host-buffer runs give the same evicted slots and the same state
 *     bit for bit as the device-buffer path;
 *   - a snapshot of the device-path handle (kvevict_save_state) loaded into a
 *     fresh handle reads back the same state bit for bit.
 * Exit status 0 on success. Build: gcc -std=c11 ... -lkvevict -lcudart. */
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "kvevict.h"

#define CHECK(call)                                                                     \
  do {                                                                                  \
    int rc_ = (call);                                                                   \
    if (rc_ != KVEVICT_OK) {                                                            \
      fprintf(stderr, "%s:%d %s -> %d (%s)\n", __FILE__, __LINE__, #call, rc_,          \
              kvevict_last_error());                                                    \
      return 1;                                                                         \
    }                                                                                   \
  } while (0)
#define CUDA(call)                                                                      \
  do {                                                                                  \
    cudaError_t e_ = (call);                                                            \
    if (e_ != cudaSuccess) {                                                            \
      fprintf(stderr, "%s:%d %s -> %s\n", __FILE__, __LINE__, #call, cudaGetErrorString(e_)); \
      return 1;                                                                         \
    }                                                                                   \
  } while (0)

enum { B = 2, L = 3, H = 2, D = 64, S = 90, T = 70, NSINK = 4, AVG = 40 };

/* fp32 -> fp16 bits, round to nearest even (normal range only; the keys here
 * stay well inside it) */
static uint16_t to_f16(float f) {
  uint32_t x;
  memcpy(&x, &f, 4);
  const uint32_t sign = (x >> 16) & 0x8000u;
  int32_t exp = (int32_t)((x >> 23) & 0xFF) - 127 + 15;
  uint32_t man = x & 0x7FFFFFu;
  if (exp <= 0) return (uint16_t)sign;          /* flush the tiny ones */
  uint32_t h = sign | ((uint32_t)exp << 10) | (man >> 13);
  const uint32_t rem = man & 0x1FFFu;
  if (rem > 0x1000u || (rem == 0x1000u && (h & 1u))) h += 1u;
  return (uint16_t)h;
}

/* deterministic pseudo-random keys in [-1, 1) (xorshift64*) */
static uint64_t state = 0x9E3779B97F4A7C15ull;
static float next_uniform(void) {
  state ^= state >> 12;
  state ^= state << 25;
  state ^= state >> 27;
  return (float)((state * 2685821657736338717ull) >> 40) / (float)(1u << 23) - 1.0f;
}

static int check_rows(kvevict_t* h, const int32_t* budgets, int64_t seen, uint16_t* keys,
                      float* sc, float* g, int32_t* pos, int32_t cap) {
  for (int b = 0; b < B; ++b)
    for (int l = 0; l < L; ++l)
      for (int hh = 0; hh < H; ++hh) {
        int32_t n = -1;
        CHECK(kvevict_read_state(h, b, l, hh, keys, sc, g, pos, &n, NULL));
        const int32_t want = (int32_t)(seen < budgets[l] ? seen : budgets[l]);
        if (n != want || n > cap) {
          fprintf(stderr, "row (%d,%d,%d): %d rows kept, expected %d\n", b, l, hh, n, want);
          return 1;
        }
        double sum = 0.0;
        for (int j = 0; j < n; ++j) {
          if (!(sc[j] >= 0.f) || !isfinite(sc[j])) {
            fprintf(stderr, "row (%d,%d,%d): score %d = %g\n", b, l, hh, j, sc[j]);
            return 1;
          }
          if (j < NSINK && pos[j] != j) {
            fprintf(stderr, "row (%d,%d,%d): sink %d holds position %d\n", b, l, hh, j, pos[j]);
            return 1;
          }
          if (j > 0 && pos[j] <= pos[j - 1]) {
            fprintf(stderr, "row (%d,%d,%d): positions not increasing at %d\n", b, l, hh, j);
            return 1;
          }
          sum += sc[j];
        }
        if (!(sum > 0.0) || sum > (double)seen * (1.0 + 1e-4)) {
          fprintf(stderr, "row (%d,%d,%d): scores sum to %g after %lld tokens\n", b, l, hh, sum,
                  (long long)seen);
          return 1;
        }
      }
  return 0;
}

int main(void) {
  kvevict_config cfg;
  memset(&cfg, 0, sizeof cfg);
  cfg.batch = B;
  cfg.n_layers = L;
  cfg.n_kv_heads = H;
  cfg.head_dim = D;
  cfg.avg_budget = AVG;
  cfg.pyramid_beta = 1.5;
  cfg.n_sink = NSINK;
  cfg.tau_init = 1.0f;
  cfg.tau_end = 2.0f;
  cfg.anneal_steps = S + T;
  cfg.rope_theta = 10000.0;
  cfg.seed = 42;
  cfg.max_prefill = S;

  int32_t budgets[L];
  CHECK(kvevict_budgets(L, AVG, NSINK, 1.5, budgets));
  int32_t cap = 0;
  for (int l = 0; l < L; ++l) cap = budgets[l] + 1 > cap ? budgets[l] + 1 : cap;

  const size_t npre = (size_t)B * L * H * S * D, ndec = (size_t)T * B * L * H * D;
  const size_t nev = (size_t)T * B * L * H;
  uint16_t* hpre = (uint16_t*)malloc(npre * 2);
  uint16_t* hdec = (uint16_t*)malloc(ndec * 2);
  int32_t* ev_dev_path = (int32_t*)malloc(nev * 4);
  int32_t* ev_host_path = (int32_t*)malloc(nev * 4);
  if (!hpre || !hdec || !ev_dev_path || !ev_host_path) return 1;
  for (size_t i = 0; i < npre; ++i) hpre[i] = to_f16(next_uniform());
  for (size_t i = 0; i < ndec; ++i) hdec[i] = to_f16(next_uniform());

  /* device-buffer path */
  uint16_t *dpre = NULL, *ddec = NULL;
  int32_t* dev = NULL;
  CUDA(cudaMalloc((void**)&dpre, npre * 2));
  CUDA(cudaMalloc((void**)&ddec, ndec * 2));
  CUDA(cudaMalloc((void**)&dev, nev * 4));
  CUDA(cudaMemcpy(dpre, hpre, npre * 2, cudaMemcpyHostToDevice));
  CUDA(cudaMemcpy(ddec, hdec, ndec * 2, cudaMemcpyHostToDevice));
  kvevict_t* h = NULL;
  CHECK(kvevict_create(&cfg, NULL, &h));
  CHECK(kvevict_prefill(h, dpre, S, NULL));
  CHECK(kvevict_decode(h, ddec, T, dev, NULL));
  CHECK(kvevict_check(h, NULL));
  int64_t p = 0;
  CHECK(kvevict_next_pos(h, &p));
  if (p != S + T) {
    fprintf(stderr, "next_pos %lld, expected %d\n", (long long)p, S + T);
    return 1;
  }
  CUDA(cudaMemcpy(ev_dev_path, dev, nev * 4, cudaMemcpyDeviceToHost));

  /* the decode kernel the library chose, and the other one forced: the same log */
  {
    int32_t kind = -1;
    CHECK(kvevict_decode_kernel_for(h, T, &kind));
    if (kind != KVEVICT_DECODE_STREAM && kind != KVEVICT_DECODE_RESIDENT) {
      fprintf(stderr, "decode_kernel_for returned %d\n", kind);
      return 1;
    }
    kvevict_config cfg2 = cfg;
    cfg2.decode_kernel = kind == KVEVICT_DECODE_STREAM ? KVEVICT_DECODE_RESIDENT : KVEVICT_DECODE_STREAM;
    kvevict_t* h2 = NULL;
    CHECK(kvevict_create(&cfg2, NULL, &h2));
    int32_t kind2 = -1;
    CHECK(kvevict_decode_kernel_for(h2, T, &kind2));
    if (kind2 != cfg2.decode_kernel) {
      fprintf(stderr, "forced decode kernel %d, got %d\n", cfg2.decode_kernel, kind2);
      return 1;
    }
    int32_t* ev_other = (int32_t*)malloc(nev * 4);
    if (!ev_other) return 1;
    CHECK(kvevict_prefill(h2, dpre, S, NULL));
    CHECK(kvevict_decode(h2, ddec, T, dev, NULL));
    CHECK(kvevict_check(h2, NULL));
    CUDA(cudaMemcpy(ev_other, dev, nev * 4, cudaMemcpyDeviceToHost));
    if (memcmp(ev_other, ev_dev_path, nev * 4) != 0) {
      fprintf(stderr, "the two decode kernels gave different eviction logs\n");
      return 1;
    }
    free(ev_other);
    CHECK(kvevict_destroy(h2));
    printf("decode kernels: the library's choice %s, the other one agrees\n",
           kind == KVEVICT_DECODE_RESIDENT ? "resident" : "streaming");
  }

  const size_t rowbuf = (size_t)cap;
  uint16_t* k1 = (uint16_t*)malloc(rowbuf * D * 2);
  uint16_t* k2 = (uint16_t*)malloc(rowbuf * D * 2);
  float *s1 = (float*)malloc(rowbuf * 4), *s2 = (float*)malloc(rowbuf * 4);
  float *g1 = (float*)malloc(rowbuf * 4), *g2 = (float*)malloc(rowbuf * 4);
  int32_t *p1 = (int32_t*)malloc(rowbuf * 4), *p2 = (int32_t*)malloc(rowbuf * 4);
  if (check_rows(h, budgets, S + T, k1, s1, g1, p1, cap)) return 1;

  /* host-buffer path on a second handle (pageable buffers) and a third
   * (page-locked buffers): same keys, same results */
  uint16_t *lpre = NULL, *ldec = NULL;
  int32_t* ev_locked = NULL;
  CUDA(cudaMallocHost((void**)&lpre, npre * 2));
  CUDA(cudaMallocHost((void**)&ldec, ndec * 2));
  CUDA(cudaMallocHost((void**)&ev_locked, nev * 4));
  memcpy(lpre, hpre, npre * 2);
  memcpy(ldec, hdec, ndec * 2);
  memset(ev_locked, 0xff, nev * 4);
  kvevict_t* hosts[2] = {NULL, NULL};
  for (int v = 0; v < 2; ++v) {
    int32_t* ev_out = v == 0 ? ev_host_path : ev_locked;
    CHECK(kvevict_create(&cfg, NULL, &hosts[v]));
    CHECK(kvevict_run_host(hosts[v], v == 0 ? hpre : lpre, S, v == 0 ? hdec : ldec, T, ev_out, NULL));
    if (memcmp(ev_dev_path, ev_out, nev * 4) != 0) {
      fprintf(stderr, "run_host (%s memory) evicted other slots than the device path\n",
              v == 0 ? "pageable" : "page-locked");
      return 1;
    }
    for (int b = 0; b < B; ++b)
      for (int l = 0; l < L; ++l)
        for (int hh = 0; hh < H; ++hh) {
          int32_t n1 = 0, n2 = 0;
          CHECK(kvevict_read_state(h, b, l, hh, k1, s1, g1, p1, &n1, NULL));
          CHECK(kvevict_read_state(hosts[v], b, l, hh, k2, s2, g2, p2, &n2, NULL));
          if (n1 != n2 || memcmp(k1, k2, (size_t)n1 * D * 2) || memcmp(s1, s2, (size_t)n1 * 4) ||
              memcmp(g1, g2, (size_t)n1 * 4) || memcmp(p1, p2, (size_t)n1 * 4)) {
            fprintf(stderr, "row (%d,%d,%d): run_host (%s memory) state differs\n", b, l, hh,
                    v == 0 ? "pageable" : "page-locked");
            return 1;
          }
        }
  }
  kvevict_t* h2 = hosts[0];

  /* checkpoint: snapshot the device-path handle, load it into a fresh one */
  size_t snap_bytes = 0;
  CHECK(kvevict_state_bytes(h, &snap_bytes));
  unsigned char* snap = (unsigned char*)malloc(snap_bytes);
  if (!snap) return 1;
  CHECK(kvevict_save_state(h, snap, snap_bytes, NULL));
  kvevict_t* h4 = NULL;
  CHECK(kvevict_create(&cfg, NULL, &h4));
  CHECK(kvevict_load_state(h4, snap, snap_bytes, NULL));
  free(snap);
  int64_t p4 = 0;
  CHECK(kvevict_next_pos(h4, &p4));
  if (p4 != S + T) {
    fprintf(stderr, "loaded next_pos %lld, expected %d\n", (long long)p4, S + T);
    return 1;
  }
  for (int b = 0; b < B; ++b)
    for (int l = 0; l < L; ++l)
      for (int hh = 0; hh < H; ++hh) {
        int32_t n1 = 0, n2 = 0;
        CHECK(kvevict_read_state(h, b, l, hh, k1, s1, g1, p1, &n1, NULL));
        CHECK(kvevict_read_state(h4, b, l, hh, k2, s2, g2, p2, &n2, NULL));
        if (n1 != n2 || memcmp(k1, k2, (size_t)n1 * D * 2) || memcmp(s1, s2, (size_t)n1 * 4) ||
            memcmp(g1, g2, (size_t)n1 * 4) || memcmp(p1, p2, (size_t)n1 * 4)) {
          fprintf(stderr, "row (%d,%d,%d): loaded snapshot differs\n", b, l, hh);
          return 1;
        }
      }
  CHECK(kvevict_destroy(h4));

  /* an invalid call is refused with a message, and the handle keeps working */
  if (kvevict_prefill(h, dpre, S, NULL) != KVEVICT_ERR_BAD_STATE || kvevict_last_error()[0] == '\0') {
    fprintf(stderr, "prefill after decode was not refused as BAD_STATE\n");
    return 1;
  }
  CHECK(kvevict_reset(h, NULL));
  CHECK(kvevict_prefill(h, dpre, S, NULL));
  CHECK(kvevict_check(h, NULL));

  CHECK(kvevict_destroy(h));
  CHECK(kvevict_destroy(h2));
  CHECK(kvevict_destroy(hosts[1]));
  cudaFreeHost(lpre);
  cudaFreeHost(ldec);
  cudaFreeHost(ev_locked);
  cudaFree(dpre);
  cudaFree(ddec);
  cudaFree(dev);
  printf("kvevict C client: ok (%d rows, %d prompt + %d decode steps)\n", B * L * H, S, T);
  return 0;
}
