/*
 * A plain C caller of libengram: a tiny bf16-table case (64 tokens in two sequences with lookback
 * rows and masked tokens; one layer of n-grams 2..3 with 4 heads, head_dim 64, hidden 256, hc 4)
 * run through engram_forward and through the four stage calls, which must agree bit for bit;
 * every id must fall in its head's bucket; engram_sync_status must report 0, then -3 after an
 * input id outside the token map. Prints "ok" and exits 0 on success.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "engram.h"

#define CK(x)                                                                      \
  do {                                                                             \
    cudaError_t e_ = (x);                                                          \
    if (e_ != cudaSuccess) {                                                       \
      fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));                     \
      return 1;                                                                    \
    }                                                                              \
  } while (0)
#define EK(x)                                                                      \
  do {                                                                             \
    int r_ = (x);                                                                  \
    if (r_ != 0) {                                                                 \
      fprintf(stderr, "%s -> %d: %s\n", #x, r_, engram_last_error());              \
      return 1;                                                                    \
    }                                                                              \
  } while (0)

static uint64_t g_state = 0x2545F4914F6CDD1Dull;
static uint64_t next_u64(void) { /* xorshift64 */
  g_state ^= g_state << 13;
  g_state ^= g_state >> 7;
  g_state ^= g_state << 17;
  return g_state;
}
static float uniform(float lo, float hi) { return lo + (hi - lo) * (float)((next_u64() >> 40) / 16777216.0); }
static uint16_t to_bf16(float f) { /* round to nearest even (finite inputs) */
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

enum { T = 64, S = 2, L = 1, MAXN = 3, HEADS = 4, C = (MAXN - 1) * HEADS, D = 64, H = 256, HC = 4 };
enum { K = C * D, N = (HC + 1) * H, RAW = 4096, VC = 1024 };

int main(void) {
  EngramDims dims = {L, MAXN, HEADS, D, H, HC, RAW, VC, 0, 1e-6f, 1e-6f};
  int64_t primes[L * C], offsets[L * C], rows[L];
  EK(engram_layout(4001, L, MAXN, HEADS, primes, offsets, rows));

  /* host inputs */
  int32_t token_map[RAW], input_ids[T], cu[S + 1] = {0, 40, T}, lookback[S * (MAXN - 1)];
  uint8_t mask[T];
  int64_t mult[L * MAXN];
  const int64_t bound = (INT64_MAX / (VC - 1)) / 2;
  for (int i = 0; i < RAW; ++i) token_map[i] = (int32_t)(next_u64() % VC);
  for (int t = 0; t < T; ++t) input_ids[t] = (int32_t)(next_u64() % RAW);
  for (int t = 0; t < T; ++t) mask[t] = (t % 17 == 5) ? 0 : 1;
  for (int i = 0; i < S * (MAXN - 1); ++i) lookback[i] = (i == 1) ? -1 : (int32_t)(next_u64() % VC);
  for (int i = 0; i < L * MAXN; ++i) mult[i] = 2 * (int64_t)(next_u64() % (uint64_t)bound) + 1;
  const int64_t R = rows[0];
  uint16_t* table = (uint16_t*)malloc((size_t)R * D * 2);
  uint16_t* wkv = (uint16_t*)malloc((size_t)N * K * 2);
  uint16_t qw[HC * H], kw[HC * H];
  float* streams = (float*)malloc((size_t)T * HC * H * 4);
  for (int64_t i = 0; i < R * D; ++i) table[i] = to_bf16(uniform(-0.05f, 0.05f));
  for (int64_t i = 0; i < (int64_t)N * K; ++i) wkv[i] = to_bf16(uniform(-0.03f, 0.03f));
  for (int i = 0; i < HC * H; ++i) {
    qw[i] = to_bf16(uniform(0.8f, 1.2f));
    kw[i] = to_bf16(uniform(0.8f, 1.2f));
  }
  for (int64_t i = 0; i < (int64_t)T * HC * H; ++i) streams[i] = uniform(-1.f, 1.f);

  /* device copies */
  int32_t *d_map, *d_ids_in, *d_cu, *d_lb, *d_ids_fwd, *d_ids_stg, *d_err;
  uint8_t* d_mask;
  int64_t *d_mult, *d_primes, *d_offsets;
  uint16_t *d_table, *d_wkv, *d_qw, *d_kw, *d_A;
  float *d_s_fwd, *d_s_stg, *d_kv;
  void* d_ws;
  const size_t ws_bytes = engram_forward_workspace_bytes(&dims, T);
  CK(cudaMalloc((void**)&d_map, sizeof(token_map)));
  CK(cudaMalloc((void**)&d_ids_in, sizeof(input_ids)));
  CK(cudaMalloc((void**)&d_cu, sizeof(cu)));
  CK(cudaMalloc((void**)&d_lb, sizeof(lookback)));
  CK(cudaMalloc((void**)&d_mask, sizeof(mask)));
  CK(cudaMalloc((void**)&d_mult, sizeof(mult)));
  CK(cudaMalloc((void**)&d_primes, sizeof(primes)));
  CK(cudaMalloc((void**)&d_offsets, sizeof(offsets)));
  CK(cudaMalloc((void**)&d_ids_fwd, (size_t)T * L * C * 4));
  CK(cudaMalloc((void**)&d_ids_stg, (size_t)T * L * C * 4));
  CK(cudaMalloc((void**)&d_err, 4));
  CK(cudaMalloc((void**)&d_table, (size_t)R * D * 2));
  CK(cudaMalloc((void**)&d_wkv, (size_t)N * K * 2));
  CK(cudaMalloc((void**)&d_qw, sizeof(qw)));
  CK(cudaMalloc((void**)&d_kw, sizeof(kw)));
  CK(cudaMalloc((void**)&d_A, (size_t)T * K * 2));
  CK(cudaMalloc((void**)&d_kv, (size_t)T * N * 4));
  CK(cudaMalloc((void**)&d_s_fwd, (size_t)T * HC * H * 4));
  CK(cudaMalloc((void**)&d_s_stg, (size_t)T * HC * H * 4));
  CK(cudaMalloc(&d_ws, ws_bytes));
  CK(cudaMemcpy(d_map, token_map, sizeof(token_map), cudaMemcpyHostToDevice));
  CK(cudaMemcpy(d_ids_in, input_ids, sizeof(input_ids), cudaMemcpyHostToDevice));
  CK(cudaMemcpy(d_cu, cu, sizeof(cu), cudaMemcpyHostToDevice));
  CK(cudaMemcpy(d_lb, lookback, sizeof(lookback), cudaMemcpyHostToDevice));
  CK(cudaMemcpy(d_mask, mask, sizeof(mask), cudaMemcpyHostToDevice));
  CK(cudaMemcpy(d_mult, mult, sizeof(mult), cudaMemcpyHostToDevice));
  CK(cudaMemcpy(d_primes, primes, sizeof(primes), cudaMemcpyHostToDevice));
  CK(cudaMemcpy(d_offsets, offsets, sizeof(offsets), cudaMemcpyHostToDevice));
  CK(cudaMemcpy(d_table, table, (size_t)R * D * 2, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(d_wkv, wkv, (size_t)N * K * 2, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(d_qw, qw, sizeof(qw), cudaMemcpyHostToDevice));
  CK(cudaMemcpy(d_kw, kw, sizeof(kw), cudaMemcpyHostToDevice));
  CK(cudaMemcpy(d_s_fwd, streams, (size_t)T * HC * H * 4, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(d_s_stg, streams, (size_t)T * HC * H * 4, cudaMemcpyHostToDevice));
  CK(cudaMemset(d_err, 0, 4));
  cudaStream_t st;
  CK(cudaStreamCreate(&st));

  /* the whole path in one call */
  EngramHashTables tabs = {d_map, d_mult, d_primes, d_offsets};
  EngramLayerWeights lw;
  memset(&lw, 0, sizeof(lw));
  lw.table_format = ENGRAM_TABLE_BF16;
  lw.table = d_table;
  lw.table_rows = R;
  lw.wkv = d_wkv;
  lw.q_weight = d_qw;
  lw.k_weight = d_kw;
  lw.wkv_format = ENGRAM_WKV_BF16;
  EngramTokens tok = {d_ids_in, T, d_cu, S, NULL, d_mask, d_lb};
  float* stream_ptrs[L] = {d_s_fwd};
  EK(engram_forward(&dims, &tabs, &lw, &tok, stream_ptrs, d_ws, ws_bytes, d_ids_fwd, d_err, st));

  /* the same through the stage calls */
  EK(engram_hash(&dims, d_ids_in, T, d_cu, S, NULL, d_mask, d_lb, d_map, d_mult, d_primes, d_offsets, d_ids_stg,
                 d_err, st));
  EK(engram_gather_dequant(ENGRAM_TABLE_BF16, d_ids_stg, L * C, T, C, D, d_table, NULL, R, d_A, d_err, st));
  EK(engram_project(d_A, d_wkv, d_kv, T, K, N, NULL, 0, d_err, st));
  EK(engram_gate(&dims, d_s_stg, d_kv, d_qw, d_kw, d_mask, T, d_err, st));
  EK(engram_sync_status(d_err, st));

  int32_t* ids_a = (int32_t*)malloc((size_t)T * L * C * 4);
  int32_t* ids_b = (int32_t*)malloc((size_t)T * L * C * 4);
  float* s_a = (float*)malloc((size_t)T * HC * H * 4);
  float* s_b = (float*)malloc((size_t)T * HC * H * 4);
  CK(cudaMemcpy(ids_a, d_ids_fwd, (size_t)T * L * C * 4, cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(ids_b, d_ids_stg, (size_t)T * L * C * 4, cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(s_a, d_s_fwd, (size_t)T * HC * H * 4, cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(s_b, d_s_stg, (size_t)T * HC * H * 4, cudaMemcpyDeviceToHost));
  if (memcmp(ids_a, ids_b, (size_t)T * L * C * 4) != 0) {
    fprintf(stderr, "ids differ between engram_forward and engram_hash\n");
    return 1;
  }
  for (int t = 0; t < T; ++t)
    for (int c = 0; c < C; ++c) {
      const int64_t id = ids_a[t * C + c];
      if (id < offsets[c] || id >= offsets[c] + primes[c]) {
        fprintf(stderr, "id %lld of token %d column %d outside its bucket\n", (long long)id, t, c);
        return 1;
      }
    }
  if (memcmp(s_a, s_b, (size_t)T * HC * H * 4) != 0) {
    fprintf(stderr, "streams differ between engram_forward and the stage calls\n");
    return 1;
  }
  int changed = 0, masked_same = 1;
  for (int t = 0; t < T; ++t)
    for (int i = 0; i < HC * H; ++i) {
      const int64_t j = (int64_t)t * HC * H + i;
      if (mask[t] && s_a[j] != streams[j]) changed = 1;
      if (!mask[t] && memcmp(&s_a[j], &streams[j], 4) != 0) masked_same = 0;
    }
  if (!changed || !masked_same) {
    fprintf(stderr, "gate: unmasked streams unchanged (%d) or masked streams changed (%d)\n", !changed,
            !masked_same);
    return 1;
  }

  /* a raw id outside the token map: hashed as pad_id, reported as ENGRAM_EDATA */
  input_ids[7] = RAW + 11;
  CK(cudaMemcpy(d_ids_in, input_ids, sizeof(input_ids), cudaMemcpyHostToDevice));
  EK(engram_hash(&dims, d_ids_in, T, d_cu, S, NULL, d_mask, d_lb, d_map, d_mult, d_primes, d_offsets, d_ids_stg,
                 d_err, st));
  const int rc = engram_sync_status(d_err, st);
  if (rc != ENGRAM_EDATA) {
    fprintf(stderr, "engram_sync_status after a bad raw id: %d, expected %d\n", rc, ENGRAM_EDATA);
    return 1;
  }
  CK(cudaStreamDestroy(st));
  printf("ok\n");
  return 0;
}
