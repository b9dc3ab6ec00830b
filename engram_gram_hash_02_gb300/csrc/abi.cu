// The extern "C" boundary of libengram: argument checks, error reporting, and the forward
// pass that chains hash -> (gather -> project -> gate) per layer on one stream.
#include <stdarg.h>
#include <stdio.h>

#include <atomic>
#include <mutex>
#include <string>

#include "internal.cuh"

namespace engram {

static thread_local std::string g_last_error;

void set_error(const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
}

int fail_cuda(cudaError_t e, const char* what) {
  set_error("%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
  return ENGRAM_ECUDA;
}

int num_sms() {
  static std::atomic<int> cache[64];        // zero-initialised (static storage); 0 = not read yet
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cache[dev].store(n, std::memory_order_relaxed);   // every thread stores the same value
  }
  return n;
}

void* PerContextOnce::current_context() {
  typedef int (*CtxGetCurrentFn)(void**);
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  void* ctx = nullptr;
  if (fn == nullptr || fn(&ctx) != 0) return nullptr;
  return ctx;
}

void set_gemm_bn_override(int bn);
void set_gemm_mx_bn_override(int bn);
void set_gemm_schedule_override(int s);

static int check_dims(const EngramDims* d, bool need_hash, bool need_gate) {
  ENGRAM_CHECK_ARG(d != nullptr, "dims is NULL");
  if (need_hash) {
    ENGRAM_CHECK_ARG(d->layers >= 1, "layers must be >= 1 (got %d)", d->layers);
    ENGRAM_CHECK_ARG(d->max_ngram >= 2 && d->max_ngram <= 8, "max_ngram must be in [2, 8] (got %d)", d->max_ngram);
    ENGRAM_CHECK_ARG(d->n_heads >= 1, "n_heads must be >= 1 (got %d)", d->n_heads);
    ENGRAM_CHECK_ARG((int64_t)d->layers * (d->max_ngram - 1) * d->n_heads <= 256,
                     "layers * n_hash_cols must be <= 256");
    ENGRAM_CHECK_ARG(d->raw_vocab >= 1, "raw_vocab must be >= 1");
    ENGRAM_CHECK_ARG(d->compressed_vocab >= 1, "compressed_vocab must be >= 1");
    ENGRAM_CHECK_ARG(d->pad_id >= 0 && d->pad_id < d->compressed_vocab, "pad_id %d outside [0, %d)", d->pad_id,
                     d->compressed_vocab);
  }
  if (need_gate) {
    ENGRAM_CHECK_ARG(d->hidden >= 8 && d->hidden <= 8192 && d->hidden % 8 == 0,
                     "hidden must be a multiple of 8 in [8, 8192] (got %d)", d->hidden);
    ENGRAM_CHECK_ARG(d->hc >= 1 && d->hc <= 8, "hc must be in [1, 8] (got %d)", d->hc);
    ENGRAM_CHECK_ARG(d->eps >= 0.f, "eps must be >= 0");
    ENGRAM_CHECK_ARG(d->clamp >= 0.f, "clamp must be >= 0");
  }
  return ENGRAM_OK;
}

static int check_gather(int32_t fmt, const int32_t* ids, int64_t ids_stride_t, int64_t T, int32_t C,
                        int32_t D, const void* table, const uint8_t* scales, int64_t num_rows,
                        const uint16_t* out) {
  ENGRAM_CHECK_ARG(T >= 0, "T must be >= 0");
  ENGRAM_CHECK_ARG(C >= 1, "C must be >= 1");
  ENGRAM_CHECK_ARG(ids_stride_t >= C, "ids_stride_t (%lld) must be >= C (%d)", (long long)ids_stride_t, C);
  ENGRAM_CHECK_ARG(num_rows >= 0, "num_rows must be >= 0");
  ENGRAM_CHECK_ARG(ids != nullptr && table != nullptr && out != nullptr, "ids, table and out must be non-NULL");
  ENGRAM_CHECK_ARG(aligned(out, 16), "out must be 16-byte aligned");
  switch (fmt) {
    case ENGRAM_TABLE_FP8_E8M0:
      ENGRAM_CHECK_ARG(D >= 32 && D % 32 == 0, "FP8 head_dim must be a multiple of 32 (got %d)", D);
      ENGRAM_CHECK_ARG(scales != nullptr, "FP8 table needs scales");
      ENGRAM_CHECK_ARG(aligned(table, 16), "FP8 table must be 16-byte aligned");
      break;
    case ENGRAM_TABLE_Q2K:
      ENGRAM_CHECK_ARG(D == 256, "Q2_K rows are 256 wide (got head_dim %d)", D);
      ENGRAM_CHECK_ARG(aligned(table, 4), "Q2_K table must be 4-byte aligned");
      break;
    case ENGRAM_TABLE_BF16:
      ENGRAM_CHECK_ARG(D >= 8 && D % 8 == 0, "bf16 head_dim must be a multiple of 8 (got %d)", D);
      ENGRAM_CHECK_ARG(aligned(table, 16), "bf16 table must be 16-byte aligned");
      break;
    default:
      ENGRAM_CHECK_ARG(false, "unknown table format %d", fmt);
  }
  return ENGRAM_OK;
}

static int check_project(const uint16_t* A, const uint16_t* wkv, const float* kv, int64_t T, int32_t K,
                         int32_t N) {
  ENGRAM_CHECK_ARG(T >= 0 && T < (int64_t)1 << 31, "T must be in [0, 2^31)");
  ENGRAM_CHECK_ARG(K >= 8 && K % 8 == 0, "K must be a positive multiple of 8 (got %d)", K);
  ENGRAM_CHECK_ARG(N >= 16 && N % 16 == 0, "N must be a positive multiple of 16 (got %d)", N);
  ENGRAM_CHECK_ARG(A != nullptr && wkv != nullptr && kv != nullptr, "A, wkv and kv must be non-NULL");
  ENGRAM_CHECK_ARG(aligned(A, 16) && aligned(wkv, 16) && aligned(kv, 16), "A, wkv and kv must be 16-byte aligned");
  return ENGRAM_OK;
}

static int check_gate(const EngramDims* d, const float* streams, const float* kv, const uint16_t* qw,
                      const uint16_t* kw, int64_t T) {
  int rc = check_dims(d, false, true);
  if (rc) return rc;
  ENGRAM_CHECK_ARG(T >= 0 && T < (int64_t)1 << 31, "T must be in [0, 2^31)");
  ENGRAM_CHECK_ARG(streams && kv && qw && kw, "streams, kv, q_weight and k_weight must be non-NULL");
  ENGRAM_CHECK_ARG(aligned(streams, 16) && aligned(kv, 16) && aligned(qw, 16) && aligned(kw, 16),
                   "streams, kv, q_weight and k_weight must be 16-byte aligned");
  return ENGRAM_OK;
}

static size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace engram

using namespace engram;

extern "C" {

const char* engram_last_error(void) { return g_last_error.c_str(); }

int engram_sync_status(const int32_t* err_flag, engram_stream_t stream) {
  ENGRAM_CHECK_ARG(err_flag != nullptr && aligned(err_flag, 4), "engram_sync_status: err_flag must be a non-NULL, "
                   "4-byte aligned device word");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, err_flag, sizeof(v), cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return fail_cuda(e, "engram_sync_status: read of err_flag");
  e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return fail_cuda(e, "engram_sync_status: stream");
  if (v & ENGRAM_ERR_PIPE_TIMEOUT) {
    set_error("engram_sync_status: a pipeline wait ran past its time limit (err_flag 0x%x): results invalid", v);
    return ENGRAM_ECUDA;
  }
  if (v != 0) {
    set_error("engram_sync_status: err_flag 0x%x:%s%s%s", v,
              (v & ENGRAM_ERR_RAW_ID) ? " raw id outside the token map (hashed as pad_id);" : "",
              (v & ENGRAM_ERR_ROW_ID) ? " row id outside the table (zero row);" : "",
              (v & ~(ENGRAM_ERR_RAW_ID | ENGRAM_ERR_ROW_ID)) ? " unknown bits;" : "");
    return ENGRAM_EDATA;
  }
  return ENGRAM_OK;
}

int engram_project_plan(int64_t T, int32_t K, int32_t N, int32_t wkv_format, int32_t num_sms,
                        EngramProjectPlan* out) {
  ENGRAM_CHECK_ARG(out != nullptr, "engram_project_plan: out is NULL");
  ENGRAM_CHECK_ARG(T >= 1 && T < (int64_t)1 << 31, "engram_project_plan: T must be in [1, 2^31)");
  ENGRAM_CHECK_ARG(N >= 16 && N % 16 == 0, "engram_project_plan: N must be a positive multiple of 16");
  ENGRAM_CHECK_ARG(num_sms >= 1 && num_sms <= 1024, "engram_project_plan: num_sms must be in [1, 1024]");
  bool ok;
  if (wkv_format == ENGRAM_WKV_BF16) {
    ENGRAM_CHECK_ARG(K >= 8 && K % 8 == 0, "engram_project_plan: K must be a positive multiple of 8");
    ok = gemm_plan_info(T, K, N, num_sms, out);
  } else if (wkv_format == ENGRAM_WKV_MXFP8) {
    ENGRAM_CHECK_ARG(K >= 128 && K % 128 == 0, "engram_project_plan: MXFP8 K must be a positive multiple of 128");
    ok = gemm_mx_plan_info(T, K, N, num_sms, out);
  } else {
    ENGRAM_CHECK_ARG(false, "engram_project_plan: unknown wkv format %d", wkv_format);
  }
  ENGRAM_CHECK_ARG(ok, "engram_project_plan: no tile plan fits (T %lld, K %d, N %d)", (long long)T, K, N);
  return ENGRAM_OK;
}
const char* engram_version(void) { return "libengram 0.1 (sm_103a)"; }

void engram_set_gemm_tile(int32_t bn) {
  set_gemm_bn_override((bn >= 16 && bn <= 256 && bn % 16 == 0) ? bn : 0);
}

void engram_set_gemm_schedule(int32_t s) { set_gemm_schedule_override((s == 1 || s == 2) ? s : 0); }

size_t engram_project_workspace_bytes(int64_t T, int32_t K, int32_t N) {
  if (T <= 0 || T >= ((int64_t)1 << 31) || K < 8 || K % 8 != 0 || N < 16 || N % 16 != 0) return 0;
  return gemm_workspace_bytes(T, K, N);
}

// Checks the hash arguments and fills its launch parameters (rc != 0: nothing to launch; T == 0
// returns ENGRAM_OK with p.T == 0).
static int hash_params(const EngramDims* dims, const int32_t* input_ids, int64_t T, const int32_t* cu_seqlens,
                       int32_t S, const int32_t* sequence_ids, const uint8_t* token_mask, const int32_t* lookback_ids,
                       const int32_t* token_map, const int64_t* multipliers, const int64_t* primes,
                       const int64_t* offsets, int32_t* out_ids, int32_t* err_flag, HashParams& p) {
  p = HashParams{};
  int rc = check_dims(dims, true, false);
  if (rc) return rc;
  ENGRAM_CHECK_ARG(T >= 0 && T < (int64_t)1 << 34, "T must be in [0, 2^34)");
  if (T == 0) return ENGRAM_OK;
  ENGRAM_CHECK_ARG(input_ids && token_map && multipliers && primes && offsets && out_ids,
                   "input_ids, token_map, multipliers, primes, offsets and out_ids must be non-NULL");
  if (cu_seqlens != nullptr) {
    ENGRAM_CHECK_ARG(S >= 1, "cu_seqlens given with S = %d", S);
  } else {
    S = 1;
  }
  p.input_ids = input_ids;
  p.cu_seqlens = cu_seqlens;
  p.sequence_ids = sequence_ids;
  p.token_mask = token_mask;
  p.lookback_ids = lookback_ids;
  p.token_map = token_map;
  p.multipliers = multipliers;
  p.primes = primes;
  p.offsets = offsets;
  p.out = out_ids;
  p.err = err_flag;
  p.T = T;
  p.S = S;
  p.layers = dims->layers;
  p.max_ngram = dims->max_ngram;
  p.n_heads = dims->n_heads;
  p.cols = (dims->max_ngram - 1) * dims->n_heads;
  p.raw_vocab = dims->raw_vocab;
  p.pad_id = dims->pad_id;
  return ENGRAM_OK;
}

static int hash_impl(const EngramDims* dims, const int32_t* input_ids, int64_t T, const int32_t* cu_seqlens,
                     int32_t S, const int32_t* sequence_ids, const uint8_t* token_mask, const int32_t* lookback_ids,
                     const int32_t* token_map, const int64_t* multipliers, const int64_t* primes,
                     const int64_t* offsets, int32_t* out_ids, int32_t* err_flag, engram_stream_t stream, bool pdl) {
  HashParams p;
  int rc = hash_params(dims, input_ids, T, cu_seqlens, S, sequence_ids, token_mask, lookback_ids, token_map,
                       multipliers, primes, offsets, out_ids, err_flag, p);
  if (rc || T == 0) return rc;
  cudaError_t e = launch_hash(p, static_cast<cudaStream_t>(stream), pdl);
  return e == cudaSuccess ? ENGRAM_OK : fail_cuda(e, "engram_hash: launch");
}

int engram_hash(const EngramDims* dims, const int32_t* input_ids, int64_t T, const int32_t* cu_seqlens,
                int32_t S, const int32_t* sequence_ids, const uint8_t* token_mask, const int32_t* lookback_ids,
                const int32_t* token_map, const int64_t* multipliers, const int64_t* primes,
                const int64_t* offsets, int32_t* out_ids, int32_t* err_flag, engram_stream_t stream) {
  return hash_impl(dims, input_ids, T, cu_seqlens, S, sequence_ids, token_mask, lookback_ids, token_map, multipliers,
                   primes, offsets, out_ids, err_flag, stream, false);
}

static int gather_impl(int32_t fmt, const int32_t* ids, int64_t ids_stride_t, int64_t T, int32_t C,
                       int32_t head_dim, const void* table, const uint8_t* scales, int64_t num_rows, uint16_t* out,
                       int32_t* err_flag, engram_stream_t stream, bool pdl) {
  if (T == 0) return ENGRAM_OK;
  int rc = check_gather(fmt, ids, ids_stride_t, T, C, head_dim, table, scales, num_rows, out);
  if (rc) return rc;
  GatherParams p{fmt, ids, ids_stride_t, T, C, head_dim, table, scales, num_rows, out, err_flag};
  cudaError_t e = launch_gather(p, static_cast<cudaStream_t>(stream), pdl);
  return e == cudaSuccess ? ENGRAM_OK : fail_cuda(e, "engram_gather_dequant: launch");
}

int engram_gather_dequant(int32_t fmt, const int32_t* ids, int64_t ids_stride_t, int64_t T, int32_t C,
                          int32_t head_dim, const void* table, const uint8_t* scales, int64_t num_rows,
                          uint16_t* out, int32_t* err_flag, engram_stream_t stream) {
  return gather_impl(fmt, ids, ids_stride_t, T, C, head_dim, table, scales, num_rows, out, err_flag, stream, false);
}

static int project_impl(const uint16_t* A, const uint16_t* wkv, float* kv, int64_t T, int32_t K, int32_t N,
                        void* workspace, size_t ws_bytes, int32_t* err_flag, engram_stream_t stream, bool pdl,
                        const GateFuse* gf = nullptr, const GateOverlap* go = nullptr) {
  if (T == 0) return ENGRAM_OK;
  int rc = check_project(A, wkv, kv, T, K, N);
  if (rc) return rc;
  ENGRAM_CHECK_ARG(workspace == nullptr || aligned(workspace, 256), "engram_project: workspace must be 256-byte aligned");
  GemmParams p{A, wkv, kv, T, K, N, err_flag, workspace, workspace != nullptr ? ws_bytes : 0};
  if (gf != nullptr) p.gf = *gf;
  if (go != nullptr) p.go = *go;
  return launch_gemm(p, static_cast<cudaStream_t>(stream), pdl);
}

int engram_project(const uint16_t* A, const uint16_t* wkv, float* kv, int64_t T, int32_t K, int32_t N,
                   void* workspace, size_t ws_bytes, int32_t* err_flag, engram_stream_t stream) {
  return project_impl(A, wkv, kv, T, K, N, workspace, ws_bytes, err_flag, stream, false);
}

static int gate_impl(const EngramDims* dims, float* streams, const float* kv, const uint16_t* q_weight,
                     const uint16_t* k_weight, const uint8_t* token_mask, int64_t T, int32_t* err_flag,
                     engram_stream_t stream, bool pdl, int32_t part_cols = 0) {
  if (T == 0) return check_dims(dims, false, true);
  int rc = check_gate(dims, streams, kv, q_weight, k_weight, T);
  if (rc) return rc;
  GateParams p{streams, kv, q_weight, k_weight, token_mask, T, dims->hidden, dims->hc, dims->eps, dims->clamp,
               err_flag, part_cols};
  cudaError_t e = launch_gate(p, static_cast<cudaStream_t>(stream), pdl);
  return e == cudaSuccess ? ENGRAM_OK : fail_cuda(e, "engram_gate: launch");
}

int engram_gate(const EngramDims* dims, float* streams, const float* kv, const uint16_t* q_weight,
                const uint16_t* k_weight, const uint8_t* token_mask, int64_t T, int32_t* err_flag,
                engram_stream_t stream) {
  return gate_impl(dims, streams, kv, q_weight, k_weight, token_mask, T, err_flag, stream, false);
}

// ---- FP8 (MXFP8) operand variant ------------------------------------------------------------

int engram_quantize_mxfp8(const uint16_t* w, int64_t N, int32_t K, uint8_t* codes, uint8_t* scales,
                          engram_stream_t stream) {
  ENGRAM_CHECK_ARG(N >= 0 && K >= 32 && K % 32 == 0, "engram_quantize_mxfp8: need N >= 0 and K a multiple of 32 (got %d)", K);
  ENGRAM_CHECK_ARG(aligned(scales, 4), "engram_quantize_mxfp8: scales must be 4-byte aligned");
  if (N == 0) return ENGRAM_OK;
  ENGRAM_CHECK_ARG(w && codes && scales, "engram_quantize_mxfp8: w, codes and scales must be non-NULL");
  cudaError_t e = launch_quantize_mxfp8(w, N, K, codes, scales, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ENGRAM_OK : fail_cuda(e, "engram_quantize_mxfp8: launch");
}

static int check_gather_codes(const int32_t* ids, int64_t ids_stride_t, int64_t T, int32_t C, int32_t D,
                              const void* table, const uint8_t* scales, int64_t num_rows, const uint8_t* codes,
                              const uint8_t* out_scales) {
  ENGRAM_CHECK_ARG(T >= 0, "T must be >= 0");
  ENGRAM_CHECK_ARG(C >= 1 && ids_stride_t >= C, "need C >= 1 and ids_stride_t >= C");
  ENGRAM_CHECK_ARG(D >= 32 && D % 32 == 0, "FP8 head_dim must be a multiple of 32 (got %d)", D);
  ENGRAM_CHECK_ARG(num_rows >= 0, "num_rows must be >= 0");
  ENGRAM_CHECK_ARG(ids && table && scales && codes && out_scales, "ids, table, scales and outputs must be non-NULL");
  ENGRAM_CHECK_ARG(aligned(table, 16) && aligned(codes, 16) && aligned(out_scales, 16),
                   "table, codes and scales must be 16-byte aligned");
  return ENGRAM_OK;
}

static int gather_codes_impl(const int32_t* ids, int64_t ids_stride_t, int64_t T, int32_t C, int32_t D,
                             const void* table, const uint8_t* scales, int64_t num_rows, uint8_t* codes,
                             uint8_t* out_scales, int32_t* err_flag, engram_stream_t stream, bool pdl) {
  if (T == 0) return ENGRAM_OK;
  int rc = check_gather_codes(ids, ids_stride_t, T, C, D, table, scales, num_rows, codes, out_scales);
  if (rc) return rc;
  GatherCodesParams p{ids, ids_stride_t, T, C, D, table, scales, num_rows, codes, out_scales, err_flag};
  cudaError_t e = launch_gather_codes(p, static_cast<cudaStream_t>(stream), pdl);
  return e == cudaSuccess ? ENGRAM_OK : fail_cuda(e, "engram_gather_fp8_codes: launch");
}

int engram_gather_fp8_codes(const int32_t* ids, int64_t ids_stride_t, int64_t T, int32_t C, int32_t head_dim,
                            const void* table, const uint8_t* table_scales, int64_t num_rows, uint8_t* codes,
                            uint8_t* scales, int32_t* err_flag, engram_stream_t stream) {
  return gather_codes_impl(ids, ids_stride_t, T, C, head_dim, table, table_scales, num_rows, codes, scales, err_flag,
                           stream, false);
}

static int check_project_mx(const uint8_t* A, const uint8_t* SA, const uint8_t* W, const uint8_t* SW, const float* kv,
                            int64_t T, int32_t K, int32_t N) {
  ENGRAM_CHECK_ARG(T >= 0 && T < (int64_t)1 << 31, "T must be in [0, 2^31)");
  ENGRAM_CHECK_ARG(K >= 128 && K % 128 == 0, "MXFP8 projection: K must be a positive multiple of 128 (got %d)", K);
  ENGRAM_CHECK_ARG(N >= 16 && N % 16 == 0, "N must be a positive multiple of 16 (got %d)", N);
  ENGRAM_CHECK_ARG(A && SA && W && SW && kv, "A, A_scales, W, W_scales and kv must be non-NULL");
  ENGRAM_CHECK_ARG(aligned(A, 16) && aligned(W, 16) && aligned(kv, 16), "A, W and kv must be 16-byte aligned");
  ENGRAM_CHECK_ARG(aligned(SA, 16) && aligned(SW, 16), "A_scales and W_scales must be 16-byte aligned");
  return ENGRAM_OK;
}

// The operand gather of the FP8 variant: the projection reads its token rows from the table itself.
struct OperandGather {
  const int32_t* ids;
  int64_t ids_stride;
  const void* table;
  int64_t table_rows;
  int32_t D;
};

static int project_mx_impl(const uint8_t* A, const uint8_t* SA, const uint8_t* W, const uint8_t* SW, float* kv,
                           int64_t T, int32_t K, int32_t N, int32_t* err_flag, engram_stream_t stream, bool pdl,
                           const GateFuse* gf = nullptr, const OperandGather* og = nullptr) {
  if (T == 0) return ENGRAM_OK;
  int rc = check_project_mx(A, SA, W, SW, kv, T, K, N);
  if (rc) return rc;
  GemmMxParams p{A, SA, W, SW, kv, T, K, N, err_flag};
  if (gf != nullptr) p.gf = *gf;
  if (og != nullptr) {
    p.ids = og->ids;
    p.ids_stride = og->ids_stride;
    p.table = static_cast<const uint8_t*>(og->table);
    p.table_rows = og->table_rows;
    p.D = og->D;
  }
  return launch_gemm_mx(p, static_cast<cudaStream_t>(stream), pdl);
}

int engram_project_mxfp8(const uint8_t* A, const uint8_t* A_scales, const uint8_t* W, const uint8_t* W_scales,
                         float* kv, int64_t T, int32_t K, int32_t N, int32_t* err_flag, engram_stream_t stream) {
  return project_mx_impl(A, A_scales, W, W_scales, kv, T, K, N, err_flag, stream, false);
}

static int g_gate_fusion = 0;   // engram_set_gate_fusion
static int g_operand_gather = 0;   // engram_set_operand_gather
static int g_gather_order = 0;     // engram_set_gather_order

void engram_set_operand_gather(int32_t on) { g_operand_gather = on ? 1 : 0; }

void engram_set_gather_order(int32_t mode) { g_gather_order = mode == 1 ? 1 : 0; }

void engram_set_gate_fusion(int32_t mode) { g_gate_fusion = (mode == 1 || mode == 2) ? mode : 0; }

void engram_set_gate_form(int32_t form) { set_gate_form_override((form == 1 || form == 2) ? form : 0); }

void engram_set_gemm_mx_tile(int32_t bn) { set_gemm_mx_bn_override((bn >= 16 && bn <= 256 && bn % 16 == 0) ? bn : 0); }

// One layer's gathered operand in the engram_forward workspace: bf16 rows [T, K], or for the
// FP8 variant the codes [T, K] followed (256-byte aligned) by the scale words [ceil(K/128)][T4][4].
static size_t a_slot_bytes(int64_t T, int64_t K) {
  const size_t rows = (size_t)(T * K * 2);
  const size_t codes = round256((size_t)(T * K)) + (size_t)((K + 127) / 128) * (size_t)((T + 3) & ~(int64_t)3) * 4;
  return round256(rows > codes ? rows : codes);
}

// Row-block counters of the overlapped gate: one word per 128 tokens and layer.
static size_t done_bytes(int64_t T, int layers) { return round256((size_t)((T + 127) / 128) * layers * 4); }

// Per layer, the table-order gathers' permutation and region counters (engram_set_gather_order).
static size_t order_bytes(int64_t T, int64_t C) { return round256((size_t)(T * C * 4)) + (size_t)kOrderBuckets * 4; }

size_t engram_forward_workspace_bytes(const EngramDims* d, int64_t T) {
  if (d == nullptr || T < 0 || d->layers < 1) return 0;
  const int64_t C = (int64_t)(d->max_ngram - 1) * d->n_heads;
  const int64_t K = C * d->head_dim;
  const int64_t N = (int64_t)d->hidden * (d->hc + 1);
  return round256((size_t)(T * d->layers * C * 4)) + (size_t)d->layers * a_slot_bytes(T, K) +
         round256((size_t)(T * N * 4)) + done_bytes(T, d->layers) + (size_t)d->layers * order_bytes(T, C);
}

}  // extern "C"

namespace {

// Events that order the side stream of engram_forward2 with the caller's stream: created once per
// device and context (no timing), and used under g_side_mutex, so one call's records and waits are
// enqueued as one sequence (a concurrent call cannot re-record an event between another call's
// record and its wait).
constexpr int kSideEvents = 33;           // the hash, then up to 32 gather launches on the side stream
constexpr int kSideDevices = 64;
std::mutex g_side_mutex;
cudaEvent_t g_side_ev[kSideDevices][kSideEvents];

int side_events(cudaEvent_t** out) {
  static PerContextOnce once;
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e, "engram_forward2: cudaGetDevice");
  ENGRAM_CHECK_ARG(dev >= 0 && dev < kSideDevices, "engram_forward2: device %d beyond the %d supported", dev,
                   kSideDevices);
  e = once.run([dev] {
    for (int i = 0; i < kSideEvents; ++i) {
      cudaError_t e1 = cudaEventCreateWithFlags(&g_side_ev[dev][i], cudaEventDisableTiming);
      if (e1 != cudaSuccess) return e1;
    }
    return cudaSuccess;
  });
  if (e != cudaSuccess) return fail_cuda(e, "engram_forward2: cudaEventCreateWithFlags");
  *out = g_side_ev[dev];
  return ENGRAM_OK;
}

// The whole path on `st`; with `side` (not NULL, not st) the gathers of the layers after the first
// run on the side stream (see engram_forward2).
int forward_core(const EngramDims* dims, const EngramHashTables* tables, const EngramLayerWeights* layers,
                 const EngramTokens* tok, float* const* streams, void* workspace, size_t ws_bytes, int32_t* out_ids,
                 int32_t* err_flag, engram_stream_t stream, cudaStream_t side) {
  int rc = check_dims(dims, true, true);
  if (rc) return rc;
  ENGRAM_CHECK_ARG(tables && layers && tok && streams, "tables, layers, tokens and streams must be non-NULL");
  const int64_t T = tok->T;
  ENGRAM_CHECK_ARG(T >= 0 && T < (int64_t)1 << 31, "T must be in [0, 2^31)");
  if (T == 0) return ENGRAM_OK;
  const int L = dims->layers;
  const int C = (dims->max_ngram - 1) * dims->n_heads;
  const int64_t K = (int64_t)C * dims->head_dim;
  const int64_t N = (int64_t)dims->hidden * (dims->hc + 1);
  ENGRAM_CHECK_ARG(K <= 0x7fffffff && N <= 0x7fffffff, "K or N too large");
  const size_t need = engram_forward_workspace_bytes(dims, T);
  ENGRAM_CHECK_ARG(workspace != nullptr && ws_bytes >= need, "workspace needs %zu bytes (got %zu)", need, ws_bytes);
  ENGRAM_CHECK_ARG(aligned(workspace, 256), "workspace must be 256-byte aligned");
  // validate every layer before launching anything
  for (int l = 0; l < L; ++l) {
    const EngramLayerWeights& w = layers[l];
    rc = check_gather(w.table_format, reinterpret_cast<const int32_t*>(16), (int64_t)L * C, T, C, dims->head_dim,
                      w.table, w.table_scales, w.table_rows, reinterpret_cast<const uint16_t*>(workspace));
    if (rc) return rc;
    if (w.wkv_format == ENGRAM_WKV_MXFP8) {
      ENGRAM_CHECK_ARG(w.table_format == ENGRAM_TABLE_FP8_E8M0,
                       "layer %d: MXFP8 wkv needs an FP8+E8M0 table (its rows are the A operand)", l);
      rc = check_gather_codes(reinterpret_cast<const int32_t*>(16), (int64_t)L * C, T, C, dims->head_dim, w.table,
                              w.table_scales, w.table_rows, static_cast<const uint8_t*>(workspace),
                              static_cast<const uint8_t*>(workspace));
      if (rc) return rc;
      rc = check_project_mx(static_cast<const uint8_t*>(workspace), static_cast<const uint8_t*>(workspace),
                            reinterpret_cast<const uint8_t*>(w.wkv), w.wkv_scales,
                            reinterpret_cast<const float*>(workspace), T, (int32_t)K, (int32_t)N);
    } else {
      ENGRAM_CHECK_ARG(w.wkv_format == ENGRAM_WKV_BF16, "layer %d: unknown wkv format %d", l, w.wkv_format);
      rc = check_project(reinterpret_cast<const uint16_t*>(workspace), w.wkv, reinterpret_cast<const float*>(workspace),
                         T, (int32_t)K, (int32_t)N);
    }
    if (rc) return rc;
    rc = check_gate(dims, streams[l], reinterpret_cast<const float*>(workspace), w.q_weight, w.k_weight, T);
    if (rc) return rc;
  }
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* ids = out_ids != nullptr ? out_ids : reinterpret_cast<int32_t*>(ws);
  // one operand slot per layer (every layer's rows are gathered before the first projection), then kv
  const size_t a_slot = a_slot_bytes(T, K);
  uint8_t* const A0 = ws + round256((size_t)(T * L * C * 4));
  auto rows_of = [&](int l) { return A0 + (size_t)l * a_slot; };                 // bf16 rows or codes
  auto scales_of = [&](int l) { return rows_of(l) + round256((size_t)(T * K)); };  // FP8 variant
  float* kv = reinterpret_cast<float*>(A0 + (size_t)L * a_slot);
  // the overlapped gate's row-block counters (after kv), cleared by the hash launch
  const int64_t nblk = (T + 127) / 128;
  uint32_t* done = reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(kv) + round256((size_t)(T * N * 4)));
  // after them, per layer: the table-order permutation and its region counters
  uint8_t* const order0 = reinterpret_cast<uint8_t*>(done) + done_bytes(T, L);
  auto perm_of = [&](int l) { return reinterpret_cast<int32_t*>(order0 + (size_t)l * order_bytes(T, C)); };
  auto hist_of = [&](int l) {
    return reinterpret_cast<uint32_t*>(order0 + (size_t)l * order_bytes(T, C) + round256((size_t)(T * C * 4)));
  };
  const bool table_order = g_gather_order == 1;
  auto overlap_gate = [&](int l) { return g_gate_fusion == 2 && layers[l].wkv_format == ENGRAM_WKV_BF16; };
  bool any_overlap = false;
  for (int l = 0; l < L; ++l) any_overlap = any_overlap || overlap_gate(l);
  // workspace beyond the minimum goes to the projection (stream-K partials)
  void* gemm_ws = ws_bytes > need ? static_cast<void*>(ws + need) : nullptr;
  const size_t gemm_ws_bytes = ws_bytes > need ? ws_bytes - need : 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  // each launch may start while its predecessor finishes (programmatic dependent launch)
  HashParams hp;
  rc = hash_params(dims, tok->input_ids, T, tok->cu_seqlens, tok->num_seqs, tok->sequence_ids, tok->token_mask,
                   tok->lookback_ids, tables->token_map, tables->multipliers, tables->primes, tables->offsets, ids,
                   err_flag, hp);
  if (rc) return rc;
  if (any_overlap) {
    hp.zero = done;
    hp.zero_n = (int32_t)(nblk * L);
  }
  // FP8-variant layers whose projection gathers its own token rows (engram_set_operand_gather):
  // the gathers before it write only the rows' scale words
  auto operand_gather = [&](int l) {
    return g_operand_gather && layers[l].wkv_format == ENGRAM_WKV_MXFP8 && dims->head_dim % 128 == 0 &&
           layers[l].table_rows < ((int64_t)1 << 31);
  };
  // the hash kernel also fetches the rows of the leading run of FP8 layers (in token order; with
  // table-order gathers every layer is gathered by a launch of its own format)
  int fused = 0;
  while (!table_order && fused < L && fused < kMaxGatherLayers &&
         layers[fused].table_format == ENGRAM_TABLE_FP8_E8M0)
    ++fused;
  if (fused > 0) {
    HashGatherParams g{};
    g.h = hp;
    g.D = dims->head_dim;
    g.layers = fused;
    for (int l = 0; l < fused; ++l) {
      g.table[l] = layers[l].table;
      g.scales[l] = layers[l].table_scales;
      g.num_rows[l] = layers[l].table_rows;
      if (layers[l].wkv_format == ENGRAM_WKV_MXFP8) {
        g.out_codes[l] = operand_gather(l) ? nullptr : rows_of(l);
        g.out_scales[l] = scales_of(l);
      } else {
        g.out_bf16[l] = reinterpret_cast<uint16_t*>(rows_of(l));
      }
    }
    cudaError_t e = launch_hash_gather(g, st, true);
    if (e != cudaSuccess) return fail_cuda(e, "engram_forward: hash + gather launch");
  } else {
    cudaError_t e = launch_hash(hp, st, true);
    if (e != cudaSuccess) return fail_cuda(e, "engram_hash: launch");
  }
  // With a side stream, the layers after the first run are gathered there (layer 0's rows, if the
  // hash did not fetch them, on `st`: they are needed first); each waits for the hash, and each
  // projection on `st` waits for its run's rows.
  const bool use_side = side != nullptr && side != st && L > (fused > 0 ? fused : 1);
  std::unique_lock<std::mutex> side_lock;
  cudaEvent_t* ev = nullptr;
  int n_ev = 0;
  int side_from = L;                          // first layer gathered on the side stream
  int wait_ev[256];                           // per layer: event its projection waits for (-1: none)
  for (int l = 0; l < L; ++l) wait_ev[l] = -1;
  if (use_side) {
    rc = side_events(&ev);
    if (rc) return rc;
    side_lock = std::unique_lock<std::mutex>(g_side_mutex);
    cudaError_t ce = cudaEventRecord(ev[n_ev++], st);          // the ids are written
    if (ce == cudaSuccess) ce = cudaStreamWaitEvent(side, ev[0], 0);
    if (ce != cudaSuccess) return fail_cuda(ce, "engram_forward2: event");
    side_from = fused > 0 ? fused : 1;
  }
  // the other layers' rows: one launch per run of consecutive layers with the same table format
  // and operand kind (bf16 rows or FP8 codes), before the first projection
  for (int l = fused; l < L;) {
    const int fmt = layers[l].table_format;
    const bool mx = layers[l].wkv_format == ENGRAM_WKV_MXFP8;
    int e = l + 1;
    const int run_end = l < side_from ? side_from : L;          // a run never crosses onto the side stream
    while (e < run_end && e - l < kMaxGatherLayers && layers[e].table_format == fmt &&
           (layers[e].wkv_format == ENGRAM_WKV_MXFP8) == mx)
      ++e;
    const bool on_side = l >= side_from && n_ev < kSideEvents;
    cudaStream_t gst = on_side ? side : st;
    const bool gpdl = !on_side;
    cudaError_t ce = cudaSuccess;
    if (table_order) {                         // each layer's rows in table order
      for (int j = l; j < e && ce == cudaSuccess; ++j)
        ce = launch_row_order(ids + (int64_t)j * C, (int64_t)L * C, T, C, layers[j].table_rows, hist_of(j),
                              perm_of(j), gst, gpdl);
      if (ce != cudaSuccess) return fail_cuda(ce, "engram_forward: table-order launch");
    }
    if (mx) {
      GatherCodesLayers m{};
      m.n = e - l;
      for (int j = l; j < e; ++j)
        m.l[j - l] = GatherCodesParams{ids + (int64_t)j * C, (int64_t)L * C, T, C, dims->head_dim, layers[j].table,
                                       layers[j].table_scales, layers[j].table_rows,
                                       operand_gather(j) ? nullptr : rows_of(j), scales_of(j), err_flag,
                                       table_order ? perm_of(j) : nullptr};
      ce = launch_gather_codes(m, gst, gpdl);
    } else {
      GatherLayers m{};
      m.n = e - l;
      for (int j = l; j < e; ++j)
        m.l[j - l] = GatherParams{fmt, ids + (int64_t)j * C, (int64_t)L * C, T, C, dims->head_dim, layers[j].table,
                                  layers[j].table_scales, layers[j].table_rows,
                                  reinterpret_cast<uint16_t*>(rows_of(j)), err_flag,
                                  table_order ? perm_of(j) : nullptr};
      ce = launch_gather(m, gst, gpdl);
    }
    if (ce != cudaSuccess) return fail_cuda(ce, "engram_forward: gather launch");
    if (on_side) {                             // this run's rows are ready for its projections
      ce = cudaEventRecord(ev[n_ev], side);
      if (ce != cudaSuccess) return fail_cuda(ce, "engram_forward2: event");
      wait_ev[l] = n_ev++;
    }
    l = e;
  }
  for (int l = 0; l < L; ++l) {
    const EngramLayerWeights& w = layers[l];
    const bool mx = w.wkv_format == ENGRAM_WKV_MXFP8;
    // the gate fused into the projection's epilogue (engram_set_gate_fusion): the keys are reduced to
    // per-tile partial sums there; needs H % 32 == 0 and tiles no wider than one stream
    GateFuse gf{};
    if (g_gate_fusion == 1 && dims->hidden % 32 == 0) {
      const int tile_cols = gemm_tile_cols(T, (int)K, (int)N, mx);
      if (tile_cols > 0 && tile_cols <= dims->hidden)
        gf = GateFuse{streams[l], w.q_weight, w.k_weight, dims->hidden, dims->hc, dims->hidden * dims->hc, tile_cols};
    }
    const GateFuse* gfp = gf.keys > 0 ? &gf : nullptr;
    if (wait_ev[l] >= 0) {
      cudaError_t ce = cudaStreamWaitEvent(st, ev[wait_ev[l]], 0);
      if (ce != cudaSuccess) return fail_cuda(ce, "engram_forward2: event wait");
    }
    if (mx) {
      // FP8 variant: the rows' codes and scales are the A operand as they are
      const OperandGather og{ids + (int64_t)l * C, (int64_t)L * C, w.table, w.table_rows, dims->head_dim};
      rc = project_mx_impl(rows_of(l), scales_of(l), reinterpret_cast<const uint8_t*>(w.wkv), w.wkv_scales, kv, T,
                           (int32_t)K, (int32_t)N, err_flag, stream, true, gfp, operand_gather(l) ? &og : nullptr);
    } else {
      GateOverlap go{};
      if (overlap_gate(l)) {
        rc = check_gate(dims, streams[l], kv, w.q_weight, w.k_weight, T);
        if (rc) return rc;
        go = GateOverlap{streams[l], w.q_weight, w.k_weight, tok->token_mask, dims->hidden, dims->hc, dims->eps,
                         dims->clamp, done + (int64_t)l * nblk};
      }
      rc = project_impl(reinterpret_cast<const uint16_t*>(rows_of(l)), w.wkv, kv, T, (int32_t)K, (int32_t)N, gemm_ws,
                        gemm_ws_bytes, err_flag, stream, true, gfp, overlap_gate(l) ? &go : nullptr);
      if (rc) return rc;
      if (overlap_gate(l)) continue;           // the projection kernel applied the gate
    }
    if (rc) return rc;
    rc = gate_impl(dims, streams[l], kv, w.q_weight, w.k_weight, tok->token_mask, T, err_flag, stream, true,
                   gf.tile_cols);
    if (rc) return rc;
  }
  return ENGRAM_OK;
}

}  // namespace

extern "C" {

int engram_forward(const EngramDims* dims, const EngramHashTables* tables, const EngramLayerWeights* layers,
                   const EngramTokens* tok, float* const* streams, void* workspace, size_t ws_bytes,
                   int32_t* out_ids, int32_t* err_flag, engram_stream_t stream) {
  return forward_core(dims, tables, layers, tok, streams, workspace, ws_bytes, out_ids, err_flag, stream, nullptr);
}

int engram_forward2(const EngramDims* dims, const EngramHashTables* tables, const EngramLayerWeights* layers,
                    const EngramTokens* tok, float* const* streams, void* workspace, size_t ws_bytes,
                    int32_t* out_ids, int32_t* err_flag, engram_stream_t stream, engram_stream_t side_stream) {
  return forward_core(dims, tables, layers, tok, streams, workspace, ws_bytes, out_ids, err_flag, stream,
                      static_cast<cudaStream_t>(side_stream));
}

}  // extern "C"
