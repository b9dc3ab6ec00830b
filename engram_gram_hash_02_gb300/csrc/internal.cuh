// Internal declarations shared by the CUDA translation units of libengram.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/engram.h"
#include "fastdiv.h"

namespace engram {

// ---- host-side error reporting -------------------------------------------------------
void set_error(const char* fmt, ...);
int fail_cuda(cudaError_t e, const char* what);

#define ENGRAM_CHECK_ARG(cond, ...)            \
  do {                                          \
    if (!(cond)) {                              \
      ::engram::set_error(__VA_ARGS__);         \
      return ENGRAM_EINVAL;                     \
    }                                           \
  } while (0)

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int num_sms();  // of the current device, cached per device

// Once-per-context set-up (kernel attributes, the static scratch address). The key is the current
// device and its current CUDA context: after cudaDeviceReset the primary context (and with it
// every module and function attribute) is re-created, so the set-up runs again. Thread-safe.
class PerContextOnce {
 public:
  // Runs fn() unless it already succeeded for the current context; returns its error, if any.
  template <typename F>
  cudaError_t run(F fn) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kDevices) return fn();
    std::lock_guard<std::mutex> g(mutex_);
    if (done_[dev] && ctx_[dev] == current_context()) return cudaSuccess;
    e = fn();
    if (e == cudaSuccess) {
      done_[dev] = true;
      ctx_[dev] = current_context();   // current by now (fn made a runtime call)
    }
    return e;
  }
  static void* current_context();   // the driver's CUcontext of this thread (nullptr if none)

 private:
  static constexpr int kDevices = 64;
  void* ctx_[kDevices] = {};
  bool done_[kDevices] = {};
  std::mutex mutex_;
};

// ---- programmatic dependent launch ----------------------------------------------------------
// Inside engram_forward each kernel is launched so that it may start while its predecessor on
// the stream is still running. Every kernel runs pdl_wait() (all prerequisite grids complete and
// their writes visible) before it reads anything a predecessor wrote or writes anything a
// predecessor reads, and every CTA runs it before exiting; pdl_trigger() comes only after the
// wait, so a dependent grid starts only once every earlier kernel but its immediate predecessor
// has finished. Launched without the attribute (the single-stage entry points), both are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename Kernel, typename... Args>
cudaError_t launch_k(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, bool pdl,
                     Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// ---- launchers (validated arguments only) ---------------------------------------------
struct HashParams {
  const int32_t* input_ids;
  const int32_t* cu_seqlens;
  const int32_t* sequence_ids;
  const uint8_t* token_mask;
  const int32_t* lookback_ids;
  const int32_t* token_map;
  const int64_t* multipliers;
  const int64_t* primes;
  const int64_t* offsets;
  int32_t* out;
  int32_t* err;
  int64_t T;
  int32_t S;
  int32_t layers, max_ngram, n_heads, cols;
  int32_t raw_vocab, pad_id;
  uint32_t* zero;             // engram_forward: words the first block clears (the overlapped gate's
  int32_t zero_n;             // row-block counters), after waiting for the preceding kernel
};
cudaError_t launch_hash(const HashParams& p, cudaStream_t stream, bool pdl = false);

// Layers whose rows one gather launch fetches (engram_forward gathers every layer's rows right
// after the hash, before the first projection)
constexpr int kMaxGatherLayers = 8;

// Hash fused with the gathers of the leading FP8_E8M0 layers (engram_forward): one CTA per token
// hashes it (all layers' ids to h.out) and gathers its rows of layers 0 .. layers-1, dequantised to
// bf16 (out_bf16[l]) or as codes and scale words (out_codes[l] / out_scales[l], the FP8 variant's
// layout).
struct HashGatherParams {
  HashParams h;
  int32_t D;
  int32_t layers;                                  // 1 .. kMaxGatherLayers
  const void* table[kMaxGatherLayers];             // e4m3 codes [num_rows, D]
  const uint8_t* scales[kMaxGatherLayers];         // [num_rows, D/32]
  int64_t num_rows[kMaxGatherLayers];
  uint16_t* out_bf16[kMaxGatherLayers];            // [T, C*D] or NULL
  uint8_t* out_codes[kMaxGatherLayers];            // [T, C*D] or NULL (with out_scales: scale words only)
  uint8_t* out_scales[kMaxGatherLayers];           // [ceil(C*D/128)][T4][4] or NULL
};
cudaError_t launch_hash_gather(const HashGatherParams& p, cudaStream_t stream, bool pdl = false);

struct GatherParams {
  int32_t fmt;
  const int32_t* ids;
  int64_t ids_stride_t;
  int64_t T;
  int32_t C, D;
  const void* table;
  const uint8_t* scales;
  int64_t num_rows;
  uint16_t* out;
  int32_t* err;
  const int32_t* perm;        // NULL: rows in token order; else row n of the gather is perm[n] (table order)
};
// n layers of the same format, T, C and D in one launch (grid y = layer); the launcher fills the
// division by C (the Q2_K gather's)
struct GatherLayers {
  int32_t n;
  GatherParams l[kMaxGatherLayers];
  FastDiv div_c;
};
cudaError_t launch_gather(const GatherLayers& p, cudaStream_t stream, bool pdl = false);
inline cudaError_t launch_gather(const GatherParams& p, cudaStream_t stream, bool pdl = false) {
  GatherLayers m{};
  m.n = 1;
  m.l[0] = p;
  return launch_gather(m, stream, pdl);
}

// The gate fused into the projection's epilogue (see tc_common.cuh): the key columns of kv are
// reduced to per-tile partial sums instead of being stored. keys == 0: the fusion is off.
struct GateFuse {
  const float* h;            // streams [M, hc, H] fp32
  const uint16_t* qw;        // q_weight [hc, H] bf16
  const uint16_t* kw;        // k_weight [hc, H] bf16
  int32_t H, hc;
  int32_t keys;              // hc * H: the key columns (0: the fusion is off)
  int32_t tile_cols;         // columns per partial slot: the tile width (set by the projection's plan)
};

// The gate run by extra warps of the projection kernel, overlapped with its tensor-core work: the
// gate of a token starts once every tile of its row block is stored (counted in `done`, one
// counter per 128-row block, zero when the projection starts).
struct GateOverlap {
  float* streams;            // [M, hc, H] fp32, updated in place (NULL: off)
  const uint16_t* qw;        // q_weight [hc, H] bf16
  const uint16_t* kw;        // k_weight [hc, H] bf16
  const uint8_t* mask;       // [M] or NULL
  int32_t H, hc;
  float eps, clamp;
  uint32_t* done;            // [ceil(M / 128)]
};

struct GemmParams {
  const uint16_t* A;
  const uint16_t* B;
  float* D;
  int64_t M;
  int32_t K, N;
  int32_t* err;
  void* workspace;      // stream-K flags (may be NULL)
  size_t ws_bytes;
  GateFuse gf;          // gf.keys > 0: gate partials instead of the key columns (data-parallel only)
  GateOverlap go;       // go.streams != NULL: the gate inside the projection (data-parallel only)
};
// returns ENGRAM_OK or an error code (sets the message)
int launch_gemm(const GemmParams& p, cudaStream_t stream, bool pdl = false);
size_t gemm_workspace_bytes(int64_t M, int K, int N);
// the plan launch_gemm / launch_gemm_mx would use on `sms` SMs (host only); false if none fits
bool gemm_plan_info(int64_t M, int K, int N, int sms, EngramProjectPlan* out);
bool gemm_mx_plan_info(int64_t M, int K, int N, int sms, EngramProjectPlan* out);

// ---- FP8 (MXFP8) operand variant of the projection -----------------------------------------
struct GatherCodesParams {
  const int32_t* ids;
  int64_t ids_stride_t;
  int64_t T;
  int32_t C, D;
  const void* table;          // e4m3 codes [rows, D]
  const uint8_t* scales;      // [rows, D/32]
  int64_t num_rows;
  uint8_t* codes;             // [T, C*D], or NULL: only the scale words (the projection gathers the codes)
  uint8_t* out_scales;        // [T, C*D/32]
  int32_t* err;
  const int32_t* perm;        // NULL: rows in token order; else row n of the gather is perm[n] (table order)
};
struct GatherCodesLayers {
  int32_t n;
  GatherCodesParams l[kMaxGatherLayers];
  FastDiv div_cpr, div_c;     // the divisions by the chunks per row and by C (filled by the launcher)
};
cudaError_t launch_gather_codes(const GatherCodesLayers& p, cudaStream_t stream, bool pdl = false);
inline cudaError_t launch_gather_codes(const GatherCodesParams& p, cudaStream_t stream, bool pdl = false) {
  GatherCodesLayers m{};
  m.n = 1;
  m.l[0] = p;
  return launch_gather_codes(m, stream, pdl);
}
// Table-order gathers (engram_set_gather_order): a permutation of one layer's T * C (token, column)
// rows sorted by table region (id >> shift, kOrderBuckets regions), so that a gather reads the
// table in address order. hist holds kOrderBuckets words of scratch. Four launches: clear, count,
// scan, scatter.
constexpr int kOrderBuckets = 16384;
cudaError_t launch_row_order(const int32_t* ids, int64_t ids_stride, int64_t T, int32_t C, int64_t num_rows,
                             uint32_t* hist, int32_t* perm, cudaStream_t stream, bool pdl);

cudaError_t launch_quantize_mxfp8(const uint16_t* w, int64_t N, int32_t K, uint8_t* codes, uint8_t* scales,
                                  cudaStream_t stream);

struct GemmMxParams {
  const uint8_t* A;           // e4m3 codes [M, K] (unused with the operand gather)
  const uint8_t* SA;          // scale bytes [M, K/32]
  const uint8_t* B;           // e4m3 codes [N, K]
  const uint8_t* SB;          // scale bytes [N, K/32]
  float* Dout;                // [M, N]
  int64_t M;
  int32_t K, N;
  int32_t* err;
  GateFuse gf;                // as GemmParams::gf
  // operand gather (ids != NULL): A row m is the concatenation of table rows ids[m * ids_stride + c],
  // c = 0 .. K/D - 1, read from the table by the projection itself (SA still holds their scales)
  const int32_t* ids;
  int64_t ids_stride;
  const uint8_t* table;       // e4m3 codes [table_rows, D]
  int64_t table_rows;
  int32_t D;
};
int launch_gemm_mx(const GemmMxParams& p, cudaStream_t stream, bool pdl = false);
// tile width the projection of this shape runs with (the partial slot width of the fused gate);
// 0 if no plan fits
int gemm_tile_cols(int64_t M, int K, int N, bool mx);

struct GateParams {
  float* streams;
  const float* kv;
  const uint16_t* q_weight;
  const uint16_t* k_weight;
  const uint8_t* token_mask;
  int64_t T;
  int32_t H, hc;
  float eps, clamp;
  int32_t* err;
  int32_t part_cols;          // > 0: the projection fused the gate's key sums (GateFuse, tile width
                              // part_cols): the key columns of kv hold per-tile partials
};
cudaError_t launch_gate(const GateParams& p, cudaStream_t stream, bool pdl = false);
cudaError_t launch_gate_persistent(const GateParams& p, cudaStream_t stream, bool pdl = false);
void set_gate_form_override(int f);

}  // namespace engram
