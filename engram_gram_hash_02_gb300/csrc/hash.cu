// Stage 1: n-gram hash ids, one warp per token (see hash_token.cuh for the per-token walk and
// mix). The NeMo "deepseek_v41.engram" page (DeepseekV41NgramHash.forward) and the vLLM
// "deepseek_v41.common.engram" page (NgramHashState.forward, EngramLayout) define it.
#include "hash_token.cuh"

namespace engram {
namespace {

constexpr int kWarpsPerBlock = 8;

__global__ void __launch_bounds__(kWarpsPerBlock * 32)
hash_kernel(const HashParams p) {
  __shared__ int32_t s_cu[kSmemCu];
  pdl_wait();                                    // inputs may come from the preceding kernel
  pdl_trigger();
  clear_words(p);
  const int lane = threadIdx.x & 31;
  const int64_t t = (int64_t)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  const bool live = t < p.T;
  TokenLoads L;
  if (live) L = hash_token_loads(p, t, lane);      // in flight while cu_seqlens is staged
  const bool cu_in_smem = stage_cu(p, s_cu);
  if (!live) return;
  hash_token_finish(p, t, lane, L, cu_in_smem, s_cu, nullptr);
}

}  // namespace

cudaError_t launch_hash(const HashParams& p, cudaStream_t stream, bool pdl) {
  const int64_t blocks = (p.T + kWarpsPerBlock - 1) / kWarpsPerBlock;
  return launch_k(hash_kernel, dim3((unsigned)blocks), dim3(kWarpsPerBlock * 32), 0, stream, pdl, p);
}

}  // namespace engram
