// Table-order gathers: the rows of one layer's gather visited in the order of their place in the
// table rather than token order, for locality in a very large table (the vLLM
// "deepseek_v41.common.engram" page sorts a lookup's ids before it reads a table in host memory,
// ParallelEngramEmbedding.lookup, _engram_lookup_thresholds). Here the table is in HBM and an
// exact sort is not needed: the (token, column) rows are grouped by table region (id >> shift, at
// most kOrderBuckets regions) with a counting pass, a scan and a scatter. The gather then walks
// the permutation and writes every row at its own place, so its output is the same as in token
// order (only the order of the reads changes).
#include "internal.cuh"

namespace engram {
namespace {

constexpr int kOrderThreads = 256;
constexpr int kScanThreads = 1024;
static_assert(kOrderBuckets % kScanThreads == 0, "regions per scan thread");

__device__ __forceinline__ int order_region(int64_t id, int64_t num_rows, int shift) {
  if (id < 0 || id >= num_rows) return 0;       // outside the table (a zero row): any region
  const int64_t b = id >> shift;
  return (int)(b < kOrderBuckets ? b : kOrderBuckets - 1);
}

__global__ void __launch_bounds__(kOrderThreads) order_clear_kernel(uint32_t* hist) {
  pdl_wait();
  pdl_trigger();
  for (int i = blockIdx.x * kOrderThreads + threadIdx.x; i < kOrderBuckets; i += gridDim.x * kOrderThreads)
    hist[i] = 0u;
}

// rows per region
__global__ void __launch_bounds__(kOrderThreads)
order_count_kernel(const int32_t* __restrict__ ids, int64_t stride, int64_t T, int C, int64_t num_rows, int shift,
                   uint32_t* hist) {
  pdl_wait();                                   // the ids come from the hash kernel
  pdl_trigger();
  const int64_t n = T * C;
  for (int64_t r = (int64_t)blockIdx.x * kOrderThreads + threadIdx.x; r < n; r += (int64_t)gridDim.x * kOrderThreads) {
    const int64_t t = r / C;
    const int col = (int)(r - t * C);
    atomicAdd(hist + order_region(__ldg(ids + t * stride + col), num_rows, shift), 1u);
  }
}

// exclusive scan of the counts, in place: hist[b] becomes the first slot of region b
__global__ void __launch_bounds__(kScanThreads) order_scan_kernel(uint32_t* hist) {
  pdl_wait();
  pdl_trigger();
  constexpr int kPer = kOrderBuckets / kScanThreads;
  __shared__ uint32_t warp_total[kScanThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t v[kPer];
  uint32_t sum = 0;
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    v[k] = hist[tid * kPer + k];
    sum += v[k];
  }
  uint32_t x = sum;                             // inclusive scan of the threads' sums in the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_total[warp] = x;
  __syncthreads();
  if (warp == 0) {                              // inclusive scan of the warps' totals
    uint32_t w = warp_total[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    warp_total[lane] = w;
  }
  __syncthreads();
  uint32_t run = x - sum + (warp > 0 ? warp_total[warp - 1] : 0u);   // rows before this thread's regions
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    hist[tid * kPer + k] = run;
    run += v[k];
  }
}

// each row to the next free slot of its region
__global__ void __launch_bounds__(kOrderThreads)
order_scatter_kernel(const int32_t* __restrict__ ids, int64_t stride, int64_t T, int C, int64_t num_rows, int shift,
                     uint32_t* hist, int32_t* perm) {
  pdl_wait();
  pdl_trigger();
  const int64_t n = T * C;
  for (int64_t r = (int64_t)blockIdx.x * kOrderThreads + threadIdx.x; r < n; r += (int64_t)gridDim.x * kOrderThreads) {
    const int64_t t = r / C;
    const int col = (int)(r - t * C);
    const uint32_t slot = atomicAdd(hist + order_region(__ldg(ids + t * stride + col), num_rows, shift), 1u);
    perm[slot] = (int32_t)r;
  }
}

}  // namespace

cudaError_t launch_row_order(const int32_t* ids, int64_t ids_stride, int64_t T, int32_t C, int64_t num_rows,
                             uint32_t* hist, int32_t* perm, cudaStream_t stream, bool pdl) {
  const int64_t n = T * C;
  if (n <= 0) return cudaSuccess;
  if (n > 0x7fffffff || num_rows < 1) return cudaErrorInvalidValue;   // perm holds int32 row numbers
  int shift = 0;
  while (((num_rows - 1) >> shift) >= kOrderBuckets) ++shift;         // regions of 2^shift rows
  int64_t blocks = (n + kOrderThreads - 1) / kOrderThreads;
  const int64_t cap = (int64_t)num_sms() * 8;
  if (blocks > cap) blocks = cap;
  cudaError_t e = launch_k(order_clear_kernel, dim3(kOrderBuckets / kOrderThreads), dim3(kOrderThreads), 0, stream,
                           pdl, hist);
  if (e == cudaSuccess)
    e = launch_k(order_count_kernel, dim3((unsigned)blocks), dim3(kOrderThreads), 0, stream, pdl, ids, ids_stride, T,
                 (int)C, num_rows, shift, hist);
  if (e == cudaSuccess) e = launch_k(order_scan_kernel, dim3(1), dim3(kScanThreads), 0, stream, pdl, hist);
  if (e == cudaSuccess)
    e = launch_k(order_scatter_kernel, dim3((unsigned)blocks), dim3(kOrderThreads), 0, stream, pdl, ids, ids_stride,
                 T, (int)C, num_rows, shift, hist, perm);
  return e;
}

}  // namespace engram
