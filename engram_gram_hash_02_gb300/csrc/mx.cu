// MXFP8 operands for the FP8 variant of the projection.
//
// The FP8 table of the vLLM "deepseek_v41.common.engram" page (ParallelEngramEmbedding: weight
// float8_e4m3fn plus one ue8m0 scale per 32 values) already is an MXFP8 operand. The variant
// therefore gathers rows without dequantising them (codes and scale bytes copied as they are)
// and stores wkv the same way, so the tensor cores read both operands with their block scales
// (tcgen05.mma kind::mxf8f6f4, see gemm_mx.cu).
//
// Weight encoding (the table's scale convention; the pages print no encoder): per row and block
// of 32 along K, the scale is the smallest power of two 2^e with max|w| / 2^e <= 448, stored as
// the byte 127 + e; each code is w / 2^e rounded to the nearest e4m3 value, ties to even. An
// all-zero block gets byte 127 and zero codes.
//
// Scale layout of both operands (the projection's own, so a stage's scales are one contiguous
// run it can bulk-copy): 32-bit words [K/128][rows4], rows4 = rows rounded up to a multiple of 4;
// word (kb, r) holds the bytes of row r's blocks 4kb .. 4kb+3, lowest byte first.
#include <type_traits>

#include "internal.cuh"

namespace engram {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// fp32 -> e4m3 code, round to nearest even, saturating at 448 (both halves of the pair carry v)
__device__ __forceinline__ uint32_t to_e4m3(float v) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %1;" : "=h"(r) : "f"(v));
  return r & 0xFFu;
}

// One warp per (row, 32-block): lane i owns element 32*blk + i.
__global__ void __launch_bounds__(kThreads)
quantize_mxfp8_kernel(const uint16_t* __restrict__ w, int64_t N, int32_t K, uint8_t* __restrict__ codes,
                      uint8_t* __restrict__ scales) {
  const int64_t blocks = N * (K / 32);
  const int64_t rows4 = (N + 3) & ~(int64_t)3;
  const int lane = threadIdx.x & 31;
  for (int64_t b = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5; b < blocks;
       b += ((int64_t)gridDim.x * kThreads) >> 5) {
    const int64_t idx = b * 32 + lane;                  // rows are K long: blocks tile them exactly
    const float x = __uint_as_float((uint32_t)__ldg(w + idx) << 16);
    float amax = fabsf(x);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    int e = 0;
    if (amax > 0.f) {
      // amax = f * 2^ex with f in [0.5, 1): 448 * 2^e >= amax holds first at e = ex - 9 when
      // f <= 0.875 (448 = 0.875 * 2^9), else at e = ex - 8
      int ex;
      const float f = frexpf(amax, &ex);
      e = f <= 0.875f ? ex - 9 : ex - 8;
      e = max(-127, min(127, e));
    }
    codes[idx] = (uint8_t)to_e4m3(ldexpf(x, -e));
    if (lane == 0) {
      const int64_t n = b / (K / 32);
      const int blk = (int)(b - n * (K / 32));
      scales[((int64_t)(blk >> 2) * rows4 + n) * 4 + (blk & 3)] = (uint8_t)(127 + e);
    }
  }
}

// FP8 rows by id, copied without dequantisation: 16 threads per 256-byte row (16-byte chunks);
// the chunk-0 thread also copies the row's scale bytes. Rows outside the table: codes 0, scale
// byte 127 (a zero row).
template <typename I>
__global__ void __launch_bounds__(kThreads)
gather_fp8_codes_kernel(const GatherCodesLayers m) {
  const GatherCodesParams& p = m.l[blockIdx.y];
  pdl_wait();                                    // ids come from the hash kernel
  pdl_trigger();
  const int chunks_per_row = p.D >> 4;
  const int sblocks = p.D >> 5;
  const int64_t total = p.T * p.C * chunks_per_row;
  const int64_t rows4 = (p.T + 3) & ~(int64_t)3;
  const uint8_t* __restrict__ weight = static_cast<const uint8_t*>(p.table);
  for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < total; i += (int64_t)gridDim.x * kThreads) {
    // index split: multiply-and-shift by the launch's constants when its indices fit in 31 bits
    // (I = uint32_t), else int64_t divisions
    // (with a permutation, the walk's row r is the row perm[r], written at that row's place)
    int64_t t, oi = i;
    int j, col;
    if constexpr (std::is_same<I, uint32_t>::value) {
      const uint32_t ii = (uint32_t)i;
      uint32_t r = fast_div(ii, m.div_cpr);
      j = (int)(ii - r * (uint32_t)chunks_per_row);
      if (p.perm != nullptr) {
        r = (uint32_t)__ldg(p.perm + r);
        oi = (int64_t)r * chunks_per_row + j;
      }
      const uint32_t tt = fast_div(r, m.div_c);
      t = tt;
      col = (int)(r - tt * (uint32_t)p.C);
    } else {
      int64_t r = i / chunks_per_row;
      j = (int)(i - r * chunks_per_row);
      if (p.perm != nullptr) {
        r = __ldg(p.perm + r);
        oi = r * chunks_per_row + j;
      }
      t = r / p.C;
      col = (int)(r - t * p.C);
    }
    const int64_t id = __ldg(p.ids + t * p.ids_stride_t + col);
    const bool ok = id >= 0 && id < p.num_rows;
    if (!ok && j == 0 && p.err != nullptr) atomicOr(p.err, ENGRAM_ERR_ROW_ID);
    if (p.codes != nullptr) {                    // NULL: scale words only (the projection gathers the codes)
      uint4 v = make_uint4(0, 0, 0, 0);
      if (ok) v = ld_stream_v4(weight + id * p.D + (j << 4));
      *reinterpret_cast<uint4*>(p.codes + (oi << 4)) = v;
    }
    // scale bytes: the row's D/32 bytes, copied by the threads of the first D/32 chunks into the
    // projection's word layout (block b of token t at byte 4 * ((b / 4) * rows4 + t) + b % 4)
    if (j < sblocks) {
      const int b = col * sblocks + j;
      p.out_scales[((int64_t)(b >> 2) * rows4 + t) * 4 + (b & 3)] = ok ? __ldg(p.scales + id * sblocks + j) : (uint8_t)127;
    }
  }
}

}  // namespace

cudaError_t launch_quantize_mxfp8(const uint16_t* w, int64_t N, int32_t K, uint8_t* codes, uint8_t* scales,
                                  cudaStream_t stream) {
  const int64_t warps = N * (K / 32);
  int64_t blocks = (warps * 32 + kThreads - 1) / kThreads;
  const int64_t cap = (int64_t)num_sms() * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return launch_k(quantize_mxfp8_kernel, dim3((unsigned)blocks), dim3(kThreads), 0, stream, false, w, N, K, codes,
                  scales);
}

cudaError_t launch_gather_codes(const GatherCodesLayers& layers, cudaStream_t stream, bool pdl) {
  if (layers.n < 1 || layers.n > kMaxGatherLayers) return cudaErrorInvalidValue;
  GatherCodesLayers m = layers;
  const GatherCodesParams& p = m.l[0];           // every layer has p's T, C and D
  if (p.C < 1 || p.D < 16) return cudaErrorInvalidValue;
  m.div_cpr = make_fastdiv((uint32_t)(p.D >> 4));
  m.div_c = make_fastdiv((uint32_t)p.C);
  const int64_t total = p.T * p.C * (p.D >> 4);
  int64_t blocks = (total + kThreads - 1) / kThreads;
  const int64_t cap = (int64_t)num_sms() * 32;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  const bool narrow = total + blocks * kThreads < ((int64_t)1 << 31);
  return launch_k(narrow ? gather_fp8_codes_kernel<uint32_t> : gather_fp8_codes_kernel<int64_t>,
                  dim3((unsigned)blocks, (unsigned)m.n), dim3(kThreads), 0, stream, pdl, m);
}

}  // namespace engram
