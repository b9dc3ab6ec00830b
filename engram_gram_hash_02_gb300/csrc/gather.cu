// Stage 2: gather table rows by id and dequantise to bf16 rows of the projection operand.
//
// FP8-E4M3 rows with one E8M0 scale per 32 values follow the vLLM "deepseek_v41.common.engram"
// page (ParallelEngramEmbedding, _engram_lookup_kernel: value * 2^(byte-127) in fp32, then
// bf16; rows outside the table read as zeros). The 84-byte Q2_K row follows the Atlas
// "engram_v41" page (stage 2, ENGRAM_ROW_BYTES), read as the public GGML Q2_K super-block.
//
// HBM-bound random row reads. FP8: one thread per 16-byte chunk of a row (16 threads per
// 256-wide row, so a row is one coalesced 256-byte read), four chunks per thread in flight,
// scales applied in registers, 32 bytes of bf16 written per chunk. Q2_K: one warp per row;
// lanes 0..20 read the 84 bytes as 21 words (one coalesced read), shuffles hand each lane
// the quants, scale nibbles and d/dmin of its 8 outputs.
#include <cuda_fp8.h>

#include <type_traits>

#include "hash_token.cuh"

namespace engram {
namespace {

constexpr int kThreads = 256;
constexpr int kChunksPerThread = 4;
constexpr int kQ2kRowsPerWarp = 4;

__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // round to nearest even
  return *reinterpret_cast<uint32_t*>(&v);
}

// two e4m3 bytes (low 16 bits of x) -> two floats, exactly
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t x) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(x & 0xFFFFu), __NV_E4M3);
  return __half22float2(*reinterpret_cast<__half2*>(&h));
}

__device__ __forceinline__ uint32_t dequant_pair(uint32_t bytes2, float scale) {
  float2 f = e4m3x2_to_float2(bytes2);
  return pack_bf16x2(f.x * scale, f.y * scale);
}

__device__ __forceinline__ void flag(int32_t* err, int32_t bit) {
  if (err != nullptr) atomicOr(err, bit);
}

// Flat chunk index i -> (row r = t * C + col, chunk j), in I: uint32_t when every index of the
// launch fits in 31 bits (a 32-bit division by a loop-invariant divisor, whose reciprocal the
// compiler keeps out of the loop), else int64_t. (The multiply-and-shift of fastdiv.h measured
// slower here at large T, though faster in the Q2_K and code gathers, which use it.)
// With a permutation (table-order gathers) the walk's row r is the row perm[r], and the chunk is
// written at that row's place (out_chunk); otherwise out_chunk = i.
template <typename I>
__device__ __forceinline__ void split_chunk(int64_t i, int chunks_per_row, int C, const int32_t* perm, I& t,
                                            int& col, int& j, int64_t& out_chunk) {
  const I ii = (I)i;
  I r = ii / (I)chunks_per_row;
  j = (int)(ii - r * (I)chunks_per_row);
  out_chunk = i;
  if (perm != nullptr) {
    r = (I)__ldg(perm + r);
    out_chunk = (int64_t)r * chunks_per_row + j;
  }
  t = r / (I)C;
  col = (int)(r - t * (I)C);
}

// ---- FP8-E4M3 + E8M0 ------------------------------------------------------------------
template <typename I>
__global__ void __launch_bounds__(kThreads)
gather_fp8_kernel(const GatherLayers m) {
  const GatherParams& p = m.l[blockIdx.y];
  pdl_wait();                                    // ids come from the hash kernel
  pdl_trigger();
  const int chunks_per_row = p.D >> 4;                 // 16 values per chunk
  const int64_t total = p.T * p.C * chunks_per_row;
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  const uint8_t* __restrict__ weight = static_cast<const uint8_t*>(p.table);
  const int sblocks = p.D >> 5;                        // scales per row

  for (int64_t base = (int64_t)blockIdx.x * kThreads + threadIdx.x; base < total;
       base += stride * kChunksPerThread) {
    uint4 v[kChunksPerThread];
    uint32_t sb[kChunksPerThread];
    bool ok[kChunksPerThread];
    int64_t oi[kChunksPerThread];               // where each chunk goes
#pragma unroll
    for (int u = 0; u < kChunksPerThread; ++u) {
      const int64_t i = base + u * stride;
      ok[u] = false;
      v[u] = make_uint4(0, 0, 0, 0);
      sb[u] = 0;
      oi[u] = i;
      if (i < total) {
        I t;
        int col, j;
        split_chunk<I>(i, chunks_per_row, p.C, p.perm, t, col, j, oi[u]);
        const int64_t id = __ldg(p.ids + (int64_t)t * p.ids_stride_t + col);
        if (id >= 0 && id < p.num_rows) {
          ok[u] = true;
          v[u] = ld_stream_v4(weight + id * p.D + (j << 4));
          sb[u] = __ldg(p.scales + id * sblocks + (j >> 1));
        } else if (j == 0) {
          flag(p.err, ENGRAM_ERR_ROW_ID);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kChunksPerThread; ++u) {
      const int64_t i = base + u * stride;
      if (i >= total) continue;
      uint4 lo = make_uint4(0, 0, 0, 0), hi = make_uint4(0, 0, 0, 0);
      if (ok[u]) {
        const float scale = __uint_as_float(sb[u] << 23);  // E8M0 byte is the fp32 exponent field
        lo.x = dequant_pair(v[u].x, scale);
        lo.y = dequant_pair(v[u].x >> 16, scale);
        lo.z = dequant_pair(v[u].y, scale);
        lo.w = dequant_pair(v[u].y >> 16, scale);
        hi.x = dequant_pair(v[u].z, scale);
        hi.y = dequant_pair(v[u].z >> 16, scale);
        hi.z = dequant_pair(v[u].w, scale);
        hi.w = dequant_pair(v[u].w >> 16, scale);
      }
      uint4* dst = reinterpret_cast<uint4*>(p.out + (oi[u] << 4));   // chunk c -> 16 bf16 at 16*c
      dst[0] = lo;
      dst[1] = hi;
    }
  }
}

// ---- bf16 rows: copy ----------------------------------------------------------------------
template <typename I>
__global__ void __launch_bounds__(kThreads)
gather_bf16_kernel(const GatherLayers m) {
  const GatherParams& p = m.l[blockIdx.y];
  pdl_wait();
  pdl_trigger();
  const int chunks_per_row = p.D >> 3;                 // 8 values per chunk
  const int64_t total = p.T * p.C * chunks_per_row;
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  const uint16_t* __restrict__ table = static_cast<const uint16_t*>(p.table);
  for (int64_t base = (int64_t)blockIdx.x * kThreads + threadIdx.x; base < total;
       base += stride * kChunksPerThread) {
    uint4 v[kChunksPerThread];
    int64_t oi[kChunksPerThread];               // where each chunk goes
#pragma unroll
    for (int u = 0; u < kChunksPerThread; ++u) {
      const int64_t i = base + u * stride;
      v[u] = make_uint4(0, 0, 0, 0);
      oi[u] = i;
      if (i < total) {
        I t;
        int col, j;
        split_chunk<I>(i, chunks_per_row, p.C, p.perm, t, col, j, oi[u]);
        const int64_t id = __ldg(p.ids + (int64_t)t * p.ids_stride_t + col);
        if (id >= 0 && id < p.num_rows) {
          v[u] = ld_stream_v4(table + id * p.D + (j << 3));
        } else if (j == 0) {
          flag(p.err, ENGRAM_ERR_ROW_ID);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kChunksPerThread; ++u) {
      const int64_t i = base + u * stride;
      if (i < total) reinterpret_cast<uint4*>(p.out)[oi[u]] = v[u];
    }
  }
}

// ---- Q2_K: one 84-byte super-block per 256-wide row ---------------------------------------
// Element e: sub-block b = e/16 (scale = low nibble, min = high nibble of byte b),
// quant = (qs[32*(e/128) + e%32] >> 2*((e%128)/32)) & 3, then d*scale*q - dmin*min.
// Lane L writes elements 8L..8L+7: half = L/16, bit pair j = (L/4)%4, l0 = 8*(L%4), b = L/2.
template <typename I>
__global__ void __launch_bounds__(kThreads)
gather_q2k_kernel(const GatherLayers m) {
  const GatherParams& p = m.l[blockIdx.y];
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
  const int64_t rows = p.T * p.C;
  const uint32_t* __restrict__ table = static_cast<const uint32_t*>(p.table);

  const int half = lane >> 4;
  const int jshift = 2 * ((lane >> 2) & 3);
  const int qword = 4 + 8 * half + 2 * (lane & 3);      // word index of qs[32*half + l0]
  const int sword = lane >> 3;                          // word holding scales[b], b = lane/2
  const int sshift = 8 * ((lane >> 1) & 3);

  for (int64_t r0 = warp * kQ2kRowsPerWarp; r0 < rows; r0 += nwarps * kQ2kRowsPerWarp) {
    uint32_t word[kQ2kRowsPerWarp];
    bool ok[kQ2kRowsPerWarp];
    int64_t orow[kQ2kRowsPerWarp];              // where each row goes (its own place in token order)
#pragma unroll
    for (int u = 0; u < kQ2kRowsPerWarp; ++u) {
      int64_t r = r0 + u;
      ok[u] = false;
      word[u] = 0;
      orow[u] = r;
      if (r < rows) {
        if (p.perm != nullptr) orow[u] = r = __ldg(p.perm + r);   // table-order walk
        I t;
        if constexpr (std::is_same<I, uint32_t>::value) t = fast_div((uint32_t)r, m.div_c);
        else t = r / p.C;
        const int col = (int)((I)r - t * (I)p.C);
        const int64_t id = __ldg(p.ids + (int64_t)t * p.ids_stride_t + col);
        ok[u] = id >= 0 && id < p.num_rows;
        if (ok[u] && lane < 21) word[u] = __ldg(table + id * 21 + lane);
        if (!ok[u] && lane == 0) flag(p.err, ENGRAM_ERR_ROW_ID);
      }
    }
#pragma unroll
    for (int u = 0; u < kQ2kRowsPerWarp; ++u) {
      const int64_t r = r0 + u;
      const uint32_t q0 = __shfl_sync(0xffffffffu, word[u], qword);
      const uint32_t q1 = __shfl_sync(0xffffffffu, word[u], qword + 1);
      const uint32_t sw = __shfl_sync(0xffffffffu, word[u], sword);
      const uint32_t dw = __shfl_sync(0xffffffffu, word[u], 20);
      if (r >= rows) continue;
      uint4 o = make_uint4(0, 0, 0, 0);
      if (ok[u]) {
        const uint32_t sc = (sw >> sshift) & 0xFFu;
        const float d = __half2float(__ushort_as_half((unsigned short)(dw & 0xFFFFu)));
        const float dmin = __half2float(__ushort_as_half((unsigned short)(dw >> 16)));
        const float dl = d * (float)(sc & 15u);       // exact
        const float nml = -(dmin * (float)(sc >> 4)); // exact
        float y[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint32_t byte = ((i < 4 ? q0 : q1) >> (8 * (i & 3))) & 0xFFu;
          const float q = (float)((byte >> jshift) & 3u);
          y[i] = fmaf(dl, q, nml);                    // dl*q exact: one rounding of the difference
        }
        o.x = pack_bf16x2(y[0], y[1]);
        o.y = pack_bf16x2(y[2], y[3]);
        o.z = pack_bf16x2(y[4], y[5]);
        o.w = pack_bf16x2(y[6], y[7]);
      }
      reinterpret_cast<uint4*>(p.out + orow[u] * 256)[lane] = o;
    }
  }
}

unsigned grid_for(int64_t work_items, int64_t per_block) {
  int64_t b = (work_items + per_block - 1) / per_block;
  if (b < 1) b = 1;
  const int64_t cap = (int64_t)num_sms() * 64;
  return (unsigned)(b < cap ? b : cap);
}

// ---- hash fused with the leading FP8 layers' gathers (engram_forward) ---------------------------
// One CTA per token: warp 0 hashes the token (its window loads in flight while the block stages
// cu_seqlens), the ids go to the global id buffer and to shared memory, then all threads fetch
// the token's rows of layers 0 .. layers-1, 16 bytes per thread and step, dequantised to bf16 or
// copied as codes, or (a layer whose projection gathers its own rows) only the scale words.
// (A form that issued every chunk load of the token at once, with 128 or 256 threads, ran faster
// alone but made the chained decode step 2 us longer; this one is kept.)
constexpr int kHgThreads = 128;

__global__ void __launch_bounds__(kHgThreads)
hash_gather_fp8_kernel(const HashGatherParams p) {
  __shared__ int32_t s_cu[kSmemCu];
  __shared__ int32_t s_ids[256];
  pdl_wait();                                    // inputs may come from the preceding kernel
  pdl_trigger();
  clear_words(p.h);
  const int64_t t = blockIdx.x;
  const int lane = threadIdx.x & 31;
  const bool hasher = threadIdx.x < 32;
  TokenLoads L;
  if (hasher) L = hash_token_loads(p.h, t, lane);
  const bool cu_in_smem = stage_cu(p.h, s_cu);
  if (hasher) hash_token_finish(p.h, t, lane, L, cu_in_smem, s_cu, s_ids);
  __syncthreads();

  const int C = p.h.cols;
  const int cpr = p.D >> 4;                     // 16-byte chunks per row
  const int sblocks = p.D >> 5;
  const int64_t K = (int64_t)C * p.D;
  const int64_t rows4 = (p.h.T + 3) & ~(int64_t)3;
#pragma unroll 1
  for (int l = 0; l < p.layers; ++l) {
    const uint8_t* __restrict__ weight = static_cast<const uint8_t*>(p.table[l]);
    const uint8_t* __restrict__ scales = p.scales[l];
    const int64_t num_rows = p.num_rows[l];
    uint16_t* const out_bf16 = p.out_bf16[l];
    uint8_t* const out_codes = p.out_codes[l];
    uint8_t* const out_scales = p.out_scales[l];
    const bool scales_only = out_bf16 == nullptr && out_codes == nullptr;
    for (int i = threadIdx.x; i < C * cpr; i += kHgThreads) {
      const int col = i / cpr;
      const int j = i - col * cpr;
      if (scales_only && j >= sblocks) continue;
      const int64_t id = s_ids[l * C + col];      // ids of token t in (layer, column) order
      const bool ok = id >= 0 && id < num_rows;
      if (!ok && j == 0) flag(p.h.err, ENGRAM_ERR_ROW_ID);
      uint4 v = make_uint4(0, 0, 0, 0);
      if (ok && !scales_only) v = ld_stream_v4(weight + id * p.D + (j << 4));
      const int64_t e0 = t * K + (int64_t)col * p.D + (j << 4);   // first element of this chunk
      if (out_bf16 != nullptr) {
        uint4 lo = make_uint4(0, 0, 0, 0), hi = make_uint4(0, 0, 0, 0);
        if (ok) {
          const float scale = __uint_as_float((uint32_t)__ldg(scales + id * sblocks + (j >> 1)) << 23);
          lo.x = dequant_pair(v.x, scale);
          lo.y = dequant_pair(v.x >> 16, scale);
          lo.z = dequant_pair(v.y, scale);
          lo.w = dequant_pair(v.y >> 16, scale);
          hi.x = dequant_pair(v.z, scale);
          hi.y = dequant_pair(v.z >> 16, scale);
          hi.z = dequant_pair(v.w, scale);
          hi.w = dequant_pair(v.w >> 16, scale);
        }
        uint4* dst = reinterpret_cast<uint4*>(out_bf16 + e0);
        dst[0] = lo;
        dst[1] = hi;
      } else {
        if (out_codes != nullptr) *reinterpret_cast<uint4*>(out_codes + e0) = v;
        if (j < sblocks) {
          const int b = col * sblocks + j;          // block of 32 along K
          out_scales[((int64_t)(b >> 2) * rows4 + t) * 4 + (b & 3)] = ok ? __ldg(scales + id * sblocks + j) : (uint8_t)127;
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_hash_gather(const HashGatherParams& p, cudaStream_t stream, bool pdl) {
  if (p.h.T > 0x7fffffff) return cudaErrorInvalidValue;
  return launch_k(hash_gather_fp8_kernel, dim3((unsigned)p.h.T), dim3(kHgThreads), 0, stream, pdl, p);
}

cudaError_t launch_gather(const GatherLayers& layers, cudaStream_t stream, bool pdl) {
  if (layers.n < 1 || layers.n > kMaxGatherLayers) return cudaErrorInvalidValue;
  GatherLayers m = layers;
  const GatherParams& p = m.l[0];                // every layer has p's format, T, C and D
  if (p.C < 1 || p.D < 16) return cudaErrorInvalidValue;
  m.div_c = make_fastdiv((uint32_t)p.C);
  const int64_t rows = p.T * p.C;
  // flat indices below 2^31 (with a stride's overshoot): 32-bit index arithmetic
  const int64_t span = rows * (p.D / 8) + 2 * (int64_t)num_sms() * 64 * kThreads * kChunksPerThread;
  const bool narrow = span < ((int64_t)1 << 31);
  switch (p.fmt) {
    case ENGRAM_TABLE_FP8_E8M0:
      return launch_k(narrow ? gather_fp8_kernel<uint32_t> : gather_fp8_kernel<int64_t>,
                      dim3(grid_for(rows * (p.D / 16), kThreads * kChunksPerThread), m.n), dim3(kThreads), 0, stream,
                      pdl, m);
    case ENGRAM_TABLE_BF16:
      return launch_k(narrow ? gather_bf16_kernel<uint32_t> : gather_bf16_kernel<int64_t>,
                      dim3(grid_for(rows * (p.D / 8), kThreads * kChunksPerThread), m.n), dim3(kThreads), 0, stream,
                      pdl, m);
    case ENGRAM_TABLE_Q2K:
      return launch_k(narrow ? gather_q2k_kernel<uint32_t> : gather_q2k_kernel<int64_t>,
                      dim3(grid_for(rows, (kThreads / 32) * kQ2kRowsPerWarp), m.n), dim3(kThreads), 0, stream, pdl,
                      m);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace engram
