// Device helpers shared by the tcgen05 projection kernels (bf16 and MXFP8): mbarrier waits with
// a bound, TMA loads, tcgen05 fences / commits / MMAs / TMEM loads, shared-memory matrix
// descriptors, and the fp32 epilogue that stores accumulators into kv with TMA.
#pragma once

#include <cuda.h>

#include "internal.cuh"

namespace engram {

// tensor maps over row-major matrices (host; defined in gemm.cu)
bool make_map_bf16(CUtensorMap* m, const void* ptr, int64_t rows, int64_t K, uint32_t box_rows);
bool make_map_u8(CUtensorMap* m, const void* ptr, int64_t rows, int64_t K, uint32_t box_rows);
bool make_map_f32(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols);

namespace {

constexpr uint64_t kWaitLimitCycles = 4000000000ull;  // wait bound in SM cycles: ~2 s at 2 GHz
constexpr int kSmemBudget = 232448;                   // 227 KB opt-in maximum per CTA
constexpr int kEpiChunk = 32;                         // columns per warp and step (128 bytes of fp32)
constexpr int kEpiWarpBytes = 32 * kEpiChunk * 4;     // one 32 x 32 fp32 staging tile (4 KB)
constexpr int kEpiBytes = 4 * kEpiWarpBytes;          // four epilogue warps

// ---- PTX wrappers ------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: false if this CTA aborted (here or in another role). The bound counts SM clock
// cycles (clock64 is a cheap local register; %globaltimer is slow to read on this part and would
// sit on the pipeline's critical path).
__device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, volatile int32_t* abort_flag,
                                            int32_t* err, uint64_t limit_cycles) {
  const uint64_t t0 = clock64();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 0) {
      if (*abort_flag) return false;
      if ((uint64_t)clock64() - t0 > limit_cycles) {
        *abort_flag = 1;
        if (err != nullptr) atomicOr(err, ENGRAM_ERR_PIPE_TIMEOUT);
        return false;
      }
    }
  }
}
// The producer and MMA threads sit on the pipeline's critical path: the common case (phase
// already complete) stays inline, the bounded spin is a call.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int32_t* abort_flag, int32_t* err,
                                          uint64_t limit_cycles) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, abort_flag, err, limit_cycles);
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// 32 lanes x 16 columns of 32-bit accumulator: thread i gets lane (quarter*32 + i)
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ unsigned long long ld_acquire(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Shared-memory matrix descriptor: K-major operand stored as 128-byte rows with the 128B
// swizzle (what TMA writes with CU_TENSOR_MAP_SWIZZLE_128B); 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);   // start address
  d |= (uint64_t)1 << 16;                      // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;            // stride byte offset: next 8-row group
  d |= (uint64_t)1 << 46;                      // descriptor version for tcgen05
  d |= (uint64_t)2 << 61;                      // 128-byte swizzle
  return d;
}

// Stores one item's fp32 accumulators into kv: this warp's 32-lane quarter of each 128-row half.
// Per 32-column chunk, tcgen05.ld gives every thread 32 columns of its row; the thread writes them
// into the warp's 32 x 128-byte staging tile in the 128B-swizzled order (16-byte piece i of row r
// at piece i ^ (r % 8): conflict-free), and one lane stores the tile with a TMA bulk tensor store,
// or a bulk reduce-add when `adder`. A 16-column tail (tile widths that are odd multiples of 16)
// is stored by the threads. With `sum_chains` (a single 128-row half), the accumulator at
// column offset acc_stride holds a second partial sum of the same tile and is added first.
__device__ __forceinline__ void store_accumulators(const CUtensorMap* tmD, float* D, int64_t M, int N, uint32_t tmem,
                                                   int q, int lane, uint32_t stg, int msub, bool sum_chains,
                                                   uint32_t acc_stride, int BN, int m0, int n0, bool adder) {
  for (int ms = 0; ms < msub; ++ms) {
    const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(ms * acc_stride);
    const int row0 = ms * 128 + q * 32;    // first row of this warp (within the item)
    const int lrow = row0 + lane;          // this thread's row (within the item)
    for (int c0 = 0; c0 < BN; c0 += kEpiChunk) {
      const bool two = c0 + 16 < BN;     // BN is a multiple of 16
      uint32_t r[32];
      tmem_ld16(tbase + c0, &r[0]);
      if (two) tmem_ld16(tbase + c0 + 16, &r[16]);
      if (sum_chains) {                    // add the second chain of this tile
        uint32_t r2[32];
        tmem_ld16(tbase + acc_stride + c0, &r2[0]);
        if (two) tmem_ld16(tbase + acc_stride + c0 + 16, &r2[16]);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) + __uint_as_float(r2[i]));
      } else {
        tmem_ld_wait();
      }
      if (!two) {
        // 16-column tail: this thread's row by plain stores (or atomic adds)
        float* dst = D + ((int64_t)m0 + lrow) * N + n0 + c0;
        if ((int64_t)m0 + lrow < M && n0 + c0 < N) {
          if (adder) {
#pragma unroll
            for (int i = 0; i < 16; ++i) atomicAdd(dst + i, __uint_as_float(r[i]));
          } else {
#pragma unroll
            for (int i = 0; i < 4; ++i)
              reinterpret_cast<float4*>(dst)[i] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                                              __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
          }
        }
        continue;
      }
      // the previous TMA store from this staging tile has read it
      if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t addr = stg + (uint32_t)(lane * 128 + ((i ^ (lane & 7)) * 16));
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(r[4 * i]), "r"(r[4 * i + 1]),
                     "r"(r[4 * i + 2]), "r"(r[4 * i + 3])
                     : "memory");
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // visible to the TMA unit
      __syncwarp();
      if (lane == 0) {
        const uint64_t map = reinterpret_cast<uint64_t>(tmD);
        if (adder)
          asm volatile(
              "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.bulk_group [%0, {%1, %2}], [%3];" ::"l"(map),
              "r"(n0 + c0), "r"(m0 + row0), "r"(stg)
              : "memory");
        else
          asm volatile(
              "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(map),
              "r"(n0 + c0), "r"(m0 + row0), "r"(stg)
              : "memory");
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
      }
    }
  }
}

}  // namespace
}  // namespace engram
