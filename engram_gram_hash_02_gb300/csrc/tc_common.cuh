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
// Columns before c_begin (a multiple of 16) are not stored.
__device__ __forceinline__ void store_accumulators(const CUtensorMap* tmD, float* D, int64_t M, int N, uint32_t tmem,
                                                   int q, int lane, uint32_t stg, int msub, bool sum_chains,
                                                   uint32_t acc_stride, int BN, int m0, int n0, bool adder,
                                                   int c_begin = 0) {
  for (int ms = 0; ms < msub; ++ms) {
    const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(ms * acc_stride);
    const int row0 = ms * 128 + q * 32;    // first row of this warp (within the item)
    const int lrow = row0 + lane;          // this thread's row (within the item)
    for (int c0 = c_begin; c0 < BN; c0 += kEpiChunk) {
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

// ---- the gate fused into the projection's epilogue ----------------------------------------------
// With the fusion on, the key columns [0, hc*H) of kv are never stored. For every token row of a
// tile, the epilogue thread that drains the row accumulates the two sums the gate needs from the
// keys, per stream j the tile covers (at most two, as the tile is at most H wide):
//     ssk_j = sum key^2          dot_j = sum (h * q_weight[j]) * (key * k_weight[j])
// over the tile's key columns of stream j, reading the stream row h from global memory (the
// epilogue warps prefetch the next tile's rows into L2 while the tensor cores run). It writes them
// as one 16-byte partial (ssk_first, dot_first, ssk_second, dot_second) at kv[t, 4 * tile_n] (the
// key columns are free). The value columns are stored as before. A finishing pass sums, for each
// (token, stream), the partials of the tiles covering the stream in tile order, adds sum h^2 and
// applies the gate.
struct RowPartials {
  float ssk[2], dot[2];
};

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Four key values (y0..y3, raw fp32 bits) with their stream values, q_weight and k_weight pairs.
__device__ __forceinline__ void gate_acc4(uint32_t y0, uint32_t y1, uint32_t y2, uint32_t y3, float4 h, uint32_t q01,
                                          uint32_t q23, uint32_t k01, uint32_t k23, float& ssk, float& dot) {
  const float a = __uint_as_float(y0), b = __uint_as_float(y1), c = __uint_as_float(y2), d = __uint_as_float(y3);
  ssk = fmaf(a, a, ssk);
  ssk = fmaf(b, b, ssk);
  ssk = fmaf(c, c, ssk);
  ssk = fmaf(d, d, ssk);
  dot = fmaf(h.x * bf16_lo(q01), a * bf16_lo(k01), dot);
  dot = fmaf(h.y * bf16_hi(q01), b * bf16_hi(k01), dot);
  dot = fmaf(h.z * bf16_lo(q23), c * bf16_lo(k23), dot);
  dot = fmaf(h.w * bf16_hi(q23), d * bf16_hi(k23), dot);
}

// The stream values of 16 columns x .. x+15 of this thread's row (one stream's: a stream boundary is
// a multiple of 32, and x a multiple of 16).
struct H16 {
  float4 a, b, c, d;
};
__device__ __forceinline__ H16 load_h16(const GateFuse& gf, int64_t row, int x) {
  const int j = x / gf.H;
  const float4* hp = reinterpret_cast<const float4*>(gf.h + (row * gf.hc + j) * (int64_t)gf.H + (x - j * gf.H));
  return H16{hp[0], hp[1], hp[2], hp[3]};
}

// 16 key values r[0..15] of this thread's row at global columns x .. x+15, with their stream
// values, into P.
__device__ __forceinline__ void gate_partial16(const GateFuse& gf, const uint32_t* r, const H16& h, int x, int j0,
                                               RowPartials& P) {
  const int j = x / gf.H;
  const int xi = x - j * gf.H;
  const uint4* qp = reinterpret_cast<const uint4*>(gf.qw + (int64_t)j * gf.H + xi);
  const uint4* kp = reinterpret_cast<const uint4*>(gf.kw + (int64_t)j * gf.H + xi);
  const uint4 q0 = __ldg(qp), q1 = __ldg(qp + 1), k0 = __ldg(kp), k1 = __ldg(kp + 1);
  float ssk = 0.f, dot = 0.f;
  gate_acc4(r[0], r[1], r[2], r[3], h.a, q0.x, q0.y, k0.x, k0.y, ssk, dot);
  gate_acc4(r[4], r[5], r[6], r[7], h.b, q0.z, q0.w, k0.z, k0.w, ssk, dot);
  gate_acc4(r[8], r[9], r[10], r[11], h.c, q1.x, q1.y, k1.x, k1.y, ssk, dot);
  gate_acc4(r[12], r[13], r[14], r[15], h.d, q1.z, q1.w, k1.z, k1.w, ssk, dot);
  if (j == j0) {                             // the tile's first stream, or its second
    P.ssk[0] += ssk;
    P.dot[0] += dot;
  } else {
    P.ssk[1] += ssk;
    P.dot[1] += dot;
  }
}

// Partials of this thread's row over the key columns of one accumulator region (columns n0 ..
// n0+cols-1 of the tile). Warp-collective (the tensor-memory loads): every lane runs it; rows past M
// only skip their global reads. The stream values of the next chunk are requested before the
// current chunk is reduced.
__device__ __forceinline__ void gate_partials_region(const GateFuse& gf, uint32_t tbase, bool sum_chains,
                                                     uint32_t acc_stride, int cols, int n0, int j0, int64_t row,
                                                     bool row_ok, RowPartials& P) {
  const int kend = min(cols, gf.keys - n0);  // key columns of this region: [0, kend)
  if (kend <= 0) return;
  H16 h0 = {}, h1 = {};
  if (row_ok) {
    h0 = load_h16(gf, row, n0);
    if (16 < kend) h1 = load_h16(gf, row, n0 + 16);
  }
  for (int c0 = 0; c0 < kend; c0 += kEpiChunk) {
    const int x = n0 + c0;
    const bool two = c0 + 16 < kend;
    uint32_t r[32];
    tmem_ld16(tbase + c0, &r[0]);
    if (two) tmem_ld16(tbase + c0 + 16, &r[16]);
    // the next chunk's stream values, in flight while this chunk is reduced
    const int c1 = c0 + kEpiChunk;
    H16 n0v = {}, n1v = {};
    if (row_ok && c1 < kend) {
      n0v = load_h16(gf, row, n0 + c1);
      if (c1 + 16 < kend) n1v = load_h16(gf, row, n0 + c1 + 16);
    }
    if (sum_chains) {
      uint32_t r2[32];
      tmem_ld16(tbase + acc_stride + c0, &r2[0]);
      if (two) tmem_ld16(tbase + acc_stride + c0 + 16, &r2[16]);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) + __uint_as_float(r2[i]));
    } else {
      tmem_ld_wait();
    }
    if (row_ok) {
      gate_partial16(gf, &r[0], h0, x, j0, P);
      if (two) gate_partial16(gf, &r[16], h1, x + 16, j0, P);
    }
    h0 = n0v;
    h1 = n1v;
  }
}

// Prefetch into L2 the stream rows a tile's key columns will need (this thread's rows).
__device__ __forceinline__ void gate_prefetch_rows(const GateFuse& gf, int64_t M, int msub, int q, int lane, int m0,
                                                   int n0, int BN) {
  const int x1 = min(n0 + BN, gf.keys);
  for (int ms = 0; ms < msub; ++ms) {
    const int64_t row = (int64_t)m0 + ms * 128 + q * 32 + lane;
    if (row >= M) continue;
    for (int x = n0; x < x1; x += 32) {      // 128-byte lines (a stream boundary is a multiple of 32)
      const int j = x / gf.H;
      const float* p = gf.h + (row * gf.hc + j) * (int64_t)gf.H + (x - j * gf.H);
      asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
    }
  }
}

// The epilogue of one tile with the gate fused: partials of the key columns, store of the value
// columns. Arguments as store_accumulators; `nsplit` 2 (two column halves of BN/2 in the two
// accumulators) or 1. BN is the tile width.
__device__ __forceinline__ void fused_gate_epilogue(const GateFuse& gf, const CUtensorMap* tmD, float* D, int64_t M,
                                                    int N, uint32_t tmem, int q, int lane, uint32_t stg, int msub,
                                                    bool sum_chains, uint32_t acc_stride, int BN, int nsplit, int m0,
                                                    int n0) {
  const int tile_n = n0 / gf.tile_cols;
  const int j0 = n0 / gf.H;                  // the first stream the tile covers
  if (n0 < gf.keys) {
    for (int ms = 0; ms < msub; ++ms) {
      const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(ms * acc_stride);
      const int64_t row = (int64_t)m0 + ms * 128 + q * 32 + lane;
      const bool row_ok = row < M;
      RowPartials P = {{0.f, 0.f}, {0.f, 0.f}};
      if (nsplit == 2) {
        const int hb = BN >> 1;
        gate_partials_region(gf, tbase, false, acc_stride, hb, n0, j0, row, row_ok, P);
        gate_partials_region(gf, tbase + acc_stride, false, acc_stride, hb, n0 + hb, j0, row, row_ok, P);
      } else {
        gate_partials_region(gf, tbase, sum_chains, acc_stride, BN, n0, j0, row, row_ok, P);
      }
      if (row_ok)
        *reinterpret_cast<float4*>(D + row * N + 4 * tile_n) = make_float4(P.ssk[0], P.dot[0], P.ssk[1], P.dot[1]);
    }
  }
  if (n0 + BN > gf.keys) {                   // value columns of this tile: stored as they are
    const int c_begin = n0 < gf.keys ? gf.keys - n0 : 0;
    if (nsplit == 2) {
      const int hb = BN >> 1;
      if (c_begin < hb)
        store_accumulators(tmD, D, M, N, tmem, q, lane, stg, 1, false, acc_stride, hb, m0, n0, false, c_begin);
      store_accumulators(tmD, D, M, N, tmem + acc_stride, q, lane, stg, 1, false, acc_stride, hb, m0, n0 + hb, false,
                         c_begin > hb ? c_begin - hb : 0);
    } else {
      store_accumulators(tmD, D, M, N, tmem, q, lane, stg, msub, sum_chains, acc_stride, BN, m0, n0, false, c_begin);
    }
  }
}

}  // namespace
}  // namespace engram
