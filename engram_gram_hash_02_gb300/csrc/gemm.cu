// Stage 3: the wkv projection kv[T, N] = A[T, K] * wkv[N, K]^T on tcgen05 tensor cores.
//
// The projection of the vLLM "deepseek_v41.common.engram" page (Engram.__init__: wkv maps
// n_hash_cols*head_dim -> dim*(hc+1); Engram.forward) and of the Atlas "engram_v41" page
// (stage 3: dense bf16 GEMM). bf16 operands, fp32 accumulation in tensor memory, fp32 out.
//
// A persistent kernel, one CTA per SM, 6 warps:
//   warp 0      TMA producer: 128B-swizzled K-major tiles of A (128 rows x 64) and of wkv
//               (BN rows x 64) into a ring of shared-memory stages (mbarrier complete_tx). Under
//               programmatic dependent launch the first ring of wkv tiles is requested before
//               waiting for the kernel that writes A.
//   warp 1      allocates tensor memory; one lane issues tcgen05.mma (M=128, N=BN, K=16,
//               kind::f16) and releases each stage with tcgen05.commit.
//   warps 2..5  epilogue: tcgen05.ld of the fp32 accumulators (each warp its 32-lane quarter),
//               staged as 32 x 32 swizzled shared tiles and written with TMA bulk tensor stores.
// Every item accumulates into two TMEM accumulators, which the tensor core runs as independent
// chains (back-to-back MMAs into one accumulator wait on each other): the two 128-row halves of
// a 256-row tile, or, for tiles of at most 128 rows, the even and odd k steps of one tile
// (summed in the epilogue).
//
// Schedules (items are (tile, k-range) pairs; the roles walk the same sequence):
//   data-parallel  CTA c takes tiles c, c + grid, ... over the whole K (many tiles);
//   stream-K       the tiles x k-blocks are split evenly over all CTAs, so a shape with fewer
//                  tiles than SMs (the decode step: 80 tiles of 256 x 256) still keeps every SM
//                  streaming wkv. A tile cut between CTAs is summed into kv in unit order: the
//                  CTA holding its first segment stores it (TMA store) and publishes an
//                  epoch-tagged flag in the caller's workspace; the CTA holding the next segment
//                  waits for that flag and adds its part with a TMA bulk reduce-add, and so on
//                  (fixed order: deterministic). Each CTA runs its segments last-first, so the
//                  segment others wait for is done early. All CTAs are co-resident (grid <= SMs)
//                  and wait only on lower-numbered CTAs.
//
// Every wait (mbarrier or flag) is bounded (~2 s of SM clock cycles); on expiry the CTA raises
// an abort flag, reports ENGRAM_ERR_PIPE_TIMEOUT, drains its in-flight copies and MMAs (again
// bounded), frees its tensor memory and exits.
#include <cuda.h>

#include <atomic>
#include <mutex>

#include "internal.cuh"

namespace engram {
namespace {

constexpr int kBK = 64;                    // k elements per stage (128 bytes = one swizzle row)
constexpr int kUmmaK = 16;                 // k per tcgen05.mma for 16-bit operands
constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;
constexpr int kMaxStages = 8;
constexpr int kATileBytes = 128 * kBK * 2;  // 16 KB
constexpr uint64_t kWaitLimitCycles = 4000000000ull;  // wait bound in SM cycles: ~2 s at 2 GHz
constexpr int kSmemBudget = 232448;        // 227 KB opt-in maximum per CTA
constexpr unsigned long long kFlagMagic = 0x5EA5C0DEull;
constexpr int kEpiChunk = 32;                        // columns per warp and step (128 bytes of fp32)
constexpr int kEpiWarpBytes = 32 * kEpiChunk * 4;    // one 32 x 32 fp32 staging tile (4 KB)
constexpr int kEpiBytes = 4 * kEpiWarpBytes;         // four epilogue warps

struct Ctl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t acc_full;                       // MMA -> epilogue: the item's accumulators are final
  uint64_t acc_empty;                      // epilogue -> MMA: tensor memory drained
  uint32_t tmem_base;
  int32_t abort_flag;
};

struct GemmArgs {
  int32_t M, K, N;
  int32_t BN, msub, stages, num_kb;
  int32_t m_tiles, n_tiles, group_m;
  int32_t stage_bytes;
  uint32_t idesc;
  uint32_t tmem_cols, acc_stride;
  int32_t stream_k;                        // 0: data-parallel tiles, 1: stream-K
  int64_t total_units;                     // tiles * num_kb
  unsigned long long* flags;               // [grid] (stream-K)
  unsigned long long epoch;
  int32_t* err;
};

struct Item {
  int tile, k0, k1;
};

// The sequence of items of CTA b. Every role constructs one and walks it in the same order.
struct Schedule {
  const GemmArgs& a;
  int b, grid;
  int next_tile;                           // data-parallel
  int64_t u_begin, u_end, cursor;          // stream-K: this CTA's unit range, walked backwards
  __device__ Schedule(const GemmArgs& args, int block, int g) : a(args), b(block), grid(g) {
    next_tile = block;
    const int64_t base = a.total_units / g, rem = a.total_units % g;
    u_begin = (int64_t)block * base + (block < rem ? block : rem);
    u_end = u_begin + base + (block < rem ? 1 : 0);
    cursor = u_end;
  }
  __device__ bool next(Item& it) {
    if (!a.stream_k) {
      if (next_tile >= a.m_tiles * a.n_tiles) return false;
      it.tile = next_tile;
      it.k0 = 0;
      it.k1 = a.num_kb;
      next_tile += grid;
      return true;
    }
    if (cursor <= u_begin) return false;
    const int64_t last = cursor - 1;
    const int tile = (int)(last / a.num_kb);
    const int64_t tile_start = (int64_t)tile * a.num_kb;
    const int64_t seg_start = tile_start > u_begin ? tile_start : u_begin;
    it.tile = tile;
    it.k0 = (int)(seg_start - tile_start);
    it.k1 = (int)(cursor - tile_start);
    cursor = seg_start;
    return true;
  }
};

__device__ __forceinline__ void tile_origin(const GemmArgs& a, int tile, int& m0, int& n0) {
  // grouped raster: consecutive tiles sweep group_m row blocks of one column block
  const int per_group = a.group_m * a.n_tiles;
  const int first_m = (tile / per_group) * a.group_m;
  const int gsize = min(a.m_tiles - first_m, a.group_m);
  const int in_group = tile % per_group;
  m0 = (first_m + in_group % gsize) * 128 * a.msub;
  n0 = (in_group / gsize) * a.BN;
}

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
__device__ __forceinline__ void epi_bar() {  // the 128 epilogue threads only
  asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
}
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

__global__ void __launch_bounds__(kThreads, 1)
wkv_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmD,
                float* __restrict__ D, const GemmArgs a) {
  // A timeout anywhere in an earlier launch sharing the flag word voids the result: skip the
  // work instead of waiting out the time limits again.
  if (a.err != nullptr && (*reinterpret_cast<volatile int32_t*>(a.err) & ENGRAM_ERR_PIPE_TIMEOUT)) {
    pdl_wait();
    return;
  }
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t tiles = (raw_base + 1023u) & ~1023u;          // swizzled tiles need 1 KB alignment
  const uint32_t epi_stage = tiles + (uint32_t)(a.stages * a.stage_bytes);   // 1 KB aligned
  Ctl* ctl = reinterpret_cast<Ctl*>(smem_raw + (tiles - raw_base) + a.stages * a.stage_bytes + kEpiBytes);
  volatile int32_t* abort_flag = &ctl->abort_flag;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(smem_u32(&ctl->full[s]), 1);
      mbar_init(smem_u32(&ctl->empty[s]), 1);
    }
    mbar_init(smem_u32(&ctl->acc_full), 1);
    mbar_init(smem_u32(&ctl->acc_empty), kEpiThreads);
    ctl->abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmD);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&ctl->tmem_base)),
                 "r"(a.tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      auto load_b = [&](int it, int kb, int n0) {
        const int s = it % a.stages;
        const uint32_t full = smem_u32(&ctl->full[s]);
        const uint32_t st = tiles + (uint32_t)(s * a.stage_bytes);
        mbar_expect_tx(full, (uint32_t)a.stage_bytes);
        tma_load_2d(st + a.msub * kATileBytes, &tmB, full, kb * kBK, n0);
      };
      auto load_a = [&](int it, int kb, int m0) {
        const int s = it % a.stages;
        const uint32_t full = smem_u32(&ctl->full[s]);
        const uint32_t st = tiles + (uint32_t)(s * a.stage_bytes);
        for (int ms = 0; ms < a.msub; ++ms) tma_load_2d(st + ms * kATileBytes, &tmA, full, kb * kBK, m0 + ms * 128);
      };
      // wkv does not come from the preceding kernel: fill the ring's weight halves before waiting
      // for the gathered rows (A) to be complete
      int early = 0;
      {
        Schedule sch(a, blockIdx.x, gridDim.x);
        Item item;
        while (early < a.stages && sch.next(item)) {
          int m0, n0;
          tile_origin(a, item.tile, m0, n0);
          for (int kb = item.k0; kb < item.k1 && early < a.stages; ++kb) load_b(early++, kb, n0);
        }
      }
      pdl_wait();
      int it = 0, issued = 0;
      bool ok = true;
      Schedule sch(a, blockIdx.x, gridDim.x);
      Item item;
      while (ok && sch.next(item)) {
        int m0, n0;
        tile_origin(a, item.tile, m0, n0);
        {
          // the next kernel may start launching once this CTA is on its last item (earlier, its
          // waiting CTAs would share the SM with a long main loop)
          Schedule peek = sch;
          Item tmp;
          if (!peek.next(tmp)) pdl_trigger();
        }
        for (int kb = item.k0; kb < item.k1; ++kb, ++it) {
          if (it < early) {
            load_a(it, kb, m0);
          } else {
            const int s = it % a.stages;
            const uint32_t ph = (uint32_t)(it / a.stages) & 1u;
            if (!mbar_wait(smem_u32(&ctl->empty[s]), ph ^ 1u, abort_flag, a.err, kWaitLimitCycles)) {
              ok = false;
              break;
            }
            load_b(it, kb, n0);
            load_a(it, kb, m0);
          }
          issued = it + 1;
        }
      }
      if (!ok) {
        // drain: the copies still in flight must land before shared memory goes away
        const int first = issued > a.stages ? issued - a.stages : 0;
        for (int j = first; j < issued; ++j) {
          volatile int32_t never = 0;
          mbar_wait(smem_u32(&ctl->full[j % a.stages]), (uint32_t)(j / a.stages) & 1u, &never, nullptr,
                    kWaitLimitCycles / 4);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      Schedule sch(a, blockIdx.x, gridDim.x);
      Item item;
      int n_items = 0;
      int slot = 0;                            // iteration mod stages
      uint32_t round = 0;                      // (iteration / stages) & 1
      bool ok = true;
      while (ok && sch.next(item)) {
        // the epilogue has drained the previous item's accumulators
        if (!mbar_wait(smem_u32(&ctl->acc_empty), (uint32_t)(n_items & 1) ^ 1u, abort_flag, a.err,
                       kWaitLimitCycles)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kb = item.k0; kb < item.k1; ++kb) {
          if (!mbar_wait(smem_u32(&ctl->full[slot]), round, abort_flag, a.err, kWaitLimitCycles)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // descriptors of the k = 0 slices; a k step of 16 elements (32 bytes) adds 2 to the
          // encoded start address, the second 128-row half (16 KB) adds 1024
          const uint32_t st = tiles + (uint32_t)(slot * a.stage_bytes);
          const uint64_t a0 = smem_desc_sw128(st);
          const uint64_t b0 = smem_desc_sw128(st + (uint32_t)(a.msub * kATileBytes));
#pragma unroll
          for (int k = 0; k < kBK / kUmmaK; ++k) {
            const uint64_t bdesc = b0 + (uint64_t)(2 * k);
            if (a.msub == 2) {
              // two chains: the two 128-row halves
              const uint32_t acc = (kb > item.k0 || k > 0) ? 1u : 0u;
              tc_mma(tmem, a0 + (uint64_t)(2 * k), bdesc, a.idesc, acc);
              tc_mma(tmem + a.acc_stride, a0 + (uint64_t)(2 * k + (kATileBytes >> 4)), bdesc, a.idesc, acc);
            } else {
              // two chains: even and odd k steps of the same tile
              tc_mma(tmem + (k & 1) * a.acc_stride, a0 + (uint64_t)(2 * k), bdesc, a.idesc,
                     (kb > item.k0 || k > 1) ? 1u : 0u);
            }
          }
          tc_commit(smem_u32(&ctl->empty[slot]));   // stage free once these MMAs have read it
          if (++slot == a.stages) {
            slot = 0;
            round ^= 1u;
          }
        }
        tc_commit(smem_u32(&ctl->acc_full));     // this item's accumulators final (or drained)
        ++n_items;
      }
      if (!ok) tc_commit(smem_u32(&ctl->acc_full));
    }
  } else {
    // ---------------- epilogue: TMEM -> registers -> shared tile -> fp32 kv --------------------
    const int q = warp & 3;                    // TMEM lane quarter this warp may access
    const int et = threadIdx.x - 64;           // 0..127
    pdl_wait();                                // kv may still be read by an earlier kernel
    Schedule sch(a, blockIdx.x, gridDim.x);
    Item item;
    int n_items = 0;
    // Each warp owns 32 rows (its TMEM lane quarter) of each 128-row half. Per 32-column chunk,
    // tcgen05.ld gives every thread 32 columns of its row; the thread writes them into the warp's
    // 32 x 128-byte staging tile in the 128B-swizzled order (16-byte piece i of row r at piece
    // i ^ (r % 8): conflict-free), and one lane stores the tile with a TMA bulk tensor store. A
    // 16-column tail (tile widths that are odd multiples of 16) is stored by the threads.
    const uint32_t stg = epi_stage + (uint32_t)(q * kEpiWarpBytes);
    while (sch.next(item)) {
      const bool ok = mbar_wait(smem_u32(&ctl->acc_full), (uint32_t)(n_items & 1), abort_flag, a.err,
                                kWaitLimitCycles);
      tc_fence_after();
      if (!ok || *abort_flag) break;
      int m0, n0;
      tile_origin(a, item.tile, m0, n0);
      // A tile cut between CTAs is summed into kv in unit order: the CTA holding its first
      // segment stores it, each later segment waits for the CTA just before it (which holds the
      // previous segment) and adds into kv. Fixed order, so results are deterministic.
      const bool adder = item.k0 > 0;                        // later segment: reduce-add into kv
      const bool publish = item.k1 < a.num_kb;               // a later segment follows: signal it
      const unsigned long long want = (a.epoch << 32) | kFlagMagic;
      if (adder) {
        const uint64_t t0 = clock64();
        while (ld_acquire(a.flags + blockIdx.x - 1) != want) {     // every lane acquires
          if (*abort_flag || (uint64_t)clock64() - t0 > kWaitLimitCycles) {
            *abort_flag = 1;
            if (a.err != nullptr) atomicOr(a.err, ENGRAM_ERR_PIPE_TIMEOUT);
            break;
          }
        }
        asm volatile("fence.proxy.async.global;" ::: "memory");   // order before our TMA adds
        __syncwarp();
        if (*abort_flag) break;
      }
      for (int ms = 0; ms < a.msub; ++ms) {
        const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(ms * a.acc_stride);
        const int row0 = ms * 128 + q * 32;    // first row of this warp (within the item)
        const int lrow = row0 + lane;          // this thread's row (within the item)
        for (int c0 = 0; c0 < a.BN; c0 += kEpiChunk) {
          const bool two = c0 + 16 < a.BN;     // BN is a multiple of 16
          uint32_t r[32];
          tmem_ld16(tbase + c0, &r[0]);
          if (two) tmem_ld16(tbase + c0 + 16, &r[16]);
          if (a.msub == 1) {                   // sum the even/odd k-step chains
            uint32_t r2[32];
            tmem_ld16(tbase + a.acc_stride + c0, &r2[0]);
            if (two) tmem_ld16(tbase + a.acc_stride + c0 + 16, &r2[16]);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) + __uint_as_float(r2[i]));
          } else {
            tmem_ld_wait();
          }
          const int npc = two ? 8 : 4;         // 16-byte pieces in this chunk
          if (!two) {
            // 16-column tail: this thread's row by plain stores (or atomic adds)
            float* dst = D + ((int64_t)m0 + lrow) * a.N + n0 + c0;
            if ((int64_t)m0 + lrow < a.M && n0 + c0 < a.N) {
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
            const uint64_t map = reinterpret_cast<uint64_t>(&tmD);
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
      // this item's stores are complete (global writes done) before the tile or flag moves on
      if (lane == 0) {
        asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
        asm volatile("fence.proxy.async.global;" ::: "memory");
      }
      __syncwarp();
      if (publish) {
        // this segment is in kv (every warp's stores complete): let the next segment's CTA add
        __threadfence();
        epi_bar();
        if (et == 0) st_release(a.flags + blockIdx.x, want);
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&ctl->acc_empty));  // tensor memory may take the next item
      ++n_items;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    if (*abort_flag) {
      // make sure no MMA is still writing the accumulators we are about to free
      volatile int32_t never = 0;
      for (int ph = 0; ph < 2; ++ph)
        mbar_wait(smem_u32(&ctl->acc_full), (uint32_t)ph, &never, nullptr, kWaitLimitCycles / 8);
    }
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(a.tmem_cols)
                 : "memory");
  }
}

// ---- host side ------------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D fp32 map over a row-major [rows, cols] matrix; box = 32 x 32 with the 128B swizzle (the
// epilogue's staging tiles)
bool make_map_f32(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 4};
  cuuint32_t box[2] = {(cuuint32_t)kEpiChunk, 32};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D bf16 map over a row-major [rows, K] matrix; box = 64 k x box_rows rows, 128B swizzle
bool make_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t K, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  cuuint32_t box[2] = {(cuuint32_t)kBK, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int g_bn_override = 0;      // engram_set_gemm_tile
int g_sched_override = 0;   // engram_set_gemm_schedule: 0 auto, 1 data-parallel, 2 stream-K
std::atomic<unsigned long long> g_epoch{1};

uint32_t pow2_at_least(uint32_t x) {
  uint32_t p = 32;
  while (p < x) p <<= 1;
  return p;
}

// tile width for the data-parallel schedule: few waves of tiles over the SMs
int pick_bn_dp(int64_t m_tiles, int N, int sms) {
  int best = 256;
  double best_cost = 1e300;
  for (int bn = 256; bn >= 64; bn -= 16) {
    const int64_t tiles = m_tiles * ((N + bn - 1) / bn);
    const int64_t waves = (tiles + sms - 1) / sms;
    const double cost = (double)waves * (bn + 48);   // a wave ~ its tile width + fixed overhead
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = bn;
    }
  }
  return best;
}

struct Plan {
  GemmArgs a;
  int grid;
  int smem;
  size_t ws_needed;   // workspace of the stream-K schedule (0 when data-parallel)
};

size_t sk_workspace(int sms) { return ((size_t)sms * 8 + 255) & ~(size_t)255; }   // one flag per CTA

// Data-parallel by default; stream-K (256-wide tiles) when asked for, the data-parallel schedule
// would leave SMs idle, and the caller's workspace holds the flags.
bool plan_gemm(int64_t M, int K, int N, int sms, size_t ws_bytes, Plan& P) {
  GemmArgs& a = P.a;
  a = GemmArgs{};
  a.M = (int32_t)M;
  a.K = K;
  a.N = N;
  a.msub = M > 128 ? 2 : 1;
  a.m_tiles = (int32_t)((M + 128 * a.msub - 1) / (128 * a.msub));
  a.num_kb = (K + kBK - 1) / kBK;
  a.group_m = 16;
  const int bn_sk = N >= 256 ? 256 : ((N + 15) / 16) * 16;
  const int64_t tiles_sk = (int64_t)a.m_tiles * ((N + bn_sk - 1) / bn_sk);
  const size_t sk_ws = sk_workspace(sms);
  // stream-K is opt-in (engram_set_gemm_schedule(2)): measured slower than data-parallel so far
  bool sk = g_sched_override == 2 && a.num_kb >= 2 && tiles_sk < 2 * (int64_t)sms;
  if (g_bn_override > 0 && g_bn_override != bn_sk) sk = false;
  if (sk && ws_bytes < sk_ws) sk = false;       // no room for the flags: data-parallel
  a.stream_k = sk ? 1 : 0;
  a.BN = sk ? bn_sk : (g_bn_override > 0 ? g_bn_override : pick_bn_dp(a.m_tiles, N, sms));
  a.n_tiles = (N + a.BN - 1) / a.BN;
  const int64_t n_tiles_total = (int64_t)a.m_tiles * a.n_tiles;
  if (n_tiles_total > 0x7fffffff) return false;
  a.total_units = n_tiles_total * a.num_kb;
  if (sk) {
    P.grid = a.total_units < sms ? (int)a.total_units : sms;
  } else {
    P.grid = n_tiles_total < sms ? (int)n_tiles_total : sms;
  }
  a.stage_bytes = a.msub * kATileBytes + a.BN * kBK * 2;
  a.stages = (kSmemBudget - 1024 - kEpiBytes - (int)sizeof(Ctl)) / a.stage_bytes;
  if (a.stages > kMaxStages) a.stages = kMaxStages;
  if (a.stages < 2) return false;
  a.acc_stride = pow2_at_least((uint32_t)a.BN);
  a.tmem_cols = a.acc_stride * 2;              // two accumulators (chains) per item
  if (a.tmem_cols > 512) return false;
  a.idesc = (1u << 4)                          // accumulate in f32
            | (1u << 7) | (1u << 10)           // A and B are bf16
            | ((uint32_t)(a.BN >> 3) << 17)    // N
            | ((uint32_t)(128 >> 4) << 24);    // M = 128; A and B K-major (bits 15, 16 = 0)
  P.smem = 1024 + a.stages * a.stage_bytes + kEpiBytes + (int)sizeof(Ctl);
  P.ws_needed = sk ? sk_ws : 0;
  return true;
}

}  // namespace

void set_gemm_bn_override(int bn) { g_bn_override = bn; }
void set_gemm_schedule_override(int s) { g_sched_override = s; }

// Workspace that lets the projection of this shape use the stream-K schedule (0 if it never would)
size_t gemm_workspace_bytes(int64_t M, int K, int N) {
  Plan P;
  const int saved = g_sched_override;
  g_sched_override = 2;
  const bool ok = plan_gemm(M, K, N, num_sms(), (size_t)-1, P);
  g_sched_override = saved;
  return ok ? P.ws_needed : 0;
}

int launch_gemm(const GemmParams& p, cudaStream_t stream, bool pdl) {
  Plan P;
  if (!plan_gemm(p.M, p.K, p.N, num_sms(), p.workspace != nullptr ? p.ws_bytes : 0, P)) {
    set_error("engram_project: no tile plan fits (T %lld, K %d, N %d)", (long long)p.M, p.K, p.N);
    return ENGRAM_EINVAL;
  }
  GemmArgs a = P.a;
  a.err = p.err;
  if (a.stream_k) {
    uint8_t* ws = static_cast<uint8_t*>(p.workspace);
    a.flags = reinterpret_cast<unsigned long long*>(ws);
    a.epoch = g_epoch.fetch_add(1) & 0xffffffffull;
  }
  static bool configured[64] = {false};     // the attribute is per device
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(wkv_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBudget);
    if (e != cudaSuccess) return fail_cuda(e, "engram_project: cudaFuncSetAttribute");
    if (dev >= 0 && dev < 64) configured[dev] = true;
  }
  CUtensorMap mA, mB, mD;
  if (!make_map(&mA, p.A, p.M, p.K, 128) || !make_map(&mB, p.B, p.N, p.K, (uint32_t)a.BN) ||
      !make_map_f32(&mD, p.D, p.M, p.N)) {
    set_error("engram_project: cuTensorMapEncodeTiled failed (driver entry point missing or bad layout)");
    return ENGRAM_ECUDA;
  }
  cudaError_t e = launch_k(wkv_gemm_kernel, dim3((unsigned)P.grid), dim3(kThreads), (size_t)P.smem, stream, pdl, mA,
                           mB, mD, p.D, a);
  if (e != cudaSuccess) return fail_cuda(e, "engram_project: launch");
  return ENGRAM_OK;
}

}  // namespace engram
