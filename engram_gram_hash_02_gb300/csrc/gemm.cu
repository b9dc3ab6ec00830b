// Stage 3: the wkv projection kv[T, N] = A[T, K] * wkv[N, K]^T on tcgen05 tensor cores.
//
// The projection of the vLLM "deepseek_v41.common.engram" page (Engram.__init__: wkv maps
// n_hash_cols*head_dim -> dim*(hc+1); Engram.forward) and of the Atlas "engram_v41" page
// (stage 3: dense bf16 GEMM). bf16 operands, fp32 accumulation in tensor memory, fp32 out.
//
// One CTA computes a tile of up to 256 rows (two 128-row accumulators) x BN columns:
//   warp 0      TMA producer: 128B-swizzled K-major tiles of A (128 rows x 64) and of wkv
//               (BN rows x 64) into a ring of shared-memory stages, mbarrier complete_tx. Under
//               programmatic dependent launch the first ring of wkv tiles is requested before
//               waiting for the kernel that writes A.
//   warp 1      allocates tensor memory; one lane issues tcgen05.mma (M=128, N=BN, K=16,
//               kind::f16) per 16-wide k step and releases a stage with tcgen05.commit.
//   warps 2..5  epilogue: tcgen05.ld of the fp32 accumulator (each warp its 32-lane quarter),
//               16-byte stores of fp32 kv (kept in fp32 for the gate's reductions).
// Both tiles of a 256-row block share each wkv tile, so wkv is read from memory once per
// column block. BN is picked per shape so the number of tiles fills the SMs in few waves.
//
// Every mbarrier wait is bounded (~2 s of SM clock cycles); on expiry the CTA raises an abort
// flag, reports ENGRAM_ERR_PIPE_TIMEOUT, drains its in-flight copies and MMAs (again
// bounded), frees its tensor memory and exits.
#include <cuda.h>

#include <mutex>

#include "internal.cuh"

namespace engram {
namespace {

constexpr int kBK = 64;                    // k elements per stage (128 bytes = one swizzle row)
constexpr int kUmmaK = 16;                 // k per tcgen05.mma for 16-bit operands
constexpr int kThreads = 192;
constexpr int kMaxStages = 8;
constexpr int kATileBytes = 128 * kBK * 2;  // 16 KB
constexpr uint64_t kWaitLimitCycles = 4000000000ull;  // wait bound in SM cycles: ~2 s at 2 GHz
constexpr int kSmemBudget = 232448;        // 227 KB opt-in maximum per CTA

struct Ctl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t acc_full;
  uint32_t tmem_base;
  int32_t abort_flag;
};

struct GemmArgs {
  int32_t M, K, N;
  int32_t cluster;
  int32_t BN, msub, stages, num_kb;
  int32_t m_tiles, n_tiles, group_m;
  int32_t stage_bytes;
  uint32_t idesc;
  uint32_t tmem_cols, acc_stride;
  int32_t* err;
};

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
__device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int32_t* abort_flag,
                                       int32_t* err, uint64_t limit_cycles) {
  if (mbar_try_wait(bar, parity)) return true;
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
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

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

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// A slice multicast into the same offset of every CTA in `mask`, each signalling its own barrier
__device__ __forceinline__ void tma_load_2d_mc(uint32_t dst, const CUtensorMap* map, uint32_t bar, int32_t x,
                                               int32_t y, uint16_t mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "h"(mask)
      : "memory");
}
// release a stage in every CTA of the cluster once this CTA's MMAs have read it
__device__ __forceinline__ void tc_commit_mc(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
wkv_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                float* __restrict__ D, const GemmArgs a) {
  const int c = a.cluster;                     // CTAs sharing one row block (launch cluster size)
  // A timeout anywhere in an earlier launch sharing the flag word voids the result: skip the
  // work instead of waiting out the time limits again. (Clustered CTAs must all take part.)
  if (c == 1 && a.err != nullptr && (*reinterpret_cast<volatile int32_t*>(a.err) & ENGRAM_ERR_PIPE_TIMEOUT)) return;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t tiles = (raw_base + 1023u) & ~1023u;          // swizzled tiles need 1 KB alignment
  Ctl* ctl = reinterpret_cast<Ctl*>(smem_raw + (tiles - raw_base) + a.stages * a.stage_bytes);
  volatile int32_t* abort_flag = &ctl->abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = c > 1 ? cluster_ctarank() : 0;
  const uint16_t all_ctas = (uint16_t)((1u << c) - 1u);

  // grouped raster over clusters: consecutive clusters sweep group_m row blocks of one group of
  // c column blocks; the CTAs of a cluster share the row block and take adjacent column blocks
  const int ct = blockIdx.x / c;
  const int n_clusters = a.n_tiles / c;        // n_tiles is padded to a multiple of c
  const int per_group = a.group_m * n_clusters;
  const int first_m = (ct / per_group) * a.group_m;
  const int gsize = min(a.m_tiles - first_m, a.group_m);
  const int in_group = ct % per_group;
  const int m_blk = first_m + in_group % gsize;
  const int n_blk = (in_group / gsize) * c + (int)rank;
  const int m0 = m_blk * 128 * a.msub;
  const int n0 = n_blk * a.BN;
  const int a_rows = 128 / c;                  // rows of each 128-row A tile this CTA loads

  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(smem_u32(&ctl->full[s]), 1);
      mbar_init(smem_u32(&ctl->empty[s]), (uint32_t)c);   // one release per consumer in the cluster
    }
    mbar_init(smem_u32(&ctl->acc_full), 1);
    ctl->abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&ctl->tmem_base)),
                 "r"(a.tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  if (c > 1) cluster_sync_all();               // peers' barriers exist before anyone multicasts
  else __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      auto load_a = [&](int kb) {
        const int s = kb % a.stages;
        const uint32_t full = smem_u32(&ctl->full[s]);
        const uint32_t st = tiles + (uint32_t)(s * a.stage_bytes);
        for (int ms = 0; ms < a.msub; ++ms) {
          const uint32_t dst = st + ms * kATileBytes + rank * (uint32_t)(a_rows * kBK * 2);
          const int y = m0 + ms * 128 + (int)rank * a_rows;
          if (c > 1) tma_load_2d_mc(dst, &tmA, full, kb * kBK, y, all_ctas);
          else tma_load_2d(dst, &tmA, full, kb * kBK, y);
        }
      };
      auto load_b = [&](int kb) {
        const int s = kb % a.stages;
        const uint32_t full = smem_u32(&ctl->full[s]);
        const uint32_t st = tiles + (uint32_t)(s * a.stage_bytes);
        mbar_expect_tx(full, (uint32_t)a.stage_bytes);
        tma_load_2d(st + a.msub * kATileBytes, &tmB, full, kb * kBK, n0);
      };
      // wkv does not come from the preceding kernel: fill the ring's weight halves before waiting
      // for the gathered rows (A) to be complete
      const int early = a.num_kb < a.stages ? a.num_kb : a.stages;
      for (int kb = 0; kb < early; ++kb) load_b(kb);
      pdl_wait();
      pdl_trigger();
      for (int kb = 0; kb < early; ++kb) load_a(kb);
      int issued = early;
      bool ok = true;
      for (int kb = early; kb < a.num_kb; ++kb) {
        const int s = kb % a.stages;
        const uint32_t ph = (uint32_t)(kb / a.stages) & 1u;
        // every consumer in the cluster has released stage s (the A slices land in all of them)
        if (!mbar_wait(smem_u32(&ctl->empty[s]), ph ^ 1u, abort_flag, a.err, kWaitLimitCycles)) {
          ok = false;
          break;
        }
        load_b(kb);
        load_a(kb);
        issued = kb + 1;
      }
      if (ok) {
        // producer tail: wait until every consumer in the cluster has released the last stages,
        // so no peer's release can arrive here after this CTA has exited
        for (int kb = a.num_kb; kb < a.num_kb + a.stages; ++kb) {
          const int s = kb % a.stages;
          const uint32_t ph = (uint32_t)(kb / a.stages) & 1u;
          if (!mbar_wait(smem_u32(&ctl->empty[s]), ph ^ 1u, abort_flag, a.err, kWaitLimitCycles)) break;
        }
      } else {
        // drain: the copies still in flight must land before shared memory goes away
        const int first = issued > a.stages ? issued - a.stages : 0;
        for (int kb = first; kb < issued; ++kb) {
          const int s = kb % a.stages;
          const uint32_t ph = (uint32_t)(kb / a.stages) & 1u;
          volatile int32_t never = 0;
          mbar_wait(smem_u32(&ctl->full[s]), ph, &never, nullptr, kWaitLimitCycles / 4);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      for (int kb = 0; kb < a.num_kb; ++kb) {
        const int s = kb % a.stages;
        const uint32_t ph = (uint32_t)(kb / a.stages) & 1u;
        if (!mbar_wait(smem_u32(&ctl->full[s]), ph, abort_flag, a.err, kWaitLimitCycles)) break;
        tc_fence_after();
        const uint32_t st = tiles + (uint32_t)(s * a.stage_bytes);
        const uint32_t b_addr = st + (uint32_t)(a.msub * kATileBytes);
#pragma unroll
        for (int k = 0; k < kBK / kUmmaK; ++k) {
          const uint64_t bdesc = smem_desc_sw128(b_addr + k * kUmmaK * 2);
          for (int ms = 0; ms < a.msub; ++ms) {
            const uint64_t adesc = smem_desc_sw128(st + ms * kATileBytes + k * kUmmaK * 2);
            tc_mma(tmem + ms * a.acc_stride, adesc, bdesc, a.idesc, (kb | k) != 0 ? 1u : 0u);
          }
        }
        if (c > 1) tc_commit_mc(smem_u32(&ctl->empty[s]), all_ctas);
        else tc_commit(smem_u32(&ctl->empty[s]));   // stage free once these MMAs have read it
      }
      tc_commit(smem_u32(&ctl->acc_full));     // accumulators final (or drained, on abort)
    }
  } else {
    // ---------------- epilogue: TMEM -> registers -> fp32 kv ----------------
    const int q = warp & 3;                    // TMEM lane quarter this warp may access
    pdl_wait();                                // kv may still be read by an earlier kernel
    const bool ok = mbar_wait(smem_u32(&ctl->acc_full), 0, abort_flag, a.err, kWaitLimitCycles);
    tc_fence_after();
    if (ok && *abort_flag == 0) {
      for (int ms = 0; ms < a.msub; ++ms) {
        const int64_t row = (int64_t)m0 + ms * 128 + q * 32 + lane;
        const bool row_ok = row < a.M;
        float* drow = D + row * (int64_t)a.N;
        const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(ms * a.acc_stride);
        for (int c0 = 0; c0 < a.BN; c0 += 32) {
          uint32_t r[32];
          const bool two = c0 + 16 < a.BN;
          tmem_ld16(tbase + c0, *reinterpret_cast<uint32_t(*)[16]>(&r[0]));
          if (two) tmem_ld16(tbase + c0 + 16, *reinterpret_cast<uint32_t(*)[16]>(&r[16]));
          tmem_ld_wait();
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int col = n0 + c0 + 16 * h;
            if (row_ok && col < a.N && (h == 0 || two)) {
              uint4* dst = reinterpret_cast<uint4*>(drow + col);
              dst[0] = make_uint4(r[16 * h + 0], r[16 * h + 1], r[16 * h + 2], r[16 * h + 3]);
              dst[1] = make_uint4(r[16 * h + 4], r[16 * h + 5], r[16 * h + 6], r[16 * h + 7]);
              dst[2] = make_uint4(r[16 * h + 8], r[16 * h + 9], r[16 * h + 10], r[16 * h + 11]);
              dst[3] = make_uint4(r[16 * h + 12], r[16 * h + 13], r[16 * h + 14], r[16 * h + 15]);
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    if (*abort_flag) {
      // make sure no MMA is still writing the accumulators we are about to free
      volatile int32_t never = 0;
      mbar_wait(smem_u32(&ctl->acc_full), 0, &never, nullptr, kWaitLimitCycles / 4);
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

int g_bn_override = 0;       // engram_set_gemm_tile
int g_cluster_override = 0;  // engram_set_gemm_cluster

int pick_bn(int64_t m_tiles, int N, int sms) {
  if (g_bn_override > 0) return g_bn_override;
  int best = 256;
  double best_cost = 1e300;
  for (int bn = 256; bn >= 64; bn -= 16) {
    const int64_t tiles = m_tiles * ((N + bn - 1) / bn);
    const int64_t waves = (tiles + sms - 1) / sms;
    // a wave costs about its tile width plus a fixed share for the A operand and setup
    const double cost = (double)waves * (bn + 48);
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = bn;
    }
  }
  return best;
}

uint32_t pow2_at_least(uint32_t x) {
  uint32_t p = 32;
  while (p < x) p <<= 1;
  return p;
}

cudaError_t launch(const CUtensorMap& mA, const CUtensorMap& mB, float* D, const GemmArgs& a, int64_t grid,
                   int smem, cudaStream_t stream, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)a.cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, wkv_gemm_kernel, mA, mB, D, a);
}

// Largest cluster (<= 4) whose clusters all fit on the GPU at once, or 2 when more than one
// wave is needed anyway; 1 when there is only one column tile.
int pick_cluster(int n_tiles, int64_t m_tiles, int smem) {
  if (g_cluster_override > 0) return g_cluster_override;
  if (n_tiles < 2) return 1;
  int best = 1;
  for (int c = 2; c <= 4; c *= 2) {
    if (n_tiles < c) break;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)c, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)c;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int active = 0;
    if (cudaOccupancyMaxActiveClusters(&active, wkv_gemm_kernel, &cfg) != cudaSuccess || active <= 0) {
      cudaGetLastError();
      break;
    }
    const int64_t clusters = m_tiles * ((n_tiles + c - 1) / c);
    if (clusters <= active) best = c;          // one wave of clusters
    else if (c == 2) best = 2;                 // several waves: pairs still halve A's L2 reads
  }
  return best;
}

}  // namespace

void set_gemm_bn_override(int bn) { g_bn_override = bn; }
void set_gemm_cluster_override(int c) { g_cluster_override = c; }

int launch_gemm(const GemmParams& p, cudaStream_t stream, bool pdl) {
  const int sms = num_sms();
  GemmArgs a{};
  a.M = (int32_t)p.M;
  a.K = p.K;
  a.N = p.N;
  a.msub = p.M > 128 ? 2 : 1;
  a.m_tiles = (int32_t)((p.M + 128 * a.msub - 1) / (128 * a.msub));
  a.BN = pick_bn(a.m_tiles, p.N, sms);
  const int n_tiles = (p.N + a.BN - 1) / a.BN;
  a.group_m = 16;
  a.num_kb = (p.K + kBK - 1) / kBK;
  a.stage_bytes = a.msub * kATileBytes + a.BN * kBK * 2;
  const int ctl_bytes = (int)sizeof(Ctl);
  a.stages = (kSmemBudget - 1024 - ctl_bytes) / a.stage_bytes;
  if (a.stages > kMaxStages) a.stages = kMaxStages;
  if (a.stages < 2) {
    set_error("engram_project: tile of %d columns does not fit shared memory", a.BN);
    return ENGRAM_EINVAL;
  }
  a.acc_stride = pow2_at_least((uint32_t)a.BN);
  a.tmem_cols = a.acc_stride * a.msub;
  a.idesc = (1u << 4)                         // accumulate in f32
            | (1u << 7) | (1u << 10)          // A and B are bf16
            | ((uint32_t)(a.BN >> 3) << 17)   // N
            | ((uint32_t)(128 >> 4) << 24);   // M = 128; A and B K-major (bits 15, 16 = 0)
  a.err = p.err;
  const int smem = 1024 + a.stages * a.stage_bytes + ctl_bytes;

  static bool configured[64] = {false};     // the attribute is per device
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(wkv_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBudget);
    if (e != cudaSuccess) return fail_cuda(e, "engram_project: cudaFuncSetAttribute");
    e = cudaFuncSetAttribute(wkv_gemm_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return fail_cuda(e, "engram_project: cudaFuncSetAttribute (cluster)");
    if (dev >= 0 && dev < 64) configured[dev] = true;
  }
  a.cluster = pick_cluster(n_tiles, a.m_tiles, smem);
  a.n_tiles = ((n_tiles + a.cluster - 1) / a.cluster) * a.cluster;   // padded tiles store nothing

  CUtensorMap mA, mB;
  if (!make_map(&mA, p.A, p.M, p.K, (uint32_t)(128 / a.cluster)) || !make_map(&mB, p.B, p.N, p.K, (uint32_t)a.BN)) {
    set_error("engram_project: cuTensorMapEncodeTiled failed (driver entry point missing or bad layout)");
    return ENGRAM_ECUDA;
  }
  const int64_t grid = (int64_t)a.m_tiles * a.n_tiles;
  if (grid > 0x7fffffff) {
    set_error("engram_project: too many tiles");
    return ENGRAM_EINVAL;
  }
  cudaError_t e = launch(mA, mB, p.D, a, grid, smem, stream, pdl);
  if (e != cudaSuccess) return fail_cuda(e, "engram_project: launch");
  return ENGRAM_OK;
}

}  // namespace engram
