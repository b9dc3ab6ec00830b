// Stage 3, FP8 operand variant: kv[T, N] = A[T, K] * W[N, K]^T with both operands MXFP8 (e4m3
// codes plus one power-of-two scale byte per 32 values along K), on tcgen05 tensor cores with
// block scaling (tcgen05.mma kind::mxf8f6f4.block_scale.scale_vec::1X), fp32 out.
//
// The A operand is the FP8 table rows of the vLLM "deepseek_v41.common.engram" page
// (ParallelEngramEmbedding: float8_e4m3fn weight, ue8m0 scale per 32 values) gathered without
// dequantisation; W is wkv encoded the same way. Each product a * 2^sa * b * 2^sb is exact, so the
// result is the projection of the dequantised operands with fp32 accumulation.
//
// A persistent data-parallel kernel, one CTA per SM, 10 warps:
//   warp 0      TMA producer: 128B-swizzled K-major tiles of codes, 128 k per stage (one swizzle
//               row per matrix row): A (128 rows per half) and W (BN rows), plus the stage's scale
//               words of both (one contiguous run each in the [K/128][rows4] word layout, 1-D bulk
//               copies). Under programmatic dependent launch the first ring of W tiles and scales
//               is requested before waiting for the kernel that writes A.
//   warp 1      allocates all 512 tensor-memory columns; one lane issues the MMAs: per stage four
//               k steps of 32, step s reading scale byte s of each 32-bit scale word.
//   warps 2..5  epilogue: fp32 accumulators -> swizzled shared tile -> TMA bulk tensor store.
//   warps 6..9  scale writers: once a stage has landed, each warp moves its scale words from shared
//               memory into that stage's scale slot of its TMEM lane quarter with tcgen05.st. Layout
//               (measured on this part): A row m reads lane m, column m / 32 of its slot; B row n
//               reads, for accumulator lanes in quarter q, lane 32q + n % 32, column n / 32. So
//               every quarter holds lane r, column c = scale word of A row r + 32c (per 128-row
//               half) and of B row r + 32c.
// A single block of at most 112 tokens loads only the token rows that exist (rounded up to 16), so
// the ring gets deeper; the MMA's reads of the other rows see whatever shared memory follows and
// only feed accumulator rows that are never stored (all inside the CTA's allocation).
// Accumulators: two independent chains (the two 128-row halves of a 256-row tile, or for tiles of
// at most 128 rows the even and odd k steps, summed in the epilogue) when tensor memory allows,
// else one. All waits are bounded (~2 s of SM clock cycles); on expiry the CTA reports
// ENGRAM_ERR_PIPE_TIMEOUT, drains what is in flight (bounded), frees tensor memory and exits.
#include <mutex>

#include "tc_common.cuh"

namespace engram {
namespace {

constexpr int kStageK = 128;                 // k per stage: one 128-byte swizzle row of codes
constexpr int kThreads = 320;
constexpr int kGatherWarps = 4;              // operand gather: warps 10..13
constexpr int kThreadsGather = kThreads + 32 * kGatherWarps;
constexpr int kEpiThreads = 128;
constexpr int kMaxStages = 8;
constexpr int kATileBytes = 128 * kStageK;   // 16 KB: 128 rows x 128 codes
constexpr int kTmemCols = 512;

struct MxCtl {
  uint64_t full[kMaxStages];                 // TMA -> MMA: the stage's A and W codes landed
  uint64_t empty[kMaxStages];                // MMA -> TMA / scale writers: stage and scale slot read
  uint64_t sf_full[kMaxStages];              // scale writers -> MMA: the slot's scales are in TMEM
  uint64_t acc_full;
  uint64_t acc_empty;
  uint32_t tmem_base;
  int32_t abort_flag;
};

struct MxArgs {
  int32_t M, K, N;
  int32_t BN, msub, chains, stages, num_kb;
  int32_t m_tiles, n_tiles, group_m;
  int32_t a_rows;                            // token rows loaded per 128-row half (128, or fewer for one short block)
  int32_t a_bytes, b_bytes;
  int32_t stage_bytes;                       // A + W codes + both scale runs, rounded to 1 KB
  int32_t rows_a4, rows_b4;                  // rows of the scale word arrays (M, N rounded up to 4)
  uint32_t idesc;
  uint32_t acc_stride;                       // column of the second accumulator chain
  uint32_t sf_base, sf_slot_w, sfb_off;      // scale slots: base column, width, W's offset in a slot
  const uint32_t* sfa;                       // [M, K/128] scale words (bytes of 4 consecutive blocks)
  const uint32_t* sfb;                       // [N, K/128]
  int32_t* err;
  GateFuse gf;                               // gf.keys > 0: the gate's key sums instead of the keys
  // operand gather (gather warps): the token tile's FP8 rows straight from the table
  const int32_t* ids;                        // ids of token m at ids + m * ids_stride, one per column
  int64_t ids_stride;
  const uint8_t* table;                      // e4m3 codes [table_rows, D]
  int64_t table_rows;
  int32_t D;                                 // table row width, a multiple of 128
};

__device__ __forceinline__ void mx_tile_origin(const MxArgs& a, int tile, int& m0, int& n0) {
  const int per_group = a.group_m * a.n_tiles;
  const int first_m = (tile / per_group) * a.group_m;
  const int gsize = min(a.m_tiles - first_m, a.group_m);
  const int in_group = tile % per_group;
  m0 = (first_m + in_group % gsize) * 128 * a.msub;
  n0 = (in_group / gsize) * a.BN;
}

__device__ __forceinline__ void tc_mma_mx(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}
// 1-D bulk copy global -> shared, completing on an mbarrier (16-byte aligned, size a multiple of 16)
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void tmem_st4(uint32_t taddr, const uint32_t* v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(v[0]), "r"(v[1]),
               "r"(v[2]), "r"(v[3])
               : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t* v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
               "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

// kFused: the gate's key sums in the epilogue (MxArgs::gf). kGatherA: the token tiles are gathered
// from the table by four more warps (MxArgs::ids): warp 10 + w serves the ring stages s with
// s % 4 == w: for each row of the tile it reads the row's id, copies the row's 128 codes of the
// stage from the table with cp.async (16 bytes a lane, 8 lanes a row) into the 128B-swizzled
// position the MMA reads (16-byte piece i of row r at piece i ^ (r % 8)), waits for its copies,
// makes them visible to the tensor cores (proxy fence) and arrives on the stage's barrier (which
// then expects the producer's copies and this arrival). Invalid ids read a zero row. Separate
// instantiations, so the plain projection keeps its own register allocation.
template <bool kFused, bool kGatherA>
__global__ void __launch_bounds__(kGatherA ? kThreadsGather : kThreads, 1)
wkv_gemm_mx_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmD, float* __restrict__ D, const MxArgs a) {
  if (a.err != nullptr && (*reinterpret_cast<volatile int32_t*>(a.err) & ENGRAM_ERR_PIPE_TIMEOUT)) {
    pdl_wait();
    return;
  }
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t tiles = (raw_base + 1023u) & ~1023u;
  const uint32_t stage_bytes = (uint32_t)a.stage_bytes;
  const uint32_t sf_off = (uint32_t)(a.a_bytes + a.b_bytes);          // scale words within a stage
  const uint32_t sfb_words_off = (uint32_t)(a.msub * 128) * 4u;
  const uint32_t epi_stage = tiles + (uint32_t)a.stages * stage_bytes;
  MxCtl* ctl = reinterpret_cast<MxCtl*>(smem_raw + (epi_stage - raw_base) + kEpiBytes);
  volatile int32_t* abort_flag = &ctl->abort_flag;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_tiles_total = a.m_tiles * a.n_tiles;

  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(smem_u32(&ctl->full[s]), kGatherA ? 2 : 1);   // producer (+ the stage's gather warp)
      mbar_init(smem_u32(&ctl->empty[s]), 1);
      mbar_init(smem_u32(&ctl->sf_full[s]), 4);
    }
    mbar_init(smem_u32(&ctl->acc_full), 1);
    mbar_init(smem_u32(&ctl->acc_empty), kEpiThreads);
    ctl->abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 0 && lane == 0) {
    if (!kGatherA) prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmD);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&ctl->tmem_base)),
                 "n"(kTmemCols)
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
      // W codes and W scales (not written by the preceding kernel); the stage's barrier expects
      // every byte of the stage, including A's that load_a brings later
      auto load_b = [&](int it, int kb, int m0, int n0) {
        const int s = it % a.stages;
        const uint32_t full = smem_u32(&ctl->full[s]);
        const uint32_t st = tiles + (uint32_t)s * stage_bytes;
        const int rows_a = min(a.msub * 128, a.rows_a4 - m0);
        const int rows_b = min(a.BN, a.rows_b4 - n0);
        const int a_code_bytes = kGatherA ? 0 : a.a_bytes;          // gathered: cp.async, not counted
        mbar_expect_tx(full, (uint32_t)(a_code_bytes + a.b_bytes + 4 * rows_a + 4 * rows_b));
        tma_load_2d(st + (uint32_t)a.a_bytes, &tmB, full, kb * kStageK, n0);
        bulk_load(st + sf_off + sfb_words_off, a.sfb + (int64_t)kb * a.rows_b4 + n0, 4u * (uint32_t)rows_b, full);
      };
      auto load_a = [&](int it, int kb, int m0) {
        const int s = it % a.stages;
        const uint32_t full = smem_u32(&ctl->full[s]);
        const uint32_t st = tiles + (uint32_t)s * stage_bytes;
        if (!kGatherA)
          for (int ms = 0; ms < a.msub; ++ms) tma_load_2d(st + ms * kATileBytes, &tmA, full, kb * kStageK, m0 + ms * 128);
        const int rows_a = min(a.msub * 128, a.rows_a4 - m0);
        bulk_load(st + sf_off, a.sfa + (int64_t)kb * a.rows_a4 + m0, 4u * (uint32_t)rows_a, full);
      };
      // W does not come from the preceding kernel: fill the ring's W halves first
      int early = 0;
      for (int tile = blockIdx.x; tile < n_tiles_total && early < a.stages; tile += gridDim.x) {
        int m0, n0;
        mx_tile_origin(a, tile, m0, n0);
        for (int kb = 0; kb < a.num_kb && early < a.stages; ++kb) load_b(early++, kb, m0, n0);
      }
      pdl_wait();
      int it = 0, issued = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < n_tiles_total; tile += gridDim.x) {
        int m0, n0;
        mx_tile_origin(a, tile, m0, n0);
        if (tile + (int)gridDim.x >= n_tiles_total) pdl_trigger();   // last tile of this CTA
        for (int kb = 0; kb < a.num_kb; ++kb, ++it) {
          if (it < early) {
            load_a(it, kb, m0);
          } else {
            const int s = it % a.stages;
            const uint32_t ph = (uint32_t)(it / a.stages) & 1u;
            if (!mbar_wait(smem_u32(&ctl->empty[s]), ph ^ 1u, abort_flag, a.err, kWaitLimitCycles)) {
              ok = false;
              break;
            }
            load_b(it, kb, m0, n0);
            load_a(it, kb, m0);
          }
          issued = it + 1;
        }
      }
      if (!ok) {
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
      int n_items = 0, slot = 0;
      uint32_t round = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < n_tiles_total; tile += gridDim.x) {
        if (!mbar_wait(smem_u32(&ctl->acc_empty), (uint32_t)(n_items & 1) ^ 1u, abort_flag, a.err,
                       kWaitLimitCycles)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < a.num_kb; ++kb) {
          if (!mbar_wait(smem_u32(&ctl->full[slot]), round, abort_flag, a.err, kWaitLimitCycles) ||
              !mbar_wait(smem_u32(&ctl->sf_full[slot]), round, abort_flag, a.err, kWaitLimitCycles)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = tiles + (uint32_t)slot * stage_bytes;
          const uint64_t a0 = smem_desc_sw128(st);
          const uint64_t b0 = smem_desc_sw128(st + (uint32_t)a.a_bytes);
          const uint32_t sfa = tmem + a.sf_base + (uint32_t)slot * a.sf_slot_w;
          const uint32_t sfb = sfa + a.sfb_off;
#pragma unroll
          for (int k = 0; k < kStageK / 32; ++k) {
            // k step of 32 codes = 32 bytes = 2 in the encoded start address; scale byte k
            const uint32_t idk = a.idesc | ((uint32_t)k << 29) | ((uint32_t)k << 4);
            const uint64_t bdesc = b0 + (uint64_t)(2 * k);
            if (a.msub == 2) {
              const uint32_t acc = (kb > 0 || k > 0) ? 1u : 0u;
              tc_mma_mx(tmem, a0 + (uint64_t)(2 * k), bdesc, idk, sfa, sfb, acc);
              tc_mma_mx(tmem + a.acc_stride, a0 + (uint64_t)(2 * k + (kATileBytes >> 4)), bdesc, idk, sfa + 4, sfb, acc);
            } else if (a.chains == 2) {
              tc_mma_mx(tmem + (k & 1) * a.acc_stride, a0 + (uint64_t)(2 * k), bdesc, idk, sfa, sfb,
                        (kb > 0 || k > 1) ? 1u : 0u);
            } else {
              tc_mma_mx(tmem, a0 + (uint64_t)(2 * k), bdesc, idk, sfa, sfb, (kb > 0 || k > 0) ? 1u : 0u);
            }
          }
          tc_commit(smem_u32(&ctl->empty[slot]));   // stage and scale slot free once read
          if (++slot == a.stages) {
            slot = 0;
            round ^= 1u;
          }
        }
        tc_commit(smem_u32(&ctl->acc_full));
        ++n_items;
      }
      if (!ok) tc_commit(smem_u32(&ctl->acc_full));
    }
  } else if (warp < 6) {
    // ---------------- epilogue ----------------
    const int q = warp & 3;
    pdl_wait();                                // kv may still be read by an earlier kernel
    const uint32_t stg = epi_stage + (uint32_t)(q * kEpiWarpBytes);
    constexpr bool fused = kFused;
    auto prefetch_tile = [&](int tile) {       // a tile's stream rows into L2 during its main loop
      if (!fused || tile >= n_tiles_total) return;
      int pm0, pn0;
      mx_tile_origin(a, tile, pm0, pn0);
      if (pn0 < a.gf.keys) gate_prefetch_rows(a.gf, a.M, a.msub, q, lane, pm0, pn0, a.BN);
    };
    prefetch_tile(blockIdx.x);
    int n_items = 0;
    for (int tile = blockIdx.x; tile < n_tiles_total; tile += gridDim.x) {
      const bool ok = mbar_wait(smem_u32(&ctl->acc_full), (uint32_t)(n_items & 1), abort_flag, a.err,
                                kWaitLimitCycles);
      tc_fence_after();
      if (!ok || *abort_flag) break;
      int m0, n0;
      mx_tile_origin(a, tile, m0, n0);
      if (fused)
        fused_gate_epilogue(a.gf, &tmD, D, a.M, a.N, tmem, q, lane, stg, a.msub, a.msub == 1 && a.chains == 2,
                            a.acc_stride, a.BN, 1, m0, n0);
      else
        store_accumulators(&tmD, D, a.M, a.N, tmem, q, lane, stg, a.msub, a.msub == 1 && a.chains == 2,
                           a.acc_stride, a.BN, m0, n0, false);
      // the accumulators are read (every tcgen05.ld has completed): tensor memory may take the next
      // tile while this one's stores are in flight (a staging tile is reused only after its store
      // has read it)
      tc_fence_before();
      mbar_arrive(smem_u32(&ctl->acc_empty));
      ++n_items;
      prefetch_tile(tile + (int)gridDim.x);
    }
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    __syncwarp();
  } else if (kGatherA && warp >= 10) {
    // ---------------- operand gather: token rows from the table ----------------
    // Stage s is always served by warp 10 + s % 4, so a warp waits only for the consumption of
    // its own previous copy into that stage (a barrier phase never more than one ahead).
    pdl_wait();                                // the ids come from the hash kernel
    const int gw = warp - 10;
    const int lr = lane >> 3;                  // row of a group of four
    const int k16 = lane & 7;                  // 16-byte piece of the row's 128 codes
    const int rows = a.msub * 128;             // tile rows: lane L holds the ids of rows L + 32 i
    int it = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < n_tiles_total; tile += gridDim.x) {
      int m0, n0;
      mx_tile_origin(a, tile, m0, n0);
      for (int kb = 0; kb < a.num_kb; ++kb, ++it) {
        const int s = it % a.stages;
        if (s % kGatherWarps != gw) continue;
        const uint32_t ph = (uint32_t)(it / a.stages) & 1u;
        if (!mbar_wait(smem_u32(&ctl->empty[s]), ph ^ 1u, abort_flag, a.err, kWaitLimitCycles)) {
          ok = false;
          break;
        }
        const uint32_t st = tiles + (uint32_t)s * stage_bytes;
        const int kcode = kb * kStageK;         // the stage's first code in the token row
        const int col = kcode / a.D;
        const int x = kcode - col * a.D + 16 * k16;
        int32_t idl[8];                         // this lane's rows' ids, all requested at once
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int R = lane + 32 * i;          // row within the tile
          const int r = R & 127;
          const int64_t m = (int64_t)m0 + R;
          idl[i] = (R < rows && r < a.a_rows && m < a.M) ? __ldg(a.ids + m * a.ids_stride + col) : 0;
        }
#pragma unroll
        for (int g = 0; g < 64; ++g) {          // rows 4g .. 4g + 3, 8 lanes a row
          const int R = 4 * g + lr;
          const int32_t id = __shfl_sync(0xffffffffu, idl[g >> 3], R & 31);   // every lane takes part
          const int ms = R >> 7, r = R & 127;
          // rows past the tile's loaded rows or past the matrix: not loaded (never stored)
          if (R >= rows || r >= a.a_rows || (int64_t)m0 + R >= a.M) continue;
          const uint32_t dst = st + (uint32_t)(ms * kATileBytes + r * 128 + ((k16 ^ (r & 7)) << 4));
          const bool valid = id >= 0 && (int64_t)id < a.table_rows;
          const uint8_t* src = a.table + (valid ? (int64_t)id * a.D + x : 0);
          // 16 bytes, or (an id outside the table) 16 zero bytes: source size 0
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
                       : "memory");
          if (!valid && k16 == 0 && a.err != nullptr) atomicOr(a.err, ENGRAM_ERR_ROW_ID);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
        asm volatile("cp.async.wait_group 0;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // visible to the tensor cores
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctl->full[s]));
      }
    }
  } else if (warp < 10) {
    // ---------------- scale writers ----------------
    const int q = warp & 3;                    // TMEM lane quarter of this warp
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
    int slot = 0;
    uint32_t round = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < n_tiles_total; tile += gridDim.x) {
      int m0, n0;
      mx_tile_origin(a, tile, m0, n0);
      for (int kb = 0; kb < a.num_kb; ++kb) {
        // the stage (codes and scale words) has landed; its slot's previous MMAs are done, since
        // the producer waited for them before loading
        if (!mbar_wait(smem_u32(&ctl->full[slot]), round, abort_flag, a.err, kWaitLimitCycles)) {
          ok = false;
          break;
        }
        const uint32_t sw = tiles + (uint32_t)slot * stage_bytes + sf_off;   // this stage's scale words
        uint32_t va[8], vb[8];
        // A row m0 + 128h + 32c + lane, W row n0 + 32c + lane; rows past the matrix read scale 1.0
        // (their codes are zero-filled)
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int r = 128 * h + 32 * c + lane;
            uint32_t v = 0x7F7F7F7Fu;
            if (h < a.msub && m0 + r < a.M) asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(sw + 4u * r));
            va[4 * h + c] = v;
          }
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const int r = 32 * c + lane;
          uint32_t v = 0x7F7F7F7Fu;
          if (r < a.BN && n0 + r < a.N) asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(sw + sfb_words_off + 4u * r));
          vb[c] = v;
        }
        const uint32_t col = a.sf_base + (uint32_t)slot * a.sf_slot_w;
        tmem_st4(lane_base + col, &va[0]);
        if (a.msub == 2) tmem_st4(lane_base + col + 4, &va[4]);
        tmem_st8(lane_base + col + a.sfb_off, vb);
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctl->sf_full[slot]));
        if (++slot == a.stages) {
          slot = 0;
          round ^= 1u;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    if (*abort_flag) {
      volatile int32_t never = 0;
      for (int ph = 0; ph < 2; ++ph)
        mbar_wait(smem_u32(&ctl->acc_full), (uint32_t)ph, &never, nullptr, kWaitLimitCycles / 8);
    }
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTmemCols) : "memory");
  }
}

// one stage: A and W code tiles, then A's and W's scale words; 1 KB aligned for the next stage
int mx_stage_bytes(int a_bytes, int msub, int bn) {
  return ((a_bytes + bn * kStageK + 4 * (msub * 128 + bn)) + 1023) & ~1023;
}

// Bytes from the ring's start to the end of the last stage's MMA reads: a full 128-row token tile
// per half (whatever was loaded), and the W tile after the loaded token rows.
int mx_mma_read_end(const MxArgs& a) {
  const int a_read = a.msub * kATileBytes;
  const int b_end = a.a_bytes + a.b_bytes;
  return (a.stages - 1) * a.stage_bytes + (a_read > b_end ? a_read : b_end);
}

struct MxPlan {
  MxArgs a;
  int grid, smem;
};

int g_mx_bn_override = 0;

// tile width: few waves of tiles over the SMs, within tensor memory (accumulator chains plus one
// scale slot per stage) and shared memory
bool plan_mx(int64_t M, int K, int N, int sms, MxPlan& P) {
  MxArgs& a = P.a;
  a = MxArgs{};
  a.M = (int32_t)M;
  a.K = K;
  a.N = N;
  a.msub = M > 128 ? 2 : 1;
  a.m_tiles = (int32_t)((M + 128 * a.msub - 1) / (128 * a.msub));
  a.num_kb = K / kStageK;
  a.group_m = 16;
  a.a_rows = (a.msub == 1 && a.m_tiles == 1 && M <= 112) ? (int32_t)((M + 15) / 16 * 16) : 128;
  a.a_bytes = a.msub * a.a_rows * kStageK;
  a.sf_slot_w = (uint32_t)(4 * a.msub + 8);
  a.sfb_off = (uint32_t)(4 * a.msub);
  const int avail = kSmemBudget - 1024 - kEpiBytes - (int)sizeof(MxCtl);
  int best = 0, best_chains = 0, best_stages = 0;
  double best_cost = 1e300;
  for (int bn = 256; bn >= 16; bn -= 16) {
    if (g_mx_bn_override > 0 && bn != g_mx_bn_override) continue;
    int stages = avail / mx_stage_bytes(a.a_bytes, a.msub, bn);
    if (stages > kMaxStages) stages = kMaxStages;
    if (stages < 2) continue;
    const int stride = ((bn + 31) / 32) * 32;
    int chains = 2;
    if (2 * stride + stages * (int)a.sf_slot_w > kTmemCols) {
      if (a.msub == 2) continue;             // both halves need their own accumulator
      chains = 1;
      if (stride + stages * (int)a.sf_slot_w > kTmemCols) continue;
    }
    const int64_t tiles = (int64_t)a.m_tiles * ((N + bn - 1) / bn);
    const int64_t waves = (tiles + sms - 1) / sms;
    const double cost = (double)waves * (bn + 48);
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = bn;
      best_chains = chains;
      best_stages = stages;
    }
  }
  if (best == 0) return false;
  a.BN = best;
  a.chains = best_chains;
  a.stages = best_stages;
  a.b_bytes = a.BN * kStageK;
  a.stage_bytes = mx_stage_bytes(a.a_bytes, a.msub, a.BN);
  a.rows_a4 = (int32_t)((M + 3) & ~(int64_t)3);
  a.rows_b4 = (N + 3) & ~3;
  a.acc_stride = (uint32_t)(((a.BN + 31) / 32) * 32);
  a.sf_base = (uint32_t)a.chains * a.acc_stride;
  a.n_tiles = (N + a.BN - 1) / a.BN;
  const int64_t tiles = (int64_t)a.m_tiles * a.n_tiles;
  if (tiles > 0x7fffffff) return false;
  P.grid = tiles < sms ? (int)tiles : sms;
  a.idesc = ((uint32_t)(a.BN >> 3) << 17)    // N
            | (1u << 23)                     // scales are UE8M0
            | ((uint32_t)(128 >> 4) << 24);  // M = 128; A and W e4m3 (format 0), K-major
  P.smem = 1024 + a.stages * a.stage_bytes + kEpiBytes + (int)sizeof(MxCtl);
  // the last stage's MMA reads (a full 128-row token tile per half, whatever was loaded) end
  // inside the allocation; 1024 bytes are kept for aligning the ring
  if (mx_mma_read_end(a) > P.smem - 1024 || P.smem > kSmemBudget) return false;
  return true;
}

}  // namespace

void set_gemm_mx_bn_override(int bn) { g_mx_bn_override = bn; }

bool gemm_mx_plan_info(int64_t M, int K, int N, int sms, EngramProjectPlan* out) {
  MxPlan P;
  if (!plan_mx(M, K, N, sms, P)) return false;
  const MxArgs& a = P.a;
  *out = EngramProjectPlan{};
  out->grid = P.grid;
  out->threads = kThreads;
  out->smem_bytes = P.smem;
  out->tile_rows = 128 * a.msub;
  out->tile_cols = a.BN;
  out->split = 1;
  out->token_rows_loaded = a.a_rows;
  out->stages = a.stages;
  out->stage_bytes = a.stage_bytes;
  out->tmem_cols = kTmemCols;
  out->stream_k = 0;
  out->mma_read_end = mx_mma_read_end(a);
  out->smem_avail = P.smem - 1024;
  return true;
}

int launch_gemm_mx(const GemmMxParams& p, cudaStream_t stream, bool pdl) {
  MxPlan P;
  if (!plan_mx(p.M, p.K, p.N, num_sms(), P)) {
    set_error("engram_project_mxfp8: no tile plan fits (T %lld, K %d, N %d)", (long long)p.M, p.K, p.N);
    return ENGRAM_EINVAL;
  }
  MxArgs a = P.a;
  a.err = p.err;
  a.gf = p.gf;
  const bool gather = p.ids != nullptr;
  if (gather) {
    if (p.D < 128 || p.D % 128 != 0 || p.table == nullptr) {
      set_error("engram_project_mxfp8: the operand gather needs table rows a multiple of 128 wide (got %d)", p.D);
      return ENGRAM_EINVAL;
    }
    a.ids = p.ids;
    a.ids_stride = p.ids_stride;
    a.table = p.table;
    a.table_rows = p.table_rows;
    a.D = p.D;
  }
  if (a.gf.keys > 0 && a.gf.tile_cols != a.BN) {
    set_error("engram_project_mxfp8: fused gate planned for tiles of %d columns, the projection runs %d",
              a.gf.tile_cols, a.BN);
    return ENGRAM_EINVAL;
  }
  a.sfa = reinterpret_cast<const uint32_t*>(p.SA);
  a.sfb = reinterpret_cast<const uint32_t*>(p.SB);
  static PerContextOnce attr;               // the attribute belongs to the context's module
  cudaError_t ae = attr.run([] {
    for (auto k : {wkv_gemm_mx_kernel<false, false>, wkv_gemm_mx_kernel<true, false>, wkv_gemm_mx_kernel<false, true>,
                   wkv_gemm_mx_kernel<true, true>}) {
      cudaError_t e1 = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBudget);
      if (e1 != cudaSuccess) return e1;
    }
    return cudaSuccess;
  });
  if (ae != cudaSuccess) return fail_cuda(ae, "engram_project_mxfp8: cudaFuncSetAttribute");
  CUtensorMap mA, mB, mD;
  // (with the operand gather the A map is not used; it is made over the table so that it is valid)
  const bool map_a = gather ? make_map_u8(&mA, p.table, p.table_rows, p.D, 1)
                            : make_map_u8(&mA, p.A, p.M, p.K, (uint32_t)a.a_rows);
  if (!map_a || !make_map_u8(&mB, p.B, p.N, p.K, (uint32_t)a.BN) || !make_map_f32(&mD, p.Dout, p.M, p.N)) {
    set_error("engram_project_mxfp8: cuTensorMapEncodeTiled failed (driver entry point missing or bad layout)");
    return ENGRAM_ECUDA;
  }
  auto kernel = a.gf.keys > 0 ? (gather ? wkv_gemm_mx_kernel<true, true> : wkv_gemm_mx_kernel<true, false>)
                               : (gather ? wkv_gemm_mx_kernel<false, true> : wkv_gemm_mx_kernel<false, false>);
  cudaError_t e = launch_k(kernel, dim3((unsigned)P.grid), dim3(gather ? kThreadsGather : kThreads), (size_t)P.smem,
                           stream, pdl, mA, mB, mD, p.Dout, a);
  if (e != cudaSuccess) return fail_cuda(e, "engram_project_mxfp8: launch");
  return ENGRAM_OK;
}

}  // namespace engram
