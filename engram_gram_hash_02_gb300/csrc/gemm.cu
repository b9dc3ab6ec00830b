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
// (summed in the epilogue), or the two column halves of a split tile (below).
//
// Short token blocks (one block of at most 112 tokens): the token tile holds only the rows that
// exist, rounded up to 16, so a stage is mostly weight tile and the ring gets deeper. The MMA
// still reads 128 rows; rows past the tile read whatever shared memory follows (the weight tile,
// later stages), which only feeds accumulator rows that are never stored (row m of the product
// depends on row m of A alone), and every such read stays inside the CTA's allocation.
//
// Split tiles (129..256 tokens, when wkv is wide): instead of one CTA per 256-row x BN tile, two
// CTAs per 128-row x 2*BN tile pair up on each column block (consecutive CTAs, so their wkv tiles
// are read from HBM once and served twice by L2). A stage then holds a 16 KB token tile and a
// 2*BN-row weight tile instead of 32 KB and BN rows: twice the weight bytes in flight per SM in
// the same shared memory.
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

#include "tc_common.cuh"

namespace engram {
namespace {

constexpr int kBK = 64;                    // k elements per stage (128 bytes = one swizzle row)
constexpr int kUmmaK = 16;                 // k per tcgen05.mma for 16-bit operands
constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;
constexpr int kMaxStages = 8;
constexpr int kATileBytes = 128 * kBK * 2;  // 16 KB
constexpr unsigned long long kFlagMagic = 0x5EA5C0DEull;


struct GemmArgs {
  int32_t M, K, N;
  int32_t BN, msub, stages, num_kb;
  int32_t nsplit;                          // 2: tile = two column halves of BN/2, one MMA each
  int32_t a_rows, a_bytes;                 // token rows loaded per 128-row half, bytes of the token tile
  int32_t m_tiles, n_tiles, group_m;
  int32_t stage_bytes;
  uint32_t idesc;
  uint32_t tmem_cols, acc_stride;
  int32_t acc_sets;                        // 2: two accumulator sets, items alternate (epilogue overlaps MMAs)
  uint32_t set_stride;                     // tensor-memory columns between the sets
  int32_t stream_k;                        // 0: data-parallel tiles, 1: stream-K
  int64_t total_units;                     // tiles * num_kb
  unsigned long long* flags;               // [grid] (stream-K)
  unsigned long long epoch;
  int32_t* err;
  GateFuse gf;                             // gf.keys > 0: the gate's key sums instead of the keys
  GateOverlap go;                          // the gate overlapped with the projection (kOverlap)
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

constexpr int kGateThreads = 256;            // gate warps of the overlapped gate (warps 6..13)
constexpr int kThreadsOverlap = kThreads + kGateThreads;
constexpr int kGateVec = 8;                  // float4 chunks of a row per gate thread (H <= 8192)
__device__ __forceinline__ void gate_bar() {  // the 256 gate threads only
  asm volatile("bar.sync 2, %0;" ::"n"(kGateThreads) : "memory");
}
__device__ __forceinline__ float gbf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float gbf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Shared state of the gate warps: the warps' partial sums (two buffers: item parity) and the
// go/stop decision of thread 0, so that every gate thread leaves the loop at the same item.
struct GateShared {
  float red[2][kGateThreads / 32][3];
  int go[2];                                 // by the parity of the row-block waits
};

struct Ctl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t acc_full[2];                    // MMA -> epilogue: an accumulator set's item is final
  uint64_t acc_empty[2];                   // epilogue -> MMA: the set is drained
  uint32_t tmem_base;
  int32_t abort_flag;
  uint32_t published;                      // stream-K: epilogue warps done with the current segment
  GateShared gate;                         // the overlapped gate's warps
};

// The gate warps of the overlapped gate: (token, stream) items round-robin over the CTAs in token
// order; before the items of a row block, thread 0 waits (bounded) until every tile of that block
// has been stored (the epilogues count them in a.go.done), then the 256 threads load the stream
// row, the key and the value into registers, reduce, and write h + g * v in place.
__device__ __forceinline__ void overlapped_gate(const GemmArgs& a, const float* kv, GateShared* gs,
                                                volatile int32_t* abort_flag) {
  const GateOverlap& g = a.go;
  const int gt = threadIdx.x - kThreads;     // 0 .. 255
  const int gl = gt & 31, gw = gt >> 5;
  const int H = g.H, H4 = H >> 2, hc = g.hc;
  const int64_t N = a.N;
  const int rows_blk = 128 * a.msub;
  const int64_t items = (int64_t)a.M * hc;
  int ready = -1;
  int n = 0;                                 // items processed: parity of the partial-sum buffer
  int waits = 0;                             // row-block waits: parity of the go word
  // Both buffers are double: a thread writes buffer p for the next use only after a gate barrier
  // that every gate thread reached after its last read of buffer p.
  for (int64_t item = blockIdx.x; item < items; item += gridDim.x) {
    const int64_t t = item / hc;
    const int j = (int)(item - t * hc);
    if (g.mask != nullptr && __ldg(g.mask + t) == 0) continue;   // masked: not read or written
    const int blk = (int)(t / rows_blk);
    if (blk > ready) {                       // the row block's kv must be complete
      if (gt == 0) {
        int ok = 1;
        const uint64_t t0 = clock64();
        for (uint32_t it = 0;; ++it) {
          uint32_t v;
          asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(g.done + blk) : "memory");
          if (v >= (uint32_t)(a.n_tiles * (kEpiThreads / 32))) break;   // every epilogue warp of every tile
          __nanosleep(128);
          if ((it & 15u) == 15u && (*abort_flag || (uint64_t)clock64() - t0 > kWaitLimitCycles)) {
            if (!*abort_flag && a.err != nullptr) atomicOr(a.err, ENGRAM_ERR_PIPE_TIMEOUT);
            *abort_flag = 1;
            ok = 0;
            break;
          }
        }
        __threadfence();
        gs->go[waits & 1] = ok;
      }
      gate_bar();
      const int go = gs->go[waits & 1];
      ++waits;
      if (!go) break;                        // the same answer in every gate thread
      ready = blk;
    }
    float4* hrow = reinterpret_cast<float4*>(g.streams + item * (int64_t)H);
    const float* kvrow = kv + t * N;
    const float4* krow = reinterpret_cast<const float4*>(kvrow + (int64_t)j * H);
    const float4* vrow = reinterpret_cast<const float4*>(kvrow + (int64_t)hc * H);
    const uint2* qrow = reinterpret_cast<const uint2*>(g.qw + (int64_t)j * H);
    const uint2* krw = reinterpret_cast<const uint2*>(g.kw + (int64_t)j * H);
    float4 x[kGateVec], v[kGateVec];
    float ssh = 0.f, ssk = 0.f, dot = 0.f;
    {
      float4 y[kGateVec];
#pragma unroll
      for (int m = 0; m < kGateVec; ++m) {
        const int c = gt + m * kGateThreads;
        if (c < H4) {
          x[m] = __ldcg(hrow + c);             // L2 only: kv was stored by other SMs in this kernel
          y[m] = __ldcg(krow + c);
          v[m] = __ldcg(vrow + c);
        }
      }
#pragma unroll
      for (int m = 0; m < kGateVec; ++m) {
        const int c = gt + m * kGateThreads;
        if (c < H4) {
          const uint2 qr = __ldg(qrow + c), kr = __ldg(krw + c);
          ssh = fmaf(x[m].x, x[m].x, ssh); ssh = fmaf(x[m].y, x[m].y, ssh);
          ssh = fmaf(x[m].z, x[m].z, ssh); ssh = fmaf(x[m].w, x[m].w, ssh);
          ssk = fmaf(y[m].x, y[m].x, ssk); ssk = fmaf(y[m].y, y[m].y, ssk);
          ssk = fmaf(y[m].z, y[m].z, ssk); ssk = fmaf(y[m].w, y[m].w, ssk);
          dot = fmaf(x[m].x * gbf16lo(qr.x), y[m].x * gbf16lo(kr.x), dot);
          dot = fmaf(x[m].y * gbf16hi(qr.x), y[m].y * gbf16hi(kr.x), dot);
          dot = fmaf(x[m].z * gbf16lo(qr.y), y[m].z * gbf16lo(kr.y), dot);
          dot = fmaf(x[m].w * gbf16hi(qr.y), y[m].w * gbf16hi(kr.y), dot);
        }
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      ssh += __shfl_xor_sync(0xffffffffu, ssh, off);
      ssk += __shfl_xor_sync(0xffffffffu, ssk, off);
      dot += __shfl_xor_sync(0xffffffffu, dot, off);
    }
    if (gl == 0) {
      gs->red[n & 1][gw][0] = ssh;
      gs->red[n & 1][gw][1] = ssk;
      gs->red[n & 1][gw][2] = dot;
    }
    gate_bar();
    float sa = 0.f, sb = 0.f, sc = 0.f;
    for (int w = 0; w < kGateThreads / 32; ++w) {   // the same order in every thread
      sa += gs->red[n & 1][w][0];
      sb += gs->red[n & 1][w][1];
      sc += gs->red[n & 1][w][2];
    }
    const float invH = 1.0f / (float)H;
    const float sv = sc * rsqrtf(sa * invH + g.eps) * rsqrtf(sb * invH + g.eps) / sqrtf((float)H);
    float ss = 0.f;                                  // sign(0) = 0
    if (sv > 0.f) ss = sqrtf(fmaxf(sv, g.clamp));
    else if (sv < 0.f) ss = -sqrtf(fmaxf(-sv, g.clamp));
    const float gate = 1.0f / (1.0f + expf(-ss));
#pragma unroll
    for (int m = 0; m < kGateVec; ++m) {
      const int c = gt + m * kGateThreads;
      if (c < H4)
        hrow[c] = make_float4(fmaf(gate, v[m].x, x[m].x), fmaf(gate, v[m].y, x[m].y), fmaf(gate, v[m].z, x[m].z),
                              fmaf(gate, v[m].w, x[m].w));
    }
    ++n;
  }
}

// kFused: the gate's key sums in the epilogue (GemmArgs::gf); a separate instantiation, so the
// plain projection keeps its own register allocation.
// kOverlap: eight more warps apply the gate to the tokens of finished row blocks while the tensor
// cores work on later tiles (GemmArgs::go).
template <bool kFused, bool kOverlap>
__global__ void __launch_bounds__(kOverlap ? kThreadsOverlap : kThreads, 1)
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
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&ctl->acc_full[b]), 1);
      mbar_init(smem_u32(&ctl->acc_empty[b]), kEpiThreads);
    }
    ctl->abort_flag = 0;
    ctl->published = 0;
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
        tma_load_2d(st + a.a_bytes, &tmB, full, kb * kBK, n0);
        if (a.nsplit == 2)
          tma_load_2d(st + a.a_bytes + (a.BN >> 1) * (kBK * 2), &tmB, full, kb * kBK, n0 + (a.BN >> 1));
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
      int set = 0;
      while (ok && sch.next(item)) {
        // the epilogue has drained this accumulator set's previous item (with two sets, the item
        // before last: its drain overlaps this item's MMAs)
        set = n_items & (a.acc_sets - 1);
        const uint32_t use = (uint32_t)(n_items >> (a.acc_sets - 1));
        if (!mbar_wait(smem_u32(&ctl->acc_empty[set]), (use & 1u) ^ 1u, abort_flag, a.err, kWaitLimitCycles)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tacc = tmem + (uint32_t)set * a.set_stride;
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
          const uint64_t b0 = smem_desc_sw128(st + (uint32_t)a.a_bytes);
#pragma unroll
          for (int k = 0; k < kBK / kUmmaK; ++k) {
            const uint64_t bdesc = b0 + (uint64_t)(2 * k);
            if (a.nsplit == 2) {
              // two chains: the two column halves (the second half's rows start BN/2 rows on)
              const uint32_t acc = (kb > item.k0 || k > 0) ? 1u : 0u;
              tc_mma(tacc, a0 + (uint64_t)(2 * k), bdesc, a.idesc, acc);
              tc_mma(tacc + a.acc_stride, a0 + (uint64_t)(2 * k), bdesc + (uint64_t)(((a.BN >> 1) * kBK * 2) >> 4),
                     a.idesc, acc);
            } else if (a.msub == 2) {
              // two chains: the two 128-row halves
              const uint32_t acc = (kb > item.k0 || k > 0) ? 1u : 0u;
              tc_mma(tacc, a0 + (uint64_t)(2 * k), bdesc, a.idesc, acc);
              tc_mma(tacc + a.acc_stride, a0 + (uint64_t)(2 * k + (kATileBytes >> 4)), bdesc, a.idesc, acc);
            } else {
              // two chains: even and odd k steps of the same tile
              tc_mma(tacc + (k & 1) * a.acc_stride, a0 + (uint64_t)(2 * k), bdesc, a.idesc,
                     (kb > item.k0 || k > 1) ? 1u : 0u);
            }
          }
          tc_commit(smem_u32(&ctl->empty[slot]));   // stage free once these MMAs have read it
          if (++slot == a.stages) {
            slot = 0;
            round ^= 1u;
          }
        }
        tc_commit(smem_u32(&ctl->acc_full[set]));   // this item's accumulators final (or drained)
        ++n_items;
      }
      if (!ok) tc_commit(smem_u32(&ctl->acc_full[set]));
    }
  } else if (warp >= 6) {
    // ---------------- the overlapped gate (kOverlap) ----------------
    if constexpr (kOverlap) {
      pdl_wait();                              // the streams may be written by an earlier kernel
      overlapped_gate(a, D, &ctl->gate, abort_flag);
    }
  } else {
    // ---------------- epilogue: TMEM -> registers -> shared tile -> fp32 kv --------------------
    const int q = warp & 3;                    // TMEM lane quarter this warp may access
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
    constexpr bool fused = kFused;
    if (fused) {                               // the first tile's stream rows, while the ring fills
      Schedule peek = sch;
      Item nx;
      if (peek.next(nx)) {
        int pm0, pn0;
        tile_origin(a, nx.tile, pm0, pn0);
        if (pn0 < a.gf.keys) gate_prefetch_rows(a.gf, a.M, a.msub, q, lane, pm0, pn0, a.BN);
      }
    }
    while (sch.next(item)) {
      const int set = n_items & (a.acc_sets - 1);
      const uint32_t use = (uint32_t)(n_items >> (a.acc_sets - 1));
      const bool ok = mbar_wait(smem_u32(&ctl->acc_full[set]), use & 1u, abort_flag, a.err, kWaitLimitCycles);
      tc_fence_after();
      if (!ok || *abort_flag) break;
      const uint32_t tacc = tmem + (uint32_t)set * a.set_stride;
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
      if (fused) {
        fused_gate_epilogue(a.gf, &tmD, D, a.M, a.N, tacc, q, lane, stg, a.msub, a.nsplit == 1 && a.msub == 1,
                            a.acc_stride, a.BN, a.nsplit, m0, n0);
      } else if (a.nsplit == 2) {
        const int hb = a.BN >> 1;
        store_accumulators(&tmD, D, a.M, a.N, tacc, q, lane, stg, 1, false, a.acc_stride, hb, m0, n0, false);
        store_accumulators(&tmD, D, a.M, a.N, tacc + a.acc_stride, q, lane, stg, 1, false, a.acc_stride, hb, m0,
                           n0 + hb, false);
      } else {
        store_accumulators(&tmD, D, a.M, a.N, tacc, q, lane, stg, a.msub, a.msub == 1, a.acc_stride, a.BN, m0, n0,
                           adder);
      }
      // The accumulators are read (every tcgen05.ld of the item has completed): the set may take
      // its next item now, while this item's stores are still in flight. (Waiting for the stores
      // first kept the tensor cores idle for the whole drain of the tile to HBM.)
      tc_fence_before();
      mbar_arrive(smem_u32(&ctl->acc_empty[set]));
      if (publish || kOverlap) {
        // the stores are complete (global writes done) before a flag or a count says so
        if (lane == 0) {
          asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
          asm volatile("fence.proxy.async.global;" ::: "memory");
        }
        __syncwarp();
      }
      if (publish) {
        // this segment is in kv once every epilogue warp's stores are complete: the last of the
        // four warps to get here lets the next segment's CTA add (a count, not a barrier, so an
        // abort that only some warps see cannot leave the others waiting)
        __threadfence();
        __syncwarp();
        if (lane == 0 && (atomicAdd(&ctl->published, 1u) & 3u) == 3u) {
          __threadfence();
          st_release(a.flags + blockIdx.x, want);
        }
      }
      if (kOverlap) {
        // this warp's quarter of the tile is in kv (its stores are complete): count it for the row
        // block, four counts a tile (no barrier across the epilogue warps, so an abort that only
        // some of them see cannot leave the others waiting)
        __threadfence();
        __syncwarp();
        if (lane == 0)
          asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(a.go.done + m0 / (128 * a.msub)) : "memory");
      }
      ++n_items;
      if (fused) {                             // the next tile's stream rows into L2 during its main loop
        Schedule peek = sch;
        Item nx;
        if (peek.next(nx)) {
          int pm0, pn0;
          tile_origin(a, nx.tile, pm0, pn0);
          if (pn0 < a.gf.keys) gate_prefetch_rows(a.gf, a.M, a.msub, q, lane, pm0, pn0, a.BN);
        }
      }
    }
    // the last stores have read their staging tiles (and are complete) before shared memory goes
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    if (*abort_flag) {
      // make sure no MMA is still writing the accumulators we are about to free
      volatile int32_t never = 0;
      for (int b = 0; b < a.acc_sets; ++b)
        for (int ph = 0; ph < 2; ++ph)
          mbar_wait(smem_u32(&ctl->acc_full[b]), (uint32_t)ph, &never, nullptr, kWaitLimitCycles / 8);
    }
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(a.tmem_cols)
                 : "memory");
  }
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

// Bytes from the ring's start to the end of the last stage's MMA reads: a full 128-row token tile
// per half (whatever was loaded), then the weight tile after the loaded token rows.
int mma_read_end(const GemmArgs& a) {
  const int a_read = a.msub * kATileBytes;
  return (a.stages - 1) * a.stage_bytes + (a_read > a.stage_bytes ? a_read : a.stage_bytes);
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
bool plan_gemm(int64_t M, int K, int N, int sms, size_t ws_bytes, Plan& P, bool allow_sk = true) {
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
  bool sk = allow_sk && g_sched_override == 2 && a.num_kb >= 2 && tiles_sk < 2 * (int64_t)sms;
  if (g_bn_override > 0 && g_bn_override != bn_sk) sk = false;
  if (sk && ws_bytes < sk_ws) sk = false;       // no room for the flags: data-parallel
  a.stream_k = sk ? 1 : 0;
  a.BN = sk ? bn_sk : (g_bn_override > 0 ? g_bn_override : pick_bn_dp(a.m_tiles, N, sms));
  a.nsplit = 1;
  if (!sk && g_bn_override == 0 && M > 128 && M <= 256) {
    // split tiles: the narrowest column half (a multiple of 16) that keeps both CTAs of every
    // column block in one wave; only for wide wkv, where the half is 128..208 columns (three or
    // more stages of 16 KB + 2 * half * 128 bytes still fit)
    int hb = 16;
    while (2 * (int64_t)((N + 2 * hb - 1) / (2 * hb)) > sms) hb += 16;
    if (hb >= 128 && hb <= 208) {
      a.nsplit = 2;
      a.msub = 1;
      a.m_tiles = (int32_t)((M + 127) / 128);
      a.BN = 2 * hb;
    }
  }
  a.n_tiles = (N + a.BN - 1) / a.BN;
  const int64_t n_tiles_total = (int64_t)a.m_tiles * a.n_tiles;
  if (n_tiles_total > 0x7fffffff) return false;
  a.total_units = n_tiles_total * a.num_kb;
  if (sk) {
    P.grid = a.total_units < sms ? (int)a.total_units : sms;
  } else {
    P.grid = n_tiles_total < sms ? (int)n_tiles_total : sms;
  }
  // token rows per half: all 128, or for a single short block only the rows that exist
  a.a_rows = (!sk && a.msub == 1 && a.m_tiles == 1 && M <= 112) ? (int32_t)((M + 15) / 16 * 16) : 128;
  a.a_bytes = a.msub * a.a_rows * kBK * 2;
  a.stage_bytes = a.a_bytes + a.BN * kBK * 2;   // split tiles: both halves
  a.stages = (kSmemBudget - 1024 - kEpiBytes - (int)sizeof(Ctl)) / a.stage_bytes;
  if (a.stages > kMaxStages) a.stages = kMaxStages;
  if (a.stages < 2) return false;
  a.acc_stride = pow2_at_least((uint32_t)(a.BN / a.nsplit));
  a.tmem_cols = a.acc_stride * 2;              // two accumulators (chains) per item
  if (a.tmem_cols > 512) return false;
  // Two accumulator sets when they fit (tiles of at most 128 columns): items alternate between
  // them, so the epilogue drains one while the tensor cores fill the other.
  a.acc_sets = 1;
  a.set_stride = 0;
  if (!sk && a.nsplit == 1 && 2 * a.tmem_cols <= 512) {
    a.acc_sets = 2;
    a.set_stride = a.tmem_cols;
    a.tmem_cols *= 2;
  }
  a.idesc = (1u << 4)                          // accumulate in f32
            | (1u << 7) | (1u << 10)           // A and B are bf16
            | ((uint32_t)((a.BN / a.nsplit) >> 3) << 17)    // N (of one MMA)
            | ((uint32_t)(128 >> 4) << 24);    // M = 128; A and B K-major (bits 15, 16 = 0)
  P.smem = 1024 + a.stages * a.stage_bytes + kEpiBytes + (int)sizeof(Ctl);
  P.ws_needed = sk ? sk_ws : 0;
  // The MMA reads 128 token rows per half from every stage, also from a short token tile (fewer
  // rows loaded): the last stage's reads must end inside the allocation (the epilogue's staging
  // tiles follow the ring). 1024 bytes are kept for aligning the ring.
  if (mma_read_end(a) > P.smem - 1024 || P.smem > kSmemBudget) return false;
  return true;
}

}  // namespace

// ---- tensor maps (shared with the MXFP8 projection) --------------------------------------------
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
bool make_map_bf16(CUtensorMap* m, const void* ptr, int64_t rows, int64_t K, uint32_t box_rows) {
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

// 2-D byte map over a row-major [rows, K] matrix of 8-bit codes; box = 128 k x box_rows rows, 128B
// swizzle (one 128-byte swizzle row per matrix row)
bool make_map_u8(CUtensorMap* m, const void* ptr, int64_t rows, int64_t K, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)K};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

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

bool gemm_plan_info(int64_t M, int K, int N, int sms, EngramProjectPlan* out) {
  Plan P;
  if (!plan_gemm(M, K, N, sms, (size_t)-1 / 2, P)) return false;
  const GemmArgs& a = P.a;
  *out = EngramProjectPlan{};
  out->grid = P.grid;
  out->threads = kThreads;
  out->smem_bytes = P.smem;
  out->tile_rows = 128 * a.msub;
  out->tile_cols = a.BN;
  out->split = a.nsplit;
  out->token_rows_loaded = a.a_rows;
  out->stages = a.stages;
  out->stage_bytes = a.stage_bytes;
  out->tmem_cols = (int32_t)a.tmem_cols;
  out->stream_k = a.stream_k;
  out->mma_read_end = mma_read_end(a);
  out->smem_avail = P.smem - 1024;
  return true;
}

int gemm_tile_cols(int64_t M, int K, int N, bool mx) {
  if (mx) {
    EngramProjectPlan info;
    return gemm_mx_plan_info(M, K, N, num_sms(), &info) ? info.tile_cols : 0;
  }
  Plan P;
  return plan_gemm(M, K, N, num_sms(), 0, P, false) ? P.a.BN : 0;
}

int launch_gemm(const GemmParams& p, cudaStream_t stream, bool pdl) {
  Plan P;
  const bool fused = p.gf.keys > 0;             // the gate's key sums need whole tiles: no stream-K
  const bool overlap = p.go.streams != nullptr;  // the gate waits for whole row blocks: no stream-K
  if (fused && overlap) {
    set_error("engram_project: the fused key sums and the overlapped gate exclude each other");
    return ENGRAM_EINVAL;
  }
  if (!plan_gemm(p.M, p.K, p.N, num_sms(), p.workspace != nullptr ? p.ws_bytes : 0, P, !fused && !overlap)) {
    set_error("engram_project: no tile plan fits (T %lld, K %d, N %d)", (long long)p.M, p.K, p.N);
    return ENGRAM_EINVAL;
  }
  GemmArgs a = P.a;
  a.err = p.err;
  a.gf = p.gf;
  a.go = p.go;
  if (overlap && (p.go.done == nullptr || p.go.H % 4 != 0 || p.go.H > 4 * kGateThreads * kGateVec)) {
    set_error("engram_project: overlapped gate needs its row-block counters and H <= %d", 4 * kGateThreads * kGateVec);
    return ENGRAM_EINVAL;
  }
  if (fused && a.gf.tile_cols != a.BN) {
    set_error("engram_project: fused gate planned for tiles of %d columns, the projection runs %d", a.gf.tile_cols,
              a.BN);
    return ENGRAM_EINVAL;
  }
  if (a.stream_k) {
    uint8_t* ws = static_cast<uint8_t*>(p.workspace);
    a.flags = reinterpret_cast<unsigned long long*>(ws);
    a.epoch = g_epoch.fetch_add(1) & 0xffffffffull;
  }
  static PerContextOnce attr;               // the attribute belongs to the context's module
  cudaError_t ae = attr.run([] {
    for (auto k : {wkv_gemm_kernel<false, false>, wkv_gemm_kernel<true, false>, wkv_gemm_kernel<false, true>}) {
      cudaError_t e1 = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBudget);
      if (e1 != cudaSuccess) return e1;
    }
    return cudaSuccess;
  });
  if (ae != cudaSuccess) return fail_cuda(ae, "engram_project: cudaFuncSetAttribute");
  CUtensorMap mA, mB, mD;
  if (!make_map_bf16(&mA, p.A, p.M, p.K, (uint32_t)a.a_rows) || !make_map_bf16(&mB, p.B, p.N, p.K, (uint32_t)(a.BN / a.nsplit)) ||
      !make_map_f32(&mD, p.D, p.M, p.N)) {
    set_error("engram_project: cuTensorMapEncodeTiled failed (driver entry point missing or bad layout)");
    return ENGRAM_ECUDA;
  }
  auto kernel = fused ? wkv_gemm_kernel<true, false> : overlap ? wkv_gemm_kernel<false, true> : wkv_gemm_kernel<false, false>;
  cudaError_t e = launch_k(kernel, dim3((unsigned)P.grid), dim3(overlap ? kThreadsOverlap : kThreads), (size_t)P.smem,
                           stream, pdl, mA, mB, mD, p.D, a);
  if (e != cudaSuccess) return fail_cuda(e, "engram_project: launch");
  return ENGRAM_OK;
}

}  // namespace engram
