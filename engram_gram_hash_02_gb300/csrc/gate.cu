// Stage 4: the Engram gate, in place on the fp32 hyper-connection highway.
//
// Follows the NeMo "deepseek_v41.engram" page (_engram_gate_core: normalised,
// signed-square-root-gated value added to every fp32 stream; masked tokens keep their
// streams), the vLLM "deepseek_v41.common.engram" page (Engram: keys first, value last in
// the wkv output, clamp 1e-6) and the Atlas "engram_v41" page (stage 4: in place on the
// fp32 highway [T, hc, H]).
//
// A persistent kernel: a few CTAs per SM, each walking a fixed share of the (token, stream)
// items (item i = t * hc + j; CTA b takes b, b + grid, ...; masked tokens are skipped before
// anything is loaded). Per item, one thread issues three 1-D bulk copies (cp.async.bulk) of
// the stream row h_j, the key_j and the shared value (4H bytes each, contiguous) into one of
// two shared-memory buffers, completing on that buffer's mbarrier; the copies of the next item
// are in flight while the CTA works on the current one. The CTA reads h and the key from shared
// memory to form sum h^2, sum key^2 and
// sum h*q*key*k, reduces them with warp shuffles, computes the gate, and writes h + g * value
// back with coalesced 16-byte stores. HBM traffic is the minimum: h read and written once, key
// read once, the value once per stream (hc - 1 of those from L2). The grid is a multiple of hc,
// so a CTA only ever sees one stream j: each thread loads its slice of q_weight[j] and
// k_weight[j] into registers once, keeping that latency off the per-item path.
//
// Under programmatic dependent launch the first items' stream rows are requested before
// waiting for the projection; every CTA waits once (not once per item). Waits on the buffers
// are bounded (~2 s of SM clock cycles); on expiry the CTA reports ENGRAM_ERR_PIPE_TIMEOUT,
// waits (bounded) for its copies in flight and exits.
#include "internal.cuh"

namespace engram {
namespace {

constexpr int kBufs = 2;
constexpr int kChunks = 4;                             // float4 chunks of a row per thread (H <= 16 * threads)
constexpr int kMaxThreads = 512;
constexpr int kMaxCtasPerSm = 8;
constexpr int kSmemBudget = 232448;                    // opt-in maximum per CTA
constexpr uint64_t kWaitLimitCycles = 4000000000ull;   // ~2 s at 2 GHz

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
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
// bounded wait on a buffer's mbarrier; false on expiry (or when another thread gave up)
__device__ __noinline__ bool wait_buffer(uint32_t bar, uint32_t parity, volatile int* abort_flag, uint64_t limit) {
  const uint64_t t0 = clock64();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 15u) == 15u && (*abort_flag || (uint64_t)clock64() - t0 > limit)) return false;
  }
}
__device__ __forceinline__ void bulk_copy(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// The CTA's items in order, masked tokens skipped: every thread walks the same sequence.
struct Items {
  const GateParams& p;
  int64_t total, stride;
  __device__ Items(const GateParams& params, int64_t s) : p(params), total(params.T * params.hc), stride(s) {}
  __device__ int64_t next(int64_t i) const {   // first unmasked item >= i on this CTA's stride
    for (; i < total; i += stride) {
      if (p.token_mask == nullptr || __ldg(p.token_mask + i / p.hc) != 0) return i;
    }
    return -1;
  }
};

// The partial sums the fused projection left for item (t, j): one 16-byte slot (ssk, dot of the
// tile's first stream, ssk, dot of its second) per tile covering stream j, tiles first .. last.
struct PartRange {
  int first, count;
};
__device__ __forceinline__ PartRange part_range(const GateParams& p, int j) {
  const int first = (j * p.H) / p.part_cols;
  const int last = ((j + 1) * p.H - 1) / p.part_cols;
  return {first, last - first + 1};
}
// Sum over the partial slots of one item, in tile order (lane i takes tiles i, i + 32, ...; then a
// fixed shuffle tree): the same order for every call. Warp-collective.
__device__ __forceinline__ void sum_partials(const GateParams& p, const float* slots, PartRange pr, int j, int lane,
                                             float& ssk, float& dot) {
  ssk = 0.f;
  dot = 0.f;
  for (int i = lane; i < pr.count; i += 32) {
    const int tt = pr.first + i;
    const int o = (((tt * p.part_cols) / p.H) == j) ? 0 : 2;   // j is the tile's first or second stream
    ssk += slots[4 * i + o];
    dot += slots[4 * i + o + 1];
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    ssk += __shfl_xor_sync(0xffffffffu, ssk, off);
    dot += __shfl_xor_sync(0xffffffffu, dot, off);
  }
}

// kFused: the projection fused the key sums (GateParams::part_cols > 0): the key slot of a buffer
// receives the item's partial slots instead of the key row.
template <bool kFused>
__global__ void __launch_bounds__(kMaxThreads, 1)
gate_kernel(const GateParams p) {
  extern __shared__ __align__(128) float buf[];          // kBufs x [h | key (or partials) | value], H floats each
  __shared__ __align__(8) uint64_t full[kBufs];
  __shared__ float red[kMaxThreads / 32][3];
  __shared__ float fused_sums[2];
  __shared__ float gate_s;
  __shared__ int abort_s;

  const int H = p.H;
  const int tid = threadIdx.x;
  const uint32_t row_bytes = 4u * (uint32_t)H;
  const int64_t N = (int64_t)(p.hc + 1) * H;
  const Items items(p, gridDim.x);

  if (tid == 0) {
    for (int b = 0; b < kBufs; ++b)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&full[b])) : "memory");
    abort_s = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  // ---- producer state (thread 0): items issued so far -------------------------------------
  int64_t ahead = items.next(blockIdx.x);                // next item to issue
  int issued = 0;
  auto buffer = [&](int n) { return smem_u32(buf) + (uint32_t)((n % kBufs) * 3) * row_bytes; };
  auto issue_h = [&](int64_t i, int n) {                 // stream row: not written by the projection
    const uint32_t bar = smem_u32(&full[n % kBufs]);
    uint32_t bytes = 3u * row_bytes;
    if (kFused) bytes = 2u * row_bytes + 16u * (uint32_t)part_range(p, (int)(i % p.hc)).count;
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
    bulk_copy(buffer(n), p.streams + i * (int64_t)H, row_bytes, bar);
  };
  auto issue_kv = [&](int64_t i, int n) {                // key (or partials) and value: the projection's output
    const uint32_t bar = smem_u32(&full[n % kBufs]);
    const int64_t t = i / p.hc;
    const int j = (int)(i - t * p.hc);
    if (kFused) {
      const PartRange pr = part_range(p, j);
      bulk_copy(buffer(n) + row_bytes, p.kv + t * N + 4 * pr.first, 16u * (uint32_t)pr.count, bar);
    } else {
      bulk_copy(buffer(n) + row_bytes, p.kv + t * N + (int64_t)j * H, row_bytes, bar);
    }
    bulk_copy(buffer(n) + 2u * row_bytes, p.kv + t * N + (int64_t)p.hc * H, row_bytes, bar);
  };
  int64_t first_items[kBufs];
  if (tid == 0) {
    for (int n = 0; n < kBufs && ahead >= 0; ++n) {
      first_items[n] = ahead;
      issue_h(ahead, n);
      ahead = items.next(ahead + gridDim.x);
      ++issued;
    }
  }
  pdl_wait();                                            // kv comes from the projection
  if (tid == 0) {
    for (int n = 0; n < issued; ++n) issue_kv(first_items[n], n);
  }

  const int lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  const int H4 = H >> 2;
  // this CTA's stream and its norm weights (grid % hc == 0: every item of the CTA has j = b % hc)
  const int jc = (int)(blockIdx.x % (unsigned)p.hc);
  uint2 qreg[kChunks], kreg[kChunks];
#pragma unroll
  for (int m = 0; m < kChunks; ++m) {
    const int c = tid + m * (int)blockDim.x;
    if (c < H4) {
      qreg[m] = __ldg(reinterpret_cast<const uint2*>(p.q_weight + (int64_t)jc * H) + c);
      kreg[m] = __ldg(reinterpret_cast<const uint2*>(p.k_weight + (int64_t)jc * H) + c);
    } else {
      qreg[m] = kreg[m] = make_uint2(0, 0);
    }
  }
  int64_t cur = items.next(blockIdx.x);
  for (int n = 0; cur >= 0; ++n) {
    const int64_t nxt = items.next(cur + gridDim.x);
    if (nxt < 0 && tid == 0) pdl_trigger();              // last item: the next kernel may launch
    const bool ok = wait_buffer(smem_u32(&full[n % kBufs]), (uint32_t)(n / kBufs) & 1u, &abort_s, kWaitLimitCycles);
    if (!ok) abort_s = 1;
    const float4* hs = reinterpret_cast<const float4*>(buf + (size_t)(n % kBufs) * 3 * H);
    const float4* ks = hs + H4;
    const float4* vs = ks + H4;
    float ssh = 0.f, ssk = 0.f, dot = 0.f;
#pragma unroll
    for (int m = 0; m < kChunks; ++m) {
      const int c = tid + m * (int)blockDim.x;
      if (c >= H4) break;
      const float4 x = hs[c];
      ssh = fmaf(x.x, x.x, ssh); ssh = fmaf(x.y, x.y, ssh); ssh = fmaf(x.z, x.z, ssh); ssh = fmaf(x.w, x.w, ssh);
      if (!kFused) {
        const float4 y = ks[c];
        const uint2 qr = qreg[m], kr = kreg[m];
        ssk = fmaf(y.x, y.x, ssk); ssk = fmaf(y.y, y.y, ssk); ssk = fmaf(y.z, y.z, ssk); ssk = fmaf(y.w, y.w, ssk);
        dot = fmaf(x.x * bf16lo(qr.x), y.x * bf16lo(kr.x), dot);
        dot = fmaf(x.y * bf16hi(qr.x), y.y * bf16hi(kr.x), dot);
        dot = fmaf(x.z * bf16lo(qr.y), y.z * bf16lo(kr.y), dot);
        dot = fmaf(x.w * bf16hi(qr.y), y.w * bf16hi(kr.y), dot);
      }
    }
    if (kFused && warp == 0) {                           // the key sums: the item's partial slots
      float fs, fd;
      sum_partials(p, reinterpret_cast<const float*>(ks), part_range(p, jc), jc, lane, fs, fd);
      if (lane == 0) {
        fused_sums[0] = fs;
        fused_sums[1] = fd;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      ssh += __shfl_xor_sync(0xffffffffu, ssh, off);
      ssk += __shfl_xor_sync(0xffffffffu, ssk, off);
      dot += __shfl_xor_sync(0xffffffffu, dot, off);
    }
    if (lane == 0) {
      red[warp][0] = ssh;
      red[warp][1] = ssk;
      red[warp][2] = dot;
    }
    __syncthreads();                                     // (1) partial sums and abort_s visible
    if (abort_s) break;
    if (tid == 0) {
      float a = 0.f, b = 0.f, c = 0.f;
      for (int w = 0; w < nwarps; ++w) {
        a += red[w][0];
        b += red[w][1];
        c += red[w][2];
      }
      if (kFused) {
        b = fused_sums[0];
        c = fused_sums[1];
      }
      const float invH = 1.0f / (float)H;
      const float rh = rsqrtf(a * invH + p.eps);
      const float rk = rsqrtf(b * invH + p.eps);
      const float s = c * rh * rk / sqrtf((float)H);
      float ss = 0.f;                                    // sign(0) = 0
      if (s > 0.f) ss = sqrtf(fmaxf(s, p.clamp));
      else if (s < 0.f) ss = -sqrtf(fmaxf(-s, p.clamp));
      gate_s = 1.0f / (1.0f + expf(-ss));
    }
    __syncthreads();                                     // (2) gate visible
    const float g = gate_s;
    float4* out = reinterpret_cast<float4*>(p.streams + cur * (int64_t)H);
    for (int c = tid; c < H4; c += blockDim.x) {
      const float4 x = hs[c], v = vs[c];
      out[c] = make_float4(fmaf(g, v.x, x.x), fmaf(g, v.y, x.y), fmaf(g, v.z, x.z), fmaf(g, v.w, x.w));
    }
    __syncthreads();                                     // (3) buffer n % kBufs read by all
    if (tid == 0 && ahead >= 0) {
      // refill this buffer with the item kBufs places ahead (issued == n + kBufs here)
      issue_h(ahead, issued);
      issue_kv(ahead, issued);
      ahead = items.next(ahead + gridDim.x);
      ++issued;
    }
    cur = nxt;
  }

  if (abort_s) {
    if (p.err != nullptr && tid == 0) atomicOr(p.err, ENGRAM_ERR_PIPE_TIMEOUT);
    // copies still in flight must land before shared memory goes away: wait (bounded) on every
    // buffer use issued but not consumed
    if (tid == 0) {
      volatile int never = 0;
      for (int n = issued > kBufs ? issued - kBufs : 0; n < issued; ++n)
        wait_buffer(smem_u32(&full[n % kBufs]), (uint32_t)(n / kBufs) & 1u, &never, kWaitLimitCycles / 4);
    }
    __syncthreads();
  }
}

// ---- small-T form: one CTA per (token, stream) item --------------------------------------------
// When there are too few items to keep a persistent grid busy (the decode step: 256 tokens x 4
// streams over 148 SMs), each item gets a CTA of its own. Each thread owns kVec float4 chunks of the
// row (chunk c = tid + m * threads): its chunks of h_j are copied into shared memory with cp.async
// before waiting for the projection (no registers held), its chunks of key_j and the value go to
// registers, all requested before any is used. A thread reads back only the chunks it copied
// itself, so the copies need no block barrier. One block barrier: the warps' partial sums meet in
// shared memory and every thread forms the gate from them (the same arithmetic in every thread),
// then writes its chunks of h + g * v. No waits on other threads' progress, so no time limit is
// needed. Registers stay within four CTAs per SM up to 4 chunks a thread (H <= 4096).
constexpr int kItemThreads = 256;

template <int kVec, bool kFused>
__global__ void __launch_bounds__(kItemThreads, kVec <= 4 ? 4 : 1)
gate_item_kernel(const GateParams p) {
  __shared__ float red[kItemThreads / 32][3];
  __shared__ float fused_sums[2];
  __shared__ __align__(16) float4 xs[kVec * kItemThreads];   // this CTA's stream row h_j
  const int H = p.H, H4 = H >> 2;
  const int tid = threadIdx.x;
  const int64_t item = blockIdx.x;
  const int64_t t = item / p.hc;
  const int j = (int)(item - t * p.hc);
  if (p.token_mask != nullptr && __ldg(p.token_mask + t) == 0) {   // masked: not read or written
    pdl_wait();
    return;
  }
  const int64_t N = (int64_t)(p.hc + 1) * H;
  float4* hrow = reinterpret_cast<float4*>(p.streams + item * (int64_t)H);
  const float4* krow = reinterpret_cast<const float4*>(p.kv + t * N + (int64_t)j * H);
  const float4* vrow = reinterpret_cast<const float4*>(p.kv + t * N + (int64_t)p.hc * H);
  const uint2* qrow = reinterpret_cast<const uint2*>(p.q_weight + (int64_t)j * H);
  const uint2* kwrow = reinterpret_cast<const uint2*>(p.k_weight + (int64_t)j * H);
  float4 y[kVec], v[kVec];
  uint2 qr[kVec], kr[kVec];
#pragma unroll
  for (int m = 0; m < kVec; ++m) {                 // not written by the projection: before the wait
    const int c = tid + m * kItemThreads;
    if (c < H4) {
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(&xs[c])), "l"(hrow + c) : "memory");
      qr[m] = __ldg(qrow + c);
      kr[m] = __ldg(kwrow + c);
    }
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
  pdl_wait();                                      // kv comes from the projection
  pdl_trigger();
#pragma unroll
  for (int m = 0; m < kVec; ++m) {
    const int c = tid + m * kItemThreads;
    if (c < H4) {
      if (!kFused) y[m] = krow[c];
      v[m] = vrow[c];
    }
  }
  const int lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  if (kFused && warp == 0) {                       // the key sums: the item's partial slots
    const PartRange pr = part_range(p, j);
    float fs, fd;
    sum_partials(p, p.kv + t * N + 4 * pr.first, pr, j, lane, fs, fd);
    if (lane == 0) {
      fused_sums[0] = fs;
      fused_sums[1] = fd;
    }
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");   // this thread's chunks of h_j have landed
  float ssh = 0.f, ssk = 0.f, dot = 0.f;
#pragma unroll
  for (int m = 0; m < kVec; ++m) {
    const int c = tid + m * kItemThreads;
    if (c < H4) {
      const float4 x = xs[c];
      ssh = fmaf(x.x, x.x, ssh); ssh = fmaf(x.y, x.y, ssh);
      ssh = fmaf(x.z, x.z, ssh); ssh = fmaf(x.w, x.w, ssh);
      if (!kFused) {
        ssk = fmaf(y[m].x, y[m].x, ssk); ssk = fmaf(y[m].y, y[m].y, ssk);
        ssk = fmaf(y[m].z, y[m].z, ssk); ssk = fmaf(y[m].w, y[m].w, ssk);
        dot = fmaf(x.x * bf16lo(qr[m].x), y[m].x * bf16lo(kr[m].x), dot);
        dot = fmaf(x.y * bf16hi(qr[m].x), y[m].y * bf16hi(kr[m].x), dot);
        dot = fmaf(x.z * bf16lo(qr[m].y), y[m].z * bf16lo(kr[m].y), dot);
        dot = fmaf(x.w * bf16hi(qr[m].y), y[m].w * bf16hi(kr[m].y), dot);
      }
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    ssh += __shfl_xor_sync(0xffffffffu, ssh, off);
    ssk += __shfl_xor_sync(0xffffffffu, ssk, off);
    dot += __shfl_xor_sync(0xffffffffu, dot, off);
  }
  if (lane == 0) {
    red[warp][0] = ssh;
    red[warp][1] = ssk;
    red[warp][2] = dot;
  }
  __syncthreads();
  float a = 0.f, b = 0.f, cdot = 0.f;
  for (int w = 0; w < nwarps; ++w) {               // the same order in every thread
    a += red[w][0];
    b += red[w][1];
    cdot += red[w][2];
  }
  if (kFused) {
    b = fused_sums[0];
    cdot = fused_sums[1];
  }
  const float invH = 1.0f / (float)H;
  const float s = cdot * rsqrtf(a * invH + p.eps) * rsqrtf(b * invH + p.eps) / sqrtf((float)H);
  float ss = 0.f;                                  // sign(0) = 0
  if (s > 0.f) ss = sqrtf(fmaxf(s, p.clamp));
  else if (s < 0.f) ss = -sqrtf(fmaxf(-s, p.clamp));
  const float g = 1.0f / (1.0f + expf(-ss));
#pragma unroll
  for (int m = 0; m < kVec; ++m) {
    const int c = tid + m * kItemThreads;
    if (c < H4) {
      const float4 x = xs[c];
      hrow[c] = make_float4(fmaf(g, v[m].x, x.x), fmaf(g, v[m].y, x.y), fmaf(g, v[m].z, x.z), fmaf(g, v[m].w, x.w));
    }
  }
}

template <int kVec>
cudaError_t launch_gate_items(const GateParams& p, cudaStream_t stream, bool pdl) {
  const int H4 = p.H / 4;
  const int threads = H4 >= kItemThreads ? kItemThreads : ((H4 + 31) / 32) * 32;
  if (p.part_cols > 0)
    return launch_k(gate_item_kernel<kVec, true>, dim3((unsigned)(p.T * p.hc)), dim3(threads), 0, stream, pdl, p);
  return launch_k(gate_item_kernel<kVec, false>, dim3((unsigned)(p.T * p.hc)), dim3(threads), 0, stream, pdl, p);
}

int g_gate_form = 0;   // engram_set_gate_form: 0 automatic, 1 persistent, 2 one CTA per item

}  // namespace

void set_gate_form_override(int f) { g_gate_form = f; }

// Items (token x stream) up to which the one-CTA-per-item form is used: about a wave and a half of
// small CTAs (below that a persistent grid leaves most of its CTAs with one or two serial items).
int64_t gate_item_threshold() { return (int64_t)num_sms() * 8; }

cudaError_t launch_gate(const GateParams& p, cudaStream_t stream, bool pdl) {
  const int64_t items = p.T * p.hc;
  const bool item_form = g_gate_form == 2 || (g_gate_form == 0 && items <= gate_item_threshold());
  if (item_form && items <= 0x7fffffff) {
    switch ((p.H / 4 + kItemThreads - 1) / kItemThreads) {     // float4 chunks per thread and row
      case 0:
      case 1: return launch_gate_items<1>(p, stream, pdl);
      case 2: return launch_gate_items<2>(p, stream, pdl);
      case 3: return launch_gate_items<3>(p, stream, pdl);
      case 4: return launch_gate_items<4>(p, stream, pdl);
      case 5: return launch_gate_items<5>(p, stream, pdl);
      case 6: return launch_gate_items<6>(p, stream, pdl);
      case 7: return launch_gate_items<7>(p, stream, pdl);
      case 8: return launch_gate_items<8>(p, stream, pdl);
      default: break;                                          // H > 8192: not reached (checked)
    }
  }
  return launch_gate_persistent(p, stream, pdl);
}

cudaError_t launch_gate_persistent(const GateParams& p, cudaStream_t stream, bool pdl) {
  const int H = p.H;
  int threads = ((H / (4 * kChunks) + 31) / 32) * 32;   // every thread covers at most kChunks chunks
  if (threads < 64) threads = 64;
  if (threads > kMaxThreads) threads = kMaxThreads;
  const size_t smem = (size_t)kBufs * 3 * 4 * (size_t)H;
  if (smem > (size_t)kSmemBudget - 2048) return cudaErrorInvalidValue;
  const bool fused = p.part_cols > 0;
  void (*kernel)(const GateParams) = fused ? gate_kernel<true> : gate_kernel<false>;
  static PerContextOnce attr;               // the attribute belongs to the context's module
  cudaError_t ae = attr.run([] {
    cudaError_t e1 = cudaFuncSetAttribute(gate_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          kSmemBudget - 2048);
    if (e1 != cudaSuccess) return e1;
    return cudaFuncSetAttribute(gate_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBudget - 2048);
  });
  if (ae != cudaSuccess) return ae;
  int per_sm = 0;                           // resident CTAs per SM (registers, shared memory)
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm > kMaxCtasPerSm) per_sm = kMaxCtasPerSm;
  if (per_sm < 1) per_sm = 1;
  const int64_t items = p.T * p.hc;
  // a multiple of hc (each CTA keeps one stream's norm weights), at most one CTA per item
  int64_t grid = ((int64_t)num_sms() * per_sm / p.hc) * p.hc;
  if (grid < p.hc) grid = p.hc;
  if (grid > items) grid = items;                       // items = T * hc: still a multiple of hc
  return launch_k(kernel, dim3((unsigned)grid), dim3(threads), smem, stream, pdl, p);
}

}  // namespace engram
