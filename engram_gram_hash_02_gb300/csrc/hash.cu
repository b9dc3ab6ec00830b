// Stage 1: n-gram hash ids, one warp per token.
//
// Follows the n-gram hash of the NeMo "deepseek_v41.engram" page
// (DeepseekV41NgramHash.forward: no lookback across document, image or padding
// boundaries) and the vLLM "deepseek_v41.common.engram" page (NgramHashState.forward,
// EngramLayout, compute_hash_multipliers; lookback ids before each chunk).
//
// Lane k < max_ngram loads window slot k (issued speculatively, alongside the block's staging
// of cu_seqlens in shared memory), then decides whether the slot may be read (its position is
// alive and in t's document, or a live lookback entry); a ballot turns the
// per-slot verdicts into the walk back from t (slot k is open only if slots 0..k all are);
// shuffles hand every lane the window. Lanes then take the (layer, column) pairs: each mixes
// its n-gram's slots with XOR of id * multiplier and reduces modulo its head's prime.
#include "internal.cuh"

namespace engram {
namespace {

constexpr int kWarpsPerBlock = 8;
constexpr int kSmemCu = 2048;   // cu_seqlens entries staged in shared memory (else searched in global)

// largest s in [0, S) with cu[s] <= t (empty sequences before t are skipped)
template <typename Load>
__device__ __forceinline__ int32_t find_sequence(Load cu, int32_t S, int64_t t) {
  int32_t lo = 0, hi = S - 1;
  while (lo < hi) {
    const int32_t mid = (lo + hi + 1) >> 1;
    if ((int64_t)cu(mid) <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__global__ void __launch_bounds__(kWarpsPerBlock * 32)
hash_kernel(const HashParams p) {
  __shared__ int32_t s_cu[kSmemCu];
  pdl_wait();                                    // inputs may come from the preceding kernel
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t t = (int64_t)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  const bool live = t < p.T;
  const int O = p.max_ngram - 1;
  const bool cu_in_smem = p.cu_seqlens != nullptr && p.S + 1 <= kSmemCu;

  // ---- speculative loads of slot k = lane (issued before the sequence start is known) --------
  const int64_t pos = t - lane;
  const bool slot = live && lane < p.max_ngram && pos >= 0;
  int32_t raw = -1, sid = 1, sid_next = 1;
  bool alive = true;
  if (slot) {
    raw = __ldg(p.input_ids + pos);
    if (p.token_mask != nullptr) alive = __ldg(p.token_mask + pos) != 0;
    if (p.sequence_ids != nullptr) {
      sid = __ldg(p.sequence_ids + pos);
      sid_next = lane > 0 ? __ldg(p.sequence_ids + pos + 1) : sid;
    }
  }
  const bool raw_ok = raw >= 0 && raw < p.raw_vocab;
  const int32_t mapped = (slot && raw_ok) ? __ldg(p.token_map + raw) : p.pad_id;

  if (cu_in_smem) {
    for (int i = threadIdx.x; i <= p.S; i += blockDim.x) s_cu[i] = __ldg(p.cu_seqlens + i);
    __syncthreads();
  }
  if (!live) return;

  int32_t s = 0;
  int64_t start = 0;
  if (cu_in_smem) {
    s = find_sequence([&](int32_t i) { return s_cu[i]; }, p.S, t);
    start = s_cu[s];
  } else if (p.cu_seqlens != nullptr) {
    s = find_sequence([&](int32_t i) { return __ldg(p.cu_seqlens + i); }, p.S, t);
    start = __ldg(p.cu_seqlens + s);
  }

  // ---- slot k = lane: may it be read, and what does it hold --------------------------------
  bool ok = false;
  int64_t val = p.pad_id;
  if (lane < p.max_ngram) {
    if (pos >= start) {
      val = mapped;                                   // pad_id for a raw id outside the map
      if (lane == 0 && !raw_ok && p.err != nullptr) atomicOr(p.err, ENGRAM_ERR_RAW_ID);
      ok = alive && sid != 0 && (lane == 0 || sid == sid_next);
    } else if (p.lookback_ids != nullptr) {
      const int64_t i = pos - start + O;              // index into the sequence's lookback row
      if (i >= 0) {
        const int32_t id = __ldg(p.lookback_ids + (int64_t)s * O + i);
        ok = id >= 0;
        val = id;
      }
    }
  }
  const uint32_t okbits = __ballot_sync(0xffffffffu, ok);

  // window slot k is open iff slots 0..k are all readable
  uint64_t w[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int64_t v = __shfl_sync(0xffffffffu, val, k);
    const uint32_t need = (2u << k) - 1u;
    w[k] = (k < p.max_ngram && (okbits & need) == need) ? (uint64_t)v : (uint64_t)p.pad_id;
  }

  // ---- lanes over (layer, column) ------------------------------------------------------
  const int LC = p.layers * p.cols;
  int32_t* out = p.out + t * LC;
  for (int idx = lane; idx < LC; idx += 32) {
    const int layer = idx / p.cols;
    const int col = idx - layer * p.cols;
    const int n = col / p.n_heads + 2;                   // n-gram size of this column
    const int64_t* m = p.multipliers + (int64_t)layer * p.max_ngram;
    uint64_t mix = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k)
      if (k < n) mix ^= w[k] * (uint64_t)__ldg(m + k);  // each product < 2^63 (bounded multipliers)
    const uint64_t prime = (uint64_t)__ldg(p.primes + idx);
    const int64_t id = __ldg(p.offsets + idx) + (int64_t)(mix % prime);
    out[idx] = (int32_t)id;
  }
}

}  // namespace

cudaError_t launch_hash(const HashParams& p, cudaStream_t stream, bool pdl) {
  const int64_t blocks = (p.T + kWarpsPerBlock - 1) / kWarpsPerBlock;
  return launch_k(hash_kernel, dim3((unsigned)blocks), dim3(kWarpsPerBlock * 32), 0, stream, pdl, p);
}

}  // namespace engram
