// Stage 1: n-gram hash ids, one warp per token.
//
// Follows the n-gram hash of the NeMo "deepseek_v41.engram" page
// (DeepseekV41NgramHash.forward: no lookback across document, image or padding
// boundaries) and the vLLM "deepseek_v41.common.engram" page (NgramHashState.forward,
// EngramLayout, compute_hash_multipliers; lookback ids before each chunk).
//
// Lane k < max_ngram decides whether window slot k may be read (its position is alive and
// in t's document, or a live lookback entry) and loads its compressed id; a ballot turns the
// per-slot verdicts into the walk back from t (slot k is open only if slots 0..k all are);
// shuffles hand every lane the window. Lanes then take the (layer, column) pairs: each mixes
// its n-gram's slots with XOR of id * multiplier and reduces modulo its head's prime.
#include "internal.cuh"

namespace engram {
namespace {

constexpr int kWarpsPerBlock = 8;

__device__ __forceinline__ int32_t find_sequence(const int32_t* __restrict__ cu, int32_t S, int64_t t) {
  // largest s in [0, S) with cu[s] <= t (empty sequences before t are skipped)
  int32_t lo = 0, hi = S - 1;
  while (lo < hi) {
    int32_t mid = (lo + hi + 1) >> 1;
    if ((int64_t)__ldg(cu + mid) <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__global__ void __launch_bounds__(kWarpsPerBlock * 32)
hash_kernel(const HashParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t t = (int64_t)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  if (t >= p.T) return;
  const int O = p.max_ngram - 1;

  int32_t s = 0;
  int64_t start = 0;
  if (p.cu_seqlens != nullptr) {
    s = find_sequence(p.cu_seqlens, p.S, t);
    start = __ldg(p.cu_seqlens + s);
  }

  // ---- slot k = lane: may it be read, and what does it hold -------------------------
  bool ok = false;
  int64_t val = p.pad_id;
  if (lane < p.max_ngram) {
    const int64_t pos = t - lane;
    if (pos >= start) {
      const int32_t raw = __ldg(p.input_ids + pos);
      if (raw >= 0 && raw < p.raw_vocab) {
        val = __ldg(p.token_map + raw);
      } else if (lane == 0 && p.err != nullptr) {
        atomicOr(p.err, ENGRAM_ERR_RAW_ID);   // hashes as pad_id
      }
      ok = (p.token_mask == nullptr || __ldg(p.token_mask + pos) != 0);
      if (p.sequence_ids != nullptr) {
        const int32_t sid = __ldg(p.sequence_ids + pos);
        ok = ok && sid != 0;
        if (lane > 0) ok = ok && sid == __ldg(p.sequence_ids + pos + 1);
      }
    } else if (p.lookback_ids != nullptr) {
      const int64_t i = pos - start + O;       // index into the sequence's lookback row
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

cudaError_t launch_hash(const HashParams& p, cudaStream_t stream) {
  const int64_t blocks = (p.T + kWarpsPerBlock - 1) / kWarpsPerBlock;
  hash_kernel<<<(unsigned)blocks, kWarpsPerBlock * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace engram
