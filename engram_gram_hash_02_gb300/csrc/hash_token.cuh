// The n-gram hash of one token, shared by the hash kernel and the fused hash + gather kernel.
//
// Follows the n-gram hash of the NeMo "deepseek_v41.engram" page
// (DeepseekV41NgramHash.forward: no lookback across document, image or padding
// boundaries) and the vLLM "deepseek_v41.common.engram" page (NgramHashState.forward,
// EngramLayout, compute_hash_multipliers; lookback ids before each chunk).
//
// One warp per token. Lane k < max_ngram loads window slot k (issued speculatively, before the
// token's sequence start is known), then decides whether the slot may be read (its position is
// alive and in t's document, or a live lookback entry); a ballot turns the per-slot answers into
// the walk back from t (slot k is open only if slots 0..k all are); shuffles hand every lane the
// window. Lanes then take the (layer, column) pairs: each mixes its n-gram's slots with XOR of
// id * multiplier and reduces modulo its head's prime.
#pragma once

#include "internal.cuh"

namespace engram {
namespace {

constexpr int kSmemCu = 2048;   // cu_seqlens entries staged in shared memory (else searched in global)

// The words engram_forward asks the hash launch to clear (block 0, after the dependency wait).
__device__ __forceinline__ void clear_words(const HashParams& p) {
  if (blockIdx.x == 0 && p.zero != nullptr)
    for (int i = threadIdx.x; i < p.zero_n; i += blockDim.x) p.zero[i] = 0u;
}

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

// Stages cu_seqlens in shared memory when it fits (all threads of the block take part; ends with a
// block barrier). Returns whether it did.
__device__ __forceinline__ bool stage_cu(const HashParams& p, int32_t* s_cu) {
  const bool in_smem = p.cu_seqlens != nullptr && p.S + 1 <= kSmemCu;
  if (in_smem) {
    for (int i = threadIdx.x; i <= p.S; i += blockDim.x) s_cu[i] = __ldg(p.cu_seqlens + i);
  }
  __syncthreads();
  return in_smem;
}

// What one lane of a token's warp loads before the token's sequence is known (issued early so it
// overlaps the block's staging of cu_seqlens).
struct TokenLoads {
  uint64_t prime[8], off[8];                 // per (layer, column) idx = lane + 32u
  int64_t pos;                               // t - lane: this lane's window slot
  int32_t raw, sid, sid_next, mapped;
  bool slot, alive, raw_ok;
};

__device__ __forceinline__ TokenLoads hash_token_loads(const HashParams& p, int64_t t, int lane) {
  TokenLoads L;
  const int LC = p.layers * p.cols;
#pragma unroll
  for (int u = 0; u < 8; ++u) {              // window-independent constants first
    const int idx = lane + 32 * u;
    L.prime[u] = idx < LC ? (uint64_t)__ldg(p.primes + idx) : 1ull;
    L.off[u] = idx < LC ? (uint64_t)__ldg(p.offsets + idx) : 0ull;
  }
  L.pos = t - lane;
  L.slot = lane < p.max_ngram && L.pos >= 0;
  L.raw = -1;
  L.sid = L.sid_next = 1;
  L.alive = true;
  if (L.slot) {
    L.raw = __ldg(p.input_ids + L.pos);
    if (p.token_mask != nullptr) L.alive = __ldg(p.token_mask + L.pos) != 0;
    if (p.sequence_ids != nullptr) {
      L.sid = __ldg(p.sequence_ids + L.pos);
      L.sid_next = lane > 0 ? __ldg(p.sequence_ids + L.pos + 1) : L.sid;
    }
  }
  L.raw_ok = L.raw >= 0 && L.raw < p.raw_vocab;
  L.mapped = (L.slot && L.raw_ok) ? __ldg(p.token_map + L.raw) : p.pad_id;
  return L;
}

// Ids of token t for every (layer, column) from the lane's early loads: written to the global
// output, and to smem_out when given. Called by all 32 lanes of one warp, after cu_seqlens was
// staged (cu_in_smem) or not.
__device__ __forceinline__ void hash_token_finish(const HashParams& p, int64_t t, int lane, const TokenLoads& L,
                                                  bool cu_in_smem, const int32_t* s_cu, int32_t* smem_out) {
  const int O = p.max_ngram - 1;
  const int LC = p.layers * p.cols;
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
    if (L.pos >= start) {
      val = L.mapped;                                 // pad_id for a raw id outside the map
      if (lane == 0 && !L.raw_ok && p.err != nullptr) atomicOr(p.err, ENGRAM_ERR_RAW_ID);
      ok = L.alive && L.sid != 0 && (lane == 0 || L.sid == L.sid_next);
    } else if (p.lookback_ids != nullptr) {
      const int64_t i = L.pos - start + O;            // index into the sequence's lookback row
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
  int32_t* out = p.out + t * LC;
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int idx = lane + 32 * u;
    if (idx >= LC) break;
    const int layer = idx / p.cols;
    const int col = idx - layer * p.cols;
    const int n = col / p.n_heads + 2;                   // n-gram size of this column
    const int64_t* m = p.multipliers + (int64_t)layer * p.max_ngram;
    uint64_t mix = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k)
      if (k < n) mix ^= w[k] * (uint64_t)__ldg(m + k);  // each product < 2^63 (bounded multipliers)
    const int32_t id = (int32_t)((int64_t)L.off[u] + (int64_t)(mix % L.prime[u]));
    out[idx] = id;
    if (smem_out != nullptr) smem_out[idx] = id;
  }
}

}  // namespace
}  // namespace engram
