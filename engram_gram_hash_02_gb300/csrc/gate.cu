// Stage 4: the Engram gate, in place on the fp32 hyper-connection highway.
//
// Follows the NeMo "deepseek_v41.engram" page (_engram_gate_core: normalised,
// signed-square-root-gated value added to every fp32 stream; masked tokens keep their
// streams), the vLLM "deepseek_v41.common.engram" page (Engram: keys first, value last in
// the wkv output, clamp 1e-6) and the Atlas "engram_v41" page (stage 4: in place on the
// fp32 highway [T, hc, H]).
//
// One CTA per (token, stream). Each thread owns two groups of 8 consecutive hidden elements;
// it reads its part of the stream, the key, the value and the two norm weights once (16-byte
// loads, all issued before any arithmetic), accumulates sum h^2, sum key^2 and
// sum h*q*key*k, and keeps the stream and the value in registers. A warp-shuffle + shared
// memory reduction gives the gate; the threads add g * value and write the stream back.
// Stream traffic is one read and one write, the minimum; the value is read once per stream
// (hc-1 of those reads hit L2).
#include "internal.cuh"

namespace engram {
namespace {

constexpr int kItems = 2;      // groups of 8 elements per thread
constexpr int kMaxThreads = 512;

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ void unpack8(const uint4 v, float (&f)[8]) {
  f[0] = bf16lo(v.x); f[1] = bf16hi(v.x);
  f[2] = bf16lo(v.y); f[3] = bf16hi(v.y);
  f[4] = bf16lo(v.z); f[5] = bf16hi(v.z);
  f[6] = bf16lo(v.w); f[7] = bf16hi(v.w);
}

__device__ __forceinline__ void load8(const float* p, float (&f)[8]) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *reinterpret_cast<const float4*>(p + 4);
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
  f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

__global__ void __launch_bounds__(kMaxThreads)
gate_kernel(const GateParams p) {
  const int64_t t = blockIdx.x / p.hc;
  const int j = blockIdx.x - (int)(t * p.hc);
  if (p.token_mask != nullptr && __ldg(p.token_mask + t) == 0) {   // gate shut: untouched
    pdl_wait();
    return;
  }

  const int H = p.H;
  const int G = H >> 3;                                  // groups of 8
  float* __restrict__ h = p.streams + (t * p.hc + j) * (int64_t)H;
  const float* __restrict__ key = p.kv + t * (int64_t)(p.hc + 1) * H + (int64_t)j * H;
  const float* __restrict__ val = p.kv + t * (int64_t)(p.hc + 1) * H + (int64_t)p.hc * H;
  const uint16_t* __restrict__ qw = p.q_weight + (int64_t)j * H;
  const uint16_t* __restrict__ kw = p.k_weight + (int64_t)j * H;

  // the stream and the norm weights do not come from the projection: load them first
  float hv[kItems][8], kv[kItems][8], vv[kItems][8];
  uint4 qraw[kItems], kraw[kItems];
#pragma unroll
  for (int it = 0; it < kItems; ++it) {
    const int g = threadIdx.x + it * blockDim.x;
    if (g < G) {
      load8(h + 8 * g, hv[it]);
      qraw[it] = __ldg(reinterpret_cast<const uint4*>(qw + 8 * g));
      kraw[it] = __ldg(reinterpret_cast<const uint4*>(kw + 8 * g));
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) hv[it][e] = 0.f;
      qraw[it] = kraw[it] = make_uint4(0, 0, 0, 0);
    }
  }
  pdl_wait();                                            // kv comes from the projection
  pdl_trigger();
#pragma unroll
  for (int it = 0; it < kItems; ++it) {
    const int g = threadIdx.x + it * blockDim.x;
    if (g < G) {
      load8(key + 8 * g, kv[it]);
      load8(val + 8 * g, vv[it]);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) kv[it][e] = vv[it][e] = 0.f;
    }
  }
  float ssh = 0.f, ssk = 0.f, dot = 0.f;
#pragma unroll
  for (int it = 0; it < kItems; ++it) {
    float q[8], k[8];
    unpack8(qraw[it], q);
    unpack8(kraw[it], k);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float x = hv[it][e], y = kv[it][e];
      ssh = fmaf(x, x, ssh);
      ssk = fmaf(y, y, ssk);
      dot = fmaf(x * q[e], y * k[e], dot);
    }
  }

  // ---- block reduction of the three sums -------------------------------------------------------
  __shared__ float red[kMaxThreads / 32][3];
  __shared__ float gate;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
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
  if (threadIdx.x == 0) {
    const int nw = blockDim.x >> 5;
    float a = 0.f, b = 0.f, c = 0.f;
    for (int w = 0; w < nw; ++w) {
      a += red[w][0];
      b += red[w][1];
      c += red[w][2];
    }
    const float invH = 1.0f / (float)H;
    const float rh = rsqrtf(a * invH + p.eps);
    const float rk = rsqrtf(b * invH + p.eps);
    const float s = c * rh * rk / sqrtf((float)H);
    float ss = 0.f;                                      // sign(0) = 0
    if (s > 0.f) ss = sqrtf(fmaxf(s, p.clamp));
    else if (s < 0.f) ss = -sqrtf(fmaxf(-s, p.clamp));
    gate = 1.0f / (1.0f + expf(-ss));
  }
  __syncthreads();
  const float g = gate;

  // ---- h += g * value ----------------------------------------------------------------------------
#pragma unroll
  for (int it = 0; it < kItems; ++it) {
    const int gi = threadIdx.x + it * blockDim.x;
    if (gi < G) {
      float4 a, b;
      a.x = fmaf(g, vv[it][0], hv[it][0]); a.y = fmaf(g, vv[it][1], hv[it][1]);
      a.z = fmaf(g, vv[it][2], hv[it][2]); a.w = fmaf(g, vv[it][3], hv[it][3]);
      b.x = fmaf(g, vv[it][4], hv[it][4]); b.y = fmaf(g, vv[it][5], hv[it][5]);
      b.z = fmaf(g, vv[it][6], hv[it][6]); b.w = fmaf(g, vv[it][7], hv[it][7]);
      *reinterpret_cast<float4*>(h + 8 * gi) = a;
      *reinterpret_cast<float4*>(h + 8 * gi + 4) = b;
    }
  }
}

}  // namespace

cudaError_t launch_gate(const GateParams& p, cudaStream_t stream, bool pdl) {
  const int groups = p.H / 8;
  int threads = (groups + kItems - 1) / kItems;
  threads = ((threads + 31) / 32) * 32;
  if (threads > kMaxThreads) return cudaErrorInvalidValue;
  const int64_t blocks = p.T * p.hc;
  if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
  return launch_k(gate_kernel, dim3((unsigned)blocks), dim3(threads), 0, stream, pdl, p);
}

}  // namespace engram
