// Stage 4: the Engram gate, in place on the fp32 hyper-connection highway.
//
// Follows the NeMo "deepseek_v41.engram" page (_engram_gate_core: normalised,
// signed-square-root-gated value added to every fp32 stream; masked tokens keep their
// streams), the vLLM "deepseek_v41.common.engram" page (Engram: keys first, value last in
// the wkv output, clamp 1e-6) and the Atlas "engram_v41" page (stage 4: in place on the
// fp32 highway [T, hc, H]).
//
// One CTA per token. Each thread owns two groups of 8 consecutive hidden elements of every
// stream; it reads the streams, keys and norm weights once (16-byte loads), accumulates the
// three reductions per stream (sum h^2, sum key^2, sum h*q*key*k), and keeps the streams in
// registers. A warp-shuffle + shared-memory reduction gives the hc gates; the threads then
// add g_j * value to their registers and write the streams back. HBM traffic is one read and
// one write of the highway plus one read of kv, the minimum.
#include "internal.cuh"

namespace engram {
namespace {

constexpr int kItems = 2;  // groups of 8 elements per thread per stream

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ void unpack8(const uint4 v, float (&f)[8]) {
  f[0] = bf16lo(v.x); f[1] = bf16hi(v.x);
  f[2] = bf16lo(v.y); f[3] = bf16hi(v.y);
  f[4] = bf16lo(v.z); f[5] = bf16hi(v.z);
  f[6] = bf16lo(v.w); f[7] = bf16hi(v.w);
}

template <int HC>
__global__ void __launch_bounds__(512)
gate_kernel(const GateParams p) {
  const int64_t t = blockIdx.x;
  if (p.token_mask != nullptr && __ldg(p.token_mask + t) == 0) return;  // gate shut: untouched

  const int H = p.H;
  const int G = H >> 3;                                  // groups of 8 per stream
  float* __restrict__ h = p.streams + t * HC * (int64_t)H;
  const uint16_t* __restrict__ kv = p.kv + t * (HC + 1) * (int64_t)H;

  float hv[HC][kItems][8];
  float ssh[HC], ssk[HC], dot[HC];
#pragma unroll
  for (int j = 0; j < HC; ++j) ssh[j] = ssk[j] = dot[j] = 0.f;

#pragma unroll
  for (int it = 0; it < kItems; ++it) {
    const int g = threadIdx.x + it * blockDim.x;
    if (g < G) {
#pragma unroll
      for (int j = 0; j < HC; ++j) {
        const float4 a = *reinterpret_cast<const float4*>(h + j * H + 8 * g);
        const float4 b = *reinterpret_cast<const float4*>(h + j * H + 8 * g + 4);
        hv[j][it][0] = a.x; hv[j][it][1] = a.y; hv[j][it][2] = a.z; hv[j][it][3] = a.w;
        hv[j][it][4] = b.x; hv[j][it][5] = b.y; hv[j][it][6] = b.z; hv[j][it][7] = b.w;
        float key[8], qw[8], kw[8];
        unpack8(__ldg(reinterpret_cast<const uint4*>(kv + j * H + 8 * g)), key);
        unpack8(__ldg(reinterpret_cast<const uint4*>(p.q_weight + j * H + 8 * g)), qw);
        unpack8(__ldg(reinterpret_cast<const uint4*>(p.k_weight + j * H + 8 * g)), kw);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float x = hv[j][it][e];
          ssh[j] = fmaf(x, x, ssh[j]);
          ssk[j] = fmaf(key[e], key[e], ssk[j]);
          dot[j] = fmaf(x * qw[e], key[e] * kw[e], dot[j]);
        }
      }
    }
  }
  uint4 vraw[kItems];
#pragma unroll
  for (int it = 0; it < kItems; ++it) {
    const int g = threadIdx.x + it * blockDim.x;
    vraw[it] = g < G ? __ldg(reinterpret_cast<const uint4*>(kv + HC * H + 8 * g)) : make_uint4(0, 0, 0, 0);
  }

  // ---- block reduction of 3*HC partial sums ------------------------------------------------
  __shared__ float red[32][3 * HC];
  __shared__ float gate[HC];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int j = 0; j < HC; ++j) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      ssh[j] += __shfl_xor_sync(0xffffffffu, ssh[j], off);
      ssk[j] += __shfl_xor_sync(0xffffffffu, ssk[j], off);
      dot[j] += __shfl_xor_sync(0xffffffffu, dot[j], off);
    }
  }
  if (lane == 0) {
#pragma unroll
    for (int j = 0; j < HC; ++j) {
      red[warp][3 * j] = ssh[j];
      red[warp][3 * j + 1] = ssk[j];
      red[warp][3 * j + 2] = dot[j];
    }
  }
  __syncthreads();
  if (threadIdx.x < HC) {
    const int j = threadIdx.x;
    const int nw = blockDim.x >> 5;
    float a = 0.f, b = 0.f, c = 0.f;
    for (int w = 0; w < nw; ++w) {
      a += red[w][3 * j];
      b += red[w][3 * j + 1];
      c += red[w][3 * j + 2];
    }
    const float invH = 1.0f / (float)H;
    const float rh = rsqrtf(a * invH + p.eps);
    const float rk = rsqrtf(b * invH + p.eps);
    const float s = c * rh * rk / sqrtf((float)H);
    float ss = 0.f;                                      // sign(0) = 0
    if (s > 0.f) ss = sqrtf(fmaxf(s, p.clamp));
    else if (s < 0.f) ss = -sqrtf(fmaxf(-s, p.clamp));
    gate[j] = 1.0f / (1.0f + expf(-ss));
  }
  __syncthreads();

  // ---- h_j += g_j * value ---------------------------------------------------------------------
#pragma unroll
  for (int it = 0; it < kItems; ++it) {
    const int g = threadIdx.x + it * blockDim.x;
    if (g < G) {
      float v[8];
      unpack8(vraw[it], v);
#pragma unroll
      for (int j = 0; j < HC; ++j) {
        const float gj = gate[j];
        float4 a, b;
        a.x = fmaf(gj, v[0], hv[j][it][0]); a.y = fmaf(gj, v[1], hv[j][it][1]);
        a.z = fmaf(gj, v[2], hv[j][it][2]); a.w = fmaf(gj, v[3], hv[j][it][3]);
        b.x = fmaf(gj, v[4], hv[j][it][4]); b.y = fmaf(gj, v[5], hv[j][it][5]);
        b.z = fmaf(gj, v[6], hv[j][it][6]); b.w = fmaf(gj, v[7], hv[j][it][7]);
        *reinterpret_cast<float4*>(h + j * H + 8 * g) = a;
        *reinterpret_cast<float4*>(h + j * H + 8 * g + 4) = b;
      }
    }
  }
}

template <int HC>
cudaError_t launch_hc(const GateParams& p, cudaStream_t stream) {
  const int groups = p.H / 8;
  int threads = (groups + kItems - 1) / kItems;
  threads = ((threads + 31) / 32) * 32;
  gate_kernel<HC><<<(unsigned)p.T, threads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gate(const GateParams& p, cudaStream_t stream) {
  switch (p.hc) {
    case 1: return launch_hc<1>(p, stream);
    case 2: return launch_hc<2>(p, stream);
    case 3: return launch_hc<3>(p, stream);
    case 4: return launch_hc<4>(p, stream);
    case 5: return launch_hc<5>(p, stream);
    case 6: return launch_hc<6>(p, stream);
    case 7: return launch_hc<7>(p, stream);
    case 8: return launch_hc<8>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace engram
