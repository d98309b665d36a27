// K1 — router of "Step3.5 Flash 大模型技术深度解析" (jsqmd.com) §3.2.2: a linear
// layer gives each routed expert a logit, a softmax over all experts turns the
// logits into probabilities, and the k most probable experts are kept.
//
// Grid (ceil(T/16), ceil(E/32)); 256 threads.  Each block computes a 16-token x
// 32-expert tile of logits in fp32 (bf16 x upcast, fp32 W_r): the 8 warps split
// K into 8 slices, each lane holds a 4x4 register tile, and the slices are summed
// in warp order through shared memory (a fixed order: the logits are
// bit-identical run to run).  The last block to finish a token tile (an atomic
// ticket per tile) runs softmax and top-k for its 16 tokens, one warp per token,
// with shuffle reductions; ties go to the lower expert index.
#include "kernels.cuh"

#include <cfloat>

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxPerLane = kMaxExperts / 32;

__device__ __forceinline__ void bf16x4_to_f32(uint2 raw, float (&v)[4]) {
  v[0] = __uint_as_float(raw.x << 16);
  v[1] = __uint_as_float(raw.x & 0xFFFF0000u);
  v[2] = __uint_as_float(raw.y << 16);
  v[3] = __uint_as_float(raw.y & 0xFFFF0000u);
}

// (v, e) is better than (ov, oe): higher probability, then lower index.
__device__ __forceinline__ bool better(float v, int e, float ov, int oe) { return v > ov || (v == ov && e < oe); }

__global__ void __launch_bounds__(kThreads) router_kernel(const bf16* __restrict__ x,
                                                          const float* __restrict__ w_router, int T, int d, int E,
                                                          int k, float* __restrict__ logits, int* tickets,
                                                          int* __restrict__ idx, float* __restrict__ prob,
                                                          float* __restrict__ gap, int* counts) {
  __shared__ float part[kWarps][kRouterTok][kRouterExp];
  __shared__ int is_last;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * kRouterTok, e0 = blockIdx.y * kRouterExp;
  const int tq = lane >> 3, eq = lane & 7;
  const int kslice = d / kWarps;  // d % 128 == 0 -> a multiple of 16
  const int kbeg = warp * kslice;

  const bf16* xr[4];
  const float* wrow[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = min(t0 + tq * 4 + i, T - 1);
    xr[i] = x + static_cast<size_t>(t) * d + kbeg;
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int e = min(e0 + eq * 4 + j, E - 1);
    wrow[j] = w_router + static_cast<size_t>(e) * d + kbeg;
  }
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

  for (int kk = 0; kk < kslice; kk += 4) {
    float4 w4[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) w4[j] = __ldg(reinterpret_cast<const float4*>(wrow[j] + kk));
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float xv[4];
      bf16x4_to_f32(__ldg(reinterpret_cast<const uint2*>(xr[i] + kk)), xv);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        acc[i][j] = fmaf(xv[0], w4[j].x, acc[i][j]);
        acc[i][j] = fmaf(xv[1], w4[j].y, acc[i][j]);
        acc[i][j] = fmaf(xv[2], w4[j].z, acc[i][j]);
        acc[i][j] = fmaf(xv[3], w4[j].w, acc[i][j]);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) part[warp][tq * 4 + i][eq * 4 + j] = acc[i][j];
  __syncthreads();

  for (int o = threadIdx.x; o < kRouterTok * kRouterExp; o += kThreads) {
    const int tl = o / kRouterExp, el = o % kRouterExp;
    float s = part[0][tl][el];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) s += part[w][tl][el];
    const int t = t0 + tl, e = e0 + el;
    if (t < T && e < E) logits[static_cast<size_t>(t) * E + e] = s;
  }

  // The last expert-tile block of this token tile does softmax and top-k.
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int v = atomicAdd(&tickets[blockIdx.x], 1);
    is_last = (v == static_cast<int>(gridDim.y) - 1);
    if (is_last) tickets[blockIdx.x] = 0;  // ready for the next call
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();

  for (int r = warp; r < kRouterTok; r += kWarps) {
    const int t = t0 + r;
    if (t >= T) break;
    const float* zrow = logits + static_cast<size_t>(t) * E;
    float p[kMaxPerLane];
    float zmax = -FLT_MAX;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) {
      const int e = lane + 32 * i;
      p[i] = (e < E) ? __ldcg(zrow + e) : -FLT_MAX;
      zmax = fmaxf(zmax, p[i]);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) zmax = fmaxf(zmax, __shfl_xor_sync(0xffffffffu, zmax, off));
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) {
      const int e = lane + 32 * i;
      p[i] = (e < E) ? expf(p[i] - zmax) : 0.f;
      s += p[i];
    }
    // xor butterfly: every lane ends with the same, bit-identical sum
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) p[i] = p[i] / s;

    uint32_t taken = 0;
    float pk = 0.f;
    for (int j = 0; j <= k; ++j) {
      float bv = -1.f;
      int be = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < kMaxPerLane; ++i) {
        const int e = lane + 32 * i;
        if (e < E && !((taken >> i) & 1u) && p[i] > bv) {  // e grows with i: '>' keeps the lower index
          bv = p[i];
          be = e;
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int oe = __shfl_xor_sync(0xffffffffu, be, off);
        if (better(ov, oe, bv, be)) {
          bv = ov;
          be = oe;
        }
      }
      if (j < k) {
        if ((be & 31) == lane) taken |= 1u << (be >> 5);
        if (lane == 0) {
          idx[static_cast<size_t>(t) * k + j] = be;
          prob[static_cast<size_t>(t) * k + j] = bv;
          atomicAdd(&counts[be], 1);
        }
        pk = bv;
      } else if (gap != nullptr && lane == 0) {
        gap[t] = (be == 0x7fffffff) ? __int_as_float(0x7f800000) : (pk - bv);
      }
    }
  }
}

}  // namespace

cudaError_t launch_router(const bf16* x, const float* w_router, int T, int d, int E, int k, float* logits,
                          int* tickets, int* idx, float* prob, float* gap, int* counts, cudaStream_t stream) {
  if (T <= 0) return cudaSuccess;
  dim3 grid((T + kRouterTok - 1) / kRouterTok, (E + kRouterExp - 1) / kRouterExp);
  router_kernel<<<grid, kThreads, 0, stream>>>(x, w_router, T, d, E, k, logits, tickets, idx, prob, gap, counts);
  return cudaGetLastError();
}

}  // namespace moe
