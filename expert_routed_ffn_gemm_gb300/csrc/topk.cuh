// Softmax and top-k of one token by one warp, shared by the routing kernels
// (router_gemm.cu) and the few-token gate/up launch that ranks the tokens
// itself (expert_gemm.cu): the same arithmetic in both, so both give the same
// bits.  "Step3.5 Flash 大模型技术深度解析" (jsqmd.com) §3.2.2: a softmax over
// all routed experts, then the k most probable (ties: the lower index).
#pragma once
#include <cfloat>
#include <cstdint>

namespace moe {

// Best slot of a lane not yet taken: highest softmax numerator, then lowest
// slot (= lowest expert index, e = lane + 32 i); -1 when none is left.
template <int NS>
__device__ __forceinline__ int lane_head(const float (&q)[NS], uint32_t taken, int lane, int E) {
  int h = -1;
  float hv = 0.f;
#pragma unroll
  for (int i = 0; i < NS; ++i) {
    const bool ok = !((taken >> i) & 1u) && lane + 32 * i < E;
    if (ok && (h < 0 || q[i] > hv)) {
      h = i;
      hv = q[i];
    }
  }
  return h;
}

// Softmax, top-k (ties: lower index), gap, per-expert counts (counts != NULL)
// and the optional per-token statistics of token t, by one warp whose lane l
// holds the summed logits of experts l, l+32, ..., l+32(NS-1) in z.  The
// ranking uses the softmax numerators q_e = exp(z_e - max z), which order the
// experts as the probabilities q_e / sum q do; each of the k+1 selection
// rounds is one warp max over the lanes' heads, then the lowest expert index
// among the heads holding it; only the winning lane finds its next head.
// renorm != 0: the k weights are divided by their sum (slot order).  tokstats
// (or NULL): the probability mass of each of n_groups equal expert groups,
// then the entropy -sum p ln p ([T][n_groups+1]).
template <int NS>
__device__ __forceinline__ void finish_token(float (&q)[NS], int t, int lane, int E, int k, int renorm,
                                             int* __restrict__ idx, float* __restrict__ prob,
                                             float* __restrict__ gap, int* counts, float* __restrict__ tokstats,
                                             int n_groups, int* sel = nullptr) {
  float zmax = -FLT_MAX;
#pragma unroll
  for (int i = 0; i < NS; ++i)
    if (lane + 32 * i < E) zmax = fmaxf(zmax, q[i]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) zmax = fmaxf(zmax, __shfl_xor_sync(0xffffffffu, zmax, off));
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < NS; ++i) {
    q[i] = (lane + 32 * i < E) ? expf(q[i] - zmax) : 0.f;
    s += q[i];
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);

  if (tokstats != nullptr) {
    // group masses (group of expert e = e / (E / n_groups)) and entropy
    const int per_group = E / n_groups;
    float* out = tokstats + static_cast<size_t>(t) * (n_groups + 1);
    for (int g = 0; g < n_groups; ++g) {
      float m = 0.f;
#pragma unroll
      for (int i = 0; i < NS; ++i) {
        const int e = lane + 32 * i;
        if (e < E && e / per_group == g) m += q[i] / s;
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m += __shfl_xor_sync(0xffffffffu, m, off);
      if (lane == 0) out[g] = m;
    }
    float h = 0.f;
#pragma unroll
    for (int i = 0; i < NS; ++i) {
      const int e = lane + 32 * i;
      const float p = q[i] / s;
      if (e < E && p > 0.f) h -= p * logf(p);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) h += __shfl_xor_sync(0xffffffffu, h, off);
    if (lane == 0) out[n_groups] = h;
  }

  // Selection rounds.  Numerators are >= 0, so their bit patterns order like
  // the values; key = bits + 1 (0 marks a lane with nothing left).
  uint32_t taken = 0u;
  int head = lane_head(q, taken, lane, E);
  float pk = 0.f, sel_sum = 0.f, my_p = 0.f;
  int my_e = 0;
  for (int j = 0; j <= k; ++j) {
    float hq = 0.f;
#pragma unroll
    for (int i = 0; i < NS; ++i)
      if (i == head) hq = q[i];
    const uint32_t hk = head >= 0 ? __float_as_uint(hq) + 1u : 0u;
    const uint32_t mk = __reduce_max_sync(0xffffffffu, hk);
    const uint32_t my_idx = head >= 0 ? static_cast<uint32_t>(lane + 32 * head) : 0x7fffffffu;
    const int be = static_cast<int>(__reduce_min_sync(0xffffffffu, (mk != 0u && hk == mk) ? my_idx : 0x7fffffffu));
    const float bv = mk ? __uint_as_float(mk - 1u) / s : -1.f;
    if (j < k) {
      if (be != 0x7fffffff && (be & 31) == lane) {  // the winner takes its head and finds the next one
        taken |= 1u << head;
        head = lane_head(q, taken, lane, E);
      }
      if (lane == j) {  // lane j keeps slot j
        my_e = be;
        my_p = bv;
      }
      sel_sum += bv;  // same value and order in every lane
      pk = bv;
    } else if (gap != nullptr && lane == 0) {
      gap[t] = (be == 0x7fffffff) ? __int_as_float(0x7f800000) : (pk - bv);
    }
  }
  if (lane < k) {
    idx[static_cast<size_t>(t) * k + lane] = my_e;
    prob[static_cast<size_t>(t) * k + lane] = renorm ? my_p / sel_sum : my_p;
    if (counts != nullptr) atomicAdd(&counts[my_e], 1);
    if (sel != nullptr) sel[t * k + lane] = my_e;
  }
}

}  // namespace moe
