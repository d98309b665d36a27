// K2 dispatch, the row gather, and K5 combine.
//
// "Step3.5 Flash 大模型技术深度解析" (jsqmd.com) §3.2.2: every token runs its 8
// chosen routed experts plus the shared expert, and the 9 outputs are summed
// with weights.  Dispatch lays the (token, expert) pairs out expert by expert so
// that each expert's rows are one contiguous block (the grouped GEMM's rows);
// combine gathers a token's rows back and sums them.  Both are deterministic:
// dispatch orders rows inside an expert by token index with block-local ranks
// (no order-dependent atomics), combine sums in a fixed order.
#include <cuda_fp8.h>

#include <mutex>

#include "../../include/moe.h"
#include "kernels.cuh"

namespace moe {
namespace {

constexpr int kDispatchThreads = 256;

// Block-wide exclusive scan of one int per thread (256 threads); returns the
// thread's exclusive prefix and writes the block total to *total.
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  int base = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kDispatchThreads / 32; ++w) {
    const int s = warp_sums[w];
    base += (w < warp) ? s : 0;
    tot += s;
  }
  __syncthreads();
  *total = tot;
  return base + incl - v;
}

// Block e < E: offset of expert e, then a stable compaction over tokens of the
// assignments (t, j) with idx[t][j] == e.  Block 0 also writes offsets[].
__global__ void __launch_bounds__(kDispatchThreads) dispatch_kernel(const int* __restrict__ idx,
                                                                    const int* __restrict__ counts, int T, int E,
                                                                    int k, int has_shared, int* __restrict__ offsets,
                                                                    int* __restrict__ perm, int* __restrict__ inv,
                                                                    int* __restrict__ chunk_base) {
  __shared__ int warp_sums[kDispatchThreads / 32];
  const int e = blockIdx.x;

  // offset of expert e = counts[0] + ... + counts[e-1]
  int part = 0;
  for (int i = threadIdx.x; i < e; i += kDispatchThreads) part += counts[i];
  int base_e;
  block_exclusive_scan(part, warp_sums, &base_e);

  if (e == 0) {
    // offsets[0..E]: each thread scans a contiguous run of experts
    const int per = (E + kDispatchThreads - 1) / kDispatchThreads;
    const int b = threadIdx.x * per;
    int local = 0;
    for (int i = b; i < min(E, b + per); ++i) local += counts[i];
    int total;
    const int pre = block_exclusive_scan(local, warp_sums, &total);
    int run = pre;
    for (int i = b; i < min(E, b + per); ++i) {
      offsets[i] = run;
      run += counts[i];
    }
    if (threadIdx.x == 0) {
      offsets[E] = total;
      offsets[E + 1] = total + (has_shared ? T : 0);
    }
    // chunk_base[0..E+1]: the same scan over ceil(count / kYpRows)
    local = 0;
    for (int i = b; i < min(E, b + per); ++i) local += (counts[i] + kYpRows - 1) / kYpRows;
    const int cpre = block_exclusive_scan(local, warp_sums, &total);
    run = cpre;
    for (int i = b; i < min(E, b + per); ++i) {
      chunk_base[i] = run;
      run += (counts[i] + kYpRows - 1) / kYpRows;
    }
    if (threadIdx.x == 0) {
      chunk_base[E] = total;
      chunk_base[E + 1] = total + (has_shared ? (T + kYpRows - 1) / kYpRows : 0);
    }
  }

  int running = 0;
  for (int t0 = 0; t0 < T; t0 += kDispatchThreads) {
    const int t = t0 + threadIdx.x;
    int jsel = -1;
    if (t < T) {
      const int* row = idx + static_cast<size_t>(t) * k;
      for (int j = 0; j < k; ++j)
        if (__ldg(row + j) == e) jsel = j;
    }
    int chunk_total;
    const int r = block_exclusive_scan(jsel >= 0 ? 1 : 0, warp_sums, &chunk_total);
    if (jsel >= 0) {
      const int pos = base_e + running + r;
      const int a = t * k + jsel;
      perm[pos] = a;
      inv[a] = pos;
    }
    running += chunk_total;
  }
}

// One warp per dispatch row: xp[pos] = x[token(pos)], 16-byte vectors; with
// to_f16 each bf16 value is rewritten as the nearest fp16.
template <bool TO_F16>
__global__ void __launch_bounds__(256) gather_kernel(const bf16* __restrict__ x, const int* __restrict__ perm,
                                                     int T, int k, int d, int rows, void* __restrict__ xp) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp >= rows) return;
  const int Tk = T * k;
  const int t = (warp < Tk) ? (__ldg(perm + warp) / k) : (warp - Tk);
  const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * d);
  uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(xp) + static_cast<size_t>(warp) * d);
  for (int c = lane; c < d / 8; c += 32) {
    uint4 v = __ldg(src + c);
    if (TO_F16) {
      uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float lo = __uint_as_float(w[i] << 16), hi = __uint_as_float(w[i] & 0xffff0000u);
        w[i] = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(lo))) |
               (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(hi))) << 16);
      }
    }
    dst[c] = v;
  }
}

constexpr int kCombineBatch = 5;  // terms whose loads are in flight together

// 2^e for an int8 exponent in [-126, 113], exact.
__device__ __forceinline__ float pow2i(int e) { return __uint_as_float(static_cast<uint32_t>(e + 127) << 23); }

// One block per token: y[t] = Yp[inv[t*k+0]] + ... + Yp[inv[t*k+k-1]] + Yp[T*k+t],
// summed in fp32 in that order.  Each term is read back exactly as h * 2^e
// (h fp16 from yp, e the int8 exponent of its feature in the row's chunk).
// d/8 threads (<= 1024): one 8-element chunk each, so every load of a token is
// in flight at once.
__global__ void __launch_bounds__(1024, 1) combine_kernel(const __half* __restrict__ yp,
                                                          const int8_t* __restrict__ yexp,
                                                          const __half* __restrict__ yp_routed,
                                                          const int8_t* __restrict__ yexp_routed,
                                                          const int* __restrict__ idx, const int* __restrict__ inv,
                                                          const int* __restrict__ offsets,
                                                          const int* __restrict__ chunk_base, int T, int k, int E,
                                                          int d, int has_shared, void* __restrict__ y,
                                                          int out_fp32) {
  const int t = blockIdx.x;
  __shared__ int pos[kMaxTopK + 1];
  __shared__ int chunk[kMaxTopK + 1];
  if (threadIdx.x <= k) {
    const int j = threadIdx.x;
    const int g = (j < k) ? __ldg(idx + static_cast<size_t>(t) * k + j) : E;
    const int p = (j < k) ? __ldg(inv + static_cast<size_t>(t) * k + j) : T * k + t;
    pos[j] = p;
    chunk[j] = __ldg(chunk_base + g) + (p - __ldg(offsets + g)) / kYpRows;
  }
  __syncthreads();
  const int nterms = k + (has_shared ? 1 : 0);
  // routed rows (slots j < k) from yp_routed / yexp_routed when given
  // (expert parallelism: the rows the experts' owners sent back)
  const __half* yp_r = yp_routed ? yp_routed : yp;
  const int8_t* ye_r = yp_routed ? yexp_routed : yexp;
  for (int c = threadIdx.x; c < d / 8; c += blockDim.x) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    // terms in batches of kCombineBatch: every load of a batch is issued
    // before any of them is summed (the sum itself stays in slot order)
    for (int j0 = 0; j0 < nterms; j0 += kCombineBatch) {
      uint4 raw[kCombineBatch];
      uint2 ex[kCombineBatch];
#pragma unroll
      for (int b = 0; b < kCombineBatch; ++b) {
        if (j0 + b < nterms) {
          const bool routed = j0 + b < k;
          raw[b] = __ldcs(reinterpret_cast<const uint4*>((routed ? yp_r : yp) + static_cast<size_t>(pos[j0 + b]) * d) +
                          c);
          ex[b] = __ldg(reinterpret_cast<const uint2*>((routed ? ye_r : yexp) + static_cast<size_t>(chunk[j0 + b]) * d) +
                        c);
        }
      }
#pragma unroll
      for (int b = 0; b < kCombineBatch; ++b) {
        if (j0 + b < nterms) {
          const uint32_t w[4] = {raw[b].x, raw[b].y, raw[b].z, raw[b].w};
          const uint32_t eb[2] = {ex[b].x, ex[b].y};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int e0 = static_cast<int8_t>((eb[i >> 1] >> (16 * (i & 1))) & 0xffu);
            const int e1 = static_cast<int8_t>((eb[i >> 1] >> (16 * (i & 1) + 8)) & 0xffu);
            acc[2 * i] += __half2float(__ushort_as_half(static_cast<unsigned short>(w[i] & 0xffffu))) * pow2i(e0);
            acc[2 * i + 1] += __half2float(__ushort_as_half(static_cast<unsigned short>(w[i] >> 16))) * pow2i(e1);
          }
        }
      }
    }
    if (out_fp32) {
      float4* dst = reinterpret_cast<float4*>(static_cast<float*>(y) + static_cast<size_t>(t) * d) + 2 * c;
      dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    } else {
      uint4 o;
      uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 pr = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
        ow[i] = *reinterpret_cast<const uint32_t*>(&pr);
      }
      reinterpret_cast<uint4*>(static_cast<bf16*>(y) + static_cast<size_t>(t) * d)[c] = o;
    }
  }
}

}  // namespace

cudaError_t launch_dispatch(const int* idx, const int* counts, int T, int E, int k, int has_shared, int* offsets,
                            int* perm, int* inv, int* chunk_base, cudaStream_t stream) {
  dispatch_kernel<<<E, kDispatchThreads, 0, stream>>>(idx, counts, T, E, k, has_shared, offsets, perm, inv,
                                                      chunk_base);
  return cudaGetLastError();
}

cudaError_t launch_gather(const bf16* x, const int* perm, int T, int k, int d, int has_shared, void* xp,
                          bool to_f16, cudaStream_t stream) {
  const int rows = T * k + (has_shared ? T : 0);
  if (rows == 0) return cudaSuccess;
  const int blocks = (rows + 7) / 8;
  if (to_f16)
    gather_kernel<true><<<blocks, 256, 0, stream>>>(x, perm, T, k, d, rows, xp);
  else
    gather_kernel<false><<<blocks, 256, 0, stream>>>(x, perm, T, k, d, rows, xp);
  return cudaGetLastError();
}

// One block per row: the row's largest magnitude by a block reduction, then
// every element divided by the scale and rounded to E4M3 (satfinite).
__global__ void __launch_bounds__(256) quantize_e4m3_kernel(const bf16* __restrict__ w, int cols,
                                                            uint8_t* __restrict__ q, float* __restrict__ s) {
  __shared__ float red[8];
  const size_t r = blockIdx.x;
  const bf16* row = w + r * cols;
  float amax = 0.f;
  for (int i = threadIdx.x; i < cols; i += 256) amax = fmaxf(amax, fabsf(__bfloat162float(row[i])));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
  const float sc = __fdiv_rn(amax, 448.0f);
  if (threadIdx.x == 0) s[r] = sc;
  for (int i = threadIdx.x; i < cols; i += 256) {
    const float v = __bfloat162float(row[i]);
    q[r * cols + i] =
        sc > 0.f ? static_cast<uint8_t>(__nv_cvt_float_to_fp8(__fdiv_rn(v, sc), __NV_SATFINITE, __NV_E4M3)) : 0;
  }
}

// One block: prefix sums over the (source, expert) groups of the rows and of
// their 16-row exponent chunks, in source-major order.
__global__ void ep_groups_kernel(const int* __restrict__ recv_counts, int S, int E_loc, int* __restrict__ offsets,
                                 int* __restrict__ chunk_base, int* __restrict__ chunks_per_source) {
  if (threadIdx.x != 0) return;
  int rows = 0, chunks = 0;
  for (int s = 0; s < S; ++s) {
    const int c0 = chunks;
    for (int e = 0; e < E_loc; ++e) {
      const int g = s * E_loc + e;
      offsets[g] = rows;
      chunk_base[g] = chunks;
      const int n = recv_counts[g];
      rows += n;
      chunks += (n + kYpRows - 1) / kYpRows;
    }
    chunks_per_source[s] = chunks - c0;
  }
  offsets[S * E_loc] = rows;
  chunk_base[S * E_loc] = chunks;
}

__global__ void gather_weights_kernel(const int* __restrict__ perm, const float* __restrict__ prob, int n,
                                      float* __restrict__ w) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) w[i] = prob[perm[i]];
}

__global__ void iota_kernel(int* __restrict__ v, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) v[i] = i;
}

cudaError_t launch_ep_groups(const int* recv_counts, int S, int E_loc, int* offsets, int* chunk_base,
                             int* chunks_per_source, cudaStream_t stream) {
  ep_groups_kernel<<<1, 32, 0, stream>>>(recv_counts, S, E_loc, offsets, chunk_base, chunks_per_source);
  return cudaGetLastError();
}

cudaError_t launch_gather_weights(const int* perm, const float* prob, int n, float* w, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  gather_weights_kernel<<<(n + 255) / 256, 256, 0, stream>>>(perm, prob, n, w);
  return cudaGetLastError();
}

cudaError_t launch_iota(int* v, int n, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  iota_kernel<<<(n + 255) / 256, 256, 0, stream>>>(v, n);
  return cudaGetLastError();
}

cudaError_t launch_quantize_e4m3(const bf16* w, long long rows, int cols, uint8_t* q, float* s,
                                 cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  if (rows > 0x7fffffffll) return cudaErrorInvalidValue;
  quantize_e4m3_kernel<<<static_cast<unsigned>(rows), 256, 0, stream>>>(w, cols, q, s);
  return cudaGetLastError();
}

cudaError_t launch_combine(const __half* yp, const int8_t* yexp, const __half* yp_routed, const int8_t* yexp_routed,
                           const int* idx, const int* inv, const int* offsets, const int* chunk_base, int T, int k,
                           int E, int d, int has_shared, void* y, int out_fp32, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const int chunks = d / 8;
  const int threads = chunks > 1024 ? 1024 : (chunks < 32 ? 32 : chunks);
  combine_kernel<<<T, threads, 0, stream>>>(yp, yexp, yp_routed, yexp_routed, idx, inv, offsets, chunk_base, T, k,
                                            E, d, has_shared, y, out_fp32);
  return cudaGetLastError();
}

// ----------------------------------------------------------------------------
// Allocation-free dispatch (moe_dispatch_noalloc in include/moe.h).
//
// Its only scratch, the per-expert row counts, lives in the file-scope device
// array below instead of a handle's workspace, so the entry point needs no
// moe_init and never allocates.  The array holds kNoAllocMaxExperts ints on
// every GPU that loads this library, for the life of the process.
namespace {

constexpr int kNoAllocMaxExperts = kMaxExperts;
__device__ __align__(256) int g_noalloc_counts[kNoAllocMaxExperts];

// counts[e] = number of entries of idx equal to e; entries outside [0, E) are skipped.
__global__ void noalloc_histogram_kernel(const int* __restrict__ idx, long long n, int E, int* counts) {
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int e = __ldg(idx + i);
    if (e >= 0 && e < E) atomicAdd(&counts[e], 1);
  }
}

// dispatch_kernel without the inverse permutation: block e < E writes the
// stable expert-major positions of expert e's rows.
__global__ void __launch_bounds__(kDispatchThreads) noalloc_dispatch_kernel(const int* __restrict__ idx,
                                                                            const int* __restrict__ counts, int T,
                                                                            int E, int k, int has_shared,
                                                                            int* __restrict__ offsets,
                                                                            int* __restrict__ perm) {
  __shared__ int warp_sums[kDispatchThreads / 32];
  const int e = blockIdx.x;
  int part = 0;
  for (int i = threadIdx.x; i < e; i += kDispatchThreads) part += counts[i];
  int base_e;
  block_exclusive_scan(part, warp_sums, &base_e);
  if (e == 0) {
    const int per = (E + kDispatchThreads - 1) / kDispatchThreads;
    const int b = threadIdx.x * per;
    int local = 0;
    for (int i = b; i < min(E, b + per); ++i) local += counts[i];
    int total;
    int run = block_exclusive_scan(local, warp_sums, &total);
    for (int i = b; i < min(E, b + per); ++i) {
      offsets[i] = run;
      run += counts[i];
    }
    if (threadIdx.x == 0) {
      offsets[E] = total;
      offsets[E + 1] = total + (has_shared ? T : 0);
    }
  }
  int running = 0;
  for (int t0 = 0; t0 < T; t0 += kDispatchThreads) {
    const int t = t0 + threadIdx.x;
    int jsel = -1;
    if (t < T) {
      const int* row = idx + static_cast<size_t>(t) * k;
      for (int j = 0; j < k; ++j)
        if (__ldg(row + j) == e) jsel = j;
    }
    int chunk_total;
    const int r = block_exclusive_scan(jsel >= 0 ? 1 : 0, warp_sums, &chunk_total);
    if (jsel >= 0) perm[base_e + running + r] = t * k + jsel;
    running += chunk_total;
  }
}

// Device address of g_noalloc_counts, looked up once per device.
constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mutex;
int* g_noalloc_ptr[kNoAllocMaxDevices] = {};

cudaError_t noalloc_counts(int** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kNoAllocMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_counts);
    if (e != cudaSuccess) return e;
    g_noalloc_ptr[dev] = static_cast<int*>(p);
  }
  *out = g_noalloc_ptr[dev];
  return cudaSuccess;
}

}  // namespace

}  // namespace moe

extern "C" int moe_dispatch_noalloc(const int* idx, int T, int n_experts, int top_k, int has_shared, int* offsets,
                                    int* perm, void* stream) {
  if (T < 0 || n_experts <= 0 || top_k <= 0 || top_k > n_experts || (has_shared != 0 && has_shared != 1))
    return MOE_ERR_INVALID_ARG;
  if (n_experts > moe::kNoAllocMaxExperts || top_k > moe::kMaxTopK) return MOE_ERR_UNSUPPORTED;
  if (static_cast<long long>(top_k + 1) * T >= (1ll << 31)) return MOE_ERR_UNSUPPORTED;
  if (offsets == nullptr || (T > 0 && (idx == nullptr || perm == nullptr))) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(idx) | reinterpret_cast<uintptr_t>(offsets) |
       reinterpret_cast<uintptr_t>(perm)) & 3u)
    return MOE_ERR_INVALID_ARG;
  int* counts = nullptr;
  if (moe::noalloc_counts(&counts) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the array keeps the previous call's counts: clear it first
  if (cudaMemsetAsync(counts, 0, sizeof(int) * n_experts, s) != cudaSuccess) return MOE_ERR_CUDA;
  const long long n = static_cast<long long>(T) * top_k;
  if (n > 0) {
    const int blocks = static_cast<int>((n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024);
    moe::noalloc_histogram_kernel<<<blocks, 256, 0, s>>>(idx, n, n_experts, counts);
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  }
  moe::noalloc_dispatch_kernel<<<n_experts, moe::kDispatchThreads, 0, s>>>(idx, counts, T, n_experts, top_k,
                                                                           has_shared, offsets, perm);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
