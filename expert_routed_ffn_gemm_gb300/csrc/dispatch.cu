// K2 dispatch, the row gather, and K5 combine.
//
// "Step3.5 Flash 大模型技术深度解析" (jsqmd.com) §3.2.2: every token runs its 8
// chosen routed experts plus the shared expert, and the 9 outputs are summed
// with weights.  Dispatch lays the (token, expert) pairs out expert by expert so
// that each expert's rows are one contiguous block (the grouped GEMM's rows);
// combine gathers a token's rows back and sums them.  Both are deterministic:
// dispatch orders rows inside an expert by token index with block-local ranks
// (no order-dependent atomics), combine sums in a fixed order.
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
                                                                    int* __restrict__ perm, int* __restrict__ inv) {
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

// One warp per dispatch row: xp[pos] = x[token(pos)], 16-byte vectors.
__global__ void __launch_bounds__(256) gather_kernel(const bf16* __restrict__ x, const int* __restrict__ perm,
                                                     int T, int k, int d, int rows, bf16* __restrict__ xp) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp >= rows) return;
  const int Tk = T * k;
  const int t = (warp < Tk) ? (__ldg(perm + warp) / k) : (warp - Tk);
  const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * d);
  uint4* dst = reinterpret_cast<uint4*>(xp + static_cast<size_t>(warp) * d);
  for (int c = lane; c < d / 8; c += 32) dst[c] = __ldg(src + c);
}

// One block per token: y[t] = Yp[inv[t*k+0]] + ... + Yp[inv[t*k+k-1]] + Yp[T*k+t],
// summed in fp32 in that order (Yp rows are fp32).  d/8 threads (<= 1024): one
// 8-element chunk each, so every load of a token is in flight at once.
__global__ void __launch_bounds__(1024) combine_kernel(const float* __restrict__ yp, const int* __restrict__ inv,
                                                      int T, int k, int d, int has_shared, void* __restrict__ y,
                                                      int out_fp32) {
  const int t = blockIdx.x;
  __shared__ int pos[kMaxTopK + 1];
  if (threadIdx.x < k) pos[threadIdx.x] = __ldg(inv + static_cast<size_t>(t) * k + threadIdx.x);
  if (threadIdx.x == 0) pos[k] = T * k + t;
  __syncthreads();
  const int nterms = k + (has_shared ? 1 : 0);
  for (int c = threadIdx.x; c < d / 8; c += blockDim.x) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int j = 0; j < nterms; ++j) {
      const float4* src = reinterpret_cast<const float4*>(yp + static_cast<size_t>(pos[j]) * d) + 2 * c;
      const float4 a = __ldcs(src), b = __ldcs(src + 1);
      acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
      acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
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
                            int* perm, int* inv, cudaStream_t stream) {
  dispatch_kernel<<<E, kDispatchThreads, 0, stream>>>(idx, counts, T, E, k, has_shared, offsets, perm, inv);
  return cudaGetLastError();
}

cudaError_t launch_gather(const bf16* x, const int* perm, int T, int k, int d, int has_shared, bf16* xp,
                          cudaStream_t stream) {
  const int rows = T * k + (has_shared ? T : 0);
  if (rows == 0) return cudaSuccess;
  const int blocks = (rows + 7) / 8;
  gather_kernel<<<blocks, 256, 0, stream>>>(x, perm, T, k, d, rows, xp);
  return cudaGetLastError();
}

cudaError_t launch_combine(const float* yp, const int* inv, int T, int k, int d, int has_shared, void* y,
                           int out_fp32, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const int chunks = d / 8;
  const int threads = chunks > 1024 ? 1024 : (chunks < 32 ? 32 : chunks);
  combine_kernel<<<T, threads, 0, stream>>>(yp, inv, T, k, d, has_shared, y, out_fp32);
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
