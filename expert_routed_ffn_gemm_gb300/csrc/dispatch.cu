// K2 dispatch, the row scatter into dispatch order, and K5 combine.
//
// "Step3.5 Flash 大模型技术深度解析" (jsqmd.com) §3.2.2: every token runs its 8
// chosen routed experts plus the shared expert, and the 9 outputs are summed
// with weights.  Dispatch lays the (token, expert) pairs out expert by expert so
// that each expert's rows are one contiguous block (the grouped GEMM's rows);
// combine gathers a token's rows back and sums them.  Both are deterministic:
// dispatch orders rows inside an expert by token index with block-local ranks
// (no order-dependent atomics), combine sums in a fixed order.
#include <cuda_fp8.h>

#include <cstdlib>
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

// offsets[0..E+1] (exclusive prefix of the counts, then the shared expert's T
// rows) and chunk_base[0..E+1] (the same over ceil(count / kYpRows), the
// shared expert's chunks from shared_chunk0(T, k, E) on), by one
// block whose threads each scan a contiguous run of experts.  base (shared
// memory, or NULL) gets offsets[0..E-1] too.
__device__ void write_offsets(const int* __restrict__ counts, int T, int E, int k, int has_shared,
                              int* __restrict__ offsets, int* __restrict__ chunk_base, int* warp_sums, int* base) {
  const int per = (E + kDispatchThreads - 1) / kDispatchThreads;
  const int b = threadIdx.x * per;
  int local = 0;
  for (int i = b; i < min(E, b + per); ++i) local += counts[i];
  int total;
  const int pre = block_exclusive_scan(local, warp_sums, &total);
  int run = pre;
  for (int i = b; i < min(E, b + per); ++i) {
    if (offsets != nullptr) offsets[i] = run;
    if (base != nullptr) base[i] = run;
    run += counts[i];
  }
  if (offsets == nullptr) return;
  if (threadIdx.x == 0) {
    offsets[E] = total;
    offsets[E + 1] = total + (has_shared ? T : 0);
  }
  local = 0;
  for (int i = b; i < min(E, b + per); ++i) local += (counts[i] + kYpRows - 1) / kYpRows;
  const int cpre = block_exclusive_scan(local, warp_sums, &total);
  run = cpre;
  for (int i = b; i < min(E, b + per); ++i) {
    chunk_base[i] = run;
    run += (counts[i] + kYpRows - 1) / kYpRows;
  }
  if (threadIdx.x == 0) {
    chunk_base[E] = shared_chunk0(T, k, E);  // the routed chunks end at total <= this
    chunk_base[E + 1] = chunk_base[E] + (has_shared ? (T + kYpRows - 1) / kYpRows : 0);
  }
}

// Block e < E: offset of expert e, then a stable compaction over tokens of the
// assignments (t, j) with idx[t][j] == e.  Block 0 also writes offsets[].
__global__ void __launch_bounds__(kDispatchThreads) dispatch_kernel(const int* __restrict__ idx,
                                                                    const int* __restrict__ counts, int T, int E,
                                                                    int k, int has_shared, int* __restrict__ offsets,
                                                                    int* __restrict__ perm, int* __restrict__ inv,
                                                                    int* __restrict__ chunk_base) {
  pdl_trigger();
  pdl_wait();
  __shared__ int warp_sums[kDispatchThreads / 32];
  const int e = blockIdx.x;

  // offset of expert e = counts[0] + ... + counts[e-1]
  int part = 0;
  for (int i = threadIdx.x; i < e; i += kDispatchThreads) part += counts[i];
  int base_e;
  block_exclusive_scan(part, warp_sums, &base_e);

  if (e == 0) write_offsets(counts, T, E, k, has_shared, offsets, chunk_base, warp_sums, nullptr);

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
      if (MOE_DBG_OK(pos >= 0 && pos < T * k)) {
        perm[pos] = a;
        inv[a] = pos;
      }
    }
    running += chunk_total;
  }
}

// Many tokens: the tokens are cut into chunks of kChunkTokens (8 warps x 32
// lanes, lane l of warp w = token chunk*256 + 32w + l).  A chunk's lane masks
// mask[w][e] (bit l: that token chose expert e; a token chooses an expert at
// most once) give every row's rank among the chunk's rows of its expert in
// token order; hist/scan turn the chunks' counts into each chunk's first row
// per expert.  Three passes, no atomics outside shared memory, and the same
// stable token order as dispatch_kernel.
constexpr int kChunkTokens = kDispatchThreads;
constexpr int kChunkWarps = kChunkTokens / 32;

__device__ __forceinline__ void chunk_masks(const int* __restrict__ idx, int T, int E, int k, uint32_t* mask) {
  for (int i = threadIdx.x; i < kChunkWarps * E; i += kChunkTokens) mask[i] = 0u;
  __syncthreads();
  const int t = blockIdx.x * kChunkTokens + threadIdx.x;
  if (t < T) {
    uint32_t* wm = mask + (threadIdx.x >> 5) * E;
    const uint32_t bit = 1u << (threadIdx.x & 31);
    const int* row = idx + static_cast<size_t>(t) * k;
    for (int j = 0; j < k; ++j) {
      const int e = __ldg(row + j);
      if (e >= 0 && e < E) atomicOr(wm + e, bit);
    }
  }
  __syncthreads();
}

// Pass 1: hist[chunk][e] = rows of expert e among the chunk's tokens.
__global__ void __launch_bounds__(kChunkTokens) chunk_hist_kernel(const int* __restrict__ idx, int T, int E, int k,
                                                                  int* __restrict__ hist) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ uint32_t mask[];
  chunk_masks(idx, T, E, k, mask);
  for (int e = threadIdx.x; e < E; e += kChunkTokens) {
    int n = 0;
#pragma unroll
    for (int w = 0; w < kChunkWarps; ++w) n += __popc(mask[w * E + e]);
    hist[static_cast<size_t>(blockIdx.x) * E + e] = n;
  }
}

// Pass 2: hist[c][e] becomes the exclusive prefix over chunks c' < c, and
// counts[e] the total.  Block = 32 experts x kScanParts runs of chunks; each
// thread sums its run, the runs' sums are scanned in shared memory, then each
// thread writes its run's prefixes.
constexpr int kScanParts = 8;
__global__ void __launch_bounds__(32 * kScanParts) chunk_scan_kernel(int* __restrict__ hist, int n_chunks, int E,
                                                                     int* __restrict__ counts) {
  pdl_trigger();
  pdl_wait();
  __shared__ int part_sum[kScanParts][32];
  const int ex = threadIdx.x & 31, part = threadIdx.x >> 5;
  const int e = blockIdx.x * 32 + ex;
  const int per = (n_chunks + kScanParts - 1) / kScanParts;
  const int c0 = part * per, c1 = min(n_chunks, c0 + per);
  int sum = 0;
  if (e < E)
    for (int c = c0; c < c1; ++c) sum += hist[static_cast<size_t>(c) * E + e];
  part_sum[part][ex] = sum;
  __syncthreads();
  int run = 0;
  for (int q = 0; q < part; ++q) run += part_sum[q][ex];
  if (e < E) {
    for (int c = c0; c < c1; ++c) {
      const int v = hist[static_cast<size_t>(c) * E + e];
      hist[static_cast<size_t>(c) * E + e] = run;
      run += v;
    }
    if (part == kScanParts - 1) counts[e] = run;
  }
}

// Pass 3: pos = offsets[e] + first row of the chunk for e + the rows of e in
// earlier warps of the chunk + the lower lanes of this warp that chose e.
// Block 0 also writes offsets[] and chunk_base[].
__global__ void __launch_bounds__(kChunkTokens) chunk_place_kernel(const int* __restrict__ idx,
                                                                   const int* __restrict__ counts,
                                                                   const int* __restrict__ chunk_first, int T, int E,
                                                                   int k, int has_shared, int* __restrict__ offsets,
                                                                   int* __restrict__ perm, int* __restrict__ inv,
                                                                   int* __restrict__ chunk_base) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ uint32_t sm[];
  __shared__ int warp_sums[kDispatchThreads / 32];
  uint32_t* mask = sm;
  int* base = reinterpret_cast<int*>(sm + kChunkWarps * E);
  const bool first = blockIdx.x == 0;
  write_offsets(counts, T, E, k, has_shared, first ? offsets : nullptr, chunk_base, warp_sums, base);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kChunkTokens) base[e] += chunk_first[static_cast<size_t>(blockIdx.x) * E + e];
  chunk_masks(idx, T, E, k, mask);  // its barriers also publish base[]
  const int t = blockIdx.x * kChunkTokens + threadIdx.x;
  if (t >= T) return;
  const int w = threadIdx.x >> 5;
  const uint32_t below = (1u << (threadIdx.x & 31)) - 1u;
  const int* row = idx + static_cast<size_t>(t) * k;
  for (int j = 0; j < k; ++j) {
    const int e = __ldg(row + j);
    if (e < 0 || e >= E) continue;
    int pos = base[e] + __popc(mask[w * E + e] & below);
    for (int q = 0; q < w; ++q) pos += __popc(mask[q * E + e]);
    const int a = t * k + j;
    if (!MOE_DBG_OK(pos >= 0 && pos < T * k)) continue;
    perm[pos] = a;
    inv[a] = pos;
  }
}

// Rows in dispatch order: xp[inv[t*k + j]] = x[t] for j < k, and with
// with_shared xp[T*k + t] = x[t] too.  One warp per (token, 1024-element
// slice of its row): the slice is read once (16-byte vectors) and written to
// each of the token's rows; with to_f16 each bf16 value is rewritten as the
// nearest fp16.  x is read exactly once, in order.
constexpr int kScatterVec = 4;  // 16-byte vectors per lane and slice
template <bool TO_F16>
__global__ void __launch_bounds__(256) scatter_rows_kernel(const bf16* __restrict__ x, const int* __restrict__ inv,
                                                           int T, int k, int d, int with_shared,
                                                           void* __restrict__ xp) {
  pdl_trigger();
  pdl_wait();
  const int n16 = d / 8;
  const int slices = (n16 + 32 * kScatterVec - 1) / (32 * kScatterVec);
  const long long w = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= static_cast<long long>(T) * slices) return;
  const int t = static_cast<int>(w / slices);
  const int c0 = static_cast<int>(w - static_cast<long long>(t) * slices) * 32 * kScatterVec + lane;
  const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * d);
  uint4 v[kScatterVec];
#pragma unroll
  for (int b = 0; b < kScatterVec; ++b) {
    if (c0 + 32 * b >= n16) continue;
    v[b] = __ldg(src + c0 + 32 * b);
    if (TO_F16) {
      uint32_t* wv = reinterpret_cast<uint32_t*>(&v[b]);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float lo = __uint_as_float(wv[i] << 16), hi = __uint_as_float(wv[i] & 0xffff0000u);
        wv[i] = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(lo))) |
                (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(hi))) << 16);
      }
    }
  }
  const int n_dst = k + (with_shared ? 1 : 0);
  for (int j = 0; j < n_dst; ++j) {
    const int row = (j < k) ? __ldg(inv + static_cast<size_t>(t) * k + j) : T * k + t;
    if (!MOE_DBG_OK(row >= 0 && row < T * k + (with_shared ? T : 0))) continue;
    uint4* dst = static_cast<uint4*>(xp) + static_cast<size_t>(row) * n16;
#pragma unroll
    for (int b = 0; b < kScatterVec; ++b)
      if (c0 + 32 * b < n16) dst[c0 + 32 * b] = v[b];
  }
}

// FP8 token rows as two E4M3 terms (see launch_scatter_x2): one block of 128
// threads per token, a pass for max|x|, then hi / lo of 8 values per thread
// and step, written to each of the token's rows.
__global__ void __launch_bounds__(128) scatter_rows_x2_kernel(const bf16* __restrict__ x,
                                                              const int* __restrict__ inv, int T, int k, int d,
                                                              int with_shared, uint8_t* __restrict__ xq,
                                                              int lo_row0, float* __restrict__ inv_s) {
  pdl_trigger();
  pdl_wait();
  __shared__ float red[4];
  const int t = blockIdx.x;
  const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * d);
  const int n8 = d / 8;
  float amax = 0.f;
  for (int c = threadIdx.x; c < n8; c += 128) {
    const uint4 v = __ldg(src + c);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
      amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w[i] << 16)), fabsf(__uint_as_float(w[i] & 0xffff0000u))));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
  // s = 2^e, the largest power of two with s * amax <= 448 = 1.75 * 2^8
  int e = 0;
  if (amax > 0.f) {
    const uint32_t b = __float_as_uint(amax);
    const int ea = static_cast<int>((b >> 23) & 0xffu) - 127;
    e = ((b & 0x7fffffu) <= 0x600000u ? 8 : 7) - ea;
    e = min(120, max(-120, e));
  }
  const float s = __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
  const int n_dst = k + (with_shared ? 1 : 0);
  for (int j = threadIdx.x; j < n_dst; j += 128) {
    const int pos = (j < k) ? __ldg(inv + static_cast<size_t>(t) * k + j) : T * k + t;
    if (!MOE_DBG_OK(pos >= 0 && pos < T * k + (with_shared ? T : 0))) continue;
    inv_s[pos] = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
  }
  for (int c = threadIdx.x; c < n8; c += 128) {
    const uint4 v = __ldg(src + c);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t hi[2], lo[2];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = make_float2(__uint_as_float(w[i] << 16) * s, __uint_as_float(w[i] & 0xffff0000u) * s);
      const __nv_fp8x2_storage_t h2 = __nv_cvt_float2_to_fp8x2(f, __NV_SATFINITE, __NV_E4M3);
      const float2 hf = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(h2, __NV_E4M3)));
      const __nv_fp8x2_storage_t l2 =
          __nv_cvt_float2_to_fp8x2(make_float2(f.x - hf.x, f.y - hf.y), __NV_SATFINITE, __NV_E4M3);
      const int word = i >> 1;
      if ((i & 1) == 0) {
        hi[word] = h2;
        lo[word] = l2;
      } else {
        hi[word] |= static_cast<uint32_t>(h2) << 16;
        lo[word] |= static_cast<uint32_t>(l2) << 16;
      }
    }
    for (int j = 0; j < n_dst; ++j) {
      const int pos = (j < k) ? __ldg(inv + static_cast<size_t>(t) * k + j) : T * k + t;
      if (!MOE_DBG_OK(pos >= 0 && pos < T * k + (with_shared ? T : 0))) continue;
      reinterpret_cast<uint2*>(xq + static_cast<size_t>(pos) * d)[c] = make_uint2(hi[0], hi[1]);
      reinterpret_cast<uint2*>(xq + static_cast<size_t>(lo_row0 + pos) * d)[c] = make_uint2(lo[0], lo[1]);
    }
  }
}

// H rows in place as two-term E4M3 rows (see launch_requant_rows_x2): one
// block of 128 threads per row; every thread reads its 8-value chunks and the
// row's largest magnitude is reduced before any byte of the row is written.
constexpr int kRequantChunks = 8;  // chunks of 8 values per thread: F <= 8192
__global__ void __launch_bounds__(128) requant_rows_x2_kernel(uint8_t* __restrict__ h, int F,
                                                              float* __restrict__ inv_s) {
  pdl_trigger();
  pdl_wait();
  __shared__ float red[4];
  uint8_t* row = h + static_cast<size_t>(blockIdx.x) * 2 * F;
  const int n8 = F / 8;
  uint4 v[kRequantChunks];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < kRequantChunks; ++i) {
    const int c = threadIdx.x + i * 128;
    if (c < n8) {
      v[i] = reinterpret_cast<const uint4*>(row)[c];
      const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[j]));
        amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
      }
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();  // also: every chunk of the row has been read
  amax = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
  int e = 0;
  if (amax > 0.f) {
    const uint32_t b = __float_as_uint(amax);
    const int ea = static_cast<int>((b >> 23) & 0xffu) - 127;
    e = ((b & 0x7fffffu) <= 0x600000u ? 8 : 7) - ea;
    e = min(120, max(-120, e));
  }
  const float s = __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
  if (threadIdx.x == 0) inv_s[blockIdx.x] = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
#pragma unroll
  for (int i = 0; i < kRequantChunks; ++i) {
    const int c = threadIdx.x + i * 128;
    if (c >= n8) continue;
    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
    uint32_t hi[2], lo[2];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&w[j]));
      const float2 f = make_float2(f0.x * s, f0.y * s);
      const __nv_fp8x2_storage_t h2 = __nv_cvt_float2_to_fp8x2(f, __NV_SATFINITE, __NV_E4M3);
      const float2 hf = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(h2, __NV_E4M3)));
      const __nv_fp8x2_storage_t l2 =
          __nv_cvt_float2_to_fp8x2(make_float2(f.x - hf.x, f.y - hf.y), __NV_SATFINITE, __NV_E4M3);
      const int word = j >> 1;
      if ((j & 1) == 0) {
        hi[word] = h2;
        lo[word] = l2;
      } else {
        hi[word] |= static_cast<uint32_t>(h2) << 16;
        lo[word] |= static_cast<uint32_t>(l2) << 16;
      }
    }
    reinterpret_cast<uint2*>(row)[c] = make_uint2(hi[0], hi[1]);
    reinterpret_cast<uint2*>(row + F)[c] = make_uint2(lo[0], lo[1]);
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
  pdl_trigger();
  const int t = blockIdx.x;
  __shared__ int pos[kMaxTopK + 1];
  __shared__ int chunk[kMaxTopK + 1];
  // the terms' rows: k routed, then the shared expert's when the layer has
  // one (a block can have fewer threads than terms: 32 threads for d = 256
  // against up to 33 terms)
  const int nterms = k + (has_shared ? 1 : 0);
  for (int j = threadIdx.x; j < nterms; j += blockDim.x) {
    int g = (j < k) ? __ldg(idx + static_cast<size_t>(t) * k + j) : E;
    int p = (j < k) ? __ldg(inv + static_cast<size_t>(t) * k + j) : T * k + t;
    if (!MOE_DBG_OK(g >= 0 && g <= E)) g = E;
    int ch = __ldg(chunk_base + g) + (p - __ldg(offsets + g)) / kYpRows;
    // the row inside its group's row block, the chunk inside its group's chunks
    if (!MOE_DBG_OK(p >= __ldg(offsets + g) && p < __ldg(offsets + g + 1) && ch < __ldg(chunk_base + g + 1))) {
      p = T * k + t;
      ch = __ldg(chunk_base + E);
    }
    pos[j] = p;
    chunk[j] = ch;
  }
  __syncthreads();
  pdl_wait();  // the expert outputs from here on (the routing results above are older, as in combine_nt_kernel)
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

// Sign-extended byte b of w.
__device__ __forceinline__ int sbyte(uint32_t w, int b) { return static_cast<int>(w << (24 - 8 * b)) >> 24; }

// acc[i] += h_i * 2^e_i for the 8 fp16 values of raw and their 8 exponents.
__device__ __forceinline__ void accum8(float (&acc)[8], const uint4& raw, const uint2& ex) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t eb = (i < 2) ? ex.x : ex.y;
    const int b = 2 * (i & 1);
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
    acc[2 * i] = fmaf(f.x, pow2i(sbyte(eb, b)), acc[2 * i]);
    acc[2 * i + 1] = fmaf(f.y, pow2i(sbyte(eb, b + 1)), acc[2 * i + 1]);
  }
}

// combine_kernel with the number of terms NT = k (+1 with the shared expert)
// fixed at compile time: the terms' row addresses are worked out once per
// token, and the loads of each half of the terms are in flight together.
// Same arithmetic and order as combine_kernel.
template <int NT>
__global__ void __launch_bounds__(512, 2) combine_nt_kernel(const __half* __restrict__ yp,
                                                            const int8_t* __restrict__ yexp,
                                                            const __half* __restrict__ yp_routed,
                                                            const int8_t* __restrict__ yexp_routed,
                                                            const int* __restrict__ idx, const int* __restrict__ inv,
                                                            const int* __restrict__ offsets,
                                                            const int* __restrict__ chunk_base, int T, int k, int E,
                                                            int d, void* __restrict__ y, int out_fp32) {
  pdl_trigger();
  constexpr int B1 = (NT + 1) / 2;
  const int t = blockIdx.x;
  __shared__ const uint4* rows[NT];
  __shared__ const uint2* exps[NT];
  if (threadIdx.x < NT) {
    const int j = threadIdx.x;
    const bool routed = j < k;
    int g = routed ? __ldg(idx + static_cast<size_t>(t) * k + j) : E;
    int p = routed ? __ldg(inv + static_cast<size_t>(t) * k + j) : T * k + t;
    if (!MOE_DBG_OK(g >= 0 && g <= E)) g = E;
    int ch = __ldg(chunk_base + g) + (p - __ldg(offsets + g)) / kYpRows;
    // the row inside its group's row block, the chunk inside its group's chunks
    if (!MOE_DBG_OK(p >= __ldg(offsets + g) && p < __ldg(offsets + g + 1) && ch < __ldg(chunk_base + g + 1))) {
      p = T * k + t;
      ch = __ldg(chunk_base + E);
    }
    const __half* ybuf = (routed && yp_routed) ? yp_routed : yp;
    const int8_t* ebuf = (routed && yp_routed) ? yexp_routed : yexp;
    rows[j] = reinterpret_cast<const uint4*>(ybuf + static_cast<size_t>(p) * d);
    exps[j] = reinterpret_cast<const uint2*>(ebuf + static_cast<size_t>(ch) * d);
  }
  __syncthreads();
  // Only now the expert outputs.  The routing and dispatch results read
  // above are older: the kernel before this one (the down GEMM) starts its
  // dependents only at its end, after its own wait for the gate/up, which
  // waited for the kernels that wrote them.
  pdl_wait();
  for (int c = threadIdx.x; c < d / 8; c += blockDim.x) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    {
      uint4 raw[B1];
      uint2 ex[B1];
#pragma unroll
      for (int j = 0; j < B1; ++j) {
        raw[j] = __ldcs(rows[j] + c);
        ex[j] = __ldg(exps[j] + c);
      }
#pragma unroll
      for (int j = 0; j < B1; ++j) accum8(acc, raw[j], ex[j]);
    }
    if (NT > B1) {
      uint4 raw[NT - B1 > 0 ? NT - B1 : 1];
      uint2 ex[NT - B1 > 0 ? NT - B1 : 1];
#pragma unroll
      for (int j = B1; j < NT; ++j) {
        raw[j - B1] = __ldcs(rows[j] + c);
        ex[j - B1] = __ldg(exps[j] + c);
      }
#pragma unroll
      for (int j = B1; j < NT; ++j) accum8(acc, raw[j - B1], ex[j - B1]);
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

MOE_DBG_DEFINE_TAKE(dbg_take_dispatch)

bool pdl_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("MOE_PDL");
    return !(v != nullptr && v[0] == '0');
  }();
  return on;
}

bool chunked_dispatch(int T) { return T >= kChunkedDispatchMinTokens; }

size_t chunk_hist_ints(int T, int E) { return static_cast<size_t>((T + kChunkTokens - 1) / kChunkTokens) * E; }

cudaError_t launch_chunk_counts(const int* idx, int T, int E, int k, int* hist, int* counts, cudaStream_t stream) {
  if (T <= 0) return cudaSuccess;
  const int n_chunks = (T + kChunkTokens - 1) / kChunkTokens;
  const cudaError_t e = launch_chain(chunk_hist_kernel, dim3(n_chunks), dim3(kChunkTokens),
                                     sizeof(uint32_t) * kChunkWarps * E, stream, idx, T, E, k, hist);
  if (e != cudaSuccess) return e;
  return launch_chain(chunk_scan_kernel, dim3((E + 31) / 32), dim3(32 * kScanParts), 0, stream, hist, n_chunks, E,
                      counts);
}

cudaError_t launch_dispatch(const int* idx, const int* counts, int T, int E, int k, int has_shared, int* offsets,
                            int* perm, int* inv, int* chunk_base, const int* chunk_first, cudaStream_t stream) {
  if (chunk_first != nullptr && chunked_dispatch(T)) {
    const int n_chunks = (T + kChunkTokens - 1) / kChunkTokens;
    return launch_chain(chunk_place_kernel, dim3(n_chunks), dim3(kChunkTokens),
                        sizeof(uint32_t) * (kChunkWarps + 1) * E, stream, idx, counts, chunk_first, T, E, k,
                        has_shared, offsets, perm, inv, chunk_base);
  }
  return launch_chain(dispatch_kernel, dim3(E), dim3(kDispatchThreads), 0, stream, idx, counts, T, E, k, has_shared,
                      offsets, perm, inv, chunk_base);
}

cudaError_t launch_gather(const bf16* x, const int* inv, int T, int k, int d, int has_shared, void* xp,
                          bool to_f16, cudaStream_t stream) {
  if (T <= 0) return cudaSuccess;
  const int n16 = d / 8;
  const long long warps = static_cast<long long>(T) * ((n16 + 32 * kScatterVec - 1) / (32 * kScatterVec));
  const long long blocks = (warps + 7) / 8;
  if (blocks > 0x7fffffffll) return cudaErrorInvalidValue;
  return launch_chain(to_f16 ? scatter_rows_kernel<true> : scatter_rows_kernel<false>,
                      dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, x, inv, T, k, d, has_shared, xp);
}

cudaError_t launch_scatter_x2(const bf16* x, const int* inv, int T, int k, int d, int has_shared, uint8_t* xq,
                              int lo_row0, float* inv_s, cudaStream_t stream) {
  if (T <= 0) return cudaSuccess;
  return launch_chain(scatter_rows_x2_kernel, dim3(T), dim3(128), 0, stream, x, inv, T, k, d, has_shared, xq,
                      lo_row0, inv_s);
}

cudaError_t launch_requant_rows_x2(void* h, int rows, int F, float* inv_s, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  if (F % 8 != 0 || F / 8 > 128 * kRequantChunks) return cudaErrorInvalidValue;
  return launch_chain(requant_rows_x2_kernel, dim3(rows), dim3(128), 0, stream, static_cast<uint8_t*>(h), F, inv_s);
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
  pdl_trigger();
  pdl_wait();
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
  pdl_trigger();
  pdl_wait();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) w[i] = prob[perm[i]];
}

__global__ void iota_kernel(int* __restrict__ v, int n) {
  pdl_trigger();
  pdl_wait();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) v[i] = i;
}

cudaError_t launch_ep_groups(const int* recv_counts, int S, int E_loc, int* offsets, int* chunk_base,
                             int* chunks_per_source, cudaStream_t stream) {
  return launch_chain(ep_groups_kernel, dim3(1), dim3(32), 0, stream, recv_counts, S, E_loc, offsets, chunk_base,
                      chunks_per_source);
}

cudaError_t launch_gather_weights(const int* perm, const float* prob, int n, float* w, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  return launch_chain(gather_weights_kernel, dim3((n + 255) / 256), dim3(256), 0, stream, perm, prob, n, w);
}

cudaError_t launch_iota(int* v, int n, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  return launch_chain(iota_kernel, dim3((n + 255) / 256), dim3(256), 0, stream, v, n);
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
  const int nterms = k + (has_shared ? 1 : 0);
  if (chunks <= 512 && (nterms == 9 || nterms == 8)) {
    const int threads = chunks < 32 ? 32 : chunks;
    return launch_chain(nterms == 9 ? combine_nt_kernel<9> : combine_nt_kernel<8>, dim3(T), dim3(threads), 0, stream,
                        yp, yexp, yp_routed, yexp_routed, idx, inv, offsets, chunk_base, T, k, E, d, y, out_fp32);
  }
  const int threads = chunks > 1024 ? 1024 : (chunks < 32 ? 32 : chunks);
  return launch_chain(combine_kernel, dim3(T), dim3(threads), 0, stream, yp, yexp, yp_routed, yexp_routed, idx, inv,
                      offsets, chunk_base, T, k, E, d, has_shared, y, out_fp32);
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
  if (cudaMemsetAsync(counts, 0, sizeof(int) * n_experts, s) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
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
