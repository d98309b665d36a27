// K1 on the tensor cores — the router of "Step3.5 Flash 大模型技术深度解析"
// (jsqmd.com) §3.2.2: one logit per routed expert from a linear layer, then a
// softmax over all experts and the k most probable ones.
//
// The logit GEMM z = x . W_r^T keeps fp32 accuracy on bf16 tensor cores: W_r
// (fp32) is held as three bf16 slices hi + mid + lo (together 24 significand
// bits, the fp32 significand), x is bf16 already, so each product x_i * slice
// is exact in fp32 and z = x.hi + x.mid + x.lo is accumulated in fp32 by
// tcgen05.mma over an effective K of 3d.  The expert rows are the MMA's M
// operand (128 per tile) and token rows its N operand, as in the expert GEMMs.
// K is split across CTAs when there are few token tiles (decode); each split
// writes its partial logits and the top-k kernel sums the splits in a fixed
// order, so results are identical run to run.
//
// Top-k: below 1024 tokens one block of four warps per token sums the K
// splits, from 1024 tokens on one warp per token does; one warp then does
// softmax and top-k with xor-shuffle butterflies (every lane ends with the same
// bits); ties go to the lower expert index.
#include "kernels.cuh"
#include "ptx.cuh"
#include "topk.cuh"

#include <algorithm>
#include <cfloat>

namespace moe {
namespace {

constexpr int kThreads = 192;
constexpr uint64_t kDrainLimitNs = 2000000000ull;
constexpr long long kPrefetchChunk = 64 * 1024;  // bytes per L2 prefetch instruction

// Two rings: token tiles (x, BN rows x 64 columns) and weight tiles (one
// 128-row slice tile each).  Every K step loads one x tile and the three
// slices' tiles of the same columns, and the three MMAs of the step read the
// one x tile: x crosses from L2 into shared memory once per K step instead of
// once per slice.
template <int BN>
struct RCfg {
  static constexpr int W_BYTES = kBlockM * kBlockK * 2;  // one slice tile
  static constexpr int X_BYTES = BN * kBlockK * 2;       // one token tile
  static constexpr int WS = 6;                           // two K steps of three slices
  static constexpr int XS_RAW = (200 * 1024 - WS * W_BYTES) / X_BYTES;
  static constexpr int XS = XS_RAW > 8 ? 8 : XS_RAW;
  static constexpr int NACC = (2 * BN <= 512) ? 2 : 1;
  static constexpr int TMEM_RAW = NACC * BN;
  static constexpr int TMEM_COLS = TMEM_RAW <= 32 ? 32 : TMEM_RAW <= 64 ? 64 : TMEM_RAW <= 128 ? 128
                                                                       : TMEM_RAW <= 256 ? 256 : 512;
  static constexpr int NUM_BARS = 2 * WS + 2 * XS + 2 * NACC + 1;
  static constexpr int SMEM_BYTES = 1024 + WS * W_BYTES + XS * X_BYTES + NUM_BARS * 8 + 16;
  static_assert(XS >= 2, "token ring too shallow");
  static_assert(SMEM_BYTES <= 232448, "exceeds shared memory per block");
  static constexpr uint32_t IDESC = idesc_bf16_f32(kBlockM, BN);
};

struct RItem {
  int tt, m, ks;
};

__device__ __forceinline__ RItem decode_ritem(int item, int m_tiles, int ksplit) {
  RItem it;
  it.ks = item % ksplit;
  const int r = item / ksplit;
  it.m = r % m_tiles;
  it.tt = r / m_tiles;
  return it;
}

__device__ __forceinline__ bool rwait(uint64_t* bar, uint32_t parity, uint64_t limit_ns, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t spins = 0;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((++spins & 15u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > limit_ns) return false;
    }
  }
}

template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    router_gemm_kernel(const __grid_constant__ CUtensorMap map_w3, const __grid_constant__ CUtensorMap map_x,
                       const RouterGemmArgs args) {
  using C = RCfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* wring = smem;
  uint8_t* xring = smem + C::WS * C::W_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(xring + C::XS * C::X_BYTES);
  uint64_t* w_full = bars;
  uint64_t* w_empty = bars + C::WS;
  uint64_t* x_full = bars + 2 * C::WS;
  uint64_t* x_empty = x_full + C::XS;
  uint64_t* acc_full = x_empty + C::XS;
  uint64_t* acc_empty = acc_full + C::NACC;
  uint64_t* drain = acc_empty + C::NACC;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + C::NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tt = (args.T + BN - 1) / BN;
  const int n_items = n_tt * args.m_tiles * args.ksplit;
  const int kd = args.d / kBlockK;                       // K steps (each with the three slices)
  const int k_per = (kd + args.ksplit - 1) / args.ksplit;  // K steps per split

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::WS; ++s) {
      mbar_init(&w_full[s], 1);
      mbar_init(&w_empty[s], 1);
    }
    for (int s = 0; s < C::XS; ++s) {
      mbar_init(&x_full[s], 1);
      mbar_init(&x_empty[s], 1);
    }
    for (int a = 0; a < C::NACC; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&map_w3);
    tma_prefetch_desc(&map_x);
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, C::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 2 && lane == 0) {
    // the shared expert's weights into L2 (chunks of kPrefetchChunk bytes,
    // CTA b taking chunks b, b + gridDim.x, ...); constant inputs, so no
    // wait on earlier work
    for (int r = 0; r < 2; ++r) {
      const char* base = static_cast<const char*>(args.pf[r]);
      const long long n = args.pf_bytes[r];
      for (long long o = static_cast<long long>(blockIdx.x) * kPrefetchChunk; o < n;
           o += static_cast<long long>(gridDim.x) * kPrefetchChunk)
        l2_prefetch_bulk(base + o, static_cast<uint32_t>(n - o < kPrefetchChunk ? n - o : kPrefetchChunk));
    }
  }
  pdl_wait();  // x and the partial-logit buffer belong to earlier work in the stream until here
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const uint64_t limit = args.wait_limit_ns;

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol = policy_evict_last();  // W slices and x are re-read by other CTAs
      uint32_t ws = 0, wph = 0, xs = 0, xph = 0;
      long w_issued = 0, x_issued = 0;
      bool ok = true;
      for (int item = blockIdx.x; ok && item < n_items && !*abort_flag; item += gridDim.x) {
        const RItem it = decode_ritem(item, args.m_tiles, args.ksplit);
        const int kb0 = it.ks * k_per, kb1 = min(kd, kb0 + k_per);
        for (int kb = kb0; ok && kb < kb1; ++kb) {
          const int kc = kb * kBlockK;
          if (!rwait(&x_empty[xs], xph ^ 1u, limit, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&x_full[xs], C::X_BYTES);
          tma_load_2d(xring + xs * C::X_BYTES, &map_x, &x_full[xs], kc, it.tt * BN, pol);
          ++x_issued;
          if (++xs == C::XS) {
            xs = 0;
            xph ^= 1u;
          }
          for (int slice = 0; slice < 3; ++slice) {
            if (!rwait(&w_empty[ws], wph ^ 1u, limit, abort_flag)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&w_full[ws], C::W_BYTES);
            tma_load_2d(wring + ws * C::W_BYTES, &map_w3, &w_full[ws], kc, slice * args.e_pad + it.m * kBlockM, pol);
            ++w_issued;
            if (++ws == C::WS) {
              ws = 0;
              wph ^= 1u;
            }
          }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(args.err, kErrWaitTimeout);
      }
      // every load issued must have landed before the CTA may exit
      for (int s = 0; s < C::WS; ++s) {
        if (w_issued <= s) break;
        const long last = s + ((w_issued - 1 - s) / C::WS) * C::WS;
        mbar_wait(&w_full[s], static_cast<uint32_t>((last / C::WS) & 1), kDrainLimitNs);
      }
      for (int s = 0; s < C::XS; ++s) {
        if (x_issued <= s) break;
        const long last = s + ((x_issued - 1 - s) / C::XS) * C::XS;
        mbar_wait(&x_full[s], static_cast<uint32_t>((last / C::XS) & 1), kDrainLimitNs);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      uint32_t ws = 0, wph = 0, xs = 0, xph = 0, acc = 0, acc_phase = 0;
      bool issued_any = false, ok = true;
      for (int item = blockIdx.x; ok && item < n_items && !*abort_flag; item += gridDim.x) {
        const RItem it = decode_ritem(item, args.m_tiles, args.ksplit);
        const int kb0 = it.ks * k_per, kb1 = min(kd, kb0 + k_per);
        if (!rwait(&acc_empty[acc], acc_phase ^ 1u, limit, abort_flag)) {
          *abort_flag = 1;
          atomicOr(args.err, kErrWaitTimeout);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = kb0; ok && kb < kb1; ++kb) {
          if (!rwait(&x_full[xs], xph, limit, abort_flag)) {
            ok = false;
            break;
          }
          const uint64_t b = smem_desc_sw128(smem_u32(xring + xs * C::X_BYTES));
          for (int slice = 0; slice < 3; ++slice) {
            if (!rwait(&w_full[ws], wph, limit, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t a = smem_desc_sw128(smem_u32(wring + ws * C::W_BYTES));
#pragma unroll
            for (int kk = 0; kk < kBlockK / 16; ++kk)
              tc_mma_bf16(d_tmem, a + 2 * kk, b + 2 * kk, C::IDESC, (kb > kb0 || slice > 0 || kk > 0) ? 1u : 0u);
            issued_any = true;
            tc_commit(&w_empty[ws]);
            if (++ws == C::WS) {
              ws = 0;
              wph ^= 1u;
            }
          }
          if (!ok) break;
          tc_commit(&x_empty[xs]);  // after the three slices' MMAs that read it
          if (++xs == C::XS) {
            xs = 0;
            xph ^= 1u;
          }
        }
        if (!ok) {
          *abort_flag = 1;
          atomicOr(args.err, kErrWaitTimeout);
          break;
        }
        tc_commit(&acc_full[acc]);
        if (++acc == C::NACC) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (issued_any) {
        tc_commit(drain);
        mbar_wait(drain, 0, kDrainLimitNs);
      }
    }
  } else {
    const int q = warp & 3;
    const int e = q * 32 + lane;  // expert row within the m tile
    uint32_t acc = 0, acc_phase = 0;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
      const RItem it = decode_ritem(item, args.m_tiles, args.ksplit);
      const int t0 = it.tt * BN;
      const int valid = min(BN, args.T - t0);
      const int expert = it.m * kBlockM + e;
      if (!__all_sync(0xffffffffu, rwait(&acc_full[acc], acc_phase, limit, abort_flag))) {
        if (lane == 0) {
          *abort_flag = 1;
          atomicOr(args.err, kErrWaitTimeout);
        }
        break;
      }
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
      float* part = args.partial + static_cast<size_t>(it.ks) * args.T * args.E;
#pragma unroll
      for (int c0 = 0; c0 < BN; c0 += 16) {
        if (c0 >= valid) break;
        uint32_t v[16];
        tmem_ld16(taddr + c0, v);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 16; ++c)
          if (c0 + c < valid && expert < args.E)
            part[static_cast<size_t>(t0 + c0 + c) * args.E + expert] = __uint_as_float(v[c]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[acc]);
      if (++acc == C::NACC) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  // dependents launch as this grid ends (past the barrier every role has
  // finished): their blocks would otherwise wait on these SMs for the whole
  // run of this persistent kernel
  pdl_trigger();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

constexpr int kTopkWarps = 4;
constexpr int kTopkWarpMinTokens = 1024;  // from this many tokens on: one warp per token


// Few tokens (decode): one block of 4 warps per token.  Warp w sums the K-split
// partials s = w, w+4, ... in increasing s; warp 0 then adds the four partial
// sums in warp order (a fixed order: logits are bit-identical run to run) and
// finishes the token alone.
template <int NS>
__global__ void __launch_bounds__(kTopkWarps * 32) router_topk_kernel(const float* __restrict__ partial, int ksplit,
                                                                      int T, int E, int k, int renorm,
                                                                      int* __restrict__ idx,
                                                                      float* __restrict__ prob,
                                                                      float* __restrict__ gap, int* counts,
                                                                      float* __restrict__ tokstats, int n_groups) {
  pdl_trigger();
  pdl_wait();
  __shared__ float zs[kTopkWarps][32 * NS];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int t = blockIdx.x;
  float p[NS];
#pragma unroll
  for (int i = 0; i < NS; ++i) p[i] = 0.f;
  // this warp's splits in batches of six whose loads are in flight together
  // (one memory latency per batch), added in increasing s
  constexpr int kBatch = 6;
  for (int s0 = warp; s0 < ksplit; s0 += kBatch * kTopkWarps) {
    float v[kBatch][NS];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int s = s0 + u * kTopkWarps;
      const float* row = partial + (static_cast<size_t>(s) * T + t) * E;
#pragma unroll
      for (int i = 0; i < NS; ++i) {
        const int e = lane + 32 * i;
        v[u][i] = (s < ksplit && e < E) ? __ldg(row + e) : 0.f;
      }
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u)
#pragma unroll
      for (int i = 0; i < NS; ++i)
        if (s0 + u * kTopkWarps < ksplit) p[i] += v[u][i];
  }
#pragma unroll
  for (int i = 0; i < NS; ++i) zs[warp][lane + 32 * i] = p[i];
  __syncthreads();
  if (warp != 0) return;
#pragma unroll
  for (int i = 0; i < NS; ++i) {
    const int e = lane + 32 * i;
    p[i] = ((zs[0][e] + zs[1][e]) + zs[2][e]) + zs[3][e];
  }
  finish_token<NS>(p, t, lane, E, k, renorm, idx, prob, gap, counts, tokstats, n_groups);
}

// Many tokens (prefill): one warp per token, kTopkTokensPerBlock tokens per
// block; the warp sums the K-split partials in increasing s and finishes the
// token, so no warp waits on another.
constexpr int kTopkTokensPerBlock = 8;
template <int NS>
__global__ void __launch_bounds__(kTopkTokensPerBlock * 32) router_topk_warp_kernel(
    const float* __restrict__ partial, int ksplit, int T, int E, int k, int renorm, int* __restrict__ idx,
    float* __restrict__ prob, float* __restrict__ gap, int* counts, float* __restrict__ tokstats, int n_groups) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kTopkTokensPerBlock + (threadIdx.x >> 5);
  if (t >= T) return;
  float p[NS];
#pragma unroll
  for (int i = 0; i < NS; ++i) p[i] = 0.f;
  // the splits in batches of four whose loads are in flight together, added
  // in increasing s
  constexpr int kBatch = 4;
  for (int s0 = 0; s0 < ksplit; s0 += kBatch) {
    float v[kBatch][NS];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const float* row = partial + (static_cast<size_t>(s0 + u) * T + t) * E;
#pragma unroll
      for (int i = 0; i < NS; ++i) {
        const int e = lane + 32 * i;
        v[u][i] = (s0 + u < ksplit && e < E) ? __ldg(row + e) : 0.f;
      }
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u)
#pragma unroll
      for (int i = 0; i < NS; ++i)
        if (s0 + u < ksplit) p[i] += v[u][i];
  }
  finish_token<NS>(p, t, lane, E, k, renorm, idx, prob, gap, counts, tokstats, n_groups);
}

// A few tokens (decode of one to kSmallRouteMaxTokens tokens): the router,
// softmax / top-k and the dispatch in one launch.  The logit GEMM is T small
// dot products per expert, bounded by reading W_r (fp32, 4.7 MB at the flash
// shape) once: block e computes expert e for every token with fp32 FMAs,
// warp w over the w-th quarter of the columns (lane l takes the float4
// columns l, l + 32, ... of it in increasing order, their loads in flight
// together), the lanes' sums meet in a fixed xor-butterfly and the four
// warps' sums are added in warp order.  The block that finishes last (an
// integer arrival count, reset for the next launch) ranks every token with
// finish_token and lays the rows out: counts, offsets and chunk bases as
// counts over the T*k picks, and each assignment a = t*k + j at offsets[e] +
// the number of earlier tokens that chose e (the stable expert, token order
// of dispatch_kernel).  With one token its k rows are copies of it whatever
// the experts, so blocks 0..k-1 copy them beside their dot products; with
// two the last block copies them.  Every result is a function of x and W_r
// alone (fixed summation orders): bit-identical run to run.  With
// ex.logits_only the blocks stop at their logits (no count, no last block):
// the gate/up launch after this one ranks the tokens itself.
constexpr int kSmallRouteWarps = 4;

template <int NS>
__global__ void __launch_bounds__(kSmallRouteWarps * 32) route_small_kernel(
    const bf16* __restrict__ x, const float* __restrict__ w_router, int T, int d, int E, int k, int renorm,
    int has_shared, float* __restrict__ logits, unsigned int* done, int* __restrict__ idx, float* __restrict__ prob,
    float* __restrict__ gap, int* __restrict__ counts, int* __restrict__ offsets, int* __restrict__ perm,
    int* __restrict__ inv, int* __restrict__ chunk_base, SmallRouteExtras ex) {
  pdl_trigger();
  __shared__ int s_last;
  __shared__ float s_part[kSmallRouteWarps][kSmallRouteMaxTokens];
  __shared__ int s_idx[kSmallRouteMaxTokens * kMaxTopK], s_first[kSmallRouteMaxTokens * kMaxTopK],
      s_pos[kSmallRouteMaxTokens * kMaxTopK];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  pdl_wait();  // x, and the routing buffers read by earlier work in the stream
  const int e = blockIdx.x;
  {
    float acc[kSmallRouteMaxTokens];
#pragma unroll
    for (int t = 0; t < kSmallRouteMaxTokens; ++t) acc[t] = 0.f;
    const int q4 = d / 16;  // float4 columns of a quarter
    const float4* wr = reinterpret_cast<const float4*>(w_router + static_cast<size_t>(e) * d) + warp * q4;
#pragma unroll 8
    for (int c = lane; c < q4; c += 32) {
      const float4 w = __ldg(wr + c);
#pragma unroll
      for (int t = 0; t < kSmallRouteMaxTokens; ++t) {
        if (t < T) {
          const uint2 xv = __ldg(reinterpret_cast<const uint2*>(x + static_cast<size_t>(t) * d) + warp * q4 + c);
          acc[t] = fmaf(__uint_as_float(xv.x << 16), w.x, acc[t]);
          acc[t] = fmaf(__uint_as_float(xv.x & 0xffff0000u), w.y, acc[t]);
          acc[t] = fmaf(__uint_as_float(xv.y << 16), w.z, acc[t]);
          acc[t] = fmaf(__uint_as_float(xv.y & 0xffff0000u), w.w, acc[t]);
        }
      }
    }
#pragma unroll
    for (int t = 0; t < kSmallRouteMaxTokens; ++t) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], off);
      if (lane == 0) s_part[warp][t] = acc[t];
    }
  }
  // One token: its k routed rows are k copies of it at dispatch positions
  // 0..k-1 whatever the experts, so blocks 0..k-1 copy them now
  if (ex.xp != nullptr && !ex.logits_only && T == 1 && e < k) {
    const uint4* src = reinterpret_cast<const uint4*>(x);
    uint4* dst = reinterpret_cast<uint4*>(static_cast<bf16*>(ex.xp) + static_cast<size_t>(e) * d);
    for (int c = threadIdx.x; c < d / 8; c += blockDim.x) dst[c] = __ldg(src + c);
  }
  // Logits only: the gate/up launch reads every group's token tile from one
  // of ex.replicas copies of the T rows (rows r*T .. r*T + T-1 of xp, CTA c
  // reading copy c mod replicas), so its CTAs do not all load the same few
  // lines; block r < replicas writes copy r
  if (ex.xp != nullptr && ex.logits_only && e < ex.replicas) {
    const uint4* src = reinterpret_cast<const uint4*>(x);
    uint4* dst = reinterpret_cast<uint4*>(static_cast<bf16*>(ex.xp) + static_cast<size_t>(e) * T * d);
    for (int c = threadIdx.x; c < T * d / 8; c += blockDim.x) dst[c] = __ldg(src + c);
  }
  __syncthreads();
  if (threadIdx.x < T)
    logits[static_cast<size_t>(threadIdx.x) * E + e] =
        ((s_part[0][threadIdx.x] + s_part[1][threadIdx.x]) + s_part[2][threadIdx.x]) + s_part[3][threadIdx.x];
  // weights every call reads whatever the routing (the shared expert's),
  // into L2 while the routing finishes — after this block's loads of W_r,
  // which they would otherwise delay: chunks of kPrefetchChunk bytes, block
  // b taking chunks b, b + gridDim.x, ...
  auto prefetch_shared = [&] {
    for (int r = 0; r < 2; ++r) {
      const char* base = static_cast<const char*>(r == 0 ? ex.pf0 : ex.pf1);
      const long long n = r == 0 ? ex.pf0_bytes : ex.pf1_bytes;
      for (long long o = static_cast<long long>(blockIdx.x) * kPrefetchChunk; o < n;
           o += static_cast<long long>(gridDim.x) * kPrefetchChunk)
        l2_prefetch_bulk(base + o, static_cast<uint32_t>(n - o < kPrefetchChunk ? n - o : kPrefetchChunk));
    }
  };
  if (ex.logits_only) {  // the gate/up launch after this one ranks the tokens
    if (threadIdx.x == 0) prefetch_shared();
    return;
  }
  // the block that finishes last sees every logit (the barrier orders this
  // block's logit stores before thread 0's release fence and count)
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const bool last = atomicAdd(done, 1u) == gridDim.x - 1;
    if (last) __threadfence();  // acquire: every block's logits are visible
    s_last = last;
    prefetch_shared();
  }
  __syncthreads();
  if (!s_last) return;
  for (int t = warp; t < T; t += kSmallRouteWarps) {
    float q[NS];
#pragma unroll
    for (int i = 0; i < NS; ++i) {
      const int ee = lane + 32 * i;
      q[i] = ee < E ? __ldcg(logits + static_cast<size_t>(t) * E + ee) : 0.f;
    }
    finish_token<NS>(q, t, lane, E, k, renorm, idx, prob, gap, nullptr, nullptr, 0, s_idx);
  }
  // The dispatch of the T * k picks.  With T <= kSmallRouteMaxTokens < 16
  // rows an expert's group takes exactly one exponent chunk when it has rows,
  // so every value is a count over the picks: offsets[e] = picks of experts
  // below e, chunk_base[e] = experts below e with a pick, and pick a = t*k + j
  // goes to offsets[e] + the earlier picks of its expert (the expert, token
  // order of dispatch_kernel; a token picks an expert at most once).
  static_assert(kSmallRouteMaxTokens < kYpRows, "one exponent chunk per group");
  const int Tk = T * k;
  __syncthreads();  // every pick in s_idx
  for (int a = threadIdx.x; a < Tk; a += blockDim.x) {
    const int e2 = s_idx[a];
    int first = 1;
    for (int a2 = 0; a2 < a; ++a2) first &= s_idx[a2] != e2;
    s_first[a] = first;
  }
  __syncthreads();
  for (int e2 = threadIdx.x; e2 < E; e2 += blockDim.x) {
    int below = 0, cnt = 0, groups = 0;
    for (int a = 0; a < Tk; ++a) {
      const int v = s_idx[a];
      below += v < e2;
      cnt += v == e2;
      groups += (v < e2) & s_first[a];
    }
    offsets[e2] = below;
    counts[e2] = cnt;
    chunk_base[e2] = groups;
  }
  if (threadIdx.x == 0) {
    offsets[E] = Tk;
    offsets[E + 1] = Tk + (has_shared ? T : 0);
    chunk_base[E] = shared_chunk0(T, k, E);  // the routed chunks end at <= Tk <= this
    chunk_base[E + 1] = chunk_base[E] + (has_shared ? (T + kYpRows - 1) / kYpRows : 0);
  }
  for (int a = threadIdx.x; a < Tk; a += blockDim.x) {
    const int e2 = s_idx[a];
    int pos = 0;
    for (int a2 = 0; a2 < Tk; ++a2) pos += (s_idx[a2] < e2) | ((a2 < a) & (s_idx[a2] == e2));
    perm[pos] = a;
    inv[a] = pos;
    s_pos[a] = pos;  // the positions of the row copy below
  }
  if (threadIdx.x == 0) *done = 0u;  // ready for the next launch
  if (ex.xp == nullptr || T == 1) return;
  // the routed rows in dispatch order, xp[pos(a)] = x[a / k], by this block:
  // each thread loads kGatherVecs 16-byte vectors of every token's row at
  // once, then stores each to the token's k positions
  __syncthreads();
  constexpr int kGatherVecs = 4;
  const int n16 = d / 8;
  const uint4* xv = reinterpret_cast<const uint4*>(x);
  uint4* xpv = reinterpret_cast<uint4*>(ex.xp);
  for (int c0 = threadIdx.x; c0 < n16; c0 += kGatherVecs * blockDim.x) {
    uint4 v[kGatherVecs][kSmallRouteMaxTokens];
#pragma unroll
    for (int u = 0; u < kGatherVecs; ++u) {
      const int c = c0 + u * blockDim.x;
#pragma unroll
      for (int t = 0; t < kSmallRouteMaxTokens; ++t)
        if (t < T && c < n16) v[u][t] = __ldg(xv + static_cast<size_t>(t) * n16 + c);
    }
#pragma unroll
    for (int u = 0; u < kGatherVecs; ++u) {
      const int c = c0 + u * blockDim.x;
      if (c >= n16) break;
#pragma unroll
      for (int t = 0; t < kSmallRouteMaxTokens; ++t) {
        if (t >= T) break;
        for (int j = 0; j < k; ++j) xpv[static_cast<size_t>(s_pos[t * k + j]) * n16 + c] = v[u][t];
      }
    }
  }
}

template <int NS>
cudaError_t launch_route_small_ns(const bf16* x, const float* w_router, int T, int d, int E, int k, int renorm,
                                  int has_shared, float* logits, unsigned int* done, int* idx, float* prob,
                                  float* gap, int* counts, int* offsets, int* perm, int* inv, int* chunk_base,
                                  const SmallRouteExtras& ex, cudaStream_t stream) {
  return launch_chain(route_small_kernel<NS>, dim3(E), dim3(kSmallRouteWarps * 32), 0, stream, x, w_router, T, d, E,
                      k, renorm, has_shared, logits, done, idx, prob, gap, counts, offsets, perm, inv, chunk_base, ex);
}

template <int NS>
cudaError_t launch_topk_ns(const float* partial, int ksplit, int T, int E, int k, int renorm, int* idx, float* prob,
                           float* gap, int* counts, float* tokstats, int n_groups, cudaStream_t stream) {
  if (T >= kTopkWarpMinTokens) {
    const int blocks = (T + kTopkTokensPerBlock - 1) / kTopkTokensPerBlock;
    return launch_chain(router_topk_warp_kernel<NS>, dim3(blocks), dim3(kTopkTokensPerBlock * 32), 0, stream,
                        partial, ksplit, T, E, k, renorm, idx, prob, gap, counts, tokstats, n_groups);
  } else {
    return launch_chain(router_topk_kernel<NS>, dim3(T), dim3(kTopkWarps * 32), 0, stream, partial, ksplit, T, E, k,
                        renorm, idx, prob, gap, counts, tokstats, n_groups);
  }
}

// Routing statistics over the tokens: group_p[g] = mean over tokens of the
// group's probability mass, summary[2] = mean entropy (both summed in token
// order per thread, then a fixed tree: bit-identical run to run);
// group_f[g] = share of the T*k rows in group g, summary[0] = L_EP =
// n_groups * sum_g f_g p_g, summary[1] = max/mean rows per expert,
// summary[3] = experts without rows.  One block of 256 threads.
__global__ void __launch_bounds__(256) route_stats_kernel(const float* __restrict__ tokstats, const int* counts,
                                                          int T, int E, int k, int n_groups, float* group_f,
                                                          float* group_p, float* summary) {
  pdl_trigger();
  pdl_wait();
  __shared__ float red[256];
  __shared__ float col_sum[kMaxStatGroups + 1];
  const int cols = n_groups + 1;
  for (int c = 0; c < cols; ++c) {
    float acc = 0.f;
    for (int t = threadIdx.x; t < T; t += 256) acc += tokstats[static_cast<size_t>(t) * cols + c];
    red[threadIdx.x] = acc;
    __syncthreads();
    for (int w = 128; w > 0; w >>= 1) {
      if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
      __syncthreads();
    }
    if (threadIdx.x == 0) col_sum[c] = red[0];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const int per_group = E / n_groups;
    const float rows = static_cast<float>(T) * k;
    float lep = 0.f;
    int max_c = 0, empty = 0;
    for (int e = 0; e < E; ++e) {
      max_c = max(max_c, counts[e]);
      empty += counts[e] == 0;
    }
    for (int g = 0; g < n_groups; ++g) {
      int cg = 0;
      for (int e = g * per_group; e < (g + 1) * per_group; ++e) cg += counts[e];
      const float f = T > 0 ? cg / rows : 0.f;
      const float pg = T > 0 ? col_sum[g] / T : 0.f;
      group_f[g] = f;
      group_p[g] = pg;
      lep += f * pg;
    }
    summary[0] = n_groups * lep;
    summary[1] = T > 0 ? max_c / (rows / E) : 0.f;
    summary[2] = T > 0 ? col_sum[n_groups] / T : 0.f;
    summary[3] = static_cast<float>(empty);
  }
}

// W_r fp32 [E][d] -> three bf16 slices [3][e_pad][d]: hi = rn(w), mid = rn(w - hi),
// lo = rn(w - hi - mid); rows E..e_pad-1 are zero.
__global__ void split_router_kernel(const float* __restrict__ w, int E, int d, int e_pad, bf16* __restrict__ w3) {
  const size_t n = static_cast<size_t>(e_pad) * d;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t row = i / d;
    const float v = row < static_cast<size_t>(E) ? w[i] : 0.f;
    const bf16 hi = __float2bfloat16_rn(v);
    const float r1 = v - __bfloat162float(hi);
    const bf16 mid = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(mid);
    w3[i] = hi;
    w3[n + i] = mid;
    w3[2 * n + i] = __float2bfloat16_rn(r2);
  }
}

template <int BN>
cudaError_t launch_rg(const CUtensorMap* map_w3, const CUtensorMap* map_x, const RouterGemmArgs& a, int grid,
                      cudaStream_t stream) {
  return launch_chain(router_gemm_kernel<BN>, dim3(grid), dim3(kThreads), RCfg<BN>::SMEM_BYTES, stream, *map_w3,
                      *map_x, a);
}

}  // namespace

cudaError_t router_gemm_prepare() {
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(router_gemm_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                RCfg<16>::SMEM_BYTES)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(router_gemm_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                RCfg<64>::SMEM_BYTES)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(router_gemm_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                RCfg<128>::SMEM_BYTES)) != cudaSuccess)
    return e;
  return cudaFuncSetAttribute(router_gemm_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              RCfg<256>::SMEM_BYTES);
}

cudaError_t launch_router_gemm(int tile_n, const CUtensorMap* map_w3, const CUtensorMap* map_x,
                               const RouterGemmArgs& a, int num_sms, cudaStream_t stream) {
  const int n_items = (a.T + tile_n - 1) / tile_n * a.m_tiles * a.ksplit;
  const int grid = n_items < num_sms ? n_items : num_sms;
  if (grid <= 0) return cudaSuccess;
  switch (tile_n) {
    case 16: return launch_rg<16>(map_w3, map_x, a, grid, stream);
    case 64: return launch_rg<64>(map_w3, map_x, a, grid, stream);
    case 128: return launch_rg<128>(map_w3, map_x, a, grid, stream);
    case 256: return launch_rg<256>(map_w3, map_x, a, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_router_topk(const float* partial, int ksplit, int T, int E, int k, int renorm, int* idx,
                               float* prob, float* gap, int* counts, float* tokstats, int n_groups,
                               cudaStream_t stream) {
  if (T <= 0) return cudaSuccess;
  // slots per lane: the fewest that hold E experts (of the instantiated widths)
  if (E <= 64)
    return launch_topk_ns<2>(partial, ksplit, T, E, k, renorm, idx, prob, gap, counts, tokstats, n_groups, stream);
  if (E <= 128)
    return launch_topk_ns<4>(partial, ksplit, T, E, k, renorm, idx, prob, gap, counts, tokstats, n_groups, stream);
  if (E <= 256)
    return launch_topk_ns<8>(partial, ksplit, T, E, k, renorm, idx, prob, gap, counts, tokstats, n_groups, stream);
  if (E <= 288)
    return launch_topk_ns<9>(partial, ksplit, T, E, k, renorm, idx, prob, gap, counts, tokstats, n_groups, stream);
  if (E <= kMaxExperts)
    return launch_topk_ns<kMaxExperts / 32>(partial, ksplit, T, E, k, renorm, idx, prob, gap, counts, tokstats,
                                            n_groups, stream);
  return cudaErrorInvalidValue;
}

bool route_small_fits(int T, int d, int E) {
  return T >= 1 && T <= kSmallRouteMaxTokens && d % 16 == 0 && E <= kMaxExperts;
}

cudaError_t launch_route_small(const bf16* x, const float* w_router, int T, int d, int E, int k, int renorm,
                               int has_shared, float* logits, unsigned int* done, int* idx, float* prob, float* gap,
                               int* counts, int* offsets, int* perm, int* inv, int* chunk_base,
                               const SmallRouteExtras& ex, cudaStream_t stream) {
  if (!route_small_fits(T, d, E)) return cudaErrorInvalidValue;
#define MOE_ROUTE_SMALL(NS_)                                                                                  \
  return launch_route_small_ns<NS_>(x, w_router, T, d, E, k, renorm, has_shared, logits, done, idx, prob, gap, \
                                    counts, offsets, perm, inv, chunk_base, ex, stream)
  if (E <= 64) MOE_ROUTE_SMALL(2);
  if (E <= 128) MOE_ROUTE_SMALL(4);
  if (E <= 256) MOE_ROUTE_SMALL(8);
  if (E <= 288) MOE_ROUTE_SMALL(9);
  MOE_ROUTE_SMALL(kMaxExperts / 32);
#undef MOE_ROUTE_SMALL
}

cudaError_t launch_route_stats(const float* tokstats, const int* counts, int T, int E, int k, int n_groups,
                               float* group_f, float* group_p, float* summary, cudaStream_t stream) {
  return launch_chain(route_stats_kernel, dim3(1), dim3(256), 0, stream, tokstats, counts, T, E, k, n_groups, group_f,
                      group_p, summary);
}

cudaError_t launch_split_router(const float* w, int E, int d, int e_pad, bf16* w3, cudaStream_t stream) {
  split_router_kernel<<<1024, 256, 0, stream>>>(w, E, d, e_pad, w3);
  return cudaGetLastError();
}

}  // namespace moe
