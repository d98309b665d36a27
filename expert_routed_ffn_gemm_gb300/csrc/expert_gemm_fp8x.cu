// K3 / K4 with FP8 expert weights and the token rows as two E4M3 terms — the
// FP8/FP16 mixed-precision inference of "Step3.5 Flash 大模型技术深度解析"
// (jsqmd.com) §8.1 applied to the gate/up and down projections of §3.2.1.
//
// The E4M3 weight codes go to the tensor cores as they are (tcgen05.mma
// kind::f8f6f4, both operands E4M3, fp32 accumulate): no widening on chip.
// Each token row x (gate/up) or h (down) arrives as two E4M3 rows,
// hi = e4m3(s*x) and lo = e4m3(s*x - hi), with one power-of-two scale s per
// row (the largest that keeps |s*x| <= 448), written by the row scatter (x)
// or by the in-place requantisation of H (h).  For an 8-bit significand (a
// bf16 x) the remainder after rounding to E4M3's 4 bits has at most 4
// significant bits, so hi + lo = s*x exactly while lo is in E4M3's normal
// range; below it lo is rounded to a multiple of 2^-9 (an error of at most
// 2^-10, against 256 <= s*max|x| <= 448).  H (fp16, 11 bits) keeps 8 bits
// this way, as the bf16 path's H does.  The hi rows and the lo rows of
// a token tile are the N operand of one MMA (N = 2*BN): column j holds the
// hi product of token j and column BN + j its lo product, and the epilogue
// adds the two, multiplies by the weight row's scale and by 1/s of the token,
// then applies the SiLU gate (K3) or the gate weight and the block-scaled
// fp16 store (K4, as expert_gemm.cu):
//   H[r, f]  = silu(sg_f/s_r * (X2[r].Qg[g, f])) * (su_f/s_r * (X2[r].Qu[g, f]))   (fp16)
//   Yp[r, o] = w_r * (sd_o/t_r * (H2[r].Qd[g, o]))
//
// Why: an M = 128, N = 16 MMA costs about the same time as one with N = 32,
// and one E4M3 MMA covers 32 K values against 16 for fp16 operands, so a
// 128-row K step of weights takes 4 MMAs here against 8 when the weights are
// widened to fp16 (the single-CTA FP8 kernel is bounded by those MMAs).
//
// Work decomposition as expert_gemm.cu (one CTA per SM, 128 weight rows per
// tile as M — K3: 64 gate + 64 up rows — token tiles of BN rows, weight tile
// fastest):
//   warp 0      TMA producer: per K step of 128, the E4M3 weight box(es) and
//               the BN x 128-byte hi and lo token boxes (the lo terms sit at
//               (lo_col0, lo_row0) from the hi terms in the token map)
//   warp 1      TMEM allocator + tcgen05.mma issuer
//   warps 2..5  epilogue (hi + lo, scales, SiLU gate or gate weight, stores)
// Every wait is bounded (wait_limit_ns); on timeout the kernel records an
// error, drains what it issued, frees tensor memory and returns.
#include "gemm_common.cuh"

namespace moe {
namespace {

using namespace gemm;

constexpr int kThreadsX = 192;
constexpr int kKStepX = kKStepE4M3;  // K elements (bytes) per stage

// E4M3 x E4M3 -> fp32 MMA from shared memory, K = 32 per instruction.
__device__ __forceinline__ void tc_mma_e4m3(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Instruction descriptor of kind::f8f6f4 with E4M3 A and B (format code 0),
// fp32 accumulation, both K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
  return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

template <bool GATEUP, int BN>
struct CfgX {
  static constexpr int A_BYTES = kBlockM * kKStepX;    // 128 weight rows x 128 E4M3
  static constexpr int B_HALF = BN * kKStepX;          // BN token rows x 128 E4M3 (hi or lo)
  static constexpr int STAGE_BYTES = A_BYTES + 2 * B_HALF;
  static constexpr int RING_BUDGET = 192 * 1024;
  static constexpr int STAGES_RAW = RING_BUDGET / STAGE_BYTES;
  static constexpr int STAGES = STAGES_RAW > 9 ? 9 : STAGES_RAW;
  static constexpr int NACC = 2;
  static constexpr int ACC_COLS = 2 * BN;  // hi columns, then lo columns
  static constexpr int TMEM_RAW = NACC * ACC_COLS;
  static constexpr int TMEM_COLS = TMEM_RAW <= 32 ? 32 : TMEM_RAW <= 64 ? 64 : TMEM_RAW <= 128 ? 128
                                                                       : TMEM_RAW <= 256 ? 256 : 512;
  static constexpr int NUM_BARS = 2 * STAGES + 2 * NACC + 1;
  static constexpr int XCHG_BYTES = GATEUP ? 2 * 2 * 64 * 8 * 4 : 0;
  static constexpr int AUX_BYTES = NUM_BARS * 8 + 16 + 32 + (kMaxGroups + 1) * 4;
  static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + XCHG_BYTES + AUX_BYTES;
  static_assert(STAGE_BYTES % 1024 == 0 && B_HALF % 1024 == 0, "stages must keep 1024-byte alignment");
  static_assert(STAGES >= 2, "ring too shallow");
  static_assert(TMEM_RAW <= 512, "accumulators exceed tensor memory");
  static_assert(SMEM_BYTES <= 232448, "exceeds shared memory per block");
  static constexpr uint32_t IDESC = idesc_e4m3_f32(kBlockM, 2 * BN);
};

template <bool GATEUP, int BN>
__global__ void __launch_bounds__(kThreadsX, 1)
    expert_gemm_fp8x_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_tok,
                            const GemmArgs args) {
  using C = CfgX<GATEUP, BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  float* xchg = reinterpret_cast<float*>(smem + C::STAGES * C::STAGE_BYTES);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES + C::XCHG_BYTES);
  uint64_t* full = bars;
  uint64_t* empty = bars + C::STAGES;
  uint64_t* acc_full = bars + 2 * C::STAGES;
  uint64_t* acc_empty = acc_full + C::NACC;
  uint64_t* drain = acc_empty + C::NACC;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + C::NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  volatile int* s_ok = reinterpret_cast<volatile int*>(tmem_holder + 4);  // [2 parities][4 warps]
  int* tile_start = reinterpret_cast<int*>(tmem_holder + 12);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = args.G;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < C::NACC; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&map_w);
    tma_prefetch_desc(&map_tok);
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, C::TMEM_COLS);
    tmem_relinquish();
  }
  pdl_wait();  // offsets, rows and outputs belong to earlier work in the stream until here
  if (warp == kEpilogueWarp0) build_tile_start(args.offsets, G, BN, tile_start, lane);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int n_base = tile_start[G] * args.m_tiles;
  // K split (token tiles <= 32, few items): part p of an item takes the K
  // steps [p * k_per, min(k_steps, (p + 1) * k_per)), the parts adjacent
  const int ks = (BN <= 32 && args.ksplit > 1 && n_base * args.ksplit <= args.ksplit_cap) ? args.ksplit : 1;
  const int n_items = n_base * ks;
  const uint64_t limit = args.wait_limit_ns;
  const int k_steps = args.K / kKStepX;
  const int k_per = (k_steps + ks - 1) / ks;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer --
      const uint64_t pol_w = policy_evict_first();   // weights: streamed once
      const uint64_t pol_act = policy_evict_last();  // token rows: re-read by the other weight tiles
      auto rows_of = [&](int item, int& row_w, int& row_act) {
        const Item it = decode_item(item / ks, args.m_tiles, tile_start, G, n_base, args.reverse);
        row_w = weight_group(args, it.g) * args.rows_per_group + it.m * (GATEUP ? kBlockM / 2 : kBlockM);
        row_act = __ldg(args.offsets + it.g) + it.n * BN;
      };
      uint32_t stage = 0, phase = 0;
      long issued = 0;
      bool ok = true;
      int next_w = 0, next_act = 0;
      if (static_cast<int>(blockIdx.x) < n_items) rows_of(blockIdx.x, next_w, next_act);
      for (int item = blockIdx.x; ok && item < n_items && !*abort_flag; item += gridDim.x) {
        const int row_w = next_w, row_act = next_act;
        const int part = item % ks;
        const int kb1 = min(k_steps, (part + 1) * k_per);
        for (int kb = part * k_per; kb < kb1; ++kb) {
          if (!wait_or_abort(&empty[stage], phase ^ 1u, limit, abort_flag)) {
            record_abort(abort_flag, args.err);
            ok = false;
            break;
          }
          uint8_t* st = ring + stage * C::STAGE_BYTES;
          mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
          tma_load_2d(st, &map_w, &full[stage], kb * kKStepX, row_w, pol_w);
          if (GATEUP) tma_load_2d(st + C::A_BYTES / 2, &map_w, &full[stage], kb * kKStepX, row_w + args.F, pol_w);
          tma_load_2d(st + C::A_BYTES, &map_tok, &full[stage], kb * kKStepX, row_act, pol_act);
          tma_load_2d(st + C::A_BYTES + C::B_HALF, &map_tok, &full[stage], args.lo_col0 + kb * kKStepX,
                      args.lo_row0 + row_act, pol_act);
          ++issued;
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
          // the next item's rows, worked out while this item's loads are in
          // flight (its offsets come from global memory)
          if (kb == part * k_per && item + static_cast<int>(gridDim.x) < n_items)
            rows_of(item + gridDim.x, next_w, next_act);
        }
      }
      for (int s = 0; s < C::STAGES; ++s) {
        if (issued <= s) break;
        const long last = s + ((issued - 1 - s) / C::STAGES) * C::STAGES;
        mbar_wait(&full[s], static_cast<uint32_t>((last / C::STAGES) & 1), kDrainLimitNs);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // --------------------------------------------------------------- MMA --
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool issued_any = false, ok = true;
      for (int item = blockIdx.x; ok && item < n_items && !*abort_flag; item += gridDim.x) {
        if (!wait_or_abort(&acc_empty[acc], acc_phase ^ 1u, limit, abort_flag)) {
          record_abort(abort_flag, args.err);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * C::ACC_COLS;
        const int part = item % ks;
        const int kb0 = part * k_per, kb1 = min(k_steps, (part + 1) * k_per);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!wait_or_abort(&full[stage], phase, limit, abort_flag)) {
            record_abort(abort_flag, args.err);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = smem_u32(ring + stage * C::STAGE_BYTES);
          const uint64_t a = smem_desc_sw128(st);
          const uint64_t b = smem_desc_sw128(st + C::A_BYTES);  // hi rows, then lo rows: N = 2*BN
#pragma unroll
          for (int kk = 0; kk < kKStepX / 32; ++kk)  // +32 B along K = +2 in the address field
            tc_mma_e4m3(d_tmem, a + 2 * kk, b + 2 * kk, C::IDESC, (kb > kb0 || kk > 0) ? 1u : 0u);
          issued_any = true;
          tc_commit(&empty[stage]);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
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
    // ------------------------------------------------------------ epilogue --
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;
    uint32_t acc = 0, acc_phase = 0, it_par = 0, chunk_par = 0;
    volatile int* s_last = reinterpret_cast<volatile int*>(tmem_holder + 2);
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
      const Item it = decode_item(item / ks, args.m_tiles, tile_start, G, n_base, args.reverse);
      const int g_row0 = __ldg(args.offsets + it.g);
      const int g_rows = __ldg(args.offsets + it.g + 1) - g_row0;
      const int row0 = g_row0 + it.n * BN;
      const int chunk0 = GATEUP ? -1 : __ldg(args.chunk_base + it.g) + it.n * (BN / kYpRows);
      const int valid = checked_valid(args, min(BN, g_rows - it.n * BN), row0, chunk0);
      const size_t wrow0 = static_cast<size_t>(weight_group(args, it.g)) * args.rows_per_group;
      // K3 rows 0..63: gate of feature 64m + row; rows 64..127: up of feature 64m + row - 64
      const float scale = GATEUP ? __ldg(args.w_scale + wrow0 + (row < 64 ? 0 : args.F) + it.m * (kBlockM / 2) +
                                         (row & 63))
                                 : __ldg(args.w_scale + wrow0 + it.m * kBlockM + row);
      // K4: the gate weight of every column times the token's 1/s
      float wreg[(BN + 31) / 32];
      if (!GATEUP) {
        load_gate_weights<BN>(wreg, row0, valid, lane, args.perm, args.prob, args.Tk);
#pragma unroll
        for (int i = 0; i < (BN + 31) / 32; ++i) {
          const int c = i * 32 + lane;
          if (c < valid) wreg[i] *= __ldg(args.tok_scale + row0 + c);
        }
      }
      if (!epilogue_wait(&acc_full[acc], acc_phase, limit, abort_flag, s_ok, it_par, q, lane, args.err)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * C::ACC_COLS;
      if constexpr (BN <= 32) {
        if (ks > 1) {
          // this part's hi + lo row to the part buffer, tensor memory back to
          // the MMA, then the last part of the item sums the parts in order
          ksplit_store_part<BN>(taddr, BN, valid, args.ksplit_part + (static_cast<size_t>(item) * kBlockM + row) * BN);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[acc]);
          if (++acc == C::NACC) {
            acc = 0;
            acc_phase ^= 1u;
          }
          const int base = item / ks;
          if (ksplit_arrive(args.ksplit_cnt + base, ks, s_last, q == 0 && lane == 0)) {
            float sum[BN];
            ksplit_sum_parts<BN>(args.ksplit_part + (static_cast<size_t>(base * ks) * kBlockM + row) * BN, ks, valid,
                                 sum);
            if (GATEUP)
              epilogue_gateup_x2<BN>(0u, row, it.m * (kBlockM / 2), row0, valid, static_cast<__half*>(args.out),
                                     args.out_ld, xchg, chunk_par, scale, args.tok_scale, BN, sum);
            else
              epilogue_down<BN>(0u, it.m * kBlockM + row, row0, valid, wreg, static_cast<__half*>(args.out),
                                args.out_exp, args.out_ld, chunk0,
                                scale, 0, sum);
            if (q == 0 && lane == 0) args.ksplit_cnt[base] = 0;  // ready for the next launch
          }
          continue;
        }
      }
      if (GATEUP)
        epilogue_gateup_x2<BN>(taddr, row, it.m * (kBlockM / 2), row0, valid, static_cast<__half*>(args.out),
                               args.out_ld, xchg, chunk_par, scale, args.tok_scale, BN);
      else
        epilogue_down<BN>(taddr, it.m * kBlockM + row, row0, valid, wreg, static_cast<__half*>(args.out),
                          args.out_exp, args.out_ld, chunk0, scale, BN);
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

template <bool GATEUP, int BN>
cudaError_t launchx_one(const CUtensorMap* map_w, const CUtensorMap* map_tok, const GemmArgs& a, int num_sms,
                        cudaStream_t stream) {
  return launch_chain(expert_gemm_fp8x_kernel<GATEUP, BN>, dim3(num_sms), dim3(kThreadsX),
                      CfgX<GATEUP, BN>::SMEM_BYTES, stream, *map_w, *map_tok, a);
}

template <bool GATEUP, int BN>
cudaError_t preparex_one() {
  return cudaFuncSetAttribute(expert_gemm_fp8x_kernel<GATEUP, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              CfgX<GATEUP, BN>::SMEM_BYTES);
}

template <bool GATEUP>
cudaError_t dispatchx(int tile_n, const CUtensorMap* map_w, const CUtensorMap* map_tok, const GemmArgs& a,
                      int num_sms, cudaStream_t stream) {
  switch (tile_n) {
    case 16: return launchx_one<GATEUP, 16>(map_w, map_tok, a, num_sms, stream);
    case 32: return launchx_one<GATEUP, 32>(map_w, map_tok, a, num_sms, stream);
    case 64: return launchx_one<GATEUP, 64>(map_w, map_tok, a, num_sms, stream);
    case 128: return launchx_one<GATEUP, 128>(map_w, map_tok, a, num_sms, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <bool GATEUP>
cudaError_t preparex_all() {
  cudaError_t e;
  if ((e = preparex_one<GATEUP, 16>()) != cudaSuccess) return e;
  if ((e = preparex_one<GATEUP, 32>()) != cudaSuccess) return e;
  if ((e = preparex_one<GATEUP, 64>()) != cudaSuccess) return e;
  return preparex_one<GATEUP, 128>();
}

}  // namespace

MOE_DBG_DEFINE_TAKE(dbg_take_expert_gemm_fp8x)

cudaError_t launch_expert_gemm_fp8x(bool gateup, int tile_n, const CUtensorMap* map_w, const CUtensorMap* map_tok,
                                    const GemmArgs& a, int num_sms, cudaStream_t stream) {
  return gateup ? dispatchx<true>(tile_n, map_w, map_tok, a, num_sms, stream)
                : dispatchx<false>(tile_n, map_w, map_tok, a, num_sms, stream);
}

cudaError_t expert_gemm_fp8x_prepare() {
  const cudaError_t e = preparex_all<true>();
  return e != cudaSuccess ? e : preparex_all<false>();
}

}  // namespace moe
