// K3 / K4 for wide token tiles on CTA pairs — the same grouped GEMMs as
// expert_gemm.cu ("Step3.5 Flash 大模型技术深度解析" (jsqmd.com) §3.2.1, §3.2.2),
// for 256 token rows per tile, run by clusters of two CTAs on two SMs with
// tcgen05.mma.cta_group::2 (M = 256 weight rows, N = 256 token rows).
//
// Why: with one CTA per tile, every K step brings a 16 KB weight tile and a
// 32 KB token tile into one SM for 128 x 256 outputs; the shared-memory fill
// bandwidth of the SM, not HBM or the tensor pipe, then sets the pace.  A pair
// splits both operands: each SM loads its 128 weight rows and 128 of the 256
// token rows (32 KB per K step) and the pair MMA reads the other half of the
// token tile from the peer, so each SM still computes 128 x 256 outputs.
//
// Roles per CTA as in the one-CTA kernel (warp 0 TMA, warp 1 MMA, warps 2..5
// epilogue), except that only the even CTA of the pair issues MMAs.  Its
// `full` barriers count the bytes of both CTAs' loads (the odd CTA's TMA
// completes on the even CTA's barrier), its commits arrive on the `empty` and
// `acc_full` barriers of both CTAs, and both CTAs' epilogue warps arrive on
// its `acc_empty`.  Each CTA's TMEM holds its 128 rows x 256 columns, double
// buffered (512 columns).  Every wait is bounded; the two CTAs meet at a
// cluster barrier before either frees tensor memory or exits.
#include "gemm_common.cuh"

namespace moe {
namespace {

using namespace gemm;

constexpr int kThreads = 192;
constexpr int kPairN = 256;  // token rows of a pair tile (N of the pair MMA)
constexpr int kHalfN = 128;  // token rows each CTA loads
// N of an M = 256 pair MMA: any multiple of 16 up to 256, so a tile's rows are
// rounded up to 16 (8 from each CTA); 32 would add 8 columns per tile on
// average at prefill sizes (~228 rows per group).
constexpr int kPairStep = 16;
constexpr int kSettleNs = 200000;

template <bool GATEUP>
struct PairCfg {
  static constexpr int A_BYTES = kBlockM * kBlockK * 2;  // this CTA's 128 weight rows
  static constexpr int B_BYTES = kHalfN * kBlockK * 2;   // this CTA's 128 token rows
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = 6;
  static constexpr int NACC = 2;
  static constexpr int TMEM_COLS = 512;
  static constexpr int NUM_BARS = 2 * STAGES + 2 * NACC + 1;
  static constexpr int XCHG_BYTES = GATEUP ? 2 * 2 * 64 * 8 * 4 : 0;
  static constexpr int AUX_BYTES = NUM_BARS * 8 + 16 + 32 + 2 * (kMaxGroups + 1) * 4;  // + tile starts, offsets
  static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + XCHG_BYTES + AUX_BYTES;
  static_assert(SMEM_BYTES <= 232448, "exceeds shared memory per block");
  static constexpr uint32_t IDESC = idesc_bf16_f32(2 * kBlockM, kPairN);
};

// try_wait with cluster-scope acquire (arrivals may come from the peer CTA).
__device__ __forceinline__ bool try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool wait_cluster(uint64_t* bar, uint32_t parity, uint64_t limit_ns,
                                             volatile int* abort_flag) {
  if (try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t spins = 0;
  while (true) {
    if (try_wait_cluster(bar, parity)) return true;
    if ((++spins & 15u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > limit_ns) return false;
    }
  }
}

template <bool GATEUP>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    expert_gemm_pair_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_act,
                            const __grid_constant__ CUtensorMap map_act2, const GemmArgs args) {
  using C = PairCfg<GATEUP>;
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
  volatile int* s_ok = reinterpret_cast<volatile int*>(tmem_holder + 4);
  int* tile_start = reinterpret_cast<int*>(tmem_holder + 12);
  int* s_off = tile_start + kMaxGroups + 1;  // the dispatch offsets, copied here once

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: issues the MMAs, 1: peer
  const int pair = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;
  const int G = args.G;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < C::NACC; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 8);  // 4 epilogue warps in each CTA
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&map_w);
    tma_prefetch_desc(&map_act);
    if (args.act2_from >= 0) tma_prefetch_desc(&map_act2);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_holder, C::TMEM_COLS);
    tmem_relinquish_pair();
  }
  pdl_wait();  // offsets, rows and outputs belong to earlier work in the stream until here
  if (warp == kEpilogueWarp0) {
    if (args.offsets != nullptr) {
      build_tile_start(args.offsets, G, kPairN, tile_start, lane, s_off);
    } else if (lane == 0) {
      // one group whose rows the host knows (G == 1): no dispatch offsets
      // needed, so the launch may run before the dispatch
      s_off[0] = args.off_const[0];
      s_off[1] = args.off_const[1];
      tile_start[0] = 0;
      tile_start[1] = (args.off_const[1] - args.off_const[0] + kPairN - 1) / kPairN;
    }
  }
  tc_fence_before();
  cluster_sync();  // barrier inits of both CTAs visible before any remote arrive
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int n_items = tile_start[G] * args.m_tiles;
  const uint64_t limit = args.wait_limit_ns;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer --
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_act = policy_evict_last();
      const int k_steps = args.K / kBlockK;
      // the rows an item loads: K3: 64 gate rows (+ the matching 64 up rows
      // at +F) per CTA, 128 features per pair tile; K4: 128 rows per CTA, 256
      // per pair tile.  The pair MMA takes N/2 token rows from each CTA: N =
      // the tile's rows rounded up to kPairStep, so the odd CTA's rows start at
      // N/2.
      auto rows_of = [&](int item, int& row_w, int& row_act) {
        const Item it = decode_item(item, args.m_tiles, tile_start, G, n_items, args.reverse);
        const int wg = weight_group(args, it.g);
        row_w = GATEUP ? wg * args.rows_per_group + it.m * kBlockM + static_cast<int>(rank) * 64
                       : wg * args.rows_per_group + it.m * 2 * kBlockM + static_cast<int>(rank) * kBlockM;
        const int g_row0 = s_off[it.g];
        const int n_mma = mma_width(s_off[it.g + 1] - g_row0 - it.n * kPairN, kPairStep, kPairN);
        row_act = g_row0 + it.n * kPairN + static_cast<int>(rank) * (n_mma / 2);
      };
      uint32_t stage = 0, phase = 0;
      long issued = 0;
      bool ok = true;
      int row_w = 0, row_act = 0, next_w = 0, next_act = 0;
      if (pair < n_items) rows_of(pair, next_w, next_act);
      for (int item = pair; ok && item < n_items && !*abort_flag; item += n_pairs) {
        row_w = next_w;
        row_act = next_act;
        for (int kb = 0; kb < k_steps; ++kb) {
          if (!wait_cluster(&empty[stage], phase ^ 1u, limit, abort_flag)) {
            record_abort(abort_flag, args.err);
            ok = false;
            break;
          }
          uint8_t* st = ring + stage * C::STAGE_BYTES;
          const uint32_t fb = mapa_shared(smem_u32(&full[stage]), 0);  // the even CTA's barrier
          if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * C::STAGE_BYTES);
          tma_load_2d_pair(st, &map_w, fb, kb * kBlockK, row_w, pol_w);
          if (GATEUP) tma_load_2d_pair(st + C::A_BYTES / 2, &map_w, fb, kb * kBlockK, row_w + args.F, pol_w);
          if (args.act2_from >= 0 && row_act >= args.act2_from)
            tma_load_2d_pair(st + C::A_BYTES, &map_act2, fb, kb * kBlockK, row_act - args.act2_from, pol_act);
          else
            tma_load_2d_pair(st + C::A_BYTES, &map_act, fb, kb * kBlockK, row_act, pol_act);
          ++issued;
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
          // the next item's rows, worked out while this item's loads are in
          // flight (its offsets come from global memory)
          if (kb == 0 && item + n_pairs < n_items) rows_of(item + n_pairs, next_w, next_act);
        }
      }
      if (rank == 0) {
        // the even CTA's barriers see every load of the pair: wait for the
        // phases this producer armed before the pair may exit
        for (int s = 0; s < C::STAGES; ++s) {
          if (issued <= s) break;
          const long last = s + ((issued - 1 - s) / C::STAGES) * C::STAGES;
          mbar_wait(&full[s], static_cast<uint32_t>((last / C::STAGES) & 1), kDrainLimitNs);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // --------------------------------------------------------------- MMA --
      const int k_steps = args.K / kBlockK;
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool issued_any = false, ok = true;
      // N of the pair MMAs: the tile's rows rounded up to kPairStep; the next
      // item's descriptor is worked out while this item's MMAs run
      uint32_t next_idesc =
          item_idesc(pair, n_items, args.reverse, args.m_tiles, tile_start, G, s_off, 2 * kBlockM, kPairStep, kPairN);
      for (int item = pair; ok && item < n_items && !*abort_flag; item += n_pairs) {
        const uint32_t idesc = next_idesc;
        if (!wait_cluster(&acc_empty[acc], acc_phase ^ 1u, limit, abort_flag)) {
          record_abort(abort_flag, args.err);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * kPairN;
        for (int kb = 0; kb < k_steps; ++kb) {
          if (!wait_cluster(&full[stage], phase, limit, abort_flag)) {
            record_abort(abort_flag, args.err);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = smem_u32(ring + stage * C::STAGE_BYTES);
          const uint64_t a = smem_desc_sw128(st);
          const uint64_t b = smem_desc_sw128(st + C::A_BYTES);
#pragma unroll
          for (int kk = 0; kk < kBlockK / 16; ++kk)
            tc_mma_bf16_pair(d_tmem, a + 2 * kk, b + 2 * kk, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
          issued_any = true;
          tc_commit_pair_multicast(&empty[stage], 0x3);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
          if (kb == 0)
            next_idesc = item_idesc(item + n_pairs, n_items, args.reverse, args.m_tiles, tile_start, G, s_off,
                                    2 * kBlockM, kPairStep, kPairN);
        }
        if (!ok) break;
        tc_commit_pair_multicast(&acc_full[acc], 0x3);
        if (++acc == C::NACC) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (issued_any) {
        tc_commit_pair(drain);
        mbar_wait(drain, 0, kDrainLimitNs);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue --
    const int q = warp & 3;
    const int row = q * 32 + lane;
    uint32_t acc = 0, acc_phase = 0, it_par = 0, chunk_par = 0;
    auto tile_rows = [&](int item, Item& it, int& row0, int& valid) {
      it = decode_item(item, args.m_tiles, tile_start, G, n_items, args.reverse);
      const int g_row0 = s_off[it.g];
      const int g_rows = s_off[it.g + 1] - g_row0;
      row0 = g_row0 + it.n * kPairN;
      valid = min(kPairN, g_rows - it.n * kPairN);
    };
    // K4: the gate weights of an item are fetched one item ahead — the
    // permutation entries while the previous item's accumulator is stored,
    // the probabilities they point at right after — so no dependent load sits
    // between an accumulator becoming ready and its stores
    float wreg[kPairN / 32];
    int pe[kPairN / 32];
    int cbase = 0, cbase_next = 0;  // the item's first exponent chunk of its group (K4)
    if (!GATEUP && pair < n_items) {
      Item it0;
      int r0, v0;
      tile_rows(pair, it0, r0, v0);
      gate_perm_entries<kPairN>(pe, r0, v0, lane, args.perm, args.Tk);
      gate_probs<kPairN>(wreg, pe, args.prob);
      cbase_next = args.chunk_base != nullptr ? __ldg(args.chunk_base + it0.g) : args.chunk_const;
    }
    for (int item = pair; item < n_items; item += n_pairs) {
      Item it;
      int row0, valid;
      tile_rows(item, it, row0, valid);
      cbase = cbase_next;
      valid = checked_valid(args, valid, row0, GATEUP ? -1 : cbase + it.n * (kPairN / kYpRows));
      const bool has_next = item + n_pairs < n_items;
      // one decision for all four epilogue warps (they meet at named barriers)
      const bool ok = __all_sync(0xffffffffu, wait_cluster(&acc_full[acc], acc_phase, limit, abort_flag));
      if (lane == 0) s_ok[it_par * 4 + q] = ok ? 1 : 0;
      named_bar_sync(kEpilogueBar, 128);
      const bool all_ok = s_ok[it_par * 4 + 0] && s_ok[it_par * 4 + 1] && s_ok[it_par * 4 + 2] &&
                          s_ok[it_par * 4 + 3];
      it_par ^= 1u;
      if (!all_ok) {
        if (lane == 0 && !ok) record_abort(abort_flag, args.err);
        break;
      }
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kPairN;
      if (GATEUP) {
        epilogue_gateup<kPairN>(taddr, row, it.m * kBlockM + static_cast<int>(rank) * 64, row0, valid,
                                static_cast<bf16*>(args.out), args.out_ld, xchg, chunk_par);
      } else {
        Item it_n;
        int row0_n = 0, valid_n = 0;
        if (has_next) {
          tile_rows(item + n_pairs, it_n, row0_n, valid_n);
          gate_perm_entries<kPairN>(pe, row0_n, valid_n, lane, args.perm, args.Tk);
          cbase_next = args.chunk_base != nullptr ? __ldg(args.chunk_base + it_n.g) : args.chunk_const;
        }
        epilogue_down_pipelined<kPairN>(taddr, it.m * 2 * kBlockM + static_cast<int>(rank) * kBlockM + row, row0,
                                        valid, wreg, static_cast<__half*>(args.out), args.out_exp, args.out_ld,
                                        cbase + it.n * (kPairN / kYpRows));
        if (has_next) gate_probs<kPairN>(wreg, pe, args.prob);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&acc_empty[acc]), 0));
      if (++acc == C::NACC) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  // After an abort, loads of the odd CTA may still be landing in its shared
  // memory (their completion is counted on the even CTA's barriers): give
  // them time before the pair exits.
  if (*abort_flag) {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < kSettleNs) {
    }
  }
  tc_fence_before();
  cluster_sync();
  // dependents launch as this grid ends (past the barrier every role has
  // finished): their blocks would otherwise wait on these SMs for the whole
  // run of this persistent kernel
  pdl_trigger();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
  }
}

}  // namespace

MOE_DBG_DEFINE_TAKE(dbg_take_expert_gemm_pair)

cudaError_t expert_gemm_pair_prepare() {
  cudaError_t e = cudaFuncSetAttribute(expert_gemm_pair_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       PairCfg<true>::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(expert_gemm_pair_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              PairCfg<false>::SMEM_BYTES);
}

cudaError_t launch_expert_gemm_pair(bool gateup, const CUtensorMap* map_w, const CUtensorMap* map_act,
                                    const CUtensorMap* map_act2, const GemmArgs& a, int num_sms,
                                    cudaStream_t stream) {
  if (map_act2 == nullptr) map_act2 = map_act;
  const int grid = num_sms & ~1;
  if (gateup)
    return launch_chain(expert_gemm_pair_kernel<true>, dim3(grid), dim3(kThreads), PairCfg<true>::SMEM_BYTES, stream,
                        *map_w, *map_act, *map_act2, a);
  return launch_chain(expert_gemm_pair_kernel<false>, dim3(grid), dim3(kThreads), PairCfg<false>::SMEM_BYTES, stream,
                      *map_w, *map_act, *map_act2, a);
}

}  // namespace moe
