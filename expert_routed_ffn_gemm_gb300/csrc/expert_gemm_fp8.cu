// K3 / K4 with FP8 expert weights — the FP8/FP16 mixed-precision inference of
// "Step3.5 Flash 大模型技术深度解析" (jsqmd.com) §8.1 applied to the experts of
// §3.2.1: the weights are stored as OCP E4M3 codes (one byte each) with one fp32
// scale per weight row, the activations (token rows X and the gate output H) as
// fp16, and the products are accumulated in fp32:
//   gate/up (K3):  H[r, f]  = silu(sg_f * X[r].Qg[g, f]) * (su_f * X[r].Qu[g, f])   (fp16)
//   down    (K4):  Yp[r, o] = w_r * (sd_o * H[r].Qd[g, o])                           (scaled fp16)
//
// Same work decomposition as expert_gemm.cu (one CTA per SM, weights as the
// M operand, token tiles of 16..128 rows as N, weight tile fastest), with the
// weights widened on chip: E4M3 -> fp16 is exact, so the tensor cores see the
// code values and the row scale is applied to the fp32 accumulator.
//   warp 0      TMA producer: per K step of 128, one 128 x 128-byte E4M3 weight
//               tile and the BN x 128 fp16 token tile (two 64-column boxes)
//   warp 1      TMEM allocator + tcgen05.mma issuer, A read from tensor memory
//   warps 2..5  epilogue (row scale, SiLU gate or gate-weight scale, stores)
//   warps 6..13 converters, two sets of four: set 0 takes the even K steps,
//               set 1 the odd ones, so two stages are widened at a time; each
//               thread takes one weight row of its stage from shared memory
//               (128 bytes), widens it to 64 fp16 pairs and stores them into a
//               ring of A tiles in tensor memory (64 columns each, above the
//               2*BN accumulator columns: 4 to 7 slots by BN)
// The widened tile never goes back to shared memory: shared-memory traffic per
// weight byte stays at one TMA write and one read.  The E4M3 tiles and the
// token tiles sit in two separate rings: a weight stage is handed back to the
// producer as soon as its converters have read it (before the MMAs run), so
// the bytes in flight from HBM are not held up by the widening and the MMAs.
// Every wait is bounded (wait_limit_ns); on timeout the kernel records an
// error, drains what it issued, frees tensor memory and returns.
#include "gemm_common.cuh"

namespace moe {
namespace {

using namespace gemm;

constexpr int kThreads8 = 448;
constexpr int kKStep8 = 128;           // K elements per stage (one 128-byte E4M3 row)
constexpr int kConvWarp0 = 6;          // warps 6..13 convert (two sets of four)
constexpr int kConvSets = 2;
constexpr uint32_t kAColsPerSlot = 64; // 128 fp16 per row = 64 columns

template <bool GATEUP, int BN>
struct Cfg8 {
  static constexpr int A8_BYTES = kBlockM * kKStep8;      // 128 rows x 128 E4M3
  static constexpr int B_HALF = BN * 128;                 // BN rows x 64 fp16
  static constexpr int B_BYTES = 2 * B_HALF;              // K 0..63 and 64..127
  // ring depths (weight stages NA, token stages NB) within 192 KB
  static constexpr int NA = BN <= 32 ? 8 : (BN == 64 ? 6 : 4);
  static constexpr int NB = BN == 16 ? 12 : (BN == 32 ? 8 : (BN == 64 ? 6 : 4));
  static constexpr int RING_BYTES = NA * A8_BYTES + NB * B_BYTES;
  static constexpr int NACC = 2;
  static constexpr int TMEM_COLS = 512;
  // A ring in tensor memory: from the first multiple of 64 columns above the
  // accumulators to column 511 (7 slots for BN <= 32, 6 for 64, 4 for 128)
  static constexpr uint32_t ACOL0 = ((NACC * BN + 63) / 64) * 64;
  static constexpr int NSLOT = (TMEM_COLS - static_cast<int>(ACOL0)) / 64;
  // a8_full[NA], a8_empty[NA], b_full[NB], b_empty[NB], a_full[4], a_empty[4],
  // acc_full[2], acc_empty[2], drain
  static constexpr int NUM_BARS = 2 * NA + 2 * NB + 2 * NSLOT + 2 * NACC + 1;
  static constexpr int XCHG_BYTES = GATEUP ? 2 * 2 * 64 * 8 * 4 : 0;
  static constexpr int AUX_BYTES = NUM_BARS * 8 + 16 + 32 + (kMaxGroups + 1) * 4;
  static constexpr int SMEM_BYTES = 1024 + RING_BYTES + XCHG_BYTES + AUX_BYTES;
  static_assert(BN <= 128, "accumulators must fit below the A ring");
  static_assert(B_BYTES % 1024 == 0, "token stages must keep 1024-byte alignment");
  static_assert(RING_BYTES <= 192 * 1024, "rings exceed their budget");
  static_assert(SMEM_BYTES <= 232448, "exceeds shared memory per block");
  static constexpr uint32_t IDESC = idesc_f16_f32(kBlockM, BN);
};

template <bool GATEUP, int BN>
__global__ void __launch_bounds__(kThreads8, 1)
    expert_gemm_fp8_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_act,
                           const GemmArgs args) {
  using C = Cfg8<GATEUP, BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring_a = smem;                          // NA x 16 KB E4M3 tiles
  uint8_t* ring_b = smem + C::NA * C::A8_BYTES;    // NB x token tiles
  float* xchg = reinterpret_cast<float*>(smem + C::RING_BYTES);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::RING_BYTES + C::XCHG_BYTES);
  uint64_t* a8_full = bars;
  uint64_t* a8_empty = a8_full + C::NA;
  uint64_t* b_full = a8_empty + C::NA;
  uint64_t* b_empty = b_full + C::NB;
  uint64_t* a_full = b_empty + C::NB;
  uint64_t* a_empty = a_full + C::NSLOT;
  uint64_t* acc_full = a_empty + C::NSLOT;
  uint64_t* acc_empty = acc_full + C::NACC;
  uint64_t* drain = acc_empty + C::NACC;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + C::NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  volatile int* s_ok = reinterpret_cast<volatile int*>(tmem_holder + 4);  // [2 parities][4 warps]
  int* tile_start = reinterpret_cast<int*>(tmem_holder + 12);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = args.G;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::NA; ++s) {
      mbar_init(&a8_full[s], 1);
      mbar_init(&a8_empty[s], 4);  // the four converter warps that read the stage
    }
    for (int s = 0; s < C::NB; ++s) {
      mbar_init(&b_full[s], 1);
      mbar_init(&b_empty[s], 1);  // the MMA commit
    }
    for (int j = 0; j < C::NSLOT; ++j) {
      mbar_init(&a_full[j], 4);
      mbar_init(&a_empty[j], 1);
    }
    for (int a = 0; a < C::NACC; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&map_w);
    tma_prefetch_desc(&map_act);
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
  const int n_items = tile_start[G] * args.m_tiles;
  const uint64_t limit = args.wait_limit_ns;
  const int k_steps = args.K / kKStep8;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer --
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_act = policy_evict_last();
      uint32_t sa = 0, pa = 0, sb = 0, pb = 0;
      long issued = 0;
      bool ok = true;
      for (int item = blockIdx.x; ok && item < n_items && !*abort_flag; item += gridDim.x) {
        const Item it = decode_item(item, args.m_tiles, tile_start, G, n_items, args.reverse);
        const int row_w = weight_group(args, it.g) * args.rows_per_group + it.m * (GATEUP ? kBlockM / 2 : kBlockM);
        const int row_act = __ldg(args.offsets + it.g) + it.n * BN;
        for (int kb = 0; kb < k_steps; ++kb) {
          if (!wait_or_abort(&a8_empty[sa], pa ^ 1u, limit, abort_flag) ||
              !wait_or_abort(&b_empty[sb], pb ^ 1u, limit, abort_flag)) {
            record_abort(abort_flag, args.err);
            ok = false;
            break;
          }
          uint8_t* sta = ring_a + sa * C::A8_BYTES;
          mbar_arrive_expect_tx(&a8_full[sa], C::A8_BYTES);
          tma_load_2d(sta, &map_w, &a8_full[sa], kb * kKStep8, row_w, pol_w);
          if (GATEUP) tma_load_2d(sta + C::A8_BYTES / 2, &map_w, &a8_full[sa], kb * kKStep8, row_w + args.F, pol_w);
          uint8_t* stb = ring_b + sb * C::B_BYTES;
          mbar_arrive_expect_tx(&b_full[sb], C::B_BYTES);
          tma_load_2d(stb, &map_act, &b_full[sb], kb * kKStep8, row_act, pol_act);
          tma_load_2d(stb + C::B_HALF, &map_act, &b_full[sb], kb * kKStep8 + 64, row_act, pol_act);
          ++issued;
          if (++sa == C::NA) {
            sa = 0;
            pa ^= 1u;
          }
          if (++sb == C::NB) {
            sb = 0;
            pb ^= 1u;
          }
        }
      }
      // every load issued must have landed before the CTA may exit
      for (int s = 0; s < C::NA; ++s) {
        if (issued <= s) break;
        const long last = s + ((issued - 1 - s) / C::NA) * C::NA;
        mbar_wait(&a8_full[s], static_cast<uint32_t>((last / C::NA) & 1), kDrainLimitNs);
      }
      for (int s = 0; s < C::NB; ++s) {
        if (issued <= s) break;
        const long last = s + ((issued - 1 - s) / C::NB) * C::NB;
        mbar_wait(&b_full[s], static_cast<uint32_t>((last / C::NB) & 1), kDrainLimitNs);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // --------------------------------------------------------------- MMA --
      uint32_t sb = 0, pb = 0, slot = 0, slot_phase = 0, acc = 0, acc_phase = 0;
      bool issued_any = false, ok = true;
      for (int item = blockIdx.x; ok && item < n_items && !*abort_flag; item += gridDim.x) {
        if (!wait_or_abort(&acc_empty[acc], acc_phase ^ 1u, limit, abort_flag)) {
          record_abort(abort_flag, args.err);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < k_steps; ++kb) {
          if (!wait_or_abort(&b_full[sb], pb, limit, abort_flag) ||
              !wait_or_abort(&a_full[slot], slot_phase, limit, abort_flag)) {
            record_abort(abort_flag, args.err);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_tmem = tmem_base + C::ACOL0 + slot * kAColsPerSlot;
          const uint32_t st_b = smem_u32(ring_b + sb * C::B_BYTES);
#pragma unroll
          for (int kk = 0; kk < kKStep8 / 16; ++kk) {
            // K 16kk..16kk+15: A columns 8kk.., B in half kk/4 at +32 B per 16 K
            const uint64_t b = smem_desc_sw128(st_b + (kk >> 2) * C::B_HALF) + 2 * (kk & 3);
            tc_mma_f16_tmem_a(d_tmem, a_tmem + 8 * kk, b, C::IDESC, (kb > 0 || kk > 0) ? 1u : 0u);
          }
          issued_any = true;
          tc_commit(&b_empty[sb]);
          tc_commit(&a_empty[slot]);
          if (++sb == C::NB) {
            sb = 0;
            pb ^= 1u;
          }
          if (++slot == C::NSLOT) {
            slot = 0;
            slot_phase ^= 1u;
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
  } else if (warp >= kConvWarp0) {
    // -------------------------------------------------------- converters --
    const int q = warp & 3;  // TMEM lane quarter
    const int set = (warp - kConvWarp0) >> 2;  // 0: even K steps, 1: odd K steps
    const int r = q * 32 + lane;  // weight row of the tile this thread widens
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    const long my_items = n_items > static_cast<int>(blockIdx.x)
                              ? (n_items - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1
                              : 0;
    const long total = my_items * k_steps;  // K steps this CTA runs, over all its items
    bool ok = true;
    for (long step = set; ok && step < total; step += kConvSets) {
      if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
      const uint32_t stage = static_cast<uint32_t>(step % C::NA);
      const uint32_t phase = static_cast<uint32_t>((step / C::NA) & 1);
      const uint32_t slot = static_cast<uint32_t>(step % C::NSLOT);
      const uint32_t slot_phase = static_cast<uint32_t>((step / C::NSLOT) & 1);
      {
        const bool got = wait_or_abort(&a8_full[stage], phase, limit, abort_flag) &&
                         wait_or_abort(&a_empty[slot], slot_phase ^ 1u, limit, abort_flag);
        if (!__all_sync(0xffffffffu, got)) {
          if (lane == 0) record_abort(abort_flag, args.err);
          ok = false;
          continue;  // leaves the loop (ok is false)
        }
        tc_fence_after();
        // row r of the 128-byte-swizzled E4M3 tile: chunk c at r*128 + ((c ^ (r & 7)) * 16)
        const uint8_t* row = ring_a + stage * C::A8_BYTES + r * 128;
        uint32_t w[32];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 v = *reinterpret_cast<const uint4*>(row + ((c ^ (r & 7)) << 4));
          w[4 * c + 0] = v.x;
          w[4 * c + 1] = v.y;
          w[4 * c + 2] = v.z;
          w[4 * c + 3] = v.w;
        }
        // widen first: once every value is in registers the stage goes back
        uint32_t h[64];  // column j: fp16 pair of K 2j, 2j+1
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          h[2 * i] = e4m3x2_to_f16x2(w[i] & 0xffffu);
          h[2 * i + 1] = e4m3x2_to_f16x2(w[i] >> 16);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&a8_empty[stage]);
        const uint32_t taddr = tmem_base + lane_base + C::ACOL0 + slot * kAColsPerSlot;
        tmem_st32(taddr, *reinterpret_cast<const uint32_t(*)[32]>(&h[0]));
        tmem_st32(taddr + 32, *reinterpret_cast<const uint32_t(*)[32]>(&h[32]));
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&a_full[slot]);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue --
    const int q = warp & 3;
    const int row = q * 32 + lane;
    uint32_t acc = 0, acc_phase = 0, it_par = 0, chunk_par = 0;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
      const Item it = decode_item(item, args.m_tiles, tile_start, G, n_items, args.reverse);
      const int g_row0 = __ldg(args.offsets + it.g);
      const int g_rows = __ldg(args.offsets + it.g + 1) - g_row0;
      const int row0 = g_row0 + it.n * BN;
      const int chunk0 = GATEUP ? -1 : __ldg(args.chunk_base + it.g) + it.n * (BN / kYpRows);
      const int valid = checked_valid(args, min(BN, g_rows - it.n * BN), row0, chunk0);
      float wreg[(BN + 31) / 32];
      if (!GATEUP) load_gate_weights<BN>(wreg, row0, valid, lane, args.perm, args.prob, args.Tk);
      // the scale of this thread's weight row
      const float scale =
          GATEUP ? __ldg(args.w_scale + static_cast<size_t>(weight_group(args, it.g)) * args.rows_per_group +
                         (row < 64 ? 0 : args.F) +
                         it.m * (kBlockM / 2) + (row & 63))
                 : __ldg(args.w_scale + static_cast<size_t>(weight_group(args, it.g)) * args.rows_per_group +
                         it.m * kBlockM + row);
      if (!epilogue_wait(&acc_full[acc], acc_phase, limit, abort_flag, s_ok, it_par, q, lane, args.err)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
      if (GATEUP) {
        epilogue_gateup<BN>(taddr, row, it.m * (kBlockM / 2), row0, valid, static_cast<__half*>(args.out),
                            args.out_ld, xchg, chunk_par, scale);
      } else {
        epilogue_down<BN>(taddr, it.m * kBlockM + row, row0, valid, wreg, static_cast<__half*>(args.out),
                          args.out_exp, args.out_ld, chunk0, scale);
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

template <bool GATEUP, int BN>
cudaError_t launch8_one(const CUtensorMap* map_w, const CUtensorMap* map_act, const GemmArgs& a, int num_sms,
                        cudaStream_t stream) {
  return launch_chain(expert_gemm_fp8_kernel<GATEUP, BN>, dim3(num_sms), dim3(kThreads8),
                      Cfg8<GATEUP, BN>::SMEM_BYTES, stream, *map_w, *map_act, a);
}

template <bool GATEUP, int BN>
cudaError_t prepare8_one() {
  return cudaFuncSetAttribute(expert_gemm_fp8_kernel<GATEUP, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              Cfg8<GATEUP, BN>::SMEM_BYTES);
}

template <bool GATEUP>
cudaError_t prepare8_all() {
  cudaError_t e;
  if ((e = prepare8_one<GATEUP, 16>()) != cudaSuccess) return e;
  if ((e = prepare8_one<GATEUP, 32>()) != cudaSuccess) return e;
  if ((e = prepare8_one<GATEUP, 64>()) != cudaSuccess) return e;
  return prepare8_one<GATEUP, 128>();
}

template <bool GATEUP>
cudaError_t dispatch8_bn(int tile_n, const CUtensorMap* map_w, const CUtensorMap* map_act, const GemmArgs& a,
                         int num_sms, cudaStream_t stream) {
  switch (tile_n) {
    case 16: return launch8_one<GATEUP, 16>(map_w, map_act, a, num_sms, stream);
    case 32: return launch8_one<GATEUP, 32>(map_w, map_act, a, num_sms, stream);
    case 64: return launch8_one<GATEUP, 64>(map_w, map_act, a, num_sms, stream);
    case 128: return launch8_one<GATEUP, 128>(map_w, map_act, a, num_sms, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

MOE_DBG_DEFINE_TAKE(dbg_take_expert_gemm_fp8)

cudaError_t launch_expert_gemm_fp8(bool gateup, int tile_n, const CUtensorMap* map_w, const CUtensorMap* map_act,
                                   const GemmArgs& a, int num_sms, cudaStream_t stream) {
  return gateup ? dispatch8_bn<true>(tile_n, map_w, map_act, a, num_sms, stream)
                : dispatch8_bn<false>(tile_n, map_w, map_act, a, num_sms, stream);
}

cudaError_t expert_gemm_fp8_prepare() {
  const cudaError_t e = prepare8_all<true>();
  return e != cudaSuccess ? e : prepare8_all<false>();
}

}  // namespace moe
