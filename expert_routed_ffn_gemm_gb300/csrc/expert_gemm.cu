// K3 / K4 — the experts of "Step3.5 Flash 大模型技术深度解析" (jsqmd.com) §3.2.1
// (each expert an independent FFN; one shared expert always on) run as grouped
// GEMMs over the dispatch order of §3.2.2, the shared expert being the last
// group:
//   gate/up (K3):  H[r, f]  = silu(X[r] . Wg[g, f]) * (X[r] . Wu[g, f])
//   down    (K4):  Yp[r, o] = w_r * (H[r] . Wd[g, o]),  w_r = the row's routing
//                  probability (1 for the shared expert); Yp is kept in fp32
// for every row r of group g.
//
// Design (sm_103a): a persistent, warp-specialised kernel, one CTA per SM.
// The weight matrix is the MMA's M operand (128 weight rows per tile) and the
// group's token rows are its N operand (16..256 columns), so that a decode-size
// group of a few tokens still streams whole 128-row weight tiles.
//   warp 0      TMA producer: weight tile(s) + token tile per K step into a
//               STAGES-deep shared-memory ring (128-byte swizzle)
//   warp 1      TMEM allocator + single-thread tcgen05.mma issuer; accumulators
//               live in tensor memory, double-buffered when they fit
//   warps 2..5  epilogue: tcgen05.ld, SiLU-gate (bf16 H) or gate-weight scale
//               (fp32 Yp)
// Work items are (group, token tile, weight tile) with the weight tile fastest,
// so the CTAs running at one time share a group's token rows in L2 while each
// weight tile is streamed from HBM once per token tile.  The per-group tile
// counts come from the device-resident dispatch offsets: no host round trip.
// Every wait is bounded (wait_limit_ns); on timeout the kernel records an error,
// drains the copies and MMAs it started, frees tensor memory and returns.
#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kThreads = 192;
constexpr int kEpilogueWarp0 = 2;
constexpr int kMaxGroups = kMaxExperts + 1;
constexpr uint64_t kDrainLimitNs = 2000000000ull;

template <bool GATEUP, int BN>
struct Cfg {
  static constexpr int A_BYTES = kBlockM * kBlockK * 2;  // one 128 x 64 bf16 weight tile
  static constexpr int NUM_A = GATEUP ? 2 : 1;           // gate + up tiles, or the down tile
  static constexpr int B_BYTES = BN * kBlockK * 2;       // BN x 64 bf16 token tile
  static constexpr int NUM_B = GATEUP ? 1 : 2;           // X rows, or the H_hi and H_lo rows
  static constexpr int STAGE_BYTES = NUM_A * A_BYTES + NUM_B * B_BYTES;  // multiple of 1024
  static constexpr int RING_BUDGET = 200 * 1024;
  static constexpr int STAGES_RAW = RING_BUDGET / STAGE_BYTES;
  static constexpr int STAGES = STAGES_RAW > 12 ? 12 : STAGES_RAW;
  static constexpr int ACC_COLS = GATEUP ? 2 * BN : BN;  // fp32 columns of one accumulator
  static constexpr int NACC = (2 * ACC_COLS <= 512) ? 2 : 1;
  static constexpr int TMEM_RAW = NACC * ACC_COLS;
  static constexpr int TMEM_COLS = TMEM_RAW <= 32 ? 32 : TMEM_RAW <= 64 ? 64 : TMEM_RAW <= 128 ? 128
                                                                       : TMEM_RAW <= 256 ? 256 : 512;
  // barriers: full[S], empty[S], acc_full[NACC], acc_empty[NACC], drain
  static constexpr int NUM_BARS = 2 * STAGES + 2 * NACC + 1;
  static constexpr int AUX_BYTES = NUM_BARS * 8 + 16 + (kMaxGroups + 1) * 4;
  static constexpr int SMEM_BYTES = 1024 /* alignment slack */ + STAGES * STAGE_BYTES + AUX_BYTES;
  static_assert(STAGE_BYTES % 1024 == 0, "stage must keep 1024-byte alignment");
  static_assert(STAGES >= 2, "ring too shallow");
  static_assert(SMEM_BYTES <= 232448, "exceeds shared memory per block");
  static constexpr uint32_t IDESC = idesc_bf16_f32(kBlockM, BN);
};

struct Item {
  int g, n, m;
};

// item -> (group, token tile inside the group, weight tile); tile_start[g] is
// the first token tile of group g (prefix over groups of ceil(rows/BN)).
__device__ __forceinline__ Item decode_item(int item, int m_tiles, const int* tile_start, int G) {
  Item it;
  const int tile = item / m_tiles;
  it.m = item - tile * m_tiles;
  int lo = 0, hi = G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tile_start[mid] <= tile)
      lo = mid;
    else
      hi = mid - 1;
  }
  it.g = lo;
  it.n = tile - tile_start[lo];
  return it;
}

__device__ __forceinline__ void record_abort(volatile int* abort_flag, uint32_t* err) {
  *abort_flag = 1;
  atomicOr(err, kErrWaitTimeout);
}

// Bounded wait that also gives up as soon as another role has aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, uint64_t limit_ns,
                                              volatile int* abort_flag) {
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

__device__ __forceinline__ float silu_mul(float g, float u) {
  return g * __frcp_rn(1.0f + __expf(-g)) * u;
}

template <bool GATEUP, int BN>
__global__ void __launch_bounds__(kThreads, 1)
    expert_gemm_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_act,
                       const __grid_constant__ CUtensorMap map_act2, const GemmArgs args) {
  using C = Cfg<GATEUP, BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
  uint64_t* full = bars;
  uint64_t* empty = bars + C::STAGES;
  uint64_t* acc_full = bars + 2 * C::STAGES;
  uint64_t* acc_empty = acc_full + C::NACC;
  uint64_t* drain = acc_empty + C::NACC;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + C::NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* tile_start = reinterpret_cast<int*>(tmem_holder + 4);

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
    tma_prefetch_desc(&map_act);
    if (!GATEUP) tma_prefetch_desc(&map_act2);
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, C::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == kEpilogueWarp0) {
    // tile_start[0..G]: each lane scans a contiguous run of groups
    const int per = (G + 31) / 32;
    const int b = lane * per, e = min(G, b + per);
    int local = 0;
    for (int g = b; g < e; ++g) {
      const int rows = __ldg(args.offsets + g + 1) - __ldg(args.offsets + g);
      local += (rows + BN - 1) / BN;
    }
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    int run = incl - local;
    for (int g = b; g < e; ++g) {
      tile_start[g] = run;
      const int rows = __ldg(args.offsets + g + 1) - __ldg(args.offsets + g);
      run += (rows + BN - 1) / BN;
    }
    if (lane == 31) tile_start[G] = incl;
  }
  tc_fence_before();
  __syncthreads();
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
      uint32_t stage = 0, phase = 0;
      long issued = 0;
      for (int item = blockIdx.x; item < n_items && !*abort_flag; item += gridDim.x) {
        const Item it = decode_item(item, args.m_tiles, tile_start, G);
        const int row_w = it.g * args.rows_per_group + it.m * kBlockM;
        const int row_act = __ldg(args.offsets + it.g) + it.n * BN;
        bool ok = true;
        for (int kb = 0; kb < k_steps; ++kb) {
          if (!wait_or_abort(&empty[stage], phase ^ 1u, limit, abort_flag)) {
            record_abort(abort_flag, args.err);
            ok = false;
            break;
          }
          uint8_t* st = ring + stage * C::STAGE_BYTES;
          mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
          tma_load_2d(st, &map_w, &full[stage], kb * kBlockK, row_w, pol_w);
          if (GATEUP) tma_load_2d(st + C::A_BYTES, &map_w, &full[stage], kb * kBlockK, row_w + args.F, pol_w);
          tma_load_2d(st + C::NUM_A * C::A_BYTES, &map_act, &full[stage], kb * kBlockK, row_act, pol_act);
          if (!GATEUP)
            tma_load_2d(st + C::NUM_A * C::A_BYTES + C::B_BYTES, &map_act2, &full[stage], kb * kBlockK, row_act,
                        pol_act);
          ++issued;
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
      }
      // Drain: the last load issued into each stage must have landed before
      // this CTA may exit (they always complete; the wait is bounded anyway).
      for (int s = 0; s < C::STAGES; ++s) {
        if (issued <= s) break;
        const long last = s + ((issued - 1 - s) / C::STAGES) * C::STAGES;
        const uint32_t par = static_cast<uint32_t>((last / C::STAGES) & 1);
        mbar_wait(&full[s], par, kDrainLimitNs);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // --------------------------------------------------------------- MMA --
      const int k_steps = args.K / kBlockK;
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool issued_any = false;
      for (int item = blockIdx.x; item < n_items && !*abort_flag; item += gridDim.x) {
        if (!wait_or_abort(&acc_empty[acc], acc_phase ^ 1u, limit, abort_flag)) {
          record_abort(abort_flag, args.err);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * C::ACC_COLS;
        bool ok = true;
        for (int kb = 0; kb < k_steps; ++kb) {
          if (!wait_or_abort(&full[stage], phase, limit, abort_flag)) {
            record_abort(abort_flag, args.err);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = smem_u32(ring + stage * C::STAGE_BYTES);
          const uint64_t a0 = smem_desc_sw128(st);
          const uint64_t a1 = smem_desc_sw128(st + C::A_BYTES);
          const uint64_t b = smem_desc_sw128(st + C::NUM_A * C::A_BYTES);
          const uint64_t b_lo = smem_desc_sw128(st + C::NUM_A * C::A_BYTES + C::B_BYTES);
#pragma unroll
          for (int kk = 0; kk < kBlockK / 16; ++kk) {
            const uint32_t accum = (kb > 0 || kk > 0) ? 1u : 0u;
            // +32 bytes along K inside the swizzle atom = +2 in the address field
            tc_mma_bf16(d_tmem, a0 + 2 * kk, b + 2 * kk, C::IDESC, accum);
            if (GATEUP) {
              tc_mma_bf16(d_tmem + BN, a1 + 2 * kk, b + 2 * kk, C::IDESC, accum);
            } else {
              // H = H_hi + H_lo: the low part goes into the same accumulator
              tc_mma_bf16(d_tmem, a0 + 2 * kk, b_lo + 2 * kk, C::IDESC, 1u);
            }
          }
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
        // every MMA of this CTA has finished before tensor memory is freed
        tc_commit(drain);
        mbar_wait(drain, 0, kDrainLimitNs);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue --
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;
    uint32_t acc = 0, acc_phase = 0;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
      const Item it = decode_item(item, args.m_tiles, tile_start, G);
      const int g_row0 = __ldg(args.offsets + it.g);
      const int g_rows = __ldg(args.offsets + it.g + 1) - g_row0;
      const int row0 = g_row0 + it.n * BN;
      const int valid = min(BN, g_rows - it.n * BN);
      // warp-uniform outcome: the tcgen05.ld below are .sync.aligned
      if (!__all_sync(0xffffffffu, wait_or_abort(&acc_full[acc], acc_phase, limit, abort_flag))) {
        if (lane == 0) record_abort(abort_flag, args.err);
        break;
      }
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * C::ACC_COLS;
      const int feat = it.m * kBlockM + row;
      for (int c0 = 0; c0 < BN && c0 < valid; c0 += 16) {
        uint32_t v[16];
        tmem_ld16(taddr + c0, v);
        if (GATEUP) {
          uint32_t u[16];
          tmem_ld16(taddr + BN + c0, u);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            if (c0 + c < valid) {
              const float h = silu_mul(__uint_as_float(v[c]), __uint_as_float(u[c]));
              const bf16 hi = __float2bfloat16_rn(h);
              const size_t o = static_cast<size_t>(row0 + c0 + c) * args.out_ld + feat;
              static_cast<bf16*>(args.out)[o] = hi;
              static_cast<bf16*>(args.out2)[o] = __float2bfloat16_rn(h - __bfloat162float(hi));
            }
          }
        } else {
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            if (c0 + c < valid) {
              const int pos = row0 + c0 + c;
              const float w = (pos < args.Tk) ? __ldg(args.prob + __ldg(args.perm + pos)) : 1.0f;
              static_cast<float*>(args.out)[static_cast<size_t>(pos) * args.out_ld + feat] =
                  w * __uint_as_float(v[c]);
            }
          }
        }
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
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

template <bool GATEUP, int BN>
cudaError_t launch_one(const CUtensorMap* map_w, const CUtensorMap* map_act, const CUtensorMap* map_act2,
                       const GemmArgs& a, int num_sms,
                       cudaStream_t stream) {
  using C = Cfg<GATEUP, BN>;
  expert_gemm_kernel<GATEUP, BN><<<num_sms, kThreads, C::SMEM_BYTES, stream>>>(*map_w, *map_act, *map_act2, a);
  return cudaGetLastError();
}

template <bool GATEUP, int BN>
cudaError_t prepare_one() {
  return cudaFuncSetAttribute(expert_gemm_kernel<GATEUP, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              Cfg<GATEUP, BN>::SMEM_BYTES);
}

template <bool GATEUP>
cudaError_t prepare_all() {
  cudaError_t e;
  if ((e = prepare_one<GATEUP, 16>()) != cudaSuccess) return e;
  if ((e = prepare_one<GATEUP, 32>()) != cudaSuccess) return e;
  if ((e = prepare_one<GATEUP, 64>()) != cudaSuccess) return e;
  if ((e = prepare_one<GATEUP, 128>()) != cudaSuccess) return e;
  return prepare_one<GATEUP, 256>();
}

template <bool GATEUP>
cudaError_t dispatch_bn(int tile_n, const CUtensorMap* map_w, const CUtensorMap* map_act, const CUtensorMap* map_act2,
                        const GemmArgs& a,
                        int num_sms, cudaStream_t stream) {
  switch (tile_n) {
    case 16: return launch_one<GATEUP, 16>(map_w, map_act, map_act2, a, num_sms, stream);
    case 32: return launch_one<GATEUP, 32>(map_w, map_act, map_act2, a, num_sms, stream);
    case 64: return launch_one<GATEUP, 64>(map_w, map_act, map_act2, a, num_sms, stream);
    case 128: return launch_one<GATEUP, 128>(map_w, map_act, map_act2, a, num_sms, stream);
    case 256: return launch_one<GATEUP, 256>(map_w, map_act, map_act2, a, num_sms, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <bool GATEUP>
int smem_bn(int tile_n) {
  switch (tile_n) {
    case 16: return Cfg<GATEUP, 16>::SMEM_BYTES;
    case 32: return Cfg<GATEUP, 32>::SMEM_BYTES;
    case 64: return Cfg<GATEUP, 64>::SMEM_BYTES;
    case 128: return Cfg<GATEUP, 128>::SMEM_BYTES;
    case 256: return Cfg<GATEUP, 256>::SMEM_BYTES;
    default: return -1;
  }
}

// A kernel that waits on a barrier nothing arrives at (bounded-wait self test).
__global__ void wait_selftest_kernel(uint32_t* err, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
    if (!mbar_wait(&bar, 0, limit_ns)) atomicOr(err, kErrWaitTimeout);
  }
}

}  // namespace

cudaError_t launch_expert_gemm(bool gateup, int tile_n, const CUtensorMap* map_w, const CUtensorMap* map_act,
                               const CUtensorMap* map_act2, const GemmArgs& a, int num_sms, cudaStream_t stream) {
  return gateup ? dispatch_bn<true>(tile_n, map_w, map_act, map_act2, a, num_sms, stream)
                : dispatch_bn<false>(tile_n, map_w, map_act, map_act2, a, num_sms, stream);
}

cudaError_t expert_gemm_prepare() {
  const cudaError_t e = prepare_all<true>();
  return e != cudaSuccess ? e : prepare_all<false>();
}

int expert_gemm_smem_bytes(bool gateup, int tile_n) { return gateup ? smem_bn<true>(tile_n) : smem_bn<false>(tile_n); }

cudaError_t launch_wait_selftest(uint32_t* err, unsigned long long limit_ns, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(err, limit_ns);
  return cudaGetLastError();
}

}  // namespace moe
