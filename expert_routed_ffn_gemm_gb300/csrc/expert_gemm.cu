// K3 / K4 — the experts of "Step3.5 Flash 大模型技术深度解析" (jsqmd.com) §3.2.1
// (each expert an independent FFN; one shared expert always on) run as grouped
// GEMMs over the dispatch order of §3.2.2, the shared expert being the last
// group:
//   gate/up (K3):  H[r, f]  = silu(X[r] . Wg[g, f]) * (X[r] . Wu[g, f])   (bf16)
//   down    (K4):  Yp[r, o] = w_r * (H[r] . Wd[g, o])   (fp32 accumulator)
// for every row r of group g, w_r = the row's routing probability (1 for the
// shared expert).  Yp is stored block-scaled: fp16 of Yp * 2^-e with one
// power-of-two exponent e per feature and 16-row chunk of a group (int8).
//
// Design (sm_103a): a persistent, warp-specialised kernel, one CTA per SM.
// The weights are the MMA's M operand (128 weight rows per tile) and the
// group's token rows its N operand (16..256 columns), so that a decode-size
// group of a few tokens still streams whole weight tiles at full width.
//   warp 0      TMA producer: one weight tile + one token tile per K step into
//               a STAGES-deep shared-memory ring (128-byte swizzle)
//   warp 1      TMEM allocator + single-thread tcgen05.mma issuer; two
//               accumulators in tensor memory so the epilogue of one work item
//               overlaps the MMAs of the next
//   warps 2..5  epilogue: tcgen05.ld, then the SiLU gate (K3) or the
//               gate-weight scale (K4), stores to global memory
// K3 builds each 128-row weight tile from 64 gate rows (tile rows 0..63) and the
// 64 up rows of the same features (rows 64..127), two TMA boxes of 64 rows, so
// one MMA produces both halves of the gate in one accumulator of N columns; the
// epilogue warps holding gate rows and those holding up rows swap half of each
// 16-column chunk through shared memory.
// Work items are (group, token tile, weight tile) with the weight tile fastest,
// so the CTAs running at one time share a group's token rows in L2 while each
// weight tile is streamed from HBM once per token tile.  The per-group tile
// counts come from the device-resident dispatch offsets: no host round trip.
// Every wait is bounded (wait_limit_ns); on timeout the kernel records an error,
// drains the copies and MMAs it started, frees tensor memory and returns.
#include "gemm_common.cuh"
#include "topk.cuh"

namespace moe {
namespace {

using namespace gemm;

constexpr int kThreads = 192;
constexpr int kPrefetchChunk = 64 * 1024;  // bytes per L2 prefetch instruction
constexpr int kRouteSlots = kMaxExperts / 32;                   // logits per lane, any E
constexpr int kRoutePicks = kSmallRouteMaxTokens * kMaxTopK;    // T*k picks at most
constexpr int kRouteAux = (4 * kRoutePicks + 4 * 16) * 4;      // their shared-memory tables

// The routing of a few tokens inside the gate/up launch (GemmArgs::route_logits):
// warp t ranks token t from its logits with the routing kernels' softmax and
// top-k (the same bits in every CTA), then every CTA works out the dispatch
// position of each pick a = t*k + j (the picks of experts below its own, then
// the earlier tokens that picked the same expert: the expert, token order of
// the dispatch) and the tile starts of the groups (each group with rows has
// one token tile: at most T*k + T rows).  CTA 0 also writes the routing and
// dispatch results where the routing kernels would.  Every thread of the CTA
// takes part (it calls __syncthreads).
__device__ void fused_route_prologue(const GemmArgs& a, int* tile_start, int* s_idx, float* s_prob, int* s_first,
                                     int* s_pos, int warp, int lane) {
  const int T = a.route_T, E = a.route_E, k = a.route_k, Tk = T * k;
  if (warp < T) {
    float q[kRouteSlots];
#pragma unroll
    for (int i = 0; i < kRouteSlots; ++i) {
      const int e = lane + 32 * i;
      q[i] = e < E ? __ldcg(a.route_logits + static_cast<size_t>(warp) * E + e) : 0.f;
    }
    finish_token<kRouteSlots>(q, warp, lane, E, k, a.route_renorm, s_idx, s_prob, nullptr, nullptr, nullptr, 0);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < Tk; i += blockDim.x) {
    const int e = s_idx[i];
    int first = 1, pos = 0;
    for (int i2 = 0; i2 < Tk; ++i2) {
      const int v = s_idx[i2];
      first &= (i2 >= i) | (v != e);
      pos += (v < e) | ((i2 < i) & (v == e));
    }
    s_first[i] = first;
    s_pos[i] = pos;
  }
  __syncthreads();
  for (int g = threadIdx.x; g <= a.G; g += blockDim.x) {
    int groups = 0;
    for (int i = 0; i < Tk; ++i) groups += (s_idx[i] < g) & s_first[i];
    tile_start[g] = groups + (g > E ? 1 : 0);  // the shared group (index E) has one tile
  }
  if (blockIdx.x == 0) {
    for (int i = threadIdx.x; i < Tk; i += blockDim.x) {
      a.route_idx[i] = s_idx[i];
      a.route_prob[i] = s_prob[i];
      a.route_perm[s_pos[i]] = i;
      a.route_inv[i] = s_pos[i];
    }
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      int below = 0, cnt = 0, groups = 0;
      for (int i = 0; i < Tk; ++i) {
        const int v = s_idx[i];
        below += v < e;
        cnt += v == e;
        groups += (v < e) & s_first[i];
      }
      a.route_offsets[e] = below;
      a.route_counts[e] = cnt;
      a.route_chunk_base[e] = groups;  // one exponent chunk per group with rows (fewer than 16 rows)
    }
    if (threadIdx.x == 0) {
      a.route_offsets[E] = Tk;
      a.route_offsets[E + 1] = Tk + (a.route_has_shared ? T : 0);
      a.route_chunk_base[E] = shared_chunk0(T, k, E);
      a.route_chunk_base[E + 1] = a.route_chunk_base[E] + (a.route_has_shared ? (T + kYpRows - 1) / kYpRows : 0);
    }
  }
  __syncthreads();
}

// The weights of the down launch's items blockIdx.x + w * gridDim.x (w <
// a.pf_waves) into L2: each item is 128 consecutive weight rows of one group,
// one contiguous block.  Items of a group's later token tiles read the same
// rows as its first and are skipped.  tile_start: this launch's token tiles,
// which the down launch shares.
__device__ __forceinline__ void prefetch_next_items(const GemmArgs& a, const int* tile_start, int G) {
  const int n_items = tile_start[G] * a.pf_m_tiles;
  const long long item_bytes = static_cast<long long>(kBlockM) * a.pf_row_bytes;
  const char* base = static_cast<const char*>(a.pf_w);
  int i = static_cast<int>(blockIdx.x);
  for (int w = 0; w < a.pf_waves && i < n_items; ++w, i += static_cast<int>(gridDim.x)) {
    const Item it = decode_item(i, a.pf_m_tiles, tile_start, G, n_items, 0);
    if (it.n > 0) continue;
    const long long row0 =
        static_cast<long long>(weight_group(a, it.g)) * a.pf_rows_per_group + static_cast<long long>(it.m) * kBlockM;
    const char* p = base + row0 * a.pf_row_bytes;
    for (long long o = 0; o < item_bytes; o += kPrefetchChunk)
      l2_prefetch_bulk(p + o, static_cast<uint32_t>(min(item_bytes - o, static_cast<long long>(kPrefetchChunk))));
  }
}

template <bool GATEUP, int BN>
struct Cfg {
  static constexpr int A_BYTES = kBlockM * kBlockK * 2;  // one 128 x 64 bf16 weight tile
  static constexpr int B_BYTES = BN * kBlockK * 2;       // BN x 64 bf16 token tile
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;  // multiple of 1024
  static constexpr int RING_BUDGET = 196 * 1024;
  static constexpr int STAGES_RAW = RING_BUDGET / STAGE_BYTES;
  static constexpr int STAGES = STAGES_RAW > 12 ? 12 : STAGES_RAW;
  static constexpr int NACC = 2;
  static constexpr int TMEM_RAW = NACC * BN;
  static constexpr int TMEM_COLS = TMEM_RAW <= 32 ? 32 : TMEM_RAW <= 64 ? 64 : TMEM_RAW <= 128 ? 128
                                                                       : TMEM_RAW <= 256 ? 256 : 512;
  // barriers: full[S], empty[S], acc_full[NACC], acc_empty[NACC], drain
  static constexpr int NUM_BARS = 2 * STAGES + 2 * NACC + 1;
  static constexpr int XCHG_BYTES = GATEUP ? 2 * 2 * 64 * 8 * 4 : 0;  // [parity][dir][64 f][8 cols] fp32
  static constexpr int AUX_BYTES = NUM_BARS * 8 + 16 + 32 + (kMaxGroups + 1) * 4 + (GATEUP ? kRouteAux : 0);
  static constexpr int SMEM_BYTES = 1024 /* alignment slack */ + STAGES * STAGE_BYTES + XCHG_BYTES + AUX_BYTES;
  static_assert(STAGE_BYTES % 1024 == 0, "stage must keep 1024-byte alignment");
  static_assert(STAGES >= 2, "ring too shallow");
  static_assert(SMEM_BYTES <= 232448, "exceeds shared memory per block");
  static constexpr uint32_t IDESC = idesc_bf16_f32(kBlockM, BN);
};

template <bool GATEUP, int BN>
__global__ void __launch_bounds__(kThreads, 1)
    expert_gemm_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_act,
                       const __grid_constant__ CUtensorMap map_act2, const GemmArgs args) {
  using C = Cfg<GATEUP, BN>;
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
  // gate/up with the routing in this launch: the picks, their weights,
  // first-of-expert flags and dispatch positions, and each epilogue warp's
  // map from token column to H row
  int* s_idx = tile_start + kMaxGroups + 1;
  float* s_prob = reinterpret_cast<float*>(s_idx + kRoutePicks);
  int* s_first = s_idx + 2 * kRoutePicks;
  int* s_pos = s_idx + 3 * kRoutePicks;
  int* s_rowmap = s_idx + 4 * kRoutePicks;  // [4 warps][16]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = args.G;
  const bool fused = GATEUP && BN <= 32 && args.route_logits != nullptr;

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
    if (args.act2_from >= 0) tma_prefetch_desc(&map_act2);
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, C::TMEM_COLS);
    tmem_relinquish();
  }
  pdl_wait();  // offsets, rows and outputs belong to earlier work in the stream until here
  if (fused)
    fused_route_prologue(args, tile_start, s_idx, s_prob, s_first, s_pos, warp, lane);
  else if (warp == kEpilogueWarp0)
    build_tile_start(args.offsets, G, BN, tile_start, lane);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int n_base = tile_start[G] * args.m_tiles;  // work items (group, token tile, weight tile)
  const int k_all = args.K / kBlockK;
  // K split (token tiles of at most 32 rows, few items): balanced ranges of K
  // steps when the host asks for them, else ksplit equal parts per item, as
  // long as the part buffer holds the parts; otherwise whole items
  int mode = kWhole;
  if (BN <= 32 && args.ksplit > 1) {
    if (args.kbalance && 2 * static_cast<int>(gridDim.x) <= args.ksplit_cap)
      mode = kBalanced;
    else if (!args.kbalance && n_base * args.ksplit <= args.ksplit_cap)
      mode = kEqualK;
  }
  const uint64_t limit = args.wait_limit_ns;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer --
      const uint64_t pol_w = policy_evict_first();   // weights: streamed once
      const uint64_t pol_act = policy_evict_last();  // token rows: re-read by the other weight tiles
      // K3: gate rows 64m.. of group g, then the up rows F + 64m..; K4: rows 128m..
      auto weight_row = [&](const Item& it) {
        return weight_group(args, it.g) * args.rows_per_group + it.m * (GATEUP ? kBlockM / 2 : kBlockM);
      };
      auto rows_of = [&](int item, int& row_w, int& row_act) {
        const Item it = decode_item(item, args.m_tiles, tile_start, G, n_base, args.reverse);
        row_w = weight_row(it);
        // routing in this launch: every group's tile is this CTA's copy of the T token rows
        row_act = fused ? static_cast<int>(blockIdx.x % max(1, args.route_replicas)) * args.route_T
                        : __ldg(args.offsets + it.g) + it.n * BN;
      };
      UnitCursor cur;
      cur.init(mode, n_base, k_all, args.ksplit);
      WorkUnit u, nu;
      bool has = cur.next(u);
      bool has_next = has && cur.next(nu);
      uint32_t stage = 0, phase = 0;
      long issued = 0;
      bool ok = true;
      int next_w = 0, next_act = 0;
      if (has) rows_of(u.item, next_w, next_act);
      while (ok && has && !*abort_flag) {
        const int row_w = next_w, row_act = next_act;
        for (int kb = u.kb0; kb < u.kb1; ++kb) {
          if (!wait_or_abort(&empty[stage], phase ^ 1u, limit, abort_flag)) {
            record_abort(abort_flag, args.err);
            ok = false;
            break;
          }
          uint8_t* st = ring + stage * C::STAGE_BYTES;
          mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
          tma_load_2d(st, &map_w, &full[stage], kb * kBlockK, row_w, pol_w);
          if (GATEUP) tma_load_2d(st + C::A_BYTES / 2, &map_w, &full[stage], kb * kBlockK, row_w + args.F, pol_w);
          if (args.act2_from >= 0 && row_act >= args.act2_from)
            tma_load_2d(st + C::A_BYTES, &map_act2, &full[stage], kb * kBlockK, row_act - args.act2_from, pol_act);
          else
            tma_load_2d(st + C::A_BYTES, &map_act, &full[stage], kb * kBlockK, row_act, pol_act);
          ++issued;
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
          // the next unit's rows, worked out while this unit's loads are in
          // flight (its offsets come from global memory)
          if (kb == u.kb0 && has_next) rows_of(nu.item, next_w, next_act);
        }
        u = nu;
        has = has_next;
        if (has) has_next = cur.next(nu);
      }
      // gate/up: every load of this CTA is issued; the down launch's first
      // weights stream in while the last stages, the epilogue and that
      // launch's start run
      if (GATEUP && ok && args.pf_w != nullptr && !*abort_flag) prefetch_next_items(args, tile_start, G);
      // Drain: the last load issued into each stage must have landed before
      // this CTA may exit (they always complete; the wait is bounded anyway).
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
      // N of the MMAs: the tile's rows rounded up to 16 (ragged tails); the
      // next unit's descriptor is worked out while this unit's MMAs run
      auto idesc_of = [&](int item) {
        if (fused) return item < n_base ? idesc_bf16_f32(kBlockM, mma_width(args.route_T, 16, BN)) : 0u;
        return item_idesc(item, n_base, args.reverse, args.m_tiles, tile_start, G, args.offsets, kBlockM, 16, BN);
      };
      UnitCursor cur;
      cur.init(mode, n_base, k_all, args.ksplit);
      WorkUnit u, nu;
      bool has = cur.next(u);
      bool has_next = has && cur.next(nu);
      uint32_t next_idesc = has ? idesc_of(u.item) : 0u;
      while (ok && has && !*abort_flag) {
        const uint32_t idesc = next_idesc;
        if (!wait_or_abort(&acc_empty[acc], acc_phase ^ 1u, limit, abort_flag)) {
          record_abort(abort_flag, args.err);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = u.kb0; kb < u.kb1; ++kb) {
          if (!wait_or_abort(&full[stage], phase, limit, abort_flag)) {
            record_abort(abort_flag, args.err);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = smem_u32(ring + stage * C::STAGE_BYTES);
          const uint64_t a = smem_desc_sw128(st);
          const uint64_t b = smem_desc_sw128(st + C::A_BYTES);
#pragma unroll
          for (int kk = 0; kk < kBlockK / 16; ++kk)  // +32 B along K = +2 in the address field
            tc_mma_bf16(d_tmem, a + 2 * kk, b + 2 * kk, idesc, (kb > u.kb0 || kk > 0) ? 1u : 0u);
          issued_any = true;
          tc_commit(&empty[stage]);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
          if (kb == u.kb0 && has_next) next_idesc = idesc_of(nu.item);
        }
        if (!ok) break;
        tc_commit(&acc_full[acc]);
        if (++acc == C::NACC) {
          acc = 0;
          acc_phase ^= 1u;
        }
        u = nu;
        has = has_next;
        if (has) has_next = cur.next(nu);
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
    uint32_t acc = 0, acc_phase = 0, it_par = 0, chunk_par = 0;
    volatile int* s_last = reinterpret_cast<volatile int*>(tmem_holder + 2);
    UnitCursor cur;
    cur.init(mode, n_base, k_all, args.ksplit);
    WorkUnit u;
    while (cur.next(u)) {
      const Item it = decode_item(u.item, args.m_tiles, tile_start, G, n_base, args.reverse);
      const int g_row0 = fused ? 0 : __ldg(args.offsets + it.g);
      const int g_rows = fused ? args.route_T : __ldg(args.offsets + it.g + 1) - g_row0;
      const int row0 = g_row0 + it.n * BN;
      const int chunk0 = GATEUP ? -1 : __ldg(args.chunk_base + it.g) + it.n * (BN / kYpRows);
      const int valid = checked_valid(args, min(BN, g_rows - it.n * BN), row0, chunk0);
      // routing in this launch: column t (token t) goes to the H row of token t's
      // pick of this group, or nowhere; the shared group's rows are T*k + t
      int* rowmap = nullptr;
      if (fused) {
        rowmap = s_rowmap + q * 16;
        __syncwarp();  // every lane has stored the previous item's columns
        if (lane < args.route_T) {
          const int k = args.route_k;
          int r = -1;
          if (it.g >= args.route_E) {
            r = args.route_T * k + lane;
          } else {
            for (int j = 0; j < k; ++j)
              if (s_idx[lane * k + j] == it.g) r = s_pos[lane * k + j];
          }
          rowmap[lane] = r;
        }
        __syncwarp();
      }
      // K4: the gate weight of every column, loaded while the MMAs still run
      float wreg[(BN + 31) / 32];
      if (!GATEUP) load_gate_weights<BN>(wreg, row0, valid, lane, args.perm, args.prob, args.Tk);
      // a part of a split item: if every other part is already stored (the
      // count, read before the wait, says so) this one is the last, and sums
      // the parts straight from tensor memory
      int others_done = 0;
      if (u.parts > 1 && q == 0 && lane == 0)
        others_done = ld_acquire_gpu(args.ksplit_cnt + u.slot0) == u.parts - 1;
      int fast = 0;
      if (!epilogue_wait(&acc_full[acc], acc_phase, limit, abort_flag, s_ok, it_par, q, lane, args.err, others_done,
                         &fast))
        break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
      if constexpr (BN <= 32) {
        if (u.parts > 1 && fast) {
          float sum[BN];
          ksplit_sum_units_own<BN>(args.ksplit_part, cur, u, row, valid, taddr, sum);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[acc]);
          if (++acc == C::NACC) {
            acc = 0;
            acc_phase ^= 1u;
          }
          if (GATEUP)
            epilogue_gateup<BN>(0u, row, it.m * (kBlockM / 2), row0, valid, static_cast<bf16*>(args.out),
                                args.out_ld, xchg, chunk_par, 1.0f, sum, rowmap);
          else
            epilogue_down<BN>(0u, it.m * kBlockM + row, row0, valid, wreg, static_cast<__half*>(args.out),
                              args.out_exp, args.out_ld, chunk0, 1.0f, 0, sum);
          if (q == 0 && lane == 0) args.ksplit_cnt[u.slot0] = 0;  // ready for the next launch
          continue;
        }
        if (u.parts > 1) {
          // this part's accumulator row to the part buffer, tensor memory back
          // to the MMA, then the last part of the item sums the parts in order
          ksplit_store_part<BN>(taddr, 0, valid,
                                args.ksplit_part + (static_cast<size_t>(u.slot) * kBlockM + row) * BN);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[acc]);
          if (++acc == C::NACC) {
            acc = 0;
            acc_phase ^= 1u;
          }
          if (ksplit_arrive(args.ksplit_cnt + u.slot0, u.parts, s_last, q == 0 && lane == 0)) {
            float sum[BN];
            ksplit_sum_units<BN>(args.ksplit_part, cur, u, row, valid, sum);
            if (GATEUP)
              epilogue_gateup<BN>(0u, row, it.m * (kBlockM / 2), row0, valid, static_cast<bf16*>(args.out),
                                  args.out_ld, xchg, chunk_par, 1.0f, sum, rowmap);
            else
              epilogue_down<BN>(0u, it.m * kBlockM + row, row0, valid, wreg, static_cast<__half*>(args.out),
                                args.out_exp, args.out_ld, chunk0,
                                1.0f, 0, sum);
            if (q == 0 && lane == 0) args.ksplit_cnt[u.slot0] = 0;  // ready for the next launch
          }
          continue;
        }
      }
      if (GATEUP) {
        // rows 0..63: gate of feature 64m + row; rows 64..127: up of feature 64m + row - 64
        epilogue_gateup<BN>(taddr, row, it.m * (kBlockM / 2), row0, valid, static_cast<bf16*>(args.out),
                            args.out_ld, xchg, chunk_par, 1.0f, nullptr, rowmap);
      } else {
        epilogue_down<BN>(taddr, it.m * kBlockM + row, row0, valid, wreg, static_cast<__half*>(args.out),
                          args.out_exp, args.out_ld, chunk0);
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
cudaError_t launch_one(const CUtensorMap* map_w, const CUtensorMap* map_act, const CUtensorMap* map_act2,
                       const GemmArgs& a, int num_sms, cudaStream_t stream) {
  return launch_chain(expert_gemm_kernel<GATEUP, BN>, dim3(num_sms), dim3(kThreads), Cfg<GATEUP, BN>::SMEM_BYTES,
                      stream, *map_w, *map_act, *map_act2, a);
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
                        const GemmArgs& a, int num_sms, cudaStream_t stream) {
  switch (tile_n) {
    case 16: return launch_one<GATEUP, 16>(map_w, map_act, map_act2, a, num_sms, stream);
    case 32: return launch_one<GATEUP, 32>(map_w, map_act, map_act2, a, num_sms, stream);
    case 64: return launch_one<GATEUP, 64>(map_w, map_act, map_act2, a, num_sms, stream);
    case 128: return launch_one<GATEUP, 128>(map_w, map_act, map_act2, a, num_sms, stream);
    case 256: return launch_one<GATEUP, 256>(map_w, map_act, map_act2, a, num_sms, stream);
    default: return cudaErrorInvalidValue;
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

MOE_DBG_DEFINE_TAKE(dbg_take_expert_gemm)

cudaError_t launch_expert_gemm(bool gateup, int tile_n, const CUtensorMap* map_w, const CUtensorMap* map_act,
                               const CUtensorMap* map_act2, const GemmArgs& a, int num_sms, cudaStream_t stream) {
  if (map_act2 == nullptr) map_act2 = map_act;
  return gateup ? dispatch_bn<true>(tile_n, map_w, map_act, map_act2, a, num_sms, stream)
                : dispatch_bn<false>(tile_n, map_w, map_act, map_act2, a, num_sms, stream);
}

cudaError_t expert_gemm_prepare() {
  const cudaError_t e = prepare_all<true>();
  return e != cudaSuccess ? e : prepare_all<false>();
}

cudaError_t launch_wait_selftest(uint32_t* err, unsigned long long limit_ns, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(err, limit_ns);
  return cudaGetLastError();
}

}  // namespace moe
