// Pieces shared by the one-CTA and the CTA-pair grouped expert GEMMs:
// work-item decoding over the groups' token tiles, bounded waits with a
// CTA-wide abort flag, and the two epilogues (SiLU gate for gate/up, gate
// weight scale for down) that read one TMEM accumulator of BN columns.
#pragma once
#include <cuda_fp16.h>

#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {
namespace gemm {

constexpr int kEpilogueWarp0 = 2;  // warps 2..5 are the epilogue
constexpr int kMaxGroups = kMaxExperts + 1;
constexpr uint64_t kDrainLimitNs = 2000000000ull;
constexpr uint32_t kEpilogueBar = 1;  // named barrier of the 4 epilogue warps

struct Item {
  int g, n, m;
};

// item -> (group, token tile inside the group, weight tile); tile_start[g] is
// the first token tile of group g (prefix over groups of ceil(rows/tile)).
// With `reverse` the items run from the last group to the first (the gate/up
// launch: the H rows it writes last are the first groups', which the down
// projection reads first).
__device__ __forceinline__ Item decode_item(int item, int m_tiles, const int* tile_start, int G, int n_items,
                                            int reverse) {
  if (reverse) item = n_items - 1 - item;
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

// tile_start[0..G] from the dispatch offsets, by one warp: lane l takes
// groups 32c + l; the tile counts of eight such runs of 32 groups are loaded
// together (coalesced, one load latency per eight runs), then each run is a
// warp prefix sum on top of the running total.
// With s_off (or NULL) the offsets[0..G] are also copied to shared memory,
// so that the roles of the kernel decode their items without a global load.
__device__ __forceinline__ void build_tile_start(const int* offsets, int G, int tile, int* tile_start, int lane,
                                                 int* s_off = nullptr) {
  constexpr int kRuns = 8;
  int carry = 0;
  for (int g0 = 0; g0 < G; g0 += 32 * kRuns) {
    int tiles[kRuns];
#pragma unroll
    for (int j = 0; j < kRuns; ++j) {
      const int g = g0 + 32 * j + lane;
      const int lo = g < G ? __ldg(offsets + g) : 0;
      const int hi = g < G ? __ldg(offsets + g + 1) : 0;
      tiles[j] = g < G ? (hi - lo + tile - 1) / tile : 0;
      if (s_off != nullptr && g < G) {
        s_off[g] = lo;
        if (g == G - 1) s_off[G] = hi;
      }
    }
#pragma unroll
    for (int j = 0; j < kRuns; ++j) {
      int incl = tiles[j];
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      const int g = g0 + 32 * j + lane;
      if (g < G) tile_start[g] = carry + incl - tiles[j];
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  if (lane == 0) tile_start[G] = carry;
}

// MMA width for a token tile with `valid` rows: the rows rounded up to a
// multiple of `step` (16 for one CTA and for a pair, 8 rows per CTA),
// at most the tile width.  Columns past it are neither loaded into the MMA
// nor computed; the epilogue only reads the valid columns.
__device__ __forceinline__ int mma_width(int valid, int step, int tile) {
  const int w = (valid + step - 1) / step * step;
  return w < tile ? w : tile;
}

// Instruction descriptor for work item `item` (M rows of weights, N = the
// item's token rows rounded up to `step`, at most `tile`); 0 past the last item.
__device__ __forceinline__ uint32_t item_idesc(int item, int n_items, int reverse, int m_tiles,
                                               const int* tile_start, int G, const int* offsets, int M, int step,
                                               int tile) {
  if (item >= n_items) return 0;
  const Item it = decode_item(item, m_tiles, tile_start, G, n_items, reverse);
  const int rows = offsets[it.g + 1] - offsets[it.g] - it.n * tile;  // global or shared memory
  return idesc_bf16_f32(M, mma_width(rows, step, tile));
}

// Debug builds: a tile's rows [row0, row0 + valid) inside the row buffers
// (a.rows_cap rows) and, for the down projection (chunk0 >= 0), its exponent
// chunks inside the exponent buffer (a.chunks_cap chunks); 0 valid rows
// (nothing stored) if not.  Release builds return `valid`.
__device__ __forceinline__ int checked_valid(const GemmArgs& a, int valid, int row0, int chunk0) {
  (void)a;
  (void)row0;
  (void)chunk0;
  return MOE_DBG_OK(valid > 0 && row0 >= 0 && row0 + valid <= a.rows_cap &&
                    (chunk0 < 0 || chunk0 + (valid + kYpRows - 1) / kYpRows <= a.chunks_cap))
             ? valid
             : 0;
}

// Weight group of row group g (expert parallelism maps (source, expert) row
// groups onto the local experts; otherwise the identity).
__device__ __forceinline__ int weight_group(const GemmArgs& a, int g) {
  return a.w_group_base + (a.w_group_mod ? g % a.w_group_mod : g);
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

// The epilogue warps' common wait on an accumulator: every warp waits, then
// all four take one decision (they meet at named barriers afterwards).
// s_ok is [2][4] ints, it_par alternates per item.  Returns false to abort.
// flag (or NULL): a yes/no of lane 0 of epilogue warp 0 (its `mine`), handed
// to all four warps through the same barrier.
__device__ __forceinline__ bool epilogue_wait(uint64_t* acc_full, uint32_t parity, uint64_t limit,
                                              volatile int* abort_flag, volatile int* s_ok, uint32_t& it_par,
                                              int q, int lane, uint32_t* err, int mine = 0, int* flag = nullptr) {
  const bool ok = __all_sync(0xffffffffu, wait_or_abort(acc_full, parity, limit, abort_flag));
  if (lane == 0) s_ok[it_par * 4 + q] = ok ? 1 + (q == 0 ? mine : 0) : 0;
  named_bar_sync(kEpilogueBar, 128);
  const bool all_ok = s_ok[it_par * 4 + 0] && s_ok[it_par * 4 + 1] && s_ok[it_par * 4 + 2] && s_ok[it_par * 4 + 3];
  if (flag != nullptr) *flag = s_ok[it_par * 4 + 0] == 2;
  it_par ^= 1u;
  if (!all_ok && lane == 0 && !ok) record_abort(abort_flag, err);
  return all_ok;
}

__device__ __forceinline__ bf16 to_out(float v, bf16*) { return __float2bfloat16_rn(v); }
__device__ __forceinline__ __half to_out(float v, __half*) { return __float2half_rn(v); }

// K3 epilogue over the `valid` columns of a BN-column accumulator whose TMEM
// rows 0..63 hold gate values and rows 64..127 the up values of the same 64
// features.  Gate-row threads keep columns 0..7 of each 16-column chunk and
// hand 8..15 to their up-row partner through xchg, which hands back 0..7;
// xchg is float4 [2 chunk parities][2 sides][2 halves][64 features], so the
// 32 lanes of a warp store and load 512 contiguous bytes per float4 (four
// shared-memory wavefronts, no bank conflicts).
// H[row0 + col][feat_base + (row & 63)] = silu(g) * u, where
// g and u are the accumulators times the `scale` of their own weight row (1
// for bf16 weights).  H is bf16 or fp16 (OutT).
// vals (or NULL): this thread's row of the accumulator, already summed over K
// parts, used in place of tensor memory.  rowmap (or NULL): the H row of each
// column in place of row0 + col (negative: the column is not stored).
template <int BN, typename OutT>
__device__ __forceinline__ void epilogue_gateup(uint32_t taddr, int row, int feat_base, int row0, int valid,
                                                OutT* H, int ldh, float* xchg, uint32_t& chunk_par,
                                                float scale = 1.0f, const float* vals = nullptr,
                                                const int* rowmap = nullptr) {
  const bool is_gate = row < 64;
  const int fl = row & 63;
  const int feat = feat_base + fl;
#pragma unroll
  for (int c0 = 0; c0 < BN; c0 += 16) {
    if (c0 >= valid) break;
    uint32_t v[16];
    if (vals != nullptr) {
#pragma unroll
      for (int c = 0; c < 16; ++c) v[c] = __float_as_uint(vals[c0 + c]);
    } else {
      tmem_ld16(taddr + c0, v);
      tmem_ld_wait();
    }
    float4* mine_out = reinterpret_cast<float4*>(xchg) + (chunk_par * 2 + (is_gate ? 1 : 0)) * 128 + fl;
    const float4* peer_in = reinterpret_cast<const float4*>(xchg) + (chunk_par * 2 + (is_gate ? 0 : 1)) * 128 + fl;
    float give[8], keep[8];  // compile-time register indices only
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      give[c] = scale * __uint_as_float(is_gate ? v[8 + c] : v[c]);
      keep[c] = scale * __uint_as_float(is_gate ? v[c] : v[8 + c]);
    }
    mine_out[0] = make_float4(give[0], give[1], give[2], give[3]);
    mine_out[64] = make_float4(give[4], give[5], give[6], give[7]);
    named_bar_sync(kEpilogueBar, 128);
    const float4 p0 = peer_in[0];
    const float4 p1 = peer_in[64];
    const float peer[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
    const int col0 = c0 + (is_gate ? 0 : 8);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const float h = is_gate ? silu_mul(keep[c], peer[c]) : silu_mul(peer[c], keep[c]);
      if (col0 + c < valid) {
        const int r = rowmap != nullptr ? rowmap[col0 + c] : row0 + col0 + c;
        if (r >= 0) H[static_cast<size_t>(r) * ldh + feat] = to_out(h, H);
      }
    }
    chunk_par ^= 1u;
  }
}

// Work units of one CTA of a persistent grouped GEMM: (item, K steps
// [kb0, kb1)), in the order the CTA's roles take them.
//   kWhole     whole items blockIdx.x, blockIdx.x + gridDim.x, ...
//   kEqualK    every item's K range in ks equal parts, the (item, part) pairs
//              dealt out the same way (part buffer slot = item * ks + part)
//   kBalanced  the launch's n_items * k_all K steps cut into gridDim.x
//              contiguous ranges of `per` steps, one per CTA: a unit is the
//              overlap of the CTA's range with one item, so every CTA streams
//              the same number of K steps whatever the item count.  The parts
//              of an item are the ranges its steps fall in (at most
//              kMaxGemmKSplit: per >= k_all / (kMaxGemmKSplit - 1)); only a
//              CTA's first and last units can be parts, so CTA c keeps them in
//              part buffer slots 2c and 2c + 1.
// A unit with parts > 1 stores its accumulator in slot `slot`; the item's
// arrival count lives at index slot0 (the slot of part 0).
enum UnitMode { kWhole = 0, kEqualK = 1, kBalanced = 2 };

struct WorkUnit {
  int item, kb0, kb1;
  int part, parts;
  int slot, slot0;
};

struct UnitCursor {
  int mode, k_all, ks, k_per, per, cta, stride;
  long long pos, end;

  __device__ __forceinline__ void init(int mode_, int n_items, int k_all_, int ks_) {
    mode = mode_;
    k_all = k_all_;
    ks = mode == kEqualK ? ks_ : 1;
    k_per = (k_all + ks - 1) / ks;
    cta = static_cast<int>(blockIdx.x);
    stride = static_cast<int>(gridDim.x);
    per = 1;
    if (mode == kBalanced) {
      const long long S = static_cast<long long>(n_items) * k_all;
      const long long even = (S + stride - 1) / stride;
      const int floor_per = (k_all + kMaxGemmKSplit - 2) / (kMaxGemmKSplit - 1);
      per = static_cast<int>(even > floor_per ? even : floor_per);
      pos = min(S, static_cast<long long>(cta) * per);
      end = min(S, static_cast<long long>(cta + 1) * per);
    } else {
      pos = cta;
      end = static_cast<long long>(n_items) * ks;
    }
  }
  // part buffer slot of CTA c's part of the item starting at K step i0
  __device__ __forceinline__ int slot_of(long long i0, int c) const {
    return 2 * c + (static_cast<long long>(c) * per < i0 ? 1 : 0);
  }
  __device__ __forceinline__ int part_slot(const WorkUnit& u, int p) const {
    if (mode != kBalanced) return u.slot0 + p;
    const long long i0 = static_cast<long long>(u.item) * k_all;
    return slot_of(i0, static_cast<int>(i0 / per) + p);
  }
  __device__ __forceinline__ bool next(WorkUnit& u) {
    if (pos >= end) return false;
    if (mode == kBalanced) {
      u.item = static_cast<int>(pos / k_all);
      const long long i0 = static_cast<long long>(u.item) * k_all;
      u.kb0 = static_cast<int>(pos - i0);
      u.kb1 = static_cast<int>(min(static_cast<long long>(k_all), end - i0));
      const int c0 = static_cast<int>(i0 / per), c1 = static_cast<int>((i0 + k_all - 1) / per);
      u.parts = c1 - c0 + 1;
      u.part = cta - c0;
      u.slot = slot_of(i0, cta);
      u.slot0 = slot_of(i0, c0);
      pos = i0 + u.kb1;
      return true;
    }
    const int idx = static_cast<int>(pos);
    pos += stride;
    u.item = idx / ks;
    u.part = idx - u.item * ks;
    u.parts = ks;
    u.kb0 = u.part * k_per;
    u.kb1 = min(k_all, u.kb0 + k_per);
    u.slot = idx;
    u.slot0 = u.item * ks;
    return true;
  }
};

// The parts of this thread's row of a unit's item (part p in slot
// cur.part_slot(u, p)), summed in part order; every part's 16 columns are
// loaded at once.
template <int BN>
__device__ __forceinline__ void ksplit_sum_units(const float* buf, const UnitCursor& cur, const WorkUnit& u, int row,
                                                 int valid, float (&sum)[BN]) {
  const float* src[kMaxGemmKSplit];
#pragma unroll
  for (int p = 0; p < kMaxGemmKSplit; ++p)
    src[p] = buf + (static_cast<size_t>(cur.part_slot(u, p < u.parts ? p : 0)) * kBlockM + row) * BN;
#pragma unroll
  for (int c0 = 0; c0 < BN; c0 += 16) {
    if (c0 >= valid) break;
    float4 f[kMaxGemmKSplit][4];
#pragma unroll
    for (int p = 0; p < kMaxGemmKSplit; ++p)
#pragma unroll
      for (int j = 0; j < 4; ++j)
        f[p][j] = p < u.parts ? __ldcg(reinterpret_cast<const float4*>(src[p] + c0 + 4 * j))
                              : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float4 a = f[0][j];
#pragma unroll
      for (int p = 1; p < kMaxGemmKSplit; ++p) {
        a.x += f[p][j].x;
        a.y += f[p][j].y;
        a.z += f[p][j].z;
        a.w += f[p][j].w;
      }
      sum[c0 + 4 * j] = a.x;
      sum[c0 + 4 * j + 1] = a.y;
      sum[c0 + 4 * j + 2] = a.z;
      sum[c0 + 4 * j + 3] = a.w;
    }
  }
}

// The same sum for the one part still in tensor memory (this thread's
// accumulator row at taddr, part u.part) when every other part is stored:
// the same values in the same order as ksplit_sum_units after storing it.
template <int BN>
__device__ __forceinline__ void ksplit_sum_units_own(const float* buf, const UnitCursor& cur, const WorkUnit& u,
                                                     int row, int valid, uint32_t taddr, float (&sum)[BN]) {
  const float* src[kMaxGemmKSplit];
#pragma unroll
  for (int p = 0; p < kMaxGemmKSplit; ++p)
    src[p] = buf + (static_cast<size_t>(cur.part_slot(u, p < u.parts ? p : 0)) * kBlockM + row) * BN;
#pragma unroll
  for (int c0 = 0; c0 < BN; c0 += 16) {
    if (c0 >= valid) break;
    uint32_t own[16];
    tmem_ld16(taddr + c0, own);
    float4 f[kMaxGemmKSplit][4];
#pragma unroll
    for (int p = 0; p < kMaxGemmKSplit; ++p)
#pragma unroll
      for (int j = 0; j < 4; ++j)
        f[p][j] = (p < u.parts && p != u.part)
                      ? __ldcg(reinterpret_cast<const float4*>(src[p] + c0 + 4 * j))
                      : make_float4(0.f, 0.f, 0.f, 0.f);
    tmem_ld_wait_regs(own);
#pragma unroll
    for (int p = 0; p < kMaxGemmKSplit; ++p)
      if (p == u.part)
#pragma unroll
        for (int j = 0; j < 4; ++j)
          f[p][j] = make_float4(__uint_as_float(own[4 * j]), __uint_as_float(own[4 * j + 1]),
                                __uint_as_float(own[4 * j + 2]), __uint_as_float(own[4 * j + 3]));
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float4 a = f[0][j];
#pragma unroll
      for (int p = 1; p < kMaxGemmKSplit; ++p) {
        a.x += f[p][j].x;
        a.y += f[p][j].y;
        a.z += f[p][j].z;
        a.w += f[p][j].w;
      }
      sum[c0 + 4 * j] = a.x;
      sum[c0 + 4 * j + 1] = a.y;
      sum[c0 + 4 * j + 2] = a.z;
      sum[c0 + 4 * j + 3] = a.w;
    }
  }
}

// K split (few work items: every item's K range in ks parts run as separate
// items).  ksplit_store_part: this thread's accumulator row of one part (the
// hi + lo sum when lo_off > 0) to the part buffer, the 16-column chunks that
// hold valid columns only.
template <int BN>
__device__ __forceinline__ void ksplit_store_part(uint32_t taddr, int lo_off, int valid, float* mine) {
#pragma unroll
  for (int c0 = 0; c0 < BN; c0 += 16) {
    if (c0 >= valid) break;
    uint32_t v[16], vl[16];
    tmem_ld16(taddr + c0, v);
    if (lo_off > 0) tmem_ld16(taddr + lo_off + c0, vl);
    tmem_ld_wait();
    float f[16];
#pragma unroll
    for (int c = 0; c < 16; ++c)
      f[c] = lo_off > 0 ? __uint_as_float(v[c]) + __uint_as_float(vl[c]) : __uint_as_float(v[c]);
#pragma unroll
    for (int c = 0; c < 16; c += 4)
      __stcg(reinterpret_cast<float4*>(mine + c0 + c), make_float4(f[c], f[c + 1], f[c + 2], f[c + 3]));
  }
}

// After every epilogue thread of the CTA stored its row of a part: one
// release (the cumulative fence after the barrier covers the other threads'
// rows) and the count of the item's finished parts.  True in every thread of
// the CTA that finished the item's last part (which then sees all parts).
__device__ __forceinline__ bool ksplit_arrive(int* cnt, int ks, volatile int* s_last, bool leader) {
  named_bar_sync(kEpilogueBar, 128);
  if (leader) {
    __threadfence();
    const int last = atomicAdd(cnt, 1) == ks - 1;
    if (last) __threadfence();  // acquire: the other parts' rows are visible
    *s_last = last;
  }
  named_bar_sync(kEpilogueBar, 128);
  return *s_last != 0;
}

// The ks parts of this thread's row (part p at src + p * 128 * BN), summed
// in part order; every part's 16 columns are loaded at once.
template <int BN>
__device__ __forceinline__ void ksplit_sum_parts(const float* src, int ks, int valid, float (&sum)[BN]) {
#pragma unroll
  for (int c0 = 0; c0 < BN; c0 += 16) {
    if (c0 >= valid) break;
    float4 f[kMaxGemmKSplit][4];
#pragma unroll
    for (int p = 0; p < kMaxGemmKSplit; ++p)
#pragma unroll
      for (int j = 0; j < 4; ++j)
        f[p][j] = p < ks ? __ldcg(reinterpret_cast<const float4*>(src + static_cast<size_t>(p) * kBlockM * BN + c0 +
                                                                   4 * j))
                         : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float4 a = f[0][j];
#pragma unroll
      for (int p = 1; p < kMaxGemmKSplit; ++p) {
        a.x += f[p][j].x;
        a.y += f[p][j].y;
        a.z += f[p][j].z;
        a.w += f[p][j].w;
      }
      sum[c0 + 4 * j] = a.x;
      sum[c0 + 4 * j + 1] = a.y;
      sum[c0 + 4 * j + 2] = a.z;
      sum[c0 + 4 * j + 3] = a.w;
    }
  }
}

// K4: the gate weight of every column of a tile, lane l holding columns
// l, l+32, ... (rows at dispatch positions >= Tk are shared-expert rows: 1).
template <int BN>
__device__ __forceinline__ void load_gate_weights(float (&wreg)[(BN + 31) / 32], int row0, int valid, int lane,
                                                  const int* perm, const float* prob, int Tk) {
#pragma unroll
  for (int i = 0; i < (BN + 31) / 32; ++i) {
    const int c = i * 32 + lane;
    const int pos = row0 + c;
    int a = -1;
    if (c < valid && pos < Tk && MOE_DBG_OK(pos >= 0)) {
      a = __ldg(perm + pos);
      if (!MOE_DBG_OK(a >= 0 && a < Tk)) a = -2;  // an assignment id outside [0, T*k)
    }
    wreg[i] = (c < valid) ? ((pos < Tk) ? (a >= 0 ? __ldg(prob + a) : 0.0f) : 1.0f) : 0.0f;
  }
}

// load_gate_weights in two phases, for fetching the next item's weights
// during this item's epilogue: gate_perm_entries loads the permutation entry
// of every column (-1: a shared-expert row, weight 1; -2: past the tile's
// valid columns, weight 0), gate_probs then the probabilities they point at.
template <int BN>
__device__ __forceinline__ void gate_perm_entries(int (&pe)[(BN + 31) / 32], int row0, int valid, int lane,
                                                  const int* perm, int Tk) {
#pragma unroll
  for (int i = 0; i < (BN + 31) / 32; ++i) {
    const int c = i * 32 + lane;
    const int pos = row0 + c;
    pe[i] = (c < valid && MOE_DBG_OK(pos >= 0)) ? ((pos < Tk) ? __ldg(perm + pos) : -1) : -2;
    if (pe[i] >= 0 && !MOE_DBG_OK(pe[i] < Tk)) pe[i] = -2;  // an assignment id outside [0, T*k)
  }
}

template <int BN>
__device__ __forceinline__ void gate_probs(float (&wreg)[(BN + 31) / 32], const int (&pe)[(BN + 31) / 32],
                                           const float* prob) {
#pragma unroll
  for (int i = 0; i < (BN + 31) / 32; ++i) wreg[i] = pe[i] >= 0 ? __ldg(prob + pe[i]) : (pe[i] == -1 ? 1.0f : 0.0f);
}

// Power-of-two exponent for a block of values whose largest magnitude has the
// fp32 bit pattern `amax`: 2^-e * amax lands in [2^14, 2^15), so every value of
// the block scaled by 2^-e is an fp16 normal or zero below 2^15 (no overflow)
// carrying 11 significant bits relative to the block's largest value.  Clamped
// to [-126, kYpExpMax] so that 2^-e and 2^e are fp32 normals.
// K3 epilogue for two-term E4M3 token rows: per 16-column chunk, the hi term
// (column c) + the lo term (column lo_off + c), times the weight row's scale
// and the token's 1/s (tok_scale of the dispatch row), then the gate/up
// exchange and h = silu(g) * u as in epilogue_gateup; H as fp16.
template <int BN>
__device__ __forceinline__ void epilogue_gateup_x2(uint32_t taddr, int row, int feat_base, int row0, int valid,
                                                   __half* H, int ldh, float* xchg, uint32_t& chunk_par,
                                                   float scale, const float* __restrict__ tok_scale, int lo_off,
                                                   const float* vals = nullptr) {
  const bool is_gate = row < 64;
  const int fl = row & 63;
  const int feat = feat_base + fl;
#pragma unroll
  for (int c0 = 0; c0 < BN; c0 += 16) {
    if (c0 >= valid) break;
    uint32_t vh[16], vl[16];
    if (vals != nullptr) {  // hi + lo already summed over the K parts
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        vh[c] = __float_as_uint(vals[c0 + c]);
        vl[c] = 0u;
      }
    } else {
      tmem_ld16(taddr + c0, vh);
      tmem_ld16(taddr + lo_off + c0, vl);
      tmem_ld_wait();
    }
    float v[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const float ts = (c0 + c < valid) ? __ldg(tok_scale + row0 + c0 + c) : 0.f;
      v[c] = (__uint_as_float(vh[c]) + __uint_as_float(vl[c])) * (scale * ts);
    }
    float4* mine_out = reinterpret_cast<float4*>(xchg) + (chunk_par * 2 + (is_gate ? 1 : 0)) * 128 + fl;
    const float4* peer_in = reinterpret_cast<const float4*>(xchg) + (chunk_par * 2 + (is_gate ? 0 : 1)) * 128 + fl;
    float give[8], keep[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      give[c] = is_gate ? v[8 + c] : v[c];
      keep[c] = is_gate ? v[c] : v[8 + c];
    }
    mine_out[0] = make_float4(give[0], give[1], give[2], give[3]);
    mine_out[64] = make_float4(give[4], give[5], give[6], give[7]);
    named_bar_sync(kEpilogueBar, 128);
    const float4 p0 = peer_in[0];
    const float4 p1 = peer_in[64];
    const float peer[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
    const int col0 = c0 + (is_gate ? 0 : 8);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const float h = is_gate ? silu_mul(keep[c], peer[c]) : silu_mul(peer[c], keep[c]);
      if (col0 + c < valid) H[static_cast<size_t>(row0 + col0 + c) * ldh + feat] = __float2half_rn(h);
    }
    chunk_par ^= 1u;
  }
}

__device__ __forceinline__ int block_exponent(uint32_t amax) {
  const int e = static_cast<int>((amax >> 23) & 0xffu) - 141;
  return e < -126 ? -126 : (e > kYpExpMax ? kYpExpMax : e);
}

// K4 epilogue: Yp[row0 + col][feat] = w_col * (row_scale * acc[col]) for the
// valid columns (row_scale: the weight row's scale, 1 for bf16 weights),
// stored scaled: the 16 columns of a chunk are kYpRows consecutive rows of the
// group, and this thread's feature over them forms one block; its exponent e
// (from the thread's own maximum, no exchange) goes to Ye[chunk0 + c0/16][feat]
// and the values to Y as fp16 of value * 2^-e.  chunk0 = the exponent chunk of
// the tile's first row (tile rows start at multiples of 16 inside the group).
// lo_off > 0: the accumulator holds two terms per column, at c and at
// lo_off + c (two-term E4M3 token rows), and acc[col] is their sum.
// One 16-column chunk of epilogue_down from its accumulator values acc[16].
template <int BN>
__device__ __forceinline__ void down_chunk(const float (&acc)[16], int c0, int feat, int row0, int valid,
                                           const float (&wreg)[(BN + 31) / 32], __half* Y, int8_t* Ye, int ldy,
                                           int chunk0, float row_scale) {
  float y[16];
  uint32_t amax = 0;
#pragma unroll
  for (int c = 0; c < 16; ++c) {
    const int col = c0 + c;
    y[c] = __shfl_sync(0xffffffffu, wreg[col >> 5], col & 31) * (row_scale * acc[c]);
    amax = max(amax, __float_as_uint(y[c]) & 0x7fffffffu);
  }
  const int e = block_exponent(amax);
  const float down = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);  // 2^-e, exact
  Ye[static_cast<size_t>(chunk0 + c0 / 16) * ldy + feat] = static_cast<int8_t>(e);
#pragma unroll
  for (int c = 0; c < 16; ++c)
    if (c0 + c < valid) Y[static_cast<size_t>(row0 + c0 + c) * ldy + feat] = __float2half_rn(y[c] * down);
}

// epilogue_down for one accumulator term read from tensor memory, with the
// next chunk's tensor-memory load in flight while a chunk is scaled and
// stored (the same arithmetic, chunk by chunk, as epilogue_down).
template <int BN>
__device__ __forceinline__ void epilogue_down_pipelined(uint32_t taddr, int feat, int row0, int valid,
                                                        const float (&wreg)[(BN + 31) / 32], __half* Y, int8_t* Ye,
                                                        int ldy, int chunk0, float row_scale = 1.0f) {
  static_assert(kYpRows == 16 && BN % 32 == 0, "16-column chunks, in pairs");
  uint32_t va[16], vb[16];
  tmem_ld16(taddr, va);
  tmem_ld_wait_regs(va);
#pragma unroll
  for (int c0 = 0; c0 < BN; c0 += 32) {
    if (c0 >= valid) break;
    const bool more_b = c0 + 16 < valid;
    if (more_b) tmem_ld16(taddr + c0 + 16, vb);
    float acc[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) acc[c] = __uint_as_float(va[c]);
    down_chunk<BN>(acc, c0, feat, row0, valid, wreg, Y, Ye, ldy, chunk0, row_scale);
    if (!more_b) break;
    tmem_ld_wait_regs(vb);
    const bool more_a = c0 + 32 < valid;
    if (more_a) tmem_ld16(taddr + c0 + 32, va);
#pragma unroll
    for (int c = 0; c < 16; ++c) acc[c] = __uint_as_float(vb[c]);
    down_chunk<BN>(acc, c0 + 16, feat, row0, valid, wreg, Y, Ye, ldy, chunk0, row_scale);
    if (!more_a) break;
    tmem_ld_wait_regs(va);
  }
}

template <int BN>
__device__ __forceinline__ void epilogue_down(uint32_t taddr, int feat, int row0, int valid,
                                              const float (&wreg)[(BN + 31) / 32], __half* Y, int8_t* Ye, int ldy,
                                              int chunk0, float row_scale = 1.0f, int lo_off = 0,
                                              const float* vals = nullptr) {
  static_assert(kYpRows == 16, "one exponent chunk per 16-column TMEM load");
#pragma unroll
  for (int c0 = 0; c0 < BN; c0 += 16) {
    if (c0 >= valid) break;
    uint32_t v[16], vl[16];
    if (vals != nullptr) {
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        v[c] = __float_as_uint(vals[c0 + c]);
        vl[c] = 0u;
      }
    } else {
      tmem_ld16(taddr + c0, v);
      if (lo_off > 0) tmem_ld16(taddr + lo_off + c0, vl);
      tmem_ld_wait();
    }
    float y[16];
    uint32_t amax = 0;
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const int col = c0 + c;
      const float acc = lo_off > 0 ? __uint_as_float(v[c]) + __uint_as_float(vl[c]) : __uint_as_float(v[c]);
      y[c] = __shfl_sync(0xffffffffu, wreg[col >> 5], col & 31) * (row_scale * acc);
      amax = max(amax, __float_as_uint(y[c]) & 0x7fffffffu);
    }
    const int e = block_exponent(amax);
    const float down = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);  // 2^-e, exact
    Ye[static_cast<size_t>(chunk0 + c0 / 16) * ldy + feat] = static_cast<int8_t>(e);
#pragma unroll
    for (int c = 0; c < 16; ++c)
      if (c0 + c < valid) Y[static_cast<size_t>(row0 + c0 + c) * ldy + feat] = __float2half_rn(y[c] * down);
  }
}

}  // namespace gemm
}  // namespace moe
