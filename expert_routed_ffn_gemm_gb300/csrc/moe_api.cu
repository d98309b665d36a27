// C ABI of libmoe.so (declared in include/moe.h): argument checks, workspace,
// TMA descriptors and the launch sequence of the layer of "Step3.5 Flash
// 大模型技术深度解析" (jsqmd.com) §3.2.1-§3.2.2:
//   router (K1) -> dispatch (K2) -> row scatter -> gate/up GEMM (K3)
//   -> down GEMM (K4) -> combine (K5),
// all enqueued on the caller's stream with no host synchronisation.
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstdio>
#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <array>
#include <mutex>
#include <new>
#include <vector>

#include "../../include/moe.h"
#include "kernels.cuh"

using moe::bf16;

constexpr int kProfStages = 6;
constexpr int kProfEvents = kProfStages + 1;
constexpr int kProfMaxCalls = 4096;
constexpr int kFusedGatherMaxTokens = 2;  // the few-token routing launch also copies the rows up to here
constexpr int kSharedOverlapMinTokens = 2048;  // the shared expert's gate/up on a second stream from here

struct moe_handle {
  uint32_t magic;
  moe_config cfg;
  moe_weights w;
  int device;
  int num_sms;
  int G;
  int tile_gateup;  // 0 = choose per call
  int tile_down;
  bool use_pairs;   // 256-row token tiles on CTA pairs (MOE_PAIR_TILES=0 turns it off)
  bool small_route; // routing and dispatch in one launch for a few tokens (MOE_SMALL_ROUTE=0 turns it off)
  // ... and with bf16 weights the top-k and dispatch in the gate/up launch
  // instead, which reads copies of the token rows (MOE_ROUTE_IN_GEMM=0 turns it off)
  bool route_in_gemm;
  // Many tokens: the shared expert's gate/up on a second stream, beside the
  // dispatch and the row scatter (MOE_SHARED_OVERLAP=0 turns it off)
  bool shared_overlap;
  cudaStream_t side = nullptr;
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
  bool fp8_x2;      // FP8 weights: gate/up on E4M3 tensor cores with two-term token rows (MOE_FP8_X2=0: off)
  int gemm_ksplit;  // K split of the bf16 expert GEMMs: -1 = by work items, 0 = balanced ranges forced,
                    // 1 = off, 2..4 = that many equal parts forced
  int pf_down_waves;  // waves of the down launch's items whose weights the single-CTA gate/up
                      // brings into L2 after its last load (MOE_PF_DOWN_WAVES; 0 = none)
  int ksplit_cap;   // work items (item, K part) the part buffer holds
  float* ksplit_part;  // [ksplit_cap][128][32] fp32 partial accumulators
  int* ksplit_cnt;     // [ksplit_cap] parts finished per item (zero between launches)
  int rows_max;     // R = (k+1)*Tmax dispatch rows the row buffer holds
  float* tok_scale; // [R] FP8 two-term token rows: 1/s of every dispatch row
  int router_tile;  // router token tile, 0 = by T (MOE_ROUTER_TILE = 16, 64, 128 or 256)
  int last_kernels;   // kernels enqueued by the last forward call
  bool fp8;           // E4M3 expert weights with per-row scales (moe_init_fp8)
  const float* s_gate_up;  // fp8: [G][2F] row scales
  const float* s_down;     // fp8: [G][d] row scales
  // expert parallelism (moe_ep_init): this rank owns routed experts
  // [ep_rank * e_loc, (ep_rank + 1) * e_loc); ep_size = 0 for a whole-layer handle
  int ep_size, ep_rank, e_loc, max_recv;
  int ep_T;                // tokens of the last moe_ep_dispatch
  int* ep_offsets;         // [ep_size * e_loc + 1] row offsets of the received (source, expert) groups
  int* ep_chunk_base;      // [ep_size * e_loc + 1] their exponent chunk bases
  int* ep_chunks_src;      // [ep_size] exponent chunks per source block
  int* ep_iota;            // [max_recv] 0, 1, 2, ... (received rows carry their own gate weight)
  unsigned long long wait_limit_ns;
  int router_m_tiles;      // ceil(E / 128)
  long long partial_rows;  // capacity of `partial` in (split, token) rows
  // workspace (one cudaMalloc)
  void* ws;
  int* counts;     // [E]
  int* chunk_hist; // [ceil(Tmax/256)][E] per-chunk rows per expert, then each chunk's first row
  float* partial;  // [partial_rows][E] router partial logits
  bf16* w3;        // [3][router_m_tiles*128][d] bf16 slices of W_r (hi, mid, lo)
  int* idx;        // [Tmax*k]
  float* prob;     // [Tmax*k]
  int* perm;       // [Tmax*k]
  int* inv;        // [Tmax*k]
  int* offsets;    // [E+2]
  void* yp;        // [(k+1)*Tmax][d] 16-bit: token rows in dispatch order (bf16), then the expert
                   // outputs (fp16, block-scaled by yexp)
  int8_t* yexp;    // [(k+1)*Tmax/16 + E + 2][d] exponents of the expert outputs (per feature and
                   // chunk of 16 rows of a group)
  int* chunk_base; // [E+2] first exponent chunk of each group
  bf16* hbuf;      // [(k+1)*Tmax][F] H
  bf16* x_stage;   // [Tmax][d] (host entry point)
  void* y_stage;   // [Tmax][d] bf16 or fp32 (host entry point)
  uint32_t* err;   // device error word
  unsigned int* route_done;  // arrival count of the few-token routing kernel, zero between launches
  float* tokstats; // [Tmax][kMaxStatGroups + 1] per-token group masses and entropy
  CUtensorMap map_w3;                   // W_r slices as [3*e_pad][d], box 64 x 128
  CUtensorMap map_wgu;                  // W_gu as [G*2F][d], box 64 x 64
  CUtensorMap map_wd;                   // W_d  as [G*d][F], box 64 x 128
                                        // (fp8: E4M3 bytes, boxes 128 x 64 / 128 x 128)
  CUtensorMap map_xp[moe::kNumTileN];   // Xp   as [Rmax][d] bf16 (in yp), box 64 x BN
  CUtensorMap map_h[moe::kNumTileN];    // H    as [Rmax][F], box 64 x BN
  CUtensorMap map_xq[moe::kNumTileN];   // FP8 two-term token rows as [2*Rmax][d] bytes, box 128 B x BN
  CUtensorMap map_hq[moe::kNumTileN];   // FP8 two-term H rows as [Rmax][2F] bytes (hi | lo), box 128 B x BN
  // per-stage timing (moe_profile_enable)
  bool profiling;
  int n_prof;
  std::vector<std::array<cudaEvent_t, kProfEvents>> prof;
};

namespace {

constexpr uint32_t kMagic = 0x4d6f4531u;  // "MoE1"
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;
constexpr int kPrefetchDownWaves = 1;  // default of MOE_PF_DOWN_WAVES

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool load_encode() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

// 2-D bf16 tensor map over a row-major [rows][cols] matrix, box = 64 columns
// (128 bytes, the swizzle width) x box_rows rows, 128-byte swizzle.
// 2-D row-major map with the 128-byte swizzle: 16-bit elements (box 64
// columns) or, with bytes = true, 8-bit codes (box 128 columns).
bool encode_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
               bool bytes = false) {
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * (bytes ? 1 : 2)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(bytes ? 128 : moe::kBlockK), box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, bytes ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                        const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool is_device_ptr(const void* p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged;
}

bool valid_handle(const moe_handle* h) { return h != nullptr && h->magic == kMagic; }

int tile_from_env(const char* name) {
  const char* v = std::getenv(name);
  if (!v) return 0;
  const int t = std::atoi(v);
  for (int i = 0; i < moe::kNumTileN; ++i)
    if (moe::kTileN[i] == t) return t;
  return 0;
}

int tile_index(int tile_n) {
  for (int i = 0; i < moe::kNumTileN; ++i)
    if (moe::kTileN[i] == tile_n) return i;
  return -1;
}

// Token-tile width for a mean of `mean_rows` rows per routed expert: the
// smallest width that holds a typical group in one tile, at most `cap`.
// Token tile width: the smallest listed width (from min_tile on) that holds
// the mean rows per group times `slack`, at most cap.  The MMAs' N follows
// each tile's actual rows (rounded up to 16), so a wider tile costs mostly its
// shared-memory ring depth (measured on GB300, one call each):
//  - bf16 weights, decode (3.6 rows per group): 32-row tiles (9 ring stages)
//    2.7-2.9 % faster than 16-row tiles (10 stages); 512 tokens (14 rows):
//    64-row tiles 1.3 % faster than 32-row ones;
//  - FP8 two-term kernel (N = 2 x tile): 64-row tiles at 2048 tokens (57 rows)
//    6 % faster than 128-row ones (4 stages of 48 KB).
int choose_tile(double mean_rows, int cap, int min_tile, double slack = 1.15) {
  for (int i = 0; i < moe::kNumTileN; ++i) {
    if (moe::kTileN[i] < min_tile) continue;
    if (moe::kTileN[i] >= cap || mean_rows * slack <= moe::kTileN[i]) return moe::kTileN[i];
  }
  return cap;
}

// MOE_TRACE_ERRORS=1 in the environment: every failing CUDA call is reported
// on stderr with its source line and error name.
bool trace_errors() {
  static const bool on = [] {
    const char* v = std::getenv("MOE_TRACE_ERRORS");
    return v != nullptr && v[0] == '1';
  }();
  return on;
}

int cuda_failed(cudaError_t e, const char* what, int line) {
  if (trace_errors()) std::fprintf(stderr, "moe: line %d: %s -> %s\n", line, what, cudaGetErrorName(e));
  return MOE_ERR_CUDA;
}

#define MOE_CUDA(call)                                   \
  do {                                                   \
    const cudaError_t moe_e_ = (call);                   \
    if (moe_e_ != cudaSuccess) {                         \
      return cuda_failed(moe_e_, #call, __LINE__);       \
    }                                                    \
  } while (0)

// Every call on a handle runs with the handle's device current in the calling
// thread (and puts the previous device back): a thread that has not used CUDA
// yet gets the device's primary context before the first driver call (the
// tensor-map encoding), and a caller working on another device is unaffected.
struct DeviceGuard {
  int prev = -1, dev;
  explicit DeviceGuard(int d) : dev(d) {
    if (cudaGetDevice(&prev) != cudaSuccess) {
      cudaGetLastError();
      prev = -1;
    }
    if (cudaSetDevice(dev) != cudaSuccess) cudaGetLastError();
  }
  ~DeviceGuard() {
    if (prev >= 0 && prev != dev) cudaSetDevice(prev);
  }
  DeviceGuard(const DeviceGuard&) = delete;
  DeviceGuard& operator=(const DeviceGuard&) = delete;
};

int check_call(const moe_handle* h, const void* x, int T) {
  if (!valid_handle(h)) return MOE_ERR_INVALID_ARG;
  if (T < 0) return MOE_ERR_INVALID_ARG;
  if (T > h->cfg.max_tokens) return MOE_ERR_TOO_MANY_TOKENS;
  if (T > 0 && (x == nullptr || !aligned(x, 16))) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

// Per-call routing choice: k experts per token (<= the handle's top_k) and
// whether the k weights are renormalised to sum to 1.
struct CallOpts {
  int k;
  int renorm;
};

// The shared expert's gate/up and down weights (pointers and bytes), or
// nothing without a shared expert: a layer call reads them whatever the
// routing, so the routing kernels prefetch them into L2.
void shared_weights(const moe_handle* h, const void* (&p)[2], long long (&n)[2]) {
  const moe_config& c = h->cfg;
  p[0] = p[1] = nullptr;
  n[0] = n[1] = 0;
  if (!c.has_shared) return;
  const size_t wb = h->fp8 ? 1 : 2, F = c.ffn_width, d = c.d_model, E = c.n_experts;
  p[0] = static_cast<const char*>(h->w.w_gate_up) + E * 2 * F * d * wb;
  n[0] = static_cast<long long>(2 * F * d * wb);
  p[1] = static_cast<const char*>(h->w.w_down) + E * d * F * wb;
  n[1] = static_cast<long long>(d * F * wb);
}

// K1: router GEMM (K split across CTAs when there are few token tiles) and
// softmax/top-k into idx/prob/gap, counts per expert; with tokstats, the
// per-token group masses and entropy for the routing statistics.
int enqueue_shared_ffn_side(moe_handle* h, const void* x, int T, int k, cudaStream_t s);

int enqueue_router(moe_handle* h, const void* x, int T, CallOpts o, int* idx, float* prob, float* gap,
                   float* tokstats, int n_groups, cudaStream_t s, bool prefetch_shared = false,
                   bool fork_shared = false) {
  const moe_config& c = h->cfg;
  // many tokens: the counts come from per-chunk histograms after the top-k
  // kernel (no atomics); otherwise the top-k kernel counts into zeroed counts
  const bool chunked = moe::chunked_dispatch(T);
  if (!chunked) MOE_CUDA(cudaMemsetAsync(h->counts, 0, sizeof(int) * c.n_experts, s));
  if (T == 0) return MOE_OK;
  const int bn = h->router_tile ? h->router_tile : (T <= 32 ? 16 : (T <= 1024 ? 64 : (T <= 4096 ? 128 : 256)));
  const int n_tt = (T + bn - 1) / bn;
  const int k_total = c.d_model / moe::kBlockK;  // K steps, each with the three weight slices
  // K splits: up to about two waves of work items, the count that fills the
  // waves best (the fewest splits among equals: every split adds a partial
  // logit pass).  At 8192 tokens this is 3 splits of 288 items on 152 SMs
  // (measured, with each slice's K steps in their own split: 8 us faster
  // than 6 and 14 us faster than 1).
  const int base_items = n_tt * h->router_m_tiles;
  const int ks_cap = std::min(moe::kMaxKSplit, std::max(1, (2 * h->num_sms + base_items - 1) / base_items));
  int ks = 1;
  double best = 0.0;
  for (int cand = 1; cand <= ks_cap; ++cand) {
    const long long items = static_cast<long long>(cand) * base_items;
    const long long waves = (items + h->num_sms - 1) / h->num_sms;
    const double fill = static_cast<double>(items) / static_cast<double>(waves * h->num_sms);
    if (fill > best + 0.02) {
      best = fill;
      ks = cand;
    }
  }
  ks = ks > k_total ? k_total : ks;
  while (ks > 1 && static_cast<long long>(ks) * T > h->partial_rows) --ks;
  // every split must own at least one K step: ks = ceil(k_total / ceil(k_total / ks))
  const int k_per = (k_total + ks - 1) / ks;
  ks = (k_total + k_per - 1) / k_per;
  CUtensorMap map_x;
  if (!encode_2d(&map_x, x, static_cast<uint64_t>(T), static_cast<uint64_t>(c.d_model), bn)) return MOE_ERR_CUDA;
  moe::RouterGemmArgs ra{};
  ra.partial = h->partial;
  ra.err = h->err;
  ra.wait_limit_ns = h->wait_limit_ns;
  ra.T = T;
  ra.d = c.d_model;
  ra.E = c.n_experts;
  ra.e_pad = h->router_m_tiles * moe::kBlockM;
  ra.m_tiles = h->router_m_tiles;
  ra.ksplit = ks;
  if (prefetch_shared) shared_weights(h, ra.pf, ra.pf_bytes);
  MOE_CUDA(moe::launch_router_gemm(bn, &h->map_w3, &map_x, ra, h->num_sms, s));
  if (fork_shared) {
    const int rc = enqueue_shared_ffn_side(h, x, T, o.k, s);
    if (rc != MOE_OK) return rc;
  }
  MOE_CUDA(moe::launch_router_topk(h->partial, ks, T, c.n_experts, o.k, o.renorm, idx, prob, gap,
                                   chunked ? nullptr : h->counts, tokstats, n_groups, s));
  if (chunked) MOE_CUDA(moe::launch_chunk_counts(idx, T, c.n_experts, o.k, h->chunk_hist, h->counts, s));
  return MOE_OK;
}

// K1 + K2 into the given buffers.
// A few tokens: K1 and K2 in one launch (the few-token routing kernel).
bool small_route(const moe_handle* h, int T) {
  return h->small_route && moe::route_small_fits(T, h->cfg.d_model, h->cfg.n_experts);
}

// Copies of the T token rows the routing launch writes to the row buffer
// when the gate/up launch finishes the routing (its CTAs read them round
// robin): up to 16, as many as the buffer's rows hold, one per block of the
// routing launch (a block per expert).
int token_replicas(const moe_handle* h, int T) {
  return std::max(1, std::min({16, h->rows_max / T, h->cfg.n_experts}));
}

int enqueue_route(moe_handle* h, const void* x, int T, CallOpts o, int* idx, float* prob, int* perm, int* offsets,
                  float* gap, cudaStream_t s) {
  const moe_config& c = h->cfg;
  if (small_route(h, T)) {
    MOE_CUDA(moe::launch_route_small(static_cast<const bf16*>(x), h->w.w_router, T, c.d_model, c.n_experts, o.k,
                                     o.renorm, c.has_shared, h->partial, h->route_done, idx, prob, gap, h->counts,
                                     offsets, perm, h->inv, h->chunk_base, moe::SmallRouteExtras{}, s));
    return MOE_OK;
  }
  const int rc = enqueue_router(h, x, T, o, idx, prob, gap, nullptr, 0, s);
  if (rc != MOE_OK) return rc;
  MOE_CUDA(moe::launch_dispatch(idx, h->counts, T, c.n_experts, o.k, c.has_shared, offsets, perm, h->inv,
                                h->chunk_base, h->chunk_hist, s));
  return MOE_OK;
}

// Options of a call: NULL = the handle's top_k, no renormalisation.
int resolve_opts(const moe_handle* h, const moe_call_options* opt, CallOpts* o) {
  o->k = h->cfg.top_k;
  o->renorm = 0;
  if (opt == nullptr) return MOE_OK;
  if (opt->top_k < 0 || opt->top_k > h->cfg.top_k) return MOE_ERR_INVALID_ARG;
  if (opt->renormalize != 0 && opt->renormalize != 1) return MOE_ERR_INVALID_ARG;
  if (opt->top_k > 0) o->k = opt->top_k;
  o->renorm = opt->renormalize;
  return MOE_OK;
}

// Event slot of this call when profiling (nullptr otherwise).
cudaEvent_t* prof_slot(moe_handle* h) {
  if (!h->profiling || h->n_prof >= kProfMaxCalls) return nullptr;
  if (h->n_prof == static_cast<int>(h->prof.size())) {
    std::array<cudaEvent_t, kProfEvents> ev{};
    for (auto& e : ev)
      if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    h->prof.push_back(ev);
  }
  return h->prof[h->n_prof++].data();
}

#define MOE_MARK(i) \
  if (ev) MOE_CUDA(cudaEventRecord(ev[i], s))

// K parts for a single-CTA bf16 or two-term E4M3 expert GEMM with token tile
// bn (k_steps: its pipeline stages along K, 16 KB of weights each).  The work
// items (weight tiles x token tiles, at most items_ub) run in waves over the
// SMs; with few items the last wave leaves SMs idle and cutting every item's
// K range into ks parts evens the load.  Estimated time: waves of part items
// x (K steps per part + a fixed cost per item worth kItemSteps K steps, which
// covers the pipeline start and the part reduction); the split is taken when
// it beats the unsplit estimate by 5 %.  Unforced, only K ranges of at least
// kMinSplitSteps steps are cut (shorter ones gain too little).  The bf16
// kernel (balanced != NULL) instead takes balanced ranges where they are
// estimated no slower: the K steps of all items in one contiguous range per
// CTA, estimated as the range's steps + kItemSteps per unit it runs;
// *balanced = 1 then.
int choose_ksplit(const moe_handle* h, int bn, long long items_ub, int k_steps, int* balanced = nullptr) {
  if (balanced != nullptr) *balanced = 0;
  if ((h->fp8 && !h->fp8_x2) || bn > 32 || h->gemm_ksplit == 1 || items_ub <= 0) return 1;
  constexpr int kMinSplitSteps = 32;
  constexpr int kBalancedMaxWaves = 20;
  const int sms = h->num_sms;
  auto fits = [&](int ks) {  // every part has a K step and the part buffer room
    return (ks - 1) * ((k_steps + ks - 1) / ks) < k_steps && items_ub * ks <= h->ksplit_cap;
  };
  if (h->gemm_ksplit >= 2) return fits(h->gemm_ksplit) ? h->gemm_ksplit : 1;
  if (h->gemm_ksplit == 0) {  // balanced ranges forced (bf16 kernel only)
    if (balanced == nullptr || 2 * sms > h->ksplit_cap) return 1;
    *balanced = 1;
    return moe::kMaxGemmKSplit;
  }
  // E4M3 items carry half the bytes of bf16 ones, so the fixed cost per part
  // outweighs the fuller last wave (T=1 gate/up: 31 us unsplit, 37 and 43 us
  // in 2 and 3 parts): split only when forced
  if (h->fp8 || k_steps < kMinSplitSteps) return 1;
  constexpr double kItemSteps = 8.0;
  auto cost = [&](int ks) {
    return static_cast<double>((items_ub * ks + sms - 1) / sms) * (static_cast<double>(k_steps) / ks + kItemSteps);
  };
  const double base = cost(1);
  if (balanced != nullptr && 2 * sms <= h->ksplit_cap) {
    // one contiguous range of K steps per CTA: the most steps any CTA streams,
    // plus the fixed cost of each unit it runs (its range starts and ends
    // inside items)
    const long long S = items_ub * k_steps;
    const long long per = std::max<long long>((S + sms - 1) / sms, (k_steps + moe::kMaxGemmKSplit - 2) /
                                                                       (moe::kMaxGemmKSplit - 1));
    const double bal = static_cast<double>(per) + static_cast<double>((per + k_steps - 1) / k_steps + 1) * kItemSteps;
    // taken where the estimate is no worse, up to kBalancedMaxWaves waves of
    // items (flash shape, gate/up, forced against unsplit: 4 tokens 119 ->
    // 108 us, 8 tokens 186 -> 184 us, 16 tokens 329 -> 327 us; 32 and 64
    // tokens about 1 % slower)
    if (bal <= base && items_ub <= kBalancedMaxWaves * sms) {
      *balanced = 1;
      return moe::kMaxGemmKSplit;
    }
    return 1;
  }
  int best = 1;
  double best_cost = base;
  for (int ks = 2; ks <= moe::kMaxGemmKSplit && fits(ks); ++ks) {
    if (cost(ks) < best_cost) {
      best = ks;
      best_cost = cost(ks);
    }
  }
  return best_cost < 0.95 * base ? best : 1;
}

// Token-tile widths and the CTA-pair choice of a grouped FFN call (mean_rows:
// mean rows per group; n_rows: the call's rows when known), and the arguments
// both of its GEMMs share.
struct FfnPlan {
  int bn1, bn2;        // token tiles of gate/up and down
  bool pair1, pair2;   // 256-row tiles on CTA pairs
  long long rows;      // rows of the call (estimated from mean_rows when not known)
};

FfnPlan plan_ffn(moe_handle* h, moe::GemmArgs& a, double mean_rows, int n_rows) {
  const moe_config& c = h->cfg;
  FfnPlan p;
  const int cap = h->fp8 ? 128 : 256;
  const int min_tile = (h->fp8 && !h->fp8_x2) || (!h->fp8 && mean_rows >= 8.0) ? 64 : 32;
  const double slack = h->fp8_x2 ? 1.0 : 1.15;
  p.bn1 = h->tile_gateup ? std::min(h->tile_gateup, cap) : choose_tile(mean_rows, cap, min_tile, slack);
  p.bn2 = h->tile_down ? std::min(h->tile_down, cap) : choose_tile(mean_rows, cap, min_tile, slack);
  p.pair1 = h->use_pairs && p.bn1 == 256;
  p.pair2 = h->use_pairs && p.bn2 == 256 && c.d_model % 256 == 0;
  a.err = h->err;
  a.wait_limit_ns = h->wait_limit_ns;
  a.F = c.ffn_width;
  // bounds of the debug build's checks: the rows of this call when known
  // (every row block lies below them), else the row buffers' capacity
  a.rows_cap = n_rows > 0 ? n_rows : h->rows_max;
  a.chunks_cap = std::max(a.rows_cap, h->rows_max) / moe::kYpRows + c.n_experts + 2;
  a.ksplit_part = h->ksplit_part;
  a.ksplit_cnt = h->ksplit_cnt;
  a.ksplit_cap = h->ksplit_cap;
  p.rows = n_rows > 0 ? n_rows : std::llround(mean_rows * a.G);
  return p;
}

// token tiles: at most one per group that has rows plus rows / bn
long long tiles_ub(const moe::GemmArgs& a, const FfnPlan& p, int bn) {
  return std::min<long long>(a.G, p.rows) + p.rows / bn;
}

// The single-CTA gate/up brings into L2, once its loads are issued, the
// weights of the first h->pf_down_waves waves of items of the down launch
// after it (see GemmArgs::pf_w), when that launch deals whole items of the
// same token tiles and has at most two waves of them.  Flash shape, one token
// (288 down items on 152 SMs): down 24.4 -> 22.4 us, the layer call about
// 1.5 us faster; from two tokens on (3.6 and more waves) the prefetch only
// takes bandwidth from the gate/up's last loads: 1-2 us slower per call.
void set_down_prefetch(const moe_handle* h, moe::GemmArgs& a, const FfnPlan& p) {
  const moe_config& c = h->cfg;
  if (h->pf_down_waves <= 0 || p.pair2 || p.bn2 != p.bn1) return;
  const long long items = tiles_ub(a, p, p.bn2) * (c.d_model / moe::kBlockM);
  int balanced = 0;
  if (items > 2LL * h->num_sms ||
      choose_ksplit(h, p.bn2, items, c.ffn_width / moe::kBlockK, &balanced) != 1)
    return;
  a.pf_w = h->w.w_down;
  a.pf_waves = h->pf_down_waves;
  a.pf_m_tiles = c.d_model / moe::kBlockM;
  a.pf_rows_per_group = c.d_model;
  a.pf_row_bytes = c.ffn_width * 2;
}

// K3: gate/up from the rows behind map_rows (one map per tile width), rows
// from a.act2_from on from rows2 [n_rows2][d], into H.
int enqueue_gateup(moe_handle* h, moe::GemmArgs a, double mean_rows, const CUtensorMap* map_rows, cudaEvent_t* ev,
                   cudaStream_t s, const void* rows2, int n_rows2, int n_rows) {
  const moe_config& c = h->cfg;
  const FfnPlan p = plan_ffn(h, a, mean_rows, n_rows);
  CUtensorMap map2;
  const CUtensorMap* map_act2 = nullptr;
  if (a.route_logits != nullptr) {
    // the routing finishes in this launch: every group's token tile is a
    // copy of the T token rows in the row buffer (written by the routing launch)
    if (h->fp8 || p.pair1 || p.bn1 > 32) return MOE_ERR_UNSUPPORTED;
    a.act2_from = -1;
  } else if (a.act2_from >= 0 && rows2 != nullptr && !h->fp8) {
    if (!encode_2d(&map2, rows2, static_cast<uint64_t>(n_rows2), static_cast<uint64_t>(c.d_model),
                   p.pair1 ? 128u : static_cast<uint32_t>(p.bn1)))
      return MOE_ERR_CUDA;
    map_act2 = &map2;
  } else {
    a.act2_from = -1;
  }
  // gate/up runs its items last group first, so the H rows it writes last are
  // those of the first groups, which the down projection (first group first)
  // then reads while they are still in L2
  a.reverse = 1;
  a.out = h->hbuf;
  a.K = c.d_model;
  a.rows_per_group = 2 * c.ffn_width;
  a.m_tiles = p.pair1 ? c.ffn_width / moe::kBlockM : c.ffn_width / (moe::kBlockM / 2);
  a.out_ld = c.ffn_width;
  const int i1 = tile_index(p.bn1), i128 = tile_index(128);
  a.w_scale = h->s_gate_up;
  a.ksplit = 1;
  a.kbalance = 0;
  if (h->fp8_x2) {
    a.tok_scale = h->tok_scale;
    a.lo_row0 = h->rows_max;
    a.lo_col0 = 0;
    a.ksplit = choose_ksplit(h, p.bn1, tiles_ub(a, p, p.bn1) * a.m_tiles, a.K / moe::kKStepE4M3);
    MOE_CUDA(moe::launch_expert_gemm_fp8x(true, p.bn1, &h->map_wgu, &h->map_xq[i1], a, h->num_sms, s));
  } else if (h->fp8)
    MOE_CUDA(moe::launch_expert_gemm_fp8(true, p.bn1, &h->map_wgu, &map_rows[i1], a, h->num_sms, s));
  else if (p.pair1)
    MOE_CUDA(moe::launch_expert_gemm_pair(true, &h->map_wgu, &map_rows[i128], map_act2, a, h->num_sms, s));
  else {
    // the second stream's launches run beside the first's: no K split there
    // (one part buffer)
    if (s != h->side) {
      a.ksplit = choose_ksplit(h, p.bn1, tiles_ub(a, p, p.bn1) * a.m_tiles, a.K / moe::kBlockK, &a.kbalance);
      set_down_prefetch(h, a, p);
    }
    MOE_CUDA(moe::launch_expert_gemm(true, p.bn1, &h->map_wgu, &map_rows[i1], map_act2, a, h->num_sms, s));
  }
  MOE_MARK(4);
  return MOE_OK;
}

// K4: down from H into yout (fp16, scaled) and yexp.
int enqueue_down(moe_handle* h, moe::GemmArgs a, double mean_rows, void* yout, int8_t* yexp, cudaEvent_t* ev,
                 cudaStream_t s, int n_rows) {
  const moe_config& c = h->cfg;
  const FfnPlan p = plan_ffn(h, a, mean_rows, n_rows);
  a.route_logits = nullptr;  // the gate/up launch has finished the routing
  a.reverse = 0;
  a.act2_from = -1;
  a.out = yout;
  a.out_exp = yexp;
  a.K = c.ffn_width;
  a.rows_per_group = c.d_model;
  a.m_tiles = p.pair2 ? c.d_model / (2 * moe::kBlockM) : c.d_model / moe::kBlockM;
  a.out_ld = c.d_model;
  a.w_scale = h->s_down;
  a.ksplit = 1;
  a.kbalance = 0;
  const int i2 = tile_index(p.bn2), i128 = tile_index(128);
  if (h->fp8_x2) {
    // H in place as two-term E4M3 rows, their 1/s in tok_scale (gate/up has
    // read the token scales by now)
    MOE_CUDA(moe::launch_requant_rows_x2(h->hbuf, n_rows, c.ffn_width, h->tok_scale, s));
    a.tok_scale = h->tok_scale;
    a.lo_row0 = 0;
    a.lo_col0 = c.ffn_width;
    a.ksplit = choose_ksplit(h, p.bn2, tiles_ub(a, p, p.bn2) * a.m_tiles, a.K / moe::kKStepE4M3);
    MOE_CUDA(moe::launch_expert_gemm_fp8x(false, p.bn2, &h->map_wd, &h->map_hq[i2], a, h->num_sms, s));
  } else if (h->fp8)
    MOE_CUDA(moe::launch_expert_gemm_fp8(false, p.bn2, &h->map_wd, &h->map_h[i2], a, h->num_sms, s));
  else if (p.pair2)
    MOE_CUDA(moe::launch_expert_gemm_pair(false, &h->map_wd, &h->map_h[i128], nullptr, a, h->num_sms, s));
  else {
    if (s != h->side)
      a.ksplit = choose_ksplit(h, p.bn2, tiles_ub(a, p, p.bn2) * a.m_tiles, a.K / moe::kBlockK, &a.kbalance);
    MOE_CUDA(moe::launch_expert_gemm(false, p.bn2, &h->map_wd, &h->map_h[i2], nullptr, a, h->num_sms, s));
  }
  MOE_MARK(5);
  return MOE_OK;
}

// The grouped FFN over the row groups of `a` (offsets, G, perm/prob/Tk for
// the gate weights, chunk_base, weight-group mapping): gate/up from the rows
// behind map_rows (one map per tile width) into H, then down into yout (fp16)
// and yexp.  mean_rows: mean rows per group (picks the token tile width).
// ev (or NULL): profiling events around the two GEMMs.
int enqueue_ffn(moe_handle* h, moe::GemmArgs a, double mean_rows, const CUtensorMap* map_rows, void* yout,
                int8_t* yexp, cudaEvent_t* ev, cudaStream_t s, const void* rows2 = nullptr, int n_rows2 = 0,
                int n_rows = 0) {
  const int rc = enqueue_gateup(h, a, mean_rows, map_rows, ev, s, rows2, n_rows2, n_rows);
  if (rc != MOE_OK) return rc;
  return enqueue_down(h, a, mean_rows, yout, yexp, ev, s, n_rows);
}

// The shared expert may run on the second stream: bf16 weights and its
// launches on CTA pairs (they take its rows from the host, not the offsets).
bool shared_overlap_ok(const moe_handle* h) {
  return h->shared_overlap && h->use_pairs && !h->fp8 && (h->tile_gateup == 0 || h->tile_gateup == 256) &&
         (h->tile_down == 0 || h->tile_down == 256);
}

// The shared expert's FFN on the handle's second stream: it needs x alone,
// so it runs on CTA pairs beside the routing's later kernels, the dispatch
// and the row copy (which use few tensor cores): gate/up into rows
// [T*k, T*k + T) of H, then down into the same rows of Yp and the exponent
// chunks from shared_chunk0 on (where the dispatch places them); ev_join
// marks its end.
int enqueue_shared_ffn_side(moe_handle* h, const void* x, int T, int k, cudaStream_t s) {
  const moe_config& c = h->cfg;
  MOE_CUDA(cudaEventRecord(h->ev_fork, s));
  MOE_CUDA(cudaStreamWaitEvent(h->side, h->ev_fork, 0));
  moe::GemmArgs sa{};
  sa.offsets = nullptr;  // one group, rows [T*k, T*k + T): known here
  sa.off_const[0] = T * k;
  sa.off_const[1] = T * k + T;
  sa.G = 1;
  sa.perm = h->perm;
  sa.prob = h->prob;
  sa.Tk = T * k;
  sa.w_group_base = c.n_experts;
  sa.act2_from = T * k;
  int rc = enqueue_gateup(h, sa, static_cast<double>(T), h->map_xp, nullptr, h->side, x, T, T * k + T);
  if (rc != MOE_OK) return rc;
  sa.chunk_base = nullptr;
  sa.chunk_const = moe::shared_chunk0(T, k, c.n_experts);
  rc = enqueue_down(h, sa, static_cast<double>(T), h->yp, h->yexp, nullptr, h->side, T * k + T);
  if (rc != MOE_OK) return rc;
  MOE_CUDA(cudaEventRecord(h->ev_join, h->side));
  return MOE_OK;
}

int enqueue_forward(moe_handle* h, const void* x, int T, CallOpts o, void* y, cudaStream_t s) {
  const moe_config& c = h->cfg;
  cudaEvent_t* ev = prof_slot(h);
  MOE_MARK(0);
  const bool fused_route = small_route(h, T);
  const bool overlap_shared = shared_overlap_ok(h) && c.has_shared && !fused_route && T >= kSharedOverlapMinTokens;
  const double mean_rows = static_cast<double>(T) * o.k / c.n_experts;
  const int n_rows = T * o.k + (c.has_shared ? T : 0);
  // bf16 weights, one CTA per SM and token tiles of at most 32 rows: the
  // few-token routing launch writes the logits (and copies of the token
  // rows) only, and the gate/up launch ranks the tokens, lays out the
  // dispatch and reads the rows from the copies (flash shape, three A/B
  // rounds against the routing launch doing it all: 1 token 0.0688 ->
  // 0.0683 ms, 2 tokens 0.1097 -> 0.1070, 3 tokens 0.1451 -> 0.1437, 4 tokens
  // 0.1723 -> 0.1714)
  bool route_in_gemm = false;
  if (fused_route && h->route_in_gemm && !h->fp8) {
    moe::GemmArgs probe{};
    const FfnPlan p = plan_ffn(h, probe, mean_rows, n_rows);
    route_in_gemm = !p.pair1 && p.bn1 <= 32;
  }
  // with one or two tokens (bf16 weights) that launch also copies the routed
  // rows into dispatch order (a handful of rows: one block is enough)
  const bool fused_gather = fused_route && !h->fp8 && !route_in_gemm && T <= kFusedGatherMaxTokens;
  if (fused_route) {
    moe::SmallRouteExtras ex{};
    const void* pf[2];
    long long pfn[2];
    shared_weights(h, pf, pfn);  // read by every call: into L2 while routing
    if (!route_in_gemm) {  // (a launch that stops at its logits ends before the prefetch could help)
      ex.pf0 = pf[0];
      ex.pf0_bytes = pfn[0];
      ex.pf1 = pf[1];
      ex.pf1_bytes = pfn[1];
    }
    ex.xp = fused_gather || route_in_gemm ? h->yp : nullptr;
    ex.logits_only = route_in_gemm ? 1 : 0;
    ex.replicas = route_in_gemm ? token_replicas(h, T) : 0;
    MOE_CUDA(moe::launch_route_small(static_cast<const bf16*>(x), h->w.w_router, T, c.d_model, c.n_experts, o.k,
                                     o.renorm, c.has_shared, h->partial, h->route_done, h->idx, h->prob, nullptr,
                                     h->counts, h->offsets, h->perm, h->inv, h->chunk_base, ex, s));
    MOE_MARK(1);
  } else {
    // many tokens: the shared expert's FFN forks off after the router GEMM
    // (see enqueue_shared_ffn_side), joined back before the combine
    const int rc = enqueue_router(h, x, T, o, h->idx, h->prob, nullptr, nullptr, 0, s, true, overlap_shared);
    if (rc != MOE_OK) return rc;
    MOE_MARK(1);
    MOE_CUDA(moe::launch_dispatch(h->idx, h->counts, T, c.n_experts, o.k, c.has_shared, h->offsets, h->perm, h->inv,
                                  h->chunk_base, h->chunk_hist, s));
  }
  MOE_MARK(2);
  // token rows in dispatch order (the yp buffer holds them until the down
  // GEMM).  bf16 weights: the routed rows only — the shared expert's rows are
  // x itself, which its gate/up reads directly.  fp8 weights: every row, as
  // fp16 (the tensor cores' input type there).
  const bool shared_from_x = !h->fp8 && c.has_shared;
  if (h->fp8_x2)
    MOE_CUDA(moe::launch_scatter_x2(static_cast<const bf16*>(x), h->inv, T, o.k, c.d_model, c.has_shared,
                                    static_cast<uint8_t*>(h->yp), h->rows_max, h->tok_scale, s));
  else if (!fused_gather && !route_in_gemm)
    MOE_CUDA(moe::launch_gather(static_cast<const bf16*>(x), h->inv, T, o.k, c.d_model,
                                shared_from_x ? 0 : c.has_shared, h->yp, h->fp8, s));
  MOE_MARK(3);
  moe::GemmArgs a{};
  a.offsets = h->offsets;
  a.perm = h->perm;
  a.prob = h->prob;
  a.G = h->G;
  a.Tk = T * o.k;
  a.chunk_base = h->chunk_base;
  a.act2_from = shared_from_x ? T * o.k : -1;
  if (route_in_gemm) {
    a.route_logits = h->partial;
    a.route_replicas = token_replicas(h, T);
    a.route_T = T;
    a.route_E = c.n_experts;
    a.route_k = o.k;
    a.route_renorm = o.renorm;
    a.route_has_shared = c.has_shared;
    a.route_idx = h->idx;
    a.route_prob = h->prob;
    a.route_counts = h->counts;
    a.route_offsets = h->offsets;
    a.route_perm = h->perm;
    a.route_inv = h->inv;
    a.route_chunk_base = h->chunk_base;
  }
  if (overlap_shared) a.G = c.n_experts;  // the routed groups; the shared one runs on the second stream
  if (int rc2 = enqueue_gateup(h, a, mean_rows, h->map_xp, ev, s, x, T, n_rows)) return rc2;
  if (int rc2 = enqueue_down(h, a, mean_rows, h->yp, h->yexp, ev, s, n_rows)) return rc2;
  if (overlap_shared) MOE_CUDA(cudaStreamWaitEvent(s, h->ev_join, 0));  // the shared expert's Yp rows
  MOE_CUDA(moe::launch_combine(static_cast<const __half*>(h->yp), h->yexp, nullptr, nullptr, h->idx, h->inv,
                               h->offsets, h->chunk_base, T, o.k, c.n_experts, c.d_model, c.has_shared, y, c.out_fp32,
                               s));
  MOE_MARK(6);
  // router GEMM, top-k, dispatch, gather, gate/up, down, combine; many
  // tokens: two more for the chunk histograms and their scan, and two more
  // for the shared expert's gate/up and down on the second stream; a few tokens:
  // routing and dispatch in one (bf16 weights: the logits and the row
  // copies, the rest in the gate/up launch; else with one or two tokens also
  // the gather); FP8 two-term rows: one more for the requantisation of H
  h->last_kernels = (fused_route ? (fused_gather || route_in_gemm ? 4 : 5) : moe::chunked_dispatch(T) ? 9 : 7) +
                    (h->fp8_x2 ? 1 : 0) + (overlap_shared ? 2 : 0);
  return MOE_OK;
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

void release_streams(moe_handle* h) {
  if (h->ev_fork) cudaEventDestroy(h->ev_fork);
  if (h->ev_join) cudaEventDestroy(h->ev_join);
  if (h->side) cudaStreamDestroy(h->side);
  h->ev_fork = h->ev_join = nullptr;
  h->side = nullptr;
}

}  // namespace

extern "C" {

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_TOO_MANY_TOKENS: return "T exceeds max_tokens of the handle";
    case MOE_ERR_UNSUPPORTED: return "unsupported layer shape";
    case MOE_ERR_CUDA: return "CUDA call failed";
    case MOE_ERR_DEVICE: return "a kernel reported a failure (pipeline wait limit exceeded)";
    case MOE_ERR_NO_DEVICE: return "no compute capability 10.3 (GB300) device is current";
    default: return "unknown status";
  }
}

}  // extern "C"

namespace {

// moe_init and moe_init_fp8: w holds the router and the two expert weight
// arrays (bf16, or E4M3 codes when s_gu / s_d, the row scales, are given).
struct EpParams {
  int size = 0, rank = 0, max_recv = 0;  // size 0: not expert-parallel
};

int init_any(const moe_config* cfg, const moe_weights* w, const float* s_gu, const float* s_d, moe_handle** out,
             EpParams ep = EpParams()) {
  if (out == nullptr) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  if (cfg == nullptr || w == nullptr) return MOE_ERR_INVALID_ARG;
  const bool fp8 = s_gu != nullptr;
  const moe_config c = *cfg;
  if (ep.size != 0) {
    if (ep.size < 1 || ep.rank < 0 || ep.rank >= ep.size || ep.max_recv < 0 || c.n_experts <= 0)
      return MOE_ERR_INVALID_ARG;
    if (c.n_experts % ep.size != 0 || fp8 || ep.max_recv > (1 << 26)) return MOE_ERR_UNSUPPORTED;
  }
  if (c.d_model <= 0 || c.n_experts <= 0 || c.top_k <= 0 || c.ffn_width <= 0 || c.max_tokens <= 0)
    return MOE_ERR_INVALID_ARG;
  if (c.has_shared != 0 && c.has_shared != 1) return MOE_ERR_INVALID_ARG;
  if (c.out_fp32 != 0 && c.out_fp32 != 1) return MOE_ERR_INVALID_ARG;
  if (c.d_model % 128 != 0 || c.ffn_width % 128 != 0 || c.n_experts > moe::kMaxExperts ||
      c.top_k > c.n_experts || c.top_k > moe::kMaxTopK || c.max_tokens > (1 << 20))
    return MOE_ERR_UNSUPPORTED;
  if (static_cast<long long>(c.top_k + 1) * c.max_tokens >= (1ll << 31)) return MOE_ERR_UNSUPPORTED;
  if (w->w_router == nullptr || w->w_gate_up == nullptr || w->w_down == nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned(w->w_router, 16) || !aligned(w->w_gate_up, 16) || !aligned(w->w_down, 16))
    return MOE_ERR_INVALID_ARG;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_NO_DEVICE;
  }
  int major = 0, minor = 0, sms = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_NO_DEVICE;
  }
  if (major != 10 || minor != 3) return MOE_ERR_NO_DEVICE;
  if (!is_device_ptr(w->w_router) || !is_device_ptr(w->w_gate_up) || !is_device_ptr(w->w_down))
    return MOE_ERR_INVALID_ARG;
  if (fp8 && (!aligned(s_gu, 4) || !aligned(s_d, 4) || !is_device_ptr(s_gu) || !is_device_ptr(s_d)))
    return MOE_ERR_INVALID_ARG;
  if (!load_encode()) return MOE_ERR_CUDA;
  if (moe::expert_gemm_prepare() != cudaSuccess || moe::expert_gemm_pair_prepare() != cudaSuccess ||
      moe::router_gemm_prepare() != cudaSuccess || moe::expert_gemm_fp8_prepare() != cudaSuccess ||
      moe::expert_gemm_fp8x_prepare() != cudaSuccess)
    return MOE_ERR_CUDA;

  moe_handle* h = new (std::nothrow) moe_handle();
  if (h == nullptr) return MOE_ERR_CUDA;
  h->cfg = c;
  h->w = *w;
  h->fp8 = fp8;
  h->s_gate_up = s_gu;
  h->s_down = s_d;
  h->device = dev;
  h->num_sms = sms;
  h->G = c.n_experts + c.has_shared;
  h->ep_size = ep.size;
  h->ep_rank = ep.rank;
  h->e_loc = ep.size ? c.n_experts / ep.size : c.n_experts;
  h->max_recv = ep.max_recv;
  h->tile_gateup = tile_from_env("MOE_TILE_N_GATEUP");
  h->tile_down = tile_from_env("MOE_TILE_N_DOWN");
  {
    const char* v = std::getenv("MOE_PAIR_TILES");
    h->use_pairs = !(v && v[0] == '0');
    const char* vs = std::getenv("MOE_SMALL_ROUTE");
    h->small_route = !(vs && vs[0] == '0');
    const char* vrg = std::getenv("MOE_ROUTE_IN_GEMM");
    h->route_in_gemm = !(vrg && vrg[0] == '0');
    const char* vo = std::getenv("MOE_SHARED_OVERLAP");
    h->shared_overlap = !(vo && vo[0] == '0');
    const char* vx = std::getenv("MOE_FP8_X2");
    // the in-place requantisation of H holds a row in registers: F <= 8192
    h->fp8_x2 = fp8 && !(vx && vx[0] == '0') && c.ffn_width <= 8192;
    const char* vk = std::getenv("MOE_GEMM_KSPLIT");
    const int ksv = vk ? std::atoi(vk) : -1;
    h->gemm_ksplit = (vk == nullptr || ksv < 0) ? -1 : (ksv <= 1 ? 1 : std::min(ksv, moe::kMaxGemmKSplit));
    if (vk != nullptr && vk[0] == 'b') h->gemm_ksplit = 0;
    const char* vp = std::getenv("MOE_PF_DOWN_WAVES");
    h->pf_down_waves = vp ? std::max(0, std::atoi(vp)) : kPrefetchDownWaves;
    const int rt = tile_from_env("MOE_ROUTER_TILE");
    h->router_tile = (rt == 16 || rt == 64 || rt == 128 || rt == 256) ? rt : 0;
  }
  h->wait_limit_ns = kDefaultWaitNs;
  h->router_m_tiles = (c.n_experts + moe::kBlockM - 1) / moe::kBlockM;

  const size_t Tmax = static_cast<size_t>(c.max_tokens);
  const size_t E = c.n_experts, k = c.top_k, d = c.d_model, F = c.ffn_width;
  const size_t R = (k + 1) * Tmax;
  // H rows: this rank's own dispatch rows, or the rows it may receive (EP)
  const size_t RH = R > static_cast<size_t>(ep.max_recv) ? R : static_cast<size_t>(ep.max_recv);
  const size_t n_epg = static_cast<size_t>(ep.size) * (ep.size ? c.n_experts / ep.size : 0) + 1;
  const size_t e_pad = static_cast<size_t>(h->router_m_tiles) * moe::kBlockM;
  // partial logits: room for kMaxKSplit K splits of Tmax tokens, at most
  // 32768 rows (the router splits K only while token tiles are few), or one
  // split of Tmax
  const size_t p_cap = 32768;
  const size_t p_rows = Tmax > p_cap ? Tmax : std::min(static_cast<size_t>(moe::kMaxKSplit) * Tmax, p_cap);
  h->partial_rows = static_cast<long long>(p_rows);
  size_t off = 0;
  auto carve = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, 256);
    return at;
  };
  // K split part buffer: up to 8 waves of part items of token tile <= 32
  h->ksplit_cap = 8 * h->num_sms;
  const size_t kcap = static_cast<size_t>(h->ksplit_cap);
  const size_t o_counts = carve(4 * E), o_err = carve(16), o_offsets = carve(4 * (E + 2)),
               o_kcnt = carve(4 * kcap), o_partial = carve(4 * p_rows * E), o_w3 = carve(2 * 3 * e_pad * d), o_idx = carve(4 * Tmax * k),
               o_prob = carve(4 * Tmax * k), o_perm = carve(4 * Tmax * k), o_inv = carve(4 * Tmax * k),
               o_yp = carve(2 * R * d), o_ye = carve((R / moe::kYpRows + E + 2) * d), o_cb = carve(4 * (E + 2)),
               o_h = carve(2 * RH * F),
               o_epo = carve(4 * n_epg), o_epc = carve(4 * n_epg), o_eps = carve(4 * (ep.size + 1)),
               o_epi = carve(4 * (static_cast<size_t>(ep.max_recv) + 1)),
               o_xs = carve(2 * Tmax * d),
               o_ys = carve((c.out_fp32 ? 4 : 2) * Tmax * d),
               o_tok = carve(4 * Tmax * (moe::kMaxStatGroups + 1)), o_tsc = carve(4 * R),
               o_ch = carve(4 * moe::chunk_hist_ints(static_cast<int>(Tmax), E)),
               o_kpart = carve(4 * kcap * moe::kBlockM * 32);
  if (cudaMalloc(&h->ws, off) != cudaSuccess) {
    cudaGetLastError();
    delete h;
    return MOE_ERR_CUDA;
  }
  char* b = static_cast<char*>(h->ws);
  h->counts = reinterpret_cast<int*>(b + o_counts);
  h->err = reinterpret_cast<uint32_t*>(b + o_err);
  h->route_done = reinterpret_cast<unsigned int*>(b + o_err + 4);  // zeroed below with the error word
  h->offsets = reinterpret_cast<int*>(b + o_offsets);
  h->partial = reinterpret_cast<float*>(b + o_partial);
  h->w3 = reinterpret_cast<bf16*>(b + o_w3);
  h->idx = reinterpret_cast<int*>(b + o_idx);
  h->prob = reinterpret_cast<float*>(b + o_prob);
  h->perm = reinterpret_cast<int*>(b + o_perm);
  h->inv = reinterpret_cast<int*>(b + o_inv);
  h->yp = b + o_yp;
  h->yexp = reinterpret_cast<int8_t*>(b + o_ye);
  h->chunk_base = reinterpret_cast<int*>(b + o_cb);
  h->hbuf = reinterpret_cast<bf16*>(b + o_h);
  h->x_stage = reinterpret_cast<bf16*>(b + o_xs);
  h->y_stage = b + o_ys;
  h->tokstats = reinterpret_cast<float*>(b + o_tok);
  h->tok_scale = reinterpret_cast<float*>(b + o_tsc);
  h->rows_max = static_cast<int>(R);
  h->chunk_hist = reinterpret_cast<int*>(b + o_ch);
  h->ksplit_cnt = reinterpret_cast<int*>(b + o_kcnt);
  h->ksplit_part = reinterpret_cast<float*>(b + o_kpart);
  h->ep_offsets = reinterpret_cast<int*>(b + o_epo);
  h->ep_chunk_base = reinterpret_cast<int*>(b + o_epc);
  h->ep_chunks_src = reinterpret_cast<int*>(b + o_eps);
  h->ep_iota = reinterpret_cast<int*>(b + o_epi);

  bool ok = cudaMemset(h->ws, 0, o_partial) == cudaSuccess;  // counts, error word, offsets, K split counters
  ok = ok && moe::launch_split_router(w->w_router, c.n_experts, c.d_model, static_cast<int>(e_pad), h->w3,
                                      nullptr) == cudaSuccess;
  // weight groups held by this handle: all, or (EP) the local experts + shared
  const size_t G = ep.size ? static_cast<size_t>(h->e_loc + c.has_shared) : static_cast<size_t>(h->G);
  ok = ok && moe::launch_iota(h->ep_iota, ep.max_recv, nullptr) == cudaSuccess;
  ok = ok && encode_2d(&h->map_w3, h->w3, 3 * e_pad, d, moe::kBlockM);
  ok = ok && encode_2d(&h->map_wgu, w->w_gate_up, G * 2 * F, d, moe::kBlockM / 2, fp8);
  ok = ok && encode_2d(&h->map_wd, w->w_down, G * d, F, moe::kBlockM, fp8);
  for (int i = 0; ok && i < moe::kNumTileN; ++i) {
    ok = ok && encode_2d(&h->map_xp[i], h->yp, R, d, moe::kTileN[i]);
    ok = ok && encode_2d(&h->map_xq[i], h->yp, 2 * R, d, moe::kTileN[i], true);
    ok = ok && encode_2d(&h->map_hq[i], h->hbuf, RH, 2 * F, moe::kTileN[i], true);
    ok = ok && encode_2d(&h->map_h[i], h->hbuf, RH, F, moe::kTileN[i]);
  }
  ok = ok && cudaStreamCreateWithFlags(&h->side, cudaStreamNonBlocking) == cudaSuccess;
  ok = ok && cudaEventCreateWithFlags(&h->ev_fork, cudaEventDisableTiming) == cudaSuccess;
  ok = ok && cudaEventCreateWithFlags(&h->ev_join, cudaEventDisableTiming) == cudaSuccess;
  ok = ok && cudaDeviceSynchronize() == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    release_streams(h);
    cudaFree(h->ws);
    delete h;
    return MOE_ERR_CUDA;
  }
  h->magic = kMagic;
  *out = h;
  return MOE_OK;
}

}  // namespace

extern "C" {

int moe_init(const moe_config* cfg, const moe_weights* w, moe_handle** out) {
  return init_any(cfg, w, nullptr, nullptr, out);
}

int moe_init_fp8(const moe_config* cfg, const moe_weights_fp8* w, moe_handle** out) {
  if (out != nullptr) *out = nullptr;
  if (w == nullptr || w->s_gate_up == nullptr || w->s_down == nullptr) return MOE_ERR_INVALID_ARG;
  const moe_weights ww{w->w_router, w->w_gate_up, w->w_down};
  return init_any(cfg, &ww, w->s_gate_up, w->s_down, out);
}

int moe_ep_init(const moe_ep_config* cfg, const moe_ep_weights* w, moe_handle** out) {
  if (out != nullptr) *out = nullptr;
  if (cfg == nullptr || w == nullptr || cfg->ep_size < 1) return MOE_ERR_INVALID_ARG;
  const moe_weights ww{w->w_router, w->w_gate_up, w->w_down};
  EpParams ep;
  ep.size = cfg->ep_size;
  ep.rank = cfg->ep_rank;
  ep.max_recv = cfg->max_recv_rows;
  return init_any(&cfg->layer, &ww, nullptr, nullptr, out, ep);
}

int moe_ep_dispatch(moe_handle* h, const void* x, int T, void* send_rows, float* send_w, int* send_counts,
                    int* rows_per_rank, void* stream) {
  int rc = check_call(h, x, T);
  if (rc != MOE_OK) return rc;
  DeviceGuard device_guard(h->device);
  if (h->ep_size == 0 || rows_per_rank == nullptr || send_counts == nullptr) return MOE_ERR_INVALID_ARG;
  const moe_config& c = h->cfg;
  const int k = c.top_k, E = c.n_experts;
  if (T > 0 && (send_rows == nullptr || send_w == nullptr || !aligned(send_rows, 16) || !aligned(send_w, 4) ||
                !is_device_ptr(x) || !is_device_ptr(send_rows) || !is_device_ptr(send_w)))
    return MOE_ERR_INVALID_ARG;
  if (!aligned(send_counts, 4) || !is_device_ptr(send_counts)) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  h->ep_T = T;
  // the routing and dispatch of the whole-layer call on the same tokens (so
  // that both give the same rows and weights)
  const bool fused_route = small_route(h, T);
  const bool overlap_shared = shared_overlap_ok(h) && c.has_shared && !fused_route && T >= kSharedOverlapMinTokens;
  if (fused_route) {
    MOE_CUDA(moe::launch_route_small(static_cast<const bf16*>(x), h->w.w_router, T, c.d_model, E, k, 0, c.has_shared,
                                     h->partial, h->route_done, h->idx, h->prob, nullptr, h->counts, h->offsets,
                                     h->perm, h->inv, h->chunk_base, moe::SmallRouteExtras{}, s));
  } else {
    rc = enqueue_router(h, x, T, CallOpts{k, 0}, h->idx, h->prob, nullptr, nullptr, 0, s);
    if (rc != MOE_OK) return rc;
  }
  MOE_CUDA(cudaMemcpyAsync(send_counts, h->counts, sizeof(int) * E, cudaMemcpyDeviceToDevice, s));
  for (int q = 0; q < h->ep_size; ++q) rows_per_rank[q] = 0;
  if (T == 0) return cudaStreamSynchronize(s) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  if (!fused_route)
    MOE_CUDA(moe::launch_dispatch(h->idx, h->counts, T, E, k, c.has_shared, h->offsets, h->perm, h->inv,
                                  h->chunk_base, h->chunk_hist, s));
  // every row in dispatch order (the shared expert's rows stay here for
  // moe_ep_combine); the routed rows, expert-major, go out rank by rank
  MOE_CUDA(moe::launch_gather(static_cast<const bf16*>(x), h->inv, T, k, c.d_model, c.has_shared, h->yp, false, s));
  const size_t Tk = static_cast<size_t>(T) * k;
  MOE_CUDA(cudaMemcpyAsync(send_rows, h->yp, Tk * c.d_model * 2, cudaMemcpyDeviceToDevice, s));
  MOE_CUDA(moe::launch_gather_weights(h->perm, h->prob, static_cast<int>(Tk), send_w, s));
  std::vector<int> off(E + 2);
  MOE_CUDA(cudaMemcpyAsync(off.data(), h->offsets, sizeof(int) * (E + 2), cudaMemcpyDeviceToHost, s));
  MOE_CUDA(cudaStreamSynchronize(s));
  for (int q = 0; q < h->ep_size; ++q) rows_per_rank[q] = off[(q + 1) * h->e_loc] - off[q * h->e_loc];
  return MOE_OK;
}

int moe_ep_experts(moe_handle* h, const void* recv_rows, const int* recv_counts, const float* recv_w, int n_recv,
                   void* out_rows, void* out_exp, int* chunks_per_source, void* stream) {
  if (!valid_handle(h) || h->ep_size == 0 || recv_counts == nullptr || chunks_per_source == nullptr)
    return MOE_ERR_INVALID_ARG;
  DeviceGuard device_guard(h->device);
  if (n_recv < 0) return MOE_ERR_INVALID_ARG;
  if (n_recv > h->max_recv) return MOE_ERR_TOO_MANY_TOKENS;
  if (!aligned(recv_counts, 4) || !is_device_ptr(recv_counts)) return MOE_ERR_INVALID_ARG;
  if (n_recv > 0 && (recv_rows == nullptr || recv_w == nullptr || out_rows == nullptr || out_exp == nullptr ||
                     !aligned(recv_rows, 16) || !aligned(recv_w, 4) || !aligned(out_rows, 16) ||
                     !aligned(out_exp, 16) || !is_device_ptr(recv_rows) || !is_device_ptr(recv_w) ||
                     !is_device_ptr(out_rows) || !is_device_ptr(out_exp)))
    return MOE_ERR_INVALID_ARG;
  const moe_config& c = h->cfg;
  const int S = h->ep_size, El = h->e_loc, G = S * El;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  MOE_CUDA(moe::launch_ep_groups(recv_counts, S, El, h->ep_offsets, h->ep_chunk_base, h->ep_chunks_src, s));
  std::vector<int> chunks(S);
  int total = 0;
  MOE_CUDA(cudaMemcpyAsync(&total, h->ep_offsets + G, sizeof(int), cudaMemcpyDeviceToHost, s));
  MOE_CUDA(cudaMemcpyAsync(chunks.data(), h->ep_chunks_src, sizeof(int) * S, cudaMemcpyDeviceToHost, s));
  MOE_CUDA(cudaStreamSynchronize(s));
  if (total != n_recv) return MOE_ERR_INVALID_ARG;  // the counts must describe exactly the rows given
  for (int q = 0; q < S; ++q) chunks_per_source[q] = chunks[q];
  if (n_recv == 0) return MOE_OK;
  CUtensorMap maps[moe::kNumTileN];
  for (int i = 0; i < moe::kNumTileN; ++i)
    if (!encode_2d(&maps[i], recv_rows, static_cast<uint64_t>(n_recv), static_cast<uint64_t>(c.d_model),
                   moe::kTileN[i]))
      return MOE_ERR_CUDA;
  // groups = (source, local expert), source-major; every row carries its own
  // gate weight (perm = identity, prob = recv_w)
  moe::GemmArgs a{};
  a.offsets = h->ep_offsets;
  a.G = G;
  a.perm = h->ep_iota;
  a.prob = recv_w;
  a.Tk = n_recv;
  a.chunk_base = h->ep_chunk_base;
  a.w_group_mod = El;
  return enqueue_ffn(h, a, static_cast<double>(n_recv) / G, maps, out_rows, static_cast<int8_t*>(out_exp), nullptr,
                     s, nullptr, 0, n_recv);
}

int moe_ep_combine(moe_handle* h, const void* ret_rows, const void* ret_exp, void* y, void* stream) {
  if (!valid_handle(h) || h->ep_size == 0) return MOE_ERR_INVALID_ARG;
  DeviceGuard device_guard(h->device);
  const moe_config& c = h->cfg;
  const int T = h->ep_T, k = c.top_k;
  if (T == 0) return MOE_OK;
  if (y == nullptr || !aligned(y, 16) || !is_device_ptr(y)) return MOE_ERR_INVALID_ARG;
  if (ret_rows == nullptr || ret_exp == nullptr || !aligned(ret_rows, 16) || !aligned(ret_exp, 8) ||
      !is_device_ptr(ret_rows) || !is_device_ptr(ret_exp))
    return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (c.has_shared) {
    // the shared expert on this rank's own tokens: one group, rows [T*k, T*k + T)
    moe::GemmArgs a{};
    a.offsets = h->offsets + c.n_experts;
    a.G = 1;
    a.perm = h->perm;
    a.prob = h->prob;
    a.Tk = T * k;
    a.chunk_base = h->chunk_base + c.n_experts;
    a.w_group_base = h->e_loc;
    if (int rc = enqueue_ffn(h, a, static_cast<double>(T), h->map_xp, h->yp, h->yexp, nullptr, s)) return rc;
  }
  MOE_CUDA(moe::launch_combine(static_cast<const __half*>(h->yp), h->yexp, static_cast<const __half*>(ret_rows),
                               static_cast<const int8_t*>(ret_exp), h->idx, h->inv, h->offsets, h->chunk_base, T, k,
                               c.n_experts, c.d_model, c.has_shared, y, c.out_fp32, s));
  return MOE_OK;
}

int moe_quantize_fp8(const void* w, long long rows, int cols, void* q, float* s, void* stream) {
  if (rows < 0 || cols <= 0 || rows > 0x7fffffffll) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  if (w == nullptr || q == nullptr || s == nullptr || !aligned(w, 2) || !aligned(s, 4)) return MOE_ERR_INVALID_ARG;
  if (!is_device_ptr(w) || !is_device_ptr(q) || !is_device_ptr(s)) return MOE_ERR_INVALID_ARG;
  MOE_CUDA(moe::launch_quantize_e4m3(static_cast<const bf16*>(w), rows, cols, static_cast<uint8_t*>(q), s,
                                     static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

int moe_route_ex(moe_handle* h, const void* x, int T, const moe_call_options* opt, int* idx, float* prob, int* perm,
                 int* offsets, float* gap, void* stream) {
  int rc = check_call(h, x, T);
  if (rc != MOE_OK) return rc;
  DeviceGuard device_guard(h->device);
  CallOpts o;
  if ((rc = resolve_opts(h, opt, &o)) != MOE_OK) return rc;
  if (idx == nullptr || prob == nullptr || perm == nullptr || offsets == nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned(idx, 4) || !aligned(prob, 4) || !aligned(perm, 4) || !aligned(offsets, 4) || !aligned(gap, 4))
    return MOE_ERR_INVALID_ARG;
  if (T > 0 && !is_device_ptr(x)) return MOE_ERR_INVALID_ARG;
  if (!is_device_ptr(idx) || !is_device_ptr(prob) || !is_device_ptr(perm) || !is_device_ptr(offsets) ||
      (gap != nullptr && !is_device_ptr(gap)))
    return MOE_ERR_INVALID_ARG;
  return enqueue_route(h, x, T, o, idx, prob, perm, offsets, gap, static_cast<cudaStream_t>(stream));
}

int moe_route(moe_handle* h, const void* x, int T, int* idx, float* prob, int* perm, int* offsets, float* gap,
              void* stream) {
  return moe_route_ex(h, x, T, nullptr, idx, prob, perm, offsets, gap, stream);
}

int moe_forward_ex(moe_handle* h, const void* x, int T, const moe_call_options* opt, void* y, void* stream) {
  int rc = check_call(h, x, T);
  if (rc != MOE_OK) return rc;
  DeviceGuard device_guard(h->device);
  if (h->ep_size != 0) return MOE_ERR_INVALID_ARG;  // an expert-parallel handle holds only its experts
  CallOpts o;
  if ((rc = resolve_opts(h, opt, &o)) != MOE_OK) return rc;
  h->last_kernels = 0;
  if (T == 0) return MOE_OK;
  if (y == nullptr || !aligned(y, 16)) return MOE_ERR_INVALID_ARG;
  if (!is_device_ptr(x) || !is_device_ptr(y)) return MOE_ERR_INVALID_ARG;
  return enqueue_forward(h, x, T, o, y, static_cast<cudaStream_t>(stream));
}

int moe_forward(moe_handle* h, const void* x, int T, void* y, void* stream) {
  return moe_forward_ex(h, x, T, nullptr, y, stream);
}

int moe_route_stats(moe_handle* h, const void* x, int T, int n_groups, int* counts, float* group_f,
                    float* group_p, float* summary, void* stream) {
  int rc = check_call(h, x, T);
  if (rc != MOE_OK) return rc;
  DeviceGuard device_guard(h->device);
  const moe_config& c = h->cfg;
  if (n_groups < 1 || n_groups > moe::kMaxStatGroups || c.n_experts % n_groups != 0) return MOE_ERR_INVALID_ARG;
  if (counts == nullptr || group_f == nullptr || group_p == nullptr || summary == nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned(counts, 4) || !aligned(group_f, 4) || !aligned(group_p, 4) || !aligned(summary, 4))
    return MOE_ERR_INVALID_ARG;
  if (T > 0 && !is_device_ptr(x)) return MOE_ERR_INVALID_ARG;
  if (!is_device_ptr(counts) || !is_device_ptr(group_f) || !is_device_ptr(group_p) || !is_device_ptr(summary))
    return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const CallOpts o{c.top_k, 0};
  rc = enqueue_router(h, x, T, o, h->idx, h->prob, nullptr, h->tokstats, n_groups, s);
  if (rc != MOE_OK) return rc;
  MOE_CUDA(moe::launch_route_stats(h->tokstats, h->counts, T, c.n_experts, c.top_k, n_groups, group_f, group_p,
                                   summary, s));
  MOE_CUDA(cudaMemcpyAsync(counts, h->counts, sizeof(int) * c.n_experts, cudaMemcpyDeviceToDevice, s));
  return MOE_OK;
}

int moe_forward_host(moe_handle* h, const void* x_host, int T, void* y_host, void* stream) {
  if (!valid_handle(h) || h->ep_size != 0) return MOE_ERR_INVALID_ARG;
  DeviceGuard device_guard(h->device);
  if (T < 0) return MOE_ERR_INVALID_ARG;
  if (T > h->cfg.max_tokens) return MOE_ERR_TOO_MANY_TOKENS;
  if (T == 0) return MOE_OK;
  if (x_host == nullptr || y_host == nullptr) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t d = h->cfg.d_model;
  const size_t xbytes = 2 * d * static_cast<size_t>(T);
  const size_t ybytes = (h->cfg.out_fp32 ? 4 : 2) * d * static_cast<size_t>(T);
  MOE_CUDA(cudaMemcpyAsync(h->x_stage, x_host, xbytes, cudaMemcpyHostToDevice, s));
  const int rc = enqueue_forward(h, h->x_stage, T, CallOpts{h->cfg.top_k, 0}, h->y_stage, s);
  if (rc != MOE_OK) return rc;
  MOE_CUDA(cudaMemcpyAsync(y_host, h->y_stage, ybytes, cudaMemcpyDeviceToHost, s));
  MOE_CUDA(cudaStreamSynchronize(s));
  return MOE_OK;
}

int moe_last_kernel_count(const moe_handle* h) {
  if (h == nullptr || h->magic != kMagic) return -1;
  return h->last_kernels;
}

int moe_check(moe_handle* h, void* stream) {
  if (!valid_handle(h)) return MOE_ERR_INVALID_ARG;
  DeviceGuard device_guard(h->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  uint32_t e = 0;
  MOE_CUDA(cudaMemcpyAsync(&e, h->err, sizeof e, cudaMemcpyDeviceToHost, s));
  MOE_CUDA(cudaMemsetAsync(h->err, 0, sizeof e, s));
  MOE_CUDA(cudaStreamSynchronize(s));
#ifdef MOE_DEBUG
  // the bounds checks' words of every kernel source (a debug build only)
  e |= moe::dbg_take_dispatch() | moe::dbg_take_expert_gemm() | moe::dbg_take_expert_gemm_pair() |
       moe::dbg_take_expert_gemm_fp8() | moe::dbg_take_expert_gemm_fp8x();
#endif
  // a GEMM that gave up may have left K split part counts behind: the next
  // call on the handle starts from zero
  if (e) MOE_CUDA(cudaMemset(h->ksplit_cnt, 0, sizeof(int) * static_cast<size_t>(h->ksplit_cap)));
  return e ? MOE_ERR_DEVICE : MOE_OK;
}

int moe_set_wait_limit(moe_handle* h, unsigned long long ns) {
  if (!valid_handle(h)) return MOE_ERR_INVALID_ARG;
  h->wait_limit_ns = ns ? ns : kDefaultWaitNs;
  return MOE_OK;
}

int moe_profile_enable(moe_handle* h, int enable) {
  if (!valid_handle(h)) return MOE_ERR_INVALID_ARG;
  h->profiling = enable != 0;
  if (!h->profiling) h->n_prof = 0;
  return MOE_OK;
}

int moe_profile_read(moe_handle* h, float* ms, int* n_calls) {
  if (!valid_handle(h) || ms == nullptr || n_calls == nullptr) return MOE_ERR_INVALID_ARG;
  DeviceGuard device_guard(h->device);
  for (int i = 0; i < kProfStages; ++i) ms[i] = 0.f;
  *n_calls = h->n_prof;
  for (int c = 0; c < h->n_prof; ++c) {
    auto& ev = h->prof[c];
    MOE_CUDA(cudaEventSynchronize(ev[kProfStages]));
    for (int i = 0; i < kProfStages; ++i) {
      float t = 0.f;
      MOE_CUDA(cudaEventElapsedTime(&t, ev[i], ev[i + 1]));
      ms[i] += t;
    }
  }
  h->n_prof = 0;
  return MOE_OK;
}

int moe_free(moe_handle* h) {
  if (!valid_handle(h)) return MOE_ERR_INVALID_ARG;
  DeviceGuard device_guard(h->device);
  h->magic = 0;
  const bool ok = cudaDeviceSynchronize() == cudaSuccess;
  for (auto& ev : h->prof)
    for (auto e : ev) cudaEventDestroy(e);
  release_streams(h);
  const bool freed = cudaFree(h->ws) == cudaSuccess;
  delete h;
  return (ok && freed) ? MOE_OK : MOE_ERR_CUDA;
}

int moe_selftest_wait_timeout(unsigned long long limit_ns, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t* err = nullptr;
  if (cudaMalloc(&err, sizeof(uint32_t)) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  uint32_t e = 0;
  bool ok = cudaMemsetAsync(err, 0, sizeof(uint32_t), s) == cudaSuccess;
  ok = ok && moe::launch_wait_selftest(err, limit_ns, s) == cudaSuccess;
  ok = ok && cudaMemcpyAsync(&e, err, sizeof e, cudaMemcpyDeviceToHost, s) == cudaSuccess;
  ok = ok && cudaStreamSynchronize(s) == cudaSuccess;
  cudaFree(err);
  if (!ok) return MOE_ERR_CUDA;
  return e ? MOE_ERR_DEVICE : MOE_OK;
}

}  // extern "C"
