// Internal interface between the C-ABI layer (moe_api.cu) and the kernels.
// Every launch_* function enqueues on `stream` and returns the launch status.
#pragma once
#include <utility>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace moe {

// Programmatic dependent launch.  The kernels of a layer call are launched
// with programmatic stream serialisation (launch_chain): a kernel may start
// while the one before it in the stream is finishing.  Each calls pdl_wait()
// before its first access to global memory that earlier work in the stream
// reads or writes (it returns once those grids have completed and their
// writes are visible) and pdl_trigger() once the next kernel may be placed:
// short kernels on entry, the persistent GEMMs at their end (without the
// launch attribute both are no-ops).  One exception: the combine reads the
// routing and dispatch results before its wait, since the down GEMM before
// it triggers only at its end, when everything older has completed.
// MOE_PDL=0 in the environment turns the attribute off.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
bool pdl_enabled();

template <typename... KArgs, typename... Args>
cudaError_t launch_chain(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                         Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}


using bf16 = __nv_bfloat16;

// Debug builds (-DMOE_DEBUG, libmoe_debug.so): the kernels check every index
// they take from the dispatch (dispatch positions, row blocks, exponent
// chunks, permutation entries) against the bounds the dispatch guarantees.  A
// failed check skips the access it guards and ORs 2 (the bounds bit) into a
// debug word of its translation unit; moe_check collects and clears the
// words (dbg_take_* below) and reports MOE_ERR_DEVICE.  Nothing traps.  In
// release builds MOE_DBG_OK(cond) is the constant true and cond is not
// evaluated.
#ifdef MOE_DEBUG
namespace {
__device__ uint32_t g_dbg_word;  // one per translation unit
__device__ __forceinline__ bool dbg_check(bool ok) {
  if (!ok) atomicOr(&g_dbg_word, 2u);
  return ok;
}
}  // namespace
#define MOE_DBG_OK(cond) (::moe::dbg_check(cond))
// Defines uint32_t name(): this translation unit's debug word, then clears it.
#define MOE_DBG_DEFINE_TAKE(name)                                                \
  uint32_t name() {                                                              \
    uint32_t v = 0;                                                              \
    if (cudaMemcpyFromSymbol(&v, g_dbg_word, sizeof v) != cudaSuccess) {         \
      cudaGetLastError();                                                        \
      return 0;                                                                  \
    }                                                                            \
    const uint32_t z = 0;                                                        \
    if (v && cudaMemcpyToSymbol(g_dbg_word, &z, sizeof z) != cudaSuccess) cudaGetLastError(); \
    return v;                                                                    \
  }
uint32_t dbg_take_dispatch();
uint32_t dbg_take_expert_gemm();
uint32_t dbg_take_expert_gemm_pair();
uint32_t dbg_take_expert_gemm_fp8();
uint32_t dbg_take_expert_gemm_fp8x();
#else
#define MOE_DBG_OK(cond) (true)
#define MOE_DBG_DEFINE_TAKE(name)
#endif

constexpr int kBlockM = 128;  // weight rows per tensor-core tile (M of tcgen05.mma)
constexpr int kBlockK = 64;   // K elements per pipeline stage (one 128-byte swizzle row)
constexpr int kMaxExperts = 512;
constexpr int kMaxTopK = 32;
constexpr int kMaxKSplit = 48;  // K splits of the router GEMM
constexpr int kMaxGemmKSplit = 4;  // K parts of the expert GEMMs (small token counts)
constexpr int kKStepE4M3 = 128;    // K per pipeline stage of the E4M3 expert GEMMs (128 bytes)
constexpr int kMaxStatGroups = 64;  // expert groups of the routing statistics

// Expert outputs Yp (one row per dispatch position) are kept as fp16 with a
// power-of-two scale per feature and chunk of kYpRows consecutive rows of one
// group: value = h * 2^e, h fp16, e int8 in [-126, kYpExpMax].  Chunks are
// numbered group by group: group g's chunks start at chunk_base[g] =
// sum over g' < g of ceil(rows(g') / kYpRows); the exponents are [chunk][d].
constexpr int kYpRows = 16;
constexpr int kYpExpMax = 113;
// The shared expert's chunks start at a place fixed by T, k and E (past every
// chunk the routed experts can have: their rows rounded up per expert), so a
// launch can write them before the dispatch has counted the routed rows.
__host__ __device__ inline int shared_chunk0(int T, int k, int E) { return (T * k + kYpRows - 1) / kYpRows + E; }

// Token-tile widths (N of tcgen05.mma) the grouped GEMMs are built for.
constexpr int kNumTileN = 5;
constexpr int kTileN[kNumTileN] = {16, 32, 64, 128, 256};

// K1 on the tensor cores: partial logits of a K split, then softmax/top-k.
struct RouterGemmArgs {
  float* partial;  // [ksplit][T][E] fp32 partial logits
  uint32_t* err;
  unsigned long long wait_limit_ns;
  int T, d, E;
  int e_pad;    // rows per slice of the split router weights (multiple of 128)
  int m_tiles;  // e_pad / 128
  int ksplit;   // K splits (1..kMaxKSplit)
  // weights to prefetch into L2 while the router runs (NULL / 0: none;
  // 16-byte multiples): the shared expert's, which every layer call reads
  const void* pf[2];
  long long pf_bytes[2];
};
cudaError_t launch_router_gemm(int tile_n, const CUtensorMap* map_w3, const CUtensorMap* map_x,
                               const RouterGemmArgs& a, int num_sms, cudaStream_t stream);
// renorm != 0 divides the k weights by their sum; tokstats (or NULL) gets per
// token the probability mass of each of n_groups expert groups and the entropy.
cudaError_t launch_router_topk(const float* partial, int ksplit, int T, int E, int k, int renorm, int* idx,
                               float* prob, float* gap, int* counts, float* tokstats, int n_groups,
                               cudaStream_t stream);
// Routing statistics from tokstats and counts (one block, fixed summation order).
cudaError_t launch_route_stats(const float* tokstats, const int* counts, int T, int E, int k, int n_groups,
                               float* group_f, float* group_p, float* summary, cudaStream_t stream);
// A few tokens: router (fp32 FMA dot products), softmax / top-k and the
// dispatch in one launch (see router_gemm.cu).  logits [T][E] scratch; done
// an unsigned int that is zero between launches.  Usable when
// route_small_fits(T, d, E).
// ex: two weight regions to prefetch into L2 while routing (pf*, NULL / 0
// for none; 16-byte multiples), and xp (or NULL): the buffer [T*k][d] bf16
// the routed rows are copied into in dispatch order.
// (up to 4 tokens: measured at 1, 2 and 4 tokens on the flash shape 4-8 %
// faster per call than the router GEMM + top-k + dispatch chain, at 8 tokens
// the same)
constexpr int kSmallRouteMaxTokens = 4;
struct SmallRouteExtras {
  const void* pf0;
  long long pf0_bytes;
  const void* pf1;
  long long pf1_bytes;
  void* xp;
  int logits_only;  // 1: the logits (and the prefetch) only; the gate/up launch ranks the tokens
  int replicas;     // logits only: copies of the T token rows written to xp for that launch
};
bool route_small_fits(int T, int d, int E);
cudaError_t launch_route_small(const bf16* x, const float* w_router, int T, int d, int E, int k, int renorm,
                               int has_shared, float* logits, unsigned int* done, int* idx, float* prob, float* gap,
                               int* counts, int* offsets, int* perm, int* inv, int* chunk_base,
                               const SmallRouteExtras& ex, cudaStream_t stream);
// W_r fp32 [E][d] -> bf16 slices [3][e_pad][d] with hi + mid + lo = W_r.
cudaError_t launch_split_router(const float* w, int E, int d, int e_pad, bf16* w3, cudaStream_t stream);
cudaError_t router_gemm_prepare();

// K2: offsets (exclusive scan of counts, shared group appended), the stable
// expert-major permutation perm / its inverse inv, and chunk_base [E+2] (the
// exponent chunks of the expert outputs, see kYpRows).
cudaError_t launch_dispatch(const int* idx, const int* counts, int T, int E, int k, int has_shared, int* offsets,
                            int* perm, int* inv, int* chunk_base, const int* chunk_first, cudaStream_t stream);
// From kChunkedDispatchMinTokens tokens on, the counts come from per-chunk
// histograms (launch_chunk_counts: hist [ceil(T/256)][E] becomes each chunk's
// first row per expert, counts [E] the totals) instead of atomics in the top-k
// kernel, and launch_dispatch places the rows chunk by chunk from them
// (chunk_first = that hist; NULL: the per-expert kernel at any T).
constexpr int kChunkedDispatchMinTokens = 1024;
bool chunked_dispatch(int T);
size_t chunk_hist_ints(int T, int E);
cudaError_t launch_chunk_counts(const int* idx, int T, int E, int k, int* hist, int* counts, cudaStream_t stream);

// Token rows into dispatch order: xp[inv[t*k + j]] = x[t] (j < k), and with
// has_shared xp[T*k + t] = x[t]; each row of x is read once and written to
// its positions.  With to_f16 the rows are written as fp16 (x's bf16 values
// rounded to nearest).
cudaError_t launch_gather(const bf16* x, const int* inv, int T, int k, int d, int has_shared, void* xp,
                          bool to_f16, cudaStream_t stream);

struct GemmArgs {
  const int* offsets;  // [G+1] row offsets of the groups in dispatch order
  const int* perm;     // [T*k] (down projection: gate weight lookup)
  const float* prob;   // [T*k] (down projection)
  void* out;           // H bf16 [R][F] (gate/up) or Yp fp16 [R][d] (down)
  int8_t* out_exp;     // down: Yp exponents [chunks][d]
  const int* chunk_base;  // down: [G+1] first exponent chunk of each group
  const float* w_scale;   // FP8 weights: scale of every weight row [G][rows_per_group]
  uint32_t* err;       // device error word
  unsigned long long wait_limit_ns;
  int G;               // groups (E + has_shared)
  int K;               // reduction length: d (gate/up) or F (down)
  int rows_per_group;  // weight rows per group: 2F (gate/up) or d (down)
  int m_tiles;         // output-feature tiles per group: F/128 or d/128
  int F;               // expert width (gate/up: offset of the up rows)
  int out_ld;          // row length of out
  int Tk;              // T*k: dispatch positions >= Tk belong to the shared expert
  int reverse;         // 1: work items in reverse order (last group first)
  int w_group_base;    // weights of group g: w_group_base + (w_group_mod ? g % w_group_mod : g)
  int w_group_mod;
  // K split (single-CTA bf16 and two-term E4M3 kernels, few work items): ksplit > 1 cuts every
  // item's K range into ksplit parts run as separate items; each part writes
  // its fp32 accumulator to ksplit_part and the last part to finish (counted
  // in ksplit_cnt, which it resets) sums the parts in part order and runs the
  // epilogue on the sum.  With more part items than ksplit_cap, or token tiles
  // wider than 32, the kernel runs unsplit.
  int ksplit;
  // single-CTA bf16 kernel: with ksplit > 1 and kbalance = 1 the K steps of
  // all items are instead cut into one contiguous range per CTA (an item's
  // parts are the ranges its steps fall in, at most kMaxGemmKSplit; CTA c
  // keeps its parts in slots 2c and 2c + 1 of the part buffer)
  int kbalance;
  int ksplit_cap;      // part items ksplit_part and ksplit_cnt hold
  float* ksplit_part;  // [ksplit_cap][128][BN]
  int* ksplit_cnt;     // [ksplit_cap], zero between launches
  const float* tok_scale;  // FP8 gate/up with two-term tokens: 1/s of every dispatch row
  int lo_row0, lo_col0;    // ... and where the lo terms of dispatch row 0 sit in the token map
  int act2_from;       // bf16 kernels: token rows from this dispatch position on come through
                       // map_act2 at row (position - act2_from); -1: all through map_act
  int rows_cap;        // rows of the dispatch-ordered buffers (token rows, H, Yp)
  int chunks_cap;      // exponent chunks the Yp exponent buffer holds
  int off_const[2];    // pair kernels with offsets == NULL: the one group's rows [off_const[0], off_const[1])
  int chunk_const;     // ... and with chunk_base == NULL (down): the group's first exponent chunk
  // Single-CTA gate/up: once a CTA has issued its last load it brings into L2
  // the weights of the down launch that follows it, which deals whole items
  // (group, weight tile of 128 rows) over the same token tiles to a grid of
  // the same size: CTA c takes that launch's items c + w * gridDim.x, w <
  // pf_waves, i.e. the first ones each of its CTAs runs.  pf_w: the down
  // weights [G][pf_rows_per_group][pf_row_bytes bytes]; NULL: no prefetch.
  const void* pf_w;
  int pf_waves;
  int pf_m_tiles;         // weight tiles per group of that launch
  int pf_rows_per_group;
  int pf_row_bytes;       // multiple of 16
  // Few tokens (at most kSmallRouteMaxTokens), bf16 gate/up on one CTA per
  // SM: the routing finished in this launch.  With route_logits [T][E] fp32
  // non-NULL every CTA ranks each token's experts from the logits (the same
  // softmax and top-k as the routing kernels), lays the dispatch out in shared
  // memory, reads every group's token tile from a copy of the T token rows
  // behind map_act (the columns of tokens that did not pick a group, and any
  // rows past the T, are computed and not stored) and stores H at the dispatch
  // positions; CTA 0 writes the routing and dispatch results (route_* below,
  // as the routing kernels lay them out) for the down projection and the
  // combine.  offsets is unused then.
  const float* route_logits;
  int route_T, route_E, route_k, route_renorm, route_has_shared;
  int route_replicas;  // copies of the T token rows behind map_act: CTA c reads rows (c mod it) * T ...
  int* route_idx;
  float* route_prob;
  int* route_counts;
  int* route_offsets;  // [E + 2]
  int* route_perm;
  int* route_inv;
  int* route_chunk_base;  // [E + 2]
};

// K3/K4: tcgen05 grouped GEMMs over the groups' row blocks.  `tile_n` must be
// one of kTileN.  gateup = true: H = silu(X Wg^T) * (X Wu^T) (map_w box: 64
// rows, m_tiles = F/64); false: Yp = w * (H Wd^T) (map_w box: 128 rows,
// m_tiles = d/128).  map_act: the token rows (X or H), box tile_n rows.
cudaError_t launch_expert_gemm(bool gateup, int tile_n, const CUtensorMap* map_w, const CUtensorMap* map_act,
                               const CUtensorMap* map_act2, const GemmArgs& a, int num_sms, cudaStream_t stream);
// Opts every grouped-GEMM instantiation into its dynamic shared memory size
// on the current device (once per device, before the first launch).
cudaError_t expert_gemm_prepare();

// K3/K4 for 256-row token tiles on CTA pairs (clusters of 2, grid = even
// number of SMs).  a.m_tiles must count pair tiles: F/128 (gate/up, map_w box
// 64 rows) or d/256 (down, map_w box 128 rows); map_act box: 128 rows.
cudaError_t launch_expert_gemm_pair(bool gateup, const CUtensorMap* map_w, const CUtensorMap* map_act,
                                    const CUtensorMap* map_act2, const GemmArgs& a, int num_sms,
                                    cudaStream_t stream);
cudaError_t expert_gemm_pair_prepare();

// K3/K4 with E4M3 weights (one fp32 scale per weight row in a.w_scale) and
// fp16 activations; tile_n in {16, 32, 64, 128}.  map_w: the E4M3 codes as
// [G * rows_per_group][K] bytes, box 128 x 64 rows (gate/up) or 128 x 128
// (down); map_act: the fp16 token rows or H, box 64 x tile_n.
cudaError_t launch_expert_gemm_fp8(bool gateup, int tile_n, const CUtensorMap* map_w, const CUtensorMap* map_act,
                                   const GemmArgs& a, int num_sms, cudaStream_t stream);
cudaError_t expert_gemm_fp8_prepare();
// K3 / K4 with E4M3 weights and two-term E4M3 token rows (tcgen05.mma
// kind::f8f6f4): map_tok is a byte map whose boxes are tile_n rows x 128 bytes,
// the hi terms of dispatch row r at row r and the lo terms at row
// a.lo_row0 + r, column a.lo_col0 on; a.tok_scale holds 1/s of every dispatch
// row.  K3 writes H as fp16, K4 writes Yp as expert_gemm.cu does.
// tile_n = 16, 32, 64 or 128.
cudaError_t launch_expert_gemm_fp8x(bool gateup, int tile_n, const CUtensorMap* map_w, const CUtensorMap* map_tok,
                                    const GemmArgs& a, int num_sms, cudaStream_t stream);
cudaError_t expert_gemm_fp8x_prepare();
// H [rows][F] fp16, rewritten in place as two-term E4M3 rows: row r's 2F
// bytes become hi (bytes 0..F-1) and lo (F..2F-1) of s_r * h, s_r the largest
// power of two with s_r * max|h_r| <= 448; inv_s[r] = 1/s_r.
cudaError_t launch_requant_rows_x2(void* h, int rows, int F, float* inv_s, cudaStream_t stream);
// Token rows for it: per token a power-of-two scale s (largest with
// s*max|x| <= 448), hi = e4m3(s*x) and lo = e4m3(s*x - hi) written to each of
// the token's dispatch rows (xq[pos], xq[lo_row0 + pos], bytes) and
// inv_s[pos] = 1/s; has_shared: also row T*k + t.
cudaError_t launch_scatter_x2(const bf16* x, const int* inv, int T, int k, int d, int has_shared, uint8_t* xq,
                              int lo_row0, float* inv_s, cudaStream_t stream);

// Per-row E4M3 quantisation of bf16 rows: s[r] = max |w[r]| / 448, q = nearest
// E4M3 (ties to even, saturating) of w / s (fp32 quotient); zero rows: s = 0, q = 0.
cudaError_t launch_quantize_e4m3(const bf16* w, long long rows, int cols, uint8_t* q, float* s,
                                 cudaStream_t stream);

// K5: y[t] = sum_j Yp[inv[t*k+j]] + Yp[T*k + t], fp32 in fixed order, each
// term read back as h * 2^e from the scaled fp16 Yp and its exponents (the
// chunk of a row found from its expert idx[t*k+j], offsets and chunk_base).
// yp_routed / yexp_routed (or NULL): where the routed rows (slots j < k) and
// their exponent chunks are, if not in yp / yexp (same positions and chunks).
cudaError_t launch_combine(const __half* yp, const int8_t* yexp, const __half* yp_routed, const int8_t* yexp_routed,
                           const int* idx, const int* inv, const int* offsets, const int* chunk_base, int T, int k,
                           int E, int d, int has_shared, void* y, int out_fp32, cudaStream_t stream);

// Expert parallelism helpers.  ep_groups: from recv_counts [S][E_loc] (rows
// per (source, local expert)), the row offsets [S*E_loc + 1] and exponent
// chunk bases [S*E_loc + 1] of the (source, expert) groups in source-major
// order, and the chunks of each source's block [S].  gather_weights:
// w[pos] = prob[perm[pos]] for pos < n.  iota: v[i] = i for i < n.
cudaError_t launch_ep_groups(const int* recv_counts, int S, int E_loc, int* offsets, int* chunk_base,
                             int* chunks_per_source, cudaStream_t stream);
cudaError_t launch_gather_weights(const int* perm, const float* prob, int n, float* w, cudaStream_t stream);
cudaError_t launch_iota(int* v, int n, cudaStream_t stream);

// Bounded-wait self test: waits on a barrier that never completes.
cudaError_t launch_wait_selftest(uint32_t* err, unsigned long long limit_ns, cudaStream_t stream);

}  // namespace moe
