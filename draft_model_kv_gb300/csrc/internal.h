// Internal interface between the C-ABI host code (api.cu) and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "../../include/dspark_ctx_kv.h"

struct dspark_bundle;

namespace dspark {

constexpr int kMaxDpPerm = 160;   // whole tiles that a launch may reorder (one wave of SMs)
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // bound on any single in-kernel wait (2 s)

// Everything the fused write needs besides the two operand tensor maps.
struct WriteParams {
  int32_t T, H, N, L, NH, D, KV;
  int32_t num_m, num_n, num_kb, num_tiles;
  // plain product mode (head_dim 0): output [T, N] rows y_stride apart in the
  // model dtype, and rowsq [T][rowsq_stride] fp32 sums of squares per N tile
  void* y;
  int64_t y_stride;
  float* rowsq;
  int32_t rowsq_stride;
  const int64_t* positions;
  const int64_t* cache_loc;
  const int32_t* commit_lens;   // null unless window mode
  int64_t loc_row_width;        // W in window mode, else 0
  const float* cos_sin;         // [max_pos, D]
  int64_t max_pos;
  int64_t pool_slots;
  const float* knorm;           // [L, D] fp32
  const void* bias;             // [N] or null
  float eps;
  uint32_t* status;             // device status word (DSPARK_FLAG_*)
  // work split: dp_tiles tiles go whole to the workers (CTAs or CTA pairs) in
  // waves; the other tiles' k-blocks (sk_units of them) are cut into
  // sk_workers equal contiguous ranges ("stream-K").  Two orders:
  //  - sk_first = 0: the whole tiles first, then the cut ranges; a cut tile is
  //    finished by the contributor holding its last k-block, which waits
  //    (bounded) for the others' parts; the others never wait
  //  - sk_first = 1: the cut ranges first, every part published; once all parts
  //    of a cut tile are published, each contributor sums and finishes its own
  //    share of the tile's rows, while its whole tiles run on the tensor cores
  int32_t dp_tiles;
  int64_t sk_units;
  int32_t sk_workers;
  int32_t sk_first;
  // optional order of the whole tiles: worker w's i-th whole tile is
  // dp_perm[w + i*workers] when that index is below dp_perm_n (else itself)
  int32_t dp_perm_n;
  // fused launch (combine_hidden_states then the write, ctx_kv_fused_kernel):
  // this problem's worker count; the grid-wide count of CTAs done with the
  // first problem (zero between launches); for the write, the first problem's
  // row sums of squares (rowsq, rowsq_stride, rowsq_n tiles) give each token
  // row's scale 1/sqrt(sum / norm_n + norm_eps)
  int32_t workers;
  int32_t* phase_count;
  int32_t rowsq_n;
  int32_t norm_n;
  float norm_eps;
  uint64_t* trace;              // null, or [gridDim.x][kTraceWords] timeline stamps
  float* workspace;             // [gridDim.x][2][kTileN/4][kTileM][4] fp32 partial tiles
  int32_t* counters;            // [gridDim.x] arrivals per cut tile, reset by the last one
  uint64_t wait_limit_ns;       // bound on any single in-kernel wait
  // waits for the parts other workers publish of a cut tile: the bound, and
  // how many arrivals beyond the real contributors they wait for (0; more
  // only in the timeout test, where no worker will reach the count)
  uint64_t split_wait_ns;
  int32_t split_wait_extra;
  int16_t dp_perm[kMaxDpPerm];
  void* k_pool[DSPARK_MAX_LAYERS];
  void* v_pool[DSPARK_MAX_LAYERS];
  int64_t k_stride[DSPARK_MAX_LAYERS];
  int64_t v_stride[DSPARK_MAX_LAYERS];
};

static_assert(sizeof(WriteParams) <= 4000, "kernel parameter space");

// Tiled tcgen05 path: one CTA per SM, 128-token x 256-column output tiles.
constexpr int kTileM = 128;
constexpr int kTileN = 256;
constexpr int kTileK = 64;     // one 128-byte swizzle row of 16-bit elements
constexpr int kTiledThreads = 384;   // 3 warpgroups: 2 epilogue, 1 control
constexpr int kLaunchRegs = 168;     // registers per thread at launch (65536 / 384, rounded down to 8)
constexpr int kGroupM = 8;     // m-blocks per raster group (L2 reuse of weight tiles)

// Output tile `tile` -> (token block, column block): tiles are rastered in
// groups of kGroupM token blocks so that weight tiles are reused from L2.
__host__ __device__ inline void tile_coords(int tile, int num_m, int num_n, int& m_blk, int& n_blk) {
  const int group_size = kGroupM * num_n;
  const int group = tile / group_size;
  const int first_m = group * kGroupM;
  const int gm = num_m - first_m < kGroupM ? num_m - first_m : kGroupM;
  const int r = tile - group * group_size;
  m_blk = first_m + r % gm;
  n_blk = r / gm;
}

constexpr int kTraceWords = 64;      // per CTA: start, end, items, 6 words per work item; last: split rows done
constexpr int kTraceItems = (kTraceWords - 3) / 6;
constexpr int kMinUnitsPerCta = 8;   // k-blocks: keeps small problems from over-splitting
constexpr int kMinSplitUnits = 2;    // k-blocks per worker of the leftover tiles (split-first order)
constexpr int kMaxLightShare = 8;    // k-blocks per V-tile worker when only those take the leftover
constexpr int kStreamAutoMaxTokens = 64;    // AUTO picks the weight-streaming kernel up to here,
constexpr int kStreamAutoCutMaxTokens = 128; // and up to here when CTA pairs would cut every tile


// Bytes of partial-tile workspace and arrival counters for a grid of `ctas`.
inline size_t workspace_bytes(int ctas) {
  return static_cast<size_t>(ctas) * 2 * kTileM * kTileN * sizeof(float);
}

// Work split of a problem of `tiles` output tiles with `num_kb` k-blocks
// each on up to `workers` workers; sets p.dp_tiles, p.sk_units, p.sk_workers
// and p.sk_first and returns the number of workers to launch.  In the order
// checked:
//  - fewer tiles than workers but at least half as many, with `whole_tiles`
//    (the tiled write): each tile goes whole to one worker and the other
//    workers stay idle.  Cut, every tile would be finished by adding a full
//    fp32 partial tile that another worker published, which costs more than
//    the idle workers' share of the products: at 256 tokens on 76 CTA pairs
//    (40 tiles) the finishers spent ~6.5 us adding the other part.
//  - one full wave and at most a third of a wave left over, with
//    `split_first` (kernels that implement it): the full wave runs whole tiles
//    and the leftover tiles are cut over the workers, at least kMinSplitUnits
//    k-blocks each, and computed first, so no worker ends on a split tile's
//    fixup.  Measured on GB300 against the other order: 10% faster with 4
//    leftover tiles on 76 pairs, 4% with 24; slower from about 44 (a tile then
//    has few contributors, each finishing many rows) and with two waves or
//    more (the other order's split-tile costs are the smaller there).
//  - other problems with fewer tiles than workers: every k-block is in the
//    stream-K range, spread over at most one worker per kMinUnitsPerCta
//    k-blocks
//  - otherwise: all but the last full wave run whole tiles and the rest (one
//    to two waves' worth) is cut over all workers
inline int plan_schedule(int tiles, int num_kb, int workers, bool split_first, WriteParams& p,
                         bool whole_tiles = false) {
  const int waves = tiles / workers;
  p.sk_first = 0;
  if (whole_tiles && tiles < workers && 2 * tiles >= workers) {
    p.dp_tiles = tiles;
    p.sk_units = 0;
    p.sk_workers = 0;
    return tiles;
  }
  if (split_first && waves == 1 && 3 * (tiles - workers) <= workers) {
    p.sk_first = 1;
    p.dp_tiles = waves * workers;
    p.sk_units = static_cast<int64_t>(tiles - p.dp_tiles) * num_kb;
    int64_t g = p.sk_units / kMinSplitUnits;
    if (g > workers) g = workers;
    if (g < 1) g = 1;
    p.sk_workers = static_cast<int32_t>(g);
    return workers;
  }
  p.dp_tiles = waves >= 2 ? (waves - 1) * workers : 0;
  p.sk_units = static_cast<int64_t>(tiles - p.dp_tiles) * num_kb;
  int grid = workers;
  if (p.dp_tiles == 0) {
    int64_t g = p.sk_units / kMinUnitsPerCta;
    if (g > workers) g = workers;
    if (g < 1) g = 1;
    grid = static_cast<int>(g);
  }
  p.sk_workers = grid;
  return grid;
}

// Split-first order with exactly one whole tile per worker: hand the leftover
// k-blocks only to the workers whose whole tile holds no K head (a V tile's
// epilogue has no norm and no rotation: it is the shorter one), so that both
// kinds of worker end together.  Reorders the whole tiles so that those
// workers come first (p.dp_perm) and narrows p.sk_workers to them; applied
// when each of them then takes kMinSplitUnits to kMaxLightShare k-blocks.
// The fused write only (head_dim 64 or 128).
inline void give_leftover_to_v_tiles(WriteParams& p, int workers) {
  if (!p.sk_first || p.D == 0 || p.dp_tiles != workers || workers > kMaxDpPerm) return;
  int16_t light[kMaxDpPerm], heavy[kMaxDpPerm];
  int nl = 0, nh = 0;
  for (int t = 0; t < p.dp_tiles; ++t) {
    int m_blk, n_blk;
    tile_coords(t, p.num_m, p.num_n, m_blk, n_blk);
    bool has_k = false;
    for (int seg = 0; seg < kTileN / p.D; ++seg) {
      const int c0 = n_blk * kTileN + seg * p.D;
      if (c0 < p.N && c0 % (2 * p.KV) < p.KV) has_k = true;
    }
    if (has_k)
      heavy[nh++] = static_cast<int16_t>(t);
    else
      light[nl++] = static_cast<int16_t>(t);
  }
  if (nl == 0 || nl >= p.sk_workers || p.sk_units < static_cast<int64_t>(nl) * kMinSplitUnits ||
      p.sk_units > static_cast<int64_t>(nl) * kMaxLightShare)
    return;
  p.sk_workers = nl;
  for (int w = 0; w < nl; ++w) p.dp_perm[w] = light[w];
  for (int w = 0; w < nh; ++w) p.dp_perm[nl + w] = heavy[w];
  p.dp_perm_n = p.dp_tiles;
}

// Launch the fused kernel for the bundle dtype (1 = bf16, 2 = fp16).  Returns
// the CUDA error of the launch.  launch_tiled: one CTA per 128 x 256 tile
// (grid = CTAs, num_m counts 128-token blocks, tmap_w box 256 rows);
// launch_pair: CTA pairs per 256 x 256 tile (grid = 2 x pairs, num_m counts
// 256-token blocks, tmap_w box 128 rows), the schedule planned over pairs.
cudaError_t launch_tiled(int device, int dtype, int head_dim, bool has_bias, const CUtensorMap& tmap_x,
                         const CUtensorMap& tmap_w, const WriteParams& p, int grid,
                         cudaStream_t stream);

cudaError_t launch_pair(int device, int dtype, int head_dim, bool has_bias, const CUtensorMap& tmap_x,
                        const CUtensorMap& tmap_w_half, const WriteParams& p, int grid,
                        cudaStream_t stream);

// Weight-streaming kernel for T <= 256 (weights as the MMA's M side).
// stream_plan: token padding, stage count and TMEM layout for T (false if T is
// out of range).  launch_stream: grid = CTAs, num_n = weight tiles of 128 rows,
// num_m = 1; tmap_x box rows = t_pad, tmap_w box 128 rows.
size_t stream_max_smem_bytes();
bool stream_plan(int64_t T, int* t_pad, int* stages, uint32_t* stage_b, uint32_t* acc_stride,
                 uint32_t* tmem_cols);
cudaError_t launch_stream(int device, int dtype, int head_dim, bool has_bias, const CUtensorMap& tmap_x,
                          const CUtensorMap& tmap_w_half, const WriteParams& p, int t_pad, int stages,
                          uint32_t stage_b, uint32_t acc_stride, uint32_t tmem_cols, int grid,
                          cudaStream_t stream);

// The same kernels in plain product mode: y[T, N] = x[T, K] . w[N, K]^T stored
// in the model dtype (p.y), with fp32 row sums of squares per 256-column tile
// (p.rowsq); tiles as launch_tiled (pair = false) or launch_pair.
cudaError_t launch_plain(int device, int dtype, const CUtensorMap& tmap_x, const CUtensorMap& tmap_w,
                         const WriteParams& p, int grid, bool pair, cudaStream_t stream);

// combine_hidden_states fused into the write, one launch of CTA pairs: p1 is
// main_proj in plain mode (token operand tmap_x1 = aux, weights tmap_w1 =
// main_proj with 128-row boxes; y and its row sums into p1.y / p1.rowsq), p
// the write whose token operand tmap_x is y and whose stacked weights are
// scaled by main_norm's weight.  grid = 2 x max(p1.workers, p.workers).
cudaError_t launch_fused(int device, int dtype, int head_dim, bool has_bias, const CUtensorMap& tmap_x1,
                         const CUtensorMap& tmap_w1, const WriteParams& p1, const CUtensorMap& tmap_x,
                         const CUtensorMap& tmap_w_half, const WriteParams& p, int grid, cudaStream_t stream);

// 2-D K-major operand map (api.cu): rows of `cols` 16-bit elements,
// `pitch_elems` apart; boxes of kTileK x box_rows with the 128-byte swizzle;
// out-of-range rows/columns read as zero.  False if the driver refuses it.
bool make_operand_map(CUtensorMap* map, const void* base, int dtype, uint64_t cols, uint64_t rows,
                      uint64_t pitch_elems, uint32_t box_rows);

// Workers that can be resident at once on `device` (0 if unknown): CTA pairs
// of the pair kernel, CTAs of the single-CTA kernel, CTAs of the streaming
// kernel with a launch's stage layout.  Grids never exceed them, since the
// split-tile waits assume that every CTA of a grid is resident.
int pair_workers(int device);
int single_workers(int device);
int stream_workers(int device, int stages, uint32_t stage_b);

// Validate the arguments of a write with bundle `b` and fill everything of p
// but the work split (dims, inputs, pools, bundle buffers, bounds).  Returns a
// dspark_status; nothing is enqueued.
int fill_write_params(const dspark_bundle* b, const void* ctx_hidden, int64_t T, int64_t hidden_row_stride,
                      int32_t hidden_dtype, const int64_t* positions, const float* cos_sin, int64_t max_pos,
                      const int64_t* cache_loc, const int32_t* commit_lens, int64_t loc_row_width,
                      int64_t num_windows, void* const* k_pools, void* const* v_pools,
                      const int64_t* k_row_strides, const int64_t* v_row_strides, int32_t pool_dtype,
                      int64_t pool_slots, WriteParams& p);

// Convert a [n] bf16 / fp16 / fp32 vector to fp32 (bundle packing).
cudaError_t launch_to_fp32(const void* src, int dtype, float* dst, int n, cudaStream_t stream);

}  // namespace dspark

// A packed bundle (dspark_pack_ctx_kv): the stacked K|V weights and their
// tensor maps, fp32 k_norm weights, and the scratch every write with it uses.
struct dspark_bundle {
  int device;
  int dtype;
  int L, H, NH, D, KV;
  int64_t N;
  int64_t w_pitch;      // elements between rows of w_all
  void* w_all;          // [N, w_pitch] in dtype
  void* bias;           // [N] in dtype or null
  float* knorm;         // [L, D] fp32
  uint32_t* status;     // device status word
  float* workspace;     // partial tiles of the stream-K split (workspace_bytes(sms))
  int32_t* counters;    // [sms] arrival counters, zero between launches
  int sms;              // SM count of the bundle's device
  uint64_t* trace;      // optional timeline buffer (dspark_set_trace_buffer)
  int variant;          // DSPARK_VARIANT_* (dspark_set_kernel_variant)
  int split_wait_extra;        // dspark_set_split_wait_test: arrivals no worker will make
  uint64_t split_wait_ns;      // bound on the waits for a cut tile's published parts
  CUtensorMap tmap_w_half;   // W_all with 128-row boxes (CTA-pair kernel)
  float eps;
  CUtensorMap tmap_w;
};
