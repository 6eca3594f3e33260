// Fused stacked-KV projection + K RMSNorm + table neox RoPE + pool scatter on
// tcgen05 tensor cores (sm_103a).
//
// One persistent CTA per SM (or CTA pair per SM pair) walks 128-token (256
// for a pair) x 256-column tiles of the stacked output Y = ctx_hidden .
// W_all^T (W_all rows: l0:K, l0:V, l1:K, ...; sglang PR #31986 summary page,
// _stacked_ctx_kv_params).  256 columns are whole heads (D = 64 or 128), so
// each tile's epilogue can finish its heads alone.  The work split
// (plan_schedule, internal.h) mixes whole tiles with tiles whose k-blocks are
// cut between workers; a cut tile is finished from the published fp32 parts
// either by the owner of its last k-block (whole tiles first) or row-wise by
// every contributor (split-first, for one wave plus a small leftover).
//
// With tcgen05.mma.cta_group::2 the leader CTA of a pair issues 256x256x16
// MMAs over both CTAs' operand halves; commits are multicast to both.
//
//   warps 0..7  epilogue, two warpgroups that take alternate heads of a tile:
//               each thread owns one token row of the accumulator
//               (tcgen05.ld 32x32b), so the RMSNorm sum of squares is a
//               per-thread sum and the neox pair (i, i + D/2) sits in the same
//               thread's registers; then 16-byte stores into the pool row
//   warp 8      TMA producer: X and W_all K-slices into a smem ring (4 stages,
//               or 5 for CTA pairs)
//   warp 9      MMA issuer: tcgen05.mma 128x256x16 (256x256x16 for a pair)
//               into one of two TMEM accumulators (2 x 256 fp32 columns);
//               owns TMEM alloc/free
//   warps 10,11 idle (they complete the control warpgroup)
// Registers are moved to the epilogue with setmaxnreg (control warpgroup 40,
// epilogue warpgroups 232 per thread).
//
// The epilogue of tile i overlaps the MMAs of tile i+1 (double-buffered TMEM).
// Per-token rules (sglang PR #31847 summary page, fused_kv_norm_rope_write):
// loc < 0 skips the token; in window mode column t mod W must be below
// commit_lens[t div W].
#include <cuda_bf16.h>
#include <atomic>
#include <cuda_fp16.h>

#include "internal.h"
#include "kernel_common.cuh"
#include "ptx.cuh"

namespace dspark {
namespace {

// Operand staging of one CTA.  Single-CTA tiles are 128 tokens x 256 columns;
// pair tiles are 256 tokens x 256 columns computed by two CTAs of a cluster
// with tcgen05.mma.cta_group::2: each CTA holds its 128 token rows of X and
// half (128 rows) of the W tile, so a stage is 32 KB; five of them (160 KB)
// measured faster than six on the large workloads (a smaller shared-memory
// carve-out leaves more L1), and no slower at 512 tokens.
template <bool kPair>
struct Geo {
  static constexpr int kTileRows = kPair ? 2 * kTileM : kTileM;   // token rows of a work tile
  static constexpr int kBRows = kPair ? kTileN / 2 : kTileN;       // W rows per CTA per stage
  static constexpr uint32_t kStageA = kTileM * kTileK * 2;         // 16 KB
  static constexpr uint32_t kStageB = kBRows * kTileK * 2;         // 16 KB (pair) or 32 KB
  static constexpr int kStages = kPair ? 5 : 4;
  static constexpr uint32_t kRingBytes = kStages * (kStageA + kStageB);
};
constexpr int kMaxStages = 5;
static_assert(Geo<false>::kStages <= kMaxStages && Geo<true>::kStages <= kMaxStages, "barrier arrays");
constexpr uint32_t kAccCols = kTileN;                    // fp32 columns per accumulator
constexpr uint32_t kTmemCols = 2 * kAccCols;             // double buffer = 512 (all of TMEM)
constexpr int kEpiWarps = 8;                             // two epilogue warpgroups
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint32_t kRegsControl = 40;
constexpr uint32_t kRegsEpilogue = 232;
static_assert(kTiledThreads == 384, "three warpgroups");
static_assert(128 * kRegsControl + 256 * kRegsEpilogue == 384 * kLaunchRegs,
              "the register split must use exactly the launch allocation");

constexpr int kRedBatch = 8;   // parts of a split tile whose loads are in flight together

struct SmemBarriers {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t drain;
  uint64_t fix[2];      // per epilogue group: bulk copies of a split tile's other parts landed
  float ss_x[kTileM];   // plain mode: the second group's row sums of squares; split rows: per-warp sums
  uint32_t tmem_base;
  int abort;
  int last_arrival;   // finisher's early look: every other part of its cut tile already published
};

// Whether token t's rows are written, with its pool slot and position (sglang
// PR #31847 summary page, fused_kv_norm_rope_write: loc < 0 skips the token;
// in window mode column t mod W must be below commit_lens[t div W]).  Range
// errors are flagged (by the caller's chosen thread) and skip the token.
__device__ __forceinline__ bool token_write(const WriteParams& p, int64_t t, bool raise, int64_t& loc,
                                            int64_t& pos) {
  loc = 0;
  pos = 0;
  if (t >= p.T) return false;
  loc = p.cache_loc[t];
  if (loc < 0) return false;
  if (p.loc_row_width > 0) {
    const int64_t b = t / p.loc_row_width;
    if (t - b * p.loc_row_width >= static_cast<int64_t>(p.commit_lens[b])) return false;
  }
  pos = p.positions[t];
  if (pos < 0 || pos >= p.max_pos) {
    if (raise) flag(p, DSPARK_FLAG_POS_RANGE);
    return false;
  }
  if (loc >= p.pool_slots) {
    if (raise) flag(p, DSPARK_FLAG_LOC_RANGE);
    return false;
  }
  return true;
}

__device__ __forceinline__ float4 add4(float4 a, float4 b) {
  return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}

// Give up after a wait ran out: report the timeout and stop this CTA's work.
// A pair stops both CTAs (the flag is also set in the peer's shared memory):
// their loads complete on the leader's barriers and are released by the
// leader's MMAs, so one CTA alone cannot wind the pipeline down.  The peer is
// still resident here: both CTAs meet at a cluster barrier before exiting.
template <bool kPair>
__device__ __forceinline__ void abort_work(const WriteParams& p, volatile int* abort_flag) {
  *abort_flag = 1;
  if constexpr (kPair)
    st_shared_cluster_u32(mapa_shared(smem_u32(const_cast<int*>(abort_flag)), cluster_ctarank() ^ 1u), 1u);
  flag(p, DSPARK_FLAG_TIMEOUT);
}

// After an abort a pair's producers may have stopped at different stages: a
// leader barrier armed for bytes the peer never loaded, or a peer load the
// leader's MMA never released, is never observed complete.  Their drain then
// ends on this bound rather than the full wait bound: every load in question
// was issued before the abort, and a tile load lands within microseconds.
constexpr uint64_t kPairAbortDrainNs = 200000;

// 1/rms over the first problem's columns of token row t (fused write): the
// row's sums of squares per 256-column tile, added in a fixed order.
__device__ __forceinline__ float row_inv_rms(const WriteParams& p, int64_t t) {
  if (t >= p.T) return 0.f;
  const float* r = p.rowsq + t * p.rowsq_stride;
  float ss = 0.f;
  for (int j = 0; j < p.rowsq_n; ++j) ss += r[j];
  return 1.0f / sqrtf(ss / static_cast<float>(p.norm_n) + p.norm_eps);
}

// Generic-proxy stores to global memory before later tensor-memory (TMA)
// loads of them, by this or another SM (with a release / acquire between).
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Fused launch: wait (bounded) until every CTA is done with the first
// problem, then order the loads that follow after it.
__device__ __forceinline__ bool wait_first_problem(const WriteParams& p, volatile int* abort_flag) {
  const int target = static_cast<int>(gridDim.x);
  const uint64_t t0 = global_timer_ns();
  while (ld_acquire_gpu(p.phase_count) < target) {
    if (*abort_flag != 0 || global_timer_ns() - t0 > p.wait_limit_ns) return false;
    __nanosleep(128);
  }
  fence_proxy_async_global();
  return true;
}

// The cut tiles of the split-first schedule (the tiles left over after the
// full wave, whose k-blocks are spread over the workers).  Every contributor
// publishes its part before any is read; then contributor i of n finishes
// rows [i*rv/n, (i+1)*rv/n) of its CTA's rows of the tile: it sums them over
// all n parts in ascending contributor order (so the bits do not depend on
// arrival order) and runs the epilogue on them -- K RMSNorm and RoPE and the
// pool scatter, or the plain product's store and row sums of squares.
//
// Rows go 8 at a time.  Lane l of a warp takes row l % 8 and, in each of two
// 16-column blocks of the tile, the float4 column group l / 8: the loads of a
// warp are four 128-byte runs of the workspace's [column group][row] layout.
// A warp's two blocks are the two halves' blocks of one rotation pair (block b
// and b + D/32 of a head), so RoPE stays inside a lane; the warps of a head
// add their parts of the sum of squares through shared memory.  It runs on the
// epilogue warps while the CTA's whole tile is on the tensor cores.  Returns
// false if a wait ran out.
template <typename E, int D, bool kBias, bool kPair, bool kRowScale>
__device__ bool finish_split_rows(const WriteParams& p, int wid, int nw, uint32_t rank, float* ss_part,
                                  volatile int* abort_flag) {
  using G = Geo<kPair>;
  constexpr bool kPlain = D == 0;
  constexpr int kRows = 8;                                    // rows per pass
  constexpr int kBH = kPlain ? 2 : D / 16;                    // 16-column blocks per head
  constexpr int kWPH = kPlain ? 1 : kBH / 2;                  // warps per head
  const int etid = threadIdx.x, warp = etid / 32, lane = etid % 32;
  const int rr = lane % kRows, gs = lane / kRows;
  const int hd = warp / kWPH;                                 // head of the tile (write mode)
  const int b1 = kPlain ? 2 * warp : kBH * hd + warp % kWPH;  // this warp's two blocks
  const int b2 = kPlain ? 2 * warp + 1 : b1 + kBH / 2;
  const int g1 = 4 * b1 + gs, g2 = 4 * b2 + gs;               // float4 column groups of the lane
  const WorkIter range = work_begin(p, wid, nw);
  if (range.cur <= range.start) return true;
  const int64_t t_lo = range.start / p.num_kb, t_hi = (range.cur - 1) / p.num_kb;
  auto cta_of = [&](int c) { return kPair ? 2 * c + static_cast<int>(rank) : c; };
  for (int64_t st = t_lo; st <= t_hi; ++st) {
    const int64_t u0 = st * p.num_kb;
    const int cf = sk_owner(p, u0), cl = sk_owner(p, u0 + p.num_kb - 1);
    if (cf == cl) continue;   // a whole tile: finished from TMEM
    const int n = cl - cf + 1;
    int32_t* counter = p.counters + cta_of(cl);
    bool ok = true;
    if (etid == 0) {
      ok = wait_count(counter, n + p.split_wait_extra, abort_flag, p.split_wait_ns);
      // second round: the last contributor past the wait resets the counter
      // for the next launch (every contributor has already read it as n)
      if (ok && atom_add_acq_rel_gpu(counter, 1) == 2 * n - 1) *counter = 0;
    }
    if (!named_barrier_and(1, kEpiThreads, ok)) return false;
    int m_blk, n_blk;
    tile_coords(p.dp_tiles + static_cast<int>(st), p.num_m, p.num_n, m_blk, n_blk);
    const int64_t row0 = static_cast<int64_t>(m_blk) * G::kTileRows + static_cast<int64_t>(rank) * kTileM;
    const int64_t left = static_cast<int64_t>(p.T) - row0;
    const int rv = left <= 0 ? 0 : (left < kTileM ? static_cast<int>(left) : kTileM);
    const int i = wid - cf;
    const int lo = i * rv / n, hi = (i + 1) * rv / n;
#pragma unroll 1
    for (int r0 = lo; r0 < hi; r0 += kRows) {
      const int row = r0 + rr;
      const bool valid = row < hi;
      float4 s1 = make_float4(0.f, 0.f, 0.f, 0.f), s2 = s1;
#pragma unroll 1
      for (int c = cf; c <= cl; c += kRedBatch) {
        float4 q1[kRedBatch], q2[kRedBatch];
#pragma unroll
        for (int j = 0; j < kRedBatch; ++j) {
          q1[j] = q2[j] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (valid && c + j <= cl) {
            const float4* src = reinterpret_cast<const float4*>(ws_slot(p, cta_of(c + j), c + j == cf ? 1 : 0));
            q1[j] = __ldcg(src + g1 * kTileM + row);
            q2[j] = __ldcg(src + g2 * kTileM + row);
          }
        }
#pragma unroll
        for (int j = 0; j < kRedBatch; ++j) {
          if (c + j <= cl) {
            s1 = c + j == cf ? q1[j] : add4(s1, q1[j]);
            s2 = c + j == cf ? q2[j] : add4(s2, q2[j]);
          }
        }
      }
      const int64_t t = row0 + row;
      if constexpr (kPlain) {
        // stored rounded to the model dtype; the sum of squares is taken over
        // the stored values
        const float4 sv[2] = {s1, s2};
        const int gg[2] = {g1, g2};
        float ss = 0.f;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const uint32_t w0 = ElemOps<E>::pack(sv[k].x, sv[k].y), w1 = ElemOps<E>::pack(sv[k].z, sv[k].w);
          float a, b, c2, d;
          ElemOps<E>::unpack(w0, a, b);
          ElemOps<E>::unpack(w1, c2, d);
          const int col = n_blk * kTileN + 4 * gg[k];
          if (col < p.N) {
            ss = fmaf(a, a, fmaf(b, b, fmaf(c2, c2, fmaf(d, d, ss))));
            if (valid)
              *reinterpret_cast<uint2*>(reinterpret_cast<E*>(p.y) + t * p.y_stride + col) = make_uint2(w0, w1);
          }
        }
        ss += __shfl_xor_sync(0xffffffffu, ss, 8);
        ss += __shfl_xor_sync(0xffffffffu, ss, 16);
        if (gs == 0) ss_part[warp * kRows + rr] = ss;
        named_barrier(1, kEpiThreads);
        if (warp == 0 && lane < kRows && r0 + lane < hi) {
          float tot = 0.f;
#pragma unroll
          for (int w = 0; w < kEpiWarps; ++w) tot += ss_part[w * kRows + lane];
          p.rowsq[(row0 + r0 + lane) * p.rowsq_stride + n_blk] = tot;
        }
      } else {
        constexpr int kHalf = D / 2;
        const int i1 = 4 * g1 - hd * D;   // column inside the head (first half); partner i1 + D/2
        const int c0 = n_blk * kTileN + hd * D;
        const bool col_ok = c0 < p.N;
        int64_t loc = 0, pos = 0;
        const bool write = valid && col_ok && token_write(p, t, warp == 0 && gs == 0, loc, pos);
        const int cv = col_ok ? c0 : 0;
        const int layer = cv / (2 * p.KV);
        const int r = cv - layer * 2 * p.KV;
        const bool is_v = r >= p.KV;
        const int head = (is_v ? r - p.KV : r) / D;
        float x1[4] = {s1.x, s1.y, s1.z, s1.w}, x2[4] = {s2.x, s2.y, s2.z, s2.w};
        if (kRowScale) {
          const float rs = row_inv_rms(p, t);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            x1[e] *= rs;
            x2[e] *= rs;
          }
        }
        if (kBias && col_ok) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            x1[e] += ElemOps<E>::load(p.bias, c0 + i1 + e);
            x2[e] += ElemOps<E>::load(p.bias, c0 + kHalf + i1 + e);
          }
        }
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) ss = fmaf(x1[e], x1[e], fmaf(x2[e], x2[e], ss));
        ss += __shfl_xor_sync(0xffffffffu, ss, 8);
        ss += __shfl_xor_sync(0xffffffffu, ss, 16);
        if (gs == 0) ss_part[warp * kRows + rr] = ss;
        named_barrier(1, kEpiThreads);
        if (!is_v) {
          float tot = 0.f;
#pragma unroll
          for (int k = 0; k < kWPH; ++k) tot += ss_part[(hd * kWPH + k) * kRows + rr];
          const float inv = rsqrtf(tot * (1.0f / D) + p.eps);
          const float* w = p.knorm + static_cast<int64_t>(layer) * D;
          const float4 w1 = *reinterpret_cast<const float4*>(w + i1);
          const float4 w2 = *reinterpret_cast<const float4*>(w + kHalf + i1);
          const float* cs = p.cos_sin + (write ? pos : 0) * D;
          const float4 c4 = *reinterpret_cast<const float4*>(cs + i1);
          const float4 s4 = *reinterpret_cast<const float4*>(cs + kHalf + i1);
          const float wa[4] = {w1.x, w1.y, w1.z, w1.w}, wb[4] = {w2.x, w2.y, w2.z, w2.w};
          const float cc[4] = {c4.x, c4.y, c4.z, c4.w}, sn[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float a = x1[e] * inv * wa[e];
            const float b = x2[e] * inv * wb[e];
            x1[e] = a * cc[e] - b * sn[e];
            x2[e] = b * cc[e] + a * sn[e];
          }
        }
        if (write) {
          E* dst = is_v ? reinterpret_cast<E*>(p.v_pool[layer]) + loc * p.v_stride[layer] + head * D
                        : reinterpret_cast<E*>(p.k_pool[layer]) + loc * p.k_stride[layer] + head * D;
          *reinterpret_cast<uint2*>(dst + i1) = make_uint2(ElemOps<E>::pack(x1[0], x1[1]), ElemOps<E>::pack(x1[2], x1[3]));
          *reinterpret_cast<uint2*>(dst + kHalf + i1) =
              make_uint2(ElemOps<E>::pack(x2[0], x2[1]), ElemOps<E>::pack(x2[2], x2[3]));
        }
      }
      named_barrier(1, kEpiThreads);   // ss_part is rewritten by the next pass
    }
  }
  return true;
}

// The kernel body.  One problem (p with its operand maps), or with kFused two
// in sequence in one launch: first p1 (the plain product main_proj, whose
// output y is p's token operand), then p, each walking its own schedule over
// the same pipeline; a grid-wide count of CTAs done with p1 orders p1's
// stores before p's loads of them.
template <typename E, int D, bool kBias, bool kPair, bool kFused>
__device__ __forceinline__ void tiled_body(const CUtensorMap& tmap_x1, const CUtensorMap& tmap_w1,
                                           const WriteParams& p1, const CUtensorMap& tmap_x,
                                           const CUtensorMap& tmap_w, const WriteParams& p) {
  using G = Geo<kPair>;
  constexpr int kStages = G::kStages;
  constexpr uint32_t kStageBytesA = G::kStageA;
  constexpr uint32_t kStageBytesB = G::kStageB;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // operand stages must sit on 1024-byte boundaries (128-byte swizzle atoms)
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* smem_a = smem;
  uint8_t* smem_b = smem + kStages * kStageBytesA;
  SmemBarriers* bars = reinterpret_cast<SmemBarriers*>(smem + G::kRingBytes);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  volatile int* abort_flag = &bars->abort;
  // a pair's two CTAs share one work sequence; rank 0 (the leader) issues MMAs
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  const int wid = kPair ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int nw = kPair ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&bars->full[s]), 1);
      mbar_init(smem_u32(&bars->empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&bars->tmem_full[b]), 1);
      // one arrival per epilogue warp (of both CTAs for a pair: the leader's
      // barrier is the one its MMA waits on)
      mbar_init(smem_u32(&bars->tmem_empty[b]), kPair ? 2 * kEpiWarps : kEpiWarps);
    }
    mbar_init(smem_u32(&bars->drain), 1);
    mbar_init(smem_u32(&bars->fix[0]), 1);
    mbar_init(smem_u32(&bars->fix[1]), 1);
    bars->abort = 0;
    fence_barrier_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tmap_x);
    tma_prefetch_desc(&tmap_w);
    if (kFused) {
      tma_prefetch_desc(&tmap_x1);
      tma_prefetch_desc(&tmap_w1);
    }
  }
  if (warp == kMmaWarp) {
    if (kPair) {
      tmem_alloc_pair(smem_u32(&bars->tmem_base), kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(&bars->tmem_base), kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncwarp();
  if (kPair) {
    cluster_sync();   // the peer's loads and commits target this CTA's barriers
  } else {
    __syncthreads();
  }
  tc_fence_after();
  const uint32_t tmem_base = bars->tmem_base;
  uint64_t* trace = p.trace != nullptr ? p.trace + static_cast<size_t>(blockIdx.x) * kTraceWords : nullptr;
  if (trace != nullptr && threadIdx.x == 0) trace[0] = global_timer_ns();

  if (warp >= kEpiWarps) {
    regs_decrease<kRegsControl>();
    if (warp == kProducerWarp) {
      // ---------------------------------------------------------- producer
      if (lane == 0) {
        // A weight tile is read once per token block.  When every token block
        // falls in one raster group (num_m <= kGroupM) those reads come close
        // together, and evict_first keeps the weights from pushing other lines
        // out of L2 (with a dirty L2 each eviction is a DRAM write): decode512
        // 45.2 -> 42.3 us.  With more token blocks the weights are kept
        // (evict_last) for the later groups.  The token rows are read by every
        // column block of their group: evict_last.
        int stage = 0;
        uint32_t phase = 0;
        uint32_t uses[kStages] = {};
        bool ok = true;
        for (int ph = kFused ? 0 : 1; ph < 2 && ok; ++ph) {
        const WriteParams& wp = ph == 0 ? p1 : p;
        const CUtensorMap* tx = ph == 0 ? &tmap_x1 : &tmap_x;
        const CUtensorMap* tw = ph == 0 ? &tmap_w1 : &tmap_w;
        const int nwq = kFused ? wp.workers : nw;
        if (kFused && wid >= nwq) continue;
        // the fused second problem reads the first one's output: every CTA
        // must be done with the first one
        if (kFused && ph == 1 && !wait_first_problem(p, abort_flag)) {
          ok = false;
          break;
        }
        const uint64_t pol_w = wp.num_m <= kGroupM ? l2_policy_evict_first() : l2_policy_evict_last();
        const uint64_t pol_x = l2_policy_evict_last();
        WorkIter it = work_begin(wp, wid, nwq);
        int tile, kb0, kb1;
        while (ok && work_next(wp, it, tile, kb0, kb1)) {
          int m_blk, n_blk;
          tile_coords(tile, wp.num_m, wp.num_n, m_blk, n_blk);
          const int a_row = m_blk * G::kTileRows + static_cast<int>(rank) * kTileM;
          const int b_row = n_blk * kTileN + static_cast<int>(rank) * G::kBRows;
          for (int kb = kb0; kb < kb1; ++kb) {
            const bool got = kPair ? mbar_wait_cluster(smem_u32(&bars->empty[stage]), phase ^ 1u,
                                                       abort_flag, wp.wait_limit_ns)
                                   : mbar_wait(smem_u32(&bars->empty[stage]), phase ^ 1u,
                                               abort_flag, wp.wait_limit_ns);
            if (!got) {
              ok = false;
              break;
            }
            const uint32_t full = smem_u32(&bars->full[stage]);
            if (kPair) {
              // both CTAs' bytes complete on the leader's barrier
              if (leader) mbar_arrive_expect_tx(full, 2 * (kStageBytesA + kStageBytesB));
              const uint32_t full_leader = mapa_shared(full, 0);
              tma_load_2d_pair(smem_u32(smem_a + stage * kStageBytesA), tx, kb * kTileK, a_row,
                               full_leader, pol_x);
              tma_load_2d_pair(smem_u32(smem_b + stage * kStageBytesB), tw, kb * kTileK, b_row,
                               full_leader, pol_w);
            } else {
              mbar_arrive_expect_tx(full, kStageBytesA + kStageBytesB);
              tma_load_2d(smem_u32(smem_a + stage * kStageBytesA), tx, kb * kTileK, a_row, full,
                          pol_x);
              tma_load_2d(smem_u32(smem_b + stage * kStageBytesB), tw, kb * kTileK, b_row, full,
                          pol_w);
            }
            ++uses[stage];
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
        }
        if (!ok) abort_work<kPair>(p, abort_flag);
        // every load issued must land before the CTA may exit (bounded by time
        // only: an abort must not cut this wait short).  A pair's peer sees its
        // loads land only through the leader's MMA releasing the stage.
        int never = 0;
        const bool short_drain = kPair && *abort_flag != 0;
        const uint64_t t_end = global_timer_ns() + (short_drain ? kPairAbortDrainNs : p.wait_limit_ns);
#pragma unroll
        for (int s = 0; s < kStages; ++s) {
          if (uses[s] == 0) continue;
          const uint64_t now = global_timer_ns();
          const uint64_t lim = short_drain ? (now < t_end ? t_end - now : 0) : p.wait_limit_ns;
          if (!kPair)
            mbar_wait(smem_u32(&bars->full[s]), (uses[s] - 1u) & 1u, &never, lim);
          else if (leader)
            mbar_wait_cluster(smem_u32(&bars->full[s]), (uses[s] - 1u) & 1u, &never, lim);
          else
            mbar_wait_cluster(smem_u32(&bars->empty[s]), (uses[s] - 1u) & 1u, &never, lim);
        }
      }
    } else if (warp == kMmaWarp) {
      // ---------------------------------------------------------- MMA issuer
      if (lane == 0 && leader) {
        constexpr uint32_t idesc = f16_instr_desc(ElemOps<E>::kFmt, G::kTileRows, kTileN);
        int stage = 0;
        uint32_t phase = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        bool ok = true;
        bool issued = false;
        for (int ph = kFused ? 0 : 1; ph < 2 && ok; ++ph) {
        const WriteParams& wp = ph == 0 ? p1 : p;
        const int nwq = kFused ? wp.workers : nw;
        if (kFused && wid >= nwq) continue;
        WorkIter it = work_begin(wp, wid, nwq);
        int tile, kb0, kb1;
        while (ok && work_next(wp, it, tile, kb0, kb1)) {
          if (!mbar_wait_cluster(smem_u32(&bars->tmem_empty[acc]), acc_phase ^ 1u, abort_flag,
                                 wp.wait_limit_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + acc * kAccCols;
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!mbar_wait_cluster(smem_u32(&bars->full[stage]), phase, abort_flag, wp.wait_limit_ns)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a0 = smem_u32(smem_a + stage * kStageBytesA);
            const uint32_t b0 = smem_u32(smem_b + stage * kStageBytesB);
#pragma unroll
            for (int k = 0; k < kTileK / 16; ++k) {
              // advancing 16 elements along K = 32 bytes inside the swizzle atom
              const uint64_t ad = sw128_kmajor_desc(a0 + k * 32), bd = sw128_kmajor_desc(b0 + k * 32);
              const uint32_t accum = (kb != kb0 || k != 0) ? 1u : 0u;
              if (kPair)
                umma_f16_pair(d_tmem, ad, bd, idesc, accum);
              else
                umma_f16(d_tmem, ad, bd, idesc, accum);
            }
            issued = true;
            if (kPair)
              umma_commit_pair(smem_u32(&bars->empty[stage]), 0x3);
            else
              umma_commit(smem_u32(&bars->empty[stage]));
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          if (kPair)
            umma_commit_pair(smem_u32(&bars->tmem_full[acc]), 0x3);
          else
            umma_commit(smem_u32(&bars->tmem_full[acc]));
          if (++acc == 2) {
            acc = 0;
            acc_phase ^= 1u;
          }
        }
        }
        if (!ok) abort_work<kPair>(p, abort_flag);
        if (issued) {
          // all MMAs issued by this thread complete before TMEM is released
          if (kPair)
            umma_commit_pair(smem_u32(&bars->drain), 0x1);
          else
            umma_commit(smem_u32(&bars->drain));
          int never = 0;
          mbar_wait(smem_u32(&bars->drain), 0, &never, p.wait_limit_ns);
        }
      }
    }
  } else {
    regs_increase<kRegsEpilogue>();
    // ------------------------------------------------------------ epilogue
    // D == 0: plain product mode (main_proj of combine_hidden_states): the
    // tile is stored in the model dtype with per-row sums of squares of the
    // stored values; no tokens, pools or heads are involved
    constexpr int kHalf = D / 2;
    // head width of the write's code paths (never run with D == 0: the plain
    // mode takes its own branch)
    constexpr int kD = D == 0 ? 128 : D;
    // cos/sin staging for the last item: measured to pay off for D = 128 only
    constexpr bool kStageCs = D == 128;
    constexpr uint32_t kCsBytes = kStageCs ? kTileM * D * 4 : 0;
    static_assert(kCsBytes <= G::kRingBytes / 2, "cos/sin staging leaves room for the fixup");
    constexpr int kChunks = kTileN / 32;            // 32-column chunks of a tile
    const int group = warp / 4;                     // warpgroup 0 or 1
    const int quarter = warp % 4;                   // TMEM lanes this warp may read
    const int row = quarter * 32 + lane;            // token row inside the tile
    const int etid = threadIdx.x;                   // 0..255 among the epilogue threads
    const int ch_lo = group * (kChunks / 2);        // this group's chunks of a cut tile
    const int ch_hi = ch_lo + kChunks / 2;
    int acc = 0;
    uint32_t acc_phase = 0;
    uint32_t fix_phase = 0;   // parity of this group's fix barrier
    int item = 0;
    bool ep_abort = false;
    for (int ph = kFused ? 0 : 1; ph < 2 && !ep_abort; ++ph) {
    const WriteParams& wp = ph == 0 ? p1 : p;
    const int nwq = kFused ? wp.workers : nw;
    // D == 0, or the first problem of a fused launch: plain product mode
    const bool plain = D == 0 || (kFused && ph == 0);
    if (kFused && ph == 1) {
      // the row scales of the second problem are the first one's row sums
      const bool got = wait_first_problem(p, abort_flag);
      if (!named_barrier_and(1, kEpiThreads, got)) {
        if (etid == 0) abort_work<kPair>(p, abort_flag);
        break;
      }
    }
    WorkIter it = work_begin(wp, wid, kFused && wid >= nwq ? 1 : nwq);
    if (kFused && wid >= nwq) it.dp_tile = wp.dp_tiles, it.cur = it.start = 0;   // no work in this problem
    int tile, kb0, kb1;
    while (work_next(wp, it, tile, kb0, kb1)) {
      int m_blk, n_blk;
      tile_coords(tile, wp.num_m, wp.num_n, m_blk, n_blk);
      // split-first schedule: after the last part of the stream-K range is
      // published, finish this worker's share of its cut tiles
      const bool reduce_after = wp.sk_first && tile >= wp.dp_tiles && it.cur <= it.start;
      bool final_item;
      {
        WorkIter peek = it;
        int t2, a2, b2;
        final_item = !work_next(wp, peek, t2, a2, b2);
      }
      // ---- per-token decision (same for every head of the tile); it does not
      // depend on the accumulator, so it runs while the MMAs are in flight
      const int64_t row0 = static_cast<int64_t>(m_blk) * G::kTileRows + static_cast<int64_t>(rank) * kTileM;
      const int64_t t = row0 + row;
      int64_t loc = 0, pos = 0;
      const bool write = !plain && token_write(wp, t, group == 0, loc, pos);
      // fused second problem: this token row's 1/rms of y (main_norm)
      const float rs = (kFused && !plain) ? row_inv_rms(wp, t) : 1.f;
      if (write) {
        // the K heads of this tile will read this token's cos/sin row
        const char* cs_row = reinterpret_cast<const char*>(wp.cos_sin + pos * D);
        for (int b = group * 128; b < D * 4; b += 256) prefetch_l2(cs_row + b);
      }
      // A tile cut between workers (whole-tiles-first order) is finished by
      // the contributor that holds its last k-block: that piece is the last
      // item of its backward walk.  The other contributors publish their parts
      // and never wait; the finisher waits (bounded) for them, so it never
      // spends a dump on its own part.  Waits only point to lower-numbered
      // workers and every CTA is resident (at most one per SM), so they end.
      // The finisher looks now, while its MMAs run, whether the other parts
      // are already published (read after the barrier below).
      const bool cut = kb0 != 0 || kb1 != wp.num_kb;
      int c_first = 0, c_last = 0;
      if (cut) {
        const int64_t u0 = static_cast<int64_t>(tile - wp.dp_tiles) * wp.num_kb;
        c_first = sk_owner(wp, u0);
        c_last = sk_owner(wp, u0 + wp.num_kb - 1);
      }
      auto cta_of = [&](int c) { return kPair ? 2 * c + static_cast<int>(rank) : c; };
      const bool designated = cut && !wp.sk_first && wid == c_last;
      if (designated && etid == 0) {
        const int seen = ld_acquire_gpu(wp.counters + cta_of(c_last));
        *reinterpret_cast<volatile int*>(&bars->last_arrival) = seen == c_last - c_first + wp.split_wait_extra;
      }
      // the outcome must be warp-uniform: tcgen05.ld below is .sync.aligned
      const bool got = mbar_wait_cluster(smem_u32(&bars->tmem_full[acc]), acc_phase, abort_flag,
                                         wp.wait_limit_ns);
      // stamps come from the thread of row 0 of the first group
      uint64_t* tr =
          (trace != nullptr && etid == 0 && item < kTraceItems) ? trace + 3 + 6 * item : nullptr;
      if (tr != nullptr) {
        tr[0] = static_cast<uint64_t>(tile);
        tr[1] = (static_cast<uint64_t>(kb0) << 16) | static_cast<uint64_t>(kb1);
        tr[2] = global_timer_ns();
        tr[3] = tr[4] = 0;
      }
      ++item;
      // every epilogue warp takes the same decision (they meet at named
      // barriers below), and every wait ends within its time bound
      if (!named_barrier_and(1, kEpiThreads, got)) {
        if (etid == 0) abort_work<kPair>(wp, abort_flag);
        ep_abort = true;
        break;
      }
      tc_fence_after();
      const uint32_t t_row = tmem_base + acc * kAccCols + (static_cast<uint32_t>(quarter * 32) << 16);

      // After the CTA's last MMA the operand ring is idle.  A last item with
      // 128-wide K heads stages its tokens' cos/sin rows there first (each
      // group copies half of every row; 16-byte units XOR-swizzled by row so
      // that the row-per-thread reads below are free of bank conflicts): the
      // rotation then reads shared memory instead of waiting on L2 per chunk.
      bool tile_has_k = false;
      if (!plain) {
        for (int seg = 0; seg < kTileN / kD; ++seg) {
          const int c0 = n_blk * kTileN + seg * kD;
          if (c0 < wp.N && c0 % (2 * wp.KV) < wp.KV) tile_has_k = true;
        }
      }
      const bool cs_stage = kStageCs && final_item && tile_has_k;
      auto stage_cs = [&]() {
        if (!cs_stage || !write) return;
        const char* src = reinterpret_cast<const char*>(wp.cos_sin + pos * D);
        const uint32_t dst = smem_u32(smem) + static_cast<uint32_t>(row) * (D * 4);
        constexpr int kUnits = D / 4;   // 16-byte units per row
#pragma unroll
        for (int u = group * (kUnits / 2); u < (group + 1) * (kUnits / 2); ++u)
          cp_async16(dst + static_cast<uint32_t>((u ^ (row & 7)) * 16), src + u * 16);
      };

      // ---- a tile cut between workers: publish this part, or (the
      // finisher) wait for the other parts and add them in contributor order
      bool finish = true;
      if (cut) {
        int32_t* counter = wp.counters + cta_of(c_last);
        finish = designated;
        if (designated) {
          const bool early = *reinterpret_cast<volatile int*>(&bars->last_arrival) != 0;
          bool ok = true;
          if (!early && etid == 0)
            ok = wait_count(counter, c_last - c_first + wp.split_wait_extra, abort_flag, wp.split_wait_ns);
          if (!named_barrier_and(1, kEpiThreads, ok)) {
            if (etid == 0) abort_work<kPair>(wp, abort_flag);
            ep_abort = true;
            break;
          }
          if (etid == 0) *counter = 0;   // no other contributor touches it again
        } else {
          float4* mine = reinterpret_cast<float4*>(ws_slot(wp, cta_of(wid), kb0 > 0 ? 0 : 1));
#pragma unroll 1
          for (int ch = ch_lo; ch < ch_hi; ch += 2) {
            uint32_t v[32], u[32];
            tmem_ld32x2(t_row + ch * 32, t_row + (ch + 1) * 32, v, u);
            if (t < wp.T) {
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                __stcg(mine + (ch * 8 + j) * kTileM + row,
                       make_float4(f32(v[4 * j]), f32(v[4 * j + 1]), f32(v[4 * j + 2]), f32(v[4 * j + 3])));
                __stcg(mine + ((ch + 1) * 8 + j) * kTileM + row,
                       make_float4(f32(u[4 * j]), f32(u[4 * j + 1]), f32(u[4 * j + 2]), f32(u[4 * j + 3])));
              }
            }
            __syncwarp();
          }
          if (tr != nullptr) tr[3] = global_timer_ns();   // dump issued
          named_barrier(1, kEpiThreads);                  // every row of the part is written
          if (etid == 0) atom_add_acq_rel_gpu(counter, 1);
          if (tr != nullptr) tr[4] = global_timer_ns();   // published
        }
        if (tr != nullptr) {
          tr[1] |= (finish ? 2ull : 1ull) << 32;
          if (finish) tr[3] = global_timer_ns();
        }
        if (finish) {
          stage_cs();
          // accumulator = sum of all parts in ascending contributor order (this
          // CTA's own part taken from TMEM at its place), so the bits do not
          // depend on timing.  Each group sums its half of the columns.
          const int64_t rows_left = static_cast<int64_t>(wp.T) - row0;
          const int rv = rows_left <= 0 ? 0 : (rows_left < kTileM ? static_cast<int>(rows_left) : kTileM);
          const int n_oth = c_last - c_first;
          // The operand ring is idle after the CTA's last MMA: the other parts
          // are staged there (each group in its own half, after the cos/sin
          // rows) with bulk copies, one per part and 32-column chunk (16 KB,
          // contiguous in a workspace slot), completing on the group's
          // mbarrier; each thread then reads its own row.  If the parts of
          // one chunk do not fit, they are read from the workspace directly.
          constexpr uint32_t kChunkBytes = 8 * kTileM * 16;
          constexpr uint32_t kHalfRing = (G::kRingBytes - kCsBytes) / 2;
          const bool staged = static_cast<uint32_t>(n_oth) * kChunkBytes <= kHalfRing;
          int cpr = kChunks / 2;   // chunks per staging round
          if (staged && n_oth > 0) {
            cpr = static_cast<int>(kHalfRing / (static_cast<uint32_t>(n_oth) * kChunkBytes));
            cpr = cpr > kChunks / 2 ? kChunks / 2 : cpr;
          }
          const uint32_t ring = smem_u32(smem) + kCsBytes + static_cast<uint32_t>(group) * kHalfRing;
          const float4* ring_f4 = reinterpret_cast<const float4*>(smem + kCsBytes + group * kHalfRing);
          const uint32_t fbar = smem_u32(&bars->fix[group]);
          const bool issuer = (etid % 128) == 0;
          bool fix_ok = true;
#pragma unroll 1
          for (int ch0 = ch_lo; ch0 < ch_hi; ch0 += cpr) {
            const int nch = (ch_hi - ch0) < cpr ? (ch_hi - ch0) : cpr;
            if (staged && n_oth > 0) {
              if (issuer) {
                // the group's reads of the previous round (generic proxy) come
                // before this round's copies (async proxy) into the same bytes
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                mbar_arrive_expect_tx(fbar, static_cast<uint32_t>(n_oth * nch) * kChunkBytes);
                int oi = 0;
                for (int c = c_first; c <= c_last; ++c) {
                  if (c == wid) continue;
                  const float* slot = ws_slot(wp, cta_of(c), c == c_first ? 1 : 0);
                  for (int cl = 0; cl < nch; ++cl)
                    bulk_load_g2s(ring + static_cast<uint32_t>(oi * nch + cl) * kChunkBytes,
                                  slot + static_cast<size_t>(ch0 + cl) * 8 * kTileM * 4, kChunkBytes, fbar);
                  ++oi;
                }
              }
              // every thread of the group waits for the round's bytes (the
              // copies read valid workspace and always complete: the wait
              // does not stop on an abort, so none is left in flight)
              int never = 0;
              fix_ok = mbar_wait(fbar, fix_phase, &never, wp.wait_limit_ns) && fix_ok;
              fix_phase ^= 1u;
            }
#pragma unroll 1
            for (int cl = 0; cl < nch; ++cl) {
              const int ch = ch0 + cl;
              uint32_t v[32];
              int oi = 0;
              for (int c = c_first; c <= c_last; ++c) {
                uint32_t part[32];
                if (c == wid) {
                  tmem_ld32(t_row + ch * 32, part);   // warp-uniform branch
                } else {
                  if (row < rv && fix_ok) {
                    const float4* src =
                        staged ? ring_f4 + (oi * nch + cl) * 8 * kTileM + row
                               : reinterpret_cast<const float4*>(ws_slot(wp, cta_of(c), c == c_first ? 1 : 0)) +
                                     ch * 8 * kTileM + row;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                      const float4 q = src[j * kTileM];
                      part[4 * j] = __float_as_uint(q.x);
                      part[4 * j + 1] = __float_as_uint(q.y);
                      part[4 * j + 2] = __float_as_uint(q.z);
                      part[4 * j + 3] = __float_as_uint(q.w);
                    }
                  } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) part[e] = 0u;
                  }
                  ++oi;
                }
#pragma unroll
                for (int e = 0; e < 32; ++e)
                  v[e] = c == c_first ? part[e] : __float_as_uint(f32(v[e]) + f32(part[e]));
              }
              __syncwarp();
              tmem_st32(t_row + ch * 32, v);
            }
            // the group's staging half is rewritten by its next round
            if (staged && n_oth > 0) named_barrier(2 + group, 128);
          }
          if (!fix_ok && etid % 128 == 0) abort_work<kPair>(wp, abort_flag);
          // both groups' sums are in TMEM before any thread reads across halves
          tc_fence_before();
          named_barrier(1, kEpiThreads);
          tc_fence_after();
        }
      }

      if (!cut) stage_cs();
      if (cs_stage && finish) {
        cp_async_wait_all();
        named_barrier(1, kEpiThreads);   // both halves of every row have landed
      }
      if (tr != nullptr && finish) tr[4] = global_timer_ns();
      if (plain) {
        if (finish) {
          // this group's 128 columns of the row: stored rounded to the model
          // dtype; the sum of squares is taken over the stored values
          const int col0 = n_blk * kTileN + group * (kTileN / 2);
          float ss = 0.f;
#pragma unroll 1
          for (int ch = 0; ch < kChunks / 2; ch += 2) {
            uint32_t v[32], u[32];
            tmem_ld32x2(t_row + (ch_lo + ch) * 32, t_row + (ch_lo + ch + 1) * 32, v, u);
            if (t < wp.T) {
#pragma unroll
              for (int half = 0; half < 2; ++half) {
                const uint32_t* src = half == 0 ? v : u;
                const int c = col0 + (ch + half) * 32;
                if (c >= wp.N) continue;
                E* dst = reinterpret_cast<E*>(wp.y) + t * wp.y_stride + c;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                  uint32_t w[4];
#pragma unroll
                  for (int e = 0; e < 4; ++e) {
                    w[e] = ElemOps<E>::pack(f32(src[8 * q + 2 * e]), f32(src[8 * q + 2 * e + 1]));
                    float lo, hi;
                    ElemOps<E>::unpack(w[e], lo, hi);
                    ss = fmaf(lo, lo, fmaf(hi, hi, ss));
                  }
                  st16(dst + 8 * q, w[0], w[1], w[2], w[3]);
                }
              }
            }
            __syncwarp();
          }
          // the two groups' halves of the row, added in a fixed order
          if (group == 1) bars->ss_x[row] = ss;
          named_barrier(1, kEpiThreads);
          if (group == 0 && t < wp.T) wp.rowsq[t * wp.rowsq_stride + n_blk] = ss + bars->ss_x[row];
          named_barrier(1, kEpiThreads);
        }
      } else if (finish) {
#pragma unroll 1
        for (int seg = group; seg < kTileN / kD; seg += 2) {
          const int c0 = n_blk * kTileN + seg * kD;
          if (c0 >= wp.N) break;
          const int layer = c0 / (2 * wp.KV);
          const int r = c0 - layer * 2 * wp.KV;
          const bool is_v = r >= wp.KV;
          const int head = (is_v ? r - wp.KV : r) / kD;
          const uint32_t t_seg = t_row + seg * D;
          if (is_v) {
            E* dst = reinterpret_cast<E*>(wp.v_pool[layer]) + loc * wp.v_stride[layer] + head * D;
#pragma unroll 1
            for (int ch = 0; ch < D / 32; ch += 2) {
              uint32_t v[32], u[32];
              tmem_ld32x2(t_seg + ch * 32, t_seg + (ch + 1) * 32, v, u);
              if (write) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                  float x[8], y[8];
#pragma unroll
                  for (int e = 0; e < 8; ++e) {
                    x[e] = f32(v[8 * q + e]) * rs;
                    y[e] = f32(u[8 * q + e]) * rs;
                  }
                  if (kBias) {
                    float bx[8], by[8];
                    load8<E>(wp.bias, c0 + ch * 32 + 8 * q, bx);
                    load8<E>(wp.bias, c0 + (ch + 1) * 32 + 8 * q, by);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                      x[e] += bx[e];
                      y[e] += by[e];
                    }
                  }
                  st16(dst + ch * 32 + 8 * q, ElemOps<E>::pack(x[0], x[1]), ElemOps<E>::pack(x[2], x[3]),
                       ElemOps<E>::pack(x[4], x[5]), ElemOps<E>::pack(x[6], x[7]));
                  st16(dst + (ch + 1) * 32 + 8 * q, ElemOps<E>::pack(y[0], y[1]),
                       ElemOps<E>::pack(y[2], y[3]), ElemOps<E>::pack(y[4], y[5]),
                       ElemOps<E>::pack(y[6], y[7]));
                }
              }
              __syncwarp();
            }
          } else {
            // RMSNorm: sum of squares over this thread's row of the head
            float ss = 0.f;
#pragma unroll 1
            for (int ch = 0; ch < D / 32; ch += 2) {
              uint32_t v[32], u[32];
              tmem_ld32x2(t_seg + ch * 32, t_seg + (ch + 1) * 32, v, u);
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                float bx[8], by[8];
                if (kBias) {
                  load8<E>(wp.bias, c0 + ch * 32 + 8 * q, bx);
                  load8<E>(wp.bias, c0 + (ch + 1) * 32 + 8 * q, by);
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                  float x = f32(v[8 * q + e]) * rs, y = f32(u[8 * q + e]) * rs;
                  if (kBias) {
                    x += bx[e];
                    y += by[e];
                  }
                  ss = fmaf(x, x, ss);
                  ss = fmaf(y, y, ss);
                }
              }
            }
            const float inv = rsqrtf(ss * (1.0f / D) + wp.eps);
            const float* w = wp.knorm + static_cast<int64_t>(layer) * D;
            const float* cs = wp.cos_sin + pos * D;
            const uint8_t* cs_smem = smem + static_cast<size_t>(row) * (D * 4);
            E* dst = reinterpret_cast<E*>(wp.k_pool[layer]) + loc * wp.k_stride[layer] + head * D;
            // rotate 16 columns of each half at a time (bounded register use)
#pragma unroll 1
            for (int hc = 0; hc < kHalf / 16; ++hc) {
              uint32_t a[16], b[16];
              tmem_ld16x2(t_seg + hc * 16, t_seg + kHalf + hc * 16, a, b);
              if (write) {
                uint32_t o1[8], o2[8];
                float b1[16], b2[16];
                if (kBias) {
                  load8<E>(wp.bias, c0 + hc * 16, *reinterpret_cast<float(*)[8]>(&b1[0]));
                  load8<E>(wp.bias, c0 + hc * 16 + 8, *reinterpret_cast<float(*)[8]>(&b1[8]));
                  load8<E>(wp.bias, c0 + kHalf + hc * 16, *reinterpret_cast<float(*)[8]>(&b2[0]));
                  load8<E>(wp.bias, c0 + kHalf + hc * 16 + 8, *reinterpret_cast<float(*)[8]>(&b2[8]));
                }
#pragma unroll
                for (int e4 = 0; e4 < 16; e4 += 4) {
                  const int i = hc * 16 + e4;
                  const float4 w1 = *reinterpret_cast<const float4*>(w + i);
                  const float4 w2 = *reinterpret_cast<const float4*>(w + kHalf + i);
                  float4 c4, s4;
                  if (cs_stage) {
                    const int sw = row & 7;
                    c4 = *reinterpret_cast<const float4*>(cs_smem + ((i / 4) ^ sw) * 16);
                    s4 = *reinterpret_cast<const float4*>(cs_smem + (((kHalf + i) / 4) ^ sw) * 16);
                  } else {
                    c4 = *reinterpret_cast<const float4*>(cs + i);
                    s4 = *reinterpret_cast<const float4*>(cs + kHalf + i);
                  }
                  const float wa[4] = {w1.x, w1.y, w1.z, w1.w};
                  const float wb[4] = {w2.x, w2.y, w2.z, w2.w};
                  const float cc[4] = {c4.x, c4.y, c4.z, c4.w};
                  const float sn[4] = {s4.x, s4.y, s4.z, s4.w};
                  float r1[4], r2[4];
#pragma unroll
                  for (int j = 0; j < 4; ++j) {
                    float x1 = f32(a[e4 + j]) * rs;
                    float x2 = f32(b[e4 + j]) * rs;
                    if (kBias) {
                      x1 += b1[e4 + j];
                      x2 += b2[e4 + j];
                    }
                    x1 = x1 * inv * wa[j];
                    x2 = x2 * inv * wb[j];
                    r1[j] = x1 * cc[j] - x2 * sn[j];
                    r2[j] = x2 * cc[j] + x1 * sn[j];
                  }
                  o1[e4 / 2] = ElemOps<E>::pack(r1[0], r1[1]);
                  o1[e4 / 2 + 1] = ElemOps<E>::pack(r1[2], r1[3]);
                  o2[e4 / 2] = ElemOps<E>::pack(r2[0], r2[1]);
                  o2[e4 / 2 + 1] = ElemOps<E>::pack(r2[2], r2[3]);
                }
                st16(dst + hc * 16, o1[0], o1[1], o1[2], o1[3]);
                st16(dst + hc * 16 + 8, o1[4], o1[5], o1[6], o1[7]);
                st16(dst + kHalf + hc * 16, o2[0], o2[1], o2[2], o2[3]);
                st16(dst + kHalf + hc * 16 + 8, o2[4], o2[5], o2[6], o2[7]);
              }
              __syncwarp();
            }
          }
        }
      }
      // accumulator fully read: hand it back to the MMA warp
      tc_fence_before();
      __syncwarp();
      if (tr != nullptr) tr[5] = global_timer_ns();
      if (lane == 0) {
        if (kPair)
          mbar_arrive_cluster(mapa_shared(smem_u32(&bars->tmem_empty[acc]), 0));
        else
          mbar_arrive(smem_u32(&bars->tmem_empty[acc]));
      }
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
      if (reduce_after) {
        const bool split_ok =
            plain ? finish_split_rows<E, 0, false, kPair, false>(wp, wid, nwq, rank, bars->ss_x, abort_flag)
                  : finish_split_rows<E, D, kBias, kPair, kFused>(wp, wid, nwq, rank, bars->ss_x, abort_flag);
        if (!split_ok) {
          if (etid == 0) abort_work<kPair>(wp, abort_flag);
          ep_abort = true;
          break;
        }
        if (trace != nullptr && etid == 0) trace[kTraceWords - 1] = global_timer_ns();   // split rows done
      }
    }
    if (kFused && ph == 0 && !ep_abort) {
      // this CTA's part of the first problem (y and its row sums) is stored:
      // make it visible to the tensor-memory loads of the second one and count
      // the CTA done
      fence_proxy_async_global();
      named_barrier(1, kEpiThreads);
      if (etid == 0) atom_add_acq_rel_gpu(p.phase_count, 1);
    }
    }
    if (kFused && !ep_abort && etid == 0) {
      // second round: the last CTA to finish resets the count for the next launch
      if (atom_add_acq_rel_gpu(p.phase_count, 1) == 2 * static_cast<int>(gridDim.x) - 1) *p.phase_count = 0;
    }
  }

  tc_fence_before();
  __syncwarp();
  if (kPair) {
    cluster_sync();   // the leader's MMAs read the peer's operands until here
  } else {
    __syncthreads();
  }
  tc_fence_after();
  if (warp == kMmaWarp) {
    if (kPair)
      tmem_dealloc_pair(tmem_base, kTmemCols);
    else
      tmem_dealloc(tmem_base, kTmemCols);
  }
  if (trace != nullptr && threadIdx.x == 0) {
    trace[1] = global_timer_ns();
    WorkIter it = work_begin(p, wid, nw);
    int tile, kb0, kb1, n = 0;
    while (work_next(p, it, tile, kb0, kb1)) ++n;
    trace[2] = static_cast<uint64_t>(n);
  }
}

template <typename E, int D, bool kBias, bool kPair>
__global__ void __launch_bounds__(kTiledThreads, 1)
    ctx_kv_tiled_kernel(const __grid_constant__ CUtensorMap tmap_x,
                        const __grid_constant__ CUtensorMap tmap_w,
                        const __grid_constant__ WriteParams p) {
  tiled_body<E, D, kBias, kPair, false>(tmap_x, tmap_w, p, tmap_x, tmap_w, p);
}

// combine_hidden_states fused into the write: main_proj (p1, plain mode, y and
// its row sums into scratch) then the write (p) over y with the stacked
// weights scaled by main_norm's weight and every token row by its 1/rms.
template <typename E, int D, bool kBias>
__global__ void __launch_bounds__(kTiledThreads, 1)
    ctx_kv_fused_kernel(const __grid_constant__ CUtensorMap tmap_x1,
                        const __grid_constant__ CUtensorMap tmap_w1,
                        const __grid_constant__ WriteParams p1,
                        const __grid_constant__ CUtensorMap tmap_x,
                        const __grid_constant__ CUtensorMap tmap_w,
                        const __grid_constant__ WriteParams p) {
  tiled_body<E, D, kBias, true, true>(tmap_x1, tmap_w1, p1, tmap_x, tmap_w, p);
}

template <bool kPair>
size_t tiled_smem_bytes() {
  return 1024 /* alignment slack */ + Geo<kPair>::kRingBytes + sizeof(SmemBarriers);
}

template <typename E, int D, bool kBias, bool kPair>
cudaError_t launch_one(int device, const CUtensorMap& tx, const CUtensorMap& tw,
                       const WriteParams& p, int grid, cudaStream_t stream) {
  auto kern = ctx_kv_tiled_kernel<E, D, kBias, kPair>;
  // the opt-in shared-memory size is set once per device and instantiation
  static std::atomic<uint64_t> attr_set{0};
  const uint64_t bit = 1ull << (device & 63);
  const size_t smem = tiled_smem_bytes<kPair>();
  if (!(attr_set.load() & bit)) {
    // setmaxnreg.inc waits until the CTA's register pool can grant it: the
    // pool the kernel launches with must cover the whole split, or it would
    // never return.  Refuse to launch otherwise.
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    if (static_cast<long>(fa.numRegs) * kTiledThreads < 128L * kRegsControl + 256L * kRegsEpilogue)
      return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attr_set.fetch_or(bit);
  }
  if (!kPair) {
    kern<<<grid, kTiledThreads, smem, stream>>>(tx, tw, p);
    return cudaGetLastError();
  }
  // CTA pairs: clusters of two along x
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kTiledThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tx, tw, p);
}

template <bool kPair>
cudaError_t dispatch(int device, int dtype, int head_dim, bool has_bias, const CUtensorMap& tx,
                     const CUtensorMap& tw, const WriteParams& p, int grid, cudaStream_t stream) {
  if (dtype == DSPARK_DTYPE_BF16) {
    if (head_dim == 128)
      return has_bias ? launch_one<__nv_bfloat16, 128, true, kPair>(device, tx, tw, p, grid, stream)
                      : launch_one<__nv_bfloat16, 128, false, kPair>(device, tx, tw, p, grid, stream);
    return has_bias ? launch_one<__nv_bfloat16, 64, true, kPair>(device, tx, tw, p, grid, stream)
                    : launch_one<__nv_bfloat16, 64, false, kPair>(device, tx, tw, p, grid, stream);
  }
  if (head_dim == 128)
    return has_bias ? launch_one<__half, 128, true, kPair>(device, tx, tw, p, grid, stream)
                    : launch_one<__half, 128, false, kPair>(device, tx, tw, p, grid, stream);
  if (head_dim == 64)
    return has_bias ? launch_one<__half, 64, true, kPair>(device, tx, tw, p, grid, stream)
                    : launch_one<__half, 64, false, kPair>(device, tx, tw, p, grid, stream);
  return cudaErrorInvalidValue;
}

template <bool kPair>
cudaError_t dispatch_plain(int device, int dtype, const CUtensorMap& tx, const CUtensorMap& tw,
                           const WriteParams& p, int grid, cudaStream_t stream) {
  return dtype == DSPARK_DTYPE_BF16 ? launch_one<__nv_bfloat16, 0, false, kPair>(device, tx, tw, p, grid, stream)
                                    : launch_one<__half, 0, false, kPair>(device, tx, tw, p, grid, stream);
}

}  // namespace


cudaError_t launch_tiled(int device, int dtype, int head_dim, bool has_bias, const CUtensorMap& tx,
                         const CUtensorMap& tw, const WriteParams& p, int grid,
                         cudaStream_t stream) {
  return dispatch<false>(device, dtype, head_dim, has_bias, tx, tw, p, grid, stream);
}

cudaError_t launch_plain(int device, int dtype, const CUtensorMap& tx, const CUtensorMap& tw, const WriteParams& p,
                         int grid, bool pair, cudaStream_t stream) {
  return pair ? dispatch_plain<true>(device, dtype, tx, tw, p, grid, stream)
              : dispatch_plain<false>(device, dtype, tx, tw, p, grid, stream);
}

namespace {

template <typename E, int D, bool kBias>
cudaError_t launch_fused_one(int device, const CUtensorMap& tx1, const CUtensorMap& tw1, const WriteParams& p1,
                             const CUtensorMap& tx, const CUtensorMap& tw, const WriteParams& p, int grid,
                             cudaStream_t stream) {
  auto kern = ctx_kv_fused_kernel<E, D, kBias>;
  static std::atomic<uint64_t> attr_set{0};
  const uint64_t bit = 1ull << (device & 63);
  const size_t smem = tiled_smem_bytes<true>();
  if (!(attr_set.load() & bit)) {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    if (static_cast<long>(fa.numRegs) * kTiledThreads < 128L * kRegsControl + 256L * kRegsEpilogue)
      return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attr_set.fetch_or(bit);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kTiledThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tx1, tw1, p1, tx, tw, p);
}

}  // namespace

cudaError_t launch_fused(int device, int dtype, int head_dim, bool has_bias, const CUtensorMap& tx1,
                         const CUtensorMap& tw1, const WriteParams& p1, const CUtensorMap& tx,
                         const CUtensorMap& tw_half, const WriteParams& p, int grid, cudaStream_t stream) {
  if (dtype == DSPARK_DTYPE_BF16) {
    if (head_dim == 128)
      return has_bias ? launch_fused_one<__nv_bfloat16, 128, true>(device, tx1, tw1, p1, tx, tw_half, p, grid, stream)
                      : launch_fused_one<__nv_bfloat16, 128, false>(device, tx1, tw1, p1, tx, tw_half, p, grid, stream);
    return has_bias ? launch_fused_one<__nv_bfloat16, 64, true>(device, tx1, tw1, p1, tx, tw_half, p, grid, stream)
                    : launch_fused_one<__nv_bfloat16, 64, false>(device, tx1, tw1, p1, tx, tw_half, p, grid, stream);
  }
  if (head_dim == 128)
    return has_bias ? launch_fused_one<__half, 128, true>(device, tx1, tw1, p1, tx, tw_half, p, grid, stream)
                    : launch_fused_one<__half, 128, false>(device, tx1, tw1, p1, tx, tw_half, p, grid, stream);
  return has_bias ? launch_fused_one<__half, 64, true>(device, tx1, tw1, p1, tx, tw_half, p, grid, stream)
                  : launch_fused_one<__half, 64, false>(device, tx1, tw1, p1, tx, tw_half, p, grid, stream);
}

cudaError_t launch_pair(int device, int dtype, int head_dim, bool has_bias, const CUtensorMap& tx,
                        const CUtensorMap& tw_half, const WriteParams& p, int grid,
                        cudaStream_t stream) {
  return dispatch<true>(device, dtype, head_dim, has_bias, tx, tw_half, p, grid, stream);
}

int single_workers(int device) {
  // CTAs of the single-CTA kernel that can be resident at once: blocks per SM
  // (one, given its shared memory) times the SM count.  The split-tile waits
  // assume every CTA of the grid is resident, so the grid never exceeds this.
  static std::atomic<int> cache[64];
  const int d = device & 63;
  int n = cache[d].load();
  if (n > 0) return n;
  auto kern = ctx_kv_tiled_kernel<__nv_bfloat16, 128, false, false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(tiled_smem_bytes<false>())) != cudaSuccess)
    return 0;
  int per_sm = 0, sms = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kTiledThreads, tiled_smem_bytes<false>()) !=
          cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || per_sm <= 0 ||
      sms <= 0)
    return 0;
  cache[d].store(per_sm * sms);
  return per_sm * sms;
}

int pair_workers(int device) {
  // every instantiation has the same block size, shared memory and registers,
  // so one of them answers for all
  static std::atomic<int> cache[64];
  const int d = device & 63;
  int n = cache[d].load();
  if (n > 0) return n;
  auto kern = ctx_kv_tiled_kernel<__nv_bfloat16, 128, false, true>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(tiled_smem_bytes<true>())) != cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kTiledThreads, 1, 1);
  cfg.dynamicSmemBytes = tiled_smem_bytes<true>();
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess || clusters <= 0) return 0;
  cache[d].store(clusters);
  return clusters;
}

}  // namespace dspark
