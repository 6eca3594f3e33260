// Weight-streaming variant of the fused context-KV write for small token
// counts (T <= 256), where the stacked weights dominate the bytes.
//
// The operands are swapped with respect to the tiled kernel: 128 rows of the
// stacked weight W_all (128 output features: one head of D = 128 or two of
// D = 64) are the M side of tcgen05.mma, and all tokens (padded to 16 or a
// multiple of 32, at most 256) are the N side.  A stage holds 16 KB of weights
// plus t_pad x 128 bytes of hidden states; up to 8 stages, so every SM keeps up
// to 128 KB of weights in flight: the weight stream runs at ~93% of the copy
// bandwidth.  Weight tiles and their k-blocks are spread over all SMs with the same
// data-parallel + backward stream-K walk as the tiled kernel.
//
//   warps 0..3  epilogue: thread r owns output feature r of the tile (TMEM lane
//               r) for every token column, so bias and k_norm weight are one
//               register each.  The per-token RMSNorm sum of squares runs
//               across the head's lanes (a warp transpose-reduce, then the
//               head's warps through shared memory); the RoPE partner feature
//               (d +- D/2) lives in another warp and is exchanged through
//               shared memory; results are transposed in shared memory so that
//               each pool row (128 features, 256 bytes) is written with 16-byte
//               stores.
//   warp 4      TMA producer
//   warp 5      MMA issuer, TMEM owner
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>

#include "internal.h"
#include "kernel_common.cuh"
#include "ptx.cuh"

namespace dspark {
namespace {

constexpr int kSRows = 128;                 // output features per tile (TMEM lanes)
constexpr int kSThreads = 192;
constexpr int kSEpiThreads = 128;
constexpr int kSProducerWarp = 4;
constexpr int kSMmaWarp = 5;
constexpr int kSMaxStages = 8;   // 128 KB of weights in flight per SM: 6 to 12 measured the same
constexpr int kSMaxTokens = 256;
constexpr uint32_t kSStageA = kSRows * kTileK * 2;   // 16 KB of weights per stage
constexpr int kSChunk = 32;                          // token columns per epilogue pass

struct StreamBarriers {
  uint64_t full[kSMaxStages];
  uint64_t empty[kSMaxStages];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int last_arrival;   // finisher's early look: every other part of its cut tile already published
};

// Epilogue scratch after the barriers.
struct StreamScratch {
  int64_t loc[kSMaxTokens];
  int64_t pos[kSMaxTokens];
  int32_t ok[kSMaxTokens];
  float red[4][kSChunk];                   // per-warp column sums of squares
  float inv[2][kSChunk];                   // per-head 1/rms of each token column
  float nbuf[kSRows][kSChunk + 1];         // normalised values (padded rows)
  uint16_t obuf[kSChunk][kSRows + 8];      // results, token-major (padded rows)
};

struct StreamCfg {
  int t_pad;           // MMA N: tokens padded to 16 or a multiple of 32
  int stages;
  uint32_t stage_b;    // bytes of hidden states per stage
  uint32_t acc_stride; // TMEM columns between the two accumulators
  uint32_t tmem_cols;
};

// One 32-lane transpose-reduce: on entry lane l holds v[j] = value of (row l,
// column j); on exit v[0] of lane l is the sum over the 32 rows of column l.
__device__ __forceinline__ float warp_column_sums(float (&v)[32], int lane) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < off; ++i) {
      const float send = upper ? v[i] : v[i + off];
      const float keep = upper ? v[i + off] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  return v[0];
}

template <typename E, int D, bool kBias>
__global__ void __launch_bounds__(kSThreads, 1)
    ctx_kv_stream_kernel(const __grid_constant__ CUtensorMap tmap_x,
                         const __grid_constant__ CUtensorMap tmap_w,
                         const __grid_constant__ WriteParams p, const StreamCfg cfg) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* smem_a = smem;
  uint8_t* smem_b = smem + cfg.stages * kSStageA;
  const uint32_t ring_bytes = cfg.stages * (kSStageA + cfg.stage_b);
  StreamBarriers* bars = reinterpret_cast<StreamBarriers*>(smem + ring_bytes);
  StreamScratch* sc = reinterpret_cast<StreamScratch*>(
      reinterpret_cast<uint8_t*>(bars) + ((sizeof(StreamBarriers) + 15) & ~size_t(15)));

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  volatile int* abort_flag = &bars->abort;
  const int wid = blockIdx.x, nw = gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < cfg.stages; ++s) {
      mbar_init(smem_u32(&bars->full[s]), 1);
      mbar_init(smem_u32(&bars->empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&bars->tmem_full[b]), 1);
      mbar_init(smem_u32(&bars->tmem_empty[b]), 4);
    }
    mbar_init(smem_u32(&bars->drain), 1);
    bars->abort = 0;
    fence_barrier_init();
  }
  if (warp == kSProducerWarp && lane == 0) {
    tma_prefetch_desc(&tmap_x);
    tma_prefetch_desc(&tmap_w);
  }
  if (warp == kSMmaWarp) {
    tmem_alloc(smem_u32(&bars->tmem_base), cfg.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncwarp();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = bars->tmem_base;
  uint64_t* trace = p.trace != nullptr ? p.trace + static_cast<size_t>(blockIdx.x) * kTraceWords : nullptr;
  if (trace != nullptr && threadIdx.x == 0) trace[0] = global_timer_ns();

  if (warp == kSProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      // the weights are read once: evict_first keeps them from pushing other
      // lines out of L2 (with a dirty L2 each eviction is a DRAM write that
      // competes with the stream: measured 8% faster at 16 and 64 tokens);
      // the hidden states are read by every SM
      const uint64_t pol_w = l2_policy_evict_first();
      const uint64_t pol_x = l2_policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t uses[kSMaxStages] = {};
      bool ok = true;
      WorkIter it = work_begin(p, wid, nw);
      int tile, kb0, kb1;
      while (ok && work_next(p, it, tile, kb0, kb1)) {
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(smem_u32(&bars->empty[stage]), phase ^ 1u, abort_flag, p.wait_limit_ns)) {
            ok = false;
            break;
          }
          const uint32_t full = smem_u32(&bars->full[stage]);
          mbar_arrive_expect_tx(full, kSStageA + cfg.stage_b);
          tma_load_2d(smem_u32(smem_a + stage * kSStageA), &tmap_w, kb * kTileK, tile * kSRows, full,
                      pol_w);
          tma_load_2d(smem_u32(smem_b + stage * cfg.stage_b), &tmap_x, kb * kTileK, 0, full, pol_x);
          ++uses[stage];
          if (++stage == cfg.stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        flag(p, DSPARK_FLAG_TIMEOUT);
      }
      int never = 0;
      for (int s = 0; s < cfg.stages; ++s)
        if (uses[s] > 0) mbar_wait(smem_u32(&bars->full[s]), (uses[s] - 1u) & 1u, &never, p.wait_limit_ns);
    }
  } else if (warp == kSMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = f16_instr_desc(ElemOps<E>::kFmt, kSRows, cfg.t_pad);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true, issued = false;
      WorkIter it = work_begin(p, wid, nw);
      int tile, kb0, kb1;
      while (ok && work_next(p, it, tile, kb0, kb1)) {
        if (!mbar_wait(smem_u32(&bars->tmem_empty[acc]), acc_phase ^ 1u, abort_flag, p.wait_limit_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * cfg.acc_stride;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(smem_u32(&bars->full[stage]), phase, abort_flag, p.wait_limit_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(smem_a + stage * kSStageA);
          const uint32_t b0 = smem_u32(smem_b + stage * cfg.stage_b);
#pragma unroll
          for (int k = 0; k < kTileK / 16; ++k)
            umma_f16(d_tmem, sw128_kmajor_desc(a0 + k * 32), sw128_kmajor_desc(b0 + k * 32), idesc,
                     (kb != kb0 || k != 0) ? 1u : 0u);
          issued = true;
          umma_commit(smem_u32(&bars->empty[stage]));
          if (++stage == cfg.stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(smem_u32(&bars->tmem_full[acc]));
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (!ok) {
        *abort_flag = 1;
        flag(p, DSPARK_FLAG_TIMEOUT);
      }
      if (issued) {
        umma_commit(smem_u32(&bars->drain));
        int never = 0;
        mbar_wait(smem_u32(&bars->drain), 0, &never, p.wait_limit_ns);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // Per-token decisions, shared by every tile of this CTA, made while the
    // producer's first loads are in flight.  Every slot is set: the epilogue
    // reads whole 32-token chunks.
    for (int t = threadIdx.x; t < kSMaxTokens; t += kSEpiThreads) {
      int64_t loc = -1, pos = 0;
      int ok = 0;
      if (t < p.T) {
        // three independent loads, then the decision
        loc = p.cache_loc[t];
        pos = p.positions[t];
        const int64_t w = p.loc_row_width;
        const int64_t committed = w > 0 ? static_cast<int64_t>(p.commit_lens[t / w]) : 0;
        ok = loc >= 0 && (w == 0 || t - (t / w) * w < committed);
        if (ok && (pos < 0 || pos >= p.max_pos)) {
          if (blockIdx.x == 0) flag(p, DSPARK_FLAG_POS_RANGE);
          ok = 0;
        } else if (ok && loc >= p.pool_slots) {
          if (blockIdx.x == 0) flag(p, DSPARK_FLAG_LOC_RANGE);
          ok = 0;
        }
        if (!ok) pos = 0;
        // the K tiles' epilogues read this token's cos/sin row
        if (ok)
          for (int b = 0; b < D * 4; b += 128) prefetch_l2(reinterpret_cast<const char*>(p.cos_sin + pos * D) + b);
      }
      sc->loc[t] = loc;
      sc->pos[t] = pos;
      sc->ok[t] = ok;
    }
    named_barrier(1, kSEpiThreads);
    constexpr int kHalf = D / 2;
    const int r = threadIdx.x;                 // output feature (TMEM lane) of the tile
    const int d = r % D;                       // element within its head
    const int hsub = r / D;                    // head within the tile (D = 64: 0 or 1)
    const int ip = d % kHalf;                  // rotation pair index
    const int partner = d < kHalf ? r + kHalf : r - kHalf;
    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(warp * 32) << 16);
    const int n_cols = cfg.t_pad;
    int acc = 0;
    uint32_t acc_phase = 0;
    int item = 0;
    WorkIter it = work_begin(p, wid, nw);
    int tile, kb0, kb1;
    while (work_next(p, it, tile, kb0, kb1)) {
      const int c0 = tile * kSRows;              // first stacked row of the tile
      const int layer = c0 / (2 * p.KV);
      const int rr = c0 - layer * 2 * p.KV;
      const bool is_v = rr >= p.KV;
      const int head0 = (is_v ? rr - p.KV : rr) / D;
      float bias = 0.f, wn = 0.f;
      if (kBias) bias = ElemOps<E>::load(p.bias, c0 + r);
      if (!is_v) wn = p.knorm[static_cast<int64_t>(layer) * D + d];

      // A split tile's last part is normally the CTA's last item: check now,
      // while its MMAs run, whether the other parts are already published, and
      // if there is exactly one, fetch its first 32 token columns as well.
      const bool cut = kb0 != 0 || kb1 != p.num_kb;
      bool final_item;
      {
        WorkIter peek = it;
        int t2, a2, b2;
        final_item = !work_next(p, peek, t2, a2, b2);
      }
      int c_first = 0, c_last = 0;
      if (cut) {
        const int64_t u0 = static_cast<int64_t>(tile - p.dp_tiles) * p.num_kb;
        c_first = sk_owner(p, u0);
        c_last = sk_owner(p, u0 + p.num_kb - 1);
      }
      // A cut tile is finished by the contributor that holds its last k-block
      // (c_last): that piece is the last item of c_last's backward walk.  The
      // others publish their parts and never wait; c_last waits (bounded) for
      // them, so it never spends a dump on its own part.  Waits only go from a
      // worker to lower-numbered ones, and every CTA is resident (one per SM),
      // so they end.  Before its accumulator is ready c_last looks whether the
      // other parts are already published and, if there is exactly one,
      // fetches its first 32 token columns.
      const bool designated = cut && wid == c_last;
      bool early = false;
      float4 pre[8];
      if (designated) {
        if (r == 0) {
          const int seen = ld_acquire_gpu(p.counters + c_last);
          *reinterpret_cast<volatile int*>(&bars->last_arrival) = seen == c_last - c_first + p.split_wait_extra;
        }
        named_barrier(1, kSEpiThreads);
        early = *reinterpret_cast<volatile int*>(&bars->last_arrival) != 0;
        if (early && c_last - c_first == 1) {
          const float4* src = reinterpret_cast<const float4*>(ws_slot(p, c_first, 1)) + r;
#pragma unroll
          for (int j = 0; j < 8; ++j)
            pre[j] = 4 * j < n_cols ? __ldcg(src + j * kSRows) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }

      const bool got = mbar_wait(smem_u32(&bars->tmem_full[acc]), acc_phase, abort_flag, p.wait_limit_ns);
      uint64_t* tr = (trace != nullptr && r == 0 && item < kTraceItems) ? trace + 3 + 6 * item : nullptr;
      if (tr != nullptr) {
        tr[0] = static_cast<uint64_t>(tile);
        tr[1] = (static_cast<uint64_t>(kb0) << 16) | static_cast<uint64_t>(kb1);
        tr[2] = global_timer_ns();
        tr[3] = tr[4] = 0;
      }
      ++item;
      if (!named_barrier_and(1, kSEpiThreads, got)) {
        if (threadIdx.x == 0) {
          *abort_flag = 1;
          flag(p, DSPARK_FLAG_TIMEOUT);
        }
        break;
      }
      tc_fence_after();
      const uint32_t t_acc = t_lane + acc * cfg.acc_stride;

      // ---- a tile cut between CTAs: publish this part, or (c_last) wait for
      // the others and add the parts in contributor order
      bool finish = true;
      if (cut) {
        int32_t* counter = p.counters + c_last;
        finish = designated;
        if (designated) {
          bool ok = true;
          if (!early && r == 0)
            ok = wait_count(counter, c_last - c_first + p.split_wait_extra, abort_flag, p.split_wait_ns);
          if (!named_barrier_and(1, kSEpiThreads, ok)) {
            if (r == 0) {
              *abort_flag = 1;
              flag(p, DSPARK_FLAG_TIMEOUT);
            }
            break;
          }
          if (r == 0) *counter = 0;   // no other contributor touches it again
        } else {
          float4* mine = reinterpret_cast<float4*>(ws_slot(p, wid, kb0 > 0 ? 0 : 1));
          for (int c = 0; c < n_cols; c += kSChunk) {
            uint32_t v[32];
            tmem_ld32(t_acc + c, v);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              if (c + 4 * j < n_cols)
                __stcg(mine + ((c / 4) + j) * kSRows + r,
                       make_float4(f32(v[4 * j]), f32(v[4 * j + 1]), f32(v[4 * j + 2]), f32(v[4 * j + 3])));
            __syncwarp();
          }
          named_barrier(1, kSEpiThreads);   // every row of the part is written
          if (threadIdx.x == 0) atom_add_acq_rel_gpu(counter, 1);
        }
        if (tr != nullptr) {
          tr[1] |= (finish ? 2ull : 1ull) << 32;
          tr[3] = global_timer_ns();
        }
        if (finish) {
          for (int c = 0; c < n_cols; c += kSChunk) {
            uint32_t v[32];
            for (int cc = c_first; cc <= c_last; ++cc) {
              uint32_t part[32];
              if (cc == wid) {
                tmem_ld32(t_acc + c, part);
              } else if (early && c == 0 && c_last - c_first == 1) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  part[4 * j] = __float_as_uint(pre[j].x);
                  part[4 * j + 1] = __float_as_uint(pre[j].y);
                  part[4 * j + 2] = __float_as_uint(pre[j].z);
                  part[4 * j + 3] = __float_as_uint(pre[j].w);
                }
              } else {
                const float4* src =
                    reinterpret_cast<const float4*>(ws_slot(p, cc, cc == c_first ? 1 : 0)) + (c / 4) * kSRows + r;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  float4 q = make_float4(0.f, 0.f, 0.f, 0.f);
                  if (c + 4 * j < n_cols) q = __ldcg(src + j * kSRows);
                  part[4 * j] = __float_as_uint(q.x);
                  part[4 * j + 1] = __float_as_uint(q.y);
                  part[4 * j + 2] = __float_as_uint(q.z);
                  part[4 * j + 3] = __float_as_uint(q.w);
                }
              }
#pragma unroll
              for (int e = 0; e < 32; ++e)
                v[e] = cc == c_first ? part[e] : __float_as_uint(f32(v[e]) + f32(part[e]));
            }
            __syncwarp();
            tmem_st32(t_acc + c, v);
          }
          tc_fence_before();
          named_barrier(1, kSEpiThreads);
          tc_fence_after();
        }
      }

      if (tr != nullptr) tr[4] = global_timer_ns();
      if (finish) {
        E* pool_base = reinterpret_cast<E*>(is_v ? p.v_pool[layer] : p.k_pool[layer]) + head0 * D;
        const int64_t stride = is_v ? p.v_stride[layer] : p.k_stride[layer];
#pragma unroll 1
        for (int c = 0; c < n_cols; c += kSChunk) {
          float x[32];
          {
            uint32_t v[32];
            tmem_ld32(t_acc + c, v);
#pragma unroll
            for (int j = 0; j < 32; ++j) x[j] = f32(v[j]) + bias;
          }
          if (!is_v) {
            // per-token sum of squares over this head's features
            float sq[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) sq[j] = x[j] * x[j];
            sc->red[warp][lane] = warp_column_sums(sq, lane);
            named_barrier(1, kSEpiThreads);
            if ((warp & (D / 32 - 1)) == 0) {
              // the first warp of each head combines its head's warps in order
              float ss = 0.f;
#pragma unroll
              for (int w = 0; w < D / 32; ++w) ss += sc->red[warp + w][lane];
              sc->inv[warp / (D / 32)][lane] = rsqrtf(ss * (1.0f / D) + p.eps);
            }
            named_barrier(1, kSEpiThreads);
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              x[j] = x[j] * sc->inv[hsub][j] * wn;
              sc->nbuf[r][j] = x[j];
            }
            named_barrier(1, kSEpiThreads);
            const float sgn = d < kHalf ? -1.f : 1.f;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float* cs = p.cos_sin + sc->pos[c + j] * D;
              const float cj = cs[ip], sj = cs[kHalf + ip];
              x[j] = x[j] * cj + sgn * sc->nbuf[partner][j] * sj;
            }
          }
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            const uint32_t pk = ElemOps<E>::pack(x[j], x[j + 1]);
            sc->obuf[j][r] = static_cast<uint16_t>(pk & 0xFFFFu);
            sc->obuf[j + 1][r] = static_cast<uint16_t>(pk >> 16);
          }
          named_barrier(1, kSEpiThreads);
          // 32 tokens x 128 features: each token's 256 bytes are one pool row
          // segment, written as 16 x 16 bytes
#pragma unroll
          for (int it2 = 0; it2 < 4; ++it2) {
            const int piece = it2 * kSEpiThreads + r;
            const int j = piece / 16, q = piece % 16;
            const int t = c + j;
            if (t < p.T && sc->ok[t]) {
              const uint4 val = *reinterpret_cast<const uint4*>(&sc->obuf[j][q * 8]);
              *reinterpret_cast<uint4*>(pool_base + sc->loc[t] * stride + q * 8) = val;
            }
          }
          named_barrier(1, kSEpiThreads);   // scratch reused by the next chunk
        }
      }
      tc_fence_before();
      __syncwarp();
      if (tr != nullptr) tr[5] = global_timer_ns();
      if (lane == 0) mbar_arrive(smem_u32(&bars->tmem_empty[acc]));
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  tc_fence_before();
  __syncwarp();
  __syncthreads();
  tc_fence_after();
  if (warp == kSMmaWarp) tmem_dealloc(tmem_base, cfg.tmem_cols);
  if (trace != nullptr && threadIdx.x == 0) {
    trace[1] = global_timer_ns();
    WorkIter it = work_begin(p, wid, nw);
    int tile, kb0, kb1, n = 0;
    while (work_next(p, it, tile, kb0, kb1)) ++n;
    trace[2] = static_cast<uint64_t>(n);
  }
}

size_t stream_smem_bytes(int stages, uint32_t stage_b) {
  return 1024 + static_cast<size_t>(stages) * (kSStageA + stage_b) +
         ((sizeof(StreamBarriers) + 15) & ~size_t(15)) + sizeof(StreamScratch);
}

template <typename E, int D, bool kBias>
cudaError_t launch_stream_one(int device, const CUtensorMap& tx, const CUtensorMap& tw,
                              const WriteParams& p, const StreamCfg& cfg, int grid, cudaStream_t stream) {
  auto kern = ctx_kv_stream_kernel<E, D, kBias>;
  static std::atomic<uint64_t> attr_set{0};
  const uint64_t bit = 1ull << (device & 63);
  if (!(attr_set.load() & bit)) {
    // the largest configuration any call uses
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(stream_max_smem_bytes()));
    if (e != cudaSuccess) return e;
    attr_set.fetch_or(bit);
  }
  kern<<<grid, kSThreads, stream_smem_bytes(cfg.stages, cfg.stage_b), stream>>>(tx, tw, p, cfg);
  return cudaGetLastError();
}

}  // namespace

size_t stream_max_smem_bytes() { return 227 * 1024; }

int stream_workers(int device, int stages, uint32_t stage_b) {
  // CTAs of the streaming kernel that can be resident at once with this
  // launch's shared memory (every instantiation has the same block size and
  // shared memory): the split-tile waits assume all of the grid is resident
  // (cached per device and token padding: stage_b = t_pad * 128 bytes)
  static std::atomic<int> cache[64][kSMaxTokens / 16 + 1];
  const int d = device & 63, k = static_cast<int>(stage_b / (16 * kTileK * 2)) % (kSMaxTokens / 16 + 1);
  int n = cache[d][k].load();
  if (n > 0) return n;
  auto kern = ctx_kv_stream_kernel<__nv_bfloat16, 128, false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(stream_max_smem_bytes())) != cudaSuccess)
    return 0;
  int per_sm = 0, sms = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kSThreads, stream_smem_bytes(stages, stage_b)) !=
          cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || per_sm <= 0 ||
      sms <= 0)
    return 0;
  // one CTA per SM at most: a second one would halve each CTA's ring
  cache[d][k].store(sms);
  return sms;
}

bool stream_plan(int64_t T, int* t_pad, int* stages, uint32_t* stage_b, uint32_t* acc_stride,
                 uint32_t* tmem_cols) {
  if (T < 1 || T > kSMaxTokens) return false;
  const int tp = T <= 16 ? 16 : static_cast<int>((T + 31) / 32 * 32);
  const uint32_t sb = static_cast<uint32_t>(tp) * kTileK * 2;
  const size_t fixed = 1024 + ((sizeof(StreamBarriers) + 15) & ~size_t(15)) + sizeof(StreamScratch);
  int st = static_cast<int>((stream_max_smem_bytes() - fixed) / (kSStageA + sb));
  if (st > kSMaxStages) st = kSMaxStages;
  if (st < 2) return false;
  const uint32_t stride = tp < 32 ? 32u : static_cast<uint32_t>(tp);
  uint32_t cols = 32;
  while (cols < 2 * stride) cols <<= 1;
  *t_pad = tp;
  *stages = st;
  *stage_b = sb;
  *acc_stride = stride;
  *tmem_cols = cols;
  return true;
}

cudaError_t launch_stream(int device, int dtype, int head_dim, bool has_bias, const CUtensorMap& tx,
                          const CUtensorMap& tw_half, const WriteParams& p, int t_pad, int stages,
                          uint32_t stage_b, uint32_t acc_stride, uint32_t tmem_cols, int grid,
                          cudaStream_t stream) {
  const StreamCfg cfg{t_pad, stages, stage_b, acc_stride, tmem_cols};
  if (dtype == DSPARK_DTYPE_BF16) {
    if (head_dim == 128)
      return has_bias ? launch_stream_one<__nv_bfloat16, 128, true>(device, tx, tw_half, p, cfg, grid, stream)
                      : launch_stream_one<__nv_bfloat16, 128, false>(device, tx, tw_half, p, cfg, grid, stream);
    return has_bias ? launch_stream_one<__nv_bfloat16, 64, true>(device, tx, tw_half, p, cfg, grid, stream)
                    : launch_stream_one<__nv_bfloat16, 64, false>(device, tx, tw_half, p, cfg, grid, stream);
  }
  if (head_dim == 128)
    return has_bias ? launch_stream_one<__half, 128, true>(device, tx, tw_half, p, cfg, grid, stream)
                    : launch_stream_one<__half, 128, false>(device, tx, tw_half, p, cfg, grid, stream);
  return has_bias ? launch_stream_one<__half, 64, true>(device, tx, tw_half, p, cfg, grid, stream)
                  : launch_stream_one<__half, 64, false>(device, tx, tw_half, p, cfg, grid, stream);
}

}  // namespace dspark
