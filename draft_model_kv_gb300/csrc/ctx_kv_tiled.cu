// Fused stacked-KV projection + K RMSNorm + table neox RoPE + pool scatter on
// tcgen05 tensor cores (sm_103a).
//
// One persistent CTA per SM walks 128-token x 256-column tiles of the stacked
// output Y = ctx_hidden . W_all^T (W_all rows: l0:K, l0:V, l1:K, ...; sglang
// PR #31986 summary page, _stacked_ctx_kv_params).  256 columns are whole
// heads (D = 64 or 128), so each tile's epilogue can finish its heads alone.
//
//   warp 0      TMA producer: X and W_all K-slices into a 4-stage smem ring
//   warp 1      MMA issuer: tcgen05.mma 128x256x16 into one of two TMEM
//               accumulators (2 x 256 fp32 columns); owns TMEM alloc/free
//   warps 2..5  epilogue: each thread owns one token row of the accumulator
//               (tcgen05.ld 32x32b), so the RMSNorm sum of squares is a
//               per-thread sum and the neox pair (i, i + D/2) sits in the same
//               thread's registers; then 16-byte stores into the pool row.
//
// The epilogue of tile i overlaps the MMAs of tile i+1 (double-buffered TMEM).
// Per-token rules (sglang PR #31847 summary page, fused_kv_norm_rope_write):
// loc < 0 skips the token; in window mode column t mod W must be below
// commit_lens[t div W].
#include <cuda_bf16.h>
#include <atomic>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace dspark {
namespace {

template <typename E>
struct ElemOps;

template <>
struct ElemOps<__nv_bfloat16> {
  static constexpr uint32_t kFmt = 1;
  __device__ static __forceinline__ uint32_t pack(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __device__ static __forceinline__ float load(const void* p, int64_t i) {
    return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i]);
  }
};

template <>
struct ElemOps<__half> {
  static constexpr uint32_t kFmt = 0;
  __device__ static __forceinline__ uint32_t pack(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __device__ static __forceinline__ float load(const void* p, int64_t i) {
    return __half2float(reinterpret_cast<const __half*>(p)[i]);
  }
};

constexpr uint32_t kStageBytesA = kTileM * kTileK * 2;   // 16 KB
constexpr uint32_t kStageBytesB = kTileN * kTileK * 2;   // 32 KB
constexpr uint32_t kAccCols = kTileN;                    // fp32 columns per accumulator
constexpr uint32_t kTmemCols = 2 * kAccCols;             // double buffer = 512 (all of TMEM)

struct SmemBarriers {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int last_arrival;   // set by the epilogue leader when this CTA finishes a cut tile
};

__device__ __forceinline__ void tile_coords(int tile, int num_m, int num_n, int& m_blk,
                                            int& n_blk) {
  const int group_size = kGroupM * num_n;
  const int group = tile / group_size;
  const int first_m = group * kGroupM;
  const int gm = min(num_m - first_m, kGroupM);
  const int r = tile - group * group_size;
  m_blk = first_m + r % gm;
  n_blk = r / gm;
}

__device__ __forceinline__ void flag(const WriteParams& p, uint32_t bits) {
  atomicOr(p.status, bits);
}

__device__ __forceinline__ float f32(uint32_t u) { return __uint_as_float(u); }

// Store 32 consecutive outputs (already rounded/packed in pairs) as 4 x 16 B.
__device__ __forceinline__ void store32(void* dst, const uint32_t (&w)[16]) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i) d[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
}

// Work of one CTA: first its whole tiles of the data-parallel waves, then its
// contiguous range of the stream-K k-block space.
struct WorkIter {
  int dp_tile;
  int64_t cur, end;
};

__device__ __forceinline__ WorkIter work_begin(const WriteParams& p) {
  WorkIter it;
  it.dp_tile = blockIdx.x;
  it.cur = static_cast<int64_t>(blockIdx.x) * p.sk_units / gridDim.x;
  it.end = static_cast<int64_t>(blockIdx.x + 1) * p.sk_units / gridDim.x;
  return it;
}

__device__ __forceinline__ bool work_next(const WriteParams& p, WorkIter& it, int& tile, int& kb0,
                                          int& kb1) {
  if (it.dp_tile < p.dp_tiles) {
    tile = it.dp_tile;
    kb0 = 0;
    kb1 = p.num_kb;
    it.dp_tile += gridDim.x;
    return true;
  }
  if (it.cur < it.end) {
    const int64_t t = it.cur / p.num_kb;
    kb0 = static_cast<int>(it.cur - t * p.num_kb);
    const int64_t rem = it.end - it.cur;
    kb1 = rem < static_cast<int64_t>(p.num_kb - kb0) ? kb0 + static_cast<int>(rem) : p.num_kb;
    it.cur += kb1 - kb0;
    tile = p.dp_tiles + static_cast<int>(t);
    return true;
  }
  return false;
}

// CTA whose stream-K range holds k-block unit u.
__device__ __forceinline__ int sk_owner(const WriteParams& p, int64_t u) {
  return static_cast<int>(((u + 1) * gridDim.x - 1) / p.sk_units);
}

// Partial-tile slot of a CTA: [kTileN/4][kTileM] float4, so that the 32 rows
// of a warp write one contiguous 512-byte run per 4 columns.
constexpr int kSlotFloats = kTileM * kTileN;

__device__ __forceinline__ float* ws_slot(const WriteParams& p, int cta, int slot) {
  return p.workspace + (static_cast<size_t>(cta) * 2 + slot) * kSlotFloats;
}

template <typename E, int D, bool kBias>
__global__ void __launch_bounds__(kTiledThreads, 1)
    ctx_kv_tiled_kernel(const __grid_constant__ CUtensorMap tmap_x,
                        const __grid_constant__ CUtensorMap tmap_w,
                        const __grid_constant__ WriteParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // operand stages must sit on 1024-byte boundaries (128-byte swizzle atoms)
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* smem_a = smem;
  uint8_t* smem_b = smem + kStages * kStageBytesA;
  SmemBarriers* bars =
      reinterpret_cast<SmemBarriers*>(smem + kStages * (kStageBytesA + kStageBytesB));

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  volatile int* abort_flag = &bars->abort;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&bars->full[s]), 1);
      mbar_init(smem_u32(&bars->empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&bars->tmem_full[b]), 1);
      mbar_init(smem_u32(&bars->tmem_empty[b]), 4);   // one arrival per epilogue warp
    }
    mbar_init(smem_u32(&bars->drain), 1);
    bars->abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmap_x);
    tma_prefetch_desc(&tmap_w);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&bars->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = bars->tmem_base;
  uint64_t* trace = p.trace != nullptr ? p.trace + static_cast<size_t>(blockIdx.x) * kTraceWords : nullptr;
  if (trace != nullptr && threadIdx.x == 0) trace[0] = global_timer_ns();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_w = l2_policy_evict_last();
      const uint64_t pol_x = l2_policy_evict_normal();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t uses[kStages] = {};
      bool ok = true;
      WorkIter it = work_begin(p);
      int tile, kb0, kb1;
      while (ok && work_next(p, it, tile, kb0, kb1)) {
        int m_blk, n_blk;
        tile_coords(tile, p.num_m, p.num_n, m_blk, n_blk);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(smem_u32(&bars->empty[stage]), phase ^ 1u, abort_flag, p.wait_limit_ns)) {
            ok = false;
            break;
          }
          const uint32_t full = smem_u32(&bars->full[stage]);
          mbar_arrive_expect_tx(full, kStageBytesA + kStageBytesB);
          tma_load_2d(smem_u32(smem_a + stage * kStageBytesA), &tmap_x, kb * kTileK,
                      m_blk * kTileM, full, pol_x);
          tma_load_2d(smem_u32(smem_b + stage * kStageBytesB), &tmap_w, kb * kTileK,
                      n_blk * kTileN, full, pol_w);
          ++uses[stage];
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        flag(p, DSPARK_FLAG_TIMEOUT);
      }
      // every load issued must land before the CTA may exit (bounded by time
      // only: an abort must not cut this wait short)
      int never = 0;
#pragma unroll
      for (int s = 0; s < kStages; ++s)
        if (uses[s] > 0) mbar_wait(smem_u32(&bars->full[s]), (uses[s] - 1u) & 1u, &never, p.wait_limit_ns);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = f16_instr_desc(ElemOps<E>::kFmt, kTileM, kTileN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      bool issued = false;
      WorkIter it = work_begin(p);
      int tile, kb0, kb1;
      while (ok && work_next(p, it, tile, kb0, kb1)) {
        if (!mbar_wait(smem_u32(&bars->tmem_empty[acc]), acc_phase ^ 1u, abort_flag,
                       p.wait_limit_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * kAccCols;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(smem_u32(&bars->full[stage]), phase, abort_flag, p.wait_limit_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(smem_a + stage * kStageBytesA);
          const uint32_t b0 = smem_u32(smem_b + stage * kStageBytesB);
#pragma unroll
          for (int k = 0; k < kTileK / 16; ++k) {
            // advancing 16 elements along K = 32 bytes inside the swizzle atom
            umma_f16(d_tmem, sw128_kmajor_desc(a0 + k * 32), sw128_kmajor_desc(b0 + k * 32),
                     idesc, (kb != kb0 || k != 0) ? 1u : 0u);
          }
          issued = true;
          umma_commit(smem_u32(&bars->empty[stage]));
          if (++stage == kStages) {
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
        // all MMAs issued by this thread complete before TMEM is released
        umma_commit(smem_u32(&bars->drain));
        int never = 0;
        mbar_wait(smem_u32(&bars->drain), 0, &never, p.wait_limit_ns);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    constexpr int kHalf = D / 2;
    const int quarter = warp % 4;                 // TMEM lanes this warp may read
    const int row = quarter * 32 + lane;          // token row inside the tile
    const int etid = threadIdx.x - 64;            // 0..127 among the epilogue threads
    int acc = 0;
    uint32_t acc_phase = 0;
    int item = 0;
    WorkIter it = work_begin(p);
    int tile, kb0, kb1;
    while (work_next(p, it, tile, kb0, kb1)) {
      int m_blk, n_blk;
      tile_coords(tile, p.num_m, p.num_n, m_blk, n_blk);
      // the outcome must be warp-uniform: tcgen05.ld below is .sync.aligned
      const bool got = mbar_wait(smem_u32(&bars->tmem_full[acc]), acc_phase, abort_flag,
                                 p.wait_limit_ns);
      uint64_t* tr = (trace != nullptr && etid == 0 && item < kTraceItems) ? trace + 3 + 4 * item : nullptr;
      if (tr != nullptr) {
        tr[0] = static_cast<uint64_t>(tile);
        tr[1] = (static_cast<uint64_t>(kb0) << 16) | static_cast<uint64_t>(kb1);
        tr[2] = global_timer_ns();
      }
      ++item;
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) {
          *abort_flag = 1;
          flag(p, DSPARK_FLAG_TIMEOUT);
        }
        break;
      }
      tc_fence_after();
      const int64_t t = static_cast<int64_t>(m_blk) * kTileM + row;
      const uint32_t t_row = tmem_base + acc * kAccCols + (static_cast<uint32_t>(quarter * 32) << 16);

      // ---- a tile cut between CTAs: publish this part; the last contributor
      // to arrive adds the other parts into its accumulator and finishes it
      bool finish = true;
      if (kb0 != 0 || kb1 != p.num_kb) {
        const int64_t u0 = static_cast<int64_t>(tile - p.dp_tiles) * p.num_kb;
        const int c_first = sk_owner(p, u0);
        const int c_last = sk_owner(p, u0 + p.num_kb - 1);
        float4* mine = reinterpret_cast<float4*>(ws_slot(p, blockIdx.x, kb0 > 0 ? 0 : 1));
#pragma unroll 1
        for (int ch = 0; ch < kTileN / 32; ++ch) {
          uint32_t v[32];
          tmem_ld32(t_row + ch * 32, v);
          if (t < p.T) {
#pragma unroll
            for (int j = 0; j < 8; ++j)
              __stcg(mine + (ch * 8 + j) * kTileM + row,
                     make_float4(f32(v[4 * j]), f32(v[4 * j + 1]), f32(v[4 * j + 2]), f32(v[4 * j + 3])));
          }
          __syncwarp();
        }
        __threadfence();
        named_barrier(1, 128);
        if (etid == 0) {
          const int old = atomicAdd(p.counters + c_last, 1);
          const int last = old == c_last - c_first;
          if (last) p.counters[c_last] = 0;   // ready for the next launch
          if (tr != nullptr) tr[1] |= (last ? 2ull : 1ull) << 32;
          __threadfence();
          *reinterpret_cast<volatile int*>(&bars->last_arrival) = last;
        }
        named_barrier(1, 128);
        // (the flag is next written only after all 128 threads pass the first
        // barrier of a later cut tile, i.e. after every thread has read it)
        finish = *reinterpret_cast<volatile int*>(&bars->last_arrival) != 0;
        if (finish) {
          // accumulator = sum of all parts in ascending contributor order
          // (this CTA's own part taken from TMEM at its place), so the result
          // does not depend on which contributor arrived last
#pragma unroll 1
          for (int ch = 0; ch < kTileN / 32; ++ch) {
            uint32_t own[32];
            tmem_ld32(t_row + ch * 32, own);
            uint32_t v[32];
            if (t < p.T) {
              for (int c = c_first; c <= c_last; ++c) {
                float part[32];
                if (c == static_cast<int>(blockIdx.x)) {
#pragma unroll
                  for (int e = 0; e < 32; ++e) part[e] = f32(own[e]);
                } else {
                  const float4* other =
                      reinterpret_cast<const float4*>(ws_slot(p, c, c == c_first ? 1 : 0));
#pragma unroll
                  for (int j = 0; j < 8; ++j) {
                    const float4 q = __ldcg(other + (ch * 8 + j) * kTileM + row);
                    part[4 * j] = q.x;
                    part[4 * j + 1] = q.y;
                    part[4 * j + 2] = q.z;
                    part[4 * j + 3] = q.w;
                  }
                }
#pragma unroll
                for (int e = 0; e < 32; ++e)
                  v[e] = c == c_first ? __float_as_uint(part[e])
                                      : __float_as_uint(f32(v[e]) + part[e]);
              }
            } else {
#pragma unroll
              for (int e = 0; e < 32; ++e) v[e] = own[e];
            }
            __syncwarp();
            tmem_st32(t_row + ch * 32, v);
          }
        }
      }

      if (finish) {
        // ---- per-token decision (same for every head of the tile)
        bool write = false;
        int64_t loc = 0, pos = 0;
        if (t < p.T) {
          loc = p.cache_loc[t];
          write = loc >= 0;
          if (write && p.loc_row_width > 0) {
            const int64_t b = t / p.loc_row_width;
            if (t - b * p.loc_row_width >= static_cast<int64_t>(p.commit_lens[b])) write = false;
          }
          if (write) {
            pos = p.positions[t];
            if (pos < 0 || pos >= p.max_pos) {
              flag(p, DSPARK_FLAG_POS_RANGE);
              write = false;
            } else if (loc >= p.pool_slots) {
              flag(p, DSPARK_FLAG_LOC_RANGE);
              write = false;
            }
          }
        }

#pragma unroll 1
        for (int seg = 0; seg < kTileN / D; ++seg) {
          const int c0 = n_blk * kTileN + seg * D;
          if (c0 >= p.N) break;
          const int layer = c0 / (2 * p.KV);
          const int r = c0 - layer * 2 * p.KV;
          const bool is_v = r >= p.KV;
          const int head = (is_v ? r - p.KV : r) / D;
          const uint32_t t_seg = t_row + seg * D;
          if (is_v) {
            E* dst = reinterpret_cast<E*>(p.v_pool[layer]) + loc * p.v_stride[layer] + head * D;
#pragma unroll
            for (int ch = 0; ch < D / 32; ++ch) {
              uint32_t v[32];
              tmem_ld32(t_seg + ch * 32, v);
              if (write) {
                uint32_t o[16];
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                  float a = f32(v[e]), b = f32(v[e + 1]);
                  if (kBias) {
                    a += ElemOps<E>::load(p.bias, c0 + ch * 32 + e);
                    b += ElemOps<E>::load(p.bias, c0 + ch * 32 + e + 1);
                  }
                  o[e / 2] = ElemOps<E>::pack(a, b);
                }
                store32(dst + ch * 32, o);
              }
              __syncwarp();
            }
          } else {
            // RMSNorm: sum of squares over this thread's row of the head
            float ss = 0.f;
#pragma unroll
            for (int ch = 0; ch < D / 32; ++ch) {
              uint32_t v[32];
              tmem_ld32(t_seg + ch * 32, v);
#pragma unroll
              for (int e = 0; e < 32; ++e) {
                float x = f32(v[e]);
                if (kBias) x += ElemOps<E>::load(p.bias, c0 + ch * 32 + e);
                ss = fmaf(x, x, ss);
              }
            }
            const float inv = rsqrtf(ss * (1.0f / D) + p.eps);
            const float* w = p.knorm + static_cast<int64_t>(layer) * D;
            const float* cs = p.cos_sin + pos * D;
            E* dst = reinterpret_cast<E*>(p.k_pool[layer]) + loc * p.k_stride[layer] + head * D;
#pragma unroll
            for (int hc = 0; hc < kHalf / 32; ++hc) {
              uint32_t a[32], b[32];
              tmem_ld32(t_seg + hc * 32, a);
              tmem_ld32(t_seg + kHalf + hc * 32, b);
              if (write) {
                uint32_t o1[16], o2[16];
#pragma unroll
                for (int e4 = 0; e4 < 32; e4 += 4) {
                  const int i = hc * 32 + e4;
                  const float4 w1 = *reinterpret_cast<const float4*>(w + i);
                  const float4 w2 = *reinterpret_cast<const float4*>(w + kHalf + i);
                  const float4 c4 = *reinterpret_cast<const float4*>(cs + i);
                  const float4 s4 = *reinterpret_cast<const float4*>(cs + kHalf + i);
                  const float wa[4] = {w1.x, w1.y, w1.z, w1.w};
                  const float wb[4] = {w2.x, w2.y, w2.z, w2.w};
                  const float cc[4] = {c4.x, c4.y, c4.z, c4.w};
                  const float sn[4] = {s4.x, s4.y, s4.z, s4.w};
                  float r1[4], r2[4];
#pragma unroll
                  for (int j = 0; j < 4; ++j) {
                    float x1 = f32(a[e4 + j]);
                    float x2 = f32(b[e4 + j]);
                    if (kBias) {
                      x1 += ElemOps<E>::load(p.bias, c0 + i + j);
                      x2 += ElemOps<E>::load(p.bias, c0 + kHalf + i + j);
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
                store32(dst + hc * 32, o1);
                store32(dst + kHalf + hc * 32, o2);
              }
              __syncwarp();
            }
          }
        }
      }
      // accumulator fully read: hand it back to the MMA warp
      tc_fence_before();
      __syncwarp();
      if (tr != nullptr) tr[3] = global_timer_ns();
      if (lane == 0) mbar_arrive(smem_u32(&bars->tmem_empty[acc]));
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
  if (trace != nullptr && threadIdx.x == 0) {
    trace[1] = global_timer_ns();
    WorkIter it = work_begin(p);
    int tile, kb0, kb1, n = 0;
    while (work_next(p, it, tile, kb0, kb1)) ++n;
    trace[2] = static_cast<uint64_t>(n);
  }
}

template <typename E, int D, bool kBias>
cudaError_t launch_one(int device, const CUtensorMap& tx, const CUtensorMap& tw,
                       const WriteParams& p, int grid, cudaStream_t stream) {
  auto kern = ctx_kv_tiled_kernel<E, D, kBias>;
  // the opt-in shared-memory size is set once per device and instantiation
  static std::atomic<uint64_t> attr_set{0};
  const uint64_t bit = 1ull << (device & 63);
  const size_t smem = tiled_smem_bytes();
  if (!(attr_set.load() & bit)) {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attr_set.fetch_or(bit);
  }
  kern<<<grid, kTiledThreads, smem, stream>>>(tx, tw, p);
  return cudaGetLastError();
}

}  // namespace

size_t tiled_smem_bytes() {
  return 1024 /* alignment slack */ + kStages * (kStageBytesA + kStageBytesB) + sizeof(SmemBarriers);
}

cudaError_t launch_tiled(int device, int dtype, int head_dim, bool has_bias, const CUtensorMap& tx,
                         const CUtensorMap& tw, const WriteParams& p, int grid,
                         cudaStream_t stream) {
  if (dtype == DSPARK_DTYPE_BF16) {
    if (head_dim == 128)
      return has_bias ? launch_one<__nv_bfloat16, 128, true>(device, tx, tw, p, grid, stream)
                      : launch_one<__nv_bfloat16, 128, false>(device, tx, tw, p, grid, stream);
    return has_bias ? launch_one<__nv_bfloat16, 64, true>(device, tx, tw, p, grid, stream)
                    : launch_one<__nv_bfloat16, 64, false>(device, tx, tw, p, grid, stream);
  }
  if (head_dim == 128)
    return has_bias ? launch_one<__half, 128, true>(device, tx, tw, p, grid, stream)
                    : launch_one<__half, 128, false>(device, tx, tw, p, grid, stream);
  return has_bias ? launch_one<__half, 64, true>(device, tx, tw, p, grid, stream)
                  : launch_one<__half, 64, false>(device, tx, tw, p, grid, stream);
}

}  // namespace dspark
