// Draft attention over the written KV pool (sglang PR #35499 summary page,
// K3 DSpark draft attention: GQA, non-causal, the context gathered from the
// pool through kv_indices, split over the context and merged).
//
// Stage 1 (one CTA per request and context split): the CTA holds the
// request's queries of every KV head in shared memory and streams its share
// of the context (then, for split 0, the block's own keys) in chunks of 16
// tokens: each token's pool row (all KV heads, contiguous) is copied with
// 16-byte asynchronous copies into a double-buffered stage, 16-byte units
// XOR-swizzled by row so that the ldmatrix reads below are conflict-free.
// Each warp owns 16 query rows of one KV head (rows = block x group, row
// i*group + hh is query i of head g*group + hh) and runs the flash-attention
// recurrence on the tensor cores (mma.sync m16n8k16: the rows are too few for
// a 128-row tcgen05 tile, and the stream of gathered 256-byte rows, not the
// MMA, bounds the kernel): S = Q K^T, online softmax in the log2 domain with
// the running max and sum in registers, O += P V with P re-packed from the S
// accumulators.  It writes its unnormalised O, max and sum to the workspace.
// Stage 2 merges the splits of each query row with the log-sum-exp weights and
// stores the output in the model dtype.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>

#include "../../include/dspark_attention.h"

namespace dspark {
namespace {

constexpr int kChunk = 16;               // keys per pipeline stage
constexpr int kMaxSplitTokens = 2048;    // context tokens per split at most
constexpr int kWaveCtas = 152;           // stage-1 CTAs resident at once (one per SM of a GB300)
constexpr int kSplitGoal = 1024;         // context tokens per split aimed for
constexpr int kMaxWarps = 16;
constexpr int kCombineWarps = 8;

struct AttnPlan {
  int splits;
  int split_tokens;
};

// Context split: about kSplitGoal tokens per split, at least two waves of
// CTAs (more splits cost workspace traffic and merge work: measured slower),
// and among up to twice that many splits the count whose CTAs fill the last
// wave best (a request's unused splits end at once, so this matters for
// equal context lengths).  Depends on the sizes only, so the workspace size
// query and the launch agree.
AttnPlan make_plan(int64_t batch, int64_t max_context) {
  AttnPlan pl;
  if (batch < 1) batch = 1;
  int64_t base = (max_context + kSplitGoal - 1) / kSplitGoal;
  const int64_t waves2 = (2 * kWaveCtas + batch - 1) / batch;
  if (base < waves2) base = waves2;
  if (base < 1) base = 1;
  int64_t best = base;
  double best_eff = 0.0;
  for (int64_t sp = base; sp <= 2 * base; ++sp) {
    const int64_t ctas = batch * sp;
    const double eff = static_cast<double>(ctas) / (((ctas + kWaveCtas - 1) / kWaveCtas) * kWaveCtas);
    if (eff > best_eff + 1e-9) {
      best_eff = eff;
      best = sp;
    }
  }
  int64_t c = (max_context + best - 1) / best;
  c = (c + kChunk - 1) / kChunk * kChunk;
  if (c < kChunk) c = kChunk;
  if (c > kMaxSplitTokens) c = kMaxSplitTokens;
  int64_t splits = (max_context + c - 1) / c;
  if (splits < 1) splits = 1;
  pl.splits = static_cast<int>(splits);
  pl.split_tokens = static_cast<int>(c);
  return pl;
}

struct AttnParams {
  const void* q;
  const void* k_ext;
  const void* v_ext;
  const void* k_pool;
  const void* v_pool;
  int64_t pool_row_stride;
  int64_t pool_slots;
  const int64_t* kv_indices;
  const int64_t* kv_start;
  int64_t batch;
  int block, nq, nkv, group, rows, splits, split_tokens;
  float scale_log2;
  void* out;
  float* ws_o;      // [batch][splits][nkv*rows][D]
  float* ws_ml;     // [batch][splits][nkv*rows][2]
  uint32_t* status;
};

template <typename E>
struct MmaOps;

template <>
struct MmaOps<__nv_bfloat16> {
  __device__ static __forceinline__ void mma(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
  __device__ static __forceinline__ uint32_t pack(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    uint32_t u;
    memcpy(&u, &h, 4);
    return u;
  }
  __device__ static __forceinline__ uint16_t one(float v) {
    __nv_bfloat16 h = __float2bfloat16_rn(v);
    uint16_t u;
    memcpy(&u, &h, 2);
    return u;
  }
};

template <>
struct MmaOps<__half> {
  __device__ static __forceinline__ void mma(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
  __device__ static __forceinline__ uint32_t pack(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    uint32_t u;
    memcpy(&u, &h, 4);
    return u;
  }
  __device__ static __forceinline__ uint16_t one(float v) {
    __half h = __float2half_rn(v);
    uint16_t u;
    memcpy(&u, &h, 2);
    return u;
  }
};

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                              uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Shared memory of stage 1 (byte offsets from a 128-byte aligned base).
struct AttnSmem {
  uint32_t q_off, kv_off, valid_off, idx_off, stage_bytes, row_bytes, total;
};

__host__ __device__ inline AttnSmem attn_smem(int D, int nkv, int rows, int split_tokens) {
  AttnSmem s;
  s.row_bytes = static_cast<uint32_t>(nkv * D * 2);                   // one token's pool row, all KV heads
  s.q_off = 0;
  s.kv_off = static_cast<uint32_t>(nkv * rows * D * 2);              // Q of every KV head
  s.stage_bytes = 2 * kChunk * s.row_bytes;                            // K then V rows of one chunk
  s.valid_off = s.kv_off + 2 * s.stage_bytes;
  s.idx_off = s.valid_off + 2 * kChunk * 4;
  s.total = s.idx_off + static_cast<uint32_t>(split_tokens) * 8;
  return s;
}

template <typename E, int D>
__global__ void __launch_bounds__(kMaxWarps * 32, 1) attn_split_kernel(const AttnParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int kUnitsD = D / 8;                 // 16-byte units of one head row
  const int nkv = p.nkv, rows = p.rows;
  const AttnSmem L = attn_smem(D, nkv, rows, p.split_tokens);
  const int units_row = nkv * kUnitsD;           // 16-byte units of one token's pool row
  uint8_t* q_s = smem + L.q_off;
  uint8_t* kv_s = smem + L.kv_off;
  int* valid_s = reinterpret_cast<int*>(smem + L.valid_off);
  int64_t* idx_s = reinterpret_cast<int64_t*>(smem + L.idx_off);

  const int tid = threadIdx.x, nthreads = blockDim.x;
  const int warp = tid / 32, lane = tid % 32;
  const int64_t b = blockIdx.y;
  const int s = blockIdx.x;
  const int64_t k0 = p.kv_start[b];
  int64_t n_b = p.kv_start[b + 1] - k0;
  const int64_t cap = static_cast<int64_t>(p.splits) * p.split_tokens;
  if (n_b > cap) {
    if (s == 0 && tid == 0 && p.status != nullptr) atomicOr(p.status, DSPARK_FLAG_CONTEXT_RANGE);
    n_b = cap;
  }
  if (n_b < 0) n_b = 0;
  const int64_t lo = static_cast<int64_t>(s) * p.split_tokens;
  const int64_t hi = lo + p.split_tokens < n_b ? lo + p.split_tokens : n_b;
  const int n_ctx = hi > lo ? static_cast<int>(hi - lo) : 0;
  const bool has_ext = s == 0;
  if (!has_ext && n_ctx == 0) return;            // nothing in this split (uniform)

  for (int t = tid; t < n_ctx; t += nthreads) idx_s[t] = p.kv_indices[k0 + lo + t];
  __syncthreads();

  const int ext_chunks = has_ext ? (p.block + kChunk - 1) / kChunk : 0;
  const int total_chunks = ext_chunks + (n_ctx + kChunk - 1) / kChunk;

  // queries of every KV head: smem row g*rows + r holds query i = r / group of
  // head g*group + r % group
  {
    const E* q = static_cast<const E*>(p.q);
    const int nunits = nkv * rows * kUnitsD;
    for (int x = tid; x < nunits; x += nthreads) {
      const int row = x / kUnitsD, u = x % kUnitsD;
      const int g = row / rows, r = row % rows;
      const int i = r / p.group, hh = r % p.group;
      const E* src = q + ((b * p.block + i) * p.nq + g * p.group + hh) * D + u * 8;
      cp_async16(smem_addr(q_s + row * (D * 2) + ((u ^ (row & 7)) * 16)), src);
    }
  }

  const bool units_fixed = nthreads % units_row == 0;
  const int my_u = tid % units_row, my_j0 = tid / units_row, j_step = nthreads / units_row;
  auto issue = [&](int ci, int stage) {
    uint8_t* ks = kv_s + stage * L.stage_bytes;
    uint8_t* vs = ks + kChunk * L.row_bytes;
    const E* kbase;
    const E* vbase;
    auto copy_unit = [&](int j, int u) {
      bool ok;
      int64_t row_off;
      if (ci < ext_chunks) {
        const int e = ci * kChunk + j;
        ok = e < p.block;
        row_off = (b * p.block + e) * static_cast<int64_t>(nkv) * D;
        kbase = static_cast<const E*>(p.k_ext);
        vbase = static_cast<const E*>(p.v_ext);
      } else {
        const int t = (ci - ext_chunks) * kChunk + j;
        ok = t < n_ctx;
        const int64_t slot = ok ? idx_s[t] : 0;
        if (ok && (slot < 0 || slot >= p.pool_slots)) {
          ok = false;
          if (u == 0 && p.status != nullptr) atomicOr(p.status, DSPARK_FLAG_LOC_RANGE);
        }
        row_off = slot * p.pool_row_stride;
        kbase = static_cast<const E*>(p.k_pool);
        vbase = static_cast<const E*>(p.v_pool);
      }
      const uint32_t off = j * L.row_bytes + ((u ^ (j & 7)) * 16);
      if (ok) {
        cp_async16(smem_addr(ks + off), kbase + row_off + u * 8);
        cp_async16(smem_addr(vs + off), vbase + row_off + u * 8);
      } else {
        *reinterpret_cast<uint4*>(ks + off) = make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(vs + off) = make_uint4(0u, 0u, 0u, 0u);
      }
      if (u == 0) valid_s[stage * kChunk + j] = ok ? 1 : 0;
    };
    if (units_fixed) {
      // the usual case: each thread copies one fixed 16-byte unit of every
      // j_step-th token row (no integer division per unit)
      for (int j = my_j0; j < kChunk; j += j_step) copy_unit(j, my_u);
    } else {
      for (int x = tid; x < kChunk * units_row; x += nthreads) copy_unit(x / units_row, x % units_row);
    }
    cp_async_commit();
  };

  // this warp: 16 query rows (mt) of KV head g
  const int tiles_per_head = rows / 16;
  const int g = warp / tiles_per_head, mt = warp % tiles_per_head;
  const bool active = warp < nkv * tiles_per_head;
  const int grp = lane / 4, tig = lane % 4;
  float acc[D / 8][4];
#pragma unroll
  for (int n = 0; n < D / 8; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

  issue(0, 0);
  for (int ci = 0; ci < total_chunks; ++ci) {
    const int stage = ci & 1;
    if (ci + 1 < total_chunks) {
      issue(ci + 1, stage ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    if (active) {
      const uint8_t* ks = kv_s + stage * L.stage_bytes;
      const uint8_t* vs = ks + kChunk * L.row_bytes;
      // ---- S = Q K^T for 16 keys
      float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      const int mi = lane / 8;
      const int qrow = g * rows + mt * 16 + (mi & 1) * 8 + lane % 8;
      const int key_b = (mi >> 1) * 8 + lane % 8;
#pragma unroll
      for (int ks16 = 0; ks16 < D / 16; ++ks16) {
        uint32_t a[4];
        const int qu = 2 * ks16 + (mi >> 1);
        ldsm_x4(smem_addr(q_s + qrow * (D * 2) + ((qu ^ (qrow & 7)) * 16)), a[0], a[1], a[2], a[3]);
        uint32_t b0, b1, b2, b3;
        const int ku = g * kUnitsD + 2 * ks16 + (mi & 1);
        ldsm_x4(smem_addr(ks + key_b * L.row_bytes + ((ku ^ (key_b & 7)) * 16)), b0, b1, b2, b3);
        MmaOps<E>::mma(sc[0], a, b0, b1);
        MmaOps<E>::mma(sc[1], a, b2, b3);
      }
      // ---- online softmax (log2 domain); masked keys get -inf
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int2 vk = *reinterpret_cast<const int2*>(valid_s + stage * kChunk + nt * 8 + 2 * tig);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const bool ok = (e == 0 ? vk.x : vk.y) != 0;
          sc[nt][e] = ok ? sc[nt][e] * p.scale_log2 : -INFINITY;
          sc[nt][2 + e] = ok ? sc[nt][2 + e] * p.scale_log2 : -INFINITY;
          mx0 = fmaxf(mx0, sc[nt][e]);
          mx1 = fmaxf(mx1, sc[nt][2 + e]);
        }
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
      const float al0 = n0 == -INFINITY ? 1.f : exp2f(m0 - n0);
      const float al1 = n1 == -INFINITY ? 1.f : exp2f(m1 - n1);
      m0 = n0;
      m1 = n1;
      float pr[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          pr[nt][e] = n0 == -INFINITY ? 0.f : exp2f(sc[nt][e] - n0);
          pr[nt][2 + e] = n1 == -INFINITY ? 0.f : exp2f(sc[nt][2 + e] - n1);
        }
      }
      l0 = l0 * al0 + pr[0][0] + pr[0][1] + pr[1][0] + pr[1][1];
      l1 = l1 * al1 + pr[0][2] + pr[0][3] + pr[1][2] + pr[1][3];
      // the running max of a row seldom changes after the first chunks: skip
      // the multiply by exactly 1
      if (al0 != 1.f || al1 != 1.f) {
#pragma unroll
        for (int n = 0; n < D / 8; ++n) {
          acc[n][0] *= al0;
          acc[n][1] *= al0;
          acc[n][2] *= al1;
          acc[n][3] *= al1;
        }
      }
      // ---- O += P V (P re-packed from the score accumulators)
      uint32_t pa[4];
      pa[0] = MmaOps<E>::pack(pr[0][0], pr[0][1]);
      pa[1] = MmaOps<E>::pack(pr[0][2], pr[0][3]);
      pa[2] = MmaOps<E>::pack(pr[1][0], pr[1][1]);
      pa[3] = MmaOps<E>::pack(pr[1][2], pr[1][3]);
      const int vkey = (mi & 1) * 8 + lane % 8;
#pragma unroll
      for (int dn = 0; dn < D / 8; dn += 2) {
        uint32_t b0, b1, b2, b3;
        const int vu = g * kUnitsD + dn + (mi >> 1);
        ldsm_x4_trans(smem_addr(vs + vkey * L.row_bytes + ((vu ^ (vkey & 7)) * 16)), b0, b1, b2, b3);
        MmaOps<E>::mma(acc[dn], pa, b0, b1);
        MmaOps<E>::mma(acc[dn + 1], pa, b2, b3);
      }
    }
    __syncthreads();   // this stage is refilled two chunks later
  }

  if (!active) return;
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  const int nrows = nkv * rows;
  const int64_t base_row = (b * p.splits + s) * static_cast<int64_t>(nrows) + g * rows + mt * 16 + grp;
  float* o0 = p.ws_o + base_row * D;
  float* o1 = o0 + 8 * D;
#pragma unroll
  for (int n = 0; n < D / 8; ++n) {
    *reinterpret_cast<float2*>(o0 + n * 8 + 2 * tig) = make_float2(acc[n][0], acc[n][1]);
    *reinterpret_cast<float2*>(o1 + n * 8 + 2 * tig) = make_float2(acc[n][2], acc[n][3]);
  }
  if (tig == 0) {
    *reinterpret_cast<float2*>(p.ws_ml + base_row * 2) = make_float2(m0, l0);
    *reinterpret_cast<float2*>(p.ws_ml + (base_row + 8) * 2) = make_float2(m1, l1);
  }
}

// Stage 2: one warp per (request, query row of a KV head): merge the splits.
template <typename E, int D>
__global__ void __launch_bounds__(kCombineWarps * 32) attn_combine_kernel(const AttnParams p) {
  const int nrows = p.nkv * p.rows;
  const int64_t wid = static_cast<int64_t>(blockIdx.x) * kCombineWarps + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (wid >= p.batch * nrows) return;
  const int64_t b = wid / nrows;
  const int row = static_cast<int>(wid % nrows);
  int64_t n_b = p.kv_start[b + 1] - p.kv_start[b];
  const int64_t cap = static_cast<int64_t>(p.splits) * p.split_tokens;
  if (n_b > cap) n_b = cap;
  if (n_b < 0) n_b = 0;
  int n_split = static_cast<int>((n_b + p.split_tokens - 1) / p.split_tokens);
  if (n_split < 1) n_split = 1;
  const int64_t r0 = b * p.splits * static_cast<int64_t>(nrows) + row;
  float M = -INFINITY;
  for (int s = 0; s < n_split; ++s) M = fmaxf(M, p.ws_ml[(r0 + static_cast<int64_t>(s) * nrows) * 2]);
  constexpr int kPer = D / 32;
  float o[kPer] = {};
  float Lsum = 0.f;
  for (int s = 0; s < n_split; ++s) {
    const int64_t r = r0 + static_cast<int64_t>(s) * nrows;
    const float m = p.ws_ml[r * 2], l = p.ws_ml[r * 2 + 1];
    const float w = m == -INFINITY ? 0.f : exp2f(m - M);
    Lsum += w * l;
    const float* src = p.ws_o + r * D + lane * kPer;
#pragma unroll
    for (int k = 0; k < kPer; ++k) o[k] += w * src[k];
  }
  const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
  const int g = row / p.rows, rr = row % p.rows;
  const int i = rr / p.group, hh = rr % p.group;
  uint16_t* dst = static_cast<uint16_t*>(p.out) + ((b * p.block + i) * p.nq + g * p.group + hh) * D + lane * kPer;
#pragma unroll
  for (int k = 0; k < kPer; ++k) dst[k] = MmaOps<E>::one(o[k] * inv);
}

template <typename E, int D>
cudaError_t launch_attention(const AttnParams& p, int warps, cudaStream_t stream) {
  const AttnSmem L = attn_smem(D, p.nkv, p.rows, p.split_tokens);
  auto k1 = attn_split_kernel<E, D>;
  cudaError_t e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(L.total));
  if (e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>(p.splits), static_cast<unsigned>(p.batch));
  k1<<<grid, warps * 32, L.total, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t rows = p.batch * p.nkv * p.rows;
  attn_combine_kernel<E, D><<<static_cast<unsigned>((rows + kCombineWarps - 1) / kCombineWarps),
                              kCombineWarps * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

int sm103_attn(int device) {
  static int cache[64] = {0};
  const int d = device & 63;
  if (cache[d] == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess)
      return 0;
    cache[d] = (major == 10 && minor == 3) ? 1 : -1;
  }
  return cache[d] > 0;
}

// Host-side shape checks shared by the size query and the call.  Returns a
// dspark_status.
int check_shape(int64_t batch, int32_t block, int32_t nq, int32_t nkv, int32_t D, int64_t max_context,
                AttnPlan* plan, int* warps, AttnSmem* smem) {
  if (batch < 0 || block < 1 || nq < 1 || nkv < 1 || max_context < 0) return DSPARK_E_INVALID_ARG;
  if (D != 64 && D != 128) return DSPARK_E_HEAD_DIM;
  if (nq % nkv != 0) return DSPARK_E_SHAPE_MISMATCH;
  const int64_t rows = static_cast<int64_t>(block) * (nq / nkv);
  if (rows % 16 != 0 || rows > 64) return DSPARK_E_SHAPE_MISMATCH;
  const int64_t w = nkv * rows / 16;
  if (w > kMaxWarps) return DSPARK_E_SHAPE_MISMATCH;
  *plan = make_plan(batch > 0 ? batch : 1, max_context);
  *warps = static_cast<int>(w);
  *smem = attn_smem(D, nkv, static_cast<int>(rows), plan->split_tokens);
  if (smem->total > 227u * 1024u) return DSPARK_E_SHAPE_MISMATCH;
  return DSPARK_OK;
}

int64_t workspace_for(int64_t batch, int32_t block, int32_t nq, int32_t D, const AttnPlan& pl) {
  const int64_t rows = batch * block * static_cast<int64_t>(nq);
  return rows * pl.splits * (static_cast<int64_t>(D) + 2) * 4;
}

}  // namespace
}  // namespace dspark

extern "C" int64_t dspark_draft_attention_workspace_bytes(int64_t batch, int32_t block, int32_t num_q_heads,
                                                          int32_t num_kv_heads, int32_t head_dim,
                                                          int64_t max_context) {
  using namespace dspark;
  AttnPlan pl;
  int warps;
  AttnSmem sm;
  if (check_shape(batch, block, num_q_heads, num_kv_heads, head_dim, max_context, &pl, &warps, &sm) != DSPARK_OK)
    return 0;
  return workspace_for(batch, block, num_q_heads, head_dim, pl);
}

extern "C" int dspark_draft_attention(const void* q, const void* k_ext, const void* v_ext, const void* k_pool,
                                      const void* v_pool, int64_t pool_row_stride, int64_t pool_slots,
                                      const int64_t* kv_indices, const int64_t* kv_start, int64_t batch,
                                      int32_t block, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                      int32_t dtype, float sm_scale, int64_t max_context, void* out,
                                      void* workspace, int64_t workspace_bytes, uint32_t* status,
                                      void* stream_) {
  using namespace dspark;
  AttnPlan pl;
  int warps;
  AttnSmem sm;
  const int st = check_shape(batch, block, num_q_heads, num_kv_heads, head_dim, max_context, &pl, &warps, &sm);
  if (st != DSPARK_OK) return st;
  if (dtype != DSPARK_DTYPE_BF16 && dtype != DSPARK_DTYPE_FP16) return DSPARK_E_DTYPE_MISMATCH;
  if (batch == 0) return DSPARK_OK;
  if (q == nullptr || k_ext == nullptr || v_ext == nullptr || k_pool == nullptr || v_pool == nullptr ||
      kv_indices == nullptr || kv_start == nullptr || out == nullptr || workspace == nullptr || pool_slots < 0 ||
      !(sm_scale > 0.f))
    return DSPARK_E_INVALID_ARG;
  if (pool_row_stride < static_cast<int64_t>(num_kv_heads) * head_dim) return DSPARK_E_POOL_LAYOUT;
  if (!aligned16(q) || !aligned16(k_ext) || !aligned16(v_ext) || !aligned16(k_pool) || !aligned16(v_pool) ||
      !aligned16(out) || !aligned16(workspace) || pool_row_stride % 8 != 0)
    return DSPARK_E_ALIGNMENT;
  if (workspace_bytes < workspace_for(batch, block, num_q_heads, head_dim, pl)) return DSPARK_E_SCRATCH_LIMIT;
  if (batch > 65535) return DSPARK_E_INVALID_ARG;   // grid y
  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess || !sm103_attn(device)) return DSPARK_E_DEVICE;

  AttnParams p;
  std::memset(&p, 0, sizeof(p));
  p.q = q;
  p.k_ext = k_ext;
  p.v_ext = v_ext;
  p.k_pool = k_pool;
  p.v_pool = v_pool;
  p.pool_row_stride = pool_row_stride;
  p.pool_slots = pool_slots;
  p.kv_indices = kv_indices;
  p.kv_start = kv_start;
  p.batch = batch;
  p.block = block;
  p.nq = num_q_heads;
  p.nkv = num_kv_heads;
  p.group = num_q_heads / num_kv_heads;
  p.rows = block * p.group;
  p.splits = pl.splits;
  p.split_tokens = pl.split_tokens;
  p.scale_log2 = sm_scale * 1.4426950408889634f;
  p.out = out;
  const int64_t rows_all = batch * static_cast<int64_t>(p.nkv) * p.rows;
  p.ws_o = static_cast<float*>(workspace);
  p.ws_ml = p.ws_o + rows_all * pl.splits * head_dim;
  p.status = status;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  cudaError_t e;
  if (dtype == DSPARK_DTYPE_BF16)
    e = head_dim == 128 ? launch_attention<__nv_bfloat16, 128>(p, warps, stream)
                        : launch_attention<__nv_bfloat16, 64>(p, warps, stream);
  else
    e = head_dim == 128 ? launch_attention<__half, 128>(p, warps, stream)
                        : launch_attention<__half, 64>(p, warps, stream);
  return e == cudaSuccess ? DSPARK_OK : DSPARK_E_CUDA;
}
