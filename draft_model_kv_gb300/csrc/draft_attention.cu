// Draft attention over the written KV pool (sglang PR #35499 summary page,
// K3 DSpark draft attention: GQA, non-causal, the context gathered from the
// pool through kv_indices, split over the context and merged).
//
// Stage 1 runs on the tcgen05 tensor cores, one CTA per (KV head, context
// split, request).  For KV head g the query rows (row r = i*group + hh: query i
// of the block, head g*group + hh) are at most 32, too few for an MMA's M, so
// the keys take the M side:
//
//   S^T[key][row]  = K_g[key] . Q_g[row]            M = 128 keys, N = rows, K = D
//   O^T[d][row]   += V_g^T[d][key] . P^T[row][key]  M = 128 (d), N = rows, K = 128 keys
//
// both accumulated in TMEM (S double-buffered; O once per group of 32 keys).
// Four producer warps gather, per 128-key chunk, each key's 2 x D x 2 bytes of
// head g (its K and V rows of the pool, or of the block's own keys for the
// last chunk of split 0) with 16-byte asynchronous copies into the
// 128-byte-swizzled layout of the MMA operands, three stages deep, a warp
// instruction covering whole rows; the copies complete on mbarriers of the K
// and V halves of a stage (the K half is free again once the scores are
// computed), and slot indices are loaded two chunks ahead.  The staged chunk
// is the K-major A operand of the first product and, read as an MN-major
// operand, the V^T of the second.  Sixteen softmax warps, four warpgroups of 8 query rows, own one
// key (TMEM lane) per thread.  Each warp keeps its own running maximum and
// sum per row over its 32 keys of every chunk (warp transpose-reductions, no
// exchange with the other warps), writes P^T (model dtype) to shared memory as
// the B operand of the second product, whose 32-key groups accumulate into
// four separate O^T, and raises its maximum only when a chunk exceeds it by
// more than 2^8; the warps of a warpgroup meet once per chunk to rescale the
// O^T of the warps whose maximum grew.  The four partial results of a row are
// merged when the split ends.  One thread issues the MMAs as their inputs
// become ready: the scores of the next landed chunk, and the product of the
// oldest chunk whose P^T is written.  Each split writes its unnormalised O,
// maximum and sum to the workspace; stage 2 merges the splits of each query
// row with the log-sum-exp weights and stores the output in the model dtype.
// Stage 2 is a programmatic dependent launch: its CTAs may start on SMs that
// stage 1's last wave leaves idle and wait there (griddepcontrol.wait) for
// stage 1 to complete.  Neither stage allocates or synchronises with the
// host, so a call can be captured in a CUDA graph.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <type_traits>

#include "../../include/dspark_attention.h"
#include "ptx.cuh"

namespace dspark {
namespace {

constexpr int kKeys = 128;               // keys per chunk: the first product's M (TMEM lanes)
constexpr int kQRows = 32;               // query rows per KV head, at most (TMEM columns per accumulator)
constexpr int kWgRows = 8;               // query rows of one softmax warpgroup
constexpr int kAttnStages = 3;           // chunks in the operand ring
constexpr int kSoftWarps = 16;           // warps 0-15: softmax, four warpgroups of 8 query rows
constexpr int kProdWarp0 = kSoftWarps;   // then the producers
constexpr int kProdWarps = 4;
constexpr int kProdThreads = kProdWarps * 32;
constexpr int kKeysPerProdWarp = kKeys / kProdWarps;
constexpr int kAttnMmaWarp = kProdWarp0 + kProdWarps;   // the MMA issuer
constexpr int kAttnThreads = (kAttnMmaWarp + 1) * 32;
constexpr int kSplitGoal = 8192;         // context tokens per split aimed for
constexpr int kMaxSplitTokens = 8192;
constexpr int kWaveCtas = 152;           // stage-1 CTAs resident at once (one per SM of a GB300)
constexpr int kCombineWarps = 8;
constexpr uint32_t kAttnTmemCols = 256;  // S0 at column 0, S1 at 32, O of key group w at 64 + 32 w
constexpr uint64_t kAttnWaitNs = 2000000000ull;
// A row's running maximum (log2 domain) is raised, and O and the sum
// rescaled, only when a chunk's maximum exceeds it by more than this: the
// weights stay below 2^8 (exact enough in the model dtype), and O seldom needs
// the previous chunk's product to be complete.
constexpr float kLazyRescale = 8.f;
constexpr int64_t kNoKey = INT64_MIN;    // a key position past the context

struct AttnPlan {
  int splits;
  int split_tokens;
};

// Context split: about kSplitGoal tokens per split (a multiple of the chunk),
// and more, shorter splits when batch x KV heads CTAs per split would not
// fill four waves.  Every CTA pays ~5 us of start and tail (the context
// bounds, then the first chunk's slot indices, then its rows, before the
// first product; the merge of its key groups and the workspace writes after
// the last), so long splits pay off while enough CTAs remain to balance the
// SMs: on 64 requests of 8 x 32 heads with contexts of 1k-32k tokens, splits
// of 2048 / 4096 / 6144-12288 / 16384 tokens took 1015 / 937 / 922 / 947 us;
// 4096-token contexts keep two splits of 2048.  Depends on the sizes only, so
// the workspace size query and the launch agree.
AttnPlan make_plan(int64_t batch, int nkv, int64_t max_context) {
  AttnPlan pl;
  if (batch < 1) batch = 1;
  int64_t splits = (max_context + kSplitGoal - 1) / kSplitGoal;
  const int64_t per_split = batch * nkv;
  const int64_t want = (4 * kWaveCtas + per_split - 1) / per_split;
  if (splits < want) splits = want;
  if (splits < 1) splits = 1;
  int64_t c = (max_context + splits - 1) / splits;
  c = (c + kKeys - 1) / kKeys * kKeys;
  if (c < kKeys) c = kKeys;
  if (c > kMaxSplitTokens) c = kMaxSplitTokens;
  splits = (max_context + c - 1) / c;
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
  int64_t max_context;   // longer contexts are cut here (and flagged)
  int block, nq, nkv, group, rows, splits, split_tokens;
  float scale_log2;
  void* out;
  float* ws_o;      // [batch][splits][nkv*rows][D]
  float* ws_ml;     // [batch][splits][nkv*rows][2]
  uint32_t* status;
  uint64_t test_wait_ns;   // diagnostics: 0, or the bound of a wait that never completes
};

template <typename E>
__device__ __forceinline__ uint16_t to_bits(float v);
template <>
__device__ __forceinline__ uint16_t to_bits<__nv_bfloat16>(float v) {
  __nv_bfloat16 h = __float2bfloat16_rn(v);
  uint16_t u;
  memcpy(&u, &h, 2);
  return u;
}
template <>
__device__ __forceinline__ uint16_t to_bits<__half>(float v) {
  __half h = __float2half_rn(v);
  uint16_t u;
  memcpy(&u, &h, 2);
  return u;
}
template <typename E>
constexpr uint32_t ab_format() {
  return std::is_same<E, __nv_bfloat16>::value ? 1u : 0u;
}

// Shared memory of stage 1 (byte offsets from a 1024-byte aligned base).  A
// staged chunk is K then V of head g, each [D/64 blocks][128 keys][128 B]
// (64 columns of a key per 128-byte row, 16-byte units XOR-swizzled by key).
struct AttnLayout {
  uint32_t stage_bytes, v_off, q_off, p_off, red_off, bar_off, total;
};

__host__ __device__ inline AttnLayout attn_layout(int D) {
  AttnLayout L;
  const uint32_t blk = kKeys * 128;                        // 64 columns of 128 keys: 16 KB
  L.v_off = static_cast<uint32_t>(D / 64) * blk;
  L.stage_bytes = 2 * L.v_off;
  L.q_off = kAttnStages * L.stage_bytes;                   // Q: [D/64][32 rows][128 B]
  L.p_off = L.q_off + static_cast<uint32_t>(D / 64) * kQRows * 128;   // P^T: 2 x [2][32 rows][128 B]
  L.red_off = L.p_off + 2 * 2 * kQRows * 128;
  L.bar_off = L.red_off + 4096;
  L.total = L.bar_off + 256 + 1024;                        // + alignment slack
  return L;
}

struct AttnBarriers {
  uint64_t full_k[kAttnStages];    // a chunk's K rows have landed
  uint64_t full_v[kAttnStages];    // its V rows have landed
  uint64_t empty_k[kAttnStages];   // its scores are computed: the K half is free
  uint64_t empty_v[kAttnStages];   // its O product is done: the V half is free
  uint64_t s_full[2];
  uint64_t s_free[2];
  uint64_t p_full[2];
  uint64_t pv_done[2];   // the O product of chunk c, per P buffer c & 1
  uint64_t q_full;
  uint64_t drain;
  uint64_t never;                   // diagnostics: a barrier nothing arrives on
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(AttnBarriers) <= 256, "barrier area");

// Shared-memory matrix descriptor of an MN-major operand in the 128-byte
// swizzle layout: 64 consecutive M elements per 128-byte row, 8 rows (K) per
// 1024-byte atom, atoms `lbo` bytes apart along M and 1024 bytes apart along
// K.  Descriptor version 1, layout type 2 (SWIZZLE_128B).
__device__ __forceinline__ uint64_t sw128_mnmajor_desc(uint32_t smem_addr, uint32_t lbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>(1024u >> 4) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}

// Transpose-reduction over a warp: on entry lane l holds v[j] = value of
// (key l, row j) for R rows; on exit the result of lane l is the reduction
// over the warp's 32 keys of row l % R.
template <bool kMax, int R>
__device__ __forceinline__ float warp_rows(float (&v)[R], int lane) {
#pragma unroll
  for (int off = R / 2; off >= 1; off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < off; ++i) {
      const float send = upper ? v[i] : v[i + off];
      const float keep = upper ? v[i + off] : v[i];
      const float other = __shfl_xor_sync(0xffffffffu, send, off);
      v[i] = kMax ? fmaxf(keep, other) : keep + other;
    }
  }
  float r = v[0];
#pragma unroll
  for (int off = R; off < 32; off <<= 1) {
    const float other = __shfl_xor_sync(0xffffffffu, r, off);
    r = kMax ? fmaxf(r, other) : r + other;
  }
  return r;
}

// 8 consecutive fp32 columns of this thread's TMEM lane (32x32b shape),
// loaded and waited for in one statement.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
      : "r"(taddr));
}

// Four runs of 8 columns, one wait: all four loads in flight together.
#define DSPARK_O8(a, i) "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]), "=r"(a[7])
__device__ __forceinline__ void tmem_ld8x4(uint32_t t0, uint32_t t1, uint32_t t2, uint32_t t3, uint32_t (&a)[8],
                                           uint32_t (&b)[8], uint32_t (&c)[8], uint32_t (&d)[8]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%32];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%8,%9,%10,%11,%12,%13,%14,%15}, [%33];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%16,%17,%18,%19,%20,%21,%22,%23}, [%34];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%24,%25,%26,%27,%28,%29,%30,%31}, [%35];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : DSPARK_O8(a, 0), DSPARK_O8(b, 0), DSPARK_O8(c, 0), DSPARK_O8(d, 0)
      : "r"(t0), "r"(t1), "r"(t2), "r"(t3));
}
#undef DSPARK_O8

// Store 8 consecutive fp32 columns of this thread's TMEM lane and wait.
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]));
}

// 2^x (PTX ex2.approx.ftz: relative error about 2^-22; 2^-inf = 0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Named barrier over `count` threads that returns how many of them passed a
// true predicate.
__device__ __forceinline__ uint32_t named_barrier_popc(uint32_t id, uint32_t count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "barrier.cta.red.popc.u32 %0, %2, %3, q;\n\t}"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "r"(id), "r"(count)
      : "memory");
  return r;
}

// The mbarrier's pending count drops by one when every asynchronous copy
// this thread issued before has landed (the init count includes it).
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// 16-byte-aligned zeros: the source of the rows of keys without a valid slot.
__device__ __align__(16) uint8_t g_attn_zero_row[256];

// Wait until the phase with the given parity has completed; a waiting thread
// sleeps in the barrier (up to kSuspendNs per try) instead of spinning, so the
// roles that have work keep the issue slots.  Gives up (false) when *abort
// becomes non-zero or after limit_ns.
constexpr uint32_t kSuspendNs = 20000;
__device__ __forceinline__ bool attn_wait(uint32_t bar, uint32_t parity, volatile int* abort, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(kSuspendNs)
        : "memory");
    if (ok) return true;
    if (*abort) return false;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}

__device__ __forceinline__ void attn_flag(const AttnParams& p, uint32_t bits) {
  if (p.status != nullptr) atomicOr(p.status, bits);
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

template <typename E, int D>
__global__ void __launch_bounds__(kAttnThreads, 1) attn_tc_kernel(const AttnParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const AttnLayout L = attn_layout(D);
  AttnBarriers* bars = reinterpret_cast<AttnBarriers*>(smem + L.bar_off);
  constexpr int kWgs = kSoftWarps / 4;
  float* alpha_s = reinterpret_cast<float*>(smem + L.red_off);   // [2 parity][kWgs][4 groups][kWgRows]
  int* resc_s = reinterpret_cast<int*>(alpha_s + 2 * kWgs * 4 * kWgRows);   // [2 parity][kWgs][4 groups]
  float* ml_s = reinterpret_cast<float*>(resc_s + 2 * kWgs * 4);    // [kWgs][4 groups][kWgRows][2]
  volatile int* abort_flag = &bars->abort;
  constexpr int kBlocksD = D / 64;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // the merge kernel (a programmatic dependent launch) may be scheduled once
  // every CTA of this grid has started; it waits for this grid's completion
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // the KV heads of one (request, split) are adjacent CTAs
  const int64_t b = blockIdx.z;
  const int g = blockIdx.x;
  const int s = blockIdx.y;
  const int64_t k0 = p.kv_start[b];
  int64_t n_b = p.kv_start[b + 1] - k0;
  if (n_b > p.max_context) {
    if (s == 0 && g == 0 && threadIdx.x == 0) attn_flag(p, DSPARK_FLAG_CONTEXT_RANGE);
    n_b = p.max_context;
  }
  if (n_b < 0) n_b = 0;
  if (p.pool_slots <= 0 && n_b > 0) {   // an empty pool: every context key is out of range
    if (s == 0 && g == 0 && threadIdx.x == 0) attn_flag(p, DSPARK_FLAG_LOC_RANGE);
    n_b = 0;
  }
  const int64_t lo = static_cast<int64_t>(s) * p.split_tokens;
  const int64_t hi = lo + p.split_tokens < n_b ? lo + p.split_tokens : n_b;
  const int n_ctx = hi > lo ? static_cast<int>(hi - lo) : 0;
  const bool has_ext = s == 0;
  if (!has_ext && n_ctx == 0) return;            // nothing in this split (uniform)
  const int ctx_chunks = (n_ctx + kKeys - 1) / kKeys;
  const int n_chunks = ctx_chunks + (has_ext ? 1 : 0);
  const int nwg = p.rows / kWgRows;              // softmax warpgroups with rows (2 or 4)

  // The first slot-index loads and the Q copies are issued before the set-up
  // barrier (Q's arrival on q_full follows it), so that their latency overlaps
  // the barrier initialisation and the TMEM allocation.
  const bool is_prod = warp >= kProdWarp0 && warp < kProdWarp0 + kProdWarps;
  const int pw = warp - kProdWarp0;               // producer warp (producers only)
  // producers: slot of key kKeysPerProdWarp*pw + lane of chunk c (checked
  // where used), kNoKey past the context, or the row of the block's own key
  auto lane_slot = [&](int c) -> int64_t {
    const int key = kKeysPerProdWarp * pw + lane;
    if (c >= n_chunks || lane >= kKeysPerProdWarp) return kNoKey;
    if (c < ctx_chunks) {
      const int64_t t = lo + static_cast<int64_t>(c) * kKeys + key;
      return t < hi ? p.kv_indices[k0 + t] : kNoKey;
    }
    return key < p.block ? b * p.block + key : kNoKey;
  };
  // softmax: slot of this thread's key (warp % 4 * 32 + lane) in context chunk c
  auto key_slot = [&](int c) -> int64_t {
    if (c >= ctx_chunks) return 0;
    const int64_t t = lo + static_cast<int64_t>(c) * kKeys + (warp % 4) * 32 + lane;
    return t < hi ? p.kv_indices[k0 + t] : -1;
  };
  int64_t pre0 = 0, pre1 = 0;
  if (is_prod) {
    const int pt = threadIdx.x - kProdWarp0 * 32;
    const E* q = static_cast<const E*>(p.q);
    // Q of head g: row r = i*group + hh, its D columns as D/64 128-byte rows
    for (int x = pt; x < p.rows * (D / 8); x += kProdThreads) {
      const int r = x / (D / 8), u = x % (D / 8);
      const E* src = q + ((b * p.block + r / p.group) * p.nq + g * p.group + r % p.group) * D + u * 8;
      const uint32_t dst = smem_u32(smem + L.q_off) + (u / 8) * (kQRows * 128) + r * 128 + (((u % 8) ^ (r & 7)) * 16);
      cp_async16(dst, src);
    }
    pre0 = lane_slot(0);
    pre1 = lane_slot(1);
  } else if (warp < kSoftWarps && warp / 4 < nwg) {
    pre0 = key_slot(0);
    pre1 = key_slot(1);
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < kAttnStages; ++i) {
      mbar_init(smem_u32(&bars->full_k[i]), kProdThreads);
      mbar_init(smem_u32(&bars->full_v[i]), kProdThreads);
      mbar_init(smem_u32(&bars->empty_k[i]), 1);
      mbar_init(smem_u32(&bars->empty_v[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bars->s_full[i]), 1);
      mbar_init(smem_u32(&bars->s_free[i]), 4 * nwg);
      mbar_init(smem_u32(&bars->p_full[i]), 4 * nwg);
      mbar_init(smem_u32(&bars->pv_done[i]), 1);
    }
    mbar_init(smem_u32(&bars->q_full), kProdThreads);
    mbar_init(smem_u32(&bars->drain), 1);
    mbar_init(smem_u32(&bars->never), 1);
    bars->abort = 0;
    fence_barrier_init();
  }
  if (warp == kAttnMmaWarp) {
    tmem_alloc(smem_u32(&bars->tmem_base), kAttnTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = bars->tmem_base;

  if (is_prod) {
    // ------------------------------------------------------------ producers
    // Every copy is a 16-byte asynchronous copy; the mbarrier of a half stage
    // (K or V rows of a chunk) completes when all 128 producer threads' copies
    // issued before their arrival on it have landed, so nothing here waits
    // for its own copies and up to three chunks are in flight.
    const int pt = threadIdx.x - kProdWarp0 * 32;   // 0..127 among the producers
    cp_async_arrive_noinc(smem_u32(&bars->q_full));   // the Q copies issued above
    // Warp pw copies kKeysPerProdWarp keys of a chunk; lane l learns the
    // slot of its key l two chunks ahead (the index load's latency under
    // the gather's DRAM load exceeds a chunk).  A warp instruction covers whole
    // K (or V) rows of 32 / (D/8) consecutive keys.  A key without a valid
    // slot gets zero rows (its weight is 0, and 0 x NaN would not be).
    constexpr int kUnits = D / 8;                 // 16-byte units of one head row
    constexpr int kPerIter = 32 / kUnits;         // keys per warp instruction
    constexpr int kXs = 8 / kPerIter;             // distinct swizzle rows of a lane's copies
    const int sub = lane / kUnits, u = lane % kUnits;
    int64_t slot_cur = pre0, slot_nxt = pre1;
    bool ok_run = true;
    for (int c = 0; c < n_chunks && ok_run; ++c) {
      const int st = c % kAttnStages;
      const bool own = c >= ctx_chunks;
      int64_t my_off = -1;
      if (slot_cur != kNoKey) {
        if (own)
          my_off = (slot_cur * p.nkv + g) * D;
        else if (slot_cur >= 0 && slot_cur < p.pool_slots)
          my_off = slot_cur * p.pool_row_stride + g * D;
        else
          attn_flag(p, DSPARK_FLAG_LOC_RANGE);
      }
      slot_cur = slot_nxt;
      slot_nxt = lane_slot(c + 2);
      // the owner lane of each key resolves its K and V row pointers (the
      // zero row for a key without a valid slot): a copy is then a shuffle, an
      // add and the copy itself
      uintptr_t my_k = reinterpret_cast<uintptr_t>(g_attn_zero_row), my_v = my_k;
      if (my_off >= 0) {
        my_k = reinterpret_cast<uintptr_t>(static_cast<const E*>(own ? p.k_ext : p.k_pool) + my_off);
        my_v = reinterpret_cast<uintptr_t>(static_cast<const E*>(own ? p.v_ext : p.v_pool) + my_off);
      }
      uint8_t* kst = smem + st * L.stage_bytes;
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        uint64_t* empty = half == 0 ? &bars->empty_k[st] : &bars->empty_v[st];
        // warp-uniform outcome: the copy loop below shuffles across the warp
        if (c >= kAttnStages &&
            !__all_sync(0xffffffffu, attn_wait(smem_u32(empty), static_cast<uint32_t>(c / kAttnStages - 1) & 1u,
                                               abort_flag, kAttnWaitNs))) {
          ok_run = false;
          break;
        }
        const unsigned long long mine = half == 0 ? my_k : my_v;
        // this lane's destinations: key kl = jj + sub of the warp's share, its
        // 16-byte unit u at (kl & 7) ^ u in the row; (kl & 7) takes kXs values
        const uint32_t lane_base = smem_u32(kst) + (half == 0 ? 0u : L.v_off) + (u / 8) * (kKeys * 128) +
                                   (kKeysPerProdWarp * pw + sub) * 128;
        uint32_t dst[kXs];
#pragma unroll
        for (int q = 0; q < kXs; ++q) dst[q] = lane_base + (((u % 8) ^ ((q * kPerIter + sub) & 7)) * 16);
#pragma unroll
        for (int jj = 0; jj < kKeysPerProdWarp; jj += kPerIter) {
          const unsigned long long src = __shfl_sync(0xffffffffu, mine, jj + sub) + static_cast<unsigned>(u * 16);
          cp_async16(dst[(jj / kPerIter) % kXs] + jj * 128, reinterpret_cast<const void*>(src));
        }
        cp_async_arrive_noinc(smem_u32(half == 0 ? &bars->full_k[st] : &bars->full_v[st]));
      }
    }
    cp_async_wait_all();   // no copy outlives the CTA
    if (!ok_run && pt == 0) {
      *abort_flag = 1;
      attn_flag(p, DSPARK_FLAG_TIMEOUT);
    }
  } else if (warp == kAttnMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // Issues whichever product is ready: the scores of the next chunk (landed,
    // its S buffer read by the softmax two chunks back) or the O product of the
    // oldest chunk whose P^T is written.  The four key groups of a chunk (32
    // keys, one softmax warp each) accumulate into their own O^T.
    if (lane == 0) {
      const uint32_t idesc_s = f16_instr_desc(ab_format<E>(), kKeys, p.rows);
      const uint32_t idesc_pv = f16_instr_desc(ab_format<E>(), kKeys, p.rows) | (1u << 15);   // A MN-major
      const uint32_t q_addr = smem_u32(smem + L.q_off);
      const uint32_t p_addr = smem_u32(smem + L.p_off);
      bool ok = attn_wait(smem_u32(&bars->q_full), 0, abort_flag, kAttnWaitNs);
      // diagnostics (dspark_draft_attention_set_wait_test): a wait that runs
      // out, so that every role takes its timeout path
      if (ok && p.test_wait_ns != 0) ok = attn_wait(smem_u32(&bars->never), 0, abort_flag, p.test_wait_ns);
      fence_proxy_async_smem();   // the copies landed through the generic proxy; the MMAs read via the async one
      bool issued = false;
      int next_s = 0, next_pv = 0;
      uint64_t t0 = global_timer_ns();
      for (uint32_t it = 1; ok && next_pv < n_chunks; ++it) {
        bool progress = false;
        if (next_s < n_chunks) {
          const int c = next_s, st = c % kAttnStages;
          if (mbar_try_wait(smem_u32(&bars->full_k[st]), static_cast<uint32_t>(c / kAttnStages) & 1u) &&
              (c < 2 || mbar_try_wait(smem_u32(&bars->s_free[c & 1]), static_cast<uint32_t>((c >> 1) - 1) & 1u))) {
            fence_proxy_async_smem();
            tc_fence_after();
            const uint32_t k_addr = smem_u32(smem + st * L.stage_bytes);
            const uint32_t t_s = tmem_base + (c & 1) * kQRows;
#pragma unroll
            for (int blk = 0; blk < kBlocksD; ++blk)
#pragma unroll
              for (int k = 0; k < 4; ++k)
                umma_f16(t_s, sw128_kmajor_desc(k_addr + blk * (kKeys * 128) + k * 32),
                         sw128_kmajor_desc(q_addr + blk * (kQRows * 128) + k * 32), idesc_s,
                         (blk != 0 || k != 0) ? 1u : 0u);
            umma_commit(smem_u32(&bars->s_full[c & 1]));
            umma_commit(smem_u32(&bars->empty_k[st]));
            issued = true;
            ++next_s;
            progress = true;
          }
        }
        if (next_pv < next_s) {
          const int j = next_pv;
          if (mbar_try_wait(smem_u32(&bars->p_full[j & 1]), static_cast<uint32_t>(j >> 1) & 1u) &&
              mbar_try_wait(smem_u32(&bars->full_v[j % kAttnStages]), static_cast<uint32_t>(j / kAttnStages) & 1u)) {
            fence_proxy_async_smem();
            tc_fence_after();
            const uint32_t v_addr = smem_u32(smem + (j % kAttnStages) * L.stage_bytes + L.v_off);
            const uint32_t pb = p_addr + (j & 1) * (2 * kQRows * 128);
#pragma unroll
            for (int kk = 0; kk < kKeys / 16; ++kk) {
              // 16 keys: two 8-key groups of the V block (1024 bytes each); P^T
              // rows hold 64 keys per 128-byte block; key group kk / 2
              const uint64_t ad = sw128_mnmajor_desc(v_addr + kk * 2048, D == 128 ? kKeys * 128 : 0);
              const uint64_t bd = sw128_kmajor_desc(pb + (kk / 4) * (kQRows * 128) + (kk % 4) * 32);
              umma_f16(tmem_base + 2 * kQRows + (kk / 2) * kQRows, ad, bd, idesc_pv,
                       (j > 0 || (kk & 1) != 0) ? 1u : 0u);
            }
            umma_commit(smem_u32(&bars->empty_v[j % kAttnStages]));
            umma_commit(smem_u32(&bars->pv_done[j & 1]));
            issued = true;
            ++next_pv;
            progress = true;
          }
        }
        if (progress) {
          t0 = global_timer_ns();
        } else if ((it & 63u) == 0u && (*abort_flag || global_timer_ns() - t0 > kAttnWaitNs)) {
          ok = false;
        }
      }
      if (!ok) {
        *abort_flag = 1;
        attn_flag(p, DSPARK_FLAG_TIMEOUT);
      }
      if (issued) {
        umma_commit(smem_u32(&bars->drain));
        int never = 0;
        attn_wait(smem_u32(&bars->drain), 0, &never, kAttnWaitNs);
      }
    }
  } else if (warp < kSoftWarps && warp / 4 < nwg) {
    // ------------------------------------------------------------ softmax
    // Warpgroup wg owns query rows wg*R .. wg*R+R-1 (R = kWgRows); warp wq of
    // it owns keys 32*wq .. 32*wq+31 of every chunk (TMEM lanes), one per
    // thread, and keeps its own running maximum and sum per row (lane l: row
    // wg*R + l % R) for its own O^T accumulator.  Per chunk the warps of a
    // warpgroup meet once, to learn whose O must be rescaled (and whether a
    // wait gave up: then all of them leave together).
    constexpr int R = kWgRows;
    const int wg = warp / 4, wq = warp % 4;
    const int k = wq * 32 + lane;
    const uint32_t bar_id = 1 + wg;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    float m_run = -INFINITY, l_run = 0.f;
    uint8_t* p_smem = smem + L.p_off;
    bool done_ok = true;
    int64_t slot_cur = pre0, slot_nxt = pre1;   // loaded two chunks early
    // byte offset in a P buffer of P^T[row wg*R + r][key k]: row Rw of block
    // k/64, 16-byte unit (k%64)/8 XOR-swizzled by the row
    uint32_t p_row[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int Rw = wg * R + r;
      p_row[r] = static_cast<uint32_t>((k / 64) * (kQRows * 128) + (k % 8) * 2 + Rw * 128 +
                                       ((((k % 64) / 8) ^ (Rw & 7)) * 16));
    }
    for (int c = 0; c < n_chunks; ++c) {
      const int par = c & 1;
      bool valid;
      if (c < ctx_chunks)
        valid = slot_cur >= 0 && slot_cur < p.pool_slots;
      else
        valid = k < p.block;
      slot_cur = slot_nxt;
      slot_nxt = key_slot(c + 2);
      bool ok = __all_sync(0xffffffffu, attn_wait(smem_u32(&bars->s_full[par]), static_cast<uint32_t>(c >> 1) & 1u,
                                                  abort_flag, kAttnWaitNs));
      bool grow = false;
      if (ok) {
        tc_fence_after();
        uint32_t sraw[R];
        tmem_ld8(tmem_base + lane_off + par * kQRows + wg * R, sraw);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars->s_free[par]));
        float x[R];
#pragma unroll
        for (int r = 0; r < R; ++r) x[r] = valid ? __uint_as_float(sraw[r]) : -INFINITY;   // raw scores
        float cm;
        {
          float t[R];
#pragma unroll
          for (int r = 0; r < R; ++r) t[r] = x[r];
          // this warp's maximum of row lane % R, in the scaled log2 domain
          cm = warp_rows<true, R>(t, lane) * p.scale_log2;
        }
        float al = 1.f;
        if (cm > m_run + kLazyRescale) {      // also the first finite maximum (m_run = -inf)
          al = m_run == -INFINITY ? 1.f : fast_exp2(m_run - cm);
          m_run = cm;
        }
        grow = __any_sync(0xffffffffu, al != 1.f);
        float pr[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const float mr = __shfl_sync(0xffffffffu, m_run, r);
          // a masked key (x = -inf) gives 2^-inf = 0; a row without a valid key
          // so far in this warp (mr = -inf) has only masked keys
          pr[r] = mr == -INFINITY ? 0.f : fast_exp2(fmaf(x[r], p.scale_log2, -mr));
        }
        // P buffer par was read by the product of chunk c - 2
        ok = c < 2 || __all_sync(0xffffffffu, attn_wait(smem_u32(&bars->pv_done[par]),
                                                        static_cast<uint32_t>((c >> 1) - 1) & 1u, abort_flag,
                                                        kAttnWaitNs));
        if (ok) {
          // P^T[row][key] in the model dtype (the row offsets of this thread's
          // key are fixed: p_row[r] below)
          uint8_t* pb = p_smem + par * (2 * kQRows * 128);
#pragma unroll
          for (int r = 0; r < R; ++r) *reinterpret_cast<uint16_t*>(pb + p_row[r]) = to_bits<E>(pr[r]);
        }
        const float sum = warp_rows<false, R>(pr, lane);
        l_run = l_run * al + sum;
        // a warp whose maximum grew publishes its factors; its accumulator may
        // be rescaled once the previous chunk's product is complete
        if (lane < R) alpha_s[((par * kWgs + wg) * 4 + wq) * R + lane] = al;
        if (ok && grow && c >= 1)
          ok = __all_sync(0xffffffffu, attn_wait(smem_u32(&bars->pv_done[(c - 1) & 1]),
                                                 static_cast<uint32_t>((c - 1) >> 1) & 1u, abort_flag, kAttnWaitNs));
      }
      if (lane == 0) {
        resc_s[(par * kWgs + wg) * 4 + wq] = (ok && grow) ? 1 : 0;
        if (!ok) *abort_flag = 1;   // the MMA issuer and the producers stop too
      }
      if (named_barrier_popc(bar_id, 128, !ok) != 0) {
        done_ok = false;
        break;
      }
      if (c >= 1) {
        // every warp rescales the grown accumulators over its own TMEM lanes
        const int* rs = resc_s + (par * kWgs + wg) * 4;
        if ((rs[0] | rs[1] | rs[2] | rs[3]) != 0) {
          tc_fence_after();
#pragma unroll 1
          for (int w = 0; w < 4; ++w) {
            if (rs[w] == 0) continue;
            const uint32_t t_ow = tmem_base + lane_off + 2 * kQRows + w * kQRows + wg * R;
            uint32_t o[R];
            tmem_ld8(t_ow, o);
#pragma unroll
            for (int r = 0; r < R; ++r)
              o[r] = __float_as_uint(__uint_as_float(o[r]) * alpha_s[((par * kWgs + wg) * 4 + w) * R + r]);
            tmem_st8(t_ow, o);
          }
        }
      }
      fence_proxy_async_smem();   // P^T (generic stores) before the tensor cores read it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars->p_full[par]));
    }
    // ---- merge the four key groups' partial results of each row: this
    // split's unnormalised O^T, maximum and sum of the warpgroup's rows
    if (done_ok && n_chunks > 0)
      done_ok = __all_sync(0xffffffffu, attn_wait(smem_u32(&bars->pv_done[(n_chunks - 1) & 1]),
                                                  static_cast<uint32_t>((n_chunks - 1) >> 1) & 1u, abort_flag,
                                                  kAttnWaitNs));
    if (lane < R) {
      ml_s[((wg * 4 + wq) * R + lane) * 2] = m_run;
      ml_s[((wg * 4 + wq) * R + lane) * 2 + 1] = l_run;
    }
    done_ok = named_barrier_and(bar_id, 128, done_ok);
    if (done_ok) {
      tc_fence_after();
      uint32_t o[4][R];
      const uint32_t t_o = tmem_base + lane_off + 2 * kQRows + wg * R;
      tmem_ld8x4(t_o, t_o + kQRows, t_o + 2 * kQRows, t_o + 3 * kQRows, o[0], o[1], o[2], o[3]);
      float acc[R];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        float mw[4];
#pragma unroll
        for (int w = 0; w < 4; ++w) mw[w] = ml_s[((wg * 4 + w) * R + r) * 2];
        const float m = fmaxf(fmaxf(mw[0], mw[1]), fmaxf(mw[2], mw[3]));
        float a = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w)
          if (mw[w] != -INFINITY) a += fast_exp2(mw[w] - m) * __uint_as_float(o[w][r]);
        acc[r] = a;
      }
      const int nrows = p.nkv * p.rows;
      const int64_t row0 = (b * p.splits + s) * static_cast<int64_t>(nrows) + static_cast<int64_t>(g) * p.rows +
                           wg * R;
      if (k < D) {
#pragma unroll
        for (int r = 0; r < R; ++r) p.ws_o[(row0 + r) * D + k] = acc[r];
      }
      if (wq == 0 && lane < R) {
        float mw[4];
#pragma unroll
        for (int w = 0; w < 4; ++w) mw[w] = ml_s[((wg * 4 + w) * R + lane) * 2];
        const float m = fmaxf(fmaxf(mw[0], mw[1]), fmaxf(mw[2], mw[3]));
        float lsum = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w)
          if (mw[w] != -INFINITY) lsum += fast_exp2(mw[w] - m) * ml_s[((wg * 4 + w) * R + lane) * 2 + 1];
        *reinterpret_cast<float2*>(p.ws_ml + (row0 + lane) * 2) = make_float2(m, lsum);
      }
    } else if (k == 0) {
      *abort_flag = 1;
      attn_flag(p, DSPARK_FLAG_TIMEOUT);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kAttnMmaWarp) tmem_dealloc(tmem_base, kAttnTmemCols);
}

// Stage 2: one warp per (request, query row of a KV head): merge the splits.
// Lane j holds split 32i + j's maximum and sum; each lane owns D/32
// consecutive columns of the row.  The first kAhead splits' partial O and the
// lanes' maxima and sums are loaded before the request's split count is known
// (the workspace holds p.splits splits, written or not; the unwritten ones are
// never used), so that a two-split row costs one round trip to memory.
template <typename E, int D>
__global__ void __launch_bounds__(kCombineWarps * 32) attn_combine_kernel(const AttnParams p) {
  constexpr int kPer = D / 32;   // 4 (D = 128) or 2 (D = 64) consecutive columns per lane
  constexpr int kAhead = 4;      // splits of partial O in flight at once
  using Vec = typename std::conditional<kPer == 4, float4, float2>::type;
  const int nrows = p.nkv * p.rows;
  const int64_t wid = static_cast<int64_t>(blockIdx.x) * kCombineWarps + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (wid >= p.batch * nrows) return;
  const int64_t b = wid / nrows;
  const int row = static_cast<int>(wid % nrows);
  const int64_t r0 = b * p.splits * static_cast<int64_t>(nrows) + row;
  const float2* ml_row = reinterpret_cast<const float2*>(p.ws_ml) + r0;
  const float* src = p.ws_o + r0 * D + lane * kPer;
  const int64_t s_stride = static_cast<int64_t>(nrows) * D;
  const int64_t kv0 = p.kv_start[b], kv1 = p.kv_start[b + 1];
  // the split kernel's workspace writes are complete and visible past here
  asm volatile("griddepcontrol.wait;" ::: "memory");
  Vec v[kAhead];
#pragma unroll
  for (int j = 0; j < kAhead; ++j)
    if (j < p.splits) v[j] = *reinterpret_cast<const Vec*>(src + j * s_stride);
  float2 ml = make_float2(-INFINITY, 0.f);
  if (lane < p.splits) ml = ml_row[static_cast<int64_t>(lane) * nrows];
  int64_t n_b = kv1 - kv0;
  if (n_b > p.max_context) n_b = p.max_context;
  if (n_b < 0 || p.pool_slots <= 0) n_b = 0;
  int n_split = static_cast<int>((n_b + p.split_tokens - 1) / p.split_tokens);
  if (n_split < 1) n_split = 1;
  if (lane >= n_split) ml = make_float2(-INFINITY, 0.f);
  float M = ml.x;
  for (int s = lane + 32; s < n_split; s += 32) M = fmaxf(M, ml_row[static_cast<int64_t>(s) * nrows].x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float o_acc[kPer] = {};
  float Lsum = 0.f;
  for (int s0 = 0; s0 < n_split; s0 += 32) {
    const int cnt = n_split - s0 < 32 ? n_split - s0 : 32;
    if (s0 > 0) ml = lane < cnt ? ml_row[static_cast<int64_t>(s0 + lane) * nrows] : make_float2(-INFINITY, 0.f);
    const float w = ml.x == -INFINITY ? 0.f : exp2f(ml.x - M);
    Lsum += w * ml.y;
    for (int j0 = 0; j0 < cnt; j0 += kAhead) {
      if (s0 > 0 || j0 > 0) {
#pragma unroll
        for (int j = 0; j < kAhead; ++j)
          if (j0 + j < cnt) v[j] = *reinterpret_cast<const Vec*>(src + (s0 + j0 + j) * s_stride);
      }
#pragma unroll
      for (int j = 0; j < kAhead; ++j) {
        const float wj = __shfl_sync(0xffffffffu, w, (j0 + j) & 31);
        if (j0 + j < cnt) {
          const float* x = reinterpret_cast<const float*>(&v[j]);
#pragma unroll
          for (int k = 0; k < kPer; ++k) o_acc[k] += wj * x[k];
        }
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) Lsum += __shfl_xor_sync(0xffffffffu, Lsum, o);
  const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
  const int g = row / p.rows, rr = row % p.rows;
  const int i = rr / p.group, hh = rr % p.group;
  uint16_t* dst = static_cast<uint16_t*>(p.out) + ((b * p.block + i) * p.nq + g * p.group + hh) * D + lane * kPer;
  uint32_t packed[kPer / 2];
#pragma unroll
  for (int k = 0; k < kPer / 2; ++k)
    packed[k] = static_cast<uint32_t>(to_bits<E>(o_acc[2 * k] * inv)) |
                (static_cast<uint32_t>(to_bits<E>(o_acc[2 * k + 1] * inv)) << 16);
  if constexpr (kPer == 4)
    *reinterpret_cast<uint2*>(dst) = make_uint2(packed[0], packed[1]);
  else
    *reinterpret_cast<uint32_t*>(dst) = packed[0];
}

template <typename E, int D>
cudaError_t launch_attention(const AttnParams& p, cudaStream_t stream) {
  const AttnLayout L = attn_layout(D);
  auto k1 = attn_tc_kernel<E, D>;
  cudaError_t e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(L.total));
  if (e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>(p.nkv), static_cast<unsigned>(p.splits), static_cast<unsigned>(p.batch));
  k1<<<grid, kAttnThreads, L.total, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // the merge is a programmatic dependent launch: its CTAs may take the SMs
  // that the split kernel's last CTAs leave idle, and wait there for it
  const int64_t rows = p.batch * p.nkv * p.rows;
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(static_cast<unsigned>((rows + kCombineWarps - 1) / kCombineWarps));
  cfg.blockDim = dim3(kCombineWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attn_combine_kernel<E, D>, p);
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

std::atomic<uint64_t> g_attn_test_wait_ns{0};   // dspark_draft_attention_set_wait_test

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
                AttnPlan* plan) {
  if (batch < 0 || block < 1 || nq < 1 || nkv < 1 || max_context < 0) return DSPARK_E_INVALID_ARG;
  if (D != 64 && D != 128) return DSPARK_E_HEAD_DIM;
  if (nq % nkv != 0) return DSPARK_E_SHAPE_MISMATCH;
  const int64_t rows = static_cast<int64_t>(block) * (nq / nkv);
  if (rows != 16 && rows != 32) return DSPARK_E_SHAPE_MISMATCH;
  if (block > kKeys) return DSPARK_E_SHAPE_MISMATCH;
  *plan = make_plan(batch > 0 ? batch : 1, nkv, max_context);
  if (attn_layout(D).total > 227u * 1024u) return DSPARK_E_SHAPE_MISMATCH;
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
  if (check_shape(batch, block, num_q_heads, num_kv_heads, head_dim, max_context, &pl) != DSPARK_OK) return 0;
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
  const int st = check_shape(batch, block, num_q_heads, num_kv_heads, head_dim, max_context, &pl);
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
  if (batch > 65535 || pl.splits > 65535) return DSPARK_E_INVALID_ARG;   // grid z and y
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
  p.max_context = max_context;
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
  p.test_wait_ns = g_attn_test_wait_ns.load();
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  cudaError_t e;
  if (dtype == DSPARK_DTYPE_BF16)
    e = head_dim == 128 ? launch_attention<__nv_bfloat16, 128>(p, stream)
                        : launch_attention<__nv_bfloat16, 64>(p, stream);
  else
    e = head_dim == 128 ? launch_attention<__half, 128>(p, stream) : launch_attention<__half, 64>(p, stream);
  return e == cudaSuccess ? DSPARK_OK : DSPARK_E_CUDA;
}

extern "C" int dspark_draft_attention_set_wait_test(uint64_t limit_ns) {
  dspark::g_attn_test_wait_ns.store(limit_ns);
  return DSPARK_OK;
}
