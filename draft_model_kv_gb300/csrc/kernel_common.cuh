// Device helpers shared by the fused context-KV kernels: 16-bit element
// access, the hybrid data-parallel / stream-K work walk and the partial-tile
// workspace layout.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstring>

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
  __device__ static __forceinline__ float to_float(__nv_bfloat16 v) { return __bfloat162float(v); }
  __device__ static __forceinline__ void unpack(uint32_t u, float& lo, float& hi) {
    __nv_bfloat162 h;
    memcpy(&h, &u, 4);
    lo = __low2float(h);
    hi = __high2float(h);
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
  __device__ static __forceinline__ float to_float(__half v) { return __half2float(v); }
  __device__ static __forceinline__ void unpack(uint32_t u, float& lo, float& hi) {
    __half2 h;
    memcpy(&h, &u, 4);
    lo = __low2float(h);
    hi = __high2float(h);
  }
};

__device__ __forceinline__ void flag(const WriteParams& p, uint32_t bits) {
  atomicOr(p.status, bits);
}

__device__ __forceinline__ float f32(uint32_t u) { return __uint_as_float(u); }

// 8 consecutive 16-bit values (one 16-byte load) widened to fp32.
template <typename E>
__device__ __forceinline__ void load8(const void* base, int64_t idx, float (&out)[8]) {
  const uint4 q = *reinterpret_cast<const uint4*>(reinterpret_cast<const E*>(base) + idx);
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint16_t lo = static_cast<uint16_t>(w[i] & 0xFFFFu), hi = static_cast<uint16_t>(w[i] >> 16);
    E a, b;
    memcpy(&a, &lo, 2);
    memcpy(&b, &hi, 2);
    out[2 * i] = ElemOps<E>::to_float(a);
    out[2 * i + 1] = ElemOps<E>::to_float(b);
  }
}

// 16-byte store of 8 packed 16-bit outputs.
__device__ __forceinline__ void st16(void* dst, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  *reinterpret_cast<uint4*>(dst) = make_uint4(a, b, c, d);
}

// Work of one worker (a CTA, or a CTA pair): its whole tiles (every nw-th
// from its index) and its contiguous range of the stream-K k-block space,
// walked from its end back to its start; whole tiles first unless the
// schedule is split-first.  In the other order the backward walk makes a
// worker begin with the (usually small) first k-blocks of the tile at the end
// of its range, publish that part while it computes the rest, and end with
// the (usually large) last part of the tile at the start of its range: it
// holds that tile's last k-block and finishes the tile from the partial tile
// it holds in TMEM plus the parts the others published.
struct WorkIter {
  int dp_tile, nw;
  int64_t start, cur;
};

__device__ __forceinline__ WorkIter work_begin(const WriteParams& p, int wid, int nw) {
  WorkIter it;
  it.dp_tile = wid;
  it.nw = nw;
  it.start = it.cur = 0;
  if (wid < p.sk_workers) {
    it.start = static_cast<int64_t>(wid) * p.sk_units / p.sk_workers;
    it.cur = static_cast<int64_t>(wid + 1) * p.sk_units / p.sk_workers;
  }
  return it;
}

__device__ __forceinline__ int dp_tile_at(const WriteParams& p, int i) {
  return i < p.dp_perm_n ? static_cast<int>(p.dp_perm[i]) : i;
}

__device__ __forceinline__ bool work_next(const WriteParams& p, WorkIter& it, int& tile, int& kb0,
                                          int& kb1) {
  if (!p.sk_first && it.dp_tile < p.dp_tiles) {
    tile = dp_tile_at(p, it.dp_tile);
    kb0 = 0;
    kb1 = p.num_kb;
    it.dp_tile += it.nw;
    return true;
  }
  if (it.cur > it.start) {
    const int64_t t = (it.cur - 1) / p.num_kb;
    const int64_t tile_start = t * p.num_kb;
    const int64_t lo = it.start > tile_start ? it.start : tile_start;
    kb0 = static_cast<int>(lo - tile_start);
    kb1 = static_cast<int>(it.cur - tile_start);
    it.cur = lo;
    tile = p.dp_tiles + static_cast<int>(t);
    return true;
  }
  if (p.sk_first && it.dp_tile < p.dp_tiles) {
    tile = dp_tile_at(p, it.dp_tile);
    kb0 = 0;
    kb1 = p.num_kb;
    it.dp_tile += it.nw;
    return true;
  }
  return false;
}

// Worker whose stream-K range holds k-block unit u.
__device__ __forceinline__ int sk_owner(const WriteParams& p, int64_t u) {
  return static_cast<int>(((u + 1) * p.sk_workers - 1) / p.sk_units);
}

// Bounded wait until *ctr >= target (acquire): the arrival count of a split
// tile's published parts.  False if this CTA aborted or the wait ran out.
__device__ __forceinline__ bool wait_count(const int32_t* ctr, int target, volatile int* abort_flag,
                                           uint64_t limit_ns) {
  const uint64_t t0 = global_timer_ns();
  while (ld_acquire_gpu(ctr) < target) {
    if (*abort_flag != 0 || global_timer_ns() - t0 > limit_ns) return false;
    __nanosleep(64);
  }
  return true;
}

// Partial-tile slot of a CTA: [kTileN/4][kTileM] float4, so that the 32 rows
// of a warp write one contiguous 512-byte run per 4 columns.
constexpr int kSlotFloats = kTileM * kTileN;

__device__ __forceinline__ float* ws_slot(const WriteParams& p, int cta, int slot) {
  return p.workspace + (static_cast<size_t>(cta) * 2 + slot) * kSlotFloats;
}

}  // namespace
}  // namespace dspark
