// In-place QK RMSNorm + table neox RoPE on a fused QKV tensor: the draft
// layers' own per-head normalisation and rotation (sglang PR #31847 summary
// page, "Key source snippets", dflash_utils.py: _table_qk_norm_rope_kernel).
//
// HBM-bound: every Q and K element is read once and written once.  Each
// thread owns 8 consecutive elements of each half of one head (two 16-byte
// loads and stores), i.e. both members of its 8 rotation pairs (element i
// and i + D/2), so a head of D = 128 is a group of 8 lanes (4 for D = 64) and
// the rotation needs no data from other lanes.  The sum of squares is
// reduced across the group with warp shuffles.  The cos/sin row of the token
// is read straight from the table (L1-cached: every head of a token shares it).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "../../include/dspark_qk_norm_rope.h"

namespace dspark {
namespace {

constexpr int kQkThreads = 256;

template <typename E>
struct QkElem;

template <>
struct QkElem<__nv_bfloat16> {
  __device__ static __forceinline__ float round_trip(float v) {
    return __bfloat162float(__float2bfloat16_rn(v));
  }
  __device__ static __forceinline__ uint32_t pack(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    uint32_t u;
    memcpy(&u, &h, 4);
    return u;
  }
  __device__ static __forceinline__ void unpack(uint32_t u, float& a, float& b) {
    __nv_bfloat162 h;
    memcpy(&h, &u, 4);
    a = __low2float(h);
    b = __high2float(h);
  }
};

template <>
struct QkElem<__half> {
  __device__ static __forceinline__ float round_trip(float v) { return __half2float(__float2half_rn(v)); }
  __device__ static __forceinline__ uint32_t pack(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    uint32_t u;
    memcpy(&u, &h, 4);
    return u;
  }
  __device__ static __forceinline__ void unpack(uint32_t u, float& a, float& b) {
    __half2 h;
    memcpy(&h, &u, 4);
    a = __low2float(h);
    b = __high2float(h);
  }
};

// At most 64 registers a thread, so that four blocks (32 warps) fit on an SM:
// the loads in flight per SM are what the HBM stream needs (measured: 79% of
// the copy bandwidth at 4 blocks against 68% at 3).
template <typename E, int D>
__global__ void __launch_bounds__(kQkThreads, 4)
    qk_norm_rope_kernel(E* __restrict__ qkv, int64_t T, int64_t row_stride, const int64_t* __restrict__ positions,
                        const E* __restrict__ q_weight, const E* __restrict__ k_weight,
                        const float* __restrict__ cos_sin, int64_t max_pos, int nq, int nh, float eps,
                        uint32_t* status) {
  constexpr int kHalf = D / 2;
  constexpr int kLanes = kHalf / 8;           // lanes of one head: each owns 8 + 8 elements
  constexpr int kHeadsPerBlock = kQkThreads / kLanes;
  const int j = threadIdx.x % kLanes;
  const int i0 = j * 8;                       // rotation index of this lane's first element
  const int64_t total = T * nh;
  // every warp runs the same number of iterations: the shuffles below always
  // involve all 32 lanes
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * kHeadsPerBlock; base < total;
       base += static_cast<int64_t>(gridDim.x) * kHeadsPerBlock) {
    const int64_t u = base + threadIdx.x / kLanes;
    const bool valid = u < total;
    const int64_t t = valid ? u / nh : 0;
    const int h = valid ? static_cast<int>(u - t * nh) : 0;
    int64_t pos = valid ? positions[t] : 0;
    const bool in_range = pos >= 0 && pos < max_pos;
    if (!in_range) pos = 0;
    E* head = qkv + t * row_stride + static_cast<int64_t>(h) * D;
    const E* w = h < nq ? q_weight : k_weight;
    const float* cs = cos_sin + pos * D;

    uint4 xa = make_uint4(0u, 0u, 0u, 0u), xb = xa, wa = xa, wb = xa;
    float4 c0 = make_float4(0.f, 0.f, 0.f, 0.f), c1 = c0, s0 = c0, s1 = c0;
    if (valid) {
      xa = *reinterpret_cast<const uint4*>(head + i0);
      xb = *reinterpret_cast<const uint4*>(head + kHalf + i0);
      wa = *reinterpret_cast<const uint4*>(w + i0);
      wb = *reinterpret_cast<const uint4*>(w + kHalf + i0);
      c0 = *reinterpret_cast<const float4*>(cs + i0);
      c1 = *reinterpret_cast<const float4*>(cs + i0 + 4);
      s0 = *reinterpret_cast<const float4*>(cs + kHalf + i0);
      s1 = *reinterpret_cast<const float4*>(cs + kHalf + i0 + 4);
    }
    float x1[8], x2[8], w1[8], w2[8];
    {
      const uint32_t q1[4] = {xa.x, xa.y, xa.z, xa.w}, q2[4] = {xb.x, xb.y, xb.z, xb.w};
      const uint32_t r1[4] = {wa.x, wa.y, wa.z, wa.w}, r2[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        QkElem<E>::unpack(q1[k], x1[2 * k], x1[2 * k + 1]);
        QkElem<E>::unpack(q2[k], x2[2 * k], x2[2 * k + 1]);
        QkElem<E>::unpack(r1[k], w1[2 * k], w1[2 * k + 1]);
        QkElem<E>::unpack(r2[k], w2[2 * k], w2[2 * k + 1]);
      }
    }
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) ss = fmaf(x2[k], x2[k], fmaf(x1[k], x1[k], ss));
#pragma unroll
    for (int off = kLanes / 2; off >= 1; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    const float inv = 1.0f / sqrtf(ss * (1.0f / D) + eps);
    const float c[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    const float s[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
    float o1[8], o2[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      // normalised values, rounded to the model dtype as the page does before
      // the rotation
      const float a = QkElem<E>::round_trip(x1[k] * inv * w1[k]);
      const float b = QkElem<E>::round_trip(x2[k] * inv * w2[k]);
      o1[k] = a * c[k] - b * s[k];
      o2[k] = b * c[k] + a * s[k];
    }
    if (valid && in_range) {
      *reinterpret_cast<uint4*>(head + i0) = make_uint4(QkElem<E>::pack(o1[0], o1[1]), QkElem<E>::pack(o1[2], o1[3]),
                                                        QkElem<E>::pack(o1[4], o1[5]), QkElem<E>::pack(o1[6], o1[7]));
      *reinterpret_cast<uint4*>(head + kHalf + i0) =
          make_uint4(QkElem<E>::pack(o2[0], o2[1]), QkElem<E>::pack(o2[2], o2[3]), QkElem<E>::pack(o2[4], o2[5]),
                     QkElem<E>::pack(o2[6], o2[7]));
    } else if (valid && status != nullptr && j == 0) {
      atomicOr(status, DSPARK_FLAG_POS_RANGE);
    }
  }
}

template <typename E, int D>
cudaError_t launch(void* qkv, int64_t T, int64_t row_stride, const int64_t* positions, const void* qw,
                   const void* kw, const float* cos_sin, int64_t max_pos, int nq, int nh, float eps,
                   uint32_t* status, int sms, cudaStream_t stream) {
  constexpr int kHeadsPerBlock = kQkThreads / (D / 16);
  const int64_t heads = T * nh;
  int64_t grid = (heads + kHeadsPerBlock - 1) / kHeadsPerBlock;
  const int64_t cap = static_cast<int64_t>(sms) * 16;   // grid-stride beyond 16 blocks per SM
  if (grid > cap) grid = cap;
  qk_norm_rope_kernel<E, D><<<static_cast<unsigned>(grid), kQkThreads, 0, stream>>>(
      static_cast<E*>(qkv), T, row_stride, positions, static_cast<const E*>(qw), static_cast<const E*>(kw),
      cos_sin, max_pos, nq, nh, eps, status);
  return cudaGetLastError();
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// SM count of the current device if it is an sm_103 part, else 0 (cached).
int sm103_sms(int device) {
  static int cache[64] = {0};
  const int d = device & 63;
  if (cache[d] == 0) {
    int major = 0, minor = 0, n = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
      return 0;
    cache[d] = (major == 10 && minor == 3) ? n : -1;
  }
  return cache[d] > 0 ? cache[d] : 0;
}

}  // namespace
}  // namespace dspark

extern "C" int dspark_qk_norm_rope(void* qkv, int64_t T, int64_t row_stride, int32_t dtype,
                                   const int64_t* positions, const void* q_weight, const void* k_weight,
                                   const float* cos_sin, int64_t max_pos, int32_t num_q_heads,
                                   int32_t num_k_heads, int32_t head_dim, float eps, uint32_t* status,
                                   void* stream_) {
  using namespace dspark;
  if (T < 0 || num_q_heads < 0 || num_k_heads < 0 || max_pos <= 0) return DSPARK_E_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return DSPARK_E_HEAD_DIM;
  if (dtype != DSPARK_DTYPE_BF16 && dtype != DSPARK_DTYPE_FP16) return DSPARK_E_DTYPE_MISMATCH;
  const int nh = num_q_heads + num_k_heads;
  if (T == 0 || nh == 0) return DSPARK_OK;
  if (qkv == nullptr || positions == nullptr || cos_sin == nullptr ||
      (num_q_heads > 0 && q_weight == nullptr) || (num_k_heads > 0 && k_weight == nullptr))
    return DSPARK_E_INVALID_ARG;
  if (row_stride < static_cast<int64_t>(nh) * head_dim) return DSPARK_E_POOL_LAYOUT;
  if (!aligned16(qkv) || row_stride % 8 != 0 || !aligned16(cos_sin) ||
      (q_weight != nullptr && !aligned16(q_weight)) || (k_weight != nullptr && !aligned16(k_weight)))
    return DSPARK_E_ALIGNMENT;
  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess) return DSPARK_E_DEVICE;
  const int sms = sm103_sms(device);
  if (sms == 0) return DSPARK_E_DEVICE;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  cudaError_t e;
  if (dtype == DSPARK_DTYPE_BF16)
    e = head_dim == 128 ? launch<__nv_bfloat16, 128>(qkv, T, row_stride, positions, q_weight, k_weight, cos_sin,
                                                     max_pos, num_q_heads, nh, eps, status, sms, stream)
                        : launch<__nv_bfloat16, 64>(qkv, T, row_stride, positions, q_weight, k_weight, cos_sin,
                                                    max_pos, num_q_heads, nh, eps, status, sms, stream);
  else
    e = head_dim == 128 ? launch<__half, 128>(qkv, T, row_stride, positions, q_weight, k_weight, cos_sin, max_pos,
                                              num_q_heads, nh, eps, status, sms, stream)
                        : launch<__half, 64>(qkv, T, row_stride, positions, q_weight, k_weight, cos_sin, max_pos,
                                             num_q_heads, nh, eps, status, sms, stream);
  return e == cudaSuccess ? DSPARK_OK : DSPARK_E_CUDA;
}
