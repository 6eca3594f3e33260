// The draft model's combine_hidden_states (vLLM PR #46995 summary page, "Key
// source snippets": main_proj, a bias-free linear layer, then main_norm, an
// RMSNorm over the hidden dimension).
//
// The product y = aux . W^T runs on the fused tcgen05 kernel in its plain
// mode (same tiles, CTA pairs and split schedule as the KV write); its
// epilogue stores y in the model dtype and the sum of squares of the stored
// values of each row per 256-column tile.  norm_apply_kernel then finishes
// the norm in place: one warp per token adds the row's tile sums in a fixed
// order, and every element becomes round(y * inv * w).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "../../include/dspark_combine.h"
#include "internal.h"

namespace dspark {
namespace {

template <typename E>
__device__ __forceinline__ void unpack2(uint32_t u, float& a, float& b);
template <>
__device__ __forceinline__ void unpack2<__nv_bfloat16>(uint32_t u, float& a, float& b) {
  __nv_bfloat162 h;
  memcpy(&h, &u, 4);
  a = __low2float(h);
  b = __high2float(h);
}
template <>
__device__ __forceinline__ void unpack2<__half>(uint32_t u, float& a, float& b) {
  __half2 h;
  memcpy(&h, &u, 4);
  a = __low2float(h);
  b = __high2float(h);
}
template <typename E>
__device__ __forceinline__ uint32_t pack2(float a, float b);
template <>
__device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  uint32_t u;
  memcpy(&u, &h, 4);
  return u;
}
template <>
__device__ __forceinline__ uint32_t pack2<__half>(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  uint32_t u;
  memcpy(&u, &h, 4);
  return u;
}

constexpr int kNormWarps = 8;

template <typename E>
__global__ void __launch_bounds__(kNormWarps * 32)
    norm_apply_kernel(E* __restrict__ x, int64_t T, int64_t stride, int hidden, const float* __restrict__ rowsq,
                      int rowsq_stride, int n_tiles, const float* __restrict__ w, float eps) {
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kNormWarps + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (t >= T) return;
  float ss = 0.f;
  for (int j = 0; j < n_tiles; ++j) ss += rowsq[t * rowsq_stride + j];   // same order in every lane
  const float inv = 1.0f / sqrtf(ss / static_cast<float>(hidden) + eps);
  E* row = x + t * stride;
  for (int c = lane * 8; c < hidden; c += 32 * 8) {
    const uint4 q = *reinterpret_cast<const uint4*>(row + c);
    const float4 w0 = *reinterpret_cast<const float4*>(w + c);
    const float4 w1 = *reinterpret_cast<const float4*>(w + c + 4);
    const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
    const uint32_t in[4] = {q.x, q.y, q.z, q.w};
    uint32_t out[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float a, b;
      unpack2<E>(in[k], a, b);
      out[k] = pack2<E>(a * inv * wv[2 * k], b * inv * wv[2 * k + 1]);
    }
    *reinterpret_cast<uint4*>(row + c) = make_uint4(out[0], out[1], out[2], out[3]);
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace dspark

using namespace dspark;

struct dspark_combine {
  int device;
  int dtype;
  int64_t hidden, aux_dim;
  float eps;
  int sms;
  float* norm_w;          // [hidden] fp32
  uint32_t* status;
  float* workspace;       // split-schedule partial tiles
  int32_t* counters;      // split-schedule arrival counters, zero between launches
  float* rowsq;           // [capacity][n_tiles]
  int64_t rowsq_capacity;
  CUtensorMap tmap_w;       // W, boxes of 256 rows (single-CTA tiles)
  CUtensorMap tmap_w_half;  // W, boxes of 128 rows (CTA pairs)
};

extern "C" {

int dspark_pack_combine(const void* weight, int64_t hidden, int64_t aux_dim, int64_t weight_row_stride,
                        int32_t dtype, const void* norm_weight, int32_t norm_dtype, float eps, void* stream_,
                        dspark_combine_t* out) {
  if (out == nullptr) return DSPARK_E_INVALID_ARG;
  *out = nullptr;
  if (weight == nullptr || norm_weight == nullptr || hidden <= 0 || aux_dim <= 0 || !(eps >= 0.f))
    return DSPARK_E_INVALID_ARG;
  if (dtype != DSPARK_DTYPE_BF16 && dtype != DSPARK_DTYPE_FP16) return DSPARK_E_DTYPE_MISMATCH;
  if (norm_dtype != DSPARK_DTYPE_BF16 && norm_dtype != DSPARK_DTYPE_FP16 && norm_dtype != DSPARK_DTYPE_FP32)
    return DSPARK_E_DTYPE_MISMATCH;
  if (hidden % 32 != 0 || aux_dim % 8 != 0 || hidden > 0x7FFFFFFF || weight_row_stride < aux_dim)
    return DSPARK_E_SHAPE_MISMATCH;
  if (!aligned16(weight) || weight_row_stride % 8 != 0) return DSPARK_E_ALIGNMENT;
  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess) return DSPARK_E_DEVICE;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, device) != cudaSuccess || prop.major != 10 || prop.minor != 3)
    return DSPARK_E_DEVICE;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  dspark_combine* c = new dspark_combine;
  std::memset(c, 0, sizeof(*c));
  c->device = device;
  c->dtype = dtype;
  c->hidden = hidden;
  c->aux_dim = aux_dim;
  c->eps = eps;
  c->sms = prop.multiProcessorCount;
  bool ok = cudaMalloc(reinterpret_cast<void**>(&c->norm_w), sizeof(float) * hidden) == cudaSuccess &&
            cudaMalloc(reinterpret_cast<void**>(&c->status), sizeof(uint32_t)) == cudaSuccess &&
            cudaMalloc(reinterpret_cast<void**>(&c->workspace), workspace_bytes(c->sms)) == cudaSuccess &&
            cudaMalloc(reinterpret_cast<void**>(&c->counters), sizeof(int32_t) * c->sms) == cudaSuccess;
  if (ok) ok = cudaMemsetAsync(c->status, 0, sizeof(uint32_t), stream) == cudaSuccess;
  if (ok) ok = cudaMemsetAsync(c->counters, 0, sizeof(int32_t) * c->sms, stream) == cudaSuccess;
  if (ok) ok = launch_to_fp32(norm_weight, norm_dtype, c->norm_w, static_cast<int>(hidden), stream) == cudaSuccess;
  if (ok) ok = cudaStreamSynchronize(stream) == cudaSuccess;
  if (ok)
    ok = make_operand_map(&c->tmap_w, weight, dtype, aux_dim, hidden, weight_row_stride, kTileN) &&
         make_operand_map(&c->tmap_w_half, weight, dtype, aux_dim, hidden, weight_row_stride, kTileN / 2);
  if (!ok) {
    dspark_free_combine(c);
    return DSPARK_E_CUDA;
  }
  *out = c;
  return DSPARK_OK;
}

int dspark_combine_hidden_states(dspark_combine_t c, const void* aux, int64_t T, int64_t aux_row_stride,
                                 void* ctx_hidden, int64_t out_row_stride, void* stream_) {
  if (c == nullptr || T < 0) return DSPARK_E_INVALID_ARG;
  if (T == 0) return DSPARK_OK;
  if (aux == nullptr || ctx_hidden == nullptr || aux_row_stride < c->aux_dim || out_row_stride < c->hidden ||
      T > 0x7FFFFFFFLL)
    return DSPARK_E_INVALID_ARG;
  if (!aligned16(aux) || !aligned16(ctx_hidden) || aux_row_stride % 8 != 0 || out_row_stride % 8 != 0)
    return DSPARK_E_ALIGNMENT;
  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess || device != c->device) return DSPARK_E_DEVICE;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  const int n_tiles = static_cast<int>((c->hidden + kTileN - 1) / kTileN);
  if (T > c->rowsq_capacity) {
    // grows with the largest token count seen; the old buffer may still be in
    // use by queued work on another stream, so wait for the device first
    if (cudaDeviceSynchronize() != cudaSuccess) return DSPARK_E_CUDA;
    if (c->rowsq != nullptr) cudaFree(c->rowsq);
    c->rowsq = nullptr;
    c->rowsq_capacity = 0;
    if (cudaMalloc(reinterpret_cast<void**>(&c->rowsq), sizeof(float) * n_tiles * T) != cudaSuccess)
      return DSPARK_E_CUDA;
    c->rowsq_capacity = T;
  }
  CUtensorMap tmap_x;
  const int pairs = pair_workers(device);
  const bool pair = pairs > 0;
  if (!make_operand_map(&tmap_x, aux, c->dtype, static_cast<uint64_t>(c->aux_dim), static_cast<uint64_t>(T),
                        static_cast<uint64_t>(aux_row_stride), kTileM))
    return DSPARK_E_CUDA;
  WriteParams p;
  std::memset(&p, 0, sizeof(p));
  p.T = static_cast<int32_t>(T);
  p.H = static_cast<int32_t>(c->aux_dim);
  p.N = static_cast<int32_t>(c->hidden);
  p.num_kb = static_cast<int32_t>((c->aux_dim + kTileK - 1) / kTileK);
  const int tile_rows = pair ? 2 * kTileM : kTileM;
  p.num_m = static_cast<int32_t>((T + tile_rows - 1) / tile_rows);
  p.num_n = n_tiles;
  p.num_tiles = p.num_m * p.num_n;
  p.status = c->status;
  p.workspace = c->workspace;
  p.counters = c->counters;
  p.wait_limit_ns = kWaitLimitNs;
  p.split_wait_ns = kWaitLimitNs;
  p.split_wait_extra = 0;
  p.y = ctx_hidden;
  p.y_stride = out_row_stride;
  p.rowsq = c->rowsq;
  p.rowsq_stride = n_tiles;
  const int workers = plan_schedule(p.num_tiles, p.num_kb, pair ? pairs : c->sms, true, p);
  cudaError_t e = launch_plain(device, c->dtype, tmap_x, pair ? c->tmap_w_half : c->tmap_w, p,
                               pair ? 2 * workers : workers, pair, stream);
  if (e != cudaSuccess) return DSPARK_E_CUDA;
  const unsigned blocks = static_cast<unsigned>((T + kNormWarps - 1) / kNormWarps);
  if (c->dtype == DSPARK_DTYPE_BF16)
    norm_apply_kernel<__nv_bfloat16><<<blocks, kNormWarps * 32, 0, stream>>>(
        static_cast<__nv_bfloat16*>(ctx_hidden), T, out_row_stride, static_cast<int>(c->hidden), c->rowsq,
        n_tiles, n_tiles, c->norm_w, c->eps);
  else
    norm_apply_kernel<__half><<<blocks, kNormWarps * 32, 0, stream>>>(
        static_cast<__half*>(ctx_hidden), T, out_row_stride, static_cast<int>(c->hidden), c->rowsq, n_tiles,
        n_tiles, c->norm_w, c->eps);
  return cudaGetLastError() == cudaSuccess ? DSPARK_OK : DSPARK_E_CUDA;
}

int dspark_combine_get_status(dspark_combine_t c, void* stream_, uint32_t* flags) {
  if (c == nullptr || flags == nullptr) return DSPARK_E_INVALID_ARG;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  uint32_t v = 0;
  if (cudaMemcpyAsync(&v, c->status, sizeof(v), cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return DSPARK_E_CUDA;
  *flags = v;
  return DSPARK_OK;
}

void dspark_free_combine(dspark_combine_t c) {
  if (c == nullptr) return;
  int prev = -1;
  cudaGetDevice(&prev);
  cudaSetDevice(c->device);
  cudaDeviceSynchronize();
  if (c->norm_w) cudaFree(c->norm_w);
  if (c->status) cudaFree(c->status);
  if (c->workspace) cudaFree(c->workspace);
  if (c->counters) cudaFree(c->counters);
  if (c->rowsq) cudaFree(c->rowsq);
  if (prev >= 0) cudaSetDevice(prev);
  delete c;
}

}  // extern "C"
