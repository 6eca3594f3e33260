// combine_hidden_states fused into the context-KV write (vLLM PR #46995
// summary page, "Key source snippets": the draft model's
// combine_hidden_states feeds every draft layer's KV projection).
//
// With y = aux . W_main^T (rounded to the model dtype) and
// ctx_hidden = y * s_t * w (s_t = 1/sqrt(mean(y_t^2) + eps), w = main_norm's
// weight), the write's projection is
//
//   ctx_hidden . W_kv^T = s_t * (y . (W_kv diag(w))^T)
//
// so the pack scales the stacked K|V weights by w once, and one launch runs
// main_proj in the tiled kernel's plain mode (y and its row sums of squares
// into scratch that stays in L2 for decode-sized batches) and then the write
// over y, each token row scaled by s_t in the epilogue before the bias, the K
// norm and the rotation.  ctx_hidden itself is never formed.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <type_traits>

#include "../../include/dspark_combine.h"
#include "internal.h"

namespace dspark {
namespace {

// W[n][j] = round(W[n][j] * w[j]) for j < cols, rows `pitch` elements apart.
template <typename E>
__global__ void scale_columns_kernel(E* w, int64_t rows, int64_t cols, int64_t pitch, const float* scale) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= rows * cols) return;
  const int64_t r = i / cols, c = i % cols;
  E* x = w + r * pitch + c;
  if constexpr (std::is_same<E, __nv_bfloat16>::value)
    *x = __float2bfloat16_rn(__bfloat162float(*x) * scale[c]);
  else
    *x = __float2half_rn(__half2float(*x) * scale[c]);
}

bool aligned16f(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace dspark

using namespace dspark;

struct dspark_fused {
  int device;
  int dtype;
  int64_t hidden, aux_dim;
  float norm_eps;
  dspark_bundle_t bundle;      // the write's bundle, stacked weights scaled by main_norm's weight
  CUtensorMap tmap_main;       // main_proj weight [hidden, aux_dim], 128-row boxes (not copied)
  int32_t* phase_count;        // CTAs done with main_proj, zero between launches
  void* y;                     // [cap, hidden] scratch in the model dtype
  float* rowsq;                // [cap][hidden / 256] sums of squares of y
  int64_t cap;
};

extern "C" {

int dspark_pack_fused_ctx_kv(const void* main_proj_weight, int64_t aux_dim, int64_t weight_row_stride,
                             const void* main_norm_weight, int32_t norm_dtype, float norm_eps,
                             const dspark_layer_desc* layers, int32_t num_layers, int32_t hidden, void* stream_,
                             dspark_fused_t* out) {
  if (out == nullptr) return DSPARK_E_INVALID_ARG;
  *out = nullptr;
  if (main_proj_weight == nullptr || main_norm_weight == nullptr || aux_dim <= 0 || !(norm_eps >= 0.f) ||
      hidden <= 0)
    return DSPARK_E_INVALID_ARG;
  if (norm_dtype != DSPARK_DTYPE_BF16 && norm_dtype != DSPARK_DTYPE_FP16 && norm_dtype != DSPARK_DTYPE_FP32)
    return DSPARK_E_DTYPE_MISMATCH;
  if (hidden % 32 != 0 || aux_dim % 8 != 0 || weight_row_stride < aux_dim) return DSPARK_E_SHAPE_MISMATCH;
  if (!aligned16f(main_proj_weight) || weight_row_stride % 8 != 0) return DSPARK_E_ALIGNMENT;
  const int chk = dspark_check_ctx_kv_layers(layers, num_layers, hidden);
  if (chk != DSPARK_OK) return chk;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  dspark_bundle_t b = nullptr;
  int st = dspark_pack_ctx_kv(layers, num_layers, hidden, stream_, &b);
  if (st != DSPARK_OK) return st;
  dspark_fused* f = new dspark_fused;
  std::memset(f, 0, sizeof(*f));
  f->device = b->device;
  f->dtype = b->dtype;
  f->hidden = hidden;
  f->aux_dim = aux_dim;
  f->norm_eps = norm_eps;
  f->bundle = b;
  float* w32 = nullptr;
  bool ok = cudaMalloc(reinterpret_cast<void**>(&w32), sizeof(float) * hidden) == cudaSuccess &&
            cudaMalloc(reinterpret_cast<void**>(&f->phase_count), sizeof(int32_t)) == cudaSuccess;
  if (ok) ok = cudaMemsetAsync(f->phase_count, 0, sizeof(int32_t), stream) == cudaSuccess;
  if (ok) ok = launch_to_fp32(main_norm_weight, norm_dtype, w32, static_cast<int>(hidden), stream) == cudaSuccess;
  if (ok) {
    const int64_t n = b->N * static_cast<int64_t>(hidden);
    const unsigned blocks = static_cast<unsigned>((n + 255) / 256);
    if (b->dtype == DSPARK_DTYPE_BF16)
      scale_columns_kernel<__nv_bfloat16><<<blocks, 256, 0, stream>>>(static_cast<__nv_bfloat16*>(b->w_all), b->N,
                                                                       hidden, b->w_pitch, w32);
    else
      scale_columns_kernel<__half><<<blocks, 256, 0, stream>>>(static_cast<__half*>(b->w_all), b->N, hidden,
                                                                b->w_pitch, w32);
    ok = cudaGetLastError() == cudaSuccess && cudaStreamSynchronize(stream) == cudaSuccess;
  }
  if (w32 != nullptr) cudaFree(w32);
  if (ok)
    ok = make_operand_map(&f->tmap_main, main_proj_weight, b->dtype, static_cast<uint64_t>(aux_dim),
                          static_cast<uint64_t>(hidden), static_cast<uint64_t>(weight_row_stride), kTileN / 2);
  if (!ok) {
    dspark_free_fused(f);
    return DSPARK_E_CUDA;
  }
  *out = f;
  return DSPARK_OK;
}

int dspark_combine_write_ctx_kv(dspark_fused_t f, const void* aux, int64_t T, int64_t aux_row_stride,
                                const int64_t* positions, const float* cos_sin, int64_t max_pos,
                                const int64_t* cache_loc, const int32_t* commit_lens, int64_t loc_row_width,
                                int64_t num_windows, void* const* k_pools, void* const* v_pools,
                                const int64_t* k_row_strides, const int64_t* v_row_strides, int32_t pool_dtype,
                                int64_t pool_slots, void* stream_) {
  if (f == nullptr || T < 0) return DSPARK_E_INVALID_ARG;
  if (T == 0) return DSPARK_OK;
  if (aux == nullptr || aux_row_stride < f->aux_dim || T > 0x7FFFFFFFLL) return DSPARK_E_INVALID_ARG;
  if (!aligned16f(aux) || aux_row_stride % 8 != 0) return DSPARK_E_ALIGNMENT;
  dspark_bundle* b = f->bundle;
  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess || device != f->device) return DSPARK_E_DEVICE;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  const int n1 = static_cast<int>((f->hidden + kTileN - 1) / kTileN);
  if (T > f->cap) {
    // the scratch grows with the largest token count seen; the old buffers
    // may still be in use by queued work, so wait for the device first
    if (cudaDeviceSynchronize() != cudaSuccess) return DSPARK_E_CUDA;
    if (f->y != nullptr) cudaFree(f->y);
    if (f->rowsq != nullptr) cudaFree(f->rowsq);
    f->y = nullptr;
    f->rowsq = nullptr;
    f->cap = 0;
    if (cudaMalloc(&f->y, static_cast<size_t>(T) * f->hidden * 2) != cudaSuccess ||
        cudaMalloc(reinterpret_cast<void**>(&f->rowsq), sizeof(float) * n1 * T) != cudaSuccess)
      return DSPARK_E_CUDA;
    f->cap = T;
  }
  // the write over y (the fused second problem)
  WriteParams p;
  int st = fill_write_params(b, f->y, T, f->hidden, f->dtype, positions, cos_sin, max_pos, cache_loc, commit_lens,
                             loc_row_width, num_windows, k_pools, v_pools, k_row_strides, v_row_strides, pool_dtype,
                             pool_slots, p);
  if (st != DSPARK_OK) return st;
  const int pairs = pair_workers(device);
  if (pairs <= 0) return DSPARK_E_CUDA;
  p.num_m = static_cast<int32_t>((T + 2 * kTileM - 1) / (2 * kTileM));
  p.num_n = static_cast<int32_t>((b->N + kTileN - 1) / kTileN);
  p.num_tiles = p.num_m * p.num_n;
  // the write takes whole tiles when they number at least half the pairs, as
  // the standalone write does
  p.workers = plan_schedule(p.num_tiles, p.num_kb, pairs, true, p, true);
  give_leftover_to_v_tiles(p, p.workers);
  p.trace = nullptr;
  p.phase_count = f->phase_count;
  p.rowsq = f->rowsq;
  p.rowsq_stride = n1;
  p.rowsq_n = n1;
  p.norm_n = static_cast<int32_t>(f->hidden);
  p.norm_eps = f->norm_eps;
  // main_proj in plain mode (the first problem): y and its row sums
  WriteParams p1;
  std::memset(&p1, 0, sizeof(p1));
  p1.T = p.T;
  p1.H = static_cast<int32_t>(f->aux_dim);
  p1.N = static_cast<int32_t>(f->hidden);
  p1.num_kb = static_cast<int32_t>((f->aux_dim + kTileK - 1) / kTileK);
  p1.num_m = p.num_m;
  p1.num_n = n1;
  p1.num_tiles = p1.num_m * p1.num_n;
  p1.workers = plan_schedule(p1.num_tiles, p1.num_kb, pairs, true, p1);
  p1.y = f->y;
  p1.y_stride = f->hidden;
  p1.rowsq = f->rowsq;
  p1.rowsq_stride = n1;
  p1.status = p.status;
  p1.workspace = p.workspace;
  p1.counters = p.counters;
  p1.wait_limit_ns = p.wait_limit_ns;
  p1.split_wait_ns = p.split_wait_ns;
  p1.split_wait_extra = p.split_wait_extra;
  p1.phase_count = f->phase_count;
  CUtensorMap tmap_aux, tmap_y;
  if (!make_operand_map(&tmap_aux, aux, f->dtype, static_cast<uint64_t>(f->aux_dim), static_cast<uint64_t>(T),
                        static_cast<uint64_t>(aux_row_stride), kTileM) ||
      !make_operand_map(&tmap_y, f->y, f->dtype, static_cast<uint64_t>(f->hidden), static_cast<uint64_t>(T),
                        static_cast<uint64_t>(f->hidden), kTileM))
    return DSPARK_E_CUDA;
  const int workers = p1.workers > p.workers ? p1.workers : p.workers;
  const cudaError_t e = launch_fused(device, f->dtype, b->D, b->bias != nullptr, tmap_aux, f->tmap_main, p1, tmap_y,
                                     b->tmap_w_half, p, 2 * workers, stream);
  return e == cudaSuccess ? DSPARK_OK : DSPARK_E_CUDA;
}

int dspark_fused_get_status(dspark_fused_t f, void* stream, uint32_t* flags) {
  if (f == nullptr) return DSPARK_E_INVALID_ARG;
  return dspark_get_device_status(f->bundle, stream, flags);
}

int dspark_fused_clear_status(dspark_fused_t f, void* stream_) {
  if (f == nullptr) return DSPARK_E_INVALID_ARG;
  const int st = dspark_clear_device_status(f->bundle, stream_);
  if (st != DSPARK_OK) return st;
  return cudaMemsetAsync(f->phase_count, 0, sizeof(int32_t), static_cast<cudaStream_t>(stream_)) == cudaSuccess
             ? DSPARK_OK
             : DSPARK_E_CUDA;
}

void dspark_free_fused(dspark_fused_t f) {
  if (f == nullptr) return;
  int prev = -1;
  cudaGetDevice(&prev);
  cudaSetDevice(f->device);
  cudaDeviceSynchronize();
  if (f->phase_count) cudaFree(f->phase_count);
  if (f->y) cudaFree(f->y);
  if (f->rowsq) cudaFree(f->rowsq);
  if (prev >= 0) cudaSetDevice(prev);
  dspark_free_bundle(f->bundle);
  delete f;
}

}  // extern "C"
