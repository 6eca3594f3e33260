// C ABI of the DSpark context-KV write: argument checks, bundle packing and
// the launch of the fused kernel.  See include/dspark_ctx_kv.h for the
// contract of every entry point.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <cstdlib>
#include <cstring>
#include <new>

#include "internal.h"

namespace dspark {
namespace {

__global__ void to_fp32_kernel(const void* src, int dtype, float* dst, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  if (dtype == DSPARK_DTYPE_BF16)
    dst[i] = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(src)[i]);
  else if (dtype == DSPARK_DTYPE_FP16)
    dst[i] = __half2float(reinterpret_cast<const __half*>(src)[i]);
  else
    dst[i] = reinterpret_cast<const float*>(src)[i];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

int device_sm_count(int device) {
  static int cache[64] = {0};
  int d = device & 63;
  if (cache[d] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return 0;
    cache[d] = n;
  }
  return cache[d];
}

}  // namespace

// 2-D K-major operand map: rows of `cols` 16-bit elements, `pitch_elems`
// apart; boxes of kTileK x box_rows with the 128-byte swizzle; out-of-range
// rows/columns read as zero.
bool make_operand_map(CUtensorMap* map, const void* base, int dtype, uint64_t cols, uint64_t rows,
                      uint64_t pitch_elems, uint32_t box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {pitch_elems * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kTileK), box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map,
                        dtype == DSPARK_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                   : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                        2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace dspark

using namespace dspark;



cudaError_t dspark::launch_to_fp32(const void* src, int dtype, float* dst, int n,
                                   cudaStream_t stream) {
  to_fp32_kernel<<<(n + 127) / 128, 128, 0, stream>>>(src, dtype, dst, n);
  return cudaGetLastError();
}

int dspark::fill_write_params(const dspark_bundle* b, const void* ctx_hidden, int64_t T,
                              int64_t hidden_row_stride, int32_t hidden_dtype, const int64_t* positions,
                              const float* cos_sin, int64_t max_pos, const int64_t* cache_loc,
                              const int32_t* commit_lens, int64_t loc_row_width, int64_t num_windows,
                              void* const* k_pools, void* const* v_pools, const int64_t* k_row_strides,
                              const int64_t* v_row_strides, int32_t pool_dtype, int64_t pool_slots,
                              WriteParams& p) {
  if (b == nullptr) return DSPARK_E_INVALID_ARG;
  if (T < 0) return DSPARK_E_INVALID_ARG;
  if ((commit_lens != nullptr) != (loc_row_width != 0)) return DSPARK_E_COMMIT_ARGS;
  if (commit_lens != nullptr) {
    if (loc_row_width < 0 || num_windows < 0) return DSPARK_E_INVALID_ARG;
    if (num_windows * loc_row_width != T) return DSPARK_E_NUMEL;
  }
  if (hidden_dtype != b->dtype || pool_dtype != b->dtype) return DSPARK_E_DTYPE_MISMATCH;
  if (ctx_hidden == nullptr || positions == nullptr || cos_sin == nullptr || cache_loc == nullptr ||
      k_pools == nullptr || v_pools == nullptr || k_row_strides == nullptr ||
      v_row_strides == nullptr)
    return DSPARK_E_INVALID_ARG;
  if (max_pos <= 0 || pool_slots <= 0 || hidden_row_stride < b->H || T > 0x7FFFFFFFLL)
    return DSPARK_E_INVALID_ARG;
  if (!aligned16(ctx_hidden) || (hidden_row_stride * 2) % 16 != 0 || !aligned16(cos_sin))
    return DSPARK_E_ALIGNMENT;
  for (int l = 0; l < b->L; ++l) {
    if (k_pools[l] == nullptr || v_pools[l] == nullptr) return DSPARK_E_INVALID_ARG;
    if (k_row_strides[l] < b->KV || v_row_strides[l] < b->KV) return DSPARK_E_POOL_LAYOUT;
    if (!aligned16(k_pools[l]) || !aligned16(v_pools[l]) || k_row_strides[l] % 8 != 0 ||
        v_row_strides[l] % 8 != 0)
      return DSPARK_E_ALIGNMENT;
  }
  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess || device != b->device) return DSPARK_E_DEVICE;
  std::memset(&p, 0, sizeof(p));
  p.T = static_cast<int32_t>(T);
  p.H = b->H;
  p.N = static_cast<int32_t>(b->N);
  p.L = b->L;
  p.NH = b->NH;
  p.D = b->D;
  p.KV = b->KV;
  p.num_kb = (b->H + kTileK - 1) / kTileK;
  p.positions = positions;
  p.cache_loc = cache_loc;
  p.commit_lens = commit_lens;
  p.loc_row_width = commit_lens != nullptr ? loc_row_width : 0;
  p.cos_sin = cos_sin;
  p.max_pos = max_pos;
  p.pool_slots = pool_slots;
  p.knorm = b->knorm;
  p.bias = b->bias;
  p.eps = b->eps;
  p.status = b->status;
  p.workspace = b->workspace;
  p.counters = b->counters;
  p.trace = b->trace;
  p.wait_limit_ns = kWaitLimitNs;
  p.split_wait_ns = b->split_wait_ns;
  p.split_wait_extra = b->split_wait_extra;
  for (int l = 0; l < b->L; ++l) {
    p.k_pool[l] = k_pools[l];
    p.v_pool[l] = v_pools[l];
    p.k_stride[l] = k_row_strides[l];
    p.v_stride[l] = v_row_strides[l];
  }
  return DSPARK_OK;
}

extern "C" {

const char* dspark_status_string(int code) {
  switch (code) {
    case DSPARK_OK: return "ok";
    case DSPARK_E_INVALID_ARG: return "invalid argument";
    case DSPARK_E_NO_LAYERS: return "no layers";
    case DSPARK_E_NOT_SLICEABLE: return "qkv weight is not sliceable (quantized or unsupported dtype)";
    case DSPARK_E_EPS_MISMATCH: return "layers disagree on the k_norm epsilon";
    case DSPARK_E_DTYPE_MISMATCH: return "dtype mismatch";
    case DSPARK_E_SHAPE_MISMATCH: return "layers disagree on q_size / num_kv_heads / head_dim, or weight too short";
    case DSPARK_E_HEAD_DIM: return "head_dim must be 64 or 128";
    case DSPARK_E_BIAS_MISMATCH: return "bias present on some layers only";
    case DSPARK_E_COMMIT_ARGS: return "commit_lens and loc_row_width must be passed together";
    case DSPARK_E_NUMEL: return "num_windows * loc_row_width != num_tokens";
    case DSPARK_E_ALIGNMENT: return "buffer or stride not 16-byte aligned";
    case DSPARK_E_POOL_LAYOUT: return "pool row stride smaller than num_kv_heads * head_dim";
    case DSPARK_E_TOO_MANY_LAYERS: return "too many layers";
    case DSPARK_E_DEVICE: return "no sm_103 device, or not the bundle's device";
    case DSPARK_E_CUDA: return "CUDA runtime error";
    case DSPARK_E_DEVICE_FAULT: return "device-side check fired";
    case DSPARK_E_SCRATCH_LIMIT: return "launch needs more scratch than the no-alloc entry point's static array holds";
    default: return "unknown status";
  }
}

int dspark_check_ctx_kv_layers(const dspark_layer_desc* layers, int32_t num_layers, int32_t hidden) {
  if (num_layers < 0 || hidden <= 0) return DSPARK_E_INVALID_ARG;
  if (num_layers == 0) return DSPARK_E_NO_LAYERS;
  if (layers == nullptr) return DSPARK_E_INVALID_ARG;
  if (num_layers > DSPARK_MAX_LAYERS) return DSPARK_E_TOO_MANY_LAYERS;
  const dspark_layer_desc& f = layers[0];
  int with_bias = 0;
  for (int l = 0; l < num_layers; ++l) {
    const dspark_layer_desc& a = layers[l];
    if (a.weight_dtype != DSPARK_DTYPE_BF16 && a.weight_dtype != DSPARK_DTYPE_FP16)
      return DSPARK_E_NOT_SLICEABLE;
    if (a.eps != f.eps) return DSPARK_E_EPS_MISMATCH;
    if (a.weight_dtype != f.weight_dtype) return DSPARK_E_DTYPE_MISMATCH;
    if (a.q_size != f.q_size || a.num_kv_heads != f.num_kv_heads || a.head_dim != f.head_dim)
      return DSPARK_E_SHAPE_MISMATCH;
    if (a.head_dim != 64 && a.head_dim != 128) return DSPARK_E_HEAD_DIM;
    if (a.q_size < 0 || a.num_kv_heads <= 0) return DSPARK_E_INVALID_ARG;
    const int64_t kv = static_cast<int64_t>(a.num_kv_heads) * a.head_dim;
    if (a.qkv_rows < a.q_size + 2 * kv) return DSPARK_E_SHAPE_MISMATCH;
    if (a.qkv_row_stride < hidden) return DSPARK_E_INVALID_ARG;
    if (a.qkv_weight == nullptr || a.k_norm_weight == nullptr) return DSPARK_E_INVALID_ARG;
    if (a.k_norm_dtype != DSPARK_DTYPE_BF16 && a.k_norm_dtype != DSPARK_DTYPE_FP16 &&
        a.k_norm_dtype != DSPARK_DTYPE_FP32)
      return DSPARK_E_INVALID_ARG;
    with_bias += a.qkv_bias != nullptr;
  }
  if (with_bias != 0 && with_bias != num_layers) return DSPARK_E_BIAS_MISMATCH;
  return DSPARK_OK;
}

int dspark_pack_ctx_kv(const dspark_layer_desc* layers, int32_t num_layers, int32_t hidden,
                       void* stream_, dspark_bundle_t* out) {
  if (out == nullptr) return DSPARK_E_INVALID_ARG;
  *out = nullptr;
  const int chk = dspark_check_ctx_kv_layers(layers, num_layers, hidden);
  if (chk != DSPARK_OK) return chk;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);

  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return DSPARK_E_DEVICE;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return DSPARK_E_DEVICE;
  if (prop.major != 10 || prop.minor != 3) return DSPARK_E_DEVICE;
  if (encode_fn() == nullptr) return DSPARK_E_CUDA;

  const dspark_layer_desc& f = layers[0];
  dspark_bundle* b = new (std::nothrow) dspark_bundle();
  if (b == nullptr) return DSPARK_E_CUDA;
  b->device = device;
  b->dtype = f.weight_dtype;
  b->L = num_layers;
  b->H = hidden;
  b->NH = f.num_kv_heads;
  b->D = f.head_dim;
  b->KV = f.num_kv_heads * f.head_dim;
  b->N = static_cast<int64_t>(num_layers) * 2 * b->KV;
  b->w_pitch = (hidden + 7) / 8 * 8;   // 16-byte row pitch for TMA
  b->eps = f.eps;
  b->split_wait_extra = 0;
  b->split_wait_ns = kWaitLimitNs;
  b->sms = device_sm_count(device);
  if (b->sms <= 0) {
    delete b;
    return DSPARK_E_CUDA;
  }

  const size_t es = 2;
  bool ok = cudaMalloc(&b->w_all, static_cast<size_t>(b->N) * b->w_pitch * es) == cudaSuccess &&
            cudaMalloc(reinterpret_cast<void**>(&b->knorm), sizeof(float) * num_layers * b->D) ==
                cudaSuccess &&
            cudaMalloc(reinterpret_cast<void**>(&b->status), sizeof(uint32_t)) == cudaSuccess &&
            cudaMalloc(reinterpret_cast<void**>(&b->workspace), workspace_bytes(b->sms)) == cudaSuccess &&
            cudaMalloc(reinterpret_cast<void**>(&b->counters), sizeof(int32_t) * b->sms) == cudaSuccess;
  if (ok && f.qkv_bias != nullptr)
    ok = cudaMalloc(&b->bias, static_cast<size_t>(b->N) * es) == cudaSuccess;
  if (ok && b->w_pitch != hidden)
    ok = cudaMemsetAsync(b->w_all, 0, static_cast<size_t>(b->N) * b->w_pitch * es, stream) == cudaSuccess;
  if (ok) ok = cudaMemsetAsync(b->status, 0, sizeof(uint32_t), stream) == cudaSuccess;
  if (ok) ok = cudaMemsetAsync(b->counters, 0, sizeof(int32_t) * b->sms, stream) == cudaSuccess;
  for (int l = 0; ok && l < num_layers; ++l) {
    const dspark_layer_desc& a = layers[l];
    const int64_t rows = 2 * b->KV;
    const char* src = static_cast<const char*>(a.qkv_weight) + static_cast<size_t>(a.q_size) * a.qkv_row_stride * es;
    char* dst = static_cast<char*>(b->w_all) + static_cast<size_t>(l) * rows * b->w_pitch * es;
    ok = cudaMemcpy2DAsync(dst, b->w_pitch * es, src, a.qkv_row_stride * es, hidden * es, rows,
                           cudaMemcpyDeviceToDevice, stream) == cudaSuccess;
    if (ok && b->bias != nullptr)
      ok = cudaMemcpyAsync(static_cast<char*>(b->bias) + static_cast<size_t>(l) * rows * es,
                           static_cast<const char*>(a.qkv_bias) + static_cast<size_t>(a.q_size) * es,
                           rows * es, cudaMemcpyDeviceToDevice, stream) == cudaSuccess;
    if (ok)
      ok = launch_to_fp32(a.k_norm_weight, a.k_norm_dtype, b->knorm + static_cast<size_t>(l) * b->D,
                          b->D, stream) == cudaSuccess;
  }
  if (ok) ok = cudaStreamSynchronize(stream) == cudaSuccess;
  if (ok)
    ok = make_operand_map(&b->tmap_w, b->w_all, b->dtype, hidden, b->N, b->w_pitch, kTileN) &&
         make_operand_map(&b->tmap_w_half, b->w_all, b->dtype, hidden, b->N, b->w_pitch, kTileN / 2);
  if (!ok) {
    dspark_free_bundle(b);
    return DSPARK_E_CUDA;
  }
  *out = b;
  return DSPARK_OK;
}

int dspark_write_ctx_kv(dspark_bundle_t b, const void* ctx_hidden, int64_t T,
                        int64_t hidden_row_stride, int32_t hidden_dtype, const int64_t* positions,
                        const float* cos_sin, int64_t max_pos, const int64_t* cache_loc,
                        const int32_t* commit_lens, int64_t loc_row_width, int64_t num_windows,
                        void* const* k_pools, void* const* v_pools, const int64_t* k_row_strides,
                        const int64_t* v_row_strides, int32_t pool_dtype, int64_t pool_slots,
                        void* stream_) {
  if (b == nullptr) return DSPARK_E_INVALID_ARG;
  if (T == 0) return DSPARK_OK;
  WriteParams p;
  const int st = fill_write_params(b, ctx_hidden, T, hidden_row_stride, hidden_dtype, positions, cos_sin, max_pos,
                                   cache_loc, commit_lens, loc_row_width, num_windows, k_pools, v_pools,
                                   k_row_strides, v_row_strides, pool_dtype, pool_slots, p);
  if (st != DSPARK_OK) return st;
  const int device = b->device;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);

  // Small token counts: stream the weights (weights as the MMA's M side).
  int t_pad = 0, stages = 0;
  uint32_t stage_b = 0, acc_stride = 0, tmem_cols = 0;
  const bool stream_ok = b->KV % 128 == 0 &&
                         stream_plan(T, &t_pad, &stages, &stage_b, &acc_stride, &tmem_cols);
  // AUTO: weight streaming up to kStreamAutoMaxTokens tokens, and up to
  // kStreamAutoCutMaxTokens when the CTA pairs would have fewer than half as
  // many tiles as pairs (every tile cut); above, the pairs take whole tiles
  bool auto_stream = T <= kStreamAutoMaxTokens;
  if (!auto_stream && T <= kStreamAutoCutMaxTokens) {
    const int pairs_avail = pair_workers(device);
    const int64_t pair_tiles = ((T + 2 * kTileM - 1) / (2 * kTileM)) * ((b->N + kTileN - 1) / kTileN);
    auto_stream = pairs_avail <= 0 || 2 * pair_tiles < pairs_avail;
  }
  const bool use_stream = stream_ok && (b->variant == DSPARK_VARIANT_STREAM ||
                                        (b->variant == DSPARK_VARIANT_AUTO && auto_stream));
  if (b->variant == DSPARK_VARIANT_STREAM && !stream_ok) return DSPARK_E_INVALID_ARG;
  if (use_stream) {
    CUtensorMap tmap_x;
    if (!make_operand_map(&tmap_x, ctx_hidden, b->dtype, b->H, T, hidden_row_stride,
                          static_cast<uint32_t>(t_pad)))
      return DSPARK_E_CUDA;
    p.num_m = 1;
    p.num_n = static_cast<int32_t>(b->N / 128);
    p.num_tiles = p.num_n;
    const int resident = stream_workers(device, stages, stage_b);
    if (resident <= 0) return DSPARK_E_CUDA;
    const int grid = plan_schedule(p.num_tiles, p.num_kb, resident < b->sms ? resident : b->sms, false, p);
    const cudaError_t e = launch_stream(device, b->dtype, b->D, b->bias != nullptr, tmap_x, b->tmap_w_half, p,
                                        t_pad, stages, stage_b, acc_stride, tmem_cols, grid, stream);
    return e == cudaSuccess ? DSPARK_OK : DSPARK_E_CUDA;
  }

  CUtensorMap tmap_x;
  if (!make_operand_map(&tmap_x, ctx_hidden, b->dtype, b->H, T, hidden_row_stride, kTileM))
    return DSPARK_E_CUDA;
  // CTA pairs (256-token tiles, tcgen05 cta_group::2) unless single-CTA tiles
  // are asked for or the device has fewer than two SMs
  const int pairs = b->variant != DSPARK_VARIANT_SINGLE ? pair_workers(device) : 0;
  const bool pair = pairs > 0;
  int singles = 0;
  if (!pair) {
    singles = single_workers(device);
    if (singles <= 0) return DSPARK_E_CUDA;
    if (singles > b->sms) singles = b->sms;
  }
  const int tile_rows = pair ? 2 * kTileM : kTileM;
  p.num_m = static_cast<int32_t>((T + tile_rows - 1) / tile_rows);
  p.num_n = static_cast<int32_t>((b->N + kTileN - 1) / kTileN);
  p.num_tiles = p.num_m * p.num_n;
  const int workers = plan_schedule(p.num_tiles, p.num_kb, pair ? pairs : singles, true, p, true);
  give_leftover_to_v_tiles(p, workers);
  const int grid = pair ? 2 * workers : workers;
  const cudaError_t e =
      pair ? launch_pair(device, b->dtype, b->D, b->bias != nullptr, tmap_x, b->tmap_w_half, p, grid, stream)
           : launch_tiled(device, b->dtype, b->D, b->bias != nullptr, tmap_x, b->tmap_w, p, grid, stream);
  return e == cudaSuccess ? DSPARK_OK : DSPARK_E_CUDA;
}

int dspark_set_kernel_variant(dspark_bundle_t b, int32_t variant) {
  if (b == nullptr) return DSPARK_E_INVALID_ARG;
  if (variant != DSPARK_VARIANT_AUTO && variant != DSPARK_VARIANT_SINGLE && variant != DSPARK_VARIANT_PAIR &&
      variant != DSPARK_VARIANT_STREAM)
    return DSPARK_E_INVALID_ARG;
  b->variant = variant;
  return DSPARK_OK;
}

int dspark_set_split_wait_test(dspark_bundle_t b, int32_t missing_arrivals, uint64_t limit_ns) {
  if (b == nullptr || missing_arrivals < 0 || missing_arrivals > 1024) return DSPARK_E_INVALID_ARG;
  if (missing_arrivals == 0) {
    b->split_wait_extra = 0;
    b->split_wait_ns = kWaitLimitNs;
    return DSPARK_OK;
  }
  if (limit_ns == 0 || limit_ns > kWaitLimitNs) return DSPARK_E_INVALID_ARG;
  b->split_wait_extra = missing_arrivals;
  b->split_wait_ns = limit_ns;
  return DSPARK_OK;
}

int dspark_get_device_status(dspark_bundle_t b, void* stream_, uint32_t* flags) {
  if (b == nullptr || flags == nullptr) return DSPARK_E_INVALID_ARG;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  uint32_t v = 0;
  if (cudaMemcpyAsync(&v, b->status, sizeof(v), cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return DSPARK_E_CUDA;
  *flags = v;
  return DSPARK_OK;
}

int dspark_clear_device_status(dspark_bundle_t b, void* stream_) {
  if (b == nullptr) return DSPARK_E_INVALID_ARG;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  // the arrival counters are reset too: a launch that timed out may leave them set
  return cudaMemsetAsync(b->status, 0, sizeof(uint32_t), stream) == cudaSuccess &&
                 cudaMemsetAsync(b->counters, 0, sizeof(int32_t) * b->sms, stream) == cudaSuccess
             ? DSPARK_OK
             : DSPARK_E_CUDA;
}

int dspark_set_trace_buffer(dspark_bundle_t b, uint64_t* buf, int64_t words) {
  if (b == nullptr) return DSPARK_E_INVALID_ARG;
  if (buf != nullptr && words < static_cast<int64_t>(b->sms) * kTraceWords) return DSPARK_E_INVALID_ARG;
  b->trace = buf;
  return DSPARK_OK;
}

int dspark_describe_schedule(int64_t tiles, int32_t num_kb, int32_t workers, int32_t split_first_allowed,
                             dspark_schedule_info* out) {
  if (out == nullptr || tiles < 1 || tiles > 0x7FFFFFFF || num_kb < 1 || workers < 1) return DSPARK_E_INVALID_ARG;
  WriteParams p;
  std::memset(&p, 0, sizeof(p));
  const int grid =
      plan_schedule(static_cast<int>(tiles), num_kb, workers, split_first_allowed != 0, p, split_first_allowed != 0);
  out->workers = grid;
  out->whole_tiles = p.dp_tiles;
  out->split_units = p.sk_units;
  out->split_workers = p.sk_workers;
  out->split_first = p.sk_first;
  return DSPARK_OK;
}

int dspark_bundle_get_info(dspark_bundle_t b, dspark_bundle_info* info) {
  if (b == nullptr || info == nullptr) return DSPARK_E_INVALID_ARG;
  info->num_layers = b->L;
  info->hidden = b->H;
  info->num_kv_heads = b->NH;
  info->head_dim = b->D;
  info->dtype = b->dtype;
  info->has_bias = b->bias != nullptr;
  info->device = b->device;
  info->eps = b->eps;
  info->stacked_rows = b->N;
  return DSPARK_OK;
}

void dspark_free_bundle(dspark_bundle_t b) {
  if (b == nullptr) return;
  int prev = -1;
  cudaGetDevice(&prev);
  cudaSetDevice(b->device);
  cudaDeviceSynchronize();
  if (b->w_all) cudaFree(b->w_all);
  if (b->bias) cudaFree(b->bias);
  if (b->knorm) cudaFree(b->knorm);
  if (b->status) cudaFree(b->status);
  if (b->workspace) cudaFree(b->workspace);
  if (b->counters) cudaFree(b->counters);
  if (prev >= 0) cudaSetDevice(prev);
  delete b;
}

}  // extern "C"
