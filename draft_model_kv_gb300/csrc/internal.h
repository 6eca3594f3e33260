// Internal interface between the C-ABI host code (api.cu) and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "../../include/dspark_ctx_kv.h"

namespace dspark {

// Everything the fused write needs besides the two operand tensor maps.
struct WriteParams {
  int32_t T, H, N, L, NH, D, KV;
  int32_t num_m, num_n, num_kb, num_tiles;
  const int64_t* positions;
  const int64_t* cache_loc;
  const int32_t* commit_lens;   // null unless window mode
  int64_t loc_row_width;        // W in window mode, else 0
  const float* cos_sin;         // [max_pos, D]
  int64_t max_pos;
  int64_t pool_slots;
  const float* knorm;           // [L, D] fp32
  const void* bias;             // [N] or null
  float eps;
  uint32_t* status;             // device status word (DSPARK_FLAG_*)
  uint64_t wait_limit_ns;       // bound on any single in-kernel wait
  void* k_pool[DSPARK_MAX_LAYERS];
  void* v_pool[DSPARK_MAX_LAYERS];
  int64_t k_stride[DSPARK_MAX_LAYERS];
  int64_t v_stride[DSPARK_MAX_LAYERS];
};

// Tiled tcgen05 path: one CTA per SM, 128-token x 256-column output tiles.
constexpr int kTileM = 128;
constexpr int kTileN = 256;
constexpr int kTileK = 64;     // one 128-byte swizzle row of 16-bit elements
constexpr int kStages = 4;
constexpr int kTiledThreads = 192;
constexpr int kGroupM = 8;     // m-blocks per raster group (L2 reuse of weight tiles)

size_t tiled_smem_bytes();

// Launch the tiled kernel for the bundle dtype (1 = bf16, 2 = fp16).  Returns
// the CUDA error of the launch.
cudaError_t launch_tiled(int device, int dtype, int head_dim, bool has_bias, const CUtensorMap& tmap_x,
                         const CUtensorMap& tmap_w, const WriteParams& p, int grid,
                         cudaStream_t stream);

// Convert a [n] bf16 / fp16 / fp32 vector to fp32 (bundle packing).
cudaError_t launch_to_fp32(const void* src, int dtype, float* dst, int n, cudaStream_t stream);

}  // namespace dspark
