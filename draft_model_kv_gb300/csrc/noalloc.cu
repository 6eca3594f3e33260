// dspark_write_ctx_kv_noalloc: the context-KV write for callers that must not
// allocate device memory.
//
// Who needs it: a host framework that owns every byte of device memory through
// its own pool allocator (a foreign cudaMalloc bypasses its accounting and can
// fragment or exhaust the pool), and latency-critical loops where cudaMalloc's
// implicit device-wide synchronisation is not acceptable.  Such callers cannot
// use dspark_pack_ctx_kv (it allocates the bundle) nor the workspace that the
// regular write keeps in the bundle.  Here the caller passes the already
// stacked weights and every input and output, and the kernel's scratch memory
// (the stream-K partial-tile workspace, its arrival counters and a fallback
// status word) lives in one file-scope device array that the library reserves
// once per GPU it is loaded on.
//
// Limits and sharing rules:
//  - the array is kNoAllocScratchBytes (16 MiB + 4 KiB) on every GPU that loads
//    the library, held until the process exits;
//  - a call runs on at most kNoAllocMaxCtas (64) SMs, the number of CTAs whose
//    partial tiles fit in the array.  The scratch a launch uses grows with its
//    CTA count only, never with the token count or the model's sizes, so with
//    this cap every problem fits; DSPARK_E_SCRATCH_LIMIT stays as a guard that
//    valid arguments never reach;
//  - a NULL status_flags sends the device flags (out-of-range positions or
//    slots, a wait that ran out) to a word inside the array that no call reads
//    back: those errors are then discarded;
//  - every call uses the same array: two calls whose kernels overlap on the GPU
//    (different streams without ordering, or two host threads) race and give
//    wrong results; keep calls on one device ordered (one stream, or events);
//  - the array keeps whatever the previous call left; the arrival counters are
//    cleared by every call before its kernel runs (stream-ordered memset, no
//    allocation);
//  - the first call on each device looks up the array's device address
//    (cudaGetSymbolAddress) and sets the kernel's shared-memory limit; make that
//    first call before any stream capture begins.
#include <cudaTypedefs.h>

#include <atomic>
#include <cstring>
#include <mutex>

#include "internal.h"

namespace dspark {
namespace {

constexpr int kNoAllocMaxCtas = 64;
constexpr size_t kNoAllocWorkspaceBytes = static_cast<size_t>(kNoAllocMaxCtas) * 2 * kTileM * kTileN * sizeof(float);
constexpr size_t kNoAllocCounterOffset = kNoAllocWorkspaceBytes;                 // int32 [kNoAllocMaxCtas]
constexpr size_t kNoAllocStatusOffset = kNoAllocWorkspaceBytes + 2048;           // uint32 fallback status word
constexpr size_t kNoAllocScratchBytes = kNoAllocWorkspaceBytes + 4096;
static_assert(kNoAllocCounterOffset + sizeof(int32_t) * kNoAllocMaxCtas <= kNoAllocStatusOffset,
              "arrival counters overlap the status word");
static_assert(kNoAllocStatusOffset + sizeof(uint32_t) <= kNoAllocScratchBytes, "status word outside the array");

// The scratch itself.  In host code this name is only a stand-in for the
// device symbol: never pass it to a kernel; use the address looked up below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

struct DeviceScratch {
  unsigned char* base = nullptr;
  int sms = 0;
  bool ready = false;
};

DeviceScratch g_dev[64];
std::mutex g_setup_mutex;

// Once per device, with that device current: the array's device address and
// the device's SM count.
int scratch_for_device(int device, DeviceScratch** out) {
  if (device < 0 || device >= 64) return DSPARK_E_DEVICE;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  DeviceScratch& d = g_dev[device];
  if (!d.ready) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
      return DSPARK_E_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || sms <= 0)
      return DSPARK_E_CUDA;
    d.base = static_cast<unsigned char*>(ptr);
    d.sms = sms;
    d.ready = true;
  }
  *out = &d;
  return DSPARK_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_tiled() {
  static std::atomic<PFN_cuTensorMapEncodeTiled_v12000> fn{nullptr};
  PFN_cuTensorMapEncodeTiled_v12000 f = fn.load();
  if (f == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      f = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
      fn.store(f);
    }
  }
  return f;
}

bool operand_map(CUtensorMap* map, const void* base, int dtype, uint64_t cols, uint64_t rows,
                 uint64_t pitch_elems, uint32_t box_rows) {
  auto fn = encode_tiled();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {pitch_elems * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kTileK), box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map,
            dtype == DSPARK_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
            2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace dspark

using namespace dspark;

extern "C" int dspark_write_ctx_kv_noalloc(
    const void* stacked_weight, int64_t weight_row_stride, const void* stacked_bias,
    const float* k_norm_weight, float eps, int32_t num_layers, int32_t hidden, int32_t num_kv_heads,
    int32_t head_dim, int32_t dtype, const void* ctx_hidden, int64_t T, int64_t hidden_row_stride,
    const int64_t* positions, const float* cos_sin, int64_t max_pos, const int64_t* cache_loc,
    const int32_t* commit_lens, int64_t loc_row_width, int64_t num_windows, void* const* k_pools,
    void* const* v_pools, const int64_t* k_row_strides, const int64_t* v_row_strides,
    int64_t pool_slots, uint32_t* status_flags, void* stream_) {
  // ---- argument checks (host only; nothing is enqueued on refusal)
  if (num_layers <= 0 || hidden <= 0 || num_kv_heads <= 0 || T < 0) return DSPARK_E_INVALID_ARG;
  if (num_layers > DSPARK_MAX_LAYERS) return DSPARK_E_TOO_MANY_LAYERS;
  if (head_dim != 64 && head_dim != 128) return DSPARK_E_HEAD_DIM;
  if (dtype != DSPARK_DTYPE_BF16 && dtype != DSPARK_DTYPE_FP16) return DSPARK_E_NOT_SLICEABLE;
  if (T == 0) return DSPARK_OK;
  if ((commit_lens != nullptr) != (loc_row_width != 0)) return DSPARK_E_COMMIT_ARGS;
  if (commit_lens != nullptr) {
    if (loc_row_width < 0 || num_windows < 0) return DSPARK_E_INVALID_ARG;
    if (num_windows * loc_row_width != T) return DSPARK_E_NUMEL;
  }
  if (stacked_weight == nullptr || k_norm_weight == nullptr || ctx_hidden == nullptr ||
      positions == nullptr || cos_sin == nullptr || cache_loc == nullptr || k_pools == nullptr ||
      v_pools == nullptr || k_row_strides == nullptr || v_row_strides == nullptr)
    return DSPARK_E_INVALID_ARG;
  if (max_pos <= 0 || pool_slots <= 0 || hidden_row_stride < hidden || weight_row_stride < hidden ||
      T > 0x7FFFFFFFLL)
    return DSPARK_E_INVALID_ARG;
  if (!aligned16(ctx_hidden) || (hidden_row_stride * 2) % 16 != 0 || !aligned16(cos_sin) ||
      !aligned16(stacked_weight) || (weight_row_stride * 2) % 16 != 0 || !aligned16(k_norm_weight))
    return DSPARK_E_ALIGNMENT;
  const int32_t KV = num_kv_heads * head_dim;
  for (int l = 0; l < num_layers; ++l) {
    if (k_pools[l] == nullptr || v_pools[l] == nullptr) return DSPARK_E_INVALID_ARG;
    if (k_row_strides[l] < KV || v_row_strides[l] < KV) return DSPARK_E_POOL_LAYOUT;
    if (!aligned16(k_pools[l]) || !aligned16(v_pools[l]) || k_row_strides[l] % 8 != 0 ||
        v_row_strides[l] % 8 != 0)
      return DSPARK_E_ALIGNMENT;
  }

  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess) return DSPARK_E_DEVICE;
  DeviceScratch* scratch = nullptr;
  const int st = scratch_for_device(device, &scratch);
  if (st != DSPARK_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);

  const int64_t N = static_cast<int64_t>(num_layers) * 2 * KV;
  WriteParams p;
  std::memset(&p, 0, sizeof(p));
  p.T = static_cast<int32_t>(T);
  p.H = hidden;
  p.N = static_cast<int32_t>(N);
  p.L = num_layers;
  p.NH = num_kv_heads;
  p.D = head_dim;
  p.KV = KV;
  p.num_m = static_cast<int32_t>((T + kTileM - 1) / kTileM);
  p.num_n = static_cast<int32_t>((N + kTileN - 1) / kTileN);
  p.num_kb = (hidden + kTileK - 1) / kTileK;
  p.num_tiles = p.num_m * p.num_n;
  const int ctas = scratch->sms < kNoAllocMaxCtas ? scratch->sms : kNoAllocMaxCtas;
  const int grid = plan_schedule(p.num_tiles, p.num_kb, ctas, true, p);
  // plan_schedule never returns more workers than it is given, so the
  // workspace of the launch fits (workspace_bytes(kNoAllocMaxCtas) is the
  // array's workspace part); the check guards that rule
  if (workspace_bytes(grid) > kNoAllocWorkspaceBytes || grid > kNoAllocMaxCtas)
    return DSPARK_E_SCRATCH_LIMIT;

  CUtensorMap tmap_x, tmap_w;
  if (!operand_map(&tmap_x, ctx_hidden, dtype, hidden, T, hidden_row_stride, kTileM) ||
      !operand_map(&tmap_w, stacked_weight, dtype, hidden, N, weight_row_stride, kTileN))
    return DSPARK_E_CUDA;

  p.positions = positions;
  p.cache_loc = cache_loc;
  p.commit_lens = commit_lens;
  p.loc_row_width = commit_lens != nullptr ? loc_row_width : 0;
  p.cos_sin = cos_sin;
  p.max_pos = max_pos;
  p.pool_slots = pool_slots;
  p.knorm = k_norm_weight;
  p.bias = stacked_bias;
  p.eps = eps;
  p.workspace = reinterpret_cast<float*>(scratch->base);
  p.counters = reinterpret_cast<int32_t*>(scratch->base + kNoAllocCounterOffset);
  p.status = status_flags != nullptr ? status_flags
                                     : reinterpret_cast<uint32_t*>(scratch->base + kNoAllocStatusOffset);
  p.trace = nullptr;
  p.wait_limit_ns = kWaitLimitNs;
  p.split_wait_ns = kWaitLimitNs;
  p.split_wait_extra = 0;
  for (int l = 0; l < num_layers; ++l) {
    p.k_pool[l] = k_pools[l];
    p.v_pool[l] = v_pools[l];
    p.k_stride[l] = k_row_strides[l];
    p.v_stride[l] = v_row_strides[l];
  }
  // counters must start at zero; a previous launch that stopped early may have
  // left some set
  if (cudaMemsetAsync(p.counters, 0, sizeof(int32_t) * kNoAllocMaxCtas, stream) != cudaSuccess)
    return DSPARK_E_CUDA;
  const cudaError_t e =
      launch_tiled(device, dtype, head_dim, stacked_bias != nullptr, tmap_x, tmap_w, p, grid, stream);
  return e == cudaSuccess ? DSPARK_OK : DSPARK_E_CUDA;
}
