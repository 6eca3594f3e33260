// The speculative verify step's accepted-draft count and bonus token (sglang
// PR #31847 summary page, "Implementation breakdown", item 2: the first
// position where draft and target disagree, one launch for the batch).
//
// One warp per request: lanes compare 32 positions at a time, a ballot of the
// mismatches gives the first one (find-first-set), and one lane writes the
// count and the target's token at it.  Launch- and latency-bound; integer
// work, so the result is exact.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/dspark_verify.h"

namespace dspark {
namespace {

constexpr int kVerifyWarps = 8;

__global__ void __launch_bounds__(kVerifyWarps * 32)
    correct_drafts_kernel(const int64_t* __restrict__ cand, int64_t cand_stride, const int64_t* __restrict__ target,
                          int64_t target_stride, int64_t batch, int block, int32_t* __restrict__ correct,
                          int64_t* __restrict__ bonus) {
  const int lane = threadIdx.x % 32;
  const int64_t b = static_cast<int64_t>(blockIdx.x) * kVerifyWarps + threadIdx.x / 32;
  if (b >= batch) return;   // whole warps only: b is warp-uniform
  const int64_t* c = cand + b * cand_stride;
  const int64_t* t = target + b * target_stride;
  int n = block - 1;        // all drafts accepted unless a mismatch is found
  for (int i0 = 0; i0 < block - 1; i0 += 32) {
    const int i = i0 + lane;
    const bool miss = i < block - 1 && c[i + 1] != t[i];
    const unsigned m = __ballot_sync(0xffffffffu, miss);
    if (m != 0u) {
      n = i0 + __ffs(static_cast<int>(m)) - 1;
      break;
    }
  }
  if (lane == 0) {
    correct[b] = n;
    bonus[b] = t[n];
  }
}

int sm103(int device) {
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

}  // namespace
}  // namespace dspark

extern "C" int dspark_correct_drafts_and_bonus(const int64_t* candidates, int64_t candidates_stride,
                                               const int64_t* target, int64_t target_stride, int64_t batch,
                                               int32_t block, int32_t* correct, int64_t* bonus, void* stream_) {
  using namespace dspark;
  if (batch < 0 || block < 1) return DSPARK_E_INVALID_ARG;
  if (batch == 0) return DSPARK_OK;
  if (candidates == nullptr || target == nullptr || correct == nullptr || bonus == nullptr ||
      candidates_stride < block || target_stride < block)
    return DSPARK_E_INVALID_ARG;
  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess || !sm103(device)) return DSPARK_E_DEVICE;
  const int64_t grid = (batch + kVerifyWarps - 1) / kVerifyWarps;
  if (grid > 0x7FFFFFFF) return DSPARK_E_INVALID_ARG;
  correct_drafts_kernel<<<static_cast<unsigned>(grid), kVerifyWarps * 32, 0, static_cast<cudaStream_t>(stream_)>>>(
      candidates, candidates_stride, target, target_stride, batch, block, correct, bonus);
  return cudaGetLastError() == cudaSuccess ? DSPARK_OK : DSPARK_E_CUDA;
}
