// Non-blocking read of a bundle's device status word (the C ABI declared in
// include/dspark_ctx_kv.h), for callers that pipeline their writes and read
// every write's status without a synchronisation per write.
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"

extern "C" int dspark_read_device_status_async(dspark_bundle_t b, void* stream_, uint32_t* flags) {
  if (b == nullptr || flags == nullptr) return DSPARK_E_INVALID_ARG;
  return cudaMemcpyAsync(flags, b->status, sizeof(uint32_t), cudaMemcpyDeviceToHost,
                         static_cast<cudaStream_t>(stream_)) == cudaSuccess
             ? DSPARK_OK
             : DSPARK_E_CUDA;
}
