// lid_internal.h -- what the library's translation units share on the host:
// the per-device facts the top-k side caches, its CUDA-error recording and its
// stream-ordered workspace allocator (defined in lid_api.cu), and the
// sparse-attention side's device error word (defined in lid_attn.cu).
#pragma once

#include <cuda_runtime.h>

namespace lid {

struct DeviceEnv {
    bool sm103;
    int sm_count;
    int smem_optin;
    unsigned long long ctx_id;  // the current context's ID (a device reset makes a new one)
};

int env_device(DeviceEnv *env);                 // LID_OK or LID_ERR_CUDA
int env_cuda_status(cudaError_t e);             // LID_OK, or LID_ERR_CUDA with the error remembered
cudaError_t env_ws_alloc(void **ptr, size_t bytes, cudaStream_t st);

// (lid_attn.cu) the sparse-attention kernels' device-side error word
int attn_device_error(int reset);

}  // namespace lid
