// kda_noalloc.cu -- kda_fwd_noalloc: the forward with scratch from a static device array.
//
// For callers that may not allocate device memory (see include/kda.h).  The scratch is a
// file-scope __device__ array; host code never uses its name as an address: the device address is
// looked up once per device with cudaGetSymbolAddress and then passed as the workspace of the
// ordinary forward entry point.
#include <mutex>

#include "kda.h"

namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[KDA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mutex;

// Device address of the scratch array on the current device (looked up on first use).
kda_status scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KDA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return KDA_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return KDA_OK;
}

}  // namespace

extern "C" kda_status kda_fwd_noalloc(const kda_dims* dims, const void* q, const void* k, const void* v,
                                      const void* g_raw, const void* beta_raw, const float* a_log,
                                      const float* dt_bias, float scale, float lower_bound, int chunk_size,
                                      const int32_t* cu_seqlens, const int32_t* cu_seqlens_host,
                                      const float* initial_state, void* out, float* final_state,
                                      cudaStream_t stream) {
    if (!dims) return KDA_ERR_INVALID_ARG;
    const size_t need = kda_fwd_workspace_size(dims, chunk_size);
    if (need == 0) {
        // invalid shape: let the ordinary entry point report the precise error
        return kda_fwd(dims, q, k, v, g_raw, beta_raw, a_log, dt_bias, scale, lower_bound, chunk_size, cu_seqlens,
                       cu_seqlens_host, initial_state, out, final_state, nullptr, 0, stream);
    }
    if (need > KDA_NOALLOC_SCRATCH_BYTES) return KDA_ERR_WORKSPACE;
    void* ws = nullptr;
    const kda_status st = scratch_address(&ws);
    if (st != KDA_OK) return st;
    return kda_fwd(dims, q, k, v, g_raw, beta_raw, a_log, dt_bias, scale, lower_bound, chunk_size, cu_seqlens,
                   cu_seqlens_host, initial_state, out, final_state, ws, KDA_NOALLOC_SCRATCH_BYTES, stream);
}
