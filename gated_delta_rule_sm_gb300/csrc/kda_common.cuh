// kda_common.cuh -- shared definitions of the KDA CUDA library (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

constexpr int kChunk = 64;      // tokens per chunk
constexpr int kSub = 16;        // tokens per decay sub-block (tensor-core path)
constexpr float kNormEps = 1e-6f;

// Everything a kernel of either path needs, passed by value.
struct Params {
    int B, T, H, K, V, N;       // N = number of segments; H = value heads
    int Hk, G;                  // key heads (q, k) and value heads per key head (H = G * Hk)
    int TT;                     // total tokens B*T
    int dtype;                  // KDA_BF16 / KDA_FP32
    int NCmax;                  // upper bound on the number of chunks
    const void *q, *k, *v, *g_raw, *beta_raw, *dout;
    const float *a_log, *dt_bias, *S0, *dST;
    const int32_t* cu;          // device cu_seqlens or nullptr
    float scale, lb;
    int gate;                   // KDA_GATE_LOWER_BOUNDED / KDA_GATE_SOFTPLUS
    void* out;
    float* ST;
    float *dq, *dk, *dv, *dg_raw, *dbeta_raw, *da_log, *ddt_bias, *dS0;
    float *dq_v, *dk_v;         // dq, dk per value head [TT, H, K]: dq / dk when G == 1, else scratch
                                // that the group sum folds into dq / dk [TT, Hk, K]
    // workspace views
    int32_t* chunk_off;         // [N+1] first chunk of each segment; chunk_off[N] = total chunks; then
                                // [N] the segments in launch order (seg_order)
    float* rec;                 // per (chunk, head) intra-chunk records (SIMT path)
    size_t rec_stride;          // floats per record
    float* states;              // [NCmax, H, K, V] chunk-entering states (backward)
    float* dstates;             // [NCmax, H, K, V] gradient w.r.t. chunk-leaving states (backward)
    float* part_dtb;            // [NCmax, H, K] per-chunk partial d dt_bias
    float* part_alog;           // [NCmax, H]    per-chunk partial d a_log
    float* scratch;             // per-CTA scratch of the SIMT gradient kernel
    size_t scratch_stride;      // floats per CTA
    int grad_ctas;              // CTAs of the SIMT gradient kernel
    void* tc;                   // tensor-core path buffers (its own layout)
    float* chunk_u;             // tensor-core backward: U per (chunk, head) [64][V] fp32, from the recompute chain
    float* chunk_du;            // tensor-core backward: dU per (chunk, head) [64][V] fp32, from the reverse chain
    float* diag;                // tensor-core forward, unbounded gate: diagonal 16 x 16 blocks of Bkk, Aqk per
                                // (chunk, head), from diag_tc_kernel
    int* status;                // device status word
};

// The segments in the order the chain kernels take them (longest first for packed documents), written by
// the planner right after the chunk table.
__host__ __device__ __forceinline__ int32_t* seg_order(const Params& p) { return p.chunk_off + p.N + 1; }

// Device status word (first error wins); `status` points at the library's word on this device.
__device__ __forceinline__ void record_error(int* status, int code) { atomicCAS(status, 0, code); }

__device__ __forceinline__ float load_act(const void* p, size_t i, int dtype) {
    if (dtype == KDA_BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i]);
    return reinterpret_cast<const float*>(p)[i];
}

__device__ __forceinline__ void store_act(void* p, size_t i, float x, int dtype) {
    if (dtype == KDA_BF16) reinterpret_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(x);
    else reinterpret_cast<float*>(p)[i] = x;
}

__device__ __forceinline__ float sigmoidf_acc(float x) { return 1.0f / (1.0f + expf(-x)); }

// log(1 + e^x) without overflow: max(x, 0) + log(1 + e^-|x|)
__device__ __forceinline__ float softplusf(float x) { return fmaxf(x, 0.f) + log1pf(expf(-fabsf(x))); }

// Log-decay of one gate element (the two gate activations of kda.h).
__device__ __forceinline__ float gate_value(const Params& p, float ea, float x, float dtb) {
    return p.gate == KDA_GATE_SOFTPLUS ? -ea * softplusf(x + dtb) : p.lb * sigmoidf_acc(ea * (x + dtb));
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Segment n spans tokens [seg_begin, seg_end) of the flattened B*T axis.
__device__ __forceinline__ int seg_begin(const Params& p, int n) { return p.cu ? p.cu[n] : n * p.T; }
__device__ __forceinline__ int seg_end(const Params& p, int n) { return p.cu ? p.cu[n + 1] : (n + 1) * p.T; }

// Segment owning global chunk c (binary search over chunk_off).
__device__ __forceinline__ int chunk_segment(const Params& p, int c) {
    int lo = 0, hi = p.N - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (p.chunk_off[mid] <= c) lo = mid; else hi = mid - 1;
    }
    return lo;
}

}  // namespace kda
