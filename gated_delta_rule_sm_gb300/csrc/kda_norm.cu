// kda_norm.cu -- the layer's output epilogue: gated RMS norm of each head's value vector.
//
// hyper-parallel "KDA context-parallel executors" (the full-layer adapter's forward) applies
// `o_norm(output, output_gate)` between the attention core and the output projection, and the
// torchtitan review describes the model's RMS norm as one reduced in fp32.  Neither prints the
// formula; the reading (the oracle's too) is, per row of V values (one token of one head),
//     y_v = o_v / sqrt(mean_u o_u^2 + eps) * w_v * sigmoid(gate_v),
// with the sum of squares in fp32.
//
// Memory-bound: one read of o and gate, one write of y (forward); reads of o, gate, dy and fp32
// writes of do, dgate (backward).  One warp per row, grid-stride over rows.  bf16 rows of 128 or 256
// values take the vector kernels (a lane owns 4 consecutive values of each 128: 8-byte loads and
// stores); other shapes the general ones, where a lane owns the values lane, lane + 32, ... (V <= 256,
// at most 8 per lane).  The backward keeps per-CTA partial sums of dweight, which a second kernel adds
// in CTA order (deterministic).
#include <math.h>
#include <string.h>

#include "kda.h"
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {

namespace {

constexpr int kNormMaxV = 256;
constexpr int kNormPer = kNormMaxV / 32;   // values per lane
constexpr int kNormThreads = 256;          // eight rows in flight per CTA
constexpr int kNormBwdCtas = 608;          // four per SM: rows of the dweight partials

struct NormArgs {
    long long rows;
    int V, dtype;
    const void* o;
    const void* gate;
    const float* w;
    float eps;
    void* y;            // forward output (dtype)
    const void* dy;     // backward input (dtype)
    float* d_o;         // [rows, V]
    float* dgate;       // [rows, V]
    float* part;        // [ctas, V] per-CTA partial sums of dweight
    float* dw;          // [V]
};

__global__ void __launch_bounds__(kNormThreads) gated_norm_fwd_kernel(NormArgs a) {
    const int lane = threadIdx.x & 31;
    const long long nw = (long long)gridDim.x * (kNormThreads / 32);
    float wv[kNormPer];
#pragma unroll
    for (int i = 0; i < kNormPer; ++i) {
        const int v = lane + 32 * i;
        wv[i] = v < a.V ? a.w[v] : 0.f;
    }
    for (long long r = (long long)blockIdx.x * (kNormThreads / 32) + (threadIdx.x >> 5); r < a.rows; r += nw) {
        const size_t base = (size_t)r * a.V;
        float ov[kNormPer], gv[kNormPer];
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < kNormPer; ++i) {
            const int v = lane + 32 * i;
            ov[i] = v < a.V ? load_act(a.o, base + v, a.dtype) : 0.f;
            gv[i] = v < a.V ? load_act(a.gate, base + v, a.dtype) : 0.f;
            ss += ov[i] * ov[i];
        }
        ss = warp_sum(ss);
        const float rn = 1.0f / sqrtf(ss / a.V + a.eps);
#pragma unroll
        for (int i = 0; i < kNormPer; ++i) {
            const int v = lane + 32 * i;
            if (v < a.V) store_act(a.y, base + v, ov[i] * rn * wv[i] * sigmoidf_acc(gv[i]), a.dtype);
        }
    }
}

// With n = o rn and s = sigmoid(gate):  dgate = dy n w s (1 - s),  dw += dy n s,  dn = dy w s,
// do = rn (dn - n mean(dn n)).
__global__ void __launch_bounds__(kNormThreads) gated_norm_bwd_kernel(NormArgs a) {
    __shared__ float sdw[kNormThreads / 32][kNormMaxV];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const long long nw = (long long)gridDim.x * (kNormThreads / 32);
    float wv[kNormPer], acc[kNormPer];
#pragma unroll
    for (int i = 0; i < kNormPer; ++i) {
        const int v = lane + 32 * i;
        wv[i] = v < a.V ? a.w[v] : 0.f;
        acc[i] = 0.f;
    }
    for (long long r = (long long)blockIdx.x * (kNormThreads / 32) + warp; r < a.rows; r += nw) {
        const size_t base = (size_t)r * a.V;
        float ov[kNormPer], sv[kNormPer], dyv[kNormPer];
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < kNormPer; ++i) {
            const int v = lane + 32 * i;
            const bool in = v < a.V;
            ov[i] = in ? load_act(a.o, base + v, a.dtype) : 0.f;
            sv[i] = in ? sigmoidf_acc(load_act(a.gate, base + v, a.dtype)) : 0.f;
            dyv[i] = in ? load_act(a.dy, base + v, a.dtype) : 0.f;
            ss += ov[i] * ov[i];
        }
        ss = warp_sum(ss);
        const float rn = 1.0f / sqrtf(ss / a.V + a.eps);
        float dot = 0.f;
#pragma unroll
        for (int i = 0; i < kNormPer; ++i) dot += dyv[i] * wv[i] * sv[i] * (ov[i] * rn);
        dot = warp_sum(dot) / a.V;
#pragma unroll
        for (int i = 0; i < kNormPer; ++i) {
            const int v = lane + 32 * i;
            if (v < a.V) {
                const float n = ov[i] * rn, dn = dyv[i] * wv[i] * sv[i];
                a.d_o[base + v] = rn * (dn - n * dot);
                a.dgate[base + v] = dyv[i] * n * wv[i] * sv[i] * (1.f - sv[i]);
                acc[i] += dyv[i] * n * sv[i];
            }
        }
    }
#pragma unroll
    for (int i = 0; i < kNormPer; ++i) {
        const int v = lane + 32 * i;
        if (v < a.V) sdw[warp][v] = acc[i];
    }
    __syncthreads();
    for (int v = threadIdx.x; v < a.V; v += kNormThreads) {
        float t = 0.f;
#pragma unroll
        for (int w = 0; w < kNormThreads / 32; ++w) t += sdw[w][v];
        a.part[(size_t)blockIdx.x * a.V + v] = t;
    }
}

// Fast path for bf16 rows of 128 or 256 values (NV = V / 128): a lane owns 4 consecutive values of each
// 128, so every access is one 8-byte load or store (bf16) or one 16-byte store (fp32) per lane and a
// row takes 3-5 memory instructions per warp instead of 3-5 per value.  Same arithmetic per value as
// the general kernels except the sigmoid (fast exponential and divide) and the order of the fp32 row
// sums.
// sigmoid with the fast exponential and divide (a few ulp): the forward rounds to bf16 and the backward's
// fp32 gradients are held to 1e-4 relative, so the accurate forms only cost issue slots here
__device__ __forceinline__ float sigmoid_fast(float x) { return __fdividef(1.f, 1.f + __expf(-x)); }

__device__ __forceinline__ void ld4_bf16(const void* p, size_t off, float* f) {
    const uint2 u = *reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(p) + off);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
    f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
}

__device__ __forceinline__ void st4_bf16(void* p, size_t off, const float* f) {
    __nv_bfloat162 a = __floats2bfloat162_rn(f[0], f[1]), b = __floats2bfloat162_rn(f[2], f[3]);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t*>(&a);
    u.y = *reinterpret_cast<const uint32_t*>(&b);
    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p) + off) = u;
}

template <int NV>
__global__ void __launch_bounds__(kNormThreads) gated_norm_fwd_vec_kernel(NormArgs a) {
    const int lane = threadIdx.x & 31;
    const long long nw = (long long)gridDim.x * (kNormThreads / 32);
    float wv[NV][4];
#pragma unroll
    for (int i = 0; i < NV; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) wv[i][e] = a.w[128 * i + 4 * lane + e];
    for (long long r = (long long)blockIdx.x * (kNormThreads / 32) + (threadIdx.x >> 5); r < a.rows; r += nw) {
        const size_t base = (size_t)r * a.V + 4 * lane;
        float ov[NV][4], gv[NV][4];
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            ld4_bf16(a.o, base + 128 * i, ov[i]);
            ld4_bf16(a.gate, base + 128 * i, gv[i]);
#pragma unroll
            for (int e = 0; e < 4; ++e) ss += ov[i][e] * ov[i][e];
        }
        ss = warp_sum(ss);
        const float rn = 1.0f / sqrtf(ss / a.V + a.eps);
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            float y[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) y[e] = ov[i][e] * rn * wv[i][e] * sigmoid_fast(gv[i][e]);
            st4_bf16(a.y, base + 128 * i, y);
        }
    }
}

template <int NV>
__global__ void __launch_bounds__(kNormThreads) gated_norm_bwd_vec_kernel(NormArgs a) {
    __shared__ float sdw[kNormThreads / 32][kNormMaxV];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const long long nw = (long long)gridDim.x * (kNormThreads / 32);
    float wv[NV][4], acc[NV][4];
#pragma unroll
    for (int i = 0; i < NV; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            wv[i][e] = a.w[128 * i + 4 * lane + e];
            acc[i][e] = 0.f;
        }
    for (long long r = (long long)blockIdx.x * (kNormThreads / 32) + warp; r < a.rows; r += nw) {
        const size_t base = (size_t)r * a.V + 4 * lane;
        float ov[NV][4], sv[NV][4], dyv[NV][4];
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            ld4_bf16(a.o, base + 128 * i, ov[i]);
            ld4_bf16(a.gate, base + 128 * i, sv[i]);
            ld4_bf16(a.dy, base + 128 * i, dyv[i]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                sv[i][e] = sigmoid_fast(sv[i][e]);
                ss += ov[i][e] * ov[i][e];
            }
        }
        ss = warp_sum(ss);
        const float rn = 1.0f / sqrtf(ss / a.V + a.eps);
        float dot = 0.f;
#pragma unroll
        for (int i = 0; i < NV; ++i)
#pragma unroll
            for (int e = 0; e < 4; ++e) dot += dyv[i][e] * wv[i][e] * sv[i][e] * (ov[i][e] * rn);
        dot = warp_sum(dot) / a.V;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            float d4[4], g4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float n = ov[i][e] * rn, dn = dyv[i][e] * wv[i][e] * sv[i][e];
                d4[e] = rn * (dn - n * dot);
                g4[e] = dyv[i][e] * n * wv[i][e] * sv[i][e] * (1.f - sv[i][e]);
                acc[i][e] += dyv[i][e] * n * sv[i][e];
            }
            *reinterpret_cast<float4*>(a.d_o + base + 128 * i) = make_float4(d4[0], d4[1], d4[2], d4[3]);
            *reinterpret_cast<float4*>(a.dgate + base + 128 * i) = make_float4(g4[0], g4[1], g4[2], g4[3]);
        }
    }
#pragma unroll
    for (int i = 0; i < NV; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) sdw[warp][128 * i + 4 * lane + e] = acc[i][e];
    __syncthreads();
    for (int v = threadIdx.x; v < a.V; v += kNormThreads) {
        float t = 0.f;
#pragma unroll
        for (int w = 0; w < kNormThreads / 32; ++w) t += sdw[w][v];
        a.part[(size_t)blockIdx.x * a.V + v] = t;
    }
}

__global__ void gated_norm_reduce_kernel(NormArgs a, int ctas) {
    const int v = blockIdx.x * blockDim.x + threadIdx.x;
    if (v >= a.V) return;
    float t = 0.f;
    for (int c = 0; c < ctas; ++c) t += a.part[(size_t)c * a.V + v];
    a.dw[v] = t;
}

kda_status norm_check(int64_t rows, int V, int dtype, const void* o, const void* gate, const float* w, float eps) {
    if (rows < 1 || V < 1) return KDA_ERR_INVALID_ARG;
    if (dtype != KDA_BF16 && dtype != KDA_FP32) return KDA_ERR_INVALID_ARG;
    if (!o || !gate || !w) return KDA_ERR_INVALID_ARG;
    // eps > 0: with eps = 0 an all-zero row would give 0 * inf = NaN in y, do and dgate
    if (!(eps > 0.f) || !isfinite(eps)) return KDA_ERR_INVALID_ARG;
    if (V > kNormMaxV) return KDA_ERR_UNSUPPORTED;
    if (rows > (1LL << 40) / V) return KDA_ERR_UNSUPPORTED;
    return KDA_OK;
}

NormArgs norm_args(int64_t rows, int V, int dtype, const void* o, const void* gate, const float* w, float eps) {
    NormArgs a;
    memset(&a, 0, sizeof(a));
    a.rows = rows; a.V = V; a.dtype = dtype; a.o = o; a.gate = gate; a.w = w; a.eps = eps;
    return a;
}

// The vector kernels' accesses: 8-byte bf16 loads and stores, 16-byte fp32 stores.
bool norm_vec_ok(const NormArgs& a) {
    auto al = [](const void* x, uintptr_t b) { return x == nullptr || (reinterpret_cast<uintptr_t>(x) % b) == 0; };
    return a.dtype == KDA_BF16 && (a.V == 128 || a.V == 256) && al(a.o, 8) && al(a.gate, 8) && al(a.y, 8) &&
           al(a.dy, 8) && al(a.d_o, 16) && al(a.dgate, 16);
}

int norm_ctas(int64_t rows, int cap) {
    const int64_t need = (rows + kNormThreads / 32 - 1) / (kNormThreads / 32);
    return (int)(need < cap ? need : cap);
}

}  // namespace

}  // namespace kda

using namespace kda;

extern "C" {

kda_status kda_gated_norm_fwd(int64_t rows, int V, kda_dtype dtype, const void* o, const void* gate,
                              const float* weight, float eps, void* y, cudaStream_t stream) {
    kda_status st = norm_check(rows, V, dtype, o, gate, weight, eps);
    if (st != KDA_OK) return st;
    if (!y) return KDA_ERR_INVALID_ARG;
    NormArgs a = norm_args(rows, V, dtype, o, gate, weight, eps);
    a.y = y;
    timing_pre(stream, K_NORM_FWD);
    const int ctas = norm_ctas(rows, 8 * 152);
    if (!norm_vec_ok(a)) gated_norm_fwd_kernel<<<ctas, kNormThreads, 0, stream>>>(a);
    else if (V == 128) gated_norm_fwd_vec_kernel<1><<<ctas, kNormThreads, 0, stream>>>(a);
    else gated_norm_fwd_vec_kernel<2><<<ctas, kNormThreads, 0, stream>>>(a);
    timing_post(stream);
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

size_t kda_gated_norm_bwd_workspace_size(int64_t rows, int V) {
    if (rows < 1 || V < 1 || V > kNormMaxV) return 0;
    return ((size_t)kNormBwdCtas * V * sizeof(float) + 255) / 256 * 256;
}

kda_status kda_gated_norm_bwd(int64_t rows, int V, kda_dtype dtype, const void* o, const void* gate,
                              const float* weight, float eps, const void* dy, float* d_o, float* dgate,
                              float* dweight, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    kda_status st = norm_check(rows, V, dtype, o, gate, weight, eps);
    if (st != KDA_OK) return st;
    if (!dy || !d_o || !dgate || !dweight) return KDA_ERR_INVALID_ARG;
    const size_t need = kda_gated_norm_bwd_workspace_size(rows, V);
    if (workspace_bytes < need || !workspace || reinterpret_cast<uintptr_t>(workspace) % 256) return KDA_ERR_WORKSPACE;
    NormArgs a = norm_args(rows, V, dtype, o, gate, weight, eps);
    a.dy = dy; a.d_o = d_o; a.dgate = dgate; a.dw = dweight;
    a.part = static_cast<float*>(workspace);
    const int ctas = norm_ctas(rows, kNormBwdCtas);
    timing_pre(stream, K_NORM_BWD);
    if (!norm_vec_ok(a)) gated_norm_bwd_kernel<<<ctas, kNormThreads, 0, stream>>>(a);
    else if (V == 128) gated_norm_bwd_vec_kernel<1><<<ctas, kNormThreads, 0, stream>>>(a);
    else gated_norm_bwd_vec_kernel<2><<<ctas, kNormThreads, 0, stream>>>(a);
    timing_post(stream);
    if (cudaGetLastError() != cudaSuccess) return KDA_ERR_CUDA;
    timing_pre(stream, K_NORM_REDUCE);
    gated_norm_reduce_kernel<<<(V + 255) / 256, 256, 0, stream>>>(a, ctas);
    timing_post(stream);
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // extern "C"
