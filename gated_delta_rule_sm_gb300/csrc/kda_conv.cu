// kda_conv.cu -- the layer's q/k/v prologue: causal depthwise short convolution + SiLU.
//
// hyper-parallel "KDA context-parallel executors" (`_run_causal_short_conv`, `_local_short_conv`,
// `_validate_layer_short_conv`): each projection passes through a depthwise Conv1d (groups =
// channels, stride 1, dilation 1, kernel_size - 1 zero padding on the left, output cut to the input
// length) and SiLU:
//     a[t, c] = bias[c] + sum_{i < W} weight[c, i] x[t - (W - 1) + i, c],    y = a * sigmoid(a)
// With packed documents every segment starts from zero history.
//
// Memory-bound: one pass over x and y (forward), x, dy and dx (backward).  A thread owns eight
// consecutive channels (one 16-byte bf16 vector) over a tile of tokens and slides a window of the
// last W - 1 inputs in registers, so every element is read once; a warp covers 256 consecutive
// channels of a token row, so each access is a full 512-byte row segment.
#include <string.h>

#include "kda.h"
#include "kda_common.cuh"
#include "kda_internal.h"
#include "kda_sm100.cuh"

namespace kda {

using namespace sm100;

namespace {

constexpr int kConvMaxW = 8;
constexpr int kConvTile = 64;       // tokens per CTA row tile
constexpr int kConvThreads = 128;   // x 8 channels = 1024 channels per CTA

struct ConvArgs {
    int TT, T, C, W, dtype, N;
    const void* x;
    const float* w;        // [C, W]
    const float* b;        // [C] or nullptr
    const int32_t* cu;     // [N + 1] or nullptr
    void* y;               // forward output (dtype)
    const void* dy;        // backward input (dtype)
    float* dx;             // [TT, C]
    float* part;           // backward partial sums [tiles][C][W + 1] (weight taps, then bias)
    float* dw;             // [C, W]
    float* db;             // [C] or nullptr
};

__device__ __forceinline__ void load8(const void* p, size_t i, int dtype, float* v) {
    if (dtype == KDA_BF16) {
        const uint4 u = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p) + i);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            v[2 * k] = __uint_as_float(w[k] << 16);
            v[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
        }
    } else {
        const float4 a = *reinterpret_cast<const float4*>(static_cast<const float*>(p) + i);
        const float4 b = *reinterpret_cast<const float4*>(static_cast<const float*>(p) + i + 4);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
}

__device__ __forceinline__ void store8(void* p, size_t i, int dtype, const float* v) {
    if (dtype == KDA_BF16) {
        *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p) + i) = pack8_bf16(v);
    } else {
        *reinterpret_cast<float4*>(static_cast<float*>(p) + i) = make_float4(v[0], v[1], v[2], v[3]);
        *reinterpret_cast<float4*>(static_cast<float*>(p) + i + 4) = make_float4(v[4], v[5], v[6], v[7]);
    }
}

__device__ __forceinline__ void store8f(float* p, size_t i, const float* v) {
    *reinterpret_cast<float4*>(p + i) = make_float4(v[0], v[1], v[2], v[3]);
    *reinterpret_cast<float4*>(p + i + 4) = make_float4(v[4], v[5], v[6], v[7]);
}

// Start of the segment holding token t and the start of the next one.
__device__ __forceinline__ void segment_of(const ConvArgs& a, int t, int& s0, int& s1) {
    if (!a.cu) {
        s0 = t / a.T * a.T;
        s1 = s0 + a.T;
        return;
    }
    int lo = 0, hi = a.N - 1;   // last n with cu[n] <= t
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.cu[mid] <= t) lo = mid; else hi = mid - 1;
    }
    s0 = a.cu[lo];
    s1 = a.cu[lo + 1];
}

template <int W>
__global__ void __launch_bounds__(kConvThreads) conv_fwd_kernel(ConvArgs a) {
    const int c0 = (blockIdx.x * kConvThreads + threadIdx.x) * 8;
    if (c0 >= a.C) return;
    const int t0 = blockIdx.y * kConvTile, t1 = min(t0 + kConvTile, a.TT);
    float w[8][W], bias[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        bias[e] = a.b ? a.b[c0 + e] : 0.f;
#pragma unroll
        for (int i = 0; i < W; ++i) w[e][i] = a.w[(size_t)(c0 + e) * W + i];
    }
    int s0, s1;
    segment_of(a, t0, s0, s1);
    float win[W][8];   // win[i] = x[t - (W - 1) + i]; the last slot is filled with the current token
#pragma unroll
    for (int i = 0; i < W - 1; ++i) {
        const int tau = t0 - (W - 1) + i;
        if (tau >= s0) load8(a.x, (size_t)tau * a.C + c0, a.dtype, win[i]);
        else
#pragma unroll
            for (int e = 0; e < 8; ++e) win[i][e] = 0.f;
    }
    for (int t = t0; t < t1; ++t) {
        if (t == s1) {   // a new segment starts: zero history
            segment_of(a, t, s0, s1);
#pragma unroll
            for (int i = 0; i < W - 1; ++i)
#pragma unroll
                for (int e = 0; e < 8; ++e) win[i][e] = 0.f;
        }
        load8(a.x, (size_t)t * a.C + c0, a.dtype, win[W - 1]);
        float y[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            float acc = bias[e];
#pragma unroll
            for (int i = 0; i < W; ++i) acc = fmaf(w[e][i], win[i][e], acc);
            y[e] = acc * __fdividef(1.f, 1.f + __expf(-acc));
        }
        store8(a.y, (size_t)t * a.C + c0, a.dtype, y);
#pragma unroll
        for (int i = 0; i < W - 1; ++i)
#pragma unroll
            for (int e = 0; e < 8; ++e) win[i][e] = win[i + 1][e];
    }
}

// Backward over a tile: da[t] for t in [t0, t1 + W - 1) (the look-ahead feeds dx of the tile's last
// tokens), scattered into a ring of the W pending dx rows; a row is final (and stored) once the
// token W - 1 after it has been processed.  The weight / bias partial sums take t in [t0, t1) only.
template <int W>
__global__ void __launch_bounds__(kConvThreads) conv_bwd_kernel(ConvArgs a) {
    const int c0 = (blockIdx.x * kConvThreads + threadIdx.x) * 8;
    if (c0 >= a.C) return;
    const int t0 = blockIdx.y * kConvTile, t1 = min(t0 + kConvTile, a.TT);
    const int tend = min(t1 + W - 1, a.TT);
    float w[8][W], bias[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        bias[e] = a.b ? a.b[c0 + e] : 0.f;
#pragma unroll
        for (int i = 0; i < W; ++i) w[e][i] = a.w[(size_t)(c0 + e) * W + i];
    }
    int s0, s1;
    segment_of(a, t0, s0, s1);
    float win[W][8], ring[W][8], pw[8][W], pb[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        pb[e] = 0.f;
#pragma unroll
        for (int i = 0; i < W; ++i) pw[e][i] = 0.f;
    }
#pragma unroll
    for (int i = 0; i < W; ++i)
#pragma unroll
        for (int e = 0; e < 8; ++e) ring[i][e] = 0.f;   // ring[i] = dx[t - (W - 1) + i]
#pragma unroll
    for (int i = 0; i < W - 1; ++i) {
        const int tau = t0 - (W - 1) + i;
        if (tau >= s0) load8(a.x, (size_t)tau * a.C + c0, a.dtype, win[i]);
        else
#pragma unroll
            for (int e = 0; e < 8; ++e) win[i][e] = 0.f;
    }
    for (int t = t0; t < tend; ++t) {
        if (t == s1) {
            segment_of(a, t, s0, s1);
#pragma unroll
            for (int i = 0; i < W - 1; ++i)
#pragma unroll
                for (int e = 0; e < 8; ++e) win[i][e] = 0.f;
        }
        load8(a.x, (size_t)t * a.C + c0, a.dtype, win[W - 1]);
        float g[8];
        load8(a.dy, (size_t)t * a.C + c0, a.dtype, g);
        const bool own = t < t1;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            float acc = bias[e];
#pragma unroll
            for (int i = 0; i < W; ++i) acc = fmaf(w[e][i], win[i][e], acc);
            const float s = __fdividef(1.f, 1.f + __expf(-acc));
            const float da = g[e] * s * (1.f + acc * (1.f - s));
#pragma unroll
            for (int i = 0; i < W; ++i) {
                // taps before the segment start do not exist: no dx there, and win[i] is zero
                if (t - (W - 1) + i >= s0) ring[i][e] = fmaf(w[e][i], da, ring[i][e]);
                if (own) pw[e][i] = fmaf(win[i][e], da, pw[e][i]);
            }
            if (own) pb[e] += da;
        }
        // no later token reaches back to t - (W - 1): its dx is complete
        const int tau = t - (W - 1);
        if (tau >= t0) store8f(a.dx, (size_t)tau * a.C + c0, ring[0]);
#pragma unroll
        for (int i = 0; i < W - 1; ++i)
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                win[i][e] = win[i + 1][e];
                ring[i][e] = ring[i + 1][e];
            }
#pragma unroll
        for (int e = 0; e < 8; ++e) ring[W - 1][e] = 0.f;
    }
    // rows the look-ahead did not reach (the end of the tokens): their dx is complete now
    for (int tau = max(tend - (W - 1), t0); tau < t1; ++tau) {
        const int k = tau - (tend - (W - 1));
        float v[8];
#pragma unroll
        for (int i = 0; i < W; ++i)
            if (i == k)
#pragma unroll
                for (int e = 0; e < 8; ++e) v[e] = ring[i][e];
        store8f(a.dx, (size_t)tau * a.C + c0, v);
    }
    float* pp = a.part + ((size_t)blockIdx.y * a.C + c0) * (W + 1);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
#pragma unroll
        for (int i = 0; i < W; ++i) pp[e * (W + 1) + i] = pw[e][i];
        pp[e * (W + 1) + W] = pb[e];
    }
}

// dweight / dbias: sum the per-tile partials in tile order (deterministic).
__global__ void conv_reduce_kernel(ConvArgs a, int tiles) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    const int per = a.W + 1;
    if (i >= a.C * per) return;
    float s = 0.f;
    for (int k = 0; k < tiles; ++k) s += a.part[(size_t)k * a.C * per + i];
    const int c = i / per, j = i - c * per;
    if (j < a.W) a.dw[(size_t)c * a.W + j] = s;
    else if (a.db) a.db[c] = s;
}

// ------------------------------------------------------------------ C ABI helpers

kda_status conv_check(int B, int T, int C, int W, int dtype, const int32_t* cu, int num_seqs, const void* x,
                      const float* weight) {
    if (B < 1 || T < 1 || C < 1 || W < 1) return KDA_ERR_INVALID_ARG;
    if (dtype != KDA_BF16 && dtype != KDA_FP32) return KDA_ERR_INVALID_ARG;
    if (!x || !weight) return KDA_ERR_INVALID_ARG;
    if (cu && (B != 1 || num_seqs < 1)) return KDA_ERR_INVALID_ARG;
    if (W > kConvMaxW || C % 8) return KDA_ERR_UNSUPPORTED;
    if ((long long)B * T > (1LL << 30) || (long long)B * T * C > (1LL << 40)) return KDA_ERR_UNSUPPORTED;
    if (reinterpret_cast<uintptr_t>(x) % 16) return KDA_ERR_UNSUPPORTED;   // 8-channel vector accesses
    return KDA_OK;
}

ConvArgs conv_args(int B, int T, int C, int W, int dtype, const int32_t* cu, int num_seqs, const void* x,
                   const float* weight, const float* bias) {
    ConvArgs a;
    memset(&a, 0, sizeof(a));
    a.TT = B * T; a.T = T; a.C = C; a.W = W; a.dtype = dtype; a.N = cu ? num_seqs : B;
    a.x = x; a.w = weight; a.b = bias; a.cu = cu;
    return a;
}

dim3 conv_grid(const ConvArgs& a) {
    return dim3((a.C / 8 + kConvThreads - 1) / kConvThreads, (a.TT + kConvTile - 1) / kConvTile);
}

}  // namespace

#define KDA_CONV_DISPATCH(KERNEL, a, grid, st)                                               \
    switch ((a).W) {                                                                         \
        case 1: KERNEL<1><<<grid, kConvThreads, 0, st>>>(a); break;                          \
        case 2: KERNEL<2><<<grid, kConvThreads, 0, st>>>(a); break;                          \
        case 3: KERNEL<3><<<grid, kConvThreads, 0, st>>>(a); break;                          \
        case 4: KERNEL<4><<<grid, kConvThreads, 0, st>>>(a); break;                          \
        case 5: KERNEL<5><<<grid, kConvThreads, 0, st>>>(a); break;                          \
        case 6: KERNEL<6><<<grid, kConvThreads, 0, st>>>(a); break;                          \
        case 7: KERNEL<7><<<grid, kConvThreads, 0, st>>>(a); break;                          \
        default: KERNEL<8><<<grid, kConvThreads, 0, st>>>(a); break;                         \
    }

}  // namespace kda

using namespace kda;

extern "C" {

kda_status kda_short_conv_fwd(int B, int T, int C, int W, kda_dtype dtype, const void* x, const float* weight,
                              const float* bias, const int32_t* cu_seqlens, int num_seqs, void* y,
                              cudaStream_t stream) {
    kda_status st = conv_check(B, T, C, W, dtype, cu_seqlens, num_seqs, x, weight);
    if (st != KDA_OK) return st;
    if (!y) return KDA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(y) % 16) return KDA_ERR_UNSUPPORTED;
    ConvArgs a = conv_args(B, T, C, W, dtype, cu_seqlens, num_seqs, x, weight, bias);
    a.y = y;
    timing_pre(stream, K_CONV_FWD);
    KDA_CONV_DISPATCH(conv_fwd_kernel, a, conv_grid(a), stream);
    timing_post(stream);
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

size_t kda_short_conv_bwd_workspace_size(int B, int T, int C, int W) {
    if (B < 1 || T < 1 || C < 1 || W < 1 || W > kConvMaxW) return 0;
    const size_t tiles = ((size_t)B * T + kConvTile - 1) / kConvTile;
    return (tiles * C * (W + 1) * sizeof(float) + 255) / 256 * 256;
}

kda_status kda_short_conv_bwd(int B, int T, int C, int W, kda_dtype dtype, const void* x, const float* weight,
                              const float* bias, const int32_t* cu_seqlens, int num_seqs, const void* dy,
                              float* dx, float* dweight, float* dbias, void* workspace, size_t workspace_bytes,
                              cudaStream_t stream) {
    kda_status st = conv_check(B, T, C, W, dtype, cu_seqlens, num_seqs, x, weight);
    if (st != KDA_OK) return st;
    if (!dy || !dx || !dweight || (bias && !dbias)) return KDA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(dy) % 16 || reinterpret_cast<uintptr_t>(dx) % 16) return KDA_ERR_UNSUPPORTED;
    const size_t need = kda_short_conv_bwd_workspace_size(B, T, C, W);
    if (workspace_bytes < need || !workspace || reinterpret_cast<uintptr_t>(workspace) % 256) return KDA_ERR_WORKSPACE;
    ConvArgs a = conv_args(B, T, C, W, dtype, cu_seqlens, num_seqs, x, weight, bias);
    a.dy = dy; a.dx = dx; a.dw = dweight; a.db = bias ? dbias : nullptr;
    a.part = static_cast<float*>(workspace);
    const dim3 g = conv_grid(a);
    timing_pre(stream, K_CONV_BWD);
    KDA_CONV_DISPATCH(conv_bwd_kernel, a, g, stream);
    timing_post(stream);
    if (cudaGetLastError() != cudaSuccess) return KDA_ERR_CUDA;
    const int outs = C * (W + 1);
    timing_pre(stream, K_CONV_REDUCE);
    conv_reduce_kernel<<<(outs + 255) / 256, 256, 0, stream>>>(a, (int)g.y);
    timing_post(stream);
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // extern "C"
