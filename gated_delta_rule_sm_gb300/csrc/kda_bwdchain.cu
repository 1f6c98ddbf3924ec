// kda_bwdchain.cu -- the two state chains of the backward on tcgen05 tensor cores (bf16 inputs,
// K = V = 128), both with tf32 operands rounded to nearest and the state in fp32 registers.
//
// Both are the affine recursion  X = Y_c + A1_c Z,  Z' = Diag(exp(Gamma_last,c)) Z + A2_c X (+ P_c)
// of the chunkwise gated delta rule ("[kimi k3] add eager reference model with FSDP2", chunk_kda):
//   * forward state recompute (REV = false): Z = S entering chunk c, A1 = -W, Y = U0, A2 = Kd^T,
//     so X = U and Z' is the state leaving the chunk;
//   * reverse chain (REV = true): Z = dS, the gradient w.r.t. the state leaving chunk c, A1 = Kd,
//     Y = scale Aqk^T dO, A2 = -W^T, P = scale Qg^T dO, so X = dU and Z' is the gradient entering
//     the chunk.
// The operand copies (records chainrec / bwrec / fwrec) and Y, P come from bwd_pre.  Every product
// runs in split precision, operand = hi + lo (both tf32), hi*hi + hi*lo + lo*hi: the gradient of
// the log-decay at the end of a chunk carries dS_end * S_end-sized terms far larger than its
// typical value, and plain tf32 chains (~2e-4 relative error in S and dS, NumPy emulation and GPU
// measurement agree) put it outside the bf16 tolerance under slowly decaying gates.
//
// One CTA of 128 threads per (segment, head, column slice of JW value columns); the columns of Z
// are independent.  Thread r owns row r of Z.  Per chunk: MMA1 (M = 64, N = JW, K = 128, three
// products) into TMEM, X = D1 + Y split into tf32 hi + lo in shared memory, MMA2 (M = 128, N = JW,
// K = 64, three products), then Z' = gC Z + D3 (+ P).  One record slot per CTA (the split operands
// fill shared memory); the next chunk's slot is copied in as soon as both MMAs are done.
#include "kda_common.cuh"
#include "kda_internal.h"
#include "kda_sm100.cuh"

namespace kda {

using namespace sm100;

namespace bwchain {
template <int JW>
struct Lay {
    static constexpr uint32_t SLOT = chainrec::SLOT;       // record slot at 0 (A1, A2, gC, A1 lo, A2 lo)
    static constexpr uint32_t ZB = SLOT;                   // Z^T tf32 hi, JW rows (j) x 128 K (c): km_f32(j, c, 4096, 128)
    static constexpr uint32_t ZL = ZB + JW * 512;          // Z^T lo
    static constexpr uint32_t XB = ZL + JW * 512;          // X^T tf32 hi, JW rows (j) x 64 K (t): km_f32(j, t, 2048, 128)
    static constexpr uint32_t XL = XB + JW * 256;          // X^T lo
    static constexpr uint32_t BAR = XL + JW * 256;         // mbarriers: full, mma1, mma2; fail flag; TMEM slot
    static constexpr uint32_t BYTES = BAR + 64;
    static constexpr uint32_t TCOLS = 2 * JW;              // D1 at column 0, D3 at column JW
};
}  // namespace bwchain

// 4 x 4 transpose inside each lane quad: on entry lane r holds v[0..3] = row (base + r), columns
// 4b .. 4b + 3; on exit it holds column 4b + r of rows base .. base + 3.
__device__ __forceinline__ void quad_transpose(float& v0, float& v1, float& v2, float& v3, int r) {
    const bool top = (r & 2) == 0, even = (r & 1) == 0;
    const float s0 = top ? v2 : v0, s1 = top ? v3 : v1;
    const float g0 = __shfl_xor_sync(0xffffffffu, s0, 2), g1 = __shfl_xor_sync(0xffffffffu, s1, 2);
    if (top) { v2 = g0; v3 = g1; } else { v0 = g0; v1 = g1; }
    const float e0 = even ? v1 : v0, e1 = even ? v3 : v2;
    const float h0 = __shfl_xor_sync(0xffffffffu, e0, 1), h1 = __shfl_xor_sync(0xffffffffu, e1, 1);
    if (even) { v1 = h0; v3 = h1; } else { v0 = h0; v2 = h1; }
}

// Where a chain finds its per-chunk inputs: slot (A1, A2, gC) of chunk c at slots + (c H + h) *
// slot_stride bytes; Y rows at ybase + (c H + h) * ystride floats (row t, 128 columns); P likewise.
struct ChainSrc {
    const uint8_t* slots;
    size_t slot_stride;
    const float* ybase;
    size_t ystride;
    const float* pbase;   // reverse chain only
    size_t pstride;
};

template <int JW, bool REV>
__global__ void __launch_bounds__(128, 1) chain_tf32_kernel(Params p, ChainSrc src) {
    using L = bwchain::Lay<JW>;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int n = blockIdx.x, h = blockIdx.y, j0 = blockIdx.z * JW;
    const int H = p.H;
    constexpr int K = 128, V = 128;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, r4 = lane & 3;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::BAR);
    uint64_t* bar1 = full + 1;
    uint64_t* bar2 = full + 2;
    int* sh_fail = reinterpret_cast<int*>(full + 3);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(full + 4);
    uint8_t* ZB = smem + L::ZB;
    uint8_t* ZL = smem + L::ZL;
    uint8_t* XB = smem + L::XB;
    uint8_t* XL = smem + L::XL;
    uint8_t* sl = smem;
    const int cb = p.chunk_off[n], ce = p.chunk_off[n + 1];
    const int nch = ce - cb;

    if (tid == 0) {
        for (int i = 0; i < 3; ++i) mbar_init(&full[i], 1);
        *sh_fail = 0;
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(tslot, L::TCOLS);
    float dS[JW];   // row tid of Z (dS for the reverse chain, S for the recompute)
    {
        const float* z0 = REV ? p.dST : p.S0;
        const float* zs = z0 ? z0 + (((size_t)n * H + h) * K + tid) * V + j0 : nullptr;
#pragma unroll
        for (int j = 0; j < JW; j += 4) {
            const float4 v = zs ? *reinterpret_cast<const float4*>(zs + j) : make_float4(0.f, 0.f, 0.f, 0.f);
            dS[j] = v.x; dS[j + 1] = v.y; dS[j + 2] = v.z; dS[j + 3] = v.w;
        }
    }
    auto write_dS_operand = [&]() {
#pragma unroll
        for (int b = 0; b < JW / 4; ++b) {
            float v0 = tf32_rn(dS[4 * b]), v1 = tf32_rn(dS[4 * b + 1]), v2 = tf32_rn(dS[4 * b + 2]),
                  v3 = tf32_rn(dS[4 * b + 3]);
            float l0 = tf32_rn(dS[4 * b] - v0), l1 = tf32_rn(dS[4 * b + 1] - v1), l2 = tf32_rn(dS[4 * b + 2] - v2),
                  l3 = tf32_rn(dS[4 * b + 3] - v3);
            quad_transpose(v0, v1, v2, v3, r4);
            quad_transpose(l0, l1, l2, l3, r4);
            const uint32_t o = km_f32(4 * b + r4, tid - r4, 4096, 128);
            *reinterpret_cast<float4*>(ZB + o) = make_float4(v0, v1, v2, v3);
            *reinterpret_cast<float4*>(ZL + o) = make_float4(l0, l1, l2, l3);
        }
    };
    write_dS_operand();
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t tD1 = tmem, tD3 = tmem + JW;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    // step s handles chunk cb + nch - 1 - s (reverse) or cb + s (forward)
    auto chunk_of = [&](int s) { return REV ? cb + nch - 1 - s : cb + s; };
    auto rec_ptr = [&](int s) { return src.slots + ((size_t)chunk_of(s) * H + h) * src.slot_stride; };
    auto y_ptr = [&](int s) { return src.ybase + ((size_t)chunk_of(s) * H + h) * src.ystride; };
    auto p_ptr = [&](int s) { return src.pbase + ((size_t)chunk_of(s) * H + h) * src.pstride; };
    auto fail_wait = [&](uint64_t* bar, uint32_t parity) {
        if (!mbar_wait(bar, parity)) atomicExch(sh_fail, 1);
    };
    if (tid == 0 && nch > 0) {
        mbar_expect_tx(full, L::SLOT);
        bulk_g2s(sl, rec_ptr(0), L::SLOT, full);
    }

    bool ok = true;
    for (int s = 0; s < nch; ++s) {
        const int c = chunk_of(s);
        const uint32_t par = s & 1;
        {   // reverse: gradient w.r.t. the state leaving chunk c; forward: the state entering chunk c
            float* dst = (REV ? p.dstates : p.states) + (((size_t)c * H + h) * K + tid) * V + j0;
#pragma unroll
            for (int j = 0; j < JW; j += 4)
                *reinterpret_cast<float4*>(dst + j) = make_float4(dS[j], dS[j + 1], dS[j + 2], dS[j + 3]);
        }
        fail_wait(full, par);
        tc_fence_after();
        if (tid == 0) {   // D1 = A1_lo Z_hi + A1_hi Z_lo + A1_hi Z_hi
            const uint32_t a = smem_u32(sl + chainrec::A1), al = smem_u32(sl + chainrec::A1_LO);
            const uint32_t b = smem_u32(ZB), bl = smem_u32(ZL);
            constexpr uint32_t id1 = idesc_tf32(64, JW);
#pragma unroll 1
            for (int kk = 0; kk < 16; ++kk)
                mma_tf32(tD1, smem_desc(al + kk * 256, 128, 4096), smem_desc(b + kk * 256, 128, 4096), id1, kk > 0);
#pragma unroll 1
            for (int kk = 0; kk < 16; ++kk)
                mma_tf32(tD1, smem_desc(a + kk * 256, 128, 4096), smem_desc(bl + kk * 256, 128, 4096), id1, 1);
#pragma unroll 1
            for (int kk = 0; kk < 16; ++kk)
                mma_tf32(tD1, smem_desc(a + kk * 256, 128, 4096), smem_desc(b + kk * 256, 128, 4096), id1, 1);
            mma_commit(bar1);
            if (s + 1 < nch) {   // warm L2 with the next chunk's Y (and P)
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(y_ptr(s + 1))),
                             "r"(64u * V * 4u)
                             : "memory");
                if (REV)
                    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(
                                     reinterpret_cast<uint64_t>(p_ptr(s + 1))),
                                 "r"(128u * V * 4u)
                                 : "memory");
            }
        }
        fail_wait(bar1, par);
        tc_fence_after();
        {
            // dU rows t = 16 warp + lane (lanes 0..15 of each warp carry the M = 64 result)
            const int t = 16 * warp + (lane & 15);
            const float* yrow = y_ptr(s) + t * V + j0;
#pragma unroll
            for (int jb = 0; jb < JW; jb += 32) {
                float d[32];
                tmem_ld16(tD1 + jb + lane_base, d);
                tmem_ld16(tD1 + jb + 16 + lane_base, d + 16);
                float y[32];
#pragma unroll
                for (int j = 0; j < 32; j += 4) {
                    const float4 v = *reinterpret_cast<const float4*>(yrow + jb + j);
                    y[j] = v.x; y[j + 1] = v.y; y[j + 2] = v.z; y[j + 3] = v.w;
                }
                tmem_ld_wait();
#pragma unroll
                for (int b = 0; b < 8; ++b) {
                    const float x0 = d[4 * b] + y[4 * b], x1 = d[4 * b + 1] + y[4 * b + 1],
                                x2 = d[4 * b + 2] + y[4 * b + 2], x3 = d[4 * b + 3] + y[4 * b + 3];
                    float v0 = tf32_rn(x0), v1 = tf32_rn(x1), v2 = tf32_rn(x2), v3 = tf32_rn(x3);
                    const uint32_t o = km_f32(jb + 4 * b + r4, t - r4, 2048, 128);
                    float l0 = tf32_rn(x0 - v0), l1 = tf32_rn(x1 - v1), l2 = tf32_rn(x2 - v2), l3 = tf32_rn(x3 - v3);
                    quad_transpose(l0, l1, l2, l3, r4);
                    quad_transpose(v0, v1, v2, v3, r4);
                    if (lane < 16) {
                        *reinterpret_cast<float4*>(XL + o) = make_float4(l0, l1, l2, l3);
                        *reinterpret_cast<float4*>(XB + o) = make_float4(v0, v1, v2, v3);
                    }
                }
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (*sh_fail) { ok = false; break; }
        if (tid == 0) {   // D3 = A2_lo X_hi + A2_hi X_lo + A2_hi X_hi
            const uint32_t a = smem_u32(sl + chainrec::A2), al = smem_u32(sl + chainrec::A2_LO);
            const uint32_t b = smem_u32(XB), bl = smem_u32(XL);
            constexpr uint32_t id2 = idesc_tf32(128, JW);
#pragma unroll 1
            for (int kk = 0; kk < 8; ++kk)
                mma_tf32(tD3, smem_desc(al + kk * 256, 128, 2048), smem_desc(b + kk * 256, 128, 2048), id2, kk > 0);
#pragma unroll 1
            for (int kk = 0; kk < 8; ++kk)
                mma_tf32(tD3, smem_desc(a + kk * 256, 128, 2048), smem_desc(bl + kk * 256, 128, 2048), id2, 1);
#pragma unroll 1
            for (int kk = 0; kk < 8; ++kk)
                mma_tf32(tD3, smem_desc(a + kk * 256, 128, 2048), smem_desc(b + kk * 256, 128, 2048), id2, 1);
            mma_commit(bar2);
        }
        fail_wait(bar2, par);
        tc_fence_after();
        {
            const float gc = reinterpret_cast<const float*>(sl + chainrec::GC)[tid];
            const float* prow = REV ? p_ptr(s) + tid * V + j0 : nullptr;
#pragma unroll
            for (int jb = 0; jb < JW; jb += 32) {
                float d[32];
                tmem_ld16(tD3 + jb + lane_base, d);
                tmem_ld16(tD3 + jb + 16 + lane_base, d + 16);
                float pv[32];
#pragma unroll
                for (int j = 0; j < 32; j += 4) {
                    const float4 v = REV ? *reinterpret_cast<const float4*>(prow + jb + j) : make_float4(0.f, 0.f, 0.f, 0.f);
                    pv[j] = v.x; pv[j + 1] = v.y; pv[j + 2] = v.z; pv[j + 3] = v.w;
                }
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j) dS[jb + j] = gc * dS[jb + j] + d[j] + pv[j];
            }
            write_dS_operand();
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (*sh_fail) { ok = false; break; }
        // both MMAs of this chunk are complete: the slot takes the next chunk
        if (tid == 0 && s + 1 < nch) {
            mbar_expect_tx(full, L::SLOT);
            bulk_g2s(sl, rec_ptr(s + 1), L::SLOT, full);
        }
    }
    __syncthreads();
    if (*sh_fail) ok = false;
    if (!ok) {
        // Record the timeout; give in-flight copies and MMAs a bounded chance to land before this CTA's
        // shared and tensor memory are released.
        if (tid == 0) {
            record_error(p.status, KDA_ERR_TIMEOUT);
            for (int b = 0; b < 3; ++b) {
                mbar_wait(&full[b], 0, 1u << 12);
                mbar_wait(&full[b], 1, 1u << 12);
            }
        }
    } else if (REV ? p.dS0 != nullptr : p.ST != nullptr) {
        float* dst = (REV ? p.dS0 : p.ST) + (((size_t)n * H + h) * K + tid) * V + j0;
#pragma unroll
        for (int j = 0; j < JW; j += 4)
            *reinterpret_cast<float4*>(dst + j) = make_float4(dS[j], dS[j + 1], dS[j + 2], dS[j + 3]);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, L::TCOLS);
}

template <int JW, bool REV>
static cudaError_t launch_chain_jw(const Params& p, const ChainSrc& src, cudaStream_t st) {
    using L = bwchain::Lay<JW>;
    static_assert(L::BYTES <= 232448, "shared memory per CTA");
    cudaError_t e = cudaFuncSetAttribute(chain_tf32_kernel<JW, REV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)L::BYTES);
    if (e != cudaSuccess) return e;
    timing_pre(st, REV ? K_CHAIN_BWD_TC : K_CHAIN_REC_TC);
    chain_tf32_kernel<JW, REV><<<dim3(p.N, p.H, 128 / JW), 128, L::BYTES, st>>>(p, src);
    timing_post(st);
    return cudaGetLastError();
}

// Column slices per (segment, head) chain: 64 value columns per CTA when the chains fill a third of
// the SMs, otherwise 32 (more parallel, shorter chains steps).
template <bool REV>
static cudaError_t launch_chain(const Params& p, const ChainSrc& src, cudaStream_t st) {
    int sms = 0, dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long chains = (long)p.N * p.H;
    if (chains * 3 >= (long)sms) return launch_chain_jw<64, REV>(p, src, st);
    return launch_chain_jw<32, REV>(p, src, st);
}

cudaError_t launch_chain_bwd_tc(const Params& p, const uint8_t* bw, cudaStream_t st) {
    ChainSrc src{bw, bwrec::BYTES, reinterpret_cast<const float*>(bw + bwrec::Y), bwrec::BYTES / 4,
                 reinterpret_cast<const float*>(bw + bwrec::P), bwrec::BYTES / 4};
    static_assert(bwrec::BYTES % 256 == 0 && fwrec::BYTES % 256 == 0, "record strides");
    return launch_chain<true>(p, src, st);
}

cudaError_t launch_chain_rec_tc(const Params& p, const uint8_t* fw, cudaStream_t st) {
    const RecLayout L = RecLayout::make(128, 128);
    ChainSrc src{fw, fwrec::BYTES, p.rec + L.U0, p.rec_stride, nullptr, 0};
    return launch_chain<false>(p, src, st);
}

}  // namespace kda
