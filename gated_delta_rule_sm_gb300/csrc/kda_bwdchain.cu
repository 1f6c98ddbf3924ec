// kda_bwdchain.cu -- reverse state chain on tcgen05 tensor cores (bf16 inputs, K = V = 128).
//
// Reverse mode of the chunk recursion of the gated delta rule ("[kimi k3] add eager reference model
// with FSDP2", chunk_kda backward).  With dS the gradient w.r.t. the state leaving chunk c,
//     dU  = Y_c + Kd_c dS                                   (64 x V)
//     dS' = Diag(exp(Gamma_last,c)) dS - W_c^T dU + P_c      (K x V), the gradient entering chunk c,
// where Y_c = scale Aqk^T dO and P_c = scale Qg^T dO do not depend on dS and come
// precomputed in the reverse-chain record (bwrec).  Both products run as kind::tf32 MMAs with
// operands rounded to nearest: the dS chain feeds every gradient, and bf16 operands for Kd dS
// lose about 0.6% of dS under slowly decaying gates.  dS stays in fp32 registers.
//
// One CTA of 128 threads per (segment, head, column slice of JW value columns); the columns of dS
// are independent.  Thread r owns row r of dS.  Per chunk: MMA1 (M = 64, N = JW, K = 128) into
// TMEM, dU = D1 + Y rounded to tf32 into shared memory, MMA2 (M = 128, N = JW, K = 64), then
// dS' = gC dS + D3 + P.  Record slots (Kd, -W^T, gC) are double buffered by bulk copies.
#include "kda_common.cuh"
#include "kda_internal.h"
#include "kda_sm100.cuh"

namespace kda {

using namespace sm100;

namespace bwchain {
template <int JW>
struct Lay {
    static constexpr uint32_t SLOT = bwrec::SLOT;          // two record slots at 0 and SLOT
    static constexpr uint32_t DSB = 2 * SLOT;              // dS^T tf32, JW rows (j) x 128 K (c): km_f32(j, c, 4096, 128)
    static constexpr uint32_t DUB = DSB + JW * 512;        // dU^T tf32, JW rows (j) x 64 K (t): km_f32(j, t, 2048, 128)
    static constexpr uint32_t BAR = DUB + JW * 256;        // mbarriers: full[2], mma1, mma2; fail flag; TMEM slot
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

template <int JW>
__global__ void __launch_bounds__(128, 1) chain_bwd_tc_kernel(Params p, const uint8_t* bw) {
    using L = bwchain::Lay<JW>;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int n = blockIdx.x, h = blockIdx.y, j0 = blockIdx.z * JW;
    const int H = p.H;
    constexpr int K = 128, V = 128;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, r4 = lane & 3;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::BAR);
    uint64_t* bar1 = full + 2;
    uint64_t* bar2 = full + 3;
    int* sh_fail = reinterpret_cast<int*>(full + 4);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(full + 5);
    uint8_t* DSB = smem + L::DSB;
    uint8_t* DUB = smem + L::DUB;
    const int cb = p.chunk_off[n], ce = p.chunk_off[n + 1];
    const int nch = ce - cb;

    if (tid == 0) {
        for (int i = 0; i < 4; ++i) mbar_init(&full[i], 1);
        *sh_fail = 0;
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(tslot, L::TCOLS);
    float dS[JW];
    {
        const float* src = p.dST ? p.dST + (((size_t)n * H + h) * K + tid) * V + j0 : nullptr;
#pragma unroll
        for (int j = 0; j < JW; j += 4) {
            const float4 v = src ? *reinterpret_cast<const float4*>(src + j) : make_float4(0.f, 0.f, 0.f, 0.f);
            dS[j] = v.x; dS[j + 1] = v.y; dS[j + 2] = v.z; dS[j + 3] = v.w;
        }
    }
    auto write_dS_operand = [&]() {
#pragma unroll
        for (int b = 0; b < JW / 4; ++b) {
            float v0 = tf32_rn(dS[4 * b]), v1 = tf32_rn(dS[4 * b + 1]), v2 = tf32_rn(dS[4 * b + 2]),
                  v3 = tf32_rn(dS[4 * b + 3]);
            quad_transpose(v0, v1, v2, v3, r4);
            *reinterpret_cast<float4*>(DSB + km_f32(4 * b + r4, tid - r4, 4096, 128)) = make_float4(v0, v1, v2, v3);
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
    auto slot_ptr = [&](int s) { return smem + (s & 1) * L::SLOT; };
    // step s handles chunk cb + nch - 1 - s
    auto rec_ptr = [&](int s) { return bw + ((size_t)(cb + nch - 1 - s) * H + h) * bwrec::BYTES; };
    auto fail_wait = [&](uint64_t* bar, uint32_t parity) {
        if (!mbar_wait(bar, parity)) atomicExch(sh_fail, 1);
    };
    if (tid == 0)
        for (int s = 0; s < 2 && s < nch; ++s) {
            mbar_expect_tx(&full[s], bwrec::SLOT);
            bulk_g2s(slot_ptr(s), rec_ptr(s), bwrec::SLOT, &full[s]);
        }

    bool ok = true;
    for (int s = 0; s < nch; ++s) {
        const int c = cb + nch - 1 - s;
        uint8_t* sl = slot_ptr(s);
        const uint32_t par = s & 1;
        {   // gradient w.r.t. the state leaving chunk c
            float* dst = p.dstates + (((size_t)c * H + h) * K + tid) * V + j0;
#pragma unroll
            for (int j = 0; j < JW; j += 4)
                *reinterpret_cast<float4*>(dst + j) = make_float4(dS[j], dS[j + 1], dS[j + 2], dS[j + 3]);
        }
        fail_wait(&full[s & 1], (s >> 1) & 1);
        tc_fence_after();
        if (tid == 0) {
            const uint32_t a = smem_u32(sl + bwrec::KDA), b = smem_u32(DSB);
#pragma unroll
            for (int kk = 0; kk < 16; ++kk)
                mma_tf32(tD1, smem_desc(a + kk * 256, 128, 4096), smem_desc(b + kk * 256, 128, 4096),
                         idesc_tf32(64, JW), kk > 0);
            mma_commit(bar1);
            if (s + 1 < nch) {   // warm L2 with the next chunk's Y and P
                const uint8_t* nx = rec_ptr(s + 1) + bwrec::Y;
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(nx)),
                             "r"(bwrec::BYTES - bwrec::Y)
                             : "memory");
            }
        }
        fail_wait(bar1, par);
        tc_fence_after();
        {
            // dU rows t = 16 warp + lane (lanes 0..15 of each warp carry the M = 64 result)
            const int t = 16 * warp + (lane & 15);
            const float* yrow = reinterpret_cast<const float*>(rec_ptr(s) + bwrec::Y) + t * V + j0;
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
                    float v0 = tf32_rn(d[4 * b] + y[4 * b]), v1 = tf32_rn(d[4 * b + 1] + y[4 * b + 1]),
                          v2 = tf32_rn(d[4 * b + 2] + y[4 * b + 2]), v3 = tf32_rn(d[4 * b + 3] + y[4 * b + 3]);
                    quad_transpose(v0, v1, v2, v3, r4);
                    if (lane < 16)
                        *reinterpret_cast<float4*>(DUB + km_f32(jb + 4 * b + r4, t - r4, 2048, 128)) =
                            make_float4(v0, v1, v2, v3);
                }
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (*sh_fail) { ok = false; break; }
        if (tid == 0) {
            const uint32_t a = smem_u32(sl + bwrec::WTN), b = smem_u32(DUB);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_tf32(tD3, smem_desc(a + kk * 256, 128, 2048), smem_desc(b + kk * 256, 128, 2048),
                         idesc_tf32(128, JW), kk > 0);
            mma_commit(bar2);
        }
        fail_wait(bar2, par);
        tc_fence_after();
        {
            const float gc = reinterpret_cast<const float*>(sl + bwrec::GC)[tid];
            const float* prow = reinterpret_cast<const float*>(rec_ptr(s) + bwrec::P) + tid * V + j0;
#pragma unroll
            for (int jb = 0; jb < JW; jb += 32) {
                float d[32];
                tmem_ld16(tD3 + jb + lane_base, d);
                tmem_ld16(tD3 + jb + 16 + lane_base, d + 16);
                float pv[32];
#pragma unroll
                for (int j = 0; j < 32; j += 4) {
                    const float4 v = *reinterpret_cast<const float4*>(prow + jb + j);
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
        // both MMAs of this chunk are complete: the slot takes the chunk two steps ahead
        if (tid == 0 && s + 2 < nch) {
            mbar_expect_tx(&full[s & 1], bwrec::SLOT);
            bulk_g2s(sl, rec_ptr(s + 2), bwrec::SLOT, &full[s & 1]);
        }
    }
    __syncthreads();
    if (*sh_fail) ok = false;
    if (!ok) {
        // Record the timeout; give in-flight copies and MMAs a bounded chance to land before this CTA's
        // shared and tensor memory are released.
        if (tid == 0) {
            record_error(p.status, KDA_ERR_TIMEOUT);
            for (int b = 0; b < 4; ++b) {
                mbar_wait(&full[b], 0, 1u << 12);
                mbar_wait(&full[b], 1, 1u << 12);
            }
        }
    } else if (p.dS0) {
        float* dst = p.dS0 + (((size_t)n * H + h) * K + tid) * V + j0;
#pragma unroll
        for (int j = 0; j < JW; j += 4)
            *reinterpret_cast<float4*>(dst + j) = make_float4(dS[j], dS[j + 1], dS[j + 2], dS[j + 3]);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, L::TCOLS);
}

template <int JW>
static cudaError_t launch_chain_bwd_jw(const Params& p, const uint8_t* bw, cudaStream_t st) {
    using L = bwchain::Lay<JW>;
    cudaError_t e = cudaFuncSetAttribute(chain_bwd_tc_kernel<JW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)L::BYTES);
    if (e != cudaSuccess) return e;
    timing_pre(st, K_CHAIN_BWD_TC);
    chain_bwd_tc_kernel<JW><<<dim3(p.N, p.H, 128 / JW), 128, L::BYTES, st>>>(p, bw);
    timing_post(st);
    return cudaGetLastError();
}

// Column slices per (segment, head) chain: one CTA per chain when the chains alone nearly fill the
// GPU's SMs, otherwise 2 or 4 narrower CTAs (shorter per-step latency, more parallel chains).
cudaError_t launch_chain_bwd_tc(const Params& p, const uint8_t* bw, cudaStream_t st) {
    int sms = 0, dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long chains = (long)p.N * p.H;
    if (chains * 3 >= (long)sms * 2) return launch_chain_bwd_jw<128>(p, bw, st);
    if (chains * 3 >= (long)sms) return launch_chain_bwd_jw<64>(p, bw, st);
    return launch_chain_bwd_jw<32>(p, bw, st);
}

}  // namespace kda
