// kda_tc.cu -- tensor-core (tcgen05 / TMEM) path for bf16 inputs with K = V = 128.
//
// Same chunkwise algebra as the SIMT path (the gated delta rule of "[kimi k3] add eager reference
// model with FSDP2", 64 tokens per chunk):
//     U = U0 - W S,   O = scale (Qg S + Aqk U),   S' = Diag(exp(Gamma_last)) S + Kd^T U.
// Precision plan (bf16 inputs, fp32 state): the products whose rounding reaches the outputs least
// run with bf16 operands (W S, Qg S: kind::f16); the ones that feed the state or the output
// directly (Aqk U, Kd^T U) run with tf32 operands rounded to nearest (kind::tf32); U0 is added in
// fp32.  The state itself stays in fp32 registers.
//
// The intra-chunk kernel writes one record per (chunk, head) in exactly the shared-memory layout
// the chain kernel's MMAs read, so the chain moves it with three bulk copies per chunk.
#include "kda_common.cuh"
#include "kda_internal.h"
#include "kda_sm100.cuh"

namespace kda {

using namespace sm100;

// ------------------------------------------------------------------ record layout (bytes)
namespace tcrec {
constexpr uint32_t WQ = 0;            // [W; Qg]  bf16  128 rows x 128 K, K-major, SBO 2048
constexpr uint32_t U0 = 32768;        // U0       fp32  4 slices x (64 rows x 32 cols), K-major core, SBO 1024
constexpr uint32_t KD = 65536;        // Kd^T     tf32  128 rows (c) x 64 K (t), K-major, SBO 2048
constexpr uint32_t AQ = 98304;        // Aqk      tf32  64 rows (t) x 64 K (s), K-major, SBO 2048
constexpr uint32_t GC = 114688;       // exp(Gamma_last) fp32 [128]
constexpr uint32_t BYTES = 115712;    // record stride (1 KB aligned)
constexpr uint32_t U0_SLICE = 8192;   // one 32-column slice of U0
constexpr uint32_t TAIL = BYTES - KD; // KD + AQ + GC, contiguous
}  // namespace tcrec

// K-major core-matrix offsets: bf16 (8 elements per 16 B row) and 32-bit (4 per row).
__host__ __device__ __forceinline__ uint32_t off_bf16(int r, int k, uint32_t sbo) {
    return static_cast<uint32_t>((r >> 3) * sbo + (k >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2);
}
__host__ __device__ __forceinline__ uint32_t off_f32(int r, int k, uint32_t sbo) {
    return static_cast<uint32_t>((r >> 3) * sbo + (k >> 2) * 128 + (r & 7) * 16 + (k & 3) * 4);
}

__device__ __forceinline__ float tf32_rn(float x) {
    uint32_t y;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(y) : "f"(x));
    return __uint_as_float(y);
}

// ------------------------------------------------------------------ intra-chunk record (SIMT math)

// One CTA per (chunk, head): the intra-chunk quantities in fp32 (direct exponentials), written as a
// tensor-core record.  Requires K = V = 128.
__global__ void __launch_bounds__(256) intra_tcrec_simt_kernel(Params p, uint8_t* recs) {
    constexpr int K = 128, V = 128, KP = K + 1;
    const int c = blockIdx.x, h = blockIdx.y;
    if (c >= p.chunk_off[p.N]) return;
    const int n = chunk_segment(p, c);
    const int tok0 = seg_begin(p, n) + (c - p.chunk_off[n]) * kChunk;
    const int len = min(kChunk, seg_end(p, n) - tok0);
    const int H = p.H;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    extern __shared__ float sm[];
    float* sQ = sm;                  // [64][KP] q_hat
    float* sK = sQ + 64 * KP;        // [64][KP] k_hat
    float* sG = sK + 64 * KP;        // [64][KP] Gamma
    float* sE = sG + 64 * KP;        // [64][KP] exp(Gamma)
    float* sA = sE + 64 * KP;        // [64][65] Aqk
    float* sB = sA + 64 * 65;        // [64][65] Bkk
    float* sN = sB + 64 * 65;        // [64][65] N
    float* sb = sN + 64 * 65;        // [64] beta
    if (tid < kChunk) {
        float b = 0.f;
        if (tid < len) b = sigmoidf_acc(load_act(p.beta_raw, (size_t)(tok0 + tid) * H + h, p.dtype));
        sb[tid] = b;
    }
    for (int t = warp; t < kChunk; t += 8) {
        const size_t base = ((size_t)(tok0 + t) * H + h) * K;
        float qv[4], kv[4], sq = 0.f, sk = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int cc = lane + 32 * i;
            qv[i] = t < len ? load_act(p.q, base + cc, p.dtype) : 0.f;
            kv[i] = t < len ? load_act(p.k, base + cc, p.dtype) : 0.f;
            sq += qv[i] * qv[i];
            sk += kv[i] * kv[i];
        }
        sq = warp_sum(sq);
        sk = warp_sum(sk);
        const float rq = 1.0f / sqrtf(sq + kNormEps), rk = 1.0f / sqrtf(sk + kNormEps);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            sQ[t * KP + lane + 32 * i] = qv[i] * rq;
            sK[t * KP + lane + 32 * i] = kv[i] * rk;
        }
    }
    const float ea = expf(p.a_log[h]);
    for (int i = tid; i < kChunk * K; i += blockDim.x) {
        const int t = i / K, cc = i % K;
        float g = 0.f;
        if (t < len) {
            const float x = load_act(p.g_raw, ((size_t)(tok0 + t) * H + h) * K + cc, p.dtype);
            g = p.lb * sigmoidf_acc(ea * (x + p.dt_bias[h * K + cc]));
        }
        sG[t * KP + cc] = g;
    }
    __syncthreads();
    for (int cc = tid; cc < K; cc += blockDim.x) {
        float acc = 0.f;
        for (int t = 0; t < kChunk; ++t) {
            acc += sG[t * KP + cc];
            sG[t * KP + cc] = acc;
            sE[t * KP + cc] = expf(acc);
        }
    }
    __syncthreads();
    for (int i = tid; i < kChunk * kChunk; i += blockDim.x) {
        const int t = i >> 6, s = i & 63;
        float aq = 0.f, ak = 0.f;
        if (s <= t) {
            for (int cc = 0; cc < K; ++cc) {
                const float e = expf(sG[t * KP + cc] - sG[s * KP + cc]);
                const float ks = sK[s * KP + cc] * e;
                aq += sQ[t * KP + cc] * ks;
                ak += sK[t * KP + cc] * ks;
            }
        }
        sA[t * 65 + s] = aq;
        sB[t * 65 + s] = (s < t) ? ak : 0.f;
        sN[t * 65 + s] = (s == t) ? 1.f : 0.f;
    }
    __syncthreads();
    for (int t = 1; t < kChunk; ++t) {
        if (tid < t) {
            float acc = 0.f;
            for (int r = tid; r < t; ++r) acc += sB[t * 65 + r] * sN[r * 65 + tid];
            sN[t * 65 + tid] = -sb[t] * acc;
        }
        __syncthreads();
    }
    uint8_t* rec = recs + ((size_t)c * H + h) * tcrec::BYTES;
    for (int i = tid; i < kChunk * K; i += blockDim.x) {
        const int t = i / K, cc = i % K;
        float w = 0.f;
        for (int s = 0; s <= t; ++s) w += sN[t * 65 + s] * sb[s] * sK[s * KP + cc] * sE[s * KP + cc];
        *reinterpret_cast<__nv_bfloat16*>(rec + tcrec::WQ + off_bf16(t, cc, 2048)) = __float2bfloat16_rn(w);
        *reinterpret_cast<__nv_bfloat16*>(rec + tcrec::WQ + off_bf16(64 + t, cc, 2048)) =
            __float2bfloat16_rn(sQ[t * KP + cc] * sE[t * KP + cc]);
        const float kd = sK[t * KP + cc] * expf(sG[63 * KP + cc] - sG[t * KP + cc]);
        *reinterpret_cast<float*>(rec + tcrec::KD + off_f32(cc, t, 2048)) = tf32_rn(kd);
    }
    for (int i = tid; i < kChunk * V; i += blockDim.x) {
        const int t = i / V, j = i % V;
        float acc = 0.f;
        for (int s = 0; s <= t && s < len; ++s)
            acc += sN[t * 65 + s] * sb[s] * load_act(p.v, ((size_t)(tok0 + s) * H + h) * V + j, p.dtype);
        *reinterpret_cast<float*>(rec + tcrec::U0 + (j >> 5) * tcrec::U0_SLICE + off_f32(t, j & 31, 1024)) = acc;
    }
    for (int i = tid; i < kChunk * kChunk; i += blockDim.x) {
        const int t = i >> 6, s = i & 63;
        *reinterpret_cast<float*>(rec + tcrec::AQ + off_f32(t, s, 2048)) = tf32_rn(sA[t * 65 + s]);
    }
    for (int cc = tid; cc < K; cc += blockDim.x)
        reinterpret_cast<float*>(rec + tcrec::GC)[cc] = sE[63 * KP + cc];
}

// ------------------------------------------------------------------ state chain (tcgen05)

namespace chainlay {
constexpr uint32_t SLOT_WQ = 0;
constexpr uint32_t SLOT_U0 = 32768;
constexpr uint32_t SLOT_KD = 40960;       // KD, AQ, GC follow contiguously (tcrec::TAIL bytes)
constexpr uint32_t SLOT_AQ = SLOT_KD + (tcrec::AQ - tcrec::KD);
constexpr uint32_t SLOT_GC = SLOT_KD + (tcrec::GC - tcrec::KD);
constexpr uint32_t SLOT_BYTES = (SLOT_KD + tcrec::TAIL + 1023) / 1024 * 1024;
constexpr uint32_t SB = 2 * SLOT_BYTES;   // S as bf16 B operand: 32 rows (j) x 128 K (c), SBO 2048
constexpr uint32_t UB = SB + 8192;        // U as tf32 B operand: 32 rows (j) x 64 K (t), SBO 2048
constexpr uint32_t BAR = UB + 8192;       // mbarriers: full[2], mma
constexpr uint32_t TSLOT = BAR + 64;
constexpr uint32_t BYTES = TSLOT + 64;
}  // namespace chainlay

constexpr uint32_t kIdescWS = idesc_bf16(128, 32, 0, 0);
// kind::tf32: A/B format 2 (TF32), f32 accumulate.
constexpr uint32_t kIdescTF32 = (1u << 4) | (2u << 7) | (2u << 10) | ((32u >> 3) << 17) | ((128u >> 4) << 24);

__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

// Issue the bulk loads of chunk record `c` (head h, slice z) into slot smem.
__device__ __forceinline__ void chain_load(uint8_t* slot, const uint8_t* rec, int z, uint64_t* bar) {
    mbar_expect_tx(bar, 32768 + tcrec::U0_SLICE + tcrec::TAIL);
    bulk_g2s(slot + chainlay::SLOT_WQ, rec + tcrec::WQ, 32768, bar);
    bulk_g2s(slot + chainlay::SLOT_U0, rec + tcrec::U0 + z * tcrec::U0_SLICE, tcrec::U0_SLICE, bar);
    bulk_g2s(slot + chainlay::SLOT_KD, rec + tcrec::KD, tcrec::TAIL, bar);
}

// One CTA per (segment, head, 32-column slice of V); 128 threads.  Thread c keeps row c of the
// state slice (32 fp32) in registers.
__global__ void __launch_bounds__(128, 1) chain_fwd_tc_kernel(Params p, const uint8_t* recs, int store_states) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int n = blockIdx.x, h = blockIdx.y, z = blockIdx.z, j0 = z * 32;
    const int H = p.H, K = 128, V = 128;
    const int tid = threadIdx.x, warp = tid >> 5;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + chainlay::BAR);
    uint64_t* mbar_mma = full + 2;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + chainlay::TSLOT);
    uint8_t* SB = smem + chainlay::SB;
    uint8_t* UB = smem + chainlay::UB;
    const int cb = p.chunk_off[n], ce = p.chunk_off[n + 1];
    const int tb = seg_begin(p, n), te = seg_end(p, n);
    const int nch = ce - cb;

    if (tid == 0) {
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        mbar_init(mbar_mma, 1);
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(tslot, 64);
    // entering state, row c = tid
    float S[32];
    {
        const float* src = p.S0 ? p.S0 + (((size_t)n * H + h) * K + tid) * V + j0 : nullptr;
#pragma unroll
        for (int j = 0; j < 32; ++j) S[j] = src ? src[j] : 0.f;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t tD1 = tmem, tD3 = tmem + 32;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    if (tid == 0) {
        for (int i = 0; i < 2 && i < nch; ++i)
            chain_load(smem + i * chainlay::SLOT_BYTES, recs + ((size_t)(cb + i) * H + h) * tcrec::BYTES, z, &full[i]);
    }
#pragma unroll
    for (int j = 0; j < 32; ++j)
        *reinterpret_cast<__nv_bfloat16*>(SB + off_bf16(j, tid, 2048)) = __float2bfloat16_rn(S[j]);
    fence_async_smem();
    __syncthreads();

    // Every wait is bounded and block-uniform: a timeout makes all threads leave the loop together.
    auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool {
        const bool mine = mbar_wait(bar, parity);
        return __syncthreads_and(mine ? 1 : 0) != 0;
    };
    uint32_t mma_phase = 0;
    bool ok = true;
    for (int i = 0; i < nch && ok; ++i) {
        const int c = cb + i;
        const int slot = i & 1;
        uint8_t* sl = smem + slot * chainlay::SLOT_BYTES;
        const int tok0 = tb + i * kChunk, len = min(kChunk, te - tok0);
        if (store_states) {
            float* dst = p.states + (((size_t)c * H + h) * K + tid) * V + j0;
#pragma unroll
            for (int j = 0; j < 32; j += 4) *reinterpret_cast<float4*>(dst + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
        }
        if (!wait_all(&full[slot], (i >> 1) & 1)) { ok = false; break; }
        // MMA1: D1 = [W; Qg] S   (bf16, M=128, N=32, K=128)
        if (tid == 0) {
            tc_fence_after();
            for (int kk = 0; kk < 8; ++kk) {
                const uint64_t a = smem_desc(smem_u32(sl + chainlay::SLOT_WQ) + kk * 256, 128, 2048);
                const uint64_t b = smem_desc(smem_u32(SB) + kk * 256, 128, 2048);
                mma_bf16(tD1, a, b, kIdescWS, kk > 0);
            }
            mma_commit(mbar_mma);
        }
        if (!wait_all(mbar_mma, mma_phase)) { ok = false; break; }
        mma_phase ^= 1;
        tc_fence_after();
        if (warp < 2) {
            // U[t][j] = U0[t][j] - (W S)[t][j], t = tid
            float d[32];
            tmem_ld16(tD1 + lane_base, d);
            tmem_ld16(tD1 + lane_base + 16, d + 16);
            tmem_ld_wait();
            const uint8_t* u0 = sl + chainlay::SLOT_U0;
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
                const float4 u = *reinterpret_cast<const float4*>(u0 + off_f32(tid, j, 1024));
                const float uu[4] = {u.x - d[j], u.y - d[j + 1], u.z - d[j + 2], u.w - d[j + 3]};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    *reinterpret_cast<float*>(UB + off_f32(j + e, tid, 2048)) = tf32_rn(uu[e]);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        // MMA2: D1 += [. ; Aqk] U  and  D3 = Kd^T U   (tf32, M=128, N=32, K=64)
        if (tid == 0) {
            tc_fence_after();
            for (int kk = 0; kk < 8; ++kk) {
                const uint64_t b = smem_desc(smem_u32(UB) + kk * 256, 128, 2048);
                const uint64_t a1 = smem_desc(smem_u32(sl + chainlay::SLOT_AQ) - 16384 + kk * 256, 128, 2048);
                mma_tf32(tD1, a1, b, kIdescTF32, 1);
                const uint64_t a2 = smem_desc(smem_u32(sl + chainlay::SLOT_KD) + kk * 256, 128, 2048);
                mma_tf32(tD3, a2, b, kIdescTF32, kk > 0);
            }
            mma_commit(mbar_mma);
        }
        if (!wait_all(mbar_mma, mma_phase)) { ok = false; break; }
        mma_phase ^= 1;
        tc_fence_after();
        const float gc = reinterpret_cast<const float*>(sl + chainlay::SLOT_GC)[tid];
        if (warp >= 2 && p.out) {
            const int t = tid - 64;
            float d[32];
            tmem_ld16(tD1 + lane_base, d);
            tmem_ld16(tD1 + lane_base + 16, d + 16);
            tmem_ld_wait();
            if (t < len) {
                __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(p.out) + ((size_t)(tok0 + t) * H + h) * V + j0;
#pragma unroll
                for (int j = 0; j < 32; j += 8) {
                    uint4 pk;
                    __nv_bfloat162 b0 = __floats2bfloat162_rn(p.scale * d[j], p.scale * d[j + 1]);
                    __nv_bfloat162 b1 = __floats2bfloat162_rn(p.scale * d[j + 2], p.scale * d[j + 3]);
                    __nv_bfloat162 b2 = __floats2bfloat162_rn(p.scale * d[j + 4], p.scale * d[j + 5]);
                    __nv_bfloat162 b3 = __floats2bfloat162_rn(p.scale * d[j + 6], p.scale * d[j + 7]);
                    pk.x = *reinterpret_cast<uint32_t*>(&b0);
                    pk.y = *reinterpret_cast<uint32_t*>(&b1);
                    pk.z = *reinterpret_cast<uint32_t*>(&b2);
                    pk.w = *reinterpret_cast<uint32_t*>(&b3);
                    *reinterpret_cast<uint4*>(o + j) = pk;
                }
            }
        }
        {
            float d[32];
            tmem_ld16(tD3 + lane_base, d);
            tmem_ld16(tD3 + lane_base + 16, d + 16);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                S[j] = gc * S[j] + d[j];
                *reinterpret_cast<__nv_bfloat16*>(SB + off_bf16(j, tid, 2048)) = __float2bfloat16_rn(S[j]);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        // the slot is free again: prefetch chunk i + 2 into it
        if (tid == 0 && i + 2 < nch)
            chain_load(sl, recs + ((size_t)(c + 2) * H + h) * tcrec::BYTES, z, &full[slot]);
    }
    if (!ok) {
        // Record the timeout, then give in-flight copies and MMAs a bounded chance to land before
        // this CTA's shared memory and tensor memory are released.
        if (tid == 0) {
            record_error(p.status, KDA_ERR_TIMEOUT);
            mbar_wait(mbar_mma, mma_phase, 1u << 16);
            for (int s2 = 0; s2 < 2; ++s2) mbar_wait(&full[s2], 0, 1u << 16);
        }
    } else if (p.ST) {
        float* dst = p.ST + (((size_t)n * H + h) * K + tid) * V + j0;
#pragma unroll
        for (int j = 0; j < 32; j += 4) *reinterpret_cast<float4*>(dst + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 64);
}

// ------------------------------------------------------------------ launchers

size_t tc_record_bytes(int NCmax, int H) { return (size_t)NCmax * H * tcrec::BYTES; }

cudaError_t launch_intra_tc(const Params& p, uint8_t* recs, cudaStream_t st) {
    const size_t smem = (size_t)(4 * 64 * 129 + 3 * 64 * 65 + 64) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(intra_tcrec_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    timing_pre(st, K_INTRA_TC);
    intra_tcrec_simt_kernel<<<dim3(p.NCmax, p.H), 256, smem, st>>>(p, recs);
    timing_post(st);
    return cudaGetLastError();
}

cudaError_t launch_chain_fwd_tc(const Params& p, const uint8_t* recs, bool store_states, cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(chain_fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)chainlay::BYTES);
    if (e != cudaSuccess) return e;
    timing_pre(st, K_CHAIN_FWD_TC);
    chain_fwd_tc_kernel<<<dim3(p.N, p.H, 4), 128, chainlay::BYTES, st>>>(p, recs, store_states ? 1 : 0);
    timing_post(st);
    return cudaGetLastError();
}

}  // namespace kda
