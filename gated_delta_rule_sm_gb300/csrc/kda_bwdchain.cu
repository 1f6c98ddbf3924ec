// kda_bwdchain.cu -- the two state chains of the backward on tcgen05 tensor cores (bf16 inputs,
// K = V = 128), state in fp32 registers.
//
// Both are the affine recursion  X = Y_c + A1_c Z,  Z' = Diag(exp(Gamma_last,c)) Z + A2_c X (+ P_c)
// of the chunkwise gated delta rule ("[kimi k3] add eager reference model with FSDP2", chunk_kda):
//   * forward state recompute (REV = false): Z = S entering chunk c, A1 = -W, Y = U0, A2 = Kd^T,
//     so X = U and Z' is the state leaving the chunk;
//   * reverse chain (REV = true): Z = dS, the gradient w.r.t. the state leaving chunk c, A1 = Kd,
//     Y = scale Aqk^T dO, A2 = -W^T, P = scale Qg^T dO, so X = dU and Z' is the gradient entering
//     the chunk.
// The operand slot (chainrec, shared by both directions) and Y, P come from bwd_pre.  Every product runs
// in split precision with bf16 halves, operand = hi + lo, hi*hi + hi*lo + lo*hi (kind::f16, relative
// error ~1e-5): the gradient of the log-decay at the end of a chunk carries dS_end * S_end-sized
// terms far larger than its typical value, and plain tf32 chains (~2e-4 relative error in S and
// dS, NumPy emulation and GPU measurement agree) put it outside the bf16 tolerance under slowly
// decaying gates.
//
// One CTA per (segment, head, column slice of JW value columns); the columns of Z are independent.
// Row r of Z belongs to threads r + 128 i, each with JH consecutive columns of the slice (bwchain::
// threads: 256 threads of JW / 2 columns for JW = 32 or 64, 512 threads of 32 columns for JW = 128), so
// the TMEM read-backs, hi / lo splits and stores of a step spread over 8 or 16 warps.  Per chunk: MMA1 (M = 64, N = JW, K = 128) into TMEM,
// X = D1 + Y split into bf16 hi + lo (MN-major, one 16-byte store per 8 columns), MMA2 (M = 128,
// N = JW, K = 64), then Z' = gC Z + D3 (+ P).  Record slots (A1, A2 hi/lo, gC) are double buffered
// by bulk copies.  X (U, or dU) and the chunk's Z are also written out per chunk for the gradient
// kernel, in x4 order (x4_off) so that every warp store covers whole 128-byte lines.
//
// Three modes (template MODE): the full pass above; for the segment-parallel backward a local pass
// (Z from zero, only the end Z written) and a transfer pass (Z from the identity, Y and P taken as
// zero, only the end Z written: the segment's transition, since K = V).  The blocks take segments
// longest first (seg_order).  K = V = 64 heads run on zero-padded 128 x 128 states that the host side
// pads and unpads with the two small kernels at the end of this file.
#include "kda_common.cuh"
#include "kda_internal.h"
#include "kda_sm100.cuh"

namespace kda {

using namespace sm100;

// Where a chain finds its per-chunk inputs: slot (chainrec) of chunk c at slots + (c H + h) *
// slot_stride bytes; the Y tile (64 rows t, 128 columns) at ybase + (c H + h) * ystride floats: in x4
// order for the reverse chain (bwd_pre's Y), row-major for the recompute (U0 of the forward record);
// the P tile (128 rows, x4 order) likewise.
struct ChainSrc {
    const uint8_t* slots;
    size_t slot_stride;
    const float* ybase;
    size_t ystride;
    const float* pbase;   // reverse chain only
    size_t pstride;
    int mode;             // BwdChainMode
    int rank_major;       // blockIdx.x = (head, slice), blockIdx.y = rank in seg_order (longest first)
};

namespace bwchain {
// Threads per CTA: 256 (two per row of Z, half the slice's columns each), or 512 for JW = 128 (four per
// row, 32 columns each).
__host__ __device__ constexpr int threads(int jw) { return jw >= 128 ? 512 : 256; }

template <int JW>
struct Lay {
    static constexpr uint32_t SLOT = chainrec::SLOT;       // two record slots at 0 and SLOT
    static constexpr uint32_t ZK = JW * 16;                // Z: bytes between its 8-row K groups
    static constexpr uint32_t XK = JW * 16;                // X: likewise
    static constexpr uint32_t ZB = 2 * SLOT;               // Z (N = j, K = c) bf16 MN-major mn_bf16(j, c, 128, ZK), hi
    static constexpr uint32_t ZL = ZB + 16 * ZK;           // Z lo (16 K groups of 8)
    static constexpr uint32_t XB = ZL + 16 * ZK;           // X (N = j, K = t) bf16 MN-major mn_bf16(j, t, 128, XK), hi
    static constexpr uint32_t XL = XB + 8 * XK;            // X lo (8 K groups)
    static constexpr uint32_t BAR = XL + 8 * XK;           // mbarriers: full[2], mma1, mma2; fail flag; TMEM slot
    static constexpr uint32_t BYTES = BAR + 64;
    static constexpr uint32_t TCOLS = 2 * JW;              // D1 at column 0, D3 at column JW
};
}  // namespace bwchain

// Eight fp32 values as bf16 hi and lo halves (lo = bf16(x - hi)).
__device__ __forceinline__ void split8_bf16(const float* x, uint4& hi, uint4& lo) {
    float h[8], l[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        h[e] = __bfloat162float(__float2bfloat16_rn(x[e]));
        l[e] = x[e] - h[e];
    }
    hi = pack8_bf16(h);
    lo = pack8_bf16(l);
}

template <int JW, bool REV, int MODE>
__global__ void __launch_bounds__(bwchain::threads(JW), 1) chain_split_kernel(Params p, ChainSrc src) {
    using L = bwchain::Lay<JW>;
    extern __shared__ __align__(1024) uint8_t smem[];
    int n, h, j0;
    if (src.rank_major) {
        constexpr int NZ = 128 / JW;
        h = blockIdx.x / NZ;
        j0 = (blockIdx.x - h * NZ) * JW;
        n = seg_order(p)[blockIdx.y];
    } else {
        n = blockIdx.x;
        h = blockIdx.y;
        j0 = blockIdx.z * JW;
    }
    const int H = p.H;
    constexpr int K = 128, V = 128;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // JW >= 64: two threads per row of Z, each with JH of the slice's columns (warps 4-7 read the same
    // TMEM lane quarters as warps 0-3, at column offset JH)
    constexpr int JH = JW / (bwchain::threads(JW) / 128);
    constexpr int BLK = JH < 32 ? JH : 32;   // columns per TMEM read-back block
    const int row = tid & 127, jo = (tid >> 7) * JH, quarter = warp & 3;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::BAR);
    uint64_t* bar1 = full + 2;
    uint64_t* bar2 = full + 3;
    int* sh_fail = reinterpret_cast<int*>(full + 4);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(full + 5);
    uint8_t* ZB = smem + L::ZB;
    uint8_t* ZL = smem + L::ZL;
    uint8_t* XB = smem + L::XB;
    uint8_t* XL = smem + L::XL;
    const int cb = p.chunk_off[n], ce = p.chunk_off[n + 1];
    const int nch = ce - cb;

    if (tid == 0) {
        for (int i = 0; i < 4; ++i) mbar_init(&full[i], 1);
        *sh_fail = 0;
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(tslot, L::TCOLS);
    // local and transfer passes write only the end state; the transfer pass takes Y and P as zero
    constexpr bool full_pass = MODE == kBwdChainFull, zero_y = MODE == kBwdChainTransfer;
    float z[JH];   // columns jo .. jo + JH - 1 of row `row` of Z (dS for the reverse chain, S for the recompute)
    {
        const float* z0 = full_pass ? (REV ? p.dST : p.S0) : nullptr;
        const float* zs = z0 ? z0 + (((size_t)n * H + h) * K + row) * V + j0 + jo : nullptr;
#pragma unroll
        for (int j = 0; j < JH; j += 4) {
            const float4 v = zs ? *reinterpret_cast<const float4*>(zs + j) : make_float4(0.f, 0.f, 0.f, 0.f);
            z[j] = v.x; z[j + 1] = v.y; z[j + 2] = v.z; z[j + 3] = v.w;
        }
        if (zero_y)   // the identity (K = V): row r has its one in column r
#pragma unroll
            for (int j = 0; j < JH; ++j) z[j] = (j0 + jo + j == row) ? 1.f : 0.f;
    }
    auto write_z_operand = [&]() {   // thread = K index c: eight j per 16-byte row of a core matrix
#pragma unroll
        for (int jg = 0; jg < JH / 8; ++jg) {
            uint4 hi, lo;
            split8_bf16(z + 8 * jg, hi, lo);
            const uint32_t o = mn_bf16(jo + 8 * jg, row, 128, L::ZK);
            *reinterpret_cast<uint4*>(ZB + o) = hi;
            *reinterpret_cast<uint4*>(ZL + o) = lo;
        }
    };
    write_z_operand();
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t tD1 = tmem, tD3 = tmem + JW;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    auto slot_ptr = [&](int s) { return smem + (s & 1) * L::SLOT; };
    // step s handles chunk cb + nch - 1 - s (reverse) or cb + s (forward)
    auto chunk_of = [&](int s) { return REV ? cb + nch - 1 - s : cb + s; };
    auto rec_ptr = [&](int s) { return src.slots + ((size_t)chunk_of(s) * H + h) * src.slot_stride; };
    auto y_ptr = [&](int s) { return src.ybase + ((size_t)chunk_of(s) * H + h) * src.ystride; };
    auto p_ptr = [&](int s) { return src.pbase + ((size_t)chunk_of(s) * H + h) * src.pstride; };
    auto fail_wait = [&](uint64_t* bar, uint32_t parity) {
        if (!mbar_wait_done(bar, parity)) atomicExch(sh_fail, 1);
    };
    if (tid == 0)
        for (int s = 0; s < 2 && s < nch; ++s) {
            mbar_expect_tx(&full[s], L::SLOT);
            bulk_g2s(slot_ptr(s), rec_ptr(s), L::SLOT, &full[s]);
        }
    // D += hi*hi + hi*lo + lo*hi, the small products first.  A: start advance per K = 16 step, LBO, SBO.
    // The slot tiles are [128 c][64 t] K-major: A2 (M = c, K = t) reads them K-major (256, 128, 1024), A1
    // (M = t, K = c) as their MN-major transpose (2048, 1024, 128); B: MN-major.
    auto mma3 = [](uint32_t d, uint32_t ah, uint32_t al, uint32_t bh, uint32_t bl, int nk, uint32_t a_step,
                   uint32_t a_lbo, uint32_t a_sbo, uint32_t b_lbo, uint32_t idesc) {
        for (int kk = 0; kk < nk; ++kk)
            mma_bf16(d, smem_desc(al + kk * a_step, a_lbo, a_sbo), smem_desc(bh + kk * 2 * b_lbo, b_lbo, 128), idesc,
                     kk > 0);
        for (int kk = 0; kk < nk; ++kk)
            mma_bf16(d, smem_desc(ah + kk * a_step, a_lbo, a_sbo), smem_desc(bl + kk * 2 * b_lbo, b_lbo, 128), idesc, 1);
        for (int kk = 0; kk < nk; ++kk)
            mma_bf16(d, smem_desc(ah + kk * a_step, a_lbo, a_sbo), smem_desc(bh + kk * 2 * b_lbo, b_lbo, 128), idesc, 1);
    };
    // this direction's operands in the shared slot
    constexpr uint32_t A1 = REV ? chainrec::KD : chainrec::WN, A1L = REV ? chainrec::KD_LO : chainrec::WN_LO;
    constexpr uint32_t A2 = REV ? chainrec::WN : chainrec::KD, A2L = REV ? chainrec::WN_LO : chainrec::KD_LO;

    bool ok = true;
    for (int s = 0; s < nch; ++s) {
        const int c = chunk_of(s);
        uint8_t* sl = slot_ptr(s);
        const uint32_t par = s & 1;
        fail_wait(&full[s & 1], (s >> 1) & 1);
        tc_fence_after();
        if (tid == 0) {   // D1 = A1 Z  (M = 64, N = JW, K = 128)
            mma3(tD1, smem_u32(sl + A1), smem_u32(sl + A1L), smem_u32(ZB), smem_u32(ZL), 8, 2048, 1024, 128, L::ZK,
                 idesc_bf16(64, JW, 1, 1));
            mma_commit(bar1);
            if (s + 1 < nch && !zero_y) {   // warm L2 with the next chunk's Y (and P)
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
        if (full_pass) {   // reverse: gradient w.r.t. the state leaving chunk c; forward: the state entering
            // chunk c (x4 order: the warp's 32 rows make 512 contiguous bytes per 16-byte store)
            float* dst = (REV ? p.dstates : p.states) + ((size_t)c * H + h) * K * V;
#pragma unroll
            for (int j = 0; j < JH; j += 4)
                *reinterpret_cast<float4*>(dst + x4_off(row, j0 + jo + j, K)) = make_float4(z[j], z[j + 1], z[j + 2], z[j + 3]);
        }
        // X rows t = 16 warp + lane (lanes 0..15 of each warp carry the M = 64 result).  The Y row is
        // read from global memory 32 columns ahead of its use: the first block before MMA1 is waited
        // for, each next block while the current one is combined.
        const int t = 16 * quarter + (lane & 15);
        // 32 columns from col of row `row` of a tile with `rows` rows, x4-ordered or row-major
        auto load32 = [](const float* tile, int row, int col, int rows, bool x4, float* dst) {   // BLK columns
            if (zero_y) {
#pragma unroll
                for (int j = 0; j < BLK; ++j) dst[j] = 0.f;
                return;
            }
#pragma unroll
            for (int j = 0; j < BLK; j += 4) {
                const float4 v = *reinterpret_cast<const float4*>(tile + (x4 ? x4_off(row, col + j, rows)
                                                                              : (size_t)row * V + col + j));
                dst[j] = v.x; dst[j + 1] = v.y; dst[j + 2] = v.z; dst[j + 3] = v.w;
            }
        };
        const float* ytile = y_ptr(s);
        float ynext[BLK];
        load32(ytile, t, j0 + jo, 64, REV, ynext);
        fail_wait(bar1, par);
        tc_fence_after();
        {
#pragma unroll
            for (int jb = 0; jb < JH; jb += BLK) {
                float d[BLK];
                tmem_ld16(tD1 + jo + jb + lane_base, d);
                if (BLK == 32) tmem_ld16(tD1 + jo + jb + 16 + lane_base, d + 16);
                float y[BLK];
#pragma unroll
                for (int j = 0; j < BLK; ++j) y[j] = ynext[j];
                if (jb + BLK < JH) load32(ytile, t, j0 + jo + jb + BLK, 64, REV, ynext);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < BLK; ++j) d[j] += y[j];
                if (full_pass && lane < 16) {   // X row t (U or dU) for the gradient kernel, x4 order
                    float* xo = (REV ? p.chunk_du : p.chunk_u) + ((size_t)c * H + h) * 64 * V;
#pragma unroll
                    for (int j = 0; j < BLK; j += 4)
                        *reinterpret_cast<float4*>(xo + x4_off(t, j0 + jo + jb + j, 64)) =
                            make_float4(d[j], d[j + 1], d[j + 2], d[j + 3]);
                }
                if (lane < 16)
#pragma unroll
                    for (int g8 = 0; g8 < BLK / 8; ++g8) {
                        uint4 hi, lo;
                        split8_bf16(d + 8 * g8, hi, lo);
                        const uint32_t o = mn_bf16(jo + jb + 8 * g8, t, 128, L::XK);
                        *reinterpret_cast<uint4*>(XB + o) = hi;
                        *reinterpret_cast<uint4*>(XL + o) = lo;
                    }
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (*sh_fail) { ok = false; break; }
        if (tid == 0) {   // D3 = A2 X  (M = 128, N = JW, K = 64)
            mma3(tD3, smem_u32(sl + A2), smem_u32(sl + A2L), smem_u32(XB), smem_u32(XL), 4, 256, 128, 1024, L::XK,
                 idesc_bf16(128, JW, 0, 1));
            mma_commit(bar2);
        }
        // the P row likewise, one 32-column block ahead (reverse chain only)
        const float* ptile = REV ? p_ptr(s) : nullptr;
        float pnext[BLK];
        if (REV) load32(ptile, row, j0 + jo, K, true, pnext);
        fail_wait(bar2, par);
        tc_fence_after();
        {
            const float gc = reinterpret_cast<const float*>(sl + chainrec::GC)[row];
#pragma unroll
            for (int jb = 0; jb < JH; jb += BLK) {
                float d[BLK];
                tmem_ld16(tD3 + jo + jb + lane_base, d);
                if (BLK == 32) tmem_ld16(tD3 + jo + jb + 16 + lane_base, d + 16);
                float pv[BLK];
#pragma unroll
                for (int j = 0; j < BLK; ++j) pv[j] = REV ? pnext[j] : 0.f;
                if (REV && jb + BLK < JH) load32(ptile, row, j0 + jo + jb + BLK, K, true, pnext);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < BLK; ++j) z[jb + j] = gc * z[jb + j] + d[j] + pv[j];
            }
            write_z_operand();
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (*sh_fail) { ok = false; break; }
        // both MMAs of this chunk are complete: the slot takes the chunk two steps ahead
        if (tid == 0 && s + 2 < nch) {
            mbar_expect_tx(&full[s & 1], L::SLOT);
            bulk_g2s(sl, rec_ptr(s + 2), L::SLOT, &full[s & 1]);
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
    } else if (REV ? p.dS0 != nullptr : p.ST != nullptr) {
        float* dst = (REV ? p.dS0 : p.ST) + (((size_t)n * H + h) * K + row) * V + j0 + jo;
#pragma unroll
        for (int j = 0; j < JH; j += 4)
            *reinterpret_cast<float4*>(dst + j) = make_float4(z[j], z[j + 1], z[j + 2], z[j + 3]);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, L::TCOLS);
}

template <int JW, bool REV>
static cudaError_t launch_chain_jw(const Params& p, const ChainSrc& src, cudaStream_t st) {
    using L = bwchain::Lay<JW>;
    static_assert(L::BYTES <= 232448, "shared memory per CTA");
    auto kern = src.mode == kBwdChainLocal      ? chain_split_kernel<JW, REV, kBwdChainLocal>
                : src.mode == kBwdChainTransfer ? chain_split_kernel<JW, REV, kBwdChainTransfer>
                                                : chain_split_kernel<JW, REV, kBwdChainFull>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::BYTES);
    if (e != cudaSuccess) return e;
    timing_pre(st, REV ? K_CHAIN_BWD_TC : K_CHAIN_REC_TC);
    ChainSrc s2 = src;
    s2.rank_major = p.N <= 65535;   // segments in launch order, longest first (grid y holds at most 65535)
    if (s2.rank_major)
        kern<<<dim3(p.H * (128 / JW), p.N), bwchain::threads(JW), L::BYTES, st>>>(p, s2);
    else
        kern<<<dim3(p.N, p.H, 128 / JW), bwchain::threads(JW), L::BYTES, st>>>(p, s2);
    timing_post(st);
    return cudaGetLastError();
}

// Column slices per (segment, head) chain: one CTA per chain when the chains alone nearly fill the
// GPU's SMs, otherwise 2 or 4 narrower CTAs (shorter per-step latency, more parallel chains).
template <bool REV>
static cudaError_t launch_chain(const Params& p, const ChainSrc& src, cudaStream_t st) {
    int sms = 0, dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long chains = (long)p.N * p.H;
    if (chains * 3 >= (long)sms * 2) return launch_chain_jw<128, REV>(p, src, st);
    if (chains * 3 >= (long)sms) return launch_chain_jw<64, REV>(p, src, st);
    return launch_chain_jw<32, REV>(p, src, st);
}

cudaError_t launch_chain_bwd_tc(const Params& p, const uint8_t* bw, cudaStream_t st, int mode) {
    const RecLayout L = RecLayout::make(128, 128);   // the slot leads each chunk's record (W, Kd, gC)
    ChainSrc src{reinterpret_cast<const uint8_t*>(p.rec + L.W), p.rec_stride * sizeof(float),
                 reinterpret_cast<const float*>(bw + bwrec::Y), bwrec::BYTES / 4,
                 reinterpret_cast<const float*>(bw + bwrec::P), bwrec::BYTES / 4, mode, 0};
    static_assert(bwrec::BYTES % 256 == 0, "record stride");
    return launch_chain<true>(p, src, st);
}

cudaError_t launch_chain_rec_tc(const Params& p, const uint8_t* bw, cudaStream_t st, int mode) {
    const RecLayout L = RecLayout::make(128, 128);
    ChainSrc src{reinterpret_cast<const uint8_t*>(p.rec + L.W), p.rec_stride * sizeof(float), p.rec + L.U0,
                 p.rec_stride, nullptr, 0, mode, 0};
    return launch_chain<false>(p, src, st);
}

}  // namespace kda

namespace kda {

// K = V = 64 heads on the tensor-core backward: the chains carry a 128 x 128 state whose upper-left
// 64 x 64 quarter is the head's state.  The caller's [N, H, K, V] states are copied into zeroed
// 128 x 128 ones before the chains (pad) and the initial-state gradient copied back after (unpad).
__global__ void state_pad_kernel(const float* __restrict__ src, float* __restrict__ dst, int K, int V, int NH) {
    const size_t total = (size_t)NH * 128 * 128;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
        const int c = (int)(i & 127), r = (int)((i >> 7) & 127);
        const size_t nh = i >> 14;
        dst[i] = (src && r < K && c < V) ? src[(nh * K + r) * V + c] : 0.f;
    }
}

__global__ void state_unpad_kernel(const float* __restrict__ src, float* __restrict__ dst, int K, int V, int NH) {
    const size_t total = (size_t)NH * K * V;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
        const int c = (int)(i % V);
        const size_t rr = i / V;
        const int r = (int)(rr % K);
        const size_t nh = rr / K;
        dst[i] = src[(nh * 128 + r) * 128 + c];
    }
}

cudaError_t launch_state_pad(const float* src, float* dst, int K, int V, int NH, cudaStream_t st) {
    const size_t total = (size_t)NH * 128 * 128;
    const int grid = (int)((total + 255) / 256 < 4096 ? (total + 255) / 256 : 4096);
    state_pad_kernel<<<grid, 256, 0, st>>>(src, dst, K, V, NH);
    return cudaGetLastError();
}

cudaError_t launch_state_unpad(const float* src, float* dst, int K, int V, int NH, cudaStream_t st) {
    const size_t total = (size_t)NH * K * V;
    const int grid = (int)((total + 255) / 256 < 4096 ? (total + 255) / 256 : 4096);
    state_unpad_kernel<<<grid, 256, 0, st>>>(src, dst, K, V, NH);
    return cudaGetLastError();
}

}  // namespace kda
