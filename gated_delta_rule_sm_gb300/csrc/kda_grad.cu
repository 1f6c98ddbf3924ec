// kda_grad.cu -- per-chunk gradients of the chunkwise KDA recurrence for K = V = 128 (K = V = 64
// heads zero-padded to 128 channels, only the real channels written out).
//
// Inputs per (chunk, head): the fp32 chunk record (Kg, N, Bkk, Gamma, q_hat, k_hat, beta, the inverse
// norms; Qg and Kd are formed from Gamma, q_hat, k_hat), the chunk-entering state S0 and the gradient
// dS_end w.r.t. the chunk-leaving
// state (both from the state chains), U and dU per chunk (written by the two backward chains), dO,
// v and g_raw.  The gradient of the chunk equations
//     U = U0 - W S0,   O = scale (Qg S0 + Aqk U),   S_end = Diag(exp(Gamma_last)) S0 + Kd^T U,
//     T = N Diag(beta), N = (I + Diag(beta) Bkk)^-1, W = T Kg, U0 = T v
// is formed here and pushed through the decayed bilinear forms, the cumulative log-decay and the
// prologue (L2 norm, sigmoid beta, the gate under either activation).
//
// Phase 1 walks the four 32-column slices of V: the slice outer products (dKg, dQg, dKd, dT, dA)
// accumulate in TMEM from tcgen05 MMAs on bf16 hi / lo operands; the small dependent products in
// between (v - Kg S0, Diag(beta) N^T dU) and those of phase 2 run as warp-level MMAs straight from
// padded shared-memory tiles, no descriptor or accumulator round trips between the many dependent
// steps.  Every one of them splits its operands (hi + lo, three products): bf16 m16n8k16 for most,
// tf32 m16n8k8 for dk_R, whose record loads run a k-step ahead; the log-decay gradient's pair terms
// cancel, so single-product rounding (~5e-4) showed up there at ~1e-2 of its RMS under mild gates.
// Row strides = 4 (mod 32) words make the fragment loads conflict-free.
#include "kda_common.cuh"
#include "kda_internal.h"
#include "kda_sm100.cuh"

namespace kda {

using namespace sm100;

namespace {

struct Tile {
    const float* p;
    int rs, cs;   // element (r, c) at p[r * rs + c * cs]
    __device__ __forceinline__ float at(int r, int c) const { return p[r * rs + c * cs]; }
};

// A bf16 tile: element (r, c) at p[r * rs + c * cs].
struct TileH {
    const __nv_bfloat16* p;
    int rs, cs;
};

// bf16 warp MMA, 16 x 8 x 16, fp32 accumulate.  Fragments (g = lane / 4, q = lane % 4): A words
// (row g, k 2q..2q+1), (row g + 8, k 2q..), (row g, k 2q + 8..), (row g + 8, k 2q + 8..); B words
// (k 2q..2q+1, col g), (k 2q + 8.., col g); the first element of a pair in the low half.  C words
// (row g, col 2q), (row g, col 2q + 1), (row g + 8, col 2q), (row g + 8, col 2q + 1), as frag_rc gives.
__device__ __forceinline__ void mma16816(float* d, const uint32_t* a, const uint32_t* b) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// (x0, x1) as bf16 pairs hi = bf16(x), lo = bf16(x - hi): hi + lo carries 16 significant bits.
__device__ __forceinline__ void split_bf16x2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = *reinterpret_cast<const uint32_t*>(&l);
}

// d[b] (16 x 8 blocks at rows m0, cols n0 + 8 b, b < NB) += sum_k A(m, k) B(k, n) over k in [k_lo, k_hi),
// both operands split into bf16 halves (hi*hi + hi*lo + lo*hi, relative error ~1e-5 where one tf32
// product gives ~5e-4); one A fragment per k-step serves the whole strip, the k-loop stays rolled to
// keep the kernel's code small.  k_lo and k_hi - k_lo multiples of 16.
template <int NB>
__device__ __forceinline__ void mma_strip3_bf16(float (&d)[NB][4], const Tile& A, const Tile& B, int m0, int n0,
                                                int k_lo, int k_hi, int lane) {
    const int g = lane >> 2, q = lane & 3;
#pragma unroll 1
    for (int k0 = k_lo; k0 < k_hi; k0 += 16) {
        uint32_t ah[4], al[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = m0 + g + 8 * (i & 1), k = k0 + 2 * q + 8 * (i >> 1);
            split_bf16x2(A.at(r, k), A.at(r, k + 1), ah[i], al[i]);
        }
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const int n = n0 + 8 * b + g;
            uint32_t bh[2], bl[2];
            split_bf16x2(B.at(k0 + 2 * q, n), B.at(k0 + 2 * q + 1, n), bh[0], bl[0]);
            split_bf16x2(B.at(k0 + 2 * q + 8, n), B.at(k0 + 2 * q + 9, n), bh[1], bl[1]);
            mma16816(d[b], al, bh);
            mma16816(d[b], ah, bl);
            mma16816(d[b], ah, bh);
        }
    }
}

// Two left operands sharing the right one, d1 += A1 B and d2 += A2 B, in the same split bf16 products
// (relative error ~1e-5, as the backward chains' split products).  k_hi - k_lo a multiple of 16.
template <int NB>
__device__ __forceinline__ void mma_strip3_pair_bf16(float (&d1)[NB][4], float (&d2)[NB][4], const Tile& A1,
                                                     const Tile& A2, const Tile& B, int m0, int n0, int k_lo,
                                                     int k_hi, int lane) {
    const int g = lane >> 2, q = lane & 3;
#pragma unroll 1
    for (int k0 = k_lo; k0 < k_hi; k0 += 16) {
        uint32_t h1[4], l1[4], h2[4], l2[4];
        const int rr[4] = {m0 + g, m0 + g + 8, m0 + g, m0 + g + 8};
        const int kk[4] = {k0 + 2 * q, k0 + 2 * q, k0 + 2 * q + 8, k0 + 2 * q + 8};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            split_bf16x2(A1.at(rr[i], kk[i]), A1.at(rr[i], kk[i] + 1), h1[i], l1[i]);
            split_bf16x2(A2.at(rr[i], kk[i]), A2.at(rr[i], kk[i] + 1), h2[i], l2[i]);
        }
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const int n = n0 + 8 * b + g;
            uint32_t bh[2], bl[2];
            split_bf16x2(B.at(k0 + 2 * q, n), B.at(k0 + 2 * q + 1, n), bh[0], bl[0]);
            split_bf16x2(B.at(k0 + 2 * q + 8, n), B.at(k0 + 2 * q + 9, n), bh[1], bl[1]);
            mma16816(d1[b], l1, bh);
            mma16816(d1[b], h1, bl);
            mma16816(d1[b], h1, bh);
            mma16816(d2[b], l2, bh);
            mma16816(d2[b], h2, bl);
            mma16816(d2[b], h2, bh);
        }
    }
}

// For a bf16 right operand (exact): d += A_lo B + A_hi B with K = 16 per instruction; A's hi + lo
// carries 16 significant bits (relative error ~1e-5).  k_hi - k_lo a multiple of 16.
// B is a row-major [k][n] bf16 tile (B.cs == 1, row stride B.rs elements, a multiple of 8, rows 16-byte
// aligned): each k-step moves two n-blocks' fragments with one ldmatrix.x4.trans (lanes 8 i .. 8 i + 7
// address rows k0 + 8 (i % 2) .. + 7 of n-block b + i / 2).  NB even, n0 a multiple of 8.
template <int NB>
__device__ __forceinline__ void mma_strip_splitA_bf16(float (&d)[NB][4], const Tile& A, const TileH& B, int m0,
                                                      int n0, int k_lo, int k_hi, int lane) {
    static_assert(NB % 2 == 0, "n-blocks in pairs");
    const int g = lane >> 2, q = lane & 3;
    const int mi = lane >> 3, ri = lane & 7;
#pragma unroll 1
    for (int k0 = k_lo; k0 < k_hi; k0 += 16) {
        uint32_t ah[4], al[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = m0 + g + 8 * (i & 1), k = k0 + 2 * q + 8 * (i >> 1);
            split_bf16x2(A.at(r, k), A.at(r, k + 1), ah[i], al[i]);
        }
#pragma unroll
        for (int b = 0; b < NB; b += 2) {
            const __nv_bfloat16* row = B.p + (k0 + 8 * (mi & 1) + ri) * B.rs + n0 + 8 * (b + (mi >> 1));
            uint32_t bb[4];
            asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                         : "=r"(bb[0]), "=r"(bb[1]), "=r"(bb[2]), "=r"(bb[3])
                         : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(row)))
                         : "memory");
            mma16816(d[b], al, bb);
            mma16816(d[b], ah, bb);
            mma16816(d[b + 1], al, bb + 2);
            mma16816(d[b + 1], ah, bb + 2);
        }
    }
}

__device__ __forceinline__ void cp_async16(float* dst, const float* src) {
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory"); }

// Eight bf16 values (16 bytes) to fp32.
__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float* f) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

constexpr int P128 = 132, P64 = 68, P32 = 36;   // padded row strides (4 mod 32)

// shared-memory plan, in floats
constexpr int O_W = 0;                      // [64][P128]  phase 1: W;     phase 2: dk accumulation
constexpr int O_KG = O_W + 64 * P128;       // [64][P128]  phase 1: Kg;    phase 2: dq accumulation
constexpr int O_KD = O_KG + 64 * P128;      // [64][P128]  phase 1: Kd;    phase 2: dGamma accumulation
constexpr int O_AQ = O_KD + 64 * P128;      // [64][P64]   Aqk (phase 2: dA)
constexpr int O_N = O_AQ + 64 * P64;        // [64][P64]   N
constexpr int O_S0 = O_N + 64 * P64;        // [128][P32]  S0 slice       (phase 2: dT / dN / dL / dB)
constexpr int O_DS = O_S0 + 128 * P32;      // [128][P32]  dS_end slice   (phase 2: k_hat * r)
constexpr int O_DO = O_DS + 128 * P32;      // [64][P32]   dO slice       (phase 2 scratch from here)
constexpr int O_U = O_DO + 64 * P32;        // [64][P32]   U slice (starts as U0)
constexpr int O_VT = O_U + 64 * P32;        // [64][P32]   v - Kg S0 slice (starts as v)
constexpr int O_DU = O_VT + 64 * P32;       // [64][P32]   dU slice
constexpr int O_DY = O_DU + 64 * P32;       // [64][P32]   dY slice
constexpr int O_BETA = O_DY + 64 * P32;     // [64]
constexpr int O_GRAW = O_DO + 64 * P64;    // bf16 [64][128] g_raw tile, phase 2 (after dB: tmp is dead)
static_assert(O_GRAW >= O_DS + 64 * P128 && O_GRAW + 64 * 128 / 2 <= O_BETA, "g_raw tile inside the free tail");
constexpr int O_GPART = O_GRAW + 64 * 128 / 2;   // [4][128] column partials of sum_t dKd Kd, phase 2
static_assert(O_GPART + 4 * 128 <= O_BETA, "partials inside the free tail");
static_assert(2 * 16 * 256 <= 64 * P128 && 16 * 256 <= 64 * P64, "diagonal-pass scratch inside the R and N tiles");
constexpr int O_RED = O_BETA + 64;          // [64] dbeta, [128] Gamma_last gradient, [8] block sums, [256] dt_bias parts
constexpr int O_MBAR = O_RED + 64 + 128 + 8 + 256;   // 8-byte mbarrier + TMEM slot (4 floats)
constexpr int SMEM_FLOATS = O_MBAR + 4;
// Phase-1 tensor-core operands (bf16, K-major over the 32 value columns of a slice: km_bf16(row, j,
// 512, 128)), in the areas that phase 2 later fills with the accumulators: W area and Kd..N area.
constexpr uint32_t B_S0 = O_W * 4;                  // S0^T slice hi / lo   [128 c][32 j]  2 x 8 KB
constexpr uint32_t B_DS = B_S0 + 16384;             // dS_end^T slice hi / lo            2 x 8 KB
constexpr uint32_t B_U = O_KD * 4;                  // U slice hi / lo      [64 t][32 j]  2 x 4 KB
constexpr uint32_t B_DU = B_U + 8192;               // dU slice hi / lo
constexpr uint32_t B_VT = B_DU + 8192;              // (v - Kg S0) slice hi / lo
constexpr uint32_t B_MDY = B_VT + 8192;             // -dY slice hi / lo
constexpr uint32_t B_DO = B_MDY + 8192;             // dO slice (bf16, exact)
static_assert(B_DS + 16384 <= (uint32_t)O_KG * 4 && B_DO + 4096 <= (uint32_t)O_N * 4, "phase-1 operand areas");
// TMEM columns of the five M = 64 accumulators (rows t in lanes (t / 16) * 32 + t % 16)
constexpr uint32_t T_KG = 0, T_QG = 128, T_KD = 256, T_T = 384, T_A = 448;

}  // namespace

// Unbounded gate: the pairs inside each diagonal sub-block, which the factorised forms left out,
// directly.  Thread = (channel, two sub-blocks).  For every pair s <= t of a sub-block one decay
// exp(Gamma_t - Gamma_s) <= 1 (it can only underflow) serves all three sums (dq_A and dk_L of row t,
// dk_R of row s); the row-t terms go straight into the thread's own column of dq, dk and dGamma in
// shared memory, and dA, dB are warp-wide broadcasts.  The sub-block's Gamma, k and q of the thread's
// channel are first copied into shared scratch ([16][256], the thread's own column, so no barrier), where
// rolled loops index them cheaply: the gradient kernel is large enough that unrolled code here costs
// more in instruction fetch than it saves, and rolled loops over global rows wait on L2 every pair.
__device__ __noinline__ void diag_pairs(const float* __restrict__ Gm, const float* __restrict__ kh,
                                        const float* __restrict__ qh, const float* dA, const float* dB, float* sdq,
                                        float* sdk, float* sdG, float* sg, float* sk, float* sq, int tid) {
    constexpr int K = 128;
    const int cc = tid & 127;
#pragma unroll 1
    for (int bb = 0; bb < 2; ++bb) {
        const int t0 = 16 * (2 * (tid >> 7) + bb);
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int gi = (t0 + u) * K + cc;
            sg[u * 256 + tid] = Gm[gi];
            sk[u * 256 + tid] = kh[gi];
            sq[u * 256 + tid] = qh[gi];
        }
#pragma unroll 1
        for (int s = 0; s < 16; ++s) {
            const float ks = sk[s * 256 + tid], gs = sg[s * 256 + tid];
            const float* ca = dA + t0 * P64 + t0 + s;   // column s of the sub-block: ca[t * P64]
            const float* cb = dB + t0 * P64 + t0 + s;
            float dr = 0.f;
#pragma unroll 2
            for (int t = s; t < 16; ++t) {
                const float E = __expf(sg[t * 256 + tid] - gs);
                const float a = ca[t * P64], b = cb[t * P64];
                const float qt = sq[t * 256 + tid], kt = sk[t * 256 + tid];
                const float x = a * ks * E, y = b * ks * E;
                const int r = (t0 + t) * P128 + cc;
                sdq[r] += x;
                sdk[r] += y;
                sdG[r] += qt * x + kt * y;
                dr += (a * qt + b * kt) * E;
            }
            const int r = (t0 + s) * P128 + cc;
            sdk[r] += dr;
            sdG[r] -= ks * dr;
        }
    }
}

// SP: the unbounded (softplus) gate, whose diagonal sub-blocks are summed pair by pair.
template <bool SP>
__global__ void __launch_bounds__(256, 1) grad_tc_kernel(Params p) {
    extern __shared__ float sm[];
    const int c = blockIdx.x, h = blockIdx.y;
    if (c >= p.chunk_off[p.N]) return;
    constexpr int K = 128, V = 128;
    const int H = p.H;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n = chunk_segment(p, c);
    const int tok0 = seg_begin(p, n) + (c - p.chunk_off[n]) * kChunk;
    const int len = min(kChunk, seg_end(p, n) - tok0);
    const RecLayout L = RecLayout::make(K, V);
    const float* rec = p.rec + ((size_t)c * H + h) * p.rec_stride;
    // the chains' per-chunk tiles, each in x4 order
    const float* S0g = p.states + ((size_t)c * H + h) * K * V;
    const float* dSg = p.dstates + ((size_t)c * H + h) * K * V;
    const float* Ug = p.chunk_u + ((size_t)c * H + h) * 64 * V;     // U = U0 - W S0 (recompute chain)
    const float* dUg = p.chunk_du + ((size_t)c * H + h) * 64 * V;   // dU = scale Aqk^T dO + Kd dS_end (reverse chain)
    float* sW = sm + O_W;
    float* sKg = sm + O_KG;
    float* sKd = sm + O_KD;
    float* sAq = sm + O_AQ;
    float* sN = sm + O_N;
    float* sS0 = sm + O_S0;
    float* sdS = sm + O_DS;
    float* sdO = sm + O_DO;
    float* sU = sm + O_U;
    float* sVt = sm + O_VT;
    float* sdU = sm + O_DU;
    float* sdY = sm + O_DY;
    float* sbeta = sm + O_BETA;
    float* sred = sm + O_RED;
    const float scale = p.scale;

    // chunk-wide operands (16-byte asynchronous copies; completed by the first slice's wait)
    // (U and dU come per slice from the two state chains, so W, Kd and A_qk are not needed here)
    for (int i = tid; i < 64 * K / 4; i += 256) {
        const int t = i >> 5, c4 = (i & 31) * 4;
        cp_async16(sKg + t * P128 + c4, rec + L.Kg + t * K + c4);
    }
    for (int i = tid; i < 64 * 64 / 4; i += 256) {
        const int t = i >> 4, s4 = (i & 15) * 4;
        cp_async16(sN + t * P64 + s4, rec + L.N + t * 64 + s4);
    }
    if (tid < 16) cp_async16(sbeta + 4 * tid, rec + L.beta + 4 * tid);
    // warm L2 with the state slices, U0, dout and v that the four V-slice loads read
    if (tid == 0) {
        const uint32_t kv = K * V * 4u;
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(S0g)), "r"(kv) : "memory");
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(dSg)), "r"(kv) : "memory");
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(Ug)), "r"(64u * V * 4u)
                     : "memory");
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(dUg)), "r"(64u * V * 4u)
                     : "memory");
        // the record fields phase 2 reads row by row from global memory, Gamma, q_hat, k_hat (adjacent),
        // requested now so they sit in L2 by then (Qg, Kg and Kd are formed from them where needed)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(rec + L.G)),
                     "r"(3u * 64u * K * 4u) : "memory");
    }
    if (tid >= 64 && tid < 64 + len) {   // one row of dout and of v per token (256 bytes, or 128 at V = 64)
        const size_t row = ((size_t)(tok0 + tid - 64) * H + h) * p.V;
        const char* po = reinterpret_cast<const char*>(static_cast<const __nv_bfloat16*>(p.dout) + row);
        const char* pv = reinterpret_cast<const char*>(static_cast<const __nv_bfloat16*>(p.v) + row);
        asm volatile("prefetch.global.L2 [%0];" ::"l"(po));
        asm volatile("prefetch.global.L2 [%0];" ::"l"(pv));
        if (p.V > 64) {
            asm volatile("prefetch.global.L2 [%0];" ::"l"(po + 128));
            asm volatile("prefetch.global.L2 [%0];" ::"l"(pv + 128));
        }
    }

    // accumulators over the four 32-column slices of V (register fragments)
    //   dKg, dQg, dKd [64 x 128]: warp w owns rows 16 (w / 2) .. +16, cols 64 (w % 2) .. +64 (8 blocks)
    //   dT, dA [64 x 64]: warp w owns rows 16 (w / 2), cols 32 (w % 2) .. +32 (4 blocks)
    // The slice contributions to dKg (-dY S0^T), dQg (dO S0^T), dKd (U dS^T), dT (dU Vt^T) and dA (dO U^T)
    // accumulate over the four slices in tensor memory: tcgen05 MMAs on bf16 hi / lo operands
    // (hi*hi + hi*lo + lo*hi; dO is bf16 and exact), ~1e-5 relative.  dKd enters dGamma twice (-dKd Kd
    // per token, +sum_t dKd Kd at Gamma_last) and the two cancel in the reverse cumulative sum, so it
    // needs that precision; the others get it for free.
    uint64_t* mbar = reinterpret_cast<uint64_t*>(sm + O_MBAR);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + O_MBAR + 2);
    uint8_t* smb = reinterpret_cast<uint8_t*>(sm);
    if (tid == 0) {
        mbar_init(mbar, 1);
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(tslot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    bool mma_ok = true;
    float dgc = 0.f;   // thread tid < 128: sum_j dS_end[c][j] S0[c][j] for channel c = tid
    const int wm0 = 16 * (warp >> 1);

    // Slice z's tiles pass through registers: x4-ordered tiles with consecutive threads on
    // consecutive rows' 16-byte chunks, dO and v one row-quarter per thread.  The next slice's loads
    // are issued as soon as the current slice is in shared memory, so they fly during its products.
    float4 ra[4], rb[4], ru[2], rdu[2];
    uint4 ro, rv;
    const int tq = tid >> 2, j8q = (tid & 3) * 8;   // dO / v: row and first column of this thread
    auto fetch_slice = [&](int z) {
        const int j0 = 32 * z;
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int i = tid + 256 * it, cc = i & (K - 1), j4 = (i / K) * 4;
            ra[it] = *reinterpret_cast<const float4*>(S0g + x4_off(cc, j0 + j4, K));
            rb[it] = *reinterpret_cast<const float4*>(dSg + x4_off(cc, j0 + j4, K));
        }
#pragma unroll
        for (int it = 0; it < 2; ++it) {
            const int i = tid + 256 * it, r = i & 63, j4 = (i >> 6) * 4;
            ru[it] = *reinterpret_cast<const float4*>(Ug + x4_off(r, j0 + j4, 64));
            rdu[it] = *reinterpret_cast<const float4*>(dUg + x4_off(r, j0 + j4, 64));
        }
        ro = rv = make_uint4(0u, 0u, 0u, 0u);
        if (tq < len && j0 + j8q < p.V) {   // (V = 64 heads: the upper value columns stay zero)
            const size_t gi = ((size_t)(tok0 + tq) * H + h) * p.V + j0 + j8q;
            ro = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.dout) + gi);
            rv = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.v) + gi);
        }
    };
    auto stage = [&]() {
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int i = tid + 256 * it, cc = i & (K - 1), j4 = (i / K) * 4;
            *reinterpret_cast<float4*>(sS0 + cc * P32 + j4) = ra[it];
            *reinterpret_cast<float4*>(sdS + cc * P32 + j4) = rb[it];
        }
#pragma unroll
        for (int it = 0; it < 2; ++it) {
            const int i = tid + 256 * it, r = i & 63, j4 = (i >> 6) * 4;
            *reinterpret_cast<float4*>(sU + r * P32 + j4) = ru[it];
            *reinterpret_cast<float4*>(sdU + r * P32 + j4) = rdu[it];
        }
        float fo[8], fv[8];
        bf16x8_to_f32(ro, fo);
        bf16x8_to_f32(rv, fv);
        *reinterpret_cast<float4*>(sdO + tq * P32 + j8q) = make_float4(fo[0], fo[1], fo[2], fo[3]);
        *reinterpret_cast<float4*>(sdO + tq * P32 + j8q + 4) = make_float4(fo[4], fo[5], fo[6], fo[7]);
        *reinterpret_cast<float4*>(sVt + tq * P32 + j8q) = make_float4(fv[0], fv[1], fv[2], fv[3]);
        *reinterpret_cast<float4*>(sVt + tq * P32 + j8q + 4) = make_float4(fv[4], fv[5], fv[6], fv[7]);
    };
    fetch_slice(0);

    for (int z = 0; z < 4; ++z) {
        const int j0 = 32 * z;
        __syncthreads();   // previous slice's readers are done
        stage();
        if (z + 1 < 4) fetch_slice(z + 1);
        if (z == 0) cp_async_wait_all();   // the record tiles requested before the loop
        __syncthreads();
        // Vt = v - Kg S0 (64 x 32): warp w takes rows 16 (w % 4), columns 16 (w / 4) .. + 16
        {
            const int m0 = 16 * (warp & 3), n0 = 16 * (warp >> 2);
            float d[2][4];
#pragma unroll
            for (int b = 0; b < 2; ++b)
#pragma unroll
                for (int e = 0; e < 4; ++e) d[b][e] = 0.f;
            mma_strip3_bf16<2>(d, Tile{sKg, P128, 1}, Tile{sS0, P32, 1}, m0, n0, 0, K, lane);
#pragma unroll
            for (int b = 0; b < 2; ++b)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    int r, cc;
                    frag_rc(lane, e, m0, n0 + 8 * b, r, cc);
                    sVt[r * P32 + cc] -= d[b][e];
                }
        }
        __syncthreads();
        // dY = Diag(beta) N^T dU  (-> dv); N is lower triangular: rows s see t >= s only
        {
            const int m0 = 16 * (warp >> 1), n0 = 16 * (warp & 1);
            float d[2][4];
#pragma unroll
            for (int b = 0; b < 2; ++b)
#pragma unroll
                for (int e = 0; e < 4; ++e) d[b][e] = 0.f;
            mma_strip3_bf16<2>(d, Tile{sN, 1, P64}, Tile{sdU, P32, 1}, m0, n0, m0, 64, lane);
#pragma unroll
            for (int b = 0; b < 2; ++b)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    int r, cc;
                    frag_rc(lane, e, m0, n0 + 8 * b, r, cc);
                    sdY[r * P32 + cc] = sbeta[r] * d[b][e];
                }
        }
        __syncthreads();
        {   // dv = dY for this slice, from the tile: 32 columns = one 128-byte row segment per 4 threads
            const int r = tid >> 2, c8 = (tid & 3) * 8;
            if (r < len && j0 + c8 < p.V) {
                float* dst = p.dv + ((size_t)(tok0 + r) * H + h) * p.V + j0 + c8;
                *reinterpret_cast<float4*>(dst) = *reinterpret_cast<const float4*>(sdY + r * P32 + c8);
                *reinterpret_cast<float4*>(dst + 4) = *reinterpret_cast<const float4*>(sdY + r * P32 + c8 + 4);
            }
        }
        // slice contributions on the tensor cores: the previous slice's MMAs must be done with the
        // operand tiles before they are rewritten
        if (z > 0 && !mbar_wait(mbar, (z - 1) & 1)) mma_ok = false;
        tc_fence_after();
        {
            // groups of 8 consecutive j of one row; 8 consecutive groups share j and take rows r..r+7
            auto put = [&](uint32_t off, const float* src, int row, int j8, float sg) {
                float x[8];
                *reinterpret_cast<float4*>(x) = *reinterpret_cast<const float4*>(src + row * P32 + j8);
                *reinterpret_cast<float4*>(x + 4) = *reinterpret_cast<const float4*>(src + row * P32 + j8 + 4);
                float hv[8], lv[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float v = sg * x[e];
                    hv[e] = __bfloat162float(__float2bfloat16_rn(v));
                    lv[e] = v - hv[e];
                }
                const uint32_t o = off + km_bf16(row, j8, 512, 128);
                *reinterpret_cast<uint4*>(smb + o) = pack8_bf16(hv);
                if (off != B_DO) *reinterpret_cast<uint4*>(smb + o + (off >= B_U ? 4096u : 8192u)) = pack8_bf16(lv);
            };
            for (int g = tid; g < 128 * 4; g += 256) {
                const int row = (g & 7) | ((g >> 5) << 3), j8 = ((g >> 3) & 3) * 8;
                put(B_S0, sS0, row, j8, 1.f);
                put(B_DS, sdS, row, j8, 1.f);
            }
            {
                const int g = tid, row = (g & 7) | ((g >> 5) << 3), j8 = ((g >> 3) & 3) * 8;   // 64 rows x 4
                put(B_U, sU, row, j8, 1.f);
                put(B_DU, sdU, row, j8, 1.f);
                put(B_VT, sVt, row, j8, 1.f);
                put(B_MDY, sdY, row, j8, -1.f);
                put(B_DO, sdO, row, j8, 1.f);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (tid == 0) {
            const uint32_t base = smem_u32(sm);
            constexpr uint32_t i128 = idesc_bf16(64, 128, 0, 0), i64 = idesc_bf16(64, 64, 0, 0);
            // D (+)= A B^T over K = 32 (two K = 16 steps); A / B K-major with 8-row groups 512 B apart
            auto mm = [&](uint32_t d, uint32_t a, uint32_t b, uint32_t id, bool first) {
                for (int kk = 0; kk < 2; ++kk)
                    mma_bf16(d, smem_desc(base + a + kk * 256, 128, 512), smem_desc(base + b + kk * 256, 128, 512), id,
                             (first && kk == 0) ? 0u : 1u);
            };
            const bool f = z == 0;
            mm(tmem + T_KG, B_MDY + 4096, B_S0, i128, f);          // -dY S0^T: lo * hi, hi * lo, hi * hi
            mm(tmem + T_KG, B_MDY, B_S0 + 8192, i128, false);
            mm(tmem + T_KG, B_MDY, B_S0, i128, false);
            mm(tmem + T_QG, B_DO, B_S0 + 8192, i128, f);           // dO S0^T (dO exact)
            mm(tmem + T_QG, B_DO, B_S0, i128, false);
            mm(tmem + T_KD, B_U + 4096, B_DS, i128, f);            // U dS^T
            mm(tmem + T_KD, B_U, B_DS + 8192, i128, false);
            mm(tmem + T_KD, B_U, B_DS, i128, false);
            mm(tmem + T_T, B_DU + 4096, B_VT, i64, f);             // dU Vt^T
            mm(tmem + T_T, B_DU, B_VT + 4096, i64, false);
            mm(tmem + T_T, B_DU, B_VT, i64, false);
            mm(tmem + T_A, B_DO, B_U + 4096, i64, f);              // dO U^T
            mm(tmem + T_A, B_DO, B_U, i64, false);
            mma_commit(mbar);
        }
        if (tid < K) {
            float acc = 0.f;
#pragma unroll 8
            for (int j = 0; j < 32; ++j) acc += sdS[tid * P32 + j] * sS0[tid * P32 + j];
            dgc += acc;
        }
    }
    __syncthreads();

    // ---- phase 2: write the accumulators out (dKg -> sW, dQg -> sKg, dKd -> sKd, dT -> sS0, dA -> sAq)
    if (!mbar_wait(mbar, 3 & 1)) mma_ok = false;
    tc_fence_after();
    if (!__syncthreads_and(mma_ok ? 1 : 0)) {
        // a tensor-core wait ran out: record it and leave (results of this chunk are void)
        if (tid == 0) record_error(p.status, KDA_ERR_TIMEOUT);
        if (tid == 0) mbar_wait(mbar, 1, 1u << 16);
        tc_fence_before();
        __syncthreads();
        if (warp == 0) tmem_dealloc(tmem, 512);
        return;
    }
    float* dKg = sW;
    float* dQg = sKg;
    float* dKdm = sKd;
    float* dT = sS0;     // [64][P64]
    float* dA = sAq;     // [64][P64]
    {
        // M = 64 accumulators: warp w reads lane quarter w % 4 (rows 16 (w % 4) + lane, lane < 16);
        // warps w and w + 4 split the columns
        const int r = 16 * (warp & 3) + (lane & 15), half = warp >> 2;
        const uint32_t lb = static_cast<uint32_t>((warp & 3) * 32) << 16;
        auto drain = [&](uint32_t col0, int ncols, float* dst, int stride, float mul, bool lower) {
            for (int cb = 0; cb < ncols; cb += 32) {
                float d[32];
                const uint32_t c0 = col0 + half * ncols + cb;
                tmem_ld16(tmem + lb + c0, d);
                tmem_ld16(tmem + lb + c0 + 16, d + 16);
                tmem_ld_wait();
                if (lane < 16)
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int cc = half * ncols + cb + j;
                        dst[r * stride + cc] = (lower && cc > r) ? 0.f : mul * d[j];
                    }
            }
        };
        drain(T_KG, 64, dKg, P128, 1.f, false);
        drain(T_QG, 64, dQg, P128, scale, false);
        drain(T_KD, 64, dKdm, P128, 1.f, false);
        drain(T_T, 32, dT, P64, 1.f, false);
        drain(T_A, 32, dA, P64, scale, true);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
    // Gamma_last gathers exp(Gamma_last) rowsum(dS_end * S0) and sum_t dKd Kd; the combine below
    // forms the second sum (partials per 16-row block in sgpart) with the Kd it uses itself
    float* sgl = sred + 64;
    float* sgpart = sm + O_GPART;   // [4][128]
    // dbeta_s = sum_t N[t][s] dT[t][s];  dN = dT Diag(beta)
    float* sdbeta = sred;
    if (tid < 64) {
        float acc = 0.f;
        for (int t = 0; t < 64; ++t) acc += sN[t * P64 + tid] * dT[t * P64 + tid];
        sdbeta[tid] = acc;
    }
    __syncthreads();
    for (int i = tid; i < 64 * 64; i += 256) {
        const int t = i >> 6, s = i & 63;
        dT[t * P64 + s] *= sbeta[s];   // dN
    }
    __syncthreads();
    // tmp = N^T dN ; dL = -(tmp N^T), strict lower ; dB = Diag(beta) dL
    float* tmp = sdO;   // [64][P64] scratch (phase-1 slice buffers are free)
    {
        float d[4][4];
#pragma unroll
        for (int b = 0; b < 4; ++b)
#pragma unroll
            for (int e = 0; e < 4; ++e) d[b][e] = 0.f;
        mma_strip3_bf16<4>(d, Tile{sN, 1, P64}, Tile{dT, P64, 1}, wm0, 32 * (warp & 1), wm0, 64, lane);   // N[t][s], t >= s
#pragma unroll
        for (int b = 0; b < 4; ++b)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                int r, cc;
                frag_rc(lane, e, wm0, 32 * (warp & 1) + 8 * b, r, cc);
                tmp[r * P64 + cc] = d[b][e];
            }
    }
    __syncthreads();
    float* dB = dT;
    {
        float d[4][4];
#pragma unroll
        for (int b = 0; b < 4; ++b)
#pragma unroll
            for (int e = 0; e < 4; ++e) d[b][e] = 0.f;
        mma_strip3_bf16<4>(d, Tile{tmp, P64, 1}, Tile{sN, 1, P64}, wm0, 32 * (warp & 1), 0, 64, lane);
        __syncwarp();
#pragma unroll
        for (int b = 0; b < 4; ++b)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                int r, cc;
                frag_rc(lane, e, wm0, 32 * (warp & 1) + 8 * b, r, cc);
                dB[r * P64 + cc] = cc < r ? -d[b][e] : 0.f;   // dL (beta applied below)
            }
    }
    __syncthreads();
    {   // dbeta_t += sum_{s<t} dL[t][s] Bkk[t][s]; warp w takes rows w, w + 8, ... (loads first)
        float bv[8][2], acc[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const float* brow = rec + L.B + (warp + 8 * u) * 64;
            bv[u][0] = brow[lane];
            bv[u][1] = brow[lane + 32];
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int t = warp + 8 * u;
            acc[u] = dB[t * P64 + lane] * bv[u][0] + dB[t * P64 + lane + 32] * bv[u][1];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
            for (int u = 0; u < 8; ++u) acc[u] += __shfl_xor_sync(0xffffffffu, acc[u], o);
        if (lane == 0)
#pragma unroll
            for (int u = 0; u < 8; ++u) sdbeta[warp + 8 * u] += acc[u];
    }
    __syncthreads();
    for (int i = tid; i < 64 * 64; i += 256) {
        const int t = i >> 6, s = i & 63;
        dB[t * P64 + s] *= sbeta[t];
    }
    // the g_raw tile of the gate backward, staged now so its latency hides behind the bilinear forms
    __nv_bfloat16* sgraw = reinterpret_cast<__nv_bfloat16*>(sm + O_GRAW);
    for (int i = tid; i < 64 * 16; i += 256) {
        const int t = i >> 4, c8 = (i & 15) * 8;
        if (t < len && c8 < p.K)
            cp_async16(reinterpret_cast<float*>(sgraw + t * 128 + c8),
                       reinterpret_cast<const float*>(static_cast<const __nv_bfloat16*>(p.g_raw) +
                                                      ((size_t)(tok0 + t) * H + h) * p.K + c8));
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    // R[s][c] = k_hat[s][c] exp(G_{b(s)+1,c} - Gamma[s][c]) (<= 1), with G_{b+1} = Gamma at the end of
    // sub-block b.  Stored in the phase-1 dS_end area: [64][P128].
    float* R = sdS;
    const float* Gm = rec + L.G;
    const float* qh = rec + L.qh;
    const float* kh = rec + L.kh;
#pragma unroll
    for (int it = 0; it < 64 * K / 4 / 256; ++it) {   // float4 per thread per trip, all loads independent
        const int i4 = tid + 256 * it, s = i4 >> 5, c4 = (i4 & 31) * 4;
        const float4 gr = *reinterpret_cast<const float4*>(Gm + (16 * (s >> 4) + 15) * K + c4);
        const float4 gs = *reinterpret_cast<const float4*>(Gm + s * K + c4);
        const float4 kv = *reinterpret_cast<const float4*>(kh + s * K + c4);
        *reinterpret_cast<float4*>(R + s * P128 + c4) =
            make_float4(kv.x * __expf(gr.x - gs.x), kv.y * __expf(gr.y - gs.y), kv.z * __expf(gr.z - gs.z),
                        kv.w * __expf(gr.w - gs.w));
    }
    __syncthreads();

    // ---- decayed bilinear forms.  For s in sub-block j: exp(Gamma_t - Gamma_s) = l_j(t) r(s) with
    // l_j(t) = exp(Gamma_t - G_{j+1}) (only t >= 16 j contribute: dA, dB are lower triangular).
    //   dq_A[t]  = sum_j l_j(t) (dA[:, J] R[J, :])[t]
    //   dk_L[t]  = sum_j l_j(t) (dB[:, J] R[J, :])[t]
    //   dk_R[s]  = r(s) sum_t (dA[t][s] q[t] + dB[t][s] k[t]) l_j(t),   s in J
    // Each warp owns the same 8 blocks (rows wm0, cols 64 (w % 2) + 8 b) of all three results.
    // Under the unbounded gate nothing bounds l_j(t) inside sub-block j itself, so there the
    // factorised forms cover only the pairs across sub-blocks and the diagonal sub-block is summed
    // directly below.
    constexpr bool sp = SP;
    float fq[8][4], fkl[8][4], fkr[8][4];
#pragma unroll
    for (int b = 0; b < 8; ++b)
#pragma unroll
        for (int e = 0; e < 4; ++e) fq[b][e] = fkl[b][e] = fkr[b][e] = 0.f;
    const int bt = warp >> 1;   // sub-block of this warp's rows
    {
        // Gamma at this thread's fragment elements (the same for every j), loaded once; Gamma at the
        // end of sub-block j for its columns, loaded before the sub-block's products so the L2
        // latency hides behind them
        float grow[8][4];
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            int r0, c0;
            frag_rc(lane, 0, wm0, 64 * (warp & 1) + 8 * b, r0, c0);   // (r0, c0 + e), (r0 + 8, c0 + e)
            const float2 x0 = *reinterpret_cast<const float2*>(Gm + r0 * K + c0);
            const float2 x1 = *reinterpret_cast<const float2*>(Gm + (r0 + 8) * K + c0);
            grow[b][0] = x0.x; grow[b][1] = x0.y; grow[b][2] = x1.x; grow[b][3] = x1.y;
        }
        for (int j = 0; j <= (sp ? bt - 1 : bt); ++j) {
            float2 gend[8];
#pragma unroll
            for (int b = 0; b < 8; ++b) {
                int r0, c0;
                frag_rc(lane, 0, wm0, 64 * (warp & 1) + 8 * b, r0, c0);
                gend[b] = *reinterpret_cast<const float2*>(Gm + (16 * j + 15) * K + c0);
            }
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {
                const int n0 = 64 * (warp & 1) + 32 * hb;
                float dq[4][4], dk[4][4];
#pragma unroll
                for (int b = 0; b < 4; ++b)
#pragma unroll
                    for (int e = 0; e < 4; ++e) dq[b][e] = dk[b][e] = 0.f;
                mma_strip3_pair_bf16<4>(dq, dk, Tile{dA, P64, 1}, Tile{dB, P64, 1}, Tile{R, P128, 1}, wm0, n0, 16 * j,
                                   16 * j + 16, lane);
#pragma unroll
                for (int b = 0; b < 4; ++b)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int bb = 4 * hb + b;
                        const float l = __expf(grow[bb][e] - ((e & 1) ? gend[bb].y : gend[bb].x));
                        fq[bb][e] += l * dq[b][e];
                        fkl[bb][e] += l * dk[b][e];
                    }
            }
        }
    }
    // dk_R: rows s of this warp's sub-block bt; sum over t >= 16 bt.  One k-step loads and splits the
    // dA / dB fragments once and feeds the eight column blocks' independent accumulators.
    {
        const int j = bt;
        const int g = lane >> 2, qd = lane & 3;
        float gref[8];
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            gref[b] = Gm[(16 * j + 15) * K + 64 * (warp & 1) + 8 * b + g];
#pragma unroll
            for (int e = 0; e < 4; ++e) fkr[b][e] = 0.f;
        }
        // the record values of the next k-step (Gamma, q_hat, k_hat at rows t1, t2 and this thread's
        // eight columns) are loaded while the current step runs its products
        float ng[2][8], nq[2][8], nk[2][8];
        auto fetch_step = [&](int k0) {
#pragma unroll
            for (int b = 0; b < 8; ++b) {
                const int cn = 64 * (warp & 1) + 8 * b + g;
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int t = k0 + qd + 4 * i;
                    ng[i][b] = Gm[t * K + cn];
                    nq[i][b] = qh[t * K + cn];
                    nk[i][b] = kh[t * K + cn];
                }
            }
        };
        const int kfirst = sp ? 16 * j + 16 : 16 * j;
        if (kfirst < 64) fetch_step(kfirst);
#pragma unroll 1
        for (int k0 = kfirst; k0 < 64; k0 += 8) {
            float cg[2][8], cq[2][8], ck[2][8];
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
                for (int b = 0; b < 8; ++b) {
                    cg[i][b] = ng[i][b];
                    cq[i][b] = nq[i][b];
                    ck[i][b] = nk[i][b];
                }
            if (k0 + 8 < 64) fetch_step(k0 + 8);
            uint32_t aAh[4], aAl[4], aBh[4], aBl[4];
            // A(m = s, k = t) = dA[t][s] (transposed access), rows s = wm0 + ...
            split_tf32(dA[(k0 + qd) * P64 + wm0 + g], aAh[0], aAl[0]);
            split_tf32(dA[(k0 + qd) * P64 + wm0 + g + 8], aAh[1], aAl[1]);
            split_tf32(dA[(k0 + qd + 4) * P64 + wm0 + g], aAh[2], aAl[2]);
            split_tf32(dA[(k0 + qd + 4) * P64 + wm0 + g + 8], aAh[3], aAl[3]);
            split_tf32(dB[(k0 + qd) * P64 + wm0 + g], aBh[0], aBl[0]);
            split_tf32(dB[(k0 + qd) * P64 + wm0 + g + 8], aBh[1], aBl[1]);
            split_tf32(dB[(k0 + qd + 4) * P64 + wm0 + g], aBh[2], aBl[2]);
            split_tf32(dB[(k0 + qd + 4) * P64 + wm0 + g + 8], aBh[3], aBl[3]);
#pragma unroll
            for (int b = 0; b < 8; ++b) {
                uint32_t bqh[2], bql[2], bkh[2], bkl[2];
                const float l1 = __expf(cg[0][b] - gref[b]), l2 = __expf(cg[1][b] - gref[b]);
                split_tf32(cq[0][b] * l1, bqh[0], bql[0]);
                split_tf32(cq[1][b] * l2, bqh[1], bql[1]);
                split_tf32(ck[0][b] * l1, bkh[0], bkl[0]);
                split_tf32(ck[1][b] * l2, bkh[1], bkl[1]);
                mma1688(fkr[b], aAl, bqh);
                mma1688(fkr[b], aAh, bql);
                mma1688(fkr[b], aAh, bqh);
                mma1688(fkr[b], aBl, bkh);
                mma1688(fkr[b], aBh, bkl);
                mma1688(fkr[b], aBh, bkh);
            }
        }
#pragma unroll
        for (int b = 0; b < 8; ++b)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                int r, cc;
                frag_rc(lane, e, wm0, 64 * (warp & 1) + 8 * b, r, cc);
                fkr[b][e] *= __expf(Gm[(16 * j + 15) * K + cc] - Gm[r * K + cc]);
            }
    }
    __syncthreads();   // dKg / dQg / dKd are read below by their owning threads only, R and dA/dB are done
    // combine: dq = dq_A + dQg e^G ; dk = dk_L + dk_R + dKg e^G + dKd e^{Gc - G} ;
    //          dGamma = q dq_A + k dk_L - k dk_R + dQg Qg + dKg Kg - dKd Kd
    float* sdq = dQg;     // in place: the owning thread reads then overwrites
    float* sdk = dKg;
    float* sdG = dKdm;
    // the record rows of block b + 1 are fetched while block b is combined (global loads: L2 latency);
    // Qg = q_hat e^Gamma, Kg = k_hat e^Gamma and Kd = k_hat e^(Gamma_last - Gamma) are formed here
    float2 G[2][2], Q[2][2], Kk[2][2];
    auto fetch = [&](int b, int buf) {
        int r0, c0;
        frag_rc(lane, 0, wm0, 64 * (warp & 1) + 8 * b, r0, c0);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int gi = (r0 + 8 * hh) * K + c0;
            G[buf][hh] = *reinterpret_cast<const float2*>(Gm + gi);
            Q[buf][hh] = *reinterpret_cast<const float2*>(qh + gi);
            Kk[buf][hh] = *reinterpret_cast<const float2*>(kh + gi);
        }
    };
    fetch(0, 0);
    float2 Gcs[8];   // Gamma_last at this thread's columns
#pragma unroll
    for (int b = 0; b < 8; ++b) {
        int r0, c0;
        frag_rc(lane, 0, wm0, 64 * (warp & 1) + 8 * b, r0, c0);
        Gcs[b] = *reinterpret_cast<const float2*>(Gm + 63 * K + c0);
    }
    // the Gamma_last gradient's sum_t dKd Kd, per column over this warp's 16 rows (the same rounded Kd
    // as the per-token term of dGamma, with which it cancels)
    float csum[8][2];
#pragma unroll
    for (int b = 0; b < 8; ++b) {
        const int cur = b & 1;
        if (b + 1 < 8) fetch(b + 1, cur ^ 1);
        const int n0 = 64 * (warp & 1) + 8 * b;
        int r0, c0;
        frag_rc(lane, 0, wm0, n0, r0, c0);   // elements (r0, c0 + e), (r0 + 8, c0 + e), e = 0, 1
        const float2 Gc = Gcs[b];
        csum[b][0] = csum[b][1] = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int hh = e >> 1, lo = e & 1;
            const int r = r0 + 8 * hh, cc = c0 + lo;
            const float g = lo ? G[cur][hh].y : G[cur][hh].x, gc = lo ? Gc.y : Gc.x;
            const float q = lo ? Q[cur][hh].y : Q[cur][hh].x, k = lo ? Kk[cur][hh].y : Kk[cur][hh].x;
            const float eG = __expf(g), eD = __expf(gc - g);
            const float qg = q * eG, kg = k * eG, kd = k * eD;
            const float vQg = dQg[r * P128 + cc], vKg = dKg[r * P128 + cc], vKd = dKdm[r * P128 + cc];
            const float dq = fq[b][e] + vQg * eG;
            const float dk = fkl[b][e] + fkr[b][e] + vKg * eG + vKd * eD;
            const float dG = q * fq[b][e] + k * fkl[b][e] - k * fkr[b][e] + vQg * qg + vKg * kg - vKd * kd;
            sdq[r * P128 + cc] = dq;
            sdk[r * P128 + cc] = dk;
            sdG[r * P128 + cc] = dG;
            csum[b][lo] += vKd * kd;
        }
    }
    // column sums over the warp's rows (lanes of equal lane % 4 share columns), one partial per
    // row block of 16 and column
#pragma unroll
    for (int b = 0; b < 8; ++b)
#pragma unroll
        for (int lo = 0; lo < 2; ++lo) {
            float v = csum[b][lo];
            v += __shfl_xor_sync(0xffffffffu, v, 4);
            v += __shfl_xor_sync(0xffffffffu, v, 8);
            v += __shfl_xor_sync(0xffffffffu, v, 16);
            if (lane < 4) sgpart[(warp >> 1) * K + 64 * (warp & 1) + 8 * b + 2 * lane + lo] = v;
        }
    __syncthreads();
    if (tid < K)
        sgl[tid] = rec[L.gC + tid] * dgc + sgpart[tid] + sgpart[K + tid] + sgpart[2 * K + tid] + sgpart[3 * K + tid];
    if (sp) {
        // scratch: the R tile's area (dead since the bilinear forms) and N's (dead since dL)
        diag_pairs(Gm, kh, qh, dA, dB, sdq, sdk, sdG, R, R + 16 * 256, sN, tid);
        __syncthreads();
    }
    // reverse cumulative sum over t (plus the Gamma_last term) gives dg
    if (tid < K) {
        float run = sgl[tid];
        for (int t = 63; t >= 0; --t) {
            run += sdG[t * P128 + tid];
            sdG[t * P128 + tid] = run;
        }
    }
    __syncthreads();
    // ---- prologue backward: L2 norms, sigmoid(beta), the gate
    for (int t0 = warp; t0 < len; t0 += 16) {   // rows t0 and t0 + 8 of this warp, interleaved
        float qv[2][4], kv[2][4], sq[2] = {0.f, 0.f}, sk[2] = {0.f, 0.f};
#pragma unroll
        for (int w2 = 0; w2 < 2; ++w2) {
            const int t = min(t0 + 8 * w2, 63);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int cc = lane + 32 * u;
                qv[w2][u] = qh[t * K + cc];
                kv[w2][u] = kh[t * K + cc];
            }
        }
#pragma unroll
        for (int w2 = 0; w2 < 2; ++w2) {
            const int t = min(t0 + 8 * w2, 63);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int cc = lane + 32 * u;
                sq[w2] += qv[w2][u] * sdq[t * P128 + cc];
                sk[w2] += kv[w2][u] * sdk[t * P128 + cc];
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
            for (int w2 = 0; w2 < 2; ++w2) {
                sq[w2] += __shfl_xor_sync(0xffffffffu, sq[w2], o);
                sk[w2] += __shfl_xor_sync(0xffffffffu, sk[w2], o);
            }
#pragma unroll
        for (int w2 = 0; w2 < 2; ++w2) {
            const int t = t0 + 8 * w2;
            if (t >= len) continue;
            const size_t row = (size_t)(tok0 + t) * H + h;
            const float rq = rec[L.rn + t], rk = rec[L.rn + 64 + t];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int cc = lane + 32 * u;
                if (cc < p.K) {   // K = 64 heads: the padded channels are not written
                    p.dq_v[row * p.K + cc] = rq * (sdq[t * P128 + cc] - qv[w2][u] * sq[w2]);
                    p.dk_v[row * p.K + cc] = rk * (sdk[t * P128 + cc] - kv[w2][u] * sk[w2]);
                }
            }
            if (lane == 0) {
                const float b = sbeta[t];
                p.dbeta_raw[row] = sdbeta[t] * b * (1.f - b);
            }
        }
    }
    // gate backward: thread (channel cc, parity hf) takes tokens hf, hf + 2, ...
    float alog_part = 0.f;
    {
        const int cc = tid & 127, hf = tid >> 7;
        const bool ch = cc < p.K;   // a real channel (K = 64 heads are padded to 128)
        const float ea = expf(p.a_log[h]);
        const float dtbv = ch ? p.dt_bias[h * p.K + cc] : 0.f;
        float* __restrict__ dgr = p.dg_raw;
        asm volatile("cp.async.wait_group 0;" ::: "memory");
        __syncthreads();
        float gv[32];
#pragma unroll
        for (int u = 0; u < 32; ++u) {
            const int t = hf + 2 * u;
            gv[u] = t < len && ch ? __bfloat162float(sgraw[t * 128 + cc]) : 0.f;
        }
        float dtb = 0.f;
#pragma unroll
        for (int u = 0; u < 32; ++u) {
            const int t = hf + 2 * u;
            if (t < len && ch && sp) {
                // g = -e^a softplus(x): dg/dx = -e^a sigmoid(x), dg/da = g
                const float x = gv[u] + dtbv;
                const float sg = __fdividef(1.f, 1.f + __expf(-x));
                const float dx = -sdG[t * P128 + cc] * ea * sg;
                dgr[((size_t)(tok0 + t) * H + h) * p.K + cc] = dx;
                dtb += dx;
                alog_part -= sdG[t * P128 + cc] * ea * (fmaxf(x, 0.f) + __logf(1.f + __expf(-fabsf(x))));
            } else if (t < len && ch) {
                const float z = ea * (gv[u] + dtbv);
                const float sg = __fdividef(1.f, 1.f + __expf(-z));   // ~2^-21 relative: ample for dg_raw
                const float dz = sdG[t * P128 + cc] * p.lb * sg * (1.f - sg);
                dgr[((size_t)(tok0 + t) * H + h) * p.K + cc] = dz * ea;
                dtb += dz * ea;
                alog_part += dz * z;
            }
        }
        float* sdtb = sred + 64 + 128 + 8;   // [256]
        sdtb[tid] = dtb;
        __syncthreads();
        if (tid < p.K) p.part_dtb[((size_t)c * H + h) * p.K + tid] = sdtb[tid] + sdtb[tid + 128];
    }
    alog_part = warp_sum(alog_part);
    float* sblk = sred + 64 + 128;
    if (lane == 0) sblk[warp] = alog_part;
    __syncthreads();
    if (tid == 0) {
        float acc = 0.f;
        for (int w = 0; w < 8; ++w) acc += sblk[w];
        p.part_alog[(size_t)c * H + h] = acc;
    }
}

// ------------------------------------------------------------------ reverse-chain operands
//
// Per (chunk, head): the dS-independent terms of the reverse recursion, Y = scale Aqk^T dO and
// P = scale Qg^T dO (bf16 warp MMAs with the left operand split into hi + lo; dO is bf16 and exact),
// into the backward workspace record (bwrec).  The chains' split bf16 operand slot (Kd and -W,
// chainrec) is written by the intra pass itself, at the head of each chunk's record.
namespace {
constexpr int PB_A = 0;                  // [64][P64]   Aqk
constexpr int PB_Q = PB_A + 64 * P64;    // [64][P128]  Qg
constexpr int PB_D = PB_Q + 64 * P128;   // bf16 [64][PD16]  dO (exact, as loaded)
constexpr int PD16 = 136;                // bf16 row stride: 272 bytes, 16-byte aligned, rows 4 banks apart
constexpr int PB_FLOATS = PB_D + 64 * PD16 / 2;
}  // namespace

__global__ void __launch_bounds__(256, 3) bwd_pre_kernel(Params p, uint8_t* bw) {
    extern __shared__ float sm[];
    const int c = blockIdx.x, h = blockIdx.y;
    if (c >= p.chunk_off[p.N]) return;
    constexpr int K = 128, V = 128;
    const int H = p.H;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n = chunk_segment(p, c);
    const int tok0 = seg_begin(p, n) + (c - p.chunk_off[n]) * kChunk;
    const int len = min(kChunk, seg_end(p, n) - tok0);
    const RecLayout L = RecLayout::make(K, V);
    const float* rec = p.rec + ((size_t)c * H + h) * p.rec_stride;
    uint8_t* out = bw + ((size_t)c * H + h) * bwrec::BYTES;
    float* sA = sm + PB_A;
    float* sQ = sm + PB_Q;
    __nv_bfloat16* sD = reinterpret_cast<__nv_bfloat16*>(sm + PB_D);
    const float scale = p.scale;

    for (int i = tid; i < 64 * K / 4; i += 256) {
        const int t = i >> 5, c4 = (i & 31) * 4;
        cp_async16(sQ + t * P128 + c4, rec + L.Qg + t * K + c4);
    }
    for (int i = tid; i < 64 * 64 / 4; i += 256) {
        const int t = i >> 4, s4 = (i & 15) * 4;
        cp_async16(sA + t * P64 + s4, rec + L.A + t * 64 + s4);
    }
    // dO rows as they are (bf16); zero past the segment and, for V = 64 heads, past the value columns
    for (int i = tid; i < 64 * V / 8; i += 256) {
        const int t = i >> 4, j8 = (i & 15) * 8;
        if (t < len && j8 < p.V)
            cp_async16(reinterpret_cast<float*>(sD + t * PD16 + j8),
                       reinterpret_cast<const float*>(static_cast<const __nv_bfloat16*>(p.dout) +
                                                      ((size_t)(tok0 + t) * H + h) * p.V + j8));
        else
            *reinterpret_cast<uint4*>(sD + t * PD16 + j8) = make_uint4(0u, 0u, 0u, 0u);
    }
    cp_async_wait_all();
    __syncthreads();
    // Y = scale Aqk^T dO (64 x 128): warp w owns rows 16 (w / 2) and columns 64 (w % 2) .. + 64.
    // Aqk is lower triangular, so rows s only see t >= s.
    {
        const int m0 = 16 * (warp >> 1), n0 = 64 * (warp & 1);
        float* Yg = reinterpret_cast<float*>(out + bwrec::Y);
        float d[8][4];
#pragma unroll
        for (int b = 0; b < 8; ++b)
#pragma unroll
            for (int e = 0; e < 4; ++e) d[b][e] = 0.f;
        mma_strip_splitA_bf16<8>(d, Tile{sA, 1, P64}, TileH{sD, PD16, 1}, m0, n0, m0, 64, lane);
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            int r, cc;
            frag_rc(lane, 0, m0, n0 + 8 * b, r, cc);
            *reinterpret_cast<float2*>(Yg + x4_off(r, cc, 64)) = make_float2(scale * d[b][0], scale * d[b][1]);
            *reinterpret_cast<float2*>(Yg + x4_off(r + 8, cc, 64)) = make_float2(scale * d[b][2], scale * d[b][3]);
        }
    }
    // P = scale Qg^T dO (128 x 128): warp w owns rows 16 w, all columns in two strips of 64
    {
        float* Pg = reinterpret_cast<float*>(out + bwrec::P);
        const int m0 = 16 * warp;
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
            float a1[8][4];
#pragma unroll
            for (int b = 0; b < 8; ++b)
#pragma unroll
                for (int e = 0; e < 4; ++e) a1[b][e] = 0.f;
            mma_strip_splitA_bf16<8>(a1, Tile{sQ, 1, P128}, TileH{sD, PD16, 1}, m0, 64 * half, 0, 64, lane);
#pragma unroll
            for (int b = 0; b < 8; ++b) {
                int r, cc;
                frag_rc(lane, 0, m0, 64 * half + 8 * b, r, cc);
                *reinterpret_cast<float2*>(Pg + x4_off(r, cc, K)) = make_float2(scale * a1[b][0], scale * a1[b][1]);
                *reinterpret_cast<float2*>(Pg + x4_off(r + 8, cc, K)) = make_float2(scale * a1[b][2], scale * a1[b][3]);
            }
        }
    }
}

cudaError_t launch_bwd_pre(const Params& p, uint8_t* bw, cudaStream_t st) {
    const size_t smem = (size_t)PB_FLOATS * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(bwd_pre_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    timing_pre(st, K_BWD_PRE);
    bwd_pre_kernel<<<dim3(p.NCmax, p.H), 256, smem, st>>>(p, bw);
    timing_post(st);
    return cudaGetLastError();
}

cudaError_t launch_grad_tc(const Params& p, cudaStream_t st) {
    const size_t smem = (size_t)SMEM_FLOATS * sizeof(float);
    auto kern = p.gate == KDA_GATE_SOFTPLUS ? grad_tc_kernel<true> : grad_tc_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    timing_pre(st, K_GRAD_TC);
    kern<<<dim3(p.NCmax, p.H), 256, smem, st>>>(p);
    timing_post(st);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_param_reduce(p, st);
}

}  // namespace kda
