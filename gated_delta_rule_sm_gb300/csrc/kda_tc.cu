// kda_tc.cu -- tensor-core (tcgen05 / TMEM) path for bf16 inputs with K = V = 128 (and K = V = 64
// heads, loaded as 128-channel tiles whose upper half is zero).
//
// Same chunkwise algebra as the SIMT path (the gated delta rule of "[kimi k3] add eager reference
// model with FSDP2", 64 tokens per chunk):
//     U = U0 - W S,   O = scale (Qg S + Aqk U),   S' = Diag(exp(Gamma_last)) S + Kd^T U.
// Precision plan (bf16 inputs, fp32 state): the chain's products run with fp16 operands (kind::f16):
// W, Qg, Kd, Aqk, S and U stay far inside fp16's range, where its 11-bit significand gives each
// product tf32-like accuracy in one MMA; U0 is added in fp32 and the state stays in fp32 registers.
//
// The intra-chunk kernels write one record per (chunk, head) in exactly the shared-memory layout the
// chain kernel's MMAs read, so the chain's load warp moves it with three bulk copies per chunk.  The
// chain's blocks take segments longest first (seg_order), the saving intra pass here also writes
// the backward record (led by the backward chains' split-bf16 Kd / -W slot, then fp32 fields), and the
// segment-parallel schedule's piece table and state combine close the file.
#include "kda_common.cuh"
#include "kda_internal.h"
#include "kda_sm100.cuh"

#include <cudaTypedefs.h>

namespace kda {

using namespace sm100;


// ------------------------------------------------------------------ intra-chunk kernel (tcgen05)
//
// Persistent: one CTA (256 threads) per SM loops over (chunk, head) items, fetching the next item's
// q, k, g, v tiles by TMA once the current item's A-matrix MMAs no longer need the tile area.
// Decay factorisation: inside a chunk, with Gamma_t the
// cumulative log-decay and 16-token sub-blocks b (Gamma at the end of sub-block b-1 is G_b),
//   exp(Gamma_t - Gamma_s) = exp(Gamma_t - G_{j+1}) * exp(G_{j+1} - Gamma_s)   for s in sub-block j.
// The right factor is <= 1; the left is <= 1 for t past sub-block j and <= exp(16 |lower_bound|)
// inside it, so every factor stays inside fp32/bf16 range for lower_bound >= -5.  Each column
// sub-block j is one MMA (M = 128: 64 k-rows and 64 q-rows, N = 16, K = 128) with its own left
// operand L^(j).  The per-token factors are running products of alpha = exp(g) inside each
// sub-block, so the exponentials per element are exp for the gate sigmoid and exp for alpha.
// Unbounded gate (g = -exp(a_log) softplus(.)): nothing bounds exp(Gamma_t - G_{j+1}) inside sub-block j,
// so for that gate the left factor of the diagonal column sub-block (j == b) is zero in the MMAs and
// diag_tc_kernel supplies those four 16 x 16 blocks of Bkk and Aqk instead.  Off the diagonal both
// factors stay <= 1 for any gate.  Per item: fp32 [2 (Bkk, Aqk)][64 t][ROW], column u = s - 16 (t / 16).
namespace diaglay {
constexpr int ROW = 20;                      // 80-byte rows: float4 reads of 8 consecutive rows hit distinct banks
constexpr int FLOATS = 2 * 64 * ROW;
constexpr uint32_t BYTES = FLOATS * 4;       // 10240
}  // namespace diaglay

namespace intralay {
constexpr uint32_t RAW_Q = 0, RAW_K = 16384, RAW_G = 32768, RAW_V = 49152;  // TMA tiles [64 t][128 c] bf16
// Left operands of the A-matrix MMAs, [k rows; q rows] 128 x 128, MN-major mn_bf16(r, c, 128, 2048),
// as a bf16 hi tile and a bf16 lo tile (v = hi + lo to ~2^-16).  Two pairs ping-pong: pair A lives
// in its own space, pair B reuses the raw tiles once the element phase has read them.
constexpr uint32_t LA_HI = 65536, LA_LO = 98304;
constexpr uint32_t LB_HI = 0, LB_LO = 32768;
constexpr uint32_t TB_HI = 131072, TB_LO = 139264;  // after the A MMAs (in the dead RB area): T split in bf16, B operand
                                                     // (N = t, K = s), km_bf16(t, s, 1024, 128); the raw area is then free
                                                     // for the next item's tiles
constexpr uint32_t SL = LA_HI;               // after the A MMAs: fp32 [64][65] Diag(beta) Bkk
constexpr uint32_t SN = LA_HI + 16640;       // fp32 [64][65] N = (I + L)^-1
constexpr uint32_t SP = LA_HI + 34816;       // fp32 [4][16][24] scratch blocks of the blocked solve
constexpr uint32_t RB_HI = 131072, RB_LO = 147456;  // B operand (N = s, K = c) 64 x 128, mn_bf16(s, c, 128, 1024), hi / lo
constexpr uint32_t KVB = 163840;             // A operand [Kg^T; V^T] 256 x 64 (K = s), km_bf16(r, s, 1024, 128)
constexpr uint32_t KGLO = 196608;            // bf16 lo half of Kg^T (128 x 64), same layout
constexpr uint32_t SMALL = 212992;           // rq[64] rk[64] beta[64] dtb[128] blk[4][128] gsum[4][128] (fp32)
constexpr uint32_t BAR = SMALL + (64 * 3 + 128 + 1024) * 4;
constexpr uint32_t DIAG = BAR + 64;          // unbounded gate: the item's diagonal blocks (diaglay), by bulk copy
constexpr uint32_t BYTES = DIAG + diaglay::BYTES;
}  // namespace intralay

// acc (a 16 x 16 block as two 16 x 8 accumulator fragments) += A B for 16 x 16 blocks A, B at row
// strides sa, sb: warp tf32 MMAs on hi / lo splits of both operands (hi*hi + hi*lo + lo*hi).
__device__ __forceinline__ void mma16_split(float (&acc)[2][4], const float* a, int sa, const float* b, int sb,
                                            int lane) {
    const int g = lane >> 2, q = lane & 3;
#pragma unroll
    for (int k0 = 0; k0 < 16; k0 += 8) {
        uint32_t ah[4], al[4];
        split_tf32(a[g * sa + k0 + q], ah[0], al[0]);
        split_tf32(a[(g + 8) * sa + k0 + q], ah[1], al[1]);
        split_tf32(a[g * sa + k0 + q + 4], ah[2], al[2]);
        split_tf32(a[(g + 8) * sa + k0 + q + 4], ah[3], al[3]);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            uint32_t bh[2], bl[2];
            split_tf32(b[(k0 + q) * sb + 8 * nt + g], bh[0], bl[0]);
            split_tf32(b[(k0 + q + 4) * sb + 8 * nt + g], bh[1], bl[1]);
            mma1688(acc[nt], al, bh);
            mma1688(acc[nt], ah, bl);
            mma1688(acc[nt], ah, bh);
        }
    }
}

// MODE 0 writes the chain record (tcrec) of the forward; MODE 1 writes the fp32 per-chunk record
// (RecLayout) that the backward's operand, chain and gradient kernels read; MODE 2 writes both (a
// forward that keeps the backward record, so the backward skips this pass).
// GATE_RT: the gate is read from Params at run time (either activation); otherwise the lower-bounded gate
// is compiled in and the unbounded gate's diagonal-block steps are left out.
// Eight consecutive t of one channel c of a chain-slot tile (chainrec: [128 c][64 t] bf16 K-major, hi,
// then lo `lo_off` bytes later), times sg: hi = bf16(x), lo = bf16(x - hi), the split the backward
// chains' products take.  One 16-byte store each.
__device__ __forceinline__ void put_slot_split8(uint8_t* slot, uint32_t off, uint32_t lo_off, const float* v, float sg) {
    float hv[8], lv[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const float x = sg * v[e];
        hv[e] = __bfloat162float(__float2bfloat16_rn(x));
        lv[e] = x - hv[e];
    }
    *reinterpret_cast<uint4*>(slot + off) = pack8_bf16(hv);
    *reinterpret_cast<uint4*>(slot + off + lo_off) = pack8_bf16(lv);
}

template <int MODE, bool GATE_RT>
__global__ void __launch_bounds__(256, 1)
    intra_tc_kernel(Params p, uint8_t* recs, const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_g,
                    const __grid_constant__ CUtensorMap tm_v) {
    using namespace intralay;
    constexpr bool BWD = MODE != 0;      // writes the fp32 backward record
    constexpr bool FWDREC = MODE != 1;   // writes the forward chain record
    extern __shared__ __align__(1024) uint8_t smem[];
    const int H = p.H;
    const int nitems = p.chunk_off[p.N] * H;   // (chunk, head) items, head fastest
    if ((int)blockIdx.x >= nitems) return;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    auto item_tok0 = [&](int it, int& h, int& c, int& tok0) {
        c = it / H;
        h = it - c * H;
        const int n = chunk_segment(p, c);
        tok0 = seg_begin(p, n) + (c - p.chunk_off[n]) * kChunk;
        return min(kChunk, seg_end(p, n) - tok0);
    };
    float* rq = reinterpret_cast<float*>(smem + SMALL);
    float* rk = rq + 64;
    float* sbeta = rk + 64;
    float* sdtb = sbeta + 64;
    float* sblk = sdtb + 128;
    float* sgsum = sblk + 512;        // per sub-block sums of g (backward record only)
    const RecLayout RL = RecLayout::make(128, 128);
    // Each MMA barrier has at most one pending phase at any time, so parity waits are unambiguous.
    uint64_t* bar_load = reinterpret_cast<uint64_t*>(smem + BAR);
    uint64_t* bar_a = bar_load + 1;   // A-matrix MMAs reading tile pair A (two issuing warps)
    uint64_t* bar_b = bar_load + 2;   // A-matrix MMAs reading tile pair B (two issuing warps)
    uint64_t* bar_w = bar_load + 3;   // the final W / U0 MMAs (two issuing warps)
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bar_load + 4);
    uint64_t* bar_diag = bar_load + 5;   // unbounded gate: the diagonal blocks of an item
    const bool sp = GATE_RT && p.gate == KDA_GATE_SOFTPLUS;   // diagonal sub-blocks from diag_tc_kernel
    auto load_diag = [&](int it) {
        mbar_expect_tx(bar_diag, diaglay::BYTES);
        bulk_g2s(smem + DIAG, p.diag + (size_t)it * diaglay::FLOATS, diaglay::BYTES, bar_diag);
    };
    // TMEM columns: A-matrix partial products p = 0..5 at 64 p + 16 j (sub-block j), W^T at 384, U0^T
    // at 448.  One thread issues a tcgen05.mma every ~100 cycles and the tensor pipe takes one about
    // every 46 at this shape, so two issuing threads keep it busy: warps 0 and 1, whose sub-block
    // writes no left operand after the first, so the other warps' operand writes for the next
    // sub-block overlap the MMAs.  The two final products go out from two warps as well.
    constexpr int NPART = 6, NISSUE = 2;
    constexpr uint32_t T_W = 384, T_U0 = 448, TCOLS = 512;
    // the raw q, k, g, v tiles of one item (64 tokens x 128 channels each, out-of-range rows zero)
    auto load_raw = [&](int it) {
        int h2, c2, t02;
        item_tok0(it, h2, c2, t02);
        mbar_expect_tx(bar_load, 4 * 16384);
        tma_load_3d(smem + RAW_Q, &tm_q, 0, h2 / p.G, t02, bar_load);   // q, k: key head of value head h2
        tma_load_3d(smem + RAW_K, &tm_k, 0, h2 / p.G, t02, bar_load);
        tma_load_3d(smem + RAW_G, &tm_g, 0, h2, t02, bar_load);
        tma_load_3d(smem + RAW_V, &tm_v, 0, h2, t02, bar_load);
    };

    if (tid == 0) {
        mbar_init(bar_load, 1);
        mbar_init(bar_a, NISSUE);
        mbar_init(bar_b, NISSUE);
        mbar_init(bar_w, 2);
        mbar_init(bar_diag, 1);
        mbar_fence_init();
        load_raw(blockIdx.x);
        if (sp) load_diag(blockIdx.x);
    }
    if (warp == 0) tmem_alloc(tslot, TCOLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    uint32_t par_a = 0, par_b = 0, par_w = 0, par_load = 0, par_diag = 0;
    bool ok = true;
    // dt_bias (thread < 128) and the beta logit (thread < 64) of an item, loaded into registers one
    // item ahead so their latency hides behind the current item
    float nx_dtb = 0.f, nx_braw = 0.f;
    auto fetch_small = [&](int it) {
        int h2, c2, t02;
        const int len2 = item_tok0(it, h2, c2, t02);
        if (tid < 128) nx_dtb = tid < p.K ? p.dt_bias[h2 * p.K + tid] : 0.f;   // K = 64: channels padded
        if (tid < 64 && tid < len2) nx_braw = load_act(p.beta_raw, (size_t)(t02 + tid) * H + h2, KDA_BF16);
    };
    fetch_small(blockIdx.x);
    // Persistent over items: each item's raw tiles were requested by the previous item (or above).
    for (int item = blockIdx.x; item < nitems; item += gridDim.x) {
    int h, c, tok0;
    const int len = item_tok0(item, h, c, tok0);
    float* frec = BWD ? p.rec + ((size_t)c * H + h) * p.rec_stride : nullptr;
    // the backward chains' operand slot, in place of the fp32 W and Kd fields (W, Kd, gC lead the record)
    uint8_t* slot = BWD ? reinterpret_cast<uint8_t*>(frec + RL.W) : nullptr;
    uint8_t* rec = FWDREC ? recs + ((size_t)c * H + h) * tcrec::BYTES : nullptr;
    if (tid < 128) sdtb[tid] = nx_dtb;
    if (tid < 64) sbeta[tid] = tid < len ? sigmoidf_acc(nx_braw) : 0.f;
    ok = __syncthreads_and(mbar_wait(bar_load, par_load) ? 1 : 0) != 0;
    par_load ^= 1;
    if (!ok) goto fail;

    // ---- per-token inverse norms (warp w: tokens 8w .. 8w+7; the 16 reductions interleave)
    {
        float ss[16];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int t = warp * 8 + u;
            const uint2 qv = *reinterpret_cast<const uint2*>(smem + RAW_Q + t * 256 + lane * 8);
            const uint2 kv = *reinterpret_cast<const uint2*>(smem + RAW_K + t * 256 + lane * 8);
            const float2 q0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&qv.x));
            const float2 q1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&qv.y));
            const float2 k0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&kv.x));
            const float2 k1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&kv.y));
            ss[u] = q0.x * q0.x + q0.y * q0.y + q1.x * q1.x + q1.y * q1.y;
            ss[8 + u] = k0.x * k0.x + k0.y * k0.y + k1.x * k1.x + k1.y * k1.y;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
            for (int i = 0; i < 16; ++i) ss[i] += __shfl_xor_sync(0xffffffffu, ss[i], o);
        if (lane < 8) {
            const int t = warp * 8 + lane;
            float sq = ss[0], sk = ss[8];
#pragma unroll
            for (int u = 1; u < 8; ++u)
                if (lane == u) { sq = ss[u]; sk = ss[8 + u]; }
            rq[t] = t < len ? 1.0f / sqrtf(sq + kNormEps) : 0.f;
            rk[t] = t < len ? 1.0f / sqrtf(sk + kNormEps) : 0.f;
        }
    }
    __syncthreads();

    {
        // ---- element phase: thread owns channels cp and cp + 64 of sub-block bi (16 tokens)
        const int cp = tid & 63, bi = tid >> 6, t0 = 16 * bi;
        const float ea = __expf(p.a_log[h]);
        float kx[2][16], qx[2][16], y[2][16], fj[2][4];
        float lg[BWD ? 2 : 1][16];          // running sum of g inside the sub-block (backward record)
        float av[2][16];                    // alpha = exp(g)
        {
            // loads and gates of both channels in one pass: independent chains for the scheduler
            const float dtb[2] = {sdtb[cp], sdtb[cp + 64]};
            float gs[2] = {0.f, 0.f};
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const int t = t0 + u;
                const float rkt = rk[t], rqt = rq[t];
#pragma unroll
                for (int ci = 0; ci < 2; ++ci) {
                    const uint32_t o = t * 256 + (cp + 64 * ci) * 2;
                    kx[ci][u] = bf16_at(smem + RAW_K, o) * rkt;
                    qx[ci][u] = bf16_at(smem + RAW_Q, o) * rqt;
                    const float z = bf16_at(smem + RAW_G, o) + dtb[ci];
                    // lower-bounded: lb sigmoid(e^a z); unbounded: -e^a softplus(z) = -e^a (max(z, 0) + log(1 + e^-|z|))
                    const float gv = sp ? -ea * (fmaxf(z, 0.f) + __logf(1.f + __expf(-fabsf(z))))
                                        : p.lb * __fdividef(1.f, 1.f + __expf(-ea * z));
                    const float g = t < len ? gv : 0.f;
                    av[ci][u] = __expf(g);
                    if (BWD) {
                        gs[ci] += g;
                        lg[BWD ? ci : 0][u] = gs[ci];
                    }
                }
            }
            if (BWD) {
                sgsum[bi * 128 + cp] = gs[0];
                sgsum[bi * 128 + cp + 64] = gs[1];
            }
        }
#pragma unroll
        for (int ci = 0; ci < 2; ++ci) {
            const int cc = cp + 64 * ci;
            const float* a = av[ci];
            float run = 1.f;
#pragma unroll
            for (int u = 15; u >= 0; --u) {     // y_t = prod_{v > t} alpha_v  (= exp(G_{b+1} - Gamma_t))
                y[ci][u] = run;
                run *= a[u];
            }
            sblk[bi * 128 + cc] = run;           // sub-block total exp(G_{b+1} - G_b)
            // R_b = k * y, split into bf16 hi + lo
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                float hi[8], lo[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float r = kx[ci][8 * hh + e] * y[ci][8 * hh + e];
                    hi[e] = __bfloat162float(__float2bfloat16_rn(r));
                    lo[e] = r - hi[e];
                }
                *reinterpret_cast<uint4*>(smem + RB_HI + mn_bf16(t0 + 8 * hh, cc, 128, 1024)) = pack8_bf16(hi);
                *reinterpret_cast<uint4*>(smem + RB_LO + mn_bf16(t0 + 8 * hh, cc, 128, 1024)) = pack8_bf16(lo);
            }
            run = 1.f;
#pragma unroll
            for (int u = 0; u < 16; ++u) {      // x_t = prod_{v <= t} alpha_v  (= exp(Gamma_t - G_b))
                run *= a[u];
                kx[ci][u] *= run;
                qx[ci][u] *= run;
            }
            // V^T rows 128 + cc of the [Kg^T; V^T] operand: an exact copy of v (zero past the segment)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                float vv[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int t = t0 + 8 * hh + e;
                    vv[e] = t < len ? bf16_at(smem + RAW_V, t * 256 + cc * 2) : 0.f;
                }
                *reinterpret_cast<uint4*>(smem + KVB + km_bf16(128 + cc, t0 + 8 * hh, 1024, 128)) = pack8_bf16(vv);
            }
        }
        __syncthreads();
        // cross-sub-block factors per channel
#pragma unroll
        for (int ci = 0; ci < 2; ++ci) {
            const int cc = cp + 64 * ci;
            const float B0 = sblk[cc], B1 = sblk[128 + cc], B2 = sblk[256 + cc], B3 = sblk[384 + cc];
            const float eG = bi == 0 ? 1.f : bi == 1 ? B0 : bi == 2 ? B0 * B1 : B0 * B1 * B2;      // exp(G_b)
            const float tail = bi == 0 ? B1 * B2 * B3 : bi == 1 ? B2 * B3 : bi == 2 ? B3 : 1.f;   // exp(Gamma_C - G_{b+1})
            const float Bi = bi == 0 ? B0 : bi == 1 ? B1 : bi == 2 ? B2 : B3;
            const float fd = sp ? 0.f : 1.f / Bi;                        // j == b (from diag_tc_kernel if sp)
            const float fm2 = bi >= 2 ? (bi == 2 ? B1 : B2) : 0.f;       // j == b - 2
            const float fm3 = bi == 3 ? B1 * B2 : 0.f;                   // j == b - 3
            // factor of L^(j) = exp(Gamma_t - G_{j+1}) / x_t for j = 0..3 (zero for j > b)
            fj[ci][0] = bi == 0 ? fd : bi == 1 ? 1.f : bi == 2 ? fm2 : fm3;
            fj[ci][1] = bi == 1 ? fd : bi == 2 ? 1.f : bi == 3 ? fm2 : 0.f;
            fj[ci][2] = bi == 2 ? fd : bi == 3 ? 1.f : 0.f;
            fj[ci][3] = bi == 3 ? fd : 0.f;
            if (FWDREC && bi == 0) reinterpret_cast<float*>(rec + tcrec::GC)[cc] = B0 * B1 * B2 * B3;
            if (BWD) {
                float gpre = 0.f;
                for (int m = 0; m < bi; ++m) gpre += sgsum[m * 128 + cc];
                if (bi == 0) frec[RL.gC + cc] = B0 * B1 * B2 * B3;
                float kdv[16];
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const int t = t0 + u;
                    const float kh = bf16_at(smem + RAW_K, t * 256 + cc * 2) * rk[t];
                    const float qh = bf16_at(smem + RAW_Q, t * 256 + cc * 2) * rq[t];
                    frec[RL.Kg + t * 128 + cc] = kx[ci][u] * eG;
                    frec[RL.Qg + t * 128 + cc] = qx[ci][u] * eG;
                    kdv[u] = kh * y[ci][u] * tail;
                    frec[RL.G + t * 128 + cc] = gpre + lg[BWD ? ci : 0][u];
                    frec[RL.qh + t * 128 + cc] = qh;
                    frec[RL.kh + t * 128 + cc] = kh;
                }
                put_slot_split8(slot, chainrec::KD + km_bf16(cc, t0, 1024, 128), chainrec::KD_LO - chainrec::KD, kdv, 1.f);
                put_slot_split8(slot, chainrec::KD + km_bf16(cc, t0 + 8, 1024, 128), chainrec::KD_LO - chainrec::KD, kdv + 8, 1.f);
            }
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int tb = t0 + 8 * hh;
                float vk[8], vq[8], vkl[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    vk[e] = kx[ci][8 * hh + e] * eG;
                    vq[e] = qx[ci][8 * hh + e] * eG;
                    vkl[e] = vk[e] - __bfloat162float(__float2bfloat16_rn(vk[e]));
                }
                *reinterpret_cast<uint4*>(smem + KVB + km_bf16(cc, tb, 1024, 128)) = pack8_bf16(vk);
                *reinterpret_cast<uint4*>(smem + KGLO + km_bf16(cc, tb, 1024, 128)) = pack8_bf16(vkl);
                if (FWDREC) *reinterpret_cast<uint4*>(rec + tcrec::WQ + mn_bf16(64 + tb, cc, 128, 2048)) = pack8_f16(vq);
            }
            // Kd^T (fp16): k * exp(Gamma_C - Gamma_t), eight tokens per 16 B (forward record only)
#pragma unroll
            for (int hh = 0; hh < (FWDREC ? 2 : 0); ++hh) {
                float kd[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int u = 8 * hh + e;
                    kd[e] = bf16_at(smem + RAW_K, (t0 + u) * 256 + cc * 2) * rk[t0 + u] * y[ci][u] * tail;
                }
                *reinterpret_cast<uint4*>(rec + tcrec::KD + km_bf16(cc, t0 + 8 * hh, 1024, 128)) = pack8_f16(kd);
            }
        }
        // L^(j) rows of this thread's sub-block (k rows t, q rows 64 + t), split into bf16 hi + lo
        auto write_L = [&](int j, uint32_t hi_off, uint32_t lo_off) {
            if (bi < j) return;
#pragma unroll
            for (int ci = 0; ci < 2; ++ci) {
                const int cc = cp + 64 * ci;
                const float f = fj[ci][0] * (j == 0) + fj[ci][1] * (j == 1) + fj[ci][2] * (j == 2) + fj[ci][3] * (j == 3);
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int tb = t0 + 8 * hh;
#pragma unroll
                    for (int part = 0; part < 2; ++part) {
                        float hi[8], lo[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const float v = (part == 0 ? kx[ci][8 * hh + e] : qx[ci][8 * hh + e]) * f;
                            hi[e] = __bfloat162float(__float2bfloat16_rn(v));
                            lo[e] = v - hi[e];
                        }
                        const uint32_t o = mn_bf16(64 * part + tb, cc, 128, 2048);
                        *reinterpret_cast<uint4*>(smem + hi_off + o) = pack8_bf16(hi);
                        *reinterpret_cast<uint4*>(smem + lo_off + o) = pack8_bf16(lo);
                    }
                }
            }
        };
        // A-matrix MMAs of column sub-block j: D_j = L_hi R_hi + L_hi R_lo + L_lo R_hi, each product
        // halved over channels: partial p = product p / 2 over channel half p % 2, summed when the
        // accumulators are read.  Warp w < 2 issues partials w, w + 2, w + 4.
        constexpr uint32_t idA = idesc_bf16(128, 16, 1, 1);
        auto issue_A = [&](int j, uint32_t hi_off, uint32_t lo_off, uint64_t* bar) {
            if (lane != 0 || warp >= NISSUE) return;
            const uint32_t lh = smem_u32(smem + hi_off), ll = smem_u32(smem + lo_off);
            const uint32_t rh = smem_u32(smem + RB_HI) + j * 256, rl = smem_u32(smem + RB_LO) + j * 256;
            for (int pp = warp; pp < NPART; pp += NISSUE) {
                const int pr = pp >> 1, k0 = 4 * (pp & 1);
                const uint32_t la = pr == 2 ? ll : lh, rb = pr == 1 ? rl : rh;
                for (int kk = k0; kk < k0 + 4; ++kk)
                    mma_bf16(tmem + 64 * pp + 16 * j, smem_desc(la + kk * 4096, 2048, 128),
                             smem_desc(rb + kk * 2048, 1024, 128), idA, kk > k0);
            }
            mma_commit(bar);
        };
        auto wait_on = [&](uint64_t* bar, uint32_t& par) -> bool {
            const bool r = __syncthreads_and(mbar_wait(bar, par) ? 1 : 0) != 0;
            par ^= 1;
            return r;
        };
        write_L(0, LA_HI, LA_LO);
        fence_async_smem();
        tc_fence_before();
        __syncthreads();                 // raw tiles are no longer read past this point
        tc_fence_after();
        issue_A(0, LA_HI, LA_LO, bar_a);
        write_L(1, LB_HI, LB_LO);
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        issue_A(1, LB_HI, LB_LO, bar_b);
        if (!wait_on(bar_a, par_a)) goto fail;      // pair A free again
        tc_fence_after();
        write_L(2, LA_HI, LA_LO);
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        issue_A(2, LA_HI, LA_LO, bar_a);
        if (!wait_on(bar_b, par_b)) goto fail;      // pair B free again
        tc_fence_after();
        write_L(3, LB_HI, LB_LO);
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        issue_A(3, LB_HI, LB_LO, bar_b);
        if (!wait_on(bar_a, par_a)) goto fail;
        if (!wait_on(bar_b, par_b)) goto fail;
        tc_fence_after();
        // the raw / pair-B area is free for the rest of this item: fetch the next item's tiles now
        if (item + (int)gridDim.x < nitems) {
            if (tid == 0) {
                fence_async_smem();
                load_raw(item + gridDim.x);
            }
            fetch_small(item + gridDim.x);
        }
    }

    {
        // ---- read the A-matrices: lanes 0-63 hold Bkk rows, lanes 64-127 hold Aqk rows
        float* SLf = reinterpret_cast<float*>(smem + SL);
        float* SNf = reinterpret_cast<float*>(smem + SN);
        float* SPf = reinterpret_cast<float*>(smem + SP);
        if (sp) {
            ok = __syncthreads_and(mbar_wait(bar_diag, par_diag) ? 1 : 0) != 0;
            par_diag ^= 1;
            if (!ok) goto fail;
        }
        {
            // warp w reads lane quarter w % 4 (rows) and columns 32 (w / 4) .. + 32 of the six partials
            const int qw = warp & 3, c0 = 32 * (warp >> 2);
            const uint32_t lb = (static_cast<uint32_t>(qw * 32) << 16) + c0;
            float d[32], e1[32], e2[32];
            tmem_ld16(tmem + lb, d);
            tmem_ld16(tmem + lb + 16, d + 16);
            tmem_ld16(tmem + lb + 64, e1);
            tmem_ld16(tmem + lb + 64 + 16, e1 + 16);
            tmem_ld_wait();
#pragma unroll
            for (int u = 0; u < 32; ++u) d[u] += e1[u];
#pragma unroll
            for (int pp = 2; pp < NPART; pp += 2) {
                tmem_ld16(tmem + lb + 64 * pp, e1);
                tmem_ld16(tmem + lb + 64 * pp + 16, e1 + 16);
                tmem_ld16(tmem + lb + 64 * (pp + 1), e2);
                tmem_ld16(tmem + lb + 64 * (pp + 1) + 16, e2 + 16);
                tmem_ld_wait();
#pragma unroll
                for (int u = 0; u < 32; ++u) d[u] += e1[u] + e2[u];
            }
            if (sp) {
                // the row's diagonal sub-block (its MMA rows had a zero left factor), if in these columns
                const int t = 32 * (qw & 1) + lane, bt = t >> 4;
                if ((bt >> 1) == (c0 >> 5)) {
                    const float4* dg = reinterpret_cast<const float4*>(smem + DIAG) + ((qw >> 1) * 64 + t) * (diaglay::ROW / 4);
                    const bool upper = bt & 1;
#pragma unroll
                    for (int u4 = 0; u4 < 4; ++u4) {
                        const float4 x = dg[u4];
                        const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            d[4 * u4 + e] += upper ? 0.f : xs[e];
                            d[16 + 4 * u4 + e] += upper ? xs[e] : 0.f;
                        }
                    }
                }
            }
            if (qw < 2) {
                const int t = 32 * qw + lane;
                const float bt = sbeta[t];
#pragma unroll
                for (int u = 0; u < 32; ++u) SLf[t * 65 + c0 + u] = c0 + u < t ? bt * d[u] : 0.f;
                if (BWD) {
                    if (c0 == 0) {
                        frec[RL.beta + t] = bt;
                        frec[RL.rn + t] = rq[t];
                        frec[RL.rn + 64 + t] = rk[t];
                    }
                    // a lane writes its own row: 16-byte stores (a warp store touches 32 rows)
#pragma unroll
                    for (int u = 0; u < 32; u += 4)
                        *reinterpret_cast<float4*>(frec + RL.B + t * 64 + c0 + u) =
                            make_float4(c0 + u < t ? d[u] : 0.f, c0 + u + 1 < t ? d[u + 1] : 0.f,
                                        c0 + u + 2 < t ? d[u + 2] : 0.f, c0 + u + 3 < t ? d[u + 3] : 0.f);
                }
            } else {
                const int t = 32 * (qw - 2) + lane;
                if (BWD) {
#pragma unroll
                    for (int u = 0; u < 32; u += 4)
                        *reinterpret_cast<float4*>(frec + RL.A + t * 64 + c0 + u) =
                            make_float4(c0 + u <= t ? d[u] : 0.f, c0 + u + 1 <= t ? d[u + 1] : 0.f,
                                        c0 + u + 2 <= t ? d[u + 2] : 0.f, c0 + u + 3 <= t ? d[u + 3] : 0.f);
                }
#pragma unroll
                for (int u = 0; u < (FWDREC ? 32 : 0); u += 8) {
                    float a8[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) a8[e] = c0 + u + e <= t ? d[u + e] : 0.f;
                    *reinterpret_cast<uint4*>(rec + tcrec::AQ + km_bf16(t, c0 + u, 1024, 128)) = pack8_f16(a8);
                }
            }
        }
        __syncthreads();
        // the diagonal-block area has been read: request the next item's
        if (sp && tid == 0 && item + (int)gridDim.x < nitems) {
            fence_async_smem();
            load_diag(item + gridDim.x);
        }
        // ---- N = (I + L)^-1, blocked: 16x16 diagonal blocks by forward substitution, then the
        // off-diagonal blocks N_ij = -N_ii sum_{m=j}^{i-1} L_im N_mj by increasing i - j.
        if (warp < 4 && lane < 16) {
            const int b = warp, s2 = lane;
            float col[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                float acc = 0.f;
#pragma unroll
                for (int m = 0; m < r; ++m) acc += SLf[(16 * b + r) * 65 + 16 * b + m] * col[m];
                col[r] = r == s2 ? 1.f : (r > s2 ? -acc : 0.f);
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) SNf[(16 * b + r) * 65 + 16 * b + s2] = col[r];
        }
        __syncthreads();
        // Off-diagonal blocks by two levels of the block lower-triangular inverse, as warp tf32 MMAs on
        // hi / lo split operands (about fp32 accuracy):
        //   level 1: N_10 = -N_11 L_10 N_00 and N_32 = -N_33 L_32 N_22;
        //   level 2: on the 32 x 32 halves, N_BL = -N_BR (L_BL N_TL).
        {
            auto blk = [&](float* base, int i, int j) { return base + (16 * i) * 65 + 16 * j; };
            constexpr int XS = 24;   // scratch row stride: conflict-free as a B operand
            float acc[2][4];
            auto zero = [&]() {
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
            };
            auto put = [&](float* d, int sd, float sgn) {
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        int r, cc;
                        frag_rc(lane, e, 0, 8 * nt, r, cc);
                        d[r * sd + cc] = sgn * acc[nt][e];
                    }
            };
            if (warp < 2) {
                const int i = warp == 0 ? 1 : 3;
                float* X = SPf + warp * 16 * XS;
                zero();
                mma16_split(acc, blk(SLf, i, i - 1), 65, blk(SNf, i - 1, i - 1), 65, lane);
                put(X, XS, 1.f);
                __syncwarp();
                zero();
                mma16_split(acc, blk(SNf, i, i), 65, X, XS, lane);
                put(blk(SNf, i, i - 1), 65, -1.f);
            }
            __syncthreads();
            const int r = 2 + (warp >> 1), cb = warp & 1;   // warps 0..3: block (r, cb) of the bottom-left half
            if (warp < 4) {
                // P_{r,cb} = sum_m L_{r,m} (N_TL)_{m,cb}, kept in scratch block 2 (r - 2) + cb
                zero();
                if (cb == 0) {
                    mma16_split(acc, blk(SLf, r, 0), 65, blk(SNf, 0, 0), 65, lane);
                    mma16_split(acc, blk(SLf, r, 1), 65, blk(SNf, 1, 0), 65, lane);
                } else {
                    mma16_split(acc, blk(SLf, r, 1), 65, blk(SNf, 1, 1), 65, lane);
                }
                put(SPf + warp * 16 * XS, XS, 1.f);
            }
            __syncthreads();
            if (warp < 4) {
                // N_{r,cb} = -sum_{m=2}^{r} N_{r,m} P_{m,cb}
                zero();
                mma16_split(acc, blk(SNf, r, 2), 65, SPf + cb * 16 * XS, XS, lane);
                if (r == 3) mma16_split(acc, blk(SNf, 3, 3), 65, SPf + (2 + cb) * 16 * XS, XS, lane);
                put(blk(SNf, r, cb), 65, -1.f);
            }
            __syncthreads();
        }
        if (BWD)
            for (int i2 = tid; i2 < 64 * 64; i2 += 256) {
                const int t = i2 >> 6, s2 = i2 & 63;
                frec[RL.N + i2] = s2 <= t ? SNf[t * 65 + s2] : 0.f;
            }
        // ---- T = N Diag(beta), split into bf16 hi + lo, as the B operand (N = t, K = s)
        {
            const int t = tid >> 2, sq = (tid & 3) * 16;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                float hi[8], lo[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int s2 = sq + 8 * hh + e;
                    const float tv = s2 <= t ? SNf[t * 65 + s2] * sbeta[s2] : 0.f;
                    hi[e] = __bfloat162float(__float2bfloat16_rn(tv));
                    lo[e] = tv - hi[e];
                }
                *reinterpret_cast<uint4*>(smem + TB_HI + km_bf16(t, sq + 8 * hh, 1024, 128)) = pack8_bf16(hi);
                *reinterpret_cast<uint4*>(smem + TB_LO + km_bf16(t, sq + 8 * hh, 1024, 128)) = pack8_bf16(lo);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        // ---- W^T = Kg^T T^T and U0^T = V^T (T_hi + T_lo)^T   (M = 128, N = 64, K = 64)
        constexpr uint32_t idW = idesc_bf16(128, 64, 0, 0);
        if (lane == 0 && warp < 2) {   // warp 0: W^T, warp 1: U0^T
            const uint32_t kvb = smem_u32(smem + KVB), thi = smem_u32(smem + TB_HI), tlo = smem_u32(smem + TB_LO);
            const uint32_t kgl = smem_u32(smem + KGLO);
            if (warp == 0) {
                // W^T = (Kg_hi + Kg_lo)^T (T_hi + T_lo)^T without the lo * lo term
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tmem + T_W, smem_desc(kvb + kk * 256, 128, 1024), smem_desc(thi + kk * 256, 128, 1024), idW,
                             kk > 0);
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tmem + T_W, smem_desc(kvb + kk * 256, 128, 1024), smem_desc(tlo + kk * 256, 128, 1024), idW, 1);
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tmem + T_W, smem_desc(kgl + kk * 256, 128, 1024), smem_desc(thi + kk * 256, 128, 1024), idW, 1);
            } else {
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tmem + T_U0, smem_desc(kvb + 16384 + kk * 256, 128, 1024),
                             smem_desc(thi + kk * 256, 128, 1024), idW, kk > 0);
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tmem + T_U0, smem_desc(kvb + 16384 + kk * 256, 128, 1024),
                             smem_desc(tlo + kk * 256, 128, 1024), idW, 1);
            }
            mma_commit(bar_w);
        }
        ok = __syncthreads_and(mbar_wait(bar_w, par_w) ? 1 : 0) != 0;
        par_w ^= 1;
        if (!ok) goto fail;
        tc_fence_after();
        // ---- record W (MN-major, thread = channel) and U0 (column-major, thread = value column)
        {
            const uint32_t lb = static_cast<uint32_t>((warp & 3) * 32) << 16;
            float d[64];
            const uint32_t col = warp < 4 ? T_W : T_U0;
            tmem_ld16(tmem + lb + col, d);
            tmem_ld16(tmem + lb + col + 16, d + 16);
            tmem_ld16(tmem + lb + col + 32, d + 32);
            tmem_ld16(tmem + lb + col + 48, d + 48);
            tmem_ld_wait();
            if (warp < 4) {
                const int cc = tid;
                if (FWDREC)
#pragma unroll
                    for (int tb = 0; tb < 64; tb += 8)
                        *reinterpret_cast<uint4*>(rec + tcrec::WQ + mn_bf16(tb, cc, 128, 2048)) = pack8_f16(d + tb);
                if (BWD)
#pragma unroll
                    for (int tb = 0; tb < 64; tb += 8)   // -W, as the chains take it
                        put_slot_split8(slot, chainrec::WN + km_bf16(cc, tb, 1024, 128), chainrec::WN_LO - chainrec::WN, d + tb, -1.f);
            } else {
                const int j = tid - 128;
                uint8_t* dst = FWDREC ? rec + tcrec::U0 + (j >> 5) * tcrec::U0_SLICE : nullptr;
                if (FWDREC)
#pragma unroll
                    for (int t = 0; t < 64; ++t) *reinterpret_cast<float*>(dst + tcrec::u0_off(t, j & 31)) = d[t];
                if (BWD)
#pragma unroll
                    for (int t = 0; t < 64; ++t) frec[RL.U0 + t * 128 + j] = d[t];
            }
        }
    }
    tc_fence_before();
    __syncthreads();   // this item's shared-memory readers are done before the next item writes
    tc_fence_after();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, TCOLS);
    return;
fail:
    // A wait gave up: record it, give outstanding copies / MMAs a bounded chance to land, release TMEM.
    if (tid == 0) {
        record_error(p.status, KDA_ERR_TIMEOUT);
        mbar_wait(bar_load, par_load, 1u << 16);
        mbar_wait(bar_a, par_a, 1u << 16);
        mbar_wait(bar_b, par_b, 1u << 16);
        mbar_wait(bar_w, par_w, 1u << 16);
        if (sp) mbar_wait(bar_diag, par_diag, 1u << 16);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, TCOLS);
}

// ------------------------------------------------------------------ diagonal blocks, unbounded gate
//
// For t, s in the same 16-token sub-block b:
//     Bkk[t,s] = sum_c k_tc k_sc prod_{s<r<=t} alpha_rc   (s < t),
//     Aqk[t,s] = sum_c q_tc k_sc prod_{s<r<=t} alpha_rc   (s <= t),
// the decay a running product of alpha = exp(g) <= 1, which cannot overflow for any gate.  One CTA of
// four warps per (chunk, head); warp b takes sub-block b, a lane channels 2 lane, 2 lane + 1 (pass 0)
// and 64 + 2 lane, 65 + 2 lane (pass 1).  The lane's partial sums of the 32 lower-triangle entries of
// columns s and 15 - s go through one warp reduce-scatter (31 shuffles), after which lane l holds one
// entry; entries above the diagonal stay zero.  Tokens past the segment have q = k = 0 and alpha = 1.
__global__ void __launch_bounds__(128, 3) diag_tc_kernel(Params p) {
    // shared: the item's q, k, g tiles [64 t][128 c] bf16 (staged by cp.async in one round trip,
    // rows past the segment zero), then the output tile
    extern __shared__ __align__(16) uint8_t dsm[];
    const __nv_bfloat162* sq2 = reinterpret_cast<const __nv_bfloat162*>(dsm);
    const __nv_bfloat162* sk2 = reinterpret_cast<const __nv_bfloat162*>(dsm + 16384);
    const __nv_bfloat162* sg2 = reinterpret_cast<const __nv_bfloat162*>(dsm + 32768);
    float* tile = reinterpret_cast<float*>(dsm + 49152);
    __shared__ float srq[64], srk[64];
    const int H = p.H;
    const int item = blockIdx.x;
    if (item >= p.chunk_off[p.N] * H) return;
    const int c = item / H, h = item - c * H;
    const int n = chunk_segment(p, c);
    const int tok0 = seg_begin(p, n) + (c - p.chunk_off[n]) * kChunk;
    const int len = min(kChunk, seg_end(p, n) - tok0);
    const int tid = threadIdx.x, lane = tid & 31, b = tid >> 5;
    {
        const uint8_t* qg = static_cast<const uint8_t*>(p.q);
        const uint8_t* kg = static_cast<const uint8_t*>(p.k);
        const uint8_t* gg = static_cast<const uint8_t*>(p.g_raw);
        // 3 tensors x 64 rows x 16 pieces of 16 bytes; a row is 256 contiguous bytes
        for (int i = tid; i < 3 * 64 * 16; i += 128) {
            const int ten = i >> 10, t = (i >> 4) & 63, piece = i & 15;
            const int tt = t < len ? t : 0;   // rows past the segment: zero-filled from a valid address
            const size_t row = ten == 2 ? (size_t)(tok0 + tt) * H + h : (size_t)(tok0 + tt) * p.Hk + h / p.G;
            const uint8_t* src = (ten == 0 ? qg : ten == 1 ? kg : gg) + row * 256 + piece * 16;
            cp_async16_zfill(dsm + ten * 16384 + t * 256 + piece * 16, src, t < len ? 16u : 0u);
        }
    }
    for (int i = tid; i < diaglay::FLOATS / 4; i += 128)
        reinterpret_cast<float4*>(tile)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    cp_async_commit_wait_all();
    __syncthreads();
    // inverse L2 norms of the sub-block's tokens
    {
        float ss[32];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int t = 16 * b + u;
            ss[u] = ss[16 + u] = 0.f;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const float2 qv = __bfloat1622float2(sq2[t * 64 + 32 * hf + lane]);
                const float2 kv = __bfloat1622float2(sk2[t * 64 + 32 * hf + lane]);
                ss[u] += qv.x * qv.x + qv.y * qv.y;
                ss[16 + u] += kv.x * kv.x + kv.y * kv.y;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
            for (int i = 0; i < 32; ++i) ss[i] += __shfl_xor_sync(0xffffffffu, ss[i], o);
        if (lane < 16) {
            const int t = 16 * b + lane;
            float sq = ss[0], sk = ss[16];
#pragma unroll
            for (int u = 1; u < 16; ++u)
                if (lane == u) { sq = ss[u]; sk = ss[16 + u]; }
            srq[t] = t < len ? 1.0f / sqrtf(sq + kNormEps) : 0.f;
            srk[t] = t < len ? 1.0f / sqrtf(sk + kNormEps) : 0.f;
        }
    }
    __syncwarp();
    const float ea = __expf(p.a_log[h]);
#pragma unroll 1
    for (int pass = 0; pass < 2; ++pass) {
        const int pr = 32 * pass + lane;   // channel pair: channels 2 pr, 2 pr + 1
        const float dt0 = p.dt_bias[h * 128 + 2 * pr], dt1 = p.dt_bias[h * 128 + 2 * pr + 1];
        float kh[2][16], qh[2][16], al[2][16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int t = 16 * b + u;
            if (t < len) {
                const float2 qv = __bfloat1622float2(sq2[t * 64 + pr]);
                const float2 kv = __bfloat1622float2(sk2[t * 64 + pr]);
                const float2 gv = __bfloat1622float2(sg2[t * 64 + pr]);
                qh[0][u] = qv.x * srq[t]; qh[1][u] = qv.y * srq[t];
                kh[0][u] = kv.x * srk[t]; kh[1][u] = kv.y * srk[t];
                // alpha = exp(-e^a softplus(z)), with the fast intrinsics the intra kernel uses for its factors
                const float z0 = gv.x + dt0, z1 = gv.y + dt1;
                al[0][u] = __expf(-ea * (fmaxf(z0, 0.f) + __logf(1.f + __expf(-fabsf(z0)))));
                al[1][u] = __expf(-ea * (fmaxf(z1, 0.f) + __logf(1.f + __expf(-fabsf(z1)))));
            } else {
                qh[0][u] = qh[1][u] = kh[0][u] = kh[1][u] = 0.f;
                al[0][u] = al[1][u] = 1.f;
            }
        }
        // Columns s and 15 - s share one reduce-scatter: column s has 16 - s Aqk and 15 - s Bkk entries
        // (rows t >= s, resp. t > s), column 15 - s has s + 1 and s, 32 in all.  Slots in that order.
#pragma unroll
        for (int sa = 0; sa < 8; ++sa) {
            const int sb = 15 - sa;
            float v[32];
#pragma unroll
            for (int col = 0; col < 2; ++col) {
                const int s = col ? sb : sa;
                const int a0 = col ? 31 - 2 * sa : 0;     // first Aqk slot of this column
                const int b0 = a0 + 16 - s;               // first Bkk slot
                float e0 = 1.f, e1 = 1.f;
#pragma unroll
                for (int t = s; t < 16; ++t) {
                    if (t > s) { e0 *= al[0][t]; e1 *= al[1][t]; }
                    const float w0 = kh[0][s] * e0, w1 = kh[1][s] * e1;
                    v[a0 + t - s] = qh[0][t] * w0 + qh[1][t] * w1;
                    if (t > s) v[b0 + t - s - 1] = kh[0][t] * w0 + kh[1][t] * w1;
                }
            }
            // reduce-scatter: each step a lane keeps the half of its values selected by its bit `w`,
            // ending with the warp's sum of slot `lane`
#pragma unroll
            for (int w = 16; w >= 1; w >>= 1) {
                const bool up = lane & w;
#pragma unroll
                for (int i = 0; i < w; ++i) {
                    const float send = up ? v[i] : v[i + w];
                    const float keep = up ? v[i + w] : v[i];
                    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
                }
            }
            // slot `lane` -> (column, matrix 0 = Bkk / 1 = Aqk, row)
            int col_s, m, t;
            if (lane < 16 - sa) { col_s = sa; m = 1; t = sa + lane; }
            else if (lane < 31 - 2 * sa) { col_s = sa; m = 0; t = lane - 15 + sa + sa; }
            else if (lane < 32 - sa) { col_s = sb; m = 1; t = sb + lane - (31 - 2 * sa); }
            else { col_s = sb; m = 0; t = sb + 1 + lane - (32 - sa); }
            float* dst = tile + (m * 64 + 16 * b + t) * diaglay::ROW + col_s;
            *dst = pass ? *dst + v[0] : v[0];
        }
    }
    __syncthreads();
    float4* dst = reinterpret_cast<float4*>(p.diag + (size_t)item * diaglay::FLOATS);
    for (int i = tid; i < diaglay::FLOATS / 4; i += 128) dst[i] = reinterpret_cast<const float4*>(tile)[i];
}

size_t diag_item_bytes() { return diaglay::BYTES; }

cudaError_t launch_diag_tc(const Params& p, cudaStream_t st) {
    constexpr int kSmem = 49152 + diaglay::BYTES;
    cudaError_t e = cudaFuncSetAttribute(diag_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    timing_pre(st, K_DIAG_TC);
    diag_tc_kernel<<<p.NCmax * p.H, 128, kSmem, st>>>(p);
    timing_post(st);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ state chain (tcgen05)

namespace chainlay {
constexpr int NSLOT = 3;                  // record slots: a chunk's copy is requested two chunks ahead
constexpr uint32_t SLOT_WQ = 0;
constexpr uint32_t SLOT_U0 = 32768;
constexpr uint32_t SLOT_KD = 40960;       // KD, AQ, GC follow contiguously (tcrec::TAIL bytes)
constexpr uint32_t SLOT_AQ = SLOT_KD + (tcrec::AQ - tcrec::KD);
constexpr uint32_t SLOT_GC = SLOT_KD + (tcrec::GC - tcrec::KD);
constexpr uint32_t SLOT_BYTES = (SLOT_KD + tcrec::TAIL + 1023) / 1024 * 1024;
constexpr uint32_t SB = NSLOT * SLOT_BYTES;   // S as fp16 B operand (N = j, K = c), MN-major: mn_bf16(j, c, 128, 512)
constexpr uint32_t UB = SB + 8192;        // U as fp16 B operand (N = j, K = t), MN-major: mn_bf16(j, t, 128, 512)
constexpr uint32_t UB_BYTES = 4096;       // two buffers (chunk parity), UB_BYTES apart
constexpr uint32_t BAR = UB + 2 * UB_BYTES; // mbarriers: full[3], empty[3], ws, s, o, u
constexpr uint32_t TSLOT = BAR + 128;
constexpr uint32_t BYTES = TSLOT + 64;
}  // namespace chainlay
static_assert(chainlay::BYTES <= 232448, "shared memory per CTA");

constexpr uint32_t kIdescWS = idesc_f16(128, 32, 1, 1);   // [W; Qg] and S both MN-major
constexpr uint32_t kIdescKU = idesc_f16(128, 32, 0, 1);   // Kd^T / Aqk K-major, U MN-major

// One CTA per (segment, head, 32-column slice of V): four compute warps (0-3), two U helper warps
// (4, 5), an MMA warp (6) and a load warp (7).  Every operand is fp16 (one kind::f16 MMA per product,
// tf32-like accuracy at these magnitudes); the state itself stays fp32 in registers.
// Compute thread c keeps row c of the state slice (32 fp32) in registers.  Per chunk the critical path
// is
//   MMA1 (W S) -> U = U0 - W S -> MMA2b (Kd^T U) -> S <- Diag(gC) S + Kd^T U -> next MMA1.
// MMA1 and MMA2b are split over K into four partial accumulators, one per compute warp (lane 0
// issues), and the epilogues add the partials.  The U step reads TMEM lanes 0..63, which only warps
// whose index is 0 or 1 modulo 4 can reach: warps 0, 1 take columns 0..15 and warps 4, 5 columns
// 16..31, which halves that step's latency.  A compute warp issues its MMA1 partial of the next chunk
// as soon as its own 32 rows of S are written (the partial contracts over exactly those rows).  The
// output is Qg S (rows 64..127 of the MMA1 partials) plus Aqk U, which the MMA warp issues into its own
// accumulator as soon as U is staged, off the critical path.  Records stream through three slots; the
// load warp refills a slot with the chunk three ahead once every reader of its chunk is done (an
// `empty` mbarrier per slot).
// flags: kChainStoreStates (write the chunk-entering states), kChainTransfer (start every segment from
// the identity and take U0 as zero: the final state is then the segment's transfer matrix, the product
// of Diag(exp(Gamma_last)) - Kd^T W over its chunks; needs K == V).
constexpr int kChainStoreStates = 1, kChainTransfer = 2, kChainRankMajor = 4;
__global__ void __launch_bounds__(256, 1) chain_fwd_tc_kernel(Params p, const uint8_t* recs, int flags) {
    const bool store_states = flags & kChainStoreStates, transfer = flags & kChainTransfer;
    extern __shared__ __align__(1024) uint8_t smem[];
    // kChainRankMajor: blockIdx.x = (head, slice), blockIdx.y = the segment's rank in seg_order (longest
    // first), so every head and slice of the longest segments start in the first wave
    int n, h, z;
    if (flags & kChainRankMajor) {
        const int nz = p.V / 32;
        h = blockIdx.x / nz;
        z = blockIdx.x - h * nz;
        n = seg_order(p)[blockIdx.y];
    } else {
        n = blockIdx.x;
        h = blockIdx.y;
        z = blockIdx.z;
    }
    const int j0 = z * 32;
    // the state slice has 128 rows in TMEM and registers; heads with K = V = 64 leave rows and columns
    // 64..127 zero (their record rows are zero) and read / write only the real ones
    const int H = p.H, K = p.K, V = p.V;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    constexpr int NS = chainlay::NSLOT;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + chainlay::BAR);   // [NS] record slots landed
    uint64_t* empty = full + NS;    // [NS] record slots released
    uint64_t* bar_ws = full + 2 * NS;       // MMA1 (4 issuers)
    uint64_t* bar_s = bar_ws + 1;   // MMA2b, state update (4 issuers)
    uint64_t* bar_o = bar_ws + 2;   // MMA2a, output (MMA warp)
    uint64_t* bar_u = bar_ws + 3;   // U of this chunk is in shared memory
    volatile int* sh_fail = reinterpret_cast<volatile int*>(smem + chainlay::TSLOT + 4);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + chainlay::TSLOT);
    uint8_t* SB = smem + chainlay::SB;
    const int cb = p.chunk_off[n], ce = p.chunk_off[n + 1];
    const int tb = seg_begin(p, n), te = seg_end(p, n);
    const int nch = ce - cb;
    constexpr uint32_t TCOLS = 512;

    if (tid == 0) {
        for (int b = 0; b < NS; ++b) mbar_init(&full[b], 1);
        // a slot is free once the four compute warps have read its exp(Gamma_last) (S step) and warp 2
        // has seen the chunk's last MMA complete (output step)
        for (int b = 0; b < NS; ++b) mbar_init(&empty[b], 5);
        mbar_init(bar_ws, 4);
        mbar_init(bar_s, 4);
        mbar_init(bar_o, 1);
        mbar_init(bar_u, 4);   // the four MMA2b issuers, each after its product is queued
        *sh_fail = 0;
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(tslot, TCOLS);
    auto slot_ptr = [&](int i) { return smem + (i % NS) * chainlay::SLOT_BYTES; };
    auto rec_ptr = [&](int i) { return recs + ((size_t)(cb + i) * H + h) * tcrec::BYTES; };
    auto ub_addr = [&](int i) { return smem_u32(smem + chainlay::UB + (i & 1) * chainlay::UB_BYTES); };
    auto fail_wait = [&](uint64_t* bar, uint32_t parity) {
        if (!mbar_wait_done(bar, parity)) atomicExch((int*)sh_fail, 1);
    };
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    // D1[b] partial w at tmem + 128 b + 32 w; D3 partial w at tmem + 256 + 32 w; Aqk U of D1[b] at 384 + 32 b
    const uint32_t tD3 = tmem + 256, tDO = tmem + 384;
    // U[t][j] = U0[t][j] - (W S)[t][j] for the 16 columns j0h .. j0h + 15 of row t (lane t % 32 of this
    // warp's lane quarter), summed over the four MMA1 partials, as fp16 into the chunk's U buffer
    auto u_half = [&](int i, int t, uint32_t lane_base, int j0h) {
        const uint32_t tD1 = tmem + 128 * (i & 1) + lane_base + j0h;
        float d[16], e[3][16];
        tmem_ld16(tD1, d);
#pragma unroll
        for (int w = 0; w < 3; ++w) tmem_ld16(tD1 + 32 * (w + 1), e[w]);
        tmem_ld_wait();
        const uint8_t* u0 = slot_ptr(i) + chainlay::SLOT_U0;
        uint8_t* UB = smem + chainlay::UB + (i & 1) * chainlay::UB_BYTES;
#pragma unroll
        for (int jg = 0; jg < 16; jg += 8) {
            float u[8];
#pragma unroll
            for (int h4 = 0; h4 < 8; h4 += 4) {
                // columns j0h + jg + h4 .. + 3 of row t: one 16-byte chunk of the swizzled U0 slice
                const float4 c4 = transfer ? make_float4(0.f, 0.f, 0.f, 0.f)
                                           : *reinterpret_cast<const float4*>(u0 + tcrec::u0_off(t, j0h + jg + h4));
                const float cv[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
                for (int e4 = 0; e4 < 4; ++e4) {
                    const int j = jg + h4 + e4;
                    u[h4 + e4] = cv[e4] - (d[j] + (e[0][j] + e[1][j]) + e[2][j]);
                }
            }
            *reinterpret_cast<uint4*>(UB + mn_bf16(j0h + jg, t, 128, 512)) = pack8_f16(u);
        }
    };

    bool ok = true;
    if (warp == 7) {
        // load warp: chunk k into slot k % NS once chunk k - NS has released it
        if (lane == 0) {
            for (int k = 0; k < nch; ++k) {
                const int sl = k % NS;
                if (k >= NS) {
                    bool got = false;
                    for (int tries = 0; tries < 64 && !got && *sh_fail == 0; ++tries)
                        got = mbar_wait(&empty[sl], ((k / NS) - 1) & 1, 1u << 16);
                    if (!got) { atomicExch((int*)sh_fail, 1); break; }
                }
                uint8_t* slot = slot_ptr(k);
                const uint8_t* rec = rec_ptr(k);
                mbar_expect_tx(&full[sl], 32768 + tcrec::U0_SLICE + tcrec::TAIL);
                bulk_g2s(slot + chainlay::SLOT_WQ, rec + tcrec::WQ, 32768, &full[sl]);
                bulk_g2s(slot + chainlay::SLOT_U0, rec + tcrec::U0 + z * tcrec::U0_SLICE, tcrec::U0_SLICE, &full[sl]);
                bulk_g2s(slot + chainlay::SLOT_KD, rec + tcrec::KD, tcrec::TAIL, &full[sl]);
            }
        }
        __syncwarp();
    } else if (warp == 6) {
        // MMA warp: Aqk U of chunk i once its U is staged (rows 0..63 of this accumulator are unused)
        if (lane == 0) {
            for (int i = 0; i < nch; ++i) {
                bool got = false;
                for (int tries = 0; tries < 64 && !got && *sh_fail == 0; ++tries) got = mbar_wait(bar_u, i & 1, 1u << 16);
                if (!got) { atomicExch((int*)sh_fail, 1); break; }
                tc_fence_after();
                const uint32_t ub = ub_addr(i);
                // an M = 128 window whose rows 64..127 are Aqk (rows 0..63: the tail of Kd^T, not read back)
                const uint32_t aq = smem_u32(slot_ptr(i) + chainlay::SLOT_AQ) - 8192;
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tDO + 32 * (i & 1), smem_desc(aq + kk * 256, 128, 1024), smem_desc(ub + kk * 1024, 512, 128),
                             kIdescKU, kk > 0);
                mma_commit(bar_o);
            }
        }
        __syncwarp();
    } else if (warp >= 4) {
        // U helpers: columns 16..31 of the U rows in lane quarter warp - 4 (t = tid - 128); warps 0 and 1
        // take columns 0..15 of the same rows, so each thread of the U step handles half a row
        const int t = tid - 128;
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        for (int i = 0; i < nch; ++i) {
            fail_wait(&full[i % NS], (i / NS) & 1);
            fail_wait(bar_ws, i & 1);
            tc_fence_after();
            u_half(i, t, lane_base, 16);
            fence_async_smem();
            tc_fence_before();
            const bool failed = named_sync_or(2, 192, *sh_fail != 0);
            tc_fence_after();
            if (failed) { ok = false; break; }
        }
    } else {
    float S[32];
    {
        const float* src = p.S0 && !transfer && tid < K ? p.S0 + (((size_t)n * H + h) * K + tid) * V + j0 : nullptr;
#pragma unroll
        for (int j = 0; j < 32; ++j) S[j] = src ? src[j] : (transfer && tid == j0 + j ? 1.f : 0.f);
    }
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const bool issuer = lane == 0;
    auto sync128 = [&]() {
        tc_fence_before();
        named_sync(1, 128);
        tc_fence_after();
    };
    // sum of the four partials 32 columns apart from base, this warp's lane quarter (one wait for all loads)
    auto ld_sum4 = [&](uint32_t base, float* d) {
        float e[3][32];
        tmem_ld16(base + lane_base, d);
        tmem_ld16(base + lane_base + 16, d + 16);
#pragma unroll
        for (int w = 0; w < 3; ++w) {
            tmem_ld16(base + 32 * (w + 1) + lane_base, e[w]);
            tmem_ld16(base + 32 * (w + 1) + lane_base + 16, e[w] + 16);
        }
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) d[j] += (e[0][j] + e[1][j]) + e[2][j];
    };
    // MMA1 partial `warp`: K rows 32 warp .. 32 warp + 31 of [W; Qg] S
    auto issue_mma1 = [&](int i) {
        fail_wait(&full[i % NS], (i / NS) & 1);
        tc_fence_after();
        const uint32_t wq = smem_u32(slot_ptr(i) + chainlay::SLOT_WQ), sb = smem_u32(SB);
        for (int q = 0; q < 2; ++q) {
            const int kk = 2 * warp + q;
            mma_bf16(tmem + 128 * (i & 1) + 32 * warp, smem_desc(wq + kk * 4096, 2048, 128),
                     smem_desc(sb + kk * 1024, 512, 128), kIdescWS, q > 0);
        }
        mma_commit(bar_ws);
    };
#pragma unroll
    for (int jg = 0; jg < 4; ++jg) *reinterpret_cast<uint4*>(SB + mn_bf16(8 * jg, tid, 128, 512)) = pack8_f16(S + 8 * jg);
    fence_async_smem();
    sync128();
    if (issuer && nch > 0) issue_mma1(0);

    for (int i = 0; i < nch; ++i) {
        const int c = cb + i;
        uint8_t* sl = slot_ptr(i);
        const uint32_t par = i & 1;
        const uint32_t tD1 = tmem + 128 * (i & 1);
        if (store_states && tid < K) {
            float* dst = p.states + (((size_t)c * H + h) * K + tid) * V + j0;
#pragma unroll
            for (int j = 0; j < 32; j += 4) *reinterpret_cast<float4*>(dst + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
        }
        fail_wait(&full[i % NS], (i / NS) & 1);   // record visible to this thread
        if (warp < 2) {
            // columns 0..15 of U rows t = tid (the helper warps take 16..31)
            fail_wait(bar_ws, par);
            tc_fence_after();
            u_half(i, tid, lane_base, 0);
        }
        fence_async_smem();
        // U staged by warps 0, 1 and the helpers.  This is the loop's one exit point: a wait that gave up
        // anywhere in the previous step is seen here by every thread of warps 0..5 at once.
        tc_fence_before();
        const bool failed = named_sync_or(2, 192, *sh_fail != 0);
        tc_fence_after();
        if (failed) { ok = false; break; }
        // MMA2b: D3 partial w = Kd^T U over t in [16 w, 16 w + 16) (one K step).  The MMA warp's output
        // product (Aqk U) is released only after these four are queued, so the state's product, on the
        // chain's critical path, does not wait behind it in the tensor pipe.
        if (issuer) {
            const uint32_t ub = ub_addr(i), kd = smem_u32(sl + chainlay::SLOT_KD);
            mma_bf16(tD3 + 32 * warp, smem_desc(kd + warp * 256, 128, 1024), smem_desc(ub + warp * 1024, 512, 128),
                     kIdescKU, 0);
            mma_commit(bar_s);
            mbar_arrive(bar_u);   // the MMA warp may read U now
        }
        fail_wait(bar_s, par);
        tc_fence_after();
        {
            const float gc = reinterpret_cast<const float*>(sl + chainlay::SLOT_GC)[tid];
            float d[32];
            ld_sum4(tD3, d);
#pragma unroll
            for (int j = 0; j < 32; ++j) S[j] = gc * S[j] + d[j];
#pragma unroll
            for (int jg = 0; jg < 4; ++jg)
                *reinterpret_cast<uint4*>(SB + mn_bf16(8 * jg, tid, 128, 512)) = pack8_f16(S + 8 * jg);
        }
        // MMA1 partial `warp` of the next chunk reads only this warp's 32 rows of S
        fence_async_smem();
        __syncwarp();
        if (issuer) mbar_arrive(&empty[i % NS]);   // this warp is done with the slot's exp(Gamma_last)
        if (issuer && i + 1 < nch) issue_mma1(i + 1);
        __syncwarp();
        if (warp >= 2) {
            // output of chunk i: rows 64..127 of its MMA1 partials plus the Aqk U accumulator
            fail_wait(bar_o, par);
            tc_fence_after();
            if (tid == 64) mbar_arrive(&empty[i % NS]);   // every reader of this chunk's slot is done
            float d[32], e[32];
            tmem_ld16(tDO + 32 * (i & 1) + lane_base, e);
            tmem_ld16(tDO + 32 * (i & 1) + lane_base + 16, e + 16);
            ld_sum4(tD1, d);
            const int t = tid - 64;
            const int tok0 = tb + i * kChunk, len = min(kChunk, te - tok0);
            if (p.out && t < len) {
                __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(p.out) + ((size_t)(tok0 + t) * H + h) * V + j0;
                float sd[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) sd[j] = p.scale * (d[j] + e[j]);
#pragma unroll
                for (int j = 0; j < 32; j += 8) *reinterpret_cast<uint4*>(o + j) = pack8_bf16(sd + j);
            }
        }
    }
    sync128();
    if (*sh_fail) ok = false;
    if (ok && p.ST && tid < K) {
        float* dst = p.ST + (((size_t)n * H + h) * K + tid) * V + j0;
#pragma unroll
        for (int j = 0; j < 32; j += 4) *reinterpret_cast<float4*>(dst + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
    }
    }
    __syncthreads();
    if (*sh_fail && tid == 0) {
        // Record the timeout; give in-flight copies and MMAs a bounded chance to land before this CTA's
        // shared and tensor memory are released.
        record_error(p.status, KDA_ERR_TIMEOUT);
        for (int b = 0; b < NS; ++b) {
            mbar_wait(&full[b], 0, 1u << 12);
            mbar_wait(&full[b], 1, 1u << 12);
        }
        for (int b = 2 * NS; b < 2 * NS + 3; ++b) {
            mbar_wait(&full[b], 0, 1u << 12);
            mbar_wait(&full[b], 1, 1u << 12);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, TCOLS);
}

// ------------------------------------------------------------------ launchers

size_t tc_record_bytes(int NCmax, int H) { return (size_t)NCmax * H * tcrec::BYTES; }

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link-time libcuda dependency).
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }
    return fn;
}

// [TT tokens][H heads][128 channels] bf16 -> boxes of 64 tokens x 1 head x 128 channels (row-major in smem).
// [TT tokens][H heads][C channels] bf16 -> boxes of 64 tokens x 1 head x 128 channels, row-major in shared
// memory; with C = 64 the upper 64 channels of every row, like tokens past the end, are filled with zeros.
static bool head_tile_map(CUtensorMap* m, const void* base, int H, int TT, int C = 128) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)C, (cuuint64_t)H, (cuuint64_t)TT};
    cuuint64_t strides[2] = {(cuuint64_t)C * 2, (cuuint64_t)H * C * 2};
    cuuint32_t box[3] = {128, 1, 64};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool head_tile_map2(CUtensorMap* m, const void* base, int H, int TT, int C) { return head_tile_map(m, base, H, TT, C); }

bool tc_inputs_aligned(const Params& p) {
    auto al = [](const void* x) { return (reinterpret_cast<uintptr_t>(x) & 15) == 0; };
    // the forward chain stores the output and the final state 16 bytes at a time, the gradient kernel dv;
    // the backward chains read the initial state and the final-state gradient and store the
    // initial-state gradient likewise (a null pointer counts as aligned)
    return al(p.q) && al(p.k) && al(p.g_raw) && al(p.v) && (p.dout == nullptr || al(p.dout)) && al(p.out) &&
           al(p.ST) && al(p.dv) && al(p.S0) && al(p.dST) && al(p.dS0);
}

cudaError_t launch_intra_tc(const Params& p, uint8_t* recs, int mode, cudaStream_t st) {
    CUtensorMap mq, mk, mg, mv;
    // K = V = 64 heads load as 128-channel tiles whose upper half the copy fills with zeros
    if (!head_tile_map(&mq, p.q, p.Hk, p.TT, p.K) || !head_tile_map(&mk, p.k, p.Hk, p.TT, p.K) ||
        !head_tile_map(&mg, p.g_raw, p.H, p.TT, p.K) || !head_tile_map(&mv, p.v, p.H, p.TT, p.V))
        return cudaErrorInvalidValue;
    const bool sp = p.gate == KDA_GATE_SOFTPLUS;
    auto kern = mode == 0 ? (sp ? intra_tc_kernel<0, true> : intra_tc_kernel<0, false>)
              : mode == 1 ? (sp ? intra_tc_kernel<1, true> : intra_tc_kernel<1, false>)
                          : (sp ? intra_tc_kernel<2, true> : intra_tc_kernel<2, false>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)intralay::BYTES);
    if (e != cudaSuccess) return e;
    timing_pre(st, K_INTRA_TC);
    // persistent: one CTA per SM (shared memory allows one), each looping over (chunk, head) items
    int sms = 0, dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long items = (long)p.NCmax * p.H;
    const int grid = (int)(items < sms ? items : sms);
    kern<<<grid, 256, intralay::BYTES, st>>>(p, recs, mq, mk, mg, mv);
    timing_post(st);
    return cudaGetLastError();
}

cudaError_t launch_chain_fwd_tc(const Params& p, const uint8_t* recs, bool store_states, cudaStream_t st,
                                bool transfer) {
    cudaError_t e = cudaFuncSetAttribute(chain_fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)chainlay::BYTES);
    if (e != cudaSuccess) return e;
    timing_pre(st, K_CHAIN_FWD_TC);
    const int flags = (store_states ? kChainStoreStates : 0) | (transfer ? kChainTransfer : 0);
    if (p.N <= 65535)   // segments in launch order, longest first (grid y holds at most 65535)
        chain_fwd_tc_kernel<<<dim3(p.H * (p.V / 32), p.N), 256, chainlay::BYTES, st>>>(p, recs,
                                                                                   flags | kChainRankMajor);
    else
        chain_fwd_tc_kernel<<<dim3(p.N, p.H, p.V / 32), 256, chainlay::BYTES, st>>>(p, recs, flags);
    timing_post(st);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ failure-detection self-test
//
// One CTA waits on an mbarrier that nothing arrives on, with the bounded wait every kernel here uses
// (a fixed number of polls), gives up and records KDA_ERR_TIMEOUT in the device status word, as the
// kernels' own fail paths do.  It shows the timeout path end to end without hanging or faulting.
__global__ void selftest_wait_kernel(int* status, uint32_t polls) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        mbar_fence_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !mbar_wait(&bar, 0, polls)) record_error(status, KDA_ERR_TIMEOUT);
}

cudaError_t launch_selftest_wait(int* status, cudaStream_t st) {
    selftest_wait_kernel<<<1, 32, 0, st>>>(status, 1u << 8);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ segment-parallel forward
//
// The chunk chain of a row is affine in its entering state: S_end = M S_begin + S_loc, with M the
// product of Diag(exp(Gamma_last)) - Kd^T W over the chunks and S_loc the end state from zero.  The
// segmented forward cuts each row into pieces, gets (M, S_loc) per piece from two chain passes run
// in parallel over pieces, propagates the true piece-entering states here, and runs the chain once
// more from them for the output.

// Pieces of the rows: row n (a document of cu_seqlens, or row n of B rows of T tokens when cu is
// null) is cut into ceil(len / L) pieces of L tokens (the last one shorter; none for an empty row).
// piece_cu[i] = first token of piece i, rows' pieces in order, row_piece[n] = first piece of row n;
// the Pmax - used unused pieces at the end are empty (piece_cu = TT).  One thread: the rows are few.
// A cu that does not start at 0, decreases or does not end at TT is reported in the status word and
// yields no pieces, so every later kernel finds nothing to do.
__global__ void piece_plan_kernel(const int32_t* cu, int rows, int T, int TT, int L, int Pmax, int32_t* piece_cu,
                                  int32_t* row_piece, int* status) {
    if (blockIdx.x != 0 || threadIdx.x != 0) return;
    bool ok = !cu || (cu[0] == 0 && cu[rows] == TT);
    for (int n = 0; ok && cu && n < rows; ++n) ok = cu[n + 1] >= cu[n];
    int np = 0;
    if (ok)
        for (int n = 0; n < rows; ++n) {
            row_piece[n] = np;
            const int b0 = cu ? cu[n] : n * T, e0 = cu ? cu[n + 1] : (n + 1) * T;
            for (int t = b0; t < e0 && np < Pmax; t += L) piece_cu[np++] = t;
        }
    else {
        record_error(status, KDA_ERR_INVALID_ARG);
        for (int n = 0; n < rows; ++n) row_piece[n] = 0;
    }
    row_piece[rows] = np;
    for (int i = np; i <= Pmax; ++i) piece_cu[i] = TT;
}
// One CTA per (row, head, slice of kCombineCols state columns); thread k owns row k of the slice
// (fp32).  For each piece of the row in order (last to first when `reverse`): record the piece's
// starting state, then S <- M S + S_loc.  M (64 KB) moves into shared memory by 16-byte cp.async
// copies, double buffered: the next piece's M is requested before this piece's product, so the
// serial walk along the row waits on the copy only when the product is shorter than the copy.  Rows
// of M are padded to 132 floats (16-byte aligned; a quarter warp's 16-byte row reads hit distinct
// banks).  The final S is the row's result: its final state, or for the reverse chain of the
// backward the gradient w.r.t. its initial state.
constexpr int kCombineCols = 4, kCombinePad = 132;
constexpr int kCombineSmem = (2 * 128 * kCombinePad + 128 * kCombineCols) * 4;
__global__ void __launch_bounds__(128) seg_combine_kernel(const float* S0, float* ST, const float* sloc,
                                                          const float* M, float* sstart, int H,
                                                          const int32_t* row_piece, int reverse) {
    extern __shared__ __align__(16) float csm[];
    float* sS = csm + 2 * 128 * kCombinePad;   // [128][kCombineCols]
    const int b = blockIdx.x, h = blockIdx.y, j0 = kCombineCols * blockIdx.z, k = threadIdx.x;
    float S[kCombineCols];
    {
        // the caller's state (4-byte alignment only): plain loads
        const float* src = S0 ? S0 + (((size_t)b * H + h) * 128 + k) * 128 + j0 : nullptr;
#pragma unroll
        for (int j = 0; j < kCombineCols; ++j) S[j] = src ? src[j] : 0.f;
    }
    const int p0 = row_piece[b], np = row_piece[b + 1] - p0;
    auto piece = [&](int i) { return reverse ? p0 + np - 1 - i : p0 + i; };
    auto fetch_m = [&](int i) {   // M of the i-th piece into buffer i & 1: 4096 chunks of 16 bytes
        const float* src = M + ((size_t)piece(i) * H + h) * 128 * 128;
        float* dst = csm + (i & 1) * 128 * kCombinePad;
        for (int c = k; c < 4096; c += 128) {
            const int r = c >> 5, c4 = (c & 31) * 4;
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(
                             __cvta_generic_to_shared(dst + r * kCombinePad + c4))),
                         "l"(src + r * 128 + c4)
                         : "memory");
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    if (np > 0) fetch_m(0);
    for (int i = 0; i < np; ++i) {
        const int pc = piece(i);
        const size_t base = ((size_t)pc * H + h) * 128 * 128;
        *reinterpret_cast<float4*>(sstart + base + (size_t)k * 128 + j0) = make_float4(S[0], S[1], S[2], S[3]);
        *reinterpret_cast<float4*>(sS + k * kCombineCols) = make_float4(S[0], S[1], S[2], S[3]);
        const float4 l = *reinterpret_cast<const float4*>(sloc + base + (size_t)k * 128 + j0);
        float acc[kCombineCols] = {l.x, l.y, l.z, l.w};
        if (i + 1 < np) {
            fetch_m(i + 1);
            asm volatile("cp.async.wait_group 1;" ::: "memory");
        } else {
            asm volatile("cp.async.wait_group 0;" ::: "memory");
        }
        __syncthreads();   // M of this piece and the slice of S are in shared memory
        const float* mrow = csm + (i & 1) * 128 * kCombinePad + k * kCombinePad;
#pragma unroll 4
        for (int kk = 0; kk < 128; kk += 4) {
            const float4 m = *reinterpret_cast<const float4*>(mrow + kk);
            const float mv[4] = {m.x, m.y, m.z, m.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float4 sv = *reinterpret_cast<const float4*>(sS + (kk + u) * kCombineCols);
                acc[0] += mv[u] * sv.x;
                acc[1] += mv[u] * sv.y;
                acc[2] += mv[u] * sv.z;
                acc[3] += mv[u] * sv.w;
            }
        }
        __syncthreads();   // every reader of this M buffer and of sS is done
#pragma unroll
        for (int j = 0; j < kCombineCols; ++j) S[j] = acc[j];
    }
    if (ST)
#pragma unroll
        for (int j = 0; j < kCombineCols; ++j) ST[(((size_t)b * H + h) * 128 + k) * 128 + j0 + j] = S[j];
}

cudaError_t launch_piece_plan(const int32_t* cu, int rows, int T, int TT, int L, int Pmax, int32_t* piece_cu,
                              int32_t* row_piece, int* status, cudaStream_t st) {
    piece_plan_kernel<<<1, 32, 0, st>>>(cu, rows, T, TT, L, Pmax, piece_cu, row_piece, status);
    return cudaGetLastError();
}
cudaError_t launch_seg_combine(const float* S0, float* ST, const float* sloc, const float* M, float* sstart, int rows,
                               int H, const int32_t* row_piece, bool reverse, cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(seg_combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kCombineSmem);
    if (e != cudaSuccess) return e;
    timing_pre(st, K_SEG_COMBINE);
    static_assert(kCombineCols == 4, "one float4 of state columns per thread");
    seg_combine_kernel<<<dim3(rows, H, 128 / kCombineCols), 128, kCombineSmem, st>>>(S0, ST, sloc, M, sstart, H,
                                                                                    row_piece, reverse ? 1 : 0);
    timing_post(st);
    return cudaGetLastError();
}

}  // namespace kda
