// kda_internal.h -- host/device layouts and launchers shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

#include "kda_common.cuh"

namespace kda {

// Per (chunk, head) record of the SIMT path, in floats.
struct RecLayout {
    size_t W, Qg, Kd, U0, A, gC;           // forward fields
    size_t Kg, N, G, qh, kh, B, beta, rn;  // backward extras (rn: 1/|q_t|, then 1/|k_t|)
    size_t fwd_size, bwd_size;
    __host__ __device__ static RecLayout make(int K, int V) {
        RecLayout r;
        size_t o = 0;
        // W, Kd and gC first and adjacent: in the tensor-core record (K = V = 128) their 66048 bytes hold
        // the backward chains' operand slot instead (chainrec: Kd and -W as bf16 hi / lo, then gC)
        r.W = o; o += 64 * (size_t)K;
        r.Kd = o; o += 64 * (size_t)K;
        r.gC = o; o += (size_t)K;
        r.Qg = o; o += 64 * (size_t)K;
        r.U0 = o; o += 64 * (size_t)V;
        r.A = o; o += 64 * 64;
        r.fwd_size = (o + 63) / 64 * 64;
        r.Kg = o; o += 64 * (size_t)K;
        r.N = o; o += 64 * 64;
        r.G = o; o += 64 * (size_t)K;
        r.qh = o; o += 64 * (size_t)K;
        r.kh = o; o += 64 * (size_t)K;
        r.B = o; o += 64 * 64;
        r.beta = o; o += 64;
        r.rn = o; o += 128;
        r.bwd_size = (o + 63) / 64 * 64;
        // (every field starts on a multiple of 4 floats: the tensor-core record pass writes rows of B and A
        // with 16-byte stores)
        return r;
    }
};

// Per-CTA scratch of the SIMT gradient kernel, in floats.
struct GradScratch {
    size_t dO, Vin, Vt, U, dU, dY, tmp;    // [64][V] (tmp: [64][max(V,64)])
    size_t dT, dA, dN, dL;                 // [64][64]
    size_t dQg, dKd, dKg, dq, dk, dG;      // [64][K]
    size_t dbeta;                          // [64]
    size_t size;
    __host__ __device__ static GradScratch make(int K, int V) {
        GradScratch z;
        size_t o = 0;
        const size_t cv = 64 * (size_t)V, ck = 64 * (size_t)K, cc = 64 * 64;
        z.dO = o; o += cv; z.Vin = o; o += cv; z.Vt = o; o += cv; z.U = o; o += cv;
        z.dU = o; o += cv; z.dY = o; o += cv;
        z.tmp = o; o += 64 * (size_t)(V > 64 ? V : 64);
        z.dT = o; o += cc; z.dA = o; o += cc; z.dN = o; o += cc; z.dL = o; o += cc;
        z.dQg = o; o += ck; z.dKd = o; o += ck; z.dKg = o; o += ck; z.dq = o; o += ck; z.dk = o; o += ck;
        z.dG = o; o += ck;
        z.dbeta = o; o += 64;
        z.size = (o + 63) / 64 * 64;
        return z;
    }
};

// Kernel ids for kda_kernel_name / kda_timing_end.
enum KernelId {
    K_PLAN = 0, K_INTRA_SIMT, K_CHAIN_FWD_SIMT, K_CHAIN_BWD_SIMT, K_GRAD_SIMT, K_PARAM_REDUCE, K_EMPTY_SEG,
    K_INTRA_TC, K_CHAIN_FWD_TC, K_GRAD_TC, K_BWD_PRE, K_CHAIN_BWD_TC, K_CHAIN_REC_TC, K_GROUP_SUM,
    K_CONV_FWD, K_CONV_BWD, K_CONV_REDUCE, K_DIAG_TC, K_SEG_COMBINE, K_NORM_FWD, K_NORM_BWD, K_NORM_REDUCE,
    K_NUM_KERNELS
};

// Chain record of the tensor-core forward, one per (chunk, head), written by the intra-chunk kernels in
// exactly the shared-memory layouts the forward chain's MMAs read (bytes).  The chain's operands are fp16:
// its values stay far inside fp16's range (|W|, |Qg|, |S|, |U|, |Kd|, |Aqk| of order 1 to 10), where the
// 11-bit significand gives every product tf32-like accuracy in one kind::f16 MMA.
namespace tcrec {
constexpr uint32_t WQ = 0;            // [W; Qg]  fp16, 128 rows x 128 K (c), MN-major: mn_bf16(r, c, 128, 2048)
constexpr uint32_t U0 = 32768;        // U0       fp32, per 32-column slice z (j in [32z, 32z+32)): [64 t][32 j] at
                                      // U0 + z U0_SLICE, 16-byte chunks of a row swizzled (u0_off)
constexpr uint32_t KD = 65536;        // Kd^T     fp16, 128 rows (c) x 64 K (t), K-major: km_bf16(c, t, 1024, 128)
constexpr uint32_t AQ = 81920;        // Aqk      fp16, 64 rows (t) x 64 K (s), K-major: km_bf16(t, s, 1024, 128)
constexpr uint32_t GC = 90112;        // exp(Gamma_last) fp32 [128]
constexpr uint32_t BYTES = 91136;     // record stride (1 KB aligned)
constexpr uint32_t U0_SLICE = 8192;   // one 32-column slice of U0
constexpr uint32_t TAIL = BYTES - KD; // KD + AQ + GC (+ padding), contiguous
// Byte offset of U0[t][j] inside its slice (j < 32 the column within the slice): row t holds 32 floats,
// its 16-byte chunk c at position c ^ (t % 8).  The writer (thread = column j) stores a whole 128-byte row
// per warp instruction; the reader (thread = row t) loads 16-byte chunks with no bank conflict.
__host__ __device__ constexpr uint32_t u0_off(int t, int j) {
    return 4u * static_cast<uint32_t>(t * 32 + ((((j >> 2) ^ (t & 7))) << 2) + (j & 3));
}
}  // namespace tcrec

// Record of the two tcgen05 state chains of the backward, per (chunk, head), K = V = 128 (bytes).
// Both chains run  X = Y + A1 Z,  Z' = Diag(exp(Gamma_last)) Z + A2 X (+ P)  with every product in
// split precision: operand = hi + lo, both bf16 (hi = bf16(x), lo = bf16(x - hi)), and the products
// hi*hi + hi*lo + lo*hi (relative error ~1e-5).  The gradient of the log-decay at the end of a chunk
// carries dS_end * S_end-sized terms far larger than its typical value, so the states and state
// gradients need far better than tf32's 2^-11.
//   forward state recompute (Z = S entering chunk c):  A1 = -W,  A2 = Kd^T,  Y = U0, no P;
//   reverse chain (Z = dS leaving chunk c):            A1 = Kd,  A2 = -W^T,  Y = scale Aqk^T dO,
//                                                      P = scale Qg^T dO.
// One slot serves both: Kd and -W are stored once as [128 c][64 t] bf16 K-major tiles
// (km_bf16(c, t, 1024, 128)), the layout in which the intra pass produces them (a thread per channel);
// read with swapped strides the same bytes are the MN-major layout of Kd and -W (M = t, K = c).  The
// slot leads each chunk's tensor-core record and moves into shared memory by one bulk copy:
namespace chainrec {
constexpr uint32_t KD = 0;           // Kd  hi
constexpr uint32_t KD_LO = 16384;    // Kd  lo
constexpr uint32_t WN = 32768;       // -W  hi
constexpr uint32_t WN_LO = 49152;    // -W  lo
constexpr uint32_t GC = 65536;       // exp(Gamma_last) fp32 [128]
constexpr uint32_t SLOT = 66048;
}  // namespace chainrec

namespace bwrec {
constexpr uint32_t Y = 0;                       // fp32 [64 t][128 j] in x4 order: scale Aqk^T dO
constexpr uint32_t P = Y + 32768;               // fp32 [128 c][128 j] in x4 order: scale Qg^T dO
constexpr uint32_t BYTES = P + 65536;           // record stride (256-byte multiple)
}  // namespace bwrec

// "x4 order" of an fp32 tile of `rows` rows and 128 value columns: element (row, j) at
// x4_off(row, j, rows) = (j / 4, row, j % 4) row-major.  Four adjacent columns of one row form a
// 16-byte chunk and the chunks of consecutive rows are adjacent, so a warp whose lanes own
// consecutive rows moves whole 128-byte lines with 16-byte accesses.  The tiles passed between the
// backward's tensor-core kernels use it: Y and P above, and the per-chunk states, state gradients,
// U and dU that the two chains write for the gradient kernel.
__host__ __device__ constexpr size_t x4_off(int row, int j, int rows) {
    return ((size_t)(j >> 2) * rows + row) * 4 + (j & 3);
}

// Launch bracketing for kda_timing_*: no-ops unless timing is active.
void timing_pre(cudaStream_t st, int kernel_id);
void timing_post(cudaStream_t st);

cudaError_t launch_plan(const Params& p, cudaStream_t st);
cudaError_t launch_intra_simt(const Params& p, bool bwd, cudaStream_t st);
cudaError_t launch_chain_fwd_simt(const Params& p, bool store_states, cudaStream_t st);
cudaError_t launch_chain_bwd_simt(const Params& p, cudaStream_t st);
cudaError_t launch_grad_simt(const Params& p, cudaStream_t st);
cudaError_t launch_param_reduce(const Params& p, cudaStream_t st);
cudaError_t launch_group_sum(const Params& p, cudaStream_t st);   // dq_v, dk_v -> dq, dk when G > 1
cudaError_t launch_grad_tc(const Params& p, cudaStream_t st);
cudaError_t launch_bwd_pre(const Params& p, uint8_t* bw, cudaStream_t st);
// The two state chains of the backward.  kBwdChainFull: from p.S0 / p.dST, writing the per-chunk
// tiles the gradient kernel reads (and p.ST / p.dS0 at the end if set); kBwdChainLocal: from zero,
// only the end state (into p.ST / p.dS0); kBwdChainTransfer: from the identity with Y and P taken as
// zero, only the end state, which is then the segment's transfer matrix.
enum BwdChainMode { kBwdChainFull = 0, kBwdChainLocal = 1, kBwdChainTransfer = 2 };
cudaError_t launch_chain_bwd_tc(const Params& p, const uint8_t* bw, cudaStream_t st, int mode = kBwdChainFull);
// K = V = 64 heads on the tensor-core backward: caller states [NH, K, V] <-> zero-padded [NH, 128, 128]
// (src == null pads zeros)
cudaError_t launch_state_pad(const float* src, float* dst, int K, int V, int NH, cudaStream_t st);
cudaError_t launch_state_unpad(const float* src, float* dst, int K, int V, int NH, cudaStream_t st);
cudaError_t launch_chain_rec_tc(const Params& p, const uint8_t* bw, cudaStream_t st, int mode = kBwdChainFull);

// tensor-core path (bf16, K = V = 128)
size_t tc_record_bytes(int NCmax, int H);
bool tc_inputs_aligned(const Params& p);
// Unbounded gate: the diagonal 16 x 16 blocks of Bkk and Aqk per (chunk, head), into p.diag
// (diag_item_bytes() each), before the intra kernel.
size_t diag_item_bytes();
cudaError_t launch_diag_tc(const Params& p, cudaStream_t st);
// mode 0: forward chain record; 1: fp32 backward record; 2: both
cudaError_t launch_intra_tc(const Params& p, uint8_t* recs, int mode, cudaStream_t st);
// the forward chain record under the lower-bounded gate, two CTAs per SM (kda_intra2.cu)
cudaError_t launch_intra2(const Params& p, uint8_t* recs, cudaStream_t st);
// transfer: start from the identity with U0 taken as zero, so that the final state is the transfer matrix
cudaError_t launch_chain_fwd_tc(const Params& p, const uint8_t* recs, bool store_states, cudaStream_t st,
                                bool transfer = false);
// segment-parallel schedule: the pieces of the rows (documents of cu, or B rows of T tokens when cu
// is null) at most L tokens long, at most Pmax of them, and the serial propagation of the pieces'
// starting states S_{k+1} = M_k S_k + S_loc,k along each row (fp32, K = V = 128), first to last, or
// last to first for the reverse chain of the backward
cudaError_t launch_piece_plan(const int32_t* cu, int rows, int T, int TT, int L, int Pmax, int32_t* piece_cu,
                              int32_t* row_piece, int* status, cudaStream_t st);
cudaError_t launch_seg_combine(const float* S0, float* ST, const float* sloc, const float* M, float* sstart, int rows,
                               int H, const int32_t* row_piece, bool reverse, cudaStream_t st);
// failure-detection self-test: a bounded wait that cannot complete records KDA_ERR_TIMEOUT
cudaError_t launch_selftest_wait(int* status, cudaStream_t st);

}  // namespace kda
