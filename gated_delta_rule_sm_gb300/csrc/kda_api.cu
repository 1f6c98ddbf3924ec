// kda_api.cu -- the extern "C" boundary: validation, workspace carving and launches.
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "kda.h"
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {

__device__ int g_status_word = 0;

static constexpr size_t kAlign = 256;
static constexpr int kGradCtas = 304;  // 2 CTAs per SM on a 152-SM GB300

static size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct Shape {
    int B, T, H, Hk, G, K, V, N, TT, NCmax, dtype, gate;
    bool varlen;
};

static kda_status check_dims(const kda_dims* d, int chunk_size, bool varlen, Shape* s) {
    if (!d) return KDA_ERR_INVALID_ARG;
    if (d->B < 1 || d->T < 1 || d->H < 1 || d->K < 1 || d->V < 1) return KDA_ERR_INVALID_ARG;
    const int Hk = d->Hk > 0 ? d->Hk : d->H;   // 0: one key head per value head
    if (d->Hk < 0 || d->H % Hk) return KDA_ERR_INVALID_ARG;
    if (d->dtype != KDA_BF16 && d->dtype != KDA_FP32) return KDA_ERR_INVALID_ARG;
    if (d->gate != KDA_GATE_LOWER_BOUNDED && d->gate != KDA_GATE_SOFTPLUS) return KDA_ERR_INVALID_ARG;
    if (chunk_size <= 0) return KDA_ERR_INVALID_ARG;
    if (d->K < 16 || d->V < 16) return KDA_ERR_INVALID_ARG;           // head dims below 16 are rejected
    // the chunk size is a blocking choice, not part of the result: 16, 32 and 64 all run the 64-token
    // kernels (segments still restart at every document start)
    if (chunk_size != 16 && chunk_size != 32 && chunk_size != kChunk) return KDA_ERR_UNSUPPORTED;
    if (d->K > 128 || d->V > 128 || d->K % 16 || d->V % 16) return KDA_ERR_UNSUPPORTED;
    const long long TT = (long long)d->B * d->T;
    if (TT > (1LL << 30) || TT * d->H * (d->K > d->V ? d->K : d->V) > (1LL << 40)) return KDA_ERR_UNSUPPORTED;
    if (varlen) {
        if (d->B != 1 || d->num_seqs < 1) return KDA_ERR_INVALID_ARG;
        if (d->num_seqs > (1 << 24)) return KDA_ERR_UNSUPPORTED;
    }
    s->B = d->B; s->T = d->T; s->H = d->H; s->K = d->K; s->V = d->V;
    s->Hk = Hk; s->G = d->H / Hk;
    s->dtype = d->dtype;
    s->gate = d->gate;
    s->varlen = varlen;
    s->N = varlen ? d->num_seqs : d->B;
    s->TT = (int)TT;
    s->NCmax = varlen ? (int)((TT + kChunk - 1) / kChunk + s->N) : d->B * ((d->T + kChunk - 1) / kChunk);
    return KDA_OK;
}

struct WsPlan {
    size_t off_chunk, off_rec, off_states, off_dstates, off_pdtb, off_palog, off_scratch, total;
    size_t off_dqv, off_dkv;   // grouped key heads: dq, dk per value head before the group sum
    size_t rec_stride, scratch_stride;
};

static WsPlan plan_simt(const Shape& s, bool bwd) {
    WsPlan w;
    memset(&w, 0, sizeof(w));
    const RecLayout L = RecLayout::make(s.K, s.V);
    w.rec_stride = bwd ? L.bwd_size : L.fwd_size;
    size_t o = 0;
    w.off_chunk = o; o = align_up(o + sizeof(int32_t) * (size_t)(2 * s.N + 1));   // chunk table, segment order
    w.off_rec = o; o = align_up(o + sizeof(float) * (size_t)s.NCmax * s.H * w.rec_stride);
    if (bwd) {
        const size_t kv = (size_t)s.K * s.V;
        w.off_states = o; o = align_up(o + sizeof(float) * (size_t)s.NCmax * s.H * kv);
        w.off_dstates = o; o = align_up(o + sizeof(float) * (size_t)s.NCmax * s.H * kv);
        w.off_pdtb = o; o = align_up(o + sizeof(float) * (size_t)s.NCmax * s.H * s.K);
        w.off_palog = o; o = align_up(o + sizeof(float) * (size_t)s.NCmax * s.H);
        w.scratch_stride = GradScratch::make(s.K, s.V).size;
        w.off_scratch = o; o = align_up(o + sizeof(float) * (size_t)kGradCtas * w.scratch_stride);
        if (s.G > 1) {
            w.off_dqv = o; o = align_up(o + sizeof(float) * (size_t)s.TT * s.H * s.K);
            w.off_dkv = o; o = align_up(o + sizeof(float) * (size_t)s.TT * s.H * s.K);
        }
    }
    w.total = o;
    return w;
}

// Tensor-core path: bf16 activations with K = V = 128.
static bool tc_eligible(const Shape& s) { return s.dtype == KDA_BF16 && s.K == 128 && s.V == 128; }
// The plain forward also takes K = V = 64 heads under the lower-bounded gate: the intra pass loads them
// as 128-channel tiles whose upper half the TMA fills with zeros, and the chain runs the two value
// slices that exist over a state whose rows 64..127 stay zero.
static bool tc_fwd_eligible(const Shape& s) {
    return tc_eligible(s) || (s.dtype == KDA_BF16 && s.K == 64 && s.V == 64 && s.gate == KDA_GATE_LOWER_BOUNDED);
}

// The tensor-core path's 16-token sub-block factorisation of the decay needs the lower-bounded
// gate with |lower_bound| <= 5 (exp of up to 16 * 5 stays inside fp32 range).  It also takes the
// unbounded gate: the diagonal sub-blocks of the intra-chunk forms then come from diag_tc_kernel,
// and the gradient kernel sums its diagonal sub-blocks pair by pair.
static bool tc_gate_ok(const Shape& s, float lb) {
    return s.gate == KDA_GATE_SOFTPLUS || (s.gate == KDA_GATE_LOWER_BOUNDED && lb >= -5.0f);
}

struct TcPlan {
    size_t off_chunk, off_rec, off_diag, total;
};

static TcPlan plan_tc_fwd(const Shape& s) {
    TcPlan w;
    size_t o = 0;
    w.off_chunk = o; o = align_up(o + sizeof(int32_t) * (size_t)(2 * s.N + 1));   // chunk table, segment order
    w.off_rec = o; o = align_up(o + tc_record_bytes(s.NCmax, s.H));
    w.off_diag = 0;
    if (s.gate == KDA_GATE_SOFTPLUS) { w.off_diag = o; o = align_up(o + diag_item_bytes() * s.NCmax * s.H); }
    w.total = o;
    return w;
}

struct TcBwdPlan {
    WsPlan simt;        // chunk table, fp32 backward records, states, partials, scratch
    size_t off_bwrec;   // reverse-chain records
    size_t off_u, off_du;   // U and dU per (chunk, head), written by the two chains
    size_t off_diag;    // unbounded gate: diagonal sub-blocks for the record pass (0 otherwise)
    size_t off_pad;     // K = V = 64 heads: three zero-padded 128 x 128 states per (row, head) (0 otherwise)
    size_t total;
};

// The tensor-core backward also takes bf16 K = V = 64 heads under the lower-bounded gate: every
// per-chunk record and tile is laid out for 128 channels, the record pass loads the heads as
// 128-channel tiles whose upper half is zero, and the chains run on zero-padded 128 x 128 states.
static bool tc_bwd_eligible(const Shape& s) {
    return tc_eligible(s) || (s.dtype == KDA_BF16 && s.K == 64 && s.V == 64 && s.gate == KDA_GATE_LOWER_BOUNDED);
}

static TcBwdPlan plan_tc_bwd(const Shape& s) {
    TcBwdPlan w;
    Shape s128 = s;   // the kernels' internal layouts are those of 128-channel heads
    s128.K = s128.V = 128;
    w.simt = plan_simt(s128, true);
    size_t o = w.simt.total;
    w.off_bwrec = o; o = align_up(o + (size_t)s.NCmax * s.H * bwrec::BYTES);
    w.off_u = o; o = align_up(o + sizeof(float) * (size_t)s.NCmax * s.H * 64 * s128.V);
    w.off_du = o; o = align_up(o + sizeof(float) * (size_t)s.NCmax * s.H * 64 * s128.V);
    w.off_diag = 0;
    if (s.gate == KDA_GATE_SOFTPLUS) { w.off_diag = o; o = align_up(o + diag_item_bytes() * s.NCmax * s.H); }
    w.off_pad = 0;
    if (s.K != 128) { w.off_pad = o; o = align_up(o + 3 * sizeof(float) * (size_t)s.N * s.H * 128 * 128); }
    w.total = o;
    return w;
}

static kda_status status_ptr(int** out) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return KDA_ERR_CUDA;
    *out = static_cast<int*>(p);
    return KDA_OK;
}

static Params base_params(const Shape& s, const void* q, const void* k, const void* v, const void* g_raw,
                          const void* beta_raw, const float* a_log, const float* dt_bias, float scale,
                          float lb, const int32_t* cu, const float* S0) {
    Params p;
    memset(&p, 0, sizeof(p));
    p.B = s.B; p.T = s.T; p.H = s.H; p.K = s.K; p.V = s.V; p.N = s.N; p.TT = s.TT;
    p.Hk = s.Hk; p.G = s.G;
    p.dtype = s.dtype; p.NCmax = s.NCmax;
    p.q = q; p.k = k; p.v = v; p.g_raw = g_raw; p.beta_raw = beta_raw;
    p.a_log = a_log; p.dt_bias = dt_bias; p.scale = scale; p.lb = lb; p.gate = s.gate;
    p.cu = cu; p.S0 = S0;
    return p;
}

static void carve(Params& p, const WsPlan& w, void* ws) {
    char* b = static_cast<char*>(ws);
    p.chunk_off = reinterpret_cast<int32_t*>(b + w.off_chunk);
    p.rec = reinterpret_cast<float*>(b + w.off_rec);
    p.rec_stride = w.rec_stride;
    if (w.off_states) {
        p.states = reinterpret_cast<float*>(b + w.off_states);
        p.dstates = reinterpret_cast<float*>(b + w.off_dstates);
        p.part_dtb = reinterpret_cast<float*>(b + w.off_pdtb);
        p.part_alog = reinterpret_cast<float*>(b + w.off_palog);
        p.scratch = reinterpret_cast<float*>(b + w.off_scratch);
        p.scratch_stride = w.scratch_stride;
        p.grad_ctas = kGradCtas;
        p.dq_v = w.off_dqv ? reinterpret_cast<float*>(b + w.off_dqv) : p.dq;
        p.dk_v = w.off_dkv ? reinterpret_cast<float*>(b + w.off_dkv) : p.dk;
    }
}

// The packed-document offsets' contract (nemo_automodel `kimi_k3.cp`, `segment_cu_seqlens` and
// `doc_ids_from_cu_seqlens`): N + 1 entries, starting at 0, never decreasing, ending at the token
// count.  Checked here when the caller hands over a host copy; plan_kernel checks the device array
// otherwise.
static kda_status check_cu_host(const Shape& s, const int32_t* cu, const int32_t* cu_host) {
    if (!cu_host) return KDA_OK;
    if (!cu) return KDA_ERR_INVALID_ARG;   // a host copy of offsets the call does not use
    if (cu_host[0] != 0 || cu_host[s.N] != s.TT) return KDA_ERR_INVALID_ARG;
    for (int n = 0; n < s.N; ++n)
        if (cu_host[n + 1] < cu_host[n]) return KDA_ERR_INVALID_ARG;
    return KDA_OK;
}

static kda_status common_checks(const kda_dims* dims, int chunk_size, const int32_t* cu, const int32_t* cu_host,
                                const void* q, const void* k, const void* v, const void* g_raw,
                                const void* beta_raw, const float* a_log, const float* dt_bias, float scale, float lb,
                                Shape* s) {
    kda_status st = check_dims(dims, chunk_size, cu != nullptr, s);
    if (st != KDA_OK) return st;
    st = check_cu_host(*s, cu, cu_host);
    if (st != KDA_OK) return st;
    if (!q || !k || !v || !g_raw || !beta_raw || !a_log || !dt_bias) return KDA_ERR_INVALID_ARG;
    if (!(lb < 0.0f) || !isfinite(lb)) return KDA_ERR_INVALID_ARG;   // lower_bound < 0 under either gate, as the page's executor checks
    if (!isfinite(scale)) return KDA_ERR_INVALID_ARG;
    return KDA_OK;
}

static kda_status check_ws(void* ws, size_t bytes, size_t need) {
    if (bytes < need) return KDA_ERR_WORKSPACE;
    if (need > 0 && (!ws || (reinterpret_cast<uintptr_t>(ws) % kAlign))) return KDA_ERR_WORKSPACE;
    return KDA_OK;
}

#define KDA_TRY_CUDA(expr)                              \
    do {                                                \
        if ((expr) != cudaSuccess) return KDA_ERR_CUDA; \
    } while (0)

static kda_status fwd_simt(const Shape& s, Params p, void* ws, size_t ws_bytes, cudaStream_t stream) {
    const WsPlan w = plan_simt(s, false);
    kda_status st = check_ws(ws, ws_bytes, w.total);
    if (st != KDA_OK) return st;
    st = status_ptr(&p.status);
    if (st != KDA_OK) return st;
    carve(p, w, ws);
    KDA_TRY_CUDA(launch_plan(p, stream));
    KDA_TRY_CUDA(launch_intra_simt(p, false, stream));
    KDA_TRY_CUDA(launch_chain_fwd_simt(p, false, stream));
    return KDA_OK;
}

// ---- kernel timing (kda_timing_*) ----
struct TimingState {
    bool active = false;
    int cap = 0, used = 0;
    bool open = false;           // a pre event is recorded, post pending
    cudaEvent_t* ev = nullptr;   // 2 * cap events
    int* ids = nullptr;
};
static TimingState g_timing;

void timing_pre(cudaStream_t st, int kernel_id) {
    TimingState& t = g_timing;
    if (!t.active || t.used >= t.cap) return;
    cudaEventRecord(t.ev[2 * t.used], st);
    t.ids[t.used] = kernel_id;
    t.open = true;
}

void timing_post(cudaStream_t st) {
    TimingState& t = g_timing;
    if (!t.active || !t.open) return;
    cudaEventRecord(t.ev[2 * t.used + 1], st);
    t.open = false;
    ++t.used;
}

static void timing_release() {
    TimingState& t = g_timing;
    if (t.ev) {
        for (int i = 0; i < 2 * t.cap; ++i) cudaEventDestroy(t.ev[i]);
        delete[] t.ev;
    }
    delete[] t.ids;
    t = TimingState();
}

static const char* kKernelNames[] = {"kda_plan",          "kda_intra_simt",   "kda_chain_fwd_simt",
                                     "kda_chain_bwd_simt", "kda_grad_simt",    "kda_param_reduce",
                                     "kda_empty_segment", "kda_intra_tc",     "kda_chain_fwd_tc",
                                     "kda_grad_tc",       "kda_bwd_pre",      "kda_chain_bwd_tc",
                                     "kda_chain_rec_tc",  "kda_group_sum",    "kda_short_conv_fwd",
                                     "kda_short_conv_bwd", "kda_short_conv_reduce", "kda_diag_tc",
                                     "kda_seg_combine",   "kda_gated_norm_fwd", "kda_gated_norm_bwd",
                                     "kda_gated_norm_reduce"};

// saved != NULL: also keep the fp32 backward record there (kda_fwd_save)
static kda_status fwd_tc(const Shape& s, Params p, void* ws, size_t ws_bytes, cudaStream_t stream,
                         float* saved = nullptr) {
    const TcPlan w = plan_tc_fwd(s);
    kda_status st = check_ws(ws, ws_bytes, w.total);
    if (st != KDA_OK) return st;
    st = status_ptr(&p.status);
    if (st != KDA_OK) return st;
    char* b = static_cast<char*>(ws);
    p.chunk_off = reinterpret_cast<int32_t*>(b + w.off_chunk);
    uint8_t* recs = reinterpret_cast<uint8_t*>(b + w.off_rec);
    if (saved) {   // the backward record, in the 128-channel layout (K = V = 64 heads padded)
        p.rec = saved;
        p.rec_stride = RecLayout::make(128, 128).bwd_size;
    }
    if (s.gate == KDA_GATE_SOFTPLUS) p.diag = reinterpret_cast<float*>(b + w.off_diag);
    KDA_TRY_CUDA(launch_plan(p, stream));
    if (p.diag) KDA_TRY_CUDA(launch_diag_tc(p, stream));
    if (!saved && !p.diag) KDA_TRY_CUDA(launch_intra2(p, recs, stream));
    else KDA_TRY_CUDA(launch_intra_tc(p, recs, saved ? 2 : 0, stream));
    KDA_TRY_CUDA(launch_chain_fwd_tc(p, recs, false, stream));
    return KDA_OK;
}

// Segment-parallel schedule: every row (a document of cu_seqlens, or one of B rows of T tokens) cut
// into pieces of at most L tokens, L a multiple of 64 so that the pieces' chunks are the rows'.  The
// pieces run as packed segments; Pmax bounds their number (unused ones are empty).
struct SegPlan {
    Shape ps;          // the pieces as packed segments
    int L, Pmax, rows;
    size_t off_piece_cu, off_row_piece, off_sloc, off_m, off_sstart;
};

static SegPlan plan_seg_shape(const Shape& s, int segments) {
    SegPlan w;
    w.rows = s.N;
    const int span = s.varlen ? s.TT : s.T;   // the longest row can be
    const int nch = (span + kChunk - 1) / kChunk;
    w.L = (nch + segments - 1) / segments * kChunk;
    // each row gives ceil(len / L) <= len / L + 1 pieces
    w.Pmax = s.varlen ? s.N + (s.TT + w.L - 1) / w.L : s.B * ((s.T + w.L - 1) / w.L);
    w.ps = s;
    w.ps.varlen = true;
    w.ps.N = w.Pmax;
    w.ps.NCmax = (int)(((long long)s.TT + kChunk - 1) / kChunk + w.Pmax);
    return w;
}

// The piece tables and the three fp32 states per piece and head (end state from zero, transfer
// matrix, true starting state), after `base` bytes of the piece problem's own workspace.
static size_t plan_seg_tail(SegPlan& w, size_t base) {
    const size_t st = sizeof(float) * (size_t)w.Pmax * w.ps.H * w.ps.K * w.ps.V;
    size_t o = base;
    w.off_piece_cu = o; o = align_up(o + sizeof(int32_t) * (size_t)(w.Pmax + 1));
    w.off_row_piece = o; o = align_up(o + sizeof(int32_t) * (size_t)(w.rows + 1));
    w.off_sloc = o; o = align_up(o + st);
    w.off_m = o; o = align_up(o + st);
    w.off_sstart = o; o = align_up(o + st);
    return o;
}

struct SegFwdPlan {
    SegPlan seg;
    TcPlan tc;
    size_t total;
};
static SegFwdPlan plan_seg_fwd(const Shape& s, int segments) {
    SegFwdPlan w;
    w.seg = plan_seg_shape(s, segments);
    w.tc = plan_tc_fwd(w.seg.ps);
    w.total = plan_seg_tail(w.seg, w.tc.total);
    return w;
}

// Params of the piece problem: the pieces as packed segments of the same chunks.
static Params piece_params(const Params& p, const SegPlan& w, char* ws) {
    Params pp = p;
    pp.N = w.ps.N;
    pp.NCmax = w.ps.NCmax;
    pp.cu = reinterpret_cast<int32_t*>(ws + w.off_piece_cu);
    return pp;
}

// Tensor-core backward.  saved == NULL: the intra kernel rebuilds the fp32 backward record in the
// workspace; otherwise the record kda_fwd_save kept is used and that pass is skipped.
static kda_status bwd_tc(const Shape& s, Params p, void* workspace, size_t workspace_bytes, cudaStream_t stream,
                         const float* saved) {
    const TcBwdPlan w = plan_tc_bwd(s);
    kda_status st = check_ws(workspace, workspace_bytes, w.total);
    if (st != KDA_OK) return st;
    st = status_ptr(&p.status);
    if (st != KDA_OK) return st;
    carve(p, w.simt, workspace);
    if (saved) p.rec = const_cast<float*>(saved);   // same layout and stride as the workspace record area
    uint8_t* bw = static_cast<uint8_t*>(workspace) + w.off_bwrec;
    p.chunk_u = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + w.off_u);
    p.chunk_du = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + w.off_du);
    Params pf = p;   // the forward state recompute writes no output and no final state
    pf.out = nullptr;
    pf.ST = nullptr;
    KDA_TRY_CUDA(launch_plan(p, stream));
    if (!saved) {
        if (s.gate == KDA_GATE_SOFTPLUS) {
            p.diag = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + w.off_diag);
            KDA_TRY_CUDA(launch_diag_tc(p, stream));
        }
        KDA_TRY_CUDA(launch_intra_tc(p, nullptr, 1, stream));
    }
    KDA_TRY_CUDA(launch_bwd_pre(p, bw, stream));
    float* user_dS0 = p.dS0;
    if (w.off_pad) {   // K = V = 64: the chains take and give zero-padded 128 x 128 states
        float* pad = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + w.off_pad);
        const size_t one = (size_t)s.N * s.H * 128 * 128;
        const int NH = s.N * s.H;
        if (p.S0) {
            KDA_TRY_CUDA(launch_state_pad(p.S0, pad, s.K, s.V, NH, stream));
            pf.S0 = pad;
        }
        if (p.dST) {
            KDA_TRY_CUDA(launch_state_pad(p.dST, pad + one, s.K, s.V, NH, stream));
            p.dST = pad + one;
        }
        if (p.dS0) p.dS0 = pad + 2 * one;
    }
    KDA_TRY_CUDA(launch_chain_rec_tc(pf, bw, stream));
    KDA_TRY_CUDA(launch_chain_bwd_tc(p, bw, stream));
    if (w.off_pad && user_dS0) KDA_TRY_CUDA(launch_state_unpad(p.dS0, user_dS0, s.K, s.V, s.N * s.H, stream));
    KDA_TRY_CUDA(launch_grad_tc(p, stream));
    return KDA_OK;
}

// Bytes of the record kda_fwd_save keeps (0 when the shape does not take the tensor-core path).
static size_t saved_bytes_for(const Shape& s) {
    if (!tc_bwd_eligible(s)) return 0;
    return sizeof(float) * (size_t)s.NCmax * s.H * RecLayout::make(128, 128).bwd_size;   // 128-channel layout
}

}  // namespace kda

using namespace kda;

extern "C" {

size_t kda_fwd_workspace_size(const kda_dims* dims, int chunk_size) {
    Shape s;
    if (!dims) return 0;
    if (check_dims(dims, chunk_size, dims->num_seqs > 0 && dims->B == 1, &s) != KDA_OK &&
        check_dims(dims, chunk_size, false, &s) != KDA_OK)
        return 0;
    // size for the varlen bound when num_seqs is given, which also covers the fixed-length layout;
    // the larger of the two paths, so either entry point can use it
    const size_t a = plan_simt(s, false).total;
    const size_t b = tc_fwd_eligible(s) ? plan_tc_fwd(s).total : 0;
    return a > b ? a : b;
}

size_t kda_bwd_workspace_size(const kda_dims* dims, int chunk_size) {
    Shape s;
    if (!dims) return 0;
    if (check_dims(dims, chunk_size, dims->num_seqs > 0 && dims->B == 1, &s) != KDA_OK &&
        check_dims(dims, chunk_size, false, &s) != KDA_OK)
        return 0;
    const size_t a = plan_simt(s, true).total;
    const size_t b = tc_bwd_eligible(s) ? plan_tc_bwd(s).total : 0;
    return a > b ? a : b;
}

kda_status kda_fwd_simt(const kda_dims* dims, const void* q, const void* k, const void* v, const void* g_raw,
                        const void* beta_raw, const float* a_log, const float* dt_bias, float scale,
                        float lower_bound, int chunk_size, const int32_t* cu_seqlens, const int32_t* cu_seqlens_host,
                        const float* initial_state, void* out, float* final_state, void* workspace,
                        size_t workspace_bytes, cudaStream_t stream) {
    Shape s;
    kda_status st = common_checks(dims, chunk_size, cu_seqlens, cu_seqlens_host, q, k, v, g_raw, beta_raw, a_log,
                                  dt_bias, scale, lower_bound, &s);
    if (st != KDA_OK) return st;
    if (!out) return KDA_ERR_INVALID_ARG;
    Params p = base_params(s, q, k, v, g_raw, beta_raw, a_log, dt_bias, scale, lower_bound, cu_seqlens,
                           initial_state);
    p.out = out;
    p.ST = final_state;
    return fwd_simt(s, p, workspace, workspace_bytes, stream);
}

kda_status kda_fwd(const kda_dims* dims, const void* q, const void* k, const void* v, const void* g_raw,
                   const void* beta_raw, const float* a_log, const float* dt_bias, float scale, float lower_bound,
                   int chunk_size, const int32_t* cu_seqlens, const int32_t* cu_seqlens_host,
                   const float* initial_state, void* out, float* final_state, void* workspace, size_t workspace_bytes,
                   cudaStream_t stream) {
    Shape s;
    kda_status st = common_checks(dims, chunk_size, cu_seqlens, cu_seqlens_host, q, k, v, g_raw, beta_raw, a_log,
                                  dt_bias, scale, lower_bound, &s);
    if (st != KDA_OK) return st;
    if (!out) return KDA_ERR_INVALID_ARG;
    Params p = base_params(s, q, k, v, g_raw, beta_raw, a_log, dt_bias, scale, lower_bound, cu_seqlens,
                           initial_state);
    p.out = out;
    p.ST = final_state;
    // the tensor-core path needs 16-byte aligned activations and outputs and a gate it can factorise
    if (!tc_fwd_eligible(s) || !tc_gate_ok(s, lower_bound) || !tc_inputs_aligned(p))
        return kda_fwd_simt(dims, q, k, v, g_raw, beta_raw, a_log, dt_bias, scale, lower_bound, chunk_size,
                            cu_seqlens, cu_seqlens_host, initial_state, out, final_state, workspace, workspace_bytes,
                            stream);
    p.out = out;
    p.ST = final_state;
    return fwd_tc(s, p, workspace, workspace_bytes, stream);
}

kda_status kda_bwd(const kda_dims* dims, const void* q, const void* k, const void* v, const void* g_raw,
                   const void* beta_raw, const float* a_log, const float* dt_bias, float scale, float lower_bound,
                   int chunk_size, const int32_t* cu_seqlens, const int32_t* cu_seqlens_host,
                   const float* initial_state, const void* dout, const float* dfinal_state, float* dq, float* dk,
                   float* dv, float* dg_raw, float* dbeta_raw, float* da_log, float* ddt_bias, float* dinitial_state,
                   void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    Shape s;
    kda_status st = common_checks(dims, chunk_size, cu_seqlens, cu_seqlens_host, q, k, v, g_raw, beta_raw, a_log,
                                  dt_bias, scale, lower_bound, &s);
    if (st != KDA_OK) return st;
    if (!dout || !dq || !dk || !dv || !dg_raw || !dbeta_raw || !da_log || !ddt_bias) return KDA_ERR_INVALID_ARG;
    Params p = base_params(s, q, k, v, g_raw, beta_raw, a_log, dt_bias, scale, lower_bound, cu_seqlens,
                           initial_state);
    p.dout = dout; p.dST = dfinal_state;
    p.dq = dq; p.dk = dk; p.dv = dv; p.dg_raw = dg_raw; p.dbeta_raw = dbeta_raw;
    p.da_log = da_log; p.ddt_bias = ddt_bias; p.dS0 = dinitial_state;
    if (tc_bwd_eligible(s) && tc_gate_ok(s, lower_bound) && tc_inputs_aligned(p))
        return bwd_tc(s, p, workspace, workspace_bytes, stream, nullptr);
    const WsPlan w = plan_simt(s, true);
    st = check_ws(workspace, workspace_bytes, w.total);
    if (st != KDA_OK) return st;
    st = status_ptr(&p.status);
    if (st != KDA_OK) return st;
    carve(p, w, workspace);
    KDA_TRY_CUDA(launch_plan(p, stream));
    KDA_TRY_CUDA(launch_intra_simt(p, true, stream));
    KDA_TRY_CUDA(launch_chain_fwd_simt(p, true, stream));
    KDA_TRY_CUDA(launch_chain_bwd_simt(p, stream));
    KDA_TRY_CUDA(launch_grad_simt(p, stream));
    return KDA_OK;
}

// Dims as the entry points read them: packed documents when num_seqs is given with B == 1 (this
// bound also covers B = 1 rows), rows otherwise.
static bool seg_shape(const kda_dims* dims, int chunk_size, int segments, Shape* s) {
    if (!dims || segments < 1) return false;
    if (check_dims(dims, chunk_size, dims->num_seqs > 0 && dims->B == 1, s) != KDA_OK &&
        check_dims(dims, chunk_size, false, s) != KDA_OK)
        return false;
    return tc_eligible(*s);
}

size_t kda_fwd_segmented_workspace_size(const kda_dims* dims, int chunk_size, int segments) {
    Shape s;
    return seg_shape(dims, chunk_size, segments, &s) ? plan_seg_fwd(s, segments).total : 0;
}

kda_status kda_fwd_segmented(const kda_dims* dims, const void* q, const void* k, const void* v, const void* g_raw,
                             const void* beta_raw, const float* a_log, const float* dt_bias, float scale,
                             float lower_bound, int chunk_size, int segments, const int32_t* cu_seqlens,
                             const int32_t* cu_seqlens_host, const float* initial_state, void* out,
                             float* final_state, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    Shape s;
    kda_status st = common_checks(dims, chunk_size, cu_seqlens, cu_seqlens_host, q, k, v, g_raw, beta_raw, a_log,
                                  dt_bias, scale, lower_bound, &s);
    if (st != KDA_OK) return st;
    if (!out || segments < 1) return KDA_ERR_INVALID_ARG;
    Params p = base_params(s, q, k, v, g_raw, beta_raw, a_log, dt_bias, scale, lower_bound, cu_seqlens,
                           initial_state);
    p.out = out;
    p.ST = final_state;
    if (!tc_eligible(s) || !tc_gate_ok(s, lower_bound) || !tc_inputs_aligned(p)) return KDA_ERR_UNSUPPORTED;
    const SegFwdPlan w = plan_seg_fwd(s, segments);
    st = check_ws(workspace, workspace_bytes, w.total);
    if (st != KDA_OK) return st;
    st = status_ptr(&p.status);
    if (st != KDA_OK) return st;
    char* b = static_cast<char*>(workspace);
    Params pp = piece_params(p, w.seg, b);
    pp.chunk_off = reinterpret_cast<int32_t*>(b + w.tc.off_chunk);
    if (s.gate == KDA_GATE_SOFTPLUS) pp.diag = reinterpret_cast<float*>(b + w.tc.off_diag);
    uint8_t* recs = reinterpret_cast<uint8_t*>(b + w.tc.off_rec);
    int32_t* row_piece = reinterpret_cast<int32_t*>(b + w.seg.off_row_piece);
    float* sloc = reinterpret_cast<float*>(b + w.seg.off_sloc);
    float* M = reinterpret_cast<float*>(b + w.seg.off_m);
    float* sstart = reinterpret_cast<float*>(b + w.seg.off_sstart);
    KDA_TRY_CUDA(launch_piece_plan(cu_seqlens, s.N, s.T, s.TT, w.seg.L, w.seg.Pmax, const_cast<int32_t*>(pp.cu),
                                   row_piece, p.status, stream));
    KDA_TRY_CUDA(launch_plan(pp, stream));
    if (pp.diag) KDA_TRY_CUDA(launch_diag_tc(pp, stream));
    if (!pp.diag) KDA_TRY_CUDA(launch_intra2(pp, recs, stream));   // the chain record, as in kda_fwd
    else KDA_TRY_CUDA(launch_intra_tc(pp, recs, 0, stream));
    Params pa = pp;   // local end states: from zero, no output
    pa.S0 = nullptr;
    pa.out = nullptr;
    pa.ST = sloc;
    KDA_TRY_CUDA(launch_chain_fwd_tc(pa, recs, false, stream));
    pa.ST = M;        // transfer matrices: from the identity with U0 taken as zero
    KDA_TRY_CUDA(launch_chain_fwd_tc(pa, recs, false, stream, true));
    KDA_TRY_CUDA(launch_seg_combine(initial_state, final_state, sloc, M, sstart, s.N, s.H, row_piece, false, stream));
    Params pc = pp;   // the output, from the true entering states
    pc.S0 = sstart;
    pc.out = out;
    pc.ST = nullptr;
    KDA_TRY_CUDA(launch_chain_fwd_tc(pc, recs, false, stream));
    return KDA_OK;
}

struct SegBwdPlan {
    SegPlan seg;
    TcBwdPlan tc;
    size_t total;
};
static SegBwdPlan plan_seg_bwd(const Shape& s, int segments) {
    SegBwdPlan w;
    w.seg = plan_seg_shape(s, segments);
    w.tc = plan_tc_bwd(w.seg.ps);
    w.total = plan_seg_tail(w.seg, w.tc.total);
    return w;
}

size_t kda_bwd_segmented_workspace_size(const kda_dims* dims, int chunk_size, int segments) {
    Shape s;
    return seg_shape(dims, chunk_size, segments, &s) ? plan_seg_bwd(s, segments).total : 0;
}

kda_status kda_bwd_segmented(const kda_dims* dims, const void* q, const void* k, const void* v, const void* g_raw,
                             const void* beta_raw, const float* a_log, const float* dt_bias, float scale,
                             float lower_bound, int chunk_size, int segments, const int32_t* cu_seqlens,
                             const int32_t* cu_seqlens_host, const float* initial_state, const void* dout,
                             const float* dfinal_state, float* dq, float* dk, float* dv, float* dg_raw,
                             float* dbeta_raw, float* da_log, float* ddt_bias, float* dinitial_state, void* workspace,
                             size_t workspace_bytes, cudaStream_t stream) {
    Shape s;
    kda_status st = common_checks(dims, chunk_size, cu_seqlens, cu_seqlens_host, q, k, v, g_raw, beta_raw, a_log,
                                  dt_bias, scale, lower_bound, &s);
    if (st != KDA_OK) return st;
    if (!dout || !dq || !dk || !dv || !dg_raw || !dbeta_raw || !da_log || !ddt_bias || segments < 1)
        return KDA_ERR_INVALID_ARG;
    Params p = base_params(s, q, k, v, g_raw, beta_raw, a_log, dt_bias, scale, lower_bound, cu_seqlens,
                           initial_state);
    p.dout = dout; p.dST = dfinal_state;
    p.dq = dq; p.dk = dk; p.dv = dv; p.dg_raw = dg_raw; p.dbeta_raw = dbeta_raw;
    p.da_log = da_log; p.ddt_bias = ddt_bias; p.dS0 = dinitial_state;
    if (!tc_eligible(s) || !tc_gate_ok(s, lower_bound) || !tc_inputs_aligned(p)) return KDA_ERR_UNSUPPORTED;
    const SegBwdPlan w = plan_seg_bwd(s, segments);
    st = check_ws(workspace, workspace_bytes, w.total);
    if (st != KDA_OK) return st;
    st = status_ptr(&p.status);
    if (st != KDA_OK) return st;
    char* b = static_cast<char*>(workspace);
    Params pp = piece_params(p, w.seg, b);
    carve(pp, w.tc.simt, workspace);
    uint8_t* bw = reinterpret_cast<uint8_t*>(b + w.tc.off_bwrec);
    pp.chunk_u = reinterpret_cast<float*>(b + w.tc.off_u);
    pp.chunk_du = reinterpret_cast<float*>(b + w.tc.off_du);
    int32_t* row_piece = reinterpret_cast<int32_t*>(b + w.seg.off_row_piece);
    float* sloc = reinterpret_cast<float*>(b + w.seg.off_sloc);
    float* M = reinterpret_cast<float*>(b + w.seg.off_m);
    float* sstart = reinterpret_cast<float*>(b + w.seg.off_sstart);
    KDA_TRY_CUDA(launch_piece_plan(cu_seqlens, s.N, s.T, s.TT, w.seg.L, w.seg.Pmax, const_cast<int32_t*>(pp.cu),
                                   row_piece, p.status, stream));
    KDA_TRY_CUDA(launch_plan(pp, stream));
    if (s.gate == KDA_GATE_SOFTPLUS) {
        pp.diag = reinterpret_cast<float*>(b + w.tc.off_diag);
        KDA_TRY_CUDA(launch_diag_tc(pp, stream));
    }
    KDA_TRY_CUDA(launch_intra_tc(pp, nullptr, 1, stream));
    KDA_TRY_CUDA(launch_bwd_pre(pp, bw, stream));
    // the states entering every chunk: local end states and transfer matrices of the pieces, the
    // pieces' true entering states along each row, then the recompute chain from those
    Params pf = pp;
    pf.out = nullptr;
    pf.ST = sloc;
    KDA_TRY_CUDA(launch_chain_rec_tc(pf, bw, stream, kBwdChainLocal));
    pf.ST = M;
    KDA_TRY_CUDA(launch_chain_rec_tc(pf, bw, stream, kBwdChainTransfer));
    KDA_TRY_CUDA(launch_seg_combine(initial_state, nullptr, sloc, M, sstart, s.N, s.H, row_piece, false, stream));
    pf.S0 = sstart;
    pf.ST = nullptr;
    KDA_TRY_CUDA(launch_chain_rec_tc(pf, bw, stream, kBwdChainFull));
    // the reverse chain likewise, last piece to first: dS leaving each piece, and the row's dS_0
    Params pr = pp;
    pr.dS0 = sloc;
    KDA_TRY_CUDA(launch_chain_bwd_tc(pr, bw, stream, kBwdChainLocal));
    pr.dS0 = M;
    KDA_TRY_CUDA(launch_chain_bwd_tc(pr, bw, stream, kBwdChainTransfer));
    KDA_TRY_CUDA(launch_seg_combine(dfinal_state, dinitial_state, sloc, M, sstart, s.N, s.H, row_piece, true, stream));
    pr.dST = sstart;
    pr.dS0 = nullptr;
    KDA_TRY_CUDA(launch_chain_bwd_tc(pr, bw, stream, kBwdChainFull));
    KDA_TRY_CUDA(launch_grad_tc(pp, stream));
    return KDA_OK;
}

size_t kda_saved_size(const kda_dims* dims, int chunk_size) {
    Shape s;
    if (!dims) return 0;
    if (check_dims(dims, chunk_size, dims->num_seqs > 0 && dims->B == 1, &s) != KDA_OK &&
        check_dims(dims, chunk_size, false, &s) != KDA_OK)
        return 0;
    return saved_bytes_for(s);
}

kda_status kda_fwd_save(const kda_dims* dims, const void* q, const void* k, const void* v, const void* g_raw,
                        const void* beta_raw, const float* a_log, const float* dt_bias, float scale,
                        float lower_bound, int chunk_size, const int32_t* cu_seqlens, const int32_t* cu_seqlens_host,
                        const float* initial_state, void* out, float* final_state, void* saved, size_t saved_bytes,
                        void* workspace,
                        size_t workspace_bytes, cudaStream_t stream) {
    Shape s;
    kda_status st = common_checks(dims, chunk_size, cu_seqlens, cu_seqlens_host, q, k, v, g_raw, beta_raw, a_log,
                                  dt_bias, scale, lower_bound, &s);
    if (st != KDA_OK) return st;
    if (!out) return KDA_ERR_INVALID_ARG;
    Params p = base_params(s, q, k, v, g_raw, beta_raw, a_log, dt_bias, scale, lower_bound, cu_seqlens,
                           initial_state);
    p.out = out;
    p.ST = final_state;
    if (!tc_bwd_eligible(s) || !tc_gate_ok(s, lower_bound) || !tc_inputs_aligned(p)) return KDA_ERR_UNSUPPORTED;
    const size_t need = saved_bytes_for(s);
    if (!saved || saved_bytes < need || (reinterpret_cast<uintptr_t>(saved) % kAlign)) return KDA_ERR_WORKSPACE;
    p.out = out;
    p.ST = final_state;
    return fwd_tc(s, p, workspace, workspace_bytes, stream, static_cast<float*>(saved));
}

kda_status kda_bwd_saved(const kda_dims* dims, const void* q, const void* k, const void* v, const void* g_raw,
                         const void* beta_raw, const float* a_log, const float* dt_bias, float scale,
                         float lower_bound, int chunk_size, const int32_t* cu_seqlens,
                         const int32_t* cu_seqlens_host, const float* initial_state, const void* dout,
                         const float* dfinal_state, float* dq, float* dk, float* dv,
                         float* dg_raw, float* dbeta_raw, float* da_log, float* ddt_bias, float* dinitial_state,
                         const void* saved, size_t saved_bytes, void* workspace, size_t workspace_bytes,
                         cudaStream_t stream) {
    Shape s;
    kda_status st = common_checks(dims, chunk_size, cu_seqlens, cu_seqlens_host, q, k, v, g_raw, beta_raw, a_log,
                                  dt_bias, scale, lower_bound, &s);
    if (st != KDA_OK) return st;
    if (!dout || !dq || !dk || !dv || !dg_raw || !dbeta_raw || !da_log || !ddt_bias) return KDA_ERR_INVALID_ARG;
    Params p = base_params(s, q, k, v, g_raw, beta_raw, a_log, dt_bias, scale, lower_bound, cu_seqlens,
                           initial_state);
    p.dout = dout; p.dST = dfinal_state;
    p.dq = dq; p.dk = dk; p.dv = dv; p.dg_raw = dg_raw; p.dbeta_raw = dbeta_raw;
    p.da_log = da_log; p.ddt_bias = ddt_bias; p.dS0 = dinitial_state;
    if (!tc_bwd_eligible(s) || !tc_gate_ok(s, lower_bound) || !tc_inputs_aligned(p)) return KDA_ERR_UNSUPPORTED;
    const size_t need = saved_bytes_for(s);
    if (!saved || saved_bytes < need || (reinterpret_cast<uintptr_t>(saved) % kAlign)) return KDA_ERR_WORKSPACE;
    return bwd_tc(s, p, workspace, workspace_bytes, stream, static_cast<const float*>(saved));
}

const char* kda_status_string(kda_status s) {
    switch (s) {
        case KDA_OK: return "ok";
        case KDA_ERR_INVALID_ARG: return "invalid argument";
        case KDA_ERR_UNSUPPORTED: return "unsupported shape or parameter";
        case KDA_ERR_CUDA: return "CUDA error";
        case KDA_ERR_TIMEOUT: return "device wait timed out";
        case KDA_ERR_WORKSPACE: return "workspace too small or misaligned";
    }
    return "unknown status";
}

kda_status kda_device_status(int reset) {
    int v = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return KDA_ERR_CUDA;
    if (cudaMemcpyFromSymbol(&v, g_status_word, sizeof(int)) != cudaSuccess) return KDA_ERR_CUDA;
    if (reset) {
        const int z = 0;
        if (cudaMemcpyToSymbol(g_status_word, &z, sizeof(int)) != cudaSuccess) return KDA_ERR_CUDA;
    }
    return static_cast<kda_status>(v);
}

kda_status kda_selftest_wait_timeout(cudaStream_t stream) {
    int* status = nullptr;
    kda_status st = status_ptr(&status);
    if (st != KDA_OK) return st;
    KDA_TRY_CUDA(launch_selftest_wait(status, stream));
    return KDA_OK;
}

int kda_version(void) { return 100; }

kda_status kda_timing_begin(int max_launches) {
    timing_release();
    if (max_launches <= 0) return KDA_ERR_INVALID_ARG;
    TimingState& t = g_timing;
    t.cap = max_launches;
    t.ev = new cudaEvent_t[2 * (size_t)max_launches];
    t.ids = new int[max_launches];
    for (int i = 0; i < 2 * max_launches; ++i) {
        if (cudaEventCreate(&t.ev[i]) != cudaSuccess) {
            t.cap = i / 2;
            for (int j = 0; j < i; ++j) cudaEventDestroy(t.ev[j]);
            delete[] t.ev;
            delete[] t.ids;
            t = TimingState();
            return KDA_ERR_CUDA;
        }
    }
    t.active = true;
    return KDA_OK;
}

int kda_timing_end(float* ms, int* kernel_ids, int cap) {
    TimingState& t = g_timing;
    if (!t.active) return 0;
    t.active = false;
    int n = t.used < cap ? t.used : cap;
    int ok = 1;
    for (int i = 0; i < n; ++i) {
        float x = 0.f;
        if (cudaEventSynchronize(t.ev[2 * i + 1]) != cudaSuccess ||
            cudaEventElapsedTime(&x, t.ev[2 * i], t.ev[2 * i + 1]) != cudaSuccess)
            ok = 0;
        if (ms) ms[i] = x;
        if (kernel_ids) kernel_ids[i] = t.ids[i];
    }
    timing_release();
    return ok ? n : -1;
}

const char* kda_kernel_name(int kernel_id) {
    if (kernel_id < 0 || kernel_id >= (int)(sizeof(kKernelNames) / sizeof(kKernelNames[0]))) return "unknown";
    return kKernelNames[kernel_id];
}

}  // extern "C"
