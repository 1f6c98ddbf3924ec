/*
 * kda.h -- C ABI of the GB300 (sm_103a) Kimi Delta Attention library.
 *
 * The operation is the chunkwise KDA gated delta rule: per head and token
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *     o_t = scale * S_t^T q_t
 *
 * ("[kimi k3] add eager reference model with FSDP2", torchtitan PR #4025:
 * chunk_kda with the gate activation, beta sigmoid and q/k L2 norm fused into
 * the kernel, checked against the explicit recurrence forward and backward).
 * The prologue is computed inside the kernels:
 *     q_hat = q / sqrt(|q|^2 + 1e-6), k_hat likewise (per head, over K)
 *     beta  = sigmoid(beta_raw)
 *     g     = lower_bound * sigmoid(exp(a_log_h) * (g_raw + dt_bias_{h,c})),  alpha = exp(g)
 * (hyper-parallel "KDA context-parallel executors", `_run_local_kda`: the
 * fused backend requires this lower-bounded gate; the exact formula is not
 * printed on the pages and is this library's reading).  The same page keeps a
 * second, unbounded gate behind `safe_gate=False` (and the torchtitan note
 * tests the kernel under each of the two gate activations); selected by
 * kda_dims.gate, it is read as
 *     g     = -exp(a_log_h) * softplus(g_raw + dt_bias_{h,c})
 * (again unprinted; the plainest unbounded form over the same ingredients).
 *
 * Layouts follow `_validate_projected_inputs` on the same page (token-first,
 * contiguous, row-major); H counts value heads and Hk key heads:
 *     q, k            [B, T, Hk, K]       dtype (bf16 or fp32)
 *     g_raw           [B, T, H, K]        dtype
 *     v, out, dout    [B, T, H, V]        dtype
 *     beta_raw        [B, T, H]           dtype
 *     a_log           [H]                 fp32
 *     dt_bias         [H * K]             fp32
 *     states          [N, H, K, V]        fp32  (initial, final and their gradients)
 *     gradients       same shape as their input, always fp32
 * Grouped key heads (the same page's checks let num_v_heads be a multiple of
 * num_k_heads): value head h reads key head h / (H / Hk); dq and dk sum over
 * the value heads of each key head.  Hk = H is the ungrouped case.
 * Packed documents (nemo_automodel `kimi_k3.cp`, `segment_cu_seqlens`): with
 * cu_seqlens != NULL, B must be 1 and segment n is tokens
 * [cu_seqlens[n], cu_seqlens[n+1]) of the T tokens; each segment is its own
 * recurrence starting from initial_state[n] (or zero).  Without cu_seqlens
 * the N = B rows are the segments.  The same page's contract for the offsets
 * (`segment_cu_seqlens`, `doc_ids_from_cu_seqlens`): N + 1 entries, the
 * first 0, never decreasing, the last equal to T (empty segments are
 * allowed and pass their state through).
 *   - cu_seqlens_host (optional, HOST memory, N + 1 int32, read during the
 *     call only): a host copy of the same offsets.  When given, the contract
 *     is checked on the host and a violation returns KDA_ERR_INVALID_ARG
 *     before anything is enqueued; it is also KDA_ERR_INVALID_ARG without
 *     cu_seqlens.  The library trusts the caller that both copies agree.
 *   - Without the host copy the device array is checked on the device by the
 *     first kernel of the call.  A violation then cannot change the return
 *     code (the call has already returned KDA_OK): the kernel records
 *     KDA_ERR_INVALID_ARG in the device status word (kda_device_status) and
 *     empties the call's chunk table, so every later kernel of the call
 *     finds no chunk to process and touches no token of any segment: out
 *     and the per-token gradients are not written, while final_state,
 *     dinitial_state and the parameter gradients get what an all-empty
 *     problem gives (the entering state, the final-state gradient, zeros).
 *     Read the status word before using the results.
 *
 * Ownership: every pointer except cu_seqlens_host is a DEVICE pointer owned
 * by the caller (cu_seqlens too).  The library allocates no memory, keeps no pointer after a call
 * returns, and enqueues all work on `stream` asynchronously; outputs are
 * fully overwritten.  Scratch memory comes from the caller's `workspace`
 * (device, 256-byte aligned, at least the size the *_workspace_size query
 * returns).
 *
 * Errors: arguments are validated on the host before anything is enqueued;
 * a failed check returns KDA_ERR_INVALID_ARG (bad shape, pointer or value),
 * KDA_ERR_UNSUPPORTED (valid but not implemented) or KDA_ERR_WORKSPACE (too
 * small / misaligned).  A CUDA launch failure returns KDA_ERR_CUDA.  Nothing
 * aborts and no C++ exception crosses this boundary.  Device-side waits are
 * bounded; one that gives up records KDA_ERR_TIMEOUT in a device status word
 * read by kda_device_status().
 */
#ifndef KDA_GB300_H
#define KDA_GB300_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1,
    KDA_ERR_UNSUPPORTED = 2,
    KDA_ERR_CUDA = 3,
    KDA_ERR_TIMEOUT = 4,
    KDA_ERR_WORKSPACE = 5
} kda_status;

typedef enum { KDA_BF16 = 0, KDA_FP32 = 1 } kda_dtype;

/* Gate activation (the page's `safe_gate` switch).  KDA_GATE_LOWER_BOUNDED, the
 * default: g = lower_bound * sigmoid(exp(a_log) * (g_raw + dt_bias)), so g lies in
 * (lower_bound, 0).  KDA_GATE_SOFTPLUS: g = -exp(a_log) * softplus(g_raw + dt_bias),
 * unbounded below; lower_bound is still validated (< 0, finite) but not used. */
typedef enum { KDA_GATE_LOWER_BOUNDED = 0, KDA_GATE_SOFTPLUS = 1 } kda_gate;

/* Problem shape.  num_seqs is the number of packed segments N when
 * cu_seqlens is given (then B == 1) and is ignored otherwise (N = B).
 * H = value heads; Hk = key heads (q, k), H a multiple of Hk, 0 meaning Hk = H;
 * H % Hk != 0 or Hk < 0 is KDA_ERR_INVALID_ARG.  gate: zero-initialised means
 * the lower-bounded gate; a value outside kda_gate is KDA_ERR_INVALID_ARG. */
typedef struct {
    int B, T, H, K, V;
    kda_dtype dtype;
    int num_seqs;
    int Hk;
    kda_gate gate;
} kda_dims;

/* Bytes of workspace kda_fwd / kda_bwd need for this shape (0 on invalid input). */
size_t kda_fwd_workspace_size(const kda_dims* dims, int chunk_size);
size_t kda_bwd_workspace_size(const kda_dims* dims, int chunk_size);

/*
 * Forward.  Writes out [B,T,H,V] (input dtype) and, if final_state != NULL,
 * final_state [N,H,K,V] fp32.  initial_state may be NULL (zero state).
 * scale is applied to the output; lower_bound must be finite and < 0;
 * chunk_size must be 16, 32 or 64 (other positive values: KDA_ERR_UNSUPPORTED).
 * The result does not depend on the chunk size in exact arithmetic; every
 * accepted value runs the same 64-token blocking, so results agree to
 * rounding with any chunk size.
 * Requirements: B,T,H >= 1; 16 <= K,V <= 128 and multiples of 16 (the pages
 * reject head dims below 16); N >= 1.
 * Paths:
 *   - bf16 with K == V == 128 and 16-byte aligned q, k, v, g_raw, out,
 *     initial_state and final_state (and dout, dv, dfinal_state and
 *     dinitial_state for kda_bwd) runs on the tcgen05 tensor-core path.  Its 16-token
 *     sub-block factorisation of the decay stays inside fp32 range only for
 *     |lower_bound| <= 5.  With the lower-bounded gate that is required of
 *     both directions.
 *   - kda_fwd, kda_bwd and the training pair (kda_fwd_save / kda_bwd_saved)
 *     also take bf16 K == V == 64 heads under the lower-bounded gate on the
 *     tensor-core path (channels padded to 128 inside the kernels, so the saved
 *     record has the 128-channel size; the backward pads the states it reads
 *     and unpads dinitial_state in its workspace).  The segmented entries
 *     refuse them.
 *   - Under the unbounded gate both directions take the tensor-core path
 *     too: the diagonal sub-blocks, where the factorisation has no bound,
 *     are formed directly (in the forward's intra-chunk forms and in the
 *     backward's decayed bilinear forms).
 *   - Every other supported shape, and fp32 inputs, run on the fp32 SIMT
 *     path.  It forms every decay as exp(Gamma_t - Gamma_s) <= 1, which holds
 *     for any gate.
 */
kda_status kda_fwd(const kda_dims* dims,
                   const void* q, const void* k, const void* v, const void* g_raw, const void* beta_raw,
                   const float* a_log, const float* dt_bias, float scale, float lower_bound, int chunk_size,
                   const int32_t* cu_seqlens, const int32_t* cu_seqlens_host, const float* initial_state,
                   void* out, float* final_state,
                   void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Same as kda_fwd but always on the fp32 SIMT kernels (any supported shape). */
kda_status kda_fwd_simt(const kda_dims* dims,
                        const void* q, const void* k, const void* v, const void* g_raw, const void* beta_raw,
                        const float* a_log, const float* dt_bias, float scale, float lower_bound, int chunk_size,
                        const int32_t* cu_seqlens, const int32_t* cu_seqlens_host, const float* initial_state,
                        void* out, float* final_state,
                        void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Backward (recomputes the forward internally; nothing is saved between
 * calls; see kda_fwd_save / kda_bwd_saved for the pair that keeps it).  Inputs as for kda_fwd plus dout [B,T,H,V] (input dtype) and
 * dfinal_state [N,H,K,V] fp32 (may be NULL = zero).  Writes fp32 gradients
 * dq, dk, dg_raw [B,T,H,K], dv [B,T,H,V], dbeta_raw [B,T,H], da_log [H],
 * ddt_bias [H*K] and, if dinitial_state != NULL, dinitial_state [N,H,K,V].
 * The parameter gradients are reduced in a fixed order (deterministic).
 */
kda_status kda_bwd(const kda_dims* dims,
                   const void* q, const void* k, const void* v, const void* g_raw, const void* beta_raw,
                   const float* a_log, const float* dt_bias, float scale, float lower_bound, int chunk_size,
                   const int32_t* cu_seqlens, const int32_t* cu_seqlens_host, const float* initial_state,
                   const void* dout, const float* dfinal_state,
                   float* dq, float* dk, float* dv, float* dg_raw, float* dbeta_raw,
                   float* da_log, float* ddt_bias, float* dinitial_state,
                   void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Human-readable name of a status code (static string). */
/*
 * Training pair: a forward that keeps what the backward would otherwise
 * recompute.  A training step runs the forward and then the backward on the
 * same inputs; kda_bwd rebuilds the per-chunk intra quantities (the WY/UT
 * transform, gates, norms) that the forward already formed.  kda_fwd_save
 * runs the forward and also writes those quantities (fp32, per chunk and
 * head, an internal layout) to the caller's `saved` buffer; kda_bwd_saved
 * takes the same arguments as kda_bwd plus that buffer and skips the
 * rebuild.  The gradients are bit-identical to kda_bwd's.  The forward
 * output agrees with kda_fwd's to rounding, not bit for bit: kda_fwd alone
 * forms the intra-chunk decayed products with tf32 operands, the saving
 * pass with split-bf16 ones.
 *
 * kda_saved_size returns the bytes `saved` must hold for these dims (0 when
 * the shape does not take the tensor-core path; then use kda_fwd / kda_bwd).
 * `saved` is a device buffer owned by the caller, 256-byte aligned; its
 * contents are only valid for the inputs of the kda_fwd_save call that wrote
 * them (same q, k, v, g_raw, beta_raw, a_log, dt_bias, lower_bound,
 * cu_seqlens), until the caller reuses the buffer.  Both calls return
 * KDA_ERR_UNSUPPORTED when the tensor-core path does not apply (dtype, K, V,
 * the lower-bounded gate with lower_bound < -5, or unaligned activations) and KDA_ERR_WORKSPACE for a
 * missing, small or misaligned `saved`.  The workspace of kda_fwd_save is
 * kda_fwd_workspace_size's, of kda_bwd_saved kda_bwd_workspace_size's.
 */
size_t kda_saved_size(const kda_dims* dims, int chunk_size);
kda_status kda_fwd_save(const kda_dims* dims,
                        const void* q, const void* k, const void* v, const void* g_raw, const void* beta_raw,
                        const float* a_log, const float* dt_bias, float scale, float lower_bound, int chunk_size,
                        const int32_t* cu_seqlens, const int32_t* cu_seqlens_host, const float* initial_state,
                        void* out, float* final_state, void* saved, size_t saved_bytes,
                        void* workspace, size_t workspace_bytes, cudaStream_t stream);
kda_status kda_bwd_saved(const kda_dims* dims,
                         const void* q, const void* k, const void* v, const void* g_raw, const void* beta_raw,
                         const float* a_log, const float* dt_bias, float scale, float lower_bound, int chunk_size,
                         const int32_t* cu_seqlens, const int32_t* cu_seqlens_host, const float* initial_state,
                         const void* dout, const float* dfinal_state,
                         float* dq, float* dk, float* dv, float* dg_raw, float* dbeta_raw,
                         float* da_log, float* ddt_bias, float* dinitial_state,
                         const void* saved, size_t saved_bytes,
                         void* workspace, size_t workspace_bytes, cudaStream_t stream);

const char* kda_status_string(kda_status s);

/* Device status word of the current device: KDA_OK, or the first error a
 * kernel recorded (e.g. KDA_ERR_TIMEOUT from a bounded wait).  Synchronises
 * the device.  reset != 0 clears the word afterwards. */
kda_status kda_device_status(int reset);

/*
 * Forward without a caller-provided workspace (no counterpart on the pages: an
 * integration aid).  Some callers cannot allocate device memory: plugin
 * hosts that own every device allocation and give their plugins no
 * allocator, and latency-critical loops that must not call cudaMalloc
 * because it can synchronise the device.  kda_fwd_noalloc takes the same
 * arguments as kda_fwd minus the workspace and uses a scratch array built
 * into this library instead: KDA_NOALLOC_SCRATCH_BYTES (32 MiB) of device
 * memory, held by every GPU that loads the library until the process exits.
 * It allocates nothing (no cudaMalloc / cudaFree, no allocating library
 * call).  Shapes whose workspace (kda_fwd_workspace_size) exceeds that size
 * return KDA_ERR_WORKSPACE.  The first call on a device looks up the
 * array's device address (cudaGetSymbolAddress) with that device current;
 * make that first call before any stream capture.  The address is kept for
 * the life of the process: after cudaDeviceReset on a device the kept
 * address no longer names the array in the new context, so do not call this
 * entry on a device that has been reset.  All calls share the one
 * array: calls that overlap on the GPU (different streams, or several host
 * threads) race and must be serialised by the caller.  No scratch content
 * needs to start at zero (every call rewrites what it reads).
 */
#define KDA_NOALLOC_SCRATCH_BYTES (32u << 20)
kda_status kda_fwd_noalloc(const kda_dims* dims,
                           const void* q, const void* k, const void* v, const void* g_raw, const void* beta_raw,
                           const float* a_log, const float* dt_bias, float scale, float lower_bound, int chunk_size,
                           const int32_t* cu_seqlens, const int32_t* cu_seqlens_host, const float* initial_state,
                           void* out, float* final_state, cudaStream_t stream);

/*
 * Segment-parallel forward for long rows with few rows x heads.  The chunk
 * chain of kda_fwd is serial per (row, head).  When B * H is small it keeps
 * only a few SMs busy however long T is.  This entry cuts every row into
 * pieces of whole chunks and works like the state-CP executor of
 * hyper-parallel "KDA context-parallel executors" (`_eager_kda_state_p2p`),
 * with pieces in place of ranks, on one GPU:
 *   1. for every piece in parallel, a summary of its chunks: the end state from
 *      zero S_loc and the transition M (the K x K product of the per-chunk
 *      maps S -> Diag(exp(Gamma_last)) S - Kd^T W S);
 *   2. the entering states, piece after piece along each row:
 *      S_{k+1} = M_k S_k + S_loc,k, from the row's initial_state (or zero);
 *      the last one is the row's final_state;
 *   3. the output of every piece from its entering state, in parallel.
 * Same arguments and results as kda_fwd plus `segments`.  A row is one of
 * the B rows of T tokens, or with cu_seqlens one packed document (the
 * documents of nemo_automodel `kimi_k3.cp`, `segment_cu_seqlens`, each
 * starting from its own initial state); cu_seqlens and cu_seqlens_host as
 * for kda_fwd.  Pieces are L = ceil(ceil(span / 64) / segments) chunks of 64
 * tokens long, span = T for rows and the total token count for documents;
 * a row of len tokens gets ceil(len / L) pieces, its last one shorter.  It
 * takes only shapes of the tensor-core forward: bf16, K = V = 128, 16-byte
 * aligned activations, the softplus gate or lower_bound >= -5; others are
 * KDA_ERR_UNSUPPORTED.  segments >= 1, else KDA_ERR_INVALID_ARG.  The
 * intra-chunk pass runs once and the chain three times, each over all
 * pieces at once.  In exact arithmetic the result equals kda_fwd's; in
 * floating point it agrees to rounding.  The workspace is
 * kda_fwd_segmented_workspace_size() bytes (0 for invalid or unsupported
 * shapes); it adds three fp32 states per piece and head to the forward's.
 * A device-only cu_seqlens with bad contents is reported, as for kda_fwd,
 * through kda_device_status, and no piece is run.
 */
size_t kda_fwd_segmented_workspace_size(const kda_dims* dims, int chunk_size, int segments);
kda_status kda_fwd_segmented(const kda_dims* dims,
                             const void* q, const void* k, const void* v, const void* g_raw, const void* beta_raw,
                             const float* a_log, const float* dt_bias, float scale, float lower_bound,
                             int chunk_size, int segments, const int32_t* cu_seqlens,
                             const int32_t* cu_seqlens_host, const float* initial_state,
                             void* out, float* final_state,
                             void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Segment-parallel backward: kda_bwd with both state chains of the
 * backward cut into the pieces of kda_fwd_segmented.  The forward state
 * recompute runs steps 1-3 above (end states from zero and transitions per
 * piece, entering states along each row, then every piece from its entering
 * state).  The reverse chain is affine in the same way, from the end of a
 * piece to its start: dS_begin = M'_k dS_end + dS_loc,k, with M'_k the
 * piece's K x K transition of dS and dS_loc,k its start value from a zero
 * end value.  Its pieces' end values follow along each row from the last
 * piece, dS_end of the last piece = dfinal_state (or zero), dS_end,k-1 =
 * M'_k dS_end,k + dS_loc,k; the first piece's dS_begin is the row's
 * dinitial_state.  This is the gradient the state-CP executor of
 * hyper-parallel "KDA context-parallel executors" (`_eager_kda_state_p2p`)
 * sends back from rank to rank.  Both chains run in the split bf16
 * precision of kda_bwd's tensor-core chains, the combines in fp32.  Same
 * arguments and results as kda_bwd plus `segments`; the same shapes as
 * kda_fwd_segmented, else KDA_ERR_UNSUPPORTED.  The gradients agree with
 * kda_bwd's to rounding.  The workspace is
 * kda_bwd_segmented_workspace_size() bytes (0 for invalid or unsupported
 * shapes).
 */
size_t kda_bwd_segmented_workspace_size(const kda_dims* dims, int chunk_size, int segments);
kda_status kda_bwd_segmented(const kda_dims* dims,
                             const void* q, const void* k, const void* v, const void* g_raw, const void* beta_raw,
                             const float* a_log, const float* dt_bias, float scale, float lower_bound,
                             int chunk_size, int segments, const int32_t* cu_seqlens,
                             const int32_t* cu_seqlens_host, const float* initial_state,
                             const void* dout, const float* dfinal_state,
                             float* dq, float* dk, float* dv, float* dg_raw, float* dbeta_raw,
                             float* da_log, float* ddt_bias, float* dinitial_state,
                             void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * The layer's output epilogue: a gated RMS norm of each head's value vector.
 * hyper-parallel "KDA context-parallel executors" applies
 * `o_norm(output, output_gate)` between the attention core and the output
 * projection.  The torchtitan review describes the model's RMS norm as one
 * reduced in fp32.  Neither prints the formula.  This library's reading, per
 * row of V values (one token of one head, rows = B * T * H):
 *     y_v = o_v / sqrt(mean_u o_u^2 + eps) * weight_v * sigmoid(gate_v)
 * Layouts (every activation in the one `dtype`; the kernels read each of
 * them with that element size, so a buffer of another type is misread):
 *   o, gate, y, dy   [rows, V] in `dtype` (bf16 or fp32);
 *   weight [V] fp32 (also when dtype is bf16), dweight [V], do, dgate [rows, V]   fp32.
 * The sum of squares and every gradient are computed in fp32.  dweight sums
 * over all rows in a fixed order, so results are deterministic.
 * Errors:
 *   - KDA_ERR_INVALID_ARG: rows < 1, V < 1, a bad dtype, a NULL pointer, or
 *     eps <= 0 or not finite (eps = 0 would turn an all-zero row into NaN);
 *   - KDA_ERR_UNSUPPORTED: V > 256;
 *   - KDA_ERR_WORKSPACE: the backward's workspace is too small or not
 *     256-byte aligned; it needs kda_gated_norm_bwd_workspace_size() bytes.
 * Every pointer is a device pointer the caller owns; nothing is kept after the
 * call, and the work is enqueued on `stream`.
 */
kda_status kda_gated_norm_fwd(int64_t rows, int V, kda_dtype dtype, const void* o, const void* gate,
                              const float* weight, float eps, void* y, cudaStream_t stream);
size_t kda_gated_norm_bwd_workspace_size(int64_t rows, int V);
kda_status kda_gated_norm_bwd(int64_t rows, int V, kda_dtype dtype, const void* o, const void* gate,
                              const float* weight, float eps, const void* dy, float* d_o, float* dgate,
                              float* dweight, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Failure-detection self-test.  Every device-side wait in this library is
 * bounded; a wait that gives up records KDA_ERR_TIMEOUT in the device status
 * word (kda_device_status) and its kernel returns, so the context stays
 * usable.  This call launches one CTA whose mbarrier wait can never complete
 * (nothing arrives on it).  The same bounded wait gives up after 256 polls,
 * milliseconds at most, and records KDA_ERR_TIMEOUT.  It neither hangs nor
 * faults.  Returns KDA_OK once launched on `stream`; read the word with
 * kda_device_status afterwards.
 */
kda_status kda_selftest_wait_timeout(cudaStream_t stream);

/* Library version, major * 10000 + minor * 100 + patch. */
int kda_version(void);

/*
 * Kernel timing for benchmarks.  After kda_timing_begin(max_launches), the
 * library records one CUDA event before and one after each kernel it
 * launches (on that launch's stream), for at most max_launches launches.
 * kda_timing_end() waits for those events, writes each launch's duration in
 * milliseconds and its kernel id (name: kda_kernel_name) into the caller's
 * host arrays (capacity `cap`), releases the events and returns how many
 * launches were recorded, or -1 on a CUDA error.  Process-wide; not meant
 * for concurrent use from several host threads.  Returns KDA_ERR_CUDA if the
 * events cannot be created.
 */
kda_status kda_timing_begin(int max_launches);
int kda_timing_end(float* ms, int* kernel_ids, int cap);
const char* kda_kernel_name(int kernel_id);

/*
 * The layer's q/k/v prologue: causal depthwise short convolution + SiLU
 * (hyper-parallel "KDA context-parallel executors", `_run_causal_short_conv`,
 * `_local_short_conv`, `_validate_layer_short_conv`: a depthwise Conv1d with
 * groups = channels, stride 1, dilation 1, kernel_size - 1 zero padding on the
 * left, output cut to the input length, then SiLU):
 *     a[t, c] = bias[c] + sum_{i < W} weight[c, i] * x[t - (W - 1) + i, c]
 *     y[t, c] = a * sigmoid(a)
 * Token-first layout: x, y, dy [B, T, C] in `dtype` (C = heads * head dim of
 * one projection); weight [C, W] fp32 (a Conv1d weight [C, 1, W]); bias [C]
 * fp32 or NULL.  With cu_seqlens (device, [num_seqs + 1], B == 1) every
 * segment starts from zero history, as in kda_fwd.  All pointers are device
 * pointers owned by the caller; nothing is allocated or retained.
 * Errors: B, T, C, W < 1, a bad dtype, NULL x / weight / y (dy, dx, dweight,
 * and dbias when bias != NULL) or cu_seqlens with B != 1 give
 * KDA_ERR_INVALID_ARG; W > 8, C not a multiple of 8 or a data pointer not
 * 16-byte aligned give KDA_ERR_UNSUPPORTED; a short or misaligned workspace
 * gives KDA_ERR_WORKSPACE.
 */
kda_status kda_short_conv_fwd(int B, int T, int C, int W, kda_dtype dtype, const void* x, const float* weight,
                              const float* bias, const int32_t* cu_seqlens, int num_seqs, void* y,
                              cudaStream_t stream);

/* Bytes of workspace kda_short_conv_bwd needs (per-tile partial sums of the weight / bias gradients). */
size_t kda_short_conv_bwd_workspace_size(int B, int T, int C, int W);

/* Reverse mode: dx [B, T, C] fp32, dweight [C, W] fp32, dbias [C] fp32 (written when bias != NULL).
 * dweight and dbias are summed over tokens in a fixed order (deterministic). */
kda_status kda_short_conv_bwd(int B, int T, int C, int W, kda_dtype dtype, const void* x, const float* weight,
                              const float* bias, const int32_t* cu_seqlens, int num_seqs, const void* dy,
                              float* dx, float* dweight, float* dbias, void* workspace, size_t workspace_bytes,
                              cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_GB300_H */
