/*
 * moe.h — C ABI of a single-GPU dropless token-choice MoE layer (forward and
 * backward) for NVIDIA GB300 (sm_103a).
 *
 * What the calls compute (sources: page title, section):
 *   moe_route           logits z = x W_g^T (+ bias), p = softmax(z), the K largest
 *                       experts per token, weights renormalised over the chosen K.
 *                       [MoEBlaze paper notes 2.1 "gating network"; Dropless MoE,
 *                       in depth, "A reference implementation"]
 *   moe_build_dispatch  expert_token_indices, expert_token_offsets and
 *                       token_index_map of the routing, built without a global
 *                       sort and without contended atomics.
 *                       [MoEBlaze paper notes 4.1 data structures, 4.2 build]
 *   moe_forward         per expert: a = x W1^T, b = x W3^T, A = SiLU(a) * b,
 *                       Y = A W2^T, read through expert_token_indices (no routed
 *                       copy of x); y_t = sum_k w_{t,k} Y_{t,k}.
 *                       [MoEBlaze paper notes 2.3, 5.1, Algorithm 1; SonicMoE 3.4.1]
 *                       Non-gated experts (moe_shape.expert = SiLU or ReLU):
 *                       A = act(a), no W3. [MoEBlaze paper notes 2.2, the
 *                       two-layer expert E_i(x) = W_2,i s(W_1,i x)]
 *   moe_backward        dx, dW_g, dW1, dW3, dW2 and the router-score gradient
 *                       dS_{t,k} = <dO_t, Y_{t,k}> (computed as <dO W2, A>).
 *                       [MoEBlaze paper notes 3.2, Algorithm 1; SonicMoE 3.4.1]
 *
 * Conventions for every call
 *   - Shapes: T tokens, d model width, E experts, K experts per token, h expert
 *     hidden width. TK = T*K.
 *   - All pointers are DEVICE pointers (cudaMalloc or equivalent), except where
 *     a comment says otherwise. bf16 arrays are passed as void* and hold IEEE
 *     bfloat16 values. All arrays are dense, row-major, 16-byte aligned.
 *   - x, dy, y, dx: [T, d] bf16. W_g, dW_g: [E, d] fp32. bias: [E] fp32.
 *     W1, W3, dW1, dW3: [E, h, d] bf16. W2, dW2: [E, d, h] bf16 (out x in).
 *     topk_ids: [T, K] int32, slot 0 = largest weight. topk_w, dS: [T, K] fp32.
 *     expert_token_indices, token_index_map: [TK] int32. offsets: [E+1] int32.
 *     H_saved: [TK, hs] bf16 with hs = 2h for SwiGLU experts (row r = (a | b) of
 *     the r-th expert-sorted row) and hs = h for non-gated experts (row r = a).
 *     Non-gated experts have no W3: W3 and dW3 are ignored and may be NULL.
 *   - Ownership: the caller allocates and owns every buffer and the workspace.
 *     The library allocates no device memory and keeps no state between calls
 *     other than the optional kernel timer below.
 *   - Execution: every call enqueues kernels on `stream` (a cudaStream_t; NULL
 *     means the legacy default stream) and returns without waiting. Per-expert
 *     counts never leave the device. Workspace contents need not survive
 *     between calls. Some kernels are launched with programmatic stream
 *     serialization (the grouped GEMMs by default; MOE_PDL=1|0|small|gemm
 *     chooses): such a kernel may be scheduled early but waits for the work
 *     before it on the stream to complete before it reads or writes memory, so
 *     stream order holds as for ordinary launches.
 *   - Errors: a call returns MOE_OK or a status code. Arguments that the host
 *     can check (null pointers, unsupported shapes, misalignment, workspace too
 *     small) are rejected before anything is launched. Errors that only the
 *     device can see (an expert id out of range or repeated within a token, a
 *     bounded wait that ran out) set a sticky device status word; kernels that
 *     start after it is set do nothing, and moe_get_error() reports it.
 *     No call traps or aborts the process.
 *   - Supported shapes: 1 <= T <= 2^24, 1 <= K <= 8, K <= E <= 256, TK < 2^31,
 *     d and h multiples of 128 (h a multiple of 256 for non-gated experts),
 *     d, h <= 32768. Buffers may exceed 2^31 elements (64-bit addressing).
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Expert function (moe_shape.expert). A zero-initialised shape is SwiGLU. */
enum moe_expert_kind {
    MOE_EXPERT_SWIGLU = 0, /* A = SiLU(x W1^T) * (x W3^T)          */
    MOE_EXPERT_SILU = 1,   /* A = SiLU(x W1^T), no W3               */
    MOE_EXPERT_RELU = 2    /* A = max(x W1^T, 0), no W3; ReLU'(0) = 0 */
};

typedef struct {
    int32_t T, d, E, K, h;
    int32_t expert; /* enum moe_expert_kind */
} moe_shape;

enum moe_status_code {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,         /* null pointer or negative size            */
    MOE_ERR_UNSUPPORTED_SHAPE = 2,   /* outside the supported shapes above       */
    MOE_ERR_WORKSPACE_TOO_SMALL = 3, /* ws_bytes < moe_workspace_size(...)       */
    MOE_ERR_CUDA = 4,                /* a CUDA runtime call failed               */
    MOE_ERR_BAD_EXPERT_ID = 5,       /* device: id out of [0,E) or repeated      */
    MOE_ERR_TIMEOUT = 6,             /* device: a bounded wait ran out           */
    MOE_ERR_MISALIGNED = 7,          /* a pointer is not 16-byte aligned         */
    MOE_ERR_NO_DEVICE = 8,           /* no usable sm_100-family device           */
    MOE_ERR_STATIC_SCRATCH_LIMIT = 9 /* shape needs more than the static scratch */
};

enum moe_workspace_kind {
    MOE_WS_ROUTE = 0,
    MOE_WS_DISPATCH = 1,
    MOE_WS_FORWARD = 2,
    MOE_WS_BACKWARD = 3,
    MOE_WS_FORWARD_SLOTWISE = 4
};

/* Bytes of device workspace that the call `which` needs for shape s (0 if the
 * shape is unsupported). Pure host function. */
size_t moe_workspace_size(moe_shape s, int which);

/* Transient-buffer bound: moe_forward runs the down projection and the
 * weighted combine (and moe_backward the dX of the up projection and the
 * token-gradient sum) in passes once T >= 1024, so the expert-output buffer
 * holds at most about a quarter of T*K*d elements, or half of them when that
 * half buffer is at most 64 MiB (small layers); never the whole routed T*K*d
 * buffer. A pass covers either a chunk of tokens (two or four chunks by that
 * rule) or, when d is a multiple of 512, a slice of the output columns (half
 * or a quarter of them by the same rule; the environment variable
 * MOE_COLUMN_PASSES=2|4 forces the column-pass count).
 * The library takes the split that re-reads fewer bytes (token chunks
 * re-read the expert weights once per pass, column chunks re-read the
 * activation operand). This function returns the tokens per token chunk.
 * Pure host function. */
int moe_chunk_tokens(moe_shape s);

/* Router. x [T,d] bf16, Wg [E,d] fp32, bias [E] fp32 or NULL.
 * Outputs: logits [T,E] fp32 (NULL to skip), topk_ids [T,K] int32 (descending
 * weight, ties to the lower id), topk_w [T,K] fp32 (sum to 1 per token).
 * Selection is on the fp32 logits z + bias; weights are exp(z_k - z_max)
 * normalised over the chosen K (equal to the renormalised softmax).
 * Workspace: moe_workspace_size(s, MOE_WS_ROUTE) bytes. For E <= 128 the
 * logits are computed on the tensor cores from three bf16 parts of W_g
 * (W_g = W0 + W1 + W2 to fp32 precision, each product with the bf16 x exact in
 * fp32, fp32 accumulation), which the call writes into the workspace
 * (3 * max(16, E rounded up to a power of two) rows of d bf16 values); a
 * workspace that is NULL or smaller returns MOE_ERR_INVALID_ARG or
 * MOE_ERR_WORKSPACE_TOO_SMALL. For E > 128 the logits are fp32 FFMA sums and
 * no workspace is needed (ws may be NULL). */
int moe_route(moe_shape s, const void* x, const float* Wg, const float* bias,
              float* logits, int32_t* topk_ids, float* topk_w,
              void* ws, size_t ws_bytes, void* stream);

/* Dispatch index from topk_ids [T,K] int32.
 * Outputs: expert_token_indices [TK] (token ids grouped by expert, ascending
 * token inside an expert), expert_token_offsets [E+1] (exclusive prefix of the
 * per-expert counts, offsets[E] = TK), token_index_map [TK] (position of
 * assignment (t,k) in expert_token_indices, at index t*K+k).
 * Bit-exact with a stable sort of the flattened ids by expert. Invalid ids set
 * MOE_ERR_BAD_EXPERT_ID on the device; the outputs are then undefined. */
int moe_build_dispatch(moe_shape s, const int32_t* topk_ids,
                       int32_t* expert_token_indices, int32_t* expert_token_offsets,
                       int32_t* token_index_map, void* ws, size_t ws_bytes, void* stream);

/* Allocation-free variant of moe_build_dispatch (the pages have no
 * counterpart; it exists for callers that cannot allocate device memory).
 *
 * Some callers cannot call cudaMalloc or hand over a workspace at this point:
 * an inference runtime or plugin host that owns every byte of device memory
 * and forbids allocation after start-up, or a latency-critical loop where an
 * allocation (which may synchronise the device) is not acceptable. This entry
 * point takes no workspace: its per-block histogram lives in a file-scope
 * device array of MOE_NOALLOC_DISPATCH_MAX_ENTRIES int32 values (4 MiB),
 * which every GPU that loads the library holds until the process exits.
 * It computes exactly what moe_build_dispatch computes, with the same inputs,
 * outputs and device-side errors.
 *   - Limit: ceil(T / 256) * E <= MOE_NOALLOC_DISPATCH_MAX_ENTRIES (for
 *     example T <= 1,048,576 tokens at E = 256); larger shapes return
 *     MOE_ERR_STATIC_SCRATCH_LIMIT and launch nothing.
 *   - The first call on a device looks up the array's device address with
 *     that device current (cudaGetSymbolAddress); make that first call
 *     before any stream capture. Under CUDA's lazy module loading (the
 *     default), that first call may also be what loads the library's device
 *     code and the array onto the device, so device memory can drop by about
 *     4 MiB at that moment (a one-time load by the driver, not an allocation
 *     by this call). Later calls do no set-up and change no device memory.
 *   - Host checks and status codes are those of moe_build_dispatch, in the
 *     same order; a failed launch returns MOE_ERR_CUDA and leaves its message
 *     for moe_last_cuda_error().
 *   - All calls on a device share the one array, and it keeps the last
 *     call's contents. Every entry a call reads is first written by the same
 *     call, so nothing needs clearing, but calls whose kernels overlap on the
 *     GPU (different streams, no ordering between them) race on the array and
 *     give wrong results. Order such calls on one stream or with events.
 * Allocates nothing: no cudaMalloc, cudaFree or allocating library call. */
#define MOE_NOALLOC_DISPATCH_MAX_ENTRIES (1 << 20)
int moe_build_dispatch_noalloc(moe_shape s, const int32_t* topk_ids,
                               int32_t* expert_token_indices, int32_t* expert_token_offsets,
                               int32_t* token_index_map, void* stream);

/* Forward. Inputs: x, W1, W3 (NULL allowed for non-gated experts), W2, the
 * routing (topk_ids, topk_w) and its dispatch index. Outputs: y [T,d] bf16
 * and H_saved [TK,hs] bf16 (the pre-activations kept for the backward; the
 * activation is recomputed there).
 * No [TK,d] copy of the routed tokens is made: expert rows are gathered from x
 * through expert_token_indices by the GEMM's loads. */
int moe_forward(moe_shape s, const void* x, const void* W1, const void* W3, const void* W2,
                const int32_t* topk_ids, const float* topk_w,
                const int32_t* expert_token_indices, const int32_t* expert_token_offsets,
                const int32_t* token_index_map,
                void* y, void* H_saved, void* ws, size_t ws_bytes, void* stream);

/* Forward with the weighted combine fused into the down projection (same
 * arguments and outputs as moe_forward; workspace MOE_WS_FORWARD_SLOTWISE).
 * The down projection runs once per routing slot k = 0..K-1 over the rows
 * (t, k) of that slot, grouped by expert; its epilogue adds w_{t,k} Y_{t,k}
 * into an fp32 accumulator row of token t (each token appears once per slot,
 * so no atomics and a fixed order), and the last slot writes bf16 y. No
 * expert-output buffer exists; the accumulator holds T*d fp32 values (K >= 2)
 * and is read and written once per slot, K*T*d*8 bytes in total, against the
 * 4*T*K*d bytes of the chunked combine. y is not rounded to bf16 between the
 * expert output and the sum (moe_forward rounds each Y row once).
 * [SonicMoE 3.4.1, O_t = sum_k s_{t,k} Y_{t,k}; MoEBlaze paper notes 5.2] */
int moe_forward_slotwise(moe_shape s, const void* x, const void* W1, const void* W3,
                         const void* W2, const int32_t* topk_ids, const float* topk_w,
                         const int32_t* expert_token_indices,
                         const int32_t* expert_token_offsets, const int32_t* token_index_map,
                         void* y, void* H_saved, void* ws, size_t ws_bytes, void* stream);

/* Backward with upstream gradient dy [T,d] bf16. Outputs: dx [T,d] bf16
 * (expert and router paths), dWg [E,d] fp32, dW1, dW3 [E,h,d] bf16 (dW3 is
 * not written, and W3 not read, for non-gated experts),
 * dW2 [E,d,h] bf16 (an expert with no tokens gets exact zeros) and
 * dS [T,K] fp32 = <dy_t, Y_{t,k}>. Gradients are written, not accumulated. */
int moe_backward(moe_shape s, const void* dy, const void* x, const float* Wg,
                 const void* W1, const void* W3, const void* W2,
                 const int32_t* topk_ids, const float* topk_w,
                 const int32_t* expert_token_indices, const int32_t* expert_token_offsets,
                 const int32_t* token_index_map, const void* H_saved,
                 void* dx, float* dWg, void* dW1, void* dW3, void* dW2, float* dS,
                 void* ws, size_t ws_bytes, void* stream);

/* ---- Token rounding and routings given as rows ----------------------------
 *
 * Token rounding (TR) replaces each expert's token-choice count f_e by the
 * nearest multiple of m_tile (a tie rounds down; at most T), so that no
 * grouped-GEMM tile is padded. Rounding down drops the expert's lowest-scoring
 * token-choice tokens; rounding up adds the best other tokens. The score of
 * (t, e) is the router probability (softmax of z_t over all experts); ties rank
 * the lower token first. [SonicMoE 3.4.4, Algorithm 4, NR-f subroutine]
 * A token can end with fewer or more than K experts; its gate weights are the
 * softmax of z_t over its final experts (renormalised over the chosen experts
 * as for top-K), and a token without experts gets y = 0 and no gradient.
 *
 * The result is a routing given as rows, consumed by moe_forward_rows and
 * moe_backward_rows:
 *   expert_token_indices [rows_cap] (first offsets[E] used; each expert's
 *     tokens ascending), expert_token_offsets [E+1],
 *   w_row [rows_cap] fp32: gate weight of each row,
 *   tok_off [T+1]: token t's entries are tok_off[t] .. tok_off[t+1] of
 *   tok_exp [rows_cap] (its experts, ascending) and tok_rows [rows_cap] (the
 *     row of each of those experts).
 * rows_cap = moe_rows_capacity(s, m_tile) bounds the rows (T*K plus fewer than
 * m_tile added tokens per expert, and at most T*E). */

/* Row capacity for token rounding with tile m_tile (0 if unsupported). */
size_t moe_rows_capacity(moe_shape s, int m_tile);

/* Workspace bytes of moe_token_rounding (0 if unsupported). */
size_t moe_token_rounding_workspace_size(moe_shape s, int m_tile);

/* Token rounding of a token-choice routing. Inputs: logits [T,E] fp32 (from
 * moe_route), topk_ids [T,K], and expert_token_indices / offsets of their
 * dispatch (moe_build_dispatch). Outputs as described above. m_tile in
 * [1, 4096]. Every output is a deterministic function of the inputs. */
int moe_token_rounding(moe_shape s, int m_tile, const float* logits, const int32_t* topk_ids,
                       const int32_t* tc_expert_token_indices,
                       const int32_t* tc_expert_token_offsets,
                       int32_t* expert_token_indices, int32_t* expert_token_offsets,
                       float* w_row, int32_t* tok_off, int32_t* tok_exp, int32_t* tok_rows,
                       void* ws, size_t ws_bytes, void* stream);

/* Workspace bytes of moe_forward_rows (which = MOE_WS_FORWARD) and
 * moe_backward_rows (MOE_WS_BACKWARD) for row capacity rows_cap. */
size_t moe_workspace_size_rows(moe_shape s, int32_t rows_cap, int which);

/* Forward on a routing given as rows (same computation as moe_forward; the
 * K slots of a token become its tok_off range). H_saved is [rows_cap, hs].
 * Down-projection passes split columns (d % 512 == 0) or run once over all
 * rows. */
int moe_forward_rows(moe_shape s, int32_t rows_cap, const void* x, const void* W1,
                     const void* W3, const void* W2, const int32_t* expert_token_indices,
                     const int32_t* expert_token_offsets, const float* w_row,
                     const int32_t* tok_off, const int32_t* tok_exp, const int32_t* tok_rows,
                     void* y, void* H_saved, void* ws, size_t ws_bytes, void* stream);

/* Backward on a routing given as rows. dS_row [rows_cap] fp32 = <dy_t, Y_r> per
 * row; the router gradient is that of w_row = softmax of z_t over the token's
 * rows: dz_r = w_r (dS_r - sum over the token's rows of w dS). */
int moe_backward_rows(moe_shape s, int32_t rows_cap, const void* dy, const void* x,
                      const float* Wg, const void* W1, const void* W3, const void* W2,
                      const int32_t* expert_token_indices, const int32_t* expert_token_offsets,
                      const float* w_row, const int32_t* tok_off, const int32_t* tok_exp,
                      const int32_t* tok_rows, const void* H_saved, void* dx, float* dWg,
                      void* dW1, void* dW3, void* dW2, float* dS_row, void* ws, size_t ws_bytes,
                      void* stream);

/* Self-test of the device failure path (no counterpart in the pages; a test
 * hook). Enqueues one CTA on `stream` that waits on a shared-memory barrier
 * that nothing ever arrives at, through the same time-bounded wait as every
 * pipelined kernel of the library; after limit_ns (1 ns .. 10 s) the wait gives
 * up and the kernel sets MOE_ERR_TIMEOUT in the device status word, then
 * returns, leaving the context usable. moe_get_error() then reports and clears
 * it. Returns MOE_ERR_INVALID_ARG for a limit out of range, else MOE_OK or
 * MOE_ERR_CUDA (launch failure). Does nothing if the status word is already
 * set. */
int moe_selftest_bounded_wait(uint64_t limit_ns, void* stream);

/* Waits for `stream`, then returns and clears the device status word of the
 * current device (MOE_OK if no device-side error happened since the last
 * call). The only call that blocks the host. */
int moe_get_error(void* stream);

/* Human-readable name of a status code (static string). */
const char* moe_status_string(int status);

/* After a call returned MOE_ERR_CUDA: "<kernel>: <CUDA error string>" of that
 * failure on the calling thread (empty if none). The pending launch error has
 * already been cleared, so later calls are not affected by it. */
const char* moe_last_cuda_error(void);

/* ---- Instrumentation (host-side; off by default) ------------------------ */

/* Number of kernels this library has launched in this process. */
long long moe_launch_count(void);

/* When on, every kernel launch is bracketed by two CUDA events on its stream
 * (recorded, not waited on). Turning it on clears earlier records. */
int moe_timing_enable(int on);

typedef struct {
    char name[32];
    int32_t launches;
    double total_ms;
} moe_kernel_time;

/* Waits for the recorded events and fills up to `max` entries (one per
 * kernel name, in first-launch order). Returns the number of names, or a
 * negative status. */
int moe_timing_collect(moe_kernel_time* out, int max);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
