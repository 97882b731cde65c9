// common.cuh — shared internals of the MoE library: device status word,
// launch bookkeeping, tensor-map encoding and the kernel launchers' signatures.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/moe.h"

namespace moe {

// ---- programmatic dependent launch
// Kernels of the layer can be launched with programmatic stream serialization
// (launch_k below and the GEMM and router launchers), so a kernel may be
// scheduled while the previous kernel on the stream still runs. Each such kernel first waits until its predecessor
// has completed and its memory is visible (pdl_wait), before it touches global
// memory, and then lets its own successor be scheduled (pdl_trigger). Waiting
// before triggering keeps the order transitive: when a kernel starts, the
// kernel two launches back has completed. Only launch latency and CTA
// scheduling overlap; no kernel reads or writes early.
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// By default only the grouped GEMMs are launched this way: measured on GB300
// (three runs each), that saved 1% of the step on the Mixtral-shaped and the
// skewed layers, while launching the small kernels this way as well cost the
// skewed layer (35 launches per step) 0.6%. MOE_PDL=1 launches every kernel of
// the layer this way, MOE_PDL=0 none, MOE_PDL=small the small kernels only
// (read at every call). gemm_launch tells which kind of launch asks.
inline bool pdl_enabled(bool gemm_launch = false) {
    const char* f = std::getenv("MOE_PDL");
    if (f == nullptr || std::strcmp(f, "gemm") == 0) return gemm_launch;
    if (std::strcmp(f, "0") == 0) return false;
    if (std::strcmp(f, "small") == 0) return !gemm_launch;
    return true;
}
// kernel<<<grid, block, smem, st>>>(args...), with programmatic stream
// serialization where pdl_enabled() says so; the kernel calls pdl_wait() before
// it touches global memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                     Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Device status word layout: the first error code that was raised wins.
__device__ __forceinline__ void raise_error(int* err, int code) {
    atomicCAS(err, 0, code);
}
__device__ __forceinline__ bool has_error(const int* err) {
    return *reinterpret_cast<const volatile int*>(err) != 0;
}

// Per-row segment of one expert inside the expert-sorted row space:
// rows [lo, hi) of A's row space; `out` is the output row of `lo` (used by the
// chunked down projection; equal to lo otherwise).
struct Seg {
    int lo, hi, out, pad;
};

// Launch bookkeeping: counts launches and (optionally) brackets them with
// events. Implemented in api.cu.
struct LaunchScope {
    LaunchScope(const char* name, cudaStream_t st);
    ~LaunchScope();
    const char* name_;
    cudaStream_t st_;
    int slot_;
};

// Tensor map of a 2D row-major bf16 array [rows, cols] with a box of
// box_cols x box_rows and a swizzle of `swizzle` bytes (128, 64, or 0 for
// none). Returns false on failure.
bool make_tmap_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                    uint32_t box_cols, uint32_t box_rows, int swizzle = 128);
// Same for a row-major fp32 array, without swizzle.
bool make_tmap_f32(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                   uint32_t box_cols, uint32_t box_rows);

int num_sms();

// Host checks shared by the entry points (api.cu): the status of a shape
// against the supported shapes (MOE_OK, MOE_ERR_INVALID_ARG or
// MOE_ERR_UNSUPPORTED_SHAPE), and the MOE_ERR_CUDA return of a failed CUDA
// call, which records "<launch>: <error>" for moe_last_cuda_error() and clears
// the pending launch error.
int check_shape_status(const moe_shape& s);
int cuda_error_status(cudaError_t e);

// Address of the current device's status word (nullptr without a device).
int* device_status_word();

// ---------------------------------------------------------------- launchers
// Every launcher enqueues on `st` and returns a cudaError_t of the launch.

// router.cu
// Whether the router logits run on the tensor cores (E <= 128; three bf16 parts
// of W_g in the route workspace) or as fp32 FFMA (E > 128). MOE_ROUTER=ffma|mma
// forces one (mma only where E <= 128); read at every call.
inline bool router_tensor_cores(const moe_shape& s) {
    const char* f = std::getenv("MOE_ROUTER");
    if (f != nullptr && std::strcmp(f, "ffma") == 0) return false;
    return s.E <= 128;
}
// Route workspace: the three bf16 parts of W_g [3 * max(16, E_pad), d] for the
// tensor-core router, else 0.
size_t router_ws_bytes(const moe_shape& s);
cudaError_t launch_router(const moe_shape& s, const __nv_bfloat16* x, const float* Wg,
                          const float* bias, float* logits, int32_t* ids, float* w, void* ws,
                          int* err, cudaStream_t st);

// dispatch.cu
int dispatch_block_tokens();
cudaError_t launch_dispatch(const moe_shape& s, const int32_t* ids, int32_t* eti,
                            int32_t* offsets, int32_t* tim, int32_t* hist, int* err,
                            cudaStream_t st);
// Per-slot lists for the slot-wise fused combine: for every slot k, the
// dispatch of the column ids[:, k] (eti_k [K][T], offsets_k [K][E+1],
// tim_k [K][T]); hist holds K * ceil(T/256) * E entries.
cudaError_t launch_slot_dispatch(const moe_shape& s, const int32_t* ids, int32_t* eti_k,
                                 int32_t* offsets_k, int32_t* tim_k, int32_t* hist, int* err,
                                 cudaStream_t st);

// Token rounding (rounding.cu). Scratch: lse [T], par [E], thr [E], n_t [T],
// w_tok [rows_max], bm [E][ceil(T/32)] (token-choice bitmap), lpT [E][T].
struct TrScratch {
    float* lse;
    int4* par;
    unsigned long long* thr;
    int32_t* n_t;
    float* w_tok;
    uint32_t* bm;
    float* lpT;  // [E][T] log-probabilities, expert-major
};
cudaError_t launch_token_rounding(const moe_shape& s, int m_tile, const float* z,
                                  const int32_t* ids, const int32_t* tc_eti,
                                  const int32_t* tc_offsets, TrScratch sc, int32_t* eti_tr,
                                  int32_t* offsets_tr, float* w_row, int32_t* tok_off,
                                  int32_t* tok_exp, int32_t* tok_rows, int* err, cudaStream_t st);

// Routing given as rows (misc.cu): token t's rows are tok_rows[tok_off[t] ..
// tok_off[t+1]) of experts tok_exp[...]; row r has weight w_row[r] (nullptr: 1).
cudaError_t launch_combine_rows(const moe_shape& s, int t0, int t1, int c0, int nc,
                                const int32_t* tok_off, const int32_t* tok_exp,
                                const int32_t* tok_rows, const float* w_row, const Seg* seg,
                                const __nv_bfloat16* Yc, __nv_bfloat16* y, int* err,
                                cudaStream_t st, const char* name);
// dS_row[r] = sum of the partials of row r; dz_row[r] = w_r (dS_r - sum over the
// token's rows of w dS).
cudaError_t launch_router_dz_rows(const moe_shape& s, int rows_cap, int nparts,
                                  const float* dS_part, const int32_t* tok_off,
                                  const int32_t* tok_rows, const float* w_row, float* dS_row,
                                  float* dz_row, int* err, cudaStream_t st);

// misc.cu
cudaError_t launch_chunk_segments(const moe_shape& s, int chunk_tokens, int nchunks,
                                  const int32_t* eti, const int32_t* offsets, Seg* segs, int* err,
                                  cudaStream_t st);
cudaError_t launch_row_weights(const moe_shape& s, const float* topk_w, const int32_t* tim,
                               float* wrow, int* err, cudaStream_t st);
// topk_w == nullptr sums with weight 1 (the token-gradient sum); `name` labels
// the launch for the kernel timer. direct: the chunk buffer holds every routed
// row in expert-sorted order (column passes, single passes), so the row of
// (t, k) is token_index_map[t*K+k] and seg is not read.
cudaError_t launch_combine(const moe_shape& s, int t0, int t1, int c0, int nc, const int32_t* ids,
                           const float* topk_w, const int32_t* tim, const Seg* seg,
                           const __nv_bfloat16* Yc, __nv_bfloat16* y, int* err, cudaStream_t st,
                           const char* name = "combine", bool direct = false);
cudaError_t launch_router_dz(const moe_shape& s, int nparts, const float* dS_part,
                             const float* topk_w, const int32_t* tim, float* dS, float* dz,
                             float* dz_row, int* err, cudaStream_t st);
// Router weight gradient dW_g = dz^T x (R2b), gathered per expert (x rows
// read through eti, fp32 sums over 32 row parts of each expert, then a
// fixed-order sum): used while x fits in L2.
int dwg_parts(const moe_shape& s);
cudaError_t launch_router_dwg(const moe_shape& s, const __nv_bfloat16* x, const int32_t* eti,
                              const int32_t* offsets, const float* dz_row, float* part,
                              float* dWg, int* err, cudaStream_t st);
// Whether the router weight gradient runs on the tensor cores: once x
// (T*d bf16) exceeds 64 MiB, so that reading it K times costs HBM traffic.
// MOE_ROUTER_DWG=mma|gather forces one path (read at every call; the
// workspace size follows it).
inline bool dwg_tensor_cores(const moe_shape& s) {
    const char* f = std::getenv("MOE_ROUTER_DWG");
    if (f != nullptr && std::strcmp(f, "mma") == 0) return true;
    if (f != nullptr && std::strcmp(f, "gather") == 0) return false;
    return static_cast<long long>(s.T) * s.d * 2 > (64ll << 20);
}
// Router weight gradient dW_g = dz^T x (R2b) as a tensor-core product: the
// dense operand B = [dz_hi | dz_lo] [T, nw] (bf16 parts of dz at each token's
// experts, zeros elsewhere; nw = 2 * e_pad), x^T B over token chunks into fp32
// partials [nchunks, d, nw], then a fixed-order sum. dwg_plan (gemm.cu) sizes it.
struct DwgPlan {
    int e_pad;    // experts padded to a multiple of 64
    int nw;       // columns of B: 2 * e_pad
    int nchunks;  // token chunks (split of the reduction over T)
    int chunk;    // tokens per chunk (multiple of 64)
};
DwgPlan dwg_plan(const moe_shape& s);
// Writes B (zeros, then hi/lo of dz_row[r] at (eti[r], expert of r) for every
// routed row r < offsets[E]), the identity token list and the chunk segments.
cudaError_t launch_dwg_operand(const moe_shape& s, const DwgPlan& dp, int rows_cap,
                               const int32_t* eti, const int32_t* offsets, const float* dz_row,
                               __nv_bfloat16* B, int32_t* iota, Seg* segs, int* err,
                               cudaStream_t st);
// dWg [E, d] = sum over chunks p of part[p][c][e] + part[p][c][e_pad + e], p ascending.
cudaError_t launch_dwg_reduce(const moe_shape& s, const DwgPlan& dp, const float* part,
                              float* dWg, int* err, cudaStream_t st);

// One CTA waits on a barrier nothing arrives at, for at most limit_ns; records
// MOE_ERR_TIMEOUT when the bounded wait gives up (moe_selftest_bounded_wait).
cudaError_t launch_selftest_wait(uint64_t limit_ns, int* err, cudaStream_t st);

// gemm.cu — the grouped tcgen05 GEMMs.
enum GemmKind { G1_UP = 0, G2_DOWN = 1, G3_DH = 2, G4_DW2 = 3, G5_DW13 = 4, G6_DX = 5,
                // Non-gated (SiLU/ReLU) variants of G1 and G3; chosen by launch_gemm
                // from moe_shape.expert, callers pass G1_UP / G3_DH.
                G1_UP_ACT = 6, G3_DH_ACT = 7,
                // Down projection of one routing slot with the combine fused
                // into its epilogue (slot-wise forward).
                G2_SLOT = 8,
                // Router weight gradient partials: x^T [dz_hi | dz_lo] over token
                // chunks (the chunks take the place of the experts), fp32 out.
                G7_DWG = 9 };

struct GemmProblem {
    GemmKind kind;
    moe_shape s;
    const Seg* segs;          // [E] rows of each expert (VM: this chunk's rows)
    const int32_t* eti;       // expert_token_indices (gather rows)
    // operands (bf16 unless noted)
    const void* a_src;        // x (G1) | A_act (G2) | dy (G3) | dy (G4) | x (G5) | dH (G6)
    const void* b_src0;       // W1 (G1) | W2 (G2) | W2 (G3) | A' (G4) | dH (G5) | W1 (G6)
    const void* b_src1;       // W3 (G1, G6)
    // epilogue
    void* out0;               // H (G1) | Yc (G2) | dH (G3) | dW2 (G4) | dW1 (G5) | dXc (G6)
    void* out1;               // A_act (G1) | A' (G3) | dW3 (G5)
    const void* aux0;         // H (G3)
    const float* wrow;        // per-row routing weight (G3)
    float* dS_part;           // [h/BN][TK] (G3)
    int n_off = 0;            // G2/G6: first output column computed by this launch
    int n_cols = 0;           // G2/G6: output columns of this launch (= row stride of out0)
    // G2_SLOT: eti = this slot's token list, a_src = A_act, b_src0 = W2, out0 = the fp32
    // accumulator [T, d], out1 = y [T, d] bf16, wrow = topk_w [T, K], tim = the routing's
    // token_index_map (A_act row of (t, k) = tim[t*K + k]).
    const int32_t* tim = nullptr;
    int slot = 0;
    int rows = 0;             // row capacity of the routed-row arrays (0: T*K)
    // G7_DWG: segs = token chunks (nseg of them), eti = identity list, a_src = x,
    // b_src0 = [dz_hi | dz_lo] [T, nw], out0 = fp32 partials [nseg * d, nw].
    int nseg = 0;
    int* err;
};
cudaError_t launch_gemm(const GemmProblem& p, cudaStream_t st);
int gemm_bn(GemmKind kind, const moe_shape& s);

}  // namespace moe
