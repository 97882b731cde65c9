// api.cu — the C ABI (include/moe.h): argument checks, workspace layout,
// the device status word, launch bookkeeping and the call sequences.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstring>
#include <initializer_list>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"

namespace moe {

// Sticky device status word (one per device that loads the library).
__device__ int g_status_word;

namespace {

constexpr int kMaxDevices = 64;
int* g_status_ptr[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};
std::mutex g_mu;

int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    return (dev >= 0 && dev < kMaxDevices) ? dev : -1;
}

int* status_ptr() {
    const int dev = current_device();
    if (dev < 0) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_status_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
        g_status_ptr[dev] = static_cast<int*>(p);
    }
    return g_status_ptr[dev];
}

// ---------------------------------------------------------------- timing
std::atomic<long long> g_launches{0};
bool g_timing = false;
struct Rec {
    std::string name;
    cudaEvent_t a, b;
};
std::vector<Rec> g_recs;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Bump allocator over the caller's workspace.
struct Carve {
    size_t off = 0;
    char* base = nullptr;
    template <class T>
    T* take(size_t count) {
        off = align_up(off, 256);
        T* p = reinterpret_cast<T*>(base ? base + off : nullptr);
        off += count * sizeof(T);
        return p;
    }
};

int check_shape(const moe_shape& s) {
    if (s.T < 1 || s.d < 1 || s.E < 1 || s.K < 1 || s.h < 1) return MOE_ERR_INVALID_ARG;
    if (s.T > (1 << 24) || s.K > 8 || s.K > s.E || s.E > 256) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (s.d % 128 != 0 || s.h % 128 != 0 || s.d > 32768 || s.h > 32768)
        return MOE_ERR_UNSUPPORTED_SHAPE;
    if (static_cast<long long>(s.T) * s.K >= (1ll << 31)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (s.expert != MOE_EXPERT_SWIGLU && s.expert != MOE_EXPERT_SILU && s.expert != MOE_EXPERT_RELU)
        return MOE_ERR_INVALID_ARG;
    // A non-gated up-projection tile is 256 columns of W1.
    if (s.expert != MOE_EXPERT_SWIGLU && s.h % 256 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    return MOE_OK;
}

bool gated(const moe_shape& s) { return s.expert == MOE_EXPERT_SWIGLU; }

// Width of the saved pre-activation H and of its gradient dH.
size_t hs_of(const moe_shape& s) { return gated(s) ? 2 * static_cast<size_t>(s.h) : s.h; }

int nchunks_of(const moe_shape& s, int tc) { return (s.T + tc - 1) / tc; }

// How a down projection (forward) or dX pass (backward) is split so that its
// transient [rows, columns] output buffer holds at most a quarter of T*K*d
// once T >= 1024. Splitting by token chunks streams the expert weights once
// per chunk; splitting by output-column chunks streams the activation
// operand once per chunk instead. The split that re-reads fewer bytes wins.
struct Plan {
    int n;         // passes
    bool by_cols;  // column chunks (else token chunks)
    int tc;        // tokens per token chunk
    int dc;        // columns per column chunk
};

Plan make_plan(const moe_shape& s, double weight_bytes, double act_bytes) {
    Plan p{1, false, s.T, s.d};
    if (s.T < 1024) return p;
    p.n = 4;
    p.tc = moe_chunk_tokens(s);
    p.n = nchunks_of(s, p.tc);
    const bool cols_ok = s.d % (4 * 128) == 0;
    if (cols_ok && act_bytes < weight_bytes) {
        p.n = 4;
        p.by_cols = true;
        p.tc = s.T;
        p.dc = s.d / 4;
    }
    return p;
}

Plan plan_down(const moe_shape& s) {
    const double TK = static_cast<double>(s.T) * s.K;
    return make_plan(s, 2.0 * s.E * s.d * s.h, 2.0 * TK * s.h);
}

Plan plan_dx(const moe_shape& s) {
    const double TK = static_cast<double>(s.T) * s.K;
    const double hs = static_cast<double>(hs_of(s));
    return make_plan(s, 2.0 * s.E * s.d * hs, 2.0 * TK * hs);
}

size_t chunk_buffer_elems(const moe_shape& s, const Plan& p) {
    const size_t TK = static_cast<size_t>(s.T) * s.K;
    return p.by_cols ? TK * p.dc : static_cast<size_t>(p.tc) * s.K * s.d;
}

struct FwdWs {
    Seg* segs;
    __nv_bfloat16* Aact;
    __nv_bfloat16* Yc;
};
struct BwdWs {
    Seg* segs;
    float* wrow;
    float* dS_part;
    float* dz;
    float* dz_row;
    __nv_bfloat16* Ap;
    __nv_bfloat16* dH;
    __nv_bfloat16* dXc;
    float* dwg_part;
};

size_t layout_fwd(const moe_shape& s, void* ws, FwdWs* o) {
    const int tc = moe_chunk_tokens(s);
    const int nc = nchunks_of(s, tc);
    const size_t TK = static_cast<size_t>(s.T) * s.K;
    Carve c;
    c.base = static_cast<char*>(ws);
    FwdWs w;
    w.segs = c.take<Seg>(static_cast<size_t>(nc + 1) * s.E);
    w.Aact = c.take<__nv_bfloat16>(TK * s.h);
    w.Yc = c.take<__nv_bfloat16>(chunk_buffer_elems(s, plan_down(s)));
    if (o) *o = w;
    return align_up(c.off, 256);
}

size_t layout_bwd(const moe_shape& s, void* ws, BwdWs* o) {
    const int tc = moe_chunk_tokens(s);
    const int nc = nchunks_of(s, tc);
    const size_t TK = static_cast<size_t>(s.T) * s.K;
    const int bn3 = gemm_bn(G3_DH, s);
    const int nparts = (s.h + bn3 - 1) / bn3;
    Carve c;
    c.base = static_cast<char*>(ws);
    BwdWs w;
    w.segs = c.take<Seg>(static_cast<size_t>(nc + 1) * s.E);
    w.wrow = c.take<float>(TK);
    w.dS_part = c.take<float>(TK * nparts);
    w.dz = c.take<float>(TK);
    w.dz_row = c.take<float>(TK);
    w.Ap = c.take<__nv_bfloat16>(TK * s.h);
    w.dH = c.take<__nv_bfloat16>(TK * hs_of(s));
    w.dXc = c.take<__nv_bfloat16>(chunk_buffer_elems(s, plan_dx(s)));
    w.dwg_part = c.take<float>(static_cast<size_t>(dwg_parts()) * s.E * s.d);
    if (o) *o = w;
    return align_up(c.off, 256);
}

struct SlotWs {
    Seg* segs;        // [E] whole-row-space segments (G1), then [K][E] per slot
    __nv_bfloat16* Aact;
    int32_t* eti_k;   // [K][T]
    int32_t* off_k;   // [K][E+1]
    int32_t* tim_k;   // [K][T] (written by the slot dispatch, unused)
    int32_t* hist;    // [K][ceil(T/256)][E]
    float* acc;       // [T, d] fp32 accumulator of y (K >= 2)
};

size_t layout_fwd_slot(const moe_shape& s, void* ws, SlotWs* o) {
    const size_t TK = static_cast<size_t>(s.T) * s.K;
    const size_t nblk = (s.T + dispatch_block_tokens() - 1) / dispatch_block_tokens();
    Carve c;
    c.base = static_cast<char*>(ws);
    SlotWs w;
    w.segs = c.take<Seg>(static_cast<size_t>(s.K + 1) * s.E);
    w.Aact = c.take<__nv_bfloat16>(TK * s.h);
    w.eti_k = c.take<int32_t>(TK);
    w.off_k = c.take<int32_t>(static_cast<size_t>(s.K) * (s.E + 1));
    w.tim_k = c.take<int32_t>(TK);
    w.hist = c.take<int32_t>(static_cast<size_t>(s.K) * nblk * s.E);
    w.acc = s.K > 1 ? c.take<float>(static_cast<size_t>(s.T) * s.d) : nullptr;
    if (o) *o = w;
    return align_up(c.off, 256);
}

size_t layout_dispatch(const moe_shape& s, void* ws, int32_t** hist) {
    const int nblk = (s.T + dispatch_block_tokens() - 1) / dispatch_block_tokens();
    Carve c;
    c.base = static_cast<char*>(ws);
    int32_t* h = c.take<int32_t>(static_cast<size_t>(nblk) * s.E);
    if (hist) *hist = h;
    return align_up(c.off, 256);
}

// Last CUDA failure of a launch sequence, for moe_last_cuda_error().
thread_local char g_last_cuda_error[160] = "";
thread_local const char* g_current_launch = "";

int record_cuda_error(cudaError_t e) {
    std::snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "%s: %s", g_current_launch,
                  cudaGetErrorString(e));
    cudaGetLastError();  // clear a non-sticky launch error so later calls start clean
    return MOE_ERR_CUDA;
}

#define MOE_TRY(expr)                                          \
    do {                                                       \
        cudaError_t _e = (expr);                               \
        if (_e != cudaSuccess) return record_cuda_error(_e);   \
    } while (0)

}  // namespace

LaunchScope::LaunchScope(const char* name, cudaStream_t st) : name_(name), st_(st), slot_(-1) {
    g_launches.fetch_add(1, std::memory_order_relaxed);
    g_current_launch = name;
    if (!g_timing) return;
    std::lock_guard<std::mutex> lk(g_mu);
    Rec r;
    r.name = name;
    if (cudaEventCreate(&r.a) != cudaSuccess) return;
    if (cudaEventCreate(&r.b) != cudaSuccess) {
        cudaEventDestroy(r.a);
        return;
    }
    cudaEventRecord(r.a, st);
    g_recs.push_back(r);
    slot_ = static_cast<int>(g_recs.size()) - 1;
}

LaunchScope::~LaunchScope() {
    if (slot_ < 0) return;
    std::lock_guard<std::mutex> lk(g_mu);
    cudaEventRecord(g_recs[slot_].b, st_);
}

bool make_tmap_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                    uint32_t box_cols, uint32_t box_rows, bool swizzle128) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t es[2] = {1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                          strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_tmap_f32(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                   uint32_t box_cols, uint32_t box_rows) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 4};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t es[2] = {1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims,
                          strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int* device_status_word() { return status_ptr(); }

int num_sms() {
    const int dev = current_device();
    if (dev < 0) return 1;
    if (g_num_sms[dev] == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        g_num_sms[dev] = n > 0 ? n : 1;
    }
    return g_num_sms[dev];
}

}  // namespace moe

using namespace moe;

extern "C" {

int moe_chunk_tokens(moe_shape s) {
    if (s.T < 1024) return std::max(1, s.T);
    return (s.T + 3) / 4;
}

size_t moe_workspace_size(moe_shape s, int which) {
    if (check_shape(s) != MOE_OK) return 0;
    switch (which) {
        case MOE_WS_ROUTE: return 0;
        case MOE_WS_DISPATCH: return layout_dispatch(s, nullptr, nullptr);
        case MOE_WS_FORWARD: return layout_fwd(s, nullptr, nullptr);
        case MOE_WS_BACKWARD: return layout_bwd(s, nullptr, nullptr);
        case MOE_WS_FORWARD_SLOTWISE: return layout_fwd_slot(s, nullptr, nullptr);
    }
    return 0;
}

int moe_route(moe_shape s, const void* x, const float* Wg, const float* bias, float* logits,
              int32_t* topk_ids, float* topk_w, void* ws, size_t ws_bytes, void* stream) {
    (void)ws;
    (void)ws_bytes;
    int rc = check_shape(s);
    if (rc) return rc;
    if (!x || !Wg || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(Wg) || (logits && !aligned16(logits)))
        return MOE_ERR_MISALIGNED;
    int* err = status_ptr();
    if (!err) return MOE_ERR_NO_DEVICE;
    MOE_TRY(launch_router(s, static_cast<const __nv_bfloat16*>(x), Wg, bias, logits, topk_ids,
                          topk_w, err, static_cast<cudaStream_t>(stream)));
    return MOE_OK;
}

int moe_build_dispatch(moe_shape s, const int32_t* topk_ids, int32_t* eti, int32_t* offsets,
                       int32_t* tim, void* ws, size_t ws_bytes, void* stream) {
    int rc = check_shape(s);
    if (rc) return rc;
    if (!topk_ids || !eti || !offsets || !tim || !ws) return MOE_ERR_INVALID_ARG;
    if (ws_bytes < layout_dispatch(s, nullptr, nullptr)) return MOE_ERR_WORKSPACE_TOO_SMALL;
    int32_t* hist = nullptr;
    layout_dispatch(s, ws, &hist);
    int* err = status_ptr();
    if (!err) return MOE_ERR_NO_DEVICE;
    MOE_TRY(launch_dispatch(s, topk_ids, eti, offsets, tim, hist, err,
                            static_cast<cudaStream_t>(stream)));
    return MOE_OK;
}

int moe_forward(moe_shape s, const void* x, const void* W1, const void* W3, const void* W2,
                const int32_t* topk_ids, const float* topk_w, const int32_t* eti,
                const int32_t* offsets, const int32_t* tim, void* y, void* H_saved, void* ws,
                size_t ws_bytes, void* stream) {
    int rc = check_shape(s);
    if (rc) return rc;
    if (!x || !W1 || (gated(s) && !W3) || !W2 || !topk_ids || !topk_w || !eti || !offsets ||
        !tim || !y || !H_saved || !ws)
        return MOE_ERR_INVALID_ARG;
    for (const void* p : std::initializer_list<const void*>{x, W1, W2, y, H_saved, ws})
        if (!aligned16(p)) return MOE_ERR_MISALIGNED;
    if (gated(s) && !aligned16(W3)) return MOE_ERR_MISALIGNED;
    if (ws_bytes < layout_fwd(s, nullptr, nullptr)) return MOE_ERR_WORKSPACE_TOO_SMALL;
    int* err = status_ptr();
    if (!err) return MOE_ERR_NO_DEVICE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    FwdWs w;
    layout_fwd(s, ws, &w);
    const int tc = moe_chunk_tokens(s);
    const int nc = nchunks_of(s, tc);
    const Plan pl = plan_down(s);
    // Column-chunked passes, and a single token chunk, use the whole-row-space
    // segments only.
    const bool per_chunk = !pl.by_cols && nc > 1;
    MOE_TRY(launch_chunk_segments(s, tc, per_chunk ? nc : 0, eti, offsets,
                                  per_chunk ? w.segs : w.segs + static_cast<size_t>(nc) * s.E,
                                  err, st));
    const Seg* full = w.segs + static_cast<size_t>(nc) * s.E;

    GemmProblem g1{};
    g1.kind = G1_UP;
    g1.s = s;
    g1.segs = full;
    g1.eti = eti;
    g1.a_src = x;
    g1.b_src0 = W1;
    g1.b_src1 = W3;
    g1.out0 = H_saved;
    g1.out1 = w.Aact;
    g1.err = err;
    MOE_TRY(launch_gemm(g1, st));

    for (int c = 0; c < pl.n; ++c) {
        const Seg* sc = per_chunk ? w.segs + static_cast<size_t>(c) * s.E : full;
        GemmProblem g2{};
        g2.kind = G2_DOWN;
        g2.s = s;
        g2.segs = sc;
        g2.eti = eti;
        g2.a_src = w.Aact;
        g2.b_src0 = W2;
        g2.out0 = w.Yc;
        g2.n_off = pl.by_cols ? c * pl.dc : 0;
        g2.n_cols = pl.by_cols ? pl.dc : s.d;
        g2.err = err;
        MOE_TRY(launch_gemm(g2, st));
        const int t0 = pl.by_cols ? 0 : c * tc, t1 = pl.by_cols ? s.T : std::min(s.T, t0 + tc);
        MOE_TRY(launch_combine(s, t0, t1, g2.n_off, g2.n_cols, topk_ids, topk_w, tim, sc, w.Yc,
                               static_cast<__nv_bfloat16*>(y), err, st));
    }
    return MOE_OK;
}

int moe_forward_slotwise(moe_shape s, const void* x, const void* W1, const void* W3,
                         const void* W2, const int32_t* topk_ids, const float* topk_w,
                         const int32_t* eti, const int32_t* offsets, const int32_t* tim, void* y,
                         void* H_saved, void* ws, size_t ws_bytes, void* stream) {
    int rc = check_shape(s);
    if (rc) return rc;
    if (!x || !W1 || (gated(s) && !W3) || !W2 || !topk_ids || !topk_w || !eti || !offsets ||
        !tim || !y || !H_saved || !ws)
        return MOE_ERR_INVALID_ARG;
    for (const void* p : std::initializer_list<const void*>{x, W1, W2, y, H_saved, ws})
        if (!aligned16(p)) return MOE_ERR_MISALIGNED;
    if (gated(s) && !aligned16(W3)) return MOE_ERR_MISALIGNED;
    if (ws_bytes < layout_fwd_slot(s, nullptr, nullptr)) return MOE_ERR_WORKSPACE_TOO_SMALL;
    int* err = status_ptr();
    if (!err) return MOE_ERR_NO_DEVICE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    SlotWs w;
    layout_fwd_slot(s, ws, &w);
    const int tc = moe_chunk_tokens(s);
    MOE_TRY(launch_chunk_segments(s, tc, 0, eti, offsets, w.segs, err, st));

    GemmProblem g1{};
    g1.kind = G1_UP;
    g1.s = s;
    g1.segs = w.segs;
    g1.eti = eti;
    g1.a_src = x;
    g1.b_src0 = W1;
    g1.b_src1 = W3;
    g1.out0 = H_saved;
    g1.out1 = w.Aact;
    g1.err = err;
    MOE_TRY(launch_gemm(g1, st));

    // Slot k's rows grouped by expert, ascending token: the dispatch of ids[:, k].
    MOE_TRY(launch_slot_dispatch(s, topk_ids, w.eti_k, w.off_k, w.tim_k, w.hist, err, st));
    for (int k = 0; k < s.K; ++k) {
        Seg* sk = w.segs + static_cast<size_t>(k + 1) * s.E;
        const int32_t* eti_k = w.eti_k + static_cast<size_t>(k) * s.T;
        MOE_TRY(launch_chunk_segments(s, tc, 0, eti_k, w.off_k + static_cast<size_t>(k) * (s.E + 1),
                                      sk, err, st));
        GemmProblem g2{};
        g2.kind = G2_SLOT;
        g2.s = s;
        g2.segs = sk;
        g2.eti = eti_k;
        g2.a_src = w.Aact;
        g2.b_src0 = W2;
        g2.out0 = w.acc;
        g2.out1 = y;
        g2.wrow = topk_w;
        g2.tim = tim;
        g2.slot = k;
        g2.err = err;
        MOE_TRY(launch_gemm(g2, st));
    }
    return MOE_OK;
}

int moe_backward(moe_shape s, const void* dy, const void* x, const float* Wg, const void* W1,
                 const void* W3, const void* W2, const int32_t* topk_ids, const float* topk_w,
                 const int32_t* eti, const int32_t* offsets, const int32_t* tim,
                 const void* H_saved, void* dx, float* dWg, void* dW1, void* dW3, void* dW2,
                 float* dS, void* ws, size_t ws_bytes, void* stream) {
    int rc = check_shape(s);
    if (rc) return rc;
    const bool gw = gated(s);  // W3 and dW3 exist
    if (!dy || !x || !Wg || !W1 || (gw && !W3) || !W2 || !topk_ids || !topk_w || !eti ||
        !offsets || !tim || !H_saved || !dx || !dWg || !dW1 || (gw && !dW3) || !dW2 || !dS || !ws)
        return MOE_ERR_INVALID_ARG;
    for (const void* p : std::initializer_list<const void*>{
             dy, x, static_cast<const void*>(Wg), W1, W2, H_saved, static_cast<const void*>(dx),
             static_cast<const void*>(dWg), static_cast<const void*>(dW1),
             static_cast<const void*>(dW2), static_cast<const void*>(ws)})
        if (!aligned16(p)) return MOE_ERR_MISALIGNED;
    if (gw && (!aligned16(W3) || !aligned16(dW3))) return MOE_ERR_MISALIGNED;
    if (ws_bytes < layout_bwd(s, nullptr, nullptr)) return MOE_ERR_WORKSPACE_TOO_SMALL;
    int* err = status_ptr();
    if (!err) return MOE_ERR_NO_DEVICE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    BwdWs w;
    layout_bwd(s, ws, &w);
    const int tc = moe_chunk_tokens(s);
    const int nc = nchunks_of(s, tc);
    const Plan pl = plan_dx(s);
    // Column-chunked passes, and a single token chunk, use the whole-row-space
    // segments only.
    const bool per_chunk = !pl.by_cols && nc > 1;
    MOE_TRY(launch_chunk_segments(s, tc, per_chunk ? nc : 0, eti, offsets,
                                  per_chunk ? w.segs : w.segs + static_cast<size_t>(nc) * s.E,
                                  err, st));
    const Seg* full = w.segs + static_cast<size_t>(nc) * s.E;
    MOE_TRY(launch_row_weights(s, topk_w, tim, w.wrow, err, st));

    GemmProblem g3{};
    g3.kind = G3_DH;
    g3.s = s;
    g3.segs = full;
    g3.eti = eti;
    g3.a_src = dy;
    g3.b_src0 = W2;
    g3.out0 = w.dH;
    g3.out1 = w.Ap;
    g3.aux0 = H_saved;
    g3.wrow = w.wrow;
    g3.dS_part = w.dS_part;
    g3.err = err;
    MOE_TRY(launch_gemm(g3, st));
    const int bn3 = gemm_bn(G3_DH, s);
    const int nparts = (s.h + bn3 - 1) / bn3;  // G3's N tiles, one dS partial each
    MOE_TRY(launch_router_dz(s, nparts, w.dS_part, topk_w, tim, dS, w.dz, w.dz_row, err, st));

    GemmProblem g4{};
    g4.kind = G4_DW2;
    g4.s = s;
    g4.segs = full;
    g4.eti = eti;
    g4.a_src = dy;
    g4.b_src0 = w.Ap;
    g4.out0 = dW2;
    g4.err = err;
    MOE_TRY(launch_gemm(g4, st));

    GemmProblem g5{};
    g5.kind = G5_DW13;
    g5.s = s;
    g5.segs = full;
    g5.eti = eti;
    g5.a_src = x;
    g5.b_src0 = w.dH;
    g5.out0 = dW1;
    g5.out1 = dW3;
    g5.err = err;
    MOE_TRY(launch_gemm(g5, st));

    for (int c = 0; c < pl.n; ++c) {
        const Seg* sc = per_chunk ? w.segs + static_cast<size_t>(c) * s.E : full;
        GemmProblem g6{};
        g6.kind = G6_DX;
        g6.s = s;
        g6.segs = sc;
        g6.eti = eti;
        g6.a_src = w.dH;
        g6.b_src0 = W1;
        g6.b_src1 = W3;
        g6.out0 = w.dXc;
        g6.wrow = w.dz_row;  // router term dz_r W_g[e] added in the epilogue
        g6.aux0 = Wg;
        g6.n_off = pl.by_cols ? c * pl.dc : 0;
        g6.n_cols = pl.by_cols ? pl.dc : s.d;
        g6.err = err;
        MOE_TRY(launch_gemm(g6, st));
        const int t0 = pl.by_cols ? 0 : c * tc, t1 = pl.by_cols ? s.T : std::min(s.T, t0 + tc);
        MOE_TRY(launch_combine(s, t0, t1, g6.n_off, g6.n_cols, topk_ids, nullptr, tim, sc, w.dXc,
                               static_cast<__nv_bfloat16*>(dx), err, st, "dx_combine"));
    }
    MOE_TRY(launch_router_dwg(s, static_cast<const __nv_bfloat16*>(x), eti, offsets, w.dz_row,
                              w.dwg_part, dWg, err, st));
    return MOE_OK;
}

int moe_get_error(void* stream) {
    int* p = status_ptr();
    if (!p) return MOE_ERR_NO_DEVICE;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return MOE_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
    if (v != 0 && cudaMemset(p, 0, sizeof(int)) != cudaSuccess) return MOE_ERR_CUDA;
    return v;
}

const char* moe_status_string(int status) {
    switch (status) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
        case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case MOE_ERR_CUDA: return "CUDA runtime error";
        case MOE_ERR_BAD_EXPERT_ID: return "expert id out of range or repeated within a token";
        case MOE_ERR_TIMEOUT: return "bounded device wait ran out";
        case MOE_ERR_MISALIGNED: return "pointer not 16-byte aligned";
        case MOE_ERR_NO_DEVICE: return "no usable CUDA device";
        case MOE_ERR_STATIC_SCRATCH_LIMIT:
            return "shape needs more scratch than the library's static device array holds";
    }
    return "unknown status";
}

long long moe_launch_count(void) { return g_launches.load(); }

const char* moe_last_cuda_error(void) { return g_last_cuda_error; }

int moe_timing_enable(int on) {
    std::lock_guard<std::mutex> lk(g_mu);
    for (auto& r : g_recs) {
        cudaEventDestroy(r.a);
        cudaEventDestroy(r.b);
    }
    g_recs.clear();
    g_timing = on != 0;
    return MOE_OK;
}

int moe_timing_collect(moe_kernel_time* out, int max) {
    std::lock_guard<std::mutex> lk(g_mu);
    std::vector<moe_kernel_time> agg;
    for (auto& r : g_recs) {
        if (cudaEventSynchronize(r.b) != cudaSuccess) return -MOE_ERR_CUDA;
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) return -MOE_ERR_CUDA;
        auto it = std::find_if(agg.begin(), agg.end(), [&](const moe_kernel_time& k) {
            return std::strncmp(k.name, r.name.c_str(), sizeof(k.name)) == 0;
        });
        if (it == agg.end()) {
            moe_kernel_time k{};
            std::strncpy(k.name, r.name.c_str(), sizeof(k.name) - 1);
            agg.push_back(k);
            it = agg.end() - 1;
        }
        it->launches += 1;
        it->total_ms += ms;
        cudaEventDestroy(r.a);
        cudaEventDestroy(r.b);
    }
    g_recs.clear();
    const int n = static_cast<int>(agg.size());
    for (int i = 0; i < n && i < max; ++i) out[i] = agg[i];
    return n;
}

}  // extern "C"
