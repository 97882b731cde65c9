// api.cu — the C ABI (include/moe.h): argument checks, workspace layout,
// the device status word, launch bookkeeping and the call sequences.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstdlib>
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

size_t tk_of(const moe_shape& s) { return static_cast<size_t>(s.T) * s.K; }

// Width of the saved pre-activation H and of its gradient dH.
size_t hs_of(const moe_shape& s) { return gated(s) ? 2 * static_cast<size_t>(s.h) : s.h; }

int nchunks_of(const moe_shape& s, int tc) { return (s.T + tc - 1) / tc; }

// How a down projection (forward) or dX pass (backward) is split so that its
// transient [rows, columns] output buffer holds at most a quarter of T*K*d
// once T >= 1024 (half of it on small layers, see column_passes and
// moe_chunk_tokens). Splitting by token chunks streams the expert weights once
// per chunk; splitting by output-column chunks streams the activation
// operand once per chunk instead. The split that re-reads fewer bytes wins.
struct Plan {
    int n;         // passes
    bool by_cols;  // column chunks (else token chunks)
    int tc;        // tokens per token chunk
    int dc;        // columns per column chunk
};

// Column passes over `rows` routed rows: two when the half-width buffer
// (rows x d/2 bf16) is at most 64 MiB, else four. On small layers each pass
// costs a launch, a pipeline fill, a tail and a short combine launch, and
// re-streams the whole activation operand, while the buffer saved is small
// next to the [rows, h] activations the layer holds anyway.
// MOE_COLUMN_PASSES=2|4 forces one count (read at every call).
int column_passes(const moe_shape& s, double rows) {
    const char* f = std::getenv("MOE_COLUMN_PASSES");
    if (f != nullptr && (f[0] == '2' || f[0] == '4') && f[1] == '\0') return f[0] - '0';
    return rows * (s.d / 2) * 2.0 <= 64.0 * 1024 * 1024 ? 2 : 4;
}

// Row mode (a routing given as rows, e.g. after token rounding): a token chunk
// may hold any number of rows, so passes split columns only (d % 512 == 0) or
// there is a single pass over all rows.
Plan make_plan(const moe_shape& s, double rows, double weight_bytes, double act_bytes,
               bool row_mode) {
    Plan p{1, false, s.T, s.d};
    if (s.T < 1024) return p;
    const bool cols_ok = s.d % (4 * 128) == 0;
    if (row_mode) {
        if (cols_ok) {
            p.n = column_passes(s, rows);
            p.by_cols = true;
            p.dc = s.d / p.n;
        }
        return p;
    }
    p.tc = moe_chunk_tokens(s);
    p.n = nchunks_of(s, p.tc);
    if (cols_ok && act_bytes < weight_bytes) {
        p.n = column_passes(s, rows);
        p.by_cols = true;
        p.tc = s.T;
        p.dc = s.d / p.n;
    }
    return p;
}

// rows: row capacity of the routing (T*K for a top-K routing).
Plan plan_down(const moe_shape& s, size_t rows, bool row_mode) {
    return make_plan(s, static_cast<double>(rows), 2.0 * s.E * s.d * s.h,
                     2.0 * static_cast<double>(rows) * s.h, row_mode);
}

Plan plan_dx(const moe_shape& s, size_t rows, bool row_mode) {
    const double hs = static_cast<double>(hs_of(s));
    return make_plan(s, static_cast<double>(rows), 2.0 * s.E * s.d * hs,
                     2.0 * static_cast<double>(rows) * hs, row_mode);
}

size_t chunk_buffer_elems(const moe_shape& s, const Plan& p, size_t rows, bool row_mode) {
    if (p.by_cols) return rows * p.dc;
    return row_mode ? rows * s.d : static_cast<size_t>(p.tc) * s.K * s.d;
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
    // router weight gradient on the tensor cores
    __nv_bfloat16* dwg_B;  // [T, nw] = [dz_hi | dz_lo]
    int32_t* dwg_iota;     // [T] identity token list
    Seg* dwg_segs;         // [nchunks] token chunks
    float* dwg_part;       // [nchunks, d, nw] fp32 partials
};

size_t layout_fwd(const moe_shape& s, size_t rows, bool row_mode, void* ws, FwdWs* o) {
    const int tc = moe_chunk_tokens(s);
    const int nc = nchunks_of(s, tc);
    Carve c;
    c.base = static_cast<char*>(ws);
    FwdWs w;
    w.segs = c.take<Seg>(static_cast<size_t>(nc + 1) * s.E);
    w.Aact = c.take<__nv_bfloat16>(rows * s.h);
    w.Yc = c.take<__nv_bfloat16>(
        chunk_buffer_elems(s, plan_down(s, rows, row_mode), rows, row_mode));
    if (o) *o = w;
    return align_up(c.off, 256);
}

size_t layout_bwd(const moe_shape& s, size_t rows, bool row_mode, void* ws, BwdWs* o) {
    const int tc = moe_chunk_tokens(s);
    const int nc = nchunks_of(s, tc);
    const size_t TK = static_cast<size_t>(s.T) * s.K;
    const int bn3 = gemm_bn(G3_DH, s);
    const int nparts = 2 * ((s.h + bn3 - 1) / bn3);  // two dS partial slots per G3 N tile
    Carve c;
    c.base = static_cast<char*>(ws);
    BwdWs w;
    w.segs = c.take<Seg>(static_cast<size_t>(nc + 1) * s.E);
    w.wrow = c.take<float>(rows);
    w.dS_part = c.take<float>(rows * nparts);
    w.dz = c.take<float>(TK);
    w.dz_row = c.take<float>(rows);
    w.Ap = c.take<__nv_bfloat16>(rows * s.h);
    w.dH = c.take<__nv_bfloat16>(rows * hs_of(s));
    w.dXc = c.take<__nv_bfloat16>(
        chunk_buffer_elems(s, plan_dx(s, rows, row_mode), rows, row_mode));
    if (dwg_tensor_cores(s)) {
        const DwgPlan dp = dwg_plan(s);
        w.dwg_B = c.take<__nv_bfloat16>(static_cast<size_t>(s.T) * dp.nw);
        w.dwg_iota = c.take<int32_t>(static_cast<size_t>(s.T));
        w.dwg_segs = c.take<Seg>(static_cast<size_t>(dp.nchunks));
        w.dwg_part = c.take<float>(static_cast<size_t>(dp.nchunks) * s.d * dp.nw);
    } else {
        w.dwg_B = nullptr;
        w.dwg_iota = nullptr;
        w.dwg_segs = nullptr;
        w.dwg_part = c.take<float>(static_cast<size_t>(dwg_parts(s)) * s.E * s.d);
    }
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

// The routing a forward or backward runs on: top-K slots (ids, topk_w, tim;
// rows = T*K) or rows with a per-token row list (tok_off, tok_exp, tok_rows,
// w_row; rows = the row capacity).
struct RouteView {
    size_t rows;
    const int32_t* eti;
    const int32_t* offsets;
    const int32_t* ids = nullptr;
    const float* topk_w = nullptr;
    const int32_t* tim = nullptr;
    const int32_t* tok_off = nullptr;
    const int32_t* tok_exp = nullptr;
    const int32_t* tok_rows = nullptr;
    const float* w_row = nullptr;
    bool row_mode() const { return tok_off != nullptr; }
};

size_t rows_capacity(const moe_shape& s, int m_tile) {
    const size_t a = tk_of(s) + static_cast<size_t>(s.E) * (m_tile - 1);
    const size_t b = static_cast<size_t>(s.T) * s.E;
    return std::min(a, b);
}

size_t layout_rounding(const moe_shape& s, int m_tile, void* ws, TrScratch* o) {
    Carve c;
    c.base = static_cast<char*>(ws);
    TrScratch w;
    w.lse = c.take<float>(s.T);
    w.par = c.take<int4>(s.E);
    w.thr = c.take<unsigned long long>(s.E);
    w.n_t = c.take<int32_t>(s.T);
    w.w_tok = c.take<float>(rows_capacity(s, m_tile));
    w.bm = c.take<uint32_t>(static_cast<size_t>(s.E) * ((s.T + 31) / 32));
    w.lpT = c.take<float>(static_cast<size_t>(s.E) * s.T);
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

int check_shape_status(const moe_shape& s) { return check_shape(s); }
int cuda_error_status(cudaError_t e) { return record_cuda_error(e); }

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
                    uint32_t box_cols, uint32_t box_rows, int swizzle) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t es[2] = {1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                          strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          swizzle == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                          : swizzle == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                          : CU_TENSOR_MAP_SWIZZLE_NONE,
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

// ---------------------------------------------------------------- call sequences
namespace moe {
namespace {

int forward_impl(const moe_shape& s, const RouteView& rv, const void* x, const void* W1,
                 const void* W3, const void* W2, void* y, void* H_saved, void* ws,
                 size_t ws_bytes, void* stream) {
    const bool rm = rv.row_mode();
    if (!x || !W1 || (gated(s) && !W3) || !W2 || !rv.eti || !rv.offsets || !y || !H_saved || !ws)
        return MOE_ERR_INVALID_ARG;
    for (const void* p : std::initializer_list<const void*>{x, W1, W2, y, H_saved, ws})
        if (!aligned16(p)) return MOE_ERR_MISALIGNED;
    if (gated(s) && !aligned16(W3)) return MOE_ERR_MISALIGNED;
    if (ws_bytes < layout_fwd(s, rv.rows, rm, nullptr, nullptr)) return MOE_ERR_WORKSPACE_TOO_SMALL;
    int* err = status_ptr();
    if (!err) return MOE_ERR_NO_DEVICE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    FwdWs w;
    layout_fwd(s, rv.rows, rm, ws, &w);
    const int nc = nchunks_of(s, moe_chunk_tokens(s));
    const Plan pl = plan_down(s, rv.rows, rm);
    // Column-chunked passes, and a single pass, use the whole-row-space
    // segments only.
    const bool per_chunk = !pl.by_cols && pl.n > 1;
    MOE_TRY(launch_chunk_segments(s, pl.tc, per_chunk ? pl.n : 0, rv.eti, rv.offsets,
                                  per_chunk ? w.segs : w.segs + static_cast<size_t>(nc) * s.E,
                                  err, st));
    const Seg* full = w.segs + static_cast<size_t>(nc) * s.E;

    GemmProblem g1{};
    g1.kind = G1_UP;
    g1.s = s;
    g1.rows = static_cast<int>(rv.rows);
    g1.segs = full;
    g1.eti = rv.eti;
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
        g2.rows = static_cast<int>(rv.rows);
        g2.segs = sc;
        g2.eti = rv.eti;
        g2.a_src = w.Aact;
        g2.b_src0 = W2;
        g2.out0 = w.Yc;
        g2.n_off = pl.by_cols ? c * pl.dc : 0;
        g2.n_cols = pl.by_cols ? pl.dc : s.d;
        g2.err = err;
        MOE_TRY(launch_gemm(g2, st));
        const int t0 = pl.by_cols ? 0 : c * pl.tc;
        const int t1 = pl.by_cols ? s.T : std::min(s.T, t0 + pl.tc);
        if (rm)
            MOE_TRY(launch_combine_rows(s, t0, t1, g2.n_off, g2.n_cols, rv.tok_off, rv.tok_exp,
                                        rv.tok_rows, rv.w_row, sc, w.Yc,
                                        static_cast<__nv_bfloat16*>(y), err, st, "combine"));
        else
            MOE_TRY(launch_combine(s, t0, t1, g2.n_off, g2.n_cols, rv.ids, rv.topk_w, rv.tim, sc,
                                   w.Yc, static_cast<__nv_bfloat16*>(y), err, st, "combine",
                                   !per_chunk));
    }
    return MOE_OK;
}

int backward_impl(const moe_shape& s, const RouteView& rv, const void* dy, const void* x,
                  const float* Wg, const void* W1, const void* W3, const void* W2,
                  const void* H_saved, void* dx, float* dWg, void* dW1, void* dW3, void* dW2,
                  float* dS, void* ws, size_t ws_bytes, void* stream) {
    const bool rm = rv.row_mode();
    const bool gw = gated(s);  // W3 and dW3 exist
    if (!dy || !x || !Wg || !W1 || (gw && !W3) || !W2 || !rv.eti || !rv.offsets || !H_saved ||
        !dx || !dWg || !dW1 || (gw && !dW3) || !dW2 || !dS || !ws)
        return MOE_ERR_INVALID_ARG;
    for (const void* p : std::initializer_list<const void*>{
             dy, x, static_cast<const void*>(Wg), W1, W2, H_saved, static_cast<const void*>(dx),
             static_cast<const void*>(dWg), static_cast<const void*>(dW1),
             static_cast<const void*>(dW2), static_cast<const void*>(ws)})
        if (!aligned16(p)) return MOE_ERR_MISALIGNED;
    if (gw && (!aligned16(W3) || !aligned16(dW3))) return MOE_ERR_MISALIGNED;
    if (ws_bytes < layout_bwd(s, rv.rows, rm, nullptr, nullptr)) return MOE_ERR_WORKSPACE_TOO_SMALL;
    int* err = status_ptr();
    if (!err) return MOE_ERR_NO_DEVICE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    BwdWs w;
    layout_bwd(s, rv.rows, rm, ws, &w);
    const int nc = nchunks_of(s, moe_chunk_tokens(s));
    const Plan pl = plan_dx(s, rv.rows, rm);
    const bool per_chunk = !pl.by_cols && pl.n > 1;
    MOE_TRY(launch_chunk_segments(s, pl.tc, per_chunk ? pl.n : 0, rv.eti, rv.offsets,
                                  per_chunk ? w.segs : w.segs + static_cast<size_t>(nc) * s.E,
                                  err, st));
    const Seg* full = w.segs + static_cast<size_t>(nc) * s.E;
    const float* wrow = rv.w_row;
    if (!rm) {
        MOE_TRY(launch_row_weights(s, rv.topk_w, rv.tim, w.wrow, err, st));
        wrow = w.wrow;
    }
    const int rows = static_cast<int>(rv.rows);

    GemmProblem g3{};
    g3.kind = G3_DH;
    g3.s = s;
    g3.rows = rows;
    g3.segs = full;
    g3.eti = rv.eti;
    g3.a_src = dy;
    g3.b_src0 = W2;
    g3.out0 = w.dH;
    g3.out1 = w.Ap;
    g3.aux0 = H_saved;
    g3.wrow = wrow;
    g3.dS_part = w.dS_part;
    g3.err = err;
    MOE_TRY(launch_gemm(g3, st));
    const int bn3 = gemm_bn(G3_DH, s);
    const int nparts = 2 * ((s.h + bn3 - 1) / bn3);  // G3's N tiles, two dS partial slots each
    if (rm)
        MOE_TRY(launch_router_dz_rows(s, rows, nparts, w.dS_part, rv.tok_off, rv.tok_rows,
                                      rv.w_row, dS, w.dz_row, err, st));
    else
        MOE_TRY(launch_router_dz(s, nparts, w.dS_part, rv.topk_w, rv.tim, dS, w.dz, w.dz_row, err,
                                 st));

    GemmProblem g4{};
    g4.kind = G4_DW2;
    g4.s = s;
    g4.rows = rows;
    g4.segs = full;
    g4.eti = rv.eti;
    g4.a_src = dy;
    g4.b_src0 = w.Ap;
    g4.out0 = dW2;
    g4.err = err;
    MOE_TRY(launch_gemm(g4, st));

    GemmProblem g5{};
    g5.kind = G5_DW13;
    g5.s = s;
    g5.rows = rows;
    g5.segs = full;
    g5.eti = rv.eti;
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
        g6.rows = rows;
        g6.segs = sc;
        g6.eti = rv.eti;
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
        const int t0 = pl.by_cols ? 0 : c * pl.tc;
        const int t1 = pl.by_cols ? s.T : std::min(s.T, t0 + pl.tc);
        if (rm)
            MOE_TRY(launch_combine_rows(s, t0, t1, g6.n_off, g6.n_cols, rv.tok_off, rv.tok_exp,
                                        rv.tok_rows, nullptr, sc, w.dXc,
                                        static_cast<__nv_bfloat16*>(dx), err, st, "dx_combine"));
        else
            MOE_TRY(launch_combine(s, t0, t1, g6.n_off, g6.n_cols, rv.ids, nullptr, rv.tim, sc,
                                   w.dXc, static_cast<__nv_bfloat16*>(dx), err, st, "dx_combine",
                                   !per_chunk));
    }
    // Router weight gradient dW_g = dz^T x: per-expert gathered sums while x
    // fits in L2; else the dense [dz_hi | dz_lo] operand, its tensor-core
    // product with x per token chunk and a fixed-order sum of the chunks.
    if (!dwg_tensor_cores(s)) {
        MOE_TRY(launch_router_dwg(s, static_cast<const __nv_bfloat16*>(x), rv.eti, rv.offsets,
                                  w.dz_row, w.dwg_part, dWg, err, st));
        return MOE_OK;
    }
    const DwgPlan dwp = dwg_plan(s);
    MOE_TRY(launch_dwg_operand(s, dwp, rows, rv.eti, rv.offsets, w.dz_row, w.dwg_B, w.dwg_iota,
                               w.dwg_segs, err, st));
    GemmProblem g7{};
    g7.kind = G7_DWG;
    g7.s = s;
    g7.segs = w.dwg_segs;
    g7.nseg = dwp.nchunks;
    g7.eti = w.dwg_iota;
    g7.a_src = x;
    g7.b_src0 = w.dwg_B;
    g7.out0 = w.dwg_part;
    g7.err = err;
    MOE_TRY(launch_gemm(g7, st));
    MOE_TRY(launch_dwg_reduce(s, dwp, w.dwg_part, dWg, err, st));
    return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

int moe_chunk_tokens(moe_shape s) {
    if (s.T < 1024) return std::max(1, s.T);
    // Two chunks when their buffer (T/2 tokens x K rows x d, bf16) is at most
    // 64 MiB, as for column passes; four otherwise.
    const long long half_bytes = static_cast<long long>(s.T) * s.K * s.d;
    const int n = half_bytes <= (64ll << 20) ? 2 : 4;
    return (s.T + n - 1) / n;
}

size_t moe_workspace_size(moe_shape s, int which) {
    if (check_shape(s) != MOE_OK) return 0;
    switch (which) {
        case MOE_WS_ROUTE: return router_ws_bytes(s);
        case MOE_WS_DISPATCH: return layout_dispatch(s, nullptr, nullptr);
        case MOE_WS_FORWARD: return layout_fwd(s, tk_of(s), false, nullptr, nullptr);
        case MOE_WS_BACKWARD: return layout_bwd(s, tk_of(s), false, nullptr, nullptr);
        case MOE_WS_FORWARD_SLOTWISE: return layout_fwd_slot(s, nullptr, nullptr);
    }
    return 0;
}

int moe_route(moe_shape s, const void* x, const float* Wg, const float* bias, float* logits,
              int32_t* topk_ids, float* topk_w, void* ws, size_t ws_bytes, void* stream) {
    int rc = check_shape(s);
    if (rc) return rc;
    if (!x || !Wg || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(Wg) || (logits && !aligned16(logits)))
        return MOE_ERR_MISALIGNED;
    const size_t need = router_ws_bytes(s);
    if (need > 0 && !ws) return MOE_ERR_INVALID_ARG;
    if (ws_bytes < need) return MOE_ERR_WORKSPACE_TOO_SMALL;
    if (need > 0 && !aligned16(ws)) return MOE_ERR_MISALIGNED;
    int* err = status_ptr();
    if (!err) return MOE_ERR_NO_DEVICE;
    MOE_TRY(launch_router(s, static_cast<const __nv_bfloat16*>(x), Wg, bias, logits, topk_ids,
                          topk_w, ws, err, static_cast<cudaStream_t>(stream)));
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
    if (!topk_ids || !topk_w || !tim) return MOE_ERR_INVALID_ARG;
    RouteView rv;
    rv.rows = tk_of(s);
    rv.eti = eti;
    rv.offsets = offsets;
    rv.ids = topk_ids;
    rv.topk_w = topk_w;
    rv.tim = tim;
    return forward_impl(s, rv, x, W1, W3, W2, y, H_saved, ws, ws_bytes, stream);
}

int moe_forward_rows(moe_shape s, int32_t rows_cap, const void* x, const void* W1,
                     const void* W3, const void* W2, const int32_t* eti, const int32_t* offsets,
                     const float* w_row, const int32_t* tok_off, const int32_t* tok_exp,
                     const int32_t* tok_rows, void* y, void* H_saved, void* ws, size_t ws_bytes,
                     void* stream) {
    int rc = check_shape(s);
    if (rc) return rc;
    if (rows_cap < 1 || static_cast<size_t>(rows_cap) > static_cast<size_t>(s.T) * s.E)
        return MOE_ERR_INVALID_ARG;
    if (!w_row || !tok_off || !tok_exp || !tok_rows) return MOE_ERR_INVALID_ARG;
    RouteView rv;
    rv.rows = static_cast<size_t>(rows_cap);
    rv.eti = eti;
    rv.offsets = offsets;
    rv.tok_off = tok_off;
    rv.tok_exp = tok_exp;
    rv.tok_rows = tok_rows;
    rv.w_row = w_row;
    return forward_impl(s, rv, x, W1, W3, W2, y, H_saved, ws, ws_bytes, stream);
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
    if (!topk_ids || !topk_w || !tim) return MOE_ERR_INVALID_ARG;
    RouteView rv;
    rv.rows = tk_of(s);
    rv.eti = eti;
    rv.offsets = offsets;
    rv.ids = topk_ids;
    rv.topk_w = topk_w;
    rv.tim = tim;
    return backward_impl(s, rv, dy, x, Wg, W1, W3, W2, H_saved, dx, dWg, dW1, dW3, dW2, dS, ws,
                         ws_bytes, stream);
}

int moe_backward_rows(moe_shape s, int32_t rows_cap, const void* dy, const void* x,
                      const float* Wg, const void* W1, const void* W3, const void* W2,
                      const int32_t* eti, const int32_t* offsets, const float* w_row,
                      const int32_t* tok_off, const int32_t* tok_exp, const int32_t* tok_rows,
                      const void* H_saved, void* dx, float* dWg, void* dW1, void* dW3, void* dW2,
                      float* dS_row, void* ws, size_t ws_bytes, void* stream) {
    int rc = check_shape(s);
    if (rc) return rc;
    if (rows_cap < 1 || static_cast<size_t>(rows_cap) > static_cast<size_t>(s.T) * s.E)
        return MOE_ERR_INVALID_ARG;
    if (!w_row || !tok_off || !tok_exp || !tok_rows) return MOE_ERR_INVALID_ARG;
    RouteView rv;
    rv.rows = static_cast<size_t>(rows_cap);
    rv.eti = eti;
    rv.offsets = offsets;
    rv.tok_off = tok_off;
    rv.tok_exp = tok_exp;
    rv.tok_rows = tok_rows;
    rv.w_row = w_row;
    return backward_impl(s, rv, dy, x, Wg, W1, W3, W2, H_saved, dx, dWg, dW1, dW3, dW2, dS_row,
                         ws, ws_bytes, stream);
}

size_t moe_rows_capacity(moe_shape s, int m_tile) {
    if (check_shape(s) != MOE_OK || m_tile < 1) return 0;
    return rows_capacity(s, m_tile);
}

size_t moe_workspace_size_rows(moe_shape s, int32_t rows_cap, int which) {
    if (check_shape(s) != MOE_OK || rows_cap < 1) return 0;
    switch (which) {
        case MOE_WS_FORWARD: return layout_fwd(s, static_cast<size_t>(rows_cap), true, nullptr, nullptr);
        case MOE_WS_BACKWARD: return layout_bwd(s, static_cast<size_t>(rows_cap), true, nullptr, nullptr);
    }
    return 0;
}

size_t moe_token_rounding_workspace_size(moe_shape s, int m_tile) {
    if (check_shape(s) != MOE_OK || m_tile < 1) return 0;
    return layout_rounding(s, m_tile, nullptr, nullptr);
}

int moe_token_rounding(moe_shape s, int m_tile, const float* logits, const int32_t* topk_ids,
                       const int32_t* tc_eti, const int32_t* tc_offsets, int32_t* eti,
                       int32_t* offsets, float* w_row, int32_t* tok_off, int32_t* tok_exp,
                       int32_t* tok_rows, void* ws, size_t ws_bytes, void* stream) {
    int rc = check_shape(s);
    if (rc) return rc;
    if (m_tile < 1 || m_tile > 4096) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!logits || !topk_ids || !tc_eti || !tc_offsets || !eti || !offsets || !w_row ||
        !tok_off || !tok_exp || !tok_rows || !ws)
        return MOE_ERR_INVALID_ARG;
    if (ws_bytes < layout_rounding(s, m_tile, nullptr, nullptr)) return MOE_ERR_WORKSPACE_TOO_SMALL;
    int* err = status_ptr();
    if (!err) return MOE_ERR_NO_DEVICE;
    TrScratch sc;
    layout_rounding(s, m_tile, ws, &sc);
    MOE_TRY(launch_token_rounding(s, m_tile, logits, topk_ids, tc_eti, tc_offsets, sc, eti,
                                  offsets, w_row, tok_off, tok_exp, tok_rows, err,
                                  static_cast<cudaStream_t>(stream)));
    return MOE_OK;
}

int moe_selftest_bounded_wait(uint64_t limit_ns, void* stream) {
    if (limit_ns == 0 || limit_ns > 10000000000ull) return MOE_ERR_INVALID_ARG;
    int* err = status_ptr();
    if (!err) return MOE_ERR_NO_DEVICE;
    MOE_TRY(launch_selftest_wait(limit_ns, err, static_cast<cudaStream_t>(stream)));
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
