// dispatch.cu — D1..D3: the dispatch index without a global sort and without
// contended atomics.
//
// Outputs (MoEBlaze paper notes 4.1, data structures of Figure 2):
//   expert_token_indices [TK]  token ids grouped by expert, ascending token
//                              order inside each expert
//   expert_token_offsets [E+1] exclusive prefix of the per-expert counts
//   token_index_map      [TK]  position of assignment (t, k), at t*K + k
// The build follows the three-step, atomic-free idea of MoEBlaze paper notes
// 4.2 (count per expert, prefix-sum into offsets, then conflict-free writes to
// precomputed positions), but replaces the dense L x E token map with
// per-block histograms:
//   D1  one CTA per block of 256 tokens. Each warp owns 32 tokens (one per
//       lane). For each slot k, __match_any_sync groups the lanes that chose
//       the same expert; the group's leader ORs the group's lane mask into the
//       warp's per-expert mask in shared memory (one writer per address, no
//       atomics). popc of the masks gives the block's per-expert counts.
//   D2  one CTA: exclusive scan of the counts over blocks for every expert
//       (block bases), then over experts (offsets).
//   D3  one CTA per block again: rebuilds the warp masks; the in-block rank of
//       (t, k) is the number of lower lanes in its warp's mask plus the counts
//       of earlier warps; position = offsets[e] + base[block][e] + rank. This
//       is exactly the order of a stable sort of the flattened ids by expert.
// Layers with E <= 16 and T*K <= 16384 take a single launch instead: one CTA
// stages the ids in shared memory and runs the same three steps with warps in
// place of blocks (dispatch_single_kernel below), which removes two launches
// and the round trips of the block histogram through global memory.
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kBlockTokens = 256;
constexpr int kWarps = kBlockTokens / 32;
constexpr int kMaxE = 256;
constexpr int kScanThreads = 1024;

// The kernels read ids[t * ld + k] for k < K: the whole routing (ld = K) or,
// with gridDim.y = K' and K = 1, one column per blockIdx.y (the slot-wise
// lists of the fused combine); blockIdx.y also selects that slot's output
// arrays.
//
// Builds masks[w][e] (bit l set when lane l of warp w chose expert e) for the
// block `blk`. Flags ids out of range or repeated within a token.
__device__ __forceinline__ void build_masks(const int32_t* __restrict__ ids, int ld, int T, int E,
                                            int K, int blk, uint32_t (*masks)[kMaxE], int* err,
                                            int (&my_e)[8]) {
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    for (int i = threadIdx.x; i < kWarps * kMaxE; i += blockDim.x) (&masks[0][0])[i] = 0u;
    __syncthreads();
    const int t = blk * kBlockTokens + warp * 32 + lane;
    const bool valid = t < T;
    bool bad = false;
    for (int k = 0; k < K; ++k) {
        int e = valid ? ids[static_cast<size_t>(t) * ld + k] : -1;
        if (valid) {
            bool dup = false;
            for (int j = 0; j < k; ++j) dup |= (my_e[j] == e);
            if (e < 0 || e >= E || dup) {
                bad = true;
                e = -1;
            }
        }
        my_e[k] = e;
        const uint32_t m = __match_any_sync(0xffffffffu, e);
        const int leader = __ffs(m) - 1;
        if (lane == leader && e >= 0) masks[warp][e] |= m;
        __syncwarp();
    }
    if (bad) raise_error(err, MOE_ERR_BAD_EXPERT_ID);
    __syncthreads();
}

__global__ void __launch_bounds__(kBlockTokens)
dispatch_hist_kernel(const int32_t* __restrict__ ids, int ld, int T, int E, int K,
                     int32_t* __restrict__ hist, int* err) {
    pdl_wait();
    pdl_trigger();
    if (has_error(err)) return;
    __shared__ uint32_t masks[kWarps][kMaxE];
    int my_e[8];
    ids += blockIdx.y;
    hist += static_cast<size_t>(blockIdx.y) * gridDim.x * E;
    build_masks(ids, ld, T, E, K, blockIdx.x, masks, err, my_e);
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int c = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) c += __popc(masks[w][e]);
        hist[static_cast<size_t>(blockIdx.x) * E + e] = c;
    }
}

// hist [nblk][E] -> exclusive scan over blocks in place (block bases), and
// offsets [E+1]. Thread (part p, expert e) scans a contiguous run of blocks.
__global__ void __launch_bounds__(kScanThreads)
dispatch_scan_kernel(int32_t* __restrict__ hist, int nblk, int E, int32_t* __restrict__ offsets,
                     int* err) {
    pdl_wait();
    pdl_trigger();
    if (has_error(err)) return;
    hist += static_cast<size_t>(blockIdx.x) * nblk * E;  // one CTA per slot view
    offsets += static_cast<size_t>(blockIdx.x) * (E + 1);
    __shared__ int32_t part_sum[kScanThreads];
    __shared__ int32_t exp_tot[kMaxE];
    const int P = kScanThreads / E;  // parts per expert (E <= 256 -> P >= 4)
    const int e = threadIdx.x % E;
    const int p = threadIdx.x / E;
    const bool active = p < P;
    const int per = (nblk + P - 1) / P;
    const int b0 = min(nblk, p * per);
    const int b1 = min(nblk, b0 + per);
    int32_t s = 0;
    if (active)
        for (int b = b0; b < b1; ++b) s += hist[static_cast<size_t>(b) * E + e];
    part_sum[threadIdx.x] = active ? s : 0;
    __syncthreads();
    if (threadIdx.x < E) {
        int32_t run = 0;
        for (int q = 0; q < P; ++q) {
            const int32_t v = part_sum[q * E + threadIdx.x];
            part_sum[q * E + threadIdx.x] = run;
            run += v;
        }
        exp_tot[threadIdx.x] = run;
    }
    __syncthreads();
    if (active) {
        int32_t run = part_sum[threadIdx.x];
        for (int b = b0; b < b1; ++b) {
            const size_t i = static_cast<size_t>(b) * E + e;
            const int32_t v = hist[i];
            hist[i] = run;
            run += v;
        }
    }
    if (threadIdx.x == 0) {
        int32_t run = 0;
        for (int q = 0; q < E; ++q) {
            offsets[q] = run;
            run += exp_tot[q];
        }
        offsets[E] = run;
    }
}

__global__ void __launch_bounds__(kBlockTokens)
dispatch_scatter_kernel(const int32_t* __restrict__ ids, int ld, int T, int E, int K,
                        const int32_t* __restrict__ base, const int32_t* __restrict__ offsets,
                        int32_t* __restrict__ eti, int32_t* __restrict__ tim, int* err) {
    pdl_wait();
    pdl_trigger();
    if (has_error(err)) return;
    __shared__ uint32_t masks[kWarps][kMaxE];
    __shared__ int32_t wbase[kWarps][kMaxE];
    int my_e[8];
    const size_t view = blockIdx.y;
    ids += view;
    base += view * gridDim.x * E;
    offsets += view * (E + 1);
    eti += view * T * K;
    tim += view * T * K;
    build_masks(ids, ld, T, E, K, blockIdx.x, masks, err, my_e);
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int32_t run = offsets[e] + base[static_cast<size_t>(blockIdx.x) * E + e];
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            wbase[w][e] = run;
            run += __popc(masks[w][e]);
        }
    }
    __syncthreads();
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int t = blockIdx.x * kBlockTokens + warp * 32 + lane;
    if (t >= T) return;
    const uint32_t lt = (1u << lane) - 1u;
    for (int k = 0; k < K; ++k) {
        const int e = my_e[k];
        if (e < 0) continue;
        const int32_t pos = wbase[warp][e] + __popc(masks[warp][e] & lt);
        eti[pos] = t;
        tim[static_cast<size_t>(t) * K + k] = pos;
    }
}

// ---------------------------------------------------------------------------
// Single-CTA build (one launch) for layers whose T*K ids fit in one CTA's
// shared memory: the same lane masks, scans and stable positions as D1..D3,
// with warps in place of blocks. The ids are staged in shared memory; warp w
// owns the contiguous tokens [w*Tw, (w+1)*Tw) (Tw a multiple of 32) and walks
// them 32 at a time.
//   pass 1  per round and slot, __match_any_sync groups the lanes that chose
//           the same expert and the group's leader adds the group's size to
//           cnt[w][e] (only warp w writes row w: no atomics);
//   scan    cnt[w][e] becomes the exclusive prefix over warps of expert e, and
//           the expert totals are scanned into offsets;
//   pass 2  per round, the slot groups' leaders OR their lane masks into
//           msk[w][e]; (t, k) lands at offsets[e] + cnt[w][e] + the number of
//           lower lanes in msk[w][e]; then cnt[w][e] advances by the round's
//           group sizes and msk[w][e] is cleared by the lanes that used it.
// Token order inside an expert is warp order, then round, then lane: ascending
// token, so the index equals that of a stable sort of the flattened ids.
constexpr int kSingleThreads = 1024;
constexpr int kSingleWarps = kSingleThreads / 32;
constexpr int kSingleMaxTK = 16384;
constexpr int kSingleMaxE = 16;  // default single-CTA builds: E <= 16
constexpr size_t kSingleMaxSmem = 200 * 1024;

size_t single_smem_bytes(int T, int E, int K) {
    const size_t tk4 = (static_cast<size_t>(T) * K + 3) / 4 * 4;
    return 4 * (tk4 + 2 * static_cast<size_t>(kSingleWarps) * E + (E + 1) + kSingleWarps + E);
}

template <int K>
__global__ void __launch_bounds__(kSingleThreads, 1)
dispatch_single_kernel(const int32_t* __restrict__ ids, int T, int E, int32_t* __restrict__ offsets,
                       int32_t* __restrict__ eti, int32_t* __restrict__ tim, int* err) {
    pdl_wait();
    pdl_trigger();
    if (has_error(err)) return;
    extern __shared__ int32_t s_dyn[];
    const int TK = T * K;
    int32_t* s_ids = s_dyn;                                         // [TK]
    int32_t* cnt = s_ids + (TK + 3) / 4 * 4;                        // [warps][E]
    uint32_t* msk = reinterpret_cast<uint32_t*>(cnt + kSingleWarps * E);  // [warps][E]
    int32_t* s_off = reinterpret_cast<int32_t*>(msk + kSingleWarps * E);  // [E + 1]
    int32_t* wsum = s_off + E + 1;                                  // [warps]
    int32_t* s_tot = wsum + kSingleWarps;                           // [E]
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    if ((reinterpret_cast<uintptr_t>(ids) & 15u) == 0) {  // 16-byte pieces, then the tail
        const int n4 = TK / 4;
        const int4* src = reinterpret_cast<const int4*>(ids);
        int4* dst = reinterpret_cast<int4*>(s_ids);
#pragma unroll 4
        for (int i = tid; i < n4; i += kSingleThreads) dst[i] = src[i];
        for (int i = 4 * n4 + tid; i < TK; i += kSingleThreads) s_ids[i] = ids[i];
    } else {
#pragma unroll 4
        for (int i = tid; i < TK; i += kSingleThreads) s_ids[i] = ids[i];
    }
    for (int i = tid; i < 2 * kSingleWarps * E; i += kSingleThreads) cnt[i] = 0;
    __syncthreads();

    const int Tw = ((T + kSingleWarps - 1) / kSingleWarps + 31) / 32 * 32;
    const int tbeg = warp * Tw;
    const int tend = min(T, tbeg + Tw);
    int32_t* my_cnt = cnt + warp * E;
    uint32_t* my_msk = msk + warp * E;
    // Expert of (t, k) for a live lane, or -1 for a lane past the end and for an
    // id out of range or repeated within the token (both passes drop the same
    // entries, so every position stays inside [0, TK)).
    auto load_slots = [&](int t, int (&e)[K]) -> bool {
        bool bad = false;
#pragma unroll
        for (int k = 0; k < K; ++k) {
            int v = t < tend ? s_ids[t * K + k] : -1;
            if (t < tend) {
                bool dup = false;
#pragma unroll
                for (int j = 0; j < k; ++j) dup |= (e[j] == v);
                if (v < 0 || v >= E || dup) {
                    bad = true;
                    v = -1;
                }
            }
            e[k] = v;
        }
        return bad;
    };

    bool bad = false;
    for (int t0 = tbeg; t0 < tend; t0 += 32) {  // warp-uniform
        int e[K];
        bad |= load_slots(t0 + lane, e);
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const uint32_t m = __match_any_sync(0xffffffffu, e[k]);
            if (e[k] >= 0 && lane == __ffs(m) - 1) my_cnt[e[k]] += __popc(m);
            __syncwarp();
        }
    }
    if (bad) raise_error(err, MOE_ERR_BAD_EXPERT_ID);
    __syncthreads();

    // Exclusive scan over warps per expert (warp e % 32 scans expert e with one
    // lane per warp of counts), then over experts.
    for (int e = warp; e < E; e += kSingleWarps) {
        const int32_t v = cnt[lane * E + e];
        int32_t run = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t u = __shfl_up_sync(0xffffffffu, run, o);
            if (lane >= o) run += u;
        }
        cnt[lane * E + e] = run - v;
        if (lane == 31) s_tot[e] = run;
    }
    __syncthreads();
    const int32_t tot = tid < E ? s_tot[tid] : 0;
    const int scan_warps = (E + 31) / 32;
    int32_t inc = tot;
    if (warp < scan_warps) {
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t v = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += v;
        }
        if (lane == 31) wsum[warp] = inc;
    }
    __syncthreads();
    if (tid < E) {
        int32_t pre = 0;
        for (int w = 0; w < warp; ++w) pre += wsum[w];
        const int32_t excl = pre + inc - tot;
        s_off[tid] = excl;
        offsets[tid] = excl;
        if (tid == E - 1) {
            s_off[E] = excl + tot;
            offsets[E] = excl + tot;
        }
    }
    __syncthreads();

    const uint32_t lt = (1u << lane) - 1u;
    for (int t0 = tbeg; t0 < tend; t0 += 32) {
        const int t = t0 + lane;
        int e[K];
        uint32_t m[K];
        load_slots(t, e);
#pragma unroll
        for (int k = 0; k < K; ++k) {
            m[k] = __match_any_sync(0xffffffffu, e[k]);
            if (e[k] >= 0 && lane == __ffs(m[k]) - 1) my_msk[e[k]] |= m[k];
            __syncwarp();
        }
#pragma unroll
        for (int k = 0; k < K; ++k) {
            if (e[k] < 0) continue;
            const int32_t pos = s_off[e[k]] + my_cnt[e[k]] + __popc(my_msk[e[k]] & lt);
            eti[pos] = t;
            tim[static_cast<size_t>(t) * K + k] = pos;
        }
        __syncwarp();
#pragma unroll
        for (int k = 0; k < K; ++k) {
            if (e[k] >= 0 && lane == __ffs(m[k]) - 1) {
                my_cnt[e[k]] += __popc(m[k]);
                my_msk[e[k]] = 0u;
            }
            __syncwarp();
        }
    }
}

// Which build a shape takes: the single CTA while E <= 16, T*K <= 16384 and its
// shared memory fits, else D1..D3. Measured on GB300 (20 calls replayed from a
// CUDA graph): 8.3 us against 9.2 us for D1..D3 at T = 4096, E = 8, K = 2, but
// 52-87 us against 14-18 us at E = 64-128, where __match_any_sync meets up to
// 32 distinct experts per warp and one SM does all the work; under ncu the
// single CTA took 10 us at T*K = 8192 and 27 us at T*K = 32768 (E = 8), where
// the three launches take about 18 us.
// MOE_DISPATCH=single|blocks forces one (single only where it fits); read at
// every call.
bool use_single(int T, int E, int K) {
    const size_t smem = single_smem_bytes(T, E, K);
    const bool fits = smem <= kSingleMaxSmem;
    const char* f = std::getenv("MOE_DISPATCH");
    if (f != nullptr && std::strcmp(f, "blocks") == 0) return false;
    if (f != nullptr && std::strcmp(f, "single") == 0) return fits;
    return fits && E <= kSingleMaxE && static_cast<long long>(T) * K <= kSingleMaxTK;
}

template <int K>
cudaError_t launch_single_k(int T, int E, const int32_t* ids, int32_t* eti, int32_t* offsets,
                            int32_t* tim, int* err, cudaStream_t st) {
    const size_t smem = single_smem_bytes(T, E, K);
    cudaError_t e = cudaFuncSetAttribute(dispatch_single_kernel<K>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    LaunchScope ls("dispatch_single", st);
    launch_k(dispatch_single_kernel<K>, dim3(1), dim3(kSingleThreads), smem, st, ids, T, E, offsets, eti, tim, err);
    return cudaGetLastError();
}

cudaError_t launch_single(int T, int E, int K, const int32_t* ids, int32_t* eti, int32_t* offsets,
                          int32_t* tim, int* err, cudaStream_t st) {
    switch (K) {
        case 1: return launch_single_k<1>(T, E, ids, eti, offsets, tim, err, st);
        case 2: return launch_single_k<2>(T, E, ids, eti, offsets, tim, err, st);
        case 3: return launch_single_k<3>(T, E, ids, eti, offsets, tim, err, st);
        case 4: return launch_single_k<4>(T, E, ids, eti, offsets, tim, err, st);
        case 5: return launch_single_k<5>(T, E, ids, eti, offsets, tim, err, st);
        case 6: return launch_single_k<6>(T, E, ids, eti, offsets, tim, err, st);
        case 7: return launch_single_k<7>(T, E, ids, eti, offsets, tim, err, st);
        case 8: return launch_single_k<8>(T, E, ids, eti, offsets, tim, err, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

int dispatch_block_tokens() { return kBlockTokens; }

namespace {
cudaError_t launch_views(int T, int E, int K, int ld, int views, const int32_t* ids,
                         int32_t* eti, int32_t* offsets, int32_t* tim, int32_t* hist, int* err,
                         cudaStream_t st, const char* n1, const char* n2, const char* n3) {
    const int nblk = (T + kBlockTokens - 1) / kBlockTokens;
    {
        LaunchScope ls(n1, st);
        launch_k(dispatch_hist_kernel, dim3(dim3(nblk, views)), dim3(kBlockTokens), 0, st, ids, ld, T, E, K, hist,
                                                                         err);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    {
        LaunchScope ls(n2, st);
        launch_k(dispatch_scan_kernel, dim3(views), dim3(kScanThreads), 0, st, hist, nblk, E, offsets, err);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    {
        LaunchScope ls(n3, st);
        launch_k(dispatch_scatter_kernel, dim3(dim3(nblk, views)), dim3(kBlockTokens), 0, st, 
            ids, ld, T, E, K, hist, offsets, eti, tim, err);
    }
    return cudaGetLastError();
}
}  // namespace

cudaError_t launch_dispatch(const moe_shape& s, const int32_t* ids, int32_t* eti,
                            int32_t* offsets, int32_t* tim, int32_t* hist, int* err,
                            cudaStream_t st) {
    if (use_single(s.T, s.E, s.K)) return launch_single(s.T, s.E, s.K, ids, eti, offsets, tim, err, st);
    return launch_views(s.T, s.E, s.K, s.K, 1, ids, eti, offsets, tim, hist, err, st,
                        "dispatch_hist", "dispatch_scan", "dispatch_scatter");
}

cudaError_t launch_slot_dispatch(const moe_shape& s, const int32_t* ids, int32_t* eti_k,
                                 int32_t* offsets_k, int32_t* tim_k, int32_t* hist, int* err,
                                 cudaStream_t st) {
    return launch_views(s.T, s.E, 1, s.K, s.K, ids, eti_k, offsets_k, tim_k, hist, err, st,
                        "slot_hist", "slot_scan", "slot_scatter");
}

}  // namespace moe

// ---------------------------------------------------------------------------
// Allocation-free dispatch build: the per-block histogram lives in a
// file-scope device array instead of the caller's workspace. In host code the
// array's name is only a host-side stand-in; its device address is looked up
// once per device (with that device current) and passed to the kernels.
namespace moe {
namespace {

static __device__ __align__(256) int32_t g_noalloc_hist[MOE_NOALLOC_DISPATCH_MAX_ENTRIES];

constexpr int kNoAllocMaxDevices = 64;
int32_t* g_noalloc_hist_ptr[kNoAllocMaxDevices] = {};
std::mutex g_noalloc_mu;

// Device address of g_noalloc_hist on the current device (set up on first use).
cudaError_t noalloc_hist_ptr(int32_t** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kNoAllocMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (g_noalloc_hist_ptr[dev] == nullptr) {
        int32_t* ptr = nullptr;
        e = cudaGetSymbolAddress(reinterpret_cast<void**>(&ptr), g_noalloc_hist);
        if (e != cudaSuccess) return e;
        g_noalloc_hist_ptr[dev] = ptr;
    }
    *out = g_noalloc_hist_ptr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace moe

extern "C" int moe_build_dispatch_noalloc(moe_shape s, const int32_t* topk_ids, int32_t* eti,
                                          int32_t* offsets, int32_t* tim, void* stream) {
    using namespace moe;
    // The same host checks, in the same order, as moe_build_dispatch.
    const int rc = check_shape_status(s);
    if (rc != MOE_OK) return rc;
    if (!topk_ids || !eti || !offsets || !tim) return MOE_ERR_INVALID_ARG;
    const long long nblk = (static_cast<long long>(s.T) + kBlockTokens - 1) / kBlockTokens;
    if (nblk * s.E > MOE_NOALLOC_DISPATCH_MAX_ENTRIES) return MOE_ERR_STATIC_SCRATCH_LIMIT;
    int* err = device_status_word();
    if (!err) return MOE_ERR_NO_DEVICE;
    int32_t* hist = nullptr;
    cudaError_t e = noalloc_hist_ptr(&hist);
    if (e != cudaSuccess) return cuda_error_status(e);
    // Every histogram entry the kernels read is written earlier in the same
    // call (one entry per block and expert), so the array is not cleared.
    e = launch_dispatch(s, topk_ids, eti, offsets, tim, hist, err,
                        static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_error_status(e);
    return MOE_OK;
}
