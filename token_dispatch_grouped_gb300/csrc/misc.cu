// misc.cu — the memory-bound kernels around the expert GEMMs.
//
//   chunk_search    per token chunk c and expert e, the sub-range of e's rows
//                   whose tokens fall in the chunk (stable order makes it one
//                   contiguous range);
//   chunk_pack      where each range lands in the chunk buffer, and the
//                   whole-row-space segments.
//   row_weights     w_row[token_index_map[t*K+k]] = topk_w[t,k].
//   combine   (C1)  y_t = sum_k w_{t,k} Y[row(t,k)], fp32, k ascending, one bf16
//                   rounding. MoEBlaze paper notes 2.3; SonicMoE 3.4.1 (O_t).
//   router_dz (R2a) dS_{t,k} = sum over N-tiles of the partial <dA'_r, A_r>;
//                   dz_k = w_k (dS_k - sum_j w_j dS_j): the Jacobian of the
//                   softmax over the chosen logits applied to dS.
//   combine also serves C2 (weights 1): dx_t = sum_k dX~'[row(t,k)], fp32, k
//                   ascending, where dX~' already holds the router term
//                   dz_{t,k} W_g[e_{t,k}] (added in the dX GEMM's epilogue).
//                   MoEBlaze paper notes 3.2 (token gradient accumulation over
//                   the K routed rows).
//   router_dwg(R2b) dW_g = dz^T x, two ways. Per-expert sums over the
//                   expert's rows (x rows gathered, partials over 32 row parts,
//                   then a fixed-order sum) while x fits in L2 (T*d*2 <= 64 MiB).
//                   Larger layers: on the tensor cores, dz split into two
//                   bf16 parts (hi = bf16(dz), lo = bf16(dz - hi), together
//                   about 16 mantissa bits) scattered into a dense operand
//                   B = [dz_hi | dz_lo] [T, 2 e_pad] (zeros where a token did
//                   not choose the expert); the grouped GEMM kind G7_DWG forms
//                   x^T B per token chunk in fp32, and dwg_reduce adds the chunk
//                   partials and the two parts in a fixed order. x is read once
//                   (a per-expert gather would read each token row K times).
// All sums run in a fixed order, so results are bit-reproducible.
#include <algorithm>

#include "common.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

// First index in [lo, hi) with a[i] >= key (hi if none), a sorted ascending.
// The warp probes 32 evenly spaced positions per round and keeps the gap where
// the predicate a[i] < key turns false: about log32(hi - lo) dependent loads.
// Every lane returns the result.
__device__ __forceinline__ int warp_lower_bound(const int32_t* __restrict__ a, int lo, int hi,
                                                int key, int lane) {
    while (hi - lo > 32) {
        const int step = (hi - lo + 31) / 32;
        const int pos = min(hi - 1, lo + (lane + 1) * step - 1);
        const unsigned below = __ballot_sync(0xffffffffu, a[pos] < key);
        const int cnt = __popc(below);  // the predicate holds on a prefix of the probes
        const int nlo = lo + cnt * step;
        hi = min(hi, lo + (cnt + 1) * step);
        lo = min(nlo, hi);
    }
    const bool below = lo + lane < hi && a[lo + lane] < key;
    return lo + __popc(__ballot_sync(0xffffffffu, below));
}

// Token-chunk ranges: one warp per (chunk c < nchunks, expert e) finds the
// rows of e whose tokens lie in [c * chunk_tokens, (c + 1) * chunk_tokens).
__global__ void chunk_search_kernel(const int32_t* __restrict__ eti,
                                    const int32_t* __restrict__ offsets, int E, int T,
                                    int chunk_tokens, int nchunks, Seg* __restrict__ segs,
                                    int* err) {
    pdl_wait();
    pdl_trigger();
    if (has_error(err)) return;
    const int lane = threadIdx.x & 31;
    const int item = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (item >= nchunks * E) return;  // warp-uniform
    const int c = item / E, e = item % E;
    const int o0 = offsets[e], o1 = offsets[e + 1];
    const int ta = c * chunk_tokens;
    const int tb = min(T, ta + chunk_tokens);
    const int lo = warp_lower_bound(eti, o0, o1, ta, lane);
    const int hi = warp_lower_bound(eti, lo, o1, tb, lane);
    if (lane == 0) segs[static_cast<size_t>(c) * E + e] = Seg{lo, hi, 0, 0};
}

// grid = nchunks + 1, block = 256. Block c < nchunks packs the chunk's ranges
// expert after expert into the chunk buffer (out = rows of the experts before
// e); the last block writes the whole-row-space segments {o_e, o_e+1, o_e}.
__global__ void chunk_pack_kernel(const int32_t* __restrict__ offsets, int E, int nchunks,
                                  Seg* __restrict__ segs, int* err) {
    pdl_wait();
    pdl_trigger();
    if (has_error(err)) return;
    __shared__ int cnt[256];
    const int c = blockIdx.x;
    const int e = threadIdx.x;
    Seg sg{0, 0, 0, 0};
    if (e < E) {
        if (c == nchunks) sg = Seg{offsets[e], offsets[e + 1], offsets[e], 0};
        else sg = segs[static_cast<size_t>(c) * E + e];
    }
    cnt[e] = sg.hi - sg.lo;
    __syncthreads();
    if (e < E) {
        if (c != nchunks) {
            int out = 0;
            for (int q = 0; q < e; ++q) out += cnt[q];
            sg.out = out;
        }
        segs[static_cast<size_t>(c) * E + e] = sg;
    }
}

__global__ void row_weights_kernel(const float* __restrict__ topk_w,
                                   const int32_t* __restrict__ tim, int TK,
                                   float* __restrict__ wrow, int* err) {
    pdl_wait();
    pdl_trigger();
    if (has_error(err)) return;
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < TK) wrow[tim[i]] = topk_w[i];
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float (&f)[8]) {
    const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float2 p = __bfloat1622float2(b[j]);
        f[2 * j] = p.x;
        f[2 * j + 1] = p.y;
    }
}

__device__ __forceinline__ uint4 f32_to_bf16x8(const float (&f)[8]) {
    uint4 v;
    __nv_bfloat162* b = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
    for (int j = 0; j < 4; ++j) b[j] = __floats2bfloat162_rn(f[2 * j], f[2 * j + 1]);
    return v;
}

constexpr int kCombThreads = 256;   // 8 warps; one warp per token at a time
constexpr int kCombWarps = kCombThreads / 32;
// A lane loads the K rows' pieces of U = max(1, 8 / K) 8-column pieces at once:
// about 8 16-byte loads (4 KB per warp) in flight before any arithmetic. (16
// loads per lane measured slower on GB300: the extra registers cut the resident
// CTAs below one wave of a 4096-token pass.)
template <int K>
constexpr int comb_u() { return K >= 8 ? 1 : 8 / K; }

// Weighted combine of one chunk. Each warp takes a token (grid-stride), reads
// its K (position, weight) pairs once, then every lane sums 8-column pieces of
// the K expert-output rows in slot order and stores bf16; a lane loads the
// pieces of all K rows for U column pieces before any arithmetic.
// The chunk buffer's rows hold columns [c0, c0 + nc) of the expert outputs.
// DIRECT (column passes and single passes: the buffer holds every routed row
// in the expert-sorted order): row(t, k) = token_index_map[t*K+k]. Otherwise
// (token chunks) row(t, k) = seg[e].out + (token_index_map[t*K+k] - seg[e].lo)
// with e = ids[t*K+k].
// A work item is (token, column slice): the 2^cs_log2 slices of a token split
// its nc columns evenly, so passes with few tokens still keep enough warps in
// flight.
template <int K, bool DIRECT>
__global__ void __launch_bounds__(kCombThreads)
combine_kernel(int t0, int t1, int c0, int nc, int d, int cs_log2, const int32_t* __restrict__ ids,
               const float* __restrict__ topk_w, const int32_t* __restrict__ tim,
               const Seg* __restrict__ seg, const __nv_bfloat16* __restrict__ Yc,
               __nv_bfloat16* __restrict__ y, int* err) {
    pdl_wait();
    pdl_trigger();
    if (has_error(err)) return;
    const int lane = threadIdx.x & 31;
    const int ncs = nc >> cs_log2;  // columns per slice
    const int items = (t1 - t0) << cs_log2;
    for (int it = blockIdx.x * kCombWarps + threadIdx.x / 32; it < items;
         it += gridDim.x * kCombWarps) {
        const int t = t0 + (it >> cs_log2);
        const int cbeg = (it & ((1 << cs_log2) - 1)) * ncs;  // first column of the slice
        size_t off = 0;
        float wl = 0.f;
        if (lane < K) {
            const size_t i = static_cast<size_t>(t) * K + lane;
            int row = tim[i];
            if constexpr (!DIRECT) {
                const Seg sg = seg[ids[i]];
                row = sg.out + (row - sg.lo);
            }
            off = static_cast<size_t>(row) * nc;
            wl = topk_w != nullptr ? topk_w[i] : 1.f;
        }
        constexpr int U = comb_u<K>();
        size_t ok[K];
        float w[K];
#pragma unroll
        for (int k = 0; k < K; ++k) {
            ok[k] = __shfl_sync(0xffffffffu, off, k);
            w[k] = __shfl_sync(0xffffffffu, wl, k);
        }
        const int cend = cbeg + ncs;
        for (int cb = cbeg + lane * 8; cb < cend; cb += 32 * 8 * U) {
            uint4 v[K][U];
#pragma unroll
            for (int k = 0; k < K; ++k)
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int c = cb + u * 256;
                    v[k][u] = c < cend ? *reinterpret_cast<const uint4*>(Yc + ok[k] + c)
                                       : make_uint4(0, 0, 0, 0);
                }
            float acc[U][8];
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[u][j] = 0.f;
#pragma unroll
            for (int k = 0; k < K; ++k)
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    float f[8];
                    bf16x8_to_f32(v[k][u], f);
#pragma unroll
                    for (int j = 0; j < 8; ++j) acc[u][j] = fmaf(w[k], f[j], acc[u][j]);
                }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = cb + u * 256;
                if (c < cend)
                    *reinterpret_cast<uint4*>(y + static_cast<size_t>(t) * d + c0 + c) =
                        f32_to_bf16x8(acc[u]);
            }
        }
    }
}

// One lane per (t, k): lanes K * j .. K * j + K - 1 of a warp hold token
// j's slots (32 / K tokens per warp). A lane sums its routed row's partials
// over the N tiles in order (loads issued 16 ahead), the token's lanes share
// sum_j w_j dS_j through shuffles in slot order, and each lane writes its dS,
// dz and the dz of its row.
__global__ void __launch_bounds__(256)
router_dz_kernel(int T, int K, int TK, int nparts, const float* __restrict__ dS_part,
                 const float* __restrict__ topk_w, const int32_t* __restrict__ tim,
                 float* __restrict__ dS, float* __restrict__ dz, float* __restrict__ dz_row,
                 int* err) {
    pdl_wait();
    pdl_trigger();
    if (has_error(err)) return;
    const int lane = threadIdx.x & 31;
    const int tpw = 32 / K;  // tokens per warp
    const int gw = static_cast<int>((static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5);
    const int t = gw * tpw + lane / K;
    const int k = lane % K;
    const bool active = lane < tpw * K && t < T;
    const size_t i = static_cast<size_t>(t) * K + k;
    float acc = 0.f, w = 0.f;
    int r = 0;
    if (active) {
        r = tim[i];
        w = topk_w[i];
        int p = 0;
        for (; p + 16 <= nparts; p += 16) {
            float v[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) v[u] = dS_part[static_cast<size_t>(p + u) * TK + r];
#pragma unroll
            for (int u = 0; u < 16; ++u) acc += v[u];
        }
        for (; p < nparts; ++p) acc += dS_part[static_cast<size_t>(p) * TK + r];
    }
    const int base = (lane / K) * K;
    float sbar = 0.f;
    for (int j = 0; j < K; ++j) {
        const float sj = __shfl_sync(0xffffffffu, acc, base + j);
        const float wj = __shfl_sync(0xffffffffu, w, base + j);
        sbar = fmaf(wj, sj, sbar);
    }
    if (active) {
        const float z = w * (acc - sbar);
        dS[i] = acc;
        dz[i] = z;
        dz_row[r] = z;
    }
}

// Combine over a row-format routing: warp per token, the token's rows in CSR
// order (ascending expert), summed in that order in fp32, one bf16 rounding;
// the weight of routed row r is w_row[r] (nullptr: 1).
// Chunk-buffer row of routed row r of expert e: seg[e].out + (r - seg[e].lo).
__global__ void __launch_bounds__(kCombThreads)
combine_rows_kernel(int t0, int t1, int c0, int nc, int d, const int32_t* __restrict__ tok_off,
                    const int32_t* __restrict__ tok_exp, const int32_t* __restrict__ tok_rows,
                    const float* __restrict__ w_row, const Seg* __restrict__ seg,
                    const __nv_bfloat16* __restrict__ Yc, __nv_bfloat16* __restrict__ y, int* err) {
    pdl_wait();
    pdl_trigger();
    if (has_error(err)) return;
    const int lane = threadIdx.x & 31;
    constexpr int U = 4;
    for (int t = t0 + blockIdx.x * kCombWarps + threadIdx.x / 32; t < t1;
         t += gridDim.x * kCombWarps) {
        const int b0 = tok_off[t], b1 = tok_off[t + 1];
        for (int cb = lane * 8; cb < nc; cb += 32 * 8 * U) {
            float acc[U][8];
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[u][j] = 0.f;
            for (int g0 = b0; g0 < b1; g0 += 32) {  // groups of 32 rows of this token
                size_t off = 0;
                float wl = 0.f;
                if (g0 + lane < b1) {
                    const int i = g0 + lane;
                    const Seg sg = seg[tok_exp[i]];
                    const int r = tok_rows[i];
                    off = static_cast<size_t>(sg.out + (r - sg.lo)) * nc;
                    wl = w_row != nullptr ? w_row[r] : 1.f;
                }
                const int n = min(32, b1 - g0);
                for (int q = 0; q < n; ++q) {
                    const size_t ok = __shfl_sync(0xffffffffu, off, q);
                    const float w = __shfl_sync(0xffffffffu, wl, q);
                    uint4 v[U];
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const int c = cb + u * 256;
                        v[u] = c < nc ? *reinterpret_cast<const uint4*>(Yc + ok + c)
                                      : make_uint4(0, 0, 0, 0);
                    }
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        float f[8];
                        bf16x8_to_f32(v[u], f);
#pragma unroll
                        for (int j = 0; j < 8; ++j) acc[u][j] = fmaf(w, f[j], acc[u][j]);
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = cb + u * 256;
                if (c < nc)
                    *reinterpret_cast<uint4*>(y + static_cast<size_t>(t) * d + c0 + c) =
                        f32_to_bf16x8(acc[u]);
            }
        }
    }
}

// Router gradient over a row-format routing: thread per token.
__global__ void router_dz_rows_kernel(int T, int rows_cap, int nparts,
                                      const float* __restrict__ dS_part,
                                      const int32_t* __restrict__ tok_off,
                                      const int32_t* __restrict__ tok_rows,
                                      const float* __restrict__ w_row, float* __restrict__ dS_row,
                                      float* __restrict__ dz_row, int* err) {
    pdl_wait();
    pdl_trigger();
    if (has_error(err)) return;
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= T) return;
    const int b0 = tok_off[t], b1 = tok_off[t + 1];
    float sbar = 0.f;
    for (int i = b0; i < b1; ++i) {
        const int r = tok_rows[i];
        float acc = 0.f;
        for (int p = 0; p < nparts; ++p) acc += dS_part[static_cast<size_t>(p) * rows_cap + r];
        dS_row[r] = acc;
        sbar = fmaf(w_row[r], acc, sbar);
    }
    for (int i = b0; i < b1; ++i) {
        const int r = tok_rows[i];
        dz_row[r] = w_row[r] * (dS_row[r] - sbar);
    }
}

constexpr int kDwgCols = 2048;     // columns per CTA (256 threads x 8)

// dW_g[e] = sum over expert e's rows r of dz_row[r] * x[eti[r]] (the router
// gradient dz^T x, with dz non-zero only at the chosen experts). grid =
// (E, ceil(d / 2048), P): CTA (e, cb, z) sums the z-th of P equal parts of
// e's rows for up to 2048 columns, 8 per thread. When d < 2048 the CTA's
// threads form G = 256 / (d / 8) groups, group g taking rows r0 + g,
// r0 + g + G, ... in ascending order; the groups' sums are then added in group
// order, so every partial has one fixed summation order. GROUPED: d < 2048.
template <bool GROUPED>
__global__ void __launch_bounds__(256)
router_dwg_part_kernel(int d, int E, int P, const __nv_bfloat16* __restrict__ x,
                       const int32_t* __restrict__ eti, const int32_t* __restrict__ offsets,
                       const float* __restrict__ dz_row, float* __restrict__ part, int* err) {
    pdl_wait();
    pdl_trigger();
    if (has_error(err)) return;  // uniform over the CTA
    const int e = blockIdx.x;
    const int z = blockIdx.z;
    const int gt = GROUPED ? d / 8 : 256;  // threads per row group
    const int G = GROUPED ? 256 / gt : 1;  // row groups
    const int g = threadIdx.x / gt;
    const int c = blockIdx.y * kDwgCols + (threadIdx.x % gt) * 8;
    const bool active = g < G && c < d;
    const int lo = offsets[e], len = offsets[e + 1] - lo;
    const int r0 = lo + static_cast<int>(static_cast<long long>(len) * z / P);
    const int r1 = lo + static_cast<int>(static_cast<long long>(len) * (z + 1) / P);
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (active) {
        int r = r0 + g;
        for (; r + 3 * G < r1; r += 4 * G) {
            uint4 v[4];
            float zz[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                v[q] = *reinterpret_cast<const uint4*>(x + static_cast<size_t>(eti[r + q * G]) * d + c);
                zz[q] = dz_row[r + q * G];
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float f[8];
                bf16x8_to_f32(v[q], f);
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[j] = fmaf(zz[q], f[j], acc[j]);
            }
        }
        for (; r < r1; r += G) {
            float f[8];
            bf16x8_to_f32(*reinterpret_cast<const uint4*>(x + static_cast<size_t>(eti[r]) * d + c), f);
            const float zq = dz_row[r];
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] = fmaf(zq, f[j], acc[j]);
        }
    }
    if constexpr (GROUPED) {
        __shared__ float red[256 * 8];
#pragma unroll
        for (int j = 0; j < 8; ++j) red[threadIdx.x * 8 + j] = acc[j];
        __syncthreads();
        if (g == 0) {
            for (int q = 1; q < G; ++q)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[j] += red[(q * gt + threadIdx.x) * 8 + j];
        }
    }
    if (g == 0 && c < d) {
        float* out = part + (static_cast<size_t>(z) * E + e) * d + c;
        *reinterpret_cast<float4*>(out) = make_float4(acc[0], acc[1], acc[2], acc[3]);
        *reinterpret_cast<float4*>(out + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
}

// dWg[i] = sum of the P partials part[q * n + i] in a fixed order. SPLIT
// (fewer than 65536 outputs, too few threads for one per output): 32 outputs
// per CTA (one per lane), warp w sums the parts q = w, w + 8, ... in ascending
// order, and the eight warp sums are added in warp order. Otherwise one thread
// per output sums q = 0, 1, ... in order.
template <bool SPLIT>
__global__ void __launch_bounds__(256)
router_dwg_reduce_kernel(int n, int P, const float* __restrict__ part, float* __restrict__ dWg,
                         int* err) {
    pdl_wait();
    pdl_trigger();
    if (has_error(err)) return;  // uniform over the CTA
    if constexpr (!SPLIT) {
        const int i = blockIdx.x * blockDim.x + threadIdx.x;
        if (i >= n) return;
        float s = 0.f;
        for (int q = 0; q < P; ++q) s += part[static_cast<size_t>(q) * n + i];
        dWg[i] = s;
        return;
    }
    __shared__ float ws[8][32];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int i = blockIdx.x * 32 + lane;
    float s = 0.f;
    if (i < n)
        for (int q = w; q < P; q += 8) s += part[static_cast<size_t>(q) * n + i];
    ws[w][lane] = s;
    __syncthreads();
    if (w == 0 && i < n) {
        float t = ws[0][lane];
#pragma unroll
        for (int q = 1; q < 8; ++q) t += ws[q][lane];
        dWg[i] = t;
    }
}

// Router-gradient operand: zero B [T, nw] (16-byte pieces), the identity
// token list and the chunk segments (chunk c = tokens [c * chunk, ...)).
__global__ void dwg_zero_kernel(int T, int nw, int chunk, int nseg, uint4* __restrict__ B,
                                int32_t* __restrict__ iota, Seg* __restrict__ segs, int* err) {
    pdl_wait();
    pdl_trigger();
    if (has_error(err)) return;
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    const size_t i0 = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const size_t n16 = static_cast<size_t>(T) * nw / 8;
    for (size_t i = i0; i < n16; i += stride) B[i] = make_uint4(0u, 0u, 0u, 0u);
    for (size_t t = i0; t < static_cast<size_t>(T); t += stride) iota[t] = static_cast<int32_t>(t);
    if (blockIdx.x == 0)
        for (int c = threadIdx.x; c < nseg; c += blockDim.x) {
            Seg sg;
            sg.lo = c * chunk;
            sg.hi = min(T, (c + 1) * chunk);
            sg.out = 0;
            sg.pad = 0;
            segs[c] = sg;
        }
}

// Routed row r < offsets[E] of expert e (the last e with offsets[e] <= r) and
// token t = eti[r]: B[t][e] = bf16(dz_r), B[t][e_pad + e] = bf16(dz_r - that).
// A token meets an expert at most once, so every element has one writer.
__global__ void dwg_scatter_kernel(int rows_cap, int E, int e_pad, int nw,
                                   const int32_t* __restrict__ eti,
                                   const int32_t* __restrict__ offsets,
                                   const float* __restrict__ dz_row, __nv_bfloat16* __restrict__ B,
                                   int* err) {
    pdl_wait();
    pdl_trigger();
    if (has_error(err)) return;
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= rows_cap || r >= offsets[E]) return;
    int lo = 0, hi = E;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (offsets[mid] <= r) lo = mid;
        else hi = mid;
    }
    const float z = dz_row[r];
    const __nv_bfloat16 zh = __float2bfloat16_rn(z);
    const __nv_bfloat16 zl = __float2bfloat16_rn(z - __bfloat162float(zh));
    __nv_bfloat16* row = B + static_cast<size_t>(eti[r]) * nw;
    row[lo] = zh;
    row[e_pad + lo] = zl;
}

// dW_g[e][c] = sum over chunks p (ascending) of part[p][c][e] + part[p][c][e_pad + e].
// Block (32, 8) owns 32 experts x 32 columns: reads run along e, the tile is
// transposed in shared memory so the writes run along c.
__global__ void __launch_bounds__(256)
dwg_reduce_kernel(int d, int E, int e_pad, int nw, int nseg, const float* __restrict__ part,
                  float* __restrict__ dWg, int* err) {
    pdl_wait();
    pdl_trigger();
    if (has_error(err)) return;
    __shared__ float tile[32][33];
    const int e0 = blockIdx.y * 32, c0 = blockIdx.x * 32;
    const int tx = threadIdx.x, ty = threadIdx.y;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int c = c0 + ty * 4 + j, e = e0 + tx;
        float acc = 0.f;
        if (c < d && e < E)
            for (int q = 0; q < nseg; ++q) {
                const float* row = part + (static_cast<size_t>(q) * d + c) * nw;
                acc += row[e];
                acc += row[e_pad + e];
            }
        tile[ty * 4 + j][tx] = acc;
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int e = e0 + ty * 4 + j, c = c0 + tx;
        if (e < E && c < d) dWg[static_cast<size_t>(e) * d + c] = tile[tx][ty * 4 + j];
    }
}

}  // namespace

cudaError_t launch_chunk_segments(const moe_shape& s, int chunk_tokens, int nchunks,
                                  const int32_t* eti, const int32_t* offsets, Seg* segs, int* err,
                                  cudaStream_t st) {
    if (nchunks > 0) {
        LaunchScope ls("chunk_search", st);
        const int warps = nchunks * s.E;
        launch_k(chunk_search_kernel, dim3((warps + 7) / 8), dim3(256), 0, st, eti, offsets, s.E, s.T,
                                                             chunk_tokens, nchunks, segs, err);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    LaunchScope ls("chunk_pack", st);
    launch_k(chunk_pack_kernel, dim3(nchunks + 1), dim3(256), 0, st, offsets, s.E, nchunks, segs, err);
    return cudaGetLastError();
}

cudaError_t launch_row_weights(const moe_shape& s, const float* topk_w, const int32_t* tim,
                               float* wrow, int* err, cudaStream_t st) {
    const int TK = s.T * s.K;
    LaunchScope ls("row_weights", st);
    launch_k(row_weights_kernel, dim3((TK + 255) / 256), dim3(256), 0, st, topk_w, tim, TK, wrow, err);
    return cudaGetLastError();
}

int comb_grid(int tokens) {
    const int per_sm = 8;  // resident 256-thread CTAs per SM
    const int need = (tokens + kCombWarps - 1) / kCombWarps;
    return std::max(1, std::min(need, num_sms() * per_sm));
}

cudaError_t launch_combine(const moe_shape& s, int t0, int t1, int c0, int nc, const int32_t* ids,
                           const float* topk_w, const int32_t* tim, const Seg* seg,
                           const __nv_bfloat16* Yc, __nv_bfloat16* y, int* err, cudaStream_t st,
                           const char* name, bool direct) {
    if (t1 <= t0) return cudaSuccess;
    LaunchScope ls(name, st);
    // Column slices per token: doubled while the pass has fewer than 24 warps'
    // worth of items per SM and each slice keeps a multiple of 256 columns (one
    // 16-byte piece per lane per row). Measured on GB300: MoEBlaze conf7's
    // passes of 2048 tokens 0.40 -> 0.44 of HBM with slices; the Mixtral-shaped
    // passes of 4096 tokens lost 1-4% with them, so they stay whole.
    int cs_log2 = 0;
    while (static_cast<long long>(t1 - t0) << cs_log2 < 24ll * num_sms() &&
           nc % (512 << cs_log2) == 0)
        ++cs_log2;
    const int grid = comb_grid((t1 - t0) << cs_log2);
    switch (s.K) {
#define MOE_COMBINE_CASE(KK)                                                                  \
    case KK:                                                                                  \
        if (direct)                                                                           \
            launch_k(combine_kernel<KK, true>, dim3(grid), dim3(kCombThreads), 0, st, t0, t1, c0, nc, s.d, cs_log2, ids, \
                                                                    topk_w, tim, seg, Yc, y,  \
                                                                    err);                     \
        else                                                                                  \
            launch_k(combine_kernel<KK, false>, dim3(grid), dim3(kCombThreads), 0, st, t0, t1, c0, nc, s.d, cs_log2, \
                                                                     ids, topk_w, tim, seg,   \
                                                                     Yc, y, err);             \
        break;
        MOE_COMBINE_CASE(1) MOE_COMBINE_CASE(2) MOE_COMBINE_CASE(3) MOE_COMBINE_CASE(4)
        MOE_COMBINE_CASE(5) MOE_COMBINE_CASE(6) MOE_COMBINE_CASE(7) MOE_COMBINE_CASE(8)
#undef MOE_COMBINE_CASE
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_router_dz(const moe_shape& s, int nparts, const float* dS_part,
                             const float* topk_w, const int32_t* tim, float* dS, float* dz,
                             float* dz_row, int* err, cudaStream_t st) {
    LaunchScope ls("router_dz", st);
    const long long warps = (static_cast<long long>(s.T) + 32 / s.K - 1) / (32 / s.K);
    launch_k(router_dz_kernel, dim3(static_cast<int>((warps * 32 + 255) / 256)), dim3(256), 0, st, 
        s.T, s.K, s.T * s.K, nparts, dS_part, topk_w, tim, dS, dz, dz_row, err);
    return cudaGetLastError();
}

cudaError_t launch_combine_rows(const moe_shape& s, int t0, int t1, int c0, int nc,
                                const int32_t* tok_off, const int32_t* tok_exp,
                                const int32_t* tok_rows, const float* w_row, const Seg* seg,
                                const __nv_bfloat16* Yc, __nv_bfloat16* y, int* err,
                                cudaStream_t st, const char* name) {
    if (t1 <= t0) return cudaSuccess;
    LaunchScope ls(name, st);
    launch_k(combine_rows_kernel, dim3(comb_grid(t1 - t0)), dim3(kCombThreads), 0, st, 
        t0, t1, c0, nc, s.d, tok_off, tok_exp, tok_rows, w_row, seg, Yc, y, err);
    return cudaGetLastError();
}

cudaError_t launch_router_dz_rows(const moe_shape& s, int rows_cap, int nparts,
                                  const float* dS_part, const int32_t* tok_off,
                                  const int32_t* tok_rows, const float* w_row, float* dS_row,
                                  float* dz_row, int* err, cudaStream_t st) {
    LaunchScope ls("router_dz", st);
    launch_k(router_dz_rows_kernel, dim3((s.T + 255) / 256), dim3(256), 0, st, s.T, rows_cap, nparts, dS_part,
                                                             tok_off, tok_rows, w_row, dS_row,
                                                             dz_row, err);
    return cudaGetLastError();
}

// Row parts per expert of the gathered router gradient: enough CTAs for
// about eight 256-thread CTAs per SM of a 152-SM GB300 (1216), at least 32 and
// at most 256. Depends on the shape alone (workspace sizes need no device).
int dwg_parts(const moe_shape& s) {
    const int cb = (s.d + kDwgCols - 1) / kDwgCols;
    const int want = (1216 + s.E * cb - 1) / (s.E * cb);
    return std::max(32, std::min(256, want));
}

cudaError_t launch_router_dwg(const moe_shape& s, const __nv_bfloat16* x, const int32_t* eti,
                              const int32_t* offsets, const float* dz_row, float* part,
                              float* dWg, int* err, cudaStream_t st) {
    const int P = dwg_parts(s);
    {
        LaunchScope ls("router_dwg", st);
        const dim3 grid(s.E, (s.d + kDwgCols - 1) / kDwgCols, P);
        if (s.d < kDwgCols)
            launch_k(router_dwg_part_kernel<true>, grid, dim3(256), 0, st, s.d, s.E, P, x, eti,
                     offsets, dz_row, part, err);
        else
            launch_k(router_dwg_part_kernel<false>, grid, dim3(256), 0, st, s.d, s.E, P, x, eti,
                     offsets, dz_row, part, err);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int n = s.E * s.d;
    LaunchScope ls("router_dwg_reduce", st);
    if (n < 65536)
        launch_k(router_dwg_reduce_kernel<true>, dim3((n + 31) / 32), dim3(256), 0, st, n, P, part,
                 dWg, err);
    else
        launch_k(router_dwg_reduce_kernel<false>, dim3((n + 255) / 256), dim3(256), 0, st, n, P,
                 part, dWg, err);
    return cudaGetLastError();
}

// Failure-path self-test: one CTA waits on an mbarrier that nothing arrives
// at, through the same bounded wait as the pipelined kernels. The wait gives
// up after limit_ns, the kernel records MOE_ERR_TIMEOUT in the status word and
// returns; the context stays usable.
__global__ void selftest_wait_kernel(uint64_t limit_ns, int* err) {
    pdl_wait();
    pdl_trigger();
    if (has_error(err)) return;
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    const uint32_t b = ptx::smem_u32(&bar);
    if (threadIdx.x == 0) {
        ptx::mbar_init(b, 1);
        abort_flag = 0;
        ptx::fence_mbar_init();
    }
    __syncthreads();
    // Phase 0 of the barrier never completes: nothing arrives on it.
    const bool ok = ptx::mbar_wait(b, 0u, &abort_flag, limit_ns);
    if (!ok && threadIdx.x == 0) raise_error(err, MOE_ERR_TIMEOUT);
}

cudaError_t launch_selftest_wait(uint64_t limit_ns, int* err, cudaStream_t st) {
    LaunchScope ls("selftest_wait", st);
    launch_k(selftest_wait_kernel, dim3(1), dim3(32), 0, st, limit_ns, err);
    return cudaGetLastError();
}

cudaError_t launch_dwg_operand(const moe_shape& s, const DwgPlan& dp, int rows_cap,
                               const int32_t* eti, const int32_t* offsets, const float* dz_row,
                               __nv_bfloat16* B, int32_t* iota, Seg* segs, int* err,
                               cudaStream_t st) {
    {
        LaunchScope ls("router_dwg_zero", st);
        const size_t n16 = static_cast<size_t>(s.T) * dp.nw / 8;
        const int grid = static_cast<int>(std::min<size_t>((n16 + 255) / 256,
                                                           static_cast<size_t>(num_sms()) * 8));
        launch_k(dwg_zero_kernel, dim3(std::max(1, grid)), dim3(256), 0, st, s.T, dp.nw, dp.chunk, dp.nchunks,
                                                           reinterpret_cast<uint4*>(B), iota,
                                                           segs, err);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    LaunchScope ls("router_dwg_scatter", st);
    launch_k(dwg_scatter_kernel, dim3((rows_cap + 255) / 256), dim3(256), 0, st, rows_cap, s.E, dp.e_pad, dp.nw,
                                                               eti, offsets, dz_row, B, err);
    return cudaGetLastError();
}

cudaError_t launch_dwg_reduce(const moe_shape& s, const DwgPlan& dp, const float* part,
                              float* dWg, int* err, cudaStream_t st) {
    LaunchScope ls("router_dwg_reduce", st);
    launch_k(dwg_reduce_kernel, dim3(dim3((s.d + 31) / 32, (s.E + 31) / 32)), dim3(dim3(32, 8)), 0, st, 
        s.d, s.E, dp.e_pad, dp.nw, dp.nchunks, part, dWg, err);
    return cudaGetLastError();
}

}  // namespace moe
