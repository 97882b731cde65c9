// misc.cu — the memory-bound kernels around the expert GEMMs.
//
//   chunk_segments  per token chunk c and expert e, the sub-range of e's rows
//                   whose tokens fall in the chunk (stable order makes it one
//                   contiguous range) and where it lands in the chunk buffer.
//   row_weights     w_row[token_index_map[t*K+k]] = topk_w[t,k].
//   combine   (C1)  y_t = sum_k w_{t,k} Y[row(t,k)], fp32, k ascending, one bf16
//                   rounding. MoEBlaze paper notes 2.3; SonicMoE 3.4.1 (O_t).
//   router_dz (R2a) dS_{t,k} = sum over N-tiles of the partial <dA'_r, A_r>;
//                   dz_k = w_k (dS_k - sum_j w_j dS_j): the Jacobian of the
//                   softmax over the chosen logits applied to dS.
//   dx_combine(C2)  dx_t = sum_k (dX~[row(t,k)] + dz_{t,k} W_g[e_{t,k}]), fp32,
//                   k ascending. MoEBlaze paper notes 3.2 (token gradient
//                   accumulation over the K routed rows).
//   router_dwg(R2b) dW_g = dz^T x, as per-chunk partials then a fixed-order sum.
// All sums run in a fixed order, so results are bit-reproducible.
#include "common.cuh"

namespace moe {
namespace {

__device__ __forceinline__ int lower_bound_i32(const int32_t* a, int lo, int hi, int key) {
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (a[mid] < key) lo = mid + 1;
        else hi = mid;
    }
    return lo;
}

// grid = nchunks + 1 (the last "chunk" is the whole row space), block = 256.
__global__ void chunk_segments_kernel(const int32_t* __restrict__ eti,
                                      const int32_t* __restrict__ offsets, int E, int T,
                                      int chunk_tokens, int nchunks, Seg* __restrict__ segs,
                                      int* err) {
    if (has_error(err)) return;
    __shared__ int cnt[256];
    const int c = blockIdx.x;
    const int e = threadIdx.x;
    int lo = 0, hi = 0;
    if (e < E) {
        const int o0 = offsets[e], o1 = offsets[e + 1];
        if (c == nchunks) {
            lo = o0;
            hi = o1;
        } else {
            const int ta = c * chunk_tokens;
            const int tb = min(T, ta + chunk_tokens);
            lo = lower_bound_i32(eti, o0, o1, ta);
            hi = lower_bound_i32(eti, lo, o1, tb);
        }
    }
    cnt[e] = hi - lo;
    __syncthreads();
    if (e < E) {
        int out = lo;
        if (c != nchunks) {
            out = 0;
            for (int q = 0; q < e; ++q) out += cnt[q];
        }
        segs[static_cast<size_t>(c) * E + e] = Seg{lo, hi, out, 0};
    }
}

__global__ void row_weights_kernel(const float* __restrict__ topk_w,
                                   const int32_t* __restrict__ tim, int TK,
                                   float* __restrict__ wrow, int* err) {
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

constexpr int kCombThreads = 128;

// One CTA per token of the chunk; each thread owns 8 columns per pass.
__global__ void __launch_bounds__(kCombThreads)
combine_kernel(int t0, int d, int E, int K, const int32_t* __restrict__ ids,
               const float* __restrict__ topk_w, const int32_t* __restrict__ tim,
               const Seg* __restrict__ seg, const __nv_bfloat16* __restrict__ Yc,
               __nv_bfloat16* __restrict__ y, int* err) {
    if (has_error(err)) return;
    const int t = t0 + blockIdx.x;
    __shared__ size_t row_off[8];
    __shared__ float wk[8];
    if (threadIdx.x < K) {
        const size_t i = static_cast<size_t>(t) * K + threadIdx.x;
        const int e = ids[i];
        const Seg sg = seg[e];
        const int r = tim[i];
        row_off[threadIdx.x] = static_cast<size_t>(sg.out + (r - sg.lo)) * d;
        wk[threadIdx.x] = topk_w[i];
    }
    __syncthreads();
    for (int c = threadIdx.x * 8; c < d; c += kCombThreads * 8) {
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int k = 0; k < K; ++k) {
            float f[8];
            bf16x8_to_f32(*reinterpret_cast<const uint4*>(Yc + row_off[k] + c), f);
            const float w = wk[k];
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] = fmaf(w, f[j], acc[j]);
        }
        *reinterpret_cast<uint4*>(y + static_cast<size_t>(t) * d + c) = f32_to_bf16x8(acc);
    }
}

__global__ void router_dz_kernel(int T, int K, int TK, int nparts, const float* __restrict__ dS_part,
                                 const float* __restrict__ topk_w, const int32_t* __restrict__ tim,
                                 float* __restrict__ dS, float* __restrict__ dz, int* err) {
    if (has_error(err)) return;
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= T) return;
    float s[8], w[8];
    float sbar = 0.f;
    for (int k = 0; k < K; ++k) {
        const size_t i = static_cast<size_t>(t) * K + k;
        const int r = tim[i];
        float acc = 0.f;
        for (int p = 0; p < nparts; ++p) acc += dS_part[static_cast<size_t>(p) * TK + r];
        s[k] = acc;
        w[k] = topk_w[i];
        sbar = fmaf(w[k], acc, sbar);
    }
    for (int k = 0; k < K; ++k) {
        const size_t i = static_cast<size_t>(t) * K + k;
        dS[i] = s[k];
        dz[i] = w[k] * (s[k] - sbar);
    }
}

__global__ void __launch_bounds__(kCombThreads)
dx_combine_kernel(int t0, int d, int E, int K, const int32_t* __restrict__ ids,
                  const float* __restrict__ dz, const int32_t* __restrict__ tim,
                  const Seg* __restrict__ seg, const __nv_bfloat16* __restrict__ dXc,
                  const float* __restrict__ Wg, __nv_bfloat16* __restrict__ dx, int* err) {
    if (has_error(err)) return;
    const int t = t0 + blockIdx.x;
    __shared__ size_t row_off[8];
    __shared__ int ek[8];
    __shared__ float zk[8];
    if (threadIdx.x < K) {
        const size_t i = static_cast<size_t>(t) * K + threadIdx.x;
        const int e = ids[i];
        const Seg sg = seg[e];
        row_off[threadIdx.x] = static_cast<size_t>(sg.out + (tim[i] - sg.lo)) * d;
        ek[threadIdx.x] = e;
        zk[threadIdx.x] = dz[i];
    }
    __syncthreads();
    for (int c = threadIdx.x * 8; c < d; c += kCombThreads * 8) {
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int k = 0; k < K; ++k) {
            float f[8];
            bf16x8_to_f32(*reinterpret_cast<const uint4*>(dXc + row_off[k] + c), f);
            const float* wg = Wg + static_cast<size_t>(ek[k]) * d + c;
            const float4 g0 = *reinterpret_cast<const float4*>(wg);
            const float4 g1 = *reinterpret_cast<const float4*>(wg + 4);
            const float gz[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
            const float z = zk[k];
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] += f[j] + z * gz[j];
        }
        *reinterpret_cast<uint4*>(dx + static_cast<size_t>(t) * d + c) = f32_to_bf16x8(acc);
    }
}

constexpr int kDwgCols = 64;
constexpr int kDwgChunk = 2048;

// grid (d / 64, nchunks); 64 threads, one column each; fp32 accumulators for
// all E experts of the CTA's 64 columns live in shared memory.
__global__ void __launch_bounds__(kDwgCols)
router_dwg_part_kernel(int T, int d, int E, int K, const __nv_bfloat16* __restrict__ x,
                       const int32_t* __restrict__ ids, const float* __restrict__ dz,
                       float* __restrict__ part, int* err) {
    if (has_error(err)) return;
    extern __shared__ float acc[];  // [E][64]
    const int c = blockIdx.x * kDwgCols + threadIdx.x;
    for (int e = 0; e < E; ++e) acc[e * kDwgCols + threadIdx.x] = 0.f;
    const int ta = blockIdx.y * kDwgChunk;
    const int tb = min(T, ta + kDwgChunk);
    for (int t = ta; t < tb; ++t) {
        const float xv = __bfloat162float(x[static_cast<size_t>(t) * d + c]);
        for (int k = 0; k < K; ++k) {
            const size_t i = static_cast<size_t>(t) * K + k;
            acc[ids[i] * kDwgCols + threadIdx.x] += dz[i] * xv;
        }
    }
    float* out = part + static_cast<size_t>(blockIdx.y) * E * d;
    for (int e = 0; e < E; ++e) out[static_cast<size_t>(e) * d + c] = acc[e * kDwgCols + threadIdx.x];
}

__global__ void router_dwg_reduce_kernel(int n, int nchunks, const float* __restrict__ part,
                                         float* __restrict__ dWg, int* err) {
    if (has_error(err)) return;
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    float s = 0.f;
    for (int q = 0; q < nchunks; ++q) s += part[static_cast<size_t>(q) * n + i];
    dWg[i] = s;
}

}  // namespace

cudaError_t launch_chunk_segments(const moe_shape& s, int chunk_tokens, int nchunks,
                                  const int32_t* eti, const int32_t* offsets, Seg* segs, int* err,
                                  cudaStream_t st) {
    LaunchScope ls("chunk_segments", st);
    chunk_segments_kernel<<<nchunks + 1, 256, 0, st>>>(eti, offsets, s.E, s.T, chunk_tokens,
                                                       nchunks, segs, err);
    return cudaGetLastError();
}

cudaError_t launch_row_weights(const moe_shape& s, const float* topk_w, const int32_t* tim,
                               float* wrow, int* err, cudaStream_t st) {
    const int TK = s.T * s.K;
    LaunchScope ls("row_weights", st);
    row_weights_kernel<<<(TK + 255) / 256, 256, 0, st>>>(topk_w, tim, TK, wrow, err);
    return cudaGetLastError();
}

cudaError_t launch_combine(const moe_shape& s, int t0, int t1, const int32_t* ids,
                           const float* topk_w, const int32_t* tim, const Seg* seg,
                           const __nv_bfloat16* Yc, __nv_bfloat16* y, int* err, cudaStream_t st) {
    if (t1 <= t0) return cudaSuccess;
    LaunchScope ls("combine", st);
    combine_kernel<<<t1 - t0, kCombThreads, 0, st>>>(t0, s.d, s.E, s.K, ids, topk_w, tim, seg, Yc,
                                                     y, err);
    return cudaGetLastError();
}

cudaError_t launch_router_dz(const moe_shape& s, int nparts, const float* dS_part,
                             const float* topk_w, const int32_t* tim, float* dS, float* dz,
                             int* err, cudaStream_t st) {
    LaunchScope ls("router_dz", st);
    router_dz_kernel<<<(s.T + 127) / 128, 128, 0, st>>>(s.T, s.K, s.T * s.K, nparts, dS_part,
                                                        topk_w, tim, dS, dz, err);
    return cudaGetLastError();
}

cudaError_t launch_dx_combine(const moe_shape& s, int t0, int t1, const int32_t* ids,
                              const float* dz, const int32_t* tim, const Seg* seg,
                              const __nv_bfloat16* dXc, const float* Wg, __nv_bfloat16* dx,
                              int* err, cudaStream_t st) {
    if (t1 <= t0) return cudaSuccess;
    LaunchScope ls("dx_combine", st);
    dx_combine_kernel<<<t1 - t0, kCombThreads, 0, st>>>(t0, s.d, s.E, s.K, ids, dz, tim, seg, dXc,
                                                        Wg, dx, err);
    return cudaGetLastError();
}

int dwg_token_chunk() { return kDwgChunk; }

cudaError_t launch_router_dwg(const moe_shape& s, const __nv_bfloat16* x, const int32_t* ids,
                              const float* dz, float* part, float* dWg, int* err,
                              cudaStream_t st) {
    const int nchunks = (s.T + kDwgChunk - 1) / kDwgChunk;
    const size_t smem = sizeof(float) * s.E * kDwgCols;
    cudaError_t e = cudaFuncSetAttribute(router_dwg_part_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    {
        LaunchScope ls("router_dwg", st);
        router_dwg_part_kernel<<<dim3(s.d / kDwgCols, nchunks), kDwgCols, smem, st>>>(
            s.T, s.d, s.E, s.K, x, ids, dz, part, err);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int n = s.E * s.d;
    LaunchScope ls("router_dwg_reduce", st);
    router_dwg_reduce_kernel<<<(n + 255) / 256, 256, 0, st>>>(n, nchunks, part, dWg, err);
    return cudaGetLastError();
}

}  // namespace moe
