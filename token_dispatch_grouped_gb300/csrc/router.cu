// router.cu — R1: router logits, top-K selection and renormalised weights.
//
// z = x W_g^T (+ bias) in fp32 (x bf16, W_g fp32); the K largest logits per
// token in descending order (ties to the lower expert id); weights
// w_k = exp(z_k - z_0) / sum_j exp(z_j - z_0) over the chosen K, which equals
// the softmax probabilities renormalised over the chosen experts.
// Sources: MoEBlaze paper notes 2.1 (TopK(softmax(W_g x))); Dropless MoE, in
// depth, "A reference implementation" (renormalise over the chosen k).
//
// Layout: one CTA of 256 threads owns BT tokens and all EP (padded) experts.
// Thread (ks, tg, eg) accumulates TT tokens x 8 experts over a 1/KS slice of
// every KC-wide chunk of the reduction; chunks of x and W_g are staged
// transposed in shared memory, and the next chunk is already in registers
// while the current one is used. The KS partial sums are added in a fixed
// order through shared memory. The EG threads of one token group sit in
// consecutive lanes of one warp, so the top-K is a butterfly arg-max over
// those lanes, repeated K times. Few tokens per CTA (16..64) keep the grid
// large for small T.
#include <cfloat>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;

template <int EP>
struct RouterCfg {
    static constexpr int EG = EP / 8;
    static constexpr int KS = EP == 8 ? 16 : EP == 16 ? 8 : EP == 32 ? 4 : EP == 64 ? 2 : 1;
    static constexpr int TG = kThreads / (EG * KS);
    static constexpr int TT = EP <= 32 ? 1 : EP == 64 ? 2 : 4;
    static constexpr int BT = TG * TT;
    static constexpr int KC = EP == 256 ? 64 : 128;
    static constexpr int XU = BT * KC / 8;    // 16-byte x units per chunk
    static constexpr int WU = EP * KC / 4;    // float4 W_g units per chunk
    static constexpr int XPT = (XU + kThreads - 1) / kThreads;
    static constexpr int WPT = (WU + kThreads - 1) / kThreads;
    static constexpr int SMEM_STAGE = (KC * BT + KC * EP) * 4;
    static constexpr int SMEM_RED = KS > 1 ? KS * BT * EP * 4 : 0;
    static constexpr int SMEM = SMEM_STAGE > SMEM_RED ? SMEM_STAGE : SMEM_RED;
};

template <int EP>
__global__ void __launch_bounds__(kThreads)
router_kernel(const __nv_bfloat16* __restrict__ x, const float* __restrict__ Wg,
              const float* __restrict__ bias, float* __restrict__ logits,
              int32_t* __restrict__ ids, float* __restrict__ wout, int T, int d, int E, int K,
              int* err) {
    using C = RouterCfg<EP>;
    if (has_error(err)) return;
    extern __shared__ __align__(16) float sm[];
    float* Xs = sm;                   // [KC][BT]
    float* Ws = sm + C::KC * C::BT;   // [KC][EP]

    const int tid = threadIdx.x;
    const int eg = tid % C::EG;
    const int tg = (tid / C::EG) % C::TG;
    const int ks = tid / (C::EG * C::TG);
    const int t0 = blockIdx.x * C::BT;

    float acc[C::TT][8];
#pragma unroll
    for (int i = 0; i < C::TT; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

    uint4 xr[C::XPT];
    float4 wr[C::WPT];
    auto fetch = [&](int k0) {
#pragma unroll
        for (int u = 0; u < C::XPT; ++u) {
            const int c = tid + u * kThreads;
            xr[u] = make_uint4(0, 0, 0, 0);
            if (c < C::XU) {
                const int r = c / (C::KC / 8);
                const int t = t0 + r;
                const int col = k0 + (c % (C::KC / 8)) * 8;  // chunks may run past d: zeros
                if (t < T && col < d)
                    xr[u] = *reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * d + col);
            }
        }
#pragma unroll
        for (int u = 0; u < C::WPT; ++u) {
            const int c = tid + u * kThreads;
            wr[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (c < C::WU) {
                const int e = c / (C::KC / 4);
                const int col = k0 + (c % (C::KC / 4)) * 4;
                if (e < E && col < d)
                    wr[u] = *reinterpret_cast<const float4*>(Wg + static_cast<size_t>(e) * d + col);
            }
        }
    };
    auto stage = [&]() {
#pragma unroll
        for (int u = 0; u < C::XPT; ++u) {
            const int c = tid + u * kThreads;
            if (c < C::XU) {
                const int r = c / (C::KC / 8);
                const int cc = (c % (C::KC / 8)) * 8;
                const __nv_bfloat16* b = reinterpret_cast<const __nv_bfloat16*>(&xr[u]);
#pragma unroll
                for (int j = 0; j < 8; ++j) Xs[(cc + j) * C::BT + r] = __bfloat162float(b[j]);
            }
        }
#pragma unroll
        for (int u = 0; u < C::WPT; ++u) {
            const int c = tid + u * kThreads;
            if (c < C::WU) {
                const int e = c / (C::KC / 4);
                const int cc = (c % (C::KC / 4)) * 4;
                Ws[(cc + 0) * EP + e] = wr[u].x;
                Ws[(cc + 1) * EP + e] = wr[u].y;
                Ws[(cc + 2) * EP + e] = wr[u].z;
                Ws[(cc + 3) * EP + e] = wr[u].w;
            }
        }
    };

    fetch(0);
    for (int k0 = 0; k0 < d; k0 += C::KC) {
        __syncthreads();  // previous chunk fully consumed
        stage();
        __syncthreads();
        if (k0 + C::KC < d) fetch(k0 + C::KC);  // in flight while this chunk is used
        constexpr int KPT = C::KC / C::KS;
#pragma unroll 8
        for (int q = 0; q < KPT; ++q) {
            const int kk = ks * KPT + q;
            const float4 w0 = *reinterpret_cast<const float4*>(Ws + kk * EP + eg * 8);
            const float4 w1 = *reinterpret_cast<const float4*>(Ws + kk * EP + eg * 8 + 4);
            const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
            for (int i = 0; i < C::TT; ++i) {
                const float xv = Xs[kk * C::BT + tg * C::TT + i];
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(xv, wv[j], acc[i][j]);
            }
        }
    }

    // Sum the KS partial results in a fixed order (ks = 0, 1, ...).
    if constexpr (C::KS > 1) {
        __syncthreads();
        float* red = sm;  // [KS][BT][EP]
#pragma unroll
        for (int i = 0; i < C::TT; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j)
                red[(ks * C::BT + tg * C::TT + i) * EP + eg * 8 + j] = acc[i][j];
        __syncthreads();
        if (ks == 0) {
#pragma unroll
            for (int i = 0; i < C::TT; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    float v = 0.f;
                    for (int q = 0; q < C::KS; ++q)
                        v += red[(q * C::BT + tg * C::TT + i) * EP + eg * 8 + j];
                    acc[i][j] = v;
                }
        }
    }
    // Threads of the warps that hold ks == 0 finish; lanes with ks != 0 in such a
    // warp take part in the shuffles but write nothing.
    if ((tid / 32) * 32 >= C::EG * C::TG) return;
    const bool owner = ks == 0;

#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int e = eg * 8 + j;
        const float b = (bias != nullptr && e < E) ? bias[e] : 0.f;
#pragma unroll
        for (int i = 0; i < C::TT; ++i) acc[i][j] += b;
    }
    if (logits != nullptr && owner) {
#pragma unroll
        for (int i = 0; i < C::TT; ++i) {
            const int t = t0 + tg * C::TT + i;
            if (t >= T) continue;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int e = eg * 8 + j;
                if (e < E) logits[static_cast<size_t>(t) * E + e] = acc[i][j];
            }
        }
    }

#pragma unroll
    for (int i = 0; i < C::TT; ++i) {
        const int t = t0 + tg * C::TT + i;
        uint32_t taken = 0;
        float zsel[8];
        int isel[8];
#pragma unroll 1
        for (int k = 0; k < K; ++k) {
            float bv = -INFINITY;
            int bi = 0x7fffffff;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int e = eg * 8 + j;
                const float v = acc[i][j];
                const bool ok = e < E && !((taken >> j) & 1u);
                if (ok && (v > bv || (v == bv && e < bi))) {
                    bv = v;
                    bi = e;
                }
            }
#pragma unroll
            for (int off = 1; off < C::EG; off <<= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
                if (ov > bv || (ov == bv && oi < bi)) {
                    bv = ov;
                    bi = oi;
                }
            }
            if (bi / 8 == eg && bi < E) taken |= 1u << (bi % 8);
            zsel[k] = bv;
            isel[k] = bi;
        }
        if (owner && eg == 0 && t < T) {
            float den = 0.f;
            float ex[8];
            for (int k = 0; k < K; ++k) {
                ex[k] = expf(zsel[k] - zsel[0]);
                den += ex[k];
            }
            const float inv = 1.f / den;
            bool bad = false;
            for (int k = 0; k < K; ++k) {
                const int e = isel[k];
                bad |= (e < 0 || e >= E);
                ids[static_cast<size_t>(t) * K + k] = e;
                wout[static_cast<size_t>(t) * K + k] = ex[k] * inv;
            }
            if (bad) raise_error(err, MOE_ERR_BAD_EXPERT_ID);
        }
    }
}

template <int EP>
cudaError_t launch_ep(const moe_shape& s, const __nv_bfloat16* x, const float* Wg,
                      const float* bias, float* logits, int32_t* ids, float* w, int* err,
                      cudaStream_t st) {
    using C = RouterCfg<EP>;
    static_assert(C::EG * C::KS * C::TG == kThreads, "thread layout");
    const size_t smem = C::SMEM;
    cudaError_t e = cudaFuncSetAttribute(router_kernel<EP>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const int grid = (s.T + C::BT - 1) / C::BT;
    LaunchScope ls("router", st);
    router_kernel<EP><<<grid, kThreads, smem, st>>>(x, Wg, bias, logits, ids, w, s.T, s.d, s.E,
                                                    s.K, err);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_router(const moe_shape& s, const __nv_bfloat16* x, const float* Wg,
                          const float* bias, float* logits, int32_t* ids, float* w, int* err,
                          cudaStream_t st) {
    if (s.E <= 8) return launch_ep<8>(s, x, Wg, bias, logits, ids, w, err, st);
    if (s.E <= 16) return launch_ep<16>(s, x, Wg, bias, logits, ids, w, err, st);
    if (s.E <= 32) return launch_ep<32>(s, x, Wg, bias, logits, ids, w, err, st);
    if (s.E <= 64) return launch_ep<64>(s, x, Wg, bias, logits, ids, w, err, st);
    if (s.E <= 128) return launch_ep<128>(s, x, Wg, bias, logits, ids, w, err, st);
    return launch_ep<256>(s, x, Wg, bias, logits, ids, w, err, st);
}

}  // namespace moe
