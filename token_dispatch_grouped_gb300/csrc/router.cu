// router.cu — R1: router logits, top-K selection and renormalised weights.
//
// z = x W_g^T (+ bias) in fp32 (x bf16, W_g fp32); the K largest logits per
// token in descending order (ties to the lower expert id); weights
// w_k = exp(z_k - z_0) / sum_j exp(z_j - z_0) over the chosen K, which equals
// the softmax probabilities renormalised over the chosen experts.
// Sources: MoEBlaze paper notes 2.1 (TopK(softmax(W_g x))); Dropless MoE, in
// depth, "A reference implementation" (renormalise over the chosen k).
//
// Layout: one CTA of 256 threads owns BT tokens and all (padded) EP experts.
// Thread (tg, eg) accumulates TT tokens x 8 experts in registers while a
// K-chunk of x and W_g is staged transposed in shared memory. The EG threads
// that share a token group sit in consecutive lanes of one warp, so the top-K
// is a butterfly arg-max over those lanes, repeated K times.
#include <cfloat>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kKC = 32;  // reduction chunk staged per step

template <int EP>
struct RouterCfg {
    static constexpr int TE = 8;
    static constexpr int EG = EP / TE;
    static constexpr int TG = kThreads / EG;
    static constexpr int TT = EP == 8 ? 1 : EP == 16 ? 1 : EP == 32 ? 2 : EP == 64 ? 4 : 8;
    static constexpr int BT = TG * TT;
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
    float* Xs = sm;                  // [kKC][BT]
    float* Ws = sm + kKC * C::BT;    // [kKC][EP]

    const int tid = threadIdx.x;
    const int eg = tid % C::EG;
    const int tg = tid / C::EG;
    const int t0 = blockIdx.x * C::BT;

    float acc[C::TT][8];
#pragma unroll
    for (int i = 0; i < C::TT; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

    for (int k0 = 0; k0 < d; k0 += kKC) {
        // x chunk: BT rows x 32 columns, 16-byte loads, stored transposed.
        for (int c = tid; c < C::BT * (kKC / 8); c += kThreads) {
            const int r = c / (kKC / 8);
            const int cc = (c % (kKC / 8)) * 8;
            const int t = t0 + r;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (t < T) v = *reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * d + k0 + cc);
            const __nv_bfloat16* b = reinterpret_cast<const __nv_bfloat16*>(&v);
#pragma unroll
            for (int j = 0; j < 8; ++j) Xs[(cc + j) * C::BT + r] = __bfloat162float(b[j]);
        }
        // W_g chunk: EP rows x 32 columns (rows >= E are zero), transposed.
        for (int c = tid; c < EP * (kKC / 4); c += kThreads) {
            const int e = c / (kKC / 4);
            const int cc = (c % (kKC / 4)) * 4;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (e < E) v = *reinterpret_cast<const float4*>(Wg + static_cast<size_t>(e) * d + k0 + cc);
            Ws[(cc + 0) * EP + e] = v.x;
            Ws[(cc + 1) * EP + e] = v.y;
            Ws[(cc + 2) * EP + e] = v.z;
            Ws[(cc + 3) * EP + e] = v.w;
        }
        __syncthreads();
#pragma unroll 4
        for (int kk = 0; kk < kKC; ++kk) {
            float xv[C::TT];
            float wv[8];
            const float4 w0 = *reinterpret_cast<const float4*>(Ws + kk * EP + eg * 8);
            const float4 w1 = *reinterpret_cast<const float4*>(Ws + kk * EP + eg * 8 + 4);
            wv[0] = w0.x; wv[1] = w0.y; wv[2] = w0.z; wv[3] = w0.w;
            wv[4] = w1.x; wv[5] = w1.y; wv[6] = w1.z; wv[7] = w1.w;
#pragma unroll
            for (int i = 0; i < C::TT; ++i) xv[i] = Xs[kk * C::BT + tg * C::TT + i];
#pragma unroll
            for (int i = 0; i < C::TT; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(xv[i], wv[j], acc[i][j]);
        }
        __syncthreads();
    }

    // Bias, optional logits output.
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int e = eg * 8 + j;
        const float b = (bias != nullptr && e < E) ? bias[e] : 0.f;
#pragma unroll
        for (int i = 0; i < C::TT; ++i) acc[i][j] += b;
    }
    if (logits != nullptr) {
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

    // Top-K per token: K rounds of a butterfly arg-max over the EG lanes.
#pragma unroll
    for (int i = 0; i < C::TT; ++i) {
        const int t = t0 + tg * C::TT + i;
        uint32_t taken = 0;
        float zsel[8];
        int isel[8];
        float z0 = 0.f;
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
            if (k == 0) z0 = bv;
        }
        if (eg == 0 && t < T) {
            float den = 0.f;
            float ex[8];
            for (int k = 0; k < K; ++k) {
                ex[k] = expf(zsel[k] - z0);
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
    const size_t smem = sizeof(float) * kKC * (C::BT + EP);
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
