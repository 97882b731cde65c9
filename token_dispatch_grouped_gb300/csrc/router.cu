// router.cu — R1: router logits, top-K selection and renormalised weights.
//
// z = x W_g^T (+ bias) in fp32 (x bf16, W_g fp32); the K largest logits per
// token in descending order (ties to the lower expert id); weights
// w_k = exp(z_k - z_0) / sum_j exp(z_j - z_0) over the chosen K, which equals
// the softmax probabilities renormalised over the chosen experts.
// Sources: MoEBlaze paper notes 2.1 (TopK(softmax(W_g x))); Dropless MoE, in
// depth, "A reference implementation" (renormalise over the chosen k).
//
// Layout: a CTA owns BT tokens and all EP (padded) experts. One producer warp
// streams KC-wide chunks of x (TMA, 128-byte swizzled rows) and W_g (TMA, plain
// rows) into a ring of shared-memory stages guarded by mbarriers; eight compute
// warps consume them without CTA-wide barriers. Compute warp w owns expert
// group eg = w % EG (TE experts) and reduction slice ks = w / EG of each chunk;
// lane l owns tokens l, l + 32, ... (TT of them), so a quarter-warp's x reads
// hit 8 rows whose swizzled 16-byte pieces sit in distinct banks, and W_g reads
// are warp-wide broadcasts. Each thread keeps TT x TE fp32 accumulators (FFMA,
// k ascending within its slice). When there are few token tiles, a cluster of
// S CTAs splits the reduction over d; partial sums meet in the first CTA's
// shared memory and are added in a fixed order (CTA rank, then slice), read
// through distributed shared memory. The top-K is a butterfly arg-max over the
// EP/8 lanes that hold a token's logits (8 each), repeated K times. Every
// mbarrier wait is bounded.
#include <algorithm>
#include <cfloat>

#include "common.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

using namespace ptx;

constexpr uint64_t kWaitNs = 2000000000ull;

template <int EP>
struct RouterCfg {
    static constexpr int TE = EP <= 64 ? 8 : EP / 8;  // experts per thread
    static constexpr int TT = EP <= 128 ? 4 : 2;      // tokens per thread
    static constexpr int EG = EP / TE;             // expert groups
    static constexpr int KS = EG >= 8 ? 1 : 8 / EG;  // reduction slices per chunk
    static constexpr int CW = EG * KS;             // compute warps (8 or 16)
    static constexpr int THREADS = 32 * CW + 32;   // plus the TMA producer warp
    static constexpr int BT = 32 * TT;             // tokens per CTA
    static constexpr int KC = 64;                 // reduction chunk: one 128-byte x row
    static constexpr int X_BYTES = BT * KC * 2;
    static constexpr int W_BYTES = EP * KC * 4;
    static constexpr int STAGE = X_BYTES + W_BYTES;
    static constexpr int BUDGET = EP <= 64 ? 98304 : 147456;
    static constexpr int STAGES = BUDGET / STAGE > 4 ? 4 : (BUDGET / STAGE < 2 ? 2 : BUDGET / STAGE);
    static constexpr int PIPE = STAGES * STAGE;
    static constexpr int EPP = EP + 1;            // floats per logit row (odd: no conflicts)
    static constexpr int RED = KS * BT * EPP * 4; // partial sums of this CTA
    static constexpr int ZS = BT * EPP * 4;       // the tile's final logits
    static constexpr int BODY = PIPE > RED + ZS ? PIPE : RED + ZS;
    static constexpr int SMEM = 1024 + BODY + 256; // 1 KB alignment slack, barriers
    static constexpr int G = EP / 8;              // lanes per token in the top-K
    static_assert((KC / KS) % 8 == 0, "slice of whole 16-byte pieces");
    static_assert(STAGE % 1024 == 0, "stages keep the 1 KB swizzle alignment");
    static_assert(16 * STAGES + 8 <= 256, "barrier region");
};

__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float (&f)[8]) {
    const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float2 p = __bfloat1622float2(b[j]);
        f[2 * j] = p.x;
        f[2 * j + 1] = p.y;
    }
}

// Warp-uniform bounded wait: every lane polls, all lanes agree on the result.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
    const bool ok = mbar_wait(bar, parity, abort, kWaitNs);
    return __all_sync(0xffffffffu, ok);
}

// Selection from a CTA's final logits zs[r * epp + e] (r < bt tokens from t0):
// adds the bias, writes the logits, picks the K largest (ties to the lower id)
// and their weights exp(z_k - z_0) / sum_j exp(z_j - z_0). G = EP / 8
// consecutive threads hold one token's logits, 8 each; the K arg-maxes are
// butterflies over those G lanes. Each lane group works on NT tokens at once,
// so that NT independent compare-and-shuffle chains overlap. nthr (a multiple
// of 32) threads take part.
template <int EP, int NT>
__device__ __forceinline__ void router_topk_tail(const float* zs, int epp, int bt, int t0, int T,
                                                 int E, int K, const float* __restrict__ bias,
                                                 float* __restrict__ logits,
                                                 int32_t* __restrict__ ids,
                                                 float* __restrict__ wout, int* err, int tid,
                                                 int nthr) {
    constexpr int G = EP / 8;
    const int groups = nthr / G;  // lane groups; each takes NT tokens per pass
    const int g = tid % G;
    float bz[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int e = g * 8 + j;
        bz[j] = (bias != nullptr && e < E) ? bias[e] : 0.f;
    }
#pragma unroll 1
    for (int base = 0; base < bt; base += groups * NT) {
        float v[NT][8];
        bool live[NT];
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            const int r = base + n * groups + tid / G;
            const int t = t0 + r;
            live[n] = r < bt && t < T;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int e = g * 8 + j;
                v[n][j] = (live[n] && e < E) ? zs[r * epp + e] + bz[j] : -INFINITY;
            }
            if (logits != nullptr && live[n]) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int e = g * 8 + j;
                    if (e < E) logits[static_cast<size_t>(t) * E + e] = v[n][j];
                }
            }
        }
        uint32_t taken[NT];
        float zsel[NT][8];
        int isel[NT][8];
#pragma unroll
        for (int n = 0; n < NT; ++n) taken[n] = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            if (k >= K) break;
            float bv[NT];
            int bi[NT];
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                bv[n] = -INFINITY;
                bi[n] = 0x7fffffff;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int e = g * 8 + j;
                    const bool ok = e < E && !((taken[n] >> j) & 1u);
                    if (ok && (v[n][j] > bv[n] || (v[n][j] == bv[n] && e < bi[n]))) {
                        bv[n] = v[n][j];
                        bi[n] = e;
                    }
                }
            }
#pragma unroll
            for (int off = 1; off < G; off <<= 1) {
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    const float ov = __shfl_xor_sync(0xffffffffu, bv[n], off);
                    const int oi = __shfl_xor_sync(0xffffffffu, bi[n], off);
                    if (ov > bv[n] || (ov == bv[n] && oi < bi[n])) {
                        bv[n] = ov;
                        bi[n] = oi;
                    }
                }
            }
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                if (bi[n] / 8 == g && bi[n] < E) taken[n] |= 1u << (bi[n] % 8);
                zsel[n][k] = bv[n];
                isel[n][k] = bi[n];
            }
        }
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            if (!(live[n] && g == 0)) continue;
            const int t = t0 + base + n * groups + tid / G;
            float den = 0.f;
            float ex[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                if (k >= K) break;
                ex[k] = expf(zsel[n][k] - zsel[n][0]);
                den += ex[k];
            }
            const float inv = 1.f / den;
            bool bad = false;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                if (k >= K) break;
                const int e = isel[n][k];
                bad |= (e < 0 || e >= E);
                ids[static_cast<size_t>(t) * K + k] = e;
                wout[static_cast<size_t>(t) * K + k] = ex[k] * inv;
            }
            if (bad) raise_error(err, MOE_ERR_BAD_EXPERT_ID);
        }
    }
}

template <int EP, int S>
__global__ void __launch_bounds__(RouterCfg<EP>::THREADS, EP <= 64 ? 2 : 1)
router_kernel(const __grid_constant__ CUtensorMap mapX, const __grid_constant__ CUtensorMap mapW,
              const float* __restrict__ bias, float* __restrict__ logits,
              int32_t* __restrict__ ids, float* __restrict__ wout, int T, int d, int E, int K,
              int* err) {
    using C = RouterCfg<EP>;
    constexpr int kCompute = 32 * C::CW;
    constexpr int kThreads = C::THREADS;
    pdl_wait();
    pdl_trigger();
    // A CTA of a cluster must not leave alone (its peers would wait at the
    // cluster barrier), so only single-CTA launches skip work after an error.
    if (S == 1 && has_error(err)) return;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;  // 128-byte swizzle wants 1 KB alignment
    uint8_t* sm = smem_raw + (sbase - raw);
    const uint32_t bar0 = sbase + C::BODY;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (C::STAGES + s); };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::BODY + 16 * C::STAGES);

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const uint32_t rank = S > 1 ? cluster_ctarank() : 0u;
    const int t0 = static_cast<int>(blockIdx.x / S) * C::BT;
    const int dS = d / S;  // this CTA's share of the reduction
    const int kbeg = static_cast<int>(rank) * dS;
    const int nchunks = dS / C::KC;

    if (tid == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), kCompute / 32);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kCompute / 32 && lane == 0) {
        prefetch_tensormap(&mapX);
        prefetch_tensormap(&mapW);
    }
    __syncthreads();

    float acc[C::TT][C::TE];
#pragma unroll
    for (int i = 0; i < C::TT; ++i)
#pragma unroll
        for (int j = 0; j < C::TE; ++j) acc[i][j] = 0.f;

    if (warp == kCompute / 32) {
        // ---- producer: one elected lane issues the TMA loads of each stage
        if (lane == 0) {
            for (int c = 0; c < nchunks; ++c) {
                const int s = c % C::STAGES;
                const uint32_t ph = (c / C::STAGES) & 1;
                if (!mbar_wait(empty_bar(s), ph ^ 1u, abort_flag, kWaitNs)) break;
                mbar_arrive_expect_tx(full_bar(s), C::STAGE);
                const uint32_t xs = sbase + s * C::STAGE;
                const int k0 = kbeg + c * C::KC;
                tma_load_2d(xs, &mapX, full_bar(s), k0, t0);              // rows >= T read as 0
                tma_load_2d(xs + C::X_BYTES, &mapW, full_bar(s), k0, 0);  // experts >= E read as 0
            }
        }
        __syncwarp();
    } else {
        // ---- compute warps
        const int eg = warp % C::EG;
        const int ks = warp / C::EG;
        for (int c = 0; c < nchunks; ++c) {
            const int s = c % C::STAGES;
            const uint32_t ph = (c / C::STAGES) & 1;
            if (!warp_wait(full_bar(s), ph, abort_flag)) break;
            const uint8_t* xs = sm + s * C::STAGE;
            const float* ws = reinterpret_cast<const float*>(xs + C::X_BYTES);
            constexpr int KPS = C::KC / C::KS;
#pragma unroll
            for (int q = 0; q < KPS; q += 8) {
                const int kk = ks * KPS + q;
                const int piece = kk >> 3;  // 16-byte piece of the 128-byte row
                float xv[C::TT][8];
#pragma unroll
                for (int i = 0; i < C::TT; ++i) {
                    const int r = lane + 32 * i;  // r & 7 == lane & 7
                    bf16x8_to_f32(*reinterpret_cast<const uint4*>(
                                      xs + r * 128 + ((piece ^ (lane & 7)) << 4)),
                                  xv[i]);
                }
#pragma unroll
                for (int j = 0; j < C::TE; ++j) {
                    const float* wr = ws + (eg * C::TE + j) * C::KC + kk;
                    const float4 w0 = *reinterpret_cast<const float4*>(wr);
                    const float4 w1 = *reinterpret_cast<const float4*>(wr + 4);
                    const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                    for (int i = 0; i < C::TT; ++i)
#pragma unroll
                        for (int m = 0; m < 8; ++m) acc[i][j] = fmaf(xv[i][m], wv[m], acc[i][j]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty_bar(s));
        }
    }
    __syncthreads();  // every stage consumed: the pipeline memory is reused below
    if (*abort_flag) {
        if (tid == 0) raise_error(err, MOE_ERR_TIMEOUT);
        // Let copies already in flight land before the memory is reused.
        const uint64_t tw = globaltimer_ns();
        while (globaltimer_ns() - tw < 5000000ull) {
        }
    }

    // Partial sums of this CTA: red[ks][token][expert].
    float* red = reinterpret_cast<float*>(sm);
    float* zs = red + C::KS * C::BT * C::EPP;
    if (warp < kCompute / 32) {
        const int eg = warp % C::EG;
        const int ks = warp / C::EG;
#pragma unroll
        for (int i = 0; i < C::TT; ++i)
#pragma unroll
            for (int j = 0; j < C::TE; ++j)
                red[(ks * C::BT + lane + 32 * i) * C::EPP + eg * C::TE + j] = acc[i][j];
    }
    if constexpr (S > 1) cluster_sync();
    else __syncthreads();
    if (rank == 0) {
        // Fixed order: CTA rank, then slice.
        for (int idx = tid; idx < C::BT * EP; idx += kThreads) {
            const int r = idx / EP, e = idx % EP;
            float parts[S * C::KS];
#pragma unroll
            for (int q = 0; q < S; ++q)
#pragma unroll
                for (int s2 = 0; s2 < C::KS; ++s2) {
                    const int off = (s2 * C::BT + r) * C::EPP + e;
                    parts[q * C::KS + s2] =
                        q == 0 ? red[off]
                               : ld_shared_cluster_f32(mapa_shared(sbase + off * 4, q));
                }
            float v = parts[0];
#pragma unroll
            for (int q = 1; q < S * C::KS; ++q) v += parts[q];
            zs[r * C::EPP + e] = v;
        }
    }
    if constexpr (S > 1) cluster_sync();  // peers keep their partials until they are read
    if (rank != 0) return;
    __syncthreads();
    if (warp >= kCompute / 32) return;

    router_topk_tail<EP, 1>(zs, C::EPP, C::BT, t0, T, E, K, bias, logits, ids, wout, err, tid,
                            kCompute);
}

// ---------------------------------------------------------------------------
// Tensor-core router (E <= 128). W_g is split into three bf16 parts,
// W_g = W0 + W1 + W2 + r with W0 = bf16(W_g), W1 = bf16(W_g - W0),
// W2 = bf16(W_g - W0 - W1) (each difference exact in fp32, |r| about 2^-24 |W_g|),
// stored as the rows of B [3 * EB, d] bf16 (row p * EB + e = part p of expert e,
// zero rows past E). x is exact in bf16, so every product x * W_p is exact in
// fp32 and the tensor cores accumulate z_p = x W_p^T in fp32 (tcgen05.mma
// kind::f16, M = 128 tokens, N = 3 * EB). The epilogue adds the three parts in
// the order W0, W1, W2. A CTA owns 128 tokens; when there are few token tiles a
// cluster of S CTAs splits the reduction over d and the partial logits meet in
// the first CTA's shared memory (fixed order: CTA rank), as in the FFMA router.
// Warps: 0 TMA producer, 1 TMEM owner and MMA issuer, 2..5 epilogue; all six
// run the top-K selection.
template <int EP>
struct RmCfg {
    static constexpr int EB = EP < 16 ? 16 : EP;       // experts per weight part
    static constexpr int NB = 3 * EB;                   // MMA N: the three parts
    static constexpr int TMEM_COLS = NB <= 64 ? 64 : NB <= 128 ? 128 : NB <= 256 ? 256 : 512;
    static constexpr int NCH = (NB + 255) / 256;        // MMAs per k-step (N <= 256 each)
    static constexpr int BOXR = NB <= 256 ? NB : NB / 2;  // B rows per TMA box
    static constexpr int BT = 128;                      // tokens per CTA (M)
    static constexpr int KC = 64;                       // reduction chunk: 128-byte rows
    static constexpr int A_BYTES = BT * KC * 2;
    static constexpr int B_BYTES = NB * KC * 2;
    static constexpr int STAGE = A_BYTES + B_BYTES;
    static constexpr int BUDGET = EP <= 32 ? 98304 : 200704;
    static constexpr int STAGES = BUDGET / STAGE > 6 ? 6 : (BUDGET / STAGE < 2 ? 2 : BUDGET / STAGE);
    static constexpr int PIPE = STAGES * STAGE;
    static constexpr int EPP = EP + 1;                  // floats per logit row
    static constexpr int RED = BT * EPP * 4;            // this CTA's (partial) logits
    static constexpr int BODY = PIPE > 2 * RED ? PIPE : 2 * RED;  // partials, then the sums
    static constexpr int SMEM = 1024 + BODY + 256;
    static constexpr int THREADS = 192;
    static_assert(STAGE % 1024 == 0 && A_BYTES % 1024 == 0, "1 KB swizzle alignment");
    static_assert(NB % 16 == 0 && (NCH == 1 || NB - 256 >= 16), "MMA N");
    static_assert(NB % BOXR == 0 && BOXR <= 256 && (BOXR * 128) % 1024 == 0, "B boxes");
    static_assert(16 * STAGES + 32 <= 256, "barrier region");
};

// Three bf16 parts of W_g: Wsp[p * EB + e][c] for e < EB (zeros past E).
__global__ void router_wsplit_kernel(const float* __restrict__ Wg, int E, int EB, int d,
                                     __nv_bfloat16* __restrict__ Wsp, int* err) {
    pdl_wait();
    pdl_trigger();
    if (has_error(err)) return;
    const size_t n = static_cast<size_t>(EB) * d;
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
        const int e = static_cast<int>(i / d);
        const float v = e < E ? Wg[i] : 0.f;
        const __nv_bfloat16 h0 = __float2bfloat16_rn(v);
        const float r1 = v - __bfloat162float(h0);
        const __nv_bfloat16 h1 = __float2bfloat16_rn(r1);
        const float r2 = r1 - __bfloat162float(h1);
        Wsp[i] = h0;
        Wsp[n + i] = h1;
        Wsp[2 * n + i] = __float2bfloat16_rn(r2);
    }
}

template <int EP, int S>
__global__ void __launch_bounds__(RmCfg<EP>::THREADS, 1)
router_mma_kernel(const __grid_constant__ CUtensorMap mapX, const __grid_constant__ CUtensorMap mapB,
                  const float* __restrict__ bias, float* __restrict__ logits,
                  int32_t* __restrict__ ids, float* __restrict__ wout, int T, int d, int E, int K,
                  int* err) {
    using C = RmCfg<EP>;
    pdl_wait();
    pdl_trigger();
    if (S == 1 && has_error(err)) return;  // a cluster's CTAs never leave alone
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (sbase - raw);
    const uint32_t bar0 = sbase + C::BODY;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (C::STAGES + s); };
    const uint32_t done_bar = bar0 + 16u * C::STAGES;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::BODY + 16 * C::STAGES + 8);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::BODY + 16 * C::STAGES + 16);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const uint32_t rank = S > 1 ? cluster_ctarank() : 0u;
    const int t0 = static_cast<int>(blockIdx.x / S) * C::BT;
    const int nkb = d / (C::KC * S);                    // k-blocks of this CTA
    const int kb0 = static_cast<int>(rank) * nkb;

    if (tid == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        mbar_init(done_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&mapX);
        prefetch_tensormap(&mapB);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            for (int kb = 0; kb < nkb; ++kb) {
                const int s = kb % C::STAGES;
                const uint32_t ph = (kb / C::STAGES) & 1;
                if (!mbar_wait(empty_bar(s), ph ^ 1u, abort_flag, kWaitNs)) break;
                mbar_arrive_expect_tx(full_bar(s), C::STAGE);
                const uint32_t as = sbase + s * C::STAGE;
                const int k0 = (kb0 + kb) * C::KC;
                tma_load_2d(as, &mapX, full_bar(s), k0, t0);  // rows >= T read as 0
#pragma unroll
                for (int j = 0; j < C::NB / C::BOXR; ++j)
                    tma_load_2d(as + C::A_BYTES + j * C::BOXR * 128, &mapB, full_bar(s), k0,
                                j * C::BOXR);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb) {
            const int s = kb % C::STAGES;
            const uint32_t ph = (kb / C::STAGES) & 1;
            if (!warp_wait(full_bar(s), ph, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (lane == 0) {
                const uint32_t as = sbase + s * C::STAGE;
                const uint32_t bs = as + C::A_BYTES;
#pragma unroll
                for (int k = 0; k < C::KC / 16; ++k) {
                    const uint64_t ad = sdesc_sw128(as + k * 32, 16, 1024);
#pragma unroll
                    for (int c = 0; c < C::NCH; ++c) {
                        const int n0 = c * 256;
                        const int nc = C::NB - n0 < 256 ? C::NB - n0 : 256;
                        const uint64_t bd = sdesc_sw128(bs + n0 * 128 + k * 32, 16, 1024);
                        mma_bf16(tmem_base + n0, ad, bd, idesc_bf16(128, nc, 0, 0),
                                 (kb | k) != 0 ? 1u : 0u);
                    }
                }
                mma_commit(empty_bar(s));
            }
            __syncwarp();
        }
        if (ok && lane == 0) mma_commit(done_bar);
        __syncwarp();
    }
    // Epilogue: token row q * 32 + lane of TMEM lane quarter q; the three parts
    // of each expert's logit are added in the order W0, W1, W2 into red.
    float* red = reinterpret_cast<float*>(sm);
    if (warp >= 2) {
        const int q = warp & 3;
        const int row = q * 32 + lane;
        if (warp_wait(done_bar, 0, abort_flag)) {
            tc_fence_after();
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll 1
            for (int c0 = 0; c0 < C::NB; c0 += 32) {
                uint32_t v[32];
                tmem_ld32(taddr + c0, v);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int c = c0 + i;
                    const int part = c / C::EB, e = c % C::EB;
                    if (c < C::NB && e < EP) {
                        float* dst = red + row * C::EPP + e;
                        const float f = __uint_as_float(v[i]);
                        *dst = part == 0 ? f : *dst + f;
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem_base, C::TMEM_COLS);
    if (*abort_flag) {
        if (tid == 0) raise_error(err, MOE_ERR_TIMEOUT);
        // Let copies already in flight land before the CTA leaves.
        const uint64_t tw = globaltimer_ns();
        while (globaltimer_ns() - tw < 5000000ull) {
        }
    }
    float* zs = red + C::BT * C::EPP;
    if constexpr (S > 1) {
        cluster_sync();
        if (rank == 0) {
            for (int idx = tid; idx < C::BT * EP; idx += C::THREADS) {
                const int r = idx / EP, e = idx % EP;
                const uint32_t off = static_cast<uint32_t>((r * C::EPP + e) * 4);
                float v = red[r * C::EPP + e];
#pragma unroll
                for (int qq = 1; qq < S; ++qq) v += ld_shared_cluster_f32(mapa_shared(sbase + off, qq));
                zs[r * C::EPP + e] = v;
            }
        }
        cluster_sync();  // peers keep their partials until they are read
        if (rank != 0) return;
        __syncthreads();
    } else {
        zs = red;
    }
    router_topk_tail<EP, (EP >= 64 ? 4 : EP >= 32 ? 2 : 1)>(zs, C::EPP, C::BT, t0, T, E, K, bias,
                                                             logits, ids, wout, err, tid,
                                                             C::THREADS);
}

template <int EP, int S>
cudaError_t launch_mma_eps(const moe_shape& s, const __nv_bfloat16* x, const __nv_bfloat16* Wsp,
                           const float* bias, float* logits, int32_t* ids, float* w, int* err,
                           cudaStream_t st) {
    using C = RmCfg<EP>;
    auto kfn = router_mma_kernel<EP, S>;
    cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    CUtensorMap mapX, mapB;
    if (!make_tmap_bf16(&mapX, x, s.T, s.d, C::KC, C::BT) ||
        !make_tmap_bf16(&mapB, Wsp, C::NB, s.d, C::KC, C::BOXR))
        return cudaErrorInvalidValue;
    const int tiles = (s.T + C::BT - 1) / C::BT;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(tiles * S);
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 2 : 1;
    LaunchScope ls("router", st);
    return cudaLaunchKernelEx(&cfg, kfn, mapX, mapB, bias, logits, ids, w, s.T, s.d, s.E, s.K, err);
}

// Cluster split of d: doubled while the grid has at most one CTA per SM and
// every CTA keeps at least two k-blocks.
template <int EP>
cudaError_t launch_mma_ep(const moe_shape& s, const __nv_bfloat16* x, const float* Wg,
                          __nv_bfloat16* Wsp, const float* bias, float* logits, int32_t* ids,
                          float* w, int* err, cudaStream_t st) {
    using C = RmCfg<EP>;
    {
        LaunchScope ls("router_wsplit", st);
        const size_t n = static_cast<size_t>(C::EB) * s.d;
        const int grid = static_cast<int>(std::min<size_t>((n + 255) / 256, 4 * 152));
        launch_k(router_wsplit_kernel, dim3(grid), dim3(256), 0, st, Wg, s.E, C::EB, s.d, Wsp, err);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int tiles = (s.T + C::BT - 1) / C::BT;
    int S = 1;
    while (S < 8 && tiles * 2 * S <= num_sms() && s.d % (2 * S * C::KC) == 0 &&
           s.d / (2 * S) >= 2 * C::KC)
        S *= 2;
    switch (S) {
        case 8: return launch_mma_eps<EP, 8>(s, x, Wsp, bias, logits, ids, w, err, st);
        case 4: return launch_mma_eps<EP, 4>(s, x, Wsp, bias, logits, ids, w, err, st);
        case 2: return launch_mma_eps<EP, 2>(s, x, Wsp, bias, logits, ids, w, err, st);
        default: return launch_mma_eps<EP, 1>(s, x, Wsp, bias, logits, ids, w, err, st);
    }
}

template <int EP, int S>
cudaError_t launch_eps(const moe_shape& s, const __nv_bfloat16* x, const float* Wg,
                       const float* bias, float* logits, int32_t* ids, float* w, int* err,
                       cudaStream_t st) {
    using C = RouterCfg<EP>;
    auto kfn = router_kernel<EP, S>;
    cudaError_t e =
        cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    CUtensorMap mapX, mapW;
    if (!make_tmap_bf16(&mapX, x, s.T, s.d, C::KC, C::BT) ||
        !make_tmap_f32(&mapW, Wg, s.E, s.d, C::KC, EP))
        return cudaErrorInvalidValue;
    const int tiles = (s.T + C::BT - 1) / C::BT;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(tiles * S);
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 2 : 1;
    LaunchScope ls("router", st);
    return cudaLaunchKernelEx(&cfg, kfn, mapX, mapW, bias, logits, ids, w, s.T, s.d, s.E, s.K,
                              err);
}

// Cluster split of the reduction: doubled while the grid has fewer than two
// CTAs per SM and every CTA keeps at least two chunks of d.
template <int EP>
cudaError_t launch_ep(const moe_shape& s, const __nv_bfloat16* x, const float* Wg,
                      const float* bias, float* logits, int32_t* ids, float* w, int* err,
                      cudaStream_t st) {
    using C = RouterCfg<EP>;
    const int tiles = (s.T + C::BT - 1) / C::BT;
    int S = 1;
    while (S < 8 && tiles * S < 2 * num_sms() && s.d % (2 * S * C::KC) == 0 &&
           s.d / (2 * S) >= 2 * C::KC)
        S *= 2;
    switch (S) {
        case 8: return launch_eps<EP, 8>(s, x, Wg, bias, logits, ids, w, err, st);
        case 4: return launch_eps<EP, 4>(s, x, Wg, bias, logits, ids, w, err, st);
        case 2: return launch_eps<EP, 2>(s, x, Wg, bias, logits, ids, w, err, st);
        default: return launch_eps<EP, 1>(s, x, Wg, bias, logits, ids, w, err, st);
    }
}

}  // namespace

size_t router_ws_bytes(const moe_shape& s) {
    if (!router_tensor_cores(s)) return 0;
    const int ep = s.E <= 8 ? 8 : s.E <= 16 ? 16 : s.E <= 32 ? 32 : s.E <= 64 ? 64 : 128;
    const int eb = ep < 16 ? 16 : ep;
    return static_cast<size_t>(3) * eb * s.d * 2;
}

cudaError_t launch_router(const moe_shape& s, const __nv_bfloat16* x, const float* Wg,
                          const float* bias, float* logits, int32_t* ids, float* w, void* ws,
                          int* err, cudaStream_t st) {
    if (router_tensor_cores(s)) {
        __nv_bfloat16* Wsp = static_cast<__nv_bfloat16*>(ws);
        if (s.E <= 8) return launch_mma_ep<8>(s, x, Wg, Wsp, bias, logits, ids, w, err, st);
        if (s.E <= 16) return launch_mma_ep<16>(s, x, Wg, Wsp, bias, logits, ids, w, err, st);
        if (s.E <= 32) return launch_mma_ep<32>(s, x, Wg, Wsp, bias, logits, ids, w, err, st);
        if (s.E <= 64) return launch_mma_ep<64>(s, x, Wg, Wsp, bias, logits, ids, w, err, st);
        return launch_mma_ep<128>(s, x, Wg, Wsp, bias, logits, ids, w, err, st);
    }
    if (s.E <= 8) return launch_ep<8>(s, x, Wg, bias, logits, ids, w, err, st);
    if (s.E <= 16) return launch_ep<16>(s, x, Wg, bias, logits, ids, w, err, st);
    if (s.E <= 32) return launch_ep<32>(s, x, Wg, bias, logits, ids, w, err, st);
    if (s.E <= 64) return launch_ep<64>(s, x, Wg, bias, logits, ids, w, err, st);
    if (s.E <= 128) return launch_ep<128>(s, x, Wg, bias, logits, ids, w, err, st);
    return launch_ep<256>(s, x, Wg, bias, logits, ids, w, err, st);
}

}  // namespace moe
