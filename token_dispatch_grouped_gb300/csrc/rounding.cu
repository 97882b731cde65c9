// rounding.cu — token rounding (TR) of a token-choice routing: every expert's
// row count becomes a multiple of M_tile (SonicMoE notes 3.4.4, Algorithm 4,
// with the NR-f round-and-sparsify subroutine).
//
// Inputs: the router logits z [T, E] (fp32), the token-choice ids [T, K] and
// the offsets of their dispatch (f_e = token-choice count of expert e).
//   R0  lse_t = log sum_e exp(z_t,e); the score of (t, e) is the log-probability
//       z_t,e - lse_t (monotone in the softmax probability S), also stored
//       expert-major for the per-expert passes.
//   R1  one CTA: per expert the nearest multiple of M_tile (a tie rounds down;
//       at most T), the number m_e of tokens to drop or add, and the offsets of
//       the rounded rows.
//   R2  one CTA per expert with m_e > 0: 64-bit radix select of the m_e-th
//       candidate in the order (score descending, token ascending), among the
//       expert's token-choice tokens (rounding down: the last m_e are dropped)
//       or among its other tokens (rounding up: the first m_e are added).
//       The key (orderable score bits << 32 | ~token) makes the order strict,
//       so the kept set is unique.
//   R3  one warp per token: its final experts (ascending id), their count, and
//       its gate weights, the softmax of z_t over the final set.
//   R4  one CTA: exclusive scan of the per-token counts.
//   R5  the same per-token pass writes tok_exp and the weights in CSR order.
//   R6  one CTA per expert: compaction of its final tokens in ascending order
//       into expert_token_indices, with each row's weight and its CSR slot.
// The expert-side kernels (R2, R6) test token choice in a bitmap [E][T/32]
// built from the routing.
// Histogram bins in R2 are counted with shared-memory atomics (exact integer
// counts); every output is order-independent and bit-reproducible.
#include <cfloat>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kSelThreads = 1024;
constexpr int kTokWarps = 8;  // warps per CTA in the per-token kernels

__device__ __forceinline__ uint32_t orderable(float f) {
    const uint32_t b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ uint64_t tr_key(float lp, int t) {
    return (static_cast<uint64_t>(orderable(lp)) << 32) | static_cast<uint32_t>(~t);
}

__device__ __forceinline__ bool is_tc(const int32_t* ids, int t, int K, int e) {
    bool r = false;
    for (int k = 0; k < K; ++k) r |= ids[static_cast<size_t>(t) * K + k] == e;
    return r;
}

// Token-choice bitmap: bit t of row e (words of 32 tokens) is set when token t
// chose expert e.
__device__ __forceinline__ bool tc_bit(const uint32_t* __restrict__ bm, int words, int t, int e) {
    return (bm[static_cast<size_t>(e) * words + (t >> 5)] >> (t & 31)) & 1u;
}

// Builds the bitmap (zeroed before) from the routing: one warp per 32 tokens,
// lane = token & 31; for each slot, the lanes that chose the same expert form
// that expert's word bits (their lane mask) and the lowest of them ORs the mask
// into the word (an integer OR gives the same word in any order).
__global__ void tr_bitmap_kernel(const int32_t* __restrict__ ids, int T, int K, int words,
                                 uint32_t* __restrict__ bm, int* err) {
    if (has_error(err)) return;
    const int lane = threadIdx.x & 31;
    const int w = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);  // word = 32 tokens
    if (w >= words) return;  // warp-uniform
    const int t = w * 32 + lane;
    for (int k = 0; k < K; ++k) {
        const int e = t < T ? ids[static_cast<size_t>(t) * K + k] : -1;
        const unsigned same = __match_any_sync(0xffffffffu, e);
        if (e >= 0 && lane == __ffs(same) - 1) atomicOr(&bm[static_cast<size_t>(e) * words + w], same);
    }
}

// R0: warp per token.
__global__ void tr_lse_kernel(const float* __restrict__ z, int T, int E, float* __restrict__ lse,
                              int* err) {
    if (has_error(err)) return;
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * kTokWarps + threadIdx.x / 32;
    if (t >= T) return;
    const float* zt = z + static_cast<size_t>(t) * E;
    float m = -INFINITY;
    for (int e = lane; e < E; e += 32) m = fmaxf(m, zt[e]);
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float s = 0.f;
    for (int e = lane; e < E; e += 32) s += expf(zt[e] - m);
    for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) lse[t] = m + logf(s);
}

// R0': lpT [E][T] = z[t, e] - lse[t], expert-major, through 32 x 32 shared
// tiles (coalesced reads of z and writes of lpT), so the per-expert passes
// read their scores contiguously.
__global__ void tr_transpose_kernel(const float* __restrict__ z, const float* __restrict__ lse,
                                    int T, int E, float* __restrict__ lpT, int* err) {
    if (has_error(err)) return;
    __shared__ float tile[32][33];
    const int t0 = blockIdx.x * 32, e0 = blockIdx.y * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8 threads
    for (int r = ty; r < 32; r += 8) {
        const int t = t0 + r, e = e0 + tx;
        tile[r][tx] = (t < T && e < E) ? z[static_cast<size_t>(t) * E + e] - lse[t] : 0.f;
    }
    __syncthreads();
    for (int r = ty; r < 32; r += 8) {
        const int e = e0 + r, t = t0 + tx;
        if (t < T && e < E) lpT[static_cast<size_t>(e) * T + t] = tile[tx][r];
    }
}

// R1: one CTA of 256 threads (E <= 256).
// par[e] = {n_e, m_e, up_e}; offsets_tr [E+1].
__global__ void tr_decide_kernel(const int32_t* __restrict__ tc_offsets, int T, int E, int m_tile,
                                 int4* __restrict__ par, int32_t* __restrict__ offsets_tr,
                                 int* err) {
    if (has_error(err)) return;
    __shared__ int cnt[256];
    const int e = threadIdx.x;
    int n = 0;
    if (e < E) {
        const int f = tc_offsets[e + 1] - tc_offsets[e];
        const int lo = (f / m_tile) * m_tile;
        const int hi = ((f + m_tile - 1) / m_tile) * m_tile;
        const bool up = (hi - f) < (f - lo);  // a tie rounds down
        n = min(up ? hi : lo, T);
        par[e] = make_int4(n, up ? n - f : f - n, up ? 1 : 0, f);
    }
    cnt[e] = n;
    __syncthreads();
    if (e == 0) {
        int run = 0;
        for (int q = 0; q < E; ++q) {
            offsets_tr[q] = run;
            run += cnt[q];
        }
        offsets_tr[E] = run;
    }
}

// R2: CTA per expert. thr[e] = the key of the m-th candidate: rounding up, the
// m-th largest key among tokens that did not choose e (keys >= thr are added);
// rounding down, the m-th smallest key among tokens that chose e (keys <= thr
// are dropped). thr = 0 when nothing changes.
__global__ void __launch_bounds__(kSelThreads)
tr_select_kernel(const float* __restrict__ lpT, const uint32_t* __restrict__ bm, int words,
                 const int32_t* __restrict__ tc_eti,
                 const int32_t* __restrict__ tc_offsets, const int4* __restrict__ par, int T,
                 int E, int K, unsigned long long* __restrict__ thr, int* err) {
    if (has_error(err)) return;
    const int e = blockIdx.x;
    const int4 pe = par[e];
    const int m = pe.y;
    const bool up = pe.z != 0;
    if (m == 0) {
        if (threadIdx.x == 0) thr[e] = 0ull;
        return;
    }
    __shared__ unsigned int hist[256];
    __shared__ uint64_t s_prefix;
    __shared__ int s_rank;
    if (threadIdx.x == 0) {
        s_prefix = 0ull;
        s_rank = m;  // 1-based rank of the wanted key in the selection order
    }
    const int o0 = tc_offsets[e];
    const int n_cand = up ? T : tc_offsets[e + 1] - o0;
    for (int pass = 0; pass < 8; ++pass) {
        const int shift = 56 - 8 * pass;
        for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0u;
        __syncthreads();
        const uint64_t prefix = s_prefix;
        const uint64_t hmask = pass == 0 ? 0ull : (~0ull << (shift + 8));
        for (int i = threadIdx.x; i < n_cand; i += blockDim.x) {
            int t;
            if (up) {
                t = i;
                if (tc_bit(bm, words, t, e)) continue;
            } else {
                t = tc_eti[o0 + i];
            }
            const uint64_t key = tr_key(lpT[static_cast<size_t>(e) * T + t], t);
            if ((key & hmask) != prefix) continue;
            // Rounding up ranks from the largest key, rounding down from the smallest.
            const unsigned int dig = static_cast<unsigned int>((key >> shift) & 0xffu);
            atomicAdd(&hist[up ? 255u - dig : dig], 1u);
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            int r = s_rank;
            int b = 0;
            for (; b < 256; ++b) {
                const int c = static_cast<int>(hist[b]);
                if (r <= c) break;
                r -= c;
            }
            const uint64_t dig = static_cast<uint64_t>(up ? 255 - b : b);
            s_prefix = prefix | (dig << shift);
            s_rank = r;
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) thr[e] = s_prefix;
}

// Final membership of (t, e), given whether token t chose e and its score lp.
__device__ __forceinline__ bool tr_member(float lp, bool tc, int t, int e,
                                          const int4* __restrict__ par,
                                          const unsigned long long* __restrict__ thr) {
    const int4 pe = par[e];
    if (pe.y == 0) return tc;
    const uint64_t key = tr_key(lp, t);
    if (pe.z) return tc || key >= thr[e];
    return tc && key > thr[e];
}

// R3 / R5: warp per token. Without tok_off: counts only (n_t). With tok_off:
// tok_exp (ascending expert id) and the gate weights w_tok in CSR order.
__global__ void tr_tokens_kernel(const float* __restrict__ z, const float* __restrict__ lse,
                                 const int32_t* __restrict__ ids, const int4* __restrict__ par,
                                 const unsigned long long* __restrict__ thr, int T, int E, int K,
                                 int32_t* __restrict__ n_t, const int32_t* __restrict__ tok_off,
                                 int32_t* __restrict__ tok_exp, float* __restrict__ w_tok,
                                 int* err) {
    if (has_error(err)) return;
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * kTokWarps + threadIdx.x / 32;
    if (t >= T) return;
    const float lt = lse[t];
    const float* zt = z + static_cast<size_t>(t) * E;  // score z - lse: as in the transpose
    int count = 0;
    float zmax = -INFINITY;
    for (int e0 = 0; e0 < E; e0 += 32) {
        const int e = e0 + lane;
        const bool mem = e < E && tr_member(zt[e] - lt, is_tc(ids, t, K, e), t, e, par, thr);
        const unsigned b = __ballot_sync(0xffffffffu, mem);
        if (mem) zmax = fmaxf(zmax, zt[e]);
        count += __popc(b);
    }
    if (tok_off == nullptr) {
        if (lane == 0) n_t[t] = count;
        return;
    }
    for (int o = 16; o; o >>= 1) zmax = fmaxf(zmax, __shfl_xor_sync(0xffffffffu, zmax, o));
    // Softmax over the final set, summed in ascending expert order by lane 0
    // of each 32-expert group and then across groups: a fixed order.
    float den = 0.f;
    for (int e0 = 0; e0 < E; e0 += 32) {
        const int e = e0 + lane;
        const bool mem = e < E && tr_member(zt[e] - lt, is_tc(ids, t, K, e), t, e, par, thr);
        float v = mem ? expf(zt[e] - zmax) : 0.f;
        for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        den += v;
    }
    const float inv = count > 0 ? 1.f / den : 0.f;
    int base = tok_off[t];
    for (int e0 = 0; e0 < E; e0 += 32) {
        const int e = e0 + lane;
        const bool mem = e < E && tr_member(zt[e] - lt, is_tc(ids, t, K, e), t, e, par, thr);
        const unsigned b = __ballot_sync(0xffffffffu, mem);
        if (mem) {
            const int slot = base + __popc(b & ((1u << lane) - 1u));
            tok_exp[slot] = e;
            w_tok[slot] = expf(zt[e] - zmax) * inv;
        }
        base += __popc(b);
    }
}

// R4: one CTA, exclusive scan of n_t into tok_off [T+1]: 1024 counts at a
// time (coalesced), warp scans, then a scan of the 32 warp totals.
__global__ void __launch_bounds__(1024)
tr_scan_kernel(const int32_t* __restrict__ n_t, int T, int32_t* __restrict__ tok_off, int* err) {
    if (has_error(err)) return;
    __shared__ int32_t wsum[32];
    __shared__ int32_t s_run;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) s_run = 0;
    __syncthreads();
    for (int t0 = 0; t0 < T; t0 += 1024) {
        const int t = t0 + threadIdx.x;
        const int32_t v = t < T ? n_t[t] : 0;
        int32_t incl = v;
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t u = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += u;
        }
        if (lane == 31) wsum[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            int32_t w = wsum[lane];
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t u = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += u;
            }
            wsum[lane] = w;  // inclusive over warps
        }
        __syncthreads();
        const int32_t base = s_run + (warp > 0 ? wsum[warp - 1] : 0);
        if (t < T) tok_off[t] = base + incl - v;
        __syncthreads();
        if (threadIdx.x == 0) s_run += wsum[31];
        __syncthreads();
    }
    if (threadIdx.x == 0) tok_off[T] = s_run;
}

// R6: CTA per expert; each thread takes 8 consecutive tokens per round
// (8192 per round), a block scan of the per-thread member counts places them
// in ascending token order.
__global__ void __launch_bounds__(kSelThreads)
tr_compact_kernel(const float* __restrict__ lpT, const uint32_t* __restrict__ bm, int words,
                  const int4* __restrict__ par, const unsigned long long* __restrict__ thr,
                  int T, int E, int K, const int32_t* __restrict__ offsets_tr,
                  const int32_t* __restrict__ tok_off, const int32_t* __restrict__ tok_exp,
                  const float* __restrict__ w_tok, int32_t* __restrict__ eti_tr,
                  float* __restrict__ w_row, int32_t* __restrict__ tok_rows, int* err) {
    if (has_error(err)) return;
    __shared__ int wsum[kSelThreads / 32];
    __shared__ int s_run;
    const int e = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x / 32;
    const int lim = offsets_tr[e + 1];
    const float* lp = lpT + static_cast<size_t>(e) * T;
    if (threadIdx.x == 0) s_run = offsets_tr[e];
    __syncthreads();
    for (int r0 = 0; r0 < T; r0 += kSelThreads * 8) {
        const int tb = r0 + threadIdx.x * 8;
        uint32_t mm = 0u;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int t = tb + j;
            if (t < T && tr_member(lp[t], tc_bit(bm, words, t, e), t, e, par, thr)) mm |= 1u << j;
        }
        const int cnt = __popc(mm);
        int incl = cnt;
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += u;
        }
        if (lane == 31) wsum[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            int v = wsum[lane];
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += u;
            }
            wsum[lane] = v;
        }
        __syncthreads();
        int pos = s_run + (warp > 0 ? wsum[warp - 1] : 0) + incl - cnt;
        for (int j = 0; j < 8; ++j) {
            if (!((mm >> j) & 1u)) continue;
            const int t = tb + j;
            if (pos >= lim) {  // more members than the decided count: inconsistent state
                raise_error(err, MOE_ERR_CUDA);
                break;
            }
            eti_tr[pos] = t;
            // e is in t's list: the same membership test wrote it.
            const int end = tok_off[t + 1];
            int slot = tok_off[t];
            while (slot < end && tok_exp[slot] != e) ++slot;
            if (slot < end) {
                tok_rows[slot] = pos;
                w_row[pos] = w_tok[slot];
            } else {
                raise_error(err, MOE_ERR_CUDA);
            }
            ++pos;
        }
        __syncthreads();
        if (threadIdx.x == 0) s_run += wsum[31];
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_token_rounding(const moe_shape& s, int m_tile, const float* z,
                                  const int32_t* ids, const int32_t* tc_eti,
                                  const int32_t* tc_offsets, TrScratch sc, int32_t* eti_tr,
                                  int32_t* offsets_tr, float* w_row, int32_t* tok_off,
                                  int32_t* tok_exp, int32_t* tok_rows, int* err,
                                  cudaStream_t st) {
    const int tok_grid = (s.T + kTokWarps - 1) / kTokWarps;
    cudaError_t e;
    {
        LaunchScope ls("tr_lse", st);
        tr_lse_kernel<<<tok_grid, kTokWarps * 32, 0, st>>>(z, s.T, s.E, sc.lse, err);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    {
        LaunchScope ls("tr_transpose", st);
        tr_transpose_kernel<<<dim3((s.T + 31) / 32, (s.E + 31) / 32), 256, 0, st>>>(
            z, sc.lse, s.T, s.E, sc.lpT, err);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    {
        LaunchScope ls("tr_decide", st);
        tr_decide_kernel<<<1, 256, 0, st>>>(tc_offsets, s.T, s.E, m_tile, sc.par, offsets_tr,
                                            err);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const int words = (s.T + 31) / 32;
    {
        LaunchScope ls("tr_bitmap", st);
        e = cudaMemsetAsync(sc.bm, 0, static_cast<size_t>(s.E) * words * sizeof(uint32_t), st);
        if (e != cudaSuccess) return e;
        tr_bitmap_kernel<<<(words + 7) / 8, 256, 0, st>>>(ids, s.T, s.K, words, sc.bm, err);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    {
        LaunchScope ls("tr_select", st);
        tr_select_kernel<<<s.E, kSelThreads, 0, st>>>(sc.lpT, sc.bm, words, tc_eti, tc_offsets,
                                                     sc.par, s.T, s.E, s.K, sc.thr, err);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    {
        LaunchScope ls("tr_tokens", st);
        tr_tokens_kernel<<<tok_grid, kTokWarps * 32, 0, st>>>(z, sc.lse, ids, sc.par, sc.thr, s.T,
                                                              s.E, s.K, sc.n_t, nullptr, nullptr,
                                                              nullptr, err);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    {
        LaunchScope ls("tr_scan", st);
        tr_scan_kernel<<<1, 1024, 0, st>>>(sc.n_t, s.T, tok_off, err);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    {
        LaunchScope ls("tr_tokens", st);
        tr_tokens_kernel<<<tok_grid, kTokWarps * 32, 0, st>>>(z, sc.lse, ids, sc.par, sc.thr, s.T,
                                                              s.E, s.K, sc.n_t, tok_off, tok_exp,
                                                              sc.w_tok, err);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    {
        LaunchScope ls("tr_compact", st);
        tr_compact_kernel<<<s.E, kSelThreads, 0, st>>>(sc.lpT, sc.bm, words, sc.par, sc.thr,
                                                      s.T, s.E, s.K, offsets_tr, tok_off, tok_exp,
                                                      sc.w_tok, eti_tr, w_row, tok_rows, err);
    }
    return cudaGetLastError();
}

}  // namespace moe
