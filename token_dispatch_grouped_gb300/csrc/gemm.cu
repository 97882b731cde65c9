// gemm.cu — grouped expert GEMMs on tcgen05 tensor cores (sm_103a).
//
// One persistent, warp-specialised kernel template serves the expert GEMMs
// of the layer (six kinds, plus the non-gated and slot-wise variants). It
// runs either one CTA per tile (CTAS = 1, M = 128) or a CTA pair per tile
// (CTAS = 2, cluster of two CTAs, tcgen05 cta_group::2, M = 256 split 128/128,
// the B tile split by N so each SM stages half of it).
// Warp roles in every CTA:
//   warp 0      producer: TMA tile loads of the operands that are stored
//               contiguously (weights, SwiGLU output, dH, A') into a ring of
//               shared-memory stages.
//   warp 1      TMEM owner; in the tile's first CTA one thread issues
//               tcgen05.mma (bf16 in, fp32 accumulate) and tcgen05.commit.
//   warps 2..5  epilogue: tcgen05.ld of the accumulator (one TMEM lane = one
//               output row per thread), fused element-wise work, stores.
//   warps 6..9  (gathering kinds) cp.async gather of the token-row operand
//               through expert_token_indices, 16 bytes per thread, written in
//               the 128-byte-swizzled layout the MMA descriptors expect; rows
//               past an expert's end are zero-filled. No routed copy of the
//               activations exists anywhere.
//   warp 10     (gathering kinds, second CTA of a pair) relays the completion
//               of that CTA's gathers to the pair's MMA issuer (cp.async can
//               only signal a barrier of its own CTA) as the byte count of a
//               16-byte bulk copy into the first CTA.
// The accumulator is double-buffered in TMEM, so the epilogue of one tile
// overlaps the main loop of the next. Tiles are dealt statically over a
// device-side tile list derived from the per-expert row ranges (counts never
// go to the host): round-robin for the row-tiled kinds, snake order over the
// experts sorted by rows for the weight gradients (see next_tile).
//
// The six GEMMs (T_e = rows of expert e, all bf16 with fp32 accumulation):
//   G1  [T_e, d] x [d, h|h]  gather x; B = W1_e, W3_e (K-major);
//       epilogue: H = (a | b) saved, A = SiLU(a) * b. (MoEBlaze paper notes 5.2
//       epilogue fusion; SonicMoE 3.4.2 SwiGLU epilogue)
//       Non-gated experts (MoEBlaze paper notes 2.2, E(x) = W2 s(W1 x)): the
//       256-column tile is 256 rows of W1 alone; H = a, A = act(a).
//   G2  [T_e, h] x [h, d]    A rows contiguous; B = W2_e (K-major); Y chunk out.
//   G3  [T_e, d] x [d, h]    gather dy; B = W2_e (MN-major): dA' = dy W2_e.
//       epilogue: recompute sigma(a), SiLU(a), A from H; partial dS = <dA', A>;
//       dA = w dA'; da = dA b SiLU'(a); db = dA SiLU(a); A' = w A.
//       Non-gated: A = act(a), da = dA act'(a), dH = da alone.
//       (SonicMoE 3.4.1 dS = <dA', A>, dA = s dA', A' = s A; MoEBlaze
//       Algorithm 1 lines for grad A, grad B with SiLU recomputed)
//   G4  dW2_e [d, h] = dy_e^T A'_e   varlen-K over T_e; gather dy (MN-major A),
//       A' rows (MN-major B). (SonicMoE 3.4.1 dW2 = A'^T dO)
//   G5  (x_e^T dH_e) [d, 2h] = [dW1_e; dW3_e]^T   varlen-K; gather x (MN-major
//       A, M = d), dH rows (MN-major B); the epilogue stores the transpose.
//       (MoEBlaze Algorithm 1, FusedBwdW). Non-gated: [d, h] = dW1_e^T.
//   G6  dX~ [T_e, d] = da W1_e + db W3_e   one accumulator over K = 2h
//       (MoEBlaze 5.2: both branches aggregated in place, no per-branch buffer);
//       the epilogue adds the router term dz_r W_g[e] of each row.
//       Non-gated: K = h, da W1_e.
//   G2_SLOT  (slot-wise forward) [T_e^k, h] x [h, d] for the rows (t, k) of one
//       routing slot k, A rows gathered through tim[t*K + k]; the epilogue adds
//       w_{t,k} Y into an fp32 accumulator row of token t (each token once per
//       slot, so no two CTAs touch one row), and the last slot writes bf16 y.
//       (SonicMoE 3.4.1: O_t = sum_k s_{t,k} Y_{t,k}, in slot order)
//   G7  (router weight gradient) partials x_c^T B_c [d, nw] of token chunk c,
//       B = [dz_hi | dz_lo] [T, nw]: the router gradient dz split into two bf16
//       parts, dense over the (padded) experts; x rows gathered through an
//       identity list (MN-major A, M = d), B rows MN-major; the epilogue writes
//       fp32 partial rows, which are summed afterwards in a fixed order
//       (dW_g = dz^T x, the router term of the backward past dS).
// The saved pre-activation H and its gradient dH are [TK, hs] with hs = 2h
// (a | b) for SwiGLU and hs = h (a) for non-gated experts.
// Rows past an expert's end are zero-filled on the gathered operand, so
// ragged tails need no padding buffers (the other operand's extra rows are
// multiplied by zeros).
#include <algorithm>
#include <cstdlib>

#include "common.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

using namespace ptx;

constexpr int BM = 128;                      // rows per CTA
constexpr int BK0 = 64;                      // K elements in one 128-byte swizzled row
constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s per wait, then give up
constexpr int kMaxE = 256;

template <GemmKind KIND>
struct Tr;
// VK: varlen-K (weight gradients); A_MN/B_MN: operand is MN-major in shared
// memory; A_G: the A operand is gathered row by row through
// expert_token_indices by the cp.async gather warps.
template <> struct Tr<G1_UP>   { static constexpr bool VK = false; static constexpr int A_MN = 0, B_MN = 0, A_G = 1; };
template <> struct Tr<G2_DOWN> { static constexpr bool VK = false; static constexpr int A_MN = 0, B_MN = 0, A_G = 0; };
template <> struct Tr<G3_DH>   { static constexpr bool VK = false; static constexpr int A_MN = 0, B_MN = 1, A_G = 1; };
template <> struct Tr<G4_DW2>  { static constexpr bool VK = true;  static constexpr int A_MN = 1, B_MN = 1, A_G = 1; };
template <> struct Tr<G5_DW13> { static constexpr bool VK = true;  static constexpr int A_MN = 1, B_MN = 1, A_G = 1; };
template <> struct Tr<G6_DX>   { static constexpr bool VK = false; static constexpr int A_MN = 0, B_MN = 1, A_G = 0; };
template <> struct Tr<G1_UP_ACT> : Tr<G1_UP> {};
template <> struct Tr<G2_SLOT> : Tr<G1_UP> {};  // gathered K-major A, K-major B
template <> struct Tr<G3_DH_ACT> : Tr<G3_DH> {};
template <> struct Tr<G7_DWG> : Tr<G4_DW2> {};  // gathered x (MN-major A), B rows MN-major

// Reduction depth per pipeline stage. A stage's handshake (barrier waits,
// expect-tx, the gather warps' arrivals, the relay) costs about the same
// whatever the stage holds, so deeper stages feed the MMA faster: measured on
// GB300 with a probe of this kernel's feed (cp.async of 128 gathered rows plus
// a TMA box per stage, one CTA per SM), 80 GB/s per SM with 32 KB stages
// against 143 GB/s with 64 KB stages. CTA pairs of the up projection, the
// weight gradients and dX take 128 (three 64 KB stages). The non-gated dH
// GEMM takes 128 (DEEP, with a two-slot H ring) when d >= 2048: measured 9-11%
// faster at d = 2048, but 5-10% slower at d = 512 and 1024, where its few
// k-blocks per tile leave the epilogue's shorter H prefetch exposed. The
// SwiGLU dH GEMM keeps 64, since its epilogue's H ring (a and b boxes) would
// leave room for two 128-deep stages only (measured 15-29% slower that way),
// and the down projections keep 64 (no gain measured). A stage holds BK / BK0 sub-blocks of 64 K elements: K-major
// operands as [rows x 64] tiles one after the other, MN-major operands as
// 64-column chunks of BK rows.
template <GemmKind KIND, int CTAS, bool DEEP = false>
__host__ __device__ constexpr int bk_of() {
    return (CTAS == 2 && (DEEP || KIND == G1_UP || KIND == G1_UP_ACT || KIND == G4_DW2 ||
                          KIND == G5_DW13 || KIND == G6_DX || KIND == G7_DWG))
               ? 128
               : 64;
}

template <int BN, int CTAS, int EPI_BOXES, int BK_>
struct Cfg {
    static constexpr int BK = BK_;
    static constexpr int KSUB = BK / BK0;           // 64-deep sub-blocks per stage
    static constexpr int BNL = BN / CTAS;           // B rows (N) staged by this CTA
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = BNL * BK * 2;
    static constexpr int SUB_A = BM * BK0 * 2;      // K-major A: bytes per sub-block
    static constexpr int SUB_B = BNL * BK0 * 2;     // K-major B: bytes per sub-block
    static constexpr int CHUNK = BK * 128;          // MN-major: bytes per 64-column chunk
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int SMEM_MISC = 7168;        // barriers, TMEM slot, segments, tile prefix
    static constexpr int SMEM_EPI = 4 * EPI_BOXES * 2048;  // per epilogue warp: 32x32 bf16 boxes
    // Pipeline stages: what the 227 KB left after alignment, misc and epilogue
    // staging holds, at most 8.
    static constexpr int STAGES_FIT = (232448 - 1024 - SMEM_MISC - SMEM_EPI) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
    static constexpr int TMEM_COLS = 2 * BN;
    static constexpr int SMEM_TILES = STAGES * STAGE_BYTES;
    static constexpr int SMEM_TOTAL = 1024 + SMEM_TILES + SMEM_MISC + SMEM_EPI;
    static_assert(STAGES >= 3 && SMEM_TOTAL <= 232448, "shared memory");
    static_assert(1024 + 16 * kMaxE + 4 * (kMaxE + 1) <= SMEM_MISC, "misc region");
    // Pipeline barriers, TMEM slot, abort flag and relay slot below 768; the
    // epilogue's H-ring barriers (4 warps x kHR) from 768 to 1024.
    static_assert(8 * (3 * STAGES + 4) + 48 <= 768, "barrier region");
};

constexpr int kGatherThreads = 128;
// G3 epilogue: chunks of H (32 rows x 32 columns of a, and of b when gated) are
// loaded by TMA into a ring of hr_of slots per warp, one slot fewer chunks
// ahead: three slots for SwiGLU (a and b boxes), two for non-gated experts (a
// alone), which leaves the shared memory for three 128-deep stages.
template <GemmKind KIND, bool DEEP = false>
__host__ __device__ constexpr int hr_of() {
    return KIND == G3_DH_ACT && DEEP ? 2 : 3;
}
constexpr int kHRMax = 3;
static_assert(768 + 8 * 4 * kHRMax <= 1024, "H-ring barriers");
// Shared 2 KB staging boxes per epilogue warp: two for the stored outputs; for
// G3 the H ring (whose boxes are rewritten in place as dH) plus one box for A'.
template <GemmKind KIND, bool DEEP = false>
__host__ __device__ constexpr int epi_boxes() {
    return KIND == G3_DH ? 2 * hr_of<KIND>() + 1 : KIND == G3_DH_ACT ? hr_of<KIND, DEEP>() + 1 : 2;
}
template <GemmKind KIND, int CTAS>
constexpr int threads_of() {
    return 192 + (Tr<KIND>::A_G ? kGatherThreads : 0) + (Tr<KIND>::A_G && CTAS == 2 ? 32 : 0);
}

struct Params {
    int T, TK, d, h, E;
    int act;       // expert function: 0 SwiGLU, 1 SiLU, 2 ReLU (moe_expert_kind)
    int Kdim;      // VM: reduction length
    int M;         // VK: rows of the output per expert
    int n_tiles;   // tiles along N
    int group_m;   // VM: M tiles per group of the tile order (0: M fastest over the expert)
    int n_half;    // G5: N tiles per half (dW1 | dW3); the last tile of a half may be partial
    int slot;      // G2_SLOT: routing slot k of this launch (of K = nslot)
    int nslot;
    const int32_t* tim;  // G2_SLOT: token_index_map
    int half;      // 1: half-height pair tiles for the last partial tile (see half_ok)
    int n_off;     // G2/G6: first output column of this launch (column chunk)
    int ldo;       // G2/G6: row stride of the output chunk buffer (elements)
    const Seg* segs;
    const int32_t* eti;
    const __nv_bfloat16* gsrc;  // gathered rows: x or dy, [T, d]
    void* out0;
    void* out1;
    const void* aux0;
    const float* wrow;
    float* dS_part;
    int* err;
};

struct Tile {
    int e, m_blk, n_blk, lo, hi, out;
};

// Tile order inside one expert: M fastest, so tiles that run at the same time
// share their B panel (a weight panel for the VM kinds, the A' or dH panel
// for the weight gradients). bmc = rows per tile (128 or 256). The weight-
// gradient kinds (vk) walk the segments sorted by row count, each carrying
// its expert in `pad`.
__device__ __forceinline__ Tile decode_tile(int tile, const int* prefix, const Seg* segs, int E,
                                            bool vk, int m_tiles_vk, int bmc, int nt, int gm) {
    int lo = 0, hi = E;  // largest e with prefix[e] <= tile
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (prefix[mid] <= tile) lo = mid;
        else hi = mid;
    }
    Tile t;
    const Seg s = segs[lo];
    t.e = vk ? s.pad : lo;
    t.lo = s.lo;
    t.hi = s.hi;
    t.out = s.out;
    const int local = tile - prefix[lo];
    const int mt = vk ? m_tiles_vk : (s.hi - s.lo + bmc - 1) / bmc;
    if (vk || gm <= 0 || mt <= gm) {
        t.m_blk = local % mt;
        t.n_blk = local / mt;
    } else {
        // Row-tiled kinds, experts of more than gm M tiles: groups of gm M tiles,
        // each walked over all nt N tiles (M fastest inside the group), so a
        // group's rows of A stay in L2 while its B panels go by.
        const int g = local / (gm * nt);
        const int r = local - g * gm * nt;
        const int gsz = min(gm, mt - g * gm);
        t.m_blk = g * gm + r % gsz;
        t.n_blk = r / gsz;
    }
    return t;
}

// Half-height pair tiles. A row-tiled CTA-pair tile whose expert has at most
// 128 rows left (its last, partial tile) is issued as M = 128 cta_group::2 MMAs:
// each CTA supplies 64 rows of A instead of 128, which halves the tile's MMA
// work. The accumulator of such an MMA is folded in each CTA's TMEM (measured on
// GB300): lanes 0..63 hold the CTA's 64 rows for the first N/2 columns and lanes
// 64..127 the same rows for the last N/2 columns. So epilogue warps 2 and 3
// (lane quarters 0, 1) take the CTA's rows 0..31 and 32..63 over the first half
// of the columns, warps 4 and 5 (quarters 2, 3) the same rows over the second.
// Kinds whose epilogue handles this set HALF. The SwiGLU up projection stages,
// for a half tile, 64 gate rows and the matching 64 up rows of B in each CTA
// (instead of 128 gate rows in one CTA and 128 up rows in the other), so every
// warp holds matched gate and up columns. The dH GEMM's two warps of a row each
// write their own dS partial (two partial slots per N tile).
template <GemmKind KIND>
__host__ __device__ constexpr bool half_ok() {
    return KIND == G1_UP || KIND == G1_UP_ACT || KIND == G2_DOWN || KIND == G3_DH ||
           KIND == G3_DH_ACT || KIND == G6_DX;
}
__device__ __forceinline__ bool half_tile(const Tile& t, int bmc) {
    return t.hi - (t.lo + t.m_blk * bmc) <= bmc / 2;
}

// Warp-uniform bounded wait: every lane polls, all lanes agree on the result.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          bool cluster_scope = false) {
    const bool ok = mbar_wait(bar, parity, abort, kWaitNs, cluster_scope);
    return __all_sync(0xffffffffu, ok);
}

// Non-gated activation and its derivative (act = 1 SiLU, 2 ReLU with
// ReLU'(0) = 0). SiLU(u) = u sigma(u), SiLU'(u) = sigma(u) + SiLU(u) (1 - sigma(u)).
__device__ __forceinline__ float act_fn(int act, float u) {
    return act == 2 ? fmaxf(u, 0.f) : __fdividef(u, 1.f + __expf(-u));
}
__device__ __forceinline__ void act_and_grad(int act, float u, float& f, float& g) {
    if (act == 2) {
        f = fmaxf(u, 0.f);
        g = u > 0.f ? 1.f : 0.f;
    } else {
        const float sg = __fdividef(1.f, 1.f + __expf(-u));
        f = u * sg;
        g = sg + f * (1.f - sg);
    }
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
}

// 32 fp32 values -> 32 bf16 at dst (64 bytes, 16-byte aligned).
__device__ __forceinline__ void store32_bf16(void* dst, const float (&v)[32]) {
    uint4* p = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint4 u;
        u.x = pack_bf16(v[8 * q + 0], v[8 * q + 1]);
        u.y = pack_bf16(v[8 * q + 2], v[8 * q + 3]);
        u.z = pack_bf16(v[8 * q + 4], v[8 * q + 5]);
        u.w = pack_bf16(v[8 * q + 6], v[8 * q + 7]);
        p[q] = u;
    }
}

__device__ __forceinline__ void tmem_ld32f(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    tmem_ld32(taddr, r);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// ---- warp-cooperative row staging for the epilogues
// A warp's 32 rows (one per lane) x 32 bf16 columns pass through a 2 KB shared
// box so that global traffic is issued four lanes per 64-byte row segment (8
// rows per instruction) instead of one lane per row. Inside the box, 16-byte
// piece c of row l sits at piece c ^ ((l >> 1) & 3): row-wise writes by the
// 32 lanes then hit 8 distinct 16-byte bank groups per 8 lanes. On a box at a
// 512-byte boundary this is the placement of TMA's 64-byte swizzle for a box of
// 64-byte rows, so TMA loads and stores of such boxes use the same layout.
__device__ __forceinline__ uint32_t box_off(int row, int c16) {
    return static_cast<uint32_t>(row * 64 + ((c16 ^ ((row >> 1) & 3)) << 4));
}

// Lane's own row (32 fp32 -> bf16) into the box.
__device__ __forceinline__ void box_put_row(uint8_t* box, int lane, const float (&v)[32]) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint4 u;
        u.x = pack_bf16(v[8 * c + 0], v[8 * c + 1]);
        u.y = pack_bf16(v[8 * c + 2], v[8 * c + 3]);
        u.z = pack_bf16(v[8 * c + 4], v[8 * c + 5]);
        u.w = pack_bf16(v[8 * c + 6], v[8 * c + 7]);
        *reinterpret_cast<uint4*>(box + box_off(lane, c)) = u;
    }
}

// Stores the box to rows base + row * ld (row < nvalid), 16 bytes per lane.
__device__ __forceinline__ void box_store_rows(const uint8_t* box, int lane, __nv_bfloat16* base,
                                               size_t ld, int nvalid) {
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int pc = lane + 32 * i;
        const int row = pc >> 2, c16 = pc & 3;
        if (row < nvalid)
            *reinterpret_cast<uint4*>(base + static_cast<size_t>(row) * ld + c16 * 8) =
                *reinterpret_cast<const uint4*>(box + box_off(row, c16));
    }
    __syncwarp();
}

__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
    const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float2 x = __bfloat1622float2(b[j]);
        f[2 * j] = x.x;
        f[2 * j + 1] = x.y;
    }
}

// Non-gated backward for one lane's 32 columns: a (packed bf16 in ua) and
// dA' (v) give dS += <dA', act(a)>, da = w dA' act'(a) into the lane's row of
// box_da and A' = w act(a) packed into ap.
template <int ACT>
__device__ __forceinline__ void ng_chunk(const uint4 (&ua)[4], const float (&v)[32], float w,
                                         float& dsum, uint8_t* box_da, uint4 (&ap4)[4],
                                         int lane) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        float a8[8];
        unpack8(ua[c], a8);
        uint32_t da[4], ap[4];
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
            float f0, g0, f1, g1;
            act_and_grad(ACT, a8[i], f0, g0);
            act_and_grad(ACT, a8[i + 1], f1, g1);
            const float v0 = v[8 * c + i], v1 = v[8 * c + i + 1];
            dsum = fmaf(v0, f0, dsum);
            dsum = fmaf(v1, f1, dsum);
            da[i / 2] = pack_bf16(w * v0 * g0, w * v1 * g1);
            ap[i / 2] = pack_bf16(w * f0, w * f1);
        }
        *reinterpret_cast<uint4*>(box_da + box_off(lane, c)) = make_uint4(da[0], da[1], da[2], da[3]);
        ap4[c] = make_uint4(ap[0], ap[1], ap[2], ap[3]);
    }
}

// SwiGLU backward for one lane's 32 columns: a, b (packed bf16) and dA' (v),
// with A = SiLU(a) b, dA = w dA', give dS += <dA', A>, da = dA b SiLU'(a) and
// db = dA SiLU(a) into the lane's rows of box_da and box_db, and A' = w A
// packed into ap.
__device__ __forceinline__ void sw_chunk(const uint4 (&ua)[4], const uint4 (&ub)[4],
                                         const float (&v)[32], float w, float& dsum,
                                         uint8_t* box_da, uint8_t* box_db, uint4 (&ap4)[4],
                                         int lane) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        float a8[8], b8[8];
        unpack8(ua[c], a8);
        unpack8(ub[c], b8);
        uint32_t da[4], db[4], ap[4];
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
            float dav[2], dbv[2], apv[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const float a = a8[i + u], b = b8[i + u], vk = v[8 * c + i + u];
                const float sg = __fdividef(1.f, 1.f + __expf(-a));
                const float si = a * sg;
                const float Av = si * b;
                dsum = fmaf(vk, Av, dsum);
                const float dA = w * vk;
                dav[u] = dA * b * (sg + si * (1.f - sg));
                dbv[u] = dA * si;
                apv[u] = w * Av;
            }
            da[i / 2] = pack_bf16(dav[0], dav[1]);
            db[i / 2] = pack_bf16(dbv[0], dbv[1]);
            ap[i / 2] = pack_bf16(apv[0], apv[1]);
        }
        *reinterpret_cast<uint4*>(box_da + box_off(lane, c)) = make_uint4(da[0], da[1], da[2], da[3]);
        *reinterpret_cast<uint4*>(box_db + box_off(lane, c)) = make_uint4(db[0], db[1], db[2], db[3]);
        ap4[c] = make_uint4(ap[0], ap[1], ap[2], ap[3]);
    }
}

// Bounded wait that ignores the abort flag: lets a warp's own copies in flight
// land before it leaves.
__device__ __forceinline__ void mbar_drain(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait_sleep(bar, parity, 20000u))
        if (globaltimer_ns() - t0 > kWaitNs) break;
}

template <GemmKind KIND, int BN, int CTAS, bool DEEP>
__global__ void __launch_bounds__(threads_of<KIND, CTAS>(), 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap mapA,
                    const __grid_constant__ CUtensorMap mapB0,
                    const __grid_constant__ CUtensorMap mapB1,
                    const __grid_constant__ CUtensorMap mapO, const Params p) {
    using TR = Tr<KIND>;
    using C = Cfg<BN, CTAS, epi_boxes<KIND, DEEP>(), bk_of<KIND, CTAS, DEEP>()>;
    constexpr bool VK = TR::VK;
    constexpr bool PAIR = CTAS == 2;
    constexpr int BMC = BM * CTAS;  // rows per tile
    constexpr int NMMA = BN;        // MMA N (for G1: 128 gate + 128 up columns)
    constexpr int BNL = C::BNL;     // N columns whose B rows this CTA stages
    constexpr int BK = C::BK;
    constexpr int KSUB = C::KSUB;
    constexpr int kHR = hr_of<KIND, DEEP>();  // G3: slots of this warp's H ring
    constexpr uint32_t IDESC = idesc_bf16(BMC, NMMA, TR::A_MN, TR::B_MN);
    // Half-height pair tiles (see half_ok): M = 128 over the pair, 64 rows per CTA.
    constexpr bool HALF = PAIR && !VK && half_ok<KIND>();
    constexpr uint32_t IDESC_HALF = idesc_bf16(BM, NMMA, TR::A_MN, TR::B_MN);
    // Bytes one CTA's TMA producer brings per stage (gather warps bring A otherwise).
    constexpr uint32_t TMA_BYTES = TR::A_G ? C::B_BYTES : C::A_BYTES + C::B_BYTES;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t base_addr = (raw_addr + 1023u) & ~1023u;
    uint8_t* base = smem_raw + (base_addr - raw_addr);
    const uint32_t sA = base_addr;
    const uint32_t sB = base_addr + C::STAGES * C::A_BYTES;
    uint8_t* misc = base + C::SMEM_TILES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(misc);
    const uint32_t bar0 = smem_u32(bars);
    // full[S], empty[S], gfull[S] (pair: this CTA's gathers), tfull[2], tempty[2]
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (C::STAGES + s); };
    auto gfull_bar = [&](int s) { return bar0 + 8u * (2 * C::STAGES + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (3 * C::STAGES + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (3 * C::STAGES + 2 + a); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 8 * (3 * C::STAGES + 4));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 8 * (3 * C::STAGES + 4) + 8);
    // 16-byte slot (16-byte aligned) for the relay's completion signal.
    const uint32_t relay_slot = (smem_u32(misc) + 8 * (3 * C::STAGES + 4) + 16 + 15) & ~15u;
    Seg* s_segs = reinterpret_cast<Seg*>(misc + 1024);
    int* s_prefix = reinterpret_cast<int*>(misc + 1024 + 16 * kMaxE);
    uint8_t* epi = misc + C::SMEM_MISC;  // epilogue staging (TMA-store source)

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int E = p.E;
    const int m_tiles_vk = VK ? p.M / BMC : 0;
    const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
    const bool leader = rank == 0;
    const int tile0 = blockIdx.x / CTAS;   // first tile of this CTA (pair)
    const int tstep = gridDim.x / CTAS;    // tiles advance by the number of pairs
    // Tiles are dealt in waves of one per pair. The weight-gradient kinds deal
    // them in snake order (even waves pairs 0..n-1, odd waves n-1..0) over the
    // experts sorted by row count, largest first: a tile's cost grows with its
    // expert's rows, and on Zipf-skewed routing this keeps the longest pair's
    // share within about 4% of the mean (11-14% in expert order). Row-tiled
    // kinds (tiles of one cost) keep a plain round-robin in expert order.
    auto next_tile = [&](int tl) -> int {
        if constexpr (VK) {
            const int w = tl / tstep + 1;
            return w * tstep + ((w & 1) ? tstep - 1 - tile0 : tile0);
        } else {
            return tl + tstep;
        }
    };

    // Programmatic dependent launch (see pdl_wait in common.cuh): wait for the
    // previous kernel, then let the next one be scheduled.
    griddep_wait();
    griddep_launch_dependents();
    // Skip the work after an earlier error; a CTA of a pair never leaves alone
    // (its peer would wait at the cluster barrier), so pairs run on.
    if (!PAIR && has_error(p.err)) return;

    // ---- setup: segments, tile prefix, barriers, TMEM
    for (int e = threadIdx.x; e < E; e += blockDim.x) s_segs[e] = p.segs[e];
    __syncthreads();
    if constexpr (VK) {
        // Segments sorted by row count, largest first, ties by index (every CTA
        // computes the same order); thread e places expert e at its rank.
        static_assert(threads_of<KIND, CTAS>() >= kMaxE, "one thread per expert");
        Seg mine{0, 0, 0, 0};
        int rk = 0;
        const int e = threadIdx.x;
        if (e < E) {
            mine = s_segs[e];
            const int rows = mine.hi - mine.lo;
            for (int f = 0; f < E; ++f) {
                const int rf = s_segs[f].hi - s_segs[f].lo;
                rk += (rf > rows || (rf == rows && f < e)) ? 1 : 0;
            }
            mine.pad = e;
        }
        __syncthreads();
        if (e < E) s_segs[rk] = mine;
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        int run = 0;
        for (int e = 0; e < E; ++e) {
            s_prefix[e] = run;
            const int rows = s_segs[e].hi - s_segs[e].lo;
            run += VK ? m_tiles_vk * p.n_tiles : ((rows + BMC - 1) / BMC) * p.n_tiles;
        }
        s_prefix[E] = run;
        for (int s = 0; s < C::STAGES; ++s) {
            // full: the producer's expect-tx arrival, this CTA's gather threads,
            // and in a pair the relay of the second CTA's gathers.
            mbar_init(full_bar(s), 1 + (TR::A_G ? kGatherThreads : 0));
            mbar_init(empty_bar(s), 1);
            mbar_init(gfull_bar(s), kGatherThreads);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), 4 * CTAS);
        }
        if constexpr (KIND == G3_DH || KIND == G3_DH_ACT)
            for (int i = 0; i < 4 * kHR; ++i) mbar_init(bar0 + 768u + 8u * i, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&mapA);
        prefetch_tensormap(&mapB0);
        prefetch_tensormap(&mapB1);
        prefetch_tensormap(&mapO);
    }
    if (warp == 1) {
        if constexpr (PAIR) {
            tmem_alloc_pair(smem_u32(tmem_slot), C::TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) cluster_sync();  // the peer's barriers exist before any remote arrive
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int num_tiles = s_prefix[E];
    // Barrier that collects a stage's loads for the MMA: the first CTA's full[s].
    auto full_target = [&](int s) { return PAIR ? mapa_shared(full_bar(s), 0) : full_bar(s); };

    if (warp == 0) {
        // =========================== TMA producer
        int stage = 0;
        uint32_t phase = 0;
        bool stop = false;
        for (int tile = tile0; tile < num_tiles && !stop; tile = next_tile(tile)) {
            const Tile t = decode_tile(tile, s_prefix, s_segs, E, VK, m_tiles_vk, BMC, p.n_tiles, p.group_m);
            const int num_kb = VK ? (t.hi - t.lo + BK - 1) / BK : p.Kdim / BK;
            const bool half = HALF && p.half && half_tile(t, BMC);
            const int row0 = t.lo + t.m_blk * BMC + rank * (half ? BM / 2 : BM);  // VM: this CTA's A rows
            // First B column of the tile inside its half (G5: dW1 | dW3), and
            // this CTA's first B column in the B tensor.
            const int nin = (KIND == G5_DW13 ? t.n_blk % p.n_half : t.n_blk) * BN;
            const int ncol = (KIND == G5_DW13 ? (t.n_blk / p.n_half) * p.h : 0) + nin + rank * BNL;
            for (int kb = 0; kb < num_kb; ++kb) {
                if (!warp_wait(empty_bar(stage), phase ^ 1u, abort_flag)) {
                    stop = true;
                    break;
                }
                if (leader && lane == 0) {
                    uint32_t bytes = CTAS * TMA_BYTES;
                    if constexpr ((KIND == G2_DOWN || KIND == G6_DX) && HALF)
                        if (half) bytes -= CTAS * (C::A_BYTES / 2);  // 64-row A boxes
                    if constexpr (KIND == G3_DH || KIND == G3_DH_ACT || KIND == G4_DW2 ||
                                  KIND == G5_DW13 || KIND == G7_DWG) {
                        // h need not be a multiple of BN: 64-column B boxes that
                        // start at or past h are not loaded (their output columns
                        // are never stored).
                        bytes = 0;
                        for (int r = 0; r < CTAS; ++r)
                            for (int l = 0; l < BNL / 64; ++l)
                                if (nin + r * BNL + l * 64 < p.h) bytes += C::CHUNK;
                    }
                    // In a gathering pair, the relay's 16-byte signal copy.
                    if constexpr (TR::A_G && PAIR) bytes += 16;
                    mbar_arrive_expect_tx(full_bar(stage), bytes);
                }
                __syncwarp();
                const uint32_t a_dst = sA + stage * C::A_BYTES;
                const uint32_t b_dst = sB + stage * C::B_BYTES;
                const uint32_t fb = full_target(stage);
                const int k0 = kb * BK;
                auto load = [&](uint32_t dst, const CUtensorMap* m, int c0, int c1) {
                    if constexpr (PAIR) tma_load_2d_pair(dst, m, fb, c0, c1);
                    else tma_load_2d(dst, m, fb, c0, c1);
                };
                if constexpr (KIND == G2_DOWN || KIND == G6_DX) {
                    // Half tiles read 64 rows (a 64-row box map in the output slot).
                    if (lane == 0)
                        for (int u = 0; u < KSUB; ++u)
                            load(a_dst + u * C::SUB_A, (HALF && half) ? &mapO : &mapA, k0 + u * BK0,
                                 row0);
                }
                if constexpr (KIND == G1_UP || KIND == G1_UP_ACT) {
                    // SwiGLU: B = 128 gate rows (W1) then 128 up rows (W3); in a
                    // pair the first CTA stages W1's rows and the second W3's.
                    // Non-gated: B = 256 consecutive rows of W1.
                    if (lane == 0) {
                        for (int u = 0; u < KSUB; ++u) {
                            const uint32_t bd = b_dst + u * C::SUB_B;
                            const int kc = k0 + u * BK0;
                            if constexpr (KIND == G1_UP) {
                                const int brow = t.e * p.h + t.n_blk * 128;
                                if (PAIR && half) {
                                    // 64 gate rows then the same 64 up rows (64-row
                                    // boxes of W1 and W3 in the A and output map slots).
                                    const int hrow = brow + static_cast<int>(rank) * 64;
                                    load(bd, &mapA, kc, hrow);
                                    load(bd + 8192, &mapO, kc, hrow);
                                } else if constexpr (PAIR) {
                                    load(bd, leader ? &mapB0 : &mapB1, kc, brow);
                                } else {
                                    load(bd, &mapB0, kc, brow);
                                    load(bd + 16384, &mapB1, kc, brow);
                                }
                            } else {
                                const int brow = t.e * p.h + t.n_blk * 256;
                                if constexpr (PAIR) {
                                    load(bd, &mapB0, kc, brow + static_cast<int>(rank) * 128);
                                } else {
                                    load(bd, &mapB0, kc, brow);
                                    load(bd + 16384, &mapB0, kc, brow + 128);
                                }
                            }
                        }
                    }
                } else if constexpr (KIND == G2_DOWN || KIND == G2_SLOT) {
                    if (lane == 0)
                        for (int u = 0; u < KSUB; ++u)
                            load(b_dst + u * C::SUB_B, &mapB0, k0 + u * BK0, t.e * p.d + p.n_off + ncol);
                } else if constexpr (KIND == G3_DH || KIND == G3_DH_ACT) {
                    if (lane < BNL / 64 && nin + static_cast<int>(rank) * BNL + lane * 64 < p.h)
                        for (int u = 0; u < KSUB; ++u)
                            load(b_dst + lane * C::CHUNK + u * 8192, &mapB0, ncol + lane * 64,
                                 t.e * p.d + k0 + u * BK0);
                } else if constexpr (KIND == G4_DW2 || KIND == G5_DW13 || KIND == G7_DWG) {
                    // B rows of this expert (A' for dW2, dH for dW1/dW3; the chunk's
                    // rows of [dz_hi | dz_lo] for the router gradient), MN-major.
                    if (lane < BNL / 64 && nin + static_cast<int>(rank) * BNL + lane * 64 < p.h)
                        for (int u = 0; u < KSUB; ++u)
                            load(b_dst + lane * C::CHUNK + u * 8192, &mapB0, ncol + lane * 64,
                                 t.lo + k0 + u * BK0);
                } else {  // G6: K = 2h, first h from W1, then W3 (non-gated: K = h, W1).
                    // h % 128 == 0, so a stage never straddles the W1 | W3 boundary.
                    if (lane < BNL / 64) {
                        const bool up = p.act == 0 && k0 >= p.h;
                        const int brow = t.e * p.h + (up ? k0 - p.h : k0);
                        for (int u = 0; u < KSUB; ++u)
                            load(b_dst + lane * C::CHUNK + u * 8192, up ? &mapB1 : &mapB0,
                                 p.n_off + ncol + lane * 64, brow + u * BK0);
                    }
                }
                if (++stage == C::STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    } else if (warp == 1) {
        // =========================== MMA issuer (first CTA of a pair)
        if (leader) {
            int stage = 0;
            uint32_t phase = 0;
            int it = 0;
            for (int tile = tile0; tile < num_tiles; tile = next_tile(tile), ++it) {
                const Tile t = decode_tile(tile, s_prefix, s_segs, E, VK, m_tiles_vk, BMC, p.n_tiles, p.group_m);
                const int num_kb = VK ? (t.hi - t.lo + BK - 1) / BK : p.Kdim / BK;
                const int acc = it & 1;
                const uint32_t acc_phase = (it >> 1) & 1;
                // In a pair, the second CTA's epilogue and relay arrive from the
                // other SM: acquire at cluster scope.
                if (!warp_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag, PAIR)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * NMMA;
                const uint32_t idesc = (HALF && p.half && half_tile(t, BMC)) ? IDESC_HALF : IDESC;
                bool ok = true;
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!warp_wait(full_bar(stage), phase, abort_flag, PAIR)) {
                        ok = false;
                        break;
                    }
                    // cp.async wrote A through the generic proxy; the MMA reads it
                    // through the async proxy.
                    if constexpr (TR::A_G) fence_proxy_async_smem();
                    tc_fence_after();
                    if (lane == 0) {
                        const uint32_t a_s = sA + stage * C::A_BYTES;
                        const uint32_t b_s = sB + stage * C::B_BYTES;
#pragma unroll
                        for (int k = 0; k < BK / 16; ++k) {
                            // K-major: sub-block k / 4, 32 bytes per 16 K; MN-major: 16
                            // rows of 128 bytes per 16 K, chunks of 64 columns CHUNK apart.
                            const uint32_t ka = (k >> 2) * C::SUB_A + (k & 3) * 32;
                            const uint32_t kb2 = (k >> 2) * C::SUB_B + (k & 3) * 32;
                            const uint64_t ad = TR::A_MN ? sdesc_sw128(a_s + k * 2048, C::CHUNK, 1024)
                                                         : sdesc_sw128(a_s + ka, 16, 1024);
                            const uint64_t bd = TR::B_MN ? sdesc_sw128(b_s + k * 2048, C::CHUNK, 1024)
                                                         : sdesc_sw128(b_s + kb2, 16, 1024);
                            if constexpr (PAIR) mma_bf16_pair(d_tmem, ad, bd, idesc, (kb | k) != 0);
                            else mma_bf16(d_tmem, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
                        }
                        if constexpr (PAIR) mma_commit_pair(empty_bar(stage));
                        else mma_commit(empty_bar(stage));
                    }
                    __syncwarp();
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                if (lane == 0) {
                    if constexpr (PAIR) mma_commit_pair(tfull_bar(acc));
                    else mma_commit(tfull_bar(acc));
                }
                __syncwarp();
            }
        }
    } else if (warp < 6) {
        // =========================== epilogue (warps 2..5)
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const int row_in_tile = q * 32 + lane;
        const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
        uint8_t* stg = epi + (warp - 2) * epi_boxes<KIND, DEEP>() * 2048;  // this warp's boxes
        int nstore = 0;                           // TMA stores issued by this warp
        // G3: this warp's H ring. Slot s holds box a (and box b when gated) of one
        // chunk; the A' box follows the ring; hc counts the chunks consumed.
        constexpr bool G3 = KIND == G3_DH || KIND == G3_DH_ACT;
        constexpr int HSLOT = (KIND == G3_DH ? 2 : 1) * 2048;
        uint8_t* box_ap = stg + kHR * HSLOT;
        const uint32_t hbar0 = bar0 + 768u + 8u * kHR * (warp - 2);
        uint32_t hc = 0;
        auto h_bar = [&](uint32_t c) { return hbar0 + 8u * (c % kHR); };
        auto h_load = [&](uint32_t c, int col, int row) {  // lane 0
            const uint32_t dst = smem_u32(stg + (c % kHR) * HSLOT);
            mbar_arrive_expect_tx(h_bar(c), HSLOT);
            tma_load_2d(dst, &mapA, h_bar(c), col, row);
            if constexpr (KIND == G3_DH) tma_load_2d(dst + 2048, &mapA, h_bar(c), p.h + col, row);
        };
        int it = 0;
        for (int tile = tile0; tile < num_tiles; tile = next_tile(tile), ++it) {
            const Tile t = decode_tile(tile, s_prefix, s_segs, E, VK, m_tiles_vk, BMC, p.n_tiles, p.group_m);
            const int acc = it & 1;
            const uint32_t acc_phase = (it >> 1) & 1;
            bool stop = false;
            // G3: the warp's first row and column of H, its chunk count, and the
            // first kHR chunks, loaded while the MMA finishes the tile.
            int hrow = 0, hn0 = 0, hn = 0, hissued = 0;
            if constexpr (G3) {
                const bool hf = HALF && p.half && half_tile(t, BMC);
                hrow = hf ? t.lo + t.m_blk * BMC + rank * (BM / 2) + (q & 1) * 32
                          : t.lo + t.m_blk * BMC + rank * BM + q * 32;
                hn0 = t.n_blk * BN + (hf ? (q >> 1) * (BN / 2) : 0);
                hn = t.hi > hrow ? max(0, min(hf ? BN / 2 : BN, p.h - hn0)) / 32 : 0;
                hissued = min(kHR, hn);
                if (lane == 0 && hn > 0) {
                    bulk_wait_group_read<0>();  // earlier stores have read their slots
                    for (int c = 0; c < hissued; ++c) h_load(hc + c, hn0 + 32 * c, hrow);
                }
                __syncwarp();
            }
            if (!warp_wait(tfull_bar(acc), acc_phase, abort_flag)) {
                for (int c = 0; c < hissued; ++c) mbar_drain(h_bar(hc + c), ((hc + c) / kHR) & 1u);
                break;
            }
            tc_fence_after();
            const uint32_t tacc = tmem_base + lane_addr + acc * NMMA;
            const int rbase = t.lo + t.m_blk * BMC + rank * BM;  // VM: first row of this CTA
            const int mbase = t.m_blk * BMC + rank * BM;         // VK: first output row
            // This warp's rows and columns: 32 rows x all NMMA columns, or, in a
            // half-height pair tile, 32 of the CTA's 64 rows x half the columns
            // (TMEM column j - ccol0 holds logical column j).
            const bool half = HALF && p.half && half_tile(t, BMC);
            const int wrow0 = half ? t.lo + t.m_blk * BMC + rank * (BM / 2) + (q & 1) * 32
                                   : rbase + q * 32;
            const int ccol0 = half ? (q >> 1) * (NMMA / 2) : 0;
            const int ncolw = half ? NMMA / 2 : NMMA;
            float v[32];
            if constexpr (KIND == G1_UP || KIND == G1_UP_ACT) {
                const int row0w = wrow0;  // this warp's first row
                const int nvalid = t.hi - row0w;
                if constexpr (KIND == G1_UP_ACT) {
                    // Non-gated: 256 columns of a; H = a, A = act(a), both [TK, h].
                    const int n0 = t.n_blk * 256;
                    const size_t r0 = static_cast<size_t>(row0w > 0 ? row0w : 0);
                    __nv_bfloat16* H = static_cast<__nv_bfloat16*>(p.out0) + r0 * p.h + n0;
                    __nv_bfloat16* Aact = static_cast<__nv_bfloat16*>(p.out1) + r0 * p.h + n0;
#pragma unroll 1
                    for (int j = ccol0; j < ccol0 + ncolw; j += 32) {
                        tmem_ld32f(tacc + (j - ccol0), v);
                        if (nvalid > 0) {
                            box_put_row(stg, lane, v);
                            box_store_rows(stg, lane, H + j, p.h, nvalid);
                            if (p.act == 2) {
#pragma unroll
                                for (int i = 0; i < 32; ++i) v[i] = act_fn(2, v[i]);
                            } else {
#pragma unroll
                                for (int i = 0; i < 32; ++i) v[i] = act_fn(1, v[i]);
                            }
                            box_put_row(stg, lane, v);
                            box_store_rows(stg, lane, Aact + j, p.h, nvalid);
                        }
                    }
                } else {
                    // Hidden units n0 .. n0 + nu of this warp; gate in TMEM columns
                    // [0, nu), up in [ub, ub + nu): 128 units with up at 128, or in
                    // a half tile 64 units with up at 64 (see the B loads).
                    const int nu = half ? 64 : 128;
                    const int n0 = t.n_blk * 128 + (q >> 1) * (half ? 64 : 0);
                    const int ub = nu;
                    __nv_bfloat16* H = static_cast<__nv_bfloat16*>(p.out0) +
                                       static_cast<size_t>(row0w > 0 ? row0w : 0) * (2 * p.h) + n0;
                    __nv_bfloat16* Aact = static_cast<__nv_bfloat16*>(p.out1) +
                                          static_cast<size_t>(row0w > 0 ? row0w : 0) * p.h + n0;
#pragma unroll 1
                    for (int j = 0; j < nu; j += 32) {
                        float b[32];
                        tmem_ld32f(tacc + j, v);
                        tmem_ld32f(tacc + ub + j, b);
                        if (nvalid > 0) {
                            box_put_row(stg, lane, v);
                            box_store_rows(stg, lane, H + j, 2 * p.h, nvalid);
                            box_put_row(stg, lane, b);
                            box_store_rows(stg, lane, H + p.h + j, 2 * p.h, nvalid);
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                v[i] = __fdividef(v[i], 1.f + __expf(-v[i])) * b[i];
                            box_put_row(stg, lane, v);
                            box_store_rows(stg, lane, Aact + j, p.h, nvalid);
                        }
                    }
                }
            } else if constexpr (KIND == G2_DOWN || KIND == G6_DX) {
                const int row0w = wrow0;
                const int nvalid = t.hi - row0w;
                __nv_bfloat16* out =
                    static_cast<__nv_bfloat16*>(p.out0) +
                    static_cast<size_t>(t.out + (row0w - t.lo)) * p.ldo + t.n_blk * BN;
                // G6 adds the router term dz_r W_g[e] of its row: every row of the
                // tile belongs to expert e, so W_g[e] is one broadcast vector.
                float dzr = 0.f;
                const float* wg = nullptr;
                if constexpr (KIND == G6_DX) {
                    const int r = row0w + lane;
                    dzr = r < t.hi ? p.wrow[r] : 0.f;
                    wg = static_cast<const float*>(p.aux0) + static_cast<size_t>(t.e) * p.d +
                         p.n_off + t.n_blk * BN;
                }
#pragma unroll 1
                for (int j = ccol0; j < ccol0 + ncolw; j += 32) {
                    tmem_ld32f(tacc + (j - ccol0), v);
                    if (nvalid > 0) {
                        if constexpr (KIND == G6_DX) {
#pragma unroll
                            for (int i = 0; i < 32; i += 4) {
                                const float4 g = *reinterpret_cast<const float4*>(wg + j + i);
                                v[i] = fmaf(dzr, g.x, v[i]);
                                v[i + 1] = fmaf(dzr, g.y, v[i + 1]);
                                v[i + 2] = fmaf(dzr, g.z, v[i + 2]);
                                v[i + 3] = fmaf(dzr, g.w, v[i + 3]);
                            }
                        }
                        box_put_row(stg, lane, v);
                        box_store_rows(stg, lane, out + j, p.ldo, nvalid);
                    }
                }
            } else if constexpr (KIND == G2_SLOT) {
                // Row r of this slot's list is token tok; y_tok accumulates
                // w_{tok,k} Y in fp32 in slot order, the last slot stores bf16.
                const int r = rbase + row_in_tile;
                const bool valid = r < t.hi;
                const int tok = valid ? p.eti[r] : 0;
                const float w = valid ? p.wrow[static_cast<size_t>(tok) * p.nslot + p.slot] : 0.f;
                const bool first = p.slot == 0, last = p.slot == p.nslot - 1;
                float* arow = static_cast<float*>(p.out0) + static_cast<size_t>(tok) * p.d +
                              t.n_blk * BN;
                __nv_bfloat16* yrow = static_cast<__nv_bfloat16*>(p.out1) +
                                      static_cast<size_t>(tok) * p.d + t.n_blk * BN;
#pragma unroll 1
                for (int j = 0; j < BN; j += 32) {
                    tmem_ld32f(tacc + j, v);
                    if (valid) {
                        float a[32];
                        if (first) {
#pragma unroll
                            for (int i = 0; i < 32; ++i) a[i] = 0.f;
                        } else {
#pragma unroll
                            for (int i = 0; i < 32; i += 4) {
                                const float4 q4 = *reinterpret_cast<const float4*>(arow + j + i);
                                a[i] = q4.x;
                                a[i + 1] = q4.y;
                                a[i + 2] = q4.z;
                                a[i + 3] = q4.w;
                            }
                        }
#pragma unroll
                        for (int i = 0; i < 32; ++i) a[i] = fmaf(w, v[i], a[i]);
                        if (last) {
                            store32_bf16(yrow + j, a);
                        } else {
#pragma unroll
                            for (int i = 0; i < 32; i += 4)
                                *reinterpret_cast<float4*>(arow + j + i) =
                                    make_float4(a[i], a[i + 1], a[i + 2], a[i + 3]);
                        }
                    }
                }
            } else if constexpr (G3) {
                // dA' = dy W2_e is in TMEM, H arrives chunk by chunk in the ring.
                // dH overwrites H in its slot; dH and A' leave by TMA when all 32
                // rows of the warp are the expert's, else by row-masked stores.
                const int r = hrow + lane;
                const bool valid = r < t.hi;
                const int nvalid = t.hi - hrow;
                const float w = valid ? p.wrow[r] : 0.f;
                const size_t hs = (KIND == G3_DH ? 2 : 1) * static_cast<size_t>(p.h);
                __nv_bfloat16* dHw = static_cast<__nv_bfloat16*>(p.out0) +
                                     static_cast<size_t>(hrow) * hs + hn0;
                __nv_bfloat16* Apw = static_cast<__nv_bfloat16*>(p.out1) +
                                     static_cast<size_t>(hrow) * p.h + hn0;
                float dsum = 0.f;
                int jj = 0;
#pragma unroll 1
                for (; jj < hn; ++jj) {
                    const uint32_t c = hc + jj;
                    uint8_t* box_a = stg + (c % kHR) * HSLOT;
                    uint8_t* box_b = box_a + 2048;  // gated
                    if (!warp_wait(h_bar(c), (c / kHR) & 1u, abort_flag)) break;
                    uint4 ua[4], ub[4], ap4[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        ua[k] = *reinterpret_cast<const uint4*>(box_a + box_off(lane, k));
                    if constexpr (KIND == G3_DH) {
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            ub[k] = *reinterpret_cast<const uint4*>(box_b + box_off(lane, k));
                    }
                    tmem_ld32f(tacc + 32 * jj, v);  // dA'
                    if constexpr (KIND == G3_DH) {
                        sw_chunk(ua, ub, v, w, dsum, box_a, box_b, ap4, lane);
                    } else {
                        if (p.act == 2) ng_chunk<2>(ua, v, w, dsum, box_a, ap4, lane);
                        else ng_chunk<1>(ua, v, w, dsum, box_a, ap4, lane);
                    }
                    // The A' box and the previous chunk's slot are free once that
                    // chunk's stores have read them.
                    if (lane == 0) bulk_wait_group_read<0>();
                    __syncwarp();
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        *reinterpret_cast<uint4*>(box_ap + box_off(lane, k)) = ap4[k];
                    fence_proxy_async_smem();
                    __syncwarp();
                    // Refill the previous chunk's slot kHR chunks ahead.
                    const bool refill = jj >= 1 && hissued < hn;
                    const int col = hn0 + 32 * jj;
                    if (lane == 0) {
                        if (refill) h_load(hc + hissued, hn0 + 32 * hissued, hrow);
                        if (nvalid >= 32) {
                            tma_store_2d(&mapO, smem_u32(box_a), col, hrow);
                            if constexpr (KIND == G3_DH)
                                tma_store_2d(&mapO, smem_u32(box_b), p.h + col, hrow);
                            tma_store_2d(&mapB1, smem_u32(box_ap), col, hrow);
                            bulk_commit_group();
                        }
                    }
                    if (refill) ++hissued;
                    if (nvalid < 32) {
                        box_store_rows(box_a, lane, dHw + 32 * jj, hs, nvalid);
                        if constexpr (KIND == G3_DH)
                            box_store_rows(box_b, lane, dHw + p.h + 32 * jj, hs, nvalid);
                        box_store_rows(box_ap, lane, Apw + 32 * jj, p.h, nvalid);
                    }
                }
                if (jj < hn) {  // gave up: let this warp's loads in flight land
                    for (int k = jj; k < hissued; ++k)
                        mbar_drain(h_bar(hc + k), ((hc + k) / kHR) & 1u);
                    stop = true;
                } else if (valid) {
                    // Two partial slots per N tile: a half tile's two warps of a row
                    // write one each; otherwise the second is zero.
                    const size_t slot = 2 * static_cast<size_t>(t.n_blk) + (half ? (q >> 1) : 0);
                    p.dS_part[slot * p.TK + r] = dsum;
                    if (!half) p.dS_part[(slot + 1) * p.TK + r] = 0.f;
                }
                hc += hn;
            } else if constexpr (KIND == G4_DW2) {
                // dW2_e [d, h]: the warp's 32 rows x 32 columns at a time go through
                // a shared-memory box and one TMA store (whole lines, asynchronous).
                const bool empty = t.hi <= t.lo;
                const int grow = t.e * p.d + mbase + q * 32;  // row in [E*d, h]
                const int ncols = min(BN, p.h - t.n_blk * BN);  // the last N tile may be partial
#pragma unroll 1
                for (int j = 0; j < ncols; j += 32, ++nstore) {
                    if (empty) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = 0.f;
                    } else {
                        tmem_ld32f(tacc + j, v);
                    }
                    uint8_t* box = stg + (nstore & 1) * 2048;
                    if (lane == 0) bulk_wait_group_read<1>();  // this box's previous store read it
                    __syncwarp();
                    store32_bf16(box + lane * 64, v);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&mapO, smem_u32(box), t.n_blk * BN + j, grow);
                        bulk_commit_group();
                    }
                }
            } else if constexpr (KIND == G7_DWG) {
                // Router-gradient partial of token chunk t.e: fp32 rows
                // t.e * d + m of [nseg * d, nw], each lane its own row, 128
                // contiguous bytes per 32 columns.
                const bool empty = t.hi <= t.lo;
                const int n0 = t.n_blk * BN;
                const int ncols = min(BN, p.h - n0);  // the last N tile may be partial
                float* orow = static_cast<float*>(p.out0) +
                              (static_cast<size_t>(t.e) * p.d + mbase + q * 32 + lane) * p.ldo + n0;
#pragma unroll 1
                for (int j = 0; j < ncols; j += 32) {
                    if (empty) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = 0.f;
                    } else {
                        tmem_ld32f(tacc + j, v);
                    }
                    float4* dst = reinterpret_cast<float4*>(orow + j);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                }
            } else {  // G5: tile of (x^T dH)_e [d, 2h]; transposed into dW1/dW3 [h, d]
                // The warp's 32 d-rows x 32 n-columns are written transposed into
                // a shared-memory box [n][m] and stored with one TMA store into
                // dW1 or dW3 viewed as [E*h, d].
                const bool empty = t.hi <= t.lo;
                const bool first_half = t.n_blk < p.n_half;
                const int n0 = (t.n_blk % p.n_half) * BN;  // first column inside the half
                const int ncols = min(BN, p.h - n0);        // the last tile of a half may be partial
                const int nrow = t.e * p.h + n0;
                const int mcol = mbase + q * 32;
#pragma unroll 1
                for (int j = 0; j < ncols; j += 32, ++nstore) {
                    if (empty) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = 0.f;
                    } else {
                        tmem_ld32f(tacc + j, v);
                    }
                    uint8_t* box = stg + (nstore & 1) * 2048;
                    if (lane == 0) bulk_wait_group_read<1>();
                    __syncwarp();
                    __nv_bfloat16* bx = reinterpret_cast<__nv_bfloat16*>(box);
#pragma unroll
                    for (int i = 0; i < 32; ++i) bx[i * 32 + lane] = __float2bfloat16_rn(v[i]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(first_half ? &mapO : &mapB1, smem_u32(box), mcol, nrow + j);
                        bulk_commit_group();
                    }
                }
            }
            if (stop) break;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if constexpr (PAIR) mbar_arrive_cluster(mapa_shared(tempty_bar(acc), 0));
                else mbar_arrive(tempty_bar(acc));
            }
        }
        if (lane == 0) bulk_wait_group<0>();
        __syncwarp();
    } else if (warp < 10) {
        if constexpr (TR::A_G) {
            // =========================== cp.async gather of A (warps 6..9)
            // Shared layout is the 128-byte swizzle that the MMA descriptors
            // expect: 16-byte chunk c of a 128-byte smem row r lives at chunk
            // c ^ (r & 7). In a pair the second CTA's gathers complete on its own
            // gfull barrier, which the relay warp forwards.
            const int g = threadIdx.x - 192;  // 0..127
            const int col16 = g & 7;
            // Gathered rows: x or dy [T, d]; for G2_SLOT the SwiGLU output [TK, h].
            const size_t rowbytes = static_cast<size_t>(KIND == G2_SLOT ? p.h : p.d) * 2;
            const char* src0 = reinterpret_cast<const char*>(p.gsrc);
            auto done_bar = [&](int s) { return leader ? full_bar(s) : gfull_bar(s); };
            int stage = 0;
            uint32_t phase = 0;
            bool stop = false;
            if constexpr (!VK) {
                // K-major A: 128 rows x 64 columns; this thread copies 16-byte chunk
                // col16 of rows rb + 16 j, j = 0..7 (the same rows for every k-block
                // of a tile). The next tile's row indices load while this one streams.
                const int rb = g >> 3;
                const uint32_t soff = static_cast<uint32_t>(rb * 128 + ((col16 ^ (rb & 7)) << 4));
                auto load_idx = [&](const Tile& tt, int (&dst)[8]) {
                    const bool hf = HALF && p.half && half_tile(tt, BMC);
                    const int rcta = tt.lo + tt.m_blk * BMC + rank * (hf ? BM / 2 : BM);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int r = rcta + rb + 16 * j;
                        // A half tile's MMA reads the first 64 rows of the stage:
                        // the rest are zero-filled without a read.
                        if (hf && rb + 16 * j >= BM / 2) {
                            dst[j] = -1;
                            continue;
                        }
                        if constexpr (KIND == G2_SLOT)
                            dst[j] = r < tt.hi ? p.tim[static_cast<size_t>(p.eti[r]) * p.nslot + p.slot]
                                               : -1;
                        else
                            dst[j] = r < tt.hi ? p.eti[r] : -1;
                    }
                };
                int idx[8], nidx[8];
                int tile = tile0;
                if (tile < num_tiles)
                    load_idx(decode_tile(tile, s_prefix, s_segs, E, VK, m_tiles_vk, BMC, p.n_tiles, p.group_m), idx);
                for (; tile < num_tiles && !stop; tile = next_tile(tile)) {
                    const int ntile = next_tile(tile);
                    if (ntile < num_tiles)
                        load_idx(decode_tile(ntile, s_prefix, s_segs, E, VK, m_tiles_vk, BMC, p.n_tiles, p.group_m),
                                 nidx);
                    const int num_kb = p.Kdim / BK;
                    for (int kb = 0; kb < num_kb; ++kb) {
                        if (!warp_wait(empty_bar(stage), phase ^ 1u, abort_flag)) {
                            stop = true;
                            break;
                        }
                        const uint32_t a_dst = sA + stage * C::A_BYTES + soff;
                        const size_t coff = static_cast<size_t>(kb * BK) * 2 + col16 * 16;
#pragma unroll
                        for (int u = 0; u < KSUB; ++u)
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                const char* src =
                                    src0 + (idx[j] >= 0 ? idx[j] * rowbytes + coff + u * 128 : 0);
                                cp_async16(a_dst + u * C::SUB_A + j * 16 * 128, src,
                                           idx[j] >= 0 ? 16u : 0u);
                            }
                        cp_async_arrive_noinc(done_bar(stage));
                        if (++stage == C::STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
#pragma unroll
                    for (int j = 0; j < 8; ++j) idx[j] = nidx[j];
                }
            } else {
                // MN-major A: BK k-rows (tokens) x 128 m-columns in two 64-column
                // chunks of BK x 128 bytes; this thread copies 16-byte chunk col16 of
                // column chunk ch for token rows rb + 8 j, j < BK / 8. Work items
                // (tile, k-block) change their row indices every k-block, so the
                // indices are loaded kLook items ahead (a ring of register slots,
                // about a microsecond of lead); tiles of experts without rows have
                // no k-blocks and are skipped.
                constexpr int NR = BK / 8;             // token rows per thread and item
                constexpr int kLook = 4 * BK0 / BK;    // items of lookahead (same lead)
                const int ch = (g >> 3) & 1;
                const int rb = g >> 4;
                const uint32_t soff =
                    static_cast<uint32_t>(ch * C::CHUNK + rb * 128 + ((col16 ^ (rb & 7)) << 4));
                struct Pos {
                    int tile, kb, nkb;
                    Tile t;
                };
                auto first_from = [&](int tile, Pos& ps) -> bool {
                    for (; tile < num_tiles; tile = next_tile(tile)) {
                        const Tile tt = decode_tile(tile, s_prefix, s_segs, E, VK, m_tiles_vk, BMC, p.n_tiles, p.group_m);
                        const int nk = (tt.hi - tt.lo + BK - 1) / BK;
                        if (nk > 0) {
                            ps.tile = tile;
                            ps.kb = 0;
                            ps.nkb = nk;
                            ps.t = tt;
                            return true;
                        }
                    }
                    return false;
                };
                auto advance = [&](Pos& ps) -> bool {  // ps := the item after ps
                    if (ps.kb + 1 < ps.nkb) {
                        ++ps.kb;
                        return true;
                    }
                    return first_from(next_tile(ps.tile), ps);
                };
                auto load_idx = [&](const Pos& ps, int (&dst)[NR]) {
#pragma unroll
                    for (int j = 0; j < NR; ++j) {
                        const int r = ps.t.lo + ps.kb * BK + rb + 8 * j;
                        dst[j] = r < ps.t.hi ? p.eti[r] : -1;
                    }
                };
                Pos slot[kLook];
                int idx[kLook][NR];
                bool have[kLook];
                Pos tail{};
                bool more = first_from(tile0, tail);  // tail: the next item to prefetch
#pragma unroll
                for (int u = 0; u < kLook; ++u) {
                    have[u] = more;
                    if (more) {
                        slot[u] = tail;
                        load_idx(tail, idx[u]);
                        more = advance(tail);
                    }
                }
                bool done = !have[0];
                while (!done && !stop) {
#pragma unroll
                    for (int u = 0; u < kLook; ++u) {
                        if (!have[u]) {  // items are assigned in order: the rest are empty
                            done = true;
                            break;
                        }
                        if (!warp_wait(empty_bar(stage), phase ^ 1u, abort_flag)) {
                            stop = true;
                            break;
                        }
                        const uint32_t a_dst = sA + stage * C::A_BYTES + soff;
                        const size_t coff =
                            static_cast<size_t>(slot[u].t.m_blk * BMC + rank * BM + ch * 64) * 2 +
                            col16 * 16;
#pragma unroll
                        for (int j = 0; j < NR; ++j) {
                            const int ix = idx[u][j];
                            const char* src = src0 + (ix >= 0 ? ix * rowbytes + coff : 0);
                            cp_async16(a_dst + j * 8 * 128, src, ix >= 0 ? 16u : 0u);
                        }
                        cp_async_arrive_noinc(done_bar(stage));
                        if (++stage == C::STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                        have[u] = more;  // refill this slot kLook items ahead
                        if (more) {
                            slot[u] = tail;
                            load_idx(tail, idx[u]);
                            more = advance(tail);
                        }
                    }
                }
            }
            cp_async_wait_all();
        }
    } else {
        if constexpr (TR::A_G && PAIR) {
            // =========================== relay (warp 10 of the second CTA)
            // Waits for this CTA's gathered stage, makes it visible to the async
            // proxy, then signals the first CTA's full barrier through the bulk-
            // copy engine: a 16-byte shared-to-shared copy whose bytes complete
            // on that barrier. The relay thread never waits on a cluster fence,
            // so the signals of consecutive stages overlap.
            if (!leader) {
                int stage = 0;
                uint32_t phase = 0;
                bool stop = false;
                const uint32_t dst = mapa_shared(relay_slot, 0);
                for (int tile = tile0; tile < num_tiles && !stop; tile = next_tile(tile)) {
                    const Tile t = decode_tile(tile, s_prefix, s_segs, E, VK, m_tiles_vk, BMC, p.n_tiles, p.group_m);
                    const int num_kb = VK ? (t.hi - t.lo + BK - 1) / BK : p.Kdim / BK;
                    for (int kb = 0; kb < num_kb; ++kb) {
                        if (!warp_wait(gfull_bar(stage), phase, abort_flag)) {
                            stop = true;
                            break;
                        }
                        fence_proxy_async_smem();
                        if (lane == 0)
                            bulk_copy_s2c(dst, relay_slot, 16, mapa_shared(full_bar(stage), 0));
                        __syncwarp();
                        if (++stage == C::STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
            }
        }
    }

    // ---- teardown
    if (*abort_flag) {
        raise_error(p.err, MOE_ERR_TIMEOUT);
        // Let copies and MMAs already in flight land before the CTA exits.
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 5000000ull) {
        }
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) cluster_sync();  // no peer still reads our smem or arrives on our barriers
    tc_fence_after();
    if (warp == 1) {
        if constexpr (PAIR) tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
        else tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

// ------------------------------------------------------------------ host side
struct Maps {
    CUtensorMap a, b0, b1, o;
};

template <GemmKind KIND, int BN, int CTAS, bool DEEP = false>
cudaError_t launch_kind(const Maps& mp, const Params& prm, int max_tiles, cudaStream_t st,
                        const char* name) {
    const bool pdl = pdl_enabled(true);
    using C = Cfg<BN, CTAS, epi_boxes<KIND, DEEP>(), bk_of<KIND, CTAS, DEEP>()>;
    auto kfn = grouped_gemm_kernel<KIND, BN, CTAS, DEEP>;
    cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_TOTAL);
    if (e != cudaSuccess) return e;
    const int units = std::max(1, std::min(num_sms() / CTAS, max_tiles));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(units * CTAS);
    cfg.blockDim = dim3(threads_of<KIND, CTAS>());
    cfg.dynamicSmemBytes = C::SMEM_TOTAL;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CTAS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    LaunchScope ls(name, st);
    return cudaLaunchKernelEx(&cfg, kfn, mp.a, mp.b0, mp.b1, mp.o, prm);
}

template <GemmKind KIND, int CTAS>
cudaError_t launch_bn(int BN, const Maps& mp, const Params& prm, int max_tiles, cudaStream_t st,
                      const char* name, bool deep) {
    if constexpr (KIND == G3_DH_ACT && CTAS == 2) {
        if (deep)
            return BN == 256 ? launch_kind<KIND, 256, CTAS, true>(mp, prm, max_tiles, st, name)
                             : launch_kind<KIND, 128, CTAS, true>(mp, prm, max_tiles, st, name);
    }
    if constexpr (KIND == G1_UP || KIND == G1_UP_ACT) {
        return launch_kind<KIND, 256, CTAS>(mp, prm, max_tiles, st, name);
    } else {
        return BN == 256 ? launch_kind<KIND, 256, CTAS>(mp, prm, max_tiles, st, name)
                         : launch_kind<KIND, 128, CTAS>(mp, prm, max_tiles, st, name);
    }
}

template <GemmKind KIND>
cudaError_t launch_ctas(int ctas, int BN, const Maps& mp, const Params& prm, int max_tiles,
                        cudaStream_t st, const char* name, bool deep = false) {
    return ctas == 2 ? launch_bn<KIND, 2>(BN, mp, prm, max_tiles, st, name, deep)
                     : launch_bn<KIND, 1>(BN, mp, prm, max_tiles, st, name, deep);
}

// CTA pairs halve each SM's share of the B tile (more stages in flight, half
// the operand bytes per SM per MMA) but double the tile height. Measured on
// GB300 (Mixtral-shaped, fine-grained and skewed layers): pairs speed up the
// row-tiled GEMMs (G1, G2, G3, G6) by 2-14% once experts hold a few hundred
// rows, and the weight-gradient GEMMs (G4, G5) by 3-5% (their tile height is
// d, so they pair whenever d % 256 == 0). MOE_GEMM_CTAS=1|2 forces one mode
// wherever it is legal.
int choose_ctas(GemmKind kind, const moe_shape& s) {
    static const char* force = std::getenv("MOE_GEMM_CTAS");
    const bool vk = kind == G4_DW2 || kind == G5_DW13 || kind == G7_DWG;
    const bool ok2 = vk ? (s.d % 256 == 0) : true;
    if (force != nullptr && (force[0] == '1' || force[0] == '2'))
        return (force[0] == '2' && ok2) ? 2 : 1;
    if (vk) return ok2 ? 2 : 1;
    // A slot-wise down projection covers one slot: T rows over the experts.
    const long long rows_per_expert =
        static_cast<long long>(s.T) * (kind == G2_SLOT ? 1 : s.K) / s.E;
    return rows_per_expert >= 384 ? 2 : 1;
}

}  // namespace

int gemm_bn(GemmKind kind, const moe_shape& s) {
    switch (kind) {
        case G1_UP: return 256;  // 128 gate + 128 up columns
        case G2_DOWN:
        case G2_SLOT:
        case G6_DX: return s.d % 256 == 0 ? 256 : 128;
        case G3_DH:
        case G4_DW2:
        case G5_DW13: return s.h >= 256 ? 256 : 128;  // the last N tile (of a half) may be partial
        case G7_DWG: return dwg_plan(s).nw >= 256 ? 256 : 128;
        default: break;
    }
    return 128;
}

// Router-gradient split: B has nw = 2 * e_pad columns; the token range is cut
// into chunks (multiples of 64 tokens, at least 256 unless T is smaller, at
// most about 8192 while that needs no more than 256 chunks) so that the tile
// count is at least about 152 (two waves of CTA pairs on a 152-SM GB300) and
// no tile's reduction runs much past 64 k-blocks. The GEMM holds at most 256
// segments (kMaxE), so layers of more than 2^21 tokens take longer chunks.
// The split depends on the shape alone, so workspace sizes need no device.
DwgPlan dwg_plan(const moe_shape& s) {
    DwgPlan p{};
    p.e_pad = (s.E + 63) / 64 * 64;
    p.nw = 2 * p.e_pad;
    const int bn = p.nw >= 256 ? 256 : 128;
    const int bmc = (s.d % 256 == 0) ? 256 : 128;  // CTA pairs when d % 256 == 0
    const int tiles_per_chunk = (s.d / bmc) * ((p.nw + bn - 1) / bn);
    int n = std::max((152 + tiles_per_chunk - 1) / tiles_per_chunk, (s.T + 8191) / 8192);
    n = std::max(1, std::min(std::min(n, s.T / 256), kMaxE));
    p.chunk = ((s.T + n - 1) / n + 63) / 64 * 64;
    p.nchunks = (s.T + p.chunk - 1) / p.chunk;
    return p;
}

namespace {

// A bytes (MiB) a group of M tiles of a row-tiled GEMM keeps in L2; 0 walks
// each expert M fastest over all its M tiles. Measured on GB300 (16, 32, 64
// MiB against 0): the long layer (32,768 rows per expert, whose x rows were
// re-read from DRAM for every N panel) 59.6 -> 56.3 ms per step, its G1 and G3
// 13% faster; the skewed layer's G1 and G3 5-6% faster; Mixtral-shaped experts
// (about 1,000 rows, all in L2) unchanged.
constexpr int kGroupMB = 32;

// One launch of a GEMM problem with `ctas` CTAs per tile.
cudaError_t launch_gemm_ctas(const GemmProblem& g, int ctas, cudaStream_t st) {
    const moe_shape& s = g.s;
    // G2/G6 may cover a column chunk; their N tile must divide it.
    const int BN = (g.kind == G2_DOWN || g.kind == G6_DX) ? (g.n_cols % 256 == 0 ? 256 : 128)
                                                          : gemm_bn(g.kind, s);
    // Row capacity of the routed-row arrays (H, A, dH, A', the chunk buffer).
    const uint64_t TK = g.rows > 0 ? static_cast<uint64_t>(g.rows) : static_cast<uint64_t>(s.T) * s.K;
    const uint64_t d = s.d, h = s.h, E = s.E;
    const bool gated = s.expert == MOE_EXPERT_SWIGLU;
    const uint64_t hs = gated ? 2 * h : h;  // width of H and dH
    const uint32_t bnl = static_cast<uint32_t>(BN / ctas);  // B rows staged per CTA
    Maps mp;
    bool ok = true;
    Params prm{};
    prm.T = s.T;
    prm.TK = static_cast<int>(TK);
    prm.d = s.d;
    prm.h = s.h;
    prm.E = s.E;
    prm.act = s.expert;
    prm.slot = g.slot;
    prm.nslot = s.K;
    prm.tim = g.tim;
    prm.segs = g.segs;
    prm.eti = g.eti;
    prm.out0 = g.out0;
    prm.out1 = g.out1;
    prm.aux0 = g.aux0;
    prm.wrow = g.wrow;
    prm.dS_part = g.dS_part;
    prm.err = g.err;
    // Half-height pair tiles for an expert's last tile of at most 128 rows;
    // MOE_GEMM_HALF=0 turns them off (read at every call).
    {
        const char* f = std::getenv("MOE_GEMM_HALF");
        prm.half = (f != nullptr && f[0] == '0' && f[1] == '\0') ? 0 : 1;
    }
    // Upper bound on the tile count (rows of all experts + one partial tile
    // per expert), only used to size the persistent grid.
    const int bmc = BM * ctas;
    const int vm_mtiles = static_cast<int>(TK / bmc) + s.E;
    int max_tiles = 0;
    switch (g.kind) {
        case G1_UP:  // A = x gathered; B = W1 | W3 [E*h, d] (or W1 alone), K-major
            prm.gsrc = static_cast<const __nv_bfloat16*>(g.a_src);
            ok &= make_tmap_bf16(&mp.b0, g.b_src0, E * h, d, 64, 128);
            if (gated) ok &= make_tmap_bf16(&mp.b1, g.b_src1, E * h, d, 64, 128);
            else mp.b1 = mp.b0;
            mp.a = mp.o = mp.b0;
            if (gated && ctas == 2) {  // half tiles: 64-row boxes of W1 and W3
                ok &= make_tmap_bf16(&mp.a, g.b_src0, E * h, d, 64, 64);
                ok &= make_tmap_bf16(&mp.o, g.b_src1, E * h, d, 64, 64);
            }
            prm.Kdim = s.d;
            prm.n_tiles = gated ? s.h / 128 : s.h / 256;
            max_tiles = vm_mtiles * prm.n_tiles;
            break;
        case G2_DOWN:  // A = SwiGLU output rows; B = W2 [E*d, h], K-major
            ok &= make_tmap_bf16(&mp.a, g.a_src, TK, h, 64, 128);
            ok &= make_tmap_bf16(&mp.b0, g.b_src0, E * d, h, 64, bnl);
            mp.b1 = mp.o = mp.b0;
            if (ctas == 2) ok &= make_tmap_bf16(&mp.o, g.a_src, TK, h, 64, 64);  // half tiles
            prm.Kdim = s.h;
            prm.n_off = g.n_off;
            prm.ldo = g.n_cols;
            prm.n_tiles = g.n_cols / BN;
            max_tiles = vm_mtiles * prm.n_tiles;
            break;
        case G2_SLOT:  // A = SwiGLU output rows gathered by slot; B = W2 [E*d, h], K-major
            prm.gsrc = static_cast<const __nv_bfloat16*>(g.a_src);
            ok &= make_tmap_bf16(&mp.b0, g.b_src0, E * d, h, 64, bnl);
            mp.a = mp.b1 = mp.o = mp.b0;
            prm.Kdim = s.h;
            prm.n_tiles = s.d / BN;
            max_tiles = (s.T / bmc + s.E) * prm.n_tiles;
            break;
        case G3_DH:  // A = dy gathered; B = W2 [E*d, h] read MN-major
            // Epilogue: H [TK, hs] loaded and dH [TK, hs], A' [TK, h] stored in
            // 32 x 32 boxes with the 64-byte swizzle of its shared staging boxes.
            prm.gsrc = static_cast<const __nv_bfloat16*>(g.a_src);
            ok &= make_tmap_bf16(&mp.b0, g.b_src0, E * d, h, 64, 64);
            ok &= make_tmap_bf16(&mp.a, g.aux0, TK, hs, 32, 32, 64);
            ok &= make_tmap_bf16(&mp.o, g.out0, TK, hs, 32, 32, 64);
            ok &= make_tmap_bf16(&mp.b1, g.out1, TK, h, 32, 32, 64);
            prm.Kdim = s.d;
            prm.n_tiles = (s.h + BN - 1) / BN;
            max_tiles = vm_mtiles * prm.n_tiles;
            break;
        case G4_DW2:  // A = dy gathered (MN-major, M = d); B = A' rows [TK, h]; TMA-stored dW2
            prm.gsrc = static_cast<const __nv_bfloat16*>(g.a_src);
            ok &= make_tmap_bf16(&mp.b0, g.b_src0, TK, h, 64, 64);
            ok &= make_tmap_bf16(&mp.o, g.out0, E * d, h, 32, 32, 0);
            mp.a = mp.b1 = mp.b0;
            prm.M = s.d;
            prm.n_tiles = (s.h + BN - 1) / BN;
            max_tiles = s.E * (s.d / bmc) * prm.n_tiles;
            break;
        case G5_DW13:  // A = x gathered (MN-major, M = d); B = dH rows [TK, hs]; TMA-stored
            prm.gsrc = static_cast<const __nv_bfloat16*>(g.a_src);
            ok &= make_tmap_bf16(&mp.b0, g.b_src0, TK, hs, 64, 64);
            ok &= make_tmap_bf16(&mp.o, g.out0, E * h, d, 32, 32, 0);  // dW1
            if (gated) ok &= make_tmap_bf16(&mp.b1, g.out1, E * h, d, 32, 32, 0);  // dW3
            else mp.b1 = mp.o;
            mp.a = mp.b0;
            prm.M = s.d;
            prm.n_half = (s.h + BN - 1) / BN;
            prm.n_tiles = (gated ? 2 : 1) * prm.n_half;
            max_tiles = s.E * (s.d / bmc) * prm.n_tiles;
            break;
        case G7_DWG: {  // A = x rows (identity list); B = [dz_hi | dz_lo] [T, nw]; fp32 partials
            const int nw = dwg_plan(s).nw;
            prm.gsrc = static_cast<const __nv_bfloat16*>(g.a_src);
            ok &= make_tmap_bf16(&mp.b0, g.b_src0, static_cast<uint64_t>(s.T), nw, 64, 64);
            mp.a = mp.b1 = mp.o = mp.b0;
            prm.E = g.nseg;  // token chunks in place of experts
            prm.h = nw;
            prm.ldo = nw;
            prm.M = s.d;
            prm.n_tiles = (nw + BN - 1) / BN;
            max_tiles = g.nseg * (s.d / bmc) * prm.n_tiles;
            break;
        }
        case G6_DX:  // A = dH rows [TK, hs]; B = W1 | W3 [E*h, d] (or W1) read MN-major
            ok &= make_tmap_bf16(&mp.a, g.a_src, TK, hs, 64, 128);
            ok &= make_tmap_bf16(&mp.b0, g.b_src0, E * h, d, 64, 64);
            if (gated) ok &= make_tmap_bf16(&mp.b1, g.b_src1, E * h, d, 64, 64);
            else mp.b1 = mp.b0;
            mp.o = mp.b0;
            if (ctas == 2) ok &= make_tmap_bf16(&mp.o, g.a_src, TK, hs, 64, 64);  // half tiles
            prm.Kdim = static_cast<int>(hs);
            prm.n_off = g.n_off;
            prm.ldo = g.n_cols;
            prm.n_tiles = g.n_cols / BN;
            max_tiles = vm_mtiles * prm.n_tiles;
            break;
    }
    if (!ok) return cudaErrorInvalidValue;
    if (prm.E < 1 || prm.E > kMaxE) return cudaErrorInvalidValue;  // segments held in shared memory
    if (g.kind == G1_UP || g.kind == G2_DOWN || g.kind == G2_SLOT || g.kind == G3_DH ||
        g.kind == G6_DX) {
        // M tiles per group of the tile order, from the A bytes a group may keep
        // in L2 (MOE_GEMM_GROUP_MB overrides, read at every call).
        const char* f = std::getenv("MOE_GEMM_GROUP_MB");
        const long long mb = f != nullptr ? std::max(0, std::atoi(f)) : kGroupMB;
        const long long a_tile = static_cast<long long>(bmc) * prm.Kdim * 2;
        prm.group_m = mb > 0 ? static_cast<int>(std::max(1ll, (mb << 20) / a_tile)) : 0;
    }
    switch (g.kind) {
        case G1_UP:
            return gated ? launch_ctas<G1_UP>(ctas, BN, mp, prm, max_tiles, st, "g1_up_swiglu")
                         : launch_ctas<G1_UP_ACT>(ctas, BN, mp, prm, max_tiles, st, "g1_up_act");
        case G2_DOWN: return launch_ctas<G2_DOWN>(ctas, BN, mp, prm, max_tiles, st, "g2_down");
        case G2_SLOT: return launch_ctas<G2_SLOT>(ctas, BN, mp, prm, max_tiles, st, "g2_slot");
        case G3_DH:
            return gated ? launch_ctas<G3_DH>(ctas, BN, mp, prm, max_tiles, st, "g3_dh")
                         : launch_ctas<G3_DH_ACT>(ctas, BN, mp, prm, max_tiles, st, "g3_dh_act",
                                                  s.d >= 2048);
        case G4_DW2: return launch_ctas<G4_DW2>(ctas, BN, mp, prm, max_tiles, st, "g4_dw2");
        case G5_DW13: return launch_ctas<G5_DW13>(ctas, BN, mp, prm, max_tiles, st, "g5_dw13");
        case G6_DX: return launch_ctas<G6_DX>(ctas, BN, mp, prm, max_tiles, st, "g6_dx");
        case G7_DWG:
            return launch_ctas<G7_DWG>(ctas, BN, mp, prm, max_tiles, st, "router_dwg_mma");
        default: break;
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_gemm(const GemmProblem& g, cudaStream_t st) {
    return launch_gemm_ctas(g, choose_ctas(g.kind, g.s), st);
}

}  // namespace moe
