// Device pieces shared by the small-M matmul kernels (single matrix with
// cluster split-K, and the grouped persistent kernel): stage geometry, the
// pair decode, the activation fragment loads and one group's MMA work.
// See w4_gemv.cu for the design.
#pragma once

#include "w4_device.cuh"

namespace w4 {
namespace gemv {

constexpr int kTiles = 4;                // 16-row tiles per CTA
constexpr int kRowsCta = 16 * kTiles;    // 64 weight rows per CTA
constexpr int kStageGroups = 4;          // groups per stage
constexpr int kMaxSplit = 8;
constexpr int kTpw = 4;  // row tiles per consumer warp: each warp takes one group of a stage for all 64 rows
constexpr int kMaxPassRows = 32;  // token rows of one pass (MT = 4)

// TPW: row tiles per consumer warp.  Consumer warp c takes group c % 4 of every
// stage for tiles (c / 4)·TPW .. +TPW-1, so 16 / TPW consumer warps per CTA.
template <int TPW>
struct Warps {
    static constexpr int kConsumers = kStageGroups * (kTiles / TPW);
    static constexpr int kThreads = 32 * (1 + kConsumers);
};
constexpr int kCodeStageBytes = kStageGroups * kRowsCta * 64;  // 16 KB: [group][row][64 B]

// MT: token tiles of 8 per pass (1..4, i.e. up to 32 token rows).
template <int MT>
struct Cfg {
    static constexpr int kXRows = 8 * MT;                               // token rows staged
    static constexpr int kXStageBytes = 2 * kStageGroups * kXRows * 128;  // [k-block][row][128 B]
    // Ring depth: two CTAs per SM must fit (a 24 KB stage at MT = 1 up to 48 KB at MT = 4).
    static constexpr int kStages = MT == 1 ? 4 : (MT == 2 ? 3 : 2);
    static constexpr int kStageBytes = kCodeStageBytes + kXStageBytes;
    // Two CTAs per SM, each with its own TMA producer (one issuing thread per
    // SM does not reach the HBM rate with copies of this size).
    static constexpr int kSmemBytes = kStages * kStageBytes + 2048;
};

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Pair i (0..3) of a stored code word as the bf16x2 value (136 + q_lo, 136 + q_hi):
// one shift and one LOP3, no subtract.  The 136·Σx offset this adds to every
// group sum is removed by starting the group's accumulator at −136·Σx.
template <int I>
__device__ __forceinline__ uint32_t biased_pair(uint32_t word) {
    uint32_t r, t = word;
    if (I != 0) asm("shr.b32 %0, %1, %2;" : "=r"(t) : "r"(word), "n"(4 * I));
    // (t & 0x000F000F) ^ 0x43084308 as one three-input logic op (LUT 0x6A = (a & b) ^ c).
    asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(r) : "r"(t), "n"(0x000F000F), "r"(0x43084308u));
    return r;
}

constexpr uint32_t kMinus136x2 = 0xC308C308u;  // bf16x2 (−136, −136)

// Activation fragments of one stage: token rows mt·8 + gid, the 64 contiguous
// bytes (32 k) of this lane's part of the group, from the 128-byte-swizzled
// [k-block][row][128 B] tile with kXRows rows per block.  The swizzle XORs the
// 16-byte chunk index with the 128-byte line's index in its 1024-byte atom
// (address bits 7..9; stages are 1024-byte aligned).  Rows at or past kXRows
// are not staged and read as zeros.
template <int MT, int kXRows>
__device__ __forceinline__ void load_x_frags(uint32_t (&xw)[MT][16], uint32_t st_x_blk, int gid, int tig) {
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
        const int r = mt * 8 + gid;
        const uint32_t rowa = st_x_blk + r * 128;
        if (kXRows < 8 && r >= kXRows) {
#pragma unroll
            for (int j = 0; j < 16; ++j) xw[mt][j] = 0u;
            continue;
        }
        const uint32_t line = (rowa >> 7) & 7u;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const uint32_t c = static_cast<uint32_t>(4 * (tig & 1) + v);
            const uint4 q = lds128(rowa + ((c ^ line) << 4));
            xw[mt][4 * v + 0] = q.x;
            xw[mt][4 * v + 1] = q.y;
            xw[mt][4 * v + 2] = q.z;
            xw[mt][4 * v + 3] = q.w;
        }
    }
}

// Word w (0..3) of a 16-byte chunk.
__device__ __forceinline__ uint32_t word_of(const uint4 v, int w) {
    return w == 0 ? v.x : w == 1 ? v.y : w == 2 ? v.z : v.w;
}

// The biased A fragment of k-step 2w + H from word w of rows gid (wa) and
// gid + 8 (wb): pairs 2H and 2H + 1 of each word.
template <int H>
__device__ __forceinline__ void biased_frag(uint32_t wa, uint32_t wb, uint32_t (&f)[4]) {
    f[0] = biased_pair<2 * H>(wa);
    f[1] = biased_pair<2 * H>(wb);
    f[2] = biased_pair<2 * H + 1>(wa);
    f[3] = biased_pair<2 * H + 1>(wb);
}

// One group of one stage for TPW row tiles: acc += d · (Σ (136 + q)·x − 136·Σx).
// The k-steps run outermost and the row tiles inside them, so an MMA's
// accumulator was last written TPW MMAs earlier (tile-by-tile order chained
// eight dependent MMAs; this order measured 2–5 % faster on the grouped
// layers), and the −136·Σx chain is added at the end instead of seeding
// every tile.
template <int MT, int TPW>
__device__ __forceinline__ void group_math(float (&acc)[TPW][MT][4], const uint32_t (&xw)[MT][16],
                                           const uint4 (&wv)[TPW][2], const float (&d)[TPW][2]) {
    float corr[MT][4];  // −136·Σ_k x[m, k] over this group, identical for every row
    float cg[TPW][MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            corr[mt][r] = 0.0f;
#pragma unroll
            for (int rt = 0; rt < TPW; ++rt) cg[rt][mt][r] = 0.0f;
        }
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
        const int w = ks >> 1;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
            mma_bf16_16816(corr[mt], kMinus136x2, kMinus136x2, kMinus136x2, kMinus136x2, xw[mt][2 * ks],
                           xw[mt][2 * ks + 1]);
#pragma unroll
        for (int rt = 0; rt < TPW; ++rt) {
            uint32_t f[4];
            if (ks & 1)
                biased_frag<1>(word_of(wv[rt][0], w), word_of(wv[rt][1], w), f);
            else
                biased_frag<0>(word_of(wv[rt][0], w), word_of(wv[rt][1], w), f);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
                mma_bf16_16816(cg[rt][mt], f[0], f[1], f[2], f[3], xw[mt][2 * ks], xw[mt][2 * ks + 1]);
        }
    }
#pragma unroll
    for (int rt = 0; rt < TPW; ++rt) {
        const float da = d[rt][0];  // rows gid and gid + 8 of the tile
        const float db = d[rt][1];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            acc[rt][mt][0] = fmaf(da, cg[rt][mt][0] + corr[mt][0], acc[rt][mt][0]);
            acc[rt][mt][1] = fmaf(da, cg[rt][mt][1] + corr[mt][1], acc[rt][mt][1]);
            acc[rt][mt][2] = fmaf(db, cg[rt][mt][2] + corr[mt][2], acc[rt][mt][2]);
            acc[rt][mt][3] = fmaf(db, cg[rt][mt][3] + corr[mt][3], acc[rt][mt][3]);
        }
    }
}

// Affine variant (group sizes 32 / 64 / 128, optional zero points): every A
// operand is dequantised, ŵ = bf16(d·((136 + c) − (136 + z'))) with c the
// stored code and z' the stored zero: the subtraction is exact, the product
// rounds once, as in the tensor-core path.  A thread's 32 codes of a group
// (one 16-byte chunk) always lie inside one group of 32 or 64, so each thread
// needs one (d, 136 + z') pair per row: d2[rt][h] and off2[rt][h] hold them as
// bf16x2 for rows gid (h = 0) and gid + 8 (h = 1).  No offset MMA chain and no
// per-group scaling: the MMA accumulates straight into acc.
__device__ __forceinline__ uint32_t affine_pair(uint32_t biased, uint32_t off2, uint32_t d2) {
    uint32_t r;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(biased), "r"(off2));
    asm("mul.rn.bf16x2 %0, %0, %1;" : "+r"(r) : "r"(d2));
    return r;
}

// One row tile of the affine variant: wa / wb are the 16-byte chunks of rows
// gid and gid + 8.
template <int MT>
__device__ __forceinline__ void tile_math_affine(float (&acc)[MT][4], const uint32_t (&xw)[MT][16], const uint4 wa4,
                                                 const uint4 wb4, uint32_t da, uint32_t db, uint32_t oa, uint32_t ob) {
    const uint32_t wa[4] = {wa4.x, wa4.y, wa4.z, wa4.w};
    const uint32_t wb[4] = {wb4.x, wb4.y, wb4.z, wb4.w};
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        const uint32_t a0 = affine_pair(biased_pair<0>(wa[w]), oa, da);
        const uint32_t a2 = affine_pair(biased_pair<1>(wa[w]), oa, da);
        const uint32_t a1 = affine_pair(biased_pair<0>(wb[w]), ob, db);
        const uint32_t a3 = affine_pair(biased_pair<1>(wb[w]), ob, db);
        const uint32_t b0 = affine_pair(biased_pair<2>(wa[w]), oa, da);
        const uint32_t b2 = affine_pair(biased_pair<3>(wa[w]), oa, da);
        const uint32_t b1 = affine_pair(biased_pair<2>(wb[w]), ob, db);
        const uint32_t b3 = affine_pair(biased_pair<3>(wb[w]), ob, db);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            mma_bf16_16816(acc[mt], a0, a1, a2, a3, xw[mt][4 * w], xw[mt][4 * w + 1]);
            mma_bf16_16816(acc[mt], b0, b1, b2, b3, xw[mt][4 * w + 2], xw[mt][4 * w + 3]);
        }
    }
}

template <int MT, int TPW>
__device__ __forceinline__ void group_math_affine(float (&acc)[TPW][MT][4], const uint32_t (&xw)[MT][16],
                                                  const uint4 (&wv)[TPW][2], const uint32_t (&d2)[TPW][2],
                                                  const uint32_t (&off2)[TPW][2]) {
    // k-steps outermost, row tiles inside (as in group_math): consecutive MMAs
    // update different tiles' accumulators (10 % faster for the affine
    // formats at 16 token rows, 1.5 % for the symmetric grouped stack).
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
        const int w = ks >> 1;
#pragma unroll
        for (int rt = 0; rt < TPW; ++rt) {
            uint32_t f[4];
            if (ks & 1)
                biased_frag<1>(word_of(wv[rt][0], w), word_of(wv[rt][1], w), f);
            else
                biased_frag<0>(word_of(wv[rt][0], w), word_of(wv[rt][1], w), f);
            f[0] = affine_pair(f[0], off2[rt][0], d2[rt][0]);
            f[1] = affine_pair(f[1], off2[rt][1], d2[rt][1]);
            f[2] = affine_pair(f[2], off2[rt][0], d2[rt][0]);
            f[3] = affine_pair(f[3], off2[rt][1], d2[rt][1]);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
                mma_bf16_16816(acc[rt][mt], f[0], f[1], f[2], f[3], xw[mt][2 * ks], xw[mt][2 * ks + 1]);
        }
    }
}

// The same with each row tile's 16-byte chunks loaded from the stage just
// before use (fewer live registers at 24 or 32 token rows).
template <int MT, int TPW>
__device__ __forceinline__ void group_math_affine_lds(float (&acc)[TPW][MT][4], const uint32_t (&xw)[MT][16],
                                                      uint32_t w_addr, const uint32_t (&d2)[TPW][2],
                                                      const uint32_t (&off2)[TPW][2]) {
#pragma unroll
    for (int rt = 0; rt < TPW; ++rt) {
        const uint4 wa = lds128(w_addr + rt * 16 * 64);
        const uint4 wb = lds128(w_addr + rt * 16 * 64 + 8 * 64);
        tile_math_affine<MT>(acc[rt], xw, wa, wb, d2[rt][0], d2[rt][1], off2[rt][0], off2[rt][1]);
    }
}

// Symmetric codes with 16 or more token rows per pass: there the legacy MMA
// pipe, not the decode, bounds the kernel, so each weight is dequantised to
// bf16(d·q) (the affine path with zero 0) instead of spending an offset MMA
// chain and per-group fp32 scaling on the 136 bias (measured 4 % faster on
// the grouped stack at M = 16, and faster at 24 and 32).
template <int MT>
struct Dequant {
    static constexpr bool value = MT >= 2;
};

}  // namespace gemv
}  // namespace w4
