// Small-M W4A16 matmul: y[m, n] = Σ_g d[n, g] · Σ_{k∈g} q[n, k] · x[m, k].
//
// Source: Qwen3.5-4B quantisation study, §1 FFN example y = W x with the
// group-quantisation equation (ŵ = d·q, one d per 128 consecutive inputs) and
// §2 settings (4-bit weights, BF16 inputs).
//
// Design (HBM-bound at M ≤ 16):
//  * One warp owns 16 output rows and a contiguous range of groups; the CTA's
//    warps split the row tile's groups (split-K) and their fp32 partials are
//    summed in shared memory in a fixed order, so results are deterministic.
//  * Each lane streams one 16-byte chunk (32 codes) per row per group straight
//    from HBM into registers, `kDepth` groups ahead of use.  The stored nibble
//    order makes every 32-bit word yield four bf16x2 pairs with one shift, one
//    LOP3 and one exact bf16x2 subtract each, with no shuffles.
//  * The products q·x go through the legacy tensor-core MMA (m16n8k16, bf16 in,
//    fp32 accumulate) from registers: the 16 rows are the MMA's M, up to 8 tokens
//    its N.  At 2 B per weight-pair of HBM traffic the SM must consume about 45
//    weights per clock; one fp32 FMA per weight and token plus the decode would
//    exceed the SM's 128 lanes already at M ≈ 2, while the MMA retires 2048
//    multiply-adds per instruction.  The tensor pipe is therefore used as an ALU
//    offload here; the kernel stays bound by HBM.
//  * q is exact in bf16 and q·x is exact in fp32, so each group's partial sum is
//    the exact-product fp32 sum; it is then scaled by d in fp32.
//  * Mapping of the MMA's k index: thread `tig` of a quad feeds, at k-step s,
//    actual group offsets 32·tig + 4s + {0,1} (MMA k = 2tig, 2tig+1) and
//    32·tig + 4s + {2,3} (MMA k = 2tig+8, 2tig+9) for both A (weights) and B (x).
//    Any consistent permutation of k leaves the sum unchanged; this one makes a
//    thread's weights one 16-byte chunk and its activations 64 contiguous bytes.
#include "w4_device.cuh"
#include "w4_internal.h"

namespace w4 {
namespace {

constexpr int kGemvMaxWarps = 8;
constexpr int kDepth = 4;  // groups of weights in flight per thread

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

struct Slot {
    uint4 wa, wb;        // 16-byte code chunks of rows gid and gid+8
    uint32_t da, db;     // their bf16 scale bits (low 16 bits)
};

// MT: token tiles of 8 (1: M ≤ 8, 2: M ≤ 16).
template <int MT>
__global__ void __launch_bounds__(32 * kGemvMaxWarps)
gemv_w4_kernel(const __nv_bfloat16* __restrict__ x, int M, int64_t N, int64_t K,
               const uint8_t* __restrict__ packed, const __nv_bfloat16* __restrict__ scales,
               __nv_bfloat16* __restrict__ y) {
    __shared__ float red[kGemvMaxWarps][MT][4][32];

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int n_warps = blockDim.x >> 5;
    const int gid = lane >> 2;
    const int tig = lane & 3;
    const int64_t G = K >> 7;
    const int64_t half_k = K >> 1;

    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * 16;
    const int64_t na = n0 + gid;
    const int64_t nb = na + 8;
    const bool va = na < N;
    const bool vb = nb < N;

    const int64_t g0 = (warp * G) / n_warps;
    const int64_t g1 = ((warp + 1) * G) / n_warps;
    const int64_t ng = g1 - g0;

    const uint8_t* pa = packed + (va ? na : 0) * half_k + tig * 16;
    const uint8_t* pb = packed + (vb ? nb : 0) * half_k + tig * 16;
    const uint16_t* sa = reinterpret_cast<const uint16_t*>(scales) + (va ? na : 0) * G;
    const uint16_t* sb = reinterpret_cast<const uint16_t*>(scales) + (vb ? nb : 0) * G;

    const __nv_bfloat16* xr[MT];
    bool xv[MT];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
        const int m = mt * 8 + gid;
        xv[mt] = m < M;
        xr[mt] = x + static_cast<int64_t>(xv[mt] ? m : 0) * K + tig * 32;
    }

    auto load_slot = [&](Slot& s, int64_t g) {
        s.wa = va ? ld_stream(pa + g * 64) : make_uint4(0, 0, 0, 0);
        s.wb = vb ? ld_stream(pb + g * 64) : make_uint4(0, 0, 0, 0);
        s.da = va ? __ldg(sa + g) : 0u;
        s.db = vb ? __ldg(sb + g) : 0u;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
            if (xv[mt]) prefetch_l1(xr[mt] + g * 128);
    };

    float acc[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[mt][r] = 0.0f;

    Slot ring[kDepth];
#pragma unroll
    for (int i = 0; i < kDepth; ++i)
        if (i < ng) load_slot(ring[i], g0 + i);

    for (int64_t it = 0; it < ng; it += kDepth) {
#pragma unroll
        for (int i = 0; i < kDepth; ++i) {
            const int64_t gi = it + i;
            if (gi < ng) {
                const Slot cur = ring[i];
                if (gi + kDepth < ng) load_slot(ring[i], g0 + gi + kDepth);
                const int64_t g = g0 + gi;

                uint32_t xw[MT][16];
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        const uint4 t = xv[mt] ? ld_cached(xr[mt] + g * 128 + v * 8)
                                               : make_uint4(0, 0, 0, 0);
                        xw[mt][4 * v + 0] = t.x;
                        xw[mt][4 * v + 1] = t.y;
                        xw[mt][4 * v + 2] = t.z;
                        xw[mt][4 * v + 3] = t.w;
                    }
                }

                float cg[MT][4];
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                    for (int r = 0; r < 4; ++r) cg[mt][r] = 0.0f;

                const uint32_t wa[4] = {cur.wa.x, cur.wa.y, cur.wa.z, cur.wa.w};
                const uint32_t wb[4] = {cur.wb.x, cur.wb.y, cur.wb.z, cur.wb.w};
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    const int w = s >> 1;
                    const int h = s & 1;
                    const uint32_t a0 = code_pair_bf16x2(wa[w], 2 * h);
                    const uint32_t a2 = code_pair_bf16x2(wa[w], 2 * h + 1);
                    const uint32_t a1 = code_pair_bf16x2(wb[w], 2 * h);
                    const uint32_t a3 = code_pair_bf16x2(wb[w], 2 * h + 1);
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt)
                        mma_bf16_16816(cg[mt], a0, a1, a2, a3, xw[mt][2 * s], xw[mt][2 * s + 1]);
                }
                const float da = bf16_lo(cur.da);
                const float db = bf16_lo(cur.db);
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    acc[mt][0] = fmaf(da, cg[mt][0], acc[mt][0]);
                    acc[mt][1] = fmaf(da, cg[mt][1], acc[mt][1]);
                    acc[mt][2] = fmaf(db, cg[mt][2], acc[mt][2]);
                    acc[mt][3] = fmaf(db, cg[mt][3], acc[mt][3]);
                }
            }
        }
    }

#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int r = 0; r < 4; ++r) red[warp][mt][r][lane] = acc[mt][r];
    __syncthreads();

    for (int e = threadIdx.x; e < MT * 4 * 32; e += blockDim.x) {
        const int mt = e / 128;
        const int r = (e / 32) & 3;
        const int l = e & 31;
        float v = 0.0f;
        for (int w = 0; w < n_warps; ++w) v += red[w][mt][r][l];
        const int64_t n = n0 + (l >> 2) + (r >= 2 ? 8 : 0);
        const int m = mt * 8 + 2 * (l & 3) + (r & 1);
        if (n < N && m < M) y[static_cast<int64_t>(m) * N + n] = __float2bfloat16_rn(v);
    }
}

}  // namespace

cudaError_t launch_gemv(const void* x, int64_t M, int64_t N, int64_t K, const void* packed,
                        const void* scales, void* y, const DeviceInfo& dev, cudaStream_t stream) {
    (void)dev;
    const int64_t G = K / 128;
    const int warps = static_cast<int>(G < kGemvMaxWarps ? G : kGemvMaxWarps);
    const int64_t blocks = (N + 15) / 16;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const auto* xb = static_cast<const __nv_bfloat16*>(x);
    auto* yb = static_cast<__nv_bfloat16*>(y);
    for (int64_t m0 = 0; m0 < M; m0 += 16) {
        const int mp = static_cast<int>(M - m0 < 16 ? M - m0 : 16);
        if (mp <= 8) {
            gemv_w4_kernel<1><<<static_cast<unsigned>(blocks), 32 * warps, 0, stream>>>(
                xb + m0 * K, mp, N, K, static_cast<const uint8_t*>(packed),
                static_cast<const __nv_bfloat16*>(scales), yb + m0 * N);
        } else {
            gemv_w4_kernel<2><<<static_cast<unsigned>(blocks), 32 * warps, 0, stream>>>(
                xb + m0 * K, mp, N, K, static_cast<const uint8_t*>(packed),
                static_cast<const __nv_bfloat16*>(scales), yb + m0 * N);
        }
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace w4
