// RTN symmetric INT4 quantiser, group 128.
//
// Computes, for each group of 128 consecutive weights of a row (Qwen3.5-4B
// quantisation study, §1 group-quantisation equation with z = 0 and the group
// paragraph; §2 settings: minmax · symmetric, no calibration data):
//   d = bf16_rne(fp32(max|w| / 7)),  q = clamp(round_half_even(fp32(w / d)), −8, 7),
// with d = +0 and q = 0 when d is zero.
//
// Work mapping (HBM-bound streaming pass, 2 B read + 0.515625 B written per weight):
//   the matrix is a flat sequence of 16-byte chunks of 8 consecutive weights;
//   a group is 16 consecutive chunks and one half-warp owns it.  Lane l loads one
//   chunk (a warp load instruction covers 512 contiguous bytes), the half-warp
//   reduces max|w| with four shuffles, and lane l writes the 32-bit code word of
//   its 8 weights.  In the stored layout that word sits at byte 4·chunk, so the
//   warp's stores are 128 contiguous bytes.  Lane 0 of the half-warp writes d.
#include "w4_device.cuh"
#include "w4_internal.h"

namespace w4 {
namespace {

constexpr int kQuantThreads = 256;
constexpr int kQuantUnroll = 4;  // chunks in flight per thread

constexpr float kRoundMagic = 12582912.0f;  // 1.5 * 2^23: x + kRoundMagic rounds x to an integer (ties to even)

// round_half_even(w / d) without a per-weight division and without a tie
// branch.  With ρ = 1/d correctly rounded (CUDA's __frcp_rn):
//   q0 = fl(w·ρ),  e = fma(−q0, d, w),  q1 = fma(e, ρ, q0)
// is one residual-correction step of the quotient (P. Markstein, "Computation
// of elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
// Dev. 34(1), 1990).  Properties used, for bf16 w and d (8-bit significands):
//  * at an exact tie w = (n + ½)·d, the real value q0 + e·ρ differs from n + ½
//    by at most |n + ½ − q0|·2^-24 < 2^-44, far below half an ulp of n + ½, so
//    q1 = n + ½ exactly, and rounding it half-to-even gives the even neighbour;
//  * otherwise w/d lies at least 1/512 from every half-integer (2w − (2n+1)·d
//    is a nonzero multiple of the coarser of the two grids), while q1 is within
//    an ulp of w/d, so rounding q1 gives round(w/d).
// Rounding uses x + 1.5·2^23: the low bits of that sum's binary32 pattern are
// the nearest integer (ties to even) in two's complement, for |x| < 2^22.
// The result is clamped to [-8, 7] only on the subnormal-scale path, where
// d's rounding can leave max|w|/d above 7.5; for d ≥ 2^-64 it never exceeds
// 7·(1 + 2^-8).
template <bool kTiny>
struct Rounder {
    float d, rcp;
    __device__ __forceinline__ explicit Rounder(float d_) {
        d = kTiny ? d_ * 0x1p64f : d_;  // exact: power-of-two scaling of a tiny scale
        rcp = __frcp_rn(d);
    }
    // round_half_even(w / d) as the rounded-magic bit pattern.
    __device__ __forceinline__ int round_bits(float w) const {
        const float x = kTiny ? w * 0x1p64f : w;
        const float q0 = __fmul_rn(x, rcp);
        const float e = __fmaf_rn(-q0, d, x);
        float q1 = __fmaf_rn(e, rcp, q0);
        if (kTiny) q1 = fminf(fmaxf(q1, -8.0f), 7.0f);
        return __float_as_int(__fadd_rn(q1, kRoundMagic));
    }
};

// Two rounded-magic patterns -> the nibble pair (bits 0-3 and 16-19) for slots
// j and j+4 of the stored word.
__device__ __forceinline__ uint32_t pair_bits(int lo, int hi) {
    return __byte_perm(lo, hi, 0x5410) & 0x000F000Fu;
}

template <bool kTiny>
__device__ __forceinline__ uint32_t quantize_chunk_t(const uint32_t (&h)[4], float d) {
    const Rounder<kTiny> R(d);
    uint32_t word = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j)
        word |= pair_bits(R.round_bits(bf16_lo(h[j])), R.round_bits(bf16_hi(h[j]))) << (4 * j);
    return word;
}

// Packs the 8 weights of one 16-byte chunk into the stored 32-bit code word:
// input word j holds weights 2j and 2j+1, which go to nibble slots j and j+4.
__device__ __forceinline__ uint32_t quantize_chunk(const uint4 v, const float d) {
    if (d == 0.0f) return 0u;
    const uint32_t h[4] = {v.x, v.y, v.z, v.w};
    return d >= 0x1p-64f ? quantize_chunk_t<false>(h, d) : quantize_chunk_t<true>(h, d);
}

// d = bf16_rne(max|w| / 7).  a/7 is never within 1/14 of a bf16 spacing of a
// bf16 rounding midpoint (2·a/7 is an integer multiple of the spacing divided
// by 7), so rounding the fp32 product a·fl(1/7), whose error is below 2^-22
// relative, to bf16 gives the same d as rounding the exact quotient.
__device__ __forceinline__ __nv_bfloat16 group_scale(float a) {
    return __float2bfloat16_rn(a * (1.0f / 7.0f));
}

// max|w| of the chunk as a bf16 bit pattern: for non-negative finite bf16,
// the order of the values is the order of the 16-bit patterns.
__device__ __forceinline__ uint32_t chunk_absmax_bits(const uint4 v) {
    const uint32_t m = __vmaxu2(__vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu),
                                __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu));
    return max(m & 0xFFFFu, m >> 16);
}

__global__ void __launch_bounds__(kQuantThreads)
quantize_rtn_kernel(const uint4* __restrict__ W, uint32_t* __restrict__ packed,
                    __nv_bfloat16* __restrict__ scales, int64_t n_chunks) {
    const int lane = threadIdx.x & 31;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t n_warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    constexpr int64_t kStep = 32 * kQuantUnroll;

    for (int64_t base = warp * kStep; base < n_chunks; base += n_warps * kStep) {
        uint4 v[kQuantUnroll];
#pragma unroll
        for (int u = 0; u < kQuantUnroll; ++u) {
            const int64_t c = base + 32 * u + lane;
            v[u] = c < n_chunks ? ld_stream(W + c) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kQuantUnroll; ++u) {
            const int64_t c = base + 32 * u + lane;
            // n_chunks is a multiple of 16, so a half-warp is wholly in or out of range.
            uint32_t a = chunk_absmax_bits(v[u]);
#pragma unroll
            for (int off = 1; off < 16; off <<= 1) a = max(a, __shfl_xor_sync(0xffffffffu, a, off));
            const __nv_bfloat16 d16 = group_scale(bf16_lo(a));
            const float d = __bfloat162float(d16);
            const uint32_t word = quantize_chunk(v[u], d);
            if (c < n_chunks) {
                packed[c] = word;
                if ((lane & 15) == 0) scales[c >> 4] = d16;
            }
        }
    }
}

}  // namespace

cudaError_t launch_quantize(const void* W, int64_t N, int64_t K, void* packed, void* scales,
                            const DeviceInfo& dev, cudaStream_t stream) {
    const int64_t n_chunks = N * K / 8;
    const int64_t per_cta = static_cast<int64_t>(kQuantThreads) * kQuantUnroll;
    int64_t blocks = (n_chunks + per_cta - 1) / per_cta;
    const int64_t cap = static_cast<int64_t>(dev.sm_count) * 8;  // 8 resident CTAs per SM
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    quantize_rtn_kernel<<<static_cast<unsigned>(blocks), kQuantThreads, 0, stream>>>(
        static_cast<const uint4*>(W), static_cast<uint32_t*>(packed),
        static_cast<__nv_bfloat16*>(scales), n_chunks);
    return cudaGetLastError();
}

}  // namespace w4
