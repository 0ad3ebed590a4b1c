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
constexpr int kRoundMagicBits = 0x4B400000;

// Codes of the two weights of one bf16x2 word, as the pair (slot j, slot j+4)
// of the stored word: bits 0-3 and 16-19 before the caller shifts by 4j.
//
// round_half_even(w / d) without a per-weight division.  With ρ = 1/d
// correctly rounded (CUDA's __frcp_rn), w·ρ differs from w/d by at most
// |w/d|·2^-23 < 2^-20.  Both w and d carry 8-bit significands, so a quotient
// that is not exactly a half-integer lies at least 1/512 away from every
// half-integer; rounding w·ρ to the nearest integer therefore gives
// round(w/d) everywhere except at exact ties.  Ties are found exactly: with
// q' the rounded value, e = w − q'·d is computed exactly by one FMA (q'·d has
// at most 12 significant bits and |e| ≤ d/2 + tiny), and |e| = d/2 holds
// precisely at a tie, where the even neighbour is then chosen.  The result is
// clamped to [-8, 7] only on the subnormal-scale path, where d's rounding can
// leave max|w|/d above 7.5; for d ≥ 2^-64 it never exceeds 7·(1 + 2^-8).
template <bool kTiny>
__device__ __forceinline__ uint32_t code_pair(uint32_t two, float d, float rcp, float half_d) {
    float w[2] = {bf16_lo(two), bf16_hi(two)};
    int t[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        float x = kTiny ? w[h] * 0x1p64f : w[h];
        float r = x * rcp;
        if (kTiny) r = fminf(fmaxf(r, -8.0f), 7.0f);
        const float tf = r + kRoundMagic;
        const float qf = tf - kRoundMagic;
        const float e = fmaf(-qf, d, x);
        int tb = __float_as_int(tf);
        if (fabsf(e) == half_d && (tb & 1)) tb += e > 0.0f ? 1 : -1;
        if (kTiny) tb = min(max(tb, kRoundMagicBits - 8), kRoundMagicBits + 7);
        t[h] = tb;
    }
    return __byte_perm(t[0], t[1], 0x5410) & 0x000F000Fu;
}

// Packs the 8 weights of one 16-byte chunk into the stored 32-bit code word:
// input word j holds weights 2j and 2j+1, which go to nibble slots j and j+4.
__device__ __forceinline__ uint32_t quantize_chunk(const uint4 v, const float d) {
    if (d == 0.0f) return 0u;
    const uint32_t h[4] = {v.x, v.y, v.z, v.w};
    uint32_t word = 0;
    if (d >= 0x1p-64f) {
        const float rcp = __frcp_rn(d);
        const float half_d = 0.5f * d;
#pragma unroll
        for (int j = 0; j < 4; ++j) word |= code_pair<false>(h[j], d, rcp, half_d) << (4 * j);
    } else {
        const float ds = d * 0x1p64f;  // exact: power-of-two scaling of a tiny scale
        const float rcp = __frcp_rn(ds);
        const float half_d = 0.5f * ds;
#pragma unroll
        for (int j = 0; j < 4; ++j) word |= code_pair<true>(h[j], ds, rcp, half_d) << (4 * j);
    }
    return word;
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
            const __nv_bfloat16 d16 = __float2bfloat16_rn(__fdiv_rn(bf16_lo(a), 7.0f));
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
