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

// Nibble slot of weight e (0..7) inside its 32-bit word: even e -> e/2, odd e -> 4 + e/2.
__device__ __forceinline__ int slot_of(int e) { return (e & 1) ? 4 + (e >> 1) : (e >> 1); }

__device__ __forceinline__ uint32_t quantize_chunk(const uint4 v, const float d) {
    const uint32_t h[4] = {v.x, v.y, v.z, v.w};
    uint32_t word = 0;
    if (d == 0.0f) return 0u;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const float w = (e & 1) ? bf16_hi(h[e >> 1]) : bf16_lo(h[e >> 1]);
        int q = __float2int_rn(__fdiv_rn(w, d));  // IEEE quotient, then ties-to-even
        q = min(7, max(-8, q));
        word |= (static_cast<uint32_t>(q) & 0xFu) << (4 * slot_of(e));
    }
    return word;
}

__device__ __forceinline__ float chunk_absmax(const uint4 v) {
    const uint32_t h[4] = {v.x, v.y, v.z, v.w};
    float a = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) a = fmaxf(a, fmaxf(fabsf(bf16_lo(h[i])), fabsf(bf16_hi(h[i]))));
    return a;
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
            float a = chunk_absmax(v[u]);
#pragma unroll
            for (int off = 1; off < 16; off <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
            const __nv_bfloat16 d16 = __float2bfloat16_rn(__fdiv_rn(a, 7.0f));
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
