// RTN symmetric INT4 quantiser, group 128.
//
// Computes, for each group of 128 consecutive weights of a row (Qwen3.5-4B
// quantisation study, §1 group-quantisation equation with z = 0 and the group
// paragraph; §2 settings: minmax · symmetric, no calibration data):
//   d = bf16_rne(fp32(max|w| / 7)),  q = clamp(round_half_even(fp32(w / d)), −8, 7),
// with d = +0 and q = 0 when d is zero.
//
// Work mapping (HBM-bound streaming pass, 2 B read + 0.515625 B written per weight):
//   the matrix is a flat sequence of 16-byte chunks of 8 consecutive weights; a
//   group is 16 consecutive chunks.  A warp takes a unit of 128 chunks (8 groups,
//   2 KB): lane l loads the 64 bytes of chunks 4l..4l+3 with two 32-byte loads
//   (each warp load instruction reads whole 32-byte sectors), four lanes reduce
//   their group's max|w| with two shuffles, and lane l writes the four 32-bit
//   code words of its chunks as one 16-byte store (the stored layout keeps the
//   word of chunk c at byte 4·c).  The first lane of each group writes d.
//   The grid is one wave of resident CTAs; warps take units in turn.
//   Instruction budget: at the HBM roofline an SM must retire about 8.6 weights
//   per clock, i.e. at most 15 warp-lane instructions per weight; the packed
//   two-lane fp32 arithmetic below keeps the kernel near 5.
#include "w4_device.cuh"
#include "w4_internal.h"

namespace w4 {
namespace {

constexpr int kQuantThreads = 256;

// x + kBiasedMagic, for |x| < 2^22, is the binary32 pattern 0x4B400008 + n with
// n = round_half_even(x): 1.5·2^23 puts the units digit in the last mantissa
// bit, and the added 8 (even, so ties still go to the even neighbour) makes
// the low 16 bits of the pattern the biased code n + 8 for n in [-8, 7].
constexpr float kBiasedMagic = 12582920.0f;  // 1.5 * 2^23 + 8

// round_half_even(w / d) without a per-weight division and without a tie
// branch.  With ρ ≈ 1/d from the hardware reciprocal (relative error at most
// 2^-23, so within 2^-22):
//   q0 = fl(w·ρ),  e = fma(−q0, d, w),  q1 = fma(e, ρ, q0)
// is one residual-correction step of the quotient (P. Markstein, "Computation
// of elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
// Dev. 34(1), 1990).  For bf16 w and d (8-bit significands):
//  * q0 = (w/d)(1 + η) with |η| < 1.3·2^-22, and w − q0·d, a multiple of
//    ulp(q0)·ulp(d) of at most |w|·|η|, needs fewer than 12 significant bits,
//    so e is exact;
//  * q0 + e·ρ = w/d + (w/d − q0)·(ρd − 1) lies within |w/d|·2^-43 of w/d;
//  * at an exact tie w/d = n + ½ that is far below half an ulp of n + ½, so
//    q1 = n + ½ exactly, and the magic addition takes the even neighbour;
//  * otherwise w/d lies at least |w/d|·2^-10 (and at least 2^-9 when
//    |w| ≥ d) from every half-integer, since 2w − (2n+1)·d is a nonzero
//    multiple of the coarser of the two bf16 grids, while q1 is within
//    |w/d|·2^-23 of w/d; so q1 rounds to round(w/d).
// For d ≥ 2^-64, max|w|/d ≤ 7·(1 + 2^-8), so |n| ≤ 7 and no clamp is needed.
// Below that the scale and weights are first multiplied by 2^64 (exact) and
// q1 is clamped to [-8, 7], which covers the subnormal scales whose rounding
// can leave max|w|/d above 7.5.
__device__ __forceinline__ float rcp_approx(float d) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(d));  // d and 1/d are normal here
    return r;
}

// Packed two-lane fp32 arithmetic (one instruction for two weights).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
// The biased codes of the two lanes as (hi << 16) | lo.
__device__ __forceinline__ uint32_t f2_biased_pair(uint64_t v) {
    uint32_t lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=r"(lo), "=r"(hi) : "l"(v));
    return __byte_perm(lo, hi, 0x5410);
}

// Pairs m[j] = (code(2j+1) + 8) << 16 | (code(2j) + 8), j = 0..3, into the
// stored word: nibble slot j holds weight 2j and slot j + 4 weight 2j + 1, in
// two's complement (biased code XOR 8).
__device__ __forceinline__ uint32_t pack_word(const uint32_t (&m)[4]) {
    const uint32_t w = ((m[3] * 16u + m[2]) * 16u + m[1]) * 16u + m[0];
    return w ^ 0x88888888u;
}

// d ≥ 2^-64: the code word of chunk h[0..3] (input word j holds weights 2j and
// 2j+1), both weights of each input word at once.
__device__ __forceinline__ uint32_t chunk_word_normal(const uint32_t* h, uint64_t R, uint64_t ND, uint64_t MG) {
    uint32_t m[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint64_t X = f2_pack(bf16_lo(h[j]), bf16_hi(h[j]));
        const uint64_t Q0 = f2_mul(X, R);
        const uint64_t E = f2_fma(Q0, ND, X);
        const uint64_t Q1 = f2_fma(E, R, Q0);
        m[j] = f2_biased_pair(f2_add(Q1, MG));
    }
    return pack_word(m);
}

// d < 2^-64 (tiny or subnormal scale, or zero): weights and scale scaled by
// 2^64 (exact), quotient clamped to [-8, 7].  A zero scale is replaced by 1:
// its group has max|w| < 7·2^-134, so every quotient rounds to 0, as required.
__device__ __forceinline__ uint32_t chunk_word_tiny(const uint32_t* h, float ds, float rho) {
    uint32_t m[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t b[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const float x = (i == 0 ? bf16_lo(h[j]) : bf16_hi(h[j])) * 0x1p64f;
            const float q0 = __fmul_rn(x, rho);
            const float e = __fmaf_rn(-q0, ds, x);
            const float q1 = fminf(fmaxf(__fmaf_rn(e, rho, q0), -8.0f), 7.0f);
            b[i] = __float_as_uint(__fadd_rn(q1, kBiasedMagic));
        }
        m[j] = __byte_perm(b[0], b[1], 0x5410);
    }
    return pack_word(m);
}

// max(|a|, |b|) per bf16 half; the sign bits of the result are not |.|'s.
__device__ __forceinline__ uint32_t max_abs2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// max|w| over a lane's 32 weights, then over the 4 lanes of its group, as a
// bf16 bit pattern (in both halves).
__device__ __forceinline__ uint32_t group_absmax_bits(const uint32_t (&h)[16]) {
    uint32_t t[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) t[i] = max_abs2(h[2 * i], h[2 * i + 1]);
#pragma unroll
    for (int i = 0; i < 4; ++i) t[i] = max_abs2(t[2 * i], t[2 * i + 1]);
    uint32_t a = max_abs2(max_abs2(t[0], t[1]), max_abs2(t[2], t[3]));
    a = max_abs2(a, __byte_perm(a, 0, 0x1032));  // both halves: max over the lane
    a = max_abs2(a, __shfl_xor_sync(0xffffffffu, a, 1));
    a = max_abs2(a, __shfl_xor_sync(0xffffffffu, a, 2));
    return a & 0x7FFF7FFFu;
}

// d = bf16_rne(max|w| / 7).  a/7 is never within 1/14 of a bf16 spacing of a
// bf16 rounding midpoint (2·a/7 is an integer multiple of the spacing divided
// by 7), so rounding the fp32 product a·fl(1/7), whose error is below 2^-22
// relative, to bf16 gives the same d as rounding the exact quotient.
__device__ __forceinline__ __nv_bfloat16 group_scale(float a) {
    return __float2bfloat16_rn(a * (1.0f / 7.0f));
}

// Lane's 64 bytes: two 32-byte loads (base 32-byte aligned) or four 16-byte ones.
template <bool kWide>
__device__ __forceinline__ void load_quarter(const uint8_t* p, uint32_t (&h)[16]) {
    if (kWide) {
#pragma unroll
        for (int i = 0; i < 2; ++i)
            asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                         : "=r"(h[8 * i]), "=r"(h[8 * i + 1]), "=r"(h[8 * i + 2]), "=r"(h[8 * i + 3]),
                           "=r"(h[8 * i + 4]), "=r"(h[8 * i + 5]), "=r"(h[8 * i + 6]), "=r"(h[8 * i + 7])
                         : "l"(p + 32 * i));
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 v = ld_stream(p + 16 * i);
            h[4 * i] = v.x;
            h[4 * i + 1] = v.y;
            h[4 * i + 2] = v.z;
            h[4 * i + 3] = v.w;
        }
    }
}

template <bool kWide>
__device__ __forceinline__ void load_quarter_or_zero(const uint8_t* W, int64_t c, int64_t n_chunks, uint32_t (&h)[16]) {
    if (c < n_chunks) {
        load_quarter<kWide>(W + c * 16, h);
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) h[i] = 0u;
    }
}

// Quantises the lane's quarter group h (chunks c..c+3) and, if valid, stores
// its code words and, from the group's first lane, its scale.  Warp-collective
// (the group max is reduced with shuffles): every lane of the warp calls it.
__device__ __forceinline__ void quantize_quarter(const uint32_t (&h)[16], int64_t c, bool valid, int lane,
                                                 uint4* __restrict__ packed, __nv_bfloat16* __restrict__ scales) {
    const uint32_t a = group_absmax_bits(h);
    const __nv_bfloat16 d16 = group_scale(bf16_lo(a));
    const float d = __bfloat162float(d16);
    uint32_t word[4];
    if (d >= 0x1p-64f) {
        const float rho = rcp_approx(d);
        const uint64_t R = f2_pack(rho, rho);
        const uint64_t ND = f2_pack(-d, -d);
        const uint64_t MG = f2_pack(kBiasedMagic, kBiasedMagic);
#pragma unroll
        for (int k = 0; k < 4; ++k) word[k] = chunk_word_normal(&h[4 * k], R, ND, MG);
    } else {
        const float ds = d == 0.0f ? 1.0f : d * 0x1p64f;
        const float rho = rcp_approx(ds);
#pragma unroll
        for (int k = 0; k < 4; ++k) word[k] = chunk_word_tiny(&h[4 * k], ds, rho);
    }
    if (valid) {
        packed[c >> 2] = make_uint4(word[0], word[1], word[2], word[3]);
        if ((lane & 3) == 0) scales[c >> 4] = d16;
    }
}

template <bool kWide>
__global__ void __launch_bounds__(kQuantThreads)
quantize_rtn_kernel(const uint8_t* __restrict__ W, uint4* __restrict__ packed,
                    __nv_bfloat16* __restrict__ scales, int64_t n_chunks) {
    const int lane = threadIdx.x & 31;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t n_warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    // Units of 128 chunks (8 groups); warp w takes units w, w + n_warps, ...,
    // so every warp gets the same count to within one, and loads its next unit
    // before it quantises the current one.  The last unit may be partial: lane
    // l's quarter group, chunks c..c+3 with c = 128·unit + 4·l, is in range for
    // all four lanes of its group or for none (n_chunks is a multiple of 16).
    const int64_t n_units = (n_chunks + 127) >> 7;
    pdl_start();
    int64_t u = warp;
    if (u >= n_units) return;
    const int64_t stride = n_warps << 7;  // chunks between a warp's units
    uint32_t A[16], B[16];
    int64_t c = (u << 7) + 4 * lane;
    load_quarter_or_zero<kWide>(W, c, n_chunks, A);
    while (true) {  // u < n_units here, so the whole warp runs each body
        if (u + n_warps < n_units) load_quarter_or_zero<kWide>(W, c + stride, n_chunks, B);
        quantize_quarter(A, c, c < n_chunks, lane, packed, scales);
        u += n_warps;
        c += stride;
        if (u >= n_units) break;
        if (u + n_warps < n_units) load_quarter_or_zero<kWide>(W, c + stride, n_chunks, A);
        quantize_quarter(B, c, c < n_chunks, lane, packed, scales);
        u += n_warps;
        c += stride;
        if (u >= n_units) break;
    }
}

template <bool kWide>
int resident_ctas_per_sm() {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, quantize_rtn_kernel<kWide>, kQuantThreads, 0) !=
            cudaSuccess ||
        n < 1) {
        cudaGetLastError();
        n = 1;
    }
    return n;
}

template <bool kWide>
cudaError_t launch_quantize_t(const void* W, int64_t n_chunks, void* packed, void* scales, const DeviceInfo& dev,
                              cudaStream_t stream) {
    const int64_t per_cta = static_cast<int64_t>(kQuantThreads / 32) * 128 * 2;
    int64_t blocks = (n_chunks + per_cta - 1) / per_cta;
    // One wave of resident CTAs, each looping over its share.
    static const int occ = resident_ctas_per_sm<kWide>();
    const int64_t cap = static_cast<int64_t>(dev.sm_count) * occ;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
    cfg.blockDim = dim3(kQuantThreads, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, quantize_rtn_kernel<kWide>, static_cast<const uint8_t*>(W),
                              static_cast<uint4*>(packed), static_cast<__nv_bfloat16*>(scales), n_chunks);
}

}  // namespace

cudaError_t launch_quantize(const void* W, int64_t N, int64_t K, void* packed, void* scales,
                            const DeviceInfo& dev, cudaStream_t stream) {
    const int64_t n_chunks = N * K / 8;
    // 32-byte loads need a 32-byte aligned base; the ABI promises 16.
    if ((reinterpret_cast<uintptr_t>(W) & 31u) == 0) return launch_quantize_t<true>(W, n_chunks, packed, scales, dev, stream);
    return launch_quantize_t<false>(W, n_chunks, packed, scales, dev, stream);
}

}  // namespace w4
