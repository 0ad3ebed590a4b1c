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
//
// Channel-scaled variant (same study, §2 AWQ equation W'_ij = W_ij·s_j): each
// loaded weight is first replaced by W' = bf16_rne(fp32(w·s_k)), with s_k the
// fp32 scale of its input channel, and W' is quantised as above.  s (K·4 bytes
// for the whole matrix) is read through L1; that kernel maps chunks to lanes
// differently (see quantize_rtn_scaled_kernel) so that the s reads coalesce.
//
// Also here: the input-side half of that equation, x'_j = x_j / s_j, as a
// streaming elementwise pass, x' = bf16_rne(fp32(x / s_k)) with the IEEE
// quotient.
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

// max|w| over a lane's 32 weights, then over the G/32 lanes of its group, as
// a bf16 bit pattern (in both halves).
template <int G = 128>
__device__ __forceinline__ uint32_t group_absmax_bits(const uint32_t (&h)[16]) {
    uint32_t t[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) t[i] = max_abs2(h[2 * i], h[2 * i + 1]);
#pragma unroll
    for (int i = 0; i < 4; ++i) t[i] = max_abs2(t[2 * i], t[2 * i + 1]);
    uint32_t a = max_abs2(max_abs2(t[0], t[1]), max_abs2(t[2], t[3]));
    a = max_abs2(a, __byte_perm(a, 0, 0x1032));  // both halves: max over the lane
    if (G >= 64) a = max_abs2(a, __shfl_xor_sync(0xffffffffu, a, 1));
    if (G >= 128) a = max_abs2(a, __shfl_xor_sync(0xffffffffu, a, 2));
    return a & 0x7FFF7FFFu;
}

// ---------------------------------------------------------------------------
// Asymmetric codes (the §1 equation with a free zero point z, the code of real
// zero): lo = min(0, min w), hi = max(0, max w), d = bf16_rne(fp32(fp32(hi −
// lo) / 15)) with IEEE fp32 subtraction and division, z = clamp(round(fp32(−lo
// / d)), 0, 15) (z = 8 where d = 0), q = clamp(round(w / d) + z, 0, 15), stored
// as the nibble q − 8 with the int8 zero z − 8.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t max2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ uint32_t min2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("min.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// lo = min(0, min w) and hi = max(0, max w) over the group (G/32 lanes).
template <int G>
__device__ __forceinline__ void group_range(const uint32_t (&h)[16], float& lo, float& hi) {
    uint32_t mx[8], mn[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        mx[i] = max2(h[2 * i], h[2 * i + 1]);
        mn[i] = min2(h[2 * i], h[2 * i + 1]);
    }
#pragma unroll
    for (int s = 4; s >= 1; s >>= 1)
#pragma unroll
        for (int i = 0; i < s; ++i) {
            mx[i] = max2(mx[2 * i], mx[2 * i + 1]);
            mn[i] = min2(mn[2 * i], mn[2 * i + 1]);
        }
    uint32_t a = max2(mx[0], __byte_perm(mx[0], 0, 0x1032));
    uint32_t b = min2(mn[0], __byte_perm(mn[0], 0, 0x1032));
    if (G >= 64) {
        a = max2(a, __shfl_xor_sync(0xffffffffu, a, 1));
        b = min2(b, __shfl_xor_sync(0xffffffffu, b, 1));
    }
    if (G >= 128) {
        a = max2(a, __shfl_xor_sync(0xffffffffu, a, 2));
        b = min2(b, __shfl_xor_sync(0xffffffffu, b, 2));
    }
    hi = fmaxf(bf16_lo(a), 0.0f);
    lo = fminf(bf16_lo(b), 0.0f);
}

// x + kBiasedMagic24, for |x| < 2^22, has low 16 bits round_half_even(x) + 24
// (the bias is even, so ties still go to the even neighbour).  With d ≥ 2^-64
// a normal bf16, |w/d| ≤ 15·(1 + 2^-8)/(1 − 2^-8) < 15.5, so those bits lie in
// [9, 39] and, after adding z ≤ 15, in [9, 54]: no carry between the halves.
constexpr float kBiasedMagic24 = 12582936.0f;  // 1.5 * 2^23 + 24
// Σ_j 24·16^j in both halves: removes the +24 of every nibble after packing.
constexpr uint32_t kPackBias24 = (24u * 0x1111u) * 0x00010001u;

// Pair (round(w/d) + 24) in both halves -> (q + 24), q = clamp(round + z, 0, 15).
__device__ __forceinline__ uint32_t asym_pair(uint32_t biased, uint32_t zz) {
    uint32_t v = biased + zz;
    asm("max.u16x2 %0, %0, %1;" : "+r"(v) : "r"(0x00180018u));
    asm("min.u16x2 %0, %0, %1;" : "+r"(v) : "r"(0x00270027u));
    return v;
}

// Pairs m[j] = (q(2j+1) + 24) << 16 | (q(2j) + 24) -> the stored word of nibbles
// q − 8 (two's complement), by linearity of the packing sum modulo 2^32.
__device__ __forceinline__ uint32_t pack_word_24(const uint32_t (&m)[4]) {
    const uint32_t w = ((m[3] * 16u + m[2]) * 16u + m[1]) * 16u + m[0];
    return (w - kPackBias24) ^ 0x88888888u;
}

// d ≥ 2^-64: the asymmetric code word of chunk h[0..3], zz = z in both halves.
__device__ __forceinline__ uint32_t chunk_word_asym(const uint32_t* h, uint64_t R, uint64_t ND, uint64_t MG,
                                                    uint32_t zz) {
    uint32_t m[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint64_t X = f2_pack(bf16_lo(h[j]), bf16_hi(h[j]));
        const uint64_t Q0 = f2_mul(X, R);
        const uint64_t E = f2_fma(Q0, ND, X);
        const uint64_t Q1 = f2_fma(E, R, Q0);
        m[j] = asym_pair(f2_biased_pair(f2_add(Q1, MG)), zz);
    }
    return pack_word_24(m);
}

// d < 2^-64 (or zero, replaced by 1): weights and scale scaled by 2^64 (exact).
// The quotient is clamped to [-16, 16] first, which leaves clamp(round + z,
// 0, 15) unchanged for any z in [0, 15].
__device__ __forceinline__ uint32_t chunk_word_asym_tiny(const uint32_t* h, float ds, float rho, uint32_t zz) {
    uint32_t m[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t b[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const float x = (i == 0 ? bf16_lo(h[j]) : bf16_hi(h[j])) * 0x1p64f;
            const float q0 = __fmul_rn(x, rho);
            const float e = __fmaf_rn(-q0, ds, x);
            const float q1 = fminf(fmaxf(__fmaf_rn(e, rho, q0), -16.0f), 16.0f);
            b[i] = __float_as_uint(__fadd_rn(q1, kBiasedMagic24));
        }
        m[j] = asym_pair(__byte_perm(b[0], b[1], 0x5410), zz);
    }
    return pack_word_24(m);
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

// Quantises the lane's 32 weights h (chunks c..c+3, in one group of G) and,
// if valid, stores its code words and, from the group's first lane, its scale
// (and zero).  Warp-collective (group reductions use shuffles): every lane of
// the warp calls it.
template <int G, bool kAsym>
__device__ __forceinline__ void quantize_quarter(const uint32_t (&h)[16], int64_t c, bool valid, int lane,
                                                 uint4* __restrict__ packed, __nv_bfloat16* __restrict__ scales,
                                                 int8_t* __restrict__ zeros) {
    __nv_bfloat16 d16;
    float d;
    uint32_t word[4];
    int z = 0;
    if (kAsym) {
        float lo, hi;
        group_range<G>(h, lo, hi);
        d16 = __float2bfloat16_rn(__fdiv_rn(__fsub_rn(hi, lo), 15.0f));
        d = __bfloat162float(d16);
        z = d == 0.0f ? 8 : min(15, max(0, __float2int_rn(__fdiv_rn(-lo, d))));
        const uint32_t zz = static_cast<uint32_t>(z) * 0x00010001u;
        if (d >= 0x1p-64f) {
            const float rho = rcp_approx(d);
            const uint64_t R = f2_pack(rho, rho);
            const uint64_t ND = f2_pack(-d, -d);
            const uint64_t MG = f2_pack(kBiasedMagic24, kBiasedMagic24);
#pragma unroll
            for (int k = 0; k < 4; ++k) word[k] = chunk_word_asym(&h[4 * k], R, ND, MG, zz);
        } else {
            const float ds = d == 0.0f ? 1.0f : d * 0x1p64f;
            const float rho = rcp_approx(ds);
#pragma unroll
            for (int k = 0; k < 4; ++k) word[k] = chunk_word_asym_tiny(&h[4 * k], ds, rho, zz);
        }
    } else {
        const uint32_t a = group_absmax_bits<G>(h);
        d16 = group_scale(bf16_lo(a));
        d = __bfloat162float(d16);
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
    }
    if (valid) {
        packed[c >> 2] = make_uint4(word[0], word[1], word[2], word[3]);
        if ((lane & (G / 32 - 1)) == 0) {
            const int64_t g = c / (G / 8);  // 8 weights per chunk
            scales[g] = d16;
            if (kAsym) zeros[g] = static_cast<int8_t>(z - 8);
        }
    }
}

template <bool kWide, int G, bool kAsym>
__global__ void __launch_bounds__(kQuantThreads)
quantize_rtn_kernel(const uint8_t* __restrict__ W, uint4* __restrict__ packed,
                    __nv_bfloat16* __restrict__ scales, int8_t* __restrict__ zeros, int64_t n_chunks) {
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
        quantize_quarter<G, kAsym>(A, c, c < n_chunks, lane, packed, scales, zeros);
        u += n_warps;
        c += stride;
        if (u >= n_units) break;
        if (u + n_warps < n_units) load_quarter_or_zero<kWide>(W, c + stride, n_chunks, A);
        quantize_quarter<G, kAsym>(B, c, c < n_chunks, lane, packed, scales, zeros);
        u += n_warps;
        c += stride;
        if (u >= n_units) break;
    }
}

// ---------------------------------------------------------------------------
// Channel-scaled variant.  Same units of 128 chunks and the same four lanes
// per group (lanes 4g..4g+3 take group g of the unit), but lane q = l mod 4 of
// a group takes its chunks q, q+4, q+8, q+12 instead of 4q..4q+3.  Then each
// warp load instruction reads, per group, 64 contiguous bytes of W and the 128
// contiguous bytes of s that belong to them (the 8 fp32 channel scales of each
// of 4 chunks), so an s read from L1 costs one wavefront per group rather than
// one per lane.  A group never crosses a row, so chunk q + 4i of the group is
// at row offset r0 + 4i, with r0 that of chunk q.
// ---------------------------------------------------------------------------
// The 8 fp32 channel scales of one chunk (32 bytes; 32-byte loads when s is
// 32-byte aligned, which makes every chunk's scales 32-byte aligned).
template <bool kWideS>
__device__ __forceinline__ void load_chunk_scales(const float* p, float (&sv)[8]) {
    if (kWideS) {
        uint32_t r[8];
        asm volatile("ld.global.nc.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                       "=r"(r[7])
                     : "l"(p));
#pragma unroll
        for (int j = 0; j < 8; ++j) sv[j] = __uint_as_float(r[j]);
    } else {
        const float4 a = __ldg(reinterpret_cast<const float4*>(p));
        const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
        sv[0] = a.x; sv[1] = a.y; sv[2] = a.z; sv[3] = a.w;
        sv[4] = b.x; sv[5] = b.y; sv[6] = b.z; sv[7] = b.w;
    }
}

// One chunk h[0..3] (h[j] holds weights 2j and 2j+1) <- bf16_rne(fp32(w·s_k)).
__device__ __forceinline__ void scale_chunk(uint32_t* h, const float (&sv)[8]) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint64_t P = f2_mul(f2_pack(bf16_lo(h[j]), bf16_hi(h[j])), f2_pack(sv[2 * j], sv[2 * j + 1]));
        float lo, hi;
        asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(P));
        const __nv_bfloat162 r = __floats2bfloat162_rn(lo, hi);
        h[j] = *reinterpret_cast<const uint32_t*>(&r);
    }
}

// The lane's chunks c0 + 4i, i = 0..3 (zeros when its group is out of range).
__device__ __forceinline__ void load_strided_or_zero(const uint4* __restrict__ W, int64_t c0, int64_t n_chunks,
                                                     uint32_t (&h)[16]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint4 v = c0 < n_chunks ? ld_stream(W + c0 + 4 * i) : make_uint4(0u, 0u, 0u, 0u);
        h[4 * i] = v.x;
        h[4 * i + 1] = v.y;
        h[4 * i + 2] = v.z;
        h[4 * i + 3] = v.w;
    }
}

// Scales, quantises and stores the lane's chunks c0 + 4i (row offset r0 + 4i).
// Warp-collective.  A group's chunks are all in range or all out of range
// (n_chunks is a multiple of 16), and the scale reads stay inside s even for
// a group out of range (r0 + 12 < row_chunks).
template <bool kWideS>
__device__ __forceinline__ void quantize_group_scaled(uint32_t (&h)[16], int64_t c0, int64_t r0, bool valid,
                                                      int lane, uint32_t* __restrict__ packed,
                                                      __nv_bfloat16* __restrict__ scales,
                                                      const float* __restrict__ s) {
    const float* sp = s + 8 * r0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float sv[8];
        load_chunk_scales<kWideS>(sp + 32 * i, sv);
        scale_chunk(&h[4 * i], sv);
    }
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
        uint32_t* out = packed + c0;
#pragma unroll
        for (int k = 0; k < 4; ++k) out[4 * k] = word[k];
        if ((lane & 3) == 0) scales[c0 >> 4] = d16;
    }
}

template <bool kWideS>
__global__ void __launch_bounds__(kQuantThreads)
quantize_rtn_scaled_kernel(const uint4* __restrict__ W, uint32_t* __restrict__ packed,
                           __nv_bfloat16* __restrict__ scales, int64_t n_chunks, const float* __restrict__ s,
                           int64_t row_chunks) {
    const int lane = threadIdx.x & 31;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t n_warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int64_t n_units = (n_chunks + 127) >> 7;
    pdl_start();
    int64_t u = warp;
    if (u >= n_units) return;
    const int64_t stride = n_warps << 7;
    // Chunk q of group g = l/4 of unit u: c0 = 128·u + 16·g + q, q = l mod 4.
    int64_t c = (u << 7) + 16 * (lane >> 2) + (lane & 3);
    // c mod row_chunks, kept up to date without a division per unit.
    int64_t r = c % row_chunks;
    const int64_t stride_r = stride % row_chunks;
    uint32_t A[16], B[16];
    load_strided_or_zero(W, c, n_chunks, A);
    while (true) {  // u < n_units here, so the whole warp runs each body
        if (u + n_warps < n_units) load_strided_or_zero(W, c + stride, n_chunks, B);
        quantize_group_scaled<kWideS>(A, c, r, c < n_chunks, lane, packed, scales, s);
        u += n_warps;
        c += stride;
        if ((r += stride_r) >= row_chunks) r -= row_chunks;
        if (u >= n_units) break;
        if (u + n_warps < n_units) load_strided_or_zero(W, c + stride, n_chunks, A);
        quantize_group_scaled<kWideS>(B, c, r, c < n_chunks, lane, packed, scales, s);
        u += n_warps;
        c += stride;
        if ((r += stride_r) >= row_chunks) r -= row_chunks;
        if (u >= n_units) break;
    }
}

template <typename Kernel>
int resident_ctas_per_sm(Kernel kernel) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kQuantThreads, 0) != cudaSuccess || n < 1) {
        cudaGetLastError();
        n = 1;
    }
    return n;
}

// One wave of resident CTAs (occ per SM), each looping over its share of units.
template <typename Kernel, typename... Args>
cudaError_t launch_one_wave(Kernel kernel, int occ, int64_t n_chunks, const DeviceInfo& dev, cudaStream_t stream,
                            Args... args) {
    const int64_t per_cta = static_cast<int64_t>(kQuantThreads / 32) * 128 * 2;
    int64_t blocks = (n_chunks + per_cta - 1) / per_cta;
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
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <bool kWide, int G, bool kAsym>
cudaError_t launch_quantize_t(const void* W, int64_t n_chunks, void* packed, void* scales, void* zeros,
                              const DeviceInfo& dev, cudaStream_t stream) {
    static const int occ = resident_ctas_per_sm(quantize_rtn_kernel<kWide, G, kAsym>);
    return launch_one_wave(quantize_rtn_kernel<kWide, G, kAsym>, occ, n_chunks, dev, stream,
                           static_cast<const uint8_t*>(W), static_cast<uint4*>(packed),
                           static_cast<__nv_bfloat16*>(scales), static_cast<int8_t*>(zeros), n_chunks);
}

template <bool kWide>
cudaError_t launch_quantize_g(const void* W, int64_t n_chunks, int group, void* packed, void* scales, void* zeros,
                              const DeviceInfo& dev, cudaStream_t stream) {
    const bool asym = zeros != nullptr;
    switch (group) {
        case 32:
            return asym ? launch_quantize_t<kWide, 32, true>(W, n_chunks, packed, scales, zeros, dev, stream)
                        : launch_quantize_t<kWide, 32, false>(W, n_chunks, packed, scales, zeros, dev, stream);
        case 64:
            return asym ? launch_quantize_t<kWide, 64, true>(W, n_chunks, packed, scales, zeros, dev, stream)
                        : launch_quantize_t<kWide, 64, false>(W, n_chunks, packed, scales, zeros, dev, stream);
        default:
            return asym ? launch_quantize_t<kWide, 128, true>(W, n_chunks, packed, scales, zeros, dev, stream)
                        : launch_quantize_t<kWide, 128, false>(W, n_chunks, packed, scales, zeros, dev, stream);
    }
}

template <bool kWideS>
cudaError_t launch_quantize_scaled_t(const void* W, int64_t n_chunks, void* packed, void* scales, const float* s,
                                     int64_t row_chunks, const DeviceInfo& dev, cudaStream_t stream) {
    static const int occ = resident_ctas_per_sm(quantize_rtn_scaled_kernel<kWideS>);
    return launch_one_wave(quantize_rtn_scaled_kernel<kWideS>, occ, n_chunks, dev, stream,
                           static_cast<const uint4*>(W), static_cast<uint32_t*>(packed),
                           static_cast<__nv_bfloat16*>(scales), n_chunks, s, row_chunks);
}

// x' = bf16_rne(fp32(x / s_k)) over x bf16 [M, K] seen as n8 vectors of 8
// consecutive k (K is a multiple of 8, so a vector never crosses a row).
constexpr int kScaleThreads = 256;

__global__ void __launch_bounds__(kScaleThreads)
scale_activations_kernel(const uint4* x, const float* __restrict__ s, uint4* out, int64_t n8, int64_t row_vecs) {
    // x and out may be the same buffer: each vector is read, then written, by one thread.
    pdl_start();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8; i += stride) {
        const uint4 v = x[i];
        const float4* sp = reinterpret_cast<const float4*>(s + 8 * (i % row_vecs));
        const float4 s0 = __ldg(sp), s1 = __ldg(sp + 1);
        const uint32_t in[4] = {v.x, v.y, v.z, v.w};
        const float sk[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const __nv_bfloat162 r = __floats2bfloat162_rn(__fdiv_rn(bf16_lo(in[j]), sk[2 * j]),
                                                           __fdiv_rn(bf16_hi(in[j]), sk[2 * j + 1]));
            o[j] = *reinterpret_cast<const uint32_t*>(&r);
        }
        out[i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

}  // namespace

cudaError_t launch_quantize(const void* W, int64_t N, int64_t K, int group, void* packed, void* scales, void* zeros,
                            const float* s, const DeviceInfo& dev, cudaStream_t stream) {
    const int64_t n_chunks = N * K / 8, row_chunks = K / 8;
    if (s) {
        if ((reinterpret_cast<uintptr_t>(s) & 31u) == 0)
            return launch_quantize_scaled_t<true>(W, n_chunks, packed, scales, s, row_chunks, dev, stream);
        return launch_quantize_scaled_t<false>(W, n_chunks, packed, scales, s, row_chunks, dev, stream);
    }
    // 32-byte loads need a 32-byte aligned base; the ABI promises 16.
    if ((reinterpret_cast<uintptr_t>(W) & 31u) == 0)
        return launch_quantize_g<true>(W, n_chunks, group, packed, scales, zeros, dev, stream);
    return launch_quantize_g<false>(W, n_chunks, group, packed, scales, zeros, dev, stream);
}

cudaError_t launch_scale_activations(const void* x, int64_t M, int64_t K, const float* s, void* out,
                                     const DeviceInfo& dev, cudaStream_t stream) {
    const int64_t n8 = M * K / 8;
    int64_t blocks = (n8 + kScaleThreads - 1) / kScaleThreads;
    const int64_t cap = static_cast<int64_t>(dev.sm_count) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
    cfg.blockDim = dim3(kScaleThreads, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, scale_activations_kernel, static_cast<const uint4*>(x), s,
                              static_cast<uint4*>(out), n8, K / 8);
}

}  // namespace w4
