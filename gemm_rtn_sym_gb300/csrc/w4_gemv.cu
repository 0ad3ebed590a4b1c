// Small-M W4A16 matmul: y[m, n] = Σ_g d[n, g] · Σ_{k∈g} q[n, k] · x[m, k].
//
// Source: Qwen3.5-4B quantisation study, §1 FFN example y = W x with the
// group-quantisation equation (ŵ = d·q, one d per 128 consecutive inputs) and
// §2 settings (4-bit weights, BF16 inputs).
//
// Design (HBM-bound at M ≤ 16):
//  * One warp owns RT tiles of 16 output rows and a contiguous range of groups;
//    the CTA's warps split the groups (split-K) and their fp32 partials are
//    summed in shared memory in a fixed order, so results are deterministic.
//  * Each lane copies one 16-byte chunk (32 codes) per row per group from HBM
//    into a per-warp shared-memory ring with cp.async, `kDepth` groups ahead of
//    use, so nothing in flight occupies registers and several CTAs fit per SM.  The stored nibble
//    order makes every 32-bit word yield four bf16x2 pairs (136 + q) with one
//    shift and one LOP3 each, with no shuffles.  The 136·Σx offset is removed
//    exactly enough (fp32, products exact) by starting each group's
//    accumulator at −136·Σx, which one extra MMA chain per group computes for
//    all rows at once.
//  * The activations of the same groups go into the same ring (only the M real
//    token rows; lanes of padding tokens use zero fragments).  The row pitch
//    and chunk order make the fragment loads conflict-free.
//  * The products q·x go through the legacy tensor-core MMA (m16n8k16, bf16 in,
//    fp32 accumulate) from registers: the 16 rows are the MMA's M, up to 8 tokens
//    its N.  At 0.5 B per weight of HBM traffic the SM must consume about 45
//    weights per clock; one fp32 FMA per weight and token plus the decode would
//    exceed the SM's 128 lanes already at M ≈ 2, while the MMA retires 2048
//    multiply-adds per instruction.  The tensor pipe is therefore used as an ALU
//    offload here; the kernel stays bound by HBM.
//  * 136 + q is exact in bf16 and (136 + q)·x is exact in fp32, so each group's
//    partial sum is an fp32 sum of exact products; it is then scaled by d in
//    fp32.  Cancelling the offset costs about 2^-22·143·Σ|x| per group, three
//    orders of magnitude inside the 4e-3·Σ|ŵx| bound.
//  * Mapping of the MMA's k index: thread `tig` of a quad feeds, at k-step s,
//    actual group offsets 32·tig + 4s + {0,1} (MMA k = 2tig, 2tig+1) and
//    32·tig + 4s + {2,3} (MMA k = 2tig+8, 2tig+9) for both A (weights) and B (x).
//    Any consistent permutation of k leaves the sum unchanged; this one makes a
//    thread's weights one 16-byte chunk and its activations 64 contiguous bytes.
#include <mutex>

#include "w4_device.cuh"
#include "w4_internal.h"

namespace w4 {
namespace {

constexpr int kGemvMaxWarps = 8;
constexpr int kXPitch = 272;    // bytes per staged token row of one group: 256 + 16 of padding

// Position of 16-byte chunk ch (0..15) of a staged x row.  With the 272-byte
// pitch this places the eight chunks one load instruction phase reads (two
// token rows x four quads) in eight different bank groups.
__device__ __forceinline__ int x_phys_chunk(int ch) { return ch ^ ((ch >> 3) << 1); }

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Right shifts by 4, 8 and 12 bits written as the high word of a product with
// 2^28, 2^24, 2^20.  The multipliers live in constant memory, so they reach the
// integer multiply-add unit (which shares the FMA pipe) instead of becoming
// shifts on the ALU pipe, which the LOP3 decode already keeps busy.
__constant__ uint32_t kShiftMul[4] = {0u, 1u << 28, 1u << 24, 1u << 20};

// Pair i (0..3) of a stored code word as the bf16x2 value (136 + q_lo, 136 + q_hi):
// one shift and one LOP3, no subtract.  The 136·Σx offset this adds to every
// group sum is removed by starting the group's accumulator at −136·Σx.
__device__ __forceinline__ uint32_t biased_pair(uint32_t word, int i) {
    const uint32_t shifted = i == 0 ? word : __umulhi(word, kShiftMul[i]);
    return (shifted & 0x000F000Fu) ^ 0x43084308u;
}

constexpr uint32_t kMinus136x2 = 0xC308C308u;  // bf16x2 (−136, −136)

// Shared-memory ring of one warp, per stage (one group):
//   [RT tiles][16 rows][64 bytes of codes]   then   [m_real token rows][272 bytes of x]
// Codes: lane (gid, tig) reads 16 bytes at row gid and row gid+8, chunk tig; one
// load phase covers two rows x 64 contiguous bytes, so reads are conflict-free.
template <int RT>
__host__ __device__ constexpr int w_stage_bytes() { return RT * 16 * 64; }

// MT: token tiles of 8 (1: M <= 8, 2: M <= 16).  RT: 16-row tiles per warp.
// kDepth: groups in flight per warp.  MINB: CTAs per SM the register allocation
// must allow.
template <int MT, int RT, int kDepth, int MINB>
__global__ void __launch_bounds__(32 * kGemvMaxWarps, MINB)
gemv_w4_kernel(const __nv_bfloat16* __restrict__ x, int M, int64_t N, int64_t K,
               const uint8_t* __restrict__ packed, const __nv_bfloat16* __restrict__ scales,
               __nv_bfloat16* __restrict__ y) {
    extern __shared__ __align__(16) uint8_t ring_raw[];
    __shared__ float red[kGemvMaxWarps][RT][MT][4][32];

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int n_warps = blockDim.x >> 5;
    const int gid = lane >> 2;
    const int tig = lane & 3;
    const int64_t G = K >> 7;
    const int64_t half_k = K >> 1;
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * 16 * RT;
    const int m_real = M < MT * 8 ? M : MT * 8;

    const int64_t g0 = (warp * G) / n_warps;
    const int64_t g1 = ((warp + 1) * G) / n_warps;
    const int ng = static_cast<int>(g1 - g0);

    const int stage = w_stage_bytes<RT>() + m_real * kXPitch;
    const uint32_t wbase = smem_addr(ring_raw) + static_cast<uint32_t>(warp * kDepth * stage);
    const uint32_t xoff = w_stage_bytes<RT>();

    // Rows past N are clamped to row N-1 (valid memory); their outputs are dropped.
    const uint8_t* pa[RT];
    const uint8_t* pb[RT];
    const uint16_t* sa[RT];
    const uint16_t* sb[RT];
#pragma unroll
    for (int rt = 0; rt < RT; ++rt) {
        int64_t na = n0 + rt * 16 + gid, nb = na + 8;
        na = na < N ? na : N - 1;
        nb = nb < N ? nb : N - 1;
        pa[rt] = packed + na * half_k + (g0 * 64 + tig * 16);
        pb[rt] = packed + nb * half_k + (g0 * 64 + tig * 16);
        sa[rt] = reinterpret_cast<const uint16_t*>(scales) + na * G + g0;
        sb[rt] = reinterpret_cast<const uint16_t*>(scales) + nb * G + g0;
    }
    const __nv_bfloat16* xg = x + g0 * 128;

    // Stage group gi of this warp's range into ring slot `slot`.
    auto issue = [&](int slot, int gi) {
        const uint32_t st = wbase + slot * stage;
#pragma unroll
        for (int rt = 0; rt < RT; ++rt) {
            cp_async16(st + (rt * 16 + gid) * 64 + tig * 16, pa[rt] + gi * 64);
            cp_async16(st + (rt * 16 + gid + 8) * 64 + tig * 16, pb[rt] + gi * 64);
        }
        for (int q = lane; q < m_real * 16; q += 32) {
            const int r = q >> 4, ch = q & 15;
            cp_async16(st + xoff + r * kXPitch + x_phys_chunk(ch) * 16,
                       xg + static_cast<int64_t>(r) * K + gi * 128 + ch * 8);
        }
    };

    float acc[RT][MT][4];
#pragma unroll
    for (int rt = 0; rt < RT; ++rt)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[rt][mt][r] = 0.0f;

#pragma unroll
    for (int i = 0; i < kDepth; ++i) {
        if (i < ng) issue(i, i);
        cp_async_commit();
    }
    // Scales one group ahead in registers.
    uint32_t d_next[RT][2];
#pragma unroll
    for (int rt = 0; rt < RT; ++rt) {
        d_next[rt][0] = ng > 0 ? __ldg(sa[rt]) : 0u;
        d_next[rt][1] = ng > 0 ? __ldg(sb[rt]) : 0u;
    }

    for (int gi = 0; gi < ng; ++gi) {
        const int slot = gi % kDepth;
        const uint32_t st = wbase + slot * stage;
        uint32_t d_cur[RT][2];
#pragma unroll
        for (int rt = 0; rt < RT; ++rt) {
            d_cur[rt][0] = d_next[rt][0];
            d_cur[rt][1] = d_next[rt][1];
            if (gi + 1 < ng) {
                d_next[rt][0] = __ldg(sa[rt] + gi + 1);
                d_next[rt][1] = __ldg(sb[rt] + gi + 1);
            }
        }
        cp_async_wait<kDepth - 1>();
        __syncwarp();
        uint4 wv[RT][2];
#pragma unroll
        for (int rt = 0; rt < RT; ++rt) {
            wv[rt][0] = lds128(st + (rt * 16 + gid) * 64 + tig * 16);
            wv[rt][1] = lds128(st + (rt * 16 + gid + 8) * 64 + tig * 16);
        }
        uint32_t xw[MT][16];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            const int row = mt * 8 + gid;
            if (row < m_real) {
                const uint32_t xr = st + xoff + row * kXPitch;
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const uint4 t = lds128(xr + x_phys_chunk(4 * tig + v) * 16);
                    xw[mt][4 * v + 0] = t.x;
                    xw[mt][4 * v + 1] = t.y;
                    xw[mt][4 * v + 2] = t.z;
                    xw[mt][4 * v + 3] = t.w;
                }
            } else {
#pragma unroll
                for (int v = 0; v < 16; ++v) xw[mt][v] = 0u;
            }
        }
        __syncwarp();
        if (gi + kDepth < ng) issue(slot, gi + kDepth);
        cp_async_commit();

        // −136·Σ_k x[m, k] over this group, identical for every row.
        float corr[MT][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
            for (int r = 0; r < 4; ++r) corr[mt][r] = 0.0f;
#pragma unroll
            for (int s = 0; s < 8; ++s)
                mma_bf16_16816(corr[mt], kMinus136x2, kMinus136x2, kMinus136x2, kMinus136x2,
                               xw[mt][2 * s], xw[mt][2 * s + 1]);
        }
#pragma unroll
        for (int rt = 0; rt < RT; ++rt) {
            // Two independent MMA chains (even and odd k-steps) per tile.
            float ce[MT][4], co[MT][4];
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    ce[mt][r] = corr[mt][r];
                    co[mt][r] = 0.0f;
                }
            const uint32_t wa[4] = {wv[rt][0].x, wv[rt][0].y, wv[rt][0].z, wv[rt][0].w};
            const uint32_t wb[4] = {wv[rt][1].x, wv[rt][1].y, wv[rt][1].z, wv[rt][1].w};
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const int w = s >> 1;
                const int h = s & 1;
                const uint32_t a0 = biased_pair(wa[w], 2 * h);
                const uint32_t a2 = biased_pair(wa[w], 2 * h + 1);
                const uint32_t a1 = biased_pair(wb[w], 2 * h);
                const uint32_t a3 = biased_pair(wb[w], 2 * h + 1);
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    if (h == 0)
                        mma_bf16_16816(ce[mt], a0, a1, a2, a3, xw[mt][2 * s], xw[mt][2 * s + 1]);
                    else
                        mma_bf16_16816(co[mt], a0, a1, a2, a3, xw[mt][2 * s], xw[mt][2 * s + 1]);
                }
            }
            const float da = bf16_lo(d_cur[rt][0]);
            const float db = bf16_lo(d_cur[rt][1]);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                acc[rt][mt][0] = fmaf(da, ce[mt][0] + co[mt][0], acc[rt][mt][0]);
                acc[rt][mt][1] = fmaf(da, ce[mt][1] + co[mt][1], acc[rt][mt][1]);
                acc[rt][mt][2] = fmaf(db, ce[mt][2] + co[mt][2], acc[rt][mt][2]);
                acc[rt][mt][3] = fmaf(db, ce[mt][3] + co[mt][3], acc[rt][mt][3]);
            }
        }
    }
    cp_async_wait<0>();

#pragma unroll
    for (int rt = 0; rt < RT; ++rt)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int r = 0; r < 4; ++r) red[warp][rt][mt][r][lane] = acc[rt][mt][r];
    __syncthreads();

    for (int e = threadIdx.x; e < RT * MT * 4 * 32; e += blockDim.x) {
        const int rt = e / (MT * 128);
        const int mt = (e / 128) % MT;
        const int r = (e / 32) & 3;
        const int l = e & 31;
        float v = 0.0f;
        for (int w = 0; w < n_warps; ++w) v += red[w][rt][mt][r][l];
        const int64_t n = n0 + rt * 16 + (l >> 2) + (r >= 2 ? 8 : 0);
        const int m = mt * 8 + 2 * (l & 3) + (r & 1);
        if (n < N && m < M) y[static_cast<int64_t>(m) * N + n] = __float2bfloat16_rn(v);
    }
}

template <int MT, int RT, int kDepth>
int gemv_smem_bytes(int warps, int m_real) {
    return warps * kDepth * (w_stage_bytes<RT>() + m_real * kXPitch);
}

std::mutex g_attr_mutex;

template <int MT, int RT, int kDepth, int MINB>
cudaError_t launch_one(const __nv_bfloat16* x, int mp, int64_t N, int64_t K, const uint8_t* packed,
                       const __nv_bfloat16* scales, __nv_bfloat16* y, int warps, cudaStream_t stream) {
    static bool attr_set[64];
    int device = 0;
    if (cudaError_t e = cudaGetDevice(&device)) return e;
    if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(g_attr_mutex);
        if (!attr_set[device]) {
            if (cudaError_t e = cudaFuncSetAttribute(gemv_w4_kernel<MT, RT, kDepth, MINB>,
                                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                     gemv_smem_bytes<MT, RT, kDepth>(kGemvMaxWarps, MT * 8)))
                return e;
            attr_set[device] = true;
        }
    }
    const int64_t blocks = (N + 16 * RT - 1) / (16 * RT);
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const int m_real = mp < MT * 8 ? mp : MT * 8;
    gemv_w4_kernel<MT, RT, kDepth, MINB><<<static_cast<unsigned>(blocks), 32 * warps,
                                           gemv_smem_bytes<MT, RT, kDepth>(warps, m_real), stream>>>(
        x, mp, N, K, packed, scales, y);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemv(const void* x, int64_t M, int64_t N, int64_t K, const void* packed,
                        const void* scales, void* y, const DeviceInfo& dev, cudaStream_t stream) {
    const int64_t G = K / 128;
    const int warps = static_cast<int>(G < kGemvMaxWarps ? G : kGemvMaxWarps);
    // Two row tiles per warp halve the x traffic per weight when there are
    // still at least two CTAs per SM.
    const bool two_tiles = (N + 31) / 32 >= 2 * static_cast<int64_t>(dev.sm_count);
    const auto* xb = static_cast<const __nv_bfloat16*>(x);
    const auto* pk = static_cast<const uint8_t*>(packed);
    const auto* sc = static_cast<const __nv_bfloat16*>(scales);
    auto* yb = static_cast<__nv_bfloat16*>(y);
    for (int64_t m0 = 0; m0 < M; m0 += 16) {
        const int mp = static_cast<int>(M - m0 < 16 ? M - m0 : 16);
        cudaError_t e;
        if (mp <= 8)
            e = two_tiles ? launch_one<1, 2, 4, 1>(xb + m0 * K, mp, N, K, pk, sc, yb + m0 * N, warps, stream)
                          : launch_one<1, 1, 4, 1>(xb + m0 * K, mp, N, K, pk, sc, yb + m0 * N, warps, stream);
        else
            e = two_tiles ? launch_one<2, 2, 4, 1>(xb + m0 * K, mp, N, K, pk, sc, yb + m0 * N, warps, stream)
                          : launch_one<2, 1, 4, 1>(xb + m0 * K, mp, N, K, pk, sc, yb + m0 * N, warps, stream);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace w4
