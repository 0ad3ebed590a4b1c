// Small-M W4A16 matmul: y[m, n] = Σ_g d[n, g] · Σ_{k∈g} q[n, k] · x[m, k].
//
// Source: Qwen3.5-4B quantisation study, §1 FFN example y = W x with the
// group-quantisation equation (ŵ = d·q, one d per 128 consecutive inputs) and
// §2 settings (4-bit weights, BF16 inputs).
//
// Design (HBM-bound at M ≤ 16):
//  * A CTA owns 64 output rows (four 16-row tiles) and a range of groups.  One
//    producer thread streams, by TMA, stages of four groups: a 16 KB code tile
//    ([group][row][64 B], from a 3-D view of the packed matrix) and the
//    matching activation tile (16-row boxes of 64-k blocks, 128-byte swizzle;
//    token rows >= M read as zeros), into a 3-4 deep shared-memory ring.  Two
//    CTAs share an SM, so two threads per SM keep the copies flowing.
//  * Four consumer warps each take one group of every stage for all four row
//    tiles, so the activation fragments are loaded once per group and reused
//    for 64 rows; the warps' fp32 partials are summed in shared memory in a
//    fixed order at the end.  Small matrices are split along K over the CTAs
//    of a thread-block cluster; each rank then adds one slice of the outputs
//    over all ranks' partials through distributed shared memory, in rank
//    order: deterministic, no global scratch.
//  * The stored nibble order makes every 32-bit word yield four bf16x2 pairs
//    (136 + q) with one shift and one LOP3 each, with no shuffles; the
//    136·Σx offset is removed by starting each group's accumulator at −136·Σx,
//    which one extra MMA chain per group computes for all rows at once.
//  * The products go through the legacy tensor-core MMA (m16n8k16, bf16 in,
//    fp32 accumulate) from registers: the 16 rows are the MMA's M, up to 8
//    tokens its N.  At 0.5 B per weight of HBM traffic each SM must consume
//    about 45 weights per clock; one fp32 FMA per weight and token plus the
//    decode would exceed the SM's lanes already at M ≈ 2.  The tcgen05 MMA is
//    no help at this size: one 128 x N x 16 instruction costs at least about
//    46 cycles for any N <= 64 (measured), i.e. at most ~44 weights per clock
//    per SM before any other work.  The legacy MMA from registers is used as
//    an ALU offload here; the kernel stays bound by HBM.
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
#include "w4_gemv_common.cuh"
#include "w4_internal.h"
#include "w4_tcgen05.cuh"

namespace w4 {
namespace {

using namespace gemv;

struct GemvArgs {
    const uint16_t* scales;
    const int8_t* zeros;  // affine variant only; nullptr: symmetric
    int64_t row_groups;   // affine variant: scales (and zeros) per row, K / group
    __nv_bfloat16* y;
    int M;  // token rows of this pass, 1..32
    int64_t N, K;
    int split;
    unsigned* status;
};

// MT: token tiles of 8 (1..4: M <= 8, 16, 24, 32 per pass).  QG: 0 for the symmetric
// group-128 format (offset MMA chain, one fp32 scaling per group); 32, 64 or
// 128 for the affine variant (group size QG, optional zero points).
template <int MT, int TPW, int QG>
__global__ void __launch_bounds__(Warps<TPW>::kThreads, 2)
gemv_w4_kernel(const __grid_constant__ CUtensorMap tmap_codes, const __grid_constant__ CUtensorMap tmap_x,
               const GemvArgs args) {
    using C = Cfg<MT>;
    constexpr int kConsumers = Warps<TPW>::kConsumers;
    constexpr int kThreads = Warps<TPW>::kThreads;
    // Every weight dequantised to bf16 before its MMA (affine formats, and the
    // symmetric format at 16 or more token rows).
    constexpr bool kDeq = QG != 0 || Dequant<MT>::value;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    const uint32_t bar_base = base + C::kStages * C::kStageBytes;
    auto full = [&](int s) { return bar_base + 8u * s; };
    auto empty = [&](int s) { return bar_base + 8u * (C::kStages + s); };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int gid = lane >> 2;
    const int tig = lane & 3;
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kRowsCta;
    const int64_t G = args.K >> 7;
    const int split = args.split;
    const uint32_t rank = split > 1 ? cluster_rank() : 0u;
    const int64_t gs = (static_cast<int64_t>(rank) * G) / split;
    const int64_t ge = (static_cast<int64_t>(rank + 1) * G) / split;
    const int ng = static_cast<int>(ge - gs);
    const int nt = (ng + kStageGroups - 1) / kStageGroups;
    const int M = args.M;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 32 * kConsumers);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_async_smem();
    }
    __syncthreads();
    pdl_start();

    bool ok = true;
    float acc[TPW][MT][4];
#pragma unroll
    for (int rt = 0; rt < TPW; ++rt)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[rt][mt][r] = 0.0f;

    if (warp == 0) {
        // -------------------------------------------------- producer: one thread, two copies per stage
        if (lane == 0) {
            int issued = 0;
            for (int t = 0; t < nt; ++t) {
                const int s = t % C::kStages;
                if (!mbar_wait_suspend(empty(s), (static_cast<uint32_t>(t / C::kStages) & 1u) ^ 1u)) {
                    ok = false;
                    break;
                }
                const uint32_t st = base + s * C::kStageBytes;
                const int g = static_cast<int>(gs + t * kStageGroups);
                mbar_arrive_expect_tx(full(s), C::kStageBytes);
                tma_load_3d(st, &tmap_codes, 0, static_cast<int>(n0), g, full(s));
                tma_load_3d(st + kCodeStageBytes, &tmap_x, 0, 0, 2 * g, full(s));
                issued = t + 1;
            }
            if (!ok) {
                record_status(args.status, kStatusTimeout);
                for (int t = issued > C::kStages ? issued - C::kStages : 0; t < issued; ++t)
                    mbar_wait(full(t % C::kStages), static_cast<uint32_t>(t / C::kStages) & 1u);
            }
        }
    } else {
        // -------------------------------------------------- consumers: decode + legacy MMA
        const int cw = (warp - 1) % kStageGroups;          // this warp's group within every stage
        const int tile0 = ((warp - 1) / kStageGroups) * TPW;  // first of its row tiles
        // Scales of rows gid / gid+8 of each tile, for this warp's group of a stage.
        // Affine variant: the group of size QG holding this thread's chunk
        // (k 32·tig .. 32·tig + 31 of the 128-k block) is 128/QG·g + sub.
        constexpr int kSub = QG == 0 ? 1 : 128 / QG;
        const int sub = QG == 32 ? tig : (QG == 64 ? (tig >> 1) : 0);
        const int64_t rg = QG == 0 ? G : args.row_groups;
        const uint16_t* srow[TPW][2];
        const int8_t* zrow[TPW][2];
#pragma unroll
        for (int rt = 0; rt < TPW; ++rt)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                int64_t n = n0 + (tile0 + rt) * 16 + gid + 8 * h;
                if (n >= args.N) n = args.N - 1;
                srow[rt][h] = args.scales + n * rg + (QG == 0 ? 0 : sub);
                zrow[rt][h] = QG != 0 && args.zeros ? args.zeros + n * rg + sub : nullptr;
            }
        // d: scale bits; for the affine variant also z: bf16 bits of 136 + z'.
        auto load_scales = [&](uint32_t (&d)[TPW][2], uint32_t (&z)[TPW][2], int t) {
            const int64_t g = gs + t * kStageGroups + cw;
            const bool in = t < nt && g < ge;
#pragma unroll
            for (int rt = 0; rt < TPW; ++rt)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    d[rt][h] = in ? __ldg(srow[rt][h] + g * kSub) : 0u;
                    if (QG != 0) {
                        const int zq = in && zrow[rt][h] ? __ldg(zrow[rt][h] + g * kSub) : 0;
                        z[rt][h] = static_cast<uint32_t>(zq);  // z' in [-8, 7], as loaded: 136 + z' is formed at use
                    }
                }
        };
        uint32_t d_cur[TPW][2], d_nxt[TPW][2], z_cur[TPW][2], z_nxt[TPW][2];
        load_scales(d_nxt, z_nxt, 0);

        // Byte offsets inside a stage.
        const uint32_t w_off = static_cast<uint32_t>(cw * kRowsCta * 64 + (tile0 * 16 + gid) * 64 + tig * 16);
        const uint32_t x_blk = static_cast<uint32_t>(kCodeStageBytes + (2 * cw + (tig >> 1)) * C::kXRows * 128);

        for (int t = 0; t < nt; ++t) {
            const int s = t % C::kStages;
#pragma unroll
            for (int rt = 0; rt < TPW; ++rt) {
                d_cur[rt][0] = d_nxt[rt][0];
                d_cur[rt][1] = d_nxt[rt][1];
                z_cur[rt][0] = z_nxt[rt][0];
                z_cur[rt][1] = z_nxt[rt][1];
            }
            load_scales(d_nxt, z_nxt, t + 1);
            const bool have = mbar_wait(full(s), static_cast<uint32_t>(t / C::kStages) & 1u);
            if (!__all_sync(0xffffffffu, have)) {
                ok = false;
                break;
            }
            const bool active = gs + t * kStageGroups + cw < ge;  // warp-uniform
            const uint32_t st = base + s * C::kStageBytes;
            // Release the stage only after its fragments have been used: the
            // shared-memory loads may still be pending when an arrive executes,
            // and the next TMA copy into this stage must not overtake them
            // (releasing right after the loads gave rare corrupted fragments).
            if (active) {
                uint32_t xw[MT][16];
                load_x_frags<MT, C::kXRows>(xw, st + x_blk, gid, tig);
                if (!kDeq) {
                    uint4 wv[TPW][2];
#pragma unroll
                    for (int rt = 0; rt < TPW; ++rt) {
                        wv[rt][0] = lds128(st + w_off + rt * 16 * 64);
                        wv[rt][1] = lds128(st + w_off + rt * 16 * 64 + 8 * 64);
                    }
                    float dv[TPW][2];
#pragma unroll
                    for (int rt = 0; rt < TPW; ++rt) {
                        dv[rt][0] = bf16_lo(d_cur[rt][0]);
                        dv[rt][1] = bf16_lo(d_cur[rt][1]);
                    }
                    group_math<MT, TPW>(acc, xw, wv, dv);
                } else {
                    uint32_t d2[TPW][2], o2[TPW][2];
#pragma unroll
                    for (int rt = 0; rt < TPW; ++rt)
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            d2[rt][h] = d_cur[rt][h] | (d_cur[rt][h] << 16);
                            o2[rt][h] = QG == 0 ? 0x43084308u : ((0x4308u + z_cur[rt][h]) | ((0x4308u + z_cur[rt][h]) << 16));
                        }
                    if (MT <= 2) {
                        // Registers allow every row tile's chunks in flight at once.
                        uint4 wv[TPW][2];
#pragma unroll
                        for (int rt = 0; rt < TPW; ++rt) {
                            wv[rt][0] = lds128(st + w_off + rt * 16 * 64);
                            wv[rt][1] = lds128(st + w_off + rt * 16 * 64 + 8 * 64);
                        }
                        group_math_affine<MT, TPW>(acc, xw, wv, d2, o2);
                    } else {
                        group_math_affine_lds<MT, TPW>(acc, xw, st + w_off, d2, o2);
                    }
                }
            }
            // Generic-proxy reads of the slot before the async-proxy TMA copy that
            // reuses it: formally ordered only by a proxy fence (about 0.5 % here).
            fence_async_smem();
            mbar_arrive(empty(s));
        }
        if (!ok) record_status(args.status, kStatusTimeout);
    }

    // ------------------------------------------------------ reduction
    // Every stage was consumed, so the stage memory is free: partials of the
    // consumer warps go there as red[warp][tile][mt][r][lane], then the CTA's
    // sum as part[m][row].
    __syncthreads();
    float* red = reinterpret_cast<float*>(gbase);  // [group][tile][mt][r][lane]
    float* part = red + kStageGroups * kTiles * MT * 4 * 32;
    if (warp >= 1) {
        const int cw = (warp - 1) % kStageGroups;
        const int tile0 = ((warp - 1) / kStageGroups) * TPW;
#pragma unroll
        for (int rt = 0; rt < TPW; ++rt)
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int r = 0; r < 4; ++r)
                    red[(((cw * kTiles + tile0 + rt) * MT + mt) * 4 + r) * 32 + lane] = acc[rt][mt][r];
    }
    __syncthreads();
    for (int e = threadIdx.x; e < kTiles * MT * 4 * 32; e += kThreads) {
        const int l = e & 31;
        const int r = (e >> 5) & 3;
        const int mt = (e >> 7) % MT;
        const int rt = e / (MT * 128);
        float v = 0.0f;
        for (int w = 0; w < kStageGroups; ++w) v += red[(((w * kTiles + rt) * MT + mt) * 4 + r) * 32 + l];
        const int rowc = rt * 16 + (l >> 2) + (r >= 2 ? 8 : 0);
        const int m = mt * 8 + 2 * (l & 3) + (r & 1);
        if (split == 1) {
            const int64_t n = n0 + rowc;
            if (n < args.N && m < M) args.y[static_cast<int64_t>(m) * args.N + n] = __float2bfloat16_rn(v);
        } else {
            part[m * kRowsCta + rowc] = v;
        }
    }
    if (split > 1) {
        // Split-K partials, summed in rank order.  Every rank of the cluster
        // takes a slice of the outputs and reads that slice from all ranks
        // through DSMEM, issuing all of an element's remote loads before the
        // first add, so the reduction costs about one DSMEM round trip instead
        // of one per rank and element.
        cluster_sync();
        const uint32_t part_addr = smem_addr(part);
        const int total = kRowsCta * M;
        const int per = (total + split - 1) / split;
        const int e_end = min(total, static_cast<int>(rank + 1) * per);
        for (int e = static_cast<int>(rank) * per + threadIdx.x; e < e_end; e += kThreads) {
            const int rowc = e % kRowsCta, m = e / kRowsCta;
            const int64_t n = n0 + rowc;
            const uint32_t a = part_addr + static_cast<uint32_t>((m * kRowsCta + rowc) * 4);
            float p[kMaxSplit];
#pragma unroll
            for (int r = 0; r < kMaxSplit; ++r) p[r] = r < split ? ld_cluster_f32(a, static_cast<uint32_t>(r)) : 0.0f;
            float v = 0.0f;
#pragma unroll
            for (int r = 0; r < kMaxSplit; ++r)
                if (r < split) v += p[r];
            if (n < args.N) args.y[static_cast<int64_t>(m) * args.N + n] = __float2bfloat16_rn(v);
        }
        cluster_sync();
    }
}

std::mutex g_attr_mutex;

template <int MT, int TPW, int QG>
cudaError_t launch_mt(const __nv_bfloat16* x, int mp, int64_t N, int64_t K, const CUtensorMap& tmap_codes,
                      const uint16_t* scales, const int8_t* zeros, __nv_bfloat16* y, const DeviceInfo& dev,
                      cudaStream_t stream) {
    using C = Cfg<MT>;
    constexpr int kThreads = Warps<TPW>::kThreads;
    static bool attr_set[64];
    int device = 0;
    if (cudaError_t e = cudaGetDevice(&device)) return e;
    if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(g_attr_mutex);
        if (!attr_set[device]) {
            if (cudaError_t e = cudaFuncSetAttribute(gemv_w4_kernel<MT, TPW, QG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                     C::kSmemBytes))
                return e;
            attr_set[device] = true;
        }
    }
    const int64_t G = K / 128;
    const int64_t row_blocks = (N + kRowsCta - 1) / kRowsCta;
    if (row_blocks > 0x7fffffffLL || K > 0x7fffffffLL) return cudaErrorInvalidConfiguration;

    // Split-K factor: the cluster size (1..8, at most G) with the least
    // modelled time, given how many clusters of that size can be resident at
    // once.
    int64_t split = 1;
    double best = 0.0;
    for (int s = 1; s <= kMaxSplit && s <= G; ++s) {
        cudaLaunchConfig_t q = {};
        q.gridDim = dim3(static_cast<unsigned>(row_blocks), static_cast<unsigned>(s), 1);
        q.blockDim = dim3(kThreads, 1, 1);
        q.dynamicSmemBytes = C::kSmemBytes;
        cudaLaunchAttribute qa[1];
        qa[0].id = cudaLaunchAttributeClusterDimension;
        qa[0].val.clusterDim.x = 1;
        qa[0].val.clusterDim.y = static_cast<unsigned>(s);
        qa[0].val.clusterDim.z = 1;
        q.attrs = qa;
        q.numAttrs = 1;
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, gemv_w4_kernel<MT, TPW, QG>, &q) != cudaSuccess || clusters < 1) {
            cudaGetLastError();
            continue;
        }
        const int64_t waves = (row_blocks + clusters - 1) / clusters;
        const int64_t stages = ((G + s - 1) / s + kStageGroups - 1) / kStageGroups;
        // Per CTA: its stages plus a fixed part (pipeline fill, epilogue) that
        // grows with the cluster reduction; fitted to timings of the layer
        // shapes on GB300 (in units of one stage, about 1.1 us).
        const double cost = static_cast<double>(waves) * (static_cast<double>(stages) + 0.5 + 0.6 * (s - 1));
        if (best == 0.0 || cost < best) {
            best = cost;
            split = s;
        }
    }

    CUtensorMap tmap_x;
    if (cudaError_t e = encode_x_stage_map(&tmap_x, x, mp, K, C::kXRows, 2 * kStageGroups)) return e;
    GemvArgs args;
    args.scales = scales;
    args.zeros = zeros;
    args.row_groups = QG == 0 ? K / 128 : K / QG;
    args.y = y;
    args.M = mp;
    args.N = N;
    args.K = K;
    args.split = static_cast<int>(split);
    args.status = dev.status;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(row_blocks), static_cast<unsigned>(split), 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = static_cast<unsigned>(split);
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, gemv_w4_kernel<MT, TPW, QG>, tmap_codes, tmap_x, args);
}

template <int QG>
cudaError_t launch_gemv_q(const void* x, int64_t M, int64_t N, int64_t K, const void* packed, const void* scales,
                          const void* zeros, void* y, const DeviceInfo& dev, cudaStream_t stream) {
    // Row tiles per consumer warp up to 8 token rows: four for the symmetric
    // format; two (eight consumer warps) for the affine formats, whose
    // per-tile (d, z') pairs and dequantising arithmetic leave four tiles per
    // warp latency-bound (on 2560×9216, asymmetric group 128: 11.3 against
    // 8.2 µs at M = 1).  From 9 to 16 token rows two tiles per warp for every
    // format (affine: 14.4 against 10.8 µs at M = 16; symmetric: 8.17
    // against 7.92 µs at M = 16, 70.9 against 70.5 µs for a 27B layer).
    constexpr int kAffineTpw = QG == 0 ? kTpw : 2;
    CUtensorMap tmap_codes;
    if (cudaError_t e = encode_codes_stage_map(&tmap_codes, packed, N, K, kRowsCta, kStageGroups, CU_TENSOR_MAP_SWIZZLE_NONE))
        return e;
    const auto* xb = static_cast<const __nv_bfloat16*>(x);
    const auto* sc = static_cast<const uint16_t*>(scales);
    const auto* zp = static_cast<const int8_t*>(zeros);
    auto* yb = static_cast<__nv_bfloat16*>(y);
    for (int64_t m0 = 0; m0 < M; m0 += kMaxPassRows) {
        const int mp = static_cast<int>(M - m0 < kMaxPassRows ? M - m0 : kMaxPassRows);
        const __nv_bfloat16* xp = xb + m0 * K;
        __nv_bfloat16* yp = yb + m0 * N;
        const cudaError_t e =
            mp <= 8    ? launch_mt<1, kAffineTpw, QG>(xp, mp, N, K, tmap_codes, sc, zp, yp, dev, stream)
            : mp <= 16 ? launch_mt<2, 2, QG>(xp, mp, N, K, tmap_codes, sc, zp, yp, dev, stream)
            : mp <= 24 ? launch_mt<3, kTpw, QG>(xp, mp, N, K, tmap_codes, sc, zp, yp, dev, stream)
                       : launch_mt<4, kTpw, QG>(xp, mp, N, K, tmap_codes, sc, zp, yp, dev, stream);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_gemv(const void* x, int64_t M, int64_t N, int64_t K, const void* packed, const void* scales,
                        void* y, const DeviceInfo& dev, cudaStream_t stream) {
    return launch_gemv_q<0>(x, M, N, K, packed, scales, nullptr, y, dev, stream);
}

cudaError_t launch_gemv_affine(const void* x, int64_t M, int64_t N, int64_t K, int group, const void* packed,
                               const void* scales, const void* zeros, void* y, const DeviceInfo& dev,
                               cudaStream_t stream) {
    switch (group) {
        case 32: return launch_gemv_q<32>(x, M, N, K, packed, scales, zeros, y, dev, stream);
        case 64: return launch_gemv_q<64>(x, M, N, K, packed, scales, zeros, y, dev, stream);
        default: return launch_gemv_q<128>(x, M, N, K, packed, scales, zeros, y, dev, stream);
    }
}

}  // namespace w4
