// Small-M W4A16 matmul on the tcgen05 tensor cores, weights as the A operand
// in tensor memory:  y[m, n] = Σ_g d[n, g] · Σ_{k∈g} q[n, k] · x[m, k].
//
// Source: Qwen3.5-4B quantisation study, §1 FFN example y = W x with the
// group-quantisation equation (ŵ = d·q, one d per 128 consecutive inputs) and
// §2 settings (4-bit weights, BF16 inputs).
//
// Why this shape: at M ≤ 16 the matmul is bound by HBM (0.5 byte per weight),
// so every SM must decode about 45 weights per clock.  The decode itself (one
// shift and one LOP3 per pair of weights) is the floor of the instruction
// stream; everything else is moved off the SM's issue slots:
//  * one thread streams, by TMA, code tiles of two groups (128 rows x 128
//    bytes, 128-byte swizzle, 16 KB per copy) into an 8-deep shared-memory
//    ring (128 KB: at the loaded HBM latency every SM needs well over 100 KB
//    in flight), another thread the matching activation tiles;
//  * 256 decoder threads, two per weight row, each read 32 bytes of their
//    row (conflict-free thanks to the swizzle), turn the 64 nibbles into 32
//    bf16x2 values 136 + q and write them with one tcgen05.st into tensor
//    memory, where they are the MMA's A operand (128 lanes = rows, one 32-bit
//    column = one pair along K);
//  * the activations of the group (16 token rows, rows ≥ M read as zeros)
//    arrive by TMA in a 128-byte-swizzled shared-memory tile, the B operand;
//  * one thread issues per group 8 MMAs of 128×16×16 with the decoded A, plus
//    8 more with a constant A tile of −136 that cancels the bias, so the fp32
//    accumulator of the group holds Σ q·x exactly up to fp32 rounding;
//  * the group accumulators (four buffers in TMEM) are read back three groups
//    behind with one tcgen05.ld per row and scaled by d in fp32 registers;
//  * waiting threads sleep in mbarrier try_wait instead of spinning.
// Split-K: the CTAs of a thread-block cluster (1 × S) take disjoint group
// ranges of the same 128 rows and sum their partials through distributed
// shared memory in a fixed rank order, so results are deterministic and no
// global scratch is used.
//
// Every mbarrier wait is bounded; a wait that runs out records a timeout in
// the status word and the CTA winds down, draining its TMA copies and MMAs
// before it frees tensor memory.
#include <mutex>

#include "w4_device.cuh"
#include "w4_internal.h"
#include "w4_tcgen05.cuh"

namespace w4 {
namespace {

constexpr int kRows = 128;          // weight rows per CTA = MMA M
constexpr int kTok = 16;            // token rows per pass = MMA N
// Warps: 0 code TMA, 1 TMEM + MMA, 2 activation TMA, 3..10 decoders (two per
// TMEM lane quarter, each decoding half of a group's k range).
constexpr int kDecoderWarp0 = 3;
constexpr int kDecoders = 256;
constexpr int kThreads = 32 * kDecoderWarp0 + kDecoders;
// A TMA copy of only 8 KB per instruction caps one issuing thread well below
// the HBM rate; 16 KB copies reach it.  So codes and activations move in
// stages of two groups (256 k): one 16 KB code copy (128 rows x 128 bytes,
// 128-byte swizzle) and one 8 KB activation copy per stage.
constexpr int kCodeSlots = 8;       // stages of codes in flight: 128 KB, most of shared memory
constexpr int kXSlots = 4;          // stages of activations (L2-resident) in flight
constexpr int kASlots = 4;          // decoded groups in TMEM
constexpr int kDBufs = 4;           // group accumulators in TMEM: read back kDBufs-1 groups behind
constexpr int kMaxSplit = 8;
constexpr int kCodeSlotBytes = kRows * 128;      // two groups of 128 rows, 128-byte swizzle
constexpr int kXSlotBytes = 4 * kTok * 128;      // four 64-k blocks of 16 rows x 128 bytes

// Tensor memory columns (one CTA per SM: the whole 512-column TMEM).
constexpr uint32_t kColD = 0;        // + 32·b: group accumulators (16 fp32 columns each)
constexpr uint32_t kColConst = 128;  // 8 columns of bf16x2 (−136, −136): K = 16 of constant A
constexpr uint32_t kColA = 256;      // + 64·slot: decoded weights of one group
constexpr uint32_t kTmemCols = 512;
constexpr int kSmemBytes = kCodeSlots * kCodeSlotBytes + kXSlots * kXSlotBytes + kTok * kRows * 4 + 1024 + 1024;

constexpr uint32_t kMinus136x2 = 0xC308C308u;

struct TmemArgs {
    const uint16_t* scales;
    __nv_bfloat16* y;
    int M;  // token rows of this pass, 1..16
    int64_t N, K;
    int split;
    unsigned* status;
};

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" :::
                     "memory");
}

__device__ __forceinline__ float ld_cluster_f32(uint32_t local_addr, uint32_t rank) {
    uint32_t remote;
    float v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

// Pair i (0..3) of a stored code word as the bf16x2 value (136 + q_lo, 136 + q_hi).
__device__ __forceinline__ uint32_t biased_pair(uint32_t word, int i) {
    return ((word >> (4 * i)) & 0x000F000Fu) ^ 0x43084308u;
}

__global__ void __launch_bounds__(kThreads, 1)
gemv_tmem_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_codes,
                 const TmemArgs args) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);

    const uint32_t code_base = base;                                  // kCodeSlots x 8 KB
    const uint32_t x_base = code_base + kCodeSlots * kCodeSlotBytes;  // kXSlots x 4 KB
    const uint32_t red_base = x_base + kXSlots * kXSlotBytes;         // 16 x 128 fp32
    const uint32_t bar_base = red_base + kTok * kRows * 4;
    auto code_full = [&](int c) { return bar_base + 8u * c; };
    auto code_empty = [&](int c) { return bar_base + 8u * (kCodeSlots + c); };
    constexpr int kB1 = 2 * kCodeSlots;
    auto x_full = [&](int c) { return bar_base + 8u * (kB1 + c); };
    auto x_empty = [&](int c) { return bar_base + 8u * (kB1 + kXSlots + c); };
    constexpr int kB2 = kB1 + 2 * kXSlots;
    auto a_full = [&](int s) { return bar_base + 8u * (kB2 + s); };
    auto a_empty = [&](int s) { return bar_base + 8u * (kB2 + kASlots + s); };
    constexpr int kB3 = kB2 + 2 * kASlots;
    auto d_full = [&](int b) { return bar_base + 8u * (kB3 + b); };
    auto d_empty = [&](int b) { return bar_base + 8u * (kB3 + kDBufs + b); };
    const uint32_t done_bar = bar_base + 8u * (kB3 + 2 * kDBufs);
    const uint32_t tmem_slot = done_bar + 8u;
    volatile uint32_t* tmem_slot_ptr = reinterpret_cast<volatile uint32_t*>(gbase + (tmem_slot - base));
    float* red = reinterpret_cast<float*>(gbase + (red_base - base));

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kRows;
    const int64_t G = args.K >> 7;
    const int split = args.split;
    const uint32_t rank = split > 1 ? cluster_rank() : 0u;
    const int64_t gs = (static_cast<int64_t>(rank) * G) / split;
    const int64_t ge = (static_cast<int64_t>(rank + 1) * G) / split;
    const int nj = static_cast<int>(ge - gs);
    const int M = args.M;

    if (threadIdx.x == 0) {
        for (int c = 0; c < kCodeSlots; ++c) {
            mbar_init(code_full(c), 1);
            mbar_init(code_empty(c), 2 * kDecoders);  // every decoder, once per group of the stage
        }
        for (int c = 0; c < kXSlots; ++c) {
            mbar_init(x_full(c), 1);
            mbar_init(x_empty(c), 2);  // one MMA commit per group of the stage
        }
        for (int s = 0; s < kASlots; ++s) {
            mbar_init(a_full(s), kDecoders);
            mbar_init(a_empty(s), 1);
        }
        for (int b = 0; b < kDBufs; ++b) {
            mbar_init(d_full(b), 1);
            mbar_init(d_empty(b), kRows);
        }
        mbar_init(done_bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_async_smem();
    }
    if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot_ptr;

    // Decoder threads: TMEM lane quarter warp % 4 (the lanes a warp may access),
    // k half `half` of every group.
    const bool decoder = warp >= kDecoderWarp0;
    const int quarter = warp & 3;
    const int half = (warp - kDecoderWarp0) >> 2;
    const int row = quarter * 32 + lane;
    const bool owner = decoder && half == 0;  // keeps the row's accumulator
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    if (owner) {
        tmem_st8(lane_base + kColConst, kMinus136x2);
        tmem_wait_st();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    bool ok = true;
    if (warp == 0) {
        // -------------------------------------------------- codes via TMA
        if (lane == 0) {
            const int nt = (nj + 1) / 2;
            int issued = 0;
            for (int t = 0; t < nt; ++t) {
                const int c = t % kCodeSlots;
                if (!mbar_wait(code_empty(c), (static_cast<uint32_t>(t / kCodeSlots) & 1u) ^ 1u)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(code_full(c), kCodeSlotBytes);
                tma_load_2d(code_base + c * kCodeSlotBytes, &tmap_codes, static_cast<int>((gs + 2 * t) * 64),
                            static_cast<int>(n0), code_full(c));
                issued = t + 1;
            }
            if (!ok) {
                record_status(args.status, kStatusTimeout);
                for (int t = issued > kCodeSlots ? issued - kCodeSlots : 0; t < issued; ++t)
                    mbar_wait(code_full(t % kCodeSlots), static_cast<uint32_t>(t / kCodeSlots) & 1u);
            }
        }
    } else if (warp == 2) {
        // -------------------------------------------------- activations via TMA
        if (lane == 0) {
            const int nt = (nj + 1) / 2;
            int issued = 0;
            for (int t = 0; t < nt; ++t) {
                const int c = t % kXSlots;
                if (!mbar_wait(x_empty(c), (static_cast<uint32_t>(t / kXSlots) & 1u) ^ 1u)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(x_full(c), kXSlotBytes);
                tma_load_3d(x_base + c * kXSlotBytes, &tmap_x, 0, 0, static_cast<int>((gs + 2 * t) * 2), x_full(c));
                issued = t + 1;
            }
            if (!ok) {
                record_status(args.status, kStatusTimeout);
                for (int t = issued > kXSlots ? issued - kXSlots : 0; t < issued; ++t)
                    mbar_wait(x_full(t % kXSlots), static_cast<uint32_t>(t / kXSlots) & 1u);
            }
        }
    } else if (warp == 1) {
        // -------------------------------------------------- MMA issue
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(kTok);
            for (int j = 0; j < nj; ++j) {
                const int t = j >> 1;
                const int c = t % kXSlots;
                const int s = j % kASlots;
                const int b = j % kDBufs;
                if (!mbar_wait(x_full(c), static_cast<uint32_t>(t / kXSlots) & 1u) ||
                    !mbar_wait(a_full(s), static_cast<uint32_t>(j / kASlots) & 1u) ||
                    (j >= kDBufs && !mbar_wait(d_empty(b), static_cast<uint32_t>(j / kDBufs - 1) & 1u))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + kColD + 32u * b;
                const uint32_t a = tmem + kColA + 64u * s;
                const uint32_t xs = x_base + c * kXSlotBytes + (j & 1) * (kXSlotBytes / 2);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint64_t bd = sw128_desc(xs + (ks >> 2) * (kTok * 128) + (ks & 3) * 32);
                    mma_bf16_tmem_a(d, a + 8u * ks, bd, idesc, ks > 0 ? 1u : 0u);
                    mma_bf16_tmem_a(d, tmem + kColConst, bd, idesc, 1u);
                }
                mma_commit(a_empty(s));
                mma_commit(x_empty(c));
                mma_commit(d_full(b));
            }
            mma_commit(done_bar);  // also tracks MMAs issued before an abort
            if (!ok) record_status(args.status, kStatusTimeout);
        }
    } else {
        // -------------------------------------------------- decode + epilogue
        int64_t n = n0 + row;
        if (n >= args.N) n = args.N - 1;  // padding rows: codes arrive as zeros, scale of a valid row
        const uint16_t* srow = args.scales + n * G + gs;
        float acc[kTok];
#pragma unroll
        for (int m = 0; m < kTok; ++m) acc[m] = 0.0f;

        // Reads group i's accumulator, scales it into acc and frees the buffer.
        auto retire = [&](int i, uint32_t dbits) {
            const int b = i % kDBufs;
            const bool got = mbar_wait(d_full(b), static_cast<uint32_t>(i / kDBufs) & 1u);
            if (!__all_sync(0xffffffffu, got)) return false;
            tc_fence_after();
            uint32_t v[16];
            tmem_ld16(lane_base + kColD + 32u * b, v);
            tc_fence_before();
            mbar_arrive(d_empty(b));
            const float d = bf16_lo(dbits);
#pragma unroll
            for (int m = 0; m < kTok; ++m)
                if (m < M) acc[m] = fmaf(d, __uint_as_float(v[m]), acc[m]);
            return true;
        };

        // This thread's two 16-byte chunks (its k half of one group) in a code
        // stage: row pitch 128 bytes, 128-byte swizzle (chunk index XOR row % 8).
        const uint32_t row_off = static_cast<uint32_t>(row * 128);
        const uint32_t sw = static_cast<uint32_t>(row & 7);
        auto chunk_off = [&](int sub, int i) {
            return row_off + ((static_cast<uint32_t>(4 * sub + 2 * half + i) ^ sw) << 4);
        };

        constexpr int kLag = kDBufs - 1;
        uint32_t d_hist[kLag + 1];  // scales of groups j-kLag .. j
#pragma unroll
        for (int i = 0; i <= kLag; ++i) d_hist[i] = 0;
        uint32_t d_next = (owner && nj > 0) ? __ldg(srow) : 0u;
        for (int j = 0; j < nj && ok; ++j) {
            const int c = (j >> 1) % kCodeSlots;
            const int s = j % kASlots;
            if (owner) {
#pragma unroll
                for (int i = 0; i < kLag; ++i) d_hist[i] = d_hist[i + 1];
                d_hist[kLag] = d_next;
                if (j + 1 < nj) d_next = __ldg(srow + j + 1);
            }
            const bool have = mbar_wait(code_full(c), static_cast<uint32_t>((j >> 1) / kCodeSlots) & 1u);
            if (!__all_sync(0xffffffffu, have)) { ok = false; break; }
            const uint32_t slot = code_base + c * kCodeSlotBytes;
            const uint4 q0 = lds128(slot + chunk_off(j & 1, 0));
            const uint4 q1 = lds128(slot + chunk_off(j & 1, 1));
            mbar_arrive(code_empty(c));

            const bool free_a = mbar_wait(a_empty(s), (static_cast<uint32_t>(j / kASlots) & 1u) ^ 1u);
            if (!__all_sync(0xffffffffu, free_a)) { ok = false; break; }
            tc_fence_after();
            const uint32_t words[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
            uint32_t v[32];
#pragma unroll
            for (int w = 0; w < 8; ++w)
#pragma unroll
                for (int p = 0; p < 4; ++p) v[4 * w + p] = biased_pair(words[w], p);
            tmem_st32(lane_base + kColA + 64u * s + 32u * half, v);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(a_full(s));
            if (owner && j >= kLag && !retire(j - kLag, d_hist[0])) ok = false;
        }
        if (owner && ok) {
            for (int i = nj - kLag < 0 ? 0 : nj - kLag; i < nj && ok; ++i)
                if (!retire(i, d_hist[kLag - (nj - 1 - i)])) ok = false;
        }
        if (!ok) record_status(args.status, kStatusTimeout);

        if (owner) {
            if (split == 1) {
                const int64_t ny = n0 + row;
                if (ny < args.N)
                    for (int m = 0; m < M; ++m)
                        args.y[static_cast<int64_t>(m) * args.N + ny] = __float2bfloat16_rn(acc[m]);
            } else {
#pragma unroll
                for (int m = 0; m < kTok; ++m) red[m * kRows + row] = acc[m];
            }
        }
    }

    // Split-K partials: rank 0 of the cluster sums them in rank order.
    if (split > 1) {
        cluster_sync();
        if (rank == 0 && owner) {
            const int64_t ny = n0 + row;
            if (ny < args.N) {
                for (int m = 0; m < M; ++m) {
                    const uint32_t addr = red_base + static_cast<uint32_t>((m * kRows + row) * 4);
                    float v = 0.0f;
                    for (int r = 0; r < split; ++r) v += ld_cluster_f32(addr, static_cast<uint32_t>(r));
                    args.y[static_cast<int64_t>(m) * args.N + ny] = __float2bfloat16_rn(v);
                }
            }
        }
        cluster_sync();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        if (lane == 0) mbar_wait(done_bar, 0);  // MMAs in flight finish before TMEM is freed
        __syncwarp();
        tmem_dealloc(tmem, kTmemCols);
    }
}

std::mutex g_attr_mutex;
bool g_attr_set[64];

}  // namespace

cudaError_t launch_gemv_tmem(const void* x, int64_t M, int64_t N, int64_t K, const void* packed,
                             const void* scales, void* y, const DeviceInfo& dev, cudaStream_t stream) {
    const int64_t G = K / 128;
    const int64_t row_blocks = (N + kRows - 1) / kRows;
    if (row_blocks > 0x7fffffffLL || K > 0x7fffffffLL || N > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    int device = 0;
    if (cudaError_t e = cudaGetDevice(&device)) return e;
    if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(g_attr_mutex);
        if (!g_attr_set[device]) {
            if (cudaError_t e = cudaFuncSetAttribute(gemv_tmem_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                     kSmemBytes))
                return e;
            g_attr_set[device] = true;
        }
    }
    // Split-K factor: the cluster size (1..8, at most G) that finishes the
    // row blocks in the fewest rounds of group work, counting how many clusters
    // of that size can be resident at once (one CTA per SM).
    int64_t split = 1;
    {
        double best = 0.0;
        for (int s = 1; s <= kMaxSplit && s <= G; ++s) {
            cudaLaunchConfig_t q = {};
            q.gridDim = dim3(static_cast<unsigned>(row_blocks), static_cast<unsigned>(s), 1);
            q.blockDim = dim3(kThreads, 1, 1);
            q.dynamicSmemBytes = kSmemBytes;
            cudaLaunchAttribute qa[1];
            qa[0].id = cudaLaunchAttributeClusterDimension;
            qa[0].val.clusterDim.x = 1;
            qa[0].val.clusterDim.y = static_cast<unsigned>(s);
            qa[0].val.clusterDim.z = 1;
            q.attrs = qa;
            q.numAttrs = 1;
            int clusters = 0;
            if (cudaOccupancyMaxActiveClusters(&clusters, gemv_tmem_kernel, &q) != cudaSuccess || clusters < 1) {
                cudaGetLastError();
                continue;
            }
            const int64_t waves = (row_blocks + clusters - 1) / clusters;
            const double cost = static_cast<double>(waves) * static_cast<double>((G + s - 1) / s);
            if (best == 0.0 || cost < best) {
                best = cost;
                split = s;
            }
        }
    }

    CUtensorMap tmap_codes;
    if (cudaError_t e = encode_codes_map(&tmap_codes, packed, N, K)) return e;
    // With an odd group count the last stage of a range reaches one group past
    // it; that copy reads valid memory (or the zero fill past K) and is never
    // consumed.
    const auto* xb = static_cast<const __nv_bfloat16*>(x);
    auto* yb = static_cast<__nv_bfloat16*>(y);
    for (int64_t m0 = 0; m0 < M; m0 += kTok) {
        const int mp = static_cast<int>(M - m0 < kTok ? M - m0 : kTok);
        CUtensorMap tmap_x;
        if (cudaError_t e = encode_x_stage_map(&tmap_x, xb + m0 * K, mp, K, kTok, 4)) return e;
        TmemArgs args;
        args.scales = static_cast<const uint16_t*>(scales);
        args.y = yb + m0 * N;
        args.M = mp;
        args.N = N;
        args.K = K;
        args.split = static_cast<int>(split);
        args.status = dev.status;

        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(row_blocks), static_cast<unsigned>(split), 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = kSmemBytes;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 1;
        attr[0].val.clusterDim.y = static_cast<unsigned>(split);
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaError_t e = cudaLaunchKernelEx(&cfg, gemv_tmem_kernel, tmap_x, tmap_codes, args)) return e;
    }
    return cudaSuccess;
}

}  // namespace w4
