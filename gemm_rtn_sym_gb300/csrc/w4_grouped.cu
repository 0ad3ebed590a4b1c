// Grouped small-M W4A16 matmul: many independent problems y_i = Ŵ_i x_i
// (for example the four matrices of a transformer layer, or every matrix of a
// stack) in one persistent launch.
//
// Source: Qwen3.5-4B quantisation study, §1 FFN example y = W x with ŵ = d·q
// (one d per 128 consecutive inputs) and §2 settings (4-bit weights, BF16
// inputs); a model applies it to every linear layer (§2: 200 quantised
// matrices).  Each problem is computed exactly as by the single-matrix kernel
// in w4_gemv.cu (same decode, same MMA, same per-group fp32 scaling), so the
// results are within the same bound.
//
// Why: a small matrix takes only a few microseconds of streaming, and a launch
// of its own adds the launch gap, the pipeline fill (one DRAM latency) and a
// split-K reduction each time.  Here the work is a list of items, one per
// (problem, 64-row block), each covering the block's whole K, so no split-K
// is needed.  The plan fixes the grid (two CTAs per SM) and assigns the items
// longest first, each to the CTA with the least work so far (LPT).
// The producer warp streams the stages of a CTA's items back to back through
// one shared-memory ring, so the pipeline fills once per CTA, not once per
// matrix.  At the end of an item the consumer warps sum their fp32 partials in
// shared memory in a fixed order and store y: results are deterministic.
//
// The plan (built once on the host, copied to device memory the caller owns)
// holds a TMA descriptor pair per problem and the item list; the kernel reads
// descriptors from global memory after a tensormap-proxy acquire fence.
#include <algorithm>
#include <cstring>
#include <mutex>
#include <queue>
#include <vector>

#include "w4_device.cuh"
#include "w4_gemv_common.cuh"
#include "w4_internal.h"
#include "w4_tcgen05.cuh"

namespace w4 {
namespace {

using namespace gemv;

// Plan memory of w4_gemm_grouped_noalloc: a file-scope device array, so that
// entry point allocates nothing.  Shared by every call on a device (see the
// race note in w4.h).
constexpr size_t kStaticPlanBytes = size_t{2} << 20;
static __device__ __align__(256) uint8_t g_static_plan[kStaticPlanBytes];

// Device layout of a plan:
//   GroupedHeader (128 B) | GroupedProblem[count] (384 B each) |
//   int32 first[n_ctas + 1] (padded to 8 B) | uint2 items[n_items]
// CTA c runs items[first[c] .. first[c + 1]).  Tensor maps stay 128-byte
// aligned when the plan is.
struct alignas(128) GroupedHeader {
    int32_t count;
    int32_t n_items;
    int32_t token_rows;   // x rows staged per 64-k block: 2, 4, 8, 16 or 24
    int32_t n_ctas;       // the grid the plan was scheduled for
    int32_t format;       // 0: symmetric group 128; 32, 64, 128: affine format of that group size
    int32_t reserved[27];
};

struct alignas(128) GroupedProblem {
    CUtensorMap codes;  // [G][N][64 B], boxes of 4 groups × 64 rows
    CUtensorMap x;      // [K/64][M][64], boxes of 8 blocks × token_rows rows, 128-byte swizzle
    const uint16_t* scales;
    __nv_bfloat16* y;
    int64_t N;
    int32_t M;
    int32_t G;
    int32_t T;  // stages per item
    int32_t pad;
    const int8_t* zeros;  // affine formats: int8 zero − 8 per group, or null
    int64_t row_groups;   // scales (and zeros) per row: K / group
    int32_t reserved[18];
};
static_assert(sizeof(GroupedHeader) == 128, "plan header");
static_assert(sizeof(GroupedProblem) == 384, "plan problem record");

__device__ __forceinline__ void tensormap_acquire(const void* map) {
    asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(map) : "memory");
}

__device__ __forceinline__ void consumer_sync(int n_threads) {
    asm volatile("bar.sync 1, %0;" ::"r"(n_threads) : "memory");
}

// Scales of one stage of the symmetric format in shared memory: 4 groups × 64
// rows of bf16.
constexpr int kScaleStageBytes = kStageGroups * kRowsCta * 2;

// Geometry of the grouped kernel for MT token tiles with XR token rows staged
// per 64-k block (XR < 8 only for one tile: a decode step of one or two tokens
// stages one or two rows, not eight), run with CPS CTAs per SM.  The ring is
// as deep as fits: per CTA about 227 KB / CPS of shared memory, of which the
// reduction buffer and barriers take 9 KB.  With one token tile three CTAs
// per SM stream faster than two (more warps to hide the decode's dependency
// latency), unless the items balance badly over that many CTAs.
template <int MT, int XR, int CPS, int QG>
struct GCfg {
    static constexpr int kXRows = XR;
    static constexpr int kXStageBytes = 2 * kStageGroups * XR * 128;  // [k-block][row][128 B]
    static constexpr int kStageBytes = kCodeStageBytes + kXStageBytes;
    // Scale slot of a stage: the symmetric format's 4 groups × 64 rows of
    // bf16; the affine formats' kE (d, z') entries per row (d bf16 as
    // [row][kE], then z' int8 as [row][kE]), kE = the stage's 512 k / QG.
    static constexpr int kE = QG == 0 ? kStageGroups : kStageGroups * 128 / QG;
    static constexpr int kScaleSlotBytes = QG == 0 ? kScaleStageBytes : kRowsCta * kE * 3;
    static constexpr int kBudget = (CPS == 3 ? 74 : 112) * 1024 - 9 * 1024;
    static constexpr int kPerStage = kStageBytes + kScaleSlotBytes;
    static constexpr int kStages = kBudget / kPerStage > 5 ? 5 : kBudget / kPerStage;
    static_assert(XR == 8 * MT || (MT == 1 && (XR == 2 || XR == 4)), "staged rows");
    static_assert(kStages >= 2, "ring depth");
};

// Row tiles per consumer warp: four, except for the affine formats up to 16
// token rows, whose per-tile (d, z') pairs and dequantising arithmetic run
// better over eight warps of two tiles (as in the single-matrix kernel: on the
// 27B-class layer asymmetric group 128 took 62 against 95 µs at M = 1 and 94
// against 122 µs at M = 16).
template <int MT, int QG>
struct GTpw {
    static constexpr int value = QG != 0 && MT <= 2 ? 2 : kTpw;
};

// Threads of a CTA: the TMA producer warp, the consumer warps and, except
// for the symmetric format at three CTAs per SM (where a sixth warp would
// leave 96 registers a thread), a warp that stages the scales (and zero points).
template <int MT, int QG, int CPS>
struct GThreads {
    static constexpr bool kStager = QG != 0 || CPS != 3;
    static constexpr int value = Warps<GTpw<MT, QG>::value>::kThreads + (kStager ? 32 : 0);
};


// QG: 0 for the symmetric group-128 format; 32, 64 or 128 for the affine
// formats (group size QG, zero points where a problem has them), which
// dequantise every weight to bf16(d·(c − z')) as the single-matrix kernel does.
template <int MT, int XR, int CPS, int QG>
__global__ void __launch_bounds__(GThreads<MT, QG, CPS>::value, CPS)
gemv_grouped_kernel(const uint8_t* __restrict__ plan, unsigned* status) {
    using C = GCfg<MT, XR, CPS, QG>;
    constexpr int TPW = GTpw<MT, QG>::value;
    constexpr bool kDeq = QG != 0 || Dequant<MT>::value;
    constexpr int kConsumers = Warps<TPW>::kConsumers;
    constexpr int kCThreads = 32 * kConsumers;
    constexpr int kRedFloats = kStageGroups * kTiles * 4 * 32;
    // Each stage's scales (and zero points) are staged in shared memory,
    // replacing the consumers' scattered global loads of them (those loads,
    // their pointers and registers measured 12–14 % of the kernel's time on
    // the 200-matrix stack, 22–26 % with zero points on the 27B-class layer).
    // Symmetric format: a transposed slot, read with one 16-byte load per
    // consumer lane.  Affine formats: the rows as stored, copied with
    // cp.async.  A warp of its own stages them (done by the producer warp, the
    // loads or copies of these small rows delay its TMA issue and every stage
    // behind it), except for the symmetric format at three CTAs per SM, where
    // the producer warp does.
    constexpr bool kSmemScales = QG == 0;
    constexpr int kE = C::kE;
    constexpr bool kStager = GThreads<MT, QG, CPS>::kStager;
    constexpr bool kProducerScales = kSmemScales && !kStager;  // the producer warp stages them
    constexpr int kStagerWarp = 1 + kConsumers;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    float* red = reinterpret_cast<float*>(gbase + C::kStages * C::kStageBytes);
    const uint32_t sc_base = base + C::kStages * C::kStageBytes + kRedFloats * 4;
    const uint32_t bar_base = sc_base + C::kStages * C::kScaleSlotBytes;
    auto full = [&](int s) { return bar_base + 8u * s; };
    auto empty = [&](int s) { return bar_base + 8u * (C::kStages + s); };
    auto sfull = [&](int s) { return bar_base + 8u * (2 * C::kStages + s); };  // the stage's scales are stored

    const GroupedHeader* hdr = reinterpret_cast<const GroupedHeader*>(plan);
    const GroupedProblem* probs = reinterpret_cast<const GroupedProblem*>(plan + sizeof(GroupedHeader));
    const int count = hdr->count;
    const int32_t* first = reinterpret_cast<const int32_t*>(plan + sizeof(GroupedHeader) + sizeof(GroupedProblem) * count);
    const uint2* items = reinterpret_cast<const uint2*>(first + ((hdr->n_ctas + 2) & ~1));
    const int i_begin = first[blockIdx.x];
    const int i_end = first[blockIdx.x + 1];

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int gid = lane >> 2;
    const int tig = lane & 3;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 32 * kConsumers);
            mbar_init(sfull(s), 32);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_async_smem();
    }
    __syncthreads();
    pdl_start();

    // Symmetric format: stage t of an item uses the scales of groups
    // 4t .. 4t + 3 of its 64 rows; the consumer warp taking group cw reads, in
    // lane (gid, tig), the scales of rows 8j + gid, j = 0..7 (row tile j / 2,
    // row half j % 2), as the 16 bytes at byte (cw·8 + gid)·16 of the stage's
    // slot.  Lane l of the staging warp stages rows l and l + 32 (j = l / 8
    // and 4 + l / 8), its global loads two stages ahead of its stores.  Rows
    // past N repeat row N − 1 (their codes are zero); groups past G stage zeros
    // (no consumer takes them).
    const uint32_t row_off = static_cast<uint32_t>(((lane & 7) * 8 + (lane >> 3)) * 2);
    int li = i_begin - 1, lt = 0, lT = 0;  // next (item, stage) whose scales to fetch; its stages
    int lG = 0;
    bool lvec = false;
    const uint16_t* lp[2] = {nullptr, nullptr};  // scales of rows l and l + 32 of item li
    auto fetch = [&](uint2 (&o)[2]) {
        if (lt == lT) {  // next item with stages
            lt = 0;
            lT = 0;
            while (lT <= 0 && ++li < i_end) lT = probs[items[li].x].T;
            if (li >= i_end) {
                lT = -1;  // fetches past the end stage zeros
            } else {
                const uint2 it = items[li];
                const GroupedProblem* pr = probs + it.x;
                lG = pr->G;
                // One 8-byte load per row where every row's and stage's start is 8-byte aligned.
                lvec = (lG & 3) == 0 && (reinterpret_cast<uintptr_t>(pr->scales) & 7u) == 0;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    int64_t n = static_cast<int64_t>(it.y) * kRowsCta + lane + 32 * h;
                    if (n >= pr->N) n = pr->N - 1;
                    lp[h] = pr->scales + n * lG;
                }
            }
        }
        o[0] = o[1] = make_uint2(0u, 0u);
        if (lT < 0) return;
        const int g0 = lt * kStageGroups;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            if (lvec) {
                o[h] = __ldg(reinterpret_cast<const uint2*>(lp[h] + g0));
            } else {
                uint32_t q[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) q[c] = g0 + c < lG ? static_cast<uint32_t>(__ldg(lp[h] + g0 + c)) : 0u;
                o[h] = make_uint2(q[0] | (q[1] << 16), q[2] | (q[3] << 16));
            }
        }
        ++lt;
    };
    auto store_sym = [&](uint32_t slot, const uint2 (&v)[2]) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t o = slot + row_off + 8u * h;  // j + 4h
            sts16(o, v[h].x);
            sts16(o + 128u, v[h].x >> 16);
            sts16(o + 256u, v[h].y);
            sts16(o + 384u, v[h].y >> 16);
        }
    };
    if (warp == 0) {
        // -------------------------------------------------- producer: stages of every item, back to back
        // Lane 0 issues the TMA copies of each stage; where the producer warp
        // stages the symmetric scales, every lane then stores its share.
        uint2 a[2], b[2], c[2];  // scales of stages k, k + 1, k + 2
        if (kProducerScales) {
            fetch(a);
            fetch(b);
        }
        int s = 0;
        uint32_t phase = 0;
        int issued = 0;  // stages issued
        bool ok = true;
        for (int i = i_begin; i < i_end && ok; ++i) {
            const uint2 it = items[i];
            const GroupedProblem* pr = probs + it.x;
            if (lane == 0) {
                tensormap_acquire(&pr->codes);
                tensormap_acquire(&pr->x);
            }
            const int row = static_cast<int>(it.y) * kRowsCta;
            for (int t = 0; t < pr->T; ++t) {
                if (kProducerScales) fetch(c);
                ok = __all_sync(0xffffffffu, mbar_wait_suspend(empty(s), phase ^ 1u));
                if (!ok) break;
                if (lane == 0) {
                    const uint32_t st = base + s * C::kStageBytes;
                    mbar_arrive_expect_tx(full(s), C::kStageBytes);
                    tma_load_3d(st, &pr->codes, 0, row, t * kStageGroups, full(s));
                    tma_load_3d(st + kCodeStageBytes, &pr->x, 0, 0, 2 * kStageGroups * t, full(s));
                }
                if (kProducerScales) {
                    store_sym(sc_base + s * C::kScaleSlotBytes, a);
                    mbar_arrive(sfull(s));
                    a[0] = b[0];
                    a[1] = b[1];
                    b[0] = c[0];
                    b[1] = c[1];
                }
                ++issued;
                if (++s == C::kStages) {
                    s = 0;
                    phase ^= 1u;
                }
            }
        }
        if (!ok && lane == 0) {
            record_status(status, kStatusTimeout);
            // Drain: every issued copy lands before the CTA may exit.
            for (int j = issued > C::kStages ? issued - C::kStages : 0; j < issued; ++j)
                mbar_wait(full(j % C::kStages), static_cast<uint32_t>(j / C::kStages) & 1u);
        }
        return;
    }

    if (kStager && kSmemScales && warp == kStagerWarp) {
        // -------------------------------------------------- symmetric stager
        uint2 a[2], b[2], c[2];  // scales of stages k, k + 1, k + 2
        fetch(a);
        fetch(b);
        int s = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int i = i_begin; i < i_end && ok; ++i) {
            const int T = probs[items[i].x].T;
            for (int t = 0; t < T; ++t) {
                fetch(c);
                ok = __all_sync(0xffffffffu, mbar_wait_suspend(empty(s), phase ^ 1u));
                if (!ok) break;
                store_sym(sc_base + s * C::kScaleSlotBytes, a);
                mbar_arrive(sfull(s));
                a[0] = b[0];
                a[1] = b[1];
                b[0] = c[0];
                b[1] = c[1];
                if (++s == C::kStages) {
                    s = 0;
                    phase ^= 1u;
                }
            }
        }
        if (!ok && lane == 0) record_status(status, kStatusTimeout);
        return;
    }

    if (!kSmemScales && warp == kStagerWarp) {
        // -------------------------------------------------- affine stager
        // Stage t of an item: the kE (d, z') entries t·kE .. of rows l and
        // l + 32 (rows past N repeat row N − 1, whose codes are zero) into the
        // stage's slot, d as [row][kE] bf16 then z' as [row][kE] int8, with
        // cp.async in the largest chunks (16, 8 or 4 bytes) that the row
        // stride, the base and a stage's entries allow, else element by
        // element; the lane's arrival on the stage's barrier is made when its
        // copies have landed.  Entries past the end of a row are not written
        // (no consumer takes them).
        auto chunk = [](int64_t stride, uintptr_t addr, int per_stage) {
            for (int c = 16; c >= 4; c >>= 1)
                if (stride % c == 0 && addr % c == 0 && per_stage % c == 0) return c;
            return 0;
        };
        int s = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int i = i_begin; i < i_end && ok; ++i) {
            const uint2 it = items[i];
            const GroupedProblem* pr = probs + it.x;
            const int64_t arg = pr->row_groups;
            const uint16_t* drow[2];
            const int8_t* zrow[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                int64_t n = static_cast<int64_t>(it.y) * kRowsCta + lane + 32 * h;
                if (n >= pr->N) n = pr->N - 1;
                drow[h] = pr->scales + n * arg;
                zrow[h] = pr->zeros ? pr->zeros + n * arg : nullptr;
            }
            const int cd = chunk(2 * arg, reinterpret_cast<uintptr_t>(pr->scales), 2 * kE);
            const int cz = pr->zeros ? chunk(arg, reinterpret_cast<uintptr_t>(pr->zeros), kE) : 0;
            for (int t = 0; t < pr->T; ++t) {
                ok = __all_sync(0xffffffffu, mbar_wait_suspend(empty(s), phase ^ 1u));
                if (!ok) break;
                const uint32_t slot = sc_base + s * C::kScaleSlotBytes;
                const int64_t e0 = static_cast<int64_t>(t) * kE;
                const int ne = static_cast<int>(arg - e0 < kE ? arg - e0 : kE);  // entries inside the row
                bool plain = false;  // some entries stored with plain stores
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint32_t r = static_cast<uint32_t>(lane + 32 * h);
                    const uint32_t dd = slot + r * (2 * kE);
                    const uint16_t* ds = drow[h] + e0;
                    if (cd) {
                        for (int b = 0; b < 2 * ne; b += cd) cp_async_n(dd + b, reinterpret_cast<const uint8_t*>(ds) + b, cd);
                    } else {
                        for (int e = 0; e < ne; ++e) sts16(dd + 2 * e, __ldg(ds + e));
                        plain = true;
                    }
                    if (zrow[h]) {
                        const uint32_t zd = slot + kRowsCta * 2 * kE + r * kE;
                        const int8_t* zs = zrow[h] + e0;
                        if (cz) {
                            for (int b = 0; b < ne; b += cz) cp_async_n(zd + b, zs + b, cz);
                        } else {
                            for (int e = 0; e < ne; ++e) sts8(zd + e, static_cast<uint32_t>(__ldg(zs + e)));
                            plain = true;
                        }
                    }
                }
                if (plain) {
                    cp_async_wait_all();
                    mbar_arrive(sfull(s));
                } else {
                    cp_async_arrive(sfull(s));
                }
                if (++s == C::kStages) {
                    s = 0;
                    phase ^= 1u;
                }
            }
        }
        if (!ok && lane == 0) record_status(status, kStatusTimeout);
        cp_async_wait_all();  // no copy of this thread outlives it
        return;
    }

    // ------------------------------------------------------ consumers
    // Every consumer warp runs the same sequence of items, stages and named
    // barriers; after a timed-out wait a warp only skips work.
    const int ctid = threadIdx.x - 32;
    const int cw = (warp - 1) % kStageGroups;
    const int tile0 = ((warp - 1) / kStageGroups) * TPW;
    const uint32_t w_off = static_cast<uint32_t>(cw * kRowsCta * 64 + (tile0 * 16 + gid) * 64 + tig * 16);
    const uint32_t x_blk = static_cast<uint32_t>(kCodeStageBytes + (2 * cw + (tig >> 1)) * C::kXRows * 128);

    int s = 0;
    uint32_t phase = 0;
    bool aborted = false;
    for (int i = i_begin; i < i_end; ++i) {
        const uint2 it = items[i];
        const GroupedProblem* pr = probs + it.x;
        const int T = pr->T;
        const int G = pr->G;
        const int64_t N = pr->N;
        const int M = pr->M;
        __nv_bfloat16* const y = pr->y;  // read once: stores to y could alias the record
        const int64_t row0 = static_cast<int64_t>(it.y) * kRowsCta;
        // Affine formats: this lane's entry of each staged row, the QG-group
        // holding its 32 codes of the warp's 128-k group (k 32·tig .. +31).
        const int sub = QG == 32 ? tig : (QG == 64 ? (tig >> 1) : 0);
        const bool has_z = QG != 0 && pr->zeros != nullptr;
        const uint32_t a_off = static_cast<uint32_t>((tile0 * 16 + gid) * kE + cw * (kE / kStageGroups) + sub);
        float acc[TPW][MT][4];
#pragma unroll
        for (int rt = 0; rt < TPW; ++rt)
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int r = 0; r < 4; ++r) acc[rt][mt][r] = 0.0f;
        for (int t = 0; t < T; ++t) {
            // d: scale bits; affine formats also z': the zero as stored (136 + z' is formed at use).
            uint32_t d_cur[TPW][2], z_cur[TPW][2];
            if (!aborted) {
                aborted = !__all_sync(0xffffffffu, mbar_wait(full(s), phase) && mbar_wait(sfull(s), phase));
                if (aborted && lane == 0) record_status(status, kStatusTimeout);
            }
            if (!aborted) {
                const bool active = t * kStageGroups + cw < G;  // warp-uniform
                if (active) {
                    const uint32_t slot = sc_base + s * C::kScaleSlotBytes;
                    if (kSmemScales) {
                        // Word rt: (row half 0, row half 1) of tile rt (TPW = 4, tile0 = 0).
                        static_assert(!kSmemScales || TPW == kTiles, "one consumer warp per group");
                        const uint4 q = lds128(slot + static_cast<uint32_t>((cw * 8 + gid) * 16));
                        const uint32_t wds[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                        for (int rt = 0; rt < TPW; ++rt) {
                            d_cur[rt][0] = wds[rt] & 0xFFFFu;
                            d_cur[rt][1] = wds[rt] >> 16;
                        }
                    } else {
                        // Row (tile0 + rt)·16 + gid + 8h of the slot: entry a_off + (16·rt + 8h)·kE.
#pragma unroll
                        for (int rt = 0; rt < TPW; ++rt)
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                const uint32_t e = a_off + static_cast<uint32_t>((16 * rt + 8 * h) * kE);
                                d_cur[rt][h] = lds_u16(slot + 2 * e);
                                z_cur[rt][h] = has_z ? static_cast<uint32_t>(lds_s8(slot + kRowsCta * 2 * kE + e)) : 0u;
                            }
                    }
                    // Release the stage only after its fragments have been used
                    // (shared-memory loads may still be pending when an arrive
                    // executes; the next TMA copy must not overtake them).
                    const uint32_t st = base + s * C::kStageBytes;
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
                                // bf16x2 (136 + z', 136 + z'); z' = 0 for symmetric codes
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
            if (++s == C::kStages) {
                s = 0;
                phase ^= 1u;
            }
        }
        // The item's sum: warp partials through shared memory, added in warp order.
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            consumer_sync(kCThreads);  // the previous readers of red are done
            if constexpr (TPW == kTiles && MT <= 2) {
                // Four warps, one per group of a stage, each holding every tile:
                // warp cw sums, for every tile, the elements acc[.][mt][cw] whose
                // own partial it holds, and writes only the other three (1–2 %
                // faster up to 16 token rows; at 24, 6 % slower).
#pragma unroll
                for (int rt = 0; rt < TPW; ++rt)
#pragma unroll
                    for (int r = 0; r < 4; ++r)
                        if (r != cw) red[((cw * kTiles + rt) * 4 + r) * 32 + lane] = acc[rt][mt][r];
                consumer_sync(kCThreads);
                const int m = mt * 8 + 2 * (lane & 3) + (cw & 1);
#pragma unroll
                for (int rt = 0; rt < TPW; ++rt) {
                    const float own = cw == 0 ? acc[rt][mt][0]
                                    : cw == 1 ? acc[rt][mt][1]
                                    : cw == 2 ? acc[rt][mt][2]
                                              : acc[rt][mt][3];
                    float v = 0.0f;
#pragma unroll
                    for (int w = 0; w < kStageGroups; ++w) v += w == cw ? own : red[((w * kTiles + rt) * 4 + cw) * 32 + lane];
                    const int64_t n = row0 + rt * 16 + (lane >> 2) + (cw >= 2 ? 8 : 0);
                    if (!aborted && n < N && m < M) y[static_cast<int64_t>(m) * N + n] = __float2bfloat16_rn(v);
                }
            } else {
#pragma unroll
                for (int rt = 0; rt < TPW; ++rt)
#pragma unroll
                    for (int r = 0; r < 4; ++r) red[((cw * kTiles + tile0 + rt) * 4 + r) * 32 + lane] = acc[rt][mt][r];
                consumer_sync(kCThreads);
                for (int e = ctid; e < kTiles * 4 * 32; e += kCThreads) {
                    const int l = e & 31;
                    const int r = (e >> 5) & 3;
                    const int rt = e >> 7;
                    float v = 0.0f;
#pragma unroll
                    for (int w = 0; w < kStageGroups; ++w) v += red[((w * kTiles + rt) * 4 + r) * 32 + l];
                    const int m = mt * 8 + 2 * (l & 3) + (r & 1);
                    const int64_t n = row0 + rt * 16 + (l >> 2) + (r >= 2 ? 8 : 0);
                    if (!aborted && n < N && m < M) y[static_cast<int64_t>(m) * N + n] = __float2bfloat16_rn(v);
                }
            }
        }
    }
}

template <int MT, int XR, int CPS, int QG>
constexpr int grouped_smem_bytes() {
    using C = GCfg<MT, XR, CPS, QG>;
    return C::kStages * (C::kStageBytes + C::kScaleSlotBytes) + kStageGroups * kTiles * 4 * 32 * 4 +
           24 * C::kStages + 1024;
}

std::mutex g_grouped_mutex;

template <int MT, int XR, int CPS, int QG>
int grouped_ctas_per_sm(int device) {
    static int per_device[64];
    std::lock_guard<std::mutex> lock(g_grouped_mutex);
    if (device < 0 || device >= 64) return 0;
    if (per_device[device] == 0) {
        int v = 0;
        if (cudaFuncSetAttribute(gemv_grouped_kernel<MT, XR, CPS, QG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 grouped_smem_bytes<MT, XR, CPS, QG>()) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, gemv_grouped_kernel<MT, XR, CPS, QG>,
                                                          GThreads<MT, QG, CPS>::value,
                                                          grouped_smem_bytes<MT, XR, CPS, QG>()) != cudaSuccess ||
            v < 1) {
            cudaGetLastError();
            return 0;
        }
        per_device[device] = v;
    }
    return per_device[device];
}

template <int MT, int XR, int CPS, int QG>
cudaError_t launch_grouped_t(const void* plan, int32_t n_ctas, const DeviceInfo& dev, cudaStream_t stream) {
    int device = 0;
    if (cudaError_t e = cudaGetDevice(&device)) return e;
    if (grouped_ctas_per_sm<MT, XR, CPS, QG>(device) < 1) return cudaErrorInvalidConfiguration;  // sets the smem attribute
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(n_ctas), 1, 1);
    cfg.blockDim = dim3(GThreads<MT, QG, CPS>::value, 1, 1);
    cfg.dynamicSmemBytes = grouped_smem_bytes<MT, XR, CPS, QG>();
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemv_grouped_kernel<MT, XR, CPS, QG>, static_cast<const uint8_t*>(plan), dev.status);
}

}  // namespace

cudaError_t static_plan_memory(void** ptr, size_t* bytes) {
    static void* per_device[64];
    int device = 0;
    if (cudaError_t e = cudaGetDevice(&device)) return e;
    if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_grouped_mutex);
    if (!per_device[device]) {
        void* p = nullptr;
        if (cudaError_t e = cudaGetSymbolAddress(&p, g_static_plan)) return e;
        per_device[device] = p;
    }
    *ptr = per_device[device];
    *bytes = kStaticPlanBytes;
    return cudaSuccess;
}

size_t grouped_plan_bytes(int32_t count, int64_t n_items, int32_t n_ctas) {
    return sizeof(GroupedHeader) + sizeof(GroupedProblem) * static_cast<size_t>(count) +
           sizeof(int32_t) * static_cast<size_t>((n_ctas + 2) & ~1) + sizeof(uint2) * static_cast<size_t>(n_items);
}

int grouped_token_rows(int64_t max_m) {
    return max_m <= 2 ? 2 : max_m <= 4 ? 4 : max_m <= 8 ? 8 : max_m <= 16 ? 16 : 24;
}

// Resident CTAs per SM of the grouped kernel for these token rows and format
// (three for one token tile of the symmetric format, two otherwise).
template <int QG>
int grouped_ctas_q(int token_rows, int device) {
    constexpr int kOne = QG == 0 ? 3 : 2;  // the affine formats run two per SM
    switch (token_rows) {
        case 2: return grouped_ctas_per_sm<1, 2, kOne, QG>(device);
        case 4: return grouped_ctas_per_sm<1, 4, kOne, QG>(device);
        case 8: return grouped_ctas_per_sm<1, 8, kOne, QG>(device);
        case 16: return grouped_ctas_per_sm<2, 16, 2, QG>(device);
        case 24: return grouped_ctas_per_sm<3, 24, 2, QG>(device);
        default: return 0;
    }
}

int grouped_ctas(int token_rows, int format, const DeviceInfo& dev) {
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) return 0;
    int per_sm = 0;
    switch (format) {
        case 0: per_sm = grouped_ctas_q<0>(token_rows, device); break;
        case 32: per_sm = grouped_ctas_q<32>(token_rows, device); break;
        case 64: per_sm = grouped_ctas_q<64>(token_rows, device); break;
        case 128: per_sm = grouped_ctas_q<128>(token_rows, device); break;
        default: return 0;
    }
    return per_sm * dev.sm_count;
}

namespace {

struct PlanItem {
    int32_t stages;
    uint2 id;
};

// Longest processing time first: items by cost (stages, plus one for the
// item's epilogue) in decreasing order, each to the least-loaded CTA (lowest
// index among equals).  Deterministic.  Returns the largest CTA load.
int64_t schedule_lpt(const std::vector<PlanItem>& sorted, int32_t n_ctas, std::vector<std::vector<uint2>>* per_cta) {
    using Load = std::pair<int64_t, int32_t>;  // (work so far, CTA)
    std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
    for (int32_t c = 0; c < n_ctas; ++c) heap.push({0, c});
    if (per_cta) per_cta->assign(static_cast<size_t>(n_ctas), {});
    int64_t makespan = 0;
    for (const PlanItem& it : sorted) {
        Load l = heap.top();
        heap.pop();
        if (per_cta) (*per_cta)[static_cast<size_t>(l.second)].push_back(it.id);
        l.first += it.stages + 1;
        makespan = std::max(makespan, l.first);
        heap.push(l);
    }
    return makespan;
}

}  // namespace

cudaError_t grouped_plan_build(const GroupedSpec* specs, int32_t count, int token_rows, int format, int32_t max_ctas,
                               int32_t sm_count, std::vector<uint8_t>* out, int64_t* n_items_out,
                               int32_t* n_ctas_out) {
    int64_t n_items = 0;
    for (int32_t i = 0; i < count; ++i) n_items += (specs[i].N + kRowsCta - 1) / kRowsCta;
    if (n_items > 0x7fffffffLL || max_ctas < 1 || sm_count < 1) return cudaErrorInvalidValue;
    std::vector<GroupedProblem> probs(static_cast<size_t>(count));
    std::vector<PlanItem> list;
    list.reserve(static_cast<size_t>(n_items));
    for (int32_t i = 0; i < count; ++i) {
        const GroupedSpec& sp = specs[i];
        GroupedProblem& pr = probs[static_cast<size_t>(i)];
        std::memset(&pr, 0, sizeof(pr));
        if (cudaError_t e = encode_codes_stage_map(&pr.codes, sp.packed, sp.N, sp.K, kRowsCta, kStageGroups,
                                                   CU_TENSOR_MAP_SWIZZLE_NONE))
            return e;
        if (cudaError_t e = encode_x_stage_map(&pr.x, sp.x, sp.M, sp.K, token_rows, 2 * kStageGroups)) return e;
        pr.scales = static_cast<const uint16_t*>(sp.scales);
        pr.y = static_cast<__nv_bfloat16*>(sp.y);
        pr.N = sp.N;
        pr.M = static_cast<int32_t>(sp.M);
        pr.G = static_cast<int32_t>(sp.K / 128);
        pr.T = (pr.G + kStageGroups - 1) / kStageGroups;
        pr.zeros = static_cast<const int8_t*>(sp.zeros);
        pr.row_groups = sp.K / (format == 0 ? 128 : format);
        const int64_t rbs = (sp.N + kRowsCta - 1) / kRowsCta;
        for (int64_t rb = 0; rb < rbs; ++rb)
            list.push_back({pr.T, make_uint2(static_cast<unsigned>(i), static_cast<unsigned>(rb))});
    }
    std::stable_sort(list.begin(), list.end(), [](const PlanItem& a, const PlanItem& b) { return a.stages > b.stages; });
    // The grid: every resident CTA, or, where three share an SM, two per SM
    // when that schedules better.  Three CTAs per SM stream about 5 % faster
    // than two (3.5–6.6 % measured on the balanced 200-matrix stack at M = 1,
    // 4, 8), so the modelled time of a grid is its largest CTA load × CTAs per
    // SM / (1.05 with three, 1 with two).  A layer with a few long items (the
    // 27B-class down matrix) balances better over fewer, longer-lived CTAs
    // (there two per SM measured 4–7 % faster than three).
    const int per_sm = std::max(1, max_ctas / sm_count);
    int32_t n_ctas = static_cast<int32_t>(std::min<int64_t>(max_ctas, n_items));
    if (per_sm >= 3) {
        const int32_t fewer = static_cast<int32_t>(std::min<int64_t>(static_cast<int64_t>(per_sm - 1) * sm_count, n_items));
        const double t_all = static_cast<double>(schedule_lpt(list, n_ctas, nullptr)) * per_sm / 1.05;
        const double t_fewer = static_cast<double>(schedule_lpt(list, fewer, nullptr)) * (per_sm - 1);
        if (t_fewer < t_all) n_ctas = fewer;
    }
    std::vector<std::vector<uint2>> per_cta;
    schedule_lpt(list, n_ctas, &per_cta);

    out->assign(grouped_plan_bytes(count, n_items, n_ctas), 0);
    GroupedHeader hdr = {};
    hdr.count = count;
    hdr.n_items = static_cast<int32_t>(n_items);
    hdr.token_rows = token_rows;
    hdr.n_ctas = n_ctas;
    hdr.format = format;
    std::memcpy(out->data(), &hdr, sizeof(hdr));
    std::memcpy(out->data() + sizeof(GroupedHeader), probs.data(), sizeof(GroupedProblem) * probs.size());
    int32_t* first = reinterpret_cast<int32_t*>(out->data() + sizeof(GroupedHeader) + sizeof(GroupedProblem) * count);
    uint2* items = reinterpret_cast<uint2*>(first + ((n_ctas + 2) & ~1));
    // The kernel loads items with 8-byte loads from a 128-byte aligned plan.
    if ((reinterpret_cast<uint8_t*>(items) - out->data()) % 8 != 0) return cudaErrorMisalignedAddress;
    int32_t k = 0;
    // The schedule's bins go to the CTAs in reverse, so that the first bins,
    // which hold the longest items, run on the CTAs launched last (measured 3–5 %
    // faster on the 27B-class layer at M = 1 and 5 and with zero points, no
    // change on the balanced 200-matrix stack; interleaving the bins over the
    // grid measured no gain).
    for (int32_t c = 0; c < n_ctas; ++c) {
        first[c] = k;
        for (const uint2& id : per_cta[static_cast<size_t>(n_ctas - 1 - c)]) items[k++] = id;
    }
    first[n_ctas] = k;
    *n_items_out = n_items;
    *n_ctas_out = n_ctas;
    return cudaSuccess;
}

namespace {

template <int QG>
cudaError_t launch_grouped_q(const void* plan, int32_t n_ctas, int token_rows, const DeviceInfo& dev,
                             cudaStream_t stream) {
    // A one-tile plan of the symmetric format scheduled over at most two CTAs
    // per SM runs the two-per-SM instance (deeper ring; exactly two fit, so
    // they spread evenly).  The affine formats always run two per SM.
    const bool two = QG != 0 || n_ctas <= 2 * dev.sm_count;
    constexpr int kOne = QG == 0 ? 3 : 2;
    switch (token_rows) {
        case 2: return two ? launch_grouped_t<1, 2, 2, QG>(plan, n_ctas, dev, stream)
                           : launch_grouped_t<1, 2, kOne, QG>(plan, n_ctas, dev, stream);
        case 4: return two ? launch_grouped_t<1, 4, 2, QG>(plan, n_ctas, dev, stream)
                           : launch_grouped_t<1, 4, kOne, QG>(plan, n_ctas, dev, stream);
        case 8: return two ? launch_grouped_t<1, 8, 2, QG>(plan, n_ctas, dev, stream)
                           : launch_grouped_t<1, 8, kOne, QG>(plan, n_ctas, dev, stream);
        case 16: return launch_grouped_t<2, 16, 2, QG>(plan, n_ctas, dev, stream);
        case 24: return launch_grouped_t<3, 24, 2, QG>(plan, n_ctas, dev, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_grouped(const void* plan, int32_t n_ctas, int token_rows, int format, const DeviceInfo& dev,
                           cudaStream_t stream) {
    if (n_ctas < 1) return cudaSuccess;
    switch (format) {
        case 0: return launch_grouped_q<0>(plan, n_ctas, token_rows, dev, stream);
        case 32: return launch_grouped_q<32>(plan, n_ctas, token_rows, dev, stream);
        case 64: return launch_grouped_q<64>(plan, n_ctas, token_rows, dev, stream);
        case 128: return launch_grouped_q<128>(plan, n_ctas, token_rows, dev, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace w4
