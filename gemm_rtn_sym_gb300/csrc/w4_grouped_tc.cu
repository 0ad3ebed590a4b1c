// Grouped tensor-core W4A16 matmul: many independent problems with M ≥ 25
// (for example the four matrices of a 70B-class layer in a speculative-verify
// pass) in one persistent launch.
//
// Source: Qwen3.5-4B quantisation study, §1 FFN example y = W x with ŵ = d·q
// (one d per 128 consecutive inputs) and §2 settings (4-bit weights, BF16
// inputs).  Every tile is computed exactly as by the single-matrix kernel in
// w4_gemm_tc.cu: bf16_rn(d·q) decoded into tensor memory as the MMA's A
// operand, the activation tile from shared memory, fp32 accumulation in TMEM
// over the whole K (no split), one bf16 rounding at the end.
//
// Why: one launch per matrix leaves SMs idle whenever a matrix has fewer
// 128-row tiles than there are SMs (a 10240-row matrix has 80), and split-K
// only partly recovers that.  Here the tiles of all problems are items
// assigned at plan time, longest first, to the least-loaded of one CTA per SM;
// each CTA keeps its TMA rings running from one tile to the next, and the MMA
// of a tile starts as soon as the previous tile's accumulator has been read.
#include <algorithm>
#include <cstring>
#include <mutex>
#include <queue>
#include <vector>

#include "w4_device.cuh"
#include "w4_internal.h"
#include "w4_tcgen05.cuh"

namespace w4 {
namespace {

constexpr int kBN = 128;            // weight rows per tile = MMA M
constexpr int kBK = 128;            // k per stage: one group
constexpr int kStages = 3;          // A (TMEM) + B (shared memory) stages
constexpr int kCodeStages = 2;      // code stages of two groups (two k stages) each
constexpr int kCodeStageBytes = 2 * kBN * 64;
// Warps: 0 activation TMA, 1 TMEM + MMA, 2 code TMA, 3 idle, 4..19 dequantise
// + epilogue (warp w takes TMEM lane quarter w % 4 and 32 k of each group).
constexpr int kCodeWarp = 2;
constexpr int kDequantWarp0 = 4;
constexpr int kDequantWarps = 16;
constexpr int kThreads = 32 * (kDequantWarp0 + kDequantWarps);
constexpr int kMaxBM = 256;
constexpr uint32_t kColA = 256;
constexpr uint32_t kTmemCols = 512;
constexpr int kMinSmemBytes = 120 * 1024;  // one CTA per SM: it takes all of TMEM

// Device layout: TcHeader | TcProblem[count] | int32 first[n_ctas + 1] (padded to
// 16 bytes, so that the 16-byte item records stay aligned) | uint4 items
struct alignas(128) TcHeader {
    int32_t count;
    int32_t n_items;
    int32_t n_ctas;
    int32_t max_bm;
    int32_t format;  // 0: symmetric group 128; 32, 64, 128: affine format of that group size
    int32_t reserved[27];
};

struct alignas(128) TcProblem {
    CUtensorMap x;      // 2-D over x [M, K]: boxes of 64 k × bm rows, 128-byte swizzle
    CUtensorMap codes;  // 3-D over codes [G][N][64 B]: boxes of 2 groups × 128 rows, 64-byte swizzle
    const uint16_t* scales;
    __nv_bfloat16* y;
    int64_t M;
    int64_t N;
    int32_t G;
    int32_t nkb;  // k stages (groups)
    int32_t bm;   // token rows per tile (multiple of 16, ≤ 256)
    int32_t pad;
    const int8_t* zeros;  // affine formats: int8 zero − 8 per group, or null
    int64_t row_groups;   // scales (and zeros) per row: K / group
    int32_t reserved[16];
};
static_assert(sizeof(TcHeader) == 128, "plan header");
static_assert(sizeof(TcProblem) == 384, "plan problem record");

// d·(c − z') for the pair i of a code word, as bf16x2: (136 + c) − (136 + z')
// is exact, the product rounds once.  off2 = bf16x2(136 + z') (136 for the
// symmetric format), d2 = bf16x2(d).  One shift, one LOP3, one subtract and
// one multiply per pair, written out in PTX (the bf16x2 arithmetic
// intrinsics cost about twice as many instructions here).
__device__ __forceinline__ uint32_t deq_pair_affine(uint32_t word, int i, uint32_t off2, uint32_t d2) {
    // (t & 0x000F000F) ^ 0x43084308 as one three-input logic op (LUT 0x6A),
    // written out: as plain C it compiled to about two LOP3s per pair.
    uint32_t t = word, biased;
    if (i != 0) asm("shr.b32 %0, %1, %2;" : "=r"(t) : "r"(word), "r"(4 * i));
    asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(biased) : "r"(t), "n"(0x000F000F), "r"(0x43084308u));
    uint32_t r;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(biased), "r"(off2));
    asm("mul.rn.bf16x2 %0, %0, %1;" : "+r"(r) : "r"(d2));
    return r;
}

__device__ __forceinline__ void tensormap_acquire(const void* map) {
    asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(map) : "memory");
}

// QG: 0 for the symmetric group-128 format; 32, 64 or 128 for the affine
// formats (group size QG, zero points where a problem has them).  Only the
// dequantisers' scale (and zero) reads differ.
template <int QG>
__global__ void __launch_bounds__(kThreads, 1)
gemm_tc_grouped_kernel(const uint8_t* __restrict__ plan, unsigned* status) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);

    const TcHeader* hdr = reinterpret_cast<const TcHeader*>(plan);
    const TcProblem* probs = reinterpret_cast<const TcProblem*>(plan + sizeof(TcHeader));
    const int32_t* first = reinterpret_cast<const int32_t*>(plan + sizeof(TcHeader) + sizeof(TcProblem) * hdr->count);
    const uint4* items = reinterpret_cast<const uint4*>(first + ((hdr->n_ctas + 4) & ~3));
    const int i_begin = first[blockIdx.x];
    const int i_end = first[blockIdx.x + 1];

    const uint32_t b_slot = static_cast<uint32_t>(hdr->max_bm) * 256u;  // two 64-k sub-tiles
    const uint32_t b_base = base;
    const uint32_t code_base = b_base + kStages * b_slot;
    const uint32_t bar_base = code_base + kCodeStages * kCodeStageBytes;
    auto full_a = [&](int s) { return bar_base + 8u * s; };
    auto full_b = [&](int s) { return bar_base + 8u * (kStages + s); };
    auto empty = [&](int s) { return bar_base + 8u * (2 * kStages + s); };
    auto code_full = [&](int c) { return bar_base + 8u * (3 * kStages + c); };
    auto code_empty = [&](int c) { return bar_base + 8u * (3 * kStages + kCodeStages + c); };
    const uint32_t accum_bar = bar_base + 8u * (3 * kStages + 2 * kCodeStages);
    const uint32_t acc_empty = accum_bar + 8u;
    const uint32_t drain_bar = accum_bar + 16u;
    const uint32_t tmem_slot = accum_bar + 24u;
    volatile uint32_t* tmem_slot_ptr = reinterpret_cast<volatile uint32_t*>(gbase + (tmem_slot - base));

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full_a(s), 32 * kDequantWarps);
            mbar_init(full_b(s), 1);
            mbar_init(empty(s), 1);
        }
        for (int c = 0; c < kCodeStages; ++c) {
            mbar_init(code_full(c), 1);
            mbar_init(code_empty(c), 32 * kDequantWarps * 2);  // every dequantiser, once per k stage
        }
        mbar_init(accum_bar, 1);
        mbar_init(acc_empty, 32 * kDequantWarps);
        mbar_init(drain_bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_async_smem();
    }
    if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_start();
    const uint32_t tmem_d = *tmem_slot_ptr;

    if (warp == 0) {
        // ------------------------------------------------ x tiles via TMA, every item back to back
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            int issued = 0;
            bool ok = true;
            for (int i = i_begin; i < i_end && ok; ++i) {
                const TcProblem* pr = probs + items[i].x;
                tensormap_acquire(&pr->x);
                const int m0 = static_cast<int>(items[i].z) * pr->bm;
                const uint32_t half_bytes = static_cast<uint32_t>(pr->bm) * 128u;
                for (int kb = 0; kb < pr->nkb; ++kb) {
                    if (!mbar_wait(empty(s), ph ^ 1u)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(full_b(s), 2u * half_bytes);
                    tma_load_2d(b_base + s * b_slot, &pr->x, kb * kBK, m0, full_b(s));
                    tma_load_2d(b_base + s * b_slot + half_bytes, &pr->x, kb * kBK + 64, m0, full_b(s));
                    ++issued;
                    if (++s == kStages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok) {
                record_status(status, kStatusTimeout);
                for (int j = issued > kStages ? issued - kStages : 0; j < issued; ++j)
                    mbar_wait(full_b(j % kStages), static_cast<uint32_t>(j / kStages) & 1u);
            }
        }
    } else if (warp == kCodeWarp) {
        // ------------------------------------------------ codes via TMA
        if (lane == 0) {
            int c = 0;
            uint32_t ph = 0;
            int issued = 0;
            bool ok = true;
            for (int i = i_begin; i < i_end && ok; ++i) {
                const TcProblem* pr = probs + items[i].x;
                tensormap_acquire(&pr->codes);
                const int n0 = static_cast<int>(items[i].y) * kBN;
                const int nst = (pr->nkb + 1) / 2;
                for (int t = 0; t < nst; ++t) {
                    if (!mbar_wait(code_empty(c), ph ^ 1u)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(code_full(c), kCodeStageBytes);
                    tma_load_3d(code_base + c * kCodeStageBytes, &pr->codes, 0, n0, 2 * t, code_full(c));
                    ++issued;
                    if (++c == kCodeStages) {
                        c = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok) {
                record_status(status, kStatusTimeout);
                for (int j = issued > kCodeStages ? issued - kCodeStages : 0; j < issued; ++j)
                    mbar_wait(code_full(j % kCodeStages), static_cast<uint32_t>(j / kCodeStages) & 1u);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issue
        // The whole warp runs the loop, so its control flow and the MMA
        // operands are warp-uniform (kept in uniform registers); one elected
        // lane issues the MMAs and the commits.  Issued from one lane's
        // divergent branch, each MMA cost about 100 cycles of issue on its
        // own (measured with clock64 stamps: 840 cycles per 8-MMA stage at
        // every token count), which bounded the tile.
        int s = 0;
        uint32_t ph = 0;
        uint32_t acc_ph = 0;
        bool ok = true;
        for (int i = i_begin; i < i_end && ok; ++i) {
            const TcProblem* pr = probs + items[i].x;
            const uint32_t idesc = idesc_bf16(pr->bm);
            const uint32_t half_bytes = static_cast<uint32_t>(pr->bm) * 128u;
            const int nkb = pr->nkb;
            // The previous item's accumulator must have been read out.
            ok = __all_sync(0xffffffffu, mbar_wait(acc_empty, acc_ph ^ 1u));
            if (!ok) break;
            acc_ph ^= 1u;
            tc_fence_after();
            for (int kb = 0; kb < nkb; ++kb) {
                ok = __all_sync(0xffffffffu, mbar_wait(full_b(s), ph) && mbar_wait(full_a(s), ph));
                if (!ok) break;
                tc_fence_after();
                const uint32_t a_s = tmem_d + kColA + 64u * s;
                const uint32_t b_s = b_base + s * b_slot;
                if (elect_one()) {
#pragma unroll
                    for (int ks = 0; ks < kBK / 16; ++ks)
                        mma_bf16_tmem_a(tmem_d, a_s + 8u * ks, sw128_desc(b_s + (ks >> 2) * half_bytes + (ks & 3) * 32),
                                        idesc, (kb | ks) != 0 ? 1u : 0u);
                    mma_commit(empty(s));
                }
                __syncwarp();
                if (++s == kStages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (ok && elect_one()) mma_commit(accum_bar);
            __syncwarp();
        }
        if (!ok && lane == 0) record_status(status, kStatusTimeout);
        // Every MMA issued has completed once this commit arrives.
        if (elect_one()) mma_commit(drain_bar);
        __syncwarp();
        mbar_wait(drain_bar, 0);
    } else if (warp >= kDequantWarp0) {
        // ------------------------------------------------ dequantisers + epilogue
        const int quarter = warp & 3;                  // TMEM lane quarter this warp may access
        const int part = (warp - kDequantWarp0) >> 2;  // which 32 k of each group
        const int t = quarter * 32 + lane;             // weight row within the tile
        const uint32_t lane_base = tmem_d + (static_cast<uint32_t>(quarter * 32) << 16);
        // Row t of a code stage: 64 bytes per group, 16-byte chunk j at j ^ ((t >> 1) & 3).
        const uint32_t row_chunk = static_cast<uint32_t>(t * 64) + (static_cast<uint32_t>(part ^ ((t >> 1) & 3)) << 4);
        int s = 0;
        uint32_t ph = 0;
        int c = 0;
        uint32_t cph = 0;
        uint32_t acc_ph = 0;
        bool ok = true;
        for (int i = i_begin; i < i_end; ++i) {
            const TcProblem* pr = probs + items[i].x;
            const int nkb = pr->nkb;
            const int bm = pr->bm;
            const int64_t n0 = static_cast<int64_t>(items[i].y) * kBN;
            const int64_t m0 = static_cast<int64_t>(items[i].z) * bm;
            const int64_t n = n0 + t < pr->N ? n0 + t : pr->N - 1;  // padding rows: zero codes, valid scale
            const int64_t rg = QG == 0 ? pr->G : pr->row_groups;
            const uint16_t* srow = pr->scales + n * rg;
            const int8_t* zrow = QG != 0 && pr->zeros ? pr->zeros + n * rg : nullptr;
            // The QG-group holding this thread's 32 k of group kb.
            auto gidx = [&](int kb) {
                return QG == 0 ? kb : kb * (128 / QG) + (QG == 64 ? (part >> 1) : (QG == 32 ? part : 0));
            };
            // Zeros as loaded (z', sign-extended); 136 + z' is formed where it is
            // used, so that the load issued a stage ahead is not waited for at once.
            auto zbits = [&](int g) { return static_cast<uint32_t>(zrow ? static_cast<int>(__ldg(zrow + g)) : 0); };
            if (ok) {
                uint32_t d_next = __ldg(srow + gidx(0));
                uint32_t z_next = QG != 0 ? zbits(gidx(0)) : 0u;
                for (int kb = 0; kb < nkb; ++kb) {
                    const int sub = kb & 1;  // group within the code stage
                    const uint32_t dbits = d_next, zb = 0x4308u + z_next;  // bf16(136 + z')
                    if (kb + 1 < nkb) {
                        d_next = __ldg(srow + gidx(kb + 1));
                        if (QG != 0) z_next = zbits(gidx(kb + 1));
                    }
                    const bool have = mbar_wait(code_full(c), cph);
                    if (!__all_sync(0xffffffffu, have)) {
                        ok = false;
                        break;
                    }
                    const uint4 q = lds128(code_base + c * kCodeStageBytes + sub * (kBN * 64) + row_chunk);
                    const uint32_t d2 = dbits | (dbits << 16), o2 = zb | (zb << 16);
                    const uint32_t words[4] = {q.x, q.y, q.z, q.w};
                    uint32_t v[16];  // column 4w + i of this thread's 16: pair i of word w
#pragma unroll
                    for (int w = 0; w < 4; ++w)
#pragma unroll
                        for (int p = 0; p < 4; ++p) v[4 * w + p] = deq_pair_affine(words[w], p, o2, d2);
                    // Release the code slot only after a proxy fence: the words were read
                    // through the generic proxy and the next TMA copy into the slot writes
                    // through the async proxy, so without the fence the copy could overtake
                    // a read still in flight (nothing keeps the decode that consumes the
                    // words ahead of the arrive).  A 40-run repeat test changed output
                    // elements in every attempt without it.
                    fence_async_smem();
                    mbar_arrive(code_empty(c));
                    if (sub == 1 || kb + 1 == nkb) {
                        // A last stage holding one group still owes one arrival.
                        if (sub == 0) mbar_arrive(code_empty(c));
                        if (++c == kCodeStages) {
                            c = 0;
                            cph ^= 1u;
                        }
                    }
                    const bool free_stage = mbar_wait(empty(s), ph ^ 1u);
                    if (!__all_sync(0xffffffffu, free_stage)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    tmem_st16(lane_base + kColA + 64u * s + 16u * part, v);
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(full_a(s));
                    if (++s == kStages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            // -------------------------------------------- epilogue of this item
            ok = __all_sync(0xffffffffu, ok);
            if (ok) ok = __all_sync(0xffffffffu, mbar_wait(accum_bar, acc_ph));
            acc_ph ^= 1u;
            if (!ok) {
                if (lane == 0) record_status(status, kStatusTimeout);
                continue;  // skip the rest; every wait from here on is skipped too
            }
            tc_fence_after();
            // The problem's fields are read once: the stores to y below could
            // alias the problem record for the compiler, which would otherwise
            // reload them after every store.
            const int64_t N = pr->N, M = pr->M;
            __nv_bfloat16* const y = pr->y;
            const int64_t ny = n0 + t;
            // The four warps of a lane quarter split the 16-column blocks.
            const int nb = bm >> 4;
            const int cbeg = ((part * nb) >> 2) << 4;
            const int cend = (((part + 1) * nb) >> 2) << 4;
            for (int c0 = cbeg; c0 < cend; c0 += 32) {
                const int nq = min(2, (cend - c0) >> 4);  // warp-uniform
                uint32_t v[2][16];
#pragma unroll
                for (int qq = 0; qq < 2; ++qq)
                    if (qq < nq) tmem_ld16_async(lane_base + static_cast<uint32_t>(c0 + 16 * qq), v[qq]);
                tmem_wait_ld();
#pragma unroll
                for (int qq = 0; qq < 2; ++qq) {
                    if (qq >= nq) continue;
                    reg_fence16(v[qq]);
                    if (ny < N) {
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const int64_t m = m0 + c0 + 16 * qq + j;
                            if (m < M) y[m * N + ny] = __float2bfloat16_rn(__uint_as_float(v[qq][j]));
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(acc_empty);  // the accumulator may be overwritten
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        __syncwarp();
        tmem_dealloc(tmem_d, kTmemCols);
    }
}

int tc_grouped_smem_bytes(int max_bm) {
    const int need = kStages * max_bm * 256 + kCodeStages * kCodeStageBytes + 8 * (3 * kStages + 2 * kCodeStages + 4) +
                     1024;
    return need > kMinSmemBytes ? need : kMinSmemBytes;
}

std::mutex g_tc_grouped_mutex;

}  // namespace

size_t tc_grouped_plan_bytes(int32_t count, int64_t n_items, int32_t n_ctas) {
    return sizeof(TcHeader) + sizeof(TcProblem) * static_cast<size_t>(count) +
           sizeof(int32_t) * static_cast<size_t>((n_ctas + 4) & ~3) + sizeof(uint4) * static_cast<size_t>(n_items);
}

int64_t tc_grouped_items(const GroupedSpec& sp) {
    const int64_t m_tiles = (sp.M + kMaxBM - 1) / kMaxBM;
    return ((sp.N + kBN - 1) / kBN) * m_tiles;
}

cudaError_t tc_grouped_plan_build(const GroupedSpec* specs, int32_t count, int format, int32_t n_ctas,
                                  std::vector<uint8_t>* out, int64_t* n_items_out, int32_t* n_ctas_out) {
    int64_t n_items = 0;
    for (int32_t i = 0; i < count; ++i) n_items += tc_grouped_items(specs[i]);
    if (n_items > 0x7fffffffLL || n_ctas < 1) return cudaErrorInvalidValue;
    if (n_ctas > n_items) n_ctas = static_cast<int32_t>(n_items);
    out->assign(tc_grouped_plan_bytes(count, n_items, n_ctas), 0);
    TcHeader hdr = {};
    hdr.count = count;
    hdr.n_items = static_cast<int32_t>(n_items);
    hdr.n_ctas = n_ctas;
    hdr.format = format;
    struct Item {
        int32_t cost;
        uint4 id;
    };
    std::vector<Item> list;
    list.reserve(static_cast<size_t>(n_items));
    int max_bm = 16;
    for (int32_t i = 0; i < count; ++i) {
        const GroupedSpec& sp = specs[i];
        const int64_t m_tiles = (sp.M + kMaxBM - 1) / kMaxBM;
        int64_t bm = (sp.M + m_tiles - 1) / m_tiles;
        bm = (bm + 15) / 16 * 16;
        max_bm = std::max(max_bm, static_cast<int>(bm));
        TcProblem pr;
        std::memset(&pr, 0, sizeof(pr));
        if (cudaError_t e = encode_x_map(&pr.x, sp.x, sp.M, sp.K, static_cast<int>(bm))) return e;
        if (cudaError_t e = encode_codes_stage_map(&pr.codes, sp.packed, sp.N, sp.K, kBN, 2, CU_TENSOR_MAP_SWIZZLE_64B))
            return e;
        pr.scales = static_cast<const uint16_t*>(sp.scales);
        pr.y = static_cast<__nv_bfloat16*>(sp.y);
        pr.M = sp.M;
        pr.N = sp.N;
        pr.G = static_cast<int32_t>(sp.K / 128);
        pr.nkb = static_cast<int32_t>(sp.K / kBK);  // groups
        pr.bm = static_cast<int32_t>(bm);
        pr.zeros = static_cast<const int8_t*>(sp.zeros);
        pr.row_groups = sp.K / (format == 0 ? 128 : format);
        std::memcpy(out->data() + sizeof(TcHeader) + sizeof(TcProblem) * i, &pr, sizeof(pr));
        const int64_t n_tiles = (sp.N + kBN - 1) / kBN;
        // Cost of a tile: its k stages, each 8 MMAs of N = bm, plus its epilogue.
        const int32_t cost = static_cast<int32_t>(pr.nkb * (bm + 32) / 16 + bm / 8);
        for (int64_t mt = 0; mt < m_tiles; ++mt)
            for (int64_t nt = 0; nt < n_tiles; ++nt)
                list.push_back({cost, make_uint4(static_cast<unsigned>(i), static_cast<unsigned>(nt),
                                                 static_cast<unsigned>(mt), 0u)});
    }
    hdr.max_bm = max_bm;
    std::memcpy(out->data(), &hdr, sizeof(hdr));
    std::stable_sort(list.begin(), list.end(), [](const Item& a, const Item& b) { return a.cost > b.cost; });
    using Load = std::pair<int64_t, int32_t>;
    std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
    for (int32_t c = 0; c < n_ctas; ++c) heap.push({0, c});
    std::vector<std::vector<uint4>> per_cta(static_cast<size_t>(n_ctas));
    for (const Item& it : list) {
        Load l = heap.top();
        heap.pop();
        per_cta[static_cast<size_t>(l.second)].push_back(it.id);
        l.first += it.cost;
        heap.push(l);
    }
    int32_t* first = reinterpret_cast<int32_t*>(out->data() + sizeof(TcHeader) + sizeof(TcProblem) * count);
    uint4* items = reinterpret_cast<uint4*>(first + ((n_ctas + 4) & ~3));
    // The kernel loads items with 16-byte loads from a 128-byte aligned plan.
    if ((reinterpret_cast<uint8_t*>(items) - out->data()) % 16 != 0) return cudaErrorMisalignedAddress;
    int32_t k = 0;
    for (int32_t c = 0; c < n_ctas; ++c) {
        first[c] = k;
        for (const uint4& id : per_cta[static_cast<size_t>(c)]) items[k++] = id;
    }
    first[n_ctas] = k;
    *n_items_out = n_items;
    *n_ctas_out = n_ctas;
    return cudaSuccess;
}

namespace {

template <int QG>
cudaError_t launch_tc_grouped_q(const void* plan, int32_t n_ctas, int max_bm, const DeviceInfo& dev,
                                cudaStream_t stream) {
    const int smem = tc_grouped_smem_bytes(max_bm);
    if (smem > dev.max_smem_optin) return cudaErrorInvalidConfiguration;
    int device = 0;
    if (cudaError_t e = cudaGetDevice(&device)) return e;
    {
        static bool attr_set[64];
        std::lock_guard<std::mutex> lock(g_tc_grouped_mutex);
        if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
        if (!attr_set[device]) {
            if (cudaError_t e = cudaFuncSetAttribute(gemm_tc_grouped_kernel<QG>,
                                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                     tc_grouped_smem_bytes(kMaxBM)))
                return e;
            attr_set[device] = true;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(n_ctas), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemm_tc_grouped_kernel<QG>, static_cast<const uint8_t*>(plan), dev.status);
}

}  // namespace

cudaError_t launch_tc_grouped(const void* plan, int32_t n_ctas, int max_bm, int format, const DeviceInfo& dev,
                              cudaStream_t stream) {
    if (n_ctas < 1) return cudaSuccess;
    switch (format) {
        case 0: return launch_tc_grouped_q<0>(plan, n_ctas, max_bm, dev, stream);
        case 32: return launch_tc_grouped_q<32>(plan, n_ctas, max_bm, dev, stream);
        case 64: return launch_tc_grouped_q<64>(plan, n_ctas, max_bm, dev, stream);
        case 128: return launch_tc_grouped_q<128>(plan, n_ctas, max_bm, dev, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace w4
