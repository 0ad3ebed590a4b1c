// Tensor-core W4A16 matmul for larger M: tcgen05.mma (kind::f16, BF16 × BF16 →
// FP32 in TMEM), weights dequantised straight into tensor memory as the MMA's
// A operand.
//
// Source: Qwen3.5-4B quantisation study, §1 FFN example y = W x with ŵ = d·q
// (one d per 128 consecutive inputs) and §2 settings (4-bit weights, BF16
// inputs).  The kernel multiplies bf16_rn(d·q), so its error per weight is at
// most 2^-9 relative; with fp32 accumulation and the final bf16 rounding the
// result stays inside 4e-3·Σ|ŵx| + 1 ulp.
//
// Tile: 128 weight rows (the MMA's M) × up to 256 tokens (the MMA's N; the
// token count is rounded up to a multiple of 16, padding rows of x read as
// zeros) per CTA, K streamed one group (128) per stage through a 3-stage ring;
// a cluster of up to 8 CTAs may split K (whole groups each) and sum its fp32
// partials over distributed shared memory.
//   warp 0      : TMA loads of x tiles (128-byte swizzle) into the ring;
//   warp 1      : allocates TMEM; the whole warp runs the stage loop and
//                 one elected lane issues 8 MMAs (K = 16 each) per stage with
//                 A read from TMEM, B from shared memory, and commits each
//                 stage back to its "empty" barrier (a 64-k stage left the
//                 barrier and commit overhead per stage as large as the MMAs'
//                 own time at N ≈ 200);
//   warp 2      : TMA loads of codes, two groups × 128 rows per copy;
//   warps 4..19 : one weight row and 32 k per thread (four warps per TMEM
//                 lane quarter) — read 16 bytes of codes from the code ring,
//                 decode nibble pairs to bf16 q, multiply by d (bf16,
//                 round-to-nearest) and store the 16 columns into the stage's
//                 A slot with tcgen05.st; after the last stage, read the
//                 accumulator back and store y (or the partial).  Sixteen
//                 dequantising warps rather than eight of 64 k each: the
//                 decode is latency-bound per warp, and with eight it set the
//                 stage time (on the grouped 27B-class layer at M = 64, 91 ->
//                 80 µs).
// Keeping A out of shared memory leaves the shared-memory port to the MMA's
// B reads and the code ring, which at 200+ tokens is what bounds the tile.
// Every mbarrier wait is bounded; a wait that runs out records a timeout in
// the status word and the CTA winds down (draining its own TMA copies and
// MMAs before freeing TMEM).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "w4_device.cuh"
#include "w4_internal.h"
#include "w4_tcgen05.cuh"

namespace w4 {
namespace {

constexpr int kBN = 128;            // weight rows per CTA = MMA M
constexpr int kBK = 128;            // k per stage: one group
constexpr int kStages = 3;          // A (decoded, in TMEM) + B (activation, shared memory) stages
constexpr int kCodeStages = 2;      // code stages of two groups (two k stages) each
constexpr int kCodeStageBytes = 2 * kBN * 64;  // 16 KB: [group][row][64 B], 64-byte swizzle
// Warps: 0 activation TMA, 1 TMEM + MMA, 2 code TMA, 3 idle, 4..19 dequantise
// + epilogue (four per TMEM lane quarter, each 32 k of the k-block).
constexpr int kCodeWarp = 2;
constexpr int kDequantWarp0 = 4;
constexpr int kDequantWarps = 16;
constexpr int kThreads = 32 * (kDequantWarp0 + kDequantWarps);
constexpr int kMaxBM = 256;
// Tensor memory: accumulator in columns [0, 256), decoded A stages of 64
// columns (128 k of bf16 pairs) from column 256.  The whole 512 columns are
// taken, so the shared memory request below keeps one CTA per SM.
constexpr uint32_t kColA = 256;
constexpr uint32_t kTmemCols = 512;
constexpr int kMinSmemBytes = 120 * 1024;

struct TcArgs {
    const uint16_t* scales;
    const int8_t* zeros;  // affine formats only; nullptr: symmetric
    int64_t row_groups;   // scales (and zeros) per row: K / group
    __nv_bfloat16* y;
    int64_t M, N, K;
    int bm;
    int split;  // CTAs of a cluster splitting K (1 = no split)
    unsigned* status;
};

// d·(c − z') for the pair i of a code word, as bf16x2: (136 + c) − (136 + z') is
// exact, the product rounds once.  off2 = bf16x2(136 + z'), d2 = bf16x2(d).
__device__ __forceinline__ uint32_t deq_pair(uint32_t word, int i, uint32_t off2, uint32_t d2) {
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

// A dequantising thread's running window over its weight row's scale (and
// zero) entries: eight consecutive entries from an 8-aligned index, loaded as
// one 16-byte (and one 8-byte) load, with the next eight requested as soon as
// the window moves onto the current ones.  Per k stage a thread needs one
// entry (its 32-k chunk's group); loaded one by one, the scale and the zero
// are two scattered load instructions per thread and stage (32 sectors per
// warp load).  Usable when a row holds a multiple of 8 entries and the scale
// (zero) row is 16- (8-) byte aligned; entries are read only inside the row.
struct ScaleWindow {
    const uint16_t* srow;
    const int8_t* zrow;  // null: no zeros (z' = 0)
    int64_t rg;          // entries per row
    int64_t base;        // index of s_cur's first entry
    uint4 s_cur, s_nxt;
    uint2 z_cur, z_nxt;

    __device__ __forceinline__ void load(int64_t at, uint4& s, uint2& z) const {
        if (at < rg) {
            s = __ldg(reinterpret_cast<const uint4*>(srow + at));
            z = zrow ? __ldg(reinterpret_cast<const uint2*>(zrow + at)) : make_uint2(0u, 0u);
        }
    }
    __device__ __forceinline__ void start(int64_t ia) {
        base = ia & ~int64_t{7};
        s_cur = s_nxt = make_uint4(0u, 0u, 0u, 0u);
        z_cur = z_nxt = make_uint2(0u, 0u);
        load(base, s_cur, z_cur);
        load(base + 8, s_nxt, z_nxt);
    }
    // Entry ia (≥ the previous call's, by at most 8): scale bits d and zero z'.
    __device__ __forceinline__ void get(int64_t ia, uint32_t& d, int& z) {
        if (ia >= base + 8) {
            s_cur = s_nxt;
            z_cur = z_nxt;
            base += 8;
            load(base + 8, s_nxt, z_nxt);
        }
        const int j = static_cast<int>(ia - base);
        const uint32_t w = j < 4 ? (j < 2 ? s_cur.x : s_cur.y) : (j < 6 ? s_cur.z : s_cur.w);
        d = (j & 1) ? (w >> 16) : (w & 0xFFFFu);
        const uint32_t zw = j < 4 ? z_cur.x : z_cur.y;
        z = static_cast<int>(static_cast<int8_t>((zw >> (8 * (j & 3))) & 0xFFu));
    }
};

// QG: 0 for the symmetric group-128 format; 32, 64 or 128 for the affine
// formats (group size QG, zero points when args.zeros is set).  Only the
// dequantisers' scale (and zero) reads differ.
template <int QG>
__global__ void __launch_bounds__(kThreads, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_codes,
               const TcArgs args) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);

    const int bm = args.bm;
    const uint32_t b_half_bytes = static_cast<uint32_t>(bm) * 128u;  // one 64-k sub-tile
    const uint32_t b_tile_bytes = 2u * b_half_bytes;
    const uint32_t b_base = base;
    const uint32_t code_base = b_base + kStages * b_tile_bytes;
    const uint32_t bar_base = code_base + kCodeStages * kCodeStageBytes;
    auto full_a = [&](int s) { return bar_base + 8u * s; };
    auto full_b = [&](int s) { return bar_base + 8u * (kStages + s); };
    auto empty = [&](int s) { return bar_base + 8u * (2 * kStages + s); };
    auto code_full = [&](int c) { return bar_base + 8u * (3 * kStages + c); };
    auto code_empty = [&](int c) { return bar_base + 8u * (3 * kStages + kCodeStages + c); };
    const uint32_t accum_bar = bar_base + 8u * (3 * kStages + 2 * kCodeStages);
    const uint32_t tmem_slot = accum_bar + 8u;
    volatile uint32_t* tmem_slot_ptr =
        reinterpret_cast<volatile uint32_t*>(gbase + (tmem_slot - base));

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kBN;
    const int64_t m0 = static_cast<int64_t>(blockIdx.y) * bm;
    const int split = args.split;
    const uint32_t rank = split > 1 ? cluster_rank() : 0u;
    const int64_t G = args.K >> 7;
    // K range of this CTA, in whole groups (a code stage holds two groups).
    const int64_t g_lo = (static_cast<int64_t>(rank) * G) / split;
    const int64_t g_hi = (static_cast<int64_t>(rank + 1) * G) / split;
    const int kb_lo = static_cast<int>(g_lo);  // stages are groups
    const int nkb = static_cast<int>(g_hi - g_lo);

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
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_async_smem();
    }
    if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_start();
    const uint32_t tmem_d = *tmem_slot_ptr;

    bool ok = true;
    if (warp == 0) {
        // ------------------------------------------------ x tiles via TMA
        if (lane == 0) {
            int issued = 0;
            for (int kb = 0; kb < nkb && ok; ++kb) {
                const int s = kb % kStages;
                const uint32_t r = static_cast<uint32_t>(kb / kStages);
                if (!mbar_wait(empty(s), (r & 1u) ^ 1u)) { ok = false; break; }
                mbar_arrive_expect_tx(full_b(s), b_tile_bytes);
                tma_load_2d(b_base + s * b_tile_bytes, &tmap_x, (kb_lo + kb) * kBK, static_cast<int>(m0), full_b(s));
                tma_load_2d(b_base + s * b_tile_bytes + b_half_bytes, &tmap_x, (kb_lo + kb) * kBK + 64,
                            static_cast<int>(m0), full_b(s));
                issued = kb + 1;
            }
            if (!ok) {
                record_status(args.status, kStatusTimeout);
                // Drain: every issued copy lands before the CTA may exit.
                for (int kb = (issued > kStages ? issued - kStages : 0); kb < issued; ++kb)
                    mbar_wait(full_b(kb % kStages), static_cast<uint32_t>(kb / kStages) & 1u);
            }
        }
    } else if (warp == kCodeWarp) {
        // ------------------------------------------------ codes via TMA
        if (lane == 0) {
            const int nst = (nkb + 1) / 2;
            int issued = 0;
            for (int t = 0; t < nst; ++t) {
                const int c = t % kCodeStages;
                if (!mbar_wait(code_empty(c), (static_cast<uint32_t>(t / kCodeStages) & 1u) ^ 1u)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(code_full(c), kCodeStageBytes);
                tma_load_3d(code_base + c * kCodeStageBytes, &tmap_codes, 0, static_cast<int>(n0),
                            static_cast<int>(g_lo + 2 * t), code_full(c));  // groups beyond g_hi are not read by this CTA
                issued = t + 1;
            }
            if (!ok) {
                record_status(args.status, kStatusTimeout);
                for (int t = issued > kCodeStages ? issued - kCodeStages : 0; t < issued; ++t)
                    mbar_wait(code_full(t % kCodeStages), static_cast<uint32_t>(t / kCodeStages) & 1u);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issue
        // The whole warp runs the loop, so its control flow and the MMA
        // operands are warp-uniform (kept in uniform registers); one elected
        // lane issues the MMAs and the commits.  Issued from one lane's
        // divergent branch, each MMA cost about 100 cycles of issue on its
        // own, which bounded the tile at every token count.
        const uint32_t idesc = idesc_bf16(bm);
        for (int kb = 0; kb < nkb; ++kb) {
            const int s = kb % kStages;
            const uint32_t par = static_cast<uint32_t>(kb / kStages) & 1u;
            ok = __all_sync(0xffffffffu, mbar_wait(full_b(s), par) && mbar_wait(full_a(s), par));
            if (!ok) break;
            tc_fence_after();
            const uint32_t a_s = tmem_d + kColA + 64u * s;
            const uint32_t b_s = b_base + s * b_tile_bytes;
            if (elect_one()) {
#pragma unroll
                for (int ks = 0; ks < kBK / 16; ++ks)
                    mma_bf16_tmem_a(tmem_d, a_s + 8u * ks,
                                    sw128_desc(b_s + (ks >> 2) * b_half_bytes + (ks & 3) * 32), idesc,
                                    (kb | ks) != 0 ? 1u : 0u);
                mma_commit(empty(s));
            }
            __syncwarp();
        }
        if (elect_one()) mma_commit(accum_bar);  // also tracks MMAs issued before an abort
        __syncwarp();
        if (!ok && lane == 0) record_status(args.status, kStatusTimeout);
    } else if (warp >= kDequantWarp0) {
        // ------------------------------------------------ dequantisers
        const int quarter = warp & 3;                  // TMEM lane quarter this warp may access
        const int part = (warp - kDequantWarp0) >> 2;  // which 32 k of each group
        const int t = quarter * 32 + lane;             // weight row within the tile
        const uint32_t lane_base = tmem_d + (static_cast<uint32_t>(quarter * 32) << 16);
        const int64_t n = n0 + t < args.N ? n0 + t : args.N - 1;  // padding rows: zero codes, valid scale
        const int64_t rg = QG == 0 ? G : args.row_groups;
        const uint16_t* srow = args.scales + n * rg;
        const int8_t* zrow = QG != 0 && args.zeros ? args.zeros + n * rg : nullptr;
        // Index of the scale (and zero) entry of this thread's 32-k chunk in k stage kb.
        auto entry = [&](int kb) -> int64_t {
            const int64_t gk = kb_lo + kb;
            return QG == 64 ? 2 * gk + (part >> 1) : (QG == 32 ? 4 * gk + part : gk);
        };
        // The scale bits and the zero of the 32-k chunk this thread
        // dequantises in k stage kb, as loaded: {d, z'} (packed into bf16x2
        // only where they are used, so that a load issued stages ahead is not
        // waited for at once).
        auto load_dz = [&](int kb, uint32_t (&o)[2]) {
            const int64_t ia = entry(kb);
            o[0] = __ldg(srow + ia);
            o[1] = static_cast<uint32_t>(zrow ? static_cast<int>(__ldg(zrow + ia)) : 0);
        };
        // Row t of a code stage: 64 bytes per group, 16-byte chunk j at j ^ ((t >> 1) & 3).
        const uint32_t row_chunk = static_cast<uint32_t>(t * 64) + (static_cast<uint32_t>(part ^ ((t >> 1) & 3)) << 4);
        // With zero points, scales and zeros through a window of eight entries
        // where the rows allow it (asymmetric group 128 / 64 / 32 on the
        // 57344×8192 matrix at M = 208: 152 → 132, 183 → 138, 181 → 145 µs);
        // else one load per stage issued two stages ahead (without zeros the
        // window measured no faster: 130 against 139 µs at group 32).
        const bool windowed = zrow != nullptr && (rg & 7) == 0 && (reinterpret_cast<uintptr_t>(srow) & 15u) == 0 &&
                              (reinterpret_cast<uintptr_t>(zrow) & 7u) == 0;
        ScaleWindow win;
        win.srow = srow;
        win.zrow = zrow;
        win.rg = rg;
        uint32_t dz1[2] = {0u, 0u};
        uint32_t dz2[2] = {0u, 0u};
        if (windowed) {
            if (nkb > 0) win.start(entry(0));
        } else {
            if (nkb > 0) load_dz(0, dz1);
            if (nkb > 1) load_dz(1, dz2);
        }
        for (int kb = 0; kb < nkb && ok; ++kb) {
            const int s = kb % kStages;
            const uint32_t r = static_cast<uint32_t>(kb / kStages);
            const int cst = (kb >> 1) % kCodeStages;
            const int sub = kb & 1;  // group within the code stage
            if (windowed) {
                int zq;
                win.get(entry(kb), dz1[0], zq);
                dz1[1] = static_cast<uint32_t>(zq);
            }
            const uint32_t zb = 0x4308u + dz1[1];  // bf16(136 + z')
            const uint32_t d2 = dz1[0] | (dz1[0] << 16), o2 = zb | (zb << 16);
            if (!windowed) {
                dz1[0] = dz2[0];
                dz1[1] = dz2[1];
                if (kb + 2 < nkb) load_dz(kb + 2, dz2);
            }
            const bool have = mbar_wait(code_full(cst), static_cast<uint32_t>((kb >> 1) / kCodeStages) & 1u);
            if (!__all_sync(0xffffffffu, have)) { ok = false; break; }
            const uint4 q = lds128(code_base + cst * kCodeStageBytes + sub * (kBN * 64) + row_chunk);
            const uint32_t words[4] = {q.x, q.y, q.z, q.w};
            uint32_t v[16];  // column 4w + i of this thread's 16: pair i of word w
#pragma unroll
            for (int w = 0; w < 4; ++w)
#pragma unroll
                for (int i = 0; i < 4; ++i) v[4 * w + i] = deq_pair(words[w], i, o2, d2);
            // Release the code slot only after a proxy fence: the words were read
            // through the generic proxy and the next TMA copy into the slot writes
            // through the async proxy, so without the fence the copy could overtake
            // a read still in flight (nothing keeps the decode that consumes the
            // words ahead of the arrive).  A 40-run repeat test changed output
            // elements in every attempt without it.
            fence_async_smem();
            mbar_arrive(code_empty(cst));
            const bool free_stage = mbar_wait(empty(s), (r & 1u) ^ 1u);
            if (!__all_sync(0xffffffffu, free_stage)) { ok = false; break; }
            tc_fence_after();
            tmem_st16(lane_base + kColA + 64u * s + 16u * part, v);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(full_a(s));
        }
        if (!ok) record_status(args.status, kStatusTimeout);

        // ------------------------------------------------ epilogue
        // tcgen05.ld is warp-collective: decide per warp, not per thread.
        ok = __all_sync(0xffffffffu, ok);
        const bool acc_ready = ok && __all_sync(0xffffffffu, mbar_wait(accum_bar, 0));
        if (acc_ready) {
            tc_fence_after();
            const int64_t ny = n0 + t;
            // With a split, the fp32 partial goes to shared memory (the rings
            // are idle now) as red[column][row], for the cluster reduction below.
            float* red = reinterpret_cast<float*>(gbase);
            // The four warps of a lane quarter split the 16-column blocks.
            const int nb = bm >> 4;
            const int cbeg = ((part * nb) >> 2) << 4;
            const int cend = (((part + 1) * nb) >> 2) << 4;
            // Up to two 16-column loads in flight per wait.
            for (int c0 = cbeg; c0 < cend; c0 += 32) {
                const int nq = min(2, (cend - c0) >> 4);  // warp-uniform
                uint32_t v[2][16];
#pragma unroll
                for (int q = 0; q < 2; ++q)
                    if (q < nq) tmem_ld16_async(lane_base + static_cast<uint32_t>(c0 + 16 * q), v[q]);
                tmem_wait_ld();
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    if (q >= nq) continue;
                    reg_fence16(v[q]);
                    const int cq = c0 + 16 * q;
                    if (split > 1) {
#pragma unroll
                        for (int j = 0; j < 16; ++j) red[(cq + j) * kBN + t] = __uint_as_float(v[q][j]);
                    } else if (ny < args.N) {
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const int64_t m = m0 + cq + j;
                            if (m < args.M)
                                args.y[m * args.N + ny] = __float2bfloat16_rn(__uint_as_float(v[q][j]));
                        }
                    }
                }
            }
        } else if (ok) {
            record_status(args.status, kStatusTimeout);
        }
    }

    if (split > 1) {
        // Split-K: CTA `rank` sums rows [rank*128/split, (rank+1)*128/split) of
        // every CTA's partial, in rank order, and stores them.
        cluster_sync();
        const int r0 = (static_cast<int>(rank) * kBN) / split;
        const int r1 = (static_cast<int>(rank + 1) * kBN) / split;
        const int rows = r1 - r0;
        const uint32_t red_addr = base;
        for (int e = threadIdx.x; e < rows * bm; e += kThreads) {
            const int rowt = r0 + e % rows;
            const int c = e / rows;
            const int64_t ny = n0 + rowt;
            const int64_t m = m0 + c;
            // All of the element's remote loads are issued before the first add.
            const uint32_t a = red_addr + static_cast<uint32_t>((c * kBN + rowt) * 4);
            float p[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) p[r] = r < split ? ld_cluster_f32(a, static_cast<uint32_t>(r)) : 0.0f;
            float v = 0.0f;
#pragma unroll
            for (int r = 0; r < 8; ++r)
                if (r < split) v += p[r];
            if (ny < args.N && m < args.M) args.y[m * args.N + ny] = __float2bfloat16_rn(v);
        }
        cluster_sync();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        // MMAs still in flight (after an abort) must finish before TMEM is freed.
        if (lane == 0) mbar_wait(accum_bar, 0);
        __syncwarp();
        tmem_dealloc(tmem_d, kTmemCols);
    }
}

// ------------------------------------------------------------------- host
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
std::mutex g_attr_mutex;

cudaError_t get_encoder() {
    std::call_once(g_encode_once, [] {
        cudaDriverEntryPointQueryResult q;
        void* fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode ? cudaSuccess : cudaErrorNotSupported;
}

}  // namespace

cudaError_t encode_x_map(CUtensorMap* map, const void* x, int64_t M, int64_t K, int box_rows) {
    if (cudaError_t e = get_encoder()) return e;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
    const cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    if (g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(x), dims, strides, box, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    return cudaSuccess;
}

cudaError_t encode_codes_stage_map(CUtensorMap* map, const void* packed, int64_t N, int64_t K, int rows,
                                   int groups, CUtensorMapSwizzle swizzle) {
    if (cudaError_t e = get_encoder()) return e;
    // codes viewed as [G groups][N rows][64 bytes]: byte (b, n, g) at n*K/2 + g*64 + b.
    const cuuint64_t dims[3] = {64u, static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(K / 128)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(K / 2), 64u};
    const cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(rows), static_cast<cuuint32_t>(groups)};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(packed), dims, strides, box, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    return cudaSuccess;
}

cudaError_t encode_x_stage_map(CUtensorMap* map, const void* x, int64_t M, int64_t K, int rows, int blocks) {
    if (cudaError_t e = get_encoder()) return e;
    // x viewed as [K/64 blocks][M rows][64 k]: element (k, m, b) at m*2K + b*128 + 2k bytes.
    const cuuint64_t dims[3] = {64u, static_cast<cuuint64_t>(M), static_cast<cuuint64_t>(K / 64)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(K) * 2, 128u};
    const cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(rows), static_cast<cuuint32_t>(blocks)};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(x), dims, strides, box, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    return cudaSuccess;
}

namespace {

int smem_bytes(int bm) {
    const int need = kStages * bm * 256 + kCodeStages * kCodeStageBytes + 8 * (3 * kStages + 2 * kCodeStages + 2) + 1024;
    const int red = bm * kBN * 4 + 1024;  // split-K partials reuse the rings
    const int n = need > red ? need : red;
    return n > kMinSmemBytes ? n : kMinSmemBytes;
}

template <int QG>
cudaError_t launch_gemm_tc_q(const void* x, int64_t M, int64_t N, int64_t K, const void* packed,
                             const void* scales, const void* zeros, void* y, const DeviceInfo& dev,
                             cudaStream_t stream) {
    static bool attr_set[64];
    const int64_t m_tiles = (M + kMaxBM - 1) / kMaxBM;
    int64_t bm = (M + m_tiles - 1) / m_tiles;
    bm = (bm + 15) / 16 * 16;
    const int64_t n_tiles = (N + kBN - 1) / kBN;
    if (n_tiles > 0x7fffffffLL || m_tiles > 65535 || M > 0x7fffffffLL || K > 0x7fffffffLL)
        return cudaErrorInvalidConfiguration;
    const int smem = smem_bytes(static_cast<int>(bm));
    if (smem > dev.max_smem_optin) return cudaErrorInvalidConfiguration;

    CUtensorMap tmap;
    if (cudaError_t e = encode_x_map(&tmap, x, M, K, static_cast<int>(bm))) return e;
    CUtensorMap tmap_codes;
    if (cudaError_t e = encode_codes_stage_map(&tmap_codes, packed, N, K, kBN, 2, CU_TENSOR_MAP_SWIZZLE_64B))
        return e;

    int device = 0;
    if (cudaError_t e = cudaGetDevice(&device)) return e;
    {
        std::lock_guard<std::mutex> lock(g_attr_mutex);
        if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
        if (!attr_set[device]) {
            if (cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<QG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                     smem_bytes(kMaxBM)))
                return e;
            attr_set[device] = true;
        }
    }
    // Split-K over a cluster when the tiles alone leave SMs idle: pick the
    // cluster size (1..8, at least 2 groups per CTA) that needs the fewest
    // rounds of k-stage work, given how many such clusters fit at once.
    const int64_t nkb_all = K / kBK;
    int split = 1;
    {
        double best = 0.0;
        for (int s = 1; s <= 8 && s * 2 <= K / 128; ++s) {
            cudaLaunchConfig_t q = {};
            q.gridDim = dim3(static_cast<unsigned>(n_tiles), static_cast<unsigned>(m_tiles), static_cast<unsigned>(s));
            q.blockDim = dim3(kThreads, 1, 1);
            q.dynamicSmemBytes = smem;
            cudaLaunchAttribute qa[1];
            qa[0].id = cudaLaunchAttributeClusterDimension;
            qa[0].val.clusterDim.x = 1;
            qa[0].val.clusterDim.y = 1;
            qa[0].val.clusterDim.z = static_cast<unsigned>(s);
            q.attrs = qa;
            q.numAttrs = 1;
            int clusters = 0;
            if (cudaOccupancyMaxActiveClusters(&clusters, gemm_tc_kernel<QG>, &q) != cudaSuccess || clusters < 1) {
                cudaGetLastError();
                continue;
            }
            const int64_t waves = (n_tiles * m_tiles + clusters - 1) / clusters;
            const double cost = static_cast<double>(waves) * static_cast<double>((nkb_all + s - 1) / s) +
                                (s > 1 ? 1.0 : 0.0);  // the reduction costs about one k stage
            if (best == 0.0 || cost < best) {
                best = cost;
                split = s;
            }
        }
    }

    TcArgs args;
    args.scales = static_cast<const uint16_t*>(scales);
    args.zeros = static_cast<const int8_t*>(zeros);
    args.row_groups = QG == 0 ? K / 128 : K / QG;
    args.y = static_cast<__nv_bfloat16*>(y);
    args.M = M;
    args.N = N;
    args.K = K;
    args.bm = static_cast<int>(bm);
    args.split = split;
    args.status = dev.status;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(n_tiles), static_cast<unsigned>(m_tiles), static_cast<unsigned>(split));
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = static_cast<unsigned>(split);
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<QG>, tmap, tmap_codes, args);
}

}  // namespace

cudaError_t launch_gemm_tc(const void* x, int64_t M, int64_t N, int64_t K, const void* packed,
                           const void* scales, void* y, const DeviceInfo& dev, cudaStream_t stream) {
    return launch_gemm_tc_q<0>(x, M, N, K, packed, scales, nullptr, y, dev, stream);
}

cudaError_t launch_gemm_tc_affine(const void* x, int64_t M, int64_t N, int64_t K, int group, const void* packed,
                                  const void* scales, const void* zeros, void* y, const DeviceInfo& dev,
                                  cudaStream_t stream) {
    switch (group) {
        case 32: return launch_gemm_tc_q<32>(x, M, N, K, packed, scales, zeros, y, dev, stream);
        case 64: return launch_gemm_tc_q<64>(x, M, N, K, packed, scales, zeros, y, dev, stream);
        default: return launch_gemm_tc_q<128>(x, M, N, K, packed, scales, zeros, y, dev, stream);
    }
}

}  // namespace w4
