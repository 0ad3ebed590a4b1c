// GPTQ quantiser into the RTN storage (packed codes + bf16 scales).
//
// Source: Qwen3.5-4B quantisation study, §2 settings table (GPTQ, same storage
// as RTN, damping 0.01, original column order, 128-column computation blocks
// whose corrections carry into later blocks), §2 H' = H + λI with
// λ = 0.01·mean(diag H), and the method table (quantise one column, then
// correct the remaining weights).  The correction rule is the published GPTQ
// algorithm (Frantar et al., 2022): with U the upper-triangular factor of
// (H')⁻¹ = UᵀU, column c's rounding error divided by U[c, c] moves every later
// column k by −err·U[c, k].
//
// Everything runs in fp64, so that each rounding decision is taken on the same
// values as in the oracle (fp32 state would differ from it by ~1e-7 and flip a
// few codes per matrix, each flip then changing the rest of its row).
//
// Factor (once per calibration statistic H, shared by every matrix that reads
// the same input).  With J the order-reversing permutation, the Cholesky
// factor L̃ of J H' J gives H' = Ũ Ũᵀ with Ũ = J L̃ J upper triangular, so
// U = Ũ⁻¹ = J L̃⁻¹ J is upper triangular with Uᵀ U = (H')⁻¹: one Cholesky and
// one triangular inverse, (2/3)·K³ flops, instead of inverting H' and
// factoring the inverse.  All in own kernels, blocked by 64:
//  1. λ, and A = J H' J = J (fp64(H) + λI) J written reversed;
//  2. right-looking Cholesky of A in place: per 64-column panel, the diagonal
//     block factored by one CTA in shared memory, the rows below solved
//     against it (one thread per row), then the trailing lower triangle
//     updated by the fp64 tile product A −= P Pᵀ;
//  3. X = L̃⁻¹ into U's memory by right-looking block substitution on the
//     identity: per 64-row block, the block row solved against the diagonal
//     block (one thread per column), then the rows below updated by the fp64
//     tile product X −= L X_block;
//  4. the reversal of X's element order, which is row-major U, in place.
// Quantise (per matrix):
//  5. W widened to fp64;
//  6. per 128-column block: the sweep kernel rounds the block's columns one
//     after another, eight threads carrying each row through the block in
//     shared memory, writes the block's codes, scales and errors E; then the
//     later columns get W[:, i2:] −= E·U[i1:i2, i2:] by the fp64 tile product,
//     which carries N·K² flops in total and bounds the call on GB300's fp64
//     rate (about 1.0 TFLOP/s measured for both DFMA and fp64 MMA, so the tile
//     product uses plain DFMA).
// A failed factorization (H' not positive definite: a pivot ≤ 0) is reported
// through the library's status word as W4_ERR_NUMERIC.
#include <mutex>

#include "w4_device.cuh"
#include "w4_internal.h"

namespace w4 {
namespace {

constexpr int kBlock = 128;              // columns per computation block
constexpr int kSweepRows = 16;           // rows per CTA
constexpr int kRowThreads = 8;           // threads per row (each owns 16 of the block's columns)
constexpr int kSweepThreads = kSweepRows * kRowThreads;
// Doubles per shared-memory column: ≡ 2 (mod 16), so the 16 lanes of a half
// warp (two rows × eight column residues) hit distinct bank pairs.
constexpr int kPitch = kSweepRows + 2;
constexpr int kSweepSmem = kBlock * kPitch * 8 + kBlock * kSweepRows;
constexpr unsigned kStatusNumeric = 6;   // W4_ERR_NUMERIC

size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

constexpr int kPanel = 64;               // factor block size (K is a multiple of 128)

// Factor workspace: λ, then A = J H' J (K×K fp64), factored in place.
struct FactorLayout {
    size_t lam, a, total;
};

FactorLayout factor_layout(int64_t K) {
    FactorLayout l;
    l.lam = 0;
    l.a = 256;
    l.total = align256(l.a + static_cast<size_t>(K) * K * 8);
    return l;
}

// Quantise workspace: fp64 copy of W and the errors of one block.
struct QuantLayout {
    size_t wd, e, total;
};

QuantLayout quant_layout(int64_t N, int64_t K) {
    QuantLayout l;
    l.wd = 0;
    l.e = align256(static_cast<size_t>(N) * K * 8);
    l.total = align256(l.e + static_cast<size_t>(N) * kBlock * 8);
    return l;
}

// λ = damp · mean(diag H), summed in fp64 in a fixed order.
__global__ void __launch_bounds__(256) diag_mean_kernel(const float* __restrict__ H, int64_t K, double damp,
                                                        double* __restrict__ lam) {
    __shared__ double part[256];
    double s = 0.0;
    for (int64_t i = threadIdx.x; i < K; i += 256) s += static_cast<double>(H[i * K + i]);
    part[threadIdx.x] = s;
    __syncthreads();
    for (int w = 128; w > 0; w >>= 1) {
        if (threadIdx.x < w) part[threadIdx.x] += part[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0) *lam = damp * part[0] / static_cast<double>(K);
}

// A = J (fp64(H) + λ I) J: element p of A is element K² − 1 − p of H'.
__global__ void damp_reversed_kernel(const float* __restrict__ H, int64_t K, const double* __restrict__ lam,
                                     double* __restrict__ A) {
    const double l = *lam;
    const int64_t n = K * K;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = i / K, c = i - r * K;
        A[i] = static_cast<double>(H[n - 1 - i]) + (r == c ? l : 0.0);
    }
}

// X (row-major, L̃⁻¹ on and below the diagonal) becomes row-major
// U[r][c] = X[K−1−r][K−1−c] in place: element p = r·K + c takes element
// K² − 1 − p, so reversing the element order is the whole permutation.
__global__ void reverse_kernel(double* __restrict__ X, int64_t K) {
    const int64_t n = K * K;
    for (int64_t p = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; p < n / 2;
         p += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t q = n - 1 - p;
        const double t = X[p];
        X[p] = X[q];
        X[q] = t;
    }
}

__global__ void widen_kernel(const uint16_t* __restrict__ W, int64_t n, double* __restrict__ Wd) {
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        Wd[i] = static_cast<double>(__uint_as_float(static_cast<uint32_t>(W[i]) << 16));
}

// ------------------------------------------------------------ factor kernels
// Cholesky of the diagonal block A[P:P+64, P:P+64] (lower triangle, in place),
// unblocked and right-looking in shared memory: per column j, the pivot's
// square root, the column below divided by it, then the trailing lower
// triangle reduced by the column's outer product.  One CTA.
constexpr int kPotrfThreads = 256;
constexpr int kSPitch = kPanel + 1;

__global__ void __launch_bounds__(kPotrfThreads)
potrf_diag_kernel(double* __restrict__ A, int64_t K, int64_t P, unsigned* status) {
    __shared__ double S[kPanel * kSPitch];
    for (int e = threadIdx.x; e < kPanel * kPanel; e += kPotrfThreads) {
        const int i = e / kPanel, k = e % kPanel;
        S[i * kSPitch + k] = A[(P + i) * K + P + k];
    }
    __syncthreads();
    for (int j = 0; j < kPanel; ++j) {
        if (threadIdx.x == 0) {
            const double p = S[j * kSPitch + j];
            if (!(p > 0.0)) record_status(status, kStatusNumeric);
            S[j * kSPitch + j] = sqrt(p);
        }
        __syncthreads();
        const double d = S[j * kSPitch + j];
        for (int i = j + 1 + threadIdx.x; i < kPanel; i += kPotrfThreads) S[i * kSPitch + j] /= d;
        __syncthreads();
        // (i, k) with j < k <= i < 64, as i = j + 1 + e / n, k = j + 1 + e % n over the
        // square and skipped above the diagonal.
        const int n = kPanel - 1 - j;
        for (int e = threadIdx.x; e < n * n; e += kPotrfThreads) {
            const int i = j + 1 + e / n, k = j + 1 + e % n;
            if (k <= i) S[i * kSPitch + k] = fma(-S[i * kSPitch + j], S[k * kSPitch + j], S[i * kSPitch + k]);
        }
        __syncthreads();
    }
    for (int e = threadIdx.x; e < kPanel * kPanel; e += kPotrfThreads) {
        const int i = e / kPanel, k = e % kPanel;
        if (k <= i) A[(P + i) * K + P + k] = S[i * kSPitch + k];
    }
}

// The rows below a factored diagonal block: for every row r >= P + 64, the
// 64 entries l = A[r, P:P+64] solve l · L_ppᵀ = a (forward substitution
// along the row, L_pp from shared memory).  One thread per row.
constexpr int kRowSolveThreads = 128;

__global__ void __launch_bounds__(kRowSolveThreads)
trsm_rows_kernel(double* __restrict__ A, int64_t K, int64_t P) {
    __shared__ double L[kPanel * kPanel];
    for (int e = threadIdx.x; e < kPanel * kPanel; e += kRowSolveThreads) {
        const int i = e / kPanel, k = e % kPanel;
        L[e] = k <= i ? A[(P + i) * K + P + k] : 0.0;
    }
    __syncthreads();
    const int64_t r = P + kPanel + static_cast<int64_t>(blockIdx.x) * kRowSolveThreads + threadIdx.x;
    if (r >= K) return;
    double* row = A + r * K + P;
    double l[kPanel];
#pragma unroll
    for (int j = 0; j < kPanel; ++j) l[j] = row[j];
#pragma unroll
    for (int j = 0; j < kPanel; ++j) {
        double s = l[j];
#pragma unroll
        for (int m = 0; m < j; ++m) s = fma(-l[m], L[j * kPanel + m], s);
        l[j] = s / L[j * kPanel + j];
    }
#pragma unroll
    for (int j = 0; j < kPanel; ++j) row[j] = l[j];
}

// X = I (the right-hand side of L X = I; every block row's solve reads its
// whole 64-row strip up to the diagonal block's last column, so the part
// above the diagonal inside that block must hold zeros too).
__global__ void identity_kernel(double* __restrict__ X, int64_t K) {
    const int64_t n = K * K;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = i / K, c = i - r * K;
        X[i] = r == c ? 1.0 : 0.0;
    }
}

// Block row I0 of X: X[I0:I0+64, c] = L_ii⁻¹ X[I0:I0+64, c] for every column
// c < I0 + 64 (forward substitution down the column, L_ii from shared
// memory).  One thread per column.
__global__ void __launch_bounds__(kRowSolveThreads)
trsm_cols_kernel(const double* __restrict__ A, double* __restrict__ X, int64_t K, int64_t I0) {
    __shared__ double L[kPanel * kPanel];
    for (int e = threadIdx.x; e < kPanel * kPanel; e += kRowSolveThreads) {
        const int i = e / kPanel, k = e % kPanel;
        L[e] = k <= i ? A[(I0 + i) * K + I0 + k] : 0.0;
    }
    __syncthreads();
    const int64_t c = static_cast<int64_t>(blockIdx.x) * kRowSolveThreads + threadIdx.x;
    if (c >= I0 + kPanel) return;
    double x[kPanel];
#pragma unroll
    for (int k = 0; k < kPanel; ++k) x[k] = X[(I0 + k) * K + c];
#pragma unroll
    for (int m = 0; m < kPanel; ++m) {
        x[m] /= L[m * kPanel + m];
#pragma unroll
        for (int k = m + 1; k < kPanel; ++k) x[k] = fma(-L[k * kPanel + m], x[m], x[k]);
    }
#pragma unroll
    for (int k = 0; k < kPanel; ++k) X[(I0 + k) * K + c] = x[k];
}

// fp64 tile product C[M×N] −= A[M×kin] · op(B), row-major operands with
// leading dimensions; op(B)[k][j] = B[k][j] (kNT false) or B[j][k] (kNT
// true).  With `lower`, tiles entirely above C's diagonal are skipped (the
// symmetric trailing update of the Cholesky keeps only the lower triangle).
// 64×64 tiles, 256 threads of 4×4 outputs, the inner dimension staged in
// chunks of 32 through shared memory.  The inner sum runs in k order from
// C's value (one fma per term), so results do not depend on the launch.
// GB300's fp64 rate (about 1.66 fma per clock per SM) makes this bound by the
// fma pipe at any tiling; the tiles only keep loads off its way.
constexpr int kGT = 64, kGK = 32, kGThreads = 256;

template <bool kNT>
__global__ void __launch_bounds__(kGThreads)
gemm_f64_kernel(double* __restrict__ C, int64_t ldc, const double* __restrict__ Am, int64_t lda,
                const double* __restrict__ Bm, int64_t ldb, int64_t M, int64_t N, int kin, bool lower) {
    __shared__ double As[kGK][kGT];  // As[k][i]
    __shared__ double Bs[kGK][kGT];  // Bs[k][j]
    const int64_t i0 = static_cast<int64_t>(blockIdx.y) * kGT, j0 = static_cast<int64_t>(blockIdx.x) * kGT;
    if (lower && j0 > i0 + kGT - 1) return;
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    double acc[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int64_t i = i0 + ty * 4 + a, j = j0 + tx * 4 + b;
            acc[a][b] = (i < M && j < N) ? C[i * ldc + j] : 0.0;
        }
    for (int k0 = 0; k0 < kin; k0 += kGK) {
        for (int e = threadIdx.x; e < kGT * kGK; e += kGThreads) {
            // A tile: row i, column k (k fastest for coalesced reads).
            const int ii = e / kGK, kk = e % kGK;
            const int64_t i = i0 + ii;
            As[kk][ii] = (i < M && k0 + kk < kin) ? Am[i * lda + k0 + kk] : 0.0;
            if (kNT) {
                const int64_t j = j0 + ii;
                Bs[kk][ii] = (j < N && k0 + kk < kin) ? Bm[j * ldb + k0 + kk] : 0.0;
            }
        }
        if (!kNT) {
            for (int e = threadIdx.x; e < kGT * kGK; e += kGThreads) {
                const int kk = e / kGT, jj = e % kGT;
                const int64_t j = j0 + jj;
                Bs[kk][jj] = (j < N && k0 + kk < kin) ? Bm[(k0 + kk) * ldb + j] : 0.0;
            }
        }
        __syncthreads();
#pragma unroll 4
        for (int kk = 0; kk < kGK; ++kk) {
            double a[4], b[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                a[t] = As[kk][ty * 4 + t];
                b[t] = Bs[kk][tx * 4 + t];
            }
#pragma unroll
            for (int p = 0; p < 4; ++p)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[p][q] = fma(-a[p], b[q], acc[p][q]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int64_t i = i0 + ty * 4 + a, j = j0 + tx * 4 + b;
            if (i < M && j < N) C[i * ldc + j] = acc[a][b];
        }
}

// One 128-column block [i1, i1 + 128) for kSweepRows rows.  Each row has
// kRowThreads threads: thread t of a row owns the block's columns k ≡ t (mod
// kRowThreads).  The block sits in shared memory column-major (W1s[k][r],
// pitch kPitch) so that one k is a contiguous run of rows.  Per column j all
// threads of the row read w_j from shared memory (after a warp barrier, since
// its owner updated it in the previous step), take the same rounding decision
// and error, and each applies the correction to its own later columns.
__global__ void __launch_bounds__(kSweepThreads)
gptq_sweep_kernel(const double* __restrict__ Wd, const double* __restrict__ U, int64_t N, int64_t K, int64_t i1,
                  int group, uint8_t* __restrict__ packed, uint16_t* __restrict__ scales, double* __restrict__ E) {
    extern __shared__ double smem_d[];
    double* W1s = smem_d;                                                     // [kBlock][kPitch]
    int8_t* Qs = reinterpret_cast<int8_t*>(smem_d + kBlock * kPitch);         // [kBlock][kSweepRows]
    const int tid = threadIdx.x;
    const int r = tid / kRowThreads;  // row within the CTA
    const int t = tid % kRowThreads;  // column residue owned by this thread
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kSweepRows;
    const int64_t n = n0 + r;

    for (int idx = tid; idx < kSweepRows * kBlock; idx += kSweepThreads) {
        const int rr = idx / kBlock, k = idx % kBlock;
        const int64_t row = n0 + rr;
        W1s[k * kPitch + rr] = row < N ? Wd[row * K + i1 + k] : 0.0;
    }
    __syncthreads();

    const double* Ub = U + i1 * K + i1;  // U[i1 + j, i1 + k] = Ub[j·K + k]
    const int64_t row_groups = K / group;
    double d = 0.0;
    for (int j = 0; j < kBlock; ++j) {
        __syncwarp();
        if (j % group == 0) {
            // The group's current weights (every later column of the block
            // already carries the corrections of the columns before j): max
            // over this thread's columns of the group, then over the row.
            double a = 0.0;
            for (int k = j + t; k < j + group; k += kRowThreads) a = fmax(a, fabs(W1s[k * kPitch + r]));
#pragma unroll
            for (int m = 1; m < kRowThreads; m <<= 1) a = fmax(a, __shfl_xor_sync(0xffffffffu, a, m));
            const __nv_bfloat16 d16 = __float2bfloat16_rn(__double2float_rn(a / 7.0));
            d = static_cast<double>(__bfloat162float(d16));
            if (n < N && t == 0) scales[n * row_groups + (i1 + j) / group] = *reinterpret_cast<const uint16_t*>(&d16);
        }
        const double wj = W1s[j * kPitch + r];
        const double q = d != 0.0 ? fmin(fmax(rint(wj / d), -8.0), 7.0) : 0.0;
        const double err = (wj - d * q) / __ldg(Ub + static_cast<int64_t>(j) * K + j);
        const double* urow = Ub + static_cast<int64_t>(j) * K;
        // This thread's columns after j: k = j + 1 + ((t − j − 1) mod kRowThreads) + kRowThreads·i.
        const int k0 = j + 1 + ((t - j - 1) & (kRowThreads - 1));
#pragma unroll 4
        for (int k = k0; k < kBlock; k += kRowThreads) W1s[k * kPitch + r] = fma(-err, __ldg(urow + k), W1s[k * kPitch + r]);
        __syncwarp();  // every thread of the row has read w_j before its owner overwrites it
        if (t == (j & (kRowThreads - 1))) {
            Qs[j * kSweepRows + r] = static_cast<int8_t>(q);
            W1s[j * kPitch + r] = err;  // column j is done: keep its error for the block update
        }
    }
    __syncthreads();

    // Errors for the later blocks, row-major [N, kBlock].
    for (int idx = tid; idx < kSweepRows * kBlock; idx += kSweepThreads) {
        const int rr = idx / kBlock, k = idx % kBlock;
        const int64_t row = n0 + rr;
        if (row < N) E[row * kBlock + k] = W1s[k * kPitch + rr];
    }
    // Codes in the stored nibble order: chunk c (k = 32c .. 32c + 31) of the
    // block, word (k mod 32)/8, slot i with offset {0,2,4,6,1,3,5,7}[i] = k mod 8.
    // Threads t < 4 of a row write chunk t as one 16-byte store.
    if (n < N && t < 4) {
        uint32_t words[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int kk = 0; kk < 32; ++kk) {
            const int e = kk % 8;
            const int slot = (e % 2 == 0) ? e / 2 : 4 + e / 2;
            const uint32_t nib = static_cast<uint32_t>(Qs[(32 * t + kk) * kSweepRows + r]) & 0xFu;
            words[kk / 8] |= nib << (4 * slot);
        }
        reinterpret_cast<uint4*>(packed + n * (K / 2) + i1 / 2)[t] = make_uint4(words[0], words[1], words[2], words[3]);
    }
}

std::mutex g_gptq_mutex;
bool g_sweep_attr[64];

int grid_for(int64_t n, const DeviceInfo& dev) {
    int64_t g = (n + 255) / 256;
    const int64_t cap = static_cast<int64_t>(dev.sm_count) * 8;
    if (g > cap) g = cap;
    return static_cast<int>(g < 1 ? 1 : g);
}

// C[M×N] −= A · op(B) (see gemm_f64_kernel); grids are at most 65535 tiles
// high, i.e. M < 4.19M rows.
template <bool kNT>
void gemm_f64(double* C, int64_t ldc, const double* A, int64_t lda, const double* B, int64_t ldb, int64_t M,
              int64_t N, int kin, bool lower, cudaStream_t stream) {
    if (M <= 0 || N <= 0) return;
    const dim3 grid(static_cast<unsigned>((N + kGT - 1) / kGT), static_cast<unsigned>((M + kGT - 1) / kGT));
    gemm_f64_kernel<kNT><<<grid, kGThreads, 0, stream>>>(C, ldc, A, lda, B, ldb, M, N, kin, lower);
}

unsigned blocks_for(int64_t n, int per) { return static_cast<unsigned>((n + per - 1) / per); }

}  // namespace

size_t gptq_factor_workspace_bytes(int64_t K) { return factor_layout(K).total; }

size_t gptq_workspace_bytes(int64_t N, int64_t K) { return quant_layout(N, K).total; }

int launch_gptq_factor(const float* H, int64_t K, double damp, double* U, void* workspace, size_t workspace_bytes,
                       const DeviceInfo& dev, cudaStream_t stream) {
    const FactorLayout l = factor_layout(K);
    if (workspace_bytes < l.total) return 2;
    if (K % kPanel != 0 || (K + kGT - 1) / kGT > 65535) return 1;
    auto* base = static_cast<uint8_t*>(workspace);
    double* lam = reinterpret_cast<double*>(base + l.lam);
    double* A = reinterpret_cast<double*>(base + l.a);
    diag_mean_kernel<<<1, 256, 0, stream>>>(H, K, damp, lam);
    damp_reversed_kernel<<<grid_for(K * K, dev), 256, 0, stream>>>(H, K, lam, A);
    // Cholesky A = L̃ L̃ᵀ, L̃ in A's lower triangle.
    for (int64_t P = 0; P < K; P += kPanel) {
        potrf_diag_kernel<<<1, kPotrfThreads, 0, stream>>>(A, K, P, dev.status);
        const int64_t rest = K - P - kPanel;
        if (rest > 0) {
            trsm_rows_kernel<<<blocks_for(rest, kRowSolveThreads), kRowSolveThreads, 0, stream>>>(A, K, P);
            const int64_t Q = P + kPanel;
            gemm_f64<true>(A + Q * K + Q, K, A + Q * K + P, K, A + Q * K + P, K, rest, rest, kPanel, true, stream);
        }
    }
    // X = L̃⁻¹ in U's memory: L̃ X = I solved block row by block row.
    identity_kernel<<<grid_for(K * K, dev), 256, 0, stream>>>(U, K);
    for (int64_t I0 = 0; I0 < K; I0 += kPanel) {
        trsm_cols_kernel<<<blocks_for(I0 + kPanel, kRowSolveThreads), kRowSolveThreads, 0, stream>>>(A, U, K, I0);
        const int64_t rest = K - I0 - kPanel;
        if (rest > 0)
            gemm_f64<false>(U + (I0 + kPanel) * K, K, A + (I0 + kPanel) * K + I0, K, U + I0 * K, K, rest,
                            I0 + kPanel, kPanel, false, stream);
    }
    // Row-major U[r][c] = X[K−1−r][K−1−c].
    reverse_kernel<<<grid_for(K * K / 2, dev), 256, 0, stream>>>(U, K);
    return cudaGetLastError() == cudaSuccess ? 0 : 1;
}

int launch_gptq(const void* W, int64_t N, int64_t K, int group, const double* U, void* packed, void* scales,
                void* workspace, size_t workspace_bytes, const DeviceInfo& dev, cudaStream_t stream) {
    const QuantLayout l = quant_layout(N, K);
    if (workspace_bytes < l.total) return 2;
    if ((N + kGT - 1) / kGT > 65535) return 1;
    {
        int device = 0;
        if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= 64) return 1;
        std::lock_guard<std::mutex> lock(g_gptq_mutex);
        if (!g_sweep_attr[device]) {
            if (cudaFuncSetAttribute(gptq_sweep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSweepSmem) !=
                cudaSuccess)
                return 1;
            g_sweep_attr[device] = true;
        }
    }
    auto* base = static_cast<uint8_t*>(workspace);
    double* Wd = reinterpret_cast<double*>(base + l.wd);
    double* E = reinterpret_cast<double*>(base + l.e);
    widen_kernel<<<grid_for(N * K, dev), 256, 0, stream>>>(static_cast<const uint16_t*>(W), N * K, Wd);
    const unsigned sweep_grid = static_cast<unsigned>((N + kSweepRows - 1) / kSweepRows);
    for (int64_t i1 = 0; i1 < K; i1 += kBlock) {
        const int64_t i2 = i1 + kBlock;
        gptq_sweep_kernel<<<sweep_grid, kSweepThreads, kSweepSmem, stream>>>(
            Wd, U, N, K, i1, group, static_cast<uint8_t*>(packed), static_cast<uint16_t*>(scales), E);
        if (cudaGetLastError() != cudaSuccess) return 1;
        // W[:, i2:] −= E · U[i1:i2, i2:].
        if (i2 < K) gemm_f64<false>(Wd + i2, K, E, kBlock, U + i1 * K + i2, K, N, K - i2, kBlock, false, stream);
    }
    return cudaGetLastError() == cudaSuccess ? 0 : 1;
}

}  // namespace w4
