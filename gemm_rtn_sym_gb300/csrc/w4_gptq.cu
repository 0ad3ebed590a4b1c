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
// factoring the inverse.
//  1. λ, and J H' J = J (fp64(H) + λI) J written reversed (own kernels);
//  2. potrf and trtri by cuSOLVER (plain library linear algebra);
//  3. the reversal and transposition back to row-major U in place (own kernel).
// Quantise (per matrix):
//  3. W widened to fp64 (own kernel);
//  4. per 128-column block: the sweep kernel (own) rounds the block's columns
//     one after another, eight threads carrying each row through the block in
//     shared memory, writes the block's codes, scales and errors E; then the
//     later columns get W[:, i2:] −= E·U[i1:i2, i2:] by cuBLAS DGEMM, which
//     carries N·K² flops in total and bounds the call on GB300's fp64 rate.
// A failed factorization (H' not positive definite) is reported through the
// library's status word as W4_ERR_NUMERIC.
#include <mutex>

#include <cublas_v2.h>
#include <cusolverDn.h>

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

// Factor workspace: λ, cuSOLVER's info word and device work space.
struct FactorLayout {
    size_t lam, info, work, total;
};

FactorLayout factor_layout(size_t work_bytes) {
    FactorLayout l;
    l.lam = 0;
    l.info = 256;
    l.work = 512;
    l.total = align256(l.work + work_bytes);
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

// The column-major lower triangle of A holds L̃⁻¹ (L̃⁻¹[i][j] at i + j·K).
// Row-major U[r][c] = L̃⁻¹[K−1−r][K−1−c] sits at K² − 1 − (r + c·K): the map
// p = r·K + c -> q = K² − 1 − (r + c·K) is an involution, so swapping each pair
// once turns A into U in place.
__global__ void reverse_transpose_kernel(double* __restrict__ A, int64_t K) {
    const int64_t n = K * K;
    for (int64_t p = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; p < n;
         p += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = p / K, c = p - r * K;
        const int64_t q = n - 1 - (r + c * K);
        if (p < q) {
            const double t = A[p];
            A[p] = A[q];
            A[q] = t;
        }
    }
}

__global__ void widen_kernel(const uint16_t* __restrict__ W, int64_t n, double* __restrict__ Wd) {
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        Wd[i] = static_cast<double>(__uint_as_float(static_cast<uint32_t>(W[i]) << 16));
}

__global__ void check_info_kernel(const int* __restrict__ info, unsigned* status) {
    if (*info != 0) record_status(status, kStatusNumeric);
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

struct Handles {
    cusolverDnHandle_t solver = nullptr;
    cublasHandle_t blas = nullptr;
    bool sweep_attr = false;
};
std::mutex g_la_mutex;
Handles g_la[64];

// Handles of the current device (created once); nullptr on failure.  The
// caller holds g_la_mutex.
Handles* handles() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    Handles& h = g_la[dev];
    if (!h.solver && cusolverDnCreate(&h.solver) != CUSOLVER_STATUS_SUCCESS) {
        h.solver = nullptr;
        return nullptr;
    }
    if (!h.blas && cublasCreate(&h.blas) != CUBLAS_STATUS_SUCCESS) {
        h.blas = nullptr;
        return nullptr;
    }
    if (!h.sweep_attr) {
        if (cudaFuncSetAttribute(gptq_sweep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSweepSmem) !=
            cudaSuccess)
            return nullptr;
        h.sweep_attr = true;
    }
    return &h;
}

// Device bytes of cuSOLVER work space for potrf and trtri at order K (trtri
// must need no host work space, which this library does not keep).
bool solver_work_bytes(Handles* h, int64_t K, size_t* bytes) {
    int a = 0;
    size_t dev_b = 0, host_b = 0;
    const int n = static_cast<int>(K);
    if (cusolverDnDpotrf_bufferSize(h->solver, CUBLAS_FILL_MODE_LOWER, n, nullptr, n, &a) != CUSOLVER_STATUS_SUCCESS ||
        cusolverDnXtrtri_bufferSize(h->solver, CUBLAS_FILL_MODE_LOWER, CUBLAS_DIAG_NON_UNIT, K, CUDA_R_64F, nullptr,
                                    K, &dev_b, &host_b) != CUSOLVER_STATUS_SUCCESS ||
        host_b != 0)
        return false;
    const size_t pa = static_cast<size_t>(a) * 8;
    *bytes = pa > dev_b ? pa : dev_b;
    return true;
}

int grid_for(int64_t n, const DeviceInfo& dev) {
    int64_t g = (n + 255) / 256;
    const int64_t cap = static_cast<int64_t>(dev.sm_count) * 8;
    if (g > cap) g = cap;
    return static_cast<int>(g < 1 ? 1 : g);
}

}  // namespace

size_t gptq_factor_workspace_bytes(int64_t K) {
    std::lock_guard<std::mutex> lock(g_la_mutex);
    Handles* h = handles();
    size_t work = 0;
    if (!h || !solver_work_bytes(h, K, &work)) return 0;
    return factor_layout(work).total;
}

size_t gptq_workspace_bytes(int64_t N, int64_t K) { return quant_layout(N, K).total; }

int launch_gptq_factor(const float* H, int64_t K, double damp, double* A, void* workspace, size_t workspace_bytes,
                       const DeviceInfo& dev, cudaStream_t stream) {
    std::lock_guard<std::mutex> lock(g_la_mutex);
    Handles* h = handles();
    size_t work_bytes = 0;
    if (!h || !solver_work_bytes(h, K, &work_bytes)) return 1;
    const FactorLayout l = factor_layout(work_bytes);
    if (workspace_bytes < l.total) return 2;
    auto* base = static_cast<uint8_t*>(workspace);
    double* lam = reinterpret_cast<double*>(base + l.lam);
    int* info = reinterpret_cast<int*>(base + l.info);
    double* work = reinterpret_cast<double*>(base + l.work);
    const int n = static_cast<int>(K);
    const int lwork = static_cast<int>(work_bytes / 8);
    if (cusolverDnSetStream(h->solver, stream) != CUSOLVER_STATUS_SUCCESS) return 1;
    diag_mean_kernel<<<1, 256, 0, stream>>>(H, K, damp, lam);
    damp_reversed_kernel<<<grid_for(K * K, dev), 256, 0, stream>>>(H, K, lam, A);
    // Column-major LOWER (the matrix is symmetric): L̃ with J H' J = L̃ L̃ᵀ
    // fills the lower triangle, then its inverse replaces it.
    if (cusolverDnDpotrf(h->solver, CUBLAS_FILL_MODE_LOWER, n, A, n, work, lwork, info) != CUSOLVER_STATUS_SUCCESS)
        return 1;
    check_info_kernel<<<1, 1, 0, stream>>>(info, dev.status);
    if (cusolverDnXtrtri(h->solver, CUBLAS_FILL_MODE_LOWER, CUBLAS_DIAG_NON_UNIT, K, CUDA_R_64F, A, K, work,
                         work_bytes, nullptr, 0, info) != CUSOLVER_STATUS_SUCCESS)
        return 1;
    check_info_kernel<<<1, 1, 0, stream>>>(info, dev.status);
    reverse_transpose_kernel<<<grid_for(K * K, dev), 256, 0, stream>>>(A, K);
    return cudaGetLastError() == cudaSuccess ? 0 : 1;
}

int launch_gptq(const void* W, int64_t N, int64_t K, int group, const double* U, void* packed, void* scales,
                void* workspace, size_t workspace_bytes, const DeviceInfo& dev, cudaStream_t stream) {
    std::lock_guard<std::mutex> lock(g_la_mutex);
    Handles* h = handles();
    if (!h) return 1;
    const QuantLayout l = quant_layout(N, K);
    if (workspace_bytes < l.total) return 2;
    auto* base = static_cast<uint8_t*>(workspace);
    double* Wd = reinterpret_cast<double*>(base + l.wd);
    double* E = reinterpret_cast<double*>(base + l.e);
    const int n = static_cast<int>(K);
    if (cublasSetStream(h->blas, stream) != CUBLAS_STATUS_SUCCESS) return 1;
    widen_kernel<<<grid_for(N * K, dev), 256, 0, stream>>>(static_cast<const uint16_t*>(W), N * K, Wd);
    const double minus_one = -1.0, one = 1.0;
    const unsigned sweep_grid = static_cast<unsigned>((N + kSweepRows - 1) / kSweepRows);
    for (int64_t i1 = 0; i1 < K; i1 += kBlock) {
        const int64_t i2 = i1 + kBlock;
        gptq_sweep_kernel<<<sweep_grid, kSweepThreads, kSweepSmem, stream>>>(
            Wd, U, N, K, i1, group, static_cast<uint8_t*>(packed), static_cast<uint16_t*>(scales), E);
        if (cudaGetLastError() != cudaSuccess) return 1;
        if (i2 < K) {
            // Row-major W[:, i2:] −= E · U[i1:i2, i2:], as the column-major
            // product Wᵀ −= Uᵀ Eᵀ.
            if (cublasDgemm(h->blas, CUBLAS_OP_N, CUBLAS_OP_N, static_cast<int>(K - i2), static_cast<int>(N), kBlock,
                            &minus_one, U + i1 * K + i2, n, E, kBlock, &one, Wd + i2, n) != CUBLAS_STATUS_SUCCESS)
                return 1;
        }
    }
    return cudaGetLastError() == cudaSuccess ? 0 : 1;
}

}  // namespace w4
