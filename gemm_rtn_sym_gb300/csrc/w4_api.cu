// C ABI of the library (declared in include/w4.h): argument checks, kernel
// choice, launches and the per-device status word of the bounded waits.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include <cuda_runtime.h>

#include "w4.h"
#include "w4_device.cuh"
#include "w4_internal.h"

namespace w4 {
namespace {

// One status word per device (written by kernels whose bounded waits ran out).
__device__ unsigned g_status_word = 0;

constexpr int kMaxDevices = 64;
DeviceInfo g_info[kMaxDevices];
bool g_info_ready[kMaxDevices];
std::mutex g_info_mutex;

// Smallest M that goes to the tensor-core kernel: under W4_PATH_AUTO for one
// matrix, and in grouped plans.  Measured crossovers on the 4B-class stack,
// the 27B-class layer and the 2560×9216 matrix (M = 17, 20, 24, 28, 32): the
// small-M kernel is faster up to M = 24 (three token tiles per pass; e.g.
// grouped stack 621 against 665 µs at M = 24), the tensor-core tile from
// M = 28 (grouped stack 665 against 815 µs; 2560×9216 alone 10.5 against
// 11.5 µs), in one launch per matrix and in grouped launches alike.
constexpr int64_t kTensorMinM = 25;
constexpr int64_t kGroupedTensorMinM = 25;

// Largest N or K of the GPTQ calls: their fp64 tile products run 64-row tiles
// on a grid at most 65535 tiles high.
constexpr int64_t kGptqMaxDim = int64_t{65535} * 64;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
    return na != 0 && nb != 0 && pa < pb + nb && pb < pa + na;
}

int check_sizes(int64_t N, int64_t K) {
    if (N < 0 || K < 0) return W4_ERR_INVALID_ARG;
    if (K % 128 != 0) return W4_ERR_UNSUPPORTED;
    if (N > 0 && K > (int64_t{1} << 62) / N) return W4_ERR_INVALID_ARG;
    return W4_OK;
}

int to_status(cudaError_t e) { return e == cudaSuccess ? W4_OK : W4_ERR_CUDA; }

bool valid_group(int32_t group) { return group == 32 || group == 64 || group == 128; }

}  // namespace

const DeviceInfo* device_info(cudaError_t* err) {
    int dev = 0;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess) return nullptr;
    if (dev < 0 || dev >= kMaxDevices) {
        *err = cudaErrorInvalidDevice;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_info_mutex);
    if (!g_info_ready[dev]) {
        DeviceInfo info;
        if ((*err = cudaDeviceGetAttribute(&info.sm_count, cudaDevAttrMultiProcessorCount, dev)) ||
            (*err = cudaDeviceGetAttribute(&info.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) ||
            (*err = cudaDeviceGetAttribute(&info.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) ||
            (*err = cudaDeviceGetAttribute(&info.max_smem_optin,
                                           cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) ||
            (*err = cudaGetSymbolAddress(reinterpret_cast<void**>(&info.status), g_status_word)))
            return nullptr;
        g_info[dev] = info;
        g_info_ready[dev] = true;
    }
    *err = cudaSuccess;
    return &g_info[dev];
}

}  // namespace w4

using namespace w4;

extern "C" {

size_t w4_packed_bytes(int64_t N, int64_t K) {
    if (check_sizes(N, K) != W4_OK) return 0;
    return static_cast<size_t>(N) * static_cast<size_t>(K) / 2;
}

size_t w4_scales_bytes(int64_t N, int64_t K, int32_t group) {
    if (!valid_group(group) || check_sizes(N, K) != W4_OK) return 0;
    return static_cast<size_t>(N) * static_cast<size_t>(K / group) * 2;
}

size_t w4_zeros_bytes(int64_t N, int64_t K, int32_t group) {
    if (!valid_group(group) || check_sizes(N, K) != W4_OK) return 0;
    return static_cast<size_t>(N) * static_cast<size_t>(K / group);
}

}  // extern "C"

namespace {

// Symmetric RTN (asym false), asymmetric RTN (zeros written), or symmetric
// RTN of the channel-scaled weights (scaled, group 128 only).
int quantize_impl(const void* W, int64_t N, int64_t K, int32_t group, const float* channel_scales,
                  bool scaled, bool asym, void* packed, void* scales, void* zeros, void* stream) {
    if (!valid_group(group) || (scaled && group != 128)) return W4_ERR_UNSUPPORTED;
    if (const int s = check_sizes(N, K)) return s;
    if (N == 0 || K == 0) return W4_OK;
    if (!W || !packed || !scales || (scaled && !channel_scales) || (asym && !zeros)) return W4_ERR_INVALID_ARG;
    if (!aligned(W, 16) || !aligned(packed, 16) || !aligned(scales, 2) ||
        (scaled && !aligned(channel_scales, 16)))
        return W4_ERR_MISALIGNED;
    const size_t wb = static_cast<size_t>(N * K) * 2, pb = w4_packed_bytes(N, K),
                 sb = w4_scales_bytes(N, K, group), cb = scaled ? static_cast<size_t>(K) * 4 : 0,
                 zb = asym ? w4_zeros_bytes(N, K, group) : 0;
    if (overlaps(W, wb, packed, pb) || overlaps(W, wb, scales, sb) || overlaps(packed, pb, scales, sb) ||
        overlaps(channel_scales, cb, packed, pb) || overlaps(channel_scales, cb, scales, sb) ||
        overlaps(zeros, zb, W, wb) || overlaps(zeros, zb, packed, pb) || overlaps(zeros, zb, scales, sb))
        return W4_ERR_INVALID_ARG;
    cudaError_t err;
    const DeviceInfo* dev = device_info(&err);
    if (!dev) return W4_ERR_CUDA;
    if (dev->cc_major < 10) return W4_ERR_UNSUPPORTED;
    return to_status(launch_quantize(W, N, K, group, packed, scales, asym ? zeros : nullptr,
                                     scaled ? channel_scales : nullptr, *dev, static_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

int w4_quantize_rtn(const void* W, int64_t N, int64_t K, int32_t group, void* packed, void* scales,
                    void* stream) {
    return quantize_impl(W, N, K, group, nullptr, false, false, packed, scales, nullptr, stream);
}

int w4_quantize_rtn_asym(const void* W, int64_t N, int64_t K, int32_t group, void* packed, void* scales,
                         void* zeros, void* stream) {
    return quantize_impl(W, N, K, group, nullptr, false, true, packed, scales, zeros, stream);
}

int w4_quantize_rtn_scaled(const void* W, int64_t N, int64_t K, int32_t group, const float* s, void* packed,
                           void* scales, void* stream) {
    return quantize_impl(W, N, K, group, s, true, false, packed, scales, nullptr, stream);
}

size_t w4_gptq_factor_workspace_bytes(int64_t K) {
    if (check_sizes(1, K) != W4_OK || K == 0 || K > kGptqMaxDim) return 0;
    return gptq_factor_workspace_bytes(K);
}

int w4_gptq_factor(const float* H, int64_t K, double damp, double* U, void* workspace, size_t workspace_bytes,
                   void* stream) {
    if (const int s = check_sizes(1, K)) return s;
    if (K == 0) return W4_OK;
    if (K > kGptqMaxDim || static_cast<double>(K) * K > 1e18) return W4_ERR_UNSUPPORTED;
    if (!(damp >= 0.0) || damp > 1e30) return W4_ERR_INVALID_ARG;
    if (!H || !U || !workspace) return W4_ERR_INVALID_ARG;
    if (!aligned(H, 4) || !aligned(U, 8) || !aligned(workspace, 256)) return W4_ERR_MISALIGNED;
    const size_t hb = static_cast<size_t>(K) * K * 4, ub = static_cast<size_t>(K) * K * 8;
    if (overlaps(H, hb, U, ub) || overlaps(workspace, workspace_bytes, H, hb) ||
        overlaps(workspace, workspace_bytes, U, ub))
        return W4_ERR_INVALID_ARG;
    cudaError_t err;
    const DeviceInfo* dev = device_info(&err);
    if (!dev) return W4_ERR_CUDA;
    if (dev->cc_major < 10) return W4_ERR_UNSUPPORTED;
    switch (launch_gptq_factor(H, K, damp, U, workspace, workspace_bytes, *dev, static_cast<cudaStream_t>(stream))) {
        case 0: return W4_OK;
        case 2: return W4_ERR_INVALID_ARG;
        default: return W4_ERR_CUDA;
    }
}

size_t w4_gptq_workspace_bytes(int64_t N, int64_t K) {
    if (check_sizes(N, K) != W4_OK || N == 0 || K == 0 || N > INT32_MAX || K > INT32_MAX) return 0;
    if (static_cast<double>(N) * K > 1e18) return 0;
    return gptq_workspace_bytes(N, K);
}

int w4_gptq_quantize(const void* W, int64_t N, int64_t K, int32_t group, const double* U, void* packed,
                     void* scales, void* workspace, size_t workspace_bytes, void* stream) {
    if (!valid_group(group)) return W4_ERR_UNSUPPORTED;
    if (const int s = check_sizes(N, K)) return s;
    if (N == 0 || K == 0) return W4_OK;
    if (N > kGptqMaxDim || K > kGptqMaxDim) return W4_ERR_UNSUPPORTED;
    if (!W || !U || !packed || !scales || !workspace) return W4_ERR_INVALID_ARG;
    if (!aligned(W, 16) || !aligned(U, 8) || !aligned(packed, 16) || !aligned(scales, 2) || !aligned(workspace, 256))
        return W4_ERR_MISALIGNED;
    const size_t wb = static_cast<size_t>(N * K) * 2, ub = static_cast<size_t>(K) * K * 8,
                 pb = w4_packed_bytes(N, K), sb = w4_scales_bytes(N, K, group);
    const void* outs[2] = {packed, scales};
    const size_t ob[2] = {pb, sb};
    for (int i = 0; i < 2; ++i)
        if (overlaps(outs[i], ob[i], W, wb) || overlaps(outs[i], ob[i], U, ub) ||
            overlaps(outs[i], ob[i], workspace, workspace_bytes))
            return W4_ERR_INVALID_ARG;
    if (overlaps(packed, pb, scales, sb) || overlaps(workspace, workspace_bytes, W, wb) ||
        overlaps(workspace, workspace_bytes, U, ub))
        return W4_ERR_INVALID_ARG;
    cudaError_t err;
    const DeviceInfo* dev = device_info(&err);
    if (!dev) return W4_ERR_CUDA;
    if (dev->cc_major < 10) return W4_ERR_UNSUPPORTED;
    switch (launch_gptq(W, N, K, group, U, packed, scales, workspace, workspace_bytes, *dev,
                        static_cast<cudaStream_t>(stream))) {
        case 0: return W4_OK;
        case 2: return W4_ERR_INVALID_ARG;
        default: return W4_ERR_CUDA;
    }
}

int w4_scale_activations(const void* x, int64_t M, int64_t K, const float* s, void* x_out, void* stream) {
    if (M < 0) return W4_ERR_INVALID_ARG;
    if (const int st = check_sizes(M, K)) return st;
    if (M == 0 || K == 0) return W4_OK;
    if (!x || !s || !x_out) return W4_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(s, 16) || !aligned(x_out, 16)) return W4_ERR_MISALIGNED;
    const size_t xb = static_cast<size_t>(M * K) * 2, cb = static_cast<size_t>(K) * 4;
    if ((x != x_out && overlaps(x, xb, x_out, xb)) || overlaps(s, cb, x_out, xb)) return W4_ERR_INVALID_ARG;
    cudaError_t err;
    const DeviceInfo* dev = device_info(&err);
    if (!dev) return W4_ERR_CUDA;
    if (dev->cc_major < 10) return W4_ERR_UNSUPPORTED;
    return to_status(launch_scale_activations(x, M, K, s, x_out, *dev, static_cast<cudaStream_t>(stream)));
}

int w4_gemm_path_for(int64_t M, int64_t N, int64_t K) {
    if (M < 0) return -W4_ERR_INVALID_ARG;
    if (const int s = check_sizes(N, K)) return -s;
    return M >= kTensorMinM ? W4_PATH_TENSOR : W4_PATH_SMALL_M;
}

namespace {

// affine: the w4_gemm_affine formats (group 32/64/128, zeros or nullptr);
// otherwise the symmetric group-128 format.
int gemm_impl(const void* x, int64_t M, int64_t N, int64_t K, int32_t group, const void* packed,
              const void* scales, const void* zeros, void* y, void* stream, int32_t path, bool affine) {
    if (affine && !valid_group(group)) return W4_ERR_UNSUPPORTED;
    if (M < 0) return W4_ERR_INVALID_ARG;
    if (const int s = check_sizes(N, K)) return s;
    if (M > 0 && K > (int64_t{1} << 62) / M) return W4_ERR_INVALID_ARG;
    if (M > 0 && N > (int64_t{1} << 62) / M) return W4_ERR_INVALID_ARG;
    if (path < W4_PATH_AUTO || path > W4_PATH_TENSOR) return W4_ERR_INVALID_ARG;
    // Tensor-map coordinates are 32-bit.
    if (N > INT32_MAX || K > INT32_MAX || M > INT32_MAX) return W4_ERR_UNSUPPORTED;
    if (M == 0 || N == 0) return W4_OK;
    if (!y) return W4_ERR_INVALID_ARG;
    if (!aligned(y, 2)) return W4_ERR_MISALIGNED;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t yb = static_cast<size_t>(M * N) * 2;
    if (K == 0) return to_status(cudaMemsetAsync(y, 0, yb, st));
    if (!x || !packed || !scales) return W4_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(packed, 16) || !aligned(scales, 2)) return W4_ERR_MISALIGNED;
    const size_t xb = static_cast<size_t>(M * K) * 2, pb = w4_packed_bytes(N, K),
                 sb = w4_scales_bytes(N, K, affine ? group : 128),
                 zb = affine && zeros ? w4_zeros_bytes(N, K, group) : 0;
    if (overlaps(y, yb, x, xb) || overlaps(y, yb, packed, pb) || overlaps(y, yb, scales, sb) ||
        overlaps(y, yb, zeros, zb))
        return W4_ERR_INVALID_ARG;
    cudaError_t err;
    const DeviceInfo* dev = device_info(&err);
    if (!dev) return W4_ERR_CUDA;
    if (dev->cc_major < 10) return W4_ERR_UNSUPPORTED;
    if (path == W4_PATH_AUTO) path = M >= kTensorMinM ? W4_PATH_TENSOR : W4_PATH_SMALL_M;
    // The symmetric group-128 format has its own kernels (offset MMA chain in
    // the small-M path); w4_gemm_affine with group 128 and no zeros uses them.
    if (affine && (group != 128 || zeros)) {
        if (path == W4_PATH_TENSOR)
            return to_status(launch_gemm_tc_affine(x, M, N, K, group, packed, scales, zeros, y, *dev, st));
        return to_status(launch_gemv_affine(x, M, N, K, group, packed, scales, zeros, y, *dev, st));
    }
    if (path == W4_PATH_TENSOR)
        return to_status(launch_gemm_tc(x, M, N, K, packed, scales, y, *dev, st));
    return to_status(launch_gemv(x, M, N, K, packed, scales, y, *dev, st));
}

}  // namespace

int w4_gemm_ex(const void* x, int64_t M, int64_t N, int64_t K, const void* packed, const void* scales,
               void* y, void* stream, int32_t path) {
    return gemm_impl(x, M, N, K, 128, packed, scales, nullptr, y, stream, path, false);
}

int w4_gemm(const void* x, int64_t M, int64_t N, int64_t K, const void* packed, const void* scales,
            void* y, void* stream) {
    return gemm_impl(x, M, N, K, 128, packed, scales, nullptr, y, stream, W4_PATH_AUTO, false);
}

int w4_gemm_affine(const void* x, int64_t M, int64_t N, int64_t K, int32_t group, const void* packed,
                   const void* scales, const void* zeros, void* y, void* stream, int32_t path) {
    return gemm_impl(x, M, N, K, group, packed, scales, zeros, y, stream, path, true);
}

namespace {

// Checks one grouped problem like w4_gemm does.
int check_grouped_problem(const w4_gemm_problem& p) {
    if (p.M < 1 || p.N < 1 || p.K < 128) return W4_ERR_INVALID_ARG;
    if (const int s = check_sizes(p.N, p.K)) return s;
    if (p.N > INT32_MAX || p.K > INT32_MAX || p.M > INT32_MAX || p.K > (int64_t{1} << 62) / p.M ||
        p.N > (int64_t{1} << 62) / p.M)
        return W4_ERR_UNSUPPORTED;
    if (!p.x || !p.packed || !p.scales || !p.y) return W4_ERR_INVALID_ARG;
    if (!aligned(p.x, 16) || !aligned(p.packed, 16) || !aligned(p.scales, 2) || !aligned(p.y, 2))
        return W4_ERR_MISALIGNED;
    return W4_OK;
}

size_t out_bytes(const w4_gemm_problem& p) { return static_cast<size_t>(p.M * p.N) * 2; }

bool is_tensor(const w4_gemm_problem& p) { return p.M >= kGroupedTensorMinM; }

size_t round128(size_t v) { return (v + 127) / 128 * 128; }

}  // namespace

namespace {

size_t grouped_plan_bytes_impl(int32_t count, const w4_gemm_problem* problems) {
    if (count < 1 || !problems) return 0;
    int64_t small_items = 0, tc_items = 0;
    int32_t n_small = 0, n_tc = 0;
    for (int32_t i = 0; i < count; ++i) {
        const w4_gemm_problem& p = problems[i];
        if (check_grouped_problem(p) != W4_OK) return 0;
        if (is_tensor(p)) {
            ++n_tc;
            tc_items += tc_grouped_items(GroupedSpec{p.x, p.M, p.N, p.K, p.packed, p.scales, p.y, nullptr});
        } else {
            ++n_small;
            small_items += (p.N + 63) / 64;
        }
    }
    if (small_items > INT32_MAX || tc_items > INT32_MAX) return 0;
    // Sized for the largest grids a plan can use (one CTA per item), so that
    // the answer does not depend on the device.
    size_t bytes = 0;
    if (n_small) bytes += round128(grouped_plan_bytes(n_small, small_items, static_cast<int32_t>(small_items)));
    if (n_tc) bytes += tc_grouped_plan_bytes(n_tc, tc_items, static_cast<int32_t>(tc_items));
    return bytes;
}

// Validates the problems (against each other and, when device_memory is not
// NULL, against the plan memory), builds the plan image and fills every field
// of *plan except device_plan.  group: the codes' group size (32, 64, 128);
// zeros: NULL, or count pointers (each NULL or int8 [N, K/group]).  Group 128
// without zeros is the symmetric format's own path (format 0).
int grouped_prepare(const void* device_memory, size_t bytes, int32_t count, const w4_gemm_problem* problems,
                    int32_t group, const void* const* zeros, std::vector<uint8_t>* image, w4_grouped_plan* plan) {
    if (!valid_group(group)) return W4_ERR_UNSUPPORTED;
    bool any_zeros = false;
    for (int32_t i = 0; zeros && i < count; ++i) any_zeros = any_zeros || zeros[i] != nullptr;
    const int format = group == 128 && !any_zeros ? 0 : group;
    int64_t max_m = 1;
    std::vector<GroupedSpec> small, tc;
    for (int32_t i = 0; i < count; ++i) {
        const w4_gemm_problem& p = problems[i];
        if (const int s = check_grouped_problem(p)) return s;
        if (p.K % group != 0) return W4_ERR_UNSUPPORTED;
        const size_t yb = out_bytes(p);
        for (int32_t j = 0; j < count; ++j) {
            const w4_gemm_problem& q = problems[j];
            const void* qz = zeros ? zeros[j] : nullptr;
            const size_t xb = static_cast<size_t>(q.M * q.K) * 2, pb = w4_packed_bytes(q.N, q.K),
                         sb = w4_scales_bytes(q.N, q.K, group), zb = qz ? w4_zeros_bytes(q.N, q.K, group) : 0;
            if (overlaps(p.y, yb, q.x, xb) || overlaps(p.y, yb, q.packed, pb) || overlaps(p.y, yb, q.scales, sb) ||
                overlaps(p.y, yb, qz, zb))
                return W4_ERR_INVALID_ARG;
            if (j != i && overlaps(p.y, yb, q.y, out_bytes(q))) return W4_ERR_INVALID_ARG;
            if (device_memory &&
                (overlaps(device_memory, bytes, q.x, xb) || overlaps(device_memory, bytes, q.packed, pb) ||
                 overlaps(device_memory, bytes, q.scales, sb) || overlaps(device_memory, bytes, q.y, out_bytes(q)) ||
                 overlaps(device_memory, bytes, qz, zb)))
                return W4_ERR_INVALID_ARG;
        }
        const GroupedSpec sp{p.x, p.M, p.N, p.K, p.packed, p.scales, p.y, zeros ? zeros[i] : nullptr};
        if (is_tensor(p)) {
            tc.push_back(sp);
        } else {
            small.push_back(sp);
            max_m = std::max(max_m, p.M);
        }
    }
    const int token_rows = grouped_token_rows(max_m);
    cudaError_t err;
    const DeviceInfo* dev = device_info(&err);
    if (!dev) return W4_ERR_CUDA;
    if (dev->cc_major < 10) return W4_ERR_UNSUPPORTED;
    std::vector<uint8_t> tc_image;
    int64_t n_items = 0, n_tc_items = 0;
    int32_t n_ctas = 0, n_tc_ctas = 0;
    image->clear();
    if (!small.empty()) {
        const int ctas = grouped_ctas(token_rows, format, *dev);
        if (ctas < 1) return W4_ERR_CUDA;
        if (grouped_plan_build(small.data(), static_cast<int32_t>(small.size()), token_rows, format, ctas,
                               dev->sm_count, image, &n_items, &n_ctas) != cudaSuccess)
            return W4_ERR_CUDA;
        image->resize(round128(image->size()), 0);
    }
    const size_t tc_offset = image->size();
    if (!tc.empty()) {
        if (tc_grouped_plan_build(tc.data(), static_cast<int32_t>(tc.size()), format, dev->sm_count, &tc_image,
                                  &n_tc_items, &n_tc_ctas) != cudaSuccess)
            return W4_ERR_CUDA;
        image->insert(image->end(), tc_image.begin(), tc_image.end());
    }
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) return W4_ERR_CUDA;
    int max_bm = 0;
    if (!tc.empty()) std::memcpy(&max_bm, tc_image.data() + 12, sizeof(int));  // TcHeader::max_bm
    plan->device_plan = nullptr;
    plan->bytes = image->size();
    plan->count = count;
    plan->device = device;
    plan->items = static_cast<int32_t>(n_items);
    plan->ctas = n_ctas;
    plan->token_rows = small.empty() ? 0 : token_rows;
    plan->tc_items = static_cast<int32_t>(n_tc_items);
    plan->tc_ctas = n_tc_ctas;
    plan->tc_max_bm = max_bm;
    plan->tc_offset = tc_offset;
    plan->format = format;
    return W4_OK;
}

int grouped_plan_init_impl(w4_grouped_plan* plan, void* device_memory, size_t bytes, int32_t count,
                           const w4_gemm_problem* problems, int32_t group, const void* const* zeros) {
    if (!plan || !device_memory || count < 1 || !problems) return W4_ERR_INVALID_ARG;
    if (!aligned(device_memory, 128)) return W4_ERR_MISALIGNED;
    std::vector<uint8_t> image;
    w4_grouped_plan p;
    if (const int s = grouped_prepare(device_memory, bytes, count, problems, group, zeros, &image, &p)) return s;
    if (bytes < image.size()) return W4_ERR_INVALID_ARG;
    if (cudaMemcpy(device_memory, image.data(), image.size(), cudaMemcpyHostToDevice) != cudaSuccess)
        return W4_ERR_CUDA;
    p.device_plan = device_memory;
    *plan = p;
    return W4_OK;
}

}  // namespace

size_t w4_grouped_plan_bytes(int32_t count, const w4_gemm_problem* problems) {
    return grouped_plan_bytes_impl(count, problems);
}

size_t w4_grouped_plan_bytes_affine(int32_t count, const w4_gemm_problem* problems, int32_t group,
                                    const void* const* zeros) {
    (void)zeros;  // the plan's size does not depend on the format
    if (!valid_group(group)) return 0;
    for (int32_t i = 0; problems && i < count; ++i)
        if (problems[i].K % group != 0) return 0;
    return grouped_plan_bytes_impl(count, problems);
}

int w4_grouped_plan_init(w4_grouped_plan* plan, void* device_memory, size_t bytes, int32_t count,
                         const w4_gemm_problem* problems) {
    return grouped_plan_init_impl(plan, device_memory, bytes, count, problems, 128, nullptr);
}

int w4_grouped_plan_init_affine(w4_grouped_plan* plan, void* device_memory, size_t bytes, int32_t count,
                                const w4_gemm_problem* problems, int32_t group, const void* const* zeros) {
    return grouped_plan_init_impl(plan, device_memory, bytes, count, problems, group, zeros);
}

int w4_gemm_grouped(const w4_grouped_plan* plan, void* stream) {
    if (!plan || !plan->device_plan) return W4_ERR_INVALID_ARG;
    const bool has_small = plan->items > 0, has_tc = plan->tc_items > 0;
    if (!has_small && !has_tc) return W4_ERR_INVALID_ARG;
    if (plan->format != 0 && !valid_group(plan->format)) return W4_ERR_INVALID_ARG;
    if (has_small && (plan->ctas < 1 || plan->ctas > plan->items ||
                      grouped_token_rows(plan->token_rows) != plan->token_rows))
        return W4_ERR_INVALID_ARG;
    if (has_tc && (plan->tc_ctas < 1 || plan->tc_ctas > plan->tc_items || plan->tc_max_bm < 16 ||
                   plan->tc_max_bm > 256 || plan->tc_offset % 128 != 0 || plan->tc_offset >= plan->bytes))
        return W4_ERR_INVALID_ARG;
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) return W4_ERR_CUDA;
    if (device != plan->device) return W4_ERR_INVALID_ARG;
    cudaError_t err;
    const DeviceInfo* dev = device_info(&err);
    if (!dev) return W4_ERR_CUDA;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (has_small)
        if (const int s = to_status(
                launch_grouped(plan->device_plan, plan->ctas, plan->token_rows, plan->format, *dev, st)))
            return s;
    if (has_tc)
        return to_status(launch_tc_grouped(static_cast<const uint8_t*>(plan->device_plan) + plan->tc_offset,
                                           plan->tc_ctas, plan->tc_max_bm, plan->format, *dev, st));
    return W4_OK;
}

int w4_gemm_grouped_noalloc(int32_t count, const w4_gemm_problem* problems, void* stream) {
    if (count < 1 || !problems) return W4_ERR_INVALID_ARG;
    std::vector<uint8_t> image;
    w4_grouped_plan p;
    if (const int s = grouped_prepare(nullptr, 0, count, problems, 128, nullptr, &image, &p)) return s;
    void* mem = nullptr;
    size_t cap = 0;
    if (static_plan_memory(&mem, &cap) != cudaSuccess) return W4_ERR_CUDA;
    if (image.size() > cap) return W4_ERR_UNSUPPORTED;
    // Stream-ordered: the copy lands after the stream's earlier work (a
    // previous call's kernels no longer read the array).  From pageable
    // memory, the source has been staged when the call returns, so `image`
    // may be released.
    if (cudaMemcpyAsync(mem, image.data(), image.size(), cudaMemcpyHostToDevice, static_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return W4_ERR_CUDA;
    p.device_plan = mem;
    return w4_gemm_grouped(&p, stream);
}

int w4_last_device_status(void* stream) {
    cudaError_t err;
    const DeviceInfo* dev = device_info(&err);
    if (!dev) return W4_ERR_CUDA;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned host = 0;
    if (cudaMemcpyAsync(&host, dev->status, sizeof(host), cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return W4_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return W4_ERR_CUDA;
    if (host != 0) {
        const unsigned zero = 0;
        if (cudaMemcpyAsync(dev->status, &zero, sizeof(zero), cudaMemcpyHostToDevice, st) != cudaSuccess ||
            cudaStreamSynchronize(st) != cudaSuccess)
            return W4_ERR_CUDA;
    }
    return static_cast<int>(host);
}

int w4_wait_probe(int64_t limit_ns, int32_t arrive, void* stream) {
    if (limit_ns < 0) return W4_ERR_INVALID_ARG;
    cudaError_t err;
    const DeviceInfo* dev = device_info(&err);
    if (!dev) return W4_ERR_CUDA;
    return to_status(launch_wait_probe(limit_ns, arrive, *dev, static_cast<cudaStream_t>(stream)));
}

const char* w4_status_string(int status) {
    switch (status) {
        case W4_OK: return "W4_OK";
        case W4_ERR_INVALID_ARG: return "W4_ERR_INVALID_ARG: invalid argument";
        case W4_ERR_UNSUPPORTED: return "W4_ERR_UNSUPPORTED: unsupported size, group or device";
        case W4_ERR_MISALIGNED: return "W4_ERR_MISALIGNED: pointer alignment";
        case W4_ERR_CUDA: return "W4_ERR_CUDA: CUDA runtime error";
        case W4_ERR_TIMEOUT: return "W4_ERR_TIMEOUT: a bounded device wait ran out";
        case W4_ERR_NUMERIC: return "W4_ERR_NUMERIC: a factorization failed (matrix not positive definite)";
        default: return "unknown w4 status";
    }
}

}  // extern "C"
