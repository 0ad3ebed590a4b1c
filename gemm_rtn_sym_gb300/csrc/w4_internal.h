// Internal declarations shared by the library's translation units (host side).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <vector>

namespace w4 {

// Device facts the launchers size their grids from (cached per device).
struct DeviceInfo {
    int sm_count = 0;
    int cc_major = 0;
    int cc_minor = 0;
    int max_smem_optin = 0;
    unsigned* status = nullptr;  // device address of this device's status word
};

// Returns nullptr (and sets *err) when the current device cannot be queried.
const DeviceInfo* device_info(cudaError_t* err);

// Launchers.  Arguments are already validated by the C ABI layer.
// group 32/64/128; zeros == nullptr: symmetric, else asymmetric (int8 z − 8 per
// group).  s != nullptr (group 128, symmetric only): RTN of bf16_rne(fp32(w·s_k)).
cudaError_t launch_quantize(const void* W, int64_t N, int64_t K, int group, void* packed, void* scales, void* zeros,
                            const float* s, const DeviceInfo& dev, cudaStream_t stream);

// x' = bf16_rne(fp32(x / s_k)) over x bf16 [M, K]; out may be x itself.
cudaError_t launch_scale_activations(const void* x, int64_t M, int64_t K, const float* s, void* out,
                                     const DeviceInfo& dev, cudaStream_t stream);

// Small-M path (TMA-fed GEMV on the legacy MMA): any M, one pass per 16 token rows.
cudaError_t launch_gemv(const void* x, int64_t M, int64_t N, int64_t K, const void* packed,
                        const void* scales, void* y, const DeviceInfo& dev, cudaStream_t stream);

// Small-M path for the affine formats: group 32/64/128, zeros (int8 z − 8 per
// group) or nullptr for symmetric codes; weights dequantised to bf16 first.
cudaError_t launch_gemv_affine(const void* x, int64_t M, int64_t N, int64_t K, int group, const void* packed,
                               const void* scales, const void* zeros, void* y, const DeviceInfo& dev,
                               cudaStream_t stream);

// Tensor-core path: tcgen05 MMA with TMEM accumulators, any M.
cudaError_t launch_gemm_tc(const void* x, int64_t M, int64_t N, int64_t K, const void* packed,
                           const void* scales, void* y, const DeviceInfo& dev, cudaStream_t stream);

// GPTQ (fp64 state): the factor U of (H + λI)⁻¹ (own blocked Cholesky and
// triangular inverse), then per matrix the sweep kernel and the fp64 tile
// product for the block updates.  Return 0, 1 on a CUDA failure, 2 when the
// workspace is too small.
size_t gptq_factor_workspace_bytes(int64_t K);
size_t gptq_workspace_bytes(int64_t N, int64_t K);
int launch_gptq_factor(const float* H, int64_t K, double damp, double* U, void* workspace, size_t workspace_bytes,
                       const DeviceInfo& dev, cudaStream_t stream);
int launch_gptq(const void* W, int64_t N, int64_t K, int group, const double* U, void* packed, void* scales,
                void* workspace, size_t workspace_bytes, const DeviceInfo& dev, cudaStream_t stream);

// Tensor-core path for the affine formats (group 32/64/128, zeros or nullptr).
cudaError_t launch_gemm_tc_affine(const void* x, int64_t M, int64_t N, int64_t K, int group, const void* packed,
                                  const void* scales, const void* zeros, void* y, const DeviceInfo& dev,
                                  cudaStream_t stream);

// 2-D tensor map over x bf16 [M, K]: boxes of 64 k x box_rows rows, 128-byte
// swizzle, rows past M read as zeros.
cudaError_t encode_x_map(CUtensorMap* map, const void* x, int64_t M, int64_t K, int box_rows);

// 3-D tensor map over x bf16 [M, K] seen as [K/64][M][64]: boxes of `blocks`
// 64-k blocks x `rows` rows, 128-byte swizzle, rows past M read as zeros.
cudaError_t encode_x_stage_map(CUtensorMap* map, const void* x, int64_t M, int64_t K, int rows, int blocks);

// 3-D tensor map over packed codes u8 [N, K/2] seen as [G][N][64]: boxes of
// `groups` groups x `rows` rows x 64 bytes; rows past N and groups past G read
// as zeros.
cudaError_t encode_codes_stage_map(CUtensorMap* map, const void* packed, int64_t N, int64_t K, int rows,
                                   int groups, CUtensorMapSwizzle swizzle);

// One problem of a grouped matmul (validated by the C ABI layer).  zeros:
// int8 zero − 8 per group of the affine formats, or null.
struct GroupedSpec {
    const void* x;
    int64_t M, N, K;
    const void* packed;
    const void* scales;
    void* y;
    const void* zeros;
};
// Plan bytes for `count` problems with `n_items` 64-row blocks in total,
// scheduled over `n_ctas` CTAs.
size_t grouped_plan_bytes(int32_t count, int64_t n_items, int32_t n_ctas);
// Token rows the grouped small-M kernel stages per pass for a largest M of
// max_m (2, 4, 8, 16 or 24; max_m ≤ 24).
int grouped_token_rows(int64_t max_m);
// CTAs the grouped kernel runs with on this device (resident at once).
// format: 0 for the symmetric group-128 format, else the affine group size.
int grouped_ctas(int token_rows, int format, const DeviceInfo& dev);
// Host image of a grouped plan: tensor maps, and the items assigned longest
// first to a grid of at most max_ctas CTAs (sm_count SMs; see the source for
// how the grid is chosen).
cudaError_t grouped_plan_build(const GroupedSpec* specs, int32_t count, int token_rows, int format, int32_t max_ctas,
                               int32_t sm_count, std::vector<uint8_t>* out, int64_t* n_items, int32_t* n_ctas_used);
// The device address and size of the library's static plan buffer on the
// current device (w4_gemm_grouped_noalloc).
cudaError_t static_plan_memory(void** ptr, size_t* bytes);
// Runs a plan already copied to device memory.
cudaError_t launch_grouped(const void* plan, int32_t n_ctas, int token_rows, int format, const DeviceInfo& dev,
                           cudaStream_t stream);

// Tensor-core grouped plan (problems with M ≥ 25): (problem, 128-row tile,
// token tile) items scheduled longest first over one CTA per SM.
size_t tc_grouped_plan_bytes(int32_t count, int64_t n_items, int32_t n_ctas);
int64_t tc_grouped_items(const GroupedSpec& sp);
cudaError_t tc_grouped_plan_build(const GroupedSpec* specs, int32_t count, int format, int32_t n_ctas,
                                  std::vector<uint8_t>* out, int64_t* n_items, int32_t* n_ctas_used);
cudaError_t launch_tc_grouped(const void* plan, int32_t n_ctas, int max_bm, int format, const DeviceInfo& dev,
                              cudaStream_t stream);

cudaError_t launch_wait_probe(int64_t spin_limit, int arrive, const DeviceInfo& dev,
                              cudaStream_t stream);

}  // namespace w4
