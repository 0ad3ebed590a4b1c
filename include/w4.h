/*
 * w4.h — C ABI of the GB300 (sm_103a) library for symmetric INT4, group-128,
 * round-to-nearest weight quantisation and the decode-time W4A16 matmul.
 *
 * What the library computes
 * -------------------------
 * Source: "Qwen3.5-4B, 작게 저장하면 무엇이 달라질까?" (Qwen3.5-4B whole-model
 * quantisation study).
 *   §1, group-quantisation equation: q = clip(round(w/d) + z, q_min, q_max),
 *       ŵ = d·(q − z); the symmetric case has z = 0.
 *   §1, paragraph under the FFN example y = W x (2560×9216): a group is 128
 *       consecutive weights of one row along the input direction (72 groups
 *       per row at 9216 inputs); every weight keeps its own 4-bit code and the
 *       group shares one restore scale d.
 *   §2, settings table: RTN, group 128, 4-bit weights and BF16 inputs, range
 *       from the group's extremes ("minmax · symmetric"), no clipping search,
 *       no calibration data.
 * Readings taken where the page is silent: d = bf16_rne(fp32(max|w| / 7)),
 * q = clamp(round_half_even(fp32(w / d)), −8, 7) with the stored bf16 d, and
 * d = +0, q = 0 for a group whose d is zero.  No flush-to-zero: subnormal
 * weights and scales are handled.  NaN/Inf weights are outside the contract
 * (outputs unspecified, never an out-of-bounds access).
 *
 * Data layout (all row-major, dense, no padding)
 * ----------------------------------------------
 *   W       bf16  [N, K]        weights, N = output features, K = input features
 *   packed  u8    [N, K/2]      4-bit two's-complement codes; the 64 bytes of
 *                               (row n, group g) start at n·K/2 + 64·g.  In that
 *                               block, 16-byte chunk j holds k = 32j..32j+31; the
 *                               32-bit little-endian word w of a chunk holds
 *                               k = 8w..8w+7 (relative to the chunk), and nibble
 *                               slot i (bits 4i..4i+3) of the word holds offset
 *                               {0,2,4,6,1,3,5,7}[i].  So slots i and i+4 hold a
 *                               consecutive pair, ready for a bf16x2 dequant.
 *   scales  bf16  [N, K/128]    d of (row n, group g) at n·(K/128) + g
 *   x       bf16  [M, K]        activations (M tokens)
 *   y       bf16  [M, N]        y[m, n] = Σ_k ŵ[n, k] · x[m, k], rounded to bf16
 *
 * Conventions for every entry point
 * ---------------------------------
 *  - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *    keeps no per-call state and allocates no device memory of its own; its
 *    only device state is a per-device status word and a 2 MB plan array (for
 *    w4_gemm_grouped_noalloc), both static __device__ variables.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Work is enqueued asynchronously on it; nothing synchronises, except
 *    w4_last_device_status(), w4_grouped_plan_init (a blocking copy of the
 *    plan) and w4_gemm_grouped_noalloc (see there).
 *  - K must be a multiple of 128; group is 128 except where an entry point
 *    says otherwise (32, 64 or 128 for the quantisers and w4_gemm_affine);
 *    N, M, K ≥ 0.  Sizes
 *    with N·K ≥ 2^62 are rejected; the matmul also needs N, M, K < 2^31
 *    (W4_ERR_UNSUPPORTED otherwise).
 *  - W, x and packed must be 16-byte aligned; scales and y 2-byte aligned.
 *  - y must not overlap x, packed or scales; packed/scales must not overlap W.
 *  - Argument errors are returned synchronously before anything is launched.
 *    A failed launch returns W4_ERR_CUDA (the CUDA error is left readable with
 *    cudaGetLastError()).
 *  - Each call uses the device that is current on the calling thread.
 */
#ifndef W4_H_
#define W4_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum w4_status {
    W4_OK = 0,
    W4_ERR_INVALID_ARG = 1, /* null pointer, negative size, overlap, overflow   */
    W4_ERR_UNSUPPORTED = 2, /* group != 128, K % 128 != 0, unsupported device    */
    W4_ERR_MISALIGNED = 3,  /* pointer alignment below what is stated above     */
    W4_ERR_CUDA = 4,        /* a CUDA runtime call or kernel launch failed       */
    W4_ERR_TIMEOUT = 5,     /* a bounded device-side wait ran out (see below)    */
    W4_ERR_NUMERIC = 6      /* a factorization failed (w4_gptq_quantize: H + λI
                               not positive definite); reported through
                               w4_last_device_status                             */
} w4_status;

/* Kernel choice for w4_gemm_ex. */
typedef enum w4_gemm_path {
    W4_PATH_AUTO = 0,    /* what w4_gemm does: picked from M (w4_gemm_path_for)  */
    W4_PATH_SMALL_M = 1, /* TMA-fed GEMV: register nibble decode, legacy MMA,
                            cluster split-K; any M (32 token rows per pass)     */
    W4_PATH_TENSOR = 2   /* tcgen05 tile: weights dequantised into tensor
                            memory as the A operand, TMEM accumulators, cluster
                            split-K; any M ≥ 1                                  */
} w4_gemm_path;

/* Bytes of the packed code buffer: N·K/2.  0 for invalid sizes. */
size_t w4_packed_bytes(int64_t N, int64_t K);

/* Bytes of the scale buffer: N·(K/group)·2 (group 32, 64 or 128).  0 for
 * invalid sizes. */
size_t w4_scales_bytes(int64_t N, int64_t K, int32_t group);

/* Bytes of the zero-point buffer of the asymmetric format: N·(K/group).  0 for
 * invalid sizes. */
size_t w4_zeros_bytes(int64_t N, int64_t K, int32_t group);

/*
 * w4_quantize_rtn — RTN symmetric INT4 quantisation of W (§1 equation with
 * z = 0; §2 settings: group 128, minmax · symmetric, no calibration).  Groups
 * of 32 or 64 (§2 settings table: smaller groups follow the range more closely
 * at the cost of more scales) apply the same rules per group.
 *   W       in : bf16 [N, K]
 *   group   in : 128 (the study's setting), 64 or 32
 *   packed  out: u8   [N, K/2]  (layout above; the same for every group size)
 *   scales  out: bf16 [N, K/group]
 * Deterministic and bit-exact: for every group, d = bf16_rne(fp32(max|w|/7))
 * and q = clamp(round_half_even(fp32(w/d)), −8, 7).  N = 0 or K = 0 is a no-op.
 * Only group 128 is read by w4_gemm; w4_gemm_affine reads every group size.
 */
int w4_quantize_rtn(const void* W, int64_t N, int64_t K, int32_t group,
                    void* packed, void* scales, void* stream);

/*
 * w4_quantize_rtn_asym — RTN asymmetric INT4 (§1 equation with a free zero
 * point z, the code of real zero in the §1 symbol table), per group of 32, 64
 * or 128:
 *   lo = min(0, min w), hi = max(0, max w),
 *   d  = bf16_rne(fp32(fp32(hi − lo) / 15))          (IEEE fp32 steps),
 *   z  = clamp(round_half_even(fp32(−lo / d)), 0, 15) (z = 8 where d = 0),
 *   q  = clamp(round_half_even(fp32(w / d)) + z, 0, 15),
 * so ŵ = d·(q − z).  Stored: the nibble q − 8 in the packed layout above and
 * the int8 z − 8 per group; ŵ = d·(stored code − stored zero).  (The symmetric
 * format is the case stored zero = 0.)
 *   W       in : bf16 [N, K]
 *   packed  out: u8   [N, K/2]
 *   scales  out: bf16 [N, K/group]
 *   zeros   out: int8 [N, K/group], any alignment
 * Bit-exact and deterministic.  N = 0 or K = 0 is a no-op.
 */
int w4_quantize_rtn_asym(const void* W, int64_t N, int64_t K, int32_t group,
                         void* packed, void* scales, void* zeros, void* stream);

/*
 * AWQ-style channel scaling (§2 AWQ equation: W'_ij = W_ij·s_j and
 * x'_j = x_j/s_j leave the product unchanged, W'x' = Wx; s_j is a per-input-
 * channel factor, distinct from the group scale d and not limited to powers of
 * two).  The caller supplies s; searching for it (the study's grid of
 * exponents over calibration statistics) is not part of this library.
 *
 * w4_quantize_rtn_scaled — quantises W' = bf16_rne(fp32(W[n,k] · s[k])) exactly
 * as w4_quantize_rtn quantises W (same d and q rules, same outputs); W' itself
 * is never stored.
 *   W       in : bf16 [N, K]
 *   s       in : fp32 [K], device, 16-byte aligned; every entry finite and > 0
 *                (not checked: other values give unspecified codes, never an
 *                out-of-bounds access).  Where W·s overflows bf16 the codes of
 *                that group are unspecified, as for Inf weights.
 *   packed  out: u8   [N, K/2]
 *   scales  out: bf16 [N, K/128]
 * s must not overlap packed or scales.
 */
int w4_quantize_rtn_scaled(const void* W, int64_t N, int64_t K, int32_t group,
                           const float* s, void* packed, void* scales, void* stream);

/*
 * w4_scale_activations — the input side: x'[m,k] = bf16_rne(fp32(x[m,k] / s[k]))
 * with the IEEE fp32 quotient, so that w4_gemm(x', packed', scales') computes
 * Ŵ'x' ≈ Wx for the outputs of w4_quantize_rtn_scaled.  With M = 1 it also
 * folds 1/s into a per-channel vector, such as the weight of the normalisation
 * that produces x.  A streaming elementwise pass (HBM-bound).
 *   x       in : bf16 [M, K], 16-byte aligned
 *   s       in : fp32 [K], 16-byte aligned, finite and > 0 (as above)
 *   x_out   out: bf16 [M, K], 16-byte aligned; x_out == x (in place) is allowed,
 *                any other overlap with x, or any overlap with s, is rejected.
 * K must be a multiple of 128; M = 0 or K = 0 is a no-op.
 */
int w4_scale_activations(const void* x, int64_t M, int64_t K, const float* s,
                         void* x_out, void* stream);

/*
 * w4_gemm — y = Ŵ x with ŵ = d·q (§1 FFN example y = W x; §2: 4-bit weights,
 * BF16 inputs).  M is the number of token rows: 1 for plain decode, K+1 for a
 * speculative-verify pass with K drafts.
 *   x       in : bf16 [M, K]
 *   packed  in : u8   [N, K/2]   as written by w4_quantize_rtn
 *   scales  in : bf16 [N, K/128]
 *   y       out: bf16 [M, N]
 * Accuracy: |y − Σ_k ŵ x| ≤ 4e-3 · Σ_k |ŵ x| + 1 bf16 ulp per element
 * (fp32 accumulation; the tensor-core path rounds d·q to bf16 first).
 * K = 0 writes zeros to y; M = 0 or N = 0 is a no-op.
 */
int w4_gemm(const void* x, int64_t M, int64_t N, int64_t K,
            const void* packed, const void* scales, void* y, void* stream);

/* w4_gemm with an explicit kernel choice (w4_gemm_path); same contract. */
int w4_gemm_ex(const void* x, int64_t M, int64_t N, int64_t K,
               const void* packed, const void* scales, void* y, void* stream,
               int32_t path);

/*
 * w4_gemm_affine — y = Ŵ x for every stored format: ŵ = d·(c − z') with c the
 * stored code, d the scale and z' the stored zero of its group (z' = 0 when
 * zeros is NULL, the symmetric format).
 *   group   in : 32, 64 or 128 (the group size the weights were quantised with)
 *   scales  in : bf16 [N, K/group]
 *   zeros   in : int8 [N, K/group] from w4_quantize_rtn_asym, or NULL
 * Same kernels, paths, accuracy and argument rules as w4_gemm_ex; group 128
 * with zeros NULL is w4_gemm_ex itself.  Other formats dequantise each weight
 * to bf16(d·(c − z')) (one rounding) before the products.
 */
int w4_gemm_affine(const void* x, int64_t M, int64_t N, int64_t K, int32_t group,
                   const void* packed, const void* scales, const void* zeros,
                   void* y, void* stream, int32_t path);

/*
 * GPTQ into the same storage as RTN (§2 settings table: GPTQ with the RTN
 * storage, damping 0.01, columns in their original order, 128-column blocks;
 * §2 H' = H + λI with λ = damp·mean(diag H); the method table: quantise one
 * column, then correct the remaining weights).  The correction is the
 * published GPTQ rule (Frantar et al., 2022): with Uᵀ U = (H')⁻¹, U upper
 * triangular, column c's error (w_c − ŵ_c) / U[c, c] moves every later column
 * k of the row by −err·U[c, k]; each group's scale is taken at its first
 * column from the group's current (corrected) weights with the RTN rules:
 * d = bf16_rne(fp32(max|w| / 7)), q = clamp(round_half_even(w / d), −8, 7).
 * All arithmetic is fp64, so the rounding decisions match an fp64 reference.
 * Two calls: the factor once per calibration statistic (every matrix that
 * reads the same input shares it), then the quantisation per matrix.
 *
 * w4_gptq_factor — U, upper triangular with Uᵀ U = (H + λI)⁻¹:
 *   H          in : fp32 [K, K], symmetric positive semi-definite (the
 *                   calibration statistic, e.g. Xᵀ X over calibration inputs
 *                   X [T, K]), 4-byte aligned
 *   damp       in : the damping fraction (the study: 0.01), ≥ 0
 *   U          out: fp64 [K, K] row-major, 8-byte aligned; its upper triangle
 *                   (diagonal included) is the factor, the rest unspecified
 * Computed as U = J L̃⁻¹ J with L̃ the Cholesky factor of J (H + λI) J (J the
 * order-reversing permutation): the library's own blocked fp64 Cholesky and
 * triangular inverse on `stream`, (2/3)·K³ flops.  A failed factorization (a
 * pivot ≤ 0) shows as W4_ERR_NUMERIC in w4_last_device_status; U is then
 * unspecified.
 *   workspace  in : w4_gptq_factor_workspace_bytes(K) bytes (= 8·K² + 256,
 *                   rounded), 256-byte aligned
 *
 * w4_gptq_quantize — codes and scales of W given U:
 *   W          in : bf16 [N, K] (not modified)
 *   group      in : 32, 64 or 128 (columns are processed in blocks of 128)
 *   U          in : as written by w4_gptq_factor for this W's input
 *   packed     out: u8   [N, K/2]
 *   scales     out: bf16 [N, K/group]
 *   workspace  in : w4_gptq_workspace_bytes(N, K) bytes (= 8·N·K + 8·N·128,
 *                   rounded), 256-byte aligned
 * Block updates by the library's own fp64 tile product on `stream`.
 *
 * Both: N, K ≤ 4,194,240 (W4_ERR_UNSUPPORTED above); workspaces owned by the caller,
 * overlapping nothing else, contents on return unspecified.
 */
size_t w4_gptq_factor_workspace_bytes(int64_t K);
int w4_gptq_factor(const float* H, int64_t K, double damp, double* U,
                   void* workspace, size_t workspace_bytes, void* stream);
size_t w4_gptq_workspace_bytes(int64_t N, int64_t K);
int w4_gptq_quantize(const void* W, int64_t N, int64_t K, int32_t group,
                     const double* U, void* packed, void* scales,
                     void* workspace, size_t workspace_bytes, void* stream);

/* The kernel W4_PATH_AUTO picks for these sizes (W4_PATH_SMALL_M for
 * M ≤ 24, W4_PATH_TENSOR above: the measured crossover for one launch per
 * matrix), or a negative w4_status for invalid sizes. */
int w4_gemm_path_for(int64_t M, int64_t N, int64_t K);

/*
 * Grouped matmul — many independent problems y_i = Ŵ_i x_i in one call (the
 * matrices of a layer, or of a whole model step).  Each problem is computed
 * as by w4_gemm's kernel for its M (same per-element results contract, K not
 * split, deterministic): problems with M ≤ 24 by the small-M kernel, whose
 * work items are (problem, 64-row block) pairs on a fixed grid of two or
 * three CTAs per SM; problems with M ≥ 25 by the tensor-core kernel (the
 * measured crossover, as for w4_gemm), whose items are
 * (problem, 128-row tile, token tile) on one CTA per SM.  Items are assigned
 * at plan time longest first to the least-loaded CTA, and each CTA streams
 * its items back to back through its TMA pipelines.  A plan with both kinds
 * launches two kernels, one after the other, on the stream.
 *
 * A plan is built once (host work plus one synchronous copy) and may then be
 * run any number of times, including inside CUDA graphs; it records the
 * problems' pointers, so their buffers must stay allocated and in place, but
 * their contents may change between runs.
 */
typedef struct w4_gemm_problem {
    const void* x;      /* bf16 [M, K]  (16-byte aligned)                       */
    int64_t M;          /* token rows, ≥ 1                                       */
    int64_t N;          /* output features, ≥ 1                                  */
    int64_t K;          /* input features, multiple of 128, ≥ 128                */
    const void* packed; /* u8 [N, K/2]  as written by w4_quantize_rtn (16-B al.) */
    const void* scales; /* bf16 [N, K/128]                                       */
    void* y;            /* bf16 [M, N]; must not overlap any other problem's    */
                        /* inputs or output                                      */
} w4_gemm_problem;

typedef struct w4_grouped_plan {
    void* device_plan;   /* the caller's device memory holding the plan           */
    size_t bytes;        /* bytes of it in use                                    */
    int32_t count;       /* problems                                              */
    int32_t device;      /* CUDA device the plan was built on                     */
    int32_t items;       /* small-M work items (0: no problem with M ≤ 24)        */
    int32_t ctas;        /* CTAs they were scheduled over (the launch grid)       */
    int32_t token_rows;  /* small-M kernel variant: token rows staged per pass,
                            the smallest of 2, 4, 8, 16, 24 ≥ the largest M      */
    int32_t tc_items;    /* tensor-core work items (0: no problem with M ≥ 25)    */
    int32_t tc_ctas;     /* CTAs they were scheduled over                         */
    int32_t tc_max_bm;   /* widest token tile                                     */
    size_t tc_offset;    /* byte offset of the tensor-core part of the plan       */
    int32_t format;      /* 0: symmetric group 128 (w4_gemm); 32, 64, 128: the
                            affine formats of w4_gemm_affine at that group size   */
} w4_grouped_plan;

/* Device bytes a plan for these problems needs (0 if any problem is invalid);
 * an upper bound that does not depend on the device. */
size_t w4_grouped_plan_bytes(int32_t count, const w4_gemm_problem* problems);

/* Validates the problems (as w4_gemm would; an output overlapping any input
 * or other output → W4_ERR_INVALID_ARG), encodes the plan and copies it
 * synchronously into `device_memory` (128-byte aligned, at least
 * w4_grouped_plan_bytes bytes, on the current device), and fills *plan.  The
 * library keeps no reference to `problems` afterwards. */
int w4_grouped_plan_init(w4_grouped_plan* plan, void* device_memory, size_t bytes,
                         int32_t count, const w4_gemm_problem* problems);

/*
 * Grouped matmul over the affine formats of w4_gemm_affine (study §1 equation
 * with a free zero point; §2 settings table: smaller groups): every problem of
 * the plan stores its codes at one group size.
 *   group  in : 32, 64 or 128 (each problem's scales are bf16 [N, K/group])
 *   zeros  in : NULL (no problem has zero points), or `count` pointers, each
 *               NULL (symmetric codes) or problem i's int8 [N, K/group] zeros
 *               from w4_quantize_rtn_asym (any alignment)
 * Each problem is computed as by w4_gemm_affine's kernel for its M (M ≤ 24:
 * the small-M kernel, M ≥ 25: the tensor-core kernel), within the same
 * bound; group 128 without zeros is exactly w4_grouped_plan_init.  The plan
 * runs with w4_gemm_grouped; sizes, checks and errors as above (zeros must
 * not overlap any output).
 */
size_t w4_grouped_plan_bytes_affine(int32_t count, const w4_gemm_problem* problems,
                                    int32_t group, const void* const* zeros);
int w4_grouped_plan_init_affine(w4_grouped_plan* plan, void* device_memory, size_t bytes,
                                int32_t count, const w4_gemm_problem* problems,
                                int32_t group, const void* const* zeros);

/* Runs every problem of the plan on `stream` (the device must be the one the
 * plan was built on).  Asynchronous; no allocation. */
int w4_gemm_grouped(const w4_grouped_plan* plan, void* stream);

/*
 * w4_gemm_grouped_noalloc — the grouped matmul without caller memory for the
 * plan: the plan is built on every call and copied into a 2 MB device array
 * compiled into the library (found once per device with
 * cudaGetSymbolAddress), then run on `stream`.  No device memory is
 * allocated.  An implementation convenience with no counterpart in the pages:
 * they describe the computation, not how its work lists are stored.
 *   W4_ERR_UNSUPPORTED  the plan for these problems exceeds the 2 MB array
 *                       (about 5000 problems, or about 250000 64-row blocks);
 *   otherwise the checks and results of w4_grouped_plan_init + w4_gemm_grouped.
 * Races: the array is shared by every call on a device.  Calls in order on
 * one stream are safe (the plan copy is ordered after the stream's earlier
 * work); calls that may overlap on the GPU — other streams or other host
 * threads — can overwrite a plan a running kernel is reading, and give wrong
 * results.  The plan is copied from pageable host memory, so the host thread
 * may block until the stream's earlier work is done.  Callers that need
 * overlapping calls use w4_grouped_plan_init + w4_gemm_grouped, with one plan
 * buffer per call.
 */
int w4_gemm_grouped_noalloc(int32_t count, const w4_gemm_problem* problems, void* stream);

/*
 * Every wait inside the library's kernels (mbarrier phases, TMA completion)
 * is bounded.  A wait that runs out records W4_ERR_TIMEOUT in a per-device
 * status word and the kernel returns early (its outputs are then undefined).
 * w4_last_device_status synchronises `stream`, returns the recorded status
 * (W4_OK if none) and clears it.  Returns W4_ERR_CUDA if synchronisation fails.
 */
int w4_last_device_status(void* stream);

/*
 * Diagnostic for the bounded-wait machinery: launches one CTA that waits on an
 * mbarrier.  With arrive = 1 the barrier is completed and the wait succeeds;
 * with arrive = 0 nothing ever completes it and the wait gives up after
 * `limit_ns` nanoseconds, records W4_ERR_TIMEOUT and exits normally.  Read
 * the outcome with w4_last_device_status.
 */
int w4_wait_probe(int64_t limit_ns, int32_t arrive, void* stream);

/* Static, human-readable name of a status code. */
const char* w4_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* W4_H_ */
