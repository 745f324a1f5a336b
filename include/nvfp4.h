/*
 * nvfp4.h -- C ABI of libnvfp4.so: NVFP4 weights x bf16 activations on one GPU.
 *
 * The operation (bw24 README, section on the NVFP4 / Q4_0 decode path; bw24
 * wiki Home, feature list, NVFP4 decode path entry; qwentin README, section
 * "How it works", wide prefill and batched verify): a weight matrix W[M][K]
 * stored as NVFP4 is multiplied by N token activations x[N][K] in bf16,
 *
 *     y[n][m] = sum_k x[n][k] * ts * e2m1(code[m][k]) * e4m3(scale[m][k/16]),
 *
 * with fp32 accumulation and fp32 (or bf16) output.  N = 1 is plain decode,
 * N = draft+1 a speculative verify that reads every weight once for all draft
 * tokens (bw24 README, speculative decoding section; qwentin README,
 * "Highlights", batched verify), and N in the hundreds to thousands a prefill
 * (qwentin README, "How it works", wide prefill where each weight is read once
 * for N tokens).
 *
 * NVFP4 layout used by every call (one tensor = three device buffers):
 *   codes        uint8 [M][K/2]  two 4-bit E2M1 codes per byte; element k = 2j
 *                                in the low nibble of byte j, k = 2j+1 in the
 *                                high nibble.  E2M1: bit 3 sign, bits 2..1
 *                                exponent (bias 1), bit 0 mantissa; magnitudes
 *                                0, .5, 1, 1.5, 2, 3, 4, 6.
 *   scales       uint8 [M][K/16] one FP8 E4M3 (OCP E4M3FN) scale per 16
 *                                consecutive k of a row, row-major.
 *   tensor_scale float [1]       one FP32 scale for the whole tensor, kept in
 *                                device memory so no call synchronises.
 * K must be a multiple of 16.  Activations x are bf16 bit patterns, row-major
 * [N][K]; outputs are row-major [N][M].
 *
 * Conventions for every entry point:
 *   - Ownership: the caller allocates and owns every buffer; the library never
 *     allocates or frees memory and keeps no pointer after a call returns.
 *   - Pointers marked "device" must be CUDA device (or managed) memory of the
 *     current device.  Codes, scales, x and outputs must be 16-byte aligned.
 *   - Asynchrony: every call enqueues kernels on `stream` (NULL = legacy default
 *     stream) and returns without synchronising.  Results are ready when the
 *     stream reaches that point.
 *   - Workspace: scratch device memory of at least nvfp4_workspace_bytes(...)
 *     bytes, 16-byte aligned (checked), owned by the caller and not used by anything
 *     else while the call's kernels run.  Calls that share a workspace must be
 *     ordered on one stream.  The products with N <= 16 (skinny path) keep
 *     split-K arrival counters in it: their workspace must be zero-filled
 *     before its first use (cudaMemsetAsync), and every such call leaves the
 *     counters at zero again, so one zeroing serves any number of skinny
 *     calls of any shapes.  Do not write to it between skinny calls (a quantise or
 *     prefill call on the same buffer counts as writing), and zero it again
 *     after a call that failed.  The quantise and prefill calls need no
 *     initialisation and leave their workspace undefined, except that the
 *     product calls keep a device status word at byte NVFP4_STATUS_WORD_OFFSET
 *     (see nvfp4_device_status).
 *   - Errors: arguments are checked on the host before anything is enqueued;
 *     a bad argument returns a nonzero nvfp4_status and nothing runs.  A
 *     failed launch returns NVFP4_ERR_CUDA.  The library never aborts or prints.
 *     Every wait inside a kernel is bounded: a pipeline that stops making
 *     progress gives up after 2 s of wall time, records a code in the
 *     workspace's status word and returns (the outputs are then undefined),
 *     so the GPU never hangs and the context stays usable; the launching call
 *     has already returned, so the code is read with nvfp4_device_status.
 *   - Determinism: the reduction order is fixed by the shapes alone (and the
 *     device's SM count), so repeated calls give bit-identical results.  For
 *     N <= 16 (skinny kernel) row n of an N-token call equals the same token in
 *     any other call with N <= 16 and the same weights, M and K (floating-point
 *     summation order is part of the contract: bw24 wiki Home, list of checks
 *     every kernel change must pass, and bw24 README, where decode and verify
 *     launch the same kernel symbols and agree bit for bit).  For N > 16 (the
 *     tensor-core prefill kernel) a single matrix whose tiles would leave the
 *     last wave of SMs poorly filled splits K across thread blocks (stream-K)
 *     in a way that depends on N, so rows of calls with different N > 16 (and
 *     across N = 16) agree within the accuracy bound below, bit for bit only
 *     when neither call splits.  A skinny call in which some token's activations are not all exact in f16 after scaling by a
 *     power of two (a dynamic range wider than f16's) switches the whole call
 *     to bf16 operands; its rows also agree within the bound.
 *   - Accuracy: every product code * scale * x is exact (bf16 operands, fp32
 *     accumulation); results satisfy |y - y_ref| <= 1e-5 * sum_k |w*x| + 1e-7
 *     against an fp64 evaluation of the formula above.
 */
#ifndef NVFP4_H
#define NVFP4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *nvfp4_stream_t; /* same handle as cudaStream_t */

/* Status codes returned by every entry point. */
typedef enum {
    NVFP4_OK = 0,
    NVFP4_ERR_INVALID_ARG = 1,       /* null pointer, negative size, misalignment, bad enum */
    NVFP4_ERR_UNSUPPORTED_SHAPE = 2, /* K % 16 != 0, N outside the call's range, size overflow */
    NVFP4_ERR_WORKSPACE = 3,         /* workspace smaller than nvfp4_workspace_bytes() */
    NVFP4_ERR_CUDA = 4,              /* a CUDA runtime call or kernel launch failed */
    NVFP4_ERR_DEVICE_TIMEOUT = 5     /* a kernel's bounded wait gave up (nvfp4_device_status) */
} nvfp4_status;

/* Operation ids for nvfp4_workspace_bytes. */
typedef enum {
    NVFP4_OP_QUANTIZE = 0,
    NVFP4_OP_GEMV_SKINNY = 1,
    NVFP4_OP_GATEUP_SWIGLU = 2,
    NVFP4_OP_GEMM_PREFILL = 3,
    NVFP4_OP_FP6_GEMM = 4,
    NVFP4_OP_FP6_GATEUP_SWIGLU = 5
} nvfp4_op;

/* Output element types. */
typedef enum { NVFP4_OUT_F32 = 0, NVFP4_OUT_BF16 = 1 } nvfp4_out_dtype;

/* Human-readable name of a status code (static string, never NULL). */
const char *nvfp4_status_string(int status);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int nvfp4_version(void);

/* Bytes of workspace the call `op` needs for these sizes (0 if none).  Host
 * only, no CUDA call; depends on (op, N, M, K) alone, not on the device.
 * Returns 0 as well for sizes the call would reject. */
size_t nvfp4_workspace_bytes(int op, int64_t N, int64_t M, int64_t K);

/* Quantise fp32 weights to NVFP4.
 * The recipe (fp32 arithmetic in this order, IEEE round-to-nearest-even):
 *   amax = max |w|;  ts = amax / 2688  (2688 = 6 * 448, the largest E2M1 value
 *   times the largest E4M3 value);  for every 16-element block of a row:
 *   scale = E4M3_rne_saturating((block_amax / 6) / ts);  d = e4m3(scale) * ts;
 *   code[k] = nearest E2M1 to w[k] / d (ties to the even code, |.| > 6 clamps
 *   to 6, the sign of w kept, so a small negative value gives 0x8).  A block
 *   with d == 0 (scale 0, or ts == 0) gets all-zero codes.
 * w            device fp32 [M][K], row-major, finite (non-finite weights give
 *              unspecified codes).
 * codes        device uint8 [M][K/2] (output)
 * scales       device uint8 [M][K/16] (output)
 * tensor_scale device float [1] (output)
 * workspace    device scratch of nvfp4_workspace_bytes(NVFP4_OP_QUANTIZE, 0, M, K).
 * The NVFP4 weights the pages use are produced this way at load time (bw24
 * README, safetensors loader, re-encoding to NVFP4 at load; qwentin README,
 * converter section, quantising and packing on the GPU through the C ABI). */
int nvfp4_quantize(const float *w, int64_t M, int64_t K,
                   uint8_t *codes, uint8_t *scales, float *tensor_scale,
                   void *workspace, size_t workspace_bytes, nvfp4_stream_t stream);

/* Quantise bf16 weights to NVFP4: the recipe of nvfp4_quantize applied to the
 * exact fp32 values of the bf16 inputs, so a bf16 matrix and its fp32 copy give
 * byte-identical codes, scales and tensor scale.  Checkpoints the pages load
 * hold bf16 weights that are re-encoded at load time (bw24 README, safetensors
 * loader; qwentin README, converter section).
 * w            device bf16 bits [M][K], row-major, finite.
 * Other arguments, workspace and errors as for nvfp4_quantize (workspace:
 * nvfp4_workspace_bytes(NVFP4_OP_QUANTIZE, 0, M, K)). */
int nvfp4_quantize_bf16(const uint16_t *w, int64_t M, int64_t K,
                        uint8_t *codes, uint8_t *scales, float *tensor_scale,
                        void *workspace, size_t workspace_bytes, nvfp4_stream_t stream);

/* Import of NVFP4 weights stored with their block scales in the blocked
 * layout that block-scaled tensor-core GEMMs read.  The pages re-encode
 * checkpoints into the engine's own layout at load time (bw24 README,
 * safetensors loader; bw24 wiki Home, NVFP4 decode path) but print no external
 * layout; this is the one the library accepts:
 *   codes        uint8 [M][K/2], exactly as in this library (element 2j in the
 *                low nibble of byte j): no repacking, use the buffer as is.
 *   scales       E4M3 bytes in 128-row x 4-column blocks, S = K/16 scale
 *                columns; blocks row-major over (ceil(M/128), ceil(S/4));
 *                inside a block the scale of row r, column c sits at byte
 *                (r % 32) * 16 + (r / 32) * 4 + c.  Entries for rows >= M or
 *                columns >= S are padding and are ignored.
 *   tensor scale the same fp32 dequantisation factor (weight = code * scale * ts).
 * nvfp4_blocked_scale_bytes gives the size of the blocked scale buffer (0 for
 * sizes the call rejects); nvfp4_import_blocked_scales rewrites it into the
 * row-major [M][K/16] scale buffer this library reads, byte for byte.
 * blocked  device uint8, nvfp4_blocked_scale_bytes(M, K) bytes, 16-byte aligned.
 * scales   device uint8 [M][K/16] (output), 16-byte aligned.
 * Errors: NVFP4_ERR_UNSUPPORTED_SHAPE for K % 16 != 0; NVFP4_ERR_INVALID_ARG
 * for negative sizes or null / misaligned pointers (M or K = 0 is a no-op). */
size_t nvfp4_blocked_scale_bytes(int64_t M, int64_t K);

int nvfp4_import_blocked_scales(const uint8_t *blocked, int64_t M, int64_t K,
                                uint8_t *scales, nvfp4_stream_t stream);

/* Skinny product, N = 1..16 tokens: y[N][M] = x[N][K] . dequant(W)^T.
 * Streams every code and scale byte from HBM once per call for all N tokens
 * (the decode and batched-verify matvec of bw24 README, NVFP4 decode path, and
 * qwentin README, batched verify reading each weight once for the tree).
 * x        device bf16 bits [N][K]
 * codes, scales, tensor_scale: the NVFP4 weight W[M][K] (device)
 * y        device [N][M], fp32 (out_dtype NVFP4_OUT_F32) or bf16 bits
 *          (NVFP4_OUT_BF16, round-to-nearest-even of the fp32 result)
 * workspace device scratch of nvfp4_workspace_bytes(NVFP4_OP_GEMV_SKINNY, N, M, K),
 *          zero-filled before first use (see Workspace above): partial sums of
 *          rows whose K range is split across thread blocks, and their
 *          arrival counters.
 * Returns NVFP4_ERR_UNSUPPORTED_SHAPE for N outside 1..16. */
int nvfp4_gemv_skinny(const uint16_t *x, int64_t N,
                      const uint8_t *codes, const uint8_t *scales,
                      const float *tensor_scale, int64_t M, int64_t K,
                      void *y, int out_dtype,
                      void *workspace, size_t workspace_bytes, nvfp4_stream_t stream);

/* Fused gate/up projection with SwiGLU, any N >= 1:
 *   g = x . dequant(Wg)^T,  u = x . dequant(Wu)^T,  h = g / (1 + exp(-g)) * u,
 * reading both weight matrices once and never writing g or u to memory (the
 * persistent-MLP GEMV of qwentin README, section on SM120 kernels, fuses the
 * MLP chain).  N <= 16 runs the skinny kernel; larger N runs the tensor-core
 * prefill kernel with a SwiGLU epilogue.
 * Wg and Wu are both [M][K] NVFP4 tensors (device buffers as above), each with
 * its own tensor scale.  h is device [N][M] fp32 or bf16 bits.
 * workspace: nvfp4_workspace_bytes(NVFP4_OP_GATEUP_SWIGLU, N, M, K). */
int nvfp4_gateup_swiglu(const uint16_t *x, int64_t N,
                        const uint8_t *gate_codes, const uint8_t *gate_scales,
                        const float *gate_tensor_scale,
                        const uint8_t *up_codes, const uint8_t *up_scales,
                        const float *up_tensor_scale,
                        int64_t M, int64_t K,
                        void *h, int out_dtype,
                        void *workspace, size_t workspace_bytes, nvfp4_stream_t stream);

/* Prefill product for any N >= 1: y[N][M] = x[N][K] . dequant(W)^T on the
 * tensor cores (weights dequantised exactly to bf16 in shared memory, bf16 x
 * bf16 products accumulated in fp32): the wide GEMM of qwentin README, "How it
 * works" (the weight read once for N tokens), and the prefill GEMM of bw24
 * README, NVFP4 decode path.  N <= 16 is forwarded to the skinny kernel, so
 * there is one entry point per operation for all N.
 * Arguments as for nvfp4_gemv_skinny; workspace:
 * nvfp4_workspace_bytes(NVFP4_OP_GEMM_PREFILL, N, M, K). */
int nvfp4_gemm_prefill(const uint16_t *x, int64_t N,
                       const uint8_t *codes, const uint8_t *scales,
                       const float *tensor_scale, int64_t M, int64_t K,
                       void *y, int out_dtype,
                       void *workspace, size_t workspace_bytes, nvfp4_stream_t stream);

/* ---------------------------------------------------------------------------
 * Skinny product lists in one launch: the decode step of a stack of layers.
 *
 * A decode step multiplies every weight matrix of every layer by the same few
 * tokens; at N = 1 one matrix streams in a few microseconds, so per-launch
 * costs would dominate.  A list of products (jobs) runs as one persistent
 * launch in which every SM streams the weights of all jobs back to back (the
 * one-replay-per-token decode of bw24 README, CUDA-graph decode, and the
 * persistent MLP chain of qwentin README, "How it works").  A job's
 * activations are a caller buffer or the bf16 output of an earlier job of the
 * list, so a dependent chain (O -> gate/up + SwiGLU -> down -> next layer)
 * runs inside the launch: a job that reads an earlier output, and every job
 * after it, waits until all jobs before it are final.
 *
 * Results: each job's output is y = x . dequant(W)^T (or silu(g) * u), within
 * the accuracy bound of nvfp4_gemv_skinny; repeated runs of a plan give
 * bit-identical outputs.  The split of K across SMs follows the whole list,
 * so bits may differ from the same product made by nvfp4_gemv_skinny.
 * Requirements: N = 1..16 tokens for every job; K % 256 == 0.
 * ------------------------------------------------------------------------- */

/* One product of a list. */
typedef struct {
    const uint16_t *x;          /* device bf16 [N][x_ld] activations (input == -1) */
    int64_t x_ld;               /* elements between token rows of x; 0 means K (multiple of 8) */
    int32_t input;              /* -1: x as given; j >= 0: x is the output of job j of the list
                                   (j earlier than this job; that output must be bf16, with
                                   M >= this K and M % 8 == 0; token n's x is its row n) */
    int32_t n_weights;          /* 1: y = x . W^T;  2: y = silu(x . Wg^T) * (x . Wu^T) */
    const uint8_t *codes[2];    /* device NVFP4 weights [M][K/2] ([0] gate, [1] up) */
    const uint8_t *scales[2];   /* device E4M3 block scales [M][K/16] */
    const float *tensor_scale[2]; /* device fp32 tensor scales */
    int64_t M, K;
    void *y;                    /* device output [N][M], fp32 or bf16 bits */
    int32_t out_dtype;          /* NVFP4_OUT_F32 or NVFP4_OUT_BF16 */
    int32_t reserved;           /* set to 0 */
} nvfp4_skinny_job;

/* Device bytes of the plan of `jobs` (0 if the list is invalid).  Host only;
 * an upper bound that holds on any device. */
size_t nvfp4_stream_plan_bytes(const nvfp4_skinny_job *jobs, int n_jobs, int64_t N);

/* Build the plan of a job list for the current device in `plan` (device
 * memory of nvfp4_stream_plan_bytes bytes, 256-byte aligned, owned by the
 * caller): the jobs' tensor maps, the split of every job's work across the
 * SMs, and the run state, zero-filled.  Copies from the host and
 * synchronises `stream`, so build plans before any stream capture.  The
 * plan holds the device pointers of the jobs: their buffers must stay where
 * they are for as long as the plan is run.
 * Errors: NVFP4_ERR_INVALID_ARG (null, misaligned, bad enum, an input that is
 * not an earlier bf16 output wide enough), NVFP4_ERR_UNSUPPORTED_SHAPE (N
 * outside 1..16, K % 256 != 0), NVFP4_ERR_WORKSPACE (plan_bytes too small),
 * NVFP4_ERR_CUDA. */
int nvfp4_stream_plan(const nvfp4_skinny_job *jobs, int n_jobs, int64_t N,
                      void *plan, size_t plan_bytes, nvfp4_stream_t stream);

/* Run every job of a plan: one kernel launch, asynchronous on `stream`,
 * capturable in a CUDA graph.  Runs of one plan must be ordered on one
 * stream; the plan is its own workspace and keeps the device status word at
 * byte NVFP4_STATUS_WORD_OFFSET (read it with nvfp4_device_status(plan, ...)).
 * After a run whose bounded wait gave up, build the plan again before the
 * next run.  NVFP4_ERR_INVALID_ARG for a null or misaligned plan or
 * plan_bytes below 256; a plan built on a device with another SM count is
 * refused on the device (status word code 31). */
int nvfp4_stream_run(void *plan, size_t plan_bytes, nvfp4_stream_t stream);

/* ---------------------------------------------------------------------------
 * FP6 E2M3 block-scaled weights: the 6-bit weight tier the pages use for
 * quality (qwentin README, "Highlights" and "How it works": E2M3 weights with
 * 128-wide block scales on the block-scaled tensor-core MMA).  Same products,
 * same activations and outputs; only the weight format differs:
 *   codes   uint8 [M][3K/4]  each row a little-endian stream of 6-bit E2M3
 *                            codes (element k at bits 6k..6k+5 of the row, so
 *                            four codes fill three bytes).  E2M3: bit 5 sign,
 *                            bits 4..3 exponent (bias 1), bits 2..0 mantissa;
 *                            exponent 0 is subnormal (m/8); largest 7.5.
 *   scales  uint8 [M][K/128] one UE8M0 scale per 128 consecutive k of a row,
 *                            value 2^(s - 127).  No tensor scale.
 * K must be a multiple of 128.  weight = e2m3(code) * 2^(s - 127), exact in
 * bf16 for every scale byte up to 252 (all the quantiser produces); the
 * accuracy bound and determinism are those of the NVFP4 calls.
 * ------------------------------------------------------------------------- */

/* Quantise fp32 (or, _bf16, bf16-bit) weights to FP6 E2M3, block by block
 * (128 k of a row), in fp32:
 *   shared = floor(log2(block amax)) - 2, raised to -127 if lower (and -127
 *            for an all-zero block);  scale byte = shared + 127;
 *   code   = nearest E2M3 value to w / 2^shared, ties to the even code,
 *            magnitudes above 7.5 saturating to 7.5, the sign of w kept.
 * (the microscaling conversion rule of the mxf8f6f4 MMA kind, with 128-wide
 * blocks).  One pass, no workspace.  w device [M][K] row-major, finite;
 * codes / scales device outputs as above; all 16-byte aligned.
 * Returns NVFP4_ERR_UNSUPPORTED_SHAPE for K % 128 != 0. */
int nvfp4_fp6_quantize(const float *w, int64_t M, int64_t K,
                       uint8_t *codes, uint8_t *scales, nvfp4_stream_t stream);
int nvfp4_fp6_quantize_bf16(const uint16_t *w, int64_t M, int64_t K,
                            uint8_t *codes, uint8_t *scales, nvfp4_stream_t stream);

/* y[N][M] = x[N][K] . dequant(W)^T for FP6 weights, any N >= 1: N <= 16 runs
 * a skinny kernel that streams every weight byte once for all N tokens, larger
 * N the tensor-core prefill kernel (the same kernels as the NVFP4 calls, with
 * the FP6 dequantiser).  x, y, out_dtype as for nvfp4_gemv_skinny; workspace:
 * nvfp4_workspace_bytes(NVFP4_OP_FP6_GEMM, N, M, K), under the same contract
 * as the NVFP4 skinny calls (zero-filled before its first use; every call
 * leaves its split-K counters zero; it may be shared with them). */
int nvfp4_fp6_gemm(const uint16_t *x, int64_t N,
                   const uint8_t *codes, const uint8_t *scales, int64_t M, int64_t K,
                   void *y, int out_dtype,
                   void *workspace, size_t workspace_bytes, nvfp4_stream_t stream);

/* Fused gate/up + SwiGLU for FP6 weights, any N >= 1:
 * h = silu(x . Wg^T) * (x . Wu^T), g and u never written to memory.
 * workspace: nvfp4_workspace_bytes(NVFP4_OP_FP6_GATEUP_SWIGLU, N, M, K). */
int nvfp4_fp6_gateup_swiglu(const uint16_t *x, int64_t N,
                            const uint8_t *gate_codes, const uint8_t *gate_scales,
                            const uint8_t *up_codes, const uint8_t *up_scales,
                            int64_t M, int64_t K, void *h, int out_dtype,
                            void *workspace, size_t workspace_bytes, nvfp4_stream_t stream);

/* Skinny product without a caller workspace, for callers that cannot allocate
 * device memory.  The source pages have no counterpart for this call: it is an
 * addition of this library.  A plain C or Fortran host program with no
 * device allocator of its own, or a latency-critical loop that must not call
 * cudaMalloc (it synchronises the whole device), can use it.
 * Same arguments, checks and results as nvfp4_gemv_skinny (N = 1..16), except
 * that the split-K scratch is a fixed array of NVFP4_NOALLOC_SCRATCH_BYTES in
 * the library's own device memory, held by every GPU that loads the library
 * until the process exits.  Nothing is allocated or freed by the call.
 *   - Set-up: the first call on each device looks up the array's device
 *     address (cudaGetSymbolAddress) with that device current and caches it;
 *     make that first call before any stream capture.
 *   - Size limit: returns NVFP4_ERR_WORKSPACE, with nothing enqueued, when the
 *     problem needs more scratch than NVFP4_NOALLOC_SCRATCH_BYTES (that is,
 *     when nvfp4_workspace_bytes(NVFP4_OP_GEMV_SKINNY, N, M, K) exceeds it).
 *   - Set-up is repeated when the current CUDA context changes (after
 *     cudaDeviceReset, or from another context on the same device): the
 *     address is cached together with the context's id.
 *   - Sharing: every call on a device uses the same array.  It starts
 *     zero-filled and every call leaves its split-K counters at zero, as the
 *     skinny workspace contract requires.  Calls whose kernels overlap on the GPU
 *     (different streams without ordering) race on the array; order them on
 *     one stream.
 *   - Failures: the array holds the device status word and the split-K
 *     counters like any skinny workspace.  After a call whose bounded wait gave
 *     up (see nvfp4_device_status), the counters may be left set and later
 *     no-allocation calls on that device can return wrong sums: read the word
 *     with nvfp4_noalloc_status and clear it (which zero-fills the array)
 *     before the next call.
 * Arguments are checked exactly as by nvfp4_gemv_skinny, before the size
 * limit and before any CUDA call. */
#define NVFP4_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)

int nvfp4_gemv_skinny_noalloc(const uint16_t *x, int64_t N,
                              const uint8_t *codes, const uint8_t *scales,
                              const float *tensor_scale, int64_t M, int64_t K,
                              void *y, int out_dtype, nvfp4_stream_t stream);

/* Status of the no-allocation array on the current device, for callers that
 * cannot pass its address to nvfp4_device_status: synchronises `stream`,
 * stores the status word in *code (if not NULL) and returns NVFP4_OK when it
 * is zero, else NVFP4_ERR_DEVICE_TIMEOUT.  With clear != 0 and a nonzero word
 * the whole array is zero-filled on `stream` (cudaMemsetAsync), which resets
 * the word and any split-K counter a failed call left set.  Allocates nothing;
 * NVFP4_ERR_CUDA if a CUDA call fails.  The source pages have no counterpart. */
int nvfp4_noalloc_status(int clear, uint32_t *code, nvfp4_stream_t stream);

/* The failure-path self-test of nvfp4_selftest_wait_timeout run against the
 * no-allocation array of the current device: after 2 s it records code 127 in
 * the array's status word, which nvfp4_noalloc_status then reports.  Faults
 * nothing; allocates nothing.  The source pages have no counterpart. */
int nvfp4_noalloc_selftest_wait_timeout(nvfp4_stream_t stream);

/* Device-side failures.  The product calls keep a 32-bit status word at byte
 * NVFP4_STATUS_WORD_OFFSET of their workspace (every product workspace is at
 * least 256 bytes).  A tensor-core kernel (skinny with K % 256 == 0, prefill)
 * whose bounded pipeline wait runs out (2 s) stores a nonzero code there and
 * returns: 1..8 from the prefill kernel, 10 from its split-mode reduction
 * (a contributor or tile outside the plan, which the host's plan rules out),
 * 11..25 from the skinny kernel, 127 from nvfp4_selftest_wait_timeout.  No
 * kernel clears the word, so it reports
 * any failure since it was last cleared; it starts clean when the workspace is
 * zero-filled (required for the skinny calls; do it for a prefill workspace
 * too before reading its status).  A quantise call overwrites the word. */
#define NVFP4_STATUS_WORD_OFFSET 128

/* Read the status word of `workspace` (device, at least
 * NVFP4_STATUS_WORD_OFFSET + 4 bytes, 16-byte aligned) after the work enqueued
 * on `stream` so far: synchronises `stream`, stores the word in *code (if
 * code is not NULL) and returns NVFP4_OK when it is zero, else
 * NVFP4_ERR_DEVICE_TIMEOUT.  With clear != 0 a nonzero word is reset to zero
 * on `stream` afterwards.  NVFP4_ERR_INVALID_ARG for a null, misaligned or too
 * small workspace; NVFP4_ERR_CUDA if the copy or the synchronisation fails. */
int nvfp4_device_status(const void *workspace, size_t workspace_bytes, int clear, uint32_t *code,
                        nvfp4_stream_t stream);

/* Test of the failure path above: enqueues one thread that waits, with the
 * kernels' own bounded wait, on a barrier that nothing completes, so after
 * 2 s it records code 127 in the status word of `workspace` and exits.  It
 * faults nothing and computes nothing; the arguments are checked as for
 * nvfp4_device_status. */
int nvfp4_selftest_wait_timeout(void *workspace, size_t workspace_bytes, nvfp4_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_H */
