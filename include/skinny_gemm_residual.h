/*
 * skinny_gemm_residual.h -- C ABI of the GB300 (sm_103a) skinny BF16
 * projection GEMM with a fused residual add.
 *
 * Operation (vLLM "benchmark_k3_cutedsl_residual.py", module docstring and
 * its correctness() reference; shape constants N = 7168, K = 3584):
 *
 *     Y[m,n] = bf16( sum_k A[m,k] * W[n,k] + R[m,n] ),  0 <= m < M, 0 <= n < N
 *
 * with FP32 accumulation and a single round-to-nearest-even to BF16 in the
 * epilogue.  The vLLM "fused_add_multicast_skinny_gemm" page rounds the FP32
 * product to BF16 before adding the residual; this library rounds once.
 *
 * Types and layouts.  A, W, R, Y hold IEEE bfloat16 values, row-major with
 * unit inner stride:
 *     A  [M, K]  row stride lda >= K      (activations)
 *     W  [N, K]  row stride K (contiguous) (nn.Linear weight layout)
 *     R  [M, N]  row stride ldr >= N      (residual)
 *     Y  [M, N]  row stride ldy >= N      (output)
 * Strides are in elements.  The plain entry point uses lda = K, ldr = ldy = N.
 * The row-strided forms cover the case on the "fused_add_multicast_skinny_gemm"
 * page where the residual is a column slice of a wider [M, hidden_dim] buffer,
 * and a chain where the next layer's A is a column slice of this layer's Y.
 *
 * Ownership.  Every pointer is a DEVICE pointer owned by the caller and must
 * stay valid until the work queued on `stream` has finished.  The library keeps
 * no reference to them after the call returns.  A per-device workspace used by
 * the tensor-core split-K path is owned by the library, allocated once per
 * device by sgr_init() (or lazily on first use) and released at process exit.
 * Calls forced onto that path (SGR_PATH_TC) share it: such calls whose
 * kernels may overlap on the GPU (different streams, graphs replayed
 * concurrently) must be serialised by the caller.  The library's own choice
 * (SGR_PATH_AUTO) never takes that path, and every other path keeps no state
 * between calls.
 *
 * Asynchrony.  Calls enqueue work on `stream` (a cudaStream_t; NULL is the
 * legacy default stream) and return without synchronising.  Kernels launch
 * with programmatic dependent launch (PDL) unless SGR_FLAG_NO_PDL is given:
 * a kernel starts streaming W while the previous kernel on the stream is still
 * finishing, and reads A and R and writes Y only after that kernel completes.
 * Contract that follows: W must not be written by the kernel queued
 * immediately before on the same stream.  A and R may be.
 *
 * CUDA graphs.  Calls may be captured into a CUDA graph after sgr_init() has
 * run for the device (the first call does it otherwise, and that first call
 * must not be inside a capture).
 *
 * Errors.  Every entry point returns an sgr_status.  Argument errors are
 * detected on the host before anything is enqueued, so nothing runs and the
 * output is untouched:
 *   SGR_ERR_NULL        a required pointer is NULL
 *   SGR_ERR_SHAPE       M, N or K negative; N or K not a multiple of 8;
 *                       a row stride smaller than its row width
 *   SGR_ERR_ALIGN       a pointer not 16-byte aligned, or a row stride that is
 *                       not a multiple of 8 elements (16 bytes)
 *   SGR_ERR_ALIAS       Y overlaps A or W, or overlaps R other than being
 *                       exactly R (Y == R with ldy == ldr, an in-place residual
 *                       update, is allowed: each element of R is read before
 *                       the same thread writes it)
 *   SGR_ERR_UNSUPPORTED a size beyond the library's limits (M <= 2^20,
 *                       N <= 2^24, K <= 2^20, row strides <= 2^36 elements),
 *                       or a forced path/config that cannot run this shape
 *   SGR_ERR_LAUNCH      the CUDA launch itself failed (cudaGetLastError)
 *   SGR_ERR_DEVICE      no usable device, or device set-up failed
 * Empty problems (M == 0 or N == 0) return SGR_OK and enqueue nothing.  This
 * is deliberate, and a departure from the plain "M >= 1" contract: an empty
 * batch (a mixture-of-experts expert to which no token was routed, the last
 * empty slice of a split batch) is a valid request with nothing to compute,
 * so it is a no-op rather than an error.  Negative sizes are errors.
 * K == 0 makes the product an empty sum, so Y = R (a device copy).
 * Device-side waits are bounded (about one second); a wait that runs out
 * records a code readable with sgr_device_error() instead of hanging.
 */
#ifndef SKINNY_GEMM_RESIDUAL_H
#define SKINNY_GEMM_RESIDUAL_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SGR_ABI_VERSION 9

typedef enum {
  SGR_OK = 0,
  SGR_ERR_NULL = 1,
  SGR_ERR_SHAPE = 2,
  SGR_ERR_ALIGN = 3,
  SGR_ERR_ALIAS = 4,
  SGR_ERR_UNSUPPORTED = 5,
  SGR_ERR_LAUNCH = 6,
  SGR_ERR_DEVICE = 7
} sgr_status;

/* Flags for the _ex / _config entry points. */
#define SGR_FLAG_NO_PDL 0x1u /* launch without programmatic dependent launch */

/* Kernel paths. */
#define SGR_PATH_AUTO 0 /* per-M table */
#define SGR_PATH_SIMT 1 /* CUDA-core streaming kernel, M <= 16 */
#define SGR_PATH_TC 2      /* tcgen05 kernel, persistent stream-K with split-K fixup */
#define SGR_PATH_TC_ROWS 3 /* tcgen05 kernel, one contiguous W row slab per CTA (M <= 256) */
#define SGR_PATH_TILE 4    /* tcgen05 kernel, 128-token x tile_n output tiles (large M) */
#define SGR_PATH_W8 5      /* tcgen05 row-slab kernel for low-bit weights, widened on chip (skinny_gemm_residual_w8
                              and _w4 only, M <= 256); both also take SGR_PATH_SIMT (CUDA-core kernel) */
#define SGR_PATH_PAIR 6    /* tcgen05 tile kernel on 2-CTA clusters (cta_group::2), 256-token x tile_n tiles (large M) */
#define SGR_PATH_W8S 7     /* FP8 weights on the FP8 tensor-core path (kind::f8f6f4), activations split exactly into
                              two E4M3 parts (skinny_gemm_residual_w8 only, M <= 16) */

/*
 * Y = bf16(A . W^T + R) with contiguous operands (lda = K, ldr = ldy = N).
 * The operation of the vLLM "benchmark_k3_cutedsl_residual.py" page
 * (module docstring), at any M >= 0 and N, K multiples of 8.
 * `stream` is a cudaStream_t.  Returns an sgr_status.
 */
int skinny_gemm_residual(const void* A, const void* W, const void* R, void* Y,
                         int M, int N, int K, void* stream);

/*
 * Same operation with row strides (elements) for A, R and Y and launch flags
 * (SGR_FLAG_*).  Row-strided residual as on the vLLM
 * "fused_add_multicast_skinny_gemm" page (its shared_shard operand has row
 * stride hidden_dim).  Returns an sgr_status.
 */
int skinny_gemm_residual_ex(const void* A, int64_t lda, const void* W,
                            const void* R, int64_t ldr, void* Y, int64_t ldy,
                            int M, int N, int K, unsigned flags, void* stream);

/*
 * Launch configuration, the analogue of the Config(block_size,
 * outputs_per_block, k_unroll, vector_width) record that the
 * "benchmark_k3_cutedsl_residual.py" page sweeps.  Zero in any field means
 * "the library's choice for this M".
 */
typedef struct {
  int path;               /* SGR_PATH_* */
  int ctas_per_sm;        /* persistent grid = SM count x ctas_per_sm */
  int stages;             /* shared-memory ring depth */
  int rows_per_stage;     /* SIMT: W rows per ring stage */
  int k_blocks_per_stage; /* TC, TC_ROWS, TILE, PAIR: 64-wide K blocks per ring stage */
  int token_tile;         /* TC, TC_ROWS: activation rows per MMA (multiple of 16, <= 256) */
  int prefetch_stages;    /* TC_ROWS, TILE, PAIR: weight stages requested before the dependency wait */
  int tile_n;             /* TILE: W rows per output tile (MMA N): 64, 128, 192 or 256;
                             PAIR: W rows per 256-token tile: 64, 96, 128, 192 or 256 */
  int k_split;            /* TILE: 1, or S = 2, 3, 4 = K split over an S-CTA cluster (one tile per cluster, all
                             clusters resident at once); tile_n 64/128/192 for S = 2, 192 for 3, 128/192/256 for 4;
                             TC_ROWS: 0 or 1, or 2 = each W slab on a 2-CTA cluster, one CTA per half of K, the
                             partial sums added in the epilogue through distributed shared memory (token tiles of
                             16-64 with at most two K blocks per MMA) */
  int reserved[2];        /* must be zero */
} sgr_config;

/*
 * As skinny_gemm_residual_ex with an explicit configuration (for sweeps and
 * tests).  A configuration that cannot run the shape returns
 * SGR_ERR_UNSUPPORTED without launching.  `cfg` may be NULL (library choice).
 */
int skinny_gemm_residual_config(const void* A, int64_t lda, const void* W,
                                const void* R, int64_t ldr, void* Y, int64_t ldy,
                                int M, int N, int K, const sgr_config* cfg,
                                unsigned flags, void* stream);

/*
 * Host-only argument check with exactly the rules the entry points apply.
 * Never touches the GPU or dereferences a pointer.  Returns an sgr_status.
 */
int sgr_validate(const void* A, int64_t lda, const void* W, const void* R,
                 int64_t ldr, const void* Y, int64_t ldy, int M, int N, int K);

/*
 * Kernel path the library chooses for this shape with SGR_PATH_AUTO
 * (SGR_PATH_SIMT, SGR_PATH_TC, SGR_PATH_TC_ROWS, SGR_PATH_TILE or SGR_PATH_PAIR), or a negative sgr_status
 * if none can run it.  Host-only.
 */
int sgr_select_path(int M, int N, int K);

/*
 * The configuration the library uses for this shape on the given path
 * (SGR_PATH_AUTO resolves first; SGR_PATH_W8 gives the FP8-weight kernel's).  Writes *cfg.  Host-only apart from a
 * device-attribute query for the SM count of `device`.  Returns an sgr_status.
 */
int sgr_default_config(int device, int M, int N, int K, int path, sgr_config* cfg);

/*
 * One-time per-device set-up: SM count, kernel attributes, split-K workspace
 * and counters, device error word.  Idempotent and thread-safe.  Call before
 * capturing calls into a CUDA graph.  Returns an sgr_status.
 */
int sgr_init(int device);

/*
 * Read (and with clear != 0, reset) the device error word of `device`, which
 * a kernel sets when one of its bounded waits runs out (0 = no error).
 * Synchronises with the device.  Allocates no device memory and does not run
 * sgr_init(), so callers of skinny_gemm_residual_noalloc can use it too.
 * Returns an sgr_status.
 */
int sgr_device_error(int device, unsigned* code, int clear);

/*
 * Resource usage of the kernel the library would launch for (path, M, K):
 * registers per thread, local (spill) bytes per thread, dynamic shared
 * memory per CTA and threads per CTA.  Like the register/spill query on the
 * "benchmark_k3_cutedsl_residual.py" page (resource_usage).  Host query.
 */
int sgr_kernel_resources(int device, int path, int M, int N, int K, int* regs,
                         int* local_bytes, int* smem_bytes, int* threads);

/* Static text for an sgr_status value. */
const char* sgr_status_string(int status);

/* SGR_ABI_VERSION of the built library; bindings compare it with their own. */
int sgr_abi_version(void);

/*
 * Allocation-free variant (no counterpart on the pages; added for callers
 * that must not allocate device memory).  Same operation, arguments and
 * errors as skinny_gemm_residual_ex, computed by the stream-K
 * tensor-core kernel, with its split-K scratch taken from a fixed array
 * inside this library instead of the workspace that sgr_init() allocates.
 * Who needs it: code that runs while a stream is being captured in a mode
 * that forbids cudaMalloc, engines that reserve all device memory up front
 * and allow no further allocation, and callers on latency-critical paths that
 * cannot risk the implicit device synchronisation an allocation may cause.
 * This entry point calls no cudaMalloc, cudaFree or allocating library
 * routine; sgr_init() is not needed and is not called.
 *
 * Limits: the scratch array is 16 KiB of tile counters plus 4 MiB of FP32
 * partial tiles, held by every GPU that loads the library until the process
 * exits.  A shape needing more (more than 4096 output tiles of 128 W rows x
 * one token tile, or more than 4 MiB of partials, which is grid x 2 x token
 * tile x 128 floats; in practice M above 16 on a 152-SM GPU) returns
 * SGR_ERR_UNSUPPORTED without launching.
 *
 * The first call on a device resolves the array's device address (with that
 * device current) and sets kernel attributes; make that first call before
 * any stream capture.  Every call on a device shares the one array: it clears
 * the counters it uses with a cudaMemsetAsync on `stream` before its kernel
 * runs, and calls whose work may overlap on the GPU (different streams, or
 * graphs replayed concurrently) race on the array and must be serialised by
 * the caller.  Because of that memset, the kernel of this call does not
 * start early under programmatic dependent launch: it runs after the
 * preceding work on `stream` has finished (W may therefore be written by
 * that work, unlike with skinny_gemm_residual_ex).  sgr_device_error() reads
 * the error word without allocating.
 */
int skinny_gemm_residual_noalloc(const void* A, int64_t lda, const void* W,
                                 const void* R, int64_t ldr, void* Y, int64_t ldy,
                                 int M, int N, int K, unsigned flags, void* stream);

/*
 * One problem of a grouped call (an expert of a mixture-of-experts layer):
 * its activations A [M, K] (row stride lda), weights W [N, K] (contiguous),
 * residual R and output Y [M, N] (row strides ldr, ldy), all device pointers
 * owned by the caller with the same rules as skinny_gemm_residual_ex.
 * M = 0 (no token routed to this expert) is allowed and skipped: its W is not
 * read.
 */
typedef struct {
  const void* A;
  int64_t lda;
  const void* W;
  const void* R;
  int64_t ldr;
  void* Y;
  int64_t ldy;
  int M;
  int reserved; /* must be zero */
} sgr_group;

/*
 * Y_g = bf16(A_g . W_g^T + R_g) for every group g, all with the same N and K,
 * in one kernel launch (per 32 groups with M > 0): the grouped expert GEMM of
 * the bitsandbytes "QLORA-2" comparison page (QLORA_GUIDE.md, "Grouped Expert
 * GEMM": all active experts batched into one launch so that the SMs stay
 * busy), here for BF16 weights on the row-slab kernel.  Each group's M must
 * be at most 256 (decode-sized expert batches); the launch configuration is
 * the library's choice for the largest M (or `cfg`, path SGR_PATH_AUTO or
 * SGR_PATH_TC_ROWS).  Errors as for skinny_gemm_residual_ex, checked for
 * every group before anything is enqueued; in addition SGR_ERR_ALIAS when a
 * group's Y overlaps another group's A, W, R or Y, and SGR_ERR_UNSUPPORTED for
 * num_groups < 0 or a group with M > 256.  `groups` is a host array read
 * during the call only.  Returns an sgr_status.
 */
int skinny_gemm_residual_grouped(const sgr_group* groups, int num_groups, int N, int K,
                                 const sgr_config* cfg, unsigned flags, void* stream);

/*
 * Low-bit weight variant: FP8 E4M3 weights with one FP32 scale per output
 * column, BF16 activations, residual and output:
 *
 *     Y[m,n] = bf16( scale[n] * sum_k A[m,k] * e4m3(Wq[n,k]) + R[m,n] )
 *
 * with FP32 accumulation and one round-to-nearest-even, the quantized-weight
 * decode kernel direction of the bitsandbytes "QLORA-2" page ("Three-Kernel
 * Strategy": weights stored in few bits, 16-bit activations, the scale
 * applied to the dot product; here per output column).  E4M3 is the OCP 8-bit
 * format (sign, 4 exponent bits with bias 7, 3 fraction bits, subnormals, no
 * infinities; the value of torch.float8_e4m3fn).  The weight bytes read per
 * call are half those of the BF16 entry points.
 *
 *     A      [M, K]  BF16, row stride lda >= K (elements, multiple of 8)
 *     Wq     [N, K]  E4M3 codes (one byte each), row stride ldw >= K bytes,
 *                    a multiple of 16; the codes 0x7F and 0xFF (NaN) must not
 *                    occur (their result is unspecified; quantisers that
 *                    saturate never write them)
 *     scale  [N]     FP32, 4-byte aligned
 *     R, Y   [M, N]  BF16, row strides ldr, ldy >= N (multiples of 8)
 *
 * M <= 256 (decode-sized batches), N and K multiples of 8.  Device pointers,
 * ownership, asynchrony, PDL (Wq and scale are read before the dependency
 * wait, like W), graph capture and errors as for skinny_gemm_residual_ex; in
 * addition SGR_ERR_ALIGN for ldw not a multiple of 16 or a misaligned scale,
 * and SGR_ERR_ALIAS when Y overlaps Wq or scale.  `cfg` may be NULL (library
 * choice).  Two kernels: SGR_PATH_W8, the tensor-core row-slab kernel (any
 * M <= 256; cfg may set stages = depth of the weight-code ring 2..16,
 * prefetch_stages = depth of the activation ring 2..8, k_blocks_per_stage =
 * 64-wide K blocks per stage, even, 2..8, token_tile, and rows_per_stage = W
 * rows per CTA, a multiple of 8 up to 128), and SGR_PATH_SIMT, the CUDA-core
 * kernel (M <= 8, contiguous code rows ldw == K, K a multiple of 16; cfg may
 * set ctas_per_sm, rows_per_stage = code rows per ring stage, stages), and
 * SGR_PATH_W8S, the FP8 tensor-core kernel (M <= 16 and the split activation
 * operand of all of K in shared memory: K <= 3584 for 9-16 tokens, 7168 for
 * up to 8; cfg may set stages 2..8, k_blocks_per_stage = 128-code K blocks
 * per stage 1..8, token_tile 8 or 16, rows_per_stage).  SGR_PATH_W8S feeds
 * the codes to the tensor core unchanged and brings the activations into
 * E4M3 instead: each token row is scaled by a power of two that puts its
 * largest magnitude in [128, 256), and each scaled value b is held as
 * hi + lo/16 with hi = e4m3(b), lo = e4m3(16 (b - hi)).  That is exact for
 * every activation within 2^13 of its row's largest magnitude; smaller ones
 * are represented with an absolute error below 2^-21 times that magnitude
 * (so a row whose values span more than 2^13 can differ from the exact
 * result by up to sum_k |scale[n] e4m3(Wq[n,k])| * 2^-21 * max_k |A[m,k]|).
 * SGR_PATH_AUTO takes SGR_PATH_W8S for M <= 8 where it can run, else the
 * CUDA-core kernel for M = 1 where it can run, else the tensor-core row-slab
 * kernel.  Returns an sgr_status.
 */
int skinny_gemm_residual_w8(const void* A, int64_t lda, const void* Wq, int64_t ldw,
                            const float* scale, const void* R, int64_t ldr, void* Y,
                            int64_t ldy, int M, int N, int K, const sgr_config* cfg,
                            unsigned flags, void* stream);

/* Host-only argument check of skinny_gemm_residual_w8 (its exact rules). */
int sgr_validate_w8(const void* A, int64_t lda, const void* Wq, int64_t ldw,
                    const float* scale, const void* R, int64_t ldr, const void* Y,
                    int64_t ldy, int M, int N, int K);

/*
 * NVFP4 weights:
 *
 *     Y[m,n] = bf16( gs * sum_k A[m,k] * e2m1(Wq4[n,k]) * e4m3(bs[n,k/16]) + R[m,n] )
 *
 * with FP32 accumulation and one round-to-nearest-even: the NVFP4 weight
 * format the bitsandbytes "QLORA-2" page builds GEMM targets for (its
 * CMakeLists NVFP4 sm100 entries), read as the published layout: 4-bit E2M1
 * codes (OCP MX FP4: sign, 2 exponent bits with bias 1, 1 fraction bit;
 * magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6), two per byte with element 2i in the
 * low nibble, one E4M3 scale per 16 consecutive elements of a row, and one
 * FP32 scale gs for the whole tensor.  The weight bytes read per call are a
 * quarter of the BF16 entry points' plus the block scales (1/16 of them).
 *
 *     A      [M, K]          BF16, row stride lda >= K (elements, multiple of 8)
 *     Wq4    [N, K/2]        bytes of two E2M1 codes, row stride ldw >= K/2 bytes, a multiple of 16
 *     bs     [N, ceil(K/16)] E4M3 block scales (one byte each, no NaN code), row stride ldbs bytes, a
 *                            multiple of 16 and >= ceil(K/16) rounded up to 16: each row is read in
 *                            16-byte units, padding included, so the buffer must hold that many bytes
 *                            from the start of every row (the last row too)
 *     gs     FP32 tensor scale (by value)
 *     R, Y   [M, N]          BF16, row strides ldr, ldy >= N (multiples of 8)
 *
 * M <= 256 (decode-sized batches), N and K multiples of 8.  Device pointers,
 * ownership, asynchrony, PDL (Wq4 and bs are read before the dependency
 * wait, like W), graph capture and errors as for skinny_gemm_residual_ex; in
 * addition SGR_ERR_ALIGN for ldw or ldbs not a multiple of 16 or a
 * misaligned Wq4 or bs, and SGR_ERR_ALIAS when Y overlaps Wq4 or bs.  `cfg`
 * may be NULL (library choice).  Two kernels, both exact in the conversion
 * (a code times its block scale has at most 6 significant bits and lies in
 * [2^-10, 2688], so FP16 and BF16 hold it exactly) and accumulating in FP32:
 * SGR_PATH_W8, the tensor-core row-slab kernel (one launch per 128 tokens;
 * the codes are converted to BF16 times their block scale on chip and fed to
 * BF16 MMAs from tensor memory; cfg may set stages = depth of the code ring
 * 2..16, prefetch_stages = depth of the activation ring 2..8,
 * k_blocks_per_stage = 64-wide K blocks per stage, 4 or 8, token_tile, and
 * rows_per_stage = W rows per CTA), and SGR_PATH_SIMT, the CUDA-core kernel
 * (K a multiple of 32 and at most 7168; 4 token rows per pass, ceil(M/4)
 * passes, each streaming the weights; cfg may set ctas_per_sm,
 * rows_per_stage = weight rows per ring stage, stages).  SGR_PATH_AUTO takes
 * the CUDA-core kernel for M = 1 where it can run, else the tensor-core
 * kernel.  The epilogue computes fmaf(sum, gs, R) and rounds once.  Returns
 * an sgr_status.
 */
int skinny_gemm_residual_w4(const void* A, int64_t lda, const void* Wq4, int64_t ldw,
                            const void* bs, int64_t ldbs, float gs, const void* R, int64_t ldr,
                            void* Y, int64_t ldy, int M, int N, int K, const sgr_config* cfg,
                            unsigned flags, void* stream);

/* Host-only argument check of skinny_gemm_residual_w4 (its exact rules). */
int sgr_validate_w4(const void* A, int64_t lda, const void* Wq4, int64_t ldw, const void* bs,
                    int64_t ldbs, const void* R, int64_t ldr, const void* Y, int64_t ldy,
                    int M, int N, int K);

/*
 * Self-test of the failure path of the kernels' bounded waits: on the
 * current device, one thread waits on an mbarrier that nothing arrives on,
 * gives up after limit_us microseconds (1..100000) of the GPU's global timer
 * and records the timeout in the device error word, as a kernel's wait does
 * after its one-second limit.  The call clears the word, runs the wait,
 * synchronises, writes the recorded code to *code (1 = a consumer gave up
 * waiting for its data) and clears the word again.  Nothing faults or hangs
 * and the context stays usable.  Returns an sgr_status.
 */
int sgr_selftest_wait_timeout(unsigned limit_us, unsigned* code);

/*
 * Self-test of the stream-K kernel's abort path (SGR_PATH_TC): one launch on
 * the current device and the legacy default stream with contiguous operands
 * (as skinny_gemm_residual), in which CTA `cta` of the persistent grid acts
 * as if its first wait for an accumulator had run out.  That CTA records
 * code 3 in the device error word, stops its copy and MMA threads at their
 * next wait, and still arrives on the split-K tile counters of its segments
 * without contributing partial sums, so that every counter is back at zero
 * when the kernel ends.  Y is unspecified afterwards.  The call clears the
 * error word, launches, synchronises the device, writes the recorded code to
 * *code and clears the word again.  Nothing faults or hangs.  Errors as for
 * skinny_gemm_residual; SGR_ERR_UNSUPPORTED when `cta` is negative or not
 * below the grid size.  Returns an sgr_status.
 */
int sgr_selftest_streamk_abort(const void* A, const void* W, const void* R, void* Y, int M, int N, int K,
                               int cta, unsigned* code);

#ifdef __cplusplus
}
#endif

#endif /* SKINNY_GEMM_RESIDUAL_H */
