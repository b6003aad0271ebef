/*
 * gated_act.h -- C ABI of the GB300 (sm_103a) fused gated-activation library.
 *
 * Fused activations over bf16 rows, each one kernel launch.  The two the
 * library is built around:
 *
 *   gelu_and_mul_sparse  Gemma3n's sparse GELU gate.  vLLM PR "[Performance]
 *       Add Triton kernel for Gemma3n sparse GELU", section "Purpose" (the
 *       fused stages: row statistics, a threshold set from them, the tanh form
 *       of GELU, the product with the up half).  For each row with gate
 *       g = columns [0, d) and up u = columns [d, 2d):
 *           mean   = sum_j g_j / d                    (fp32 accumulation)
 *           std    = sqrt(sum_j (g_j - mean)^2 / d)   (population std)
 *           cutoff = mean + std * z,   z = inverse normal CDF of the target
 *                                      sparsity (0.95 -> 1.6448536269514722)
 *           out_j  = gelu_tanh(max(g_j - cutoff, 0)) * u_j
 *           gelu_tanh(x) = 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)))
 *       computed in fp32 and rounded once to bf16 (nearest even).
 *
 *   silu_and_mul  the MoE expert activation of Megatron-LM PR "Size MoE
 *       activation kernel grid to the row count", section "What changed and
 *       why": out_j = silu(g_j) * u_j, silu(x) = x / (1 + exp(-x)), fp32 math,
 *       bf16 out.
 *
 * Conventions shared by every entry point
 *   - bf16 means 2-byte IEEE bfloat16 storage.  Pointers are owned by the
 *     caller and address memory the current device can read and write:
 *     device (or managed) memory, or page-locked host memory (cudaHostAlloc /
 *     cudaHostRegister).  Host buffers are read and written by the kernels in
 *     place, over the CPU-GPU link, with no separate copy (the bulk-copy
 *     geometries, tma rows and pipe rows, are then not used).  An address
 *     the CUDA runtime does not know -- pageable host memory, or no
 *     allocation at all -- gives GATED_ACT_ERR_HOST, and device memory of
 *     another GPU than the current one gives GATED_ACT_ERR_DEVICE, both with
 *     nothing launched.
 *     The activations allocate no memory, never synchronize the host and
 *     launch only on `stream` (0 = the legacy default stream), so every call
 *     is asynchronous and can be captured in a CUDA graph.  The library keeps
 *     three pieces of device state per GPU, all in its own static device
 *     memory: a status word that the bulk-copy kernels set when a bounded
 *     wait gives up (gated_act_device_status), the 256-byte scratch array of
 *     gelu_and_mul_sparse_ws_static, and the native mode's 64 KB tables (see
 *     gelu_and_mul_sparse_native).  No other device state outlives a call.
 *   - The launch geometry depends only on the arguments, the pointers'
 *     alignment and the device's SM count.
 *   - 16-byte vector paths are taken when `in`, `out`, the row stride and d
 *     allow 16-byte aligned rows (pointers 16-byte aligned, row_stride and d
 *     multiples of 8); any other layout runs the scalar path -- slower, same
 *     results -- never an error.
 *   - Return value: GATED_ACT_OK (0) or a negative gated_act_status.  A
 *     negative value other than GATED_ACT_ERR_CUDA means nothing was launched.
 *     A zero-row call (T == 0 or M == 0) launches nothing and returns 0.
 *   - NaN/Inf follow IEEE arithmetic: a NaN anywhere in a gate row makes that
 *     whole output row NaN (it reaches the mean); a NaN in up stays in its
 *     element.
 */
#ifndef GATED_ACT_H
#define GATED_ACT_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gated_act_status {
    GATED_ACT_OK = 0,
    GATED_ACT_ERR_NULL = -1,       /* null in/out with a non-empty problem       */
    GATED_ACT_ERR_SIZE = -2,       /* T or M < 0, or d <= 0                      */
    GATED_ACT_ERR_STRIDE = -3,     /* row_stride < 2 d                           */
    GATED_ACT_ERR_TOO_LARGE = -4,  /* d > 2^30 or a byte range overflows int64   */
    GATED_ACT_ERR_OVERLAP = -5,    /* the bytes out writes overlap the bytes in reads */
    GATED_ACT_ERR_VARIANT = -6,    /* a forced variant/cluster size does not fit the call */
    GATED_ACT_ERR_CUDA = -7,       /* the CUDA runtime reported an error at launch */
    GATED_ACT_ERR_ALIGN = -8,      /* a pointer is not aligned to its element size */
    GATED_ACT_ERR_DTYPE = -9,      /* unknown element type                        */
    GATED_ACT_ERR_HOST = -10,      /* memory the CUDA runtime does not know       */
    GATED_ACT_ERR_SCRATCH = -11,   /* more scratch than the static array holds    */
    GATED_ACT_ERR_DEVICE = -12     /* device memory of a GPU other than the current one */
} gated_act_status;

/* Element types of the typed entry point (in and out share one type). */
typedef enum gated_act_dtype {
    GATED_ACT_BF16 = 0,
    GATED_ACT_F16 = 1,
    GATED_ACT_F32 = 2
} gated_act_dtype;

/*
 * gelu_and_mul_sparse -- fused sparse GELU gate (definition above).
 *   out        [T, d] bf16, contiguous (row r at out + r*d).  Written only.
 *   in         [T, row_stride] bf16; row r: gate = in[r*row_stride + j],
 *              up = in[r*row_stride + d + j], j in [0, d).  Columns past 2d
 *              are never read.  Read only; must not overlap out.
 *   T          rows, >= 0.       d  gate/up width, >= 1.
 *   row_stride elements between consecutive input rows, >= 2d.
 *   z          threshold in standard deviations (applied in fp32).
 *   stream     CUDA stream to launch on.
 * Accuracy (against an fp64 evaluation of the definition): every element
 * within 1e-2 |ref| + 2e-3; the zero pattern equals {g > cutoff} except where
 * |g - cutoff| < 1e-3 std.  A row whose gate is constant gives exact zeros
 * for d <= 65536 (its fp32 sum is exact).
 */
int gelu_and_mul_sparse(void *out, const void *in, int64_t T, int64_t d,
                        int64_t row_stride, double z, cudaStream_t stream);

/*
 * silu_and_mul -- out = silu(gate) * up, elementwise.
 *   out  [M, d] bf16 contiguous, written only.
 *   in   [M, 2d] bf16 contiguous: gate = columns [0, d), up = [d, 2d).
 *   M    rows, >= 0.   d >= 1.
 * Accuracy: within one bf16 ulp of the correctly rounded result.
 */
int silu_and_mul(void *out, const void *in, int64_t M, int64_t d,
                 cudaStream_t stream);

/*
 * Launch one empty kernel on `stream` with the same launch attributes as the
 * activations (programmatic stream serialization, waiting for the preceding
 * grid like they do).  For measuring launch overhead; no other effect.
 */
int gated_act_noop(cudaStream_t stream);

/*
 * Launch mode.  Every kernel is launched with programmatic stream
 * serialization: it waits for the preceding grid in `stream` to complete and
 * its writes to be visible before touching memory, and lets the next such
 * launch in the stream begin early, so launch latency overlaps the previous
 * kernel's tail.  Setting the environment variable GATED_ACT_PDL=0 before the
 * first launch turns the attribute off (plain stream order).
 */

/*
 * silu_and_mul_bounded -- silu_and_mul over the live rows only.
 * Megatron-LM PR "Size MoE activation kernel grid to the row count", section
 * "What changed and why": under CUDA graphs the grid is fixed by the
 * capture-time bound M while the number of live MoE rows changes per step;
 * the live count is read on the device, and CTAs past it exit early.
 *   out, in, M, d  as silu_and_mul (M is the buffer bound).
 *   n_rows         DEVICE pointer to one int32, the live row count, read by
 *                  the kernel after the preceding work in `stream`; clamped to
 *                  [0, M].  Output rows >= the live count are not written.
 * The launch depends only on M and d, so one capture serves every count.
 */
int silu_and_mul_bounded(void *out, const void *in, int64_t M, int64_t d,
                         const int32_t *n_rows, cudaStream_t stream);

/*
 * gelu_and_mul -- the dense form of the sparse-GELU activation (no
 * threshold): out = gelu_tanh(gate) * up, fp32 math, bf16 out.
 *   out  [T, d] bf16 contiguous;  in [T, row_stride] bf16, gate = [0, d),
 *   up = [d, 2d), row_stride >= 2d.
 * Accuracy: within one bf16 ulp of the correctly rounded result.
 */
int gelu_and_mul(void *out, const void *in, int64_t T, int64_t d,
                 int64_t row_stride, cudaStream_t stream);

/*
 * squared_relu -- out = max(x, 0)^2 elementwise, not gated (the sibling MoE
 * activation in Megatron-LM PR "Size MoE activation kernel grid to the row
 * count", section "Scope and risks").
 *   out [M, d] bf16 contiguous;  in [M, d] bf16 contiguous; no overlap.
 * Exact: x^2 of a bf16 value is exact in fp32, so the output is the correctly
 * rounded bf16 of max(x, 0)^2.
 */
int squared_relu(void *out, const void *in, int64_t M, int64_t d,
                 cudaStream_t stream);

/* Human-readable text for a status code (static storage; never NULL). */
const char *gated_act_status_string(int status);

/* The cudaError_t behind the calling thread's last GATED_ACT_ERR_CUDA (0 if none). */
int gated_act_last_cuda_error(void);

/*
 * Device-side status of the library's kernels on the current device since
 * the last call, then cleared.  *flags bit 0: a kernel's bounded wait (1 s)
 * for one of its own bulk copies gave up; the rows that CTA had not finished
 * were left unwritten.  No other bit is used.  Synchronizes the device
 * (it copies a status word), so call it outside stream capture.
 */
int gated_act_device_status(unsigned int *flags);

/* ------------------------------------------------------------------------
 * Launch-geometry control, for tests and measurements.
 *
 * gelu_and_mul_sparse picks one of these geometries; the choice never changes
 * the definition, only the fp32 summation order (results agree within the
 * accuracy bound above; rows with the same geometry agree bitwise).
 * ------------------------------------------------------------------------ */
typedef enum gated_act_variant {
    GATED_ACT_VARIANT_AUTO = 0,      /* the library's own choice                   */
    GATED_ACT_VARIANT_WARP_ROWS = 1, /* one warp per row, several rows per CTA     */
    GATED_ACT_VARIANT_CTA_ROW = 2,   /* one CTA, or a cluster of CTAs, per row;
                                        row held in registers                       */
    GATED_ACT_VARIANT_SCALAR = 3,    /* any layout: one CTA per row, 2-byte loads   */
    GATED_ACT_VARIANT_TMA_ROWS = 4,  /* persistent CTAs; gate/up half-rows stream
                                        through shared memory by bulk copy          */
    GATED_ACT_VARIANT_PIPE_ROWS = 5, /* as TMA_ROWS, with one producer lane that
                                        issues the copies and picks rows while the
                                        other warps finish rows                      */
    GATED_ACT_VARIANT_SPLIT_ROWS = 6 /* a few wide rows: C = 2, 4 or 8 independent
                                        CTAs per row, each reading the whole gate
                                        half-row for the statistics and finishing
                                        1/C of the columns (device memory, rows of
                                        up to 4096 16-byte vectors)                 */
} gated_act_variant;

typedef struct gated_act_plan {
    int32_t variant;        /* gated_act_variant actually used                */
    int32_t cluster;        /* CTAs that share one row (1 = none): a cluster in
                               CTA_ROW, independent CTAs in SPLIT_ROWS          */
    int32_t threads;        /* threads per CTA                                 */
    int32_t vec_per_thread; /* 16-byte vectors of gate per thread (0: scalar)  */
    int32_t rows_per_cta;   /* rows one CTA handles at a time                  */
    int32_t stages;         /* shared-memory slots per CTA (TMA and pipe
                               rows), else 0                                   */
    int32_t ctas_per_sm;    /* resident CTAs per SM the grid is sized for
                               (TMA and pipe rows), else 0                     */
    int32_t dynamic_rows;   /* 1: with a workspace (gelu_and_mul_sparse_ws)
                               the bulk-copy CTAs take rows from an atomic
                               counter; 0: rows are assigned round-robin    */
    int64_t grid;           /* CTAs launched                                   */
    int64_t smem_bytes;     /* dynamic shared memory per CTA                   */
} gated_act_plan;

/*
 * Describe the launch gelu_and_mul_sparse(_ex, _typed) would make, without
 * launching.  dtype a gated_act_dtype; variant/cluster as in
 * gelu_and_mul_sparse_ex.  out/in are never dereferenced: they are inspected
 * for alignment, and classified with cudaPointerGetAttributes (page-locked
 * host memory rules out the bulk-copy geometry; a pointer the runtime cannot
 * classify, or 0 for out, plans as device memory).  sm_count > 0 plans for a
 * device with that many SMs; sm_count <= 0 queries the current device.
 * Returns 0 and fills *plan, or a negative status (GATED_ACT_ERR_VARIANT when
 * the forced geometry does not fit).
 */
int gelu_and_mul_sparse_plan(const void *out, const void *in, int64_t T,
                             int64_t d, int64_t row_stride, int dtype,
                             int variant, int cluster, int sm_count,
                             gated_act_plan *plan);

/*
 * gelu_and_mul_sparse_plan for either kind of call: with_workspace = 0 the
 * plain call (as gelu_and_mul_sparse_plan), nonzero a call with a workspace
 * (gelu_and_mul_sparse_ws or gelu_and_mul_sparse_ws_static), whose automatic
 * choice may differ (see "Dynamic rows" below).
 */
int gelu_and_mul_sparse_plan_ex(const void *out, const void *in, int64_t T,
                                int64_t d, int64_t row_stride, int dtype,
                                int variant, int cluster, int sm_count,
                                int with_workspace, gated_act_plan *plan);

/*
 * gelu_and_mul_sparse with a forced geometry.
 *   variant  a gated_act_variant; AUTO behaves like gelu_and_mul_sparse.
 *            TMA_ROWS and PIPE_ROWS need the 16-byte layout and d <= 32768;
 *            the first launch of such a kernel shape on a device raises that
 *            kernel's shared-memory limit (cudaFuncSetAttribute), so make one
 *            call per device before capturing such launches in a graph.
 *   cluster  for GATED_ACT_VARIANT_CTA_ROW: CTAs per row, a power of two
 *            in [1, 8]; for GATED_ACT_VARIANT_TMA_ROWS: CTAs per SM, a power
 *            of two in [1, 16] (threads per CTA = 1024 / that); for
 *            GATED_ACT_VARIANT_PIPE_ROWS: CTAs per SM, a power of two in
 *            [1, 8]; 0 lets the library choose for those three; for
 *            GATED_ACT_VARIANT_SPLIT_ROWS: CTAs per row, 2, 4 or 8 (no
 *            default: other values return GATED_ACT_ERR_VARIANT; device
 *            memory and rows of up to 4096 16-byte vectors only); ignored by
 *            the other variants.
 * Returns GATED_ACT_ERR_VARIANT when the layout cannot use that geometry
 * (vector variants need the 16-byte layout above; a row slice must fit the
 * CTA's registers).
 */
int gelu_and_mul_sparse_ex(void *out, const void *in, int64_t T, int64_t d,
                           int64_t row_stride, double z, int variant,
                           int cluster, cudaStream_t stream);

/*
 * gelu_and_mul_sparse on fp16 or fp32 rows as well as bf16.  The
 * sparse-GELU page, "Cross-architecture warp and dtype validation", checks
 * the op in FP32, FP16 and BF16.
 *   dtype    a gated_act_dtype shared by in and out.  Sizes and strides are
 *            in elements; pointers aligned to the element size.
 *   variant, cluster as in gelu_and_mul_sparse_ex.  fp16 and fp32 run the
 *            CTA-row, split-row or scalar geometries only: WARP_ROWS,
 *            TMA_ROWS and PIPE_ROWS return GATED_ACT_ERR_VARIANT for them.
 * Math is fp32 throughout; the fp32 output evaluates tanh-GELU as
 * s / (1 + e^{-2y}) on the hardware exponential and reciprocal (relative
 * error about 2^-21), the 16-bit outputs use the hardware tanh.  Accuracy against an fp64 evaluation:
 * bf16 1e-2 |ref| + 2e-3; fp16 1e-3 |ref| + 1e-5; fp32 1e-5 |ref| + 1e-5;
 * the zero pattern as for gelu_and_mul_sparse.
 */
int gelu_and_mul_sparse_typed(void *out, const void *in, int64_t T, int64_t d,
                              int64_t row_stride, double z, int dtype,
                              int variant, int cluster, cudaStream_t stream);

/*
 * gelu_and_mul_sparse in native-rounding mode: the op computed as the
 * composition of separate element-type ops does it, every intermediate
 * rounded to the element type -- what the sparse-GELU page's kernel does to
 * match PyTorch's own sequence of ops ("Cross-architecture warp and dtype
 * validation").  Each op
 * runs in fp32 and its result is rounded (nearest even) to the element type:
 *   m = R(mean g), sd = R(population std g), t = R(sd * z), c = R(m + t),
 *   s = relu(R(g - c)), a = R(gelu_tanh(s)), out = R(a * u).
 *   dtype  GATED_ACT_BF16 or GATED_ACT_F16 (fp32 ops round to fp32 anyway:
 *          GATED_ACT_ERR_DTYPE).  Other arguments as gelu_and_mul_sparse.
 * Accuracy: the zero pattern is exactly {g > c}; where the kernel's fp32 row
 * statistics round to the same c as an exact evaluation (all but rare rows),
 * each output is within one element-type ulp of that evaluation.
 * a = R(gelu_tanh(s)) depends only on the 16-bit pattern of s, so it is
 * tabulated: the first native launch on a device that finds the table of its
 * element type missing builds it (32768 entries, 64 KB per type, in the
 * library's device memory; that launch computes a directly) and later
 * launches read it through the read-only cache.  Table and direct
 * evaluation give the same bits.  Rows run one CTA per row (the geometry
 * with the most L1 for the table), or, for a few wide rows, split over 8 or
 * 4 CTAs (2 above d = 16384) that each compute the row's statistics, or in
 * an 8-CTA cluster.
 */
int gelu_and_mul_sparse_native(void *out, const void *in, int64_t T, int64_t d,
                               int64_t row_stride, double z, int dtype,
                               cudaStream_t stream);

/*
 * The launch gelu_and_mul_sparse_native would make, without launching; the
 * arguments as gelu_and_mul_sparse_plan without the variant, cluster and
 * workspace (dtype GATED_ACT_BF16 or GATED_ACT_F16; GATED_ACT_ERR_DTYPE
 * otherwise).
 */
int gelu_and_mul_sparse_native_plan(const void *out, const void *in, int64_t T,
                                    int64_t d, int64_t row_stride, int dtype,
                                    int sm_count, gated_act_plan *plan);

/* ------------------------------------------------------------------------
 * Dynamic rows through a caller-owned workspace.
 *
 * The bulk-copy geometries run one persistent CTA (or a few) per SM.  Given
 * round-robin rows, each CTA ends when its own share is done, and the SMs
 * that stream more slowly set the end of the launch.  With a workspace the
 * CTAs instead take rows from an atomic counter in it, so every SM stays
 * busy to the end; at d >= 32768 pipe rows also run the last wave of rows
 * as two half jobs each (both compute the row's statistics in full, each
 * writes half of its output).  Within one geometry the results are
 * identical: every row's statistics and outputs are computed in the same
 * order either way.  The automatic choice can differ with a workspace: for
 * rows wider than 16384 it prefers pipe rows, which gain most from dynamic
 * rows, where the plain call keeps tma rows (d >= 28672 from 8 rows per SM
 * on).  Then the two calls agree within the accuracy bound rather than
 * bitwise; gelu_and_mul_sparse_plan_ex tells.
 * ------------------------------------------------------------------------ */

/* Bytes of workspace gelu_and_mul_sparse_ws needs (a constant, 16). */
size_t gelu_and_mul_sparse_workspace_bytes(void);

/*
 * gelu_and_mul_sparse_typed with a workspace.
 *   workspace  device (or managed) memory of
 *              gelu_and_mul_sparse_workspace_bytes() bytes, 8-byte aligned,
 *              disjoint from in and out, all zero before its first use.
 *              A call that completes leaves it all zero again, so one
 *              workspace serves any number of calls that run one after
 *              another on the GPU (one stream, or streams ordered by events;
 *              replays of one CUDA graph are ordered too).  Calls that may
 *              overlap on the GPU need workspaces of their own: two running
 *              launches sharing one would take each other's row tickets.
 *              The library only reads and writes it from the GPU.
 *   Other arguments as gelu_and_mul_sparse_typed.  Rows are taken
 *   dynamically when the plan's dynamic_rows is 1: pipe rows always, tma
 *   rows at six or more rows per CTA or whenever they are forced; other
 *   geometries ignore the workspace.
 * Errors as gelu_and_mul_sparse_typed, plus GATED_ACT_ERR_NULL (no
 * workspace), GATED_ACT_ERR_ALIGN (not 8-byte aligned), GATED_ACT_ERR_OVERLAP
 * (it overlaps in or out) and GATED_ACT_ERR_HOST (host memory).
 */
int gelu_and_mul_sparse_ws(void *out, const void *in, int64_t T, int64_t d,
                           int64_t row_stride, double z, int dtype,
                           int variant, int cluster, void *workspace,
                           cudaStream_t stream);

/*
 * gelu_and_mul_sparse_ws_static -- gelu_and_mul_sparse_ws for callers that
 * cannot allocate device memory.  Neither the sparse-GELU page nor the
 * MoE-activation page defines such an entry point.  Some callers cannot
 * call cudaMalloc at all: an inference engine that reserved every free byte
 * for its own pool at start-up, or a plugin host that hands a kernel only
 * its inputs and outputs.  For them even a 16-byte workspace is out of
 * reach, and cudaMalloc/cudaFree may also synchronize the device.  This
 * entry point allocates nothing.  Its row counters live in a 256-byte
 * scratch array inside the library, which every GPU that loads the library
 * holds until the process exits.
 *   Arguments as gelu_and_mul_sparse_ws, without the workspace.  The caller
 *   still owns in and out.
 *   Set-up: the array's device address belongs to one CUDA context, so it is
 *   looked up (cudaGetSymbolAddress) by the first call on a device in each
 *   context, with that device current, and kept for that context.  A new
 *   context -- after cudaDeviceReset, or one the caller made current through
 *   the driver API -- gets its own lookup.  Make the first call on each
 *   device before any stream capture.
 *   Only calls whose plan takes rows from a counter use the array
 *   (gelu_and_mul_sparse_plan_ex with with_workspace = 1 reports
 *   dynamic_rows = 1): such a call first zeroes the counters on `stream`,
 *   then launches.  Every such call shares the one array per device, and it
 *   keeps the last call's contents.  Calls that overlap on the GPU (other
 *   streams, other threads) race on the counters and can hand rows to the
 *   wrong launch: order such calls on the GPU, or use gelu_and_mul_sparse_ws
 *   with a workspace each.  A call whose plan takes no counter neither reads
 *   nor clears the array.
 *   A call that would need more scratch than the array holds returns
 *   GATED_ACT_ERR_SCRATCH.  This op needs 16 bytes at any size.
 * Results and other errors as gelu_and_mul_sparse_ws.
 */
int gelu_and_mul_sparse_ws_static(void *out, const void *in, int64_t T,
                                  int64_t d, int64_t row_stride, double z,
                                  int dtype, int variant, int cluster,
                                  cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GATED_ACT_H */
