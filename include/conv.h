/*
 * conv.h -- C ABI of the GB300 implicit-GEMM convolution-forward library
 * (libconvfwd.so).
 *
 * The operation (page "composable_kernel dispatcher/heuristics/LEARNINGS_GROUPED_CONV.md",
 * introduction and section 2; page "[ET-VK] conv1d runs at ~3% of the GPU's matmul
 * throughput ...", sections "Measurements", "The conv2d path already solves this" and
 * "Suggested fix"):
 *
 *   y[n, o, g, k] = act( bias[g, k] + sum_{t, c} x[n, o*stride + t*dilation - pad, g, c] * w[g, k, t, c] )
 *
 * a dense or grouped cross-correlation over 1, 2 or 3 spatial dimensions with stride,
 * symmetric zero padding and dilation; act is the identity or the exact (erf) GELU.
 * A 1D problem is run as the H = 1 (and D = 1) case of the same path, never by a
 * separate kernel; a 2D problem is the D = 1 case.
 *
 * Layouts (channels last, dense, row major):
 *   x      N  [D] [H] W  G C        (conv1d: N L C with G = 1)
 *   w      G  K  [Z] [Y] X  C       (conv1d: K kw C)
 *   y      N  [Do][Ho] Wo G K
 *   bias   G*K
 * Output size per spatial dimension: O = floor((I + 2*pad - dil*(F-1) - 1) / stride) + 1.
 *
 * Arithmetic: bf16 I/O multiplies bf16 on the tensor cores (tcgen05) and accumulates
 * in fp32.  fp32 I/O runs by default on the tensor cores as 3xTF32: each operand splits
 * into a TF32 high part and an fp32 remainder, and lo*hi + hi*lo + hi*hi are accumulated
 * in fp32; what it drops (lo*lo, and the low bits of lo that TF32 does not carry) is
 * below 2^-20 |x*w| per term (both splits truncate), so the result stays within 1e-5 of
 * sum |x*w|, the bound an fp32 FFMA sum meets.  The FFMA kernel (plain fp32) takes the
 * problems no tensor-core plan can express (channel counts that are not multiples of 8
 * for bf16 or of 4 for fp32, fp32 inputs the TMA gather cannot address) and plans forced
 * onto it.  The epilogue (bias, GELU) runs in fp32 and a bf16 output is rounded once, to
 * nearest even.
 *
 * Conventions for every call:
 *  - Ownership: the caller allocates and frees every device buffer (x, w, w_packed,
 *    bias, y, workspace).  A plan owns only host memory; it never allocates device
 *    memory.
 *  - Pointers: x, w, w_packed, bias, y and the workspace are device pointers and must
 *    be 16-byte aligned (CONV_ERR_ALIGNMENT otherwise).
 *  - Streams: `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  Calls enqueue work and return; they never synchronise.  conv_fwd makes
 *    no allocation and no host-device copy, so it may be captured in a CUDA graph.
 *  - Errors: every call returns a conv_status.  Launch failures return CONV_ERR_CUDA.
 *    A kernel that gives up on a pipeline wait (a bounded spin) records the fact in a
 *    device-side error word and exits; conv_plan_check() reads and clears it.
 *  - Threads: a plan may be used from several host threads and streams at once as long
 *    as calls that use a workspace are given disjoint workspaces.
 */
#ifndef CONVFWD_CONV_H
#define CONVFWD_CONV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    CONV_OK = 0,
    CONV_ERR_INVALID_ARG = 1,   /* a size, count or pointer argument is out of range   */
    CONV_ERR_UNSUPPORTED = 2,   /* well formed, but outside what the library implements */
    CONV_ERR_ALIGNMENT = 3,     /* a pointer or a channel count breaks 16-byte alignment */
    CONV_ERR_WORKSPACE = 4,     /* the plan needs a workspace and none (or too small) set */
    CONV_ERR_CUDA = 5,          /* a CUDA runtime call or a kernel launch failed          */
    CONV_ERR_TIMEOUT = 6        /* a kernel abandoned a pipeline wait (see conv_plan_check) */
} conv_status;

typedef enum { CONV_F32 = 0, CONV_BF16 = 1 } conv_dtype;   /* I/O type of x, w, bias, y */

typedef enum {
    CONV_EPI_NONE = 0,        /* y = acc                         */
    CONV_EPI_BIAS = 1,        /* y = acc + bias                  */
    CONV_EPI_BIAS_GELU = 2,   /* y = GELU(acc + bias), erf form  */
    CONV_EPI_GELU = 3         /* y = GELU(acc)                   */
} conv_epilogue;

typedef struct conv_plan* conv_plan_t;

/*
 * Build a plan: validate the problem, normalise it to three spatial dimensions
 * (conv1d -> D = H = 1, conv2d -> D = 1; page "[ET-VK] conv1d ...", "Suggested fix"),
 * form the GEMM view per group (M = N*Do*Ho*Wo, N_gemm = K, K_gemm = taps*C) and pick
 * the kernel variant and tiling (page "onnxruntime PR #33639", "Description": large
 * tiles for large problems, split-K where tiles alone cannot fill the GPU, each choice
 * checked against the device's limits).
 *   ndim      1, 2 or 3
 *   N G C K   batch, groups, input channels per group, output channels per group (>= 1)
 *   spatial   ndim input extents, outermost first (D, H, W)
 *   filter    ndim filter extents (Z, Y, X)
 *   stride, pad, dilation   ndim values each; stride >= 1, pad >= 0, dilation >= 1
 * bf16 problems with C and K multiples of 8 run on the tensor cores (kind::f16); fp32
 * problems with C and K multiples of 4 whose input the TMA gather can address run on the
 * tensor cores as 3xTF32 (kind::tf32, three products per useful product); everything
 * else runs on the FFMA kernel.  conv_plan_describe names the choice ("variant=tc_bf16",
 * "tc_tf32x3", "simt_bf16" or "simt_f32") and, for tensor-core plans, the gather (per-tap
 * boxes or slabs), the tile, the ring stages and whether tiles of 256 rows run on a pair of
 * SMs ("cta_pair=m256": the two CTAs of a cluster issue .cta_group::2 MMAs, each holding half
 * of every weight tile) or y leaves through a TMA tensor store ("store=tma").  Results are the
 * same bits either way: every output is one sum in a fixed order.
 * Returns CONV_ERR_INVALID_ARG for a bad argument or an empty output,
 * CONV_ERR_UNSUPPORTED when an index would overflow the kernels' 32-bit coordinates.  The plan queries the current
 * device's SM count; without a device it plans for 152 SMs.  *out is set only on CONV_OK.
 */
conv_status conv_plan_create(conv_plan_t* out, int ndim, int64_t N, int64_t G, int64_t C, int64_t K,
                             const int64_t* spatial, const int64_t* filter, const int64_t* stride,
                             const int64_t* pad, const int64_t* dilation, conv_dtype dtype,
                             conv_epilogue epilogue);

/* Output extents (ndim values, outermost first) into out_spatial: per dimension
 * O = floor((I + 2*pad - dil*(F-1) - 1) / stride) + 1, the size that gives the page's
 * printed lengths 3000 (k3 s1 p1) and 1500 (k3 s2 p1) from L = 3000 (page "[ET-VK]
 * conv1d ...", "Measurements").  out_spatial: caller-owned host array of ndim int64.
 * CONV_ERR_INVALID_ARG on a NULL plan or array. */
conv_status conv_plan_output_shape(conv_plan_t plan, int64_t* out_spatial);

/* Bytes of the prepacked weight buffer that conv_prepack_weights writes (0 on a NULL plan). */
size_t conv_prepacked_weight_bytes(conv_plan_t plan);

/* Bytes of device workspace conv_fwd needs: 0 unless the plan splits the reduction over
 * K and sums the partial sums in a second kernel (splits x M x G*K fp32 values); split
 * plans whose splits share a thread-block cluster need none.  Split-K is the small-
 * problem variant of page "onnxruntime PR #33639", "Description" (it fills the GPU
 * better than large tiles).  0 on a NULL plan. */
size_t conv_workspace_bytes(conv_plan_t plan);

/*
 * Attach a caller-owned device workspace of at least conv_workspace_bytes(plan) bytes.
 * The plan keeps the pointer, not the memory.  CONV_ERR_WORKSPACE if too small.
 */
conv_status conv_plan_set_workspace(conv_plan_t plan, void* workspace, size_t bytes);

/*
 * Weight prepack, once per weight tensor (page "[ET-VK] conv1d ...", "Suggested fix":
 * weight prepacking is part of the conv2d machinery the conv1d case reuses).
 * Reads w (layout G K [Z][Y] X C, the plan's dtype) and writes the plan-specific packed
 * image into w_packed (conv_prepacked_weight_bytes(plan) bytes): for the tensor-core
 * variant, per group, per N tile and per 64-element K block, a 128-byte-swizzled
 * K-major tile that is copied into shared memory verbatim; for the FFMA variant, a
 * (taps*C) x K_padded row-major matrix.  Asynchronous on `stream`.
 */
conv_status conv_prepack_weights(conv_plan_t plan, const void* w, void* w_packed, void* stream);

/*
 * The forward pass (the hot path): the operation at the top of this file, computed as an
 * implicit GEMM whose activation tiles are gathered from x with no im2col matrix in
 * memory (page "[ET-VK] conv1d ...", "The conv2d path already solves this": conv as
 * im2col + GEMM; page "composable_kernel ... LEARNINGS_GROUPED_CONV.md", introduction:
 * NHWGC x GKYXC -> NHWGK).  x, w_packed (from conv_prepack_weights with the same plan),
 * bias (G*K values of the plan's dtype; required when the epilogue adds a bias, ignored
 * otherwise) and y are device pointers; y must not overlap x.  Enqueues the kernel(s)
 * on `stream` and returns; launch errors come back as CONV_ERR_CUDA, a missing or small
 * workspace as CONV_ERR_WORKSPACE, a NULL or backward plan or a missing bias as
 * CONV_ERR_INVALID_ARG, a pointer off 16 bytes as CONV_ERR_ALIGNMENT; all of these are
 * checked before anything is launched.  Plans that split the reduction need a workspace
 * set first.  Each call encodes the activation tensor map for this x on the host.
 */
conv_status conv_fwd(conv_plan_t plan, const void* x, const void* w_packed, const void* bias, void* y,
                     void* stream);

/*
 * Synchronise `stream`, then read and clear the device error word.  Returns
 * CONV_ERR_TIMEOUT if a kernel abandoned a pipeline wait since the last check,
 * CONV_ERR_CUDA if the stream reports an error, CONV_OK otherwise.  (The pages have no
 * counterpart: their dispatches report nothing; this is how the library's bounded waits
 * surface instead of hanging a stream.)  The error word is one per device and shared by
 * every plan, so a check after several plans' calls reports a timeout in any of them.
 */
conv_status conv_plan_check(conv_plan_t plan, void* stream);

/* Free the plan's host memory.  NULL is accepted. */
conv_status conv_plan_destroy(conv_plan_t plan);

/* Static string naming a status code. */
const char* conv_status_string(conv_status status);

/*
 * Static-per-plan description of the choice made: variant, tile, stages, splits,
 * grid, gather mode, CTA pairs and tensor-map stores.  Valid until the plan is destroyed.
 */
const char* conv_plan_describe(conv_plan_t plan);

/*
 * Useful FLOPs of one conv_fwd: 2 * N*Do*Ho*Wo * G*K * taps*C, padded taps counted
 * (the convention of page "[ET-VK] conv1d ...", "Measurements": 31.3 GFLOP/s for the
 * 80 -> 384 layer at 17.7 ms).  0 on a NULL plan.
 */
double conv_plan_flops(conv_plan_t plan);

/*
 * Let consecutive kernels of a chain overlap (programmatic dependent launch).  With
 * enable != 0, the kernels conv_fwd launches for this plan are marked so that each may
 * start while the kernel before it on the stream is still running, when that kernel
 * allows it (the library's own kernels allow it as soon as each of their CTAs is set
 * up).  A kernel that starts early builds its shared-memory pipeline and loads the
 * packed weights, then waits for the previous kernel to complete before it reads x or
 * bias or writes y or the workspace.  So the overlap is safe whenever w_packed is not
 * written by the kernel launched just before conv_fwd on the same stream; x, bias and y
 * may be (a chain of layers, each reading the previous layer's output, is the intended
 * use).  The pages' first "next step" asks for exactly this chaining of the Whisper
 * frontend (page "[ET-VK] conv1d ...", "The conv2d path already solves this": the two
 * convs and their GELUs run as dependent dispatches).  Default: off.  Returns
 * CONV_ERR_INVALID_ARG on a NULL plan.
 */
conv_status conv_plan_set_overlap(conv_plan_t plan, int enable);

/*
 * Backward passes (the "bwd_data" and "bwd_weight" variants that page "Learnings --
 * Grouped-Conv Heuristic (Forward, 2D + 3D)", section 6, names for the same NHWGC x
 * GKYXC -> NHWGK layouts).  Both take the FORWARD problem's description, exactly as
 * conv_plan_create does (ndim, N, G, C, K, input extents, filter, stride, pad, dilation,
 * dtype), and return CONV_ERR_INVALID_ARG / CONV_ERR_UNSUPPORTED on the same inputs.
 * dy is the gradient of a loss with respect to the forward output y (N Do Ho Wo G K,
 * the dtype of the plan); they differentiate the convolution's linear part only (bias
 * and GELU are elementwise and outside it):
 *
 *   dx[n,i,g,c] = sum over k and taps t of dy[n,o,g,k] * w[g,k,t,c], over the o with
 *                 o*stride - pad + t*dil = i in every spatial dimension
 *   dw[g,k,t,c] = sum over n and output positions o of dy[n,o,g,k] * x[n, o*stride - pad + t*dil, g, c]
 *
 * accumulated in fp32 and rounded once to the plan's dtype.  conv_plan_output_shape
 * returns the forward output extents (dy's), conv_plan_flops the forward problem's
 * useful FLOPs (each backward pass performs as many), conv_plan_describe the variant.
 * Workspaces (conv_workspace_bytes / conv_plan_set_workspace), conv_plan_check,
 * conv_plan_set_overlap and conv_plan_destroy work as for forward plans; conv_fwd and
 * conv_fwd_static_scratch refuse backward plans with CONV_ERR_INVALID_ARG.
 */

/*
 * Backward-data plan.  Its packed weight comes from conv_prepack_weights(plan, w, ...)
 * with w in the forward layout G K Z Y X C (conv_prepacked_weight_bytes gives the size).
 * At unit stride (and pad <= dil*(F-1) per dimension) dx is the forward convolution of
 * dy with every tap axis flipped, C and K swapped and padding dil*(F-1) - pad, and the
 * plan runs the forward kernels on that problem; otherwise an FFMA kernel gathers, for
 * each input pixel, the dy positions that map onto it.
 */
conv_status conv_bwd_data_plan_create(conv_plan_t* out, int ndim, int64_t N, int64_t G, int64_t C, int64_t K,
                                      const int64_t* spatial, const int64_t* filter, const int64_t* stride,
                                      const int64_t* pad, const int64_t* dilation, conv_dtype dtype);

/*
 * dx (N D H W G C, device) from dy (N Do Ho Wo G K, device) and the packed weight.  All
 * three 16-byte aligned.  Asynchronous on `stream`; errors as conv_fwd
 * (CONV_ERR_INVALID_ARG for NULL pointers or a plan of another direction).
 */
conv_status conv_bwd_data(conv_plan_t plan, const void* dy, const void* w_packed, void* dx, void* stream);

/*
 * Backward-weight plan.  No packed weight (conv_prepack_weights returns
 * CONV_ERR_INVALID_ARG).  The output pixels are split across CTAs, whose fp32 partial sums
 * live in the workspace; fp32 plans also stage x and dy there as three bf16 planes each (the
 * tensor cores then accumulate six plane products per tile).  Attach a workspace of
 * conv_workspace_bytes(plan) whenever that is non-zero.
 */
conv_status conv_bwd_weight_plan_create(conv_plan_t* out, int ndim, int64_t N, int64_t G, int64_t C, int64_t K,
                                        const int64_t* spatial, const int64_t* filter, const int64_t* stride,
                                        const int64_t* pad, const int64_t* dilation, conv_dtype dtype);

/*
 * dw (G K Z Y X C, device) from x (N D H W G C) and dy (N Do Ho Wo G K), all device and
 * 16-byte aligned; dw is overwritten (not accumulated into).  Asynchronous on `stream`;
 * errors as conv_fwd.
 */
conv_status conv_bwd_weight(conv_plan_t plan, const void* x, const void* dy, void* dw, void* stream);

/*
 * Measured kernel selection.  conv_plan_create picks a variant and tiling by fixed rules
 * from the problem's geometry.  The selector instead times the candidate plans of one
 * problem on this device and keeps the fastest, in a process-wide table that later
 * conv_plan_create calls for the same problem consult.  The table's key holds every
 * feature that changes the best kernel: N, G, C, K, the input extents, filter, stride,
 * padding and dilation per axis, dtype, epilogue and the SM count (page "Learnings --
 * Grouped-Conv Heuristic (Forward, 2D + 3D)", section 2: dilation must be a feature or
 * dilated 3D problems are indistinguishable).  Each entry records the whole choice (N
 * tile, split factor, gather mode, slab streaming and tile pairs, epilogue width, cluster
 * reduction, FFMA kernel), not a bucket of it (same page, section 1: aliased kernel
 * names capped the predictor's top-1 accuracy).  Precedence in conv_plan_create: the
 * CONV_FORCE_* test variables, then the table, then the rules.
 */

/*
 * Device bytes conv_plan_tune needs as scratch: the largest packed weight of any
 * candidate (rounded up to 256 bytes) plus that candidate's split-K workspace.  0 on a
 * NULL plan.
 */
size_t conv_tune_scratch_bytes(conv_plan_t plan);

/*
 * Time every candidate plan for this problem and switch `plan` to the fastest.
 *   x, y:     device input (as conv_fwd) and an output buffer of the plan's output shape;
 *             y is overwritten (many times) with valid conv outputs.
 *   w:        device weight in the unpacked layout conv_prepack_weights reads.
 *   bias:     device bias (required for the bias epilogues, else may be NULL).
 *   scratch:  device buffer of at least conv_tune_scratch_bytes(plan) bytes, 16-byte
 *             aligned; each candidate's packed weight and workspace are placed in it.
 *   iters:    timed calls per candidate (>= 1), after two untimed ones; CUDA events on
 *             `stream` time them.
 * Synchronizes `stream` once per candidate.  A candidate whose kernels report a wait
 * timeout is skipped.  On success the plan's variant, tiling, packed-weight layout and
 * workspace size may all have changed: the caller must query conv_prepacked_weight_bytes
 * and conv_workspace_bytes again, re-run conv_prepack_weights and re-attach a workspace
 * before the next conv_fwd.  The choice is also entered in the process-wide table.
 * Errors: CONV_ERR_INVALID_ARG (NULL plan, x, w, y or scratch; missing bias; iters < 1),
 * CONV_ERR_ALIGNMENT, CONV_ERR_WORKSPACE (no candidate fits `scratch`), CONV_ERR_CUDA
 * (a launch or synchronization failed; the plan is unchanged).
 */
conv_status conv_plan_tune(conv_plan_t plan, const void* x, const void* w, const void* bias, void* y,
                           void* scratch, size_t scratch_bytes, int iters, void* stream);

/*
 * Write the selector's table to a text file, one problem per line ("<key> | <choice>",
 * then " | us=<time per call>" for a choice measured in this process), each measured
 * problem followed by one comment line per candidate timed ("#", tab, "us=<time>", tab,
 * the candidate's conv_plan_describe text).  CONV_ERR_INVALID_ARG if the file cannot be
 * written.
 */
conv_status conv_tune_table_save(const char* path);

/*
 * Merge a file written by conv_tune_table_save into the table (entries for the same key
 * are replaced).  A file with any malformed line changes nothing and returns
 * CONV_ERR_INVALID_ARG, as does a file that cannot be read.  Entries only affect plans
 * created afterwards.
 */
conv_status conv_tune_table_load(const char* path);

/* Empty the selector's table (plans created afterwards use the rules). */
conv_status conv_tune_table_clear(void);

/*
 * Forward pass for callers that cannot allocate device memory.  (The pages have no
 * counterpart: this is an interface convenience of this library.)
 *
 * Some callers cannot call cudaMalloc: a plugin or custom operator that a host
 * framework hands only its input and output buffers and no allocator, or a
 * latency-critical loop that must not allocate after start-up (cudaMalloc may
 * synchronise the device).  Such callers cannot provide the split-K workspace that
 * conv_fwd needs for small problems.  This entry point computes the same result as
 * conv_fwd, but keeps the split-K partial sums in a device array that is part of the
 * library itself (CONV_STATIC_SCRATCH_BYTES bytes, reserved on every GPU that loads
 * the library, until the process exits).  The caller still passes x, w_packed, bias
 * and y; the plan's own workspace, if any, is not used.
 *
 *  - Limit: a plan whose conv_workspace_bytes() exceeds CONV_STATIC_SCRATCH_BYTES is
 *    rejected with CONV_ERR_WORKSPACE before anything is launched.  Plans that do not
 *    split the reduction need no scratch and always run.
 *  - No allocation: the call makes no cudaMalloc, cudaFree or other allocating call.
 *  - Set-up: the first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current) and caches it; make that first
 *    call before any stream capture begins.
 *  - Sharing: every call in the process uses the same array.  It keeps whatever the
 *    last call left in it; nothing in it has to start at zero, because every split
 *    writes its whole partial sum before the reduction reads it.  Calls that overlap on
 *    the GPU (on different streams, or from different host threads) race on the array
 *    and give wrong results: serialise them.
 * Errors as for conv_fwd.
 */
#define CONV_STATIC_SCRATCH_BYTES ((size_t)16 << 20)
conv_status conv_fwd_static_scratch(conv_plan_t plan, const void* x, const void* w_packed, const void* bias,
                                    void* y, void* stream);

/* The size of that array in the library as built (CONV_STATIC_SCRATCH_BYTES when the
 * library and this header agree), so that a binding need not restate the constant. */
size_t conv_static_scratch_bytes(void);

#ifdef __cplusplus
}
#endif

#endif /* CONVFWD_CONV_H */
