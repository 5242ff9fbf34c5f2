/*
 * wgrad.h — C ABI of libwgrad.so: grouped-convolution backward-weight (wgrad)
 * on one NVIDIA GB300 (sm_103a), lowered as an implicit GEMM.
 *
 * Operation (weight gradient of a grouped convolution):
 *
 *   dW[g,k,(z),(y),x,c] = sum over n,(od),(oh),ow of
 *        dY[n,(od),(oh),ow,g,k] * X[n,(od*sd-pld+z*dd),(oh*sh-plh+y*dh),ow*sw-plw+x*dw,g,c]
 *
 * where terms whose input position falls outside the image are zero (implicit
 * zero padding).  Layouts, one per spatial rank, are those of the
 * GroupedConvBwdWeightKernelArgs constructors in "Composable Kernel:
 * grouped_convolution_backward_weight_kernel.hpp Source File":
 *   1-D  X = NWGC,   dW = GKXC,   dY = NWGK
 *   2-D  X = NHWGC,  dW = GKYXC,  dY = NHWGK
 *   3-D  X = NDHWGC, dW = GKZYXC, dY = NDHWGK
 * all packed (no custom strides), C and K being the channels of one group.
 * The implicit GEMM of that page has GemmM = K, GemmN = C*Z*Y*X,
 * GemmK = N*Do*Ho*Wo and GemmBatch = G.
 *
 * Conventions for every entry point below:
 *  - Pointers x, dy, dw and workspace are DEVICE pointers on the current CUDA
 *    device, owned by the caller (wg_conv_bwd_weight_host also takes the
 *    host buffers x_host, dy_host and dw_host).  The library allocates no
 *    device memory.
 *  - x, dy, dw and workspace must be 16-byte aligned (WG_ERR_MISALIGNED).
 *  - dW is overwritten (beta = 0) in every mode.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  All device work is stream-ordered; return codes report host-side
 *    validation and launch errors only.  Device-side errors (a bounded wait
 *    that ran out) are reported by wg_check_status.
 *  - On a non-zero return, wg_last_error() gives a one-line reason.
 *  - Thread-safe: calls keep no state between them except the device status
 *    word read by wg_check_status.
 */
#ifndef WGRAD_H
#define WGRAD_H

#include <stddef.h>

#if defined(__GNUC__)
#define WG_API __attribute__((visibility("default")))
#else
#define WG_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { WG_BF16 = 0, WG_FP16 = 1, WG_FP32 = 2 } wg_dtype;

/* How split-K partial sums are combined.
 *  DIRECT:        no split (split_k must be 1 or 0); dW = cast(sum).
 *  ATOMIC:        dW is zeroed on the stream first (the Preprocess memset of the
 *                 CK page; here a kernel whose successor, the split-K kernel,
 *                 waits for it only before its first add), then every split
 *                 adds its fp32 partial with a global atomic.  A 16-bit dW is
 *                 accumulated the same way in an fp32 copy in the workspace
 *                 (4 bytes per dW element), which a last kernel casts (round
 *                 to nearest even) to dW.  Not bitwise reproducible.
 *  DETERMINISTIC: two-stage: every split writes an fp32 partial to the
 *                 workspace, then a second kernel sums the splits in a fixed
 *                 order (for S >= 8: four contiguous ranges of splits, each in
 *                 index order, then the range sums in range order; for S < 8:
 *                 index order) and casts (round to nearest even) to dW.
 *                 Bitwise reproducible for a given problem and split degree.
 *  AUTO:          DIRECT when the chosen split degree is 1; otherwise ATOMIC
 *                 for an fp32 dW and DETERMINISTIC for a 16-bit dW (each
 *                 measured the faster for its dtype on GB300: the 16-bit
 *                 atomic path has one more kernel).  Ask for DETERMINISTIC
 *                 explicitly when bitwise reproducibility matters. */
typedef enum {
    WG_MODE_AUTO = 0,
    WG_MODE_DIRECT = 1,
    WG_MODE_ATOMIC = 2,
    WG_MODE_DETERMINISTIC = 3
} wg_mode;

typedef enum {
    WG_OK = 0,
    WG_ERR_INVALID_ARGUMENT = 1, /* non-positive size, derived output <= 0, out[] mismatch, NULL pointer */
    WG_ERR_NOT_SUPPORTED = 2,    /* valid problem outside what the kernels handle (IsSupportedArgument = false) */
    WG_ERR_MISALIGNED = 3,       /* a base pointer is not 16-byte aligned */
    WG_ERR_WORKSPACE = 4,        /* workspace missing or smaller than wg_workspace_size */
    WG_ERR_CUDA = 5,             /* a CUDA runtime/driver call failed */
    WG_ERR_DEVICE_TIMEOUT = 6    /* a kernel's bounded wait ran out, or (an internal error) a kernel
                                    found its launch inconsistent; reported by wg_check_status */
} wg_status;

/* Problem record (the host arguments of the CK page: G_, N_, C_, K_, spatial
 * lengths, strides, dilations, left/right pads).
 * Spatial arrays use their first `ndim` entries, outermost dimension first
 * (D, H, W for 3-D; H, W for 2-D; W for 1-D); the other entries are ignored. */
typedef struct {
    int ndim;              /* 1, 2 or 3 */
    int G, N, C, K;        /* groups, batch, channels per group (input C, output K) */
    int in[3];             /* input spatial lengths */
    int filt[3];           /* filter spatial lengths */
    int out[3];            /* output lengths: 0 = derive; non-zero must equal the derived value */
    int stride[3], dil[3]; /* >= 1 */
    int pad_l[3], pad_r[3];/* >= 0 */
    wg_dtype in_dtype;     /* X and dY: WG_BF16 or WG_FP16 (both the same) */
    wg_dtype out_dtype;    /* dW: WG_FP32, WG_BF16 or WG_FP16 */
} wg_problem;

/* Which kernel computes the contraction.
 *  AUTO:       the depthwise kernel where it applies (C = K = 1, 1-D or 2-D,
 *              at most 9 taps, G a multiple of 8), else the tensor-core kernel.
 *  IGEMM:      the tensor-core implicit GEMM for every problem.  For small C
 *              and K it folds several groups into one tile and keeps only the
 *              diagonal blocks (the merged-tile design of the CK page's group
 *              merging), so depthwise problems run on it too.  The planner
 *              picks the tile form (below) from its cost model.
 *  DEPTHWISE:  the CUDA-core depthwise kernel; WG_ERR_NOT_SUPPORTED where it
 *              does not apply.
 *  IGEMM_TAPS_M:  the tensor-core kernel with every filter tap on the MMA rows:
 *              D[(tap, c), k] (the CK page's GemmN = C*YX, transposed).
 *  IGEMM_TAPS_MN: the tensor-core kernel with the filter's x taps moved to the
 *              MMA columns: D[(z, y, c), (x, k)], summed over pixels q shifted
 *              by x along W (dY read at q - x*dil, X at q - pad), which turns
 *              K = 64 into 64*X columns per MMA.  Needs stride 1, a k window
 *              that is a multiple of 64 (K, or K times the groups folded into
 *              one tile when C and K are small), 2 <= X <= 4 and no cluster;
 *              WG_ERR_NOT_SUPPORTED otherwise.  One CTA per M-tile.
 *  IGEMM_PAIR: the IGEMM_TAPS_MN tile with a split's two M-tiles on the two
 *              CTAs of a thread-block cluster sharing M = 256 MMAs
 *              (tcgen05 .cta_group::2), each CTA staging half of the output
 *              channels of dY.  Needs what IGEMM_TAPS_MN needs, plus K = 64
 *              with no group folding, C <= 64, a 2-D filter with 3 or 4 taps
 *              along h; WG_ERR_NOT_SUPPORTED otherwise.  IGEMM and AUTO choose
 *              between the forms by the planner's cost model. */
typedef enum {
    WG_KERNEL_AUTO = 0,
    WG_KERNEL_IGEMM = 1,
    WG_KERNEL_DEPTHWISE = 2,
    WG_KERNEL_IGEMM_TAPS_M = 3,
    WG_KERNEL_IGEMM_TAPS_MN = 4,
    WG_KERNEL_IGEMM_PAIR = 5
} wg_kernel;

/* Per-call options (the CK page's k_batch, plus the two ways of combining splits).
 *  split_k:     0 = choose automatically, 1 = no split, S > 1 = S splits of GemmK.
 *  mode:        see wg_mode.
 *  group_merge: depthwise problems only (C = K = 1): channels handled per thread
 *               vector (1, 2, 4 or 8); 0 = choose automatically.  Must be 0 or 1
 *               for other problems.
 *  cluster:     tensor-core path only: consecutive splits run as thread-block
 *               clusters of this many CTAs (2, 4 or 8), which add their partial
 *               sums in distributed shared memory (in cluster-rank order) before
 *               anything leaves the SMs, so only S / cluster partial sums per dW
 *               element reach memory.  0 or 1 = no clusters (the default:
 *               distributed shared memory is slow enough on GB300 that this was
 *               slower than the two-stage path on every workload measured).
 *               Must divide split_k; must be 0 or 1 for the depthwise kernel.
 *               With S == cluster the sums are final: mode DIRECT then accepts
 *               the split, and no workspace is needed.
 *  kernel:      see wg_kernel. */
typedef struct {
    int split_k;
    wg_mode mode;
    int group_merge;
    int cluster;
    wg_kernel kernel;
} wg_options;

/* Validate `p` and fill p->out[] with the derived output lengths
 * (out = floor((in + pad_l + pad_r - dil*(filt-1) - 1) / stride) + 1 per dim).
 * Returns WG_OK or WG_ERR_INVALID_ARGUMENT.  Host only. */
WG_API int wg_problem_normalize(wg_problem* p);

/* Bytes of device workspace that wg_conv_bwd_weight needs for (p, opt): the
 * caller-visible workspace sizing of the two-stage (deterministic split-K)
 * path, sized from the unmerged dimensions as the PR #12359 page ("add group
 * merging (Gm) for depthwise grouped conv", PR #12951's
 * wgrad_two_stage_workspace_nbytes) states it.  0 unless the chosen mode is
 * DETERMINISTIC with more than one partial sum reaching memory, where it is
 * (partials) * G*K*Z*Y*X*C * 4 bytes, each (g, k) row of Z*Y*X*C rounded up to
 * whole reduction slices, or ATOMIC with a 16-bit dW, where it is the fp32
 * copy of dW (G*K*Z*Y*X*C rounded up to a multiple of 4, times 4 bytes).
 * opt may be NULL (all defaults).
 * Returns WG_OK, WG_ERR_INVALID_ARGUMENT or WG_ERR_NOT_SUPPORTED.  Host only. */
WG_API int wg_workspace_size(const wg_problem* p, const wg_options* opt, size_t* bytes);

/* Compute dW for problem p on `stream`.
 *  x:  input activations, in_dtype, layout N(D)(H)WGC
 *  dy: output gradient,   in_dtype, layout N(Do)(Ho)WoGK
 *  dw: weight gradient,  out_dtype, layout GK(Z)(Y)XC — overwritten
 *  workspace / ws_bytes: at least wg_workspace_size bytes (may be NULL when that is 0)
 * Returns WG_OK or an error status; nothing is launched on an error. */
WG_API int wg_conv_bwd_weight(const wg_problem* p, const void* x, const void* dy, void* dw, const wg_options* opt,
                       void* workspace, size_t ws_bytes, void* stream);

/* Synchronise `stream`, then read and clear the device status word that the
 * kernels set when a bounded wait runs out.  Returns WG_OK,
 * WG_ERR_DEVICE_TIMEOUT or WG_ERR_CUDA. */
WG_API int wg_check_status(void* stream);

/* Human-readable plan for (p, opt): kernel, tiles, split degree, mode, grid,
 * shared memory, workspace.  Writes at most n bytes including the NUL.
 * Returns WG_OK or a validation status.  Host only. */
WG_API int wg_plan_string(const wg_problem* p, const wg_options* opt, char* buf, size_t n);

/* Static name of a status code. */
WG_API const char* wg_status_string(int status);

/* One-line reason for the last non-zero return on the calling thread. */
WG_API const char* wg_last_error(void);

/* wg_conv_bwd_weight for callers that cannot allocate device memory (no
 * counterpart in the CK page: it is a property of this library's API).
 *
 * Who needs it: wg_conv_bwd_weight asks the caller for the split-K workspace.
 * A caller that cannot call cudaMalloc -- a plug-in whose host application owns
 * all device memory through its own allocator, code held to a fixed device
 * memory budget, a latency-critical path that cannot take cudaMalloc's implicit
 * synchronisation -- cannot supply one.  This entry point takes the workspace
 * from a 16 MiB array compiled into the library instead (every GPU that loads
 * the library holds it until the process exits) and allocates nothing.
 *
 * Arguments and results are those of wg_conv_bwd_weight without the workspace.
 * With split_k = 0 the split degree is capped so that the partial sums fit the
 * array (with clusters of Q splits, Q times as many splits fit); when not even
 * two partial sums of dW fit, the call runs one split (one cluster), which
 * needs no workspace.  An explicit split_k whose partial sums need more than
 * 16 MiB returns WG_ERR_WORKSPACE with the sizes in wg_last_error().
 *
 * The first call on a device looks up the array's device address (with that
 * device current) and caches it for the rest of the process; make that first
 * call before any stream capture, and make no call on a device after a
 * cudaDeviceReset of it (the cached address belongs to the context the reset
 * destroyed).  All calls share the one array and it keeps the last call's
 * contents; the kernels write every element they later read, so nothing needs
 * clearing, but calls whose work overlaps on the GPU (other streams, other
 * threads) race on it and must be serialised by the caller. */
WG_API int wg_conv_bwd_weight_noalloc(const wg_problem* p, const void* x, const void* dy, void* dw,
                                      const wg_options* opt, void* stream);

/* wg_conv_bwd_weight with the inputs and the result in host memory (no
 * counterpart in the CK page: it is a property of this library's API).
 *
 *  x_host, dy_host: X and dY in host memory, layouts as for wg_conv_bwd_weight.
 *    Page-locked memory (cudaHostAlloc, cudaHostRegister) is copied
 *    asynchronously; pageable memory goes through the driver's staging (the
 *    call then returns only after it has been read).
 *  dw_host: host memory that receives dW (out_dtype).
 *  x_dev, dy_dev, dw_dev: device buffers of the sizes of X, dY and dW that the
 *    call copies into and computes from (caller-owned, 16-byte aligned).
 *  opt, workspace, ws_bytes, stream: as for wg_conv_bwd_weight.
 *
 * Enqueues on `stream`: the copies of X and dY to the device buffers, the
 * computation exactly as wg_conv_bwd_weight on those buffers, and the copy of
 * dW to dw_host, which holds dW once `stream` has completed the call.
 * (Copying in image chunks overlapped with the main kernel's split ranges was
 * measured slower on GB300 than copying first: 181 us against 162 us per call
 * for the 56x56 C = K = 64 problem, so the copies run first.)  Returns WG_OK
 * or an error status; nothing is enqueued on an error. */
WG_API int wg_conv_bwd_weight_host(const wg_problem* p, const void* x_host, const void* dy_host, void* dw_host,
                                   void* x_dev, void* dy_dev, void* dw_dev, const wg_options* opt, void* workspace,
                                   size_t ws_bytes, void* stream);

/* Self-test of failure detection (no counterpart in the CK page).  Launches
 * one thread on `stream` that waits on an mbarrier which nothing completes:
 * the wait is bounded like every wait in the library's kernels, runs out
 * after the library's limit (2 s), sets the device status word and returns.
 * The next wg_check_status then returns WG_ERR_DEVICE_TIMEOUT (and clears
 * the word); the context stays usable.  Returns WG_OK or WG_ERR_CUDA (launch). */
WG_API int wg_selftest_timeout(void* stream);

/* Measurement hook (no counterpart in the CK page: it exists so that the
 * kernels of one call can be timed separately with CUDA events).  While
 * `event` (a cudaEvent_t owned by the caller, valid while set) is non-NULL,
 * every wg_conv_bwd_weight / wg_conv_bwd_weight_noalloc call made by this host
 * thread records it on the call's stream right after the call's main kernel
 * (the tensor-core or depthwise kernel), before the split-K reduction kernel
 * if the plan has one.  Between those two kernels the record takes away the
 * reduction's early launch (programmatic dependent launch), so a step timed
 * with it set is slightly slower.  NULL turns it off.  Returns WG_OK.  Host only. */
WG_API int wg_set_mark_event(void* event);

/* Backward-data (dgrad) of the same grouped convolution, the step beside the
 * weight gradient in training (the pages' "dgrad" section: dY, NHWGK, read
 * with its contiguous K channels as the reduction axis; W read as KYXC):
 *
 *   dX[n,(d),(h),w,g,c] = sum over k and taps (z,y,x) with
 *       (d + pad_l - z*dil, h + pad_l - y*dil, w + pad_l - x*dil) / stride integral
 *       and inside the output, of dY[n, that position, g, k] * W[g,k,z,y,x,c]
 *
 *  p:  the convolution, as for wg_conv_bwd_weight; here in_dtype is the dtype
 *      of dY and W (WG_BF16 or WG_FP16) and out_dtype that of dX (WG_FP32,
 *      WG_BF16 or WG_FP16).
 *  dy: N(Do)(Ho)WoGK, w: GK(Z)(Y)XC (in_dtype), dx: N(D)(H)WGC (out_dtype),
 *      device pointers, 16-byte aligned, owned by the caller.  dX is
 *      overwritten (every element is written once).
 *  workspace / ws_bytes: at least wg_bwd_data_workspace_size bytes (may be NULL
 *      when that is 0).  For small C and K several groups share one tile and the
 *      kernel reads a block-diagonal copy of W that a first kernel writes here;
 *      its contents need not be preserved between calls.
 * Supported: strides up to 8, any dilation and pads, up to 32 taps per
 * dimension, G*C and G*K multiples of 8, and without a group fold C a multiple
 * of 8 and K a multiple of 8 when G > 1; otherwise WG_ERR_NOT_SUPPORTED.  Input
 * positions that no (output position, tap) pair reaches (a stride larger than
 * the dilated filter) get 0.
 * Returns WG_OK or an error status; nothing is launched on an error.  The
 * kernels run on `stream` (a cudaStream_t). */
WG_API int wg_conv_bwd_data(const wg_problem* p, const void* dy, const void* w, void* dx, void* workspace,
                            size_t ws_bytes, void* stream);

/* Bytes of workspace wg_conv_bwd_data needs for p (0 when no group fold). */
WG_API int wg_bwd_data_workspace_size(const wg_problem* p, size_t* bytes);

/* Human-readable plan of wg_conv_bwd_data for p.  Host only. */
WG_API int wg_bwd_data_plan_string(const wg_problem* p, char* buf, size_t n);

#ifdef __cplusplus
}
#endif

#endif /* WGRAD_H */
