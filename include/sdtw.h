/*
 * sdtw.h -- C ABI of the GB300 (sm_103a) batched Soft-DTW library (libsdtw.so).
 *
 * The operation is Soft-DTW of Cuturi & Blondel (ICML 2017), the method named
 * in the "Acknowledgments" of the SoftDTW-CUDA (PyTorch + Numba) README, with
 * the squared Euclidean cost and the log-space backward of the SoftDTW-CUDA-Torch
 * paper (abstract, contributions (1)-(3)):
 *
 *   C[b,i,j] = sum_k (x[b,i,k] - y[b,j,k])^2
 *   R[0,0] = 0, R[i,0] = R[0,j] = +inf,
 *   R[i,j] = C[i,j] + softmin_g(R[i-1,j-1], R[i-1,j], R[i,j-1]),
 *   softmin_g(a) = -g log sum exp(-a/g),  loss[b] = R[N,M]  (may be negative),
 *   E = dR[N,M]/dC from the backward recursion done in log space,
 *   grad_x[b,i] = grad_loss[b] * 2 sum_j E[i,j] (x_i - y_j),
 *   grad_y[b,j] = grad_loss[b] * 2 sum_i E[i,j] (y_j - x_i).
 *
 * Conventions shared by every entry point
 *  - Tensors are fp32, row-major and contiguous: x (B,N,D), y (B,M,D),
 *    grad_x like x, grad_y like y, loss and grad_loss (B,).
 *  - Every tensor pointer and the workspace are DEVICE pointers owned by the
 *    caller, except the tensors of sdtw_value_and_grad_host, which are HOST
 *    pointers. The library allocates no memory.
 *  - `ws` is a caller-owned device workspace of at least
 *    sdtw_workspace_bytes(...) bytes, 256-byte aligned. sdtw_forward leaves in
 *    it the state that the matching sdtw_backward reads, so the caller keeps it
 *    unchanged between the two calls (as autograd keeps saved tensors).
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *    stream). Argument errors are returned synchronously before any launch.
 *    A launch failure returns SDTW_ERR_CUDA. A device-side wait that runs out
 *    of time is reported later by sdtw_last_device_status.
 *  - No CPU fallback exists: every step runs in this library's CUDA kernels.
 *  - Inputs containing NaN or inf are not checked; results are then NaN.
 */
#ifndef SDTW_H
#define SDTW_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Distance handling. UNFUSED precomputes the (B,N,M) cost tensor in the
 * workspace before the DP (README, "Basic (Unfused)"; review page, "proposed
 * method", fourth bullet). FUSED recomputes the cost inside the DP kernels and
 * keeps no cost tensor (README, "Fused Mode"; paper abstract, contribution (3)). */
typedef enum { SDTW_UNFUSED = 0, SDTW_FUSED = 1 } sdtw_mode;

/* Precision flag, OR-ed into the mode of every entry point except
 * sdtw_forward_noalloc. Long sequences at small gamma make the gradient react
 * to cost perturbations below fp32 resolution (at N=M=8192, gamma=0.01 even an
 * fp64 DP fed correctly rounded fp32 costs misses rel 1e-3), and on rows where two
 * alignments nearly tie the fp32 state's rounding moves a gradient entry by more
 * than abs 1e-5 at O(1) upstream weights. With this flag the cost and the forward
 * DP state are carried as double-floats (hi + lo fp32 pairs; the costs for
 * D <= 400 from exact fixed-point digit products on the tensor cores) and the
 * forward stores per-cell transition log-probabilities for the backward; the
 * workspace grows from 12 to 20 bytes per cell (unfused: 16 to 28). Without it
 * the DP runs in fp32 difference form, which met the tolerances on the tested
 * workloads for gamma >= 0.05, N, M < 4096 and D <= 64 at batch-mean weights of
 * at most 1/32 (or D <= 4 at any weight), but is not guaranteed to on near ties. */
#define SDTW_EXTENDED 2

/* Checkpoint flag, OR-ed into SDTW_FUSED for sdtw_forward / sdtw_backward and
 * their padded-batch forms (fp32, D <= 64 only; otherwise SDTW_ERR_ARG). The fused
 * forward then keeps only the boundary row of each band of 128 rows (the
 * checkpoints, 8 bytes per band row and column) and the state of the last band.
 * The backward walks the bands from the last up: it recomputes a band's state from
 * the row above it (on a helper stream, while the band below runs its backward)
 * and runs that band's backward, then its gradient terms (on a second helper
 * stream, overlapping the next band's backward). The per-cell workspace shrinks
 * to two bands of every problem (12 bytes per cell of a band); the bands'
 * backward wavefronts run one after another, so the backward's time grows with
 * N/128 (measured at B=32, N=M=512, D=64: workspace 142 -> 78 MiB, forward +
 * backward with gradients 0.32 -> 0.47 ms). SoftDTW-CUDA-Torch paper,
 * abstract, contribution (3): fused memory O(B(N+M)) rather than O(BNM). */
#define SDTW_CHECKPOINT 4

typedef enum {
    SDTW_OK = 0,
    SDTW_ERR_ARG = 1,        /* null pointer, bad mode, bad op, bad step number   */
    SDTW_ERR_GAMMA = 2,      /* gamma not > 0 or not finite                        */
    SDTW_ERR_EMPTY = 3,      /* B, N, M or D < 1 (empty sequences)                 */
    SDTW_ERR_SHAPE = 4,      /* shape mismatch (normalized needs equal shapes)     */
    SDTW_ERR_WORKSPACE = 5,  /* workspace NULL, misaligned or smaller than needed  */
    SDTW_ERR_CUDA = 6,       /* a CUDA runtime call or a launch failed             */
    SDTW_ERR_TIMEOUT = 7,    /* a device-side wait ran out of time (device status) */
    SDTW_ERR_TOO_LARGE = 8   /* sizes overflow the library's 32-bit index limits   */
} sdtw_status;

/* Operation codes for sdtw_workspace_bytes. */
#define SDTW_OP_FWD_BWD 0    /* sdtw_forward followed by sdtw_backward           */
#define SDTW_OP_NORMALIZED 1 /* sdtw_normalized (N == M)                          */
#define SDTW_OP_BARYCENTER 2 /* sdtw_barycenter_step: B = K sequences, N = T, M = T2 */
#define SDTW_OP_COST 3       /* sdtw_forward_cost followed by sdtw_backward_cost; D is ignored */
#define SDTW_OP_NORMALIZED_UNEQUAL 4 /* sdtw_normalized_unequal: x (B,N,D), y (B,M,D)     */

/* Bytes of device workspace needed by `op` for these sizes and mode; 0 when the
 * arguments are invalid. Pure host function, no CUDA call. */
size_t sdtw_workspace_bytes(int op, int B, int N, int M, int D, sdtw_mode mode);

/* Squared Euclidean cost C (B,N,M), row-major, into `C` (device). The unfused
 * distance step on its own (README, "Tests": distance correctness). */
sdtw_status sdtw_distance(const float* x, const float* y, int B, int N, int M, int D,
                          float* C, void* stream);

/* Forward pass: loss[b] = R_b[N,M] (B,) for every pair (x_b, y_b). Leaves the
 * DP state for sdtw_backward in `ws`. */
sdtw_status sdtw_forward(const float* x, const float* y, int B, int N, int M, int D, float gamma,
                         sdtw_mode mode, float* loss, void* ws, size_t ws_bytes, void* stream);

/* Backward pass for the same (x, y, B, N, M, D, gamma, mode) as the preceding
 * sdtw_forward on this workspace. grad_loss (B,) is dL/dloss. grad_x and/or
 * grad_y may be NULL when not wanted; they are overwritten, not accumulated. */
sdtw_status sdtw_backward(const float* x, const float* y, int B, int N, int M, int D, float gamma,
                          sdtw_mode mode, const float* grad_loss, float* grad_x, float* grad_y,
                          void* ws, size_t ws_bytes, void* stream);

/* sdtw_forward / sdtw_backward on a padded batch of unequal lengths (SoftDTW
 * README: sequences of any length; the pages show no padded-batch interface, the
 * one adopted is this). x_lengths and y_lengths are DEVICE int arrays (B,):
 * problem b aligns x_b[0, N_b) with y_b[0, M_b), N_b = x_lengths[b], M_b =
 * y_lengths[b], so loss[b] = R_b[N_b, M_b]; lengths are clamped to [1, N] and
 * [1, M] on the device (they are not read on the host). Gradients of padded
 * rows are 0; the padding of x and y must be finite (zeros are fine). Either
 * array may be NULL (full length). The workspace is that of sdtw_forward for
 * the padded sizes, and the backward must get the same lengths. */
sdtw_status sdtw_forward_varlen(const float* x, const float* y, const int* x_lengths, const int* y_lengths,
                                int B, int N, int M, int D, float gamma, sdtw_mode mode, float* loss,
                                void* ws, size_t ws_bytes, void* stream);
sdtw_status sdtw_backward_varlen(const float* x, const float* y, const int* x_lengths,
                                 const int* y_lengths, int B, int N, int M, int D, float gamma,
                                 sdtw_mode mode, const float* grad_loss, float* grad_x, float* grad_y,
                                 void* ws, size_t ws_bytes, void* stream);

/* Normalized Soft-DTW (README, "Normalization"):
 *   loss[b] = s(x_b,y_b) - (s(x_b,x_b) + s(y_b,y_b)) / 2,  x and y both (B,N,D).
 * The three problems run as one batch of 3B. When grad_loss is non-NULL the
 * input gradients are written too (grad_x/grad_y may be NULL individually). */
sdtw_status sdtw_normalized(const float* x, const float* y, int B, int N, int D, float gamma,
                            sdtw_mode mode, float* loss, const float* grad_loss, float* grad_x,
                            float* grad_y, void* ws, size_t ws_bytes, void* stream);

/* Backward of normalized Soft-DTW, for a caller that ran sdtw_normalized without
 * grad_loss (the forward only) and kept its workspace unchanged since, as autograd
 * keeps saved tensors: the three backward wavefronts and the ordered gradient
 * combination of sdtw_normalized, on the forward's state, without running the
 * forward again. Same arguments as that call; grad_loss (B,) is required,
 * grad_x / grad_y may be NULL individually (overwritten, not accumulated). */
sdtw_status sdtw_normalized_backward(const float* x, const float* y, int B, int N, int D, float gamma,
                                     sdtw_mode mode, const float* grad_loss, float* grad_x, float* grad_y,
                                     void* ws, size_t ws_bytes, void* stream);

/* Normalized Soft-DTW of sequences of different lengths, x (B,N,D) and y (B,M,D):
 * the README's "Normalization" definition, loss[b] = s(x_b,y_b) - (s(x_b,x_b) +
 * s(y_b,y_b)) / 2, applied unchanged to N != M (the README's own interface takes
 * equal shapes only; this entry lifts that restriction). The three terms are three
 * batches of different shapes (N x M, N x N, M x M) whose wavefronts run side by
 * side on internal streams ordered against `stream`; N == M gives the same values
 * as sdtw_normalized. Arguments as for sdtw_normalized: when grad_loss is non-NULL
 * the input gradients are written (grad_x (B,N,D) and grad_y (B,M,D), either may
 * be NULL). Workspace: sdtw_workspace_bytes(SDTW_OP_NORMALIZED_UNEQUAL, B, N, M, D,
 * mode); its status word gathers the three batches' device status. */
sdtw_status sdtw_normalized_unequal(const float* x, const float* y, int B, int N, int M, int D,
                                    float gamma, sdtw_mode mode, float* loss, const float* grad_loss,
                                    float* grad_x, float* grad_y, void* ws, size_t ws_bytes,
                                    void* stream);

/* Backward of sdtw_normalized_unequal run without grad_loss, on its unchanged
 * workspace: as sdtw_normalized_backward, for the three batches of their own
 * shapes. */
sdtw_status sdtw_normalized_unequal_backward(const float* x, const float* y, int B, int N, int M, int D,
                                             float gamma, sdtw_mode mode, const float* grad_loss,
                                             float* grad_x, float* grad_y, void* ws, size_t ws_bytes,
                                             void* stream);

/* One Adam step of a Soft-DTW barycenter (README, "Time Series Barycenters
 * (Averaging)"; review page, "proposed method", fifth bullet):
 *   L(z) = (1/K) sum_k s(z, X_k),  g = dL/dz,
 *   m <- b1 m + (1-b1) g;  v <- b2 v + (1-b2) g^2;
 *   z <- z - lr (m / (1-b1^t)) / (sqrt(v / (1-b2^t)) + eps).
 * z, m, v are (T,D) and updated in place; X is (K,T2,D); t >= 1 is the step
 * number. loss_out (nullable, one float) receives L at the incoming z. */
sdtw_status sdtw_barycenter_step(float* z, float* m, float* v, int t, const float* X, int K, int T,
                                 int T2, int D, float gamma, float lr, float beta1, float beta2,
                                 float eps, sdtw_mode mode, float* loss_out, void* ws,
                                 size_t ws_bytes, void* stream);

/* sdtw_barycenter_step with the gradient clipped by its global L2 norm first
 * (README, "Time Series Barycenters": gradient clipping for stability; the page
 * gives no rule, the one adopted is g <- g * min(1, max_grad_norm / ||g||)).
 * max_grad_norm = 0 is the unclipped step; negative or NaN is SDTW_ERR_ARG.
 * Same workspace (SDTW_OP_BARYCENTER). */
sdtw_status sdtw_barycenter_step_clipped(float* z, float* m, float* v, int t, const float* X, int K, int T,
                                         int T2, int D, float gamma, float lr, float beta1, float beta2,
                                         float eps, float max_grad_norm, sdtw_mode mode, float* loss_out,
                                         void* ws, size_t ws_bytes, void* stream);

/* Forward pass that allocates nothing and takes no workspace. No page of the
 * method has a counterpart: it exists for callers that cannot allocate device
 * memory -- a host program with no device allocator of its own (no PyTorch, no
 * memory pool), or a latency-critical loop that must not call cudaMalloc/
 * cudaFree, which synchronize the device. The caller passes inputs and
 * outputs as in sdtw_forward; the scratch comes from one 64 MiB file-scope
 * device array inside the library, which every GPU that loads the library
 * holds until the process exits.
 *  - Sizes whose forward scratch exceeds 64 MiB return SDTW_ERR_TOO_LARGE
 *    before any launch (for example B=4, N=M=64 fits; B=32, N=M=512 does not).
 *  - The first call on each device, with that device current, looks up the
 *    array's device address (cudaGetSymbolAddress); make that first call
 *    before any stream capture.
 *  - The looked-up address belongs to the device's current context: it is not
 *    valid across cudaDeviceReset (the array may move when the module loads
 *    again).
 *  - All calls share the array and it keeps the last call's contents; the
 *    control words are cleared at the start of each call. Calls that overlap
 *    on the GPU (other streams, other host threads) race on it.
 *  - No state is left for sdtw_backward. A device-side wait that runs out of
 *    time makes every loss of the call NaN (there is no workspace status word
 *    to read); sdtw_debug_set_wait applies to this entry too. */
sdtw_status sdtw_forward_noalloc(const float* x, const float* y, int B, int N, int M, int D,
                                 float gamma, sdtw_mode mode, float* loss, void* stream);

/* Soft-DTW on a caller-supplied cost tensor C (B,N,M), row-major: any
 * discrepancy, not only the squared Euclidean one (the SoftDTW README's `dist=`
 * argument, "Usage"; Soft-DTW paper, section 2). loss[b] = R_b[N,M] with
 * R[i,j] = C[b,i,j] + softmin_g(R[i-1,j-1], R[i-1,j], R[i,j-1]).
 * mode: SDTW_UNFUSED, optionally OR-ed with SDTW_EXTENDED; SDTW_FUSED is
 * SDTW_ERR_ARG (there is no cost to fuse). Workspace: op SDTW_OP_COST. Leaves the
 * DP state for sdtw_backward_cost in `ws`. */
sdtw_status sdtw_forward_cost(const float* C, int B, int N, int M, float gamma, sdtw_mode mode,
                              float* loss, void* ws, size_t ws_bytes, void* stream);

/* Backward pass of sdtw_forward_cost on the same workspace and arguments:
 * grad_C[b,i,j] = grad_loss[b] * E_b[i,j] = dL/dC[b,i,j] (B,N,M), row-major,
 * overwritten. */
sdtw_status sdtw_backward_cost(const float* C, int B, int N, int M, float gamma, sdtw_mode mode,
                               const float* grad_loss, float* grad_C, void* ws, size_t ws_bytes,
                               void* stream);

/* Bytes of device workspace needed by sdtw_value_and_grad_host; 0 when the
 * arguments are invalid. Pure host function, no CUDA call. */
size_t sdtw_host_workspace_bytes(int B, int N, int M, int D, sdtw_mode mode, int chunks);

/* Loss and input gradients of a batch that lives in HOST memory: the training
 * step of the SoftDTW README's "Usage" (loss of a batch, then its backward) with
 * the host<->device copies included. x (B,N,D), y (B,M,D) and grad_loss (B,)
 * are read from host memory; loss (B,), grad_x (B,N,D) and grad_y (B,M,D) are
 * written to host memory (grad_x / grad_y may be NULL; grad_loss may be NULL
 * only when both are). Use page-locked host memory (cudaHostAlloc): pageable
 * buffers give the same results without overlap.
 * The batch is cut into `chunks` groups of problems (<= 0: 2; at most 8 and at
 * most B), each run on a stream of its own that copies its inputs in, runs
 * sdtw_forward and sdtw_backward and copies its outputs out, so the copies of one
 * chunk overlap the kernels of the others; each chunk's wavefronts are sized
 * for its share of the SMs. The wavefronts of a small batch are latency-bound
 * (each chunk takes about as long as the whole batch), so there more chunks
 * only delay the last one; large batches gain from more. The call is asynchronous on `stream` like every
 * other: the host outputs are complete once the stream reaches this point, and
 * the host inputs must stay unchanged until then.
 * `ws` (device, 256-byte aligned) holds at least sdtw_host_workspace_bytes(B, N,
 * M, D, mode, chunks) bytes; its status word (offset 0) gathers the chunks'
 * device status, so sdtw_last_device_status(ws, stream) reports a timed-out
 * wait of any chunk. */
sdtw_status sdtw_value_and_grad_host(const float* x, const float* y, const float* grad_loss, int B, int N,
                                     int M, int D, float gamma, sdtw_mode mode, float* loss,
                                     float* grad_x, float* grad_y, int chunks, void* ws,
                                     size_t ws_bytes, void* stream);

/* Synchronizes `stream`, then reports (and clears) the device status word kept
 * in `ws`: SDTW_OK, or SDTW_ERR_TIMEOUT when a DP kernel gave up waiting for a
 * neighbouring tile. */
sdtw_status sdtw_last_device_status(void* ws, void* stream);

/* Static description of a status code. */
const char* sdtw_status_string(sdtw_status s);

/* Testing hook. Sets the time limit of every device-side wait (seconds; <= 0
 * restores the default of 2 s) and, when `skip_publish` is non-zero, makes the
 * next sdtw_forward withhold the ready flags of the first strip so that waiting
 * tiles run out of time and the call reports SDTW_ERR_TIMEOUT through
 * sdtw_last_device_status. No GPU fault is involved. Process-wide. */
void sdtw_debug_set_wait(double seconds, int skip_publish);

/* Testing hook. Forces choices the library otherwise makes itself, so that tests
 * reach every kernel on small inputs: warps_fwd / warps_bwd > 0 fix the warps per
 * wavefront CTA of the forward / backward (and with them the number of strips of
 * a problem, whose boundaries pass through global memory); dist_simt / fused_simt
 * non-zero select the difference-form cost kernels instead of the tensor-core
 * ones in the unfused / fused modes, fp32 and extended (with fused_simt the
 * checkpoint flag is SDTW_ERR_ARG). All zeros restore the library's own choices. Process-wide, read
 * by the calls that follow; set it while no other host thread calls the library. */
void sdtw_debug_set_options(int warps_fwd, int warps_bwd, int dist_simt, int fused_simt);

/* Testing hook. Caps the CTAs per thread-block cluster of the fused fp32 forward
 * with tensor-core costs: consecutive strips of a problem in one cluster pass their
 * boundary rows through each other's shared memory instead of global memory (the
 * other wavefront kernels always use global memory between strips). 0: the
 * library's own choice (up to 4, when every cluster of the launch can be resident
 * at once); 1: no clusters; 2: at most 2. Process-wide, read by the calls that
 * follow; set it while no other host thread calls the library. */
void sdtw_debug_set_clusters(int max_cluster);

/* Testing hook. out[i] = 2^x[i] (n device floats each) by the library's own
 * exponential of the double-float path: Cody & Waite reduction x = k + f, k the
 * nearest integer, |f| <= 1/2, then a degree-7 polynomial in f fitted to 2^f,
 * exponent added to the bits. Its error bound, stated for x in [-125, 0]:
 * within 2 ulp of the correctly rounded value; 0 for x < -125. */
sdtw_status sdtw_debug_exp2_neg(const float* x, float* out, int n, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* SDTW_H */
