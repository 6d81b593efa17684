// kernels.h -- host-side declarations of the library's kernel launchers.
#pragma once
#include <cuda_runtime.h>

#include "common.cuh"

namespace sdtw {

// Parameters of the two wavefront kernels. All pointers are device pointers
// into the caller's tensors or the caller's workspace.
struct WaveParams {
    Problems pr;
    int P;            // problems in the batch
    int N, M, D;
    int NB;           // 32-row blocks per problem, ceil(N/32)
    int S;            // strips (CTAs) per problem, ceil(N / (32 W))
    int W;            // warps per CTA
    int smem_fixed;   // bytes of dynamic shared memory before the fused buffers
    float scale;      // log2(e) / gamma
    float unscale;    // gamma * ln(2)
    const float* Dsk; // unfused: raw cost, skewed layout; fused: nullptr
    float2* VH;       // (vl, hu) per cell, skewed layout (extended: float4 log2-probabilities)
    float* E;         // alignment matrix, skewed layout (backward output)
    Slot* edge_f;     // [P][S][M]     boundary rows between forward strips (tagged)
    Slot* edge_b;     // [P][S][M][2]  boundary messages between backward strips (tagged)
    int* ticket_f;    // forward strip ticket
    int* ticket_b;    // backward strip ticket
    int* done;        // [P]         finished forward strips
    double* colsum;   // [P][NB]
    double* rowsum;   // [P]  (unused)
    float* rowbuf;    // [P][M]      h of the last row, for the loss
    float* loss;      // [P]
    int* status;      // device status word
    unsigned long long wait_ns;
    int skip_publish; // test hook: strip 0 withholds its forward ready counter
    int ext;          // 1: extended-precision forward state (wavefront_x.cu)
    const int* lens_n; // per-problem lengths of x and y (device, P each), or null: every
    const int* lens_m; // problem spans N x M. A problem aligns its leading N_b x M_b block.
    // Band launches of the checkpointed backward: this launch covers strips
    // [strip0, strip0 + S) of S_all strips per problem, and VH / E hold only row
    // blocks [vh_rb0, vh_rb0 + vh_nb) of every problem. Zeros: the whole problem.
    int strip0, S_all, vh_rb0, vh_nb;
    int no_loss;       // 1: a recompute of stored boundary rows; no loss is assembled
    // Fused tensor-core forward: CTAs per thread-block cluster (1: none). A cluster
    // takes one ticket and runs C consecutive strips of a problem, by cluster rank;
    // the boundary row between two of them goes through the consumer CTA's shared
    // memory. The other wavefront kernels ignore it.
    int C;
};

// Strips per problem for the boundary-row buffers.
__host__ __device__ inline int strips_all(const WaveParams& q) { return q.S_all > 0 ? q.S_all : q.S; }

// Index of (problem p, row block rb, step 0, lane) in the VH / E buffers: the skewed
// layout restricted to the launch's band of row blocks.
__host__ __device__ inline long long band_index(const WaveParams& q, int p, int rb, int lane, int T)
{
    const int nb = q.vh_nb > 0 ? q.vh_nb : q.NB;
    return ((long long)p * nb + (rb - q.vh_rb0)) * T * 32 + lane;
}

// Device-wait settings of sdtw_debug_set_wait (api.cu): the time limit of every
// bounded wait, and the one-shot request that the next forward's first strip
// withhold its ready flags (read and cleared by the call that launches it).
unsigned long long debug_wait_ns();
int debug_take_skip_publish();

size_t wave_smem_fixed(int W, bool backward);
size_t wave_smem_fused_per_warp(int D);
size_t wave_smem_floor();
size_t wavex_smem_fused_per_warp(int D);
cudaError_t launch_forward_x(WaveParams q, bool fused, cudaStream_t st);
cudaError_t launch_dist_skewed_x(const Problems& pr, int P, int N, int M, int D, float2* Dsk, cudaStream_t st);
cudaError_t launch_forward(WaveParams q, bool fused, cudaStream_t st);
// The double-float backward takes at most 12 warps per CTA: its ~166 registers per
// thread fit 384 threads (a 512-thread build, capped at 128 registers, spills).
constexpr int kMaxWarpsBwdExt = 12;
cudaError_t launch_backward(WaveParams q, cudaStream_t st);

// Unfused cost: raw squared Euclidean distances into the skewed layout.
cudaError_t launch_dist_skewed(const Problems& pr, int P, int N, int M, int D, float* Dsk,
                               cudaStream_t st);
// Cost matrix (P,N,M) row-major.
cudaError_t launch_dist_rowmajor(const Problems& pr, int P, int N, int M, int D, float* C,
                                 cudaStream_t st);

// Gradient contractions from the skewed alignment matrix.
//   row part, for each problem p and row i:
//     out_x[p][i,:] (+)= coef * w[p] * 2 * (sum_j E[i,j] x_i - sum_j E[i,j] y_j)
//   column part, for each problem p and column j:
//     out_y[p][j,:] (+)= coef * w[p] * 2 * (sum_i E[i,j] y_j - sum_i E[i,j] x_i)
// w[p] = grad_loss[p % wmod] (1 when grad_loss is NULL). out + (p % omod) * stride.
struct GradParams {
    Problems pr;
    int P, N, M, D;
    const float* E;
    const float* grad_loss;
    int wmod;
    float coef;
    float* out;
    long long out_stride;
    int omod;
    int accumulate;
    // per problem and 32-row block, the column range [x, y] where E may be non-zero
    // (launch_ebounds); null: every column
    const int2* bounds;
};
cudaError_t launch_grad_rows(const GradParams& g, cudaStream_t st);
// The column ranges of GradParams::bounds for the g.P problems of g.E (difference-form
// contractions visit only the tiles inside them).
cudaError_t launch_ebounds(const GradParams& g, int2* bounds, cudaStream_t st);
// The same contractions on the tensor cores (tcgen05, 3xTF32); cols selects grad_y.
// Pre-split B operand images: [Y | 1] into img_rows (for grad_x) and [X | 1]
// into img_cols (for grad_y), one launch; a null pointer skips that image.
// Each buffer takes egemm_bimg_bytes(P, K, D) with K = M (rows) or N (cols).
cudaError_t launch_bimg(const GradParams& g, float* img_rows, float* img_cols, cudaStream_t st);
// bimg: the image for this orientation, written by launch_bimg before.
cudaError_t launch_grad_tc(const GradParams& g, bool cols, const float* bimg, int* status, cudaStream_t st);
size_t egemm_bimg_bytes(int P, int K, int D);

// Tensor-core cost tensor (dist_tc.cu), D <= kTcKFeat * kMaxTcKBlocks: operand
// images of x and y (simg_bytes each), their squared row norms (snorm_bytes each),
// then the skewed cost tensor. status receives kStatusTimeout if a bounded wait
// expires. Beyond that width the difference-form kernels compute the costs.
constexpr int kTcKFeat = 64;      // features per K-block of the bf16 operand images
constexpr int kMaxTcKBlocks = 1;  // D <= 64: the fp32 state's parity needs exact costs beyond
size_t simg_bytes(int P, int L, int D);
// Operand image layout (bytes): per problem, per K-block of 64 features, the three
// bf16 parts v = v0 + v1 + v2, each Lpad = roundup(L, 128) rows of 128 bytes (64
// bf16; 16-byte chunks swizzled by row mod 8); row norms (fp32) at p * Lpad + r.
__host__ __device__ inline size_t simg_offset(int p, int KB, int kb, int part, int Lpad, int r)
{
    return ((((size_t)p * KB + kb) * 3 + part) * (size_t)Lpad + (size_t)r) * 128;
}
__host__ __device__ inline int simg_pad(int L) { return (L + 127) / 128 * 128; }
size_t snorm_bytes(int P, int L);
cudaError_t launch_simg(const Problems& pr, int P, int N, int M, int D, void* ximg, void* yimg, float* xnorm,
                        float* ynorm, cudaStream_t st);
cudaError_t launch_dist_tc(int P, int N, int M, int D, const void* ximg, const void* yimg, const float* xnorm,
                           const float* ynorm, float* Dsk, int* status, cudaStream_t st);

// Exact fixed-point operand images for the extended fused forward (wavefront_x.cu),
// per problem, per K-block of 64 features, NS = xtc_slices(D) bf16 digit slices
// (5 up to D = 128, 6 above), each Lpad rows of 128 bytes
// (swizzled as the bf16 images above); per row the info (norm hi, norm lo, scale
// exponent as int bits, 0).
constexpr int kMaxXtcD = 400;    // exact tensor-core costs, both modes (six digits above D = 128)
int xtc_slices(int D);
__host__ __device__ inline size_t oimg_offset(int p, int KB, int kb, int NS, int slice, int Lpad, int r)
{
    return ((((size_t)p * KB + kb) * NS + slice) * (size_t)Lpad + (size_t)r) * 128;
}
size_t oimg_bytes(int P, int L, int D);
size_t oinfo_bytes(int P, int L);
cudaError_t launch_oimg(const Problems& pr, int P, int N, int M, int D, void* ximg, void* yimg, void* xinfo,
                        void* yinfo, cudaStream_t st);
// Extended unfused cost tensor from the exact tensor-core level sums (D <= kMaxXtcD):
// raw double-float costs (hi, lo) in the skewed layout.
cudaError_t launch_dist_xtc(int P, int N, int M, int D, const void* ximg, const void* yimg, const void* xinfo,
                            const void* yinfo, float2* Dsk, int* status, cudaStream_t st);
// Extended fused forward with exact tensor-core cost tiles (D <= kMaxXtcD): q.W must be 4.
cudaError_t launch_forward_xtc(WaveParams q, const void* ximg, const void* yimg, const void* xinfo,
                               const void* yinfo, cudaStream_t st);

// Fused forward with tensor-core cost tiles (wavefront_tc.cu): q.W must be 4
// (128-row strips), D <= 64; the operand images and norms as for launch_dist_tc.
cudaError_t launch_forward_tc(WaveParams q, const void* ximg, const void* yimg, const float* xnorm,
                              const float* ynorm, cudaStream_t st);
size_t wave_tc_smem(int D);

// Caller-supplied costs (cost.cu): C (P,N,M) row-major into the skewed cost slots
// (float, or (c, 0) pairs when ext), and grad_C = grad_loss[p] * E back out.
// Barycenter Adam step with the gradient clipped by its global L2 norm
// (max_norm > 0); partials: ceil(n/256) floats of scratch.
cudaError_t launch_adam_clipped(float* z, float* m, float* v, float* gparts, int K, int n, float lr, float beta1,
                                float beta2, float eps, float bc1, float bc2, float max_norm, float* partials,
                                const float* losses, float* loss_out, cudaStream_t st);

cudaError_t launch_skew_cost(const float* C, int P, int N, int M, bool ext, float* Dsk, cudaStream_t st);
cudaError_t launch_unskew_grad(const float* E, int P, int N, int M, const float* grad_loss, float* gC,
                               cudaStream_t st);
cudaError_t launch_grad_cols(const GradParams& g, cudaStream_t st);

// Barycenter: grad = (1/K) sum_k gparts[k]; Adam update of z, m, v; mean loss.
cudaError_t launch_adam(float* z, float* m, float* v, const float* gparts, int K, int n,
                        float lr, float beta1, float beta2, float eps, float bc1, float bc2,
                        const float* losses, float* loss_out, cudaStream_t st);

}  // namespace sdtw
