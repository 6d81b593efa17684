// grad.cu -- input gradients from the alignment matrix in difference form, and
// the barycenter Adam step.
//
// Chain rule through the squared Euclidean cost C[i,j] = |x_i - y_j|^2:
//   dL/dx_i = g * 2 * sum_j E[i,j] (x_i - y_j),   dL/dy_j = g * 2 * sum_i E[i,j] (y_j - x_i).
// These kernels keep the difference form term by term. The GEMM form
// rowsum_i(E) x_i - (E y)_i (egemm.cu) cancels badly where one row aligns to
// many columns (stretched warps, rowsum >> 1): at N=M=8192 its fp32 sums miss
// rel 1e-3 on such rows while the difference form does not. The extended
// precision path therefore uses these kernels.
// E arrives in the skewed layout of the wavefront; each CTA un-skews 32x32
// tiles into shared memory and contracts them with the matching x or y rows.
#include "common.cuh"
#include "kernels.h"

namespace sdtw {

namespace {

constexpr int kKC = 64;   // k-slice per CTA (16 per warp)
constexpr int kYS = kKC + 4;

// Un-skew the 32x32 tile (rows of block rb, columns c0..c0+31) into es.
// ROW_MAJOR: es[r*32 + c]; otherwise es[c*32 + r]. Entries outside the matrix are 0.
// Returns whether this thread stored a non-zero value: away from the alignment
// path E underflows to exactly 0, and a tile that is all zero adds nothing.
// The tile spans 63 skewed rows of 32 lanes; each of the kGradThreads threads
// issues all of its loads before any store, so a tile costs one memory latency.
constexpr int kGradThreads = 128;
template <bool ROW_MAJOR>
__device__ __forceinline__ bool load_tile(const float* __restrict__ Esk, int N, int M, int p, int rb, int c0,
                                          float* es)
{
    constexpr int kIters = (63 * 32 + kGradThreads - 1) / kGradThreads;
    const float* base = Esk + skew_index(N, M, p, rb, 0, 0);
    float v[kIters];
#pragma unroll
    for (int u = 0; u < kIters; ++u) {
        const int idx = threadIdx.x + u * kGradThreads;
        const int tt = idx >> 5, rr = idx & 31;
        const int c = tt - rr;
        const bool ok = idx < 63 * 32 && c >= 0 && c < 32 && (c0 + c < M) && (rb * 32 + rr < N);
        v[u] = ok ? base[(long long)(c0 + tt) * 32 + rr] : 0.f;
    }
    bool nz = false;
#pragma unroll
    for (int u = 0; u < kIters; ++u) {
        const int idx = threadIdx.x + u * kGradThreads;
        const int tt = idx >> 5, rr = idx & 31;
        const int c = tt - rr;
        if (idx < 63 * 32 && c >= 0 && c < 32) {
            nz = nz || (v[u] != 0.f);
            if (ROW_MAJOR) es[rr * 32 + c] = v[u];
            else es[c * 32 + rr] = v[u];
        }
    }
    return nz;
}

// Column range of the non-zero E of each 32-row block: away from the alignment path
// E underflows to exactly 0, so the contractions below need only the tiles between
// the first and the last non-zero column of a row block. One warp scans kBoundSeg
// skewed rows of one block (its loads in batches of 8); atomics combine the segments.
constexpr int kBoundSeg = 512;
__global__ void ebounds_init_kernel(int2* b, int n)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) b[i] = make_int2(0x7fffffff, -1);
}

// grid (ceil(NB/8), P, ceil(T/kBoundSeg)), block 256.
__global__ void __launch_bounds__(256) ebounds_kernel(const float* __restrict__ Esk, int N, int M, int2* bounds)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NB = (N + 31) / 32, T = skew_T(M);
    const int rb = blockIdx.x * 8 + warp, p = blockIdx.y;
    if (rb >= NB) return;
    const int t0 = blockIdx.z * kBoundSeg, t1 = min(T, t0 + kBoundSeg);
    const bool row_ok = rb * 32 + lane < N;
    const float* base = Esk + skew_index(N, M, p, rb, 0, lane);
    int lo = 0x7fffffff, hi = -1;
    for (int t = t0; t < t1; t += 8) {
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = (t + u < t1) ? base[(long long)(t + u) * 32] : 0.f;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int j = t + u - lane;
            if (v[u] != 0.f && row_ok && j >= 0 && j < M) {
                lo = min(lo, j);
                hi = max(hi, j);
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
        hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    if (lane == 0 && hi >= 0) {
        int* b = reinterpret_cast<int*>(bounds + (size_t)p * NB + rb);
        atomicMin(b, lo);
        atomicMax(b + 1, hi);
    }
}

// grid (NB, P, ceil(D/64)), block 128.
__global__ void __launch_bounds__(kGradThreads, 4) grad_rows_kernel(const GradParams g)
{
    __shared__ float es[32 * 32];
    __shared__ __align__(16) float ys[32 * kYS];
    const int rb = blockIdx.x, p = blockIdx.y, kb = blockIdx.z * kKC;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int N = g.N, M = g.M, D = g.D;
    const float* yb = g.pr.y(p);
    const int i = rb * 32 + lane;
    float xi[16];
    const float* xrow = g.pr.x(p) + (size_t)min(i, N - 1) * D;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const int kk = kb + warp * 16 + k;
        xi[k] = (kk < D) ? xrow[kk] : 0.f;
    }
    float acc[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) acc[k] = 0.f;
    int c_first = 0, c_last = M - 1;   // the block's non-zero columns (CTA-uniform)
    if (g.bounds) {
        const int2 bb = g.bounds[(size_t)p * ((N + 31) / 32) + rb];
        c_first = bb.x & ~31;
        c_last = bb.y;
    }
    for (int c0 = c_first; c0 <= c_last; c0 += 32) {
        if (!__syncthreads_or(load_tile<false>(g.E, N, M, p, rb, c0, es))) continue;  // an all-zero tile
        {   // the tile's 32 y rows, k-slice kb: all loads before the stores
            float v[32 * kKC / kGradThreads];
#pragma unroll
            for (int u = 0; u < 32 * kKC / kGradThreads; ++u) {
                const int idx = threadIdx.x + u * kGradThreads, c = idx / kKC, kk = idx - c * kKC;
                v[u] = (c0 + c < M && kb + kk < D) ? yb[(size_t)(c0 + c) * D + kb + kk] : 0.f;
            }
#pragma unroll
            for (int u = 0; u < 32 * kKC / kGradThreads; ++u) {
                const int idx = threadIdx.x + u * kGradThreads, c = idx / kKC, kk = idx - c * kKC;
                ys[c * kYS + kk] = v[u];
            }
        }
        __syncthreads();
#pragma unroll 4
        for (int c = 0; c < 32; ++c) {
            const float e = es[c * 32 + lane];
            const float4* yv = reinterpret_cast<const float4*>(ys + c * kYS + warp * 16);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 w = yv[q];
                acc[4 * q + 0] = fmaf(e, xi[4 * q + 0] - w.x, acc[4 * q + 0]);
                acc[4 * q + 1] = fmaf(e, xi[4 * q + 1] - w.y, acc[4 * q + 1]);
                acc[4 * q + 2] = fmaf(e, xi[4 * q + 2] - w.z, acc[4 * q + 2]);
                acc[4 * q + 3] = fmaf(e, xi[4 * q + 3] - w.w, acc[4 * q + 3]);
            }
        }
        __syncthreads();
    }
    if (i >= N) return;
    const float w = g.coef * 2.f * (g.grad_loss ? g.grad_loss[p % g.wmod] : 1.f);
    float* out = g.out + (long long)(p % g.omod) * g.out_stride + (size_t)i * D;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const int kk = kb + warp * 16 + k;
        if (kk < D) {
            const float val = w * acc[k];
            out[kk] = g.accumulate ? out[kk] + val : val;
        }
    }
}

// grid (ceil(M/32), P, ceil(D/64)), block 128.
__global__ void __launch_bounds__(kGradThreads, 4) grad_cols_kernel(const GradParams g)
{
    __shared__ float es[32 * 32];
    __shared__ __align__(16) float xs[32 * kYS];
    const int c0 = blockIdx.x * 32, p = blockIdx.y, kb = blockIdx.z * kKC;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int N = g.N, M = g.M, D = g.D;
    const float* xb = g.pr.x(p);
    const int j = c0 + lane;
    float yj[16];
    const float* yrow = g.pr.y(p) + (size_t)min(j, M - 1) * D;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const int kk = kb + warp * 16 + k;
        yj[k] = (kk < D) ? yrow[kk] : 0.f;
    }
    float acc[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) acc[k] = 0.f;
    const int NB = (N + 31) / 32;
    __shared__ int2 s_bnd[kGradThreads];   // the bounds of the next kGradThreads row blocks
    for (int rb = 0; rb < NB; ++rb) {
        if (g.bounds) {   // row blocks whose non-zero columns miss this column tile add nothing
            if ((rb % kGradThreads) == 0) {
                __syncthreads();
                const int r = rb + (int)threadIdx.x;
                s_bnd[threadIdx.x] = r < NB ? g.bounds[(size_t)p * NB + r] : make_int2(0x7fffffff, -1);
                __syncthreads();
            }
            const int2 bb = s_bnd[rb % kGradThreads];
            if (bb.y < c0 || bb.x > c0 + 31) continue;   // CTA-uniform
        }
        if (!__syncthreads_or(load_tile<true>(g.E, N, M, p, rb, c0, es))) continue;  // an all-zero tile
        {   // the tile's 32 x rows, k-slice kb: all loads before the stores
            float v[32 * kKC / kGradThreads];
#pragma unroll
            for (int u = 0; u < 32 * kKC / kGradThreads; ++u) {
                const int idx = threadIdx.x + u * kGradThreads, r = idx / kKC, kk = idx - r * kKC;
                const int i = rb * 32 + r;
                v[u] = (i < N && kb + kk < D) ? xb[(size_t)i * D + kb + kk] : 0.f;
            }
#pragma unroll
            for (int u = 0; u < 32 * kKC / kGradThreads; ++u) {
                const int idx = threadIdx.x + u * kGradThreads, r = idx / kKC, kk = idx - r * kKC;
                xs[r * kYS + kk] = v[u];
            }
        }
        __syncthreads();
#pragma unroll 4
        for (int r = 0; r < 32; ++r) {
            const float e = es[r * 32 + lane];
            const float4* xv = reinterpret_cast<const float4*>(xs + r * kYS + warp * 16);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 w = xv[q];
                acc[4 * q + 0] = fmaf(e, yj[4 * q + 0] - w.x, acc[4 * q + 0]);
                acc[4 * q + 1] = fmaf(e, yj[4 * q + 1] - w.y, acc[4 * q + 1]);
                acc[4 * q + 2] = fmaf(e, yj[4 * q + 2] - w.z, acc[4 * q + 2]);
                acc[4 * q + 3] = fmaf(e, yj[4 * q + 3] - w.w, acc[4 * q + 3]);
            }
        }
        __syncthreads();
    }
    if (j >= M) return;
    const float w = g.coef * 2.f * (g.grad_loss ? g.grad_loss[p % g.wmod] : 1.f);
    float* out = g.out + (long long)(p % g.omod) * g.out_stride + (size_t)j * D;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const int kk = kb + warp * 16 + k;
        if (kk < D) {
            const float val = w * acc[k];
            out[kk] = g.accumulate ? out[kk] + val : val;
        }
    }
}

// Barycenter: g = sum_k gparts[k] (each part already carries its 1/K), then Adam.
__global__ void adam_kernel(float* __restrict__ z, float* __restrict__ m, float* __restrict__ v,
                            const float* __restrict__ gparts, int K, int n, float lr, float b1, float b2,
                            float eps, float bc1, float bc2, const float* __restrict__ losses,
                            float* __restrict__ loss_out)
{
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e == 0 && loss_out) {
        double s = 0.0;
        for (int k = 0; k < K; ++k) s += losses[k];
        *loss_out = (float)(s / K);
    }
    if (e >= n) return;
    float gsum = 0.f;
    for (int k = 0; k < K; ++k) gsum += gparts[(size_t)k * n + e];
    const float mm = b1 * m[e] + (1.f - b1) * gsum;
    const float vv = b2 * v[e] + (1.f - b2) * gsum * gsum;
    m[e] = mm;
    v[e] = vv;
    z[e] -= lr * (mm / bc1) / (sqrtf(vv / bc2) + eps);
}

// Gradient clipping (by global L2 norm) for the barycenter step, in two launches:
// gsum_kernel sums the K parts of each element into part 0 (k order as in
// adam_kernel) and writes one partial sum of squares per block (fixed tree order);
// adam_clip_kernel adds the partials in block order, scales the gradient by
// min(1, max_norm / ||g||) and applies Adam. grid ceil(n/256), block 256.
__global__ void __launch_bounds__(256) gsum_kernel(float* __restrict__ gparts, int K, int n,
                                                   float* __restrict__ partials)
{
    __shared__ float red[256];
    const int e = blockIdx.x * 256 + threadIdx.x;
    float g = 0.f;
    if (e < n) {
        for (int k = 0; k < K; ++k) g += gparts[(size_t)k * n + e];
        gparts[e] = g;
    }
    red[threadIdx.x] = g * g;
    __syncthreads();
    for (int o = 128; o > 0; o >>= 1) {
        if (threadIdx.x < o) red[threadIdx.x] += red[threadIdx.x + o];
        __syncthreads();
    }
    if (threadIdx.x == 0) partials[blockIdx.x] = red[0];
}

__global__ void __launch_bounds__(256) adam_clip_kernel(float* __restrict__ z, float* __restrict__ m,
                                                        float* __restrict__ v, const float* __restrict__ g, int n,
                                                        float lr, float b1, float b2, float eps, float bc1, float bc2,
                                                        const float* __restrict__ partials, int nparts,
                                                        float max_norm, int K, const float* __restrict__ losses,
                                                        float* __restrict__ loss_out)
{
    __shared__ float s_scale;
    if (threadIdx.x == 0) {
        double s2 = 0.0;
        for (int b = 0; b < nparts; ++b) s2 += partials[b];
        const float nrm = (float)sqrt(s2);
        s_scale = (max_norm > 0.f && nrm > max_norm) ? max_norm / nrm : 1.f;
        if (blockIdx.x == 0 && loss_out) {
            double l = 0.0;
            for (int k = 0; k < K; ++k) l += losses[k];
            *loss_out = (float)(l / K);
        }
    }
    __syncthreads();
    const int e = blockIdx.x * 256 + threadIdx.x;
    if (e >= n) return;
    const float gg = g[e] * s_scale;
    const float mm = b1 * m[e] + (1.f - b1) * gg;
    const float vv = b2 * v[e] + (1.f - b2) * gg * gg;
    m[e] = mm;
    v[e] = vv;
    z[e] -= lr * (mm / bc1) / (sqrtf(vv / bc2) + eps);
}

}  // namespace

cudaError_t launch_adam_clipped(float* z, float* m, float* v, float* gparts, int K, int n, float lr, float beta1,
                                float beta2, float eps, float bc1, float bc2, float max_norm, float* partials,
                                const float* losses, float* loss_out, cudaStream_t st)
{
    const int blocks = (n + 255) / 256;
    gsum_kernel<<<blocks, 256, 0, st>>>(gparts, K, n, partials);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    adam_clip_kernel<<<blocks, 256, 0, st>>>(z, m, v, gparts, n, lr, beta1, beta2, eps, bc1, bc2, partials, blocks,
                                             max_norm, K, losses, loss_out);
    return cudaGetLastError();
}

cudaError_t launch_grad_rows(const GradParams& g, cudaStream_t st)
{
    dim3 grid((g.N + 31) / 32, g.P, (g.D + kKC - 1) / kKC);
    grad_rows_kernel<<<grid, kGradThreads, 0, st>>>(g);
    return cudaGetLastError();
}

cudaError_t launch_ebounds(const GradParams& g, int2* bounds, cudaStream_t st)
{
    const int NB = (g.N + 31) / 32, n = g.P * NB;
    ebounds_init_kernel<<<(n + 255) / 256, 256, 0, st>>>(bounds, n);
    dim3 grid((NB + 7) / 8, g.P, (skew_T(g.M) + kBoundSeg - 1) / kBoundSeg);
    ebounds_kernel<<<grid, 256, 0, st>>>(g.E, g.N, g.M, bounds);
    return cudaGetLastError();
}

cudaError_t launch_grad_cols(const GradParams& g, cudaStream_t st)
{
    dim3 grid((g.M + 31) / 32, g.P, (g.D + kKC - 1) / kKC);
    grad_cols_kernel<<<grid, kGradThreads, 0, st>>>(g);
    return cudaGetLastError();
}

cudaError_t launch_adam(float* z, float* m, float* v, const float* gparts, int K, int n, float lr,
                        float beta1, float beta2, float eps, float bc1, float bc2, const float* losses,
                        float* loss_out, cudaStream_t st)
{
    const int threads = 256;
    const int blocks = (n + threads - 1) / threads;
    adam_kernel<<<blocks > 0 ? blocks : 1, threads, 0, st>>>(z, m, v, gparts, K, n, lr, beta1, beta2, eps, bc1,
                                                             bc2, losses, loss_out);
    return cudaGetLastError();
}

}  // namespace sdtw
