// dist.cu -- squared Euclidean cost for the unfused mode.
//
// C[i,j] = sum_k (x_i[k] - y_j[k])^2, computed in the difference form (every
// term is a square, so the fp32 sum has no cancellation), written straight into
// the skewed layout that the forward wavefront reads one 128-byte row per step.
// (SoftDTW-CUDA (PyTorch + Numba) README, "Notes" and "Basic (Unfused)"; review
// page, "proposed method", fourth bullet: the unfused mode precomputes and
// stores the full distance tensor.)
#include "common.cuh"
#include "kernels.h"

namespace sdtw {

namespace {

constexpr int kDistT = 64;      // skewed rows per CTA
constexpr int kDistWarps = 8;   // each warp covers kDistT / kDistWarps skewed rows

// grid: (ceil((M+31)/kDistT), NB, P), block: 32*kDistWarps.
__global__ void __launch_bounds__(32 * kDistWarps) dist_skew_kernel(Problems pr, int N, int M, int D,
                                                                   float* __restrict__ Dsk)
{
    extern __shared__ float sm[];
    const int XS = D + 1;
    float* xs = sm;                     // [32][XS]
    float* ys = sm + 32 * XS;           // [kDistT + 31][XS], y rows jbase .. jbase + kDistT + 30
    const int p = blockIdx.z, rb = blockIdx.y, t0 = blockIdx.x * kDistT;
    const int T = M + 31;
    const int r0 = rb * 32, jbase = t0 - 31;
    const float* xb = pr.x(p);
    const float* yb = pr.y(p);
    for (int e = threadIdx.x; e < 32 * D; e += blockDim.x) {
        const int r = e / D, k = e - r * D;
        xs[r * XS + k] = (r0 + r < N) ? xb[(size_t)(r0 + r) * D + k] : 0.f;
    }
    const int ny = kDistT + 31;
    for (int e = threadIdx.x; e < ny * D; e += blockDim.x) {
        const int r = e / D, k = e - r * D;
        const int j = jbase + r;
        ys[r * XS + k] = (j >= 0 && j < M) ? yb[(size_t)j * D + k] : 0.f;
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int TPW = kDistT / kDistWarps;
    DistAcc acc[TPW];
    const int tw = t0 + warp * TPW;
    // lane handles row r0+lane, columns j = t - lane for t in [tw, tw+TPW)
    const int yrow0 = tw - lane - jbase;  // ys row of the first column, in [0, ny)
    for (int k0 = 0; k0 < D; k0 += kDistBlock) {
        const int k1 = min(k0 + kDistBlock, D);
        float blk[TPW];
#pragma unroll
        for (int u = 0; u < TPW; ++u) blk[u] = 0.f;
        for (int k = k0; k < k1; ++k) {
            const float xv = xs[lane * XS + k];
#pragma unroll
            for (int u = 0; u < TPW; ++u) {
                const float a = xv - ys[(yrow0 + u) * XS + k];
                blk[u] = fmaf(a, a, blk[u]);
            }
        }
#pragma unroll
        for (int u = 0; u < TPW; ++u) acc[u].add_block(blk[u]);
    }
    float* out = Dsk + skew_index(N, M, p, rb, 0, lane);
#pragma unroll
    for (int u = 0; u < TPW; ++u) {
        const int t = tw + u;
        if (t < T) out[(long long)t * 32] = acc[u].value();
    }
}

// grid: (ceil(M/32), ceil(N/8), P), block (32, 8).
__global__ void dist_rowmajor_kernel(Problems pr, int N, int M, int D, float* __restrict__ C)
{
    const int p = blockIdx.z;
    const int j = blockIdx.x * 32 + threadIdx.x;
    const int i = blockIdx.y * 8 + threadIdx.y;
    if (i >= N || j >= M) return;
    const float* xi = pr.x(p) + (size_t)i * D;
    const float* yj = pr.y(p) + (size_t)j * D;
    DistAcc acc;
    for (int k0 = 0; k0 < D; k0 += kDistBlock) {
        float blk = 0.f;
        for (int k = k0; k < min(k0 + kDistBlock, D); ++k) {
            const float a = xi[k] - yj[k];
            blk = fmaf(a, a, blk);
        }
        acc.add_block(blk);
    }
    C[((size_t)p * N + i) * M + j] = acc.value();
}

}  // namespace

cudaError_t launch_dist_skewed(const Problems& pr, int P, int N, int M, int D, float* Dsk, cudaStream_t st)
{
    const int T = M + 31;
    dim3 grid((T + kDistT - 1) / kDistT, (N + 31) / 32, P);
    const size_t smem = (size_t)(32 + kDistT + 31) * (D + 1) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(dist_skew_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dist_skew_kernel<<<grid, 32 * kDistWarps, smem, st>>>(pr, N, M, D, Dsk);
    return cudaGetLastError();
}

cudaError_t launch_dist_rowmajor(const Problems& pr, int P, int N, int M, int D, float* C, cudaStream_t st)
{
    dim3 grid((M + 31) / 32, (N + 7) / 8, P);
    dist_rowmajor_kernel<<<grid, dim3(32, 8), 0, st>>>(pr, N, M, D, C);
    return cudaGetLastError();
}

}  // namespace sdtw
