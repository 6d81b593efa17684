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

constexpr int kDistWarps = 8;   // column tiles of 32 per CTA (one per warp), at most

// grid: (ceil(M / (32*nw)), NB, P), block 32*nw (nw <= kDistWarps warps).
// A CTA takes one 32-row block and 32*nw columns. Lane j of warp w holds
// the y row of column c0 = 32*(blockIdx.x*kDistWarps + w) + j in registers
// (DX > 0) and walks the 32 x rows, read from shared memory by every lane at
// once (broadcast); the 32x32 tile then goes through shared memory into the
// skewed layout. Rows are zero-padded to D32 = roundup(D, 32) components.
template <int DX>
__global__ void __launch_bounds__(32 * kDistWarps) dist_skew_kernel(Problems pr, int N, int M, int D,
                                                                   float* __restrict__ Dsk)
{
    extern __shared__ __align__(16) float sm[];
    const int D32 = (D + 31) & ~31, XS = D32 + 4;
    float* xs = sm;                                  // [32][XS] rows of the block
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float* tile = sm + 32 * XS + warp * 32 * 32;     // [32 rows][32 cols] per warp
    const int nw = blockDim.x >> 5;
    float* yw = sm + 32 * XS + nw * 1024 + warp * 32 * XS;  // [32][XS] y rows (DX == 0)
    const int p = blockIdx.z, rb = blockIdx.y;
    const int c0 = 32 * (blockIdx.x * nw + warp);
    const int r0 = rb * 32;
    const float* xb = pr.x(p);
    const float* yb = pr.y(p);
    stage_rows(xs, XS, xb, D, r0, 32, D32, N, threadIdx.x, blockDim.x);
    const int j = c0 + lane;
    float yr[DX > 0 ? DX : 1];
    if constexpr (DX > 0) {
#pragma unroll
        for (int k = 0; k < DX; ++k) yr[k] = (j < M && k < D) ? yb[(size_t)j * D + k] : 0.f;
    } else {
        stage_rows(yw, XS, yb, D, c0, 32, D32, M, lane, 32);
    }
    __syncthreads();
    if (c0 < M) {
        // d(x_i, y_j): the same arithmetic as the fused forward (x minus y)
        for (int i = 0; i < 32; ++i) {
            float v;
            if constexpr (DX > 0) {
                // dist_reg subtracts the shared row from the register row; (y - x)^2 == (x - y)^2
                v = dist_reg<DX>(yr, xs + i * XS);
            } else {
                v = dist_rows(xs + i * XS, yw + lane * XS, D32);
            }
            tile[i * 32 + lane] = v;
        }
        __syncwarp();
        // skewed slot t = col + row: lane = row, t = c0 + to
        float* out = Dsk + skew_index(N, M, p, rb, 0, lane);
        for (int to = 0; to < 63; ++to) {
            const int cc = to - lane;  // column within the tile for this lane's row
            if (cc >= 0 && cc < 32 && c0 + cc < M && r0 + lane < N)
                out[(long long)(c0 + to) * 32] = tile[lane * 32 + cc];
        }
    }
}

}  // namespace

namespace {

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
    const int D32 = (D + 31) & ~31, XS = D32 + 4;
    const int dx = (D <= 32) ? 32 : (D <= 64 ? 64 : 0);
    auto bytes = [&](int nw) {
        size_t b = (size_t)(32 * XS + nw * 1024) * sizeof(float);
        if (dx == 0) b += (size_t)nw * 32 * XS * sizeof(float);
        return b;
    };
    int nw = kDistWarps;
    while (nw > 1 && bytes(nw) > 220 * 1024) --nw;
    const size_t smem = bytes(nw);
    dim3 grid((M + 32 * nw - 1) / (32 * nw), (N + 31) / 32, P);
    auto go = [&](auto kern) -> cudaError_t {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        kern<<<grid, 32 * nw, smem, st>>>(pr, N, M, D, Dsk);
        return cudaGetLastError();
    };
    return dx == 32 ? go(dist_skew_kernel<32>) : dx == 64 ? go(dist_skew_kernel<64>) : go(dist_skew_kernel<0>);
}

cudaError_t launch_dist_rowmajor(const Problems& pr, int P, int N, int M, int D, float* C, cudaStream_t st)
{
    dim3 grid((M + 31) / 32, (N + 7) / 8, P);
    dist_rowmajor_kernel<<<grid, dim3(32, 8), 0, st>>>(pr, N, M, D, C);
    return cudaGetLastError();
}

}  // namespace sdtw
