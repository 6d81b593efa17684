// cost.cu -- Soft-DTW on a caller-supplied cost tensor.
//
// The recursion of the forward and backward wavefronts does not care where the
// cost comes from: any (B,N,M) tensor C can be aligned (the pages' `dist=`
// argument of SoftDTW, SoftDTW-CUDA (PyTorch + Numba) README, "Usage"; Soft-DTW
// paper, section 2, where the discrepancy matrix is any cost). The two kernels
// here move between the caller's row-major tensors and the skewed layout the
// wavefronts read and write:
//   skew_cost_kernel   C (row-major)  -> cost slots (float, or (c, 0) pairs for the
//                                         extended precision mode)
//   unskew_grad_kernel E slots        -> grad_C[b,i,j] = grad_loss[b] * E[b,i,j]
// Each CTA moves one 32x32 tile through shared memory: the row-major side is read
// or written a 128-byte row at a time, the skewed side one 128-byte slot row at a
// time (partial at the tile's left and right edges).
#include "common.cuh"
#include "kernels.h"

namespace sdtw {

namespace {

// grid (ceil(M/32), NB, P), block (32, 8).
template <bool EXT>
__global__ void __launch_bounds__(256) skew_cost_kernel(const float* __restrict__ C, int N, int M, float* __restrict__ Dsk)
{
    __shared__ float tile[32][33];
    const int p = blockIdx.z, rb = blockIdx.y, c0 = blockIdx.x * 32;
    const int tx = threadIdx.x, ty = threadIdx.y;
    for (int r = ty; r < 32; r += 8) {
        const int i = rb * 32 + r, j = c0 + tx;
        tile[r][tx] = (i < N && j < M) ? C[((size_t)p * N + i) * M + j] : 0.f;
    }
    __syncthreads();
    // slot c0 + t of block rb holds column (t - lane) of row (32 rb + lane)
    const int lane = tx;
    const int i = rb * 32 + lane;
    const long long base = skew_index(N, M, p, rb, c0, lane);
    for (int t = ty; t < 63; t += 8) {
        const int jj = t - lane;
        if (jj >= 0 && jj < 32 && c0 + jj < M && i < N) {
            const float v = tile[lane][jj];
            if (EXT) reinterpret_cast<float2*>(Dsk)[base + (long long)t * 32] = make_float2(v, 0.f);
            else Dsk[base + (long long)t * 32] = v;
        }
    }
}

// grid (ceil(M/32), NB, P), block (32, 8).
__global__ void __launch_bounds__(256) unskew_grad_kernel(const float* __restrict__ E, int N, int M,
                                                          const float* __restrict__ grad_loss,
                                                          float* __restrict__ gC)
{
    __shared__ float tile[32][33];
    const int p = blockIdx.z, rb = blockIdx.y, c0 = blockIdx.x * 32;
    const int tx = threadIdx.x, ty = threadIdx.y;
    const int lane = tx;
    const int i = rb * 32 + lane;
    const long long base = skew_index(N, M, p, rb, c0, lane);
    for (int t = ty; t < 63; t += 8) {
        const int jj = t - lane;
        if (jj >= 0 && jj < 32 && c0 + jj < M && i < N) tile[lane][jj] = E[base + (long long)t * 32];
    }
    __syncthreads();
    const float g = grad_loss[p];
    for (int r = ty; r < 32; r += 8) {
        const int ii = rb * 32 + r, j = c0 + tx;
        if (ii < N && j < M) gC[((size_t)p * N + ii) * M + j] = g * tile[r][tx];
    }
}

}  // namespace

cudaError_t launch_skew_cost(const float* C, int P, int N, int M, bool ext, float* Dsk, cudaStream_t st)
{
    dim3 grid((M + 31) / 32, (N + 31) / 32, P), block(32, 8);
    if (ext) skew_cost_kernel<true><<<grid, block, 0, st>>>(C, N, M, Dsk);
    else skew_cost_kernel<false><<<grid, block, 0, st>>>(C, N, M, Dsk);
    return cudaGetLastError();
}

cudaError_t launch_unskew_grad(const float* E, int P, int N, int M, const float* grad_loss, float* gC, cudaStream_t st)
{
    dim3 grid((M + 31) / 32, (N + 31) / 32, P), block(32, 8);
    unskew_grad_kernel<<<grid, block, 0, st>>>(E, N, M, grad_loss, gC);
    return cudaGetLastError();
}

}  // namespace sdtw
