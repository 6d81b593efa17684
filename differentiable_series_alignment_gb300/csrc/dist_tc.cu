// dist_tc.cu -- the pairwise cost tensor on the tensor cores, for feature widths
// up to 64 in the fp32 modes.
//
//   C[i,j] = |x_i|^2 + |y_j|^2 - 2 x_i . y_j
//
// (the expansion of the squared Euclidean distance; Soft-DTW paper, section 2,
// squared Euclidean discrepancy; SoftDTW-CUDA (PyTorch + Numba) README, "Basic
// (Unfused)", where the unfused mode materialises the whole cost tensor.)
//
// The dot products are a batched GEMM x . y^T with K = D. Each sequence is first
// written once as an operand image (simg_kernel): every row split into tf32
// hi + lo parts (round to nearest), stored in the 128-byte-swizzled K-major
// layout that tcgen05.mma reads, in K-blocks of 32 features, together with the
// squared norm of the row (compensated fp32: exact squares, TwoSum partial
// sums). A cost CTA (dist_tc_kernel) bulk-copies the 128 x-rows and 128 y-rows of its tile into
// shared memory and one thread issues the 3xTF32 products
//   x_hi . [y_hi ; y_lo]  (N = 256)   and   x_lo . y_hi  (N = 128)
// per 8-wide K step into tensor memory. Eight warps read the accumulators back,
// form the cost, clamp it at 0 and write the skewed layout of the wavefront
// through a per-warp shared staging tile, so every global store is a 128-byte
// slot row.
//
// Precision: the dot carries ~2^-21 of sum_k |x_k y_k|, and the final fp32
// combination a few ulps of C; at D <= 64 that keeps the gradient of the
// unit-variance workloads far inside rel 1e-3 / abs 1e-5 (wider features use the
// exact difference-form kernel in dist.cu).
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace sdtw {

namespace {

using namespace tc;

constexpr int kTile = 128;                   // rows and columns per cost CTA
constexpr int kTcThreads = 256;              // 8 warps
constexpr uint32_t kBlockBytes = kTile * 128;  // one K-block of 128 rows (32 tf32 each)
constexpr int kStg = 63 * 32;                // per-warp skew staging (floats)

// grid (Lpad/32, P, 2): z = 0 writes the x image, z = 1 the y image. block 256.
// Rows past the sequence end are zero (image and norm). KB <= 2: every thread
// issues all of its loads (at most 8) before the first shared store.
__global__ void __launch_bounds__(256) simg_kernel(Problems pr, int N, int M, int D, int KB, float* __restrict__ ximg,
                                                   float* __restrict__ yimg, float* __restrict__ xnorm,
                                                   float* __restrict__ ynorm)
{
    extern __shared__ float t[];  // [32][D32 + 1]
    const bool isy = blockIdx.z == 1;
    const int p = blockIdx.y, r0 = blockIdx.x * 32;
    const int L = isy ? M : N;
    const int Lpad = (L + kTile - 1) / kTile * kTile;
    if (r0 >= Lpad) return;
    const float* src = isy ? pr.y(p) : pr.x(p);
    float* img = isy ? yimg : ximg;
    float* nrm = isy ? ynorm : xnorm;
    const int D32 = 32 * KB, ld = D32 + 1;
    const int n = 32 * D32 / 256;  // values per thread: 4 or 8
    float v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const int idx = threadIdx.x + 256 * u;
        const int r = idx / D32, k = idx - r * D32;
        v[u] = (u < n && r0 + r < L && k < D) ? src[(size_t)(r0 + r) * D + k] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const int idx = threadIdx.x + 256 * u;
        const int r = idx / D32, k = idx - r * D32;
        if (u < n) t[r * ld + k] = v[u];
    }
    __syncthreads();
    {
        // squared norm of row tid/8: eight threads take every eighth feature (exact
        // squares by fma, TwoSum partial sums), then pairwise TwoSum across the eight
        const int r = threadIdx.x >> 3, part = threadIdx.x & 7;
        float s = 0.f, c = 0.f;
        for (int k = part; k < D; k += 8) {
            const float x = t[r * ld + k];
            const float sq = x * x;
            float sn, err;
            two_sum(s, sq, sn, err);
            s = sn;
            c += err + fmaf(x, x, -sq);
        }
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
            const float so = __shfl_xor_sync(0xffffffffu, s, o), co = __shfl_xor_sync(0xffffffffu, c, o);
            float sn, err;
            two_sum(s, so, sn, err);
            s = sn;
            c += co + err;
        }
        if (part == 0) nrm[(size_t)p * Lpad + r0 + r] = s + c;
    }
    // a warp writes one 128-byte image row (32 features of one row) per pass
    for (int idx = threadIdx.x; idx < 32 * D32; idx += blockDim.x) {
        const int k = idx & 31, r = (idx >> 5) & 31, kb = idx >> 10;
        float h, l;
        split_tf32(t[r * ld + kb * 32 + k], h, l);
        const uint32_t o = (uint32_t)((((k >> 2) ^ (r & 7)) << 4) + (k & 3) * 4) / 4;
        img[simg_offset(p, KB, kb, 0, Lpad, r0 + r) + o] = h;
        img[simg_offset(p, KB, kb, 1, Lpad, r0 + r) + o] = l;
    }
}

// grid (ceil(M/128), ceil(N/128), P), block 256. One 128 x 128 cost tile.
template <int KB>
__global__ void __launch_bounds__(kTcThreads, 1)
    dist_tc_kernel(int N, int M, const float* __restrict__ ximg, const float* __restrict__ yimg,
                   const float* __restrict__ xnorm, const float* __restrict__ ynorm, float* __restrict__ Dsk,
                   int* status)
{
    extern __shared__ unsigned char smem_dyn[];
    __shared__ uint64_t s_load, s_mma;
    __shared__ uint32_t s_tmem;
    __shared__ float s_ny[kTile];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int p = blockIdx.z, r0 = blockIdx.y * kTile, c0 = blockIdx.x * kTile;
    const int Npad = (N + kTile - 1) / kTile * kTile, Mpad = (M + kTile - 1) / kTile * kTile;
    const int NB = (N + 31) / 32;

    // shared memory (1 KiB aligned): A_hi[KB], A_lo[KB], B[KB] = [y_hi ; y_lo], staging
    unsigned char* base = smem_dyn + ((1024u - (smem_u32(smem_dyn) & 1023u)) & 1023u);
    unsigned char* a_hi = base;
    unsigned char* a_lo = base + KB * kBlockBytes;
    unsigned char* bst = base + 2 * KB * kBlockBytes;
    float* stg = reinterpret_cast<float*>(bst + 2 * KB * kBlockBytes) + warp * kStg;

    if (tid == 0) {
        mbar_init(smem_u32(&s_load), 1);
        mbar_init(smem_u32(&s_mma), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) tmem_alloc(&s_tmem, 256);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = s_tmem;

    bool ok = true;
    if (tid == 0) {
        mbar_expect_tx(smem_u32(&s_load), 4u * KB * kBlockBytes);
        for (int kb = 0; kb < KB; ++kb) {
            bulk_g2s(smem_u32(a_hi + kb * kBlockBytes), ximg + simg_offset(p, KB, kb, 0, Npad, r0), kBlockBytes,
                     smem_u32(&s_load));
            bulk_g2s(smem_u32(a_lo + kb * kBlockBytes), ximg + simg_offset(p, KB, kb, 1, Npad, r0), kBlockBytes,
                     smem_u32(&s_load));
            bulk_g2s(smem_u32(bst + kb * 2 * kBlockBytes), yimg + simg_offset(p, KB, kb, 0, Mpad, c0), kBlockBytes,
                     smem_u32(&s_load));
            bulk_g2s(smem_u32(bst + kb * 2 * kBlockBytes + kBlockBytes), yimg + simg_offset(p, KB, kb, 1, Mpad, c0),
                     kBlockBytes, smem_u32(&s_load));
        }
    }
    if (tid < kTile) s_ny[tid] = ynorm[(size_t)p * Mpad + c0 + tid];
    if (tid == 0) {
        wait_ok(ok, smem_u32(&s_load), 0u, status);
        if (!ok) {
            // no copy may still be writing shared memory when the CTA exits
            bool drained = true;
            wait_ok(drained, smem_u32(&s_load), 0u, status);
        }
        fence_after_sync();
        const uint32_t id2 = idesc_tf32(kTile, 2 * kTile), id1 = idesc_tf32(kTile, kTile);
#pragma unroll
        for (int kb = 0; kb < KB; ++kb) {
            const uint32_t ah = smem_u32(a_hi + kb * kBlockBytes), al = smem_u32(a_lo + kb * kBlockBytes);
            const uint32_t bh = smem_u32(bst + kb * 2 * kBlockBytes);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                const uint32_t ko = ks * 32;  // 8 tf32 = 32 bytes along K
                mma_tf32(tmem, sdesc(ah + ko), sdesc(bh + ko), id2, (kb > 0 || ks > 0) ? 1u : 0u);
                mma_tf32(tmem, sdesc(al + ko), sdesc(bh + ko), id1, 1u);
            }
        }
        mma_commit(smem_u32(&s_mma));
    }
    __syncthreads();  // s_ny
    wait_ok(ok, smem_u32(&s_mma), 0u, status);
    fence_after_sync();

    // ---- epilogue: warp w reads rows 32(w mod 4) + lane (its TMEM lane quarter) and
    // columns [64 (w / 4), 64 (w / 4) + 64) in two chunks of 32
    const int q = warp & 3, half = warp >> 2;
    const int rb = (r0 >> 5) + q;
    const int row = r0 + 32 * q + lane;
    const float nx = xnorm[(size_t)p * Npad + row];
    const uint32_t trow = tmem + ((uint32_t)(32 * q) << 16);
    float* out = (rb < NB) ? Dsk + skew_index(N, M, p, rb, 0, lane) : nullptr;
    const bool skip = out == nullptr || !__all_sync(0xffffffffu, ok);  // warp-uniform
#pragma unroll 1
    for (int cc = 0; cc < 2; ++cc) {
        const int ch = 2 * half + cc;
        float a[32], b[32];
        tmem_ld32(trow + (uint32_t)(32 * ch), a);
        tmem_ld32(trow + (uint32_t)(kTile + 32 * ch), b);
        if (skip) continue;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const float c = fmaxf(nx + s_ny[32 * ch + j] - 2.f * (a[j] + b[j]), 0.f);
            stg[(j + lane) * 32 + lane] = c;
        }
        __syncwarp();
        // skewed slot c0 + 32 ch + t holds column (t - lane) of this chunk for this lane's row
        const int cb = c0 + 32 * ch;
        for (int t = 0; t < 63; ++t) {
            const int j = t - lane;
            if (j >= 0 && j < 32 && cb + j < M && row < N) out[(long long)(cb + t) * 32] = stg[t * 32 + lane];
        }
        __syncwarp();
    }

    fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        fence_after_sync();
        tmem_dealloc(tmem, 256);
    }
}

}  // namespace

size_t simg_bytes(int P, int L, int D)
{
    const int KB = (D + 31) / 32;
    const int Lpad = (L + kTile - 1) / kTile * kTile;
    return (size_t)P * KB * 2 * Lpad * 128;
}

size_t snorm_bytes(int P, int L)
{
    const int Lpad = (L + kTile - 1) / kTile * kTile;
    return (size_t)P * Lpad * sizeof(float);
}

cudaError_t launch_simg(const Problems& pr, int P, int N, int M, int D, float* ximg, float* yimg, float* xnorm,
                        float* ynorm, cudaStream_t st)
{
    const int KB = (D + 31) / 32;
    const int Lmax = ((N > M ? N : M) + kTile - 1) / kTile * kTile;
    const size_t smem = sizeof(float) * 32 * (32 * KB + 1);
    simg_kernel<<<dim3(Lmax / 32, P, 2), 256, smem, st>>>(pr, N, M, D, KB, ximg, yimg, xnorm, ynorm);
    return cudaGetLastError();
}

cudaError_t launch_dist_tc(int P, int N, int M, int D, const float* ximg, const float* yimg, const float* xnorm,
                           const float* ynorm, float* Dsk, int* status, cudaStream_t st)
{
    const int KB = (D + 31) / 32;
    if (KB < 1 || KB > 2) return cudaErrorInvalidValue;
    const size_t smem = 1024 + 4 * (size_t)KB * kBlockBytes + 8 * kStg * sizeof(float);
    dim3 grid((M + kTile - 1) / kTile, (N + kTile - 1) / kTile, P);
    auto go = [&](auto kern) -> cudaError_t {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        kern<<<grid, kTcThreads, smem, st>>>(N, M, ximg, yimg, xnorm, ynorm, Dsk, status);
        return cudaGetLastError();
    };
    return KB == 1 ? go(dist_tc_kernel<1>) : go(dist_tc_kernel<2>);
}

}  // namespace sdtw
