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
// written once as an operand image (simg_kernel): every value split exactly into
// three bf16 parts v = v0 + v1 + v2 (8 significant bits each), stored in the
// 128-byte-swizzled K-major layout that tcgen05.mma reads, in K-blocks of 64
// features, together with the squared norm of the row (compensated fp32: exact
// squares, TwoSum partial sums, rounded once). The dot is the sum of all nine
// part products, each exact in fp32,
//   x0 . [y0 ; y1 ; y2]  +  x1 . [y0 ; y1 ; y2]  +  x2 . [y0 ; y1 ; y2],
// three bf16 MMAs per 16-wide K step with the y parts stacked along N, all
// accumulating in fp32 in tensor memory; the three column groups are summed in
// the epilogue, so the dot carries only the fp32 accumulation.
//
// A cost CTA (dist_tc_kernel) owns 128 x rows and walks the y columns in tiles
// of 64; one thread issues the copies and MMAs into one of two tensor-memory
// slots while eight warps drain the other: they read the accumulators back, form
// the cost, clamp it at 0 and write the skewed layout of the wavefront through a
// per-warp shared staging tile, so every global store is a 128-byte slot row.
// The x rows (one K-block: D <= 64) stay in shared memory. Wider features take the
// exact difference-form kernel of dist.cu: beyond one K-block the fp32
// accumulation of the dot in tensor memory adds errors of a few ulps of the cost,
// which the fp32 DP state's gradients do not absorb at the tolerance.
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace sdtw {

namespace {

using namespace tc;

constexpr int kTile = 128;                     // x rows per cost CTA (the MMA height)
constexpr int kColTile = 64;                   // y columns per cost tile
constexpr int kTcWarps = 8;                    // epilogue warps; warp 8 copies and issues the MMAs
constexpr int kTcThreads = (kTcWarps + 1) * 32;
constexpr uint32_t kPartBytes = kTile * 128;   // one bf16 part of one K-block of 128 x rows
constexpr uint32_t kABytes = 3 * kPartBytes;   // the three parts of one K-block of x rows
constexpr uint32_t kYPart = kColTile * 128;    // one part of one K-block of 64 y rows
constexpr uint32_t kBBytes = 3 * kYPart;       // [y0 ; y1 ; y2] of one K-block of a y tile
constexpr int kSlotCols = 3 * kColTile;        // tensor-memory columns of one tile: three part groups
constexpr int kStg = 63 * 32;                  // per-warp skew staging (floats)

// grid (Lpad/32, P, 2): z = 0 writes the x image, z = 1 the y image. block 256.
// Rows past the sequence end are zero (image and norm). Each thread loads its
// values in batches of 8, all issued before their shared stores.
// Eight CTAs of 256 threads per SM (32 registers a thread): a batch's images are one wave.
__global__ void __launch_bounds__(256, 8) simg_kernel(Problems pr, int N, int M, int D, int KB,
                                                   unsigned char* __restrict__ ximg, unsigned char* __restrict__ yimg,
                                                   float* __restrict__ xnorm, float* __restrict__ ynorm)
{
    extern __shared__ float t[];  // [32][D64 + 1]
    const bool isy = blockIdx.z == 1;
    const int p = blockIdx.y, r0 = blockIdx.x * 32;
    const int L = isy ? M : N;
    const int Lpad = simg_pad(L);
    if (r0 >= Lpad) return;
    const float* src = isy ? pr.y(p) : pr.x(p);
    unsigned char* img = isy ? yimg : ximg;
    float* nrm = isy ? ynorm : xnorm;
    const int D64 = kTcKFeat * KB, ld = D64 + 1;
    const int n = 32 * D64 / 256;  // values per thread: 8 per K-block
    for (int u0 = 0; u0 < n; u0 += 8) {
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int idx = threadIdx.x + 256 * (u0 + u);
            const int r = idx / D64, k = idx - r * D64;
            v[u] = (r0 + r < L && k < D) ? src[(size_t)(r0 + r) * D + k] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int idx = threadIdx.x + 256 * (u0 + u);
            const int r = idx / D64, k = idx - r * D64;
            t[r * ld + k] = v[u];
        }
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
    // one 16-byte chunk (8 features) of all three parts per thread and pass: eight
    // threads write one 128-byte image row per part (its chunks permuted by the
    // swizzle), a warp four rows
    const size_t part_bytes = (size_t)Lpad * 128;   // between the parts of a K-block
    for (int idx = threadIdx.x; idx < 32 * D64 / 8; idx += blockDim.x) {
        const int c8 = idx & 7, r = (idx >> 3) & 31, kb = idx >> 8;
        const float* src8 = t + r * ld + kb * kTcKFeat + 8 * c8;
        uint16_t h0[8], h1[8], h2[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) split_bf16x3(src8[q], h0[q], h1[q], h2[q]);
        uint4 w0, w1, w2;
        w0.x = h0[0] | ((uint32_t)h0[1] << 16); w0.y = h0[2] | ((uint32_t)h0[3] << 16);
        w0.z = h0[4] | ((uint32_t)h0[5] << 16); w0.w = h0[6] | ((uint32_t)h0[7] << 16);
        w1.x = h1[0] | ((uint32_t)h1[1] << 16); w1.y = h1[2] | ((uint32_t)h1[3] << 16);
        w1.z = h1[4] | ((uint32_t)h1[5] << 16); w1.w = h1[6] | ((uint32_t)h1[7] << 16);
        w2.x = h2[0] | ((uint32_t)h2[1] << 16); w2.y = h2[2] | ((uint32_t)h2[3] << 16);
        w2.z = h2[4] | ((uint32_t)h2[5] << 16); w2.w = h2[6] | ((uint32_t)h2[7] << 16);
        unsigned char* row = img + simg_offset(p, KB, kb, 0, Lpad, r0 + r) + 16 * (c8 ^ (r & 7));
        *reinterpret_cast<uint4*>(row) = w0;
        *reinterpret_cast<uint4*>(row + part_bytes) = w1;
        *reinterpret_cast<uint4*>(row + 2 * part_bytes) = w2;
    }
}

// Epilogue warps 0-7 of the cost kernels: warp w reads TMEM lane quarter w mod 4
// (rows r0 + 32(w mod 4) + lane) and the 32-column half w / 4 of each 64-column
// tile from its three part groups, releases the slot, forms C = |x|^2 + |y|^2 -
// 2 x.y clamped at 0 and writes the skewed layout through a per-warp staging tile
// (128-byte rows).
__device__ __forceinline__ void cost_epilogue(int N, int M, int p, int r0, int nC, uint32_t tmem,
                                              uint64_t* s_tfull, uint64_t* s_tfree, const float* __restrict__ xnorm,
                                              const float* __restrict__ ynorm, float* __restrict__ Dsk, float* stg,
                                              bool& ok, int* status)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Npad = simg_pad(N), Mpad = simg_pad(M);
    const int NB = (N + 31) / 32;
    const int q = warp & 3, half = warp >> 2;
    const int rb = (r0 >> 5) + q;
    const int row = r0 + 32 * q + lane;
    const float nx = xnorm[(size_t)p * Npad + row];
    const uint32_t trow = tmem + ((uint32_t)(32 * q) << 16);
    float* out = (rb < NB) ? Dsk + skew_index(N, M, p, rb, 0, lane) : nullptr;
    for (int c = 0; c < nC; ++c) {
        const int t = c & 1;
        wait_ok(ok, smem_u32(&s_tfull[t]), (uint32_t)((c >> 1) & 1), status);
        if (!__all_sync(0xffffffffu, ok)) break;
        fence_after_sync();
        float a[32], b[32], e[32];
        const uint32_t col = trow + (uint32_t)(t * kSlotCols + 32 * half);
        tmem_ld32(col, a);
        tmem_ld32(col + kColTile, b);
        tmem_ld32(col + 2 * kColTile, e);
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&s_tfree[t]));
        const int cb = c * kColTile + 32 * half;  // first column of this warp's chunk
        if (out == nullptr || cb >= M) continue;  // warp-uniform
        const float nyv = ynorm[(size_t)p * Mpad + cb + lane];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const float ny = __shfl_sync(0xffffffffu, nyv, j);
            stg[(j + lane) * 32 + lane] = fmaxf(nx + ny - 2.f * (a[j] + (b[j] + e[j])), 0.f);
        }
        __syncwarp();
        // skewed slot cb + tt holds column (tt - lane) of this chunk for this lane's row
        for (int tt = 0; tt < 63; ++tt) {
            const int j = tt - lane;
            if (j >= 0 && j < 32 && cb + j < M && row < N) out[(long long)(cb + tt) * 32] = stg[tt * 32 + lane];
        }
        __syncwarp();
    }
}

// grid (ceil(N/128), P), block 288: one CTA per 128-row block of x and problem,
// walking the y columns in tiles of 64. Warp 8 (lane 0) copies the x rows once
// (one K-block: D <= 64) and each y tile into a two-entry ring, and issues every
// tile's MMAs into one of two tensor-memory slots; warps 0-7 drain a slot
// (epilogue) while the next tile's MMAs run. Hand-offs (all bounded mbarrier
// waits):
//   s_bfull[e]  y tile in entry e      s_bempty[e] its MMAs are done
//   s_tfull[t]  costs in TMEM slot t   s_tfree[t]  the 8 epilogue warps read slot t
__global__ void __launch_bounds__(kTcThreads, 1)
    dist_tc_kernel(int N, int M, const unsigned char* __restrict__ ximg, const unsigned char* __restrict__ yimg,
                   const float* __restrict__ xnorm, const float* __restrict__ ynorm, float* __restrict__ Dsk,
                   int* status)
{
    extern __shared__ unsigned char smem_dyn[];
    __shared__ uint64_t s_a, s_done, s_bfull[2], s_bempty[2], s_tfull[2], s_tfree[2];
    __shared__ uint32_t s_tmem;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int p = blockIdx.y, r0 = blockIdx.x * kTile;
    const int Npad = simg_pad(N), Mpad = simg_pad(M);
    const int nC = (M + kColTile - 1) / kColTile;

    // shared memory (1 KiB aligned): A [x0 | x1 | x2], 2 y entries [y0 ; y1 ; y2], staging
    unsigned char* base = smem_dyn + ((1024u - (smem_u32(smem_dyn) & 1023u)) & 1023u);
    unsigned char* a_img = base;
    unsigned char* yring = base + kABytes;
    float* stg = reinterpret_cast<float*>(yring + 2 * kBBytes) + warp * kStg;

    if (tid == 0) {
        mbar_init(smem_u32(&s_a), 1);
        mbar_init(smem_u32(&s_done), 1);
        for (int e = 0; e < 2; ++e) {
            mbar_init(smem_u32(&s_bfull[e]), 1);
            mbar_init(smem_u32(&s_bempty[e]), 1);
            mbar_init(smem_u32(&s_tfull[e]), 1);
            mbar_init(smem_u32(&s_tfree[e]), kTcWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) tmem_alloc(&s_tmem, 512);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = s_tmem;
    bool ok = true;

    if (warp == kTcWarps) {
        if (lane == 0) {
            mbar_expect_tx(smem_u32(&s_a), kABytes);
            for (int part = 0; part < 3; ++part)
                bulk_g2s(smem_u32(a_img + part * kPartBytes), ximg + simg_offset(p, 1, 0, part, Npad, r0), kPartBytes,
                         smem_u32(&s_a));
            int y_last[2] = {-1, -1};
            auto issue_y = [&](int c) {
                const int e = c & 1;
                unsigned char* dst = yring + e * kBBytes;
                mbar_expect_tx(smem_u32(&s_bfull[e]), kBBytes);
                for (int part = 0; part < 3; ++part)
                    bulk_g2s(smem_u32(dst + part * kYPart), yimg + simg_offset(p, 1, 0, part, Mpad, c * kColTile),
                             kYPart, smem_u32(&s_bfull[e]));
                y_last[e] = c;
            };
            for (int c = 0; c < 2 && c < nC; ++c) issue_y(c);
            wait_ok(ok, smem_u32(&s_a), 0u, status);
            for (int c = 0; c < nC && ok; ++c) {
                const int e = c & 1, t = c & 1;
                wait_ok(ok, smem_u32(&s_bfull[e]), (uint32_t)((c >> 1) & 1), status);
                if (c >= 2) wait_ok(ok, smem_u32(&s_tfree[t]), (uint32_t)(((c - 2) >> 1) & 1), status);
                if (!ok) break;
                fence_after_sync();
                const uint32_t d = tmem + (uint32_t)(t * kSlotCols);
                const uint32_t a = smem_u32(a_img), b = smem_u32(yring + e * kBBytes);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)  // 16 bf16 = 32 bytes along K per step
                    mma_bf16x3(d, a, b, kTile, kColTile, kPartBytes, ks * 32, ks > 0 ? 1u : 0u);
                mma_commit(smem_u32(&s_tfull[t]));
                mma_commit(smem_u32(&s_bempty[e]));
                if (c + 2 < nC) {  // entry e takes tile c + 2 once MMA(c) has read it
                    wait_ok(ok, smem_u32(&s_bempty[e]), (uint32_t)((c >> 1) & 1), status);
                    if (!ok) break;
                    issue_y(c + 2);
                }
            }
            // no MMA may still be running, and no copy still writing shared memory, at exit
            mma_commit(smem_u32(&s_done));
            bool fin = true;
            wait_ok(fin, smem_u32(&s_done), 0u, status);
            for (int e = 0; e < 2; ++e)
                if (y_last[e] >= 0) wait_ok(fin, smem_u32(&s_bfull[e]), (uint32_t)((y_last[e] >> 1) & 1), status);
        }
        __syncwarp();
    } else {
        cost_epilogue(N, M, p, r0, nC, tmem, s_tfull, s_tfree, xnorm, ynorm, Dsk, stg, ok, status);
    }

    fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        fence_after_sync();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

size_t simg_bytes(int P, int L, int D)
{
    const int KB = (D + kTcKFeat - 1) / kTcKFeat;
    return (size_t)P * KB * 3 * simg_pad(L) * 128;
}

size_t snorm_bytes(int P, int L) { return (size_t)P * simg_pad(L) * sizeof(float); }

cudaError_t launch_simg(const Problems& pr, int P, int N, int M, int D, void* ximg, void* yimg, float* xnorm,
                        float* ynorm, cudaStream_t st)
{
    const int KB = (D + kTcKFeat - 1) / kTcKFeat;
    const int Lmax = simg_pad(N > M ? N : M);
    const size_t smem = sizeof(float) * 32 * (kTcKFeat * KB + 1);
    cudaError_t e = cudaFuncSetAttribute(simg_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    simg_kernel<<<dim3(Lmax / 32, P, 2), 256, smem, st>>>(pr, N, M, D, KB, static_cast<unsigned char*>(ximg),
                                                          static_cast<unsigned char*>(yimg), xnorm, ynorm);
    return cudaGetLastError();
}

cudaError_t launch_dist_tc(int P, int N, int M, int D, const void* ximg, const void* yimg, const float* xnorm,
                           const float* ynorm, float* Dsk, int* status, cudaStream_t st)
{
    const int KB = (D + kTcKFeat - 1) / kTcKFeat;
    if (KB < 1 || KB > kMaxTcKBlocks) return cudaErrorInvalidValue;
    dim3 grid((N + kTile - 1) / kTile, P);
    const size_t stg = (size_t)kTcWarps * kStg * sizeof(float);
    const auto* xi = static_cast<const unsigned char*>(ximg);
    const auto* yi = static_cast<const unsigned char*>(yimg);
    const size_t smem = 1024 + kABytes + 2 * (size_t)kBBytes + stg;
    cudaError_t e = cudaFuncSetAttribute(dist_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dist_tc_kernel<<<grid, kTcThreads, smem, st>>>(N, M, xi, yi, xnorm, ynorm, Dsk, status);
    return cudaGetLastError();
}

}  // namespace sdtw
