// egemm.cu -- input gradients as tensor-core contractions of the alignment matrix.
//
//   grad_x[i,:] = g * 2 * (sum_j E[i,j] x_i - sum_j E[i,j] y_j)    (rows:    E   . [Y | 1])
//   grad_y[j,:] = g * 2 * (sum_i E[i,j] y_j - sum_i E[i,j] x_i)    (columns: E^T . [X | 1])
//
// One CTA computes 128 output rows (tcgen05 M = 128) against all D+1 output
// columns (the extra column of ones yields the row or column sums of E in the
// same MMA). The reduction runs over the other sequence in K-tiles of 32. Each
// A-tile's skewed rows of E arrive by bulk copy (cp.async.bulk) and the CTA's
// threads un-skew them, split each value into tf32 hi + lo parts (round to
// nearest) and store both in the 128-byte-swizzled K-major layout. The B tiles
// ([Y | 1] or [X | 1]) are the same for every CTA of a problem, so a small
// kernel writes them once, already split and swizzled, and each CTA fetches a
// K-tile's B image with one bulk copy. One thread issues the 3xTF32 products
// hi*hi + lo*hi + hi*lo with tcgen05.mma (fp32 accumulation in tensor memory),
// committed to an mbarrier. Two smem stages let the copies and un-skew of tile
// k+1 overlap the MMAs of tile k. The epilogue reads the accumulators back with
// tcgen05.ld.
//
// Precision: each split product carries ~2^-21 relative error, so E . y keeps
// ~1e-6 relative accuracy; the gradient is a difference of two such sums that
// can cancel by ~100x, which leaves it well inside rel 1e-3.
#include "common.cuh"
#include "kernels.h"

namespace sdtw {

namespace {

constexpr int kBM = 128;       // output rows per CTA (MMA M)
constexpr int kBK = 32;        // reduction elements per K-tile (128 bytes of fp32 per smem row)
constexpr int kThreads = 256;  // 8 warps; warps w and w+4 share TMEM lane quarter w

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Byte offset of element (r, k) in a K-major tile of 32 fp32 per row, 128-byte
// swizzle: 16-byte chunk index XOR (row mod 8) inside each 8-row, 1 KiB atom.
__device__ __forceinline__ uint32_t sw128(int r, int k) {
    return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((((k >> 2) ^ r) & 7) << 4) + (k & 3) * 4);
}

// fp32 -> tf32 hi (round to nearest) and the tf32-rounded remainder.
__device__ __forceinline__ void split_tf32(float v, float& hi, float& lo) {
    hi = __uint_as_float((__float_as_uint(v) + 0x1000u) & 0xFFFFE000u);
    const float r = v - hi;
    lo = __uint_as_float((__float_as_uint(r) + 0x1000u) & 0xFFFFE000u);
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups 1 KiB apart.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)1 << 16;              // leading byte offset (unused with swizzled K-major)
    d |= (uint64_t)(1024 >> 4) << 32;    // stride byte offset: next 8-row group
    d |= (uint64_t)1 << 46;              // descriptor version
    d |= (uint64_t)2 << 61;              // 128-byte swizzle
    return d;
}

// Instruction descriptor: D fp32, A and B tf32, both K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void mbar_init(uint32_t bar, int count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.b32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the given phase parity of an mbarrier (all threads).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int* status) {
    if (mbar_test(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_test(bar, parity)) {
        if (global_ns() - t0 > 2000000000ull) {
            atomicOr(status, kStatusTimeout);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int q = 0; q < 16; ++q) v[q] = __uint_as_float(r[q]);
}

// Stores the split value into the hi and lo tiles of a stage.
__device__ __forceinline__ void put(unsigned char* hi_tile, unsigned char* lo_tile, int r, int k, float v) {
    float h, l;
    split_tf32(v, h, l);
    const uint32_t o = sw128(r, k);
    *reinterpret_cast<float*>(hi_tile + o) = h;
    *reinterpret_cast<float*>(lo_tile + o) = l;
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// One TMA bulk copy global -> shared (16-byte aligned addresses, size multiple of 16).
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// Skewed rows of E that one K-tile needs, per row block.
//   rows (grad_x): for each of the 4 row blocks, slots t in [k0, k0+63)   -> 64 rows copied
//   cols (grad_y): one row block k0/32, slots t in [m0, m0+159)           -> 160 rows copied
template <bool COLS>
struct Raw {
    static constexpr int kRows = COLS ? 160 : 4 * 64;
    static constexpr uint32_t kBytes = kRows * 128;
};

// Issue the bulk copies of K-tile kt's skewed rows of E into raw buffer rawA
// (completion on `bar`). Called by one thread.
template <bool COLS>
__device__ __forceinline__ void issue_a(const float* Ekp, int N, int M, int T, int m0, int kt, unsigned char* rawA,
                                        uint32_t bar)
{
    const int k0 = kt * kBK;
    const int NB = (N + 31) / 32;
    uint32_t bytes = 0;
    if (!COLS) {
        for (int b = 0; b < 4; ++b) {
            if ((m0 >> 5) + b >= NB) break;
            bytes += min(64, T - k0) * 128;
        }
    } else {
        bytes = (uint32_t)min(160, T - m0) * 128;
    }
    mbar_expect_tx(bar, bytes);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (!COLS) {
        for (int b = 0; b < 4; ++b) {
            const int rb = (m0 >> 5) + b;
            if (rb >= NB) break;
            const int rows = min(64, T - k0);
            bulk_g2s(smem_u32(rawA + b * 64 * 128), Ekp + ((size_t)rb * T + k0) * 32, rows * 128, bar);
        }
    } else {
        const int rb = k0 >> 5;
        const int rows = min(160, T - m0);
        bulk_g2s(smem_u32(rawA), Ekp + ((size_t)rb * T + m0) * 32, rows * 128, bar);
    }
}

// B operand image of K-tile kt: hi then lo tiles (n_total rows x 128 B each),
// already split and swizzled; one bulk copy into the tile stage.
__device__ __forceinline__ void issue_b(const float* img, int n_total, int kt, unsigned char* B_hi, uint32_t bar)
{
    const uint32_t bytes = 2u * (uint32_t)n_total * 128u;
    mbar_expect_tx(bar, bytes);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    bulk_g2s(smem_u32(B_hi), img + (size_t)kt * (bytes / 4), bytes, bar);
}

// COLS = false: grad_x rows (A = E rows i, K = j, B = [Y | 1]).
// COLS = true : grad_y rows (A = E columns j, K = i, B = [X | 1]).
// bimg: per problem, per K-tile, the pre-split B image (bimg_kernel).
template <bool COLS>
__global__ void __launch_bounds__(kThreads, 1)
    egemm_kernel(const GradParams g, const float* __restrict__ bimg, int n_total, int tstages, int* status)
{
    extern __shared__ unsigned char smem_dyn[];
    __shared__ uint64_t s_mma[2];   // MMA completion per tile stage
    __shared__ uint64_t s_raw[2];   // A bulk copies per raw buffer
    __shared__ uint64_t s_bim[2];   // B image copies per tile stage
    __shared__ uint32_t s_tmem;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, half = warp >> 2;
    const int p = blockIdx.y;
    const int m0 = blockIdx.x * kBM;
    const int N = g.N, M = g.M, D = g.D, T = skew_T(M);
    const int rows = COLS ? M : N;     // output rows
    const int kdim = COLS ? N : M;     // reduction length
    const int NB = (N + 31) / 32;
    const int nK = (kdim + kBK - 1) / kBK;
    const float* Ekp = g.E + skew_index(N, M, p, 0, 0, 0);
    const float* xb = g.pr.x(p);
    const float* yb = g.pr.y(p);
    const float* bimg_p = bimg + (size_t)p * nK * 2 * n_total * 32;

    // Shared memory (1 KiB aligned): tile stages [A hi | A lo | B hi | B lo], then 2 raw A buffers.
    const uint32_t a_bytes = kBM * 128, b_bytes = (uint32_t)n_total * 128;
    const uint32_t stage_bytes = 2 * a_bytes + 2 * b_bytes;
    const uint32_t rawA_bytes = Raw<COLS>::kBytes;
    unsigned char* base = smem_dyn + ((1024u - (smem_u32(smem_dyn) & 1023u)) & 1023u);
    unsigned char* raw0 = base + tstages * stage_bytes;
    auto stage = [&](int st) { return base + st * stage_bytes; };
    auto rawA = [&](int r) { return raw0 + r * rawA_bytes; };

    if (tid == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&s_mma[b]), 1);
            mbar_init(smem_u32(&s_raw[b]), 1);
            mbar_init(smem_u32(&s_bim[b]), 1);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    int ncols = 32;
    while (ncols < n_total) ncols <<= 1;
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                     "r"(ncols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = s_tmem;

    uint32_t mma_ph[2] = {0u, 0u}, raw_ph[2] = {0u, 0u}, bim_ph[2] = {0u, 0u};
    bool ok = true;
    if (tid == 0) {
        issue_a<COLS>(Ekp, N, M, T, m0, 0, rawA(0), smem_u32(&s_raw[0]));
        issue_b(bimg_p, n_total, 0, stage(0) + 2 * a_bytes, smem_u32(&s_bim[0]));
    }
    for (int kt = 0; kt < nK; ++kt) {
        const int r = kt & 1;
        const int s = (tstages == 2) ? (kt & 1) : 0;
        // A raw rows and the B image of tile kt have landed
        ok = mbar_wait(smem_u32(&s_raw[r]), raw_ph[r], status) && ok;
        raw_ph[r] ^= 1u;
        ok = mbar_wait(smem_u32(&s_bim[s]), bim_ph[s], status) && ok;
        bim_ph[s] ^= 1u;
        __syncthreads();
        // prefetch the A rows of tile kt+1 into the other raw buffer (last read before the
        // barrier that ended iteration kt-1)
        if (tid == 0 && kt + 1 < nK) issue_a<COLS>(Ekp, N, M, T, m0, kt + 1, rawA(r ^ 1), smem_u32(&s_raw[r ^ 1]));
        unsigned char* A_hi = stage(s);
        unsigned char* A_lo = A_hi + a_bytes;
        const int k0 = kt * kBK;
        const float* ra = reinterpret_cast<const float*>(rawA(r));

        // ---- A tile: un-skew and split (zero outside the matrix)
        if (!COLS) {
            // warps w, w+4: row block m0/32 + (w mod 4), columns split in halves; lane = row
            const int rb = (m0 >> 5) + quarter;
            const int i = m0 + 32 * quarter + lane;
            const float* rw = ra + quarter * 64 * 32;
#pragma unroll 8
            for (int cc = 0; cc < kBK / 2; ++cc) {
                const int c = half * (kBK / 2) + cc;
                const int j = k0 + c;
                const float v = (rb < NB && i < N && j < M) ? rw[(c + lane) * 32 + lane] : 0.f;
                put(A_hi, A_lo, 32 * quarter + lane, c, v);
            }
        } else {
            // raw row tt holds slot m0 + tt of block k0/32; lane = K index i - k0; output row r = tt - lane
            const int i = k0 + lane;
#pragma unroll 4
            for (int rr = warp; rr < kBM; rr += 8) {
                const int j = m0 + rr;
                const float v = (i < N && j < M) ? ra[(rr + lane) * 32 + lane] : 0.f;
                put(A_hi, A_lo, rr, lane, v);
            }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();

        if (tid == 0) {
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const uint32_t ah = smem_u32(A_hi), al = smem_u32(A_lo);
            const uint32_t bh = smem_u32(A_hi + 2 * a_bytes), bl = bh + b_bytes;
            for (int n0 = 0; n0 < n_total; n0 += 256) {
                const int nn = min(256, n_total - n0);
                const uint32_t id = idesc_tf32(kBM, nn);
                const uint32_t d = tmem + (uint32_t)n0;
                const uint32_t boff = (uint32_t)n0 * 128;
#pragma unroll
                for (int ks = 0; ks < kBK / 8; ++ks) {
                    const uint32_t ko = ks * 32;  // 8 tf32 = 32 bytes along K
                    const uint32_t first = (kt > 0 || ks > 0) ? 1u : 0u;
                    mma_tf32(d, sdesc(ah + ko), sdesc(bh + boff + ko), id, first);
                    mma_tf32(d, sdesc(al + ko), sdesc(bh + boff + ko), id, 1u);
                    mma_tf32(d, sdesc(ah + ko), sdesc(bl + boff + ko), id, 1u);
                }
            }
            mma_commit(smem_u32(&s_mma[s]));
            // the B image of tile kt+1 goes to the stage it will use, once the MMAs that
            // last read that stage (tile kt-1 with two stages, tile kt with one) are done;
            // this wait also orders the next A writes into that stage after those MMAs
            if (kt + 1 < nK) {
                const int sn = (tstages == 2) ? (s ^ 1) : 0;
                if (tstages == 1 || kt >= 1) {
                    ok = mbar_wait(smem_u32(&s_mma[sn]), mma_ph[sn], status) && ok;
                    mma_ph[sn] ^= 1u;
                }
                issue_b(bimg_p, n_total, kt + 1, stage(sn) + 2 * a_bytes, smem_u32(&s_bim[sn]));
            }
        }
    }
    // Every thread waits for the last commit; it covers every MMA issued before it.
    {
        const int s = (tstages == 2) ? ((nK - 1) & 1) : 0;
        const int commits = (tstages == 2) ? ((nK - 1 - s) / 2 + 1) : nK;  // commits on stage s
        ok = mbar_wait(smem_u32(&s_mma[s]), (uint32_t)((commits - 1) & 1), status) && ok;
    }
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");

    // ---- epilogue: warp w (and w+4) hold output rows m0 + 32(w mod 4) + lane in TMEM lane quarter w mod 4;
    // warps 0-3 write columns [0, Dh), warps 4-7 columns [Dh, D)
    const int row = m0 + 32 * quarter + lane;
    const uint32_t trow = tmem + ((uint32_t)(32 * quarter) << 16);
    float sums[16];
    tmem_ld16(trow + (uint32_t)(D & ~15), sums);
    float sum = 0.f;
#pragma unroll
    for (int q = 0; q < 16; ++q) sum = (q == (D & 15)) ? sums[q] : sum;
    const float w = g.coef * 2.f * (g.grad_loss ? g.grad_loss[p % g.wmod] : 1.f);
    const float* own = (COLS ? yb : xb) + (size_t)row * D;
    float* out = g.out + (long long)(p % g.omod) * g.out_stride + (size_t)row * D;
    const int nchunks = (D + 15) / 16;
    const int cbeg = half ? (nchunks + 1) / 2 : 0, cend = half ? nchunks : (nchunks + 1) / 2;
    for (int ch = cbeg; ch < cend; ++ch) {
        const int c0 = ch * 16;
        float acc[16];
        tmem_ld16(trow + (uint32_t)c0, acc);
        if (ok && row < rows) {
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                const int n = c0 + q;
                if (n < D) {
                    const float val = w * (sum * own[n] - acc[q]);
                    out[n] = g.accumulate ? out[n] + val : val;
                }
            }
        }
    }

    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(ncols) : "memory");
    }
}

// Pre-split B operand images: for problem p and K-tile kt, rows n < D hold
// coordinate n of the other sequence's rows kt*32 .. kt*32+31, row D holds ones;
// written as the hi then lo tf32 tiles in the swizzled smem layout. A 32x32
// shared tile turns the row-major reads and the K-major writes into full lines.
// grid (nK, P), block 256.
__global__ void __launch_bounds__(256) bimg_kernel(const GradParams g, bool cols, int n_total, float* __restrict__ img)
{
    __shared__ float t[32][33];
    const int kt = blockIdx.x, p = blockIdx.y;
    const int D = g.D;
    const int kdim = cols ? g.N : g.M;
    const int nK = (kdim + kBK - 1) / kBK;
    const float* vb = cols ? g.pr.x(p) : g.pr.y(p);
    unsigned char* hi = reinterpret_cast<unsigned char*>(img + ((size_t)p * nK + kt) * 2 * n_total * 32);
    unsigned char* lo = hi + (size_t)n_total * 128;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    for (int n0 = 0; n0 < n_total; n0 += 32) {
        for (int k = ty; k < 32; k += 8) {
            const int kk = kt * kBK + k, n = n0 + tx;
            float v = 0.f;
            if (kk < kdim) v = (n < D) ? vb[(size_t)kk * D + n] : (n == D ? 1.f : 0.f);
            t[k][tx] = v;
        }
        __syncthreads();
        for (int nn = ty; nn < 32; nn += 8) {
            const int n = n0 + nn;
            if (n < n_total) put(hi, lo, n, tx, t[tx][nn]);
        }
        __syncthreads();
    }
}

}  // namespace

// Shared-memory plan: tile stages (hi/lo of A and B) and two raw A buffers;
// two tile stages when they fit in 220 KiB.
static void egemm_plan(int D, bool cols, int* tstages, size_t* bytes)
{
    const int n_total = ((D + 1 + 15) / 16) * 16;
    const size_t stage = 2 * (size_t)kBM * 128 + 2 * (size_t)n_total * 128;
    const size_t raw = 2 * (size_t)(cols ? Raw<true>::kBytes : Raw<false>::kBytes);
    const int t = (1024 + 2 * stage + raw <= 220 * 1024) ? 2 : 1;
    *tstages = t;
    *bytes = 1024 + t * stage + raw;
}

size_t egemm_smem_bytes(int D)
{
    int t;
    size_t a, b;
    egemm_plan(D, false, &t, &a);
    egemm_plan(D, true, &t, &b);
    return a > b ? a : b;
}

size_t egemm_bimg_bytes(int P, int N, int M, int D)
{
    const int n_total = ((D + 1 + 15) / 16) * 16;
    const int nK = ((N > M ? N : M) + kBK - 1) / kBK;
    return (size_t)P * nK * 2 * n_total * 128;
}

cudaError_t launch_grad_tc(const GradParams& g, bool cols, float* bimg, int* status, cudaStream_t st)
{
    const int n_total = ((g.D + 1 + 15) / 16) * 16;
    const int kdim = cols ? g.N : g.M;
    const int nK = (kdim + kBK - 1) / kBK;
    bimg_kernel<<<dim3(nK, g.P), 256, 0, st>>>(g, cols, n_total, bimg);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    int tstages;
    size_t smem;
    egemm_plan(g.D, cols, &tstages, &smem);
    const int rows = cols ? g.M : g.N;
    dim3 grid((rows + kBM - 1) / kBM, g.P);
    if (cols) {
        e = cudaFuncSetAttribute(egemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        egemm_kernel<true><<<grid, kThreads, smem, st>>>(g, bimg, n_total, tstages, status);
    } else {
        e = cudaFuncSetAttribute(egemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        egemm_kernel<false><<<grid, kThreads, smem, st>>>(g, bimg, n_total, tstages, status);
    }
    return cudaGetLastError();
}

}  // namespace sdtw
