// egemm.cu -- input gradients as tensor-core contractions of the alignment matrix.
//
//   grad_x[i,:] = g * 2 * (sum_j E[i,j] x_i - sum_j E[i,j] y_j)    (rows:    E   . [Y | 1])
//   grad_y[j,:] = g * 2 * (sum_i E[i,j] y_j - sum_i E[i,j] x_i)    (columns: E^T . [X | 1])
//
// One CTA computes 128 output rows (tcgen05 M = 128) against all D+1 output
// columns (the extra column of ones yields the row or column sums of E in the
// same MMA). The reduction runs over the other sequence in K-tiles of 32. Each
// A-tile's skewed rows of E arrive by bulk copy (cp.async.bulk); eight worker
// warps un-skew them, split each value into tf32 hi + lo parts (round to
// nearest) and store both in the 128-byte-swizzled K-major layout. The B tiles
// ([Y | 1] or [X | 1]) are the same for every CTA of a problem, so a small
// kernel writes them once, already split and swizzled, and each CTA fetches a
// K-tile's B image with one bulk copy. One warp issues the 3xTF32 products
// hi*hi + lo*hi + hi*lo with tcgen05.mma (fp32 accumulation in tensor memory)
// and two more issue the bulk copies; all hand buffers over through mbarriers, so
// the un-skew of tile k+1 overlaps the MMAs of tile k and the copies run two to
// four K-tiles ahead. The epilogue reads the accumulators back with tcgen05.ld
// and writes the gradient rows through a shared-memory tile.
//
// Precision: each split product carries ~2^-21 relative error, so E . y keeps
// ~1e-6 relative accuracy; the gradient is a difference of two such sums that
// can cancel by ~100x, which leaves it well inside rel 1e-3.
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace sdtw {

namespace {

using namespace tc;

constexpr int kBM = 128;       // output rows per CTA (MMA M)
constexpr int kBK = 32;        // reduction elements per K-tile (128 bytes of fp32 per smem row)
constexpr size_t kSmemLimit = 227 * 1024 - 256;  // opt-in dynamic shared memory, minus static

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
// already split and swizzled; one bulk copy. Called by one thread.
__device__ __forceinline__ void issue_b(const float* img, int n_total, int kt, unsigned char* B_hi, uint32_t bar)
{
    const uint32_t bytes = 2u * (uint32_t)n_total * 128u;
    mbar_expect_tx(bar, bytes);
    bulk_g2s(smem_u32(B_hi), img + (size_t)kt * (bytes / 4), bytes, bar);
}

// Pipeline depths (egemm_plan): ts A-tile stages, pb B-image buffers, pa raw-A buffers.
struct Pipe {
    int ts, pb, pa;
};

constexpr int kMaxRing = 4;
constexpr int kWorkers = 256;            // warps 0-7: un-skew and epilogue
constexpr int kMmaWarp = 8;              // warp 8: tcgen05.mma issue (lane 0)
constexpr int kCopyAWarp = 9;            // warp 9: bulk copies of the skewed E rows (lane 0)
constexpr int kCopyBWarp = 10;           // warp 10: bulk copies of the B images (lane 0)
constexpr int kThreadsTotal = kWorkers + 3 * 32;
constexpr int kStageStride = 65;         // epilogue staging row stride (floats)

__device__ __forceinline__ void workers_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kWorkers) : "memory");
}

// COLS = false: grad_x rows (A = E rows i, K = j, B = [Y | 1]).
// COLS = true : grad_y rows (A = E columns j, K = i, B = [X | 1]).
// bimg: per problem, per K-tile, the pre-split B image (bimg_kernel).
//
// Warp-specialised pipeline, all hand-offs through mbarriers:
//   MMA warp   : MMAs of tile kt once its A stage is full and its B image has landed,
//                committed to the A-stage and B-buffer "empty" barriers.
//   copy warps : raw E rows of tile k once the workers released entry k % pa; the B
//                image of tile k once MMA(k - pb) has freed buffer k % pb.
//   workers    : wait for raw A of tile kt and for A stage kt%ts to be empty (MMA(kt-ts)),
//             un-skew + split into the stage, then each warp arrives on "raw empty" and
//             "A full". After the last commit they stage the accumulators through shared
//             memory and write the gradient rows with coalesced stores.
// Barrier parities: entry e of a ring of depth P serves tiles e, e+P, ...; tile k's
// phase has parity (k/P)&1 and every wait is for the oldest phase not yet reused.
template <bool COLS>
__global__ void __launch_bounds__(kThreadsTotal, 1)
    egemm_kernel(const GradParams g, const float* __restrict__ bimg, int n_total, Pipe pp, int* status)
{
    extern __shared__ unsigned char smem_dyn[];
    __shared__ uint64_t s_raw_full[kMaxRing], s_raw_empty[kMaxRing];
    __shared__ uint64_t s_b_full[kMaxRing], s_b_empty[kMaxRing];
    __shared__ uint64_t s_a_full[kMaxRing], s_a_empty[kMaxRing];
    __shared__ uint64_t s_acc;
    __shared__ uint32_t s_tmem;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int p = blockIdx.y;
    const int m0 = blockIdx.x * kBM;
    const int N = g.N, M = g.M, D = g.D, T = skew_T(M);
    const int rows = COLS ? M : N;     // output rows
    const int kdim = COLS ? N : M;     // reduction length
    const int NB = (N + 31) / 32;
    const int nK = (kdim + kBK - 1) / kBK;
    const int ts = pp.ts, pb = pp.pb, pa = pp.pa;
    // [B_hi; B_lo] as one operand of 2*n_total rows: A_hi x [B_hi; B_lo] + A_lo x B_hi
    const bool stacked = 2 * n_total <= 256;
    const float* Ekp = g.E + skew_index(N, M, p, 0, 0, 0);
    const float* bimg_p = bimg + (size_t)p * nK * 2 * n_total * 32;

    // Shared memory (1 KiB aligned): ts A stages [hi | lo], pb B images [hi | lo], pa raw A buffers.
    const uint32_t a_bytes = kBM * 128, b_bytes = (uint32_t)n_total * 128;
    const uint32_t rawA_bytes = Raw<COLS>::kBytes;
    unsigned char* base = smem_dyn + ((1024u - (smem_u32(smem_dyn) & 1023u)) & 1023u);
    unsigned char* bbase = base + ts * 2 * a_bytes;
    unsigned char* rbase = bbase + pb * 2 * b_bytes;
    auto astage = [&](int kt) { return base + (kt % ts) * 2 * a_bytes; };
    auto bbuf = [&](int kt) { return bbase + (kt % pb) * 2 * b_bytes; };
    auto rawA = [&](int kt) { return rbase + (kt % pa) * rawA_bytes; };

    if (tid == 0) {
        for (int b = 0; b < kMaxRing; ++b) {
            mbar_init(smem_u32(&s_raw_full[b]), 1);
            mbar_init(smem_u32(&s_raw_empty[b]), kWorkers / 32);
            mbar_init(smem_u32(&s_b_full[b]), 1);
            mbar_init(smem_u32(&s_b_empty[b]), 1);
        }
        for (int b = 0; b < kMaxRing; ++b) {
            mbar_init(smem_u32(&s_a_full[b]), kWorkers / 32);
            mbar_init(smem_u32(&s_a_empty[b]), 1);
        }
        mbar_init(smem_u32(&s_acc), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    int ncols = 32;
    while (ncols < (stacked ? 2 * n_total : n_total)) ncols <<= 1;
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
    bool ok = true;

    if (warp == kMmaWarp) {
        if (lane == 0) {
            for (int kt = 0; kt < nK && ok; ++kt) {
                wait_ok(ok, smem_u32(&s_a_full[kt % ts]), (uint32_t)((kt / ts) & 1), status);
                wait_ok(ok, smem_u32(&s_b_full[kt % pb]), (uint32_t)((kt / pb) & 1), status);
                if (!ok) break;
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t ah = smem_u32(astage(kt)), al = ah + a_bytes;
                const uint32_t bh = smem_u32(bbuf(kt)), bl_ = bh + b_bytes;
                if (stacked) {
                    const uint32_t id2 = idesc_tf32(kBM, 2 * n_total), id1 = idesc_tf32(kBM, n_total);
#pragma unroll
                    for (int ks = 0; ks < kBK / 8; ++ks) {
                        const uint32_t ko = ks * 32;  // 8 tf32 = 32 bytes along K
                        mma_tf32(tmem, sdesc(ah + ko), sdesc(bh + ko), id2, (kt > 0 || ks > 0) ? 1u : 0u);
                        mma_tf32(tmem, sdesc(al + ko), sdesc(bh + ko), id1, 1u);
                    }
                } else {
                    for (int n0 = 0; n0 < n_total; n0 += 256) {
                        const int nn = min(256, n_total - n0);
                        const uint32_t id = idesc_tf32(kBM, nn);
                        const uint32_t d = tmem + (uint32_t)n0;
                        const uint32_t boff = (uint32_t)n0 * 128;
#pragma unroll
                        for (int ks = 0; ks < kBK / 8; ++ks) {
                            const uint32_t ko = ks * 32;
                            mma_tf32(d, sdesc(ah + ko), sdesc(bh + boff + ko), id, (kt > 0 || ks > 0) ? 1u : 0u);
                            mma_tf32(d, sdesc(al + ko), sdesc(bh + boff + ko), id, 1u);
                            mma_tf32(d, sdesc(ah + ko), sdesc(bl_ + boff + ko), id, 1u);
                        }
                    }
                }
                mma_commit(smem_u32(&s_a_empty[kt % ts]));
                mma_commit(smem_u32(&s_b_empty[kt % pb]));
            }
            // releases the workers once every MMA issued above has completed
            mma_commit(smem_u32(&s_acc));
        }
        __syncwarp();
    } else if (warp == kCopyAWarp) {
        // raw E rows of tile k into entry k % pa, once the workers released tile k - pa
        if (lane == 0) {
            int last[kMaxRing];
            for (int e = 0; e < kMaxRing; ++e) last[e] = -1;
            for (int k = 0; k < nK && ok; ++k) {
                if (k >= pa) wait_ok(ok, smem_u32(&s_raw_empty[k % pa]), (uint32_t)(((k - pa) / pa) & 1), status);
                if (!ok) break;
                issue_a<COLS>(Ekp, N, M, T, m0, k, rawA(k), smem_u32(&s_raw_full[k % pa]));
                last[k % pa] = k;
            }
            bool drained = true;  // no copy may still be writing shared memory when the CTA exits
            for (int e = 0; e < kMaxRing; ++e)
                if (last[e] >= 0) wait_ok(drained, smem_u32(&s_raw_full[e]), (uint32_t)((last[e] / pa) & 1), status);
        }
        __syncwarp();
    } else if (warp == kCopyBWarp) {
        // B image of tile k into buffer k % pb, once MMA(k - pb) has read it
        if (lane == 0) {
            int last[kMaxRing];
            for (int e = 0; e < kMaxRing; ++e) last[e] = -1;
            for (int k = 0; k < nK && ok; ++k) {
                if (k >= pb) wait_ok(ok, smem_u32(&s_b_empty[k % pb]), (uint32_t)(((k - pb) / pb) & 1), status);
                if (!ok) break;
                issue_b(bimg_p, n_total, k, bbuf(k), smem_u32(&s_b_full[k % pb]));
                last[k % pb] = k;
            }
            bool drained = true;
            for (int e = 0; e < kMaxRing; ++e)
                if (last[e] >= 0) wait_ok(drained, smem_u32(&s_b_full[e]), (uint32_t)((last[e] / pb) & 1), status);
        }
        __syncwarp();
    } else {
        const int quarter = warp & 3, half = warp >> 2;
        for (int kt = 0; kt < nK; ++kt) {
            wait_ok(ok, smem_u32(&s_raw_full[kt % pa]), (uint32_t)((kt / pa) & 1), status);
            if (kt >= ts) wait_ok(ok, smem_u32(&s_a_empty[kt % ts]), (uint32_t)(((kt - ts) / ts) & 1), status);
            unsigned char* A_hi = astage(kt);
            unsigned char* A_lo = A_hi + a_bytes;
            const int k0 = kt * kBK;
            const float* ra = reinterpret_cast<const float*>(rawA(kt));
            if (!COLS) {
                // warps w, w+4: row block m0/32 + (w mod 4), lane = row, 16-byte chunks
                // 4*half .. 4*half+3 of the row. The skewed reads hit bank `lane`; in the
                // swizzled stores each 8-lane phase covers the 8 chunk slots of one atom.
                const int rb = (m0 >> 5) + quarter;
                const int rloc = 32 * quarter + lane;
                const bool rowok = rb < NB && m0 + rloc < N;
                const float* rw = ra + quarter * 64 * 32 + lane * 33;   // slot (c + lane), entry lane
                const uint32_t rowoff = (uint32_t)((rloc >> 3) * 1024 + (rloc & 7) * 128);
                // all 16 values first: the stage stores could alias the raw buffer for the
                // compiler, which would otherwise chain every load behind the previous store
                float vals[16];
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const int c = 4 * (half * 4 + (u >> 2)) + (u & 3);
                    vals[u] = (rowok && k0 + c < M) ? rw[c * 32] : 0.f;
                }
#pragma unroll
                for (int cq = 0; cq < 4; ++cq) {
                    const int kc = half * 4 + cq;
                    float4 hi, lo;
                    float* h = &hi.x;
                    float* l = &lo.x;
#pragma unroll
                    for (int q = 0; q < 4; ++q) split_tf32(vals[4 * cq + q], h[q], l[q]);
                    const uint32_t o = rowoff + (uint32_t)(((kc ^ rloc) & 7) << 4);
                    *reinterpret_cast<float4*>(A_hi + o) = hi;
                    *reinterpret_cast<float4*>(A_lo + o) = lo;
                }
            } else {
                // raw row tt holds slot m0 + tt of block k0/32; lane = K index i - k0. Warp w
                // takes output rows rr = w + 8*it, so rr mod 8 = w and the swizzled offset
                // is it*1024 plus a per-thread constant.
                const bool iok = k0 + lane < N;
                const float* rp = ra + (warp + lane) * 32 + lane;
                const uint32_t coff = (uint32_t)(warp * 128 + ((((lane >> 2) ^ warp) & 7) << 4) + (lane & 3) * 4);
                float vals[kBM / 8];
#pragma unroll
                for (int it = 0; it < kBM / 8; ++it) vals[it] = (iok && m0 + warp + 8 * it < M) ? rp[it * 8 * 32] : 0.f;
#pragma unroll
                for (int it = 0; it < kBM / 8; ++it) {
                    float h, l;
                    split_tf32(vals[it], h, l);
                    *reinterpret_cast<float*>(A_hi + coff + it * 1024) = h;
                    *reinterpret_cast<float*>(A_lo + coff + it * 1024) = l;
                }
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(smem_u32(&s_raw_empty[kt % pa]));
                mbar_arrive(smem_u32(&s_a_full[kt % ts]));
            }
        }
        // The epilogue's first batch of loads (own rows, and the output when it
        // accumulates) does not depend on the products: it goes out before the wait.
        constexpr int kR = 16;  // rows per batch of epilogue loads
        const float* own = COLS ? g.pr.y(p) : g.pr.x(p);
        float* out = g.out + (long long)(p % g.omod) * g.out_stride;
        float ov0[kR], pv0[kR];
        {
            const int c = tid & 63, r0 = tid >> 6;
            if (c < D) {
#pragma unroll
                for (int k = 0; k < kR; ++k) {
                    const size_t o = (size_t)min(m0 + r0 + 4 * k, rows - 1) * D + c;
                    ov0[k] = own[o];
                    pv0[k] = g.accumulate ? out[o] : 0.f;
                }
            }
        }
        // every MMA has completed (and every copy has landed) once s_acc fires
        {
            bool fin = true;
            wait_ok(fin, smem_u32(&s_acc), 0u, status);
            ok = ok && fin;
        }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");

        // ---- epilogue: warp w holds output rows m0 + 32(w mod 4) + lane in TMEM lane quarter w mod 4.
        // Accumulators go to a [128 x 64] shared tile per group of 64 columns, then all
        // workers write the group row by row with coalesced loads of own[] and stores.
        float* stg = reinterpret_cast<float*>(base);
        float* ssum = stg + kBM * kStageStride;
        const int r_own = 32 * quarter + lane;
        const uint32_t trow = tmem + ((uint32_t)(32 * quarter) << 16);
        if (half == 0) {
            float v[16];
            float s = 0.f;
            tmem_ld16(trow + (uint32_t)(D & ~15), v);
#pragma unroll
            for (int q = 0; q < 16; ++q) s += (q == (D & 15)) ? v[q] : 0.f;
            if (stacked) {
                tmem_ld16(trow + (uint32_t)(n_total + (D & ~15)), v);
#pragma unroll
                for (int q = 0; q < 16; ++q) s += (q == (D & 15)) ? v[q] : 0.f;
            }
            ssum[r_own] = s;
        }
        const float w = g.coef * 2.f * (g.grad_loss ? g.grad_loss[p % g.wmod] : 1.f);
        for (int g0 = 0; g0 < D; g0 += 64) {
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const int c0 = g0 + (2 * half + cc) * 16;
                if (c0 < D) {
                    float v[16];
                    tmem_ld16(trow + (uint32_t)c0, v);
                    if (stacked) {
                        float u[16];
                        tmem_ld16(trow + (uint32_t)(n_total + c0), u);
#pragma unroll
                        for (int q = 0; q < 16; ++q) v[q] += u[q];
                    }
#pragma unroll
                    for (int q = 0; q < 16; ++q) stg[r_own * kStageStride + (c0 - g0) + q] = v[q];
                }
            }
            workers_sync();
            // thread: column g0 + (tid mod 64) of rows (tid / 64) + 4k; every load of the
            // group is issued before the first store
            const int c = tid & 63, r0 = tid >> 6;
            if (ok && c < D - g0) {
                for (int rb0 = 0; rb0 < kBM; rb0 += 4 * kR) {
                    float ov[kR], pv[kR];
                    if (g0 == 0 && rb0 == 0) {  // loaded before the wait
#pragma unroll
                        for (int k = 0; k < kR; ++k) {
                            ov[k] = ov0[k];
                            pv[k] = pv0[k];
                        }
                    } else {
#pragma unroll
                        for (int k = 0; k < kR; ++k) {
                            const int row = m0 + rb0 + r0 + 4 * k;
                            const size_t o = (size_t)min(row, rows - 1) * D + g0 + c;
                            ov[k] = own[o];
                            pv[k] = g.accumulate ? out[o] : 0.f;
                        }
                    }
#pragma unroll
                    for (int k = 0; k < kR; ++k) {
                        const int r = rb0 + r0 + 4 * k;
                        if (m0 + r < rows)
                            out[(size_t)(m0 + r) * D + g0 + c] =
                                pv[k] + w * (ssum[r] * ov[k] - stg[r * kStageStride + c]);
                    }
                }
            }
            workers_sync();
        }
    }

    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(ncols) : "memory");
    }
}

// Pre-split B operand images, both orientations in one launch (blockIdx.z = 0:
// [Y | 1] for grad_x, 1: [X | 1] for grad_y): for problem p and K-tile kt, rows
// n < D hold coordinate n of the other sequence's rows kt*32 .. kt*32+31, row D
// holds ones; written as the hi then lo tf32 tiles in the swizzled smem layout.
// The 32 source rows are contiguous: every thread loads its share into a
// [32 x (n_total+1)] shared tile first, then warps write 128-byte image rows.
// grid (max K-tiles, P, 2), block 256, dynamic smem 32*(n_total+1)*4; a null
// image pointer skips that orientation.
__global__ void __launch_bounds__(256) bimg_kernel(const GradParams g, int n_total, float* __restrict__ img_rows,
                                                   float* __restrict__ img_cols)
{
    extern __shared__ float t[];
    const bool cols = blockIdx.z == 1;
    const int kt = blockIdx.x, p = blockIdx.y;
    const int D = g.D;
    const int kdim = cols ? g.N : g.M;
    const int nK = (kdim + kBK - 1) / kBK;
    if (kt >= nK) return;
    const float* src = (cols ? g.pr.x(p) : g.pr.y(p)) + (size_t)kt * kBK * D;
    float* img = cols ? img_cols : img_rows;
    if (img == nullptr) return;
    unsigned char* hi = reinterpret_cast<unsigned char*>(img + ((size_t)p * nK + kt) * 2 * n_total * 32);
    unsigned char* lo = hi + (size_t)n_total * 128;
    const int ld = n_total + 1;
    const int here = min(kBK, kdim - kt * kBK);
    // loads in batches of 16 per thread, all issued before their shared stores
    for (int base = 0; base < kBK * n_total; base += 256 * 16) {
        float v[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int idx = base + threadIdx.x + 256 * u;
            const int k = idx / n_total, n = idx - k * n_total;
            float x = 0.f;
            if (idx < kBK * n_total && k < here) x = (n < D) ? src[(size_t)k * D + n] : (n == D ? 1.f : 0.f);
            v[u] = x;
        }
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int idx = base + threadIdx.x + 256 * u;
            const int k = idx / n_total, n = idx - k * n_total;
            if (idx < kBK * n_total) t[k * ld + n] = v[u];
        }
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < kBK * n_total; idx += 256) {
        const int n = idx >> 5, k = idx & 31;
        put(hi, lo, n, k, t[k * ld + n]);
    }
}

}  // namespace

// Shared-memory plan: the deepest pipeline (A stages, B images, raw A buffers)
// that fits in the opt-in limit, preferring two A stages and three-deep rings.
static size_t egemm_bytes(int D, bool cols, Pipe pp)
{
    const int n_total = ((D + 1 + 15) / 16) * 16;
    const size_t a = 2 * (size_t)kBM * 128, b = 2 * (size_t)n_total * 128;
    const size_t raw = cols ? Raw<true>::kBytes : Raw<false>::kBytes;
    return 1024 + pp.ts * a + pp.pb * b + pp.pa * raw;
}

static Pipe egemm_plan(int D, bool cols)
{
    static const Pipe order[] = {{3, 3, 3}, {3, 3, 2}, {2, 3, 3}, {2, 2, 3}, {2, 2, 2}, {1, 2, 2}, {1, 1, 2}};
    for (const Pipe& pp : order)
        if (egemm_bytes(D, cols, pp) <= kSmemLimit) return pp;
    return order[6];
}

size_t egemm_bimg_bytes(int P, int K, int D)
{
    const int n_total = ((D + 1 + 15) / 16) * 16;
    const int nK = (K + kBK - 1) / kBK;
    return (size_t)P * nK * 2 * n_total * 128;
}

cudaError_t launch_bimg(const GradParams& g, float* img_rows, float* img_cols, cudaStream_t st)
{
    const int n_total = ((g.D + 1 + 15) / 16) * 16;
    const int nK = ((g.N > g.M ? g.N : g.M) + kBK - 1) / kBK;
    const size_t smem = sizeof(float) * kBK * (n_total + 1);
    cudaError_t e = cudaFuncSetAttribute(bimg_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    bimg_kernel<<<dim3(nK, g.P, 2), 256, smem, st>>>(g, n_total, img_rows, img_cols);
    return cudaGetLastError();
}

cudaError_t launch_grad_tc(const GradParams& g, bool cols, const float* bimg, int* status, cudaStream_t st)
{
    const int n_total = ((g.D + 1 + 15) / 16) * 16;
    cudaError_t e;
    const Pipe pp = egemm_plan(g.D, cols);
    const size_t smem = egemm_bytes(g.D, cols, pp);
    const int rows = cols ? g.M : g.N;
    dim3 grid((rows + kBM - 1) / kBM, g.P);
    if (cols) {
        e = cudaFuncSetAttribute(egemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        egemm_kernel<true><<<grid, kThreadsTotal, smem, st>>>(g, bimg, n_total, pp, status);
    } else {
        e = cudaFuncSetAttribute(egemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        egemm_kernel<false><<<grid, kThreadsTotal, smem, st>>>(g, bimg, n_total, pp, status);
    }
    return cudaGetLastError();
}

}  // namespace sdtw
