// wavefront_tc.cu -- fused forward wavefront whose costs come from the tensor
// cores (fp32 mode, D <= 64).
//
// Same recursion, strip decomposition and boundary channels as the forward in
// wavefront.cu (difference form, one warp per 32-row block, tagged slots
// between warps and strips). What changes is where the cost of a cell comes
// from: no cost tensor is stored (SoftDTW-CUDA (PyTorch + Numba) README,
// "Fused Mode"), and instead of every DP lane summing D squared differences per
// step, the CTA computes its 128 rows x 32 columns cost tiles as a tcgen05 GEMM:
//
//   C[i,j] = |x_i|^2 + |y_j|^2 - 2 x_i . y_j,
//
// from the exact three-part bf16 operand images of dist_tc.cu (all nine part
// products). The x rows of the CTA stay in
// shared memory and 32-row y tiles stream in by bulk copy. A fifth warp issues
// the copies and MMAs into a ring of
// tensor-memory tiles (three 32-column groups each); at the start of every
// 32-step period each DP warp loads its 32 rows of the next tile (tcgen05.ld),
// releases the tile, and writes the costs into its 64-column shared ring in the
// order its lanes read them. The DP step itself then costs one shared load.
//
// Hand-offs (all mbarriers, all waits bounded):
//   s_bfull[e]  y tile copies landed       (issuer waits)
//   s_bempty[e] MMAs reading entry e done  (issuer waits before refilling)
//   s_tfull[t]  cost tile t in TMEM        (DP warps wait)
//   s_tfree[t]  every DP warp with rows has loaded tile t (issuer waits)
#include "channel.cuh"
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

#include <mutex>

namespace sdtw {

namespace {

using namespace tc;

constexpr int kDpWarps = 4;               // 128 rows per CTA: the MMA tile height
constexpr int kIssuerWarp = kDpWarps;     // warp 4: bulk copies and MMAs
constexpr int kSlotCols = 96;             // tensor-memory columns of a cost tile: the y0, y1, y2 groups
constexpr int kRT = 5;                    // cost tiles in tensor memory
constexpr int kTmemCols = 512;            // the whole tensor memory of the SM (kRT * kSlotCols rounded up)
constexpr int kRB = 3;                    // y tiles in shared memory
constexpr uint32_t kAPart = 128 * 128;    // one bf16 part of one K-block of the CTA's 128 x rows (bytes)
constexpr uint32_t kABlock = 3 * kAPart;  // the three parts [x0 | x1 | x2] of one K-block
constexpr uint32_t kBPart = 32 * 128;     // one part of one K-block of 32 y rows
constexpr uint32_t kBBlock = 3 * kBPart;  // [y0 ; y1 ; y2] of one K-block of a y tile

}  // namespace

size_t wave_tc_smem(int D)
{
    const int KB = (D + kTcKFeat - 1) / kTcKFeat;
    const size_t operands = (size_t)KB * kABlock + (size_t)kRB * KB * kBBlock;
    // per DP warp: a 64-column cost ring and two tiles' y norms
    return wave_smem_fixed(kDpWarps, false) + 1024 + operands + (size_t)kDpWarps * (64 + 2) * 32 * sizeof(float);
}

namespace {

// Thread-block clusters: the strips of one problem that share a cluster hand their
// boundary rows over through distributed shared memory. cluster_map gives the
// generic address of the same shared variable in CTA `rank` of the cluster; the
// slot loads and stores (generic, volatile) work on it unchanged.
__device__ __forceinline__ unsigned cluster_rank() {
    unsigned r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
template <typename T>
__device__ __forceinline__ T* cluster_map(T* p, unsigned rank) {
    unsigned long long a;
    asm volatile("mapa.u64 %0, %1, %2;" : "=l"(a) : "l"(p), "r"(rank));
    return reinterpret_cast<T*>(a);
}
// Barrier of every thread of the cluster (each calls it twice per kernel: after
// the set-up and before leaving, on every path): the writes before it are visible
// to the reads after it in every CTA of the cluster.
__device__ __forceinline__ void cluster_barrier() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// 4-byte asynchronous global -> shared copy (completion: cp.async.wait_group).
__device__ __forceinline__ void cp_async4(float* dst, const float* src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

// STORE: 0, no per-cell state (a checkpointed forward keeps the strips' boundary
// rows only); 1, the state of every row; 2, the state of the row blocks
// [q.vh_rb0, q.vh_rb0 + q.vh_nb) only (one band: the checkpointed forward keeps its
// last band, a band's recompute its own).
template <int STORE, bool CL>
__global__ void __launch_bounds__((kDpWarps + 1) * 32, 1)
    fwd_tc_kernel(const WaveParams q, const unsigned char* __restrict__ ximg, const unsigned char* __restrict__ yimg,
                  const float* __restrict__ xnorm, const float* __restrict__ ynorm)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    constexpr int W = kDpWarps;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    Slot* ring = reinterpret_cast<Slot*>(smem_raw);                          // [W][kRing], by producer warp
    volatile int* cons = reinterpret_cast<volatile int*>(ring + W * kRing);  // [W] columns consumed
    __shared__ int s_tk;
    __shared__ double s_red[kMaxWarps];
    __shared__ int s_last;
    __shared__ uint64_t s_a, s_fin, s_bfull[kRB], s_bempty[kRB], s_tfull[kRT], s_tfree[kRT];
    __shared__ uint32_t s_tmem;
    __shared__ Slot s_xring[CL ? kRing : 1];  // boundary row from the previous CTA of the cluster
    __shared__ int s_xcons;                   // columns of this CTA's boundary row the next CTA consumed
    const int C = CL ? q.C : 1;
    const unsigned crank = C > 1 ? cluster_rank() : 0u;

    if (threadIdx.x == 0 && crank == 0) s_tk = atomicAdd(q.ticket_f, 1);
    if (threadIdx.x < W) cons[threadIdx.x] = 0;
    if (threadIdx.x == 0) s_xcons = 0;
    for (int k = threadIdx.x; k < W * kRing; k += blockDim.x) ring[k].tag = 0u;
    if (CL)
        for (int k = threadIdx.x; k < kRing; k += blockDim.x) s_xring[k].tag = 0u;
    __syncthreads();
    if (C > 1) cluster_barrier();  // every CTA of the cluster initialised; rank 0's ticket visible

    const int tk = C > 1 ? *cluster_map(reinterpret_cast<volatile int*>(&s_tk), 0u) : s_tk;
    const int o = C > 1 ? (tk / q.P) * C + (int)crank : tk / q.P;  // strip in processing order
    if (o >= q.S) {  // a CTA of the cluster past the last strip: no rows, and no peer writes to it
        if (C > 1) cluster_barrier();  // the cluster's final barrier
        return;
    }
    const int p = tk % q.P, strip = q.strip0 + o;
    const int N = q.N, M = q.M, T = skew_T(M);
    const int KB = (q.D + kTcKFeat - 1) / kTcKFeat;
    const int Npad = simg_pad(N), Mpad = simg_pad(M);
    const int rs0 = strip * W * 32;                              // first row of the CTA
    const int nact = min(W, max(1, (N - rs0 + 31) / 32));       // DP warps with rows
    const int nT = (M + 31) / 32;                                // cost tiles

    unsigned char* tcb = smem_raw + q.smem_fixed;
    unsigned char* base = tcb + ((1024u - (smem_u32(tcb) & 1023u)) & 1023u);
    unsigned char* a_img = base;                                  // [KB][x0 | x1 | x2]
    unsigned char* bring = base + KB * kABlock;                   // [kRB][KB][y0 ; y1 ; y2]
    float* dts = reinterpret_cast<float*>(bring + kRB * KB * kBBlock);
    float* nys = dts + W * 64 * 32;                                // [W][2][32] y norms of the next tiles

    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&s_a), 1);
        mbar_init(smem_u32(&s_fin), 1);
        for (int e = 0; e < kRB; ++e) {
            mbar_init(smem_u32(&s_bfull[e]), 1);
            mbar_init(smem_u32(&s_bempty[e]), 1);
        }
        for (int t = 0; t < kRT; ++t) {
            mbar_init(smem_u32(&s_tfull[t]), 1);
            mbar_init(smem_u32(&s_tfree[t]), nact);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) tmem_alloc(&s_tmem, kTmemCols);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = s_tmem;
    int* status = q.status;

    float c0 = 0.f;  // scaled d(i, 0)
    bool active = false;

    if (warp == kIssuerWarp) {
        if (lane == 0) {
            bool ok = true;
            int y_last[kRB];
            for (int e = 0; e < kRB; ++e) y_last[e] = -1;
            mbar_expect_tx(smem_u32(&s_a), (uint32_t)KB * kABlock);
            for (int kb = 0; kb < KB; ++kb)
                for (int part = 0; part < 3; ++part)
                    bulk_g2s(smem_u32(a_img + kb * kABlock + part * kAPart),
                             ximg + simg_offset(p, KB, kb, part, Npad, rs0), kAPart, smem_u32(&s_a));
            auto issue_y = [&](int c) {
                const int e = c % kRB;
                mbar_expect_tx(smem_u32(&s_bfull[e]), (uint32_t)KB * kBBlock);
                for (int kb = 0; kb < KB; ++kb) {
                    unsigned char* dst = bring + (e * KB + kb) * kBBlock;
                    for (int part = 0; part < 3; ++part)
                        bulk_g2s(smem_u32(dst + part * kBPart), yimg + simg_offset(p, KB, kb, part, Mpad, 32 * c),
                                 kBPart, smem_u32(&s_bfull[e]));
                }
                y_last[e] = c;
            };
            for (int c = 0; c < kRB - 1 && c < nT; ++c) issue_y(c);
            wait_ok_sleep(ok, smem_u32(&s_a), 0u, status);
            for (int c = 0; c < nT && ok; ++c) {
                const int t = c % kRT, e = c % kRB;
                if (c >= kRT) wait_ok_sleep(ok, smem_u32(&s_tfree[t]), (uint32_t)(((c - kRT) / kRT) & 1), status);
                wait_ok_sleep(ok, smem_u32(&s_bfull[e]), (uint32_t)((c / kRB) & 1), status);
                if (!ok) break;
                fence_after_sync();
                const uint32_t d = tmem + (uint32_t)(t * kSlotCols);
                for (int kb = 0; kb < KB; ++kb) {
                    const uint32_t a = smem_u32(a_img + kb * kABlock), b = smem_u32(bring + (e * KB + kb) * kBBlock);
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)  // 16 bf16 = 32 bytes along K per step
                        mma_bf16x3(d, a, b, 128, 32, kAPart, ks * 32, (kb > 0 || ks > 0) ? 1u : 0u);
                }
                mma_commit(smem_u32(&s_tfull[t]));
                mma_commit(smem_u32(&s_bempty[e]));
                // y tile c + kRB - 1 goes to entry (c - 1) % kRB, last read by MMA(c - 1)
                const int cy = c + kRB - 1;
                if (cy < nT) {
                    if (c >= 1) wait_ok_sleep(ok, smem_u32(&s_bempty[(c - 1) % kRB]), (uint32_t)(((c - 1) / kRB) & 1), status);
                    if (!ok) break;
                    issue_y(cy);
                }
            }
            // every MMA issued above has completed before tensor memory is released,
            // and no copy is still writing shared memory when the CTA exits
            mma_commit(smem_u32(&s_fin));
            bool fin = true;
            wait_ok_sleep(fin, smem_u32(&s_fin), 0u, status);
            for (int e = 0; e < kRB; ++e)
                if (y_last[e] >= 0) wait_ok_sleep(fin, smem_u32(&s_bfull[e]), (uint32_t)((y_last[e] / kRB) & 1), status);
        }
        __syncwarp();
    } else {
        const int rb = strip * W + warp, r0 = rb * 32, i = r0 + lane;
        active = r0 < N;
        const bool has_top = active && r0 > 0;
        const bool top_x = has_top && warp == 0 && crank > 0;  // from the previous CTA of the cluster
        const bool top_global = has_top && warp == 0 && !top_x;
        const bool has_bot = active && (r0 + 32 < N);
        const bool bot_x = has_bot && warp == W - 1 && (int)crank < C - 1;  // to the next CTA of the cluster
        const bool bot_global = has_bot && warp == W - 1 && !bot_x;
        const bool row0_lane = (i == 0);
        // this problem's own lengths (a padded batch): it aligns rows < Nb, columns < Mb
        const int Nb = q.lens_n ? min(max(q.lens_n[p], 1), N) : N;
        const int Mb = q.lens_m ? min(max(q.lens_m[p], 1), M) : M;
        const bool last_lane = (i == Nb - 1);
        const float scale = q.scale;
        float* rowbuf = q.rowbuf + (size_t)p * M;
        float* dt = dts + warp * 64 * 32;  // [64][32] raw cost, slot (col & 63), lane
        const float nx = xnorm[(size_t)p * Npad + i];
        const float* nyp = ynorm + (size_t)p * Mpad;
        // the 32 y norms of a cost tile reach shared memory one period ahead (cp.async),
        // so no global load is waited for at the start of a period
        float* nyw = nys + warp * 2 * 32;
        const uint32_t tq = tmem + ((uint32_t)(32 * warp) << 16);
        if (active) {
            cp_async4(nyw + lane, nyp + lane);
            asm volatile("cp.async.commit_group;" ::: "memory");
        }

        if (active) {
            const bool store_rows = STORE == 1 || (STORE == 2 && rb >= q.vh_rb0 && rb < q.vh_rb0 + q.vh_nb);
            float2* vhp = store_rows ? q.VH + band_index(q, p, rb, lane, T) : nullptr;
            Slot* ring_out = ring + warp * kRing;
            const Slot* ring_in = top_x ? s_xring : ring + (warp - 1) * kRing;
            Slot* edge_out = q.edge_f + ((size_t)p * strips_all(q) + strip) * M;
            const Slot* edge_in = q.edge_f + ((size_t)p * strips_all(q) + strip - 1) * M;
            const bool chan_lane =
                has_bot && lane == 31 && !(q.skip_publish && strip == 0 && (bot_global || bot_x));
            Slot* chan_out = bot_global ? edge_out : (bot_x ? cluster_map(s_xring, crank + 1) : ring_out);
            volatile int* bot_cons = bot_x ? reinterpret_cast<volatile int*>(&s_xcons) : cons + warp;
            const int chan_mask = bot_global ? 0x7fffffff : (kRing - 1);
            Slot nxt[1];
            nxt[0].v = 0.f;
            nxt[0].tag = 0u;
            if (top_global && lane < kGroup && lane < M) nxt[0] = slot_load(edge_in + lane);

            float h_prev = 0.f, v_prev = 0.f;
            bool tc_ok = true;
            int cons_seen = 0;  // last count read from the next warp's consumption counter
            const int nG = T / kGroup;
            for (int g = 0; g < nG; ++g) {
                const int s0 = g * kGroup;
                if ((s0 & 31) == 0 && (s0 >> 5) < nT) {
                    // Period c = s0/32 reads columns of tiles c-1 and c: bring tile c in. Its
                    // ring slots last held tile c-2, whose last read was at step s0-2.
                    const int c = s0 >> 5, t = c % kRT;
                    wait_ok(tc_ok, smem_u32(&s_tfull[t]), (uint32_t)((c / kRT) & 1), status);
                    if (!__all_sync(kFull, tc_ok)) break;
                    fence_after_sync();
                    float a[32], b[32], e[32];
                    tmem_ld32(tq + (uint32_t)(t * kSlotCols), a);
                    tmem_ld32(tq + (uint32_t)(t * kSlotCols + 32), b);
                    tmem_ld32(tq + (uint32_t)(t * kSlotCols + 64), e);
                    fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&s_tfree[t]));
                    asm volatile("cp.async.wait_group 0;" ::: "memory");
                    __syncwarp();
                    const float nyv = nyw[(c & 1) * 32 + lane];
                    if (c + 1 < nT) {  // its buffer was last read in period c - 1
                        cp_async4(nyw + ((c + 1) & 1) * 32 + lane, nyp + 32 * (c + 1) + lane);
                        asm volatile("cp.async.commit_group;" ::: "memory");
                    }
#pragma unroll
                    for (int u = 0; u < 32; ++u) {
                        const float ny = __shfl_sync(kFull, nyv, u);
                        dt[((32 * c + u) & 63) * 32 + lane] = fmaxf(nx + ny - 2.f * (a[u] + (b[u] + e[u])), 0.f);
                    }
                    __syncwarp();
                }

                // Upper-neighbour values for lane 0: lane q holds column s0 + q.
                float topv = 0.f;
                bool ok = true;
                if (has_top && s0 < M) {
                    const int col = s0 + lane;
                    const unsigned want = (lane < kGroup && col < M) ? (unsigned)(col + 1) : 0u;
                    Slot cur[1];
                    if (top_global) {
                        cur[0] = nxt[0];
                        ok = validate(cur, edge_in + col, want, q);
                        const int ncol = col + kGroup;
                        if (ok && lane < kGroup && ncol < M) nxt[0] = slot_load(edge_in + ncol);
                    } else {
                        cur[0].v = 0.f;
                        cur[0].tag = 0u;
                        if (want) cur[0] = slot_load(ring_in + (col & (kRing - 1)));
                        ok = validate(cur, ring_in + (col & (kRing - 1)), want, q);
                    }
                    topv = cur[0].v;
                }
                if (ok && has_bot && !bot_global) {
                    const int need = s0 + kGroup - 31 - kRing;  // ring slots this group overwrites are free
                    if (need > cons_seen) ok = wait_smem(bot_cons, need, q, cons_seen);
                }
                if (!ok) break;

#pragma unroll
                for (int u = 0; u < kGroup; ++u) {
                    const int s = s0 + u;
                    const int j = s - lane;
                    const float hs = __shfl_up_sync(kFull, h_prev, 1);
                    const float tv = __shfl_sync(kFull, topv, u);
                    const float hu = (lane == 0) ? tv : hs;
                    const float vl = v_prev;
                    const float d = dt[(j & 63) * 32 + lane] * scale;
                    float lo, mid, hi;
                    sort3(0.f, vl, hu, lo, mid, hi);
                    const float lz = lg2((1.f + ex2(lo - mid)) + ex2(lo - hi));
                    const float tt = (d + lo) - lz;
                    const bool col0 = (j == 0);
                    // border values picked off the dependency chain: one select follows tt
                    const bool border = col0 || row0_lane;
                    const float hb = col0 ? -kBig : d, vb = row0_lane ? -kBig : d;
                    const float h = border ? hb : tt - vl;
                    const float v = border ? vb : tt - hu;
                    const float svl = col0 ? kBig : (row0_lane ? -kBig : vl);
                    const float shu = row0_lane ? kBig : (col0 ? -kBig : hu);
                    c0 = col0 ? d : c0;
                    if constexpr (STORE == 1) vhp[(long long)s * 32] = make_float2(svl, shu);
                    if constexpr (STORE == 2) {
                        if (store_rows) vhp[(long long)s * 32] = make_float2(svl, shu);
                    }
                    const bool valid = (unsigned)j < (unsigned)M;
                    slot_store_if(chan_lane && valid, chan_out + (j & chan_mask), h, (unsigned)(j + 1));
                    if (last_lane && (unsigned)j < (unsigned)Mb) rowbuf[j] = h;
                    h_prev = h;
                    v_prev = v;
                }

                if (has_top && !top_global && lane == 0) {
                    const int used = min(s0 + kGroup, M);
                    if (top_x) *cluster_map(reinterpret_cast<volatile int*>(&s_xcons), crank - 1) = used;
                    else cons[warp - 1] = used;
                }
            }
            asm volatile("cp.async.wait_all;" ::: "memory");  // none in flight past an early exit
        }
    }

    // Loss: R[N,M] = sum_i d(i,0) + sum_{j>=1} h(N-1, j), scaled units (not in a recompute).
    if (!q.no_loss) {
    const int Nb = q.lens_n ? min(max(q.lens_n[p], 1), N) : N;
    const int Mb = q.lens_m ? min(max(q.lens_m[p], 1), M) : M;
    double part = (active && warp < W && rs0 + 32 * warp + lane < Nb) ? (double)c0 : 0.0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(kFull, part, o);
    if (lane == 0) s_red[warp] = part;
    __threadfence();
    __syncthreads();
    float* rowbuf = q.rowbuf + (size_t)p * M;
    if (threadIdx.x == 0) {
        double cs = 0.0;
        for (int w = 0; w < W; ++w) cs += s_red[w];
        q.colsum[(size_t)p * q.NB + strip] = cs;
        __threadfence();
        s_last = (atomicAdd(&q.done[p], 1) == strips_all(q) - 1);
    }
    __syncthreads();
    if (s_last) {  // the last strip of problem p to finish assembles its loss
        __threadfence();
        double acc = 0.0;
        for (int j = 1 + (int)threadIdx.x; j < Mb; j += blockDim.x) acc += (double)__ldcg(rowbuf + j);
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(kFull, acc, o);
        if (lane == 0) s_red[warp] = acc;
        __syncthreads();
        if (threadIdx.x == 0) {
            double tot = 0.0;
            for (int w = 0; w <= W; ++w) tot += s_red[w];
            for (int k = 0; k < strips_all(q); ++k) tot += __ldcg(&q.colsum[(size_t)p * q.NB + k]);
            q.loss[p] = (float)(tot * (double)q.unscale);
        }
    }
    }

    fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
    if (C > 1) cluster_barrier();  // no CTA leaves while a peer may still write its shared memory
}

}  // namespace

namespace {

// Cluster size (1, 2 or 4) for a fused forward launch of kern, q.C being the
// caller's limit: clusters only when the strips are the whole problem (no band
// launch) and every cluster of the launch can be resident at once (a launch of
// several waves keeps every SM).
int tc_cluster(const WaveParams& q, const void* kern, int threads, size_t smem)
{
    if (q.C < 2 || q.S < 2 || q.strip0 != 0 || (q.S_all != 0 && q.S_all != q.S)) return 1;
    struct Entry { const void* kern; int C, threads; size_t smem; int clusters; };
    static Entry cache[32];
    static int used = 0;
    static std::mutex mu;
    for (int C = q.C >= 4 ? 4 : 2; C >= 2; C >>= 1) {
        if (C > q.S) continue;
        const long long grid = (long long)q.P * ((q.S + C - 1) / C) * C;
        int clusters = -1;
        {
            std::lock_guard<std::mutex> lk(mu);
            for (int k = 0; k < used; ++k)
                if (cache[k].kern == kern && cache[k].C == C && cache[k].threads == threads && cache[k].smem == smem)
                    clusters = cache[k].clusters;
        }
        if (clusters < 0) {
            cudaLaunchConfig_t cfg{};
            cudaLaunchAttribute at[1];
            at[0].id = cudaLaunchAttributeClusterDimension;
            at[0].val.clusterDim.x = (unsigned)C;
            at[0].val.clusterDim.y = 1;
            at[0].val.clusterDim.z = 1;
            cfg.gridDim = dim3((unsigned)C);
            cfg.blockDim = dim3((unsigned)threads);
            cfg.dynamicSmemBytes = smem;
            cfg.attrs = at;
            cfg.numAttrs = 1;
            if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess) {
                cudaGetLastError();
                clusters = 0;
            }
            std::lock_guard<std::mutex> lk(mu);
            if (used < 32) cache[used++] = Entry{kern, C, threads, smem, clusters};
        }
        if ((long long)clusters * C >= grid) return C;
    }
    return 1;
}

}  // namespace

cudaError_t launch_forward_tc(WaveParams q, const void* ximg, const void* yimg, const float* xnorm,
                              const float* ynorm, cudaStream_t st)
{
    if (q.W != kDpWarps || q.D > kTcKFeat * kMaxTcKBlocks) return cudaErrorInvalidValue;
    q.smem_fixed = (int)wave_smem_fixed(kDpWarps, false);
    // more than half of the SM's shared memory: one CTA per SM, which the
    // 512-column tensor-memory allocation relies on
    int dev = 0, per_sm = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess || per_sm <= 0)
        per_sm = 228 * 1024;
    const size_t smem = max(wave_tc_smem(q.D), (size_t)per_sm / 2 + 1024);
    // A checkpointed forward (STORE 0 or 2) keeps every strip's boundary row in the
    // global edge buffer for the band recomputes: no clusters there.
    // kern_cl: the build with the cluster paths; kern: without them (every cluster
    // branch compiled out), which runs when no cluster is used.
    auto go = [&](auto kern_cl, auto kern, bool may_cluster) -> cudaError_t {
        constexpr int threads = (kDpWarps + 1) * 32;
        const unsigned char* xi = static_cast<const unsigned char*>(ximg);
        const unsigned char* yi = static_cast<const unsigned char*>(yimg);
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e == cudaSuccess && may_cluster)
            e = cudaFuncSetAttribute(kern_cl, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        q.C = may_cluster ? tc_cluster(q, reinterpret_cast<const void*>(kern_cl), threads, smem) : 1;
        if (q.C <= 1) {
            kern<<<q.P * q.S, threads, smem, st>>>(q, xi, yi, xnorm, ynorm);
            return cudaGetLastError();
        }
        cudaLaunchConfig_t cfg{};
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = (unsigned)q.C;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3((unsigned)(q.P * ((q.S + q.C - 1) / q.C) * q.C));
        cfg.blockDim = dim3((unsigned)threads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = st;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, kern_cl, q, xi, yi, xnorm, ynorm);
    };
    if (q.VH == nullptr) return go(fwd_tc_kernel<0, false>, fwd_tc_kernel<0, false>, false);
    if (q.vh_nb > 0) return go(fwd_tc_kernel<2, false>, fwd_tc_kernel<2, false>, false);
    return go(fwd_tc_kernel<1, true>, fwd_tc_kernel<1, false>, true);
}

}  // namespace sdtw
