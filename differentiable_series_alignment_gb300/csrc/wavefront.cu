// wavefront.cu -- single-launch wavefront kernels for the Soft-DTW DP.
//
// Forward: the soft-min recursion of Cuturi & Blondel (ICML 2017), carried in
// the difference form described in common.cuh. Backward: the alignment matrix
// E by the reverse recursion done in log space, exponentiated only after the
// log-domain DP (SoftDTW-CUDA-Torch paper, abstract, contribution (2)).
//
// Work decomposition (the same for both directions):
//  * A warp owns 32 consecutive rows (lane = row) and walks the anti-diagonals
//    of its 32-row block: at step s lane l handles column s - l (forward) or
//    column M-1 - (s - (31-l)) (backward). The left (right) neighbour stays in
//    a register, the upper (lower) neighbour arrives by one warp shuffle.
//  * A CTA owns a strip of W warps = 32W rows. Adjacent warps exchange the
//    boundary row through a shared-memory ring of tagged slots (value and
//    column tag in one 64-bit word, so no fence or ready counter is needed).
//  * Strips exchange their boundary row through tagged slots in global memory,
//    loaded one group ahead of use. Strips are handed out by an atomic ticket
//    in dependency order, so a CTA only ever waits on a strip already owned by
//    a running CTA; this holds whatever the grid size and residency.
//  * Every wait is bounded (global timer); on expiry the kernel sets the
//    device status word and every other wait then gives up too.
//
// This replaces the per-anti-diagonal kernel launches of the pages' design
// (review page, "proposed method", first bullet) by one launch per direction.
#include "channel.cuh"
#include "common.cuh"
#include "kernels.h"

#include <type_traits>

namespace sdtw {

namespace {

struct FusedSmem {
    float* xs;  // [32][XS]     rows of this warp, zero padded to D4
    float* ys;  // [2][32][XS]  y rows of the next two 32-column tiles (cp.async double buffer)
    float* dt;  // [64][32]     raw cost of two 32-column tiles, slot (col & 63), lane
};

__device__ __forceinline__ void cp_async16(float* dst, const float* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async4f(float* dst, const float* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src)
                 : "memory");
}

// Stage y rows [c0, c0+32) of one problem into a [32][XS] tile (zero padded).
// Asynchronous (cp.async); the caller waits with cp.async.wait_all + __syncwarp.
__device__ __forceinline__ void stage_y_tile(float* tile, const float* yb, int c0, int M, int D, int D4, int XS,
                                             int lane)
{
    const bool vec = ((D & 3) == 0) && ((reinterpret_cast<uintptr_t>(yb) & 15) == 0);
    if (vec) {
        const int per = D4 >> 2;  // float4 per (padded) row
        for (int e = lane; e < 32 * per; e += 32) {
            const int r = e / per, q = e - r * per;
            float* dst = tile + r * XS + 4 * q;
            if (c0 + r < M && 4 * q < D) cp_async16(dst, yb + (size_t)(c0 + r) * D + 4 * q);
            else *reinterpret_cast<float4*>(dst) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    } else {
        for (int e = lane; e < 32 * D4; e += 32) {
            const int r = e / D4, k = e - r * D4;
            float* dst = tile + r * XS + k;
            if (c0 + r < M && k < D) cp_async4f(dst, yb + (size_t)(c0 + r) * D + k);
            else *dst = 0.f;
        }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
}

}  // namespace

// ---------------------------------------------------------------------------
// Forward
// ---------------------------------------------------------------------------
// DX (fused only): 32 or 64 keeps the warp's x rows in registers, padded to DX
// components (D <= DX); 0 reads them from shared memory (D > 64).
template <bool FUSED, int DX>
__global__ void __launch_bounds__(FUSED ? 256 : kMaxWarps * 32, 1) fwd_kernel(const WaveParams q)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int W = q.W;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    Slot* ring = reinterpret_cast<Slot*>(smem_raw);                      // [W][kRing], by producer warp
    volatile int* cons = reinterpret_cast<volatile int*>(ring + W * kRing);  // [W] columns consumed
    __shared__ int s_tk;
    __shared__ double s_red[kMaxWarps];
    __shared__ int s_last;

    if (threadIdx.x == 0) s_tk = atomicAdd(q.ticket_f, 1);
    if (threadIdx.x < W) cons[threadIdx.x] = 0;
    for (int k = threadIdx.x; k < W * kRing; k += blockDim.x) ring[k].tag = 0u;
    __syncthreads();

    const int tk = s_tk;
    const int p = tk % q.P, strip = tk / q.P;
    const int N = q.N, M = q.M, T = skew_T(M);
    const int rb = strip * W + warp, r0 = rb * 32, i = r0 + lane;
    const bool active = r0 < N;
    const bool has_top = active && r0 > 0;
    const bool top_global = has_top && warp == 0;
    const bool has_bot = active && (r0 + 32 < N);
    const bool bot_global = has_bot && warp == W - 1;
    // this problem's own lengths (a padded batch): it aligns rows < Nb, columns < Mb
    const int Nb = q.lens_n ? min(max(q.lens_n[p], 1), N) : N;
    const int Mb = q.lens_m ? min(max(q.lens_m[p], 1), M) : M;
    const bool row0_lane = (i == 0);
    const bool last_lane = (i == Nb - 1);
    const float scale = q.scale;
    float* rowbuf = q.rowbuf + (size_t)p * M;

    float c0 = 0.f;  // scaled d(i, 0)

    // Fused: each warp keeps its 32 rows of x, y rows of the next two 32-column
    // tiles and the raw costs of two tiles. The cost of column s+32 is computed
    // for all 32 rows during DP step s, one column per step, interleaved with the
    // latency-bound recursion.
    FusedSmem fz{};
    int XS = 0, D4 = 0;
    const float* yb = q.pr.y(p);
    if (FUSED) {
        const int D = q.D;
        D4 = (D + 31) & ~31;   // rows zero-padded to whole 32-component groups
        XS = D4 + 4;
        float* base = reinterpret_cast<float*>(smem_raw + q.smem_fixed);
        float* mine = base + (size_t)warp * (96 * XS + 64 * 32);
        fz.xs = mine;
        fz.ys = mine + 32 * XS;
        fz.dt = mine + 96 * XS;
        const float* xb = q.pr.x(p);
        for (int e = lane; e < 32 * D4; e += 32) {
            const int r = e / D4, k = e - r * D4;
            fz.xs[r * XS + k] = (r0 + r < N && k < D) ? xb[(size_t)(r0 + r) * D + k] : 0.f;
        }
        if (active) {
            stage_y_tile(fz.ys, yb, 0, M, D, D4, XS, lane);             // tile 0 -> buffer 0
            stage_y_tile(fz.ys + 32 * XS, yb, 32, M, D, D4, XS, lane);  // tile 1 -> buffer 1
            asm volatile("cp.async.wait_group 1;" ::: "memory");
            __syncwarp();
        }
    }
    float xr[DX > 0 ? DX : 1];
    if constexpr (FUSED && DX > 0) {
#pragma unroll
        for (int k = 0; k < DX; ++k) xr[k] = fz.xs[lane * XS + k];
    }
    if (FUSED && active) {
        for (int c = 0; c < 32 && c < M; ++c) {  // costs of tile 0
            if constexpr (DX > 0) fz.dt[c * 32 + lane] = dist_reg<DX>(xr, fz.ys + c * XS);
            else fz.dt[c * 32 + lane] = dist_rows(fz.xs + lane * XS, fz.ys + c * XS, D4);
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
    }
    if (FUSED) __syncwarp();

    if (active) {
        const long long sk = skew_index(N, M, p, rb, 0, lane);
        float2* vhp = q.VH + sk;
        const float* dp = FUSED ? nullptr : q.Dsk + sk;
        Slot* ring_out = ring + warp * kRing;
        const Slot* ring_in = ring + (warp - 1) * kRing;
        Slot* edge_out = q.edge_f + ((size_t)p * q.S + strip) * M;
        const Slot* edge_in = q.edge_f + ((size_t)p * q.S + strip - 1) * M;
        // Boundary row out of this warp (lane 31), tagged column + 1: into the
        // shared ring of the next warp or the global edge buffer of the next strip.
        const bool chan_lane = has_bot && lane == 31 && !(q.skip_publish && strip == 0 && bot_global);
        Slot* chan_out = bot_global ? edge_out : ring_out;
        const int chan_mask = bot_global ? 0x7fffffff : (kRing - 1);
        // Upper-boundary values of the first group (global channel: loaded one group ahead).
        Slot nxt[1];
        nxt[0].v = 0.f;
        nxt[0].tag = 0u;
        if (top_global && lane < kGroup && lane < M) nxt[0] = slot_load(edge_in + lane);

        float h_prev = 0.f, v_prev = 0.f;
        // Raw costs: a group's 16 skewed slot rows of this warp are one contiguous 2 KB
        // block; it is copied one group ahead into a per-warp double buffer in shared
        // memory with cp.async (no register scoreboard stays pending across the DP
        // steps), then read into registers at the start of its group.
        float* dsm = FUSED ? nullptr : reinterpret_cast<float*>(smem_raw + q.smem_fixed) + warp * 2 * kGroup * 32;
        const float* dwarp = FUSED ? nullptr : dp - lane;
        auto stage_costs = [&](int g) {  // group g -> buffer g & 1, 64 bytes per lane
            float* dst = dsm + (g & 1) * kGroup * 32 + lane * 16;
            const float* src = dwarp + (long long)g * kGroup * 32 + lane * 16;
#pragma unroll
            for (int c = 0; c < 4; ++c) cp_async16(dst + 4 * c, src + 4 * c);
            asm volatile("cp.async.commit_group;" ::: "memory");
        };
        if (!FUSED) stage_costs(0);
        int cons_seen = 0;  // last count read from the next warp's consumption counter
        const int nG = T / kGroup;
        for (int g = 0; g < nG; ++g) {
            const int s0 = g * kGroup;
            float dcur[kGroup];
            if (!FUSED) {  // the next group's copy goes out, then this group's costs are read
                if (g + 1 < nG) {
                    stage_costs(g + 1);
                    asm volatile("cp.async.wait_group 1;" ::: "memory");
                } else {
                    asm volatile("cp.async.wait_group 0;" ::: "memory");
                }
                __syncwarp();
                const float* cur = dsm + (g & 1) * kGroup * 32 + lane;
#pragma unroll
                for (int u = 0; u < kGroup; ++u) dcur[u] = cur[u * 32];
            }
            if (FUSED && (s0 & 31) == 0) {
                // New period s0/32: the y rows of tile s0/32 + 1 (costed during this
                // period) have arrived; the buffer of tile s0/32, whose costs are
                // complete, is restaged with tile s0/32 + 2. Each lane reads and
                // writes only its own row's cost slots, so the costs need no barrier.
                asm volatile("cp.async.wait_all;" ::: "memory");
                __syncwarp();
                const int cnext = s0 + 64;  // first column of tile s0/32 + 2
                if (cnext < M)
                    stage_y_tile(fz.ys + ((cnext >> 5) & 1) * 32 * XS, yb, cnext, M, q.D, D4, XS, lane);
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
                if (need > cons_seen) ok = wait_smem(&cons[warp], need, q, cons_seen);
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
                float draw;
                if (FUSED) {
                    draw = fz.dt[(j & 63) * 32 + lane];
                    // cost of column s+32 (past the last column it is computed from zero rows
                    // and never read): branch-free, so it interleaves with the DP chain
                    const int cn = s + 32;
                    const float* yrow = fz.ys + ((cn >> 5) & 1) * 32 * XS + (cn & 31) * XS;
                    if constexpr (DX > 0) fz.dt[(cn & 63) * 32 + lane] = dist_reg<DX>(xr, yrow);
                    else fz.dt[(cn & 63) * 32 + lane] = dist_rows(fz.xs + lane * XS, yrow, D4);
                } else {
                    draw = dcur[u];
                }
                const float d = draw * scale;
                // t = d + softmin(0, vl, hu) = d + lo - log2(1 + 2^(lo-mid) + 2^(lo-hi))
                float lo, mid, hi;
                sort3(0.f, vl, hu, lo, mid, hi);
                const float lz = lg2((1.f + ex2(lo - mid)) + ex2(lo - hi));
                const float tt = (d + lo) - lz;
                // first column / first row: a single predecessor (R borders are +inf)
                const bool col0 = (j == 0);
                // border values picked off the dependency chain: one select follows tt
                const bool border = col0 || row0_lane;
                const float hb = col0 ? -kBig : d, vb = row0_lane ? -kBig : d;
                const float h = border ? hb : tt - vl;
                const float v = border ? vb : tt - hu;
                const float svl = col0 ? kBig : (row0_lane ? -kBig : vl);
                const float shu = row0_lane ? kBig : (col0 ? -kBig : hu);
                c0 = col0 ? d : c0;
                vhp[(long long)s * 32] = make_float2(svl, shu);
                const bool valid = (unsigned)j < (unsigned)M;
                slot_store_if(chan_lane && valid, chan_out + (j & chan_mask), h, (unsigned)(j + 1));
                if (last_lane && (unsigned)j < (unsigned)Mb) rowbuf[j] = h;
                h_prev = h;
                v_prev = v;
            }

            if (has_top && !top_global && lane == 0) cons[warp - 1] = min(s0 + kGroup, M);
        }
    }

    // Loss: R[N,M] = sum_i d(i,0) + sum_{j>=1} h(N-1, j), scaled units.
    double part = (active && i < Nb) ? (double)c0 : 0.0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(kFull, part, o);
    if (lane == 0) s_red[warp] = part;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        double cs = 0.0;
        for (int w = 0; w < W; ++w) cs += s_red[w];
        q.colsum[(size_t)p * q.NB + strip] = cs;
        __threadfence();
        s_last = (atomicAdd(&q.done[p], 1) == q.S - 1);
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
            for (int w = 0; w < W; ++w) tot += s_red[w];
            for (int k = 0; k < q.S; ++k) tot += __ldcg(&q.colsum[(size_t)p * q.NB + k]);
            q.loss[p] = (float)(tot * (double)q.unscale);
        }
    }
}

// ---------------------------------------------------------------------------
// Backward (log space)
// ---------------------------------------------------------------------------
// EXT: the extended forward stored the three transition log2-probabilities of
// each cell (float4: diag, left, up), and the log-sum-exp of the messages uses
// the unbiased exp2_neg / log2f; otherwise the (vl, hu) pair from which they are
// recomputed, and the MUFU ex2 / lg2.
// MAXT: the block size the kernel is compiled for. Strips of at most 8 warps take
// the 256-thread build, whose register budget holds the prefetched state of a
// whole group without spilling.
template <bool EXT, int MAXT>
__global__ void __launch_bounds__(MAXT, 1) bwd_kernel(const WaveParams q)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int W = q.W;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    Slot* ring = reinterpret_cast<Slot*>(smem_raw);                       // [W][kRing][2], by producer warp
    volatile int* cons = reinterpret_cast<volatile int*>(ring + 2 * W * kRing);  // [W] slots consumed
    __shared__ int s_tk;

    if (threadIdx.x == 0) s_tk = atomicAdd(q.ticket_b, 1);
    if (threadIdx.x < W) cons[threadIdx.x] = 0;
    for (int k = threadIdx.x; k < 2 * W * kRing; k += blockDim.x) ring[k].tag = 0u;
    __syncthreads();

    const int tk = s_tk;
    const int p = tk % q.P, strip = q.strip0 + q.S - 1 - tk / q.P;
    const int N = q.N, M = q.M, T = skew_T(M);
    const int off = T - (M + 31);   // leading padding steps of the reverse walk
    const int rb = strip * W + warp, r0 = rb * 32, i = r0 + lane;
    const bool active = r0 < N;
    if (!active) return;
    const bool has_below = r0 + 32 < N;                // producer: the warp (or strip) below
    const bool below_global = has_below && warp == W - 1;
    const bool has_above = r0 > 0;                     // consumer: the warp (or strip) above
    const bool above_global = has_above && warp == 0;
    // this problem's own lengths (a padded batch): it aligns rows < Nb, columns < Mb
    const int Nb = q.lens_n ? min(max(q.lens_n[p], 1), N) : N;
    const int Mb = q.lens_m ? min(max(q.lens_m[p], 1), M) : M;
    const bool last_lane = (i == Nb - 1);
    const bool row_in = i < Nb;

    using VT = typename std::conditional<EXT, float4, float2>::type;
    const long long sk = band_index(q, p, rb, lane, T);
    const VT* vhp = reinterpret_cast<const VT*>(q.VH) + sk;
    float* ep = q.E + sk;
    Slot* ring_out = ring + 2 * warp * kRing;
    const Slot* ring_in = ring + 2 * (warp + 1) * kRing;
    const int S_all = strips_all(q);
    Slot* edge_out = q.edge_b + 2 * ((size_t)p * S_all + strip) * M;
    const Slot* edge_in = q.edge_b + 2 * ((size_t)p * S_all + strip + 1) * M;
    // Messages to the row above (lane 0), slot k = column M-1-k, a pair of
    // tagged slots (msg_up, msg_diag) with tag k + 1: into the shared ring of
    // the warp above or the global edge buffer of the strip above.
    const bool chan_lane = has_above && lane == 0;
    Slot* chan_out = above_global ? edge_out : ring_out;
    const int chan_mask = above_global ? 0x7fffffff : (kRing - 1);
    Slot nxt[2];
    nxt[0].v = nxt[1].v = -kBig;
    nxt[0].tag = nxt[1].tag = 0u;
    if (below_global && lane < kGroup) {
        const int k = lane - off;
        if (k >= 0 && k < M) { nxt[0] = slot_load(edge_in + 2 * k); nxt[1] = slot_load(edge_in + 2 * k + 1); }
    }

    float ml = -kBig, su = -kBig, sd = -kBig, rd_hold = -kBig;
    // E leaves in bursts of kEB steps' values kept in registers: per-step stores
    // interleaved with the chain slow every step (a warp issues in order; measured:
    // a whole group per burst is fastest, delaying each store by one step is not).
    // The wider builds have fewer registers to spare; the 384-thread double-float
    // one is fastest storing at once.
    constexpr int kEB = MAXT <= 256 ? kGroup : (EXT ? 1 : 8);
    // Per-step state of the next kGroup steps; slot u is refilled with the
    // following group's value as soon as step u has consumed it.
    VT buf[kGroup];
#pragma unroll
    for (int u = 0; u < kGroup; ++u) buf[u] = vhp[(long long)(T - 1 - u) * 32];
    int cons_seen = 0;  // last count read from the next warp's consumption counter
    const int nG = T / kGroup;
    for (int g = 0; g < nG; ++g) {
        const int t0 = g * kGroup;   // first reverse step of the group
        const int k0 = t0 - off;     // channel slot read by lane 31 at that step
        VT bcur[EXT ? 1 : kGroup];
        float eg[kEB];  // E of the steps not yet stored
        if (!EXT) {  // this group's state; the next group's loads go out now
#pragma unroll
            for (int u = 0; u < kGroup; ++u) bcur[u] = buf[u];
            if (g + 1 < nG) {
#pragma unroll
                for (int u = 0; u < kGroup; ++u) buf[u] = vhp[(long long)(T - 1 - (t0 + kGroup + u)) * 32];
            }
        }
        // Messages of the row below for lane 31: lane q holds slot k0 + q.
        float2 botv = make_float2(-kBig, -kBig);
        bool ok = true;
        if (has_below && k0 + kGroup > 0 && k0 < M) {
            const int k = k0 + lane;
            const unsigned want = (lane < kGroup && k >= 0 && k < M) ? (unsigned)(k + 1) : 0u;
            Slot cur[2];
            if (below_global) {
                cur[0] = nxt[0];
                cur[1] = nxt[1];
                ok = validate(cur, edge_in + 2 * k, want, q);
                const int nk = k + kGroup;
                if (ok && lane < kGroup && nk >= 0 && nk < M) {
                    nxt[0] = slot_load(edge_in + 2 * nk);
                    nxt[1] = slot_load(edge_in + 2 * nk + 1);
                }
            } else {
                const Slot* src = ring_in + 2 * (k & (kRing - 1));
                cur[0].tag = cur[1].tag = 0u;
                cur[0].v = cur[1].v = -kBig;
                if (want) { cur[0] = slot_load(src); cur[1] = slot_load(src + 1); }
                ok = validate(cur, src, want, q);
            }
            if (want) botv = make_float2(cur[0].v, cur[1].v);
        }
        if (ok && has_above && !above_global) {
            const int need = k0 + kGroup - 31 - kRing;
            if (need > cons_seen) ok = wait_smem(&cons[warp], need, q, cons_seen);
        }
        if (!ok) break;

#pragma unroll
        for (int u = 0; u < kGroup; ++u) {
            const int t = T - 1 - (t0 + u);
            const int j = t - lane;
            const float rs = __shfl_down_sync(kFull, su, 1);
            const float rds = __shfl_down_sync(kFull, sd, 1);
            const float bx = __shfl_sync(kFull, botv.x, u);
            const float by = __shfl_sync(kFull, botv.y, u);
            const float rd = (lane == 31) ? by : rds;  // msg_diag from (i+1, j), used next step
            const float a1 = (j < Mb - 1) ? ml : -kBig;                    // from (i, j+1)
            // from (i+1, j): msg_up of the row below (lane 31: from the next warp), none
            // past the last row; one select follows the shuffle
            const bool a2k = last_lane || lane == 31;
            const float a2 = a2k ? (last_lane ? -kBig : bx) : rs;
            const float a3 = (last_lane || j >= Mb - 1) ? -kBig : rd_hold; // from (i+1, j+1)
            rd_hold = rd;
            float lo, mid, hi;
            sort3(a1, a2, a3, lo, mid, hi);
            float lE = hi + dp_log2<EXT>((1.f + dp_exp2<EXT>(mid - hi)) + dp_exp2<EXT>(lo - hi));
            lE = (last_lane && j == Mb - 1) ? 0.f : lE;
            VT cur;
            if (EXT) {  // single buffer (register budget): refill slot u right after use
                cur = buf[u];
                buf[u] = vhp[(long long)(T - 1 - min(t0 + kGroup + u, T - 1)) * 32];
            } else {
                cur = bcur[u];
            }
            float wl, wu, wd;  // transition log2-probabilities of this cell to its left/up/diag predecessors
            if (EXT) {
                const float4 st = reinterpret_cast<const float4&>(cur);
                wd = st.x; wl = st.y; wu = st.z;
            } else {
                // log2 normaliser of this cell's own soft-min: the log-probabilities
                // to its diag/left/up predecessors are -Lz, -vl-Lz, -hu-Lz.
                const float2 st = reinterpret_cast<const float2&>(cur);
                float wlo, wmid, whi;
                sort3(0.f, st.x, st.y, wlo, wmid, whi);
                const float Lz = lg2((1.f + ex2(wlo - wmid)) + ex2(wlo - whi)) - wlo;
                wl = -st.x - Lz; wu = -st.y - Lz; wd = -Lz;
            }
            ml = lE + wl;
            su = lE + wu;
            sd = lE + wd;
            // cells outside this problem's own N_b x M_b block carry no alignment
            eg[u % kEB] = (row_in && (unsigned)j < (unsigned)Mb) ? ex2(lE) : 0.f;
            if (u % kEB == kEB - 1) {
#pragma unroll
                for (int v = 0; v < kEB; ++v) ep[(long long)(t + kEB - 1 - v) * 32] = eg[v];
            }
            {
                const bool pub = chan_lane && (unsigned)j < (unsigned)M;
                const int k = M - 1 - j;
                Slot* dst = chan_out + 2 * (k & chan_mask);
                slot_store_if(pub, dst, su, (unsigned)(k + 1));
                slot_store_if(pub, dst + 1, sd, (unsigned)(k + 1));
            }
        }

        if (has_below && !below_global && lane == 31) cons[warp + 1] = min(max(k0 + kGroup, 0), M);
    }
}

// ---------------------------------------------------------------------------
// Host launchers
// ---------------------------------------------------------------------------
size_t wave_smem_fixed(int W, bool backward)
{
    const size_t ring = (size_t)W * kRing * sizeof(Slot) * (backward ? 2 : 1);
    const size_t ctr = (size_t)W * sizeof(int);
    return (ring + ctr + 15) & ~(size_t)15;
}

size_t wave_smem_fused_per_warp(int D)
{
    const int D4 = (D + 31) & ~31;
    const int XS = D4 + 4;
    return (size_t)(96 * XS + 64 * 32) * sizeof(float);
}

// Dynamic shared memory requested by every wavefront CTA, at least. The DP is
// latency-bound: CTAs must not share an SM, or the warps of the co-resident
// CTAs split the issue slots and every step slows down. Requesting more than
// half of an SM's shared memory keeps the block scheduler from packing them.
size_t wave_smem_floor()
{
    static size_t floor_bytes = 0;
    if (floor_bytes == 0) {
        int dev = 0, per_sm = 0;
        cudaGetDevice(&dev);
        if (cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
            per_sm <= 0)
            per_sm = 228 * 1024;
        floor_bytes = (size_t)per_sm / 2 + 1024;
    }
    return floor_bytes;
}

cudaError_t launch_forward(WaveParams q, bool fused, cudaStream_t st)
{
    const int grid = q.P * q.S;
    q.smem_fixed = (int)wave_smem_fixed(q.W, false);
    size_t smem = q.smem_fixed;
    if (fused) smem += (size_t)q.W * wave_smem_fused_per_warp(q.D);
    else smem += (size_t)q.W * 2 * kGroup * 32 * sizeof(float);  // staged raw costs
    smem = max(smem, wave_smem_floor());
    auto go = [&](auto kern) -> cudaError_t {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        kern<<<grid, q.W * 32, smem, st>>>(q);
        return cudaGetLastError();
    };
    if (fused) {
        const int dx = (q.D <= 32) ? 32 : (q.D <= 64 ? 64 : 0);
        return dx == 32 ? go(fwd_kernel<true, 32>) : dx == 64 ? go(fwd_kernel<true, 64>) : go(fwd_kernel<true, 0>);
    }
    return go(fwd_kernel<false, 0>);
}

cudaError_t launch_backward(WaveParams q, cudaStream_t st)
{
    const int grid = q.P * q.S;
    q.smem_fixed = (int)wave_smem_fixed(q.W, true);
    const size_t smem = max((size_t)q.smem_fixed, wave_smem_floor());
    auto go = [&](auto kern) -> cudaError_t {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        kern<<<grid, q.W * 32, smem, st>>>(q);
        return cudaGetLastError();
    };
    if (q.W <= 8) return q.ext ? go(bwd_kernel<true, 256>) : go(bwd_kernel<false, 256>);
    if (q.ext) return q.W <= kMaxWarpsBwdExt ? go(bwd_kernel<true, kMaxWarpsBwdExt * 32>) : cudaErrorInvalidValue;
    return go(bwd_kernel<false, kMaxWarps * 32>);
}

}  // namespace sdtw
