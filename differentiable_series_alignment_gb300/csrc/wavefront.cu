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
//    boundary row through a shared-memory ring with producer/consumer counters.
//  * Strips exchange their boundary row through global memory with
//    release/acquire ready counters. Strips are handed out by an atomic ticket
//    in dependency order, so a CTA only ever waits on a strip already owned by
//    a running CTA; this holds whatever the grid size and residency.
//  * Every wait is bounded (global timer); on expiry the kernel sets the
//    device status word and every other wait then gives up too.
//
// This replaces the per-anti-diagonal kernel launches of the pages' design
// (review page, "proposed method", first bullet) by one launch per direction.
#include "common.cuh"
#include "kernels.h"

namespace sdtw {

namespace {

constexpr unsigned kFull = 0xffffffffu;

// Bounded wait on a shared-memory counter. Warp-uniform result.
__device__ __forceinline__ bool wait_smem(const volatile int* cnt, int target, const WaveParams& q) {
    bool ok = true;
    if (*cnt < target) {
        const unsigned long long t0 = global_ns();
        unsigned it = 0;
        while (*cnt < target) {
            if ((++it & 31u) == 0) {
                if (ld_volatile_global(q.status) != 0) { ok = false; break; }
                if (global_ns() - t0 > q.wait_ns) { atomicOr(q.status, kStatusTimeout); ok = false; break; }
            }
        }
    }
    ok = __shfl_sync(kFull, ok, 0);
    __threadfence_block();
    return ok;
}

// Bounded wait on a global ready counter (acquire). Warp-uniform result.
__device__ __forceinline__ bool wait_global(const int* cnt, int target, const WaveParams& q) {
    bool ok = true;
    if (ld_acquire_gpu(cnt) < target) {
        const unsigned long long t0 = global_ns();
        while (ld_acquire_gpu(cnt) < target) {
            if (ld_volatile_global(q.status) != 0) { ok = false; break; }
            if (global_ns() - t0 > q.wait_ns) { atomicOr(q.status, kStatusTimeout); ok = false; break; }
        }
    }
    return __shfl_sync(kFull, ok, 0);
}

struct FusedSmem {
    float* xs;  // [32][XS]  rows of this warp, zero padded
    float* ys;  // [32][XS]  current 32 columns of y
    float* dt;  // [64][32]  two tiles of raw cost, slot (col & 63), lane
};

}  // namespace

// ---------------------------------------------------------------------------
// Forward
// ---------------------------------------------------------------------------
template <bool FUSED>
__global__ void __launch_bounds__(kMaxWarps * 32) fwd_kernel(const WaveParams q)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int W = q.W;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float* ring = reinterpret_cast<float*>(smem_raw);                    // [W][kRing]
    volatile int* prod = reinterpret_cast<volatile int*>(ring + W * kRing);
    volatile int* cons = prod + W;
    __shared__ int s_tk;
    __shared__ double s_red[kMaxWarps];

    if (threadIdx.x == 0) s_tk = atomicAdd(q.ticket_f, 1);
    if (threadIdx.x < W) { prod[threadIdx.x] = 0; cons[threadIdx.x] = 0; }
    __syncthreads();

    const int tk = s_tk;
    const int p = tk % q.P, strip = tk / q.P;
    const int N = q.N, M = q.M, T = M + 31;
    const int rb = strip * W + warp, r0 = rb * 32, i = r0 + lane;
    const bool active = r0 < N;
    const bool has_top = active && r0 > 0;
    const bool top_global = has_top && warp == 0;
    const bool has_bot = active && (r0 + 32 < N);
    const bool bot_global = has_bot && warp == W - 1;
    const float scale = q.scale;

    float c0 = 0.f;              // scaled d(i, 0)
    float rsum = 0.f, rcmp = 0.f;  // Kahan sum of h over the last row

    FusedSmem fz{};
    int XS = 0;
    const float* yb = q.pr.y(p);
    if (FUSED) {
        const int D = q.D, D4 = (D + 3) & ~3;
        XS = D4 + 4;
        float* base = reinterpret_cast<float*>(smem_raw + q.smem_fixed);
        float* mine = base + (size_t)warp * (64 * XS + 64 * 32);
        fz.xs = mine;
        fz.ys = mine + 32 * XS;
        fz.dt = mine + 64 * XS;
        const float* xb = q.pr.x(p);
        for (int e = lane; e < 32 * D4; e += 32) {
            const int r = e / D4, k = e - r * D4;
            fz.xs[r * XS + k] = (r0 + r < N && k < D) ? xb[(size_t)(r0 + r) * D + k] : 0.f;
        }
        __syncwarp();
    }

    if (active) {
        const long long sk = skew_index(N, M, p, rb, 0, lane);
        float2* vhp = q.VH + sk;
        const float* dp = FUSED ? nullptr : q.Dsk + sk;
        float* ring_out = ring + warp * kRing;
        const float* ring_in = ring + (warp - 1) * kRing;
        float* edge_out = q.edge_f + ((size_t)p * q.NB + strip) * M;
        const float* edge_in = q.edge_f + ((size_t)p * q.NB + strip - 1) * M;
        int* prog_out = q.prog_f + (size_t)p * q.NB + strip;
        const int* prog_in = q.prog_f + (size_t)p * q.NB + strip - 1;
        const bool publish_ok = !(q.skip_publish && strip == 0);

        float h_prev = 0.f, v_prev = 0.f;
        float dn[kGroup];
        if (!FUSED) {
#pragma unroll
            for (int u = 0; u < kGroup; ++u) dn[u] = (u < T) ? dp[(long long)u * 32] : 0.f;
        }
        const int nG = (T + kGroup - 1) / kGroup;
        for (int g = 0; g < nG; ++g) {
            const int s0 = g * kGroup;
            float dc[kGroup];
            if (!FUSED) {
#pragma unroll
                for (int u = 0; u < kGroup; ++u) dc[u] = dn[u];
                if (g + 1 < nG) {
#pragma unroll
                    for (int u = 0; u < kGroup; ++u) {
                        const int t = s0 + kGroup + u;
                        dn[u] = (t < T) ? dp[(long long)t * 32] : 0.f;
                    }
                }
            } else if ((s0 & 31) == 0 && s0 < M) {
                // Raw cost of columns [s0, s0+32) for this warp's 32 rows.
                const int D = q.D, D4 = (D + 3) & ~3;
                __syncwarp();
                for (int e = lane; e < 32 * D4; e += 32) {
                    const int r = e / D4, k = e - r * D4;
                    const int col = s0 + r;
                    fz.ys[r * XS + k] = (col < M && k < D) ? yb[(size_t)col * D + k] : 0.f;
                }
                __syncwarp();
                float acc[32];
#pragma unroll
                for (int cc = 0; cc < 32; ++cc) acc[cc] = 0.f;
                for (int k4 = 0; k4 < D4; k4 += 4) {
                    const float4 xv = *reinterpret_cast<const float4*>(fz.xs + lane * XS + k4);
#pragma unroll
                    for (int cc = 0; cc < 32; ++cc) {
                        const float4 yv = *reinterpret_cast<const float4*>(fz.ys + cc * XS + k4);
                        float a = xv.x - yv.x;
                        acc[cc] = fmaf(a, a, acc[cc]);
                        a = xv.y - yv.y;
                        acc[cc] = fmaf(a, a, acc[cc]);
                        a = xv.z - yv.z;
                        acc[cc] = fmaf(a, a, acc[cc]);
                        a = xv.w - yv.w;
                        acc[cc] = fmaf(a, a, acc[cc]);
                    }
                }
#pragma unroll
                for (int cc = 0; cc < 32; ++cc) fz.dt[((s0 + cc) & 63) * 32 + lane] = acc[cc];
                __syncwarp();
            }

            // Upper-neighbour values for lane 0: columns [s0, s0+kGroup).
            float topv = 0.f;
            bool ok = true;
            if (has_top) {
                const int need = min(s0 + kGroup, M);
                if (s0 < M) {
                    if (top_global) {
                        ok = wait_global(prog_in, need, q);
                        if (ok && lane < kGroup && s0 + lane < M) topv = __ldcg(edge_in + s0 + lane);
                    } else {
                        ok = wait_smem(&prod[warp - 1], need, q);
                        if (ok && lane < kGroup) topv = ring_in[(s0 + lane) & (kRing - 1)];
                    }
                }
            }
            if (ok && has_bot && !bot_global) {
                const int need = s0 + kGroup - 31 - kRing;  // ring slots this group overwrites are free
                if (need > 0) ok = wait_smem(&cons[warp], need, q);
            }
            if (!ok) break;

#pragma unroll
            for (int u = 0; u < kGroup; ++u) {
                const int s = s0 + u;
                const int j = s - lane;
                float hu = __shfl_up_sync(kFull, h_prev, 1);
                const float tv = __shfl_sync(kFull, topv, u);
                if (lane == 0) hu = tv;
                const float vl = v_prev;
                const float d = FUSED ? fz.dt[(j & 63) * 32 + lane] * scale : dc[u] * scale;
                const float m = fminf(fminf(0.f, vl), hu);
                const float S = ex2(m) + ex2(m - vl) + ex2(m - hu);
                const float tt = d + m - lg2(S);
                float h = tt - vl, v = tt - hu;
                float svl = vl, shu = hu;
                if (i == 0) {
                    if (j == 0) { h = -kBig; v = -kBig; svl = kBig; shu = kBig; }
                    else { h = d; v = -kBig; svl = -kBig; shu = kBig; }
                } else if (j == 0) {
                    v = d; h = -kBig; svl = kBig; shu = -kBig;
                }
                if (j == 0) c0 = d;
                const bool valid = (i < N) && (j >= 0) && (j < M);
                if (s < T) vhp[(long long)s * 32] = make_float2(svl, shu);
                if (has_bot && lane == 31 && valid) {
                    if (bot_global) edge_out[j] = h;
                    else ring_out[j & (kRing - 1)] = h;
                }
                if (i == N - 1 && valid && j >= 1) {  // Kahan
                    const float yk = h - rcmp;
                    const float tk2 = rsum + yk;
                    rcmp = (tk2 - rsum) - yk;
                    rsum = tk2;
                }
                h_prev = h;
                v_prev = v;
            }

            if (has_bot && lane == 31) {
                int cnt = min(max(s0 + kGroup - 31, 0), M);
                if (g == nG - 1) cnt = M;
                if (bot_global) {
                    if (publish_ok) st_release_gpu(prog_out, cnt);
                } else {
                    __threadfence_block();
                    prod[warp] = cnt;
                }
            }
            if (has_top && !top_global && lane == 0) cons[warp - 1] = min(s0 + kGroup, M);
        }
    }

    // Loss assembly: R[N,M] = sum_i d(i,0) + sum_{j>=1} h(N-1, j), in scaled units.
    double part = (active && i < N) ? (double)c0 : 0.0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(kFull, part, o);
    if (lane == 0) s_red[warp] = part;
    if (active && i == N - 1) q.rowsum[p] = (double)rsum - (double)rcmp;
    __syncthreads();
    if (threadIdx.x == 0) {
        double cs = 0.0;
        for (int w = 0; w < W; ++w) cs += s_red[w];
        q.colsum[(size_t)p * q.NB + strip] = cs;
        __threadfence();
        const int prev = atomicAdd(&q.done[p], 1);
        if (prev == q.S - 1) {
            __threadfence();
            double tot = *reinterpret_cast<volatile double*>(&q.rowsum[p]);
            for (int k = 0; k < q.S; ++k) tot += *reinterpret_cast<volatile double*>(&q.colsum[(size_t)p * q.NB + k]);
            q.loss[p] = (float)(tot * (double)q.unscale);
        }
    }
}

// ---------------------------------------------------------------------------
// Backward (log space)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kMaxWarps * 32) bwd_kernel(const WaveParams q)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int W = q.W;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float2* ring = reinterpret_cast<float2*>(smem_raw);                   // [W][kRing], by producer
    volatile int* prod = reinterpret_cast<volatile int*>(ring + W * kRing);
    volatile int* cons = prod + W;
    __shared__ int s_tk;

    if (threadIdx.x == 0) s_tk = atomicAdd(q.ticket_b, 1);
    if (threadIdx.x < W) { prod[threadIdx.x] = 0; cons[threadIdx.x] = 0; }
    __syncthreads();

    const int tk = s_tk;
    const int p = tk % q.P, strip = q.S - 1 - tk / q.P;
    const int N = q.N, M = q.M, T = M + 31;
    const int rb = strip * W + warp, r0 = rb * 32, i = r0 + lane;
    const bool active = r0 < N;
    if (!active) return;
    const bool has_below = r0 + 32 < N;                // producer: the warp (or strip) below
    const bool below_global = has_below && warp == W - 1;
    const bool has_above = r0 > 0;                     // consumer: the warp (or strip) above
    const bool above_global = has_above && warp == 0;

    const long long sk = skew_index(N, M, p, rb, 0, lane);
    const float2* vhp = q.VH + sk;
    float* ep = q.E + sk;
    float2* ring_out = ring + warp * kRing;
    const float2* ring_in = ring + (warp + 1) * kRing;
    float2* edge_out = q.edge_b + ((size_t)p * q.NB + strip) * M;
    const float2* edge_in = q.edge_b + ((size_t)p * q.NB + strip + 1) * M;
    int* prog_out = q.prog_b + (size_t)p * q.NB + strip;
    const int* prog_in = q.prog_b + (size_t)p * q.NB + strip + 1;

    float ml = -kBig, su = -kBig, sd = -kBig, rd_hold = -kBig;
    float2 vn[kGroup];
#pragma unroll
    for (int u = 0; u < kGroup; ++u) vn[u] = (u < T) ? vhp[(long long)(T - 1 - u) * 32] : make_float2(0.f, 0.f);
    const int nG = (T + kGroup - 1) / kGroup;
    for (int g = 0; g < nG; ++g) {
        const int t0 = g * kGroup;  // first backward step of the group
        float2 vc[kGroup];
#pragma unroll
        for (int u = 0; u < kGroup; ++u) vc[u] = vn[u];
        if (g + 1 < nG) {
#pragma unroll
            for (int u = 0; u < kGroup; ++u) {
                const int tau = t0 + kGroup + u;
                vn[u] = (tau < T) ? vhp[(long long)(T - 1 - tau) * 32] : make_float2(0.f, 0.f);
            }
        }
        // Messages of the row below for lane 31: slots [t0, t0+kGroup), slot k = column M-1-k.
        float2 botv = make_float2(-kBig, -kBig);
        bool ok = true;
        if (has_below && t0 < M) {
            const int need = min(t0 + kGroup, M);
            if (below_global) {
                ok = wait_global(prog_in, need, q);
                if (ok && lane < kGroup && t0 + lane < M) {
                    const float2* src = edge_in + t0 + lane;
                    botv = __ldcg(src);
                }
            } else {
                ok = wait_smem(&prod[warp + 1], need, q);
                if (ok && lane < kGroup) botv = ring_in[(t0 + lane) & (kRing - 1)];
            }
        }
        if (ok && has_above && !above_global) {
            const int need = t0 + kGroup - 31 - kRing;
            if (need > 0) ok = wait_smem(&cons[warp], need, q);
        }
        if (!ok) break;

#pragma unroll
        for (int u = 0; u < kGroup; ++u) {
            const int tau = t0 + u;
            const int t = T - 1 - tau;
            const int j = t - lane;
            float ru = __shfl_down_sync(kFull, su, 1);
            float rd = __shfl_down_sync(kFull, sd, 1);
            const float bx = __shfl_sync(kFull, botv.x, u);
            const float by = __shfl_sync(kFull, botv.y, u);
            if (lane == 31) { ru = bx; rd = by; }
            const float a1 = (j < M - 1) ? ml : -kBig;
            const float a2 = (i < N - 1) ? ru : -kBig;
            const float a3 = (i < N - 1 && j < M - 1) ? rd_hold : -kBig;
            rd_hold = rd;
            const float mx = fmaxf(fmaxf(a1, a2), a3);
            float lE = mx + lg2(ex2(a1 - mx) + ex2(a2 - mx) + ex2(a3 - mx));
            if (i == N - 1 && j == M - 1) lE = 0.f;
            const float2 st = vc[u];
            const float m = fminf(fminf(0.f, st.x), st.y);
            const float Lz = lg2(ex2(m) + ex2(m - st.x) + ex2(m - st.y)) - m;
            ml = lE + (-st.x - Lz);
            su = lE + (-st.y - Lz);
            sd = lE - Lz;
            if (t >= 0) ep[(long long)t * 32] = ex2(lE);
            if (has_above && lane == 0 && j >= 0 && j < M) {
                const float2 msg = make_float2(su, sd);
                const int k = M - 1 - j;
                if (above_global) edge_out[k] = msg;
                else ring_out[k & (kRing - 1)] = msg;
            }
        }

        if (has_above && lane == 0) {
            int cnt = min(max(t0 + kGroup - 31, 0), M);
            if (g == nG - 1) cnt = M;
            if (above_global) {
                st_release_gpu(prog_out, cnt);
            } else {
                __threadfence_block();
                prod[warp] = cnt;
            }
        }
        if (has_below && !below_global && lane == 31) cons[warp + 1] = min(t0 + kGroup, M);
    }
}

// ---------------------------------------------------------------------------
// Host launchers
// ---------------------------------------------------------------------------
size_t wave_smem_fixed(int W, bool backward)
{
    const size_t ring = (size_t)W * kRing * (backward ? sizeof(float2) : sizeof(float));
    const size_t ctr = 2 * (size_t)W * sizeof(int);
    return (ring + ctr + 15) & ~(size_t)15;
}

size_t wave_smem_fused_per_warp(int D)
{
    const int D4 = (D + 3) & ~3;
    const int XS = D4 + 4;
    return (size_t)(64 * XS + 64 * 32) * sizeof(float);
}

cudaError_t launch_forward(WaveParams q, bool fused, cudaStream_t st)
{
    const int grid = q.P * q.S;
    q.smem_fixed = (int)wave_smem_fixed(q.W, false);
    size_t smem = q.smem_fixed;
    if (fused) smem += (size_t)q.W * wave_smem_fused_per_warp(q.D);
    cudaError_t e;
    if (fused) {
        e = cudaFuncSetAttribute(fwd_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        fwd_kernel<true><<<grid, q.W * 32, smem, st>>>(q);
    } else {
        e = cudaFuncSetAttribute(fwd_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        fwd_kernel<false><<<grid, q.W * 32, smem, st>>>(q);
    }
    return cudaGetLastError();
}

cudaError_t launch_backward(WaveParams q, cudaStream_t st)
{
    const int grid = q.P * q.S;
    const size_t smem = wave_smem_fixed(q.W, true);
    q.smem_fixed = (int)smem;
    cudaError_t e = cudaFuncSetAttribute(bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    bwd_kernel<<<grid, q.W * 32, smem, st>>>(q);
    return cudaGetLastError();
}

}  // namespace sdtw
