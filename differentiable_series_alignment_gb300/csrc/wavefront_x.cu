// wavefront_x.cu -- the extended-precision forward (SDTW_EXTENDED).
//
// Long sequences at small gamma make the gradient sensitive to cost
// perturbations below fp32 resolution: at N=M=8192, gamma=0.01, even an fp64
// DP fed the correctly rounded fp32 costs misses rel 1e-3 on some gradient
// elements. This forward therefore keeps
//   * the cost C[i,j] as a double-float (hi + lo), summed from exact
//     differences x - y (TwoSum) and exact squares (FMA product error),
//   * the difference-form DP state h, v as double-floats,
// and stores per cell the three transition log2-probabilities to the diag,
// left and up predecessors (fp32: each is computed from an exact double-float
// difference, rounded once), which the backward reads directly. The loss and
// the recursion follow wavefront.cu; only the arithmetic is wider.
#include "channel.cuh"
#include "common.cuh"
#include "kernels.h"

namespace sdtw {

namespace {

struct dd {
    float hi, lo;
};
__device__ __forceinline__ dd mk(float h, float l) { return dd{h, l}; }
__device__ __forceinline__ dd fast2(float a, float b) {
    const float s = a + b;
    return dd{s, b - (s - a)};
}
__device__ __forceinline__ dd add(dd a, dd b) {
    float s, e;
    two_sum(a.hi, b.hi, s, e);
    e += a.lo + b.lo;
    return fast2(s, e);
}
__device__ __forceinline__ dd sub(dd a, dd b) { return add(a, dd{-b.hi, -b.lo}); }
__device__ __forceinline__ dd sub_f(dd a, float f) {
    float s, e;
    two_sum(a.hi, -f, s, e);
    e += a.lo;
    return fast2(s, e);
}
__device__ __forceinline__ float to_f(dd a) { return a.hi + a.lo; }
__device__ __forceinline__ bool less(dd a, dd b) { return a.hi < b.hi || (a.hi == b.hi && a.lo < b.lo); }
__device__ __forceinline__ dd sel(bool c, dd a, dd b) { return dd{c ? a.hi : b.hi, c ? a.lo : b.lo}; }
__device__ __forceinline__ void sort3dd(dd a, dd b, dd c, dd& lo, dd& mid, dd& hi) {
    const bool ab = less(a, b);
    const dd t1 = sel(ab, a, b), t2 = sel(ab, b, a);
    lo = sel(less(c, t1), c, t1);
    const bool c2 = less(t2, c);
    hi = sel(c2, c, t2);
    const dd m2 = sel(c2, t2, c);
    mid = sel(less(t1, m2), m2, t1);
}

// Double-float squared distance accumulator: exact differences and squares.
struct DistDD {
    float s = 0.f, c = 0.f;
    __device__ __forceinline__ void add_term(float x, float y) {
        float a, ae;
        two_sum(x, -y, a, ae);            // a + ae == x - y
        const float p = a * a;
        float pe = fmaf(a, a, -p);        // p + pe == a*a
        pe = fmaf(2.f * a, ae, pe);       // + 2 a ae  (ae^2 below resolution)
        float t, e;
        two_sum(s, p, t, e);
        s = t;
        c += e + pe;
    }
    __device__ __forceinline__ dd value() const { return fast2(s, c); }
};

// dd cost times the fp32 scale log2(e)/gamma.
__device__ __forceinline__ dd scale_dd(dd d, float k) {
    const float p = d.hi * k;
    const float pe = fmaf(d.hi, k, -p);
    return fast2(p, fmaf(d.lo, k, pe));
}

}  // namespace

// ---------------------------------------------------------------------------
// Cost tensor for the unfused extended forward: (hi, lo) per slot, raw (unscaled).
// grid: (ceil(T/64), NB, P), block 256
__global__ void __launch_bounds__(256) distx_kernel(Problems pr, int N, int M, int D, float2* __restrict__ Dsk)
{
    extern __shared__ float sm[];
    const int XS = D + 1;
    float* xs = sm;               // [32][XS]
    float* ys = sm + 32 * XS;     // [95][XS]
    const int p = blockIdx.z, rb = blockIdx.y, t0 = blockIdx.x * 64;
    const int T = M + 31;
    const int r0 = rb * 32, jbase = t0 - 31;
    const float* xb = pr.x(p);
    const float* yb = pr.y(p);
    for (int e = threadIdx.x; e < 32 * D; e += blockDim.x) {
        const int r = e / D, k = e - r * D;
        xs[r * XS + k] = (r0 + r < N) ? xb[(size_t)(r0 + r) * D + k] : 0.f;
    }
    for (int e = threadIdx.x; e < 95 * D; e += blockDim.x) {
        const int r = e / D, k = e - r * D;
        const int j = jbase + r;
        ys[r * XS + k] = (j >= 0 && j < M) ? yb[(size_t)j * D + k] : 0.f;
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tw = t0 + warp * 8;
    const int yrow0 = tw - lane - jbase;
    DistDD acc[8];
    for (int k = 0; k < D; ++k) {
        const float xv = xs[lane * XS + k];
#pragma unroll
        for (int u = 0; u < 8; ++u) acc[u].add_term(xv, ys[(yrow0 + u) * XS + k]);
    }
    float2* out = Dsk + skew_index(N, M, p, rb, 0, lane);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const int t = tw + u;
        const dd v = acc[u].value();
        if (t < T) out[(long long)t * 32] = make_float2(v.hi, v.lo);
    }
}

// ---------------------------------------------------------------------------
// Extended forward. Same decomposition and channels as fwd_kernel, with the
// boundary h carried as a (hi, lo) pair of tagged slots.
template <bool FUSED>
__global__ void __launch_bounds__(kMaxWarps * 32, 1) fwdx_kernel(const WaveParams q)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int W = q.W;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    Slot* ring = reinterpret_cast<Slot*>(smem_raw);                           // [W][kRing][2]
    volatile int* cons = reinterpret_cast<volatile int*>(ring + 2 * W * kRing);  // [W]
    __shared__ int s_tk;
    __shared__ double s_red[kMaxWarps];
    __shared__ int s_last;

    if (threadIdx.x == 0) s_tk = atomicAdd(q.ticket_f, 1);
    if (threadIdx.x < W) cons[threadIdx.x] = 0;
    for (int k = threadIdx.x; k < 2 * W * kRing; k += blockDim.x) ring[k].tag = 0u;
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
    const bool row0_lane = (i == 0);
    // this problem's own lengths (a padded batch): it aligns rows < Nb, columns < Mb
    const int Nb = q.lens_n ? min(max(q.lens_n[p], 1), N) : N;
    const int Mb = q.lens_m ? min(max(q.lens_m[p], 1), M) : M;
    const bool last_lane = (i == Nb - 1);
    const float scale = q.scale;
    float2* rowbuf = reinterpret_cast<float2*>(q.rowbuf) + (size_t)p * M;
    const dd zero = mk(0.f, 0.f), nbig = mk(-kBig, 0.f);

    dd c0 = zero;  // scaled d(i, 0)

    // fused: per warp x rows [32][XS], y rows [32][XS], costs [64][32] (hi) + [64][32] (lo)
    int XS = 0;
    float *fxs = nullptr, *fys = nullptr, *fdh = nullptr, *fdl = nullptr;
    const float* yb = q.pr.y(p);
    if (FUSED) {
        const int D = q.D;
        XS = D + 1;
        float* base = reinterpret_cast<float*>(smem_raw + q.smem_fixed);
        float* mine = base + (size_t)warp * (64 * XS + 2 * 64 * 32);
        fxs = mine;
        fys = mine + 32 * XS;
        fdh = mine + 64 * XS;
        fdl = fdh + 64 * 32;
        const float* xb = q.pr.x(p);
        for (int e = lane; e < 32 * D; e += 32) {
            const int r = e / D, k = e - r * D;
            fxs[r * XS + k] = (r0 + r < N) ? xb[(size_t)(r0 + r) * D + k] : 0.f;
        }
        __syncwarp();
    }

    if (active) {
        const long long sk = skew_index(N, M, p, rb, 0, lane);
        float4* lpp = reinterpret_cast<float4*>(q.VH) + sk;
        const float2* dp = FUSED ? nullptr : reinterpret_cast<const float2*>(q.Dsk) + sk;
        Slot* ring_out = ring + 2 * warp * kRing;
        const Slot* ring_in = ring + 2 * (warp - 1) * kRing;
        Slot* edge_out = q.edge_f + 2 * ((size_t)p * q.S + strip) * M;
        const Slot* edge_in = q.edge_f + 2 * ((size_t)p * q.S + strip - 1) * M;
        const bool chan_lane = has_bot && lane == 31 && !(q.skip_publish && strip == 0 && bot_global);
        Slot* chan_out = bot_global ? edge_out : ring_out;
        const int chan_mask = bot_global ? 0x7fffffff : (kRing - 1);
        Slot nxt[2];
        nxt[0].v = nxt[1].v = 0.f;
        nxt[0].tag = nxt[1].tag = 0u;
        if (top_global && lane < kGroup && lane < M) {
            nxt[0] = slot_load(edge_in + 2 * lane);
            nxt[1] = slot_load(edge_in + 2 * lane + 1);
        }

        dd h_prev = zero, v_prev = zero;
        int cons_seen = 0;  // last count read from the next warp's consumption counter
        const int nG = T / kGroup;
        for (int g = 0; g < nG; ++g) {
            const int s0 = g * kGroup;
            if (FUSED && (s0 & 31) == 0 && s0 < M) {
                // double-float costs of columns [s0, s0+32) for this warp's rows
                const int D = q.D;
                __syncwarp();
                for (int e = lane; e < 32 * D; e += 32) {
                    const int r = e / D, k = e - r * D;
                    const int col = s0 + r;
                    fys[r * XS + k] = (col < M) ? yb[(size_t)col * D + k] : 0.f;
                }
                __syncwarp();
                for (int half = 0; half < 32; half += 8) {
                    DistDD acc[8];
                    for (int k = 0; k < D; ++k) {
                        const float xv = fxs[lane * XS + k];
#pragma unroll
                        for (int cc = 0; cc < 8; ++cc) acc[cc].add_term(xv, fys[(half + cc) * XS + k]);
                    }
#pragma unroll
                    for (int cc = 0; cc < 8; ++cc) {
                        const dd v = acc[cc].value();
                        const int slot = ((s0 + half + cc) & 63) * 32 + lane;
                        fdh[slot] = v.hi;
                        fdl[slot] = v.lo;
                    }
                }
                __syncwarp();
            }

            // Upper-neighbour h for lane 0: lane q holds column s0 + q as a (hi, lo) slot pair.
            dd topv = zero;
            bool ok = true;
            if (has_top && s0 < M) {
                const int col = s0 + lane;
                const unsigned want = (lane < kGroup && col < M) ? (unsigned)(col + 1) : 0u;
                Slot cur[2];
                if (top_global) {
                    cur[0] = nxt[0];
                    cur[1] = nxt[1];
                    ok = validate(cur, edge_in + 2 * col, want, q);
                    const int ncol = col + kGroup;
                    if (ok && lane < kGroup && ncol < M) {
                        nxt[0] = slot_load(edge_in + 2 * ncol);
                        nxt[1] = slot_load(edge_in + 2 * ncol + 1);
                    }
                } else {
                    const Slot* src = ring_in + 2 * (col & (kRing - 1));
                    cur[0].v = cur[1].v = 0.f;
                    cur[0].tag = cur[1].tag = 0u;
                    if (want) { cur[0] = slot_load(src); cur[1] = slot_load(src + 1); }
                    ok = validate(cur, src, want, q);
                }
                topv = mk(cur[0].v, cur[1].v);
            }
            if (ok && has_bot && !bot_global) {
                const int need = s0 + kGroup - 31 - kRing;
                if (need > cons_seen) ok = wait_smem(&cons[warp], need, q, cons_seen);
            }
            if (!ok) break;

            float2 dc[kGroup];
            if (!FUSED) {
#pragma unroll
                for (int u = 0; u < kGroup; ++u) dc[u] = dp[(long long)(s0 + u) * 32];
            }
#pragma unroll
            for (int u = 0; u < kGroup; ++u) {
                const int s = s0 + u;
                const int j = s - lane;
                const float hs_hi = __shfl_up_sync(kFull, h_prev.hi, 1);
                const float hs_lo = __shfl_up_sync(kFull, h_prev.lo, 1);
                const float tv_hi = __shfl_sync(kFull, topv.hi, u);
                const float tv_lo = __shfl_sync(kFull, topv.lo, u);
                const dd hu = (lane == 0) ? mk(tv_hi, tv_lo) : mk(hs_hi, hs_lo);
                const dd vl = v_prev;
                dd d;
                if (FUSED) {
                    const int slot = (j & 63) * 32 + lane;
                    d = scale_dd(mk(fdh[slot], fdl[slot]), scale);
                } else {
                    d = scale_dd(mk(dc[u].x, dc[u].y), scale);
                }
                dd lo, mid, hi;
                sort3dd(zero, vl, hu, lo, mid, hi);
                const float e1 = to_f(sub(lo, mid)), e2 = to_f(sub(lo, hi));
                const float L = log2f((1.f + exp2_neg(e1)) + exp2_neg(e2));
                const dd tt = sub_f(add(d, lo), L);
                dd h = sub(tt, vl), v = sub(tt, hu);
                float lpd = to_f(lo) - L;
                float lpl = to_f(sub(lo, vl)) - L;
                float lpu = to_f(sub(lo, hu)) - L;
                const bool col0 = (j == 0);
                if (col0) {        // first column: only the upper predecessor (or none at (0,0))
                    h = nbig;
                    v = row0_lane ? nbig : d;
                    lpd = -kBig; lpl = -kBig; lpu = row0_lane ? -kBig : 0.f;
                } else if (row0_lane) {  // first row: only the left predecessor
                    h = d;
                    v = nbig;
                    lpd = -kBig; lpl = 0.f; lpu = -kBig;
                }
                c0 = col0 ? d : c0;
                lpp[(long long)s * 32] = make_float4(lpd, lpl, lpu, 0.f);
                const bool valid = (unsigned)j < (unsigned)M;
                if (chan_lane && valid) {
                    Slot* dst = chan_out + 2 * (j & chan_mask);
                    slot_store(dst, h.hi, (unsigned)(j + 1));
                    slot_store(dst + 1, h.lo, (unsigned)(j + 1));
                }
                if (last_lane && (unsigned)j < (unsigned)Mb) rowbuf[j] = make_float2(h.hi, h.lo);
                h_prev = h;
                v_prev = v;
            }
            if (has_top && !top_global && lane == 0) cons[warp - 1] = min(s0 + kGroup, M);
        }
    }

    // Loss: R[N,M] = sum_i d(i,0) + sum_{j>=1} h(N-1, j), scaled units, in fp64.
    double part = (active && i < Nb) ? (double)c0.hi + (double)c0.lo : 0.0;
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
    if (s_last) {
        __threadfence();
        double acc = 0.0;
        for (int j = 1 + (int)threadIdx.x; j < Mb; j += blockDim.x) {
            const float2 hv = __ldcg(rowbuf + j);
            acc += (double)hv.x + (double)hv.y;
        }
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

size_t wavex_smem_fused_per_warp(int D)
{
    return (size_t)(64 * (D + 1) + 2 * 64 * 32) * sizeof(float);
}

cudaError_t launch_forward_x(WaveParams q, bool fused, cudaStream_t st)
{
    const int grid = q.P * q.S;
    q.smem_fixed = (int)(((size_t)q.W * kRing * 2 * sizeof(Slot) + (size_t)q.W * sizeof(int) + 15) & ~(size_t)15);
    size_t smem = q.smem_fixed;
    if (fused) smem += (size_t)q.W * wavex_smem_fused_per_warp(q.D);
    smem = max(smem, wave_smem_floor());
    auto go = [&](auto kern) -> cudaError_t {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        kern<<<grid, q.W * 32, smem, st>>>(q);
        return cudaGetLastError();
    };
    return fused ? go(fwdx_kernel<true>) : go(fwdx_kernel<false>);
}

cudaError_t launch_dist_skewed_x(const Problems& pr, int P, int N, int M, int D, float2* Dsk, cudaStream_t st)
{
    const int T = M + 31;
    dim3 grid((T + 63) / 64, (N + 31) / 32, P);
    const size_t smem = (size_t)(32 + 95) * (D + 1) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(distx_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    distx_kernel<<<grid, 256, smem, st>>>(pr, N, M, D, Dsk);
    return cudaGetLastError();
}

}  // namespace sdtw
