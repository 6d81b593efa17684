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
#include "tc.cuh"

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

// The double-float forwards run a 16-step group as short chunks in a rolled loop:
// the unrolled double-float step is long, and a fully unrolled group misses the
// instruction cache. Measured on the fused forward (nine warps of three roles) at
// 16 / 8 / 4 / 2 steps per chunk: 1.20 / 0.62 / 0.42 / 0.40 ms at the 32 x 512^2
// headline shape, 52 / 21 / 14.6 / 10.6 ms at 8 x 8192^2. The unfused forward takes
// its chunk's costs by selects among the group's registers, which grow with the
// chunk count: 4 steps there (8192^2: 14.5 ms at 4, 15.4 at 2).
constexpr int kXChunkFused = 2;
constexpr int kXChunk = 4;

// One cell of the double-float recursion: d the scaled cost, vl = v[i,j-1] and
// hu = h[i-1,j] the incoming differences (relative to the diagonal predecessor).
// Gives h, v and the three transition log2-probabilities to the diag, left and up
// predecessors (float4 x, y, z); the first column and the first row have a single
// predecessor (R borders are +inf).
//
// The soft-min is factored around the predecessor with the smallest leading part:
//   t = d + lo - log2(2^-d0 + 2^-dl + 2^-du),  dk = a_k - lo >= 0,
// exact for any choice of lo among the three, so comparing the hi parts suffices.
// The offsets dk only feed the fp32 log and the fp32 log-probabilities: formed as
// (a.hi - lo.hi) + (a.lo - lo.lo), the first difference is exact whenever it is
// small (Sterbenz), and a large one leaves a negligible term. The results are
// formed as h = (d + lo - v_left) - L and v = (d + lo - h_up) - L: the bracketed
// double-float sums do not depend on the log, so they run beside the exp2/log2
// chain and only one double-float step follows it. The borders are selects.
__device__ __forceinline__ void xcell(dd d, dd vl, dd hu, bool col0, bool row0_lane, dd& h, dd& v, float4& lp)
{
    const dd nbig = mk(-kBig, 0.f);
    const dd m = (hu.hi < vl.hi) ? hu : vl;
    const dd lo = (m.hi < 0.f) ? m : mk(0.f, 0.f);
    const float d0 = (0.f - lo.hi) - lo.lo;
    const float dl = (vl.hi - lo.hi) + (vl.lo - lo.lo);
    const float du = (hu.hi - lo.hi) + (hu.lo - lo.lo);
    const dd dlo = add(d, lo);
    const dd ph = sub(dlo, vl), pv = sub(dlo, hu);
    const float L = log2f((exp2_neg(-d0) + exp2_neg(-dl)) + exp2_neg(-du));
    const dd hh = sub_f(ph, L), vv = sub_f(pv, L);
    // first column: only the upper predecessor (none at (0,0)); first row: only the left
    h = col0 ? nbig : (row0_lane ? d : hh);
    v = row0_lane ? nbig : (col0 ? d : vv);
    lp.x = (col0 || row0_lane) ? -kBig : -d0 - L;
    lp.y = col0 ? -kBig : (row0_lane ? 0.f : -dl - L);
    lp.z = row0_lane ? -kBig : (col0 ? 0.f : -du - L);
    lp.w = 0.f;
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
    stage_rows(xs, XS, xb, D, r0, 32, D, N, threadIdx.x, blockDim.x);
    stage_rows(ys, XS, yb, D, jbase, 95, D, M, threadIdx.x, blockDim.x);
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

            // the group's 16 costs into registers before any of its stores (the compiler
            // keeps loads behind stores it cannot prove apart)
            float2 dc[kGroup];
#pragma unroll
            for (int u = 0; u < kGroup; ++u) {
                if (FUSED) {
                    const int slot = ((s0 + u - lane) & 63) * 32 + lane;
                    dc[u] = make_float2(fdh[slot], fdl[slot]);
                } else {
                    dc[u] = dp[(long long)(s0 + u) * 32];
                }
            }
            // rolled chunks of kXChunk steps; a chunk takes its costs from dc by selects
            // between fixed indices, so dc stays in registers
#pragma unroll 1
            for (int h8 = 0; h8 < kGroup; h8 += kXChunk) {
#pragma unroll
                for (int uu = 0; uu < kXChunk; ++uu) {
                    const int u = h8 + uu;
                    const int s = s0 + u;
                    const int j = s - lane;
                    const float hs_hi = __shfl_up_sync(kFull, h_prev.hi, 1);
                    const float hs_lo = __shfl_up_sync(kFull, h_prev.lo, 1);
                    const float tv_hi = __shfl_sync(kFull, topv.hi, u);
                    const float tv_lo = __shfl_sync(kFull, topv.lo, u);
                    const dd hu = (lane == 0) ? mk(tv_hi, tv_lo) : mk(hs_hi, hs_lo);
                    const dd vl = v_prev;
                    float2 cu = dc[uu];
#pragma unroll
                    for (int q = 1; q < kGroup / kXChunk; ++q) cu = (h8 == q * kXChunk) ? dc[uu + q * kXChunk] : cu;
                    const dd d = scale_dd(mk(cu.x, cu.y), scale);
                    const bool col0 = (j == 0);
                    dd h, v;
                    float4 lp;
                    xcell(d, vl, hu, col0, row0_lane, h, v, lp);
                    c0 = col0 ? d : c0;
                    lpp[(long long)s * 32] = lp;
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

// ---------------------------------------------------------------------------
// Exact cost tiles on the tensor cores for the extended modes (D <= 400): the fused
// forward's tiles and the unfused cost tensor
//
// The double-float DP needs each cost to ~1e-9 of itself, beyond any fp32 split
// product (whose fp32 accumulation rounds). The dot x_i . y_j is therefore made
// exact in fixed point and evaluated on the tensor cores in integer arithmetic:
// every row v of x or y is scaled by its own power of two s = 2^e > max |v_k| and
// rounded to F = NS * b bits of fixed point, V_k = rint(v_k 2^(F-1) / s), so
// |v_k - s V_k 2^-(F-1)| <= s 2^-F, and V_k is written as NS balanced base-2^b
// digits,
//   V_k = sum_l a_l 2^(b (NS-1-l)),  |a_l| <= 2^(b-1),
// each an integer that bf16 holds exactly (oimg_kernel). Then
//   x . y = s_x s_y sum_sigma 2^(2 - 2b - b sigma) S_sigma,
//   S_sigma = sum_{l+m=sigma} sum_k a_l,k b_m,k,
// and the level sums S_sigma for sigma <= NS-1 are bf16 MMAs accumulated in fp32
// in tensor memory: every partial sum is an integer of magnitude below
// NS D 2^(2b-2) < 2^24, so fp32 holds it exactly (checked on the GB300 up to
// 2^23.98 against int64 sums) and the level sums are exact. Two digit sets:
// NS = 5 digits of b = 8 bits (F = 40) for D <= 128 (5 * 128 * 2^14 < 2^24), and
// NS = 6 digits of b = 7 bits (F = 42) up to D = 400 (6 * 400 * 2^12 < 2^24). The
// MMA of x digit l multiplies the stacked y digits [b_0 ; ... ; b_(NS-1-l)] into
// tensor-memory columns starting at level l, so product (l, m) lands in level
// l + m: NS MMAs (N = 32 NS, ..., 32 columns) per 16-wide K step. Error bound of
// x . y: the fixed-point rounding of both rows, D (|y|_max s_x + |x|_max s_y) 2^-F
// <= 2 D s_x s_y 2^-F, plus the dropped levels sigma >= NS, below
// (NS+2) D s_x s_y 2^-F: at D = 128, s <= 4 (unit-variance data) and F = 40, below
// 2e-8 absolute, ~1e-10 of a cost. The DP warps combine the level sums, the
// exponents and the double-float row norms into C = |x|^2 + |y|^2 - 2 x . y as a
// double-float.
namespace {

constexpr int kXDpWarps = 4;                   // 128 rows per CTA: the MMA tile height
constexpr int kXIssuer = kXDpWarps;            // warp 4: bulk copies and MMAs
constexpr uint32_t kXAPart = 128 * 128;        // one digit of one K-block of 128 x rows
constexpr uint32_t kXBPart = 32 * 128;         // one digit of one K-block of 32 y rows

// The digit sets: NS = 5 digits of DB = 8 bits (D <= 128) or NS = 6 digits of
// DB = 7 bits (D <= 400). SlotCols: the tensor-memory columns of one cost tile (its
// NS level sums for 32 y columns).
template <int NS> struct XDigits {
    static_assert(NS == 5 || NS == 6, "five 8-bit or six 7-bit digits");
    static constexpr int DB = NS == 5 ? 8 : 7;            // bits per digit
    static constexpr int SlotCols = NS * 32;
    static constexpr uint32_t A = NS * kXAPart;           // all digits of one K-block of the x rows
    static constexpr uint32_t B = NS * kXBPart;           // [b_0 ; ... ; b_(NS-1)] of one K-block of a y tile
};

// Shared memory of the operand region: one K-block keeps the x digits resident
// with a two-entry ring of y tiles; more K-blocks stream through one stage.
__host__ __device__ inline uint32_t xtc_region(int NS, int KB)
{
    const uint32_t a = NS * kXAPart, b = NS * kXBPart;
    return KB == 1 ? a + 2 * b : a + b;
}

// bf16 bit pattern of a small integer (|v| <= 256: exact)
__device__ __forceinline__ uint32_t bf16_int(int v)
{
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn((float)v));
}

// grid (Lpad/32, P, 2): z = 0 writes the x image, z = 1 the y image. block 256.
// Per row: its digits (five bf16 slices per K-block of 64 features, 128-byte
// swizzled K-major rows), and info = (|v|^2 hi, |v|^2 lo, exponent e as int bits, 0).
template <int NS>
__global__ void __launch_bounds__(256) oimg_kernel(Problems pr, int N, int M, int D, int KB,
                                                   unsigned char* __restrict__ ximg, unsigned char* __restrict__ yimg,
                                                   float4* __restrict__ xinfo, float4* __restrict__ yinfo)
{
    extern __shared__ float t[];  // [32][D64 + 1]
    __shared__ int s_exp[32];
    const bool isy = blockIdx.z == 1;
    const int p = blockIdx.y, r0 = blockIdx.x * 32;
    const int L = isy ? M : N;
    const int Lpad = simg_pad(L);
    if (r0 >= Lpad) return;
    const float* src = isy ? pr.y(p) : pr.x(p);
    unsigned char* img = isy ? yimg : ximg;
    float4* info = isy ? yinfo : xinfo;
    const int D64 = kTcKFeat * KB, ld = D64 + 1;
    const int n = 32 * D64 / 256;
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
        // row norm as a double-float (exact squares, TwoSum sums) and the row's scale
        // exponent: eight threads per row, then a TwoSum / max reduction across them
        const int r = threadIdx.x >> 3, part = threadIdx.x & 7;
        DistDD acc;
        float mx = 0.f;
        for (int k = part; k < D; k += 8) {
            const float x = t[r * ld + k];
            acc.add_term(x, 0.f);
            mx = fmaxf(mx, fabsf(x));
        }
        float s = acc.s, c = acc.c;
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
            const float so = __shfl_xor_sync(0xffffffffu, s, o), co = __shfl_xor_sync(0xffffffffu, c, o);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            float sn, err;
            two_sum(s, so, sn, err);
            s = sn;
            c += co + err;
        }
        int e = 0;
        if (mx > 0.f) frexpf(mx, &e);   // mx < 2^e
        if (part == 0) {
            const dd nrm = fast2(s, c);
            info[(size_t)p * Lpad + r0 + r] = make_float4(nrm.hi, nrm.lo, __int_as_float(e), 0.f);
            s_exp[r] = e;
        }
    }
    __syncthreads();
    // digits: one 16-byte chunk (8 features) of all NS slices per thread and pass
    constexpr int DB = XDigits<NS>::DB, F = NS * DB, HALF = 1 << (DB - 1), MASK = (1 << DB) - 1;
    const size_t slice_bytes = (size_t)Lpad * 128;
    for (int idx = threadIdx.x; idx < 32 * D64 / 8; idx += blockDim.x) {
        const int c8 = idx & 7, r = (idx >> 3) & 31, kb = idx >> 8;
        const float* src8 = t + r * ld + kb * kTcKFeat + 8 * c8;
        const double sc = ldexp(1.0, F - 1 - s_exp[r]);   // exact power of two
        uint32_t w[NS][4];
#pragma unroll
        for (int q = 0; q < 8; q += 2) {
            uint32_t lo[NS], hi[NS];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                long long X = __double2ll_rn((double)src8[q + h] * sc);   // |X| <= 2^(F-1)
                uint32_t* dst = h ? hi : lo;
#pragma unroll
                for (int l = NS - 1; l > 0; --l) {
                    const int d = (int)((X + HALF) & MASK) - HALF;        // balanced digit
                    dst[l] = bf16_int(d);
                    X = (X - d) >> DB;
                }
                dst[0] = bf16_int((int)X);                                 // |a_0| <= 2^(DB-1)
            }
#pragma unroll
            for (int l = 0; l < NS; ++l) w[l][q / 2] = lo[l] | (hi[l] << 16);
        }
        unsigned char* row = img + oimg_offset(p, KB, kb, NS, 0, Lpad, r0 + r) + 16 * (c8 ^ (r & 7));
#pragma unroll
        for (int l = 0; l < NS; ++l)
            *reinterpret_cast<uint4*>(row + l * slice_bytes) = make_uint4(w[l][0], w[l][1], w[l][2], w[l][3]);
    }
}

// x . y from its exact level sums S[0..NS-1]: sum_sigma 2^(-DB sigma) S_sigma as a
// double-float (each scaled term is exact in fp32), smallest first, times 2^k.
// 2^k for k in the normal range [-126, 127], exactly.
__device__ __forceinline__ float pow2i(int k) { return __int_as_float((k + 127) << 23); }

// The scale 2^k (k = e_x + e_y + 2 - 2 DB, the row exponents of two finite rows)
// as two in-range powers of two: exact, branch-free, for k in [-252, 254]; below,
// the dot is under 2^-220 and flushes to 0 like any fp32 value that small.
template <int NS>
__device__ __forceinline__ dd levels_dd(const float (&S)[NS], int k)
{
    constexpr int DB = XDigits<NS>::DB;
    dd a = mk(S[NS - 1] * pow2i(-DB * (NS - 1)), 0.f);
#pragma unroll
    for (int l = NS - 2; l >= 0; --l) a = add(a, mk(S[l] * pow2i(-DB * l), 0.f));
    k = min(max(k, -252), 254);
    const int k1 = k / 2;
    const float f1 = pow2i(k1), f2 = pow2i(k - k1);
    return mk(a.hi * f1 * f2, a.lo * f1 * f2);
}

// Extended fused forward with the exact tensor-core cost tiles. Same recursion,
// channels and loss as fwdx_kernel<true>. A CTA owns 128 rows (four DP warps, the
// MMA height) of one problem as a strip of the wavefront. Warp 4 (lane 0) copies
// the digits (the x digits once for one K-block, else x and y streamed per K-block
// through one stage) and issues the level MMAs of each 32-column tile into a ring
// of three tensor-memory tiles. Warps 5-8 are converters, one per TMEM lane
// quarter: as soon as a tile is in TMEM and the shared cost ring of the DP warp
// with the same rows has room, converter q combines its 32 rows' level sums into
// double-float costs in that ring (hi and lo planes) and releases the tile.
//
// Why converters. A DP warp starts its 16-step group at s0 only after the warp
// above has finished step s0 + 46, so warp 3 trails warp 0 by ~94 steps. Were the
// DP warps to read the tiles themselves, tile c - 3 would be released only when
// warp 3 reached it, at warp 0's step 32 c - 2: warp 0 would wait on warp 3 at
// every tile, with no slack (three tiles of five levels fill the tensor memory).
// With converters a tile waits on DP progress only for ring room. The rings hold
// 3, 3, 3, 4 tiles (warps 0-3): a converter can fill tile c + 1 while its DP warp
// runs period c (which reads tiles c - 1 and c). With three tensor-memory tiles (five
// digits) the tile warp 0 needs at step 32 c waits on warps 1-3 having finished
// periods c - 5, c - 5 and c - 6 (warp 0 near step 32 c - 66 at the latest); with two
// (six digits, 192 columns each) on periods c - 4, c - 4 and c - 5 (near step
// 32 c - 34). The conversion also leaves the DP warps' critical path. Six digits
// stage the x digits of a K-block in two fills of three (72 KB with the y digits).
//
// Hand-offs (every wait bounded):
//   s_a                      x digits resident
//   s_sfull / s_sempty       stage copies landed / the MMAs reading it are done
//   s_tfull[t] / s_tfree[t]  levels of tile t in TMEM / the 4 converters read them
//   s_conv[q]                tiles converted into ring q (converter q -> DP warp q)
//   s_used[q]                tiles DP warp q no longer needs (DP warp q -> converter q)
constexpr int kXConvWarps = 4;
constexpr int kXFusedThreads = (kXDpWarps + 1 + kXConvWarps) * 32;
constexpr int kXTileFloats = 32 * 32;                       // one plane of a 32-column ring tile
__host__ __device__ constexpr int xring_tiles(int w) { return w < 3 ? 3 : 4; }
__host__ __device__ constexpr int xring_first(int w) { return 3 * w; }
constexpr int kXRingTiles = 13;                             // xring_first(3) + xring_tiles(3)
constexpr size_t kXRingBytes = (size_t)kXRingTiles * 2 * kXTileFloats * sizeof(float);

template <int NS>
__global__ void __launch_bounds__(kXFusedThreads, 1)
    fwdx_tc_kernel(const WaveParams q, const unsigned char* __restrict__ ximg, const unsigned char* __restrict__ yimg,
                   const float4* __restrict__ xinfo, const float4* __restrict__ yinfo)
{
    using X = XDigits<NS>;
    // five digits: three tiles of 160 TMEM columns, all x digits of a K-block in one
    // fill; six digits: two tiles of 192 columns, x digits in two fills of three
    constexpr int kXRT = NS == 5 ? 3 : 2, kXSlotCols = X::SlotCols, kXSlices = NS;
    constexpr int kAH = NS == 5 ? 5 : 3, kH = NS / kAH;       // x digits per fill, fills per K-block
    constexpr uint32_t kXA = X::A, kXAH = kAH * kXAPart, kXB = X::B;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    constexpr int W = kXDpWarps;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    Slot* ring = reinterpret_cast<Slot*>(smem_raw);                              // [W][kRing][2]
    volatile int* cons = reinterpret_cast<volatile int*>(ring + 2 * W * kRing);  // [W]
    __shared__ int s_tk;
    __shared__ double s_red[kMaxWarps];
    __shared__ int s_last;
    __shared__ uint64_t s_a, s_sfull, s_sempty, s_fin, s_tfull[kXRT], s_tfree[kXRT];
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_conv[kXDpWarps], s_used[kXDpWarps];

    if (threadIdx.x == 0) s_tk = atomicAdd(q.ticket_f, 1);
    if (threadIdx.x < W) {
        cons[threadIdx.x] = 0;
        s_conv[threadIdx.x] = 0;
        s_used[threadIdx.x] = 0;
    }
    for (int k = threadIdx.x; k < 2 * W * kRing; k += blockDim.x) ring[k].tag = 0u;
    __syncthreads();

    const int tk = s_tk;
    const int p = tk % q.P, strip = tk / q.P;
    const int N = q.N, M = q.M, T = skew_T(M);
    const int KB = (q.D + kTcKFeat - 1) / kTcKFeat;
    const bool resident = KB == 1 && kH == 1;   // one K-block (five digits): the x digits stay in shared memory
    const int Npad = simg_pad(N), Mpad = simg_pad(M);
    const int rs0 = strip * W * 32;
    const int nT = (M + 31) / 32;

    unsigned char* tcb = smem_raw + q.smem_fixed;
    unsigned char* stage = tcb + ((1024u - (tc::smem_u32(tcb) & 1023u)) & 1023u);   // [x digits | y digits]
    float* rings = reinterpret_cast<float*>(stage + kXAH + kXB);                   // cost rings of the DP warps

    if (threadIdx.x == 0) {
        tc::mbar_init(tc::smem_u32(&s_a), 1);
        tc::mbar_init(tc::smem_u32(&s_sfull), 1);
        tc::mbar_init(tc::smem_u32(&s_sempty), 1);
        tc::mbar_init(tc::smem_u32(&s_fin), 1);
        for (int t = 0; t < kXRT; ++t) {
            tc::mbar_init(tc::smem_u32(&s_tfull[t]), 1);
            tc::mbar_init(tc::smem_u32(&s_tfree[t]), kXConvWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) tc::tmem_alloc(&s_tmem, 512);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = s_tmem;
    int* status = q.status;
    const dd zero = mk(0.f, 0.f);

    dd c0 = zero;  // scaled d(i, 0)
    bool active = false;

    // the level MMAs of one 16-wide K step for x digits l0 .. l0 + kAH - 1 (staged from
    // a): digit l against the stacked y digits [b_0 ; ... ; b_(NS-1-l)], into the level
    // columns l .. NS-1
    auto level_mmas = [&](uint32_t d0, uint32_t a, uint32_t b, uint32_t ko, int l0, bool acc0) {
#pragma unroll
        for (int la = 0; la < kAH; ++la) {
            const int l = l0 + la;
            tc::mma_bf16(d0 + (uint32_t)(l * 32), tc::sdesc(a + la * kXAPart + ko), tc::sdesc(b + ko),
                         tc::idesc_bf16(128, (kXSlices - l) * 32), (acc0 || l > 0) ? 1u : 0u);
        }
    };

    if (warp == kXIssuer) {
        if (lane == 0) {
            bool ok = true;
            int issued = -1, landed = -1;   // stage fills issued / waited for
            if (resident) {
                const uint32_t abar = tc::smem_u32(&s_a);
                tc::mbar_expect_tx(abar, kXA);
                for (int l = 0; l < kXSlices; ++l)
                    tc::bulk_g2s(tc::smem_u32(stage + l * kXAPart), ximg + oimg_offset(p, 1, 0, NS, l, Npad, rs0),
                                 kXAPart, abar);
                tc::wait_ok_sleep(ok, abar, 0u, status);
            }
            // stage fill g = (c * KB + kb) * kH + h: y tile c's digits of K-block kb (with
            // h = 0) and, streamed, x digits h kAH .. h kAH + kAH - 1 of that K-block, once
            // the MMAs of fill g - 1 have read the stage
            const int G = nT * KB * kH;
            for (int g = 0; g < G && ok; ++g) {
                const int c = g / (KB * kH), r = g - c * KB * kH, kb = r / kH, h = r - kb * kH;
                const int t = c % kXRT;
                if (g >= 1) tc::wait_ok_sleep(ok, tc::smem_u32(&s_sempty), (uint32_t)((g - 1) & 1), status);
                if (!ok) break;
                const uint32_t bar = tc::smem_u32(&s_sfull);
                tc::mbar_expect_tx(bar, (resident ? 0u : kXAH) + (h == 0 ? kXB : 0u));
                if (!resident)
                    for (int la = 0; la < kAH; ++la)
                        tc::bulk_g2s(tc::smem_u32(stage + la * kXAPart),
                                     ximg + oimg_offset(p, KB, kb, NS, h * kAH + la, Npad, rs0), kXAPart, bar);
                if (h == 0)
                    for (int l = 0; l < kXSlices; ++l)
                        tc::bulk_g2s(tc::smem_u32(stage + kXAH + l * kXBPart),
                                     yimg + oimg_offset(p, KB, kb, NS, l, Mpad, 32 * c), kXBPart, bar);
                issued = g;
                if (kb == 0 && h == 0 && c >= kXRT)   // TMEM tile t free: the converters have read tile c - kXRT
                    tc::wait_ok_sleep(ok, tc::smem_u32(&s_tfree[t]), (uint32_t)(((c - kXRT) / kXRT) & 1), status);
                tc::wait_ok_sleep(ok, bar, (uint32_t)(g & 1), status);
                if (!ok) break;
                landed = g;
                tc::fence_after_sync();
                const uint32_t d0 = tmem + (uint32_t)(t * kXSlotCols);
                const uint32_t a = tc::smem_u32(stage), b = a + kXAH;
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) level_mmas(d0, a, b, ks * 32, h * kAH, kb > 0 || ks > 0);
                tc::mma_commit(tc::smem_u32(&s_sempty));
                if (kb == KB - 1 && h == kH - 1) tc::mma_commit(tc::smem_u32(&s_tfull[t]));
            }
            // every MMA has completed before tensor memory is released, and no copy is
            // still writing shared memory when the CTA exits
            tc::mma_commit(tc::smem_u32(&s_fin));
            bool fin = true;
            tc::wait_ok_sleep(fin, tc::smem_u32(&s_fin), 0u, status);
            if (issued > landed) tc::wait_ok_sleep(fin, tc::smem_u32(&s_sfull), (uint32_t)(issued & 1), status);
        }
        __syncwarp();
    } else if (warp > kXIssuer) {
        // converter of TMEM lane quarter qd, feeding DP warp qd's ring
        const int qd = warp & 3;
        const bool rows = rs0 + 32 * qd < N;   // DP warp qd has rows (else: read and release only)
        const int R = xring_tiles(qd);
        float* dh = rings + xring_first(qd) * 2 * kXTileFloats;   // [32 R][32] cost hi, slot (col mod 32 R), lane
        float* dl = dh + R * kXTileFloats;                        // [32 R][32] cost lo
        const float4 xi = xinfo[(size_t)p * Npad + rs0 + 32 * qd + lane];
        const int ex = __float_as_int(xi.z);
        const uint32_t tq = tmem + ((uint32_t)(32 * qd) << 16);
        bool ok = true;
        int used_seen = 0;
        // a tile's y row info is loaded one tile ahead (rows padded to Mpad >= 32 nT)
        const float4* yvp = yinfo + (size_t)p * Mpad + lane;
        float4 yv_next = yvp[0];
        for (int c = 0; c < nT; ++c) {
            const int t = c % kXRT;
            const float4 yv = yv_next;
            if (c + 1 < nT) yv_next = yvp[32 * (c + 1)];
            // ring slot of tile c held tile c - R: DP warp qd must be done with it
            if (rows && c - R + 1 > used_seen) ok = wait_smem_sleep(&s_used[qd], c - R + 1, q, used_seen, 128);
            if (!ok) break;
            tc::wait_ok_sleep(ok, tc::smem_u32(&s_tfull[t]), (uint32_t)((c / kXRT) & 1), status);
            if (!__all_sync(kFull, ok)) break;
            tc::fence_after_sync();
            const uint32_t tt0 = tq + (uint32_t)(t * kXSlotCols);
#pragma unroll 1
            for (int q8 = 0; q8 < 4; ++q8) {   // 8 columns at a time: NS x 8 level sums in registers
                uint32_t S[NS][8];
#pragma unroll
                for (int l = 0; l < NS; ++l) tc::tmem_ld8_nowait(tt0 + l * 32 + 8 * q8, S[l]);
                tc::tmem_wait_ld();
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int col = 8 * q8 + u;
                    const float nyh = __shfl_sync(kFull, yv.x, col), nyl = __shfl_sync(kFull, yv.y, col);
                    const int ey = __shfl_sync(kFull, __float_as_int(yv.z), col);
                    float Su[NS];
#pragma unroll
                    for (int l = 0; l < NS; ++l) Su[l] = __uint_as_float(S[l][u]);
                    const dd xy = levels_dd<NS>(Su, ex + ey + 2 - 2 * X::DB);
                    dd cst = sub(add(mk(xi.x, xi.y), mk(nyh, nyl)), mk(2.f * xy.hi, 2.f * xy.lo));
                    if (cst.hi < 0.f) cst = zero;
                    if (rows) {
                        const int slot = (32 * (c % R) + col) * 32 + lane;
                        dh[slot] = cst.hi;
                        dl[slot] = cst.lo;
                    }
                }
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(tc::smem_u32(&s_tfree[t]));
            if (rows) {   // the costs are visible to DP warp qd before the count
                __threadfence_block();
                __syncwarp();
                if (lane == 0) s_conv[qd] = c + 1;
            }
        }
    } else {
        const int rb = strip * W + warp, r0 = rb * 32, i = r0 + lane;
        active = r0 < N;
        const bool has_top = active && r0 > 0;
        const bool top_global = has_top && warp == 0;
        const bool has_bot = active && (r0 + 32 < N);
        const bool bot_global = has_bot && warp == W - 1;
        const bool row0_lane = (i == 0);
        const int Nb = q.lens_n ? min(max(q.lens_n[p], 1), N) : N;
        const int Mb = q.lens_m ? min(max(q.lens_m[p], 1), M) : M;
        const bool last_lane = (i == Nb - 1);
        const float scale = q.scale;
        float2* rowbuf = reinterpret_cast<float2*>(q.rowbuf) + (size_t)p * M;
        const int rcols = 32 * xring_tiles(warp);   // ring columns: slot of column j is j mod rcols
        const float* dh = rings + xring_first(warp) * 2 * kXTileFloats;
        const float* dl = dh + xring_tiles(warp) * kXTileFloats;

        if (active) {
            float4* lpp = reinterpret_cast<float4*>(q.VH) + skew_index(N, M, p, rb, 0, lane);
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
            int cons_seen = 0, conv_seen = 0;
            const int nG = T / kGroup;
            for (int g = 0; g < nG; ++g) {
                const int s0 = g * kGroup;
                if ((s0 & 31) == 0 && (s0 >> 5) < nT) {
                    // period c = s0/32 reads columns of tiles c-1 and c: tiles below c - 1
                    // are free for the converter, tile c must be in the ring
                    const int c = s0 >> 5;
                    if (c >= 2 && lane == 0) s_used[warp] = c - 1;
                    if (conv_seen < c + 1 && !wait_smem(&s_conv[warp], c + 1, q, conv_seen)) break;
                    __threadfence_block();
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

                // the group in rolled chunks of kXChunkFused steps (nine warps' code shares the
                // instruction cache); each chunk's costs go into registers before any of its
                // stores (the compiler keeps loads behind stores it cannot prove apart)
                int col = (s0 - lane + rcols) % rcols;   // column s0 - lane >= -31 in the ring
#pragma unroll 1
                for (int h8 = 0; h8 < kGroup; h8 += kXChunkFused) {
                    float2 dc[kXChunkFused];
#pragma unroll
                    for (int uu = 0; uu < kXChunkFused; ++uu) {
                        dc[uu] = make_float2(dh[col * 32 + lane], dl[col * 32 + lane]);
                        col = (col + 1 == rcols) ? 0 : col + 1;
                    }
#pragma unroll
                    for (int uu = 0; uu < kXChunkFused; ++uu) {
                        const int u = h8 + uu;
                        const int s = s0 + u;
                        const int j = s - lane;
                        const float hs_hi = __shfl_up_sync(kFull, h_prev.hi, 1);
                        const float hs_lo = __shfl_up_sync(kFull, h_prev.lo, 1);
                        const float tv_hi = __shfl_sync(kFull, topv.hi, u);
                        const float tv_lo = __shfl_sync(kFull, topv.lo, u);
                        const dd hu = (lane == 0) ? mk(tv_hi, tv_lo) : mk(hs_hi, hs_lo);
                        const dd vl = v_prev;
                        const dd d = scale_dd(mk(dc[uu].x, dc[uu].y), scale);
                        const bool col0 = (j == 0);
                        dd h, v;
                        float4 lp;
                        xcell(d, vl, hu, col0, row0_lane, h, v, lp);
                        c0 = col0 ? d : c0;
                        lpp[(long long)s * 32] = lp;
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
                }
                if (has_top && !top_global && lane == 0) cons[warp - 1] = min(s0 + kGroup, M);
            }
        }
    }

    // Loss: R[N,M] = sum_i d(i,0) + sum_{j>=1} h(N-1, j), scaled units, in fp64.
    const int nwarps = (int)(blockDim.x >> 5);
    const int Nb = q.lens_n ? min(max(q.lens_n[p], 1), N) : N;
    const int Mb = q.lens_m ? min(max(q.lens_m[p], 1), M) : M;
    double part = (active && warp < W && rs0 + 32 * warp + lane < Nb) ? (double)c0.hi + (double)c0.lo : 0.0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(kFull, part, o);
    if (lane == 0) s_red[warp] = part;
    __threadfence();
    __syncthreads();
    float2* rowbuf = reinterpret_cast<float2*>(q.rowbuf) + (size_t)p * M;
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
        for (int j = 1 + (int)threadIdx.x; j < Mb; j += blockDim.x) {
            const float2 hv = __ldcg(rowbuf + j);
            acc += (double)hv.x + (double)hv.y;
        }
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(kFull, acc, o);
        if (lane == 0) s_red[warp] = acc;
        __syncthreads();
        if (threadIdx.x == 0) {
            double tot = 0.0;
            for (int w = 0; w < nwarps; ++w) tot += s_red[w];
            for (int k = 0; k < q.S; ++k) tot += __ldcg(&q.colsum[(size_t)p * q.NB + k]);
            q.loss[p] = (float)(tot * (double)q.unscale);
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 512);
    }
}

// The extended unfused cost tensor from the exact level sums. One CTA per 128 x
// rows and problem walks the y columns in tiles of 32: warp 8 (lane 0) copies the
// digits (x resident for one K-block, else both streamed per K-block through one
// stage) and issues each tile's level MMAs into one of two tensor-memory slots;
// epilogue warps 0-7 drain the other. Warp w reads TMEM lane quarter w mod 4 and
// the 16-column half w / 4 of the tile, combines the NS level sums of each column
// with the exponents and the double-float norms into C = |x|^2 + |y|^2 - 2 x . y
// (clamped at 0) and writes the skewed layout through a per-warp staging tile.
// No DP runs behind the tiles, so two slots keep the MMAs ahead of the epilogue
// and six digits (two slots of 192 columns) fit as well. Hand-offs (bounded
// mbarrier waits):
//   s_a         x digits resident       s_bfull[e] / s_bempty[e]  y ring (one K-block)
//   s_sfull     stage landed            s_sempty   its MMAs are done (K-blocks streamed)
//   s_tfull[t]  levels in TMEM slot t   s_tfree[t] the 8 epilogue warps read slot t
constexpr int kXdWarps = 8;
constexpr int kXdStg = 47 * 32;   // per-warp staging: skewed rows of a 16-column chunk (float2)

template <int NS>
__global__ void __launch_bounds__((kXdWarps + 1) * 32, 1)
    distx_tc_kernel(int N, int M, int D, const unsigned char* __restrict__ ximg, const unsigned char* __restrict__ yimg,
                    const float4* __restrict__ xinfo, const float4* __restrict__ yinfo, float2* __restrict__ Dsk,
                    int* status)
{
    using X = XDigits<NS>;
    constexpr int kSlot = X::SlotCols;
    constexpr uint32_t kA = X::A, kB = X::B;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __shared__ uint64_t s_a, s_sfull, s_sempty, s_fin, s_bfull[2], s_bempty[2], s_tfull[2], s_tfree[2];
    __shared__ uint32_t s_tmem;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int p = blockIdx.y, r0 = blockIdx.x * 128;
    const int KB = (D + kTcKFeat - 1) / kTcKFeat;
    const bool resident = KB == 1;
    const int Npad = simg_pad(N), Mpad = simg_pad(M);
    const int nT = (M + 31) / 32;
    unsigned char* stage = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
    float2* stg = reinterpret_cast<float2*>(stage + xtc_region(NS, KB)) + warp * kXdStg;

    if (threadIdx.x == 0) {
        tc::mbar_init(tc::smem_u32(&s_a), 1);
        tc::mbar_init(tc::smem_u32(&s_sfull), 1);
        tc::mbar_init(tc::smem_u32(&s_sempty), 1);
        tc::mbar_init(tc::smem_u32(&s_fin), 1);
        for (int e = 0; e < 2; ++e) {
            tc::mbar_init(tc::smem_u32(&s_bfull[e]), 1);
            tc::mbar_init(tc::smem_u32(&s_bempty[e]), 1);
            tc::mbar_init(tc::smem_u32(&s_tfull[e]), 1);
            tc::mbar_init(tc::smem_u32(&s_tfree[e]), kXdWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) tc::tmem_alloc(&s_tmem, 512);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = s_tmem;
    bool ok = true;

    // the level MMAs of one 16-wide K step: x digit l against the stacked y digits
    // [b_0 ; ... ; b_(NS-1-l)], into the level columns l .. NS-1
    auto level_mmas = [&](uint32_t d0, uint32_t a, uint32_t b, uint32_t ko, bool acc0) {
#pragma unroll
        for (int l = 0; l < NS; ++l)
            tc::mma_bf16(d0 + (uint32_t)(l * 32), tc::sdesc(a + l * kXAPart + ko), tc::sdesc(b + ko),
                         tc::idesc_bf16(128, (NS - l) * 32), (acc0 || l > 0) ? 1u : 0u);
    };

    if (warp == kXdWarps) {
        if (lane == 0) {
            if (resident) {
                int y_last[2] = {-1, -1};
                const uint32_t abar = tc::smem_u32(&s_a);
                tc::mbar_expect_tx(abar, kA);
                for (int l = 0; l < NS; ++l)
                    tc::bulk_g2s(tc::smem_u32(stage + l * kXAPart), ximg + oimg_offset(p, 1, 0, NS, l, Npad, r0),
                                 kXAPart, abar);
                auto issue_y = [&](int c) {
                    const int e = c & 1;
                    const uint32_t bar = tc::smem_u32(&s_bfull[e]);
                    tc::mbar_expect_tx(bar, kB);
                    for (int l = 0; l < NS; ++l)
                        tc::bulk_g2s(tc::smem_u32(stage + kA + e * kB + l * kXBPart),
                                     yimg + oimg_offset(p, 1, 0, NS, l, Mpad, 32 * c), kXBPart, bar);
                    y_last[e] = c;
                };
                for (int c = 0; c < 2 && c < nT; ++c) issue_y(c);
                tc::wait_ok(ok, abar, 0u, status);
                for (int c = 0; c < nT && ok; ++c) {
                    const int e = c & 1;
                    if (c >= 2) tc::wait_ok(ok, tc::smem_u32(&s_tfree[e]), (uint32_t)(((c - 2) >> 1) & 1), status);
                    tc::wait_ok(ok, tc::smem_u32(&s_bfull[e]), (uint32_t)((c >> 1) & 1), status);
                    if (!ok) break;
                    tc::fence_after_sync();
                    const uint32_t d0 = tmem + (uint32_t)(e * kSlot);
                    const uint32_t a = tc::smem_u32(stage), b = a + kA + e * kB;
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) level_mmas(d0, a, b, ks * 32, ks > 0);
                    tc::mma_commit(tc::smem_u32(&s_bempty[e]));
                    tc::mma_commit(tc::smem_u32(&s_tfull[e]));
                    if (c + 2 < nT) {   // entry e takes tile c + 2 once MMA(c) has read it
                        tc::wait_ok(ok, tc::smem_u32(&s_bempty[e]), (uint32_t)((c >> 1) & 1), status);
                        if (!ok) break;
                        issue_y(c + 2);
                    }
                }
                tc::mma_commit(tc::smem_u32(&s_fin));
                bool fin = true;
                tc::wait_ok(fin, tc::smem_u32(&s_fin), 0u, status);
                for (int e = 0; e < 2; ++e)
                    if (y_last[e] >= 0)
                        tc::wait_ok(fin, tc::smem_u32(&s_bfull[e]), (uint32_t)((y_last[e] >> 1) & 1), status);
            } else {
                // stage g = c * KB + kb: K-block kb of the x rows' and of y tile c's digits
                const int G = nT * KB;
                int g_last = -1;
                for (int g = 0; g < G && ok; ++g) {
                    const int c = g / KB, kb = g - c * KB, t = c & 1;
                    if (kb == 0 && c >= 2)
                        tc::wait_ok(ok, tc::smem_u32(&s_tfree[t]), (uint32_t)(((c - 2) >> 1) & 1), status);
                    if (g >= 1) tc::wait_ok(ok, tc::smem_u32(&s_sempty), (uint32_t)((g - 1) & 1), status);
                    if (!ok) break;
                    const uint32_t bar = tc::smem_u32(&s_sfull);
                    tc::mbar_expect_tx(bar, kA + kB);
                    for (int l = 0; l < NS; ++l)
                        tc::bulk_g2s(tc::smem_u32(stage + l * kXAPart), ximg + oimg_offset(p, KB, kb, NS, l, Npad, r0),
                                     kXAPart, bar);
                    for (int l = 0; l < NS; ++l)
                        tc::bulk_g2s(tc::smem_u32(stage + kA + l * kXBPart),
                                     yimg + oimg_offset(p, KB, kb, NS, l, Mpad, 32 * c), kXBPart, bar);
                    g_last = g;
                    tc::wait_ok(ok, bar, (uint32_t)(g & 1), status);
                    if (!ok) break;
                    tc::fence_after_sync();
                    const uint32_t d0 = tmem + (uint32_t)(t * kSlot);
                    const uint32_t a = tc::smem_u32(stage), b = a + kA;
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) level_mmas(d0, a, b, ks * 32, kb > 0 || ks > 0);
                    tc::mma_commit(tc::smem_u32(&s_sempty));
                    if (kb == KB - 1) tc::mma_commit(tc::smem_u32(&s_tfull[t]));
                }
                tc::mma_commit(tc::smem_u32(&s_fin));
                bool fin = true;
                tc::wait_ok(fin, tc::smem_u32(&s_fin), 0u, status);
                if (g_last >= 0) tc::wait_ok(fin, tc::smem_u32(&s_sfull), (uint32_t)(g_last & 1), status);
            }
        }
        __syncwarp();
    } else {
        const int qd = warp & 3, half = warp >> 2;
        const int rb = (r0 >> 5) + qd, row = r0 + 32 * qd + lane;
        const int NB = (N + 31) / 32;
        const float4 xi = xinfo[(size_t)p * Npad + row];
        const int ex = __float_as_int(xi.z);
        const uint32_t tq = tmem + ((uint32_t)(32 * qd) << 16);
        float2* out = (rb < NB) ? Dsk + skew_index(N, M, p, rb, 0, lane) : nullptr;
        for (int c = 0; c < nT; ++c) {
            const int t = c & 1;
            tc::wait_ok(ok, tc::smem_u32(&s_tfull[t]), (uint32_t)((c >> 1) & 1), status);
            if (!__all_sync(kFull, ok)) break;
            tc::fence_after_sync();
            const int cb = 32 * c + 16 * half;   // first column of this warp's chunk
            const float4 yv = yinfo[(size_t)p * Mpad + cb + (lane & 15)];
            const uint32_t tt0 = tq + (uint32_t)(t * kSlot + 16 * half);
#pragma unroll
            for (int h8 = 0; h8 < 2; ++h8) {   // 8 columns at a time: NS x 8 level sums in registers
                uint32_t S[NS][8];
#pragma unroll
                for (int l = 0; l < NS; ++l) tc::tmem_ld8_nowait(tt0 + l * 32 + 8 * h8, S[l]);
                tc::tmem_wait_ld();
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int col = 8 * h8 + u;
                    const float nyh = __shfl_sync(kFull, yv.x, col), nyl = __shfl_sync(kFull, yv.y, col);
                    const int ey = __shfl_sync(kFull, __float_as_int(yv.z), col);
                    float Su[NS];
#pragma unroll
                    for (int l = 0; l < NS; ++l) Su[l] = __uint_as_float(S[l][u]);
                    const dd xy = levels_dd<NS>(Su, ex + ey + 2 - 2 * X::DB);
                    dd cst = sub(add(mk(xi.x, xi.y), mk(nyh, nyl)), mk(2.f * xy.hi, 2.f * xy.lo));
                    if (cst.hi < 0.f) cst = mk(0.f, 0.f);
                    stg[(col + lane) * 32 + lane] = make_float2(cst.hi, cst.lo);
                }
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(tc::smem_u32(&s_tfree[t]));
            if (out != nullptr && cb < M) {   // warp-uniform
                // skewed slot cb + tt holds column cb + tt - lane of this lane's row
                for (int tt = 0; tt < 47; ++tt) {
                    const int j = tt - lane;
                    if (j >= 0 && j < 16 && cb + j < M && row < N) out[(long long)(cb + tt) * 32] = stg[tt * 32 + lane];
                }
            }
            __syncwarp();
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 512);
    }
}

}  // namespace

// digits per value of the exact cost tiles for a feature width
int xtc_slices(int D) { return D <= 128 ? 5 : 6; }

size_t oimg_bytes(int P, int L, int D)
{
    const int KB = (D + kTcKFeat - 1) / kTcKFeat;
    return (size_t)P * KB * xtc_slices(D) * simg_pad(L) * 128;
}

size_t oinfo_bytes(int P, int L) { return (size_t)P * simg_pad(L) * sizeof(float4); }

cudaError_t launch_oimg(const Problems& pr, int P, int N, int M, int D, void* ximg, void* yimg, void* xinfo,
                        void* yinfo, cudaStream_t st)
{
    const int KB = (D + kTcKFeat - 1) / kTcKFeat;
    const int Lmax = simg_pad(N > M ? N : M);
    const size_t smem = sizeof(float) * 32 * (kTcKFeat * KB + 1);
    auto go = [&](auto kern) -> cudaError_t {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        kern<<<dim3(Lmax / 32, P, 2), 256, smem, st>>>(pr, N, M, D, KB, static_cast<unsigned char*>(ximg),
                                                       static_cast<unsigned char*>(yimg), static_cast<float4*>(xinfo),
                                                       static_cast<float4*>(yinfo));
        return cudaGetLastError();
    };
    return xtc_slices(D) == 5 ? go(oimg_kernel<5>) : go(oimg_kernel<6>);
}

cudaError_t launch_forward_xtc(WaveParams q, const void* ximg, const void* yimg, const void* xinfo,
                               const void* yinfo, cudaStream_t st)
{
    if (q.W != kXDpWarps || q.D > kMaxXtcD) return cudaErrorInvalidValue;
    const int grid = q.P * q.S;
    q.smem_fixed = (int)(((size_t)kXDpWarps * kRing * 2 * sizeof(Slot) + (size_t)kXDpWarps * sizeof(int) + 15) &
                         ~(size_t)15);
    auto go = [&](auto kern, size_t stage) -> cudaError_t {
        const size_t need = q.smem_fixed + 1024 + stage + kXRingBytes;
        const size_t smem = max(need, wave_smem_floor());   // one CTA per SM: the whole tensor memory
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        kern<<<grid, kXFusedThreads, smem, st>>>(q, static_cast<const unsigned char*>(ximg),
                                                 static_cast<const unsigned char*>(yimg),
                                                 static_cast<const float4*>(xinfo), static_cast<const float4*>(yinfo));
        return cudaGetLastError();
    };
    // the stage: all five x digits of a K-block, or three of six, and the y tile's digits
    return xtc_slices(q.D) == 5 ? go(fwdx_tc_kernel<5>, XDigits<5>::A + XDigits<5>::B)
                                : go(fwdx_tc_kernel<6>, 3 * kXAPart + XDigits<6>::B);
}

cudaError_t launch_dist_xtc(int P, int N, int M, int D, const void* ximg, const void* yimg, const void* xinfo,
                            const void* yinfo, float2* Dsk, int* status, cudaStream_t st)
{
    if (D < 1 || D > kMaxXtcD) return cudaErrorInvalidValue;
    const int KB = (D + kTcKFeat - 1) / kTcKFeat;
    const int NS = xtc_slices(D);
    const size_t smem = 1024 + xtc_region(NS, KB) + (size_t)kXdWarps * kXdStg * sizeof(float2);
    if (smem > 227 * 1024) return cudaErrorInvalidValue;
    const dim3 grid((N + 127) / 128, P);
    auto go = [&](auto kern) -> cudaError_t {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        kern<<<grid, (kXdWarps + 1) * 32, smem, st>>>(N, M, D, static_cast<const unsigned char*>(ximg),
                                                      static_cast<const unsigned char*>(yimg),
                                                      static_cast<const float4*>(xinfo),
                                                      static_cast<const float4*>(yinfo), Dsk, status);
        return cudaGetLastError();
    };
    return NS == 5 ? go(distx_tc_kernel<5>) : go(distx_tc_kernel<6>);
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
