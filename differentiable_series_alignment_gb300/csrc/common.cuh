// common.cuh -- device helpers and data layouts shared by the library's kernels.
//
// Units. The DP runs in "scaled base-2" units: every cost and every R
// difference is multiplied by s = log2(e) / gamma, so that
//   softmin_gamma(a, b, c) * s = -log2(2^-a' + 2^-b' + 2^-c')
// and the exponentials are single MUFU ex2 / lg2 instructions.
//
// Difference form. Instead of R itself the forward carries, per cell,
//   h[i,j] = R[i,j] - R[i,j-1]   and   v[i,j] = R[i,j] - R[i-1,j],
// and, with a = R[i-1,j-1] as reference, the recursion becomes
//   t = d[i,j] + softmin(0, vl, hu),  h = t - vl,  v = t - hu,
//   vl = v[i,j-1],  hu = h[i-1,j].
// Neighbouring differences are small numbers, so fp32 keeps them to ~1e-7
// relative, whereas fp32 R itself loses the low bits that the backward's
// transition probabilities exp((R[s]-C[s]-R[p])/gamma) depend on.
//
// Skewed ("anti-diagonal major") layout. Rows are grouped in blocks of 32 (one
// warp, lane = row within the block). Within a block, entry (t, lane) holds the
// cell (32*rb + lane, t - lane), t in [0, M+31). A warp that walks the
// wavefront touches one contiguous 128-byte row (t) per step.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace sdtw {

constexpr float kBig = 1e30f;          // stands for +inf in stored differences
constexpr int kGroup = 16;             // wavefront steps between channel synchronizations
constexpr int kRing = 256;             // entries of a shared-memory channel between warps
constexpr int kMaxWarps = 16;          // warps (32-row blocks) per wavefront CTA
constexpr int kStatusTimeout = 1;      // bit in the device status word

// Batch of independent problems. Problem p uses set s = p / B and element
// b = p % B; its inputs are xs[s] + b*xstride[s] (N,D) and ys[s] + b*ystride[s]
// (M,D). A stride of 0 broadcasts one sequence over the batch.
struct Problems {
    const float* xs[3];
    const float* ys[3];
    long long xstride[3];
    long long ystride[3];
    int B;
    // Selects rather than xs[s]: indexing the kernel-parameter arrays by a run-time
    // value would make every thread copy them to local memory first.
    __host__ __device__ __forceinline__ const float* x(int p) const {
        const int s = p / B, b = p - s * B;
        const float* base = s == 0 ? xs[0] : (s == 1 ? xs[1] : xs[2]);
        const long long st = s == 0 ? xstride[0] : (s == 1 ? xstride[1] : xstride[2]);
        return base + (long long)b * st;
    }
    __host__ __device__ __forceinline__ const float* y(int p) const {
        const int s = p / B, b = p - s * B;
        const float* base = s == 0 ? ys[0] : (s == 1 ? ys[1] : ys[2]);
        const long long st = s == 0 ? ystride[0] : (s == 1 ? ystride[1] : ystride[2]);
        return base + (long long)b * st;
    }
};

// Skewed layout geometry for one problem: NB blocks of skew_T(M) x 32 slots,
// skew_T(M) = M + 31 rounded up to a whole number of wavefront groups (the
// padding slots hold no cell, so the step loops need no bounds checks).
__host__ __device__ __forceinline__ int skew_T(int M) {
    return ((M + 31 + kGroup - 1) / kGroup) * kGroup;
}
__host__ __device__ __forceinline__ long long skew_slots(int N, int M) {
    return (long long)((N + 31) / 32) * (long long)skew_T(M) * 32;
}
__host__ __device__ __forceinline__ long long skew_index(int N, int M, int p, int rb, int t, int lane) {
    return (long long)p * skew_slots(N, M) + ((long long)rb * skew_T(M) + t) * 32 + lane;
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float lg2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// 2^x for x <= 0; 0 for x < -125 (and for x = -inf). Cody & Waite range
// reduction x = n + f, n = rint(x), f in [-1/2, 1/2], then a degree-7
// polynomial for 2^f fitted for this library (fit_exp2.py: relative fit error
// 2.6e-9, mean -4e-10). Its error is dominated by round-to-nearest, so it has
// no systematic bias, unlike the hardware approximation: the DP recursions add
// ~N+M of these terms along every path, and a biased exponential would drift
// the alignment matrix.
__device__ __forceinline__ float exp2_neg(float x) {
    const float magic = 12582912.0f;  // 1.5 * 2^23: x + magic rounds x to an integer
    const float t = x + magic;
    const float n = t - magic;
    const float f = x - n;
    float p = 1.5165811419137754e-05f;
    p = fmaf(p, f, 0.00015466917830053717f);
    p = fmaf(p, f, 0.001333407941274345f);
    p = fmaf(p, f, 0.00961803738027811f);
    p = fmaf(p, f, 0.055504102259874344f);
    p = fmaf(p, f, 0.24022650718688965f);
    p = fmaf(p, f, 0.6931471824645996f);
    p = fmaf(p, f, 1.0f);
    const int scale = (__float_as_int(t) - 0x4B400000) << 23;  // n << 23
    const float r = __int_as_float(__float_as_int(p) + scale);
    return (x < -125.0f) ? 0.0f : r;
}

// Math of the DP kernels: the double-float path (flag set) takes the unbiased
// exp2_neg above and log2f, the fp32 path the MUFU approximations.
template <bool EXT> __device__ __forceinline__ float dp_exp2(float x) { return EXT ? exp2_neg(x) : ex2(x); }
template <bool EXT> __device__ __forceinline__ float dp_log2(float x) { return EXT ? log2f(x) : lg2(x); }

// Error-free sum (Knuth's TwoSum): s + e == a + b exactly.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
    s = a + b;
    const float bb = s - a;
    e = (a - (s - bb)) + (b - bb);
}

// Squared Euclidean distance accumulator. Terms are summed in fp32 over blocks
// of kDistBlock components; block sums are added into a (hi, lo) pair with
// TwoSum, so the result is within about one rounding of the exact sum. A plain
// sequential fp32 sum over D components is ~5x less accurate, and the
// gradient reacts to cost errors at that level (the alignment matrix moves by
// ~1e-4 relative), which the rel 1e-3 gradient tolerance does not absorb where
// the terms of sum_j E[i,j] (x_i - y_j) cancel.
constexpr int kDistBlock = 8;
struct DistAcc {
    float hi = 0.f, lo = 0.f;
    __device__ __forceinline__ void add_block(float blk) {
        float s, e;
        two_sum(hi, blk, s, e);
        hi = s;
        lo += e;
    }
    __device__ __forceinline__ float value() const { return hi + lo; }
};

// Packed fp32 pairs (f32x2 instructions: one issue slot for two lanes' worth
// of arithmetic per thread).
__device__ __forceinline__ unsigned long long pk2(float a, float b) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void upk2(unsigned long long v, float& a, float& b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ unsigned long long sub2(unsigned long long a, unsigned long long b) {
    unsigned long long r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b, unsigned long long c) {
    unsigned long long r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

// Squared distance of two zero-padded rows of D32 (multiple of 32) floats,
// 16-byte aligned. Each 32-component group feeds four independent block sums
// of 8 components (packed fp32 pairs); each block sum enters its own TwoSum
// (hi, lo) pair, and the four pairs are combined at the end. Four independent
// chains keep the latency short enough to hide inside a DP step. Shared by the
// unfused cost kernel and the fused forward, so both see identical costs.
__device__ __forceinline__ unsigned long long blk8(const float4* x4, const float4* y4) {
    const float4 xa = x4[0], ya = y4[0], xb = x4[1], yb = y4[1];
    unsigned long long d = sub2(pk2(xa.x, xa.y), pk2(ya.x, ya.y));
    unsigned long long b = fma2(d, d, pk2(0.f, 0.f));
    d = sub2(pk2(xa.z, xa.w), pk2(ya.z, ya.w));
    b = fma2(d, d, b);
    d = sub2(pk2(xb.x, xb.y), pk2(yb.x, yb.y));
    b = fma2(d, d, b);
    d = sub2(pk2(xb.z, xb.w), pk2(yb.z, yb.w));
    return fma2(d, d, b);
}
__device__ __forceinline__ void fold(DistAcc& a, unsigned long long b) {
    float e0, e1;
    upk2(b, e0, e1);
    a.add_block(e0 + e1);
}
__device__ __forceinline__ float dist_rows(const float* __restrict__ xr, const float* __restrict__ yr, int D32) {
    const float4* x4 = reinterpret_cast<const float4*>(xr);
    const float4* y4 = reinterpret_cast<const float4*>(yr);
    DistAcc a0, a1, a2, a3;
    for (int q = 0; q < (D32 >> 2); q += 8) {
        fold(a0, blk8(x4 + q, y4 + q));
        fold(a1, blk8(x4 + q + 2, y4 + q + 2));
        fold(a2, blk8(x4 + q + 4, y4 + q + 4));
        fold(a3, blk8(x4 + q + 6, y4 + q + 6));
    }
    float s01, e01, s23, e23, s, e;
    two_sum(a0.hi, a1.hi, s01, e01);
    two_sum(a2.hi, a3.hi, s23, e23);
    two_sum(s01, s23, s, e);
    return s + (e + ((e01 + e23) + ((a0.lo + a1.lo) + (a2.lo + a3.lo))));
}

// The same arithmetic as dist_rows with one row held in registers (DX = 32 or
// 64 padded components) and the other row read from shared memory: `r` minus
// the shared row, in the same block order, so the results are bit-identical.
template <int DX>
__device__ __forceinline__ unsigned long long blk8r(const float (&r)[DX], int o, const float4* y4) {
    const float4 ya = y4[0], yb = y4[1];
    unsigned long long d = sub2(pk2(r[o], r[o + 1]), pk2(ya.x, ya.y));
    unsigned long long b = fma2(d, d, pk2(0.f, 0.f));
    d = sub2(pk2(r[o + 2], r[o + 3]), pk2(ya.z, ya.w));
    b = fma2(d, d, b);
    d = sub2(pk2(r[o + 4], r[o + 5]), pk2(yb.x, yb.y));
    b = fma2(d, d, b);
    d = sub2(pk2(r[o + 6], r[o + 7]), pk2(yb.z, yb.w));
    return fma2(d, d, b);
}
template <int DX>
__device__ __forceinline__ float dist_reg(const float (&r)[DX], const float* __restrict__ yr) {
    const float4* y4 = reinterpret_cast<const float4*>(yr);
    DistAcc a0, a1, a2, a3;
#pragma unroll
    for (int q = 0; q < DX / 4; q += 8) {
        fold(a0, blk8r(r, 4 * q, y4 + q));
        fold(a1, blk8r(r, 4 * q + 8, y4 + q + 2));
        fold(a2, blk8r(r, 4 * q + 16, y4 + q + 4));
        fold(a3, blk8r(r, 4 * q + 24, y4 + q + 6));
    }
    float s01, e01, s23, e23, s, e;
    two_sum(a0.hi, a1.hi, s01, e01);
    two_sum(a2.hi, a3.hi, s23, e23);
    two_sum(s01, s23, s, e);
    return s + (e + ((e01 + e23) + ((a0.lo + a1.lo) + (a2.lo + a3.lo))));
}

// Sort three values: lo <= mid <= hi.
__device__ __forceinline__ void sort3(float a, float b, float c, float& lo, float& mid, float& hi) {
    const float t1 = fminf(a, b), t2 = fmaxf(a, b);
    lo = fminf(t1, c);
    hi = fmaxf(t2, c);
    mid = fmaxf(t1, fminf(t2, c));
}

// A channel slot: a value and the tag that validates it (tag = column + 1;
// 0 = not written yet). Written and read as one 64-bit access, which is
// single-copy atomic, so a reader that sees the expected tag also sees the
// value and neither side needs a fence or a separate ready counter.
struct __align__(8) Slot {
    float v;
    unsigned tag;
};
// A slot publishes one value and nothing else, so its store needs no ordering
// against other memory operations of the producer (no "memory" clobber): the
// consumer reads only the slot itself and accepts it once the tag matches.
__device__ __forceinline__ void slot_store(Slot* p, float v, unsigned tag) {
    asm volatile("st.volatile.v2.b32 [%0], {%1, %2};" ::"l"(p), "f"(v), "r"(tag));
}
// slot_store under a per-lane predicate, as one predicated instruction: a branch
// around the store would diverge (one lane publishes) in every DP step.
__device__ __forceinline__ void slot_store_if(bool pred, Slot* p, float v, unsigned tag) {
    asm volatile(
        "{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %3, 0;\n\t@q st.volatile.v2.b32 [%0], {%1, %2};\n\t}"
        ::"l"(p), "f"(v), "r"(tag), "r"((unsigned)pred));
}
__device__ __forceinline__ Slot slot_load(const Slot* p) {
    Slot s;
    asm volatile("ld.volatile.v2.b32 {%0, %1}, [%2];" : "=f"(s.v), "=r"(s.tag) : "l"(p) : "memory");
    return s;
}

// Stage rows [row0, row0 + rows) of a row-major (., D) fp32 matrix into shared
// memory rows of ld floats (columns [0, cols): zero past D and for rows outside
// [0, rows_valid)), cooperatively over nthreads threads (this one is tid). Each
// thread issues its loads in batches of 8 before the batch's stores, so a batch
// costs one memory latency instead of eight.
__device__ __forceinline__ void stage_rows(float* dst, int ld, const float* src, int D, int row0, int rows,
                                           int cols, int rows_valid, int tid, int nthreads)
{
    const int n = rows * cols;
    for (int e0 = tid; e0 < n; e0 += 8 * nthreads) {
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int e = e0 + u * nthreads;
            const int r = e / cols, k = e - r * cols;
            const int row = row0 + r;
            v[u] = (e < n && row >= 0 && row < rows_valid && k < D) ? src[(size_t)row * D + k] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int e = e0 + u * nthreads;
            const int r = e / cols, k = e - r * cols;
            if (e < n) dst[r * ld + k] = v[u];
        }
    }
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ int ld_volatile_global(const int* p) {
    return *reinterpret_cast<const volatile int*>(p);
}

}  // namespace sdtw
