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
    __host__ __device__ __forceinline__ const float* x(int p) const {
        int s = p / B, b = p - s * B;
        return xs[s] + (long long)b * xstride[s];
    }
    __host__ __device__ __forceinline__ const float* y(int p) const {
        int s = p / B, b = p - s * B;
        return ys[s] + (long long)b * ystride[s];
    }
};

// Skewed layout geometry for one problem: NB blocks of (M+31) x 32 slots.
__host__ __device__ __forceinline__ long long skew_slots(int N, int M) {
    return (long long)((N + 31) / 32) * (long long)(M + 31) * 32;
}
__host__ __device__ __forceinline__ long long skew_index(int N, int M, int p, int rb, int t, int lane) {
    return (long long)p * skew_slots(N, M) + ((long long)rb * (M + 31) + t) * 32 + lane;
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
__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_gpu(int* p, int v) {
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_volatile_global(const int* p) {
    return *reinterpret_cast<const volatile int*>(p);
}

}  // namespace sdtw
