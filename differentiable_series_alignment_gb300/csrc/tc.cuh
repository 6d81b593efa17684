// tc.cuh -- tcgen05 / TMA / mbarrier building blocks shared by the tensor-core
// kernels (gradient contraction, cost tiles): shared-memory descriptors for the
// 128-byte-swizzled K-major layout, the tf32 instruction descriptor, the 3xTF32
// hi/lo split, bounded mbarrier waits, bulk copies and tensor-memory loads.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

#include "common.cuh"

namespace sdtw {
namespace tc {

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

// Instruction descriptor of kind::f16 with bf16 A and B (both K-major), fp32 D, M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

// The three MMAs of one 16-wide K step (byte offset ko along K) of the exact
// product of split operands: a = [x0 | x1 | x2], the three parts of M rows each,
// part_a bytes apart; b = [y0 ; y1 ; y2] stacked along N, `rows` y rows per part,
// contiguous. Each x part multiplies all three y parts, so every one of the nine
// part products (each exact in fp32: 8 x 8 significant bits) enters; tensor-memory
// columns [0, rows), [rows, 2 rows) and [2 rows, 3 rows) of d receive the y0, y1
// and y2 terms, whose sum is x . y up to the fp32 accumulation.
__device__ __forceinline__ void mma_bf16x3(uint32_t d, uint32_t a, uint32_t b, int M, int rows, uint32_t part_a,
                                           uint32_t ko, uint32_t acc)
{
    const uint32_t id = idesc_bf16(M, 3 * rows);
    mma_bf16(d, sdesc(a + ko), sdesc(b + ko), id, acc);
    mma_bf16(d, sdesc(a + part_a + ko), sdesc(b + ko), id, 1u);
    mma_bf16(d, sdesc(a + 2 * part_a + ko), sdesc(b + ko), id, 1u);
}

// fp32 -> three bf16 parts with v == b0 + b1 + b2 exactly: each part takes the
// next 8 significant bits (round to nearest), and the remainders are exact in
// fp32 (24 = 3 x 8 bits). Packed as raw 16-bit patterns.
__device__ __forceinline__ void split_bf16x3(float v, uint16_t& b0, uint16_t& b1, uint16_t& b2) {
    const __nv_bfloat16 h0 = __float2bfloat16_rn(v);
    const float r1 = v - __bfloat162float(h0);
    const __nv_bfloat16 h1 = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(h1);
    const __nv_bfloat16 h2 = __float2bfloat16_rn(r2);
    b0 = __bfloat16_as_ushort(h0);
    b1 = __bfloat16_as_ushort(h1);
    b2 = __bfloat16_as_ushort(h2);
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

// tcgen05.ld of 8 columns without the wait: issue several, then tmem_wait_ld()
// once before reading any of them.
__device__ __forceinline__ void tmem_ld8_nowait(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

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

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Sticky bounded wait: after one timeout the caller stops waiting (the status word
// already carries the error) so the kernel ends in bounded time.
__device__ __forceinline__ void wait_ok(bool& ok, uint32_t bar, uint32_t parity, int* status) {
    if (ok) ok = mbar_wait(bar, parity, status);
}

// The same bounded wait, sleeping between tests: for warps whose waits are off the
// critical path (an issuer or a converter running ahead), which would otherwise
// take issue slots from the DP warp on their scheduler while they poll.
__device__ __forceinline__ bool mbar_wait_sleep(uint32_t bar, uint32_t parity, int* status, unsigned ns) {
    if (mbar_test(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_test(bar, parity)) {
        __nanosleep(ns);
        if (global_ns() - t0 > 2000000000ull) {
            atomicOr(status, kStatusTimeout);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ void wait_ok_sleep(bool& ok, uint32_t bar, uint32_t parity, int* status,
                                              unsigned ns = 128) {
    if (ok) ok = mbar_wait_sleep(bar, parity, status, ns);
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int q = 0; q < 32; ++q) v[q] = __uint_as_float(r[q]);
}

__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, int ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t tmem, int ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(ncols) : "memory");
}

__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

}  // namespace tc
}  // namespace sdtw
