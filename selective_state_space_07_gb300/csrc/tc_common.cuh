// Shared helpers of the tcgen05 kernels (kind::f16 products with operands in
// 128-byte-swizzled shared memory and fp32 accumulators in TMEM): operand
// layouts and descriptors, product issue, TMEM loads and stores, fences,
// bf16 packing and a bounded mbarrier wait.
#pragma once
#include "ssm_common.cuh"

namespace ssm {
namespace tc {

// Byte offset of element (row, col) in a K-major, 128-byte-swizzled bf16
// operand of `rows` rows.
__device__ __forceinline__ int swz(int row, int col, int rows) {
    return (col >> 6) * rows * 128 + (row >> 3) * 1024 + (row & 7) * 128 + ((((col >> 3) & 7) ^ (row & 7)) << 4) +
           ((col & 7) << 1);
}

// Shared-memory matrix descriptors, 128-byte swizzle. K-major: 8-row groups
// 1024 bytes apart (SBO), K advancing inside the 128-byte rows. MN-major
// (the operand stored as rows of K, M or N contiguous): the same 1024-byte
// atoms with the roles swapped -- a 128-byte row holds 64 elements of M or
// N, 8 rows of K make an atom; SBO = 1024 between 8-row groups of K, LBO =
// 8192 between the 64-element blocks of M or N. That is the image
// swz(k, mn, 64) writes, and what a 128-byte-swizzled TMA box of 64 columns
// x 64 rows lands as.
__device__ __forceinline__ uint64_t desc_sw128(unsigned addr) {
    return (uint64_t)((addr >> 4) & 0x3FFFu) | (1ull << 16) | ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) |
           (2ull << 61);
}
__device__ __forceinline__ uint64_t desc_sw128_mn(unsigned addr) {
    return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)(8192 >> 4) << 16) | ((uint64_t)(1024 >> 4) << 32) |
           (1ull << 46) | (2ull << 61);
}

// kind::f16 instruction descriptor: fp32 accumulator, bf16 A and B, M = 128,
// N = n; A and B K-major unless a_mn / b_mn (bits 15 / 16: MN-major).
__host__ __device__ constexpr uint32_t idesc_m128(int n, bool a_mn = false, bool b_mn = false) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
           ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

// D[128 x n] (+)= A[128 x kdim] B[kdim x n]. A K-major (128 rows) or, with
// a_mn, MN-major (the swz(k, m, 64) image); B K-major with its 64-wide K
// atoms laid out for b_rows rows or, with b_mn, MN-major (swz(k, n, 64)).
__device__ __forceinline__ void mma_issue(unsigned d_tmem, unsigned a, unsigned b, int b_rows, int n, int kdim,
                                          bool accumulate, bool a_mn = false, bool b_mn = false) {
    const uint32_t id = idesc_m128(n, a_mn, b_mn);
    for (int j = 0; j < kdim / 16; ++j) {  // K = 16 per instruction
        // K-major: atom j/4, 32-byte step j%4; MN-major: two 8-row K groups per step
        const uint64_t ad = a_mn ? desc_sw128_mn(a + j * 2048) : desc_sw128(a + (j >> 2) * 128 * 128 + (j & 3) * 32);
        const uint64_t bd = b_mn ? desc_sw128_mn(b + j * 2048) : desc_sw128(b + (j >> 2) * b_rows * 128 + (j & 3) * 32);
        const unsigned acc = (accumulate || j > 0) ? 1u : 0u;
        asm volatile(
            "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
            " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
            "l"(ad), "l"(bd), "r"(id), "r"(acc)
            : "memory");
    }
}

__device__ __forceinline__ void tmem_ld32(unsigned taddr, float* v) {
    unsigned r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 / 16 consecutive columns of this warp's 32 TMEM lanes without waiting:
// the registers are valid after tmem_wait_ld(), so several loads can be in flight.
__device__ __forceinline__ void tmem_ld32_nw(unsigned taddr, unsigned* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld16_nw(unsigned taddr, unsigned* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }
// After tmem_wait_ld(): ties n registers of a no-wait load to the wait, so no use moves above it.
template <int N> __device__ __forceinline__ void tmem_regs_ready(unsigned* r) {
#pragma unroll
    for (int i = 0; i < N; ++i) asm volatile("" : "+r"(r[i]));
}

// Two consecutive columns of this warp's 32 TMEM lanes (one value per lane each).
__device__ __forceinline__ void tmem_ld2(unsigned taddr, float* v) {
    unsigned r0, r1;
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x2.b32 {%0,%1}, [%2];\n" : "=r"(r0), "=r"(r1) : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
    v[0] = __uint_as_float(r0);
    v[1] = __uint_as_float(r1);
}

__device__ __forceinline__ void tmem_st32(unsigned taddr, const float* v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
        "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
        "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
        "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
        "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
        : "memory");
}

__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }
__device__ __forceinline__ void tc_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void tc_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }

__device__ __forceinline__ unsigned pack_bf2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<unsigned*>(&h);
}
// 8 consecutive bf16 of a K-major swizzled row (one 16-byte chunk): col % 8 == 0.
__device__ __forceinline__ void st8(char* base, int row, int col, int rows, const float* v) {
    *reinterpret_cast<uint4*>(base + swz(row, col, rows)) =
        make_uint4(pack_bf2(v[0], v[1]), pack_bf2(v[2], v[3]), pack_bf2(v[4], v[5]), pack_bf2(v[6], v[7]));
}
__device__ __forceinline__ void st1(char* base, int row, int col, int rows, float v) {
    *reinterpret_cast<__nv_bfloat16*>(base + swz(row, col, rows)) = __float2bfloat16_rn(v);
}
// two consecutive bf16 (col even) of a K-major swizzled row
__device__ __forceinline__ void st2(char* base, int row, int col, int rows, float a, float b) {
    *reinterpret_cast<unsigned*>(base + swz(row, col, rows)) = pack_bf2(a, b);
}
__device__ __forceinline__ void unpack8(uint4 u, float* f) {
    const unsigned w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}
__device__ __forceinline__ void ld8(const char* base, int row, int col, int rows, float* f) {
    unpack8(*reinterpret_cast<const uint4*>(base + swz(row, col, rows)), f);
}


// Wait until phase `parity` of the barrier completes (mbarrier.try_wait,
// which suspends the thread for a while in hardware between checks), at most
// limit_ns; returns whether it completed.
__device__ __forceinline__ bool mbar_try(unsigned bar, unsigned parity) {
    unsigned done = 0;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}
__device__ __forceinline__ bool mbar_wait_try(unsigned bar, unsigned parity, unsigned long long limit_ns) {
    if (mbar_try(bar, parity)) return true;  // the usual case: no clock read
    const unsigned long long t0 = global_ns();
    while (true) {
        if (mbar_try(bar, parity)) return true;
        if (global_ns() - t0 > limit_ns) return false;
    }
}

}  // namespace tc
}  // namespace ssm
