// Device-side building blocks shared by the forward, backward and step
// kernels of the S6 selective scan (sm_103a).
//
// Scan definition (rustytorch commit log, "MambaBlock" S6 forward commit):
//   Delta = softplus(dt + dt_bias); a = exp(Delta*A[d,n]);
//   h = a*h + (Delta*x)*Bm[t,n];  y = (sum_n Cm[t,n]*h + D*x) * silu(z).
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ssm_internal.h"

namespace ssm {

constexpr int kN = 16;         // d_state supported by the kernels
constexpr int kCK = 16;        // tokens per staged forward tile
constexpr int kCkpt = 8;       // tokens between saved forward states (backward chunk)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;

__host__ __device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }

// ------------------------------------------------------------ MUFU wrappers
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// 2^x without the MUFU (XU) pipe, for a kernel whose XU pipe binds: a
// Cody-Waite split x = n + f, n = x rounded to the nearest integer by adding
// and subtracting 1.5 * 2^23 (exact for |x| < 2^22; f = x - n in [-0.5, 0.5]
// is exact too), 2^f by the degree-6 polynomial that interpolates it at the
// Chebyshev nodes of [-0.5, 0.5] (coefficients from csrc/exp2_poly.py;
// largest relative error 1.1e-7 in float32), and n added to the exponent
// field: the shifted sum's bits hold 0x4B400000 + n, whose low nine bits
// shifted up by 23 are n << 23 (mod 2^32). 13 instructions on the FMA and ALU
// pipes. Arguments below -125.5 give 0 (the result would not be a normal
// number: flushed as ex2.approx.ftz flushes); arguments must be <= 127.
__device__ __forceinline__ float ex2_fma(float x) {
    const float xc = fmaxf(x, -127.f);
    const float sh = __fadd_rn(xc, 12582912.f);
    const float f = __fsub_rn(xc, __fsub_rn(sh, 12582912.f));
    float p = 1.5461444854736328e-4f;
    p = __fmaf_rn(p, f, 1.3400427997112274e-3f);
    p = __fmaf_rn(p, f, 9.618056938052177e-3f);
    p = __fmaf_rn(p, f, 5.550327152013779e-2f);
    p = __fmaf_rn(p, f, 2.4022650718688965e-1f);
    p = __fmaf_rn(p, f, 6.931471824645996e-1f);
    p = __fmaf_rn(p, f, 1.0f);
    const float r = __int_as_float((int)((unsigned)__float_as_int(sh) * (1u << 23) + (unsigned)__float_as_int(p)));
    return xc < -125.5f ? 0.f : r;
}
__device__ __forceinline__ float lg2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ------------------------------------------------------------ I/O types
template <typename IO> struct IOT;
template <> struct IOT<float> {
    // fp32 I/O: per-token helpers call CUDA's full-precision expf/log1pf and
    // use IEEE division.
    static constexpr bool kFast = false;
    __device__ static float to_f(float v) { return v; }
    __device__ static float from_f(float v) { return v; }
};
template <> struct IOT<__nv_bfloat16> {
    // bf16 I/O: outputs carry 8 significant bits, so the per-token helpers
    // use the MUFU forms (relative error ~1e-6 or better where it matters).
    static constexpr bool kFast = true;
    __device__ static float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
    __device__ static __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
};

// ------------------------------------------------------------ per-token math
// softplus(v) = max(v,0) + log1p(exp(-|v|)) ("numerically-stable softplus").
// Also returns sigmoid(v), which the backward needs for d(dt). Every
// rounding step is explicit so that each kernel that inlines these helpers
// gets the same bits (the compiler may not contract them differently).
template <bool FAST>
__device__ __forceinline__ float softplus_sig(float v, float* sig) {
    if (FAST) {
        const float e = ex2(__fmul_rn(-fabsf(v), kLog2e));  // exp(-|v|) in (0, 1]
        const float w = __fadd_rn(1.0f, e);
        if (sig) {
            const float r = rcp(w);
            *sig = v >= 0.0f ? r : __fmul_rn(e, r);
        }
        return __fmaf_rn(kLn2, lg2(w), fmaxf(v, 0.0f));
    } else {
        const float e = expf(-fabsf(v));
        const float w = __fadd_rn(1.0f, e);
        if (sig) *sig = v >= 0.0f ? __fdiv_rn(1.0f, w) : __fdiv_rn(e, w);
        return __fadd_rn(fmaxf(v, 0.0f), log1pf(e));
    }
}
template <bool FAST> __device__ __forceinline__ float softplus(float v) {
    return softplus_sig<FAST>(v, nullptr);
}
// Logistic sigmoid; exp(-z) may overflow to +inf for very negative z,
// which gives 1/inf = 0 as required.
template <bool FAST> __device__ __forceinline__ float sigmoid(float z) {
    if (FAST) return rcp(__fadd_rn(1.0f, ex2(__fmul_rn(-z, kLog2e))));
    return __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-z)));
}
// Delta of one token.
template <bool FAST>
__device__ __forceinline__ float token_delta(float dtv, float bias, bool sp) {
    const float v = __fadd_rn(dtv, bias);
    return sp ? softplus<FAST>(v) : v;
}

// ------------------------------------------------------------ cp.async staging
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool valid) {
    unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    int n = valid ? 16 : 0;  // 0 source bytes => the 16 destination bytes are zero-filled
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(n)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N> __device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// Stage a [rows x chunks*16 bytes] block whose rows are `gstride` bytes
// apart in global memory into shared memory rows `sstride` bytes apart.
// Rows >= valid_rows and chunks >= valid_chunks are zero-filled (their
// global address is never formed).
template <int NT>
__device__ __forceinline__ void stage_block(char* sdst, int sstride, const char* gsrc, int64_t gstride,
                                            int rows, int chunks, int valid_rows, int valid_chunks) {
    for (int idx = threadIdx.x; idx < rows * chunks; idx += NT) {
        const int r = idx / chunks, ch = idx - r * chunks;
        const bool v = r < valid_rows && ch < valid_chunks;
        const char* src = v ? gsrc + (int64_t)r * gstride + ch * 16 : gsrc;
        cp_async16(sdst + r * sstride + ch * 16, src, v);
    }
}

__device__ __forceinline__ void red_add_v4(float* gptr, float4 v) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};\n" ::"l"(gptr), "f"(v.x), "f"(v.y),
                 "f"(v.z), "f"(v.w)
                 : "memory");
}

// y for one token from the channel's full readout p (lanes combined).
template <bool FAST>
__device__ __forceinline__ float gate_out(float p, float Dd, float xv, float zv, bool has_z) {
    const float pp = __fmaf_rn(Dd, xv, p);
    if (!has_z) return pp;
    return __fmul_rn(pp, __fmul_rn(zv, sigmoid<FAST>(zv)));
}

// ------------------------------------------------------------ channel-pair (f32x2) forms
// The same roundings as the scalar helpers above, applied to two channels at
// once with packed fp32 instructions (each half of a packed add, multiply or
// fused multiply-add rounds exactly as the scalar instruction does), so a
// kernel using these and one using the scalar forms get identical bits.
__device__ __forceinline__ float2 pk(float a, float b) { return make_float2(a, b); }

template <bool FAST>
__device__ __forceinline__ float2 delta2(float2 dtv, float2 bias, bool sp) {
    const float2 v = __fadd2_rn(dtv, bias);
    if (!sp) return v;
    if (FAST) {
        const float2 arg = __fmul2_rn(pk(-fabsf(v.x), -fabsf(v.y)), pk(kLog2e, kLog2e));
        const float2 w = __fadd2_rn(pk(1.0f, 1.0f), pk(ex2(arg.x), ex2(arg.y)));
        return __ffma2_rn(pk(kLn2, kLn2), pk(lg2(w.x), lg2(w.y)), pk(fmaxf(v.x, 0.0f), fmaxf(v.y, 0.0f)));
    }
    return pk(softplus<false>(v.x), softplus<false>(v.y));
}
// Delta and sigmoid(dt + bias) of two channels (the backward's d(dt) factor).
template <bool FAST>
__device__ __forceinline__ float2 delta_sig2(float2 dtv, float2 bias, bool sp, float2* sig) {
    const float2 v = __fadd2_rn(dtv, bias);
    if (!sp) {
        *sig = pk(1.0f, 1.0f);
        return v;
    }
    if (FAST) {
        const float2 arg = __fmul2_rn(pk(-fabsf(v.x), -fabsf(v.y)), pk(kLog2e, kLog2e));
        const float2 e = pk(ex2(arg.x), ex2(arg.y));
        const float2 w = __fadd2_rn(pk(1.0f, 1.0f), e);
        const float2 r = pk(rcp(w.x), rcp(w.y));
        const float2 er = __fmul2_rn(e, r);
        *sig = pk(v.x >= 0.0f ? r.x : er.x, v.y >= 0.0f ? r.y : er.y);
        return __ffma2_rn(pk(kLn2, kLn2), pk(lg2(w.x), lg2(w.y)), pk(fmaxf(v.x, 0.0f), fmaxf(v.y, 0.0f)));
    }
    float s0, s1;
    const float d0 = softplus_sig<false>(v.x, &s0), d1 = softplus_sig<false>(v.y, &s1);
    *sig = pk(s0, s1);
    return pk(d0, d1);
}
template <bool FAST> __device__ __forceinline__ float2 sigmoid2(float2 z) {
    if (FAST) {
        const float2 arg = __fmul2_rn(pk(-z.x, -z.y), pk(kLog2e, kLog2e));
        const float2 w = __fadd2_rn(pk(1.0f, 1.0f), pk(ex2(arg.x), ex2(arg.y)));
        return pk(rcp(w.x), rcp(w.y));
    }
    return pk(sigmoid<false>(z.x), sigmoid<false>(z.y));
}

// Two adjacent channels of a staged row (byte offset `off`) as fp32, and the
// store of two adjacent outputs in the I/O dtype.
template <typename IO> __device__ __forceinline__ float2 ld2(const char* p);
template <> __device__ __forceinline__ float2 ld2<float>(const char* p) { return *reinterpret_cast<const float2*>(p); }
template <> __device__ __forceinline__ float2 ld2<__nv_bfloat16>(const char* p) {
    const unsigned w = *reinterpret_cast<const unsigned*>(p);  // low half: the first channel
    return pk(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
template <typename IO> __device__ __forceinline__ void st2(IO* p, float2 v);
template <> __device__ __forceinline__ void st2<float>(float* p, float2 v) { *reinterpret_cast<float2*>(p) = v; }
template <> __device__ __forceinline__ void st2<__nv_bfloat16>(__nv_bfloat16* p, float2 v) {
    *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(v.x, v.y);
}

__device__ __forceinline__ void flag_nonfinite(unsigned* status, float acc) {
    // acc accumulates y*0 over the outputs: 0 unless one of them was Inf/NaN.
    const bool bad = !(acc == 0.0f);
    if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0 && status) atomicOr(status, kStatusNonFinite);
}


// ------------------------------------------------------------ mbarriers and TMA
__device__ __forceinline__ unsigned smem_u32(const void* p) { return (unsigned)__cvta_generic_to_shared(p); }
constexpr unsigned long long kWaitNs = 1000000000ull;  // 1 s: how long a thread waits on an mbarrier

__device__ __forceinline__ void mbar_init(unsigned bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory"); }
__device__ __forceinline__ void mbar_expect_tx(unsigned bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_test(unsigned bar, unsigned parity) {
    unsigned ok = 0;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
    return t;
}
// Wait (non-blocking polls with a short sleep) until phase `parity` of the
// barrier completes or `limit_ns` have passed; returns whether it completed.
__device__ __forceinline__ bool mbar_wait_bounded(unsigned bar, unsigned parity,
                                                  unsigned long long limit_ns = kWaitNs) {
    if (mbar_test(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_test(bar, parity)) {
        if (global_ns() - t0 > limit_ns) return false;
        __nanosleep(32);
    }
    return true;
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, unsigned bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}


}  // namespace ssm
