// Backward (reverse-time) pass of the S6 selective scan on sm_103a.
//
// The analytic VJP of the rustytorch "MambaBlock" commits ("reverse-time
// recurrence over the cached h trajectory ... summed over the batch"), for
// loss = <dy, y> + <dh_last, h_last>. Per (b, d) channel and state n:
//   p_t  = sum_n C h_t + D x_t,   dp_t = dy_t * silu(z_t),
//   dz_t = dy_t * p_t * silu'(z_t)
//   G_t  = a_{t+1} G_{t+1} + dp_t C_t        (adjoint of h_t; G_{L-1} += dh_last)
//   dx_t = dp_t D + Delta_t sum_n G B
//   dDelta_t = sum_n G (B x_t + A a_t h_{t-1}),  d(dt)_t = dDelta_t * sigmoid(dt_t + dt_bias)
//   dA  += Delta_t G a_t h_{t-1}   (over b, t)      dD += dp_t x_t
//   dB[b,t,n] += G u_t,  dC[b,t,n] += dp_t h_t      (over d)
//
// Work split: a CTA owns CH channels x one L-group and walks the group's
// 16-token sub-chunks from last to first. For each sub-chunk it restarts
// the forward from the checkpoint the forward pass saved, one state at a
// time: the 16 values of a_t and h_t of that state live in registers, the
// reverse recurrence runs over them at once, and the per-token sums over
// states (sum G B, sum A G a h, sum C h) accumulate in registers. dB / dC
// contributions go through a per-warp shared-memory transpose (channel
// reduction), then a per-CTA sum over warps, then one vector atomic per
// 4 outputs. dA, dD, d_dt_bias accumulate in registers over the whole
// group and leave with one atomic each.
#include "ssm_common.cuh"
#include "ssm_internal.h"

namespace ssm {

namespace {

template <typename IO, int NSPLIT> struct BwdLayout {
    static constexpr int NT = kBwdThreads;
    static constexpr int NW = NT / 32;
    static constexpr int CH = NT / NSPLIT;
    static constexpr int NS = kN / NSPLIT;
    static constexpr int ES = sizeof(IO);
    // tokens per recompute pass: the whole 16-token sub-chunk, or (with 4
    // lanes per channel, where registers are capped at 128) two halves
    static constexpr int HALF = NSPLIT >= 4 ? kCK / 2 : kCK;
    static constexpr int NH = kCK / HALF;                      // passes per sub-chunk
    static constexpr int SPR = kCK / HALF;                     // states per transpose reduction
    static constexpr int XROW = CH * ES + 16;
    static constexpr int DTROW = CH * 4 + 16;
    static constexpr int BCROW = kN * ES;
    static constexpr int OFF_X = 0;
    static constexpr int OFF_Z = OFF_X + kCK * XROW;
    static constexpr int OFF_DY = OFF_Z + kCK * XROW;
    static constexpr int OFF_DT = OFF_DY + kCK * XROW;
    static constexpr int OFF_B = OFF_DT + kCK * DTROW;
    static constexpr int OFF_C = OFF_B + kCK * BCROW;
    static constexpr int OFF_H = OFF_C + kCK * BCROW;         // checkpoint tile [CH][16] fp32
    static constexpr int STAGE = OFF_H + CH * kN * 4;
    static constexpr int OFF_T = 2 * STAGE;                    // per-token [5][16 tokens][CH] fp32
    static constexpr int NTOK = 5;                             // Delta, u, dp, sigmoid(v), dy*silu'(z)
    static constexpr int SMEM = OFF_T + NTOK * kCK * CH * 4;   // dynamic shared memory
    static constexpr int WROW = 36;                            // floats per lane row of the transpose buffer
    static constexpr int WFLOATS = NW * 32 * WROW;
    static constexpr int SFLOATS = 3 * HALF * CH * NSPLIT;     // lane partial state sums [3][8][CH][NSPLIT]
    static constexpr int UFLOATS = WFLOATS > SFLOATS ? WFLOATS : SFLOATS;
    static constexpr int MINB = NSPLIT == 4 ? 4 : (NSPLIT == 2 ? 2 : 1);
};

__device__ __forceinline__ float2 f2(float a, float b) { return make_float2(a, b); }

// One CTA: CH channels of one batch row over one L-group; lane k of a
// channel owns states k, k+NSPLIT, ... Each 16-token sub-chunk (walked from
// last to first) is processed in NH passes of HALF tokens, last pass first:
//   A  per (token, channel): Delta, u, dp, sigmoid(v), dy*silu'(z); B/C^T
//   P1 (two passes only) per lane: each state's forward over the first half
//      from the checkpoint, giving the state at the middle of the sub-chunk
//   C  per pass, per state: forward over the pass (a, h in registers), then
//      the reverse E_t = a_{t+1} E_{t+1} + dp_t C_t; dB/dC contributions go
//      through a per-warp transpose every SPR states; per-token state sums
//      accumulate in registers and leave through shared memory
//   E  per (token, channel) of the pass: dx, dz, d(dt) in place, dD and
//      d_dt_bias partials; dB/dC of the pass leave as vector atomics
template <typename IO, int NSPLIT>
__global__ void __launch_bounds__(kBwdThreads, BwdLayout<IO, NSPLIT>::MINB) ssm_bwd_kernel(const BwdParams p) {
    using Ly = BwdLayout<IO, NSPLIT>;
    constexpr int NT = Ly::NT, CH = Ly::CH, NS = Ly::NS, ES = Ly::ES, HALF = Ly::HALF, NH = Ly::NH, SPR = Ly::SPR;
    constexpr bool FAST = IOT<IO>::kFast;
    extern __shared__ __align__(16) char smem[];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = tid / NSPLIT, k = tid % NSPLIT;   // scan role: channel c, states k, k+NSPLIT, ...
    const int ce = tid % CH;                         // per-token role: channel ce
    const int64_t D = p.D, L = p.L;
    const int64_t d0 = (int64_t)blockIdx.x * CH, d = d0 + c, de = d0 + ce;
    const bool dv = d < D, dve = de < D;
    const int g = blockIdx.y;
    const int64_t b = blockIdx.z;
    const int64_t tb0 = (int64_t)g * p.Lg;
    const int64_t tb1 = min64(L, tb0 + p.Lg);
    const int nsub = (int)((tb1 - tb0 + kCK - 1) / kCK);
    const int64_t nck = (L + kCK - 1) / kCK;
    const bool has_z = p.has_z != 0, sp = p.sp != 0;

    float Gc[NS], dAacc[NS];
    const float* Arow = p.A + (dv ? d : 0) * kN;
#pragma unroll
    for (int j = 0; j < NS; ++j) {
        const int n = k + NSPLIT * j;
        float gi = 0.f;
        if (dv && p.gstart)
            gi = p.G == 1 ? p.gstart[(b * D + d) * kN + n] : p.gstart[((b * p.G + g) * D + d) * kN + n];
        Gc[j] = gi;
        dAacc[j] = 0.f;
    }
    const float Dde = (dve && p.Dskip) ? p.Dskip[de] : 0.f;
    const float biase = (dve && p.dt_bias) ? p.dt_bias[de] : 0.f;
    float dDacc = 0.f, dbacc = 0.f, nf = 0.f;

    const int vchx = (int)(min64(CH, D - d0) * ES / 16);
    const int vchd = (int)(min64(CH, D - d0) * 4 / 16);
    const int vchh = (int)(min64(CH, D - d0) * kN * 4 / 16);
    auto issue = [&](int s, char* st) {
        const int64_t t0 = tb0 + (int64_t)s * kCK;
        const int rows = (int)min64(kCK, tb1 - t0);
        const int64_t row0 = b * L + t0;
        stage_block<NT>(st + Ly::OFF_X, Ly::XROW, (const char*)p.x + (row0 * D + d0) * ES, D * ES, kCK,
                        CH * ES / 16, rows, vchx);
        if (has_z)
            stage_block<NT>(st + Ly::OFF_Z, Ly::XROW, (const char*)p.z + (row0 * D + d0) * ES, D * ES, kCK,
                            CH * ES / 16, rows, vchx);
        stage_block<NT>(st + Ly::OFF_DY, Ly::XROW, (const char*)p.dy + (row0 * D + d0) * ES, D * ES, kCK,
                        CH * ES / 16, rows, vchx);
        stage_block<NT>(st + Ly::OFF_DT, Ly::DTROW, (const char*)p.dt + (row0 * D + d0) * 4, D * 4, kCK,
                        CH * 4 / 16, rows, vchd);
        stage_block<NT>(st + Ly::OFF_B, Ly::BCROW, (const char*)p.Bm + row0 * kN * ES, kN * ES, kCK,
                        Ly::BCROW / 16, rows, Ly::BCROW / 16);
        stage_block<NT>(st + Ly::OFF_C, Ly::BCROW, (const char*)p.Cm + row0 * kN * ES, kN * ES, kCK,
                        Ly::BCROW / 16, rows, Ly::BCROW / 16);
        stage_block<NT>(st + Ly::OFF_H, CH * kN * 4, (const char*)(p.ckpt + ((b * nck + t0 / kCK) * D + d0) * kN),
                        CH * kN * 4, 1, CH * kN * 4 / 16, 1, vchh);
        cp_async_commit();
    };

    // B^T / C^T tiles, the transpose buffer (reused for the lane partial
    // state sums), and the per-warp reduced outputs are separate shared
    // objects so the compiler can reorder loads from one across stores to
    // another.
    __shared__ __align__(16) float BT[kN * kCK];                // [16 states][16 tokens]
    __shared__ __align__(16) float CT[kN * kCK];
    __shared__ __align__(16) float WU[Ly::UFLOATS];
    __shared__ __align__(16) float wo[Ly::NW * 2 * kN * HALF];  // [NW][2][16 states][8 tokens]
    float* TL = reinterpret_cast<float*>(smem + Ly::OFF_T);   // [5][16][CH]
    float* wb = WU + warp * 32 * Ly::WROW;
    float* SS = WU;                                            // [3][8][CH][NSPLIT]
    constexpr int TS = kCK * CH;                              // stride between the per-token arrays

    if (nsub > 0) issue(nsub - 1, smem);
    for (int it = 0; it < nsub; ++it) {
        const int s = nsub - 1 - it;
        char* st = smem + (it & 1) * Ly::STAGE;
        if (s > 0) {
            issue(s - 1, smem + ((it + 1) & 1) * Ly::STAGE);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const int64_t t0 = tb0 + (int64_t)s * kCK;
        const int rows = (int)min64(kCK, tb1 - t0);

        // ---- A: B/C to fp32 (transposed), per-token quantities once per (token, channel)
        {
            const IO* Braw = reinterpret_cast<const IO*>(st + Ly::OFF_B);
            const IO* Craw = reinterpret_cast<const IO*>(st + Ly::OFF_C);
            for (int i = tid; i < kCK * kN; i += NT) {
                const int n = i / kCK, tok = i % kCK;
                BT[i] = IOT<IO>::to_f(Braw[tok * kN + n]);
                CT[i] = IOT<IO>::to_f(Craw[tok * kN + n]);
            }
#pragma unroll
            for (int r = 0; r < kCK * CH / NT; ++r) {
                const int t = tid / CH + (NT / CH) * r;
                const float xv = IOT<IO>::to_f(reinterpret_cast<const IO*>(st + Ly::OFF_X + t * Ly::XROW)[ce]);
                const float dyv = IOT<IO>::to_f(reinterpret_cast<const IO*>(st + Ly::OFF_DY + t * Ly::XROW)[ce]);
                const float v = __fadd_rn(reinterpret_cast<const float*>(st + Ly::OFF_DT + t * Ly::DTROW)[ce], biase);
                float sg = 1.f, delta = v;
                if (sp) delta = softplus_sig<FAST>(v, &sg);
                float dpv = dyv, dyds = 0.f;
                if (has_z) {
                    const float zv = IOT<IO>::to_f(reinterpret_cast<const IO*>(st + Ly::OFF_Z + t * Ly::XROW)[ce]);
                    const float sz = sigmoid<FAST>(zv);
                    dpv = __fmul_rn(dyv, __fmul_rn(zv, sz));
                    dyds = dyv * (sz * (1.0f + zv * (1.0f - sz)));
                }
                const bool live = t < rows;  // tokens past the end act as identity (a = 1, no input)
                TL[0 * TS + t * CH + ce] = live ? delta : 0.f;
                TL[1 * TS + t * CH + ce] = live ? __fmul_rn(delta, xv) : 0.f;
                TL[2 * TS + t * CH + ce] = live ? dpv : 0.f;
                TL[3 * TS + t * CH + ce] = sg;
                TL[4 * TS + t * CH + ce] = dyds;
            }
        }
        __syncthreads();
        const float* hck = reinterpret_cast<const float*>(st + Ly::OFF_H) + c * kN;

        // ---- P1: the state at the middle of the sub-chunk, per lane state
        float hmid[NS];
        if constexpr (NH == 2) {
            float2 Dl[HALF / 2], Ul[HALF / 2];
#pragma unroll
            for (int m = 0; m < HALF / 2; ++m) {
                Dl[m] = f2(TL[0 * TS + (2 * m) * CH + c], TL[0 * TS + (2 * m + 1) * CH + c]);
                Ul[m] = f2(TL[1 * TS + (2 * m) * CH + c], TL[1 * TS + (2 * m + 1) * CH + c]);
            }
#pragma unroll
            for (int j = 0; j < NS; ++j) {
                const int n = k + NSPLIT * j;
                const float A2 = __fmul_rn(dv ? __ldg(Arow + n) : 0.f, kLog2e);
                const float2 A2p = f2(A2, A2);
                float hp = hck[n];
#pragma unroll
                for (int q = 0; q < HALF / 4; ++q) {
                    const float4 b4 = *reinterpret_cast<const float4*>(BT + n * kCK + 4 * q);
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        const int m = 2 * q + h2;
                        const float2 bb = h2 ? f2(b4.z, b4.w) : f2(b4.x, b4.y);
                        const float2 arg = __fmul2_rn(Dl[m], A2p);
                        const float2 ub = __fmul2_rn(Ul[m], bb);
                        hp = __fmaf_rn(ex2(arg.x), hp, ub.x);
                        hp = __fmaf_rn(ex2(arg.y), hp, ub.y);
                    }
                }
                hmid[j] = hp;
            }
        }

#pragma unroll
        for (int half = NH - 1; half >= 0; --half) {
            const int i0 = HALF * half;
            float2 Dl[HALF / 2], Ul[HALF / 2], Pl[HALF / 2];
#pragma unroll
            for (int m = 0; m < HALF / 2; ++m) {
                const int ta = i0 + 2 * m;
                Dl[m] = f2(TL[0 * TS + ta * CH + c], TL[0 * TS + (ta + 1) * CH + c]);
                Ul[m] = f2(TL[1 * TS + ta * CH + c], TL[1 * TS + (ta + 1) * CH + c]);
                Pl[m] = f2(TL[2 * TS + ta * CH + c], TL[2 * TS + (ta + 1) * CH + c]);
            }
            float2 S1[HALF / 2], S2[HALF / 2], S3[HALF / 2];
#pragma unroll
            for (int m = 0; m < HALF / 2; ++m) S1[m] = S2[m] = S3[m] = f2(0.f, 0.f);

#pragma unroll
            for (int j = 0; j < NS; ++j) {
                const int n = k + NSPLIT * j;
                const float* Bn = BT + n * kCK + i0;
                const float* Cn = CT + n * kCK + i0;
                const float An = dv ? __ldg(Arow + n) : 0.f;
                const float A2 = __fmul_rn(An, kLog2e);
                const float2 A2p = f2(A2, A2), Ap = f2(An, An);
                float2 a[HALF / 2], hh[HALF / 2];
                float hp = (NH == 2 && half == 1) ? hmid[j] : hck[n];
#pragma unroll
                for (int q = 0; q < HALF / 4; ++q) {
                    const float4 b4 = *reinterpret_cast<const float4*>(Bn + 4 * q);
                    const float4 c4 = *reinterpret_cast<const float4*>(Cn + 4 * q);
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        const int m = 2 * q + h2;
                        const float2 bb = h2 ? f2(b4.z, b4.w) : f2(b4.x, b4.y);
                        const float2 cc = h2 ? f2(c4.z, c4.w) : f2(c4.x, c4.y);
                        const float2 arg = __fmul2_rn(Dl[m], A2p);
                        a[m] = f2(ex2(arg.x), ex2(arg.y));
                        const float2 ub = __fmul2_rn(Ul[m], bb);
                        const float h0v = __fmaf_rn(a[m].x, hp, ub.x);
                        const float h1v = __fmaf_rn(a[m].y, h0v, ub.y);
                        hp = h1v;
                        hh[m] = f2(h0v, h1v);
                        S3[m] = __ffma2_rn(cc, hh[m], S3[m]);
                    }
                }
                // adjoint E_t = a_{t+1} E_{t+1} + dp_t C_t; the carry Gc holds a_{t+1} E_{t+1}
                float E = Gc[j];
                float anext = 1.f;
                float dAj = 0.f;
                const int jj = j % SPR;
#pragma unroll
                for (int q = HALF / 4 - 1; q >= 0; --q) {
                    const float4 b4 = *reinterpret_cast<const float4*>(Bn + 4 * q);
                    const float4 c4 = *reinterpret_cast<const float4*>(Cn + 4 * q);
                    float2 vb[2], vc[2];
#pragma unroll
                    for (int h2 = 1; h2 >= 0; --h2) {
                        const int m = 2 * q + h2;
                        const float2 bb = h2 ? f2(b4.z, b4.w) : f2(b4.x, b4.y);
                        const float2 rr = __fmul2_rn(Pl[m], h2 ? f2(c4.z, c4.w) : f2(c4.x, c4.y));
                        const float e1 = __fmaf_rn(anext, E, rr.y);
                        const float e0 = __fmaf_rn(a[m].y, e1, rr.x);
                        E = e0;
                        anext = a[m].x;
                        const float2 E2 = f2(e0, e1);
                        vb[h2] = __fmul2_rn(E2, Ul[m]);
                        vc[h2] = __fmul2_rn(Pl[m], hh[m]);
                        S1[m] = __ffma2_rn(E2, bb, S1[m]);
                        // a_t h_{t-1} = h_t - u_t B_t
                        const float2 qv = __ffma2_rn(f2(-Ul[m].x, -Ul[m].y), bb, hh[m]);
                        const float2 w = __fmul2_rn(E2, qv);
                        const float2 dw = __fmul2_rn(Dl[m], w);
                        dAj = __fadd_rn(dAj, __fadd_rn(dw.x, dw.y));
                        S2[m] = __ffma2_rn(Ap, w, S2[m]);
                    }
                    // row layout per reduction group: [state jj][vb 0..HALF-1 | vc 0..HALF-1]
                    *reinterpret_cast<float4*>(wb + lane * Ly::WROW + jj * 2 * HALF + 4 * q) =
                        make_float4(vb[0].x, vb[0].y, vb[1].x, vb[1].y);
                    *reinterpret_cast<float4*>(wb + lane * Ly::WROW + jj * 2 * HALF + HALF + 4 * q) =
                        make_float4(vc[0].x, vc[0].y, vc[1].x, vc[1].y);
                }
                Gc[j] = __fmul_rn(anext, E);  // carried to the previous half: a_{t_first} E_{t_first}
                dAacc[j] += dAj;
                if (jj == SPR - 1 || j == NS - 1) {
                    __syncwarp();
                    // Sum the transpose buffer over the channel lanes that hold
                    // these states: lane = (quad qd of the 32 values, part kk,
                    // row block hpb); rows (hpb*8 + r)*NSPLIT + kk, r = 0..7.
                    const int qd = lane & 7, rest = lane >> 3, kk = rest % NSPLIT, hpb = rest / NSPLIT;
                    float2 acc0 = f2(0.f, 0.f), acc1 = f2(0.f, 0.f);
#pragma unroll
                    for (int r = 0; r < 8; ++r) {
                        const int row = (hpb * 8 + r) * NSPLIT + kk;
                        const float4 v = *reinterpret_cast<const float4*>(wb + row * Ly::WROW + 4 * qd);
                        acc0 = __fadd2_rn(acc0, f2(v.x, v.y));
                        acc1 = __fadd2_rn(acc1, f2(v.z, v.w));
                    }
#pragma unroll
                    for (int off = 8 * NSPLIT; off < 32; off <<= 1) {
                        acc0.x += __shfl_xor_sync(0xffffffffu, acc0.x, off);
                        acc0.y += __shfl_xor_sync(0xffffffffu, acc0.y, off);
                        acc1.x += __shfl_xor_sync(0xffffffffu, acc1.x, off);
                        acc1.y += __shfl_xor_sync(0xffffffffu, acc1.y, off);
                    }
                    const int sj = qd / (HALF / 2), type = (qd / (HALF / 4)) & 1, iq = (qd % (HALF / 4)) * 4;
                    const int jbase = j - jj;
                    if (hpb == 0 && jbase + sj < NS) {
                        const int nk = kk + NSPLIT * (jbase + sj);
                        *reinterpret_cast<float4*>(wo + ((warp * 2 + type) * kN + nk) * HALF + iq) =
                            make_float4(acc0.x, acc0.y, acc1.x, acc1.y);
                    }
                    __syncwarp();
                }
            }
            __syncthreads();  // every warp is done with its transpose buffer
            // lane partial per-token state sums -> shared memory [3][8][CH][NSPLIT]
#pragma unroll
            for (int m = 0; m < HALF / 2; ++m) {
                SS[((0 * HALF + 2 * m) * CH + c) * NSPLIT + k] = S1[m].x;
                SS[((0 * HALF + 2 * m + 1) * CH + c) * NSPLIT + k] = S1[m].y;
                SS[((1 * HALF + 2 * m) * CH + c) * NSPLIT + k] = S2[m].x;
                SS[((1 * HALF + 2 * m + 1) * CH + c) * NSPLIT + k] = S2[m].y;
                SS[((2 * HALF + 2 * m) * CH + c) * NSPLIT + k] = S3[m].x;
                SS[((2 * HALF + 2 * m + 1) * CH + c) * NSPLIT + k] = S3[m].y;
            }
            __syncthreads();

            // ---- E: per-token outputs of the half, written in place into the staged tiles
#pragma unroll
            for (int r = 0; r < HALF * CH / NT; ++r) {
                const int ti = tid / CH + (NT / CH) * r;  // 0..7 within the half
                const int t = i0 + ti;
                if (t < rows) {
                    IO* xs = reinterpret_cast<IO*>(st + Ly::OFF_X + t * Ly::XROW);
                    IO* zs = reinterpret_cast<IO*>(st + Ly::OFF_Z + t * Ly::XROW);
                    IO* dys = reinterpret_cast<IO*>(st + Ly::OFF_DY + t * Ly::XROW);
                    float* dts = reinterpret_cast<float*>(st + Ly::OFF_DT + t * Ly::DTROW);
                    const float xv = IOT<IO>::to_f(xs[ce]);
                    const float delta = TL[0 * TS + t * CH + ce], dpv = TL[2 * TS + t * CH + ce];
                    const float sg = TL[3 * TS + t * CH + ce], dyds = TL[4 * TS + t * CH + ce];
                    float s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
                    for (int kk = 0; kk < NSPLIT; ++kk) {
                        s1 += SS[((0 * HALF + ti) * CH + ce) * NSPLIT + kk];
                        s2 += SS[((1 * HALF + ti) * CH + ce) * NSPLIT + kk];
                        s3 += SS[((2 * HALF + ti) * CH + ce) * NSPLIT + kk];
                    }
                    if (has_z) {
                        const float dzv = __fmaf_rn(Dde, xv, s3) * dyds;
                        nf = __fmaf_rn(dzv, 0.0f, nf);
                        zs[ce] = IOT<IO>::from_f(dzv);
                    }
                    const float dxv = __fmaf_rn(dpv, Dde, delta * s1);
                    const float ddelta = __fmaf_rn(xv, s1, s2);
                    const float ddtv = sp ? ddelta * sg : ddelta;
                    dDacc = __fmaf_rn(dpv, xv, dDacc);
                    dbacc += ddtv;
                    nf = __fmaf_rn(dxv, 0.0f, nf);
                    nf = __fmaf_rn(ddtv, 0.0f, nf);
                    dys[ce] = IOT<IO>::from_f(dxv);
                    dts[ce] = ddtv;
                }
            }
            // dB / dC of the half: sum the warps, one vector atomic per 4 outputs
            for (int o = tid; o < 2 * HALF * (kN / 4); o += NT) {
                const int type = o / (HALF * kN / 4), rem = o % (HALF * kN / 4);
                const int n0 = (rem / HALF) * 4, ti = rem % HALF;
                if (i0 + ti < rows) {
                    float4 s4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int w = 0; w < Ly::NW; ++w) {
                        const float* src = wo + ((w * 2 + type) * kN + n0) * HALF + ti;
                        s4.x += src[0]; s4.y += src[HALF]; s4.z += src[2 * HALF]; s4.w += src[3 * HALF];
                    }
                    float* dst = (type == 0 ? p.dB : p.dC) + (b * L + t0 + i0 + ti) * kN + n0;
                    red_add_v4(dst, s4);
                }
            }
            __syncthreads();
        }

        // ---- copy dx, dz, d_dt out
        {
            constexpr int CHX = CH * ES / 16, CHD = CH * 4 / 16;
            for (int i = tid; i < rows * CHX; i += NT) {
                const int r = i / CHX, ch = i - r * CHX;
                if (ch < vchx) {
                    const int64_t off = ((b * L + t0 + r) * D + d0) * ES + ch * 16;
                    *reinterpret_cast<int4*>((char*)p.dx + off) =
                        *reinterpret_cast<const int4*>(st + Ly::OFF_DY + r * Ly::XROW + ch * 16);
                    if (has_z)
                        *reinterpret_cast<int4*>((char*)p.dz + off) =
                            *reinterpret_cast<const int4*>(st + Ly::OFF_Z + r * Ly::XROW + ch * 16);
                }
            }
            for (int i = tid; i < rows * CHD; i += NT) {
                const int r = i / CHD, ch = i - r * CHD;
                if (ch < vchd)
                    *reinterpret_cast<int4*>((char*)p.ddt + ((b * L + t0 + r) * D + d0) * 4 + ch * 16) =
                        *reinterpret_cast<const int4*>(st + Ly::OFF_DT + r * Ly::DTROW + ch * 16);
            }
        }
        __syncthreads();
    }

    // ---- reductions over the group
    if (dv) {
#pragma unroll
        for (int j = 0; j < NS; ++j) atomicAdd(p.dA + d * kN + k + NSPLIT * j, dAacc[j]);
        if (g == 0 && p.dh0) {
#pragma unroll
            for (int j = 0; j < NS; ++j) p.dh0[(b * D + d) * kN + k + NSPLIT * j] = Gc[j];
        }
    }
    if (dve) {
        atomicAdd(p.dD + de, dDacc);
        atomicAdd(p.ddt_bias + de, dbacc);
    }
    flag_nonfinite(p.status, nf);
}

// Chunk aggregate of the reverse recurrence for groups 1..G-1: with the
// adjoint carry set to zero at the group's end, run G <- (G + dp*C)*a back to
// the group's start; publish that value (Q) and the group's sum of Delta.
// The carry entering group g-1 from the right is then
// exp(A*sum Delta_g) * carry_g + Q_g.
template <typename IO, int NSPLIT> constexpr int bwd_agg_smem() {
    constexpr int CH = kBwdThreads / NSPLIT, ES = sizeof(IO);
    constexpr int XROW = CH * ES + 16, DTROW = CH * 4 + 16, BCROW = kN * ES;
    return 2 * (2 * kCK * XROW + kCK * DTROW + kCK * BCROW) + kCK * kN * 4;
}

template <typename IO, int NSPLIT>
__global__ void __launch_bounds__(kBwdThreads) ssm_bwd_agg_kernel(const BwdParams p) {
    constexpr int NT = kBwdThreads, CH = NT / NSPLIT, NS = kN / NSPLIT, ES = sizeof(IO);
    constexpr bool FAST = IOT<IO>::kFast;
    constexpr int XROW = CH * ES + 16, DTROW = CH * 4 + 16, BCROW = kN * ES;
    constexpr int OFF_Z = 0, OFF_DY = kCK * XROW, OFF_DT = 2 * kCK * XROW, OFF_C = OFF_DT + kCK * DTROW;
    constexpr int STAGE = OFF_C + kCK * BCROW;
    extern __shared__ __align__(16) char smem[];
    float* Cf = reinterpret_cast<float*>(smem + 2 * STAGE);

    const int tid = threadIdx.x, lane = tid & 31, c = tid / NSPLIT, k = tid % NSPLIT;
    const int base = lane & ~(NSPLIT - 1);
    const int64_t D = p.D, L = p.L;
    const int64_t d0 = (int64_t)blockIdx.x * CH, d = d0 + c;
    const bool dv = d < D;
    const int g = blockIdx.y + 1;  // groups 1..G-1
    const int64_t b = blockIdx.z;
    const int64_t tb0 = (int64_t)g * p.Lg, tb1 = min64(L, tb0 + p.Lg);
    const int ntile = (int)((tb1 - tb0 + kCK - 1) / kCK);
    const bool has_z = p.has_z != 0, sp = p.sp != 0;

    float2 A2[NS / 2], Gv[NS / 2];
#pragma unroll
    for (int j = 0; j < NS / 2; ++j) {
        const int n = k * NS + 2 * j;
        A2[j] = dv ? make_float2(__fmul_rn(p.A[d * kN + n], kLog2e), __fmul_rn(p.A[d * kN + n + 1], kLog2e))
                   : make_float2(0.f, 0.f);
        Gv[j] = make_float2(0.f, 0.f);
    }
    const float bias = (dv && p.dt_bias) ? p.dt_bias[d] : 0.f;
    const int vchx = (int)(min64(CH, D - d0) * ES / 16);
    const int vchd = (int)(min64(CH, D - d0) * 4 / 16);
    auto issue = [&](int j, char* st) {
        const int64_t t0 = tb0 + (int64_t)j * kCK;
        const int rows = (int)min64(kCK, tb1 - t0);
        const int64_t row0 = b * L + t0;
        if (has_z)
            stage_block<NT>(st + OFF_Z, XROW, (const char*)p.z + (row0 * D + d0) * ES, D * ES, kCK, CH * ES / 16, rows,
                            vchx);
        stage_block<NT>(st + OFF_DY, XROW, (const char*)p.dy + (row0 * D + d0) * ES, D * ES, kCK, CH * ES / 16, rows,
                        vchx);
        stage_block<NT>(st + OFF_DT, DTROW, (const char*)p.dt + (row0 * D + d0) * 4, D * 4, kCK, CH * 4 / 16, rows,
                        vchd);
        stage_block<NT>(st + OFF_C, BCROW, (const char*)p.Cm + row0 * kN * ES, kN * ES, kCK, BCROW / 16, rows,
                        BCROW / 16);
        cp_async_commit();
    };
    float ssum = 0.f;
    if (ntile > 0) issue(ntile - 1, smem);
    for (int it = 0; it < ntile; ++it) {
        const int j = ntile - 1 - it;
        char* st = smem + (it & 1) * STAGE;
        if (j > 0) {
            issue(j - 1, smem + ((it + 1) & 1) * STAGE);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        for (int i = tid; i < kCK * kN; i += NT) Cf[i] = IOT<IO>::to_f(reinterpret_cast<const IO*>(st + OFF_C)[i]);
        __syncthreads();
        const int rows = (int)min64(kCK, tb1 - (tb0 + (int64_t)j * kCK));
#pragma unroll
        for (int tb = kCK - NSPLIT; tb >= 0; tb -= NSPLIT) {
            const int tm = tb + k;
            const float dtv = reinterpret_cast<const float*>(st + OFF_DT + tm * DTROW)[c];
            const float dyv = IOT<IO>::to_f(reinterpret_cast<const IO*>(st + OFF_DY + tm * XROW)[c]);
            const float delta = token_delta<FAST>(dtv, bias, sp);
            float dpv = dyv;
            if (has_z) {
                const float zv = IOT<IO>::to_f(reinterpret_cast<const IO*>(st + OFF_Z + tm * XROW)[c]);
                dpv = __fmul_rn(dyv, __fmul_rn(zv, sigmoid<FAST>(zv)));
            }
#pragma unroll
            for (int jj = NSPLIT - 1; jj >= 0; --jj) {
                const float dj = NSPLIT == 1 ? delta : __shfl_sync(0xffffffffu, delta, base + jj);
                const float pj = NSPLIT == 1 ? dpv : __shfl_sync(0xffffffffu, dpv, base + jj);
                if (tb + jj < rows) {
                    ssum = __fadd_rn(ssum, dj);
                    const float2 d2 = make_float2(dj, dj), p2 = make_float2(pj, pj);
                    const float* Ct = Cf + (tb + jj) * kN + k * NS;
#pragma unroll
                    for (int q = 0; q < NS / 2; ++q) {
                        const float2 arg = __fmul2_rn(d2, A2[q]);
                        const float2 a = make_float2(ex2(arg.x), ex2(arg.y));
                        const float2 cc = *reinterpret_cast<const float2*>(Ct + 2 * q);
                        Gv[q] = __fmul2_rn(__ffma2_rn(p2, cc, Gv[q]), a);
                    }
                }
            }
        }
        __syncthreads();
    }
    if (dv) {
        float* Q = p.aggQ + ((b * p.G + g) * D + d) * kN + k * NS;
#pragma unroll
        for (int q = 0; q < NS / 2; ++q) {
            Q[2 * q] = Gv[q].x;
            Q[2 * q + 1] = Gv[q].y;
        }
        if (k == 0) p.aggS[(b * p.G + g) * D + d] = ssum;
    }
}

template <typename IO, int NSPLIT> int launch_bwd_t(const BwdParams& p, cudaStream_t s) {
    using Ly = BwdLayout<IO, NSPLIT>;
    auto kern = ssm_bwd_kernel<IO, NSPLIT>;
    static unsigned long long mask = 0;
    if (!ensure_smem(kern, Ly::SMEM, mask)) return -1;
    if (p.B == 0 || p.D == 0 || p.G == 0) return 0;
    dim3 grid((unsigned)((p.D + Ly::CH - 1) / Ly::CH), (unsigned)p.G, (unsigned)p.B);
    kern<<<grid, kBwdThreads, Ly::SMEM, s>>>(p);
    return cudaGetLastError() == cudaSuccess ? 1 : -1;
}

template <typename IO, int NSPLIT> int launch_bwd_agg_t(const BwdParams& p, cudaStream_t s) {
    constexpr int CH = kBwdThreads / NSPLIT;
    constexpr int SMEM = bwd_agg_smem<IO, NSPLIT>();
    auto kern = ssm_bwd_agg_kernel<IO, NSPLIT>;
    static unsigned long long mask = 0;
    if (!ensure_smem(kern, SMEM, mask)) return -1;
    if (p.B == 0 || p.D == 0 || p.G <= 1) return 0;
    dim3 grid((unsigned)((p.D + CH - 1) / CH), (unsigned)(p.G - 1), (unsigned)p.B);
    kern<<<grid, kBwdThreads, SMEM, s>>>(p);
    return cudaGetLastError() == cudaSuccess ? 1 : -1;
}

}  // namespace

int launch_bwd(int io, int nsplit, const BwdParams& p, cudaStream_t s) {
    if (io == 0) {
        if (nsplit == 1) return launch_bwd_t<float, 1>(p, s);
        if (nsplit == 2) return launch_bwd_t<float, 2>(p, s);
        return launch_bwd_t<float, 4>(p, s);
    }
    if (nsplit == 1) return launch_bwd_t<__nv_bfloat16, 1>(p, s);
    if (nsplit == 2) return launch_bwd_t<__nv_bfloat16, 2>(p, s);
    return launch_bwd_t<__nv_bfloat16, 4>(p, s);
}

int launch_bwd_agg(int io, int nsplit, const BwdParams& p, cudaStream_t s) {
    if (io == 0) {
        if (nsplit == 1) return launch_bwd_agg_t<float, 1>(p, s);
        if (nsplit == 2) return launch_bwd_agg_t<float, 2>(p, s);
        return launch_bwd_agg_t<float, 4>(p, s);
    }
    if (nsplit == 1) return launch_bwd_agg_t<__nv_bfloat16, 1>(p, s);
    if (nsplit == 2) return launch_bwd_agg_t<__nv_bfloat16, 2>(p, s);
    return launch_bwd_agg_t<__nv_bfloat16, 4>(p, s);
}

}  // namespace ssm
