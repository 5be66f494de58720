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
    static constexpr int OFF_BT = 2 * STAGE;                   // fp32 B^T [16 states][16 tokens]
    static constexpr int OFF_CT = OFF_BT + kN * kCK * 4;       // fp32 C^T
    static constexpr int WROW = 36;                            // floats per lane row of the transpose buffer
    static constexpr int OFF_W = OFF_CT + kN * kCK * 4;        // [NW][32][WROW]
    static constexpr int OFF_O = OFF_W + NW * 32 * WROW * 4;   // [NW][2][16 states][16 tokens]
    static constexpr int SMEM = OFF_O + NW * 2 * kN * kCK * 4;
};

template <int NSPLIT> __device__ __forceinline__ float pick(const float (&a)[kCK], int m, int k) {
    // a[NSPLIT*m + k] with m static and k the lane's part index
    if constexpr (NSPLIT == 1) return a[m];
    else if constexpr (NSPLIT == 2) return k ? a[2 * m + 1] : a[2 * m];
    else {
        const float lo = (k & 1) ? a[4 * m + 1] : a[4 * m];
        const float hi = (k & 1) ? a[4 * m + 3] : a[4 * m + 2];
        return (k & 2) ? hi : lo;
    }
}

template <typename IO, int NSPLIT>
__global__ void __launch_bounds__(kBwdThreads) ssm_bwd_kernel(const BwdParams p) {
    using Ly = BwdLayout<IO, NSPLIT>;
    constexpr int NT = Ly::NT, CH = Ly::CH, NS = Ly::NS, ES = Ly::ES;
    constexpr int MI = kCK / NSPLIT;  // tokens whose per-token work this lane does
    constexpr bool FAST = IOT<IO>::kFast;
    extern __shared__ __align__(16) char smem[];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = tid / NSPLIT, k = tid % NSPLIT;
    const int base = lane & ~(NSPLIT - 1);
    const int64_t D = p.D, L = p.L;
    const int64_t d0 = (int64_t)blockIdx.x * CH, d = d0 + c;
    const bool dv = d < D;
    const int g = blockIdx.y;
    const int64_t b = blockIdx.z;
    const int64_t tb0 = (int64_t)g * p.Lg;
    const int64_t tb1 = min64(L, tb0 + p.Lg);
    const int nsub = (int)((tb1 - tb0 + kCK - 1) / kCK);
    const int64_t nck = (L + kCK - 1) / kCK;
    const bool has_z = p.has_z != 0, sp = p.sp != 0;

    float An[NS], A2n[NS], Gc[NS], dAacc[NS];
#pragma unroll
    for (int j = 0; j < NS; ++j) {
        const int n = k * NS + j;
        An[j] = dv ? p.A[d * kN + n] : 0.f;
        A2n[j] = __fmul_rn(An[j], kLog2e);
        float gi = 0.f;
        if (dv && p.gstart)
            gi = p.G == 1 ? p.gstart[(b * D + d) * kN + n] : p.gstart[((b * p.G + g) * D + d) * kN + n];
        Gc[j] = gi;
        dAacc[j] = 0.f;
    }
    const float Dd = (dv && p.Dskip) ? p.Dskip[d] : 0.f;
    const float bias = (dv && p.dt_bias) ? p.dt_bias[d] : 0.f;
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

    float* BT = reinterpret_cast<float*>(smem + Ly::OFF_BT);
    float* CT = reinterpret_cast<float*>(smem + Ly::OFF_CT);
    float* wb = reinterpret_cast<float*>(smem + Ly::OFF_W) + warp * 32 * Ly::WROW;
    float* wo = reinterpret_cast<float*>(smem + Ly::OFF_O);

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
        {
            const IO* Braw = reinterpret_cast<const IO*>(st + Ly::OFF_B);
            const IO* Craw = reinterpret_cast<const IO*>(st + Ly::OFF_C);
            for (int i = tid; i < kCK * kN; i += NT) {
                const int tok = i / kN, n = i % kN;  // raw is [token][state]; store [state][token]
                BT[n * kCK + tok] = IOT<IO>::to_f(Braw[i]);
                CT[n * kCK + tok] = IOT<IO>::to_f(Craw[i]);
            }
        }
        __syncthreads();

        const int64_t t0 = tb0 + (int64_t)s * kCK;
        const int rows = (int)min64(kCK, tb1 - t0);

        // ---- per-token quantities: this lane prepares tokens k, k+NSPLIT, ...
        float Dl[kCK], Ul[kCK], Pl[kCK];
        {
            float md[MI], mu[MI], mp[MI];
#pragma unroll
            for (int m = 0; m < MI; ++m) {
                const int i = NSPLIT * m + k;
                const float xv = IOT<IO>::to_f(reinterpret_cast<const IO*>(st + Ly::OFF_X + i * Ly::XROW)[c]);
                const float dyv = IOT<IO>::to_f(reinterpret_cast<const IO*>(st + Ly::OFF_DY + i * Ly::XROW)[c]);
                const float dtv = reinterpret_cast<const float*>(st + Ly::OFF_DT + i * Ly::DTROW)[c];
                float delta = token_delta<FAST>(dtv, bias, sp);
                float dpv = dyv;
                if (has_z) {
                    const float zv = IOT<IO>::to_f(reinterpret_cast<const IO*>(st + Ly::OFF_Z + i * Ly::XROW)[c]);
                    dpv = __fmul_rn(dyv, __fmul_rn(zv, sigmoid<FAST>(zv)));
                }
                const bool live = i < rows;  // tokens past the end act as identity
                md[m] = live ? delta : 0.f;
                mu[m] = live ? __fmul_rn(delta, xv) : 0.f;
                mp[m] = live ? dpv : 0.f;
            }
#pragma unroll
            for (int i = 0; i < kCK; ++i) {
                const int m = i / NSPLIT, src = base + i % NSPLIT;
                Dl[i] = NSPLIT == 1 ? md[m] : __shfl_sync(0xffffffffu, md[m], src);
                Ul[i] = NSPLIT == 1 ? mu[m] : __shfl_sync(0xffffffffu, mu[m], src);
                Pl[i] = NSPLIT == 1 ? mp[m] : __shfl_sync(0xffffffffu, mp[m], src);
            }
        }

        float S1[kCK], S2[kCK], S3[kCK];
#pragma unroll
        for (int i = 0; i < kCK; ++i) S1[i] = S2[i] = S3[i] = 0.f;
        const float* hck = reinterpret_cast<const float*>(st + Ly::OFF_H) + c * kN;

#pragma unroll
        for (int j = 0; j < NS; ++j) {
            const int n = k * NS + j;
            const float* Bn = BT + n * kCK;
            const float* Cn = CT + n * kCK;
            const float hstart = hck[n];
            float a[kCK], hh[kCK];
            float hp = hstart;
#pragma unroll
            for (int q = 0; q < kCK / 4; ++q) {
                const float4 b4 = *reinterpret_cast<const float4*>(Bn + 4 * q);
                const float4 c4 = *reinterpret_cast<const float4*>(Cn + 4 * q);
                const float bq[4] = {b4.x, b4.y, b4.z, b4.w}, cq[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int i = 4 * q + r;
                    a[i] = ex2(__fmul_rn(Dl[i], A2n[j]));
                    hh[i] = __fmaf_rn(a[i], hp, __fmul_rn(Ul[i], bq[r]));
                    hp = hh[i];
                    S3[i] = __fmaf_rn(cq[r], hh[i], S3[i]);
                }
            }
            float G = Gc[j];
#pragma unroll
            for (int q = kCK / 4 - 1; q >= 0; --q) {
                const float4 b4 = *reinterpret_cast<const float4*>(Bn + 4 * q);
                const float4 c4 = *reinterpret_cast<const float4*>(Cn + 4 * q);
                const float bq[4] = {b4.x, b4.y, b4.z, b4.w}, cq[4] = {c4.x, c4.y, c4.z, c4.w};
                float vb[4], vc[4];
#pragma unroll
                for (int r = 3; r >= 0; --r) {
                    const int i = 4 * q + r;
                    const float Gn = __fmaf_rn(Pl[i], cq[r], G);
                    vb[r] = __fmul_rn(Gn, Ul[i]);
                    vc[r] = __fmul_rn(Pl[i], hh[i]);
                    S1[i] = __fmaf_rn(Gn, bq[r], S1[i]);
                    const float hprev = i > 0 ? hh[i - 1] : hstart;
                    const float w = __fmul_rn(Gn, __fmul_rn(a[i], hprev));
                    dAacc[j] = __fmaf_rn(Dl[i], w, dAacc[j]);
                    S2[i] = __fmaf_rn(An[j], w, S2[i]);
                    G = __fmul_rn(Gn, a[i]);
                }
                *reinterpret_cast<float4*>(wb + lane * Ly::WROW + 4 * q) = make_float4(vb[0], vb[1], vb[2], vb[3]);
                *reinterpret_cast<float4*>(wb + lane * Ly::WROW + kCK + 4 * q) =
                    make_float4(vc[0], vc[1], vc[2], vc[3]);
            }
            Gc[j] = G;
            __syncwarp();
            {
                // Sum the transpose buffer over the channel lanes that share
                // this state: lane = (quad qd of the 32 values, part kk, row
                // block hpb); rows (hpb*8 + r)*NSPLIT + kk, r = 0..7.
                const int qd = lane & 7, rest = lane >> 3, kk = rest % NSPLIT, hpb = rest / NSPLIT;
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    const int row = (hpb * 8 + r) * NSPLIT + kk;
                    const float4 v = *reinterpret_cast<const float4*>(wb + row * Ly::WROW + 4 * qd);
                    acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
                }
#pragma unroll
                for (int off = 8 * NSPLIT; off < 32; off <<= 1) {
                    acc.x += __shfl_xor_sync(0xffffffffu, acc.x, off);
                    acc.y += __shfl_xor_sync(0xffffffffu, acc.y, off);
                    acc.z += __shfl_xor_sync(0xffffffffu, acc.z, off);
                    acc.w += __shfl_xor_sync(0xffffffffu, acc.w, off);
                }
                if (hpb == 0) {
                    const int nk = kk * NS + j, type = qd >> 2, i0 = (qd & 3) * 4;
                    *reinterpret_cast<float4*>(wo + ((warp * 2 + type) * kN + nk) * kCK + i0) = acc;
                }
            }
            __syncwarp();
        }

        // ---- per-token sums over the lane's states -> over all 16 states
#pragma unroll
        for (int i = 0; i < kCK; ++i) {
            if constexpr (NSPLIT >= 2) {
                S1[i] += __shfl_xor_sync(0xffffffffu, S1[i], 1);
                S2[i] += __shfl_xor_sync(0xffffffffu, S2[i], 1);
                S3[i] += __shfl_xor_sync(0xffffffffu, S3[i], 1);
            }
            if constexpr (NSPLIT >= 4) {
                S1[i] += __shfl_xor_sync(0xffffffffu, S1[i], 2);
                S2[i] += __shfl_xor_sync(0xffffffffu, S2[i], 2);
                S3[i] += __shfl_xor_sync(0xffffffffu, S3[i], 2);
            }
        }

        // ---- per-token outputs of this lane's tokens, written in place
#pragma unroll
        for (int m = 0; m < MI; ++m) {
            const int i = NSPLIT * m + k;
            if (i < rows) {
                IO* xs = reinterpret_cast<IO*>(st + Ly::OFF_X + i * Ly::XROW);
                IO* zs = reinterpret_cast<IO*>(st + Ly::OFF_Z + i * Ly::XROW);
                IO* dys = reinterpret_cast<IO*>(st + Ly::OFF_DY + i * Ly::XROW);
                float* dts = reinterpret_cast<float*>(st + Ly::OFF_DT + i * Ly::DTROW);
                const float xv = IOT<IO>::to_f(xs[c]);
                const float dyv = IOT<IO>::to_f(dys[c]);
                float sg = 1.f;
                const float v = __fadd_rn(dts[c], bias);
                float delta = v;
                if (sp) delta = softplus_sig<FAST>(v, &sg);
                const float s1 = pick<NSPLIT>(S1, m, k), s2 = pick<NSPLIT>(S2, m, k), s3 = pick<NSPLIT>(S3, m, k);
                const float pr = __fmaf_rn(Dd, xv, s3);
                float dpv = dyv;
                if (has_z) {
                    const float zv = IOT<IO>::to_f(zs[c]);
                    const float sz = sigmoid<FAST>(zv);
                    dpv = __fmul_rn(dyv, __fmul_rn(zv, sz));
                    const float dsilu = sz * (1.0f + zv * (1.0f - sz));
                    const float dzv = dyv * pr * dsilu;
                    nf = __fmaf_rn(dzv, 0.0f, nf);
                    zs[c] = IOT<IO>::from_f(dzv);
                }
                const float dxv = __fmaf_rn(dpv, Dd, delta * s1);
                const float ddelta = __fmaf_rn(xv, s1, s2);
                const float ddtv = sp ? ddelta * sg : ddelta;
                dDacc = __fmaf_rn(dpv, xv, dDacc);
                dbacc += ddtv;
                nf = __fmaf_rn(dxv, 0.0f, nf);
                nf = __fmaf_rn(ddtv, 0.0f, nf);
                dys[c] = IOT<IO>::from_f(dxv);
                dts[c] = ddtv;
            }
        }
        __syncthreads();

        // ---- copy dx, dz, d_dt out; dB / dC: sum the warps, one atomic per 4
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
            // 2 types x 16 tokens x 4 state-quads = 128 float4 outputs
            for (int o = tid; o < 2 * kCK * (kN / 4); o += NT) {
                const int type = o / (kCK * kN / 4), rem = o % (kCK * kN / 4);
                const int i = rem / (kN / 4), n0 = (rem % (kN / 4)) * 4;
                if (i < rows) {
                    float4 s4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int w = 0; w < Ly::NW; ++w) {
                        const float* src = wo + ((w * 2 + type) * kN + n0) * kCK + i;
                        s4.x += src[0]; s4.y += src[kCK]; s4.z += src[2 * kCK]; s4.w += src[3 * kCK];
                    }
                    float* dst = (type == 0 ? p.dB : p.dC) + (b * L + t0 + i) * kN + n0;
                    red_add_v4(dst, s4);
                }
            }
        }
        __syncthreads();
    }

    // ---- reductions over the group
    if (dv) {
#pragma unroll
        for (int j = 0; j < NS; ++j) atomicAdd(p.dA + d * kN + k * NS + j, dAacc[j]);
        if (g == 0 && p.dh0) {
#pragma unroll
            for (int j = 0; j < NS; ++j) p.dh0[(b * D + d) * kN + k * NS + j] = Gc[j];
        }
    }
    if constexpr (NSPLIT >= 2) {
        dDacc += __shfl_xor_sync(0xffffffffu, dDacc, 1);
        dbacc += __shfl_xor_sync(0xffffffffu, dbacc, 1);
    }
    if constexpr (NSPLIT >= 4) {
        dDacc += __shfl_xor_sync(0xffffffffu, dDacc, 2);
        dbacc += __shfl_xor_sync(0xffffffffu, dbacc, 2);
    }
    if (dv && k == 0) {
        atomicAdd(p.dD + d, dDacc);
        atomicAdd(p.ddt_bias + d, dbacc);
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
