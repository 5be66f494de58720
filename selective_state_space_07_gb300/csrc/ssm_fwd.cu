// Forward scan, chunk-aggregate pass, chunk-carry scan and single-token step
// of the S6 selective scan on sm_103a.
//
// Recurrence (rustytorch commit log, "MambaBlock" S6 forward commit:
// "sequential scan h=dA.h+dBu, y=sum C.h + D.u -> gate by SiLU(z)"):
// per (b, d) channel the 16 states are an independent first-order linear
// recurrence in t. Each channel is owned by NSPLIT adjacent lanes of a warp
// (lane k holds states [k*16/NSPLIT, (k+1)*16/NSPLIT)) and walks its tokens
// sequentially with the state in registers. Tiles of 16 tokens x CH
// channels of x, z, dt and the 16-wide B_t / C_t rows are staged into shared
// memory with cp.async (double-buffered), B/C are widened to fp32 once per
// tile, and y leaves through a shared-memory tile as 16-byte stores.
//
// Parallelism along L: the sequence splits into G groups. A first pass
// (AGG) runs every group but the last from a zero state and publishes its
// end state and sum of Delta; a warp-shuffle associative scan of the affine
// maps h -> exp(A*sum Delta)*h + H_end across groups produces each group's
// carry-in; the main pass then reruns every group from its carry.
#include "ssm_common.cuh"
#include "ssm_internal.h"

namespace ssm {

namespace {

template <typename IO, int NSPLIT> struct FwdLayout {
    static constexpr int NT = kFwdThreads;
    static constexpr int CH = NT / NSPLIT;        // channels per CTA
    static constexpr int NS = kN / NSPLIT;        // states per lane
    static constexpr int ES = sizeof(IO);
    static constexpr int XROW = CH * ES + 16;     // padded shared row (bytes) of x / z / y
    static constexpr int DTROW = CH * 4 + 16;     // padded shared row of dt
    static constexpr int BCROW = kN * ES;         // one token of B or C
    static constexpr int OFF_X = 0;
    static constexpr int OFF_Z = OFF_X + kCK * XROW;
    static constexpr int OFF_DT = OFF_Z + kCK * XROW;
    static constexpr int OFF_B = OFF_DT + kCK * DTROW;
    static constexpr int OFF_C = OFF_B + kCK * BCROW;
    static constexpr int STAGE = OFF_C + kCK * BCROW;
    // cp.async pipeline depth: enough tiles in flight to cover DRAM latency
    static constexpr int NSTAGE = STAGE <= 12 * 1024 ? 4 : 2;
    static constexpr int SMEM = NSTAGE * STAGE;                 // staged tiles (dynamic shared memory)
};


// Full readout of one (token, channel) from its NSPLIT lane partials, in the
// canonical tree ((lane0 + lane1) + (lane2 + lane3)) -- the association
// readout_allreduce uses in the step form.
template <int NSPLIT> __device__ __forceinline__ float combine_partials(const float* P) {
    if constexpr (NSPLIT == 1) return P[0];
    else if constexpr (NSPLIT == 2) {
        const float2 v = *reinterpret_cast<const float2*>(P);
        return __fadd_rn(v.x, v.y);
    } else {
        const float4 v = *reinterpret_cast<const float4*>(P);
        return __fadd_rn(__fadd_rn(v.x, v.y), __fadd_rn(v.z, v.w));
    }
}

// One CTA: CH channels of one batch row over one L-group, 16 tokens per
// staged tile. Per tile: (A) every thread prepares (Delta, u) and the gate
// factor for (token, channel) pairs; (B) each lane advances its NS states
// through the tile's tokens and leaves its partial readouts in shared
// memory; (E) every thread combines the partials of (token, channel)
// pairs, applies skip and gate and stages y.
template <typename IO, int NSPLIT, bool AGG>
__global__ void __launch_bounds__(kFwdThreads) ssm_fwd_kernel(const FwdParams p) {
    using Ly = FwdLayout<IO, NSPLIT>;
    constexpr int NT = Ly::NT, CH = Ly::CH, NS = Ly::NS, ES = Ly::ES;
    constexpr bool FAST = IOT<IO>::kFast;
    extern __shared__ __align__(16) char smem[];

    const int tid = threadIdx.x;
    // lane role: channel c, states [k*NS, k*NS+NS). Lanes sharing k sit in
    // the same quarter / half of the warp, so the per-token B/C loads of a
    // quarter-warp hit one address (a broadcast takes half the wavefronts of
    // four interleaved addresses).
    constexpr int CPW = 32 / NSPLIT;  // channels per warp
    const int c = (tid >> 5) * CPW + (tid & (CPW - 1)), k = (tid & 31) / CPW;
    const int ce = tid % CH;                        // per-token role: channel ce
    const int64_t D = p.D, L = p.L;
    const int64_t d0 = (int64_t)blockIdx.x * CH, d = d0 + c, de = d0 + ce;
    const bool dv = d < D, dve = de < D;
    const int g = blockIdx.y;
    const int64_t b = blockIdx.z;
    const int64_t tb0 = (int64_t)g * p.Lg;
    const int64_t tb1 = min64(L, tb0 + p.Lg);
    const int ntile = (int)((tb1 - tb0 + kCK - 1) / kCK);
    const int64_t nck = (L + kCkpt - 1) / kCkpt;  // saved states per sequence
    const bool has_z = !AGG && p.has_z;
    const bool sp = p.sp != 0;

    float2 A2[NS / 2], h[NS / 2];
#pragma unroll
    for (int j = 0; j < NS / 2; ++j) {
        const int n = k * NS + 2 * j;
        A2[j] = dv ? make_float2(__fmul_rn(p.A[d * kN + n], kLog2e), __fmul_rn(p.A[d * kN + n + 1], kLog2e))
                   : make_float2(0.f, 0.f);
        float2 hv = make_float2(0.f, 0.f);
        if (!AGG && dv && p.hstart) {
            const float* hs = p.G == 1 ? p.hstart + (b * D + d) * kN : p.hstart + ((b * p.G + g) * D + d) * kN;
            hv = make_float2(hs[n], hs[n + 1]);
        }
        h[j] = hv;
    }
    const float Dde = (dve && p.Dskip) ? p.Dskip[de] : 0.f;
    const float biase = (dve && p.dt_bias) ? p.dt_bias[de] : 0.f;

    const int vchx = (int)(min64(CH, D - d0) * ES / 16);  // valid 16-byte chunks per x row
    const int vchd = (int)(min64(CH, D - d0) * 4 / 16);
    auto issue = [&](int j, char* st) {
        const int64_t t0 = tb0 + (int64_t)j * kCK;
        const int rows = (int)min64(kCK, tb1 - t0);
        const int64_t row0 = b * L + t0;
        stage_block<NT>(st + Ly::OFF_X, Ly::XROW, (const char*)p.x + (row0 * D + d0) * ES, D * ES, kCK,
                        CH * ES / 16, rows, vchx);
        if (has_z)
            stage_block<NT>(st + Ly::OFF_Z, Ly::XROW, (const char*)p.z + (row0 * D + d0) * ES, D * ES, kCK,
                            CH * ES / 16, rows, vchx);
        stage_block<NT>(st + Ly::OFF_DT, Ly::DTROW, (const char*)p.dt + (row0 * D + d0) * 4, D * 4, kCK,
                        CH * 4 / 16, rows, vchd);
        stage_block<NT>(st + Ly::OFF_B, Ly::BCROW, (const char*)p.Bm + row0 * kN * ES, kN * ES, kCK,
                        Ly::BCROW / 16, rows, Ly::BCROW / 16);
        if (!AGG)
            stage_block<NT>(st + Ly::OFF_C, Ly::BCROW, (const char*)p.Cm + row0 * kN * ES, kN * ES, kCK,
                            Ly::BCROW / 16, rows, Ly::BCROW / 16);
        cp_async_commit();
    };

    // per-tile working arrays: each its own shared object, so the compiler
    // knows loads from one never alias stores to another
    __shared__ __align__(16) float Bf[kCK * kN];
    __shared__ __align__(16) float Cf[kCK * kN];
    __shared__ __align__(16) float2 DU[kCK * CH];
    __shared__ __align__(16) float GZ[AGG ? 1 : kCK * CH];
    __shared__ __align__(16) float PB[AGG ? 1 : kCK * CH * NSPLIT];
    __shared__ __align__(16) char ys[AGG ? 16 : kCK * Ly::XROW];
    float nf = 0.f;     // Inf/NaN detector
    float ssum = 0.f;   // AGG: sum of Delta over the group

    // prologue: tiles 0 .. NSTAGE-2 in flight (one commit group per tile,
    // empty groups past the end keep the group count uniform)
#pragma unroll
    for (int q = 0; q < Ly::NSTAGE - 1; ++q) {
        if (q < ntile) issue(q, smem + q * Ly::STAGE);
        else cp_async_commit();
    }
    for (int j = 0; j < ntile; ++j) {
        char* st = smem + (j % Ly::NSTAGE) * Ly::STAGE;
        {
            const int jn = j + Ly::NSTAGE - 1;  // refill the slot tile j-1 used
            if (jn < ntile) issue(jn, smem + (jn % Ly::NSTAGE) * Ly::STAGE);
            else cp_async_commit();
        }
        cp_async_wait<Ly::NSTAGE - 1>();
        __syncthreads();
        const int64_t t0 = tb0 + (int64_t)j * kCK;
        const int rows = (int)min64(kCK, tb1 - t0);
        // ---- (A) per (token, channel): Delta, u, gate factor; B/C to fp32
        {
            const IO* Braw = reinterpret_cast<const IO*>(st + Ly::OFF_B);
            const IO* Craw = reinterpret_cast<const IO*>(st + Ly::OFF_C);
            for (int i = tid; i < kCK * kN; i += NT) {
                Bf[i] = IOT<IO>::to_f(Braw[i]);
                if (!AGG) Cf[i] = IOT<IO>::to_f(Craw[i]);
            }
#pragma unroll
            for (int r = 0; r < kCK * CH / NT; ++r) {
                const int t = tid / CH + (NT / CH) * r;
                const float xv = IOT<IO>::to_f(reinterpret_cast<const IO*>(st + Ly::OFF_X + t * Ly::XROW)[ce]);
                const float dtv = reinterpret_cast<const float*>(st + Ly::OFF_DT + t * Ly::DTROW)[ce];
                const float delta = token_delta<FAST>(dtv, biase, sp);
                DU[t * CH + ce] = make_float2(delta, __fmul_rn(delta, xv));
                if (has_z) {
                    const float zv = IOT<IO>::to_f(reinterpret_cast<const IO*>(st + Ly::OFF_Z + t * Ly::XROW)[ce]);
                    GZ[t * CH + ce] = __fmul_rn(zv, sigmoid<FAST>(zv));
                }
            }
        }
        __syncthreads();
        // ---- (B) the lane's states through the tile's tokens; partial
        // readouts stay in registers until the tile is done
        float Pt[kCK];
#pragma unroll
        for (int t = 0; t < kCK; ++t) {
            Pt[t] = 0.f;
            if (!AGG && t % kCkpt == 0 && t < rows && p.ckpt && dv) {
                // state before token t0+t: ckpt[b][(t0+t)/8][n][d]
                float* cp = p.ckpt + ((b * nck + (t0 + t) / kCkpt) * kN + k * NS) * D + d;
#pragma unroll
                for (int q = 0; q < NS / 2; ++q) {
                    cp[(2 * q) * D] = h[q].x;
                    cp[(2 * q + 1) * D] = h[q].y;
                }
            }
            if (t < rows) {
                const float2 du = DU[t * CH + c];
                const float* Bt = Bf + t * kN + k * NS;
                if (AGG) {
                    token_update<NS>(h, A2, du.x, du.y, Bt);
                    ssum = __fadd_rn(ssum, du.x);
                } else {
                    Pt[t] = token_states<NS>(h, A2, du.x, du.y, Bt, Cf + t * kN + k * NS);
                }
            }
        }
        if (!AGG) {
#pragma unroll
            for (int t = 0; t < kCK; ++t) PB[(t * CH + c) * NSPLIT + k] = Pt[t];
        }
        if (!AGG) {
            __syncthreads();
            // ---- (E) per (token, channel): combine partials, skip term, gate
#pragma unroll
            for (int r = 0; r < kCK * CH / NT; ++r) {
                const int t = tid / CH + (NT / CH) * r;
                if (t < rows) {
                    const float pr = combine_partials<NSPLIT>(PB + (t * CH + ce) * NSPLIT);
                    const float xv = IOT<IO>::to_f(reinterpret_cast<const IO*>(st + Ly::OFF_X + t * Ly::XROW)[ce]);
                    const float pp = __fmaf_rn(Dde, xv, pr);
                    const float yv = has_z ? __fmul_rn(pp, GZ[t * CH + ce]) : pp;
                    nf = __fmaf_rn(yv, 0.0f, nf);
                    reinterpret_cast<IO*>(ys + t * Ly::XROW)[ce] = IOT<IO>::from_f(yv);
                }
            }
            __syncthreads();
            constexpr int CHX = CH * ES / 16;
            for (int i = tid; i < rows * CHX; i += NT) {
                const int r = i / CHX, ch = i - r * CHX;
                if (ch < vchx)
                    *reinterpret_cast<int4*>((char*)p.y + (((b * L + t0 + r) * D + d0) * ES + ch * 16)) =
                        *reinterpret_cast<const int4*>(ys + r * Ly::XROW + ch * 16);
            }
        }
        __syncthreads();
    }

    if (AGG) {
        if (dv) {
            float* H = p.aggH + ((b * p.G + g) * D + d) * kN + k * NS;
#pragma unroll
            for (int q = 0; q < NS / 4; ++q)
                reinterpret_cast<float4*>(H)[q] = make_float4(h[2 * q].x, h[2 * q].y, h[2 * q + 1].x, h[2 * q + 1].y);
            if (k == 0) p.aggS[(b * p.G + g) * D + d] = ssum;
        }
    } else {
        if (g == p.G - 1 && p.h_last && dv) {
            float* hl = p.h_last + (b * D + d) * kN + k * NS;
#pragma unroll
            for (int q = 0; q < NS / 4; ++q)
                reinterpret_cast<float4*>(hl)[q] = make_float4(h[2 * q].x, h[2 * q].y, h[2 * q + 1].x, h[2 * q + 1].y);
        }
        flag_nonfinite(p.status, nf);
    }
}

// Carries along L. One warp per (b, d, n); lanes take the groups in windows
// of 32 and run an inclusive warp-shuffle scan of the affine maps
// f_g(h) = a_g*h + v_g (a_g = exp(A*sum Delta_g)), composed as
// (a2, v2) o (a1, v1) = (a2*a1, a2*v1 + v2). Forward: map g takes the
// state at the start of group g to its end; out[g] = state entering group g.
// Reverse (backward pass): map m takes the adjoint carry at the end of group
// G-1-m to the end of group G-2-m; out[g] = carry entering group g from
// the right.
__global__ void ssm_carry_kernel(int64_t B, int64_t D, int G, int reverse, const float* __restrict__ A,
                                 const float* __restrict__ start, const float* __restrict__ aggV,
                                 const float* __restrict__ aggS, float* __restrict__ out) {
    const int64_t wid = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (wid >= B * D * kN) return;  // whole warp leaves together
    const int n = (int)(wid % kN);
    const int64_t bd = wid / kN, d = bd % D, b = bd / D;
    const float An = A[d * kN + n];
    float carry = start ? start[(b * D + d) * kN + n] : 0.f;
    const int nmaps = G - 1;
    for (int w0 = 0; w0 < G; w0 += 32) {
        const int m = w0 + lane;
        float a = 1.f, v = 0.f;
        if (m < nmaps) {
            const int gsrc = reverse ? G - 1 - m : m;
            a = expf(An * aggS[(b * G + gsrc) * D + d]);
            v = aggV[((b * G + gsrc) * D + d) * kN + n];
        }
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float ap = __shfl_up_sync(0xffffffffu, a, off);
            const float vp = __shfl_up_sync(0xffffffffu, v, off);
            if (lane >= off) {
                v = fmaf(a, vp, v);
                a = a * ap;
            }
        }
        const float after = fmaf(a, carry, v);  // value after map m
        // value entering position w0 is `carry`; after map m it enters position m+1
        if (lane == 0) {
            const int gdst = reverse ? G - 1 - w0 : w0;
            out[((b * G + gdst) * D + d) * kN + n] = carry;
        }
        if (lane < 31 && m + 1 < G) {
            const int gdst = reverse ? G - 2 - m : m + 1;
            out[((b * G + gdst) * D + d) * kN + n] = after;
        }
        carry = __shfl_sync(0xffffffffu, after, 31);
    }
}

// One token for every (b, d): the same per-token arithmetic as the forward
// (token_delta, token_states, readout tree, gate_out).
template <typename IO, int NSPLIT>
__global__ void __launch_bounds__(kFwdThreads) ssm_step_kernel(const StepParams p) {
    constexpr int CH = kFwdThreads / NSPLIT, NS = kN / NSPLIT;
    constexpr bool FAST = IOT<IO>::kFast;
    __shared__ __align__(16) float Bs[kN], Cs[kN];
    const int tid = threadIdx.x, c = tid / NSPLIT, k = tid % NSPLIT;
    const int64_t D = p.D, b = blockIdx.y, d = (int64_t)blockIdx.x * CH + c;
    const bool dv = d < D;
    if (tid < kN) {
        Bs[tid] = IOT<IO>::to_f(reinterpret_cast<const IO*>(p.Bm)[b * kN + tid]);
        Cs[tid] = IOT<IO>::to_f(reinterpret_cast<const IO*>(p.Cm)[b * kN + tid]);
    }
    __syncthreads();
    float2 A2[NS / 2], h[NS / 2];
    float* st = p.state + (b * D + (dv ? d : 0)) * kN + k * NS;
#pragma unroll
    for (int j = 0; j < NS / 2; ++j) {
        const int n = k * NS + 2 * j;
        A2[j] = dv ? make_float2(__fmul_rn(p.A[d * kN + n], kLog2e), __fmul_rn(p.A[d * kN + n + 1], kLog2e))
                   : make_float2(0.f, 0.f);
        h[j] = dv ? make_float2(st[2 * j], st[2 * j + 1]) : make_float2(0.f, 0.f);
    }
    const int64_t i = b * D + (dv ? d : 0);
    const float xv = dv ? IOT<IO>::to_f(reinterpret_cast<const IO*>(p.x)[i]) : 0.f;
    const float dtv = dv ? p.dt[i] : 0.f;
    const float bias = (dv && p.dt_bias) ? p.dt_bias[d] : 0.f;
    const float Dd = (dv && p.Dskip) ? p.Dskip[d] : 0.f;
    const float delta = token_delta<FAST>(dtv, bias, p.sp != 0);
    const float u = __fmul_rn(delta, xv);
    const float P = token_states<NS>(h, A2, delta, u, Bs + k * NS, Cs + k * NS);
    const float pr = readout_allreduce<NSPLIT>(P);
    const bool has_z = p.has_z != 0;
    const float zv = (has_z && dv) ? IOT<IO>::to_f(reinterpret_cast<const IO*>(p.z)[i]) : 0.f;
    const float yv = gate_out<FAST>(pr, Dd, xv, zv, has_z);
    if (dv) {
#pragma unroll
        for (int j = 0; j < NS / 2; ++j) {
            st[2 * j] = h[j].x;
            st[2 * j + 1] = h[j].y;
        }
        if (k == 0) reinterpret_cast<IO*>(p.y)[i] = IOT<IO>::from_f(yv);
    }
    flag_nonfinite(p.status, __fmaf_rn(yv, 0.0f, 0.0f));
}

template <typename IO, int NSPLIT, bool AGG> int launch_fwd_t(const FwdParams& p, cudaStream_t s) {
    using Ly = FwdLayout<IO, NSPLIT>;
    static unsigned long long mask = 0;
    auto kern = ssm_fwd_kernel<IO, NSPLIT, AGG>;
    if (!ensure_smem(kern, Ly::SMEM, mask)) return -1;
    const int gy = AGG ? p.G - 1 : p.G;
    if (gy <= 0 || p.B == 0 || p.D == 0) return 0;
    dim3 grid((unsigned)((p.D + Ly::CH - 1) / Ly::CH), (unsigned)gy, (unsigned)p.B);
    kern<<<grid, kFwdThreads, Ly::SMEM, s>>>(p);
    return cudaGetLastError() == cudaSuccess ? 1 : -1;
}

template <typename IO, int NSPLIT> int launch_step_t(const StepParams& p, cudaStream_t s) {
    constexpr int CH = kFwdThreads / NSPLIT;
    if (p.B == 0 || p.D == 0) return 0;
    dim3 grid((unsigned)((p.D + CH - 1) / CH), (unsigned)p.B);
    ssm_step_kernel<IO, NSPLIT><<<grid, kFwdThreads, 0, s>>>(p);
    return cudaGetLastError() == cudaSuccess ? 1 : -1;
}

template <bool AGG> int dispatch_fwd(int io, int nsplit, const FwdParams& p, cudaStream_t s) {
    if (io == 0) {
        if (nsplit == 1) return launch_fwd_t<float, 1, AGG>(p, s);
        if (nsplit == 2) return launch_fwd_t<float, 2, AGG>(p, s);
        return launch_fwd_t<float, 4, AGG>(p, s);
    }
    if (nsplit == 1) return launch_fwd_t<__nv_bfloat16, 1, AGG>(p, s);
    if (nsplit == 2) return launch_fwd_t<__nv_bfloat16, 2, AGG>(p, s);
    return launch_fwd_t<__nv_bfloat16, 4, AGG>(p, s);
}

}  // namespace

int launch_fwd(int io, int nsplit, const FwdParams& p, cudaStream_t s) { return dispatch_fwd<false>(io, nsplit, p, s); }
int launch_fwd_agg(int io, int nsplit, const FwdParams& p, cudaStream_t s) { return dispatch_fwd<true>(io, nsplit, p, s); }

int launch_carry(int64_t B, int64_t D, int G, bool reverse, const float* A, const float* start, const float* aggV,
                 const float* aggS, float* out, cudaStream_t s) {
    const int64_t warps = B * D * kN;
    if (warps == 0) return 0;
    const int threads = 256;
    const int64_t blocks = (warps * 32 + threads - 1) / threads;
    ssm_carry_kernel<<<(unsigned)blocks, threads, 0, s>>>(B, D, G, reverse ? 1 : 0, A, start, aggV, aggS, out);
    return cudaGetLastError() == cudaSuccess ? 1 : -1;
}

int launch_step(int io, int nsplit, const StepParams& p, cudaStream_t s) {
    if (io == 0) {
        if (nsplit == 1) return launch_step_t<float, 1>(p, s);
        if (nsplit == 2) return launch_step_t<float, 2>(p, s);
        return launch_step_t<float, 4>(p, s);
    }
    if (nsplit == 1) return launch_step_t<__nv_bfloat16, 1>(p, s);
    if (nsplit == 2) return launch_step_t<__nv_bfloat16, 2>(p, s);
    return launch_step_t<__nv_bfloat16, 4>(p, s);
}

}  // namespace ssm
