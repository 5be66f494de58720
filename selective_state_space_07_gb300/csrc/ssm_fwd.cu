// Forward scan, chunk-aggregate pass, chunk-carry scan and single-token step
// of the S6 selective scan on sm_103a.
//
// Recurrence (rustytorch commit log, "MambaBlock" S6 forward commit:
// "sequential scan h=dA.h+dBu, y=sum C.h + D.u -> gate by SiLU(z)"):
// per (b, d) channel the 16 states are an independent first-order linear
// recurrence in t. Lanes l and l^16 of a warp share one channel: lane l
// holds states 8*(l>>4) .. 8*(l>>4)+7 in registers and walks the tokens in
// order. Tiles of 16 tokens x 64 channels of x, z, dt and the 16-wide B_t /
// C_t rows are staged into shared memory by TMA (one thread issues a tile's
// boxes onto the stage's mbarrier; four tiles in flight); B/C are widened to
// fp32 and transposed (state-major) once per
// tile, so a half-warp reads one state's row of 4 tokens with one broadcast
// 16-byte load. Delta*A, u*B and the readout are packed over token pairs
// (f32x2); each state's update is a scalar fused multiply-add chain.
//
// Per tile: (A) each lane prepares Delta, u and the gate factor for its 8
// tokens (one lane of the pair per token, two tokens per packed f32x2
// operation) and shares Delta/u with its partner through shared memory;
// (S) the lane's 8 state recurrences advance side by side through the 16
// tokens (independent chains for the scheduler) while the readout chain
// takes the states in order; (E) the two half-readouts of each token are
// added and each lane gates and writes y for its 8 tokens.
//
// One block barrier per tile: the tables a tile writes (B^T, C^T, Delta/u)
// are double-buffered by tile parity, so the barrier after (A) of tile j
// also orders every write of tile j+1 after the reads of tile j-1; the
// stage a tile used is refilled at the top of the next tile, after that
// barrier. The per-warp half-readout exchange of (E) synchronises the warp
// only.
//
// Canonical readout order (the step kernel evaluates the same operations):
// each half of the states is a sequential fused multiply-add chain
// C_0 h_0 -> fma(C_1, h_1, .) -> ... -> fma(C_7, h_7, .), and the two halves
// are added; p + D x is fused, then multiplied by z * sigmoid(z).
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

template <typename IO> struct FwdLayout {
    static constexpr int NT = kFwdThreads;
    static constexpr int CH = NT / 2;             // channels per CTA (a lane pair per channel)
    static constexpr int ES = sizeof(IO);
    static constexpr int XROW = CH * ES;          // staged row of x / z (bytes)
    static constexpr int DTROW = CH * 4;          // staged row of dt
    static constexpr int BCROW = kN * ES;         // one token of B or C
    static constexpr int OFF_X = 0;
    static constexpr int OFF_Z = OFF_X + kCK * XROW;
    static constexpr int OFF_DT = OFF_Z + kCK * XROW;
    static constexpr int OFF_B = OFF_DT + kCK * DTROW;
    static constexpr int OFF_C = OFF_B + kCK * BCROW;
    static constexpr int STAGE = OFF_C + kCK * BCROW;
    static constexpr int NSTAGE = 4;              // tiles in flight
    static constexpr int SMEM = NSTAGE * STAGE + 128;  // dynamic shared memory (+ slack for 128-byte alignment)
    static_assert(OFF_Z % 128 == 0 && OFF_DT % 128 == 0 && OFF_B % 128 == 0 && OFF_C % 128 == 0 &&
                      STAGE % 128 == 0, "TMA destinations on 128-byte boundaries");
    static constexpr int ROW = 2 * kCK + 4;       // per-channel row of DU / PB (floats, padded)
};

__device__ __forceinline__ float2 f2(float a, float b) { return make_float2(a, b); }

// TMA descriptors of a tile's inputs: x, z, dt [B*L, D] in boxes of CH
// channels x 16 tokens; B, C [B*L, 16] (rows bcs elements apart) in boxes of
// 16 x 16. Elements past the last token or channel read as zero.
struct FwdMaps {
    CUtensorMap x, z, dt, b, c;
};

// MINB: resident CTAs per SM the register budget is cut for (3 when the grid
// can use a third CTA per SM; 1 -- no cut -- when one L-group's grid fits in
// two CTAs per SM, which leaves the scheduler registers for the interleaved
// state chains).
template <typename IO, bool AGG, int MINB>
__global__ void __launch_bounds__(kFwdThreads, MINB)
    ssm_fwd_kernel(const FwdParams p, const __grid_constant__ FwdMaps mp) {
    using Ly = FwdLayout<IO>;
    constexpr int NT = Ly::NT, CH = Ly::CH, ES = Ly::ES, T = kCK, NS = kN / 2;
    constexpr bool FAST = IOT<IO>::kFast;
    extern __shared__ __align__(128) char smem_raw[];
    char* smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);  // the TMA destinations
    __shared__ __align__(8) uint64_t fullb[Ly::NSTAGE];          // a stage's copies landed
    // tables of a tile, double-buffered by tile parity so that one barrier
    // per tile orders every write after the reads of two tiles before
    __shared__ __align__(16) float BT[2][kN * T];                 // B^T of the tile [state][token]
    __shared__ __align__(16) float CT[2][AGG ? 4 : kN * T];
    __shared__ __align__(16) float DU[2][CH * Ly::ROW];           // per channel [Delta 0..15 | u 0..15]
    __shared__ __align__(16) float PB[AGG ? 4 : CH * Ly::ROW];    // per channel [half-0 readouts | half-1]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int hk = lane >> 4;                 // states 8*hk .. 8*hk+7; tokens 8*hk .. 8*hk+7 of the tile
    const int c = warp * 16 + (lane & 15);    // channel within the CTA
    const int64_t D = p.D, L = p.L;
    const int64_t d0 = (int64_t)blockIdx.x * CH, d = d0 + c;
    const bool dv = d < D;
    const int g = blockIdx.y;
    const int64_t b = blockIdx.z;
    const int64_t tb0 = (int64_t)g * p.Lg;
    const int64_t tb1 = min64(L, tb0 + p.Lg);
    const int ntile = (int)((tb1 - tb0 + T - 1) / T);
    const int64_t nck = (L + kCkpt - 1) / kCkpt;  // saved states per sequence
    const bool has_z = !AGG && p.has_z;
    const bool sp = p.sp != 0;

    float A2[NS], h[NS];
#pragma unroll
    for (int s = 0; s < NS; ++s) {
        const int n = NS * hk + s;
        A2[s] = dv ? __fmul_rn(p.A[d * kN + n], kLog2e) : 0.f;
        float hv = 0.f;
        if (!AGG && dv && p.hstart)
            hv = p.G == 1 ? p.hstart[(b * D + d) * kN + n] : p.hstart[((b * p.G + g) * D + d) * kN + n];
        h[s] = hv;
    }
    const float Dd = (dv && p.Dskip) ? p.Dskip[d] : 0.f;
    const float bias = (dv && p.dt_bias) ? p.dt_bias[d] : 0.f;

    const float2 D2 = f2(Dd, Dd), bias2 = f2(bias, bias);
    const unsigned long long wait_ns = p.wait_ns ? p.wait_ns : kWaitNs;

    // one thread loads a tile's inputs with TMA onto the stage's mbarrier;
    // rows past the group's last token are loaded too (or read as zero past
    // the tensor's end) and ignored: they act as identity tokens below
    const unsigned stage_bytes =
        (unsigned)(T * (Ly::XROW * (has_z ? 2 : 1) + Ly::DTROW + Ly::BCROW * (AGG ? 1 : 2)));
    auto issue = [&](int j) {
        const int slot = j % Ly::NSTAGE;
        char* st = smem + slot * Ly::STAGE;
        const int y = (int)(b * L + tb0 + (int64_t)j * T);  // first token row of the tile in [B*L]
        const unsigned bar = smem_u32(&fullb[slot]);
        mbar_expect_tx(bar, stage_bytes);
        if (j + 1 == p.fault_tile1) return;  // test hook: the barrier is armed, the copies never come
        tma_load_2d(st + Ly::OFF_X, &mp.x, (int)d0, y, bar);
        if (has_z) tma_load_2d(st + Ly::OFF_Z, &mp.z, (int)d0, y, bar);
        tma_load_2d(st + Ly::OFF_DT, &mp.dt, (int)d0, y, bar);
        tma_load_2d(st + Ly::OFF_B, &mp.b, 0, y, bar);
        if (!AGG) tma_load_2d(st + Ly::OFF_C, &mp.c, 0, y, bar);
    };
    if (tid == 0) {
        for (int q = 0; q < Ly::NSTAGE; ++q) mbar_init(smem_u32(&fullb[q]), 1);
        mbar_fence_init();
    }
    __syncthreads();

    float nf = 0.f;     // Inf/NaN detector
    float ssum = 0.f;   // AGG: this lane's part of the sum of Delta over the group

    // prologue: tiles 0 .. NSTAGE-2 in flight
    if (tid == 0)
        for (int q = 0; q < Ly::NSTAGE - 1 && q < ntile; ++q) issue(q);
    int j = 0;
    bool aborted = false;
    for (; j < ntile; ++j) {
        const int buf = j & 1;
        const char* st = smem + (j % Ly::NSTAGE) * Ly::STAGE;
        // refill the slot tile j-1 used: every thread passed tile j-1's
        // barrier, after its last read of that stage
        if (tid == 0 && j + Ly::NSTAGE - 1 < ntile) issue(j + Ly::NSTAGE - 1);
        // every thread waits for the tile itself (bounded); the barrier below
        // tells every thread whether any wait ran out
        const bool late = !mbar_wait_bounded(smem_u32(&fullb[j % Ly::NSTAGE]), (unsigned)((j / Ly::NSTAGE) & 1), wait_ns);
        const int64_t t0 = tb0 + (int64_t)j * T;
        const int rows = (int)min64(T, tb1 - t0);

        // ---- B/C to fp32, state-major
        {
            const IO* Braw = reinterpret_cast<const IO*>(st + Ly::OFF_B);
            const IO* Craw = reinterpret_cast<const IO*>(st + Ly::OFF_C);
            for (int i = tid; i < kN * T; i += NT) {
                const int n = i / T, tok = i - n * T;
                const bool live = tok < rows;  // rows past the end belong to other tokens: zero, not read
                BT[buf][i] = live ? IOT<IO>::to_f(Braw[tok * kN + n]) : 0.f;
                if (!AGG) CT[buf][i] = live ? IOT<IO>::to_f(Craw[tok * kN + n]) : 0.f;
            }
        }
        // ---- A: Delta, u and the gate factor of this lane's 8 tokens, a
        // token pair at a time; tokens past the end act as identity (Delta = u = 0)
        float* du = DU[buf] + c * Ly::ROW;
        float2 xo[NS / 2], gz[NS / 2];
        {
            float2 dl[NS / 2], ul[NS / 2];
#pragma unroll
            for (int i = 0; i < NS / 2; ++i) {
                const int t = NS * hk + 2 * i;
                const char* xr = st + Ly::OFF_X + t * Ly::XROW;
                const float2 xv = f2(IOT<IO>::to_f(reinterpret_cast<const IO*>(xr)[c]),
                                     IOT<IO>::to_f(reinterpret_cast<const IO*>(xr + Ly::XROW)[c]));
                const char* dr = st + Ly::OFF_DT + t * Ly::DTROW;
                const float2 dtv = f2(reinterpret_cast<const float*>(dr)[c], reinterpret_cast<const float*>(dr + Ly::DTROW)[c]);
                const float2 delta = delta2<FAST>(dtv, bias2, sp);
                const bool l0 = t < rows, l1 = t + 1 < rows;
                dl[i] = f2(l0 ? delta.x : 0.f, l1 ? delta.y : 0.f);
                const float2 u = __fmul2_rn(delta, xv);
                ul[i] = f2(l0 ? u.x : 0.f, l1 ? u.y : 0.f);
                xo[i] = xv;
                if (AGG) ssum = __fadd_rn(__fadd_rn(ssum, dl[i].x), dl[i].y);
                if (has_z) {
                    const char* zr = st + Ly::OFF_Z + t * Ly::XROW;
                    const float2 zv = f2(IOT<IO>::to_f(reinterpret_cast<const IO*>(zr)[c]),
                                         IOT<IO>::to_f(reinterpret_cast<const IO*>(zr + Ly::XROW)[c]));
                    gz[i] = __fmul2_rn(zv, sigmoid2<FAST>(zv));
                }
            }
            *reinterpret_cast<float4*>(du + NS * hk) = make_float4(dl[0].x, dl[0].y, dl[1].x, dl[1].y);
            *reinterpret_cast<float4*>(du + NS * hk + 4) = make_float4(dl[2].x, dl[2].y, dl[3].x, dl[3].y);
            *reinterpret_cast<float4*>(du + T + NS * hk) = make_float4(ul[0].x, ul[0].y, ul[1].x, ul[1].y);
            *reinterpret_cast<float4*>(du + T + NS * hk + 4) = make_float4(ul[2].x, ul[2].y, ul[3].x, ul[3].y);
        }
        if (__syncthreads_or(late)) {  // the tables of this tile are ready -- unless a copy never came
            aborted = true;
            break;
        }
        float2 Dl[T / 2], Ul[T / 2];
#pragma unroll
        for (int q = 0; q < T / 4; ++q) {
            const float4 dq = *reinterpret_cast<const float4*>(du + 4 * q);
            const float4 uq = *reinterpret_cast<const float4*>(du + T + 4 * q);
            Dl[2 * q] = f2(dq.x, dq.y);
            Dl[2 * q + 1] = f2(dq.z, dq.w);
            Ul[2 * q] = f2(uq.x, uq.y);
            Ul[2 * q + 1] = f2(uq.z, uq.w);
        }

        // ---- S: per state, the tile's 16 tokens; the readout chain runs
        // over this lane's 8 states
        const bool ck = !AGG && p.ckpt && dv;
        // checkpoint [B][nck][8 state pairs][D][2]: pair (n, n+1) of channel d
        float* ckp = ck ? p.ckpt + (((b * nck + t0 / kCkpt) * (kN / 2) + NS * hk / 2) * D + d) * 2 : nullptr;
        const float* BTb = BT[buf];
        const float* CTb = CT[buf];
        float2 acc[T / 2];
        // SI states advance together through the tokens (independent chains
        // for the scheduler); the readout chain still takes the states in order
        constexpr int SI = 8;
#pragma unroll
        for (int s = 0; s < NS; s += SI) {
            const int n = NS * hk + s;
            float2 A2p[SI];
            float hp[SI];
#pragma unroll
            for (int i = 0; i < SI; ++i) {
                A2p[i] = f2(A2[s + i], A2[s + i]);
                hp[i] = h[s + i];
            }
            if (ck) {  // states before token t0
#pragma unroll
                for (int i = 0; i < SI; i += 2) *reinterpret_cast<float2*>(ckp + (int64_t)((s + i) / 2) * D * 2) = f2(hp[i], hp[i + 1]);
            }
#pragma unroll
            for (int q = 0; q < T / 4; ++q) {
                float4 b4[SI], c4[SI];
#pragma unroll
                for (int i = 0; i < SI; ++i) {
                    b4[i] = *reinterpret_cast<const float4*>(BTb + (n + i) * T + 4 * q);
                    if (!AGG) c4[i] = *reinterpret_cast<const float4*>(CTb + (n + i) * T + 4 * q);
                }
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const int m = 2 * q + h2;
                    float hv0[SI], hv1[SI];
#pragma unroll
                    for (int i = 0; i < SI; ++i) {
                        const float2 bb = h2 ? f2(b4[i].z, b4[i].w) : f2(b4[i].x, b4[i].y);
                        const float2 arg = __fmul2_rn(Dl[m], A2p[i]);
                        const float a0 = ex2(arg.x), a1 = ex2(arg.y);
                        const float2 ub = __fmul2_rn(Ul[m], bb);
                        hv0[i] = __fmaf_rn(a0, hp[i], ub.x);
                        hv1[i] = __fmaf_rn(a1, hv0[i], ub.y);
                        hp[i] = hv1[i];
                    }
                    if (!AGG) {
                        float2 r = acc[m];
#pragma unroll
                        for (int i = 0; i < SI; ++i) {
                            const float2 cc = h2 ? f2(c4[i].z, c4[i].w) : f2(c4[i].x, c4[i].y);
                            r = (s + i == 0) ? __fmul2_rn(cc, f2(hv0[i], hv1[i])) : __ffma2_rn(cc, f2(hv0[i], hv1[i]), r);
                        }
                        acc[m] = r;
                    }
                }
                if (q == 1 && ck && rows > kCkpt) {  // states before token t0+8
#pragma unroll
                    for (int i = 0; i < SI; i += 2)
                        *reinterpret_cast<float2*>(ckp + (int64_t)((s + i) / 2) * D * 2 + (int64_t)kN * D) = f2(hp[i], hp[i + 1]);
                }
            }
#pragma unroll
            for (int i = 0; i < SI; ++i) h[s + i] = hp[i];
        }
        if (!AGG) {
            // ---- E: half readouts -> full readout of this lane's 8 tokens
            float* pb = PB + c * Ly::ROW;
            __syncwarp();  // the previous tile's reads of PB are done
            *reinterpret_cast<float4*>(pb + T * hk) = make_float4(acc[0].x, acc[0].y, acc[1].x, acc[1].y);
            *reinterpret_cast<float4*>(pb + T * hk + 4) = make_float4(acc[2].x, acc[2].y, acc[3].x, acc[3].y);
            *reinterpret_cast<float4*>(pb + T * hk + 8) = make_float4(acc[4].x, acc[4].y, acc[5].x, acc[5].y);
            *reinterpret_cast<float4*>(pb + T * hk + 12) = make_float4(acc[6].x, acc[6].y, acc[7].x, acc[7].y);
            __syncwarp();
            const float4 p0a = *reinterpret_cast<const float4*>(pb + NS * hk);
            const float4 p0b = *reinterpret_cast<const float4*>(pb + NS * hk + 4);
            const float4 p1a = *reinterpret_cast<const float4*>(pb + T + NS * hk);
            const float4 p1b = *reinterpret_cast<const float4*>(pb + T + NS * hk + 4);
            const float2 P0[NS / 2] = {f2(p0a.x, p0a.y), f2(p0a.z, p0a.w), f2(p0b.x, p0b.y), f2(p0b.z, p0b.w)};
            const float2 P1[NS / 2] = {f2(p1a.x, p1a.y), f2(p1a.z, p1a.w), f2(p1b.x, p1b.y), f2(p1b.z, p1b.w)};
            IO* yrow = reinterpret_cast<IO*>(p.y) + (b * L + t0) * D + d;
#pragma unroll
            for (int i = 0; i < NS / 2; ++i) {
                const int t = NS * hk + 2 * i;
                const float2 pr = __fadd2_rn(P0[i], P1[i]);
                const float2 pp = __ffma2_rn(D2, xo[i], pr);
                const float2 yv = has_z ? __fmul2_rn(pp, gz[i]) : pp;
                if (dv && t < rows) {
                    nf = __fmaf_rn(yv.x, 0.0f, nf);
                    yrow[(int64_t)t * D] = IOT<IO>::from_f(yv.x);
                }
                if (dv && t + 1 < rows) {
                    nf = __fmaf_rn(yv.y, 0.0f, nf);
                    yrow[(int64_t)(t + 1) * D] = IOT<IO>::from_f(yv.y);
                }
            }
        }
    }

    if (aborted) {
        // every thread stops at tile j; thread 0 waits (bounded) for the
        // copies still in flight (tiles j .. j + NSTAGE - 1) before the block leaves
        if (tid == 0) {
            const int last = min(j + Ly::NSTAGE - 1, ntile - 1);
            for (int jj = j; jj <= last; ++jj)
                (void)mbar_wait_bounded(smem_u32(&fullb[jj % Ly::NSTAGE]), (unsigned)((jj / Ly::NSTAGE) & 1), wait_ns);
            if (p.status) atomicOr(p.status, kStatusTimeout);
        }
        return;
    }
    if (AGG) {
        ssum = __fadd_rn(ssum, __shfl_xor_sync(0xffffffffu, ssum, 16));
        if (dv) {
            float* H = p.aggH + ((b * p.G + g) * D + d) * kN + NS * hk;
#pragma unroll
            for (int s = 0; s < NS; ++s) H[s] = h[s];
            if (hk == 0) p.aggS[(b * p.G + g) * D + d] = ssum;
        }
    } else {
        if (g == p.G - 1 && p.h_last && dv) {
            float* hl = p.h_last + (b * D + d) * kN + NS * hk;
#pragma unroll
            for (int s = 0; s < NS; ++s) hl[s] = h[s];
        }
        flag_nonfinite(p.status, nf);
    }
}

// Carries along L. A segment of W lanes (W = the power of two >= G, at most
// 32) serves one (b, d, n); a warp holds 32/W segments. Lanes take the groups
// in windows of W and run an inclusive segmented warp-shuffle scan of the
// affine maps f_g(h) = a_g*h + v_g (a_g = exp(A*sum Delta_g)), composed as
// (a2, v2) o (a1, v1) = (a2*a1, a2*v1 + v2). Forward: map g takes the state
// at the start of group g to its end; out[g] = state entering group g.
// Reverse (backward pass): map m takes the adjoint carry at the end of group
// G-1-m to the end of group G-2-m; out[g] = carry entering group g from
// the right.
template <int W>
__global__ void ssm_carry_kernel(int64_t B, int64_t D, int G, int reverse, const float* __restrict__ A,
                                 const float* __restrict__ start, const float* __restrict__ aggV,
                                 const float* __restrict__ aggS, float* __restrict__ out) {
    const int lane = threadIdx.x & 31, sl = lane & (W - 1);
    const int64_t item = (((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5) * (32 / W) + lane / W;
    const bool valid = item < B * D * kN;  // invalid segments still shuffle (full-warp masks)
    const int n = (int)(item % kN);
    const int64_t bd = valid ? item / kN : 0, d = bd % D, b = bd / D;
    const float An = valid ? A[d * kN + n] : 0.f;
    float carry = (valid && start) ? start[(b * D + d) * kN + n] : 0.f;
    const int nmaps = G - 1;
    for (int w0 = 0; w0 < G; w0 += W) {
        const int m = w0 + sl;
        float a = 1.f, v = 0.f;
        if (valid && m < nmaps) {
            const int gsrc = reverse ? G - 1 - m : m;
            a = expf(An * aggS[(b * G + gsrc) * D + d]);
            v = aggV[((b * G + gsrc) * D + d) * kN + n];
        }
#pragma unroll
        for (int off = 1; off < W; off <<= 1) {
            const float ap = __shfl_up_sync(0xffffffffu, a, off, W);
            const float vp = __shfl_up_sync(0xffffffffu, v, off, W);
            if (sl >= off) {
                v = fmaf(a, vp, v);
                a = a * ap;
            }
        }
        const float after = fmaf(a, carry, v);  // value after map m
        if (valid) {
            // value entering position w0 is `carry`; after map m it enters position m+1
            if (sl == 0) {
                const int gdst = reverse ? G - 1 - w0 : w0;
                out[((b * G + gdst) * D + d) * kN + n] = carry;
            }
            if (sl < W - 1 && m + 1 < G) {
                const int gdst = reverse ? G - 2 - m : m + 1;
                out[((b * G + gdst) * D + d) * kN + n] = after;
            }
        }
        carry = __shfl_sync(0xffffffffu, after, W - 1, W);
    }
}

// One token for every (b, d) channel with the forward's arithmetic and
// canonical readout order: NSPLIT = 1 (a lane per channel, both half chains)
// or 2 (adjacent lanes take the two halves).
template <typename IO, int NSPLIT>
__global__ void __launch_bounds__(kFwdThreads) ssm_step_kernel(const StepParams p) {
    constexpr int CH = kFwdThreads / NSPLIT;
    constexpr bool FAST = IOT<IO>::kFast;
    __shared__ __align__(16) float Bs[kN], Cs[kN];
    const int tid = threadIdx.x, c = tid / NSPLIT, k = tid % NSPLIT;
    const int64_t D = p.D, b = blockIdx.y, d = (int64_t)blockIdx.x * CH + c;
    const bool dv = d < D;
    if (tid < kN) {
        Bs[tid] = IOT<IO>::to_f(reinterpret_cast<const IO*>(p.Bm)[b * p.bcs + tid]);
        Cs[tid] = IOT<IO>::to_f(reinterpret_cast<const IO*>(p.Cm)[b * p.bcs + tid]);
    }
    __syncthreads();
    const int64_t i = b * D + (dv ? d : 0);
    const float xv = dv ? IOT<IO>::to_f(reinterpret_cast<const IO*>(p.x)[i]) : 0.f;
    const float dtv = dv ? p.dt[i] : 0.f;
    const float bias = (dv && p.dt_bias) ? p.dt_bias[d] : 0.f;
    const float Dd = (dv && p.Dskip) ? p.Dskip[d] : 0.f;
    const float delta = token_delta<FAST>(dtv, bias, p.sp != 0);
    const float u = __fmul_rn(delta, xv);
    float* st = p.state + (b * D + (dv ? d : 0)) * kN;
    float half[2] = {0.f, 0.f};
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
        if (NSPLIT == 2 && hf != k) continue;
        float acc = 0.f;
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            const int n = 8 * hf + s;
            const float A2 = dv ? __fmul_rn(p.A[d * kN + n], kLog2e) : 0.f;
            const float a = ex2(__fmul_rn(delta, A2));
            const float ub = __fmul_rn(u, Bs[n]);
            const float hv = __fmaf_rn(a, dv ? st[n] : 0.f, ub);
            if (dv) st[n] = hv;
            acc = s == 0 ? __fmul_rn(Cs[n], hv) : __fmaf_rn(Cs[n], hv, acc);
        }
        half[hf] = acc;
    }
    float pr;
    if (NSPLIT == 1) {
        pr = __fadd_rn(half[0], half[1]);
    } else {
        const float mine = half[k];
        pr = __fadd_rn(mine, __shfl_xor_sync(0xffffffffu, mine, 1));  // addition commutes: same bits in both lanes
    }
    const bool has_z = p.has_z != 0;
    const float zv = (has_z && dv) ? IOT<IO>::to_f(reinterpret_cast<const IO*>(p.z)[i]) : 0.f;
    const float yv = gate_out<FAST>(pr, Dd, xv, zv, has_z);
    if (dv && k == 0) reinterpret_cast<IO*>(p.y)[i] = IOT<IO>::from_f(yv);
    flag_nonfinite(p.status, __fmaf_rn(yv, 0.0f, 0.0f));
}

template <typename IO, bool AGG, int MINB>
int launch_fwd_v(const FwdParams& p, const FwdMaps& mp, dim3 grid, cudaStream_t s) {
    using Ly = FwdLayout<IO>;
    static unsigned long long mask = 0;
    auto kern = ssm_fwd_kernel<IO, AGG, MINB>;
    if (!ensure_smem(kern, Ly::SMEM, mask)) return -1;
    kern<<<grid, kFwdThreads, Ly::SMEM, s>>>(p, mp);
    return cudaGetLastError() == cudaSuccess ? 1 : -1;
}

template <typename IO> bool encode_fwd_maps(const FwdParams& p, bool with_c, FwdMaps* mp) {
    using Ly = FwdLayout<IO>;
    const CUtensorMapDataType io = sizeof(IO) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    const int64_t rows = p.B * p.L, ES = sizeof(IO);
    const CUtensorMapSwizzle none = CU_TENSOR_MAP_SWIZZLE_NONE;
    if (!encode_2d(&mp->x, io, p.x, p.D, rows, p.D * ES, Ly::CH, kCK, none) ||
        !encode_2d(&mp->dt, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, p.dt, p.D, rows, p.D * 4, Ly::CH, kCK, none) ||
        !encode_2d(&mp->b, io, p.Bm, kN, rows, p.bcs * ES, kN, kCK, none))
        return false;
    mp->z = mp->x;
    mp->c = mp->b;
    if (p.has_z && !encode_2d(&mp->z, io, p.z, p.D, rows, p.D * ES, Ly::CH, kCK, none)) return false;
    if (with_c && !encode_2d(&mp->c, io, p.Cm, kN, rows, p.bcs * ES, kN, kCK, none)) return false;
    return true;
}

template <typename IO, bool AGG> int launch_fwd_t(const FwdParams& p, cudaStream_t s) {
    using Ly = FwdLayout<IO>;
    const int gy = AGG ? p.G - 1 : p.G;
    if (gy <= 0 || p.B == 0 || p.D == 0) return 0;
    FwdMaps mp;
    if (!encode_fwd_maps<IO>(p, !AGG, &mp)) return -1;
    dim3 grid((unsigned)((p.D + Ly::CH - 1) / Ly::CH), (unsigned)gy, (unsigned)p.B);
    const int64_t ctas = (int64_t)grid.x * grid.y * grid.z;
    if (!AGG && p.G == 1 && ctas <= 2 * (int64_t)sm_count()) return launch_fwd_v<IO, AGG, 1>(p, mp, grid, s);
    return launch_fwd_v<IO, AGG, 3>(p, mp, grid, s);
}

template <typename IO, int NSPLIT> int launch_step_t(const StepParams& p, cudaStream_t s) {
    constexpr int CH = kFwdThreads / NSPLIT;
    if (p.B == 0 || p.D == 0) return 0;
    dim3 grid((unsigned)((p.D + CH - 1) / CH), (unsigned)p.B);
    ssm_step_kernel<IO, NSPLIT><<<grid, kFwdThreads, 0, s>>>(p);
    return cudaGetLastError() == cudaSuccess ? 1 : -1;
}

}  // namespace

namespace {
template <typename K> int blocks_per_sm(K kern, int threads, int smem, int* cache) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    int& c = cache[dev & 63];
    if (c == 0) {
        int v = 0;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, kern, threads, smem) != cudaSuccess || v < 1)
            v = 1;
        c = v;
    }
    return c;
}
}  // namespace

int fwd_blocks_per_sm(int io) {
    static int cache_f[64] = {0}, cache_b[64] = {0};
    // the variant that runs whenever the grid can use more than 2 CTAs per SM
    return io == 0 ? blocks_per_sm(ssm_fwd_kernel<float, false, 3>, kFwdThreads, FwdLayout<float>::SMEM, cache_f)
                   : blocks_per_sm(ssm_fwd_kernel<__nv_bfloat16, false, 3>, kFwdThreads,
                                   FwdLayout<__nv_bfloat16>::SMEM, cache_b);
}
int fwd_channels_per_cta() { return FwdLayout<float>::CH; }

int sm_count() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 152;
    int& c = cache[dev & 63];
    if (c == 0) {
        int v = 0;
        c = (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0) ? v : 152;
    }
    return c;
}

int launch_fwd(int io, const FwdParams& p, cudaStream_t s) {
    return io == 0 ? launch_fwd_t<float, false>(p, s) : launch_fwd_t<__nv_bfloat16, false>(p, s);
}
int launch_fwd_agg(int io, const FwdParams& p, cudaStream_t s) {
    return io == 0 ? launch_fwd_t<float, true>(p, s) : launch_fwd_t<__nv_bfloat16, true>(p, s);
}

template <int W>
int launch_carry_w(int64_t B, int64_t D, int G, bool reverse, const float* A, const float* start,
                   const float* aggV, const float* aggS, float* out, cudaStream_t s) {
    const int64_t warps = (B * D * kN + 32 / W - 1) / (32 / W);
    const int threads = 256;
    const int64_t blocks = (warps * 32 + threads - 1) / threads;
    ssm_carry_kernel<W><<<(unsigned)blocks, threads, 0, s>>>(B, D, G, reverse ? 1 : 0, A, start, aggV, aggS, out);
    return cudaGetLastError() == cudaSuccess ? 1 : -1;
}

int launch_carry(int64_t B, int64_t D, int G, bool reverse, const float* A, const float* start, const float* aggV,
                 const float* aggS, float* out, cudaStream_t s) {
    if (B * D == 0) return 0;
    if (G <= 2) return launch_carry_w<2>(B, D, G, reverse, A, start, aggV, aggS, out, s);
    if (G <= 4) return launch_carry_w<4>(B, D, G, reverse, A, start, aggV, aggS, out, s);
    if (G <= 8) return launch_carry_w<8>(B, D, G, reverse, A, start, aggV, aggS, out, s);
    if (G <= 16) return launch_carry_w<16>(B, D, G, reverse, A, start, aggV, aggS, out, s);
    return launch_carry_w<32>(B, D, G, reverse, A, start, aggV, aggS, out, s);
}

int launch_step(int io, int nsplit, const StepParams& p, cudaStream_t s) {
    if (io == 0) return nsplit == 1 ? launch_step_t<float, 1>(p, s) : launch_step_t<float, 2>(p, s);
    return nsplit == 1 ? launch_step_t<__nv_bfloat16, 1>(p, s) : launch_step_t<__nv_bfloat16, 2>(p, s);
}

}  // namespace ssm
