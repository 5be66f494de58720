// Forward scan, chunk-aggregate pass, chunk-carry scan and single-token step
// of the S6 selective scan on sm_103a.
//
// Recurrence (rustytorch commit log, "MambaBlock" S6 forward commit:
// "sequential scan h=dA.h+dBu, y=sum C.h + D.u -> gate by SiLU(z)"):
// per (b, d) channel the 16 states are an independent first-order linear
// recurrence in t. kFwdLPC lanes of a warp share one channel (lanes l,
// l + 32/kFwdLPC, ...): each holds 16/kFwdLPC of its states in registers and
// walks the tokens in order. Tiles of 16 tokens x 32 channels of x, z, dt and
// the 16-wide B_t /
// C_t rows are staged into shared memory by TMA (one thread issues a tile's
// boxes onto the stage's mbarrier; four tiles in flight); B/C are widened to
// fp32 and transposed (state-major) once per
// tile, so a half-warp reads one state's row of 4 tokens with one broadcast
// 16-byte load. Delta*A, u*B and the readout are packed over token pairs
// (f32x2); each state's update is a scalar fused multiply-add chain.
//
// Per tile: (A) each lane prepares Delta, u and the gate factor for its
// share of the tokens (one lane of the channel per token, two tokens per
// packed f32x2 operation) and shares Delta/u with the channel's other lanes
// through shared memory; (S) the lane's state recurrences advance side by
// side through the 16 tokens (independent chains for the scheduler) while
// its readout chain takes them in order; (E) the partial readouts of each
// token are summed and each lane gates and writes y for its tokens.
//
// One block barrier per tile: the tables a tile writes (B^T, C^T, Delta/u)
// are double-buffered by tile parity, so the barrier after (A) of tile j
// also orders every write of tile j+1 after the reads of tile j-1; the
// stage a tile used is refilled at the top of the next tile, after that
// barrier. The per-warp half-readout exchange of (E) synchronises the warp
// only.
//
// Canonical readout order (the step kernel evaluates the same operations):
// the states split into kFwdLPC blocks of 16/kFwdLPC consecutive states; each
// block is a sequential fused multiply-add chain C_n h_n -> fma(C_n+1,
// h_n+1, .) -> ...; the blocks are summed as a balanced binary tree in state
// order ((b0 + b1) + (b2 + b3) for four blocks); p + D x is fused, then
// multiplied by z * sigmoid(z).
//
// Parallelism along L: the sequence splits into G groups. A first pass
// (AGG) computes, for every group but the last, its end state from a zero
// state and its sum of Delta; a warp-shuffle associative scan of the affine
// maps h -> exp(A*sum Delta)*h + H_end across groups produces each group's
// carry-in; the main pass then reruns every group from its carry. The
// aggregate needs no per-token state: per tile, h <- exp(A sum Delta) h +
// sum_t exp(A S_t) u_t B_t with S_t the sum of Delta over the tile's later
// tokens (the product of the decays after t), so its terms are independent
// of one another instead of one multiply-add chain per state.
#include "ssm_common.cuh"
#include "ssm_internal.h"

namespace ssm {

namespace {

// Lane layout: the kFwdLPC lanes l, l + 32/kFwdLPC, ... of a warp share one
// channel; each holds NS = 16/kFwdLPC of its states and does the per-token
// work of TPL = 16/kFwdLPC of a tile's tokens.
constexpr int kLPC = kFwdLPC;
constexpr int kCPW = 32 / kLPC;  // channels per warp

// AGG stages neither z nor C: its stages are smaller (more CTAs per SM).
template <typename IO, bool AGG = false> struct FwdLayout {
    static constexpr int NT = kFwdCtaThreads;
    static constexpr int CH = NT / kLPC;          // channels per CTA
    static constexpr int ES = sizeof(IO);
    static constexpr int XROW = CH * ES;          // staged row of x / z (bytes)
    static constexpr int DTROW = CH * 4;          // staged row of dt
    static constexpr int BCROW = kN * ES;         // one token of B or C
    static constexpr int OFF_X = 0;
    static constexpr int OFF_Z = OFF_X + kCK * XROW;
    static constexpr int OFF_DT = OFF_Z + (AGG ? 0 : kCK * XROW);
    static constexpr int OFF_B = OFF_DT + kCK * DTROW;
    static constexpr int OFF_C = OFF_B + kCK * BCROW;
    static constexpr int STAGE = OFF_C + (AGG ? 0 : kCK * BCROW);
    static constexpr int NSTAGE = 4;              // tiles in flight
    static constexpr int SMEM = NSTAGE * STAGE + 128;  // dynamic shared memory (+ slack for 128-byte alignment)
    static_assert(OFF_Z % 128 == 0 && OFF_DT % 128 == 0 && OFF_B % 128 == 0 && OFF_C % 128 == 0 &&
                      STAGE % 128 == 0, "TMA destinations on 128-byte boundaries");
    static constexpr int ROW = 2 * kCK + 4;       // per-channel row of DU: [Delta 0..15 | u 0..15], padded
    static constexpr int PROW = kLPC * kCK + 4;   // per-channel row of PB: one 16-token row per lane, padded
};

__device__ __forceinline__ float2 f2(float a, float b) { return make_float2(a, b); }

// Sum of a channel's kLPC partial readouts in the canonical order: a
// balanced binary tree over the lanes' state blocks, in state order.
template <int P> __device__ __forceinline__ float2 tree2(const float2* q) {
    if constexpr (P == 1) {
        return q[0];
    } else {
        return __fadd2_rn(tree2<P / 2>(q), tree2<P / 2>(q + P / 2));
    }
}

// TMA descriptors of a tile's inputs: x, z, dt [B*L, D] in boxes of CH
// channels x 16 tokens; B, C [B*L, 16] (rows bcs elements apart) in boxes of
// 16 x 16. Elements past the last token or channel read as zero.
struct FwdMaps {
    CUtensorMap x, z, dt, b, c;
};

// MINB: resident CTAs per SM the register budget is cut for.
template <typename IO, bool AGG, int MINB>
__global__ void __launch_bounds__(kFwdCtaThreads, MINB)
    ssm_fwd_kernel(const FwdParams p, const __grid_constant__ FwdMaps mp) {
    using Ly = FwdLayout<IO, AGG>;
    constexpr int NT = Ly::NT, CH = Ly::CH, T = kCK, NS = kN / kLPC, TPL = kCK / kLPC, RB = kReadBlock;
    static_assert(NS % RB == 0, "whole readout blocks per lane");
    constexpr bool FAST = IOT<IO>::kFast;
    static_assert(NS % 2 == 0 && TPL % 4 == 0, "states and tokens per lane in pairs / quads");
    extern __shared__ __align__(128) char smem_raw[];
    char* smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);  // the TMA destinations
    __shared__ __align__(8) uint64_t fullb[Ly::NSTAGE];          // a stage's copies landed
    // tables of a tile, double-buffered by tile parity so that one barrier
    // per tile orders every write after the reads of two tiles before
    __shared__ __align__(16) float BT[2][kN * T];                 // B^T of the tile [state][token]
    __shared__ __align__(16) float CT[2][AGG ? 4 : kN * T];
    __shared__ __align__(16) float DU[2][CH * Ly::ROW];           // per channel [Delta 0..15 | u 0..15]
    __shared__ __align__(16) float PB[AGG ? 4 : CH * Ly::PROW];   // per channel, per lane: partial readouts

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int hk = lane / kCPW;                    // states NS*hk ..; tokens TPL*hk .. of the tile
    const int c = warp * kCPW + (lane % kCPW);     // channel within the CTA
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

    float nf = 0.f;        // Inf/NaN detector
    float ssum = 0.f;      // AGG: the sum of Delta over the group (the same in every lane of a channel)
    float tile_sum = 0.f;  // AGG: the sum of Delta over the current tile

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
        // ---- A: Delta, u and the gate factor of this lane's TPL tokens, a
        // token pair at a time; tokens past the end act as identity (Delta = u = 0)
        float* du = DU[buf] + c * Ly::ROW;
        float2 xo[TPL / 2], gz[TPL / 2];
        {
            float2 dl[TPL / 2], ul[TPL / 2];
#pragma unroll
            for (int i = 0; i < TPL / 2; ++i) {
                const int t = TPL * hk + 2 * i;
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
                if (has_z) {
                    const char* zr = st + Ly::OFF_Z + t * Ly::XROW;
                    const float2 zv = f2(IOT<IO>::to_f(reinterpret_cast<const IO*>(zr)[c]),
                                         IOT<IO>::to_f(reinterpret_cast<const IO*>(zr + Ly::XROW)[c]));
                    gz[i] = __fmul2_rn(zv, sigmoid2<FAST>(zv));
                }
            }
            if constexpr (AGG) {
                // the Delta row becomes, per token, the sum of Delta over the
                // tile's later tokens (exclusive suffix): the lane's own tokens,
                // then the totals of the channel's later lane blocks
                float sf[TPL];
                sf[TPL - 1] = 0.f;
#pragma unroll
                for (int k = TPL - 2; k >= 0; --k)
                    sf[k] = __fadd_rn(sf[k + 1], (k + 1) & 1 ? dl[(k + 1) / 2].y : dl[(k + 1) / 2].x);
                const float own = __fadd_rn(sf[0], dl[0].x);
                float after = 0.f, tot = 0.f;
#pragma unroll
                for (int r = 0; r < kLPC; ++r) {
                    const float tr = __shfl_sync(0xffffffffu, own, (lane % kCPW) + kCPW * r);
                    tot = __fadd_rn(tot, tr);  // the same order in every lane of the channel
                    if (r > hk) after = __fadd_rn(after, tr);
                }
#pragma unroll
                for (int i = 0; i < TPL / 2; ++i) dl[i] = f2(__fadd_rn(sf[2 * i], after), __fadd_rn(sf[2 * i + 1], after));
                tile_sum = tot;
                ssum = __fadd_rn(ssum, tot);
            }
#pragma unroll
            for (int i = 0; i < TPL / 4; ++i) {
                *reinterpret_cast<float4*>(du + TPL * hk + 4 * i) =
                    make_float4(dl[2 * i].x, dl[2 * i].y, dl[2 * i + 1].x, dl[2 * i + 1].y);
                *reinterpret_cast<float4*>(du + T + TPL * hk + 4 * i) =
                    make_float4(ul[2 * i].x, ul[2 * i].y, ul[2 * i + 1].x, ul[2 * i + 1].y);
            }
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

        // ---- S: this lane's NS states advance together through the tile's
        // 16 tokens; the readout chain takes them in order
        const bool ck = !AGG && p.ckpt && dv;
        // checkpoint [B][nck][8 state pairs][D][2]: pair (n, n+1) of channel d
        float* ckp = ck ? p.ckpt + (((b * nck + t0 / kCkpt) * (kN / 2) + NS * hk / 2) * D + d) * 2 : nullptr;
        const float* BTb = BT[buf];
        const float* CTb = CT[buf];
        const int n0 = NS * hk;
        float2 acc[T / 2];
        float2 A2p[NS];
        float hp[NS];
#pragma unroll
        for (int i = 0; i < NS; ++i) {
            A2p[i] = f2(A2[i], A2[i]);
            hp[i] = h[i];
        }
        if (ck) {  // states before token t0
#pragma unroll
            for (int i = 0; i < NS; i += 2) *reinterpret_cast<float2*>(ckp + (int64_t)(i / 2) * D * 2) = f2(hp[i], hp[i + 1]);
        }
        if constexpr (AGG) {
            // the group's end state from a zero start, tile by tile: h <- exp(A
            // sum Delta) h + sum_t exp(A S_t) u_t B_t, S_t the sum of Delta over
            // the tile's tokens after t -- no term of the sum waits for another
            float2 ha[NS];
#pragma unroll
            for (int i = 0; i < NS; ++i) ha[i] = f2(0.f, 0.f);
#pragma unroll
            for (int q = 0; q < T / 4; ++q) {
#pragma unroll
                for (int i = 0; i < NS; ++i) {
                    const float4 b4 = *reinterpret_cast<const float4*>(BTb + (n0 + i) * T + 4 * q);
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        const int m = 2 * q + h2;
                        const float2 bb = h2 ? f2(b4.z, b4.w) : f2(b4.x, b4.y);
                        const float2 arg = __fmul2_rn(Dl[m], A2p[i]);
                        const float2 ub = __fmul2_rn(Ul[m], bb);
                        ha[i] = __ffma2_rn(f2(ex2(arg.x), ex2(arg.y)), ub, ha[i]);
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < NS; ++i) h[i] = __fmaf_rn(ex2(__fmul_rn(A2[i], tile_sum)), h[i], __fadd_rn(ha[i].x, ha[i].y));
        } else {
#pragma unroll
            for (int q = 0; q < T / 4; ++q) {
                float4 b4[NS], c4[NS];
#pragma unroll
                for (int i = 0; i < NS; ++i) {
                    b4[i] = *reinterpret_cast<const float4*>(BTb + (n0 + i) * T + 4 * q);
                    if (!AGG) c4[i] = *reinterpret_cast<const float4*>(CTb + (n0 + i) * T + 4 * q);
                }
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const int m = 2 * q + h2;
                    float hv0[NS], hv1[NS];
#pragma unroll
                    for (int i = 0; i < NS; ++i) {
                        const float2 bb = h2 ? f2(b4[i].z, b4[i].w) : f2(b4[i].x, b4[i].y);
                        const float2 arg = __fmul2_rn(Dl[m], A2p[i]);
                        const float a0 = ex2(arg.x), a1 = ex2(arg.y);
                        const float2 ub = __fmul2_rn(Ul[m], bb);
                        hv0[i] = __fmaf_rn(a0, hp[i], ub.x);
                        hv1[i] = __fmaf_rn(a1, hv0[i], ub.y);
                        hp[i] = hv1[i];
                    }
                    if (!AGG) {
                        // the lane's NS/RB readout blocks: sequential chains of RB
                        // states, then summed as a balanced tree in state order
                        float2 r[NS / RB];
#pragma unroll
                        for (int i = 0; i < NS; ++i) {
                            const float2 cc = h2 ? f2(c4[i].z, c4[i].w) : f2(c4[i].x, c4[i].y);
                            r[i / RB] = (i % RB == 0) ? __fmul2_rn(cc, f2(hv0[i], hv1[i]))
                                                      : __ffma2_rn(cc, f2(hv0[i], hv1[i]), r[i / RB]);
                        }
                        acc[m] = tree2<NS / RB>(r);
                    }
                }
                if (q == 1 && ck && rows > kCkpt) {  // states before token t0+8
#pragma unroll
                    for (int i = 0; i < NS; i += 2)
                        *reinterpret_cast<float2*>(ckp + (int64_t)(i / 2) * D * 2 + (int64_t)kN * D) = f2(hp[i], hp[i + 1]);
                }
            }
#pragma unroll
            for (int i = 0; i < NS; ++i) h[i] = hp[i];
            if (!AGG) {
                // ---- E: the kLPC partial readouts of this lane's TPL tokens
                float* pb = PB + c * Ly::PROW;
                __syncwarp();  // the previous tile's reads of PB are done
#pragma unroll
                for (int q = 0; q < T / 4; ++q)
                    *reinterpret_cast<float4*>(pb + T * hk + 4 * q) =
                        make_float4(acc[2 * q].x, acc[2 * q].y, acc[2 * q + 1].x, acc[2 * q + 1].y);
                __syncwarp();
                IO* yrow = reinterpret_cast<IO*>(p.y) + (b * L + t0) * D + d;
#pragma unroll
                for (int i = 0; i < TPL / 4; ++i) {
                    float2 qa[kLPC], qb[kLPC];  // tokens TPL*hk + 4i + (0, 1) and (2, 3), one per lane block
#pragma unroll
                    for (int r = 0; r < kLPC; ++r) {
                        const float4 v = *reinterpret_cast<const float4*>(pb + T * r + TPL * hk + 4 * i);
                        qa[r] = f2(v.x, v.y);
                        qb[r] = f2(v.z, v.w);
                    }
                    const float2 pr[2] = {tree2<kLPC>(qa), tree2<kLPC>(qb)};
#pragma unroll
                    for (int k2 = 0; k2 < 2; ++k2) {
                        const int t = TPL * hk + 4 * i + 2 * k2;
                        const float2 pp = __ffma2_rn(D2, xo[2 * i + k2], pr[k2]);
                        const float2 yv = has_z ? __fmul2_rn(pp, gz[2 * i + k2]) : pp;
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
    // the lane's states and row of A, every load issued before anything is
    // stored (16-byte vectors; the state is updated in place)
    constexpr int NL = kN / NSPLIT;          // states of this lane
    const int nb0 = NSPLIT == 2 ? k * NL : 0;
    float hs[NL], As[NL];
#pragma unroll
    for (int q = 0; q < NL; q += 4) {
        const float4 h4 = dv ? *reinterpret_cast<const float4*>(st + nb0 + q) : make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 a4 = dv ? *reinterpret_cast<const float4*>(p.A + d * kN + nb0 + q) : make_float4(0.f, 0.f, 0.f, 0.f);
        hs[q] = h4.x; hs[q + 1] = h4.y; hs[q + 2] = h4.z; hs[q + 3] = h4.w;
        As[q] = a4.x; As[q + 1] = a4.y; As[q + 2] = a4.z; As[q + 3] = a4.w;
    }
    // the forward's readout order: blocks of BS states, each a sequential
    // fused multiply-add chain C_0 h_0 -> fma(C_1, h_1, .) -> ...; the blocks
    // summed as a balanced binary tree in state order (its top level: one
    // half of the blocks + the other)
    constexpr int BS = kReadBlock, NB = kN / kReadBlock, HB = NB / 2;
    float part[NB];
#pragma unroll
    for (int blk = 0; blk < NB; ++blk) part[blk] = 0.f;
#pragma unroll
    for (int blk = 0; blk < NB; ++blk) {
        if (NSPLIT == 2 && blk / HB != k) continue;
        float acc = 0.f;
#pragma unroll
        for (int s = 0; s < BS; ++s) {
            // j: the state's slot in this lane's registers (the lane holds states nb0 .. nb0 + NL - 1, nb0 a
            // multiple of NL, so j = n mod NL: known at compile time)
            const int n = BS * blk + s, j = n & (NL - 1);
            const float A2 = __fmul_rn(As[j], kLog2e);
            const float a = ex2(__fmul_rn(delta, A2));
            const float ub = __fmul_rn(u, Bs[n]);
            const float hv = __fmaf_rn(a, hs[j], ub);
            hs[j] = hv;
            acc = s == 0 ? __fmul_rn(Cs[n], hv) : __fmaf_rn(Cs[n], hv, acc);
        }
        part[blk] = acc;
    }
    if (dv) {
#pragma unroll
        for (int q = 0; q < NL; q += 4)
            *reinterpret_cast<float4*>(st + nb0 + q) = make_float4(hs[q], hs[q + 1], hs[q + 2], hs[q + 3]);
    }
#pragma unroll
    for (int w = 1; w < HB; w <<= 1)
#pragma unroll
        for (int i = 0; i < NB; i += 2 * w) part[i] = __fadd_rn(part[i], part[i + w]);
    float pr;
    if (NSPLIT == 1) {
        pr = __fadd_rn(part[0], part[HB]);
    } else {
        const float mine = part[k * HB];
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
    using Ly = FwdLayout<IO, AGG>;
    static unsigned long long mask = 0;
    auto kern = ssm_fwd_kernel<IO, AGG, MINB>;
    if (!ensure_smem(kern, Ly::SMEM, mask)) return -1;
    kern<<<grid, kFwdCtaThreads, Ly::SMEM, s>>>(p, mp);
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
    // the register budget: uncut when one L-group's grid fits in two CTAs
    // per SM (the scheduler gets registers for the interleaved state
    // chains), else cut to three CTAs per SM; the aggregate pass (no readout)
    // fits four
    if constexpr (AGG) {
        return launch_fwd_v<IO, AGG, 4>(p, mp, grid, s);
    } else {
        if (p.G == 1 && ctas <= 2 * (int64_t)sm_count()) return launch_fwd_v<IO, AGG, 1>(p, mp, grid, s);
        return launch_fwd_v<IO, AGG, 3>(p, mp, grid, s);
    }
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
    // the variant that runs whenever the grid can use more than 2 CTAs per SM
    return io == 0 ? blocks_per_sm(ssm_fwd_kernel<float, false, 3>, kFwdCtaThreads, FwdLayout<float>::SMEM, cache_f)
                   : blocks_per_sm(ssm_fwd_kernel<__nv_bfloat16, false, 3>, kFwdCtaThreads,
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
