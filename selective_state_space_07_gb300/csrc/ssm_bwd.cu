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
// Work split. A CTA owns 128 channels x one L-group and walks the group's
// 8-token chunks (one per saved forward state) from last to first. Lanes l
// and l^16 of a warp share the channel pair {l, l^16}: each works on both
// channels for half of the 16 states (8*(l>>4) ...), so its dB/dC
// contributions are summed over two channels in registers before they leave
// the lane. Per chunk:
//   A  each lane computes Delta, u, dp (and sigmoid(v), dy*silu'(z)) for its
//      own channel and swaps Delta, u, dp with its partner (shuffle);
//   S  per state, the two channels side by side: forward from the
//      checkpoint over the 8 tokens (a_t, h_t in registers) and the reverse
//      recurrence over them, the forward of state n+1 interleaved with the
//      reverse of state n (four independent chains in flight);
//      per-token state sums stay in registers; dB/dC contributions go
//      through a per-warp shared-memory transpose every 4 states, then a
//      per-CTA sum over warps and one vector atomic per 4 outputs;
//   E  the partners add their per-token state sums (shuffle) and each lane
//      writes dx, dz, d(dt) of its own channel.
// dA, dD, d_dt_bias accumulate in registers over the whole group.
#include "ssm_common.cuh"
#include "ssm_internal.h"

namespace ssm {

namespace {

template <typename IO> struct BwdLayout {
    static constexpr int NT = kBwdThreads;
    static constexpr int NW = NT / 32;
    static constexpr int CH = NT;                  // channels per CTA (one own channel per lane)
    static constexpr int ES = sizeof(IO);
    static constexpr int T = kCkpt;                // tokens per chunk
    static constexpr int XROW = CH * ES;           // staged row of x / z / dy (bytes)
    static constexpr int DTROW = CH * 4;
    static constexpr int BCROW = kN * ES;
    static constexpr int HROW = CH * 4;            // one state of the checkpoint tile
    static constexpr int OFF_X = 0;
    static constexpr int OFF_Z = OFF_X + T * XROW;
    static constexpr int OFF_DY = OFF_Z + T * XROW;
    static constexpr int OFF_DT = OFF_DY + T * XROW;
    static constexpr int OFF_B = OFF_DT + T * DTROW;
    static constexpr int OFF_C = OFF_B + T * BCROW;
    static constexpr int OFF_H = OFF_C + T * BCROW;
    static constexpr int STAGE = OFF_H + kN * HROW;
    static constexpr int NSTAGE = 2;
    // transpose buffer: per lane a row [4 states][dB | dC][T tokens] plus 4
    // floats of padding (row stride 68 floats: conflict-free 16-byte stores
    // down a column and 16-byte loads along a row)
    static constexpr int SPB = 4;                  // states per transpose
    static constexpr int TBROW = SPB * 2 * T + 4;
    // the reduction gives each lane of a half-warp one 4-float column of a row
    static_assert(SPB * 2 * T == 16 * 4, "a transpose row must hold 16 column quads");
    static constexpr int OFF_TB = NSTAGE * STAGE;
    static constexpr int SMEM = OFF_TB + NW * 32 * TBROW * 4 + 128;  // + slack for 128-byte alignment
    static_assert(OFF_Z % 128 == 0 && OFF_DY % 128 == 0 && OFF_DT % 128 == 0 && OFF_B % 128 == 0 &&
                      OFF_C % 128 == 0 && OFF_H % 128 == 0 && STAGE % 128 == 0, "TMA destinations on 128-byte boundaries");
};

__device__ __forceinline__ float2 f2(float a, float b) { return make_float2(a, b); }

// Column c of two consecutive staged rows (`row` bytes apart) as fp32.
template <typename IO> __device__ __forceinline__ float2 ld_pair(const char* p, int row, int c) {
    return f2(IOT<IO>::to_f(reinterpret_cast<const IO*>(p)[c]), IOT<IO>::to_f(reinterpret_cast<const IO*>(p + row)[c]));
}

// TMA descriptors of a chunk's inputs: x, z, dy, dt [B*L, D] in boxes of CH
// channels x T tokens; B, C [B*L, 16] (rows bcs elements apart) in boxes of
// 16 x T; the checkpoints [B*ceil(L/8)*8, 2D] (state pairs) in boxes of 2CH x 8.
// Elements past the last token or channel read as zero.
struct BwdMaps {
    CUtensorMap x, z, dy, dt, b, c, h;
};

template <typename IO>
__global__ void __launch_bounds__(kBwdThreads, 2)
    ssm_bwd_kernel(const BwdParams p, const __grid_constant__ BwdMaps mp) {
    using Ly = BwdLayout<IO>;
    constexpr int NT = Ly::NT, CH = Ly::CH, T = Ly::T, SPB = Ly::SPB;
    constexpr int NS = kN / 2;  // states per lane
    constexpr bool FAST = IOT<IO>::kFast;
    extern __shared__ __align__(128) char smem_raw[];
    char* smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);  // the TMA destinations
    __shared__ __align__(8) uint64_t fullb[Ly::NSTAGE];      // a chunk's copies landed
    __shared__ int aborted;                                   // a copy did not arrive within the time bound
    __shared__ __align__(16) float AT[kN * CH];               // A^T of the CTA's channels
    // double-buffered by chunk parity: a chunk's tables are written while the
    // previous chunk's are still read, and its dB/dC rows while the previous
    // chunk's are summed (one CTA barrier per chunk)
    constexpr int OBSZ = Ly::NW * 2 * T * kN;
    __shared__ __align__(16) float BT[2 * kN * T];            // B^T, C^T of the chunk (fp32)
    __shared__ __align__(16) float CT[2 * kN * T];
    __shared__ __align__(16) float OB[2 * OBSZ];              // per-warp dB/dC [warp][dB|dC][token][state]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int hk = lane >> 4;                   // states 8*hk .. 8*hk+7
    const int cO = tid;                         // own channel (slot 0)
    const int cP = (warp << 5) + (lane ^ 16);   // partner's channel (slot 1)
    const int64_t D = p.D, L = p.L;
    const int64_t d0 = (int64_t)blockIdx.x * CH;
    const int64_t dO = d0 + cO, dP = d0 + cP;
    const bool vO = dO < D, vP = dP < D;
    const int g = blockIdx.y;
    const int64_t b = blockIdx.z;
    const int64_t tb0 = (int64_t)g * p.Lg;
    const int64_t tb1 = min64(L, tb0 + p.Lg);
    const int nsub = (int)((tb1 - tb0 + T - 1) / T);
    const int64_t nck = (L + T - 1) / T;
    const bool has_z = p.has_z != 0, sp = p.sp != 0;
    float* TB = reinterpret_cast<float*>(smem + Ly::OFF_TB) + warp * 32 * Ly::TBROW;

    for (int i = tid; i < kN * CH; i += NT) {
        const int n = i / CH, c = i - n * CH;
        AT[i] = d0 + c < D ? p.A[(d0 + c) * kN + n] : 0.f;
    }
    float Gc[2][NS], dA[2][NS];
#pragma unroll
    for (int s = 0; s < NS; ++s) {
        const int n = NS * hk + s;
        float g0 = 0.f, g1 = 0.f;
        if (p.gstart) {
            const int64_t base = p.G == 1 ? b * D : (b * p.G + g) * D;
            if (vO) g0 = p.gstart[(base + dO) * kN + n];
            if (vP) g1 = p.gstart[(base + dP) * kN + n];
        }
        Gc[0][s] = g0;
        Gc[1][s] = g1;
        dA[0][s] = dA[1][s] = 0.f;
    }
    const float Dd = (vO && p.Dskip) ? p.Dskip[dO] : 0.f;
    const float bias = (vO && p.dt_bias) ? p.dt_bias[dO] : 0.f;
    const float2 D2 = f2(Dd, Dd), bias2 = f2(bias, bias);
    float2 dD2 = f2(0.f, 0.f), db2 = f2(0.f, 0.f), nf2 = f2(0.f, 0.f);  // even / odd tokens

    // one thread loads a chunk's inputs with TMA onto the buffer's mbarrier;
    // rows past the group's last token are loaded too (or read as zero past
    // the tensor's end) and ignored: they act as identity tokens below
    const unsigned chunk_bytes =
        (unsigned)(T * (Ly::XROW * (has_z ? 3 : 2) + Ly::DTROW + 2 * Ly::BCROW) + kN * Ly::HROW);
    auto issue = [&](int s, int buf) {
        if (tid != 0) return;
        char* st = smem + buf * Ly::STAGE;
        const int64_t t0 = tb0 + (int64_t)s * T;
        const int y = (int)(b * L + t0);                 // the chunk's first token row in [B*L]
        const int yh = (int)((b * nck + t0 / T) * (kN / 2));  // its checkpoint's first state-pair row
        const unsigned bar = smem_u32(&fullb[buf]);
        mbar_expect_tx(bar, chunk_bytes);
        tma_load_2d(st + Ly::OFF_X, &mp.x, (int)d0, y, bar);
        if (has_z) tma_load_2d(st + Ly::OFF_Z, &mp.z, (int)d0, y, bar);
        tma_load_2d(st + Ly::OFF_DY, &mp.dy, (int)d0, y, bar);
        tma_load_2d(st + Ly::OFF_DT, &mp.dt, (int)d0, y, bar);
        tma_load_2d(st + Ly::OFF_B, &mp.b, 0, y, bar);
        tma_load_2d(st + Ly::OFF_C, &mp.c, 0, y, bar);
        tma_load_2d(st + Ly::OFF_H, &mp.h, (int)(2 * d0), yh, bar);
    };
    if (tid == 0) {
        for (int q = 0; q < Ly::NSTAGE; ++q) mbar_init(smem_u32(&fullb[q]), 1);
        mbar_fence_init();
        aborted = 0;
    }
    __syncthreads();

    // dB / dC of chunk s from its per-warp rows: sum the warps, one vector atomic per 4 outputs
    auto flush_dbdc = [&](int s, const float* ob) {
        if (tid >= 2 * T * (kN / 4)) return;
        const int64_t t0 = tb0 + (int64_t)s * T;
        const int rows = (int)min64(T, tb1 - t0);
        const int type = tid / (T * kN / 4), rem = tid % (T * kN / 4);
        const int tk = rem / (kN / 4), n0 = (rem % (kN / 4)) * 4;
        if (tk < rows) {
            float4 s4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int w = 0; w < Ly::NW; ++w) {
                const float4 v = *reinterpret_cast<const float4*>(ob + ((w * 2 + type) * T + tk) * kN + n0);
                s4.x += v.x; s4.y += v.y; s4.z += v.z; s4.w += v.w;
            }
            red_add_v4((type == 0 ? p.dB : p.dC) + (b * L + t0 + tk) * kN + n0, s4);
        }
    };

    if (nsub > 0) issue(nsub - 1, 0);
    for (int it = 0; it < nsub; ++it) {
        const int s_ = nsub - 1 - it, cb = it & 1;
        char* st = smem + cb * Ly::STAGE;
        float* BTc = BT + cb * kN * T;
        float* CTc = CT + cb * kN * T;
        float* OBc = OB + cb * OBSZ;
        // every thread waits for the chunk (bounded); after a timeout the block
        // stops waiting but keeps the barrier sequence (its results are flagged invalid)
        if (!aborted && !mbar_wait_bounded(smem_u32(&fullb[cb]), (unsigned)((it >> 1) & 1))) {
            aborted = 1;
            if (p.status) atomicOr(p.status, kStatusTimeout);
        }
        const int64_t t0 = tb0 + (int64_t)s_ * T;
        const int rows = (int)min64(T, tb1 - t0);
        {
            const IO* Braw = reinterpret_cast<const IO*>(st + Ly::OFF_B);
            const IO* Craw = reinterpret_cast<const IO*>(st + Ly::OFF_C);
            for (int i = tid; i < kN * T; i += NT) {
                const int n = i / T, tok = i - n * T;
                const bool live = tok < rows;  // rows past the end belong to other tokens: zero, not read
                BTc[i] = live ? IOT<IO>::to_f(Braw[tok * kN + n]) : 0.f;
                CTc[i] = live ? IOT<IO>::to_f(Craw[tok * kN + n]) : 0.f;
            }
        }

        // ---- A: per-token quantities of the own channel, a token pair at a
        // time (packed f32x2); tokens past the end act as identity (a = 1, no
        // input, no adjoint input, nothing accumulated)
        const bool full = rows == T;
        float2 Dl[2][T / 2], Ul[2][T / 2], Pl[2][T / 2];
        float2 sgp[T / 2], ddp[T / 2], Xl[T / 2];  // x stays in registers for phase E
#pragma unroll
        for (int m = 0; m < T / 2; ++m) {
            const int t = 2 * m;
            const float2 xv = ld_pair<IO>(st + Ly::OFF_X + t * Ly::XROW, Ly::XROW, cO);
            const float2 dyv = ld_pair<IO>(st + Ly::OFF_DY + t * Ly::XROW, Ly::XROW, cO);
            const float2 dtv = ld_pair<float>(st + Ly::OFF_DT + t * Ly::DTROW, Ly::DTROW, cO);
            float2 sgv;
            float2 dl = delta_sig2<FAST>(dtv, bias2, sp, &sgv);
            float2 pl = dyv, dyds = f2(0.f, 0.f);
            if (has_z) {
                const float2 zv = ld_pair<IO>(st + Ly::OFF_Z + t * Ly::XROW, Ly::XROW, cO);
                const float2 sz = sigmoid2<FAST>(zv);
                pl = __fmul2_rn(dyv, __fmul2_rn(zv, sz));
                // dy * silu'(z) = dy * s (1 + z (1 - s))
                const float2 one = f2(1.f, 1.f);
                dyds = __fmul2_rn(dyv, __fmul2_rn(sz, __ffma2_rn(zv, __fadd2_rn(one, f2(-sz.x, -sz.y)), one)));
            }
            float2 ul = __fmul2_rn(dl, xv);
            Xl[m] = xv;
            if (!full) {
                const bool l0 = t < rows, l1 = t + 1 < rows;
                dl = f2(l0 ? dl.x : 0.f, l1 ? dl.y : 0.f);
                ul = f2(l0 ? ul.x : 0.f, l1 ? ul.y : 0.f);
                pl = f2(l0 ? pl.x : 0.f, l1 ? pl.y : 0.f);
                sgv = f2(l0 ? sgv.x : 0.f, l1 ? sgv.y : 0.f);
                dyds = f2(l0 ? dyds.x : 0.f, l1 ? dyds.y : 0.f);
            }
            Dl[0][m] = dl;
            Ul[0][m] = ul;
            Pl[0][m] = pl;
            sgp[m] = sgv;
            ddp[m] = dyds;
        }
#pragma unroll
        for (int m = 0; m < T / 2; ++m) {
            Dl[1][m] = f2(__shfl_xor_sync(0xffffffffu, Dl[0][m].x, 16), __shfl_xor_sync(0xffffffffu, Dl[0][m].y, 16));
            Ul[1][m] = f2(__shfl_xor_sync(0xffffffffu, Ul[0][m].x, 16), __shfl_xor_sync(0xffffffffu, Ul[0][m].y, 16));
            Pl[1][m] = f2(__shfl_xor_sync(0xffffffffu, Pl[0][m].x, 16), __shfl_xor_sync(0xffffffffu, Pl[0][m].y, 16));
        }
        // the chunk's B^T / C^T are ready; every thread is done with the previous
        // chunk (its staging buffer is free, its dB/dC rows are complete)
        __syncthreads();
        if (s_ > 0) issue(s_ - 1, cb ^ 1);  // into the buffer the previous chunk used
        if (it > 0) flush_dbdc(s_ + 1, OB + (cb ^ 1) * OBSZ);

        // ---- S: per state, both channels; per-token state sums in registers
        float2 S1[2][T / 2], S2[2][T / 2], S3[2][T / 2];
#pragma unroll
        for (int sl = 0; sl < 2; ++sl)
#pragma unroll
            for (int m = 0; m < T / 2; ++m) S1[sl][m] = S2[sl][m] = S3[sl][m] = f2(0.f, 0.f);
        const float* hck = reinterpret_cast<const float*>(st + Ly::OFF_H);

        // the forward recomputation of state s+1 runs interleaved with the
        // reverse recurrence of state s (independent chains for the scheduler)
        float2 aS[2][2][T / 2], hS[2][2][T / 2], bS[2][T / 2];  // [state parity][channel slot][token pair]
        float A2s[2][2], hps[2][2];
        auto load_state = [&](int n, int k) {
            const float4 b4a = *reinterpret_cast<const float4*>(BTc + n * T);
            const float4 b4b = *reinterpret_cast<const float4*>(BTc + n * T + 4);
            bS[k][0] = f2(b4a.x, b4a.y); bS[k][1] = f2(b4a.z, b4a.w);
            bS[k][2] = f2(b4b.x, b4b.y); bS[k][3] = f2(b4b.z, b4b.w);
#pragma unroll
            for (int sl = 0; sl < 2; ++sl) {
                const int c = sl ? cP : cO;
                A2s[k][sl] = __fmul_rn(AT[n * CH + c], kLog2e);
                hps[k][sl] = hck[((n >> 1) * CH + c) * 2 + (n & 1)];  // [state pair][channel][2]
            }
        };
        auto fwd_pair = [&](int k, int m) {
#pragma unroll
            for (int sl = 0; sl < 2; ++sl) {
                const float2 arg = __fmul2_rn(Dl[sl][m], f2(A2s[k][sl], A2s[k][sl]));
                aS[k][sl][m] = f2(ex2(arg.x), ex2(arg.y));
                const float2 ub = __fmul2_rn(Ul[sl][m], bS[k][m]);
                const float h0v = __fmaf_rn(aS[k][sl][m].x, hps[k][sl], ub.x);
                const float h1v = __fmaf_rn(aS[k][sl][m].y, h0v, ub.y);
                hps[k][sl] = h1v;
                hS[k][sl][m] = f2(h0v, h1v);
            }
        };
        load_state(NS * hk, 0);
#pragma unroll
        for (int m = 0; m < T / 2; ++m) fwd_pair(0, m);

#pragma unroll
        for (int s = 0; s < NS; ++s) {
            const int n = NS * hk + s, k = s & 1;
            const bool more = s + 1 < NS;
            const float4 c4a = *reinterpret_cast<const float4*>(CTc + n * T);
            const float4 c4b = *reinterpret_cast<const float4*>(CTc + n * T + 4);
            const float2 cc[4] = {f2(c4a.x, c4a.y), f2(c4a.z, c4a.w), f2(c4b.x, c4b.y), f2(c4b.z, c4b.w)};
            float2 Ap[2];
#pragma unroll
            for (int sl = 0; sl < 2; ++sl) {
                const float An = AT[n * CH + (sl ? cP : cO)];
                Ap[sl] = f2(An, An);
            }
            if (more) load_state(n + 1, k ^ 1);
            float2 vb[T / 2], vc[T / 2];
            // reverse: E_t = a_{t+1} E_{t+1} + dp_t C_t, carry Gc = a_{t+1} E_{t+1}
            float E[2] = {Gc[0][s], Gc[1][s]}, anext[2] = {1.f, 1.f};
            float2 dAp[2] = {f2(0.f, 0.f), f2(0.f, 0.f)};
#pragma unroll
            for (int m = T / 2 - 1; m >= 0; --m) {
#pragma unroll
                for (int sl = 0; sl < 2; ++sl) {
                    const float2 rr = __fmul2_rn(Pl[sl][m], cc[m]);
                    const float e1 = __fmaf_rn(anext[sl], E[sl], rr.y);
                    const float e0 = __fmaf_rn(aS[k][sl][m].y, e1, rr.x);
                    E[sl] = e0;
                    anext[sl] = aS[k][sl][m].x;
                    const float2 E2 = f2(e0, e1);
                    if (sl == 0) {
                        vb[m] = __fmul2_rn(E2, Ul[0][m]);
                        vc[m] = __fmul2_rn(Pl[0][m], hS[k][0][m]);
                    } else {
                        vb[m] = __ffma2_rn(E2, Ul[1][m], vb[m]);
                        vc[m] = __ffma2_rn(Pl[1][m], hS[k][1][m], vc[m]);
                    }
                    S1[sl][m] = __ffma2_rn(E2, bS[k][m], S1[sl][m]);
                    // a_t h_{t-1} = h_t - u_t B_t
                    const float2 q = __ffma2_rn(f2(-Ul[sl][m].x, -Ul[sl][m].y), bS[k][m], hS[k][sl][m]);
                    const float2 w = __fmul2_rn(E2, q);
                    dAp[sl] = __ffma2_rn(Dl[sl][m], w, dAp[sl]);
                    S2[sl][m] = __ffma2_rn(Ap[sl], w, S2[sl][m]);
                    S3[sl][m] = __ffma2_rn(cc[m], hS[k][sl][m], S3[sl][m]);
                }
                if (more) fwd_pair(k ^ 1, T / 2 - 1 - m);
            }
#pragma unroll
            for (int sl = 0; sl < 2; ++sl) {
                Gc[sl][s] = __fmul_rn(anext[sl], E[sl]);
                dA[sl][s] += __fadd_rn(dAp[sl].x, dAp[sl].y);
            }
            // dB/dC contributions of this state, summed over the two channels
            const int sb = s % SPB;
            float* row = TB + lane * Ly::TBROW + sb * 2 * T;
            *reinterpret_cast<float4*>(row + 0) = make_float4(vb[0].x, vb[0].y, vb[1].x, vb[1].y);
            *reinterpret_cast<float4*>(row + 4) = make_float4(vb[2].x, vb[2].y, vb[3].x, vb[3].y);
            *reinterpret_cast<float4*>(row + T) = make_float4(vc[0].x, vc[0].y, vc[1].x, vc[1].y);
            *reinterpret_cast<float4*>(row + T + 4) = make_float4(vc[2].x, vc[2].y, vc[3].x, vc[3].y);
            if (sb == SPB - 1) {
                __syncwarp();
                // lane (hk, o) sums its half-warp's 16 rows at column quad o:
                // state s-3 + o/4, dB or dC by (o/2)&1, tokens 4*(o&1) .. +3
                const int o = lane & 15;
                const float* col = TB + (16 * hk) * Ly::TBROW + 4 * o;
                float4 acc = *reinterpret_cast<const float4*>(col);
#pragma unroll
                for (int r = 1; r < 16; ++r) {
                    const float4 v = *reinterpret_cast<const float4*>(col + r * Ly::TBROW);
                    const float2 lo = __fadd2_rn(f2(acc.x, acc.y), f2(v.x, v.y));
                    const float2 hi = __fadd2_rn(f2(acc.z, acc.w), f2(v.z, v.w));
                    acc = make_float4(lo.x, lo.y, hi.x, hi.y);
                }
                const int nn = NS * hk + s - (SPB - 1) + (o >> 2), type = (o >> 1) & 1, tk = (o & 1) * 4;
                float* ob = OBc + ((warp * 2 + type) * T + tk) * kN + nn;
                ob[0] = acc.x;
                ob[kN] = acc.y;
                ob[2 * kN] = acc.z;
                ob[3 * kN] = acc.w;
                __syncwarp();
            }
        }

        // ---- E: the partners add their per-token state sums; each lane
        // finishes its own channel
#pragma unroll
        for (int m = 0; m < T / 2; ++m) {
            S1[0][m] = __fadd2_rn(S1[0][m], f2(__shfl_xor_sync(0xffffffffu, S1[1][m].x, 16),
                                               __shfl_xor_sync(0xffffffffu, S1[1][m].y, 16)));
            S2[0][m] = __fadd2_rn(S2[0][m], f2(__shfl_xor_sync(0xffffffffu, S2[1][m].x, 16),
                                               __shfl_xor_sync(0xffffffffu, S2[1][m].y, 16)));
            S3[0][m] = __fadd2_rn(S3[0][m], f2(__shfl_xor_sync(0xffffffffu, S3[1][m].x, 16),
                                               __shfl_xor_sync(0xffffffffu, S3[1][m].y, 16)));
        }
        if (vO) {
#pragma unroll
            for (int m = 0; m < T / 2; ++m) {
                const int t = 2 * m;
                float2 xv = Xl[m];
                if (!full) xv = f2(t < rows ? xv.x : 0.f, t + 1 < rows ? xv.y : 0.f);
                const float2 s1 = S1[0][m], s2 = S2[0][m];
                const float2 dxv = __ffma2_rn(Pl[0][m], D2, __fmul2_rn(Dl[0][m], s1));
                const float2 ddelta = __ffma2_rn(xv, s1, s2);
                float2 ddtv = sp ? __fmul2_rn(ddelta, sgp[m]) : ddelta;
                if (!full) ddtv = f2(t < rows ? ddtv.x : 0.f, t + 1 < rows ? ddtv.y : 0.f);
                dD2 = __ffma2_rn(Pl[0][m], xv, dD2);
                db2 = __fadd2_rn(db2, ddtv);
                nf2 = __ffma2_rn(dxv, f2(0.f, 0.f), __ffma2_rn(ddtv, f2(0.f, 0.f), nf2));
                IO* dxp = reinterpret_cast<IO*>(p.dx) + (b * L + t0 + t) * D + dO;
                float* ddp_ = p.ddt + (b * L + t0 + t) * D + dO;
                IO* dzp = reinterpret_cast<IO*>(p.dz) + (b * L + t0 + t) * D + dO;
                float2 dzv = f2(0.f, 0.f);
                if (has_z) {
                    dzv = __fmul2_rn(__ffma2_rn(D2, xv, S3[0][m]), ddp[m]);
                    nf2 = __ffma2_rn(dzv, f2(0.f, 0.f), nf2);
                }
                if (full || t < rows) {
                    dxp[0] = IOT<IO>::from_f(dxv.x);
                    ddp_[0] = ddtv.x;
                    if (has_z) dzp[0] = IOT<IO>::from_f(dzv.x);
                }
                if (full || t + 1 < rows) {
                    dxp[D] = IOT<IO>::from_f(dxv.y);
                    ddp_[D] = ddtv.y;
                    if (has_z) dzp[D] = IOT<IO>::from_f(dzv.y);
                }
            }
        }
    }
    __syncthreads();  // the last chunk's dB/dC rows are complete
    if (nsub > 0) flush_dbdc(0, OB + ((nsub - 1) & 1) * OBSZ);

    // ---- reductions over the group
#pragma unroll
    for (int s = 0; s < NS; ++s) {
        const int n = NS * hk + s;
        if (vO) atomicAdd(p.dA + dO * kN + n, dA[0][s]);
        if (vP) atomicAdd(p.dA + dP * kN + n, dA[1][s]);
        if (g == 0 && p.dh0) {
            if (vO) p.dh0[(b * D + dO) * kN + n] = Gc[0][s];
            if (vP) p.dh0[(b * D + dP) * kN + n] = Gc[1][s];
        }
    }
    if (vO) {
        atomicAdd(p.dD + dO, __fadd_rn(dD2.x, dD2.y));
        atomicAdd(p.ddt_bias + dO, __fadd_rn(db2.x, db2.y));
    }
    flag_nonfinite(p.status, __fadd_rn(nf2.x, nf2.y));
}

// Chunk aggregate of the reverse recurrence for groups 1..G-1: with the
// adjoint carry set to zero at the group's end, the carry the group passes to
// its left neighbour is Q = a_{t0} E_{t0}, and unrolling E_t = a_{t+1} E_{t+1}
// + dp_t C_t gives it in closed form,
//   Q_n = sum_t exp(A_n Lambda_t) dp_t C_t,n,  Lambda_t = Delta_{t0} + ... + Delta_t,
// every term independent of the others (the product of the decays up to t is
// the exponential of A times the prefix sum of Delta). The kernel walks the
// group from its start, keeps the running Lambda per channel and publishes
// Q and the group's sum of Delta. The carry entering group g-1 from the right
// is then exp(A*sum Delta_g) * carry_g + Q_g. Layout as in the forward: a lane
// pair per channel, each lane 8 states and 8 of a tile's 16 tokens for the
// per-token work; C staged state-major (broadcast loads).
template <typename IO> struct BwdAggLayout {
    static constexpr int NT = kBwdThreads;
    static constexpr int CH = NT / 2;
    static constexpr int ES = sizeof(IO);
    static constexpr int XROW = CH * ES, DTROW = CH * 4, BCROW = kN * ES;
    static constexpr int OFF_Z = 0, OFF_DY = kCK * XROW, OFF_DT = 2 * kCK * XROW, OFF_C = OFF_DT + kCK * DTROW;
    static constexpr int STAGE = OFF_C + kCK * BCROW;
    static constexpr int NSTAGE = 3;
    static constexpr int SMEM = NSTAGE * STAGE + 128;  // + slack for 128-byte alignment
    static constexpr int ROW = 2 * kCK + 4;  // per-channel row [Lambda 0..15 | dp 0..15], padded
    static_assert(OFF_DY % 128 == 0 && OFF_DT % 128 == 0 && OFF_C % 128 == 0 && STAGE % 128 == 0,
                  "TMA destinations on 128-byte boundaries");
};

// TMA descriptors of a tile's inputs: z, dy, dt [B*L, D] in boxes of CH
// channels x 16 tokens, C [B*L, 16] in boxes of 16 x 16.
struct AggMaps {
    CUtensorMap z, dy, dt, c;
};

template <typename IO>
__global__ void __launch_bounds__(kBwdThreads) ssm_bwd_agg_kernel(const BwdParams p, const __grid_constant__ AggMaps mp) {
    using Ly = BwdAggLayout<IO>;
    constexpr int NT = Ly::NT, CH = Ly::CH, T = kCK, NS = kN / 2;
    constexpr bool FAST = IOT<IO>::kFast;
    extern __shared__ __align__(128) char smem_raw[];
    char* smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);  // the TMA destinations
    __shared__ __align__(8) uint64_t fullb[Ly::NSTAGE];
    __shared__ int aborted;
    // C^T double-buffered by tile parity (one CTA barrier per tile); a
    // channel's Lambda / dp row is shared by its lane pair only (warp syncs)
    __shared__ __align__(16) float CT2[2 * kN * T];
    __shared__ __align__(16) float DP[CH * Ly::ROW];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int hk = lane >> 4;
    const int c = warp * 16 + (lane & 15);
    const int64_t D = p.D, L = p.L;
    const int64_t d0 = (int64_t)blockIdx.x * CH, d = d0 + c;
    const bool dv = d < D;
    const int g = blockIdx.y + 1;  // groups 1..G-1
    const int64_t b = blockIdx.z;
    const int64_t tb0 = (int64_t)g * p.Lg, tb1 = min64(L, tb0 + p.Lg);
    const int ntile = (int)((tb1 - tb0 + T - 1) / T);
    const bool has_z = p.has_z != 0, sp = p.sp != 0;

    float2 A2p[NS], acc[NS];  // A log2(e) twice; per state the even- and odd-token partial sums of Q
#pragma unroll
    for (int s = 0; s < NS; ++s) {
        const float a2 = dv ? __fmul_rn(p.A[d * kN + NS * hk + s], kLog2e) : 0.f;
        A2p[s] = make_float2(a2, a2);
        acc[s] = make_float2(0.f, 0.f);
    }
    const float bias = (dv && p.dt_bias) ? p.dt_bias[d] : 0.f;
    const unsigned tile_bytes = (unsigned)(T * (Ly::XROW * (has_z ? 2 : 1) + Ly::DTROW + Ly::BCROW));
    auto issue = [&](int j) {  // tile j counted from the group's start
        if (tid != 0) return;
        const int slot = j % Ly::NSTAGE;
        char* st = smem + slot * Ly::STAGE;
        const int y = (int)(b * L + tb0 + (int64_t)j * T);
        const unsigned bar = smem_u32(&fullb[slot]);
        mbar_expect_tx(bar, tile_bytes);
        if (has_z) tma_load_2d(st + Ly::OFF_Z, &mp.z, (int)d0, y, bar);
        tma_load_2d(st + Ly::OFF_DY, &mp.dy, (int)d0, y, bar);
        tma_load_2d(st + Ly::OFF_DT, &mp.dt, (int)d0, y, bar);
        tma_load_2d(st + Ly::OFF_C, &mp.c, 0, y, bar);
    };
    if (tid == 0) {
        for (int q = 0; q < Ly::NSTAGE; ++q) mbar_init(smem_u32(&fullb[q]), 1);
        mbar_fence_init();
        aborted = 0;
    }
    __syncthreads();
    float* dp = DP + c * Ly::ROW;
    float lam = 0.f;  // Lambda at the end of the previous tile (the same in both lanes of a pair)
#pragma unroll
    for (int q = 0; q < Ly::NSTAGE - 1; ++q)
        if (q < ntile) issue(q);
    for (int j = 0; j < ntile; ++j) {
        char* st = smem + (j % Ly::NSTAGE) * Ly::STAGE;
        if (j + Ly::NSTAGE - 1 < ntile) issue(j + Ly::NSTAGE - 1);
        if (!aborted && !mbar_wait_bounded(smem_u32(&fullb[j % Ly::NSTAGE]), (unsigned)((j / Ly::NSTAGE) & 1))) {
            aborted = 1;
            if (p.status) atomicOr(p.status, kStatusTimeout);
        }
        float* CT = CT2 + (j & 1) * kN * T;
        const int64_t t0 = tb0 + (int64_t)j * T;
        const int rows = (int)min64(T, tb1 - t0);
        {
            const IO* Craw = reinterpret_cast<const IO*>(st + Ly::OFF_C);
            for (int i = tid; i < kN * T; i += NT) {
                const int n = i / T, tok = i - n * T;
                CT[i] = tok < rows ? IOT<IO>::to_f(Craw[tok * kN + n]) : 0.f;  // rows past the end: zero
            }
        }
        {
            // Delta and dp of this lane's 8 tokens, a token pair at a time;
            // tokens past the end add nothing to Lambda and have dp = 0
            const float2 bias2 = make_float2(bias, bias);
            float dl[NS], pl[NS];
#pragma unroll
            for (int i = 0; i < NS / 2; ++i) {
                const int t = NS * hk + 2 * i;
                const float2 dtv = ld_pair<float>(st + Ly::OFF_DT + t * Ly::DTROW, Ly::DTROW, c);
                const float2 dyv = ld_pair<IO>(st + Ly::OFF_DY + t * Ly::XROW, Ly::XROW, c);
                const float2 delta = delta2<FAST>(dtv, bias2, sp);
                float2 dpv = dyv;
                if (has_z) {
                    const float2 zv = ld_pair<IO>(st + Ly::OFF_Z + t * Ly::XROW, Ly::XROW, c);
                    dpv = __fmul2_rn(dyv, __fmul2_rn(zv, sigmoid2<FAST>(zv)));
                }
                const bool l0 = t < rows, l1 = t + 1 < rows;
                dl[2 * i] = l0 ? delta.x : 0.f;
                dl[2 * i + 1] = l1 ? delta.y : 0.f;
                pl[2 * i] = l0 ? dpv.x : 0.f;
                pl[2 * i + 1] = l1 ? dpv.y : 0.f;
            }
            // the lane's inclusive prefix over its 8 tokens; the second lane
            // of the pair starts after the first lane's 8
#pragma unroll
            for (int i = 1; i < NS; ++i) dl[i] = __fadd_rn(dl[i - 1], dl[i]);
            const float own = dl[NS - 1], other = __shfl_xor_sync(0xffffffffu, own, 16);
            const float base = hk ? __fadd_rn(lam, other) : lam;
#pragma unroll
            for (int i = 0; i < NS; ++i) dl[i] = __fadd_rn(base, dl[i]);
            lam = __fadd_rn(lam, __fadd_rn(own, other));  // the same in both lanes: s0 + s1 = s1 + s0
            *reinterpret_cast<float4*>(dp + NS * hk) = make_float4(dl[0], dl[1], dl[2], dl[3]);
            *reinterpret_cast<float4*>(dp + NS * hk + 4) = make_float4(dl[4], dl[5], dl[6], dl[7]);
            *reinterpret_cast<float4*>(dp + T + NS * hk) = make_float4(pl[0], pl[1], pl[2], pl[3]);
            *reinterpret_cast<float4*>(dp + T + NS * hk + 4) = make_float4(pl[4], pl[5], pl[6], pl[7]);
        }
        // the tile's C^T and Lambda / dp rows are ready; every thread is done
        // with the previous tile (so its staging slot may be refilled)
        __syncthreads();
        float2 Lm[T / 2], Pl[T / 2];
#pragma unroll
        for (int q = 0; q < T / 4; ++q) {
            const float4 lq = *reinterpret_cast<const float4*>(dp + 4 * q);
            const float4 pq = *reinterpret_cast<const float4*>(dp + T + 4 * q);
            Lm[2 * q] = make_float2(lq.x, lq.y);
            Lm[2 * q + 1] = make_float2(lq.z, lq.w);
            Pl[2 * q] = make_float2(pq.x, pq.y);
            Pl[2 * q + 1] = make_float2(pq.z, pq.w);
        }
        // Q_n += exp2(A_n log2(e) Lambda_t) * dp_t C_t,n: no term waits for another.
        // The first SSM_AGG_FMA_STATES of a lane's states take the FMA-pipe 2^x
        // instead of the MUFU (0 = none).
#ifndef SSM_AGG_FMA_STATES
#define SSM_AGG_FMA_STATES 0
#endif
        constexpr int kAggFma = SSM_AGG_FMA_STATES;
#pragma unroll
        for (int s = 0; s < NS; ++s) {
            const int n = NS * hk + s;
#pragma unroll
            for (int q = 0; q < T / 4; ++q) {
                const float4 c4 = *reinterpret_cast<const float4*>(CT + n * T + 4 * q);
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const int m = 2 * q + h2;
                    const float2 cc = h2 ? make_float2(c4.z, c4.w) : make_float2(c4.x, c4.y);
                    const float2 arg = __fmul2_rn(Lm[m], A2p[s]);
                    const float2 r = __fmul2_rn(Pl[m], cc);
                    const float2 e = s < kAggFma ? make_float2(ex2_fma(arg.x), ex2_fma(arg.y))
                                                 : make_float2(ex2(arg.x), ex2(arg.y));
                    acc[s] = __ffma2_rn(e, r, acc[s]);
                }
            }
        }
        __syncwarp();  // the lane pair is done with its Lambda / dp row before the next tile rewrites it
    }
    if (dv) {
        float* Q = p.aggQ + ((b * p.G + g) * D + d) * kN + NS * hk;
#pragma unroll
        for (int s = 0; s < NS; ++s) Q[s] = __fadd_rn(acc[s].x, acc[s].y);
        if (hk == 0) p.aggS[(b * p.G + g) * D + d] = lam;
    }
}

template <typename IO> constexpr CUtensorMapDataType io_map_type() {
    return sizeof(IO) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
}

template <typename IO> int launch_bwd_t(const BwdParams& p, cudaStream_t s) {
    using Ly = BwdLayout<IO>;
    auto kern = ssm_bwd_kernel<IO>;
    static unsigned long long mask = 0;
    if (!ensure_smem(kern, Ly::SMEM, mask)) return -1;
    if (p.B == 0 || p.D == 0 || p.G == 0) return 0;
    const CUtensorMapDataType io = io_map_type<IO>(), f32 = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    const CUtensorMapSwizzle none = CU_TENSOR_MAP_SWIZZLE_NONE;
    const int64_t rows = p.B * p.L, ES = sizeof(IO), hrows = p.B * ((p.L + Ly::T - 1) / Ly::T) * (kN / 2);
    BwdMaps mp;
    if (!encode_2d(&mp.x, io, p.x, p.D, rows, p.D * ES, Ly::CH, Ly::T, none) ||
        !encode_2d(&mp.dy, io, p.dy, p.D, rows, p.D * ES, Ly::CH, Ly::T, none) ||
        !encode_2d(&mp.dt, f32, p.dt, p.D, rows, p.D * 4, Ly::CH, Ly::T, none) ||
        !encode_2d(&mp.b, io, p.Bm, kN, rows, p.bcs * ES, kN, Ly::T, none) ||
        !encode_2d(&mp.c, io, p.Cm, kN, rows, p.bcs * ES, kN, Ly::T, none) ||
        !encode_2d(&mp.h, f32, p.ckpt, 2 * p.D, hrows, p.D * 8, 2 * Ly::CH, kN / 2, none))
        return -1;
    mp.z = mp.x;
    if (p.has_z && !encode_2d(&mp.z, io, p.z, p.D, rows, p.D * ES, Ly::CH, Ly::T, none)) return -1;
    dim3 grid((unsigned)((p.D + Ly::CH - 1) / Ly::CH), (unsigned)p.G, (unsigned)p.B);
    kern<<<grid, kBwdThreads, Ly::SMEM, s>>>(p, mp);
    return cudaGetLastError() == cudaSuccess ? 1 : -1;
}

template <typename IO> int launch_bwd_agg_t(const BwdParams& p, cudaStream_t s) {
    using Ly = BwdAggLayout<IO>;
    auto kern = ssm_bwd_agg_kernel<IO>;
    static unsigned long long mask = 0;
    if (!ensure_smem(kern, Ly::SMEM, mask)) return -1;
    if (p.B == 0 || p.D == 0 || p.G <= 1) return 0;
    const CUtensorMapDataType io = io_map_type<IO>(), f32 = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    const CUtensorMapSwizzle none = CU_TENSOR_MAP_SWIZZLE_NONE;
    const int64_t rows = p.B * p.L, ES = sizeof(IO);
    AggMaps mp;
    if (!encode_2d(&mp.dy, io, p.dy, p.D, rows, p.D * ES, Ly::CH, kCK, none) ||
        !encode_2d(&mp.dt, f32, p.dt, p.D, rows, p.D * 4, Ly::CH, kCK, none) ||
        !encode_2d(&mp.c, io, p.Cm, kN, rows, p.bcs * ES, kN, kCK, none))
        return -1;
    mp.z = mp.dy;
    if (p.has_z && !encode_2d(&mp.z, io, p.z, p.D, rows, p.D * ES, Ly::CH, kCK, none)) return -1;
    dim3 grid((unsigned)((p.D + Ly::CH - 1) / Ly::CH), (unsigned)(p.G - 1), (unsigned)p.B);
    kern<<<grid, kBwdThreads, Ly::SMEM, s>>>(p, mp);
    return cudaGetLastError() == cudaSuccess ? 1 : -1;
}

}  // namespace

int bwd_blocks_per_sm(int io) {
    static int cache[2][64] = {{0}};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    int& c = cache[io ? 1 : 0][dev & 63];
    if (c == 0) {
        int v = 0;
        cudaError_t e;
        if (io == 0) {
            auto kern = ssm_bwd_kernel<float>;
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, BwdLayout<float>::SMEM);
            if (e == cudaSuccess)
                e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, kern, kBwdThreads, BwdLayout<float>::SMEM);
        } else {
            auto kern = ssm_bwd_kernel<__nv_bfloat16>;
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     BwdLayout<__nv_bfloat16>::SMEM);
            if (e == cudaSuccess)
                e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, kern, kBwdThreads,
                                                                  BwdLayout<__nv_bfloat16>::SMEM);
        }
        c = (e == cudaSuccess && v > 0) ? v : 1;
    }
    return c;
}
int bwd_channels_per_cta() { return BwdLayout<float>::CH; }

int launch_bwd(int io, const BwdParams& p, cudaStream_t s) {
    return io == 0 ? launch_bwd_t<float>(p, s) : launch_bwd_t<__nv_bfloat16>(p, s);
}

int launch_bwd_agg(int io, const BwdParams& p, cudaStream_t s) {
    return io == 0 ? launch_bwd_agg_t<float>(p, s) : launch_bwd_agg_t<__nv_bfloat16>(p, s);
}

}  // namespace ssm
