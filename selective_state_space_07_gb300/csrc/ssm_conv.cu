// Causal depthwise conv1d + SiLU in front of the S6 scan, on sm_103a.
//
// rustytorch commit log, "MambaBlock" S6 forward commit: "in_proj -> causal
// depthwise conv1d -> SiLU -> x_proj -> ..."; the MambaRecurrence commit
// carries the "conv-ring" state between steps. Per (b, d) channel, with the
// K-1 inputs before t = 0 in `state` (zeros when absent):
//   pre_t = bias[d] + sum_{k<K} w[d,k] * in_{t-(K-1)+k},   x_t = pre_t * sigmoid(pre_t)
// Backward for loss = <dx, x>:
//   dpre_t = dx_t * silu'(pre_t);  dxin_s = sum_k w[d,k] * dpre_{s+(K-1)-k}
//   dw[d,k] = sum_{b,t} dpre_t * in_{t-(K-1)+k};  dbias[d] = sum_{b,t} dpre_t
//
// The op streams [B,L,D] activations once each way, so it is bound by HBM,
// and what decides its speed is how many bytes are in flight. Work is cut
// per warp: a warp owns a column of 256 channels (8 per lane: one 16-byte
// bf16 vector per token row, a 512-byte row per warp) of one batch row and
// an even share of its tokens, with the number of shares picked so that one
// wave of resident warps covers the whole problem. Each lane streams its own
// bytes of the rows through a 3-stage shared-memory ring with cp.async (the
// copies are the lane's own, so per-thread wait_group is the only
// synchronisation), keeping two stages of rows in flight without holding
// registers for them. The K-1 inputs before a share come from the halo rows
// (or the carried state) with plain loads; channel pairs are computed as
// packed f32x2 arithmetic. The backward streams xin and dx together, walks
// K-1 rows past its share to finish dxin of its last tokens, writes the
// state's gradient from the share that starts at t = 0, and folds dw / dbias
// into registers with one vector reduction per channel at the end.
#include "ssm_common.cuh"
#include "ssm_internal.h"

namespace ssm {

namespace {

constexpr int kConvWarps = kConvThreads / 32;
constexpr int kConvStage = 4096;  // bytes of one ring stage of a warp

// Per-lane row geometry for CL channels of I/O type IO: VB bytes per token
// row, moved as NV vectors of VS bytes; P channel pairs.
template <typename IO, int CL> struct Lane {
    static constexpr int VB = (int)sizeof(IO) * CL;
    static constexpr int VS = VB < 16 ? VB : 16;
    static constexpr int NV = VB / VS;
    static constexpr int W = VB / 4;  // 32-bit words
    static constexpr int P = CL / 2;
    static_assert(VS == 8 || VS == 16, "8- or 16-byte vectors");
};

// Ring geometry per warp: NS stages of 4 KB; a stage holds R token rows of
// each stream; one stream's row is NV vectors per lane stored
// [vector][lane], so every shared load of a warp reads 32 * VS contiguous
// bytes. NS-1 stages are in flight while one is read.
template <typename IO, int STREAMS, int CL, int STAGES> struct ConvTile {
    using G = Lane<IO, CL>;
    static constexpr int ROW = G::NV * 32 * G::VS;
    static constexpr int R = kConvStage / (STREAMS * ROW);
    static constexpr int NS = STAGES;
    static constexpr int WARP = NS * kConvStage;
    static constexpr int SMEM = kConvWarps * WARP;
    static constexpr int WARP_CH = 32 * CL;
    static_assert(R >= 1 && R * STREAMS * ROW == kConvStage, "whole rows per stage");
};

// Both passes keep 8 channels per lane (16-byte bf16 rows; 4 per lane
// measured slower: twice the per-row overhead per channel). The forward
// fits 3 CTAs per SM and keeps 3 of its 4 stages in flight (144 KB of rows
// per SM); the backward, whose dw / dbias accumulators take 218 registers,
// fits 2 CTAs and keeps 2 of its 3 two-stream stages in flight.
constexpr int kFwdCL = 8, kBwdCL = 8;
constexpr int kFwdMinBlocks = 3, kBwdMinBlocks = 2;
constexpr int kFwdStages = 4, kBwdStages = 3;

struct ConvParams {
    int64_t B, L, D, groups, splits;  // groups: warp columns across D; splits: token shares per column
    const void* xin;
    const float *w, *bias, *state_in;
    void* x;
    float* state_out;
    const void* dx;
    void* dxin;
    float *dw, *dbias, *dstate;
    unsigned* status;
};

__device__ __forceinline__ float2 splat(float v) { return make_float2(v, v); }

template <int VS> __device__ __forceinline__ void ld_shared_vec(const char* p, unsigned* w) {
    if constexpr (VS == 16) {
        const uint4 q = *reinterpret_cast<const uint4*>(p);
        w[0] = q.x; w[1] = q.y; w[2] = q.z; w[3] = q.w;
    } else {
        const uint2 q = *reinterpret_cast<const uint2*>(p);
        w[0] = q.x; w[1] = q.y;
    }
}
template <int VS> __device__ __forceinline__ void ld_global_vec(const char* p, unsigned* w) {
    if constexpr (VS == 16) {
        const uint4 q = __ldg(reinterpret_cast<const uint4*>(p));
        w[0] = q.x; w[1] = q.y; w[2] = q.z; w[3] = q.w;
    } else {
        const uint2 q = __ldg(reinterpret_cast<const uint2*>(p));
        w[0] = q.x; w[1] = q.y;
    }
}
template <int VS> __device__ __forceinline__ void st_global_vec(char* p, const unsigned* w) {
    if constexpr (VS == 16)
        *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
    else
        *reinterpret_cast<uint2*>(p) = make_uint2(w[0], w[1]);
}
// VS bytes global -> shared, zero-filled when !valid (no source bytes read)
template <int VS> __device__ __forceinline__ void cp_async_vec(char* smem, const char* gmem, bool valid) {
    if constexpr (VS == 16) {
        cp_async16(smem, gmem, valid);
    } else {
        const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
        const int n = valid ? 8 : 0;
        asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;\n" ::"r"(s), "l"(gmem), "r"(n) : "memory");
    }
}

// CL channels of one row <-> P channel pairs
template <typename IO, int CL> struct Row {
    using G = Lane<IO, CL>;
    __device__ static void unpack(const unsigned (&w)[G::W], float2 (&v)[G::P]) {
#pragma unroll
        for (int i = 0; i < G::P; ++i) {
            if constexpr (sizeof(IO) == 2)
                v[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
            else
                v[i] = make_float2(__uint_as_float(w[2 * i]), __uint_as_float(w[2 * i + 1]));
        }
    }
    __device__ static void ld_shared(const char* p, float2 (&v)[G::P]) {
        unsigned w[G::W];
#pragma unroll
        for (int n = 0; n < G::NV; ++n) ld_shared_vec<G::VS>(p + n * 32 * G::VS, w + n * (G::VS / 4));
        unpack(w, v);
    }
    __device__ static void ld_global(const IO* p, float2 (&v)[G::P]) {
        unsigned w[G::W];
#pragma unroll
        for (int n = 0; n < G::NV; ++n)
            ld_global_vec<G::VS>(reinterpret_cast<const char*>(p) + n * G::VS, w + n * (G::VS / 4));
        unpack(w, v);
    }
    __device__ static void st_global(IO* p, const float2 (&v)[G::P]) {
        unsigned w[G::W];
#pragma unroll
        for (int i = 0; i < G::P; ++i) {
            if constexpr (sizeof(IO) == 2) {
                const __nv_bfloat162 h = __floats2bfloat162_rn(v[i].x, v[i].y);
                w[i] = *reinterpret_cast<const unsigned*>(&h);
            } else {
                w[2 * i] = __float_as_uint(v[i].x);
                w[2 * i + 1] = __float_as_uint(v[i].y);
            }
        }
#pragma unroll
        for (int n = 0; n < G::NV; ++n) st_global_vec<G::VS>(reinterpret_cast<char*>(p) + n * G::VS, w + n * (G::VS / 4));
    }
};

// sigmoid of a channel pair: the scan's sigmoid (MUFU forms for bf16 I/O)
template <bool FAST> __device__ __forceinline__ float2 sigmoid2(float2 v) {
    if (FAST) {
        const float2 m = __fmul2_rn(v, splat(-kLog2e));
        const float2 den = __fadd2_rn(make_float2(ex2(m.x), ex2(m.y)), splat(1.0f));
        return make_float2(rcp(den.x), rcp(den.y));
    }
    return make_float2(sigmoid<false>(v.x), sigmoid<false>(v.y));
}

// Copy rows row0 .. row0+R-1 of each stream into ring slot `slot`; rows at
// or past `rend` are zero-filled (their address is never formed).
template <typename IO, int STREAMS, int CL, int STAGES>
__device__ __forceinline__ void issue_stage(char* ring, int slot, const IO* const (&src)[STREAMS], int64_t D,
                                            int64_t row0, int64_t rend, int lane) {
    using T = ConvTile<IO, STREAMS, CL, STAGES>;
    using G = Lane<IO, CL>;
#pragma unroll
    for (int r = 0; r < T::R; ++r) {
        const bool valid = row0 + r < rend;
#pragma unroll
        for (int s = 0; s < STREAMS; ++s) {
            const char* g = reinterpret_cast<const char*>(valid ? src[s] + (row0 + r) * D : src[s]);
#pragma unroll
            for (int n = 0; n < G::NV; ++n)
                cp_async_vec<G::VS>(ring + slot * kConvStage + (r * STREAMS + s) * T::ROW + n * 32 * G::VS + lane * G::VS,
                                    g + n * G::VS, valid);
        }
    }
}

// seq[0 .. K-2] <- the K-1 inputs before token t0: halo rows, or the
// carried state (zeros when absent) where t < 0.
template <typename IO, int K, int CL, int S>
__device__ __forceinline__ void load_window(const ConvParams& p, const IO* xin, int64_t b, int64_t d0, int64_t t0,
                                            float2 (&seq)[S][CL / 2]) {
#pragma unroll
    for (int j = 0; j < K - 1; ++j) {
        const int64_t t = t0 - (K - 1) + j;
        if (t >= 0) {
            Row<IO, CL>::ld_global(xin + t * p.D, seq[j]);
        } else {
#pragma unroll
            for (int i = 0; i < CL / 2; ++i) {
                const int64_t at = (b * p.D + d0 + 2 * i) * (K - 1) + (K - 1 + t);
                seq[j][i] = p.state_in ? make_float2(p.state_in[at], p.state_in[at + (K - 1)]) : splat(0.f);
            }
        }
    }
}

template <int K, int P>
__device__ __forceinline__ void load_weights(const ConvParams& p, int64_t d0, float2 (&w2)[K][P], float2 (&b2)[P]) {
#pragma unroll
    for (int i = 0; i < P; ++i) {
#pragma unroll
        for (int k = 0; k < K; ++k) w2[k][i] = make_float2(p.w[(d0 + 2 * i) * K + k], p.w[(d0 + 2 * i + 1) * K + k]);
        b2[i] = p.bias ? make_float2(p.bias[d0 + 2 * i], p.bias[d0 + 2 * i + 1]) : splat(0.f);
    }
}

template <int NS> __device__ __forceinline__ int next_slot(int s) { return s + 1 == NS ? 0 : s + 1; }

template <typename IO, int K>
__global__ void __launch_bounds__(kConvThreads, kFwdMinBlocks) ssm_conv_fwd_kernel(const ConvParams p) {
    constexpr int CL = kFwdCL, P = CL / 2;
    using T = ConvTile<IO, 1, CL, kFwdStages>;
    using G = Lane<IO, CL>;
    constexpr int R = T::R;
    constexpr bool FAST = IOT<IO>::kFast;
    extern __shared__ __align__(16) char conv_smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    char* ring = conv_smem + warp * T::WARP;
    const char* mine = ring + lane * G::VS;
    const int64_t D = p.D, L = p.L, items = p.B * p.groups * p.splits;
    float2 nf = splat(0.f);
    for (int64_t item = (int64_t)blockIdx.x * kConvWarps + warp; item < items;
         item += (int64_t)gridDim.x * kConvWarps) {
        const int64_t j = item % p.splits, col = item / p.splits;
        const int64_t b = col / p.groups, d0 = (col % p.groups) * T::WARP_CH + lane * CL;
        const bool dv = d0 < D;  // lanes past D copy nothing and store nothing (no early exit: warp votes)
        const int64_t dd0 = dv ? d0 : 0;
        const int64_t t0 = L * j / p.splits, t1 = L * (j + 1) / p.splits;
        const IO* const src[1] = {reinterpret_cast<const IO*>(p.xin) + b * L * D + dd0};
        IO* x = reinterpret_cast<IO*>(p.x) + b * L * D + dd0;
        const int64_t nst = (t1 - t0 + R - 1) / R, rend = dv ? t1 : t0;
#pragma unroll
        for (int s = 0; s < T::NS - 1; ++s) {
            if (s < nst) issue_stage<IO, 1, CL, kFwdStages>(ring, s, src, D, t0 + s * R, rend, lane);
            cp_async_commit();
        }
        float2 w2[K][P], b2[P], seq[K - 1 + R][P];
        load_weights<K, P>(p, dd0, w2, b2);
#pragma unroll
        for (int jj = 0; jj < K - 1; ++jj)
#pragma unroll
            for (int i = 0; i < P; ++i) seq[jj][i] = splat(0.f);
        if (dv) load_window<IO, K, CL>(p, src[0], b, d0, t0, seq);
        int slot = 0, fill = T::NS - 1;
        for (int64_t st = 0; st < nst; ++st) {
            if (st + T::NS - 1 < nst) issue_stage<IO, 1, CL, kFwdStages>(ring, fill, src, D, t0 + (st + T::NS - 1) * R, rend, lane);
            cp_async_commit();
            cp_async_wait<T::NS - 1>();
#pragma unroll
            for (int u = 0; u < R; ++u) {
                Row<IO, CL>::ld_shared(mine + slot * kConvStage + u * T::ROW, seq[K - 1 + u]);
                float2 out[P];
#pragma unroll
                for (int i = 0; i < P; ++i) {
                    float2 s = b2[i];
#pragma unroll
                    for (int k = 0; k < K; ++k) s = __ffma2_rn(w2[k][i], seq[u + k][i], s);
                    out[i] = __fmul2_rn(s, sigmoid2<FAST>(s));
                }
                {  // Inf / NaN in any output survives the sum
                    float2 a = out[0];
#pragma unroll
                    for (int i = 1; i < P; ++i) a = __fadd2_rn(a, out[i]);
                    nf = __ffma2_rn(a, splat(0.f), nf);
                }
                const int64_t t = t0 + st * R + u;
                if (t < rend) Row<IO, CL>::st_global(x + t * D, out);
            }
#pragma unroll
            for (int jj = 0; jj < K - 1; ++jj)
#pragma unroll
                for (int i = 0; i < P; ++i) seq[jj][i] = seq[R + jj][i];
            slot = next_slot<T::NS>(slot);
            fill = next_slot<T::NS>(fill);
        }
        cp_async_wait<0>();
        // the share holding the last token writes the last K-1 inputs; all
        // are read before any is written, so state_out may be state_in
        // (the launch then gives each column one share)
        if (dv && p.state_out && t1 == L && K > 1) {
            float2 last[K > 1 ? K - 1 : 1][P];
            load_window<IO, K, CL>(p, src[0], b, d0, L, last);
#pragma unroll
            for (int i = 0; i < P; ++i)
#pragma unroll
                for (int jj = 0; jj < K - 1; ++jj) {
                    const int64_t at = (b * D + d0 + 2 * i) * (K - 1) + jj;
                    p.state_out[at] = last[jj][i].x;
                    p.state_out[at + (K - 1)] = last[jj][i].y;
                }
        }
    }
    flag_nonfinite(p.status, nf.x + nf.y);
}

template <typename IO, int K>
__global__ void __launch_bounds__(kConvThreads, kBwdMinBlocks) ssm_conv_bwd_kernel(const ConvParams p) {
    constexpr int CL = kBwdCL, P = CL / 2;
    using T = ConvTile<IO, 2, CL, kBwdStages>;
    using G = Lane<IO, CL>;
    constexpr int R = T::R;
    constexpr bool FAST = IOT<IO>::kFast;
    extern __shared__ __align__(16) char conv_smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    char* ring = conv_smem + warp * T::WARP;
    const char* mine = ring + lane * G::VS;
    const int64_t D = p.D, L = p.L, items = p.B * p.groups * p.splits;
    float2 nf = splat(0.f);
    for (int64_t item = (int64_t)blockIdx.x * kConvWarps + warp; item < items;
         item += (int64_t)gridDim.x * kConvWarps) {
        const int64_t j = item % p.splits, col = item / p.splits;
        const int64_t b = col / p.groups, d0 = (col % p.groups) * T::WARP_CH + lane * CL;
        const bool dv = d0 < D;
        const int64_t dd0 = dv ? d0 : 0;
        const int64_t t0 = L * j / p.splits, t1 = L * (j + 1) / p.splits;
        // rows t0 .. t1+K-2: the share's tokens and the K-1 after it, whose
        // dpre finish dxin of the share's last inputs (none past the end)
        const int64_t rend = dv ? min64(L, t1 + (K - 1)) : t0;
        const int64_t nst = (t1 + (K - 1) - t0 + R - 1) / R;
        const IO* const src[2] = {reinterpret_cast<const IO*>(p.xin) + b * L * D + dd0,
                                  reinterpret_cast<const IO*>(p.dx) + b * L * D + dd0};
        IO* dxin = reinterpret_cast<IO*>(p.dxin) + b * L * D + dd0;
#pragma unroll
        for (int s = 0; s < T::NS - 1; ++s) {
            if (s < nst) issue_stage<IO, 2, CL, kBwdStages>(ring, s, src, D, t0 + s * R, rend, lane);
            cp_async_commit();
        }
        float2 w2[K][P], b2[P], gw[K][P], gb[P];
        float2 seq[K - 1 + R][P], dseq[K - 1 + R][P];  // inputs / dpre of tokens t-(K-1) .. t+R-1
        load_weights<K, P>(p, dd0, w2, b2);
#pragma unroll
        for (int i = 0; i < P; ++i) {
            gb[i] = splat(0.f);
#pragma unroll
            for (int k = 0; k < K; ++k) gw[k][i] = splat(0.f);
#pragma unroll
            for (int jj = 0; jj < K - 1; ++jj) {
                dseq[jj][i] = splat(0.f);  // dxin below t0 is not this share's
                seq[jj][i] = splat(0.f);
            }
        }
        if (dv) load_window<IO, K, CL>(p, src[0], b, d0, t0, seq);
        int slot = 0, fill = T::NS - 1;
        for (int64_t st = 0; st < nst; ++st) {
            if (st + T::NS - 1 < nst) issue_stage<IO, 2, CL, kBwdStages>(ring, fill, src, D, t0 + (st + T::NS - 1) * R, rend, lane);
            cp_async_commit();
            cp_async_wait<T::NS - 1>();
            const char* sp = mine + slot * kConvStage;
#pragma unroll
            for (int u = 0; u < R; ++u) {
                float2 g[P];
                Row<IO, CL>::ld_shared(sp + (2 * u) * T::ROW, seq[K - 1 + u]);
                Row<IO, CL>::ld_shared(sp + (2 * u + 1) * T::ROW, g);
                const int64_t t = t0 + st * R + u;
#pragma unroll
                for (int i = 0; i < P; ++i) {
                    float2 v = b2[i];
#pragma unroll
                    for (int k = 0; k < K; ++k) v = __ffma2_rn(w2[k][i], seq[u + k][i], v);
                    const float2 sg = sigmoid2<FAST>(v);
                    // silu'(v) = s * (1 + v * (1 - s)); rows past the end hold dx = 0
                    const float2 inner = __ffma2_rn(v, __ffma2_rn(sg, splat(-1.0f), splat(1.0f)), splat(1.0f));
                    dseq[K - 1 + u][i] = __fmul2_rn(g[i], __fmul2_rn(sg, inner));
                }
                if (t < t1) {  // the look-ahead rows add no dw / dbias terms
#pragma unroll
                    for (int i = 0; i < P; ++i) {
#pragma unroll
                        for (int k = 0; k < K; ++k) gw[k][i] = __ffma2_rn(dseq[K - 1 + u][i], seq[u + k][i], gw[k][i]);
                        gb[i] = __fadd2_rn(gb[i], dseq[K - 1 + u][i]);
                    }
                }
                // input s = t-(K-1) feeds tokens s .. s+K-1: dxin_s = sum_k w[k] * dpre_{s+(K-1)-k}
                const int64_t s_ = t - (K - 1);
                float2 o[P];
#pragma unroll
                for (int i = 0; i < P; ++i) {
                    float2 a = __fmul2_rn(w2[0][i], dseq[u + K - 1][i]);
#pragma unroll
                    for (int k = 1; k < K; ++k) a = __ffma2_rn(w2[k][i], dseq[u + K - 1 - k][i], a);
                    o[i] = a;
                }
                if (s_ >= t0 && s_ < t1) {
                    if (dv) Row<IO, CL>::st_global(dxin + s_ * D, o);
                } else if (s_ < 0 && p.dstate && dv) {
                    // the share starting at t = 0: entry K-1+s_ of the carried state's gradient
#pragma unroll
                    for (int i = 0; i < P; ++i) {
                        const int64_t at = (b * D + d0 + 2 * i) * (K - 1) + (K - 1 + s_);
                        p.dstate[at] = o[i].x;
                        p.dstate[at + (K - 1)] = o[i].y;
                    }
                }
            }
#pragma unroll
            for (int jj = 0; jj < K - 1; ++jj)
#pragma unroll
                for (int i = 0; i < P; ++i) {
                    seq[jj][i] = seq[R + jj][i];
                    dseq[jj][i] = dseq[R + jj][i];
                }
            slot = next_slot<T::NS>(slot);
            fill = next_slot<T::NS>(fill);
        }
        cp_async_wait<0>();
        // every output is a w-weighted sum of dpre values, and every dpre of
        // this share's tokens is in gb: Inf / NaN anywhere shows there
#pragma unroll
        for (int i = 0; i < P; ++i) nf = __ffma2_rn(gb[i], splat(0.f), nf);
        if (dv) {
#pragma unroll
            for (int i = 0; i < P; ++i) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float* dst = p.dw + (d0 + 2 * i + h) * K;
                    if constexpr (K == 4) {
                        red_add_v4(dst, h ? make_float4(gw[0][i].y, gw[1][i].y, gw[2][i].y, gw[3][i].y)
                                          : make_float4(gw[0][i].x, gw[1][i].x, gw[2][i].x, gw[3][i].x));
                    } else {
#pragma unroll
                        for (int k = 0; k < K; ++k) atomicAdd(dst + k, h ? gw[k][i].y : gw[k][i].x);
                    }
                }
            }
            if (p.dbias) {
#pragma unroll
                for (int i = 0; i < P; i += 2)
                    red_add_v4(p.dbias + d0 + 2 * i, make_float4(gb[i].x, gb[i].y, gb[i + 1].x, gb[i + 1].y));
            }
        }
    }
    flag_nonfinite(p.status, nf.x + nf.y);
}

template <typename KERN> int conv_blocks_per_sm(KERN kern, int smem, int* cache) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    int& c = cache[dev & 63];
    if (c == 0) {
        int v = 0;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, kern, kConvThreads, smem) != cudaSuccess || v < 1)
            v = 1;
        c = v;
    }
    return c;
}

template <typename IO, int K> int launch_conv_t(bool bwd, ConvParams p, cudaStream_t s) {
    if (p.B == 0 || p.L == 0 || p.D == 0) return 0;
    static int cache_f[64] = {0}, cache_b[64] = {0};
    const int smem = bwd ? ConvTile<IO, 2, kBwdCL, kBwdStages>::SMEM : ConvTile<IO, 1, kFwdCL, kFwdStages>::SMEM;
    const int bps = bwd ? conv_blocks_per_sm(ssm_conv_bwd_kernel<IO, K>, smem, cache_b)
                        : conv_blocks_per_sm(ssm_conv_fwd_kernel<IO, K>, smem, cache_f);
    const int64_t resident = (int64_t)sm_count() * bps;
    const int64_t warp_ch = 32 * (bwd ? kBwdCL : kFwdCL);
    p.groups = (p.D + warp_ch - 1) / warp_ch;
    p.splits = conv_splits(p.B * p.groups, p.L, resident * kConvWarps,
                           !bwd && p.state_out != nullptr && p.state_out == p.state_in);
    const int64_t items = p.B * p.groups * p.splits;
    const int64_t grid = min64((items + kConvWarps - 1) / kConvWarps, resident);
    if (bwd)
        ssm_conv_bwd_kernel<IO, K><<<(unsigned)grid, kConvThreads, smem, s>>>(p);
    else
        ssm_conv_fwd_kernel<IO, K><<<(unsigned)grid, kConvThreads, smem, s>>>(p);
    return cudaGetLastError() == cudaSuccess ? 1 : -1;
}

template <typename IO> int launch_conv_k(bool bwd, int K, const ConvParams& p, cudaStream_t s) {
    switch (K) {
        case 1: return launch_conv_t<IO, 1>(bwd, p, s);
        case 2: return launch_conv_t<IO, 2>(bwd, p, s);
        case 3: return launch_conv_t<IO, 3>(bwd, p, s);
        default: return launch_conv_t<IO, 4>(bwd, p, s);
    }
}

}  // namespace

int launch_conv(int io, bool bwd, int64_t B, int64_t L, int64_t D, int K, const void* xin, const float* w,
                const float* bias, const float* state_in, void* x, float* state_out, const void* dx, void* dxin,
                float* dw, float* dbias, float* dstate, unsigned* status, cudaStream_t s) {
    ConvParams p{};
    p.B = B; p.L = L; p.D = D;
    p.xin = xin; p.w = w; p.bias = bias; p.state_in = state_in;
    p.x = x; p.state_out = state_out;
    p.dx = dx; p.dxin = dxin; p.dw = dw; p.dbias = dbias; p.dstate = dstate;
    p.status = status;
    return io == 0 ? launch_conv_k<float>(bwd, K, p, s) : launch_conv_k<__nv_bfloat16>(bwd, K, p, s);
}

}  // namespace ssm
