// mLSTM stabilized chunkwise forward on the sm_103a tensor cores
// (Evil-Inference-Code, README_FIX_RUST.md, "mLSTM Equivalence Fixes (Rust
// vs Python)": the cell whose recurrent step must match its parallel form,
// with the stabilized denominator max(|q . n|, exp(-m)), the cumulative sum
// of log forget gates by iteration and m starting at 0).
//
// One CTA per (batch, head) walks the sequence chunk by chunk (64 tokens,
// K = V = 128). The stabilized state stays on chip the whole time: C^T in
// 128 TMEM columns (lane = value channel v, column = key channel), n and m
// in shared memory / registers (fp32). Products are tcgen05.mma (kind::f16,
// bf16 operands, fp32 accumulation, M = 128) on 128-byte-swizzled operands;
// q, k and v arrive by TMA one chunk ahead, v as the MN-major operand of
// every product that contracts over tokens (no transposes).
//
// Per chunk, with F the chunk's inclusive cumulative log forget gates,
// g_s = log i_s - F_s, mx_t = max(m_prev, max_{s<=t} g_s) and m_t = F_t +
// mx_t (the recurrent stabilizer unrolled):
//  0. gate pass (one warp, for the next chunk, during this chunk's round 2;
//     two table sets): F by a warp scan, the running maximum of g, and
//     alpha_t = exp(m_prev - mx_t), gamma_s = exp(g_s - mx_last), the
//     state's decay beta = alpha_last and m_new = m_last;
//  1. as soon as q and k land, [S | q.n] = q [k; n_hi; n_lo]^T (n rides as
//     two bf16 rows of the k operand, so q.n needs no reduction); under it
//     the row pass: gamma * k (MN-major) and the per-warp partial sums of
//     gamma * k (n's increment);
//  2. C^T q^T (the state's share of the output, scaled by alpha_t * scale
//     in step 5), issued by a thread of another warp (issuing blocks the
//     issuing thread while the tensor pipe works); every other thread waits
//     for S by itself;
//  3. P = S * scale * exp(g_s - mx_t) on and below the diagonal, held as two
//     bf16 parts P = P_hi + P_lo (the normaliser divides by a sum of signed
//     terms that can nearly cancel, so P's one bf16 rounding would reach the
//     output at up to 4e-2; the two parts carry 16 bits), and its row sums:
//     every warp a quarter of the columns of 32 rows (S is in TMEM twice);
//     C^T <- beta C^T in TMEM;
//  4. MMA out^T = V^T P_hi^T + V^T P_lo^T and C^T += V^T (gamma k), while
//     the gate pass runs, 64 threads form 1 / max(|alpha_t q.n + rowsum_t|,
//     exp(-m_t)) and 128 threads n <- beta n + sum gamma_s k_s;
//  5. h_t = (alpha_t scale (C^T q^T)_t + (P v)_t) times that reciprocal,
//     staged as rows and (with weights) normalised per token over V, eight
//     tokens per warp at once; the bf16 copy of C^T that the next chunk's
//     product reads is refreshed from TMEM.
// Every exponent is <= 0 (mx is a running maximum), so no gate overflows.
//
// Every wait (copies, tensor-core completions) is bounded (1 s); a wait that
// runs out sets the timeout status bit, the CTA waits (bounded) for its
// copies still in flight and stops.
#include <math.h>

#include "ssm_common.cuh"
#include "ssm_internal.h"
#include "tc_common.cuh"
#include "../../include/mlstm.h"

namespace ssm {

namespace {

using namespace tc;

constexpr int kMC = 64;    // tokens per chunk
constexpr int kMK = 128;   // key channels
constexpr int kMV = 128;   // value channels
constexpr int kMThreads = 256;
constexpr int kGateWarp = 1;  // runs the gate passes (during round 2, where it has no other work)
constexpr int kCqWarp = 7;    // a thread of it issues the state term C^T q^T

// Shared-memory regions (bytes from a 1024-byte aligned base).
constexpr int kKR = 80;                 // rows of the k operand: k (64), n_hi, n_lo, zeros (N = 80)
constexpr int kQ = 0;                   // [q; q]             128 rows x K=128 (q by TMA into both halves)
constexpr int kKB = kQ + 32768;         // [k; n_hi; n_lo; 0]  80 rows x K=128 (k by TMA into rows 0-63)
constexpr int kVB = kKB + 2 * kKR * 128;  // v                 MN-major [64 tokens][128] (TMA)
constexpr int kCT = kVB + 16384;        // C^T (bf16)         128 rows x K=128
constexpr int kKP = kCT + 32768;        // gamma*k             MN-major [64 tokens][128]
constexpr int kP = kKP + 16384;         // P_hi                64 rows x K=64
constexpr int kP2 = kP + 8192;          // P_lo = P - P_hi     64 rows x K=64
constexpr int kOS = kP2 + 8192;         // output rows fp32 [64][kOSR]
constexpr int kOSR = kMV + 4;           // padded row (floats)
constexpr int kMisc = kOS + kMC * kOSR * 4;
// misc (floats): two sets (chunk parity) of the gate tables g, mx, alpha, m_t, gamma [64 each] and beta, m_new
// [4]; then q.n [64], row sums [4][64], 1/denominator [64], n [128], per-warp partial n increments [8][128];
// then mbarriers, TMEM slot
constexpr int kGateSet = 5 * kMC + 4;
constexpr int kMiscFloats = 2 * kGateSet + kMC + 4 * kMC + kMC + kMK + 8 * kMK;
constexpr int kBarOff = kMisc + kMiscFloats * 4;
constexpr int kMSmem = kBarOff + 64 + 1024;  // + slack for the 1024-byte alignment
static_assert(kMSmem <= 227 * 1024, "shared memory");
static_assert(kBarOff % 8 == 0, "mbarriers 8-byte aligned");
static_assert(kKB % 1024 == 0 && kVB % 1024 == 0 && kCT % 1024 == 0 && kKP % 1024 == 0 &&
                  kP % 1024 == 0 && kP2 % 1024 == 0 && (kKR * 128) % 1024 == 0,
              "swizzled operands and copy destinations on 1024-byte boundaries");
constexpr unsigned kQBytes = 4 * 64 * 64 * 2, kKBytes = 2 * 64 * 64 * 2, kVBytes = 2 * 64 * 64 * 2;

// TMEM columns: C^T; per chunk S (twice: lanes 0-63 and 64-127) with q.n_hi, q.n_lo in columns 64, 65, the
// chunk's own share of out^T (P v) and the state's share (C^T q^T, scaled per token in the epilogue).
constexpr unsigned kTC = 0, kTS = 128, kTO = 256, kTQ = 320, kTCols = 512;

struct MlstmParams {
    int64_t B, H, T;
    float scale, norm_eps;
    const float* igate;
    const float* fgate;
    const float* C_in;
    const float* n_in;
    const float* m_in;
    const float* norm_weight;
    __nv_bfloat16* h;
    float* C_out;
    float* n_out;
    float* m_out;
    unsigned* status;
    unsigned long long wait_ns;  // bound of every wait (kWaitNs unless a test armed a fault)
    int64_t fault_chunk1;        // tests: chunk fault_chunk1 - 1's q copy is not issued (0: none)
};
struct MlstmMaps {
    CUtensorMap q, k, v;  // rows = B*H*T tokens; 64-column swizzled boxes of 64 rows
};

// log(sigmoid(x)) = min(x, 0) - log(1 + exp(-|x|)), finite for every finite x
__device__ __forceinline__ float log_sigmoid(float x) { return fminf(x, 0.f) - log1pf(expf(-fabsf(x))); }

__device__ __forceinline__ float bf16_round(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

__global__ void __launch_bounds__(kMThreads, 1)
    mlstm_chunk_fwd_kernel(const MlstmParams p, const __grid_constant__ MlstmMaps mp) {
    extern __shared__ __align__(1024) char m_smem_raw[];
    char* sm = m_smem_raw + ((1024u - (smem_u32(m_smem_raw) & 1023u)) & 1023u);
    // gate tables of chunk parity b: g = log i_s - F_s (-inf past the chunk's end), mx = max(m_prev, max_{s<=t}
    // g_s), alpha = exp(m_prev - mx), m_t = F_t + mx, gamma = exp(g_s - mx_last); then beta, m_new
    float* s_gate = reinterpret_cast<float*>(sm + kMisc);
    auto G_g = [&](int b) { return s_gate + b * kGateSet; };
    auto G_mx = [&](int b) { return s_gate + b * kGateSet + kMC; };
    auto G_al = [&](int b) { return s_gate + b * kGateSet + 2 * kMC; };
    auto G_mt = [&](int b) { return s_gate + b * kGateSet + 3 * kMC; };
    auto G_gam = [&](int b) { return s_gate + b * kGateSet + 4 * kMC; };
    auto G_sc = [&](int b) { return s_gate + b * kGateSet + 5 * kMC; };
    float* s_qn = s_gate + 2 * kGateSet;  // scale * q_t . n (n before the chunk)
    float* s_rs = s_qn + kMC;             // row sums of P_hi + P_lo, per column quarter [4][64]
    float* s_rd = s_rs + 4 * kMC;         // 1 / max(|den_t|, exp(-m_t))
    float* s_n = s_rd + kMC;              // n [K]
    float* s_np = s_n + kMK;              // per-warp partial sums of gamma_s k_s [8][K]
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kBarOff);  // round 2, q, k, v, product S, state term Cq
    unsigned* tslot = reinterpret_cast<unsigned*>(bars + 6);
    float* s_os = reinterpret_cast<float*>(sm + kOS);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, whalf = warp >> 2;  // TMEM lanes 32*quarter..; column half
    const int64_t bh = blockIdx.x;
    const int64_t T = p.T;
    const int nchunks = (int)((T + kMC - 1) / kMC);
    const unsigned sbase = smem_u32(sm);
    const unsigned mbar = smem_u32(bars), bar_q = smem_u32(bars + 1), bar_k = smem_u32(bars + 2),
                   bar_v = smem_u32(bars + 3), mbar_s = smem_u32(bars + 4), mbar_c = smem_u32(bars + 5);
    constexpr float L2E = 1.4426950408889634f;

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_u32(tslot)),
                     "r"(kTCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    }
    // the copies of chunk cj (issued by kTmaThread); rows past the end of the
    // whole tensor read as zero, rows of the next (batch, head) on the ragged
    // last chunk are zeroed before any product reads them
    auto row_of = [&](int cj) { return (int)(bh * T + (int64_t)cj * kMC); };
    auto q_skipped = [&](int cj) { return (int64_t)cj + 1 == p.fault_chunk1; };
    auto issue = [&](int b, int cj) {
        const int y = row_of(cj);
        if (b == 0) {
            if (q_skipped(cj)) return;
            mbar_expect_tx(bar_q, kQBytes);
            for (int at = 0; at < 4; ++at) tma_load_2d(sm + kQ + at * 8192, &mp.q, (at >> 1) * 64, y, bar_q);
        } else if (b == 1) {
            mbar_expect_tx(bar_k, kKBytes);
            for (int at = 0; at < 2; ++at) tma_load_2d(sm + kKB + at * kKR * 128, &mp.k, at * 64, y, bar_k);
        } else {
            mbar_expect_tx(bar_v, kVBytes);
            for (int at = 0; at < 2; ++at) tma_load_2d(sm + kVB + at * 8192, &mp.v, at * 64, y, bar_v);
        }
    };
    // thread kTmaThread (warp 2) issues the copies; thread 0 the products
    constexpr int kTmaThread = 64;
    if (tid == kTmaThread) {
        const CUtensorMap* maps[3] = {&mp.q, &mp.k, &mp.v};
        for (int m = 0; m < 3; ++m)
            asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(maps[m])) : "memory");
    }
    if (tid == 0) {
        for (int b = 0; b < 6; ++b) mbar_init(smem_u32(bars + b), 1);
        mbar_fence_init();
    }
    // zero for the whole run: rows 66-79 of the k operand (the copies fill rows 0-63; rows 64 and 65
    // get n below)
    for (int i = tid; i < 2 * 2048 / 16; i += kMThreads) {
        const int at = i / (2048 / 16), o = i % (2048 / 16);
        *reinterpret_cast<uint4*>(sm + kKB + at * kKR * 128 + 8192 + o * 16) = make_uint4(0u, 0u, 0u, 0u);
    }
    __syncthreads();
    if (tid == kTmaThread && nchunks > 0)
        for (int b = 0; b < 3; ++b) issue(b, 0);
    tc_before();
    __syncthreads();
    tc_after();
    const unsigned tmem = *tslot;
    const unsigned tlane = (unsigned)(quarter * 32) << 16;  // this warp's TMEM lane quarter
    const int vrow = quarter * 32 + lane;                    // the TMEM lane (row) this thread reads

    // n as the two bf16 rows (hi, lo) of the k operand: the first product then also gives q . n
    auto put_n = [&](int kc, float nv) {
        const float hi = bf16_round(nv);
        st1(sm + kKB, 64, kc, kKR, hi);
        st1(sm + kKB, 65, kc, kKR, nv - hi);
    };
    // ---- the initial state: C^T into TMEM and its bf16 copy; n; m (0 without a state)
    {
        const float* c0 = p.C_in ? p.C_in + bh * kMK * kMV : nullptr;
        for (int c = 0; c < 2; ++c) {
            const int k0 = whalf * 64 + c * 32;
            float vals[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) vals[i] = c0 ? c0[(int64_t)(k0 + i) * kMV + vrow] : 0.f;
            tmem_st32(tmem + tlane + kTC + (unsigned)k0, vals);
#pragma unroll
            for (int i = 0; i < 32; i += 8) st8(sm + kCT, vrow, k0 + i, 128, vals + i);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
        if (tid < kMK) {
            const float nv = p.n_in ? p.n_in[bh * kMK + tid] : 0.f;
            s_n[tid] = nv;
            put_n(tid, nv);
        }
    }

    // ---- the gate pass (warp kGateWarp; lane: tokens 2*lane, 2*lane + 1): chunk cj's tables into set b,
    // from the pre-activations in ig, fg and the stabilizer m_in before the chunk; returns m after it
    auto gate_pass = [&](int cj, int b, float m_in, const float* ig, const float* fg) -> float {
        const int c = (int)min64(kMC, T - (int64_t)cj * kMC);
        float lf[2], li[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const bool live = 2 * lane + e < c;  // tokens past the end: f = 1, i = 0
            lf[e] = live ? log_sigmoid(fg[e]) : 0.f;
            li[e] = live ? ig[e] : -INFINITY;
        }
        // F: inclusive cumulative sum over the chunk (the pair, then a scan over lanes)
        const float pair = lf[0] + lf[1];
        float inc = pair;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, inc, off);
            if (lane >= off) inc += y;
        }
        float before = __shfl_up_sync(0xffffffffu, inc, 1);
        if (lane == 0) before = 0.f;
        const float F[2] = {before + lf[0], before + pair};
        const float g[2] = {li[0] - F[0], li[1] - F[1]};
        // running maximum of g over the chunk, then mx = max(m_in, .)
        float mxi = fmaxf(g[0], g[1]);
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, mxi, off);
            if (lane >= off) mxi = fmaxf(mxi, y);
        }
        float mb = __shfl_up_sync(0xffffffffu, mxi, 1);
        if (lane == 0) mb = -INFINITY;
        const float M0 = fmaxf(mb, g[0]), M1 = fmaxf(M0, g[1]);
        const float mx[2] = {fmaxf(m_in, M0), fmaxf(m_in, M1)};
        const float al[2] = {ex2((m_in - mx[0]) * L2E), ex2((m_in - mx[1]) * L2E)};
        const int last = c - 1;
        const float mxL = __shfl_sync(0xffffffffu, (last & 1) ? mx[1] : mx[0], last >> 1);
        const float FL = __shfl_sync(0xffffffffu, (last & 1) ? F[1] : F[0], last >> 1);
        const float alL = __shfl_sync(0xffffffffu, (last & 1) ? al[1] : al[0], last >> 1);
        const float gm[2] = {ex2((g[0] - mxL) * L2E), ex2((g[1] - mxL) * L2E)};  // 0 past the end (g = -inf)
        const int t = 2 * lane;
        *reinterpret_cast<float2*>(G_g(b) + t) = make_float2(g[0], g[1]);
        *reinterpret_cast<float2*>(G_mx(b) + t) = make_float2(mx[0], mx[1]);
        *reinterpret_cast<float2*>(G_al(b) + t) = make_float2(al[0], al[1]);
        *reinterpret_cast<float2*>(G_mt(b) + t) = make_float2(F[0] + mx[0], F[1] + mx[1]);
        *reinterpret_cast<float2*>(G_gam(b) + t) = make_float2(gm[0], gm[1]);
        if (lane == 0) {
            G_sc(b)[0] = alL;       // beta: the state's decay over the chunk
            G_sc(b)[1] = FL + mxL;  // m at the chunk's last token
        }
        return FL + mxL;
    };
    // the gate pre-activations of the chunk whose gate pass comes next (warp kGateWarp)
    float ig_nx[2] = {0.f, 0.f}, fg_nx[2] = {0.f, 0.f};
    auto load_gates = [&](int cj) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int64_t t = (int64_t)cj * kMC + 2 * lane + e;
            ig_nx[e] = t < T ? p.igate[bh * T + t] : 0.f;
            fg_nx[e] = t < T ? p.fgate[bh * T + t] : 0.f;
        }
    };
    // m after the last chunk whose gate pass has run (warp kGateWarp); the first chunk's pass runs here,
    // every later one during the previous chunk's round 2
    float m_run = p.m_in ? p.m_in[bh] : 0.f;
    if (warp == kGateWarp && nchunks > 0) {
        load_gates(0);
        m_run = gate_pass(0, 0, m_run, ig_nx, fg_nx);
        if (nchunks > 1) load_gates(1);
    }
    fence_async_smem();
    tc_before();
    __syncthreads();

    unsigned phase = 0, phase_s = 0, phase_c = 0;
    // copies issued / waited for, per barrier (q, k, v); uniform over the CTA
    int issued[3] = {nchunks > 0 && !q_skipped(0), nchunks > 0, nchunks > 0}, waited[3] = {0, 0, 0};
    const unsigned tbar[3] = {bar_q, bar_k, bar_v};
    float nf = 0.f;
    auto fail = [&]() {
        if (tid == 0 && p.status) atomicOr(p.status, kStatusTimeout);
    };
    // every thread waits for a commit (the product S on its own barrier: one commit per barrier per
    // chunk, so no phase is missed); false if it never came
    auto mma_wait = [&](unsigned bar, unsigned& ph) -> bool {
        const bool ok = mbar_wait_try(bar, ph & 1u, p.wait_ns);
        ph++;
        if (!ok) fail();
        return __syncthreads_and(ok) != 0;
    };
    auto copies_wait = [&]() -> bool {  // the chunk's three copies, one CTA barrier
        bool ok = true;
        for (int b = 0; b < 3; ++b) ok = ok && mbar_wait_try(tbar[b], (unsigned)(waited[b] & 1), p.wait_ns);
        if (!ok) fail();
        const bool all = __syncthreads_and(ok) != 0;
        if (all)
            for (int b = 0; b < 3; ++b) waited[b]++;
        return all;
    };
    auto commit = [&](unsigned bar) {
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar)
                     : "memory");
    };
    auto refill = [&](int b, int cj) {  // next chunk's copy into a buffer every thread is done reading
        if (cj >= nchunks) return;
        if (tid == kTmaThread) {
            fence_async_smem();
            issue(b, cj);
        }
        issued[b] += (b == 0 && q_skipped(cj)) ? 0 : 1;
    };

    // the head-wise norm's weights for this lane's output channels 4 (lane % 8) + 32 u, u = 0..3
    const bool has_norm = p.norm_weight != nullptr;
    float4 w4[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
        w4[u] = has_norm ? *reinterpret_cast<const float4*>(p.norm_weight + (bh % p.H) * kMV + 4 * (lane & 7) + 32 * u)
                         : make_float4(1.f, 1.f, 1.f, 1.f);

    bool ok = true;
    for (int ci = 0; ci < nchunks && ok; ++ci) {
        const int gb = ci & 1;                  // this chunk's gate tables
        const int64_t t0 = (int64_t)ci * kMC;
        const int c = (int)min64(kMC, T - t0);  // live tokens; tokens c..63 are identity (f = 1, i = 0)
        const int64_t row0 = bh * T + t0;      // first token row of the chunk in [B*H*T]
        const float* g_g = G_g(gb);
        const float* g_mx = G_mx(gb);
        const float* g_al = G_al(gb);
        const float* g_mt = G_mt(gb);
        const float* g_gam = G_gam(gb);

        // the chunk's copies (one CTA barrier)
        if (!(ok = copies_wait())) break;

        // ---- 1a. [S | q.n_hi | q.n_lo] = [q; q] [k; n_hi; n_lo; 0]^T (S twice: lanes 0-63 and 64-127) from the
        // copies as they landed, under the row pass (columns of tokens past the chunk's end reach only rows past
        // it, which are never stored)
        if (tid == 0) {
            tc_after();
            mma_issue(tmem + kTS, sbase + kQ, sbase + kKB, kKR, kKR, kMK, false);
            commit(mbar_s);
        }

        // ---- 1b. row pass (thread = token r, channels cc..cc+7): gamma*k (MN-major) and the per-warp
        // partial sums of gamma*k over tokens (n's increment); v rows past the chunk's end zeroed
        {
            const int cc = (tid & 15) * 8;
            float np[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 2
            for (int it = 0; it < 4; ++it) {
                const int r = (tid >> 4) + it * (kMThreads >> 4);
                const bool live = r < c;
                float kv[8];
                ld8(sm + kKB, r, cc, kKR, kv);
                const float gm = g_gam[r];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    kv[i] = live ? kv[i] * gm : 0.f;
                    np[i] += kv[i];
                }
                st8(sm + kKP, r, cc, 64, kv);
                if (!live) {
                    const float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                    st8(sm + kVB, r, cc, 64, z);
                }
            }
            // lanes l and l ^ 16 hold the same channels for other tokens
#pragma unroll
            for (int i = 0; i < 8; ++i) np[i] += __shfl_xor_sync(0xffffffffu, np[i], 16);
            if (lane < 16) {
                *reinterpret_cast<float4*>(s_np + warp * kMK + cc) = make_float4(np[0], np[1], np[2], np[3]);
                *reinterpret_cast<float4*>(s_np + warp * kMK + cc + 4) = make_float4(np[4], np[5], np[6], np[7]);
            }
        }
        fence_async_smem();
        tc_before();
        __syncthreads();

        // ---- 2. the state's share of the output, C^T q^T (the rows of q are its N operand; alpha_t * scale is
        // applied per token in phase 5), issued by a thread of warp kCqWarp once S has had the tensor pipe to
        // itself (issuing blocks the issuing thread while the pipe works); every other thread waits for S by
        // itself (no CTA barrier: the outcome is agreed at the end of phase 3) and goes on
        if (tid == kCqWarp * 32) {
            tc_after();
            mma_issue(tmem + kTQ, sbase + kCT, sbase + kQ, 128, 64, kMK, false);
            commit(mbar_c);
        }
        const bool ok_s = mbar_wait_try(mbar_s, phase_s & 1u, p.wait_ns);
        phase_s++;
        if (!ok_s) fail();
        tc_after();

        // ---- 3. P as two bf16 parts and its row sums, every warp a quarter of the columns of 32 rows
        // (rows 0-31 on lanes 0-31 and 64-95, rows 32-63 on lanes 32-63 and 96-127); q.n; then C^T *= beta
        const float beta = G_sc(gb)[0];
        {
            const int t = (quarter & 1) * 32 + lane;  // 0..63
            const int cg = (quarter >> 1) * 2 + whalf, sb = cg * 16;
            const float mxt = g_mx[t];
            unsigned sr[16];
            tmem_ld16_nw(tmem + tlane + kTS + (unsigned)sb, sr);
            float qn[2];
            if (cg == 0) tmem_ld2(tmem + tlane + kTS + 64u, qn);  // waits for both loads
            else tmem_wait_ld();
            tmem_regs_ready<16>(sr);
            float hi[16], lo[16], rs = 0.f;
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
                const int s = sb + jj;
                const float pv = s <= t ? __uint_as_float(sr[jj]) * p.scale * ex2((g_g[s] - mxt) * L2E) : 0.f;
                hi[jj] = bf16_round(pv);
                lo[jj] = bf16_round(pv - hi[jj]);
                rs += hi[jj] + lo[jj];
            }
#pragma unroll
            for (int jj = 0; jj < 16; jj += 8) {
                st8(sm + kP, t, sb + jj, 64, hi + jj);
                st8(sm + kP2, t, sb + jj, 64, lo + jj);
            }
            s_rs[cg * kMC + t] = rs;
            if (cg == 0) s_qn[t] = (qn[0] + qn[1]) * p.scale;
        }
        {
            unsigned cr[64];
            tmem_ld32_nw(tmem + tlane + kTC + (unsigned)(whalf * 64), cr);
            tmem_ld32_nw(tmem + tlane + kTC + (unsigned)(whalf * 64 + 32), cr + 32);
            tmem_wait_ld();
            tmem_regs_ready<64>(cr);
            float cv[64];
#pragma unroll
            for (int i = 0; i < 64; ++i) cv[i] = __uint_as_float(cr[i]) * beta;
            tmem_st32(tmem + tlane + kTC + (unsigned)(whalf * 64), cv);
            tmem_st32(tmem + tlane + kTC + (unsigned)(whalf * 64 + 32), cv + 32);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
        fence_async_smem();
        tc_before();
        // one barrier agrees on the waits for S and for the state's share (which must have read q and the
        // bf16 copy of C^T before q's buffer is refilled and phase 5 rewrites the copy)
        {
            const bool ok_c = mbar_wait_try(mbar_c, phase_c & 1u, p.wait_ns);
            phase_c++;
            if (!ok_c) fail();
            if (!(ok = __syncthreads_and(ok_s && ok_c) != 0)) break;
        }
        refill(0, ci + 1);  // q has been read (by the two products only)
        refill(1, ci + 1);  // k has been read

        // ---- 4. out^T += V^T P_hi^T + V^T P_lo^T;  C^T += V^T (gamma*k); meanwhile the next chunk's
        // gate pass, the per-token reciprocal of the stabilized denominator and n (the first product,
        // which read n's rows of the k operand, is complete)
        if (tid == 0) {
            tc_after();
            mma_issue(tmem + kTO, sbase + kVB, sbase + kP, 64, 64, kMC, false, true, false);
            mma_issue(tmem + kTO, sbase + kVB, sbase + kP2, 64, 64, kMC, true, true, false);
            mma_issue(tmem + kTC, sbase + kVB, sbase + kKP, 0, kMK, kMC, true, true, true);
            commit(mbar);
        }
        if (warp == kGateWarp && ci + 1 < nchunks) {  // the next chunk's gate tables
            m_run = gate_pass(ci + 1, gb ^ 1, m_run, ig_nx, fg_nx);
            if (ci + 2 < nchunks) load_gates(ci + 2);
        } else if (tid >= 64 && tid < 64 + kMC) {
            const int t = tid - 64;
            const float rs = (s_rs[t] + s_rs[kMC + t]) + (s_rs[2 * kMC + t] + s_rs[3 * kMC + t]);
            const float den = __fmaf_rn(g_al[t], s_qn[t], rs);
            s_rd[t] = 1.f / fmaxf(fabsf(den), ex2(-g_mt[t] * L2E));  // exp(-m_t)
        } else if (tid >= 128) {  // n <- beta n + sum gamma_s k_s, and its rows of the k operand
            const int kc = tid - 128;
            float a = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w) a += s_np[w * kMK + kc];
            const float nv = __fmaf_rn(beta, s_n[kc], a);
            s_n[kc] = nv;
            put_n(kc, nv);
        }
        if (!(ok = mma_wait(mbar, phase))) break;
        tc_after();
        refill(2, ci + 1);  // v has been read

        // ---- 5. h = (alpha * scale * C^T q^T + P v) / max(|den|, exp(-m)) into the staging rows; the bf16
        // copy of C^T
        {
            const int tb = whalf * 32, k0 = whalf * 64;
            unsigned orr[32], oqr[32], cr[64];
            tmem_ld32_nw(tmem + tlane + kTO + (unsigned)tb, orr);
            tmem_ld32_nw(tmem + tlane + kTQ + (unsigned)tb, oqr);
            tmem_ld32_nw(tmem + tlane + kTC + (unsigned)k0, cr);
            tmem_ld32_nw(tmem + tlane + kTC + (unsigned)(k0 + 32), cr + 32);
            tmem_wait_ld();
            tmem_regs_ready<32>(orr);
            tmem_regs_ready<32>(oqr);
            tmem_regs_ready<64>(cr);
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
                const int t = tb + jj;
                const float o = __fmaf_rn(g_al[t] * p.scale, __uint_as_float(oqr[jj]), __uint_as_float(orr[jj]));
                s_os[t * kOSR + vrow] = o * s_rd[t];
            }
            float cv[64];
#pragma unroll
            for (int i = 0; i < 64; ++i) cv[i] = __uint_as_float(cr[i]);
#pragma unroll
            for (int i = 0; i < 64; i += 8) st8(sm + kCT, vrow, k0 + i, 128, cv + i);
        }
        __syncthreads();
        // rows: warp w takes tokens w, w + 8, ..., w + 56, four at a time on lane groups of 8 (group g the
        // token w + 8 (4 it + g); lane j of it channels 4j + 32u, u = 0..3), so the norm's two sums take
        // three shuffle rounds per four tokens
        {
            const int g = lane >> 3, j = lane & 7;
#pragma unroll
            for (int it = 0; it < 2; ++it) {
                const int t = warp + 8 * (4 * it + g);
                float4 x[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) x[u] = *reinterpret_cast<const float4*>(s_os + t * kOSR + 4 * j + 32 * u);
                if (has_norm) {
                    float sum = 0.f;
#pragma unroll
                    for (int u = 0; u < 4; ++u) sum += (x[u].x + x[u].y) + (x[u].z + x[u].w);
#pragma unroll
                    for (int off = 4; off >= 1; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
                    const float mean = sum * (1.f / kMV);
                    float sq = 0.f;
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        x[u] = make_float4(x[u].x - mean, x[u].y - mean, x[u].z - mean, x[u].w - mean);
                        sq += (x[u].x * x[u].x + x[u].y * x[u].y) + (x[u].z * x[u].z + x[u].w * x[u].w);
                    }
#pragma unroll
                    for (int off = 4; off >= 1; off >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, off);
                    const float rstd = rsqrtf(sq * (1.f / kMV) + p.norm_eps);
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        x[u] = make_float4(x[u].x * rstd * w4[u].x, x[u].y * rstd * w4[u].y, x[u].z * rstd * w4[u].z,
                                           x[u].w * rstd * w4[u].w);
                }
                if (t < c) {
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        nf = __fmaf_rn((x[u].x + x[u].y) + (x[u].z + x[u].w), 0.f, nf);
                        *reinterpret_cast<uint2*>(p.h + (row0 + t) * kMV + 4 * j + 32 * u) =
                            make_uint2(pack_bf2(x[u].x, x[u].y), pack_bf2(x[u].z, x[u].w));
                    }
                }
            }
        }
        fence_async_smem();
        tc_before();
        __syncthreads();
    }

    if (!ok) {  // a wait ran out: let the copies still in flight land before the CTA exits
        if (tid == kTmaThread)
            for (int b = 0; b < 3; ++b)
                for (; waited[b] < issued[b]; ++waited[b])
                    if (!mbar_wait_try(tbar[b], (unsigned)(waited[b] & 1), p.wait_ns)) break;
    } else if (p.C_out) {
        float* co = p.C_out + bh * kMK * kMV;
        for (int cc = 0; cc < 2; ++cc) {
            const int k0 = whalf * 64 + cc * 32;
            float s[32];
            tmem_ld32(tmem + tlane + kTC + (unsigned)k0, s);
#pragma unroll
            for (int i = 0; i < 32; ++i) co[(int64_t)(k0 + i) * kMV + vrow] = s[i];
        }
        if (tid < kMK) p.n_out[bh * kMK + tid] = s_n[tid];
        if (tid == kGateWarp * 32) p.m_out[bh] = m_run;  // m after the last chunk (this warp ran every gate pass)
    }
    flag_nonfinite(p.status, nf);
    tc_before();
    __syncthreads();
    if (warp == 0) {
        tc_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(kTCols) : "memory");
    }
}

// ---------------------------------------------------------------- one token: the recurrent step
struct MlstmStepParams {
    int64_t H;
    float scale, norm_eps;
    const __nv_bfloat16* q;
    const __nv_bfloat16* k;
    const __nv_bfloat16* v;
    const float* igate;
    const float* fgate;
    float* C;
    float* n;
    float* m;
    const float* norm_weight;
    __nv_bfloat16* h;
    unsigned* status;
};

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

// One CTA of 256 threads per (batch, head); everything in fp32. Thread (v = tid % 128, kh = tid / 128)
// updates C[k][v] for the 64 key channels kh*64.. (rows of C are read and written coalesced) and keeps its
// share of q . C'[:, v]; the two shares, q . n' and the norm's mean and variance meet in shared memory.
__global__ void __launch_bounds__(kMThreads) mlstm_step_kernel(const MlstmStepParams p) {
    __shared__ float s_q[kMK], s_k[kMK];
    __shared__ float s_part[2][kMV];
    __shared__ float s_red[8];
    __shared__ float s_rd;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t bh = blockIdx.x;
    if (tid < kMK) {
        s_q[tid] = __bfloat162float(p.q[bh * kMK + tid]) * p.scale;
        s_k[tid] = __bfloat162float(p.k[bh * kMK + tid]);
    }
    // the stabilizer and the two decays (the same scalars in every thread)
    const float lf = log_sigmoid(p.fgate[bh]), li = p.igate[bh], m0 = p.m[bh];
    const float m1 = fmaxf(lf + m0, li);
    const float fs = expf(lf + m0 - m1), is = expf(li - m1);
    __syncthreads();
    // n' = f' n + i' k and the partial sums of q . n'
    float qn = 0.f, nv = 0.f;
    if (tid < kMK) {
        nv = __fmaf_rn(fs, p.n[bh * kMK + tid], is * s_k[tid]);
        qn = s_q[tid] * nv;
    }
    // C' = f' C + i' k v^T and this thread's share of q . C'[:, v]
    const int v = tid & (kMV - 1), kh = tid >> 7;
    const float iv = is * __bfloat162float(p.v[bh * kMV + v]);
    float* Cb = p.C + bh * kMK * kMV;
    const int k0 = kh * (kMK / 2);
    float cv[kMK / 2];  // every load in flight before the first use
#pragma unroll
    for (int kk = 0; kk < kMK / 2; ++kk) cv[kk] = Cb[(int64_t)(k0 + kk) * kMV + v];
    float acc = 0.f;
#pragma unroll
    for (int kk = 0; kk < kMK / 2; ++kk) {
        const float c = __fmaf_rn(fs, cv[kk], iv * s_k[k0 + kk]);
        Cb[(int64_t)(k0 + kk) * kMV + v] = c;
        acc = __fmaf_rn(s_q[k0 + kk], c, acc);
    }
    s_part[kh][v] = acc;
    qn = warp_sum(qn);
    if (lane == 0 && warp < 4) s_red[warp] = qn;
    __syncthreads();
    if (tid == 0) {
        s_rd = 1.f / fmaxf(fabsf((s_red[0] + s_red[1]) + (s_red[2] + s_red[3])), expf(-m1));
        p.m[bh] = m1;
    }
    if (tid < kMK) p.n[bh * kMK + tid] = nv;
    __syncthreads();
    float hv = tid < kMV ? (s_part[0][tid] + s_part[1][tid]) * s_rd : 0.f;
    if (p.norm_weight) {  // the head-wise norm over the V values held by threads 0-127
        const float sum = warp_sum(hv);
        if (lane == 0 && warp < 4) s_red[4 + warp] = sum;
        __syncthreads();
        const float mean = ((s_red[4] + s_red[5]) + (s_red[6] + s_red[7])) * (1.f / kMV);
        const float d = tid < kMV ? hv - mean : 0.f;
        const float sq = warp_sum(d * d);
        if (lane == 0 && warp < 4) s_red[warp] = sq;
        __syncthreads();
        const float var = ((s_red[0] + s_red[1]) + (s_red[2] + s_red[3])) * (1.f / kMV);
        hv = tid < kMV ? d * rsqrtf(var + p.norm_eps) * p.norm_weight[(bh % p.H) * kMV + tid] : 0.f;
    }
    if (tid < kMV) p.h[bh * kMV + tid] = __float2bfloat16_rn(hv);
    flag_nonfinite(p.status, __fmaf_rn(hv, 0.f, 0.f));
}

bool misaligned(const void* q, uintptr_t a) { return q && (reinterpret_cast<uintptr_t>(q) & (a - 1)) != 0; }

}  // namespace
}  // namespace ssm

namespace {
// One-shot wait fault for this thread's next mlstm_chunk_fwd (tests).
thread_local int64_t g_mlstm_fault_chunk1 = 0;
thread_local unsigned long long g_mlstm_fault_wait_ns = 0;
}  // namespace

extern "C" int mlstm_debug_arm_wait_fault(int64_t chunk, uint64_t wait_ns) {
    if (wait_ns > 10000000000ull) return SSM_ERR_INVALID_ARG;
    g_mlstm_fault_chunk1 = chunk < 0 ? 0 : chunk + 1;
    g_mlstm_fault_wait_ns = chunk < 0 ? 0 : wait_ns;
    return SSM_OK;
}

extern "C" int mlstm_chunk_fwd(const mlstm_fwd_args* a, void* stream) {
    ssm::reset_launches();
    // an armed fault applies to this call only
    const int64_t fault_chunk1 = g_mlstm_fault_chunk1;
    const unsigned long long fault_wait_ns = g_mlstm_fault_wait_ns;
    g_mlstm_fault_chunk1 = 0;
    g_mlstm_fault_wait_ns = 0;
    if (!a) return SSM_ERR_INVALID_ARG;
    if (a->B < 0 || a->H < 0 || a->T < 0) return SSM_ERR_INVALID_ARG;
    if (a->K != ssm::kMK || a->V != ssm::kMV || (a->chunk != 0 && a->chunk != ssm::kMC)) return SSM_ERR_UNSUPPORTED;
    if (!(fabsf(a->scale) <= 3.0e38f)) return SSM_ERR_INVALID_ARG;              // NaN or infinite scale
    if (!(a->norm_eps >= 0.f && a->norm_eps <= 3.0e38f)) return SSM_ERR_INVALID_ARG;  // NaN, negative or infinite
    if (a->B * a->H > 0x7fffffff) return SSM_ERR_INVALID_ARG;
    // token rows are addressed by 32-bit copy coordinates
    if (a->T > 0x7fffffff || a->B * a->H * a->T > 0x7fffffff - 2 * ssm::kMC) return SSM_ERR_UNSUPPORTED;
    const bool in_all = a->C_in && a->n_in && a->m_in, in_none = !a->C_in && !a->n_in && !a->m_in;
    const bool out_all = a->C_out && a->n_out && a->m_out, out_none = !a->C_out && !a->n_out && !a->m_out;
    if (!(in_all || in_none) || !(out_all || out_none)) return SSM_ERR_INVALID_ARG;
    const bool work = a->B > 0 && a->H > 0 && a->T > 0;
    if (work && (!a->q || !a->k || !a->v || !a->igate || !a->fgate || !a->h)) return SSM_ERR_INVALID_ARG;
    const void* p16[] = {a->q, a->k, a->v, a->C_in, a->norm_weight, a->h, a->C_out, a->workspace};
    for (const void* q : p16)
        if (ssm::misaligned(q, 16)) return SSM_ERR_ALIGNMENT;
    const void* p4[] = {a->igate, a->fgate, a->n_in, a->m_in, a->n_out, a->m_out};
    for (const void* q : p4)
        if (ssm::misaligned(q, 4)) return SSM_ERR_ALIGNMENT;
    cudaStream_t s = (cudaStream_t)stream;
    const int64_t BH = a->B * a->H;
    if (!work) {  // the final state is the initial one
        if (out_all && BH > 0) {
            const size_t cb = (size_t)BH * ssm::kMK * ssm::kMV * sizeof(float), nb = (size_t)BH * ssm::kMK * sizeof(float),
                         mb = (size_t)BH * sizeof(float);
            cudaError_t e = cudaSuccess;
            if (in_all) {
                if (e == cudaSuccess) e = cudaMemcpyAsync(a->C_out, a->C_in, cb, cudaMemcpyDeviceToDevice, s);
                if (e == cudaSuccess) e = cudaMemcpyAsync(a->n_out, a->n_in, nb, cudaMemcpyDeviceToDevice, s);
                if (e == cudaSuccess) e = cudaMemcpyAsync(a->m_out, a->m_in, mb, cudaMemcpyDeviceToDevice, s);
            } else {
                if (e == cudaSuccess) e = cudaMemsetAsync(a->C_out, 0, cb, s);
                if (e == cudaSuccess) e = cudaMemsetAsync(a->n_out, 0, nb, s);
                if (e == cudaSuccess) e = cudaMemsetAsync(a->m_out, 0, mb, s);
            }
            if (e != cudaSuccess) return SSM_ERR_CUDA;
        }
        return SSM_OK;
    }
    static unsigned long long mask = 0;
    if (!ssm::ensure_smem(ssm::mlstm_chunk_fwd_kernel, ssm::kMSmem, mask)) return SSM_ERR_CUDA;
    ssm::MlstmParams p{};
    p.B = a->B; p.H = a->H; p.T = a->T;
    p.scale = a->scale; p.norm_eps = a->norm_eps;
    p.igate = a->igate; p.fgate = a->fgate;
    p.C_in = a->C_in; p.n_in = a->n_in; p.m_in = a->m_in;
    p.norm_weight = a->norm_weight;
    p.h = (__nv_bfloat16*)a->h;
    p.C_out = a->C_out; p.n_out = a->n_out; p.m_out = a->m_out;
    p.status = (unsigned*)a->workspace;
    p.fault_chunk1 = fault_chunk1;
    p.wait_ns = fault_chunk1 > 0 && fault_wait_ns > 0 ? fault_wait_ns : ssm::kWaitNs;
    const int64_t rows = BH * a->T;
    ssm::MlstmMaps mp{};
    const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const bool enc =
        ssm::encode_2d(&mp.q, bf, a->q, ssm::kMK, rows, ssm::kMK * 2, 64, ssm::kMC, CU_TENSOR_MAP_SWIZZLE_128B) &&
        ssm::encode_2d(&mp.k, bf, a->k, ssm::kMK, rows, ssm::kMK * 2, 64, ssm::kMC, CU_TENSOR_MAP_SWIZZLE_128B) &&
        ssm::encode_2d(&mp.v, bf, a->v, ssm::kMV, rows, ssm::kMV * 2, 64, ssm::kMC, CU_TENSOR_MAP_SWIZZLE_128B);
    if (!enc) return SSM_ERR_CUDA;
    ssm::mlstm_chunk_fwd_kernel<<<(unsigned)BH, ssm::kMThreads, ssm::kMSmem, s>>>(p, mp);
    return ssm::count_launches(cudaGetLastError() == cudaSuccess ? 1 : -1);
}

extern "C" int mlstm_step(const mlstm_step_args* a, void* stream) {
    ssm::reset_launches();
    if (!a) return SSM_ERR_INVALID_ARG;
    if (a->B < 0 || a->H < 0) return SSM_ERR_INVALID_ARG;
    if (a->K != ssm::kMK || a->V != ssm::kMV) return SSM_ERR_UNSUPPORTED;
    if (!(fabsf(a->scale) <= 3.0e38f)) return SSM_ERR_INVALID_ARG;
    if (!(a->norm_eps >= 0.f && a->norm_eps <= 3.0e38f)) return SSM_ERR_INVALID_ARG;
    if (a->B * a->H > 0x7fffffff) return SSM_ERR_INVALID_ARG;
    const int64_t BH = a->B * a->H;
    if (BH == 0) return SSM_OK;
    if (!a->q || !a->k || !a->v || !a->igate || !a->fgate || !a->C || !a->n || !a->m || !a->h) return SSM_ERR_INVALID_ARG;
    const void* p16[] = {a->q, a->k, a->v, a->C, a->norm_weight, a->h, a->workspace};
    for (const void* q : p16)
        if (ssm::misaligned(q, 16)) return SSM_ERR_ALIGNMENT;
    const void* p4[] = {a->igate, a->fgate, a->n, a->m};
    for (const void* q : p4)
        if (ssm::misaligned(q, 4)) return SSM_ERR_ALIGNMENT;
    ssm::MlstmStepParams p{};
    p.H = a->H; p.scale = a->scale; p.norm_eps = a->norm_eps;
    p.q = (const __nv_bfloat16*)a->q; p.k = (const __nv_bfloat16*)a->k; p.v = (const __nv_bfloat16*)a->v;
    p.igate = a->igate; p.fgate = a->fgate; p.C = a->C; p.n = a->n; p.m = a->m;
    p.norm_weight = a->norm_weight; p.h = (__nv_bfloat16*)a->h; p.status = (unsigned*)a->workspace;
    ssm::mlstm_step_kernel<<<(unsigned)BH, ssm::kMThreads, 0, (cudaStream_t)stream>>>(p);
    return ssm::count_launches(cudaGetLastError() == cudaSuccess ? 1 : -1);
}
