// Gated DeltaNet-2 chunkwise forward on the sm_103a tensor cores
// (docs.rs, burn-gdn2 0.1.4, src/forward.rs, chunk_wy_forward).
//
// One CTA per (batch, head) walks the sequence chunk by chunk (64 tokens,
// K = V = 128); the [K, V] state stays on chip in fp32 the whole time, as
// its transpose S^T in 128 TMEM columns (lane = value channel v, column =
// key channel n). Every product is a tcgen05.mma (kind::f16: bf16 operands,
// fp32 accumulation, M = 128) whose operands one thread points at in shared
// memory in the tensor core's 128-byte-swizzled layouts (rows of 128 bytes =
// 64 bf16, 8-row groups 1024 bytes apart, the 16-byte chunks of row r
// permuted by r % 8; rows along M or N for K-major operands, along K for
// MN-major ones).
//
// Inputs arrive by TMA, one chunk ahead: q, k and b straight into the first
// product's operands, v and w as the same 128-byte-swizzled 64-column boxes,
// g into a staging buffer; each copy is issued as soon as the buffer it
// lands in has been read for the current chunk, so it runs under the
// current chunk's work. Operands whose contraction runs over tokens (b*k*
// exp G, k*exp(G[last] - G), w*v) are kept row-major, token by channel, and
// handed to the tensor core as MN-major operands -- no transposes.
//
// Per chunk (the page's steps, with the products arranged so that M = 128):
//  0. column pass (thread = one key channel, 32 tokens): G = cumsum of g,
//     E+ = exp(G - G[m]) about the middle token m (fp32, in place of g).
//     Row pass (thread = 8 channels of a token): [E+; E+], E- = 1/E+ (in
//     place of v), q*exp(G)*scale, b*k, b*k*exp(G), k*exp(G[last] - G), w*v;
//  1. MMA [q; b*k] k^T and [E+; E+] E-^T (K * decay in both lane halves:
//     the key-mean of exp(G[i] - G[j]) = E+[i] . E-[j] / K); then, from
//     the state before the chunk, out^T = S^T (q*exp(G)*scale)^T (the
//     output's inter-chunk term) and Y^T = S^T (b*k*exp(G))^T;
//  2. aqk = qk * decay * scale (j <= i), akk = (bk)k^T * decay (j < i);
//     Z = w*v - Y (the page's u - W S before the triangular solve: with
//     (I + akk) W = b*k*exp(G) and (I + akk) U = w*v, v_new = U - W S is
//     (I + akk)^-1 Z);
//  3. T = (I + akk)^-1 by 2 x 2 block inversion (16 x 16 diagonal blocks
//     by forward substitution, the off-diagonal blocks as warp-level tf32
//     products: T is rounded to bf16 for the product that uses it);
//     MMA v_new^T = Z^T T^T;
//  4. S^T scaled column-wise by exp(G[last]); MMA out^T += v_new^T aqk^T and
//     S^T += v_new^T (k*exp(G[last]-G)).
// The state's bf16 copy that the products read is refreshed from TMEM
// after every chunk.
//
// Every wait (copies, tensor-core completions) is bounded (1 s); a wait that
// runs out sets the timeout status bit, the CTA waits (bounded) for its
// copies still in flight and stops.
#include "ssm_common.cuh"
#include "ssm_internal.h"
#include "tc_common.cuh"
#include "../../include/gdn2.h"

namespace ssm {

namespace {

using namespace tc;

constexpr int kGC = 64;    // tokens per chunk
constexpr int kGK = 128;   // key channels
constexpr int kGV = 128;   // value channels
constexpr int kGThreads = 256;

// Shared-memory regions (bytes from a 1024-byte aligned base). Regions used
// in disjoint phases of a chunk share space.
constexpr int kA1 = 0;                  // [q; b*k]            128 rows x K=128 (q, b by TMA)
constexpr int kB1 = kA1 + 32768;        // k                    64 rows x K=128 (TMA)
constexpr int kA2 = kB1 + 16384;        // [E+; E+]            128 rows x K=128
constexpr int kA3 = kA2 + 32768;        // b*k*exp(G)          [64 tokens][128] (then Z^T, then v_new^T)
constexpr int kA4 = kA3 + 16384;        // w (TMA), then w*v   MN-major [64 tokens][128]
constexpr int kA5 = kA4 + 16384;        // S^T (bf16)          128 rows x K=128
constexpr int kB7 = kA5 + 32768;        // q*exp(G)*scale       64 rows x K=128
constexpr int kB8 = kB7 + 16384;        // k*exp(Glast-G)      MN-major [64 tokens][128]
constexpr int kGS = kB8 + 16384;        // g staging fp32 [64][128] (TMA) -> E+; then T fp32
constexpr int kVS = kGS + 32768;        // v staging, swz(token, channel, 64) image (TMA); then E- 64 rows x K=128
constexpr int kMisc = kVS + 16384;      // em, egl, elm [128] fp32; mbarriers; TMEM slot
constexpr int kB6 = kA2;                // aqk                  64 rows x K=64
constexpr int kB3 = kA2 + 8192;         // T                    64 rows x K=64 (as A: 128 rows, the rest unused)
constexpr int kAKK = kA2 + 16384;       // akk fp32 [64][64], row-major, float4 chunks permuted per row
constexpr int kAZ = kA3;                // Z^T = (w*v - b*k*exp(G) S)^T  128 rows x K=64
constexpr int kA6 = kA3;                // v_new^T             128 rows x K=64
constexpr int kGSmem = kMisc + 1536 + 64 + 1024;  // + slack for the 1024-byte alignment
static_assert(kGSmem <= 227 * 1024, "shared memory");
constexpr unsigned kQkbBytes = 3 * 2 * 64 * 128;  // q, b, k: two 64-column boxes each
constexpr unsigned kGBytes = kGC * kGK * 4, kVBytes = kGC * kGV * 2;

// TMEM columns: S^T; per chunk qk|bkk, the decay, out^T, Y^T = (b*k*exp(G) S)^T and v_new^T.
constexpr unsigned kTS = 0, kTD1 = 128, kTD2 = 192, kTDOUT = 256, kTDY = 320, kTDV = 384;

// D[16 x 8] += A[16 x 8] B[8 x 8] on the warp's tensor-core path (tf32
// operands, fp32 accumulation); g = lane / 4, t = lane % 4 hold
// a = {A[g][t], A[g+8][t], A[g][t+4], A[g+8][t+4]}, b = {B[t][g], B[t+4][g]},
// d = {D[g][2t], D[g][2t+1], D[g+8][2t], D[g+8][2t+1]}.
__device__ __forceinline__ unsigned tf32(float x) {
    unsigned u;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(u) : "f"(x));
    return u;
}
__device__ __forceinline__ void mma_tf32(float* d, const float* a, const float* b) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(tf32(a[0])), "r"(tf32(a[1])), "r"(tf32(a[2])), "r"(tf32(a[3])), "r"(tf32(b[0])), "r"(tf32(b[1])));
}

struct Gdn2Params {
    int64_t B, H, T;
    float scale;
    unsigned* status;
    unsigned long long wait_ns;  // bound of every wait (kWaitNs unless a test armed a fault)
    int64_t fault_chunk1;        // tests: chunk fault_chunk1 - 1's q, k, b copies are not issued (0: none)
};
struct Gdn2Maps {
    CUtensorMap q, k, b, g, v, w;  // rows = B*H*T tokens; q, k, b, v, w: 64-column swizzled boxes; g: whole rows
};

__global__ void __launch_bounds__(kGThreads, 1)
    gdn2_chunk_fwd_kernel(const Gdn2Params p, const float* __restrict__ state_in, __nv_bfloat16* __restrict__ out,
                          float* __restrict__ state_out, const __grid_constant__ Gdn2Maps mp) {
    extern __shared__ __align__(1024) char g_smem_raw[];
    char* sm = g_smem_raw + ((1024u - (smem_u32(g_smem_raw) & 1023u)) & 1023u);
    float* s_em = reinterpret_cast<float*>(sm + kMisc);  // exp(G[m]) per key channel
    float* s_egl = s_em + kGK;                           // exp(G[last])
    float* s_elm = s_egl + kGK;                          // exp(G[last] - G[m])
    uint64_t* bars = reinterpret_cast<uint64_t*>(s_elm + kGK);  // mma, qkb, g, v, w, mma (second batch)
    unsigned* tslot = reinterpret_cast<unsigned*>(bars + 6);
    float* s_gm = reinterpret_cast<float*>(sm + kA2);    // column-pass exchange (A2 is written after it)
    float* s_e = reinterpret_cast<float*>(sm + kGS);     // g, then E+ [64][128]; then T (fp32) and scratch
    float* s_akk = reinterpret_cast<float*>(sm + kAKK);
    // akk[i][j]: row i, its float4 chunks permuted by i % 16 (conflict-free row writes, one per lane)
    auto akk_at = [&](int i, int j) -> float* { return s_akk + i * kGC + ((((j >> 2) ^ (i & 15)) << 2) | (j & 3)); };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, whalf = warp >> 2;  // TMEM lanes 32*quarter..; column half
    const int64_t bh = blockIdx.x;
    const int64_t T = p.T;
    const int nchunks = (int)((T + kGC - 1) / kGC);
    const unsigned sbase = smem_u32(sm);
    const unsigned mbar = smem_u32(bars), bar_qkb = smem_u32(bars + 1), bar_g = smem_u32(bars + 2),
                   bar_v = smem_u32(bars + 3), bar_w = smem_u32(bars + 4), mbar2 = smem_u32(bars + 5);
    constexpr float L2E = 1.4426950408889634f;

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_u32(tslot)),
                     "r"(512)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    }
    // the copies of chunk cj (issued by kTmaThread); rows past the end of the
    // whole tensor read as zero, rows of the next (batch, head) are zeroed or
    // ignored on the ragged last chunk
    auto row_of = [&](int cj) { return (int)(bh * T + (int64_t)cj * kGC); };
    // a test-armed fault: this chunk's q, k, b copies are never issued, so the
    // bounded wait for them runs out
    auto qkb_skipped = [&](int cj) { return (int64_t)cj + 1 == p.fault_chunk1; };
    auto issue_qkb = [&](int cj) {
        if (qkb_skipped(cj)) return;
        const int y = row_of(cj);
        mbar_expect_tx(bar_qkb, kQkbBytes);
#pragma unroll
        for (int at = 0; at < 2; ++at) {  // x = 0, 64: 128-byte aligned
            tma_load_2d(sm + kA1 + at * 16384, &mp.q, at * 64, y, bar_qkb);
            tma_load_2d(sm + kA1 + at * 16384 + 8192, &mp.b, at * 64, y, bar_qkb);
            tma_load_2d(sm + kB1 + at * 8192, &mp.k, at * 64, y, bar_qkb);
        }
    };
    auto issue_one = [&](unsigned bar, int off, const CUtensorMap* m, unsigned bytes, int cj) {
        mbar_expect_tx(bar, bytes);
        tma_load_2d(sm + off, m, 0, row_of(cj), bar);
    };
    auto issue_sw = [&](unsigned bar, int off, const CUtensorMap* m, int cj) {  // two 64-column swizzled boxes
        mbar_expect_tx(bar, kVBytes);
        tma_load_2d(sm + off, m, 0, row_of(cj), bar);
        tma_load_2d(sm + off + 8192, m, 64, row_of(cj), bar);
    };
    // thread kTmaThread (warp 2, idle while the first two lane quarters run the
    // epilogues) issues the copies; thread 0 issues the products
    constexpr int kTmaThread = 64;
    if (tid == kTmaThread) {
        const CUtensorMap* maps[6] = {&mp.q, &mp.k, &mp.b, &mp.g, &mp.v, &mp.w};
        for (int m = 0; m < 6; ++m)
            asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(maps[m])) : "memory");
    }
    if (tid == 0) {
        for (int b = 0; b < 6; ++b) mbar_init(smem_u32(bars + b), 1);
        mbar_fence_init();
    }
    __syncthreads();
    if (tid == kTmaThread) {
        if (nchunks > 0) {
            issue_qkb(0);
            issue_one(bar_g, kGS, &mp.g, kGBytes, 0);
            issue_sw(bar_v, kVS, &mp.v, 0);
            issue_sw(bar_w, kA4, &mp.w, 0);
        }
    }
    tc_before();
    __syncthreads();
    tc_after();
    const unsigned tmem = *tslot;
    const unsigned tlane = (unsigned)(quarter * 32) << 16;  // this warp's TMEM lane quarter
    const int vrow = quarter * 32 + lane;                    // the TMEM lane (row) this thread reads

    // ---- the initial state: S^T into TMEM (lane v, column n) and its bf16 copy
    {
        const float* s0 = state_in ? state_in + bh * kGK * kGV : nullptr;
        for (int c = 0; c < 2; ++c) {
            const int n0 = whalf * 64 + c * 32;
            float vals[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) vals[i] = s0 ? s0[(int64_t)(n0 + i) * kGV + vrow] : 0.f;
            tmem_st32(tmem + tlane + kTS + (unsigned)n0, vals);
#pragma unroll
            for (int i = 0; i < 32; i += 8) st8(sm + kA5, vrow, n0 + i, 128, vals + i);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
    }
    fence_async_smem();
    tc_before();
    __syncthreads();

    // Tensor-core completions: `mbar` for the rounds waited in order, `mbar2`
    // for the second batch of round 1 (committed right after the first, so on
    // one barrier the two could complete two phases before anyone polls).
    unsigned phase = 0, phase2 = 0;
    // copies issued / waited for, per barrier (qkb, g, v, w); uniform over the CTA
    int issued[4] = {nchunks > 0 && !qkb_skipped(0), nchunks > 0, nchunks > 0, nchunks > 0}, waited[4] = {0, 0, 0, 0};
    const unsigned tbar[4] = {bar_qkb, bar_g, bar_v, bar_w};
    float nf = 0.f;
    auto fail = [&]() {
        if (tid == 0 && p.status) atomicOr(p.status, kStatusTimeout);
    };
    auto mma_wait = [&]() -> bool {  // every thread waits for the last commit; false if it never came
        const bool ok = mbar_wait_try(mbar, phase & 1u, p.wait_ns);
        phase++;
        if (!ok) fail();
        return __syncthreads_and(ok) != 0;
    };
    auto mma_wait2 = [&]() -> bool {  // the second batch of round 1
        const bool ok = mbar_wait_try(mbar2, phase2 & 1u, p.wait_ns);
        phase2++;
        if (!ok) fail();
        return __syncthreads_and(ok) != 0;
    };
    auto copies_wait = [&](int b0, int b1) -> bool {  // copies b0..b1 of the current chunk, one CTA barrier
        bool ok = true;
        for (int b = b0; b <= b1; ++b) ok = ok && mbar_wait_try(tbar[b], (unsigned)(waited[b] & 1), p.wait_ns);
        if (!ok) fail();
        const bool all = __syncthreads_and(ok) != 0;
        if (all)
            for (int b = b0; b <= b1; ++b) waited[b]++;
        return all;
    };
    auto commit_to = [&](unsigned bar) {
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar)
                     : "memory");
    };
    auto commit = [&]() { commit_to(mbar); };
    auto refill = [&](int b, int cj) {  // next chunk's copy into a buffer all threads are done reading
        if (cj >= nchunks) return;
        if (tid == kTmaThread) {
            fence_async_smem();
            if (b == 0) issue_qkb(cj);
            else if (b == 1) issue_one(bar_g, kGS, &mp.g, kGBytes, cj);
            else if (b == 2) issue_sw(bar_v, kVS, &mp.v, cj);
            else issue_sw(bar_w, kA4, &mp.w, cj);
        }
        issued[b] += (b == 0 && qkb_skipped(cj)) ? 0 : 1;
    };

    bool ok = true;
    for (int ci = 0; ci < nchunks && ok; ++ci) {
        const int64_t t0 = (int64_t)ci * kGC;
        const int c = (int)min64(kGC, T - t0);  // live tokens; rows c..63 are zero (identity tokens)
        const int64_t row0 = bh * T + t0;      // first token row of the chunk in [B*H*T]

        // ---- 0. column pass (thread = key channel n, tokens 32*hf ..+31):
        // G = cumsum(g) and E+ = exp(G - G[m]) in place of g; per-channel
        // exp(G[m]), exp(G[last]), exp(G[last] - G[m])
        if (!(ok = copies_wait(0, 3))) break;
        {
            const int n = tid & (kGK - 1), hf = tid >> 7, j0 = hf * 32;
            float G[32];
            float acc = 0.f;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                acc = __fadd_rn(acc, j0 + i < c ? s_e[(j0 + i) * kGK + n] : 0.f);
                G[i] = acc;
            }
            if (hf == 0) s_gm[n] = acc;  // G at the middle token m = 31
            __syncthreads();
            const float Gm = s_gm[n];
            if (hf == 1) {
#pragma unroll
                for (int i = 0; i < 32; ++i) G[i] = __fadd_rn(G[i], Gm);
                const float Gl = G[31];  // G at the last row (= the last live token: later rows add zeros)
                s_em[n] = ex2(Gm * L2E);
                s_egl[n] = ex2(Gl * L2E);
                s_elm[n] = ex2((Gl - Gm) * L2E);
            }
#pragma unroll
            for (int i = 0; i < 32; ++i) s_e[(j0 + i) * kGK + n] = ex2((G[i] - Gm) * L2E);  // same thread's entries
        }
        __syncthreads();  // E+; the exp tables
        // ---- 0c. row pass (thread = token r, channels cc..cc+7): [E+; E-],
        // q*exp(G)*scale, b*k in place of b, and the MN-major operands
        // b*k*exp(G), k*exp(G[last] - G), w*v (in place of w). Rows past the
        // chunk's tokens: b*k, k, w*v zeroed (identity tokens); q's rows there
        // only reach outputs that are not stored.
        {
        const int cc = (tid & 15) * 8;  // the thread's channels, the same for its four tokens
        float em8[8], elm8[8];
        *reinterpret_cast<float4*>(em8) = *reinterpret_cast<const float4*>(s_em + cc);
        *reinterpret_cast<float4*>(em8 + 4) = *reinterpret_cast<const float4*>(s_em + cc + 4);
        *reinterpret_cast<float4*>(elm8) = *reinterpret_cast<const float4*>(s_elm + cc);
        *reinterpret_cast<float4*>(elm8 + 4) = *reinterpret_cast<const float4*>(s_elm + cc + 4);
#pragma unroll 2
        for (int it = 0; it < 4; ++it) {
            const int r = (tid >> 4) + it * (kGThreads >> 4);
            const bool live = r < c;
            float ep[8], en[8], qv[8], kv[8], bv[8], wv[8], vv[8];
            *reinterpret_cast<float4*>(ep) = *reinterpret_cast<const float4*>(s_e + r * kGK + cc);
            *reinterpret_cast<float4*>(ep + 4) = *reinterpret_cast<const float4*>(s_e + r * kGK + cc + 4);
            ld8(sm + kA1, r, cc, 128, qv);
            ld8(sm + kA1, 64 + r, cc, 128, bv);
            ld8(sm + kB1, r, cc, 64, kv);
            ld8(sm + kA4, r, cc, 64, wv);
            ld8(sm + kVS, r, cc, 64, vv);
            float qg[8], bk[8], rk[8], kp[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                en[i] = rcp(ep[i]);
                const float eg = ep[i] * em8[i];  // exp(G)
                qg[i] = qv[i] * eg * p.scale;
                const float kk = live ? kv[i] : 0.f;
                kv[i] = kk;
                bk[i] = live ? bv[i] * kk : 0.f;
                rk[i] = bk[i] * eg;
                kp[i] = kk * (en[i] * elm8[i]);  // k*exp(G[last] - G)
                wv[i] = live ? wv[i] * vv[i] : 0.f;
            }
            st8(sm + kA2, r, cc, 128, ep);
            st8(sm + kA2, 64 + r, cc, 128, ep);
            st8(sm + kVS, r, cc, 64, en);  // in place of v (same thread, same chunk of the image)
            st8(sm + kB7, r, cc, 64, qg);
            st8(sm + kA1, 64 + r, cc, 128, bk);
            if (!live) st8(sm + kB1, r, cc, 64, kv);
            st8(sm + kA3, r, cc, 64, rk);
            st8(sm + kB8, r, cc, 64, kp);
            st8(sm + kA4, r, cc, 64, wv);
        }
        }
        fence_async_smem();
        tc_before();
        __syncthreads();

        // ---- 1. qk^T | (bk)k^T and [E+; E+] E-^T (K * decay in both lane halves); then the
        // products that need only the state before the chunk: out^T = S^T (q exp(G) scale)^T
        // and Y^T = S^T (b k exp(G))^T, committed separately
        if (tid == 0) {
            tc_after();
            mma_issue(tmem + kTD1, sbase + kA1, sbase + kB1, 64, 64, kGK, false);
            mma_issue(tmem + kTD2, sbase + kA2, sbase + kVS, 64, 64, kGK, false);
            commit();
        } else if (tid == 32) {  // a second issuing thread: its commit covers its own products
            tc_after();
            mma_issue(tmem + kTDOUT, sbase + kA5, sbase + kB7, 64, 64, kGK, false);
            mma_issue(tmem + kTDY, sbase + kA5, sbase + kA3, 64, 64, kGK, false);
            commit_to(mbar2);
        }
        if (!(ok = mma_wait())) break;
        tc_after();
        refill(0, ci + 1);  // q, k, b have been read
        refill(2, ci + 1);  // E- (in v's buffer) has been read

        // ---- 2. aqk (lanes 0-63) and akk (lanes 64-127), the decay in both lane halves
        {
            const int jb = whalf * 32;
            float d1[32], d2[32];
            tmem_ld32(tmem + tlane + kTD1 + (unsigned)jb, d1);
            tmem_ld32(tmem + tlane + kTD2 + (unsigned)jb, d2);
            if (quarter < 2) {
                const int i = vrow;
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) d1[jj] = (jb + jj <= i) ? d1[jj] * d2[jj] * (p.scale / kGK) : 0.f;
#pragma unroll
                for (int jj = 0; jj < 32; jj += 8) st8(sm + kB6, i, jb + jj, 64, d1 + jj);
            } else {
                const int i = vrow - 64;
#pragma unroll
                for (int jj = 0; jj < 32; jj += 4) {
                    float a4[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) a4[e] = (jb + jj + e < i) ? d1[jj + e] * d2[jj + e] * (1.f / kGK) : 0.f;
                    *reinterpret_cast<float4*>(akk_at(i, jb + jj)) = make_float4(a4[0], a4[1], a4[2], a4[3]);
                }
            }
        }
        // Z^T = (w v)^T - Y^T (lane v, tokens j), the right-hand side of v_new = T Z
        if (!(ok = mma_wait2())) break;
        tc_after();
        {
            const int jb = whalf * 32;
            float y[32];
            tmem_ld32(tmem + tlane + kTDY + (unsigned)jb, y);
#pragma unroll
            for (int jj = 0; jj < 32; ++jj)
                y[jj] = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(sm + kA4 + swz(jb + jj, vrow, 64))) - y[jj];
#pragma unroll
            for (int jj = 0; jj < 32; jj += 8) st8(sm + kAZ, vrow, jb + jj, 128, y + jj);
        }
        tc_before();
        __syncthreads();
        refill(3, ci + 1);  // w*v has been read: the next w can land in its buffer

        // ---- 3. T = (I + akk)^-1 by blocks; then v_new = T Z
        // The inverse of the unit lower-triangular I + akk by blocks: for
        // [[A, 0], [C, B]] the inverse is [[A^-1, 0], [-B^-1 C A^-1, B^-1]].
        // (a) the four diagonal 16 x 16 blocks by forward substitution (one
        // thread per column); (b) the two off-diagonal 16 x 16 blocks inside
        // the 32 x 32 halves; (c) the lower 32 x 32 block. fp32 throughout; every
        // block is also written as the bf16 K-major operand T (rows r, K = column).
        constexpr int TS = kGC + 4;   // row stride of T: rows 4 banks apart
        float* TT = s_e;              // T fp32 [64][TS], row-major (g's staging buffer is free)
        float* TY = s_e + kGC * TS;   // scratch products
        if (tid < kGC) {  // (a): thread = column cl of diagonal block base/16, rows in order
            const int base = (tid >> 4) * 16, cl = tid & 15;
            float x[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                float acc0 = r == cl ? 1.f : 0.f, acc1 = 0.f;
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    if (4 * q4 < r) {
                        const float4 a = *reinterpret_cast<const float4*>(akk_at(base + r, base + 4 * q4));
                        const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            if (4 * q4 + e < r) {
                                if (e & 1) acc1 = __fmaf_rn(-av[e], x[4 * q4 + e], acc1);
                                else acc0 = __fmaf_rn(-av[e], x[4 * q4 + e], acc0);
                            }
                    }
                }
                x[r] = acc0 + acc1;
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                TT[(base + r) * TS + base + cl] = x[r];
                st1(sm + kB3, base + r, base + cl, 64, x[r]);
            }
        } else {  // zeros above the diagonal blocks: blocks (0,1), (2,3) and the upper 32 x 32
            for (int e = tid - kGC; e < 1024 + 512; e += kGThreads - kGC) {
                int r, cc;
                if (e < 1024) {  // rows 0-31, columns 32-63
                    r = e >> 5;
                    cc = 32 + (e & 31);
                } else {         // block (0,1) (rows 0-15, columns 16-31) or (2,3) (rows 32-47, columns 48-63)
                    const int f = e - 1024, blk = f >> 8;
                    r = 32 * blk + ((f >> 4) & 15);
                    cc = 32 * blk + 16 + (f & 15);
                }
                TT[r * TS + cc] = 0.f;
                st1(sm + kB3, r, cc, 64, 0.f);
            }
        }
        __syncthreads();
        {   // (b) T[R0+r][C0+c] = -D_hi (L D_lo), R0 = 16 + 32p, C0 = 32p: warps 0-3,
            // problem p = warp / 2, 8-column tile nj = warp % 2, two k-steps of 8
            const int g = lane >> 2, t = lane & 3;
            const int pb = (warp >> 1) & 1, nj = warp & 1;
            const int R0 = 16 + 32 * pb, C0 = 32 * pb;
            float d[4] = {0.f, 0.f, 0.f, 0.f};
            if (warp < 4) {
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) {
                    const int k0 = 8 * ks;
                    const float av[4] = {*akk_at(R0 + g, C0 + k0 + t), *akk_at(R0 + g + 8, C0 + k0 + t),
                                         *akk_at(R0 + g, C0 + k0 + t + 4), *akk_at(R0 + g + 8, C0 + k0 + t + 4)};
                    const float bv[2] = {TT[(C0 + k0 + t) * TS + C0 + 8 * nj + g],
                                         TT[(C0 + k0 + t + 4) * TS + C0 + 8 * nj + g]};
                    mma_tf32(d, av, bv);
                }
                float* y = TY + pb * 256 + 8 * nj + 2 * t;  // Y [16][16] per problem
                y[g * 16] = d[0]; y[g * 16 + 1] = d[1]; y[(g + 8) * 16] = d[2]; y[(g + 8) * 16 + 1] = d[3];
            }
            __syncthreads();
            if (warp < 4) {
                d[0] = d[1] = d[2] = d[3] = 0.f;
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) {
                    const int k0 = 8 * ks;
                    const float* dh = TT + (R0 + g) * TS + R0 + k0 + t;
                    const float av[4] = {-dh[0], -dh[8 * TS], -dh[4], -dh[8 * TS + 4]};
                    const float* yb = TY + pb * 256 + (k0 + t) * 16 + 8 * nj + g;
                    const float bv[2] = {yb[0], yb[4 * 16]};
                    mma_tf32(d, av, bv);
                }
                float* o = TT + (R0 + g) * TS + C0 + 8 * nj + 2 * t;
                o[0] = d[0]; o[1] = d[1]; o[8 * TS] = d[2]; o[8 * TS + 1] = d[3];
                st2(sm + kB3, R0 + g, C0 + 8 * nj + 2 * t, 64, d[0], d[1]);
                st2(sm + kB3, R0 + g + 8, C0 + 8 * nj + 2 * t, 64, d[2], d[3]);
            }
        }
        __syncthreads();
        {   // (c) T[32+r][c] = -E1 (L E0), E0 = T[0:32][0:32], E1 = T[32:64][32:64]:
            // 16-row tile mi = warp / 4, 8-column tile nj = warp % 4, four k-steps
            const int g = lane >> 2, t = lane & 3;
            const int mi = warp >> 2, nj = warp & 3;
            const int r0 = 16 * mi, cc = 8 * nj;
            float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                const int k0 = 8 * ks;
                const float av[4] = {*akk_at(32 + r0 + g, k0 + t), *akk_at(32 + r0 + g + 8, k0 + t),
                                     *akk_at(32 + r0 + g, k0 + t + 4), *akk_at(32 + r0 + g + 8, k0 + t + 4)};
                const float bv[2] = {TT[(k0 + t) * TS + cc + g], TT[(k0 + t + 4) * TS + cc + g]};
                mma_tf32(d, av, bv);
            }
            float* y = TY + (r0 + g) * 32 + cc + 2 * t;  // Y [32][32]
            y[0] = d[0]; y[1] = d[1]; y[8 * 32] = d[2]; y[8 * 32 + 1] = d[3];
            __syncthreads();
            d[0] = d[1] = d[2] = d[3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                const int k0 = 8 * ks;
                const float* e1 = TT + (32 + r0 + g) * TS + 32 + k0 + t;
                const float av[4] = {-e1[0], -e1[8 * TS], -e1[4], -e1[8 * TS + 4]};
                const float bv[2] = {TY[(k0 + t) * 32 + cc + g], TY[(k0 + t + 4) * 32 + cc + g]};
                mma_tf32(d, av, bv);
            }
            float* o = TT + (32 + r0 + g) * TS + cc + 2 * t;
            o[0] = d[0]; o[1] = d[1]; o[8 * TS] = d[2]; o[8 * TS + 1] = d[3];
            st2(sm + kB3, 32 + r0 + g, cc + 2 * t, 64, d[0], d[1]);
            st2(sm + kB3, 32 + r0 + g + 8, cc + 2 * t, 64, d[2], d[3]);
        }
        fence_async_smem();
        tc_before();
        __syncthreads();
        refill(1, ci + 1);  // g's buffer (E+, then T) has been read
        if (tid == 0) {
            tc_after();
            mma_issue(tmem + kTDV, sbase + kAZ, sbase + kB3, 64, 64, kGC, false);  // v_new^T = Z^T T^T
            commit();
        }
        if (!(ok = mma_wait())) break;
        tc_after();
        {
            float u[32];
            const int i0 = whalf * 32;
            tmem_ld32(tmem + tlane + kTDV + (unsigned)i0, u);
#pragma unroll
            for (int ii = 0; ii < 32; ii += 8) st8(sm + kA6, vrow, i0 + ii, 128, u + ii);
            // S^T columns n scaled by exp(G[last][n]) before the update is added
            for (int cc = 0; cc < 2; ++cc) {
                const int n0 = whalf * 64 + cc * 32;
                float s[32];
                tmem_ld32(tmem + tlane + kTS + (unsigned)n0, s);
#pragma unroll
                for (int nn = 0; nn < 32; ++nn) s[nn] *= s_egl[n0 + nn];
                tmem_st32(tmem + tlane + kTS + (unsigned)n0, s);
            }
            asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
        }
        fence_async_smem();
        tc_before();
        __syncthreads();

        // ---- 5. out^T += v_new^T aqk^T (the inter-chunk term is in already);  S^T += v_new^T (k exp(Glast - G))
        if (tid == 0) {
            tc_after();
            mma_issue(tmem + kTDOUT, sbase + kA6, sbase + kB6, 64, 64, kGC, true);
            mma_issue(tmem + kTS, sbase + kA6, sbase + kB8, 0, 128, kGC, true, false, true);
            commit();
        }
        if (!(ok = mma_wait())) break;
        tc_after();
        {
            float o[32];
            const int i0 = whalf * 32;
            tmem_ld32(tmem + tlane + kTDOUT + (unsigned)i0, o);
#pragma unroll
            for (int ii = 0; ii < 32; ++ii) {
                if (i0 + ii < c) {
                    nf = __fmaf_rn(o[ii], 0.f, nf);
                    out[(row0 + i0 + ii) * kGV + vrow] = __float2bfloat16_rn(o[ii]);
                }
            }
            // the bf16 copy of the updated state for the next chunk's products
            for (int cc = 0; cc < 2; ++cc) {
                const int n0 = whalf * 64 + cc * 32;
                float s[32];
                tmem_ld32(tmem + tlane + kTS + (unsigned)n0, s);
#pragma unroll
                for (int nn = 0; nn < 32; nn += 8) st8(sm + kA5, vrow, n0 + nn, 128, s + nn);
            }
        }
        fence_async_smem();
        tc_before();
        __syncthreads();
    }

    if (!ok) {  // a wait ran out: let the copies still in flight land before the CTA exits
        if (tid == kTmaThread)
            for (int b = 0; b < 4; ++b)
                for (; waited[b] < issued[b]; ++waited[b])
                    if (!mbar_wait_try(tbar[b], (unsigned)(waited[b] & 1), p.wait_ns)) break;
    } else if (state_out) {
        float* so = state_out + bh * kGK * kGV;
        for (int cc = 0; cc < 2; ++cc) {
            const int n0 = whalf * 64 + cc * 32;
            float s[32];
            tmem_ld32(tmem + tlane + kTS + (unsigned)n0, s);
#pragma unroll
            for (int nn = 0; nn < 32; ++nn) so[(int64_t)(n0 + nn) * kGV + vrow] = s[nn];
        }
    }
    flag_nonfinite(p.status, nf);
    tc_before();
    __syncthreads();
    if (warp == 0) {
        tc_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(512) : "memory");
    }
}

// ---------------------------------------------------------------- one token: the per-token form
struct Gdn2StepParams {
    float scale;
    const __nv_bfloat16* q;
    const __nv_bfloat16* k;
    const __nv_bfloat16* v;
    const float* g;
    const __nv_bfloat16* b;
    const __nv_bfloat16* w;
    float* S;
    __nv_bfloat16* out;
    unsigned* status;
};

// One CTA of 256 threads per (batch, head), fp32. Thread (v = tid % 128, kh = tid / 128) holds the 64 entries
// S[k][v] of its key half in registers: one pass decays them and sums (b k)^T S for v_new, a second adds
// k v_new^T, writes them back and sums q^T S; the key halves meet in shared memory.
__global__ void __launch_bounds__(kGThreads) gdn2_step_kernel(const Gdn2StepParams p) {
    __shared__ float s_eg[kGK], s_bk[kGK], s_k[kGK], s_q[kGK];
    __shared__ float s_part[2][kGV];
    __shared__ float s_vn[kGV];
    const int tid = threadIdx.x;
    const int64_t bh = blockIdx.x;
    if (tid < kGK) {
        const int64_t i = bh * kGK + tid;
        const float kk = __bfloat162float(p.k[i]);
        s_eg[tid] = expf(p.g[i]);
        s_k[tid] = kk;
        s_bk[tid] = __bfloat162float(p.b[i]) * kk;
        s_q[tid] = __bfloat162float(p.q[i]) * p.scale;
    }
    __syncthreads();
    const int v = tid & (kGV - 1), kh = tid >> 7, k0 = kh * (kGK / 2);
    float* Sb = p.S + bh * kGK * kGV;
    float sv[kGK / 2];
    float acc = 0.f;
#pragma unroll
    for (int kk = 0; kk < kGK / 2; ++kk) {
        sv[kk] = Sb[(int64_t)(k0 + kk) * kGV + v] * s_eg[k0 + kk];
        acc = __fmaf_rn(s_bk[k0 + kk], sv[kk], acc);
    }
    s_part[kh][v] = acc;
    __syncthreads();
    if (tid < kGV) {
        const int64_t i = bh * kGV + tid;
        s_vn[tid] = __bfloat162float(p.w[i]) * __bfloat162float(p.v[i]) - (s_part[0][tid] + s_part[1][tid]);
    }
    __syncthreads();
    const float vn = s_vn[v];
    acc = 0.f;
#pragma unroll
    for (int kk = 0; kk < kGK / 2; ++kk) {
        const float x = __fmaf_rn(s_k[k0 + kk], vn, sv[kk]);
        Sb[(int64_t)(k0 + kk) * kGV + v] = x;
        acc = __fmaf_rn(s_q[k0 + kk], x, acc);
    }
    __syncthreads();  // every thread has read s_part before it is reused
    s_part[kh][v] = acc;
    __syncthreads();
    float o = 0.f;
    if (tid < kGV) {
        o = s_part[0][tid] + s_part[1][tid];
        p.out[bh * kGV + tid] = __float2bfloat16_rn(o);
    }
    flag_nonfinite(p.status, __fmaf_rn(o, 0.f, 0.f));
}

bool misaligned16(const void* q) { return q && (reinterpret_cast<uintptr_t>(q) & 15u) != 0; }

}  // namespace
}  // namespace ssm

namespace {
// One-shot wait fault for this thread's next gdn2_chunk_fwd (tests).
thread_local int64_t g_gdn2_fault_chunk1 = 0;
thread_local unsigned long long g_gdn2_fault_wait_ns = 0;
}  // namespace

extern "C" int gdn2_debug_arm_wait_fault(int64_t chunk, uint64_t wait_ns) {
    if (wait_ns > 10000000000ull) return SSM_ERR_INVALID_ARG;
    g_gdn2_fault_chunk1 = chunk < 0 ? 0 : chunk + 1;
    g_gdn2_fault_wait_ns = chunk < 0 ? 0 : wait_ns;
    return SSM_OK;
}

extern "C" int gdn2_chunk_fwd(const gdn2_fwd_args* a, void* stream) {
    ssm::reset_launches();
    // an armed fault applies to this call only
    const int64_t fault_chunk1 = g_gdn2_fault_chunk1;
    const unsigned long long fault_wait_ns = g_gdn2_fault_wait_ns;
    g_gdn2_fault_chunk1 = 0;
    g_gdn2_fault_wait_ns = 0;
    if (!a) return SSM_ERR_INVALID_ARG;
    if (a->B < 0 || a->H < 0 || a->T < 0) return SSM_ERR_INVALID_ARG;
    if (a->K != ssm::kGK || a->V != ssm::kGV || (a->chunk != 0 && a->chunk != ssm::kGC)) return SSM_ERR_UNSUPPORTED;
    if (!(fabsf(a->scale) <= 3.0e38f)) return SSM_ERR_INVALID_ARG;  // NaN or infinite scale
    if (a->B * a->H > 0x7fffffff) return SSM_ERR_INVALID_ARG;
    // token rows are addressed by 32-bit copy coordinates
    if (a->T > 0x7fffffff || a->B * a->H * a->T > 0x7fffffff - 2 * ssm::kGC) return SSM_ERR_UNSUPPORTED;
    const bool work = a->B > 0 && a->H > 0 && a->T > 0;
    if (work && (!a->q || !a->k || !a->v || !a->g || !a->b || !a->w || !a->out)) return SSM_ERR_INVALID_ARG;
    const void* ptrs[] = {a->q, a->k, a->v, a->g, a->b, a->w, a->state_in, a->out, a->state_out, a->workspace};
    for (const void* q : ptrs)
        if (ssm::misaligned16(q)) return SSM_ERR_ALIGNMENT;
    cudaStream_t s = (cudaStream_t)stream;
    const int64_t BH = a->B * a->H;
    if (!work) {
        if (a->state_out && BH > 0) {
            const size_t bytes = (size_t)BH * ssm::kGK * ssm::kGV * sizeof(float);
            cudaError_t e = a->state_in ? cudaMemcpyAsync(a->state_out, a->state_in, bytes, cudaMemcpyDeviceToDevice, s)
                                        : cudaMemsetAsync(a->state_out, 0, bytes, s);
            if (e != cudaSuccess) return SSM_ERR_CUDA;
        }
        return SSM_OK;
    }
    static unsigned long long mask = 0;
    if (!ssm::ensure_smem(ssm::gdn2_chunk_fwd_kernel, ssm::kGSmem, mask)) return SSM_ERR_CUDA;
    ssm::Gdn2Params p{};
    p.B = a->B; p.H = a->H; p.T = a->T; p.scale = a->scale;
    p.status = (unsigned*)a->workspace;
    p.fault_chunk1 = fault_chunk1;
    p.wait_ns = fault_chunk1 > 0 && fault_wait_ns > 0 ? fault_wait_ns : ssm::kWaitNs;
    const int64_t rows = BH * a->T;
    ssm::Gdn2Maps mp{};
    const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, f32 = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    const bool enc =
        ssm::encode_2d(&mp.q, bf, a->q, ssm::kGK, rows, ssm::kGK * 2, 64, ssm::kGC, CU_TENSOR_MAP_SWIZZLE_128B) &&
        ssm::encode_2d(&mp.k, bf, a->k, ssm::kGK, rows, ssm::kGK * 2, 64, ssm::kGC, CU_TENSOR_MAP_SWIZZLE_128B) &&
        ssm::encode_2d(&mp.b, bf, a->b, ssm::kGK, rows, ssm::kGK * 2, 64, ssm::kGC, CU_TENSOR_MAP_SWIZZLE_128B) &&
        ssm::encode_2d(&mp.g, f32, a->g, ssm::kGK, rows, ssm::kGK * 4, ssm::kGK, ssm::kGC, CU_TENSOR_MAP_SWIZZLE_NONE) &&
        ssm::encode_2d(&mp.v, bf, a->v, ssm::kGV, rows, ssm::kGV * 2, 64, ssm::kGC, CU_TENSOR_MAP_SWIZZLE_128B) &&
        ssm::encode_2d(&mp.w, bf, a->w, ssm::kGV, rows, ssm::kGV * 2, 64, ssm::kGC, CU_TENSOR_MAP_SWIZZLE_128B);
    if (!enc) return SSM_ERR_CUDA;
    ssm::gdn2_chunk_fwd_kernel<<<(unsigned)BH, ssm::kGThreads, ssm::kGSmem, s>>>(
        p, a->state_in, (__nv_bfloat16*)a->out, a->state_out, mp);
    return ssm::count_launches(cudaGetLastError() == cudaSuccess ? 1 : -1);
}

extern "C" int gdn2_step(const gdn2_step_args* a, void* stream) {
    ssm::reset_launches();
    if (!a) return SSM_ERR_INVALID_ARG;
    if (a->B < 0 || a->H < 0) return SSM_ERR_INVALID_ARG;
    if (a->K != ssm::kGK || a->V != ssm::kGV) return SSM_ERR_UNSUPPORTED;
    if (!(fabsf(a->scale) <= 3.0e38f)) return SSM_ERR_INVALID_ARG;
    if (a->B * a->H > 0x7fffffff) return SSM_ERR_INVALID_ARG;
    const int64_t BH = a->B * a->H;
    if (BH == 0) return SSM_OK;
    if (!a->q || !a->k || !a->v || !a->g || !a->b || !a->w || !a->state || !a->out) return SSM_ERR_INVALID_ARG;
    const void* ptrs[] = {a->q, a->k, a->v, a->g, a->b, a->w, a->state, a->out, a->workspace};
    for (const void* q : ptrs)
        if (ssm::misaligned16(q)) return SSM_ERR_ALIGNMENT;
    ssm::Gdn2StepParams p{};
    p.scale = a->scale;
    p.q = (const __nv_bfloat16*)a->q; p.k = (const __nv_bfloat16*)a->k; p.v = (const __nv_bfloat16*)a->v;
    p.g = a->g; p.b = (const __nv_bfloat16*)a->b; p.w = (const __nv_bfloat16*)a->w;
    p.S = a->state; p.out = (__nv_bfloat16*)a->out; p.status = (unsigned*)a->workspace;
    ssm::gdn2_step_kernel<<<(unsigned)BH, ssm::kGThreads, 0, (cudaStream_t)stream>>>(p);
    return ssm::count_launches(cudaGetLastError() == cudaSuccess ? 1 : -1);
}
