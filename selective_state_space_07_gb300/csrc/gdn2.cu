// Gated DeltaNet-2 chunkwise forward on the sm_103a tensor cores
// (docs.rs, burn-gdn2 0.1.4, src/forward.rs, chunk_wy_forward).
//
// One CTA per (batch, head) walks the sequence chunk by chunk (64 tokens,
// K = V = 128); the [K, V] state stays on chip in fp32 the whole time, as
// its transpose S^T in 128 TMEM columns (lane = value channel v, column =
// key channel n). Every product is a tcgen05.mma (kind::f16: bf16 operands,
// fp32 accumulation, M = 128) whose operands one thread points at in shared
// memory in the tensor core's 128-byte-swizzled K-major layout (rows of
// 128 bytes = 64 bf16 of K, 8-row groups 1024 bytes apart, the 16-byte
// chunks of row r permuted by r % 8); the CTA's threads write those
// operands with ordinary stores, then fence them to the async proxy.
//
// Per chunk (the page's steps, with the products arranged so that M = 128):
//  1. load q, k, b*k (bf16) and w*v; the column threads form G = cumsum of
//     g, and from it E+ = exp(G - G[m]), E- = exp(G[m] - G) about the
//     middle token m, q*exp(G)*scale, (b*k*exp(G))^T and
//     (k*exp(G[last] - G))^T;
//  2. MMA [q; b*k] k^T and [E+; E+] E-^T (the second / K is the key-mean
//     of exp(G[i] - G[j]) = the decay, in both lane halves);
//  3. aqk = qk * decay * scale (j <= i) and akk = (bk)k^T * decay (j < i);
//  4. T = (I + akk)^-1 by forward substitution, one column per thread
//     (unit lower-triangular); then MMA W^T = (b*k*exp(G))^T T^T and
//     U^T = (w*v)^T T^T (the page's row-by-row WY substitution, as
//     (I + akk) W = rhs);
//  5. MMA (W S)^T = S^T W^T; v_new = U - W S;
//  6. MMA out^T = v_new^T aqk^T + S^T (q*exp(G)*scale)^T, and, after S^T
//     is scaled column-wise by exp(G[last]), S^T += v_new^T (k*exp(G[last]-G)).
// The state's bf16 copy that the products read is refreshed from TMEM
// after every chunk.
//
// Every wait on a tensor-core completion is bounded (1 s); a wait that runs
// out sets the timeout status bit and the CTA stops.
#include "ssm_common.cuh"
#include "ssm_internal.h"
#include "../../include/gdn2.h"

namespace ssm {

namespace {

constexpr int kGC = 64;    // tokens per chunk
constexpr int kGK = 128;   // key channels
constexpr int kGV = 128;   // value channels
constexpr int kGThreads = 256;

// Shared-memory regions (bytes from a 1024-byte aligned base). Regions used
// in disjoint phases of a chunk share space.
constexpr int kA1 = 0;                  // [q; b*k]            128 rows x K=128
constexpr int kB1 = kA1 + 32768;        // k                    64 rows x K=128   (then akk^T fp32 [64][64])
constexpr int kA2 = kB1 + 16384;        // [E+; E+]            128 rows x K=128   (then W, v_new^T)
constexpr int kB2 = kA2 + 32768;        // E-                   64 rows x K=128   (then aqk, T)
constexpr int kA3 = kB2 + 16384;        // (b*k*exp G)^T       128 rows x K=64
constexpr int kA4 = kA3 + 16384;        // (w*v)^T             128 rows x K=64
constexpr int kA5 = kA4 + 16384;        // S^T (bf16)          128 rows x K=128
constexpr int kB7 = kA5 + 32768;        // q*exp(G)*scale       64 rows x K=128
constexpr int kB8 = kB7 + 16384;        // (k*exp(Glast-G))^T  128 rows x K=64
constexpr int kMisc = kB8 + 16384;      // gsum[128], glast[128] (fp32), mbarrier, TMEM slot
constexpr int kB5 = kA2;                // W                    64 rows x K=128
constexpr int kA6 = kA2 + 16384;        // v_new^T             128 rows x K=64
constexpr int kB6 = kB2;                // aqk                  64 rows x K=64
constexpr int kB3 = kB2 + 8192;         // T                    64 rows x K=64
constexpr int kAKK = kB1;               // akk^T fp32 [64][64]
constexpr int kGSmem = kMisc + 2048 + 1024;  // misc (1040 bytes used) + slack for the 1024-byte alignment

// TMEM columns
constexpr unsigned kTS = 0, kTD1 = 128, kTD2 = 192, kTDW = 256, kTDU = 320, kTDWS = 384, kTDOUT = 448;

// Byte offset of element (row, col) in a K-major, 128-byte-swizzled bf16
// operand of `rows` rows.
__device__ __forceinline__ int swz(int row, int col, int rows) {
    return (col >> 6) * rows * 128 + (row >> 3) * 1024 + (row & 7) * 128 + ((((col >> 3) & 7) ^ (row & 7)) << 4) +
           ((col & 7) << 1);
}

// Shared-memory matrix descriptor: 128-byte swizzled K-major layout, SBO 1024.
__device__ __forceinline__ uint64_t desc_sw128(unsigned addr) {
    return (uint64_t)((addr >> 4) & 0x3FFFu) | (1ull << 16) | ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) |
           (2ull << 61);
}

// kind::f16 instruction descriptor: fp32 accumulator, bf16 A and B, both K-major, M = 128, N = n.
__host__ __device__ constexpr uint32_t idesc_m128(int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

// D[128 x n] (+)= A[128 x kdim] B[n x kdim]^T, both operands K-major swizzled in shared memory.
__device__ __forceinline__ void mma_issue(unsigned d_tmem, unsigned a, unsigned b, int b_rows, int n, int kdim,
                                          bool accumulate) {
    const uint32_t id = idesc_m128(n);
    for (int j = 0; j < kdim / 16; ++j) {  // K = 16 per instruction: atom j/4, 32-byte step j%4
        const uint64_t ad = desc_sw128(a + (j >> 2) * 128 * 128 + (j & 3) * 32);
        const uint64_t bd = desc_sw128(b + (j >> 2) * b_rows * 128 + (j & 3) * 32);
        const unsigned acc = (accumulate || j > 0) ? 1u : 0u;
        asm volatile(
            "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
            " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
            "l"(ad), "l"(bd), "r"(id), "r"(acc)
            : "memory");
    }
}

__device__ __forceinline__ void tmem_ld32(unsigned taddr, float* v) {
    unsigned r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(unsigned taddr, const float* v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
        "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
        "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
        "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
        "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
        : "memory");
}

__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }
__device__ __forceinline__ void tc_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void tc_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }

// 8 consecutive bf16 of a K-major swizzled row (one 16-byte chunk): col % 8 == 0.
__device__ __forceinline__ void st8(char* base, int row, int col, int rows, const float* v) {
    uint4 u;
    __nv_bfloat162 p0 = __floats2bfloat162_rn(v[0], v[1]), p1 = __floats2bfloat162_rn(v[2], v[3]),
                   p2 = __floats2bfloat162_rn(v[4], v[5]), p3 = __floats2bfloat162_rn(v[6], v[7]);
    u.x = *reinterpret_cast<unsigned*>(&p0);
    u.y = *reinterpret_cast<unsigned*>(&p1);
    u.z = *reinterpret_cast<unsigned*>(&p2);
    u.w = *reinterpret_cast<unsigned*>(&p3);
    *reinterpret_cast<uint4*>(base + swz(row, col, rows)) = u;
}
__device__ __forceinline__ void st1(char* base, int row, int col, int rows, float v) {
    *reinterpret_cast<__nv_bfloat16*>(base + swz(row, col, rows)) = __float2bfloat16_rn(v);
}
__device__ __forceinline__ float ld1(const char* base, int row, int col, int rows) {
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(base + swz(row, col, rows)));
}
__device__ __forceinline__ void unpack8(uint4 u, float* f) {
    const unsigned w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

struct Gdn2Params {
    int64_t B, H, T;
    float scale;
    const __nv_bfloat16 *q, *k, *v, *b, *w;
    const float* g;
    const float* state_in;
    __nv_bfloat16* out;
    float* state_out;
    unsigned* status;
};

__global__ void __launch_bounds__(kGThreads, 1) gdn2_chunk_fwd_kernel(const Gdn2Params p) {
    extern __shared__ __align__(1024) char g_smem_raw[];
    char* sm = g_smem_raw + ((1024u - (smem_u32(g_smem_raw) & 1023u)) & 1023u);
    float* gsum = reinterpret_cast<float*>(sm + kMisc);
    float* glast = gsum + kGK;                       // exp(G[last]) per key channel
    uint64_t* bar = reinterpret_cast<uint64_t*>(glast + kGK);
    unsigned* tslot = reinterpret_cast<unsigned*>(bar + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, whalf = warp >> 2;  // TMEM lanes 32*quarter..; column half
    const int64_t bh = blockIdx.x;
    const int64_t T = p.T;
    const int nchunks = (int)((T + kGC - 1) / kGC);
    const unsigned sbase = smem_u32(sm);
    const unsigned mbar = smem_u32(bar);

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_u32(tslot)),
                     "r"(512)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    }
    if (tid == 0) {
        mbar_init(mbar, 1);
        mbar_fence_init();
    }
    tc_before();
    __syncthreads();
    tc_after();
    const unsigned tmem = *tslot;
    const unsigned tlane = (unsigned)(quarter * 32) << 16;  // this warp's TMEM lane quarter
    const int vrow = quarter * 32 + lane;                    // the TMEM lane (row) this thread reads

    // ---- the initial state: S^T into TMEM (lane v, column n) and its bf16 copy
    {
        const float* s0 = p.state_in ? p.state_in + bh * kGK * kGV : nullptr;
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

    unsigned phase = 0;
    float nf = 0.f;
    auto mma_wait = [&]() -> bool {  // every thread waits for the last commit; false if it never came
        const bool ok = mbar_wait_bounded(mbar, phase & 1u);
        phase++;
        if (!ok && tid == 0 && p.status) atomicOr(p.status, kStatusTimeout);
        return __syncthreads_and(ok) != 0;
    };
    auto commit = [&]() {
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(mbar)
                     : "memory");
    };

    bool ok = true;
    for (int ci = 0; ci < nchunks && ok; ++ci) {
        const int64_t t0 = (int64_t)ci * kGC;
        const int c = (int)min64(kGC, T - t0);  // live tokens; rows c..63 are zero (identity tokens)
        const int64_t row0 = bh * T + t0;      // first token row of the chunk in [B*H*T]

        // ---- 1a. q, k, b*k into the product operands; (w*v)^T
        for (int e = tid; e < kGC * (kGK / 8); e += kGThreads) {
            const int r = e >> 4, cc = (e & 15) * 8;
            float qv[8], kv[8], bv[8];
            if (r < c) {
                const int64_t off = (row0 + r) * kGK + cc;
                unpack8(*reinterpret_cast<const uint4*>(p.q + off), qv);
                unpack8(*reinterpret_cast<const uint4*>(p.k + off), kv);
                unpack8(*reinterpret_cast<const uint4*>(p.b + off), bv);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) qv[i] = kv[i] = bv[i] = 0.f;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) bv[i] *= kv[i];
            st8(sm + kA1, r, cc, 128, qv);
            st8(sm + kA1, 64 + r, cc, 128, bv);
            st8(sm + kB1, r, cc, 64, kv);
        }
        for (int e = tid; e < kGC * (kGV / 8); e += kGThreads) {
            const int r = e >> 4, cc = (e & 15) * 8;
            float vv[8], wv[8];
            if (r < c) {
                const int64_t off = (row0 + r) * kGV + cc;
                unpack8(*reinterpret_cast<const uint4*>(p.v + off), vv);
                unpack8(*reinterpret_cast<const uint4*>(p.w + off), wv);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) vv[i] = wv[i] = 0.f;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) st1(sm + kA4, cc + i, r, 128, vv[i] * wv[i]);  // (w*v)^T: row v, column j
        }
        // ---- 1b. the column threads: G = cumsum(g) over the chunk's tokens,
        // rows 32*half .. +31 of key channel kc
        const int kc = tid & (kGK - 1), half = tid >> 7;
        float G[32];
        {
            float acc = 0.f;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int r = half * 32 + i;
                const float gv = r < c ? p.g[(row0 + r) * kGK + kc] : 0.f;
                acc = __fadd_rn(acc, gv);
                G[i] = acc;
            }
            if (half == 0) gsum[kc] = acc;  // G at the middle token m = 31
        }
        __syncthreads();  // gsum; the q / k / b*k operands
        const float Gm = gsum[kc];
        if (half == 1) {
#pragma unroll
            for (int i = 0; i < 32; ++i) G[i] = __fadd_rn(G[i], Gm);
            glast[kc] = G[31];  // G at the last row (= the last live token: later rows add zeros)
        }
        __syncthreads();
        {
            const float Gl = glast[kc];
            const float em = expf(Gm), elm = expf(Gl - Gm);  // exp(G[m]), exp(G[last] - G[m])
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int r = half * 32 + i;
                const float ep = expf(G[i] - Gm);    // E+ = exp(G - G[m])
                const float en = expf(Gm - G[i]);    // E- = exp(G[m] - G)
                const float eg = ep * em;            // exp(G)
                st1(sm + kA2, r, kc, 128, ep);
                st1(sm + kA2, 64 + r, kc, 128, ep);
                st1(sm + kB2, r, kc, 64, en);
                st1(sm + kB7, r, kc, 64, ld1(sm + kA1, r, kc, 128) * eg * p.scale);   // q * exp(G) * scale
                st1(sm + kA3, kc, r, 128, ld1(sm + kA1, 64 + r, kc, 128) * eg);       // (b*k*exp G)^T
                st1(sm + kB8, kc, r, 128, ld1(sm + kB1, r, kc, 64) * (elm * en));     // (k*exp(Glast - G))^T
            }
        }
        __syncthreads();
        if (half == 0) glast[kc] = expf(glast[kc]);  // from here on: exp(G[last])
        fence_async_smem();
        tc_before();
        __syncthreads();

        // ---- 2. qk^T and (bk)k^T in one product; the decay (x K) in both lane halves
        if (tid == 0) {
            tc_after();
            mma_issue(tmem + kTD1, sbase + kA1, sbase + kB1, 64, 64, kGK, false);
            mma_issue(tmem + kTD2, sbase + kA2, sbase + kB2, 64, 64, kGK, false);
            commit();
        }
        if (!(ok = mma_wait())) break;
        tc_after();

        // ---- 3. aqk (rows 0-63) and akk^T (rows 64-127, fp32, transposed)
        {
            float d1[32], d2[32];
            const int j0 = whalf * 32;
            tmem_ld32(tmem + tlane + kTD1 + (unsigned)j0, d1);
            tmem_ld32(tmem + tlane + kTD2 + (unsigned)j0, d2);
            if (vrow < 64) {
                const int i = vrow;
                float a[32];
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) a[jj] = (j0 + jj <= i) ? d1[jj] * d2[jj] * (p.scale / kGK) : 0.f;
#pragma unroll
                for (int jj = 0; jj < 32; jj += 8) st8(sm + kB6, i, j0 + jj, 64, a + jj);
            } else {
                const int i = vrow - 64;
                float* akkT = reinterpret_cast<float*>(sm + kAKK);
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) akkT[(j0 + jj) * kGC + i] = (j0 + jj < i) ? d1[jj] * d2[jj] * (1.f / kGK) : 0.f;
            }
        }
        tc_before();
        __syncthreads();

        // ---- 4. T = (I + akk)^-1 by forward substitution: four threads per
        // column (column tid/4, rows 16*(tid%4) ..+15); at step i the owner of
        // x[i] passes it to the other three, which update their later rows
        {
            const float* akkT = reinterpret_cast<const float*>(sm + kAKK);
            const int col = tid >> 2, part = tid & 3, r0 = part * 16;
            float x[16];
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) x[rr] = (r0 + rr == col) ? 1.f : 0.f;
#pragma unroll
            for (int i = 0; i < kGC - 1; ++i) {
                const float xi = __shfl_sync(0xffffffffu, x[i & 15], (lane & ~3) | (i >> 4));
                if (r0 + 15 > i) {
                    const float4* row = reinterpret_cast<const float4*>(akkT + i * kGC + r0);  // akk[r0.., i]
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const float4 a4 = row[q4];
                        const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            if (r0 + 4 * q4 + e > i) x[4 * q4 + e] = __fmaf_rn(-av[e], xi, x[4 * q4 + e]);
                    }
                }
            }
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) st1(sm + kB3, r0 + rr, col, 64, x[rr]);  // T[r][col]
        }
        fence_async_smem();
        tc_before();
        __syncthreads();
        if (tid == 0) {
            tc_after();
            mma_issue(tmem + kTDW, sbase + kA3, sbase + kB3, 64, 64, kGC, false);  // W^T = rhs_k^T T^T
            mma_issue(tmem + kTDU, sbase + kA4, sbase + kB3, 64, 64, kGC, false);  // U^T = rhs_v^T T^T
            commit();
        }
        if (!(ok = mma_wait())) break;
        tc_after();
        {   // W (rows i, K = n) from W^T (lane n, column i)
            float wt[32];
            const int i0 = whalf * 32;
            tmem_ld32(tmem + tlane + kTDW + (unsigned)i0, wt);
#pragma unroll
            for (int ii = 0; ii < 32; ++ii) st1(sm + kB5, i0 + ii, vrow, 64, wt[ii]);
        }
        fence_async_smem();
        tc_before();
        __syncthreads();

        // ---- 5. (W S)^T = S^T W^T; v_new^T = U^T - (W S)^T
        if (tid == 0) {
            tc_after();
            mma_issue(tmem + kTDWS, sbase + kA5, sbase + kB5, 64, 64, kGK, false);
            commit();
        }
        if (!(ok = mma_wait())) break;
        tc_after();
        {
            float u[32], ws[32];
            const int i0 = whalf * 32;
            tmem_ld32(tmem + tlane + kTDU + (unsigned)i0, u);
            tmem_ld32(tmem + tlane + kTDWS + (unsigned)i0, ws);
#pragma unroll
            for (int ii = 0; ii < 32; ++ii) u[ii] -= ws[ii];
#pragma unroll
            for (int ii = 0; ii < 32; ii += 8) st8(sm + kA6, vrow, i0 + ii, 128, u + ii);
            // S^T columns n scaled by exp(G[last][n]) before the update is added
            for (int cc = 0; cc < 2; ++cc) {
                const int n0 = whalf * 64 + cc * 32;
                float s[32];
                tmem_ld32(tmem + tlane + kTS + (unsigned)n0, s);
#pragma unroll
                for (int nn = 0; nn < 32; ++nn) s[nn] *= glast[n0 + nn];
                tmem_st32(tmem + tlane + kTS + (unsigned)n0, s);
            }
            asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
        }
        fence_async_smem();
        tc_before();
        __syncthreads();

        // ---- 6. out^T = v_new^T aqk^T + S^T (q exp(G) scale)^T;  S^T += v_new^T (k exp(Glast - G))
        if (tid == 0) {
            tc_after();
            mma_issue(tmem + kTDOUT, sbase + kA6, sbase + kB6, 64, 64, kGC, false);
            mma_issue(tmem + kTDOUT, sbase + kA5, sbase + kB7, 64, 64, kGK, true);
            mma_issue(tmem + kTS, sbase + kA6, sbase + kB8, 128, 128, kGC, true);
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
                    p.out[(row0 + i0 + ii) * kGV + vrow] = __float2bfloat16_rn(o[ii]);
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

    if (ok && p.state_out) {
        float* so = p.state_out + bh * kGK * kGV;
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

bool misaligned16(const void* q) { return q && (reinterpret_cast<uintptr_t>(q) & 15u) != 0; }

}  // namespace
}  // namespace ssm

extern "C" int gdn2_chunk_fwd(const gdn2_fwd_args* a, void* stream) {
    ssm::reset_launches();
    if (!a) return SSM_ERR_INVALID_ARG;
    if (a->B < 0 || a->H < 0 || a->T < 0) return SSM_ERR_INVALID_ARG;
    if (a->K != ssm::kGK || a->V != ssm::kGV || (a->chunk != 0 && a->chunk != ssm::kGC)) return SSM_ERR_UNSUPPORTED;
    if (!(fabsf(a->scale) <= 3.0e38f)) return SSM_ERR_INVALID_ARG;  // NaN or infinite scale
    if (a->B * a->H > 0x7fffffff || a->B * a->H * a->T > (int64_t(1) << 40)) return SSM_ERR_INVALID_ARG;
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
    p.q = (const __nv_bfloat16*)a->q; p.k = (const __nv_bfloat16*)a->k; p.v = (const __nv_bfloat16*)a->v;
    p.b = (const __nv_bfloat16*)a->b; p.w = (const __nv_bfloat16*)a->w; p.g = a->g;
    p.state_in = a->state_in; p.out = (__nv_bfloat16*)a->out; p.state_out = a->state_out;
    p.status = (unsigned*)a->workspace;
    ssm::gdn2_chunk_fwd_kernel<<<(unsigned)BH, ssm::kGThreads, ssm::kGSmem, s>>>(p);
    return ssm::count_launches(cudaGetLastError() == cudaSuccess ? 1 : -1);
}
