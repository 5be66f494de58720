// The dt projection in front of the S6 scan with the softplus fused into the
// GEMM's epilogue, on the sm_103a tensor cores (tcgen05, TMEM accumulators).
//
// rustytorch commit log, "MambaBlock" S6 forward commit:
// "delta=softplus(dt.dt_proj+dt_bias)", where dt is the first dt_rank
// columns of the x_proj output. With a = those columns [M = B*L, R] (rows
// read in place from the x_proj buffer), w the projection weight [D, R]:
//   forward:  delta[m,d] = softplus(bias[d] + sum_r a[m,r] w[d,r])
//   backward: dpre[m,d]  = ddelta[m,d] * sigmoid(pre[m,d]),  dbias[d] = sum_m dpre[m,d]
// (the pre-activation is recomputed; the two weight/input gradients that
// follow are plain GEMMs of dpre and are left to the caller's BLAS).
//
// One CTA computes a 128-token x 256-channel tile. One thread loads the a
// rows and w rows (bf16, K-major) with TMA: per 16-byte column of K one 2D
// box of [8 elements x 128 (or 256) rows], which lands as a stack of the
// tensor core's no-swizzle core matrices (8 rows x 16 bytes): SBO = 128 bytes
// between 8-row groups, LBO = rows*16 bytes between core matrices along K;
// rows past M or D are zero-filled by the copy. The same thread issues the R/16 `tcgen05.mma ...
// kind::f16` (M = 128, N = 256, K = 16 each) into a 256-column TMEM
// accumulator and commits them to an mbarrier; every warp then reads 32
// TMEM lanes (rows; two warps per lane quarter, alternate 32-column chunks)
// with `tcgen05.ld`, transposes 32x32 blocks through
// shared memory so that each store instruction writes whole 128-byte row
// segments, and applies the epilogue. The op is bound by writing the fp32
// [M, D] result (K = R is small: 2*R flops per 4 output bytes), so the
// epilogue's stores are what the design serves.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "ssm_common.cuh"
#include "ssm_internal.h"

namespace ssm {

namespace {

constexpr int kTM = 128;           // tokens per tile: MMA M, TMEM lanes
constexpr int kTN = 256;           // channels per tile: MMA N, TMEM columns
constexpr int kDPThreads = 256;    // warp w reads TMEM lanes 32(w%4) .. +31 and every (warps/4)-th 32-column chunk
constexpr int kDPMinBlocks = 2;    // CTAs per SM (each holds kTN of the SM's 512 TMEM columns)
constexpr int kDPWarps = kDPThreads / 32;
constexpr int kChunkStep = kDPWarps / 4;
static_assert(kDPWarps % 4 == 0 && kDPMinBlocks * kTN <= 512, "lane quarters; TMEM columns");
constexpr int kStgRow = 36;        // floats per row of a warp's 32x32 transpose block (padded)
constexpr int kStgBytes = kDPWarps * 32 * kStgRow * 4;
constexpr unsigned long long kWaitNs = 1000000000ull;  // 1 s: how long a thread waits for the MMAs

struct DtProjParams {
    int64_t M, D, R, a_stride;     // a rows are a_stride elements apart
    int64_t tiles_n;               // tiles across D
    const __nv_bfloat16* a;        // [M, R] (rows strided)
    const __nv_bfloat16* w;        // [D, R]
    const float* bias;             // [D] or null
    float* out;                    // forward: delta [M,D]; backward: dpre [M,D]
    const float* dout;             // backward: ddelta [M,D] (may alias out)
    float* dbias;                  // backward: [D] (zeroed on the stream first) or null
    int softplus;
    unsigned* status;
};

// Every CTA holds kTN TMEM columns, so the shared memory request is large
// enough that no more than 512 / kTN CTAs fit on an SM (228 KB each), and
// tcgen05.alloc never has to wait for columns.
constexpr int kMinOperandSmem = ((228 * 1024) / (512 / kTN + 1) + 1024 + 127) / 128 * 128;
__host__ __device__ constexpr int operand_bytes(int64_t R) { return (int)((kTM + kTN) * R * 2); }
__host__ __device__ constexpr int dtproj_smem(int64_t R) {
    return (operand_bytes(R) > kMinOperandSmem ? operand_bytes(R) : kMinOperandSmem) + kTN * 4 + 32;
}
static_assert(kMinOperandSmem >= kStgBytes, "the transpose blocks fit in the operand region");
// the dbias sums, the two mbarriers and the TMEM slot follow the operand
// region, which must end on a 16-byte boundary for them to be aligned
static_assert(kMinOperandSmem % 128 == 0 && operand_bytes(16) % 128 == 0, "aligned tail of shared memory");

__device__ __forceinline__ unsigned smem_u32(const void* p) { return (unsigned)__cvta_generic_to_shared(p); }

// Shared-memory matrix descriptor: no swizzle, K-major canonical layout
// (start, LBO = core-matrix step along K, SBO = 8-row-group step), version 1.
__device__ __forceinline__ uint64_t smem_desc(unsigned addr, unsigned lbo, unsigned sbo) {
    return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}

// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, N = kTN, M = kTM.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kTN >> 3) << 17) |
                            ((uint32_t)(kTM >> 4) << 24);

__device__ __forceinline__ bool mbar_test(unsigned bar, unsigned parity) {
    unsigned ok = 0;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
    return t;
}
// Wait (non-blocking polls with a short sleep) until phase `parity` of the
// barrier completes or kWaitNs have passed; returns whether it completed.
__device__ __forceinline__ bool mbar_wait_bounded(unsigned bar, unsigned parity) {
    const unsigned long long t0 = global_ns();
    while (!mbar_test(bar, parity)) {
        if (global_ns() - t0 > kWaitNs) return false;
        __nanosleep(64);
    }
    return true;
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, unsigned bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// The bf16-operand path uses the scan's MUFU forms of softplus and sigmoid
// (the ones its bf16 path applies to dt + dt_bias).
__device__ __forceinline__ float4 softplus4(float4 v) {
    return make_float4(softplus<true>(v.x), softplus<true>(v.y), softplus<true>(v.z), softplus<true>(v.w));
}
__device__ __forceinline__ float4 dsoftplus4(float4 g, float4 v) {
    return make_float4(g.x * sigmoid<true>(v.x), g.y * sigmoid<true>(v.y), g.z * sigmoid<true>(v.z),
                       g.w * sigmoid<true>(v.w));
}

template <bool BWD>
__global__ void __launch_bounds__(kDPThreads, kDPMinBlocks)
    ssm_dtproj_kernel(const DtProjParams p, const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmB) {
    extern __shared__ __align__(128) char dp_smem[];
    const int64_t R = p.R;
    char* sA = dp_smem;
    char* sB = dp_smem + (int64_t)kTM * R * 2;
    float* stg = reinterpret_cast<float*>(dp_smem);  // reused after the MMAs have read the operands
    float* sDB = reinterpret_cast<float*>(dp_smem + (dtproj_smem(R) - kTN * 4 - 32));
    uint64_t* barT = reinterpret_cast<uint64_t*>(dp_smem + (dtproj_smem(R) - 32));  // operands landed
    uint64_t* bar = reinterpret_cast<uint64_t*>(dp_smem + (dtproj_smem(R) - 24));   // MMAs done
    unsigned* tslot = reinterpret_cast<unsigned*>(dp_smem + (dtproj_smem(R) - 16));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t tm = blockIdx.x / p.tiles_n, tn = blockIdx.x % p.tiles_n;
    const int64_t m0 = tm * kTM, n0 = tn * kTN;

    if (warp == 0) {  // the accumulator: 256 TMEM columns x 128 lanes of fp32
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_u32(tslot)),
                     "r"(kTN)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    }
    if (threadIdx.x == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(smem_u32(barT)) : "memory");
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(smem_u32(bar)) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    if (BWD)
        for (int i = threadIdx.x; i < kTN; i += kDPThreads) sDB[i] = 0.f;
    asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
    const unsigned tmem = *tslot;

    if (threadIdx.x == 0) {  // the operands: one box per 16-byte column of K, x = 8*kc (16-byte aligned)
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(barT)),
                     "r"((unsigned)operand_bytes(R))
                     : "memory");
        for (int kc = 0; kc < (int)(R / 8); ++kc) {
            tma_load_2d(sA + kc * kTM * 16, &tmA, kc * 8, (int)m0, smem_u32(barT));
            tma_load_2d(sB + kc * kTN * 16, &tmB, kc * 8, (int)n0, smem_u32(barT));
        }
    }
    bool landed = mbar_wait_bounded(smem_u32(barT), 0);
    if (!landed) {
        if (threadIdx.x == 0 && p.status) atomicOr(p.status, kStatusTimeout);
        landed = mbar_wait_bounded(smem_u32(barT), 0);
    }

    if (threadIdx.x == 0 && landed) {
        const unsigned a0 = smem_u32(sA), b0 = smem_u32(sB);
        for (int j = 0; j < (int)(R / 16); ++j) {  // K = 16 per instruction: two core matrices along K
            const uint64_t ad = smem_desc(a0 + j * 2 * kTM * 16, kTM * 16, 128);
            const uint64_t bd = smem_desc(b0 + j * 2 * kTN * 16, kTN * 16, 128);
            const unsigned acc = j > 0;
            asm volatile(
                "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
                " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem),
                "l"(ad), "l"(bd), "r"(kIdesc), "r"(acc)
                : "memory");
        }
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
                         smem_u32(bar))
                     : "memory");
    }
    // every thread waits for the accumulator (bounded: a stuck MMA becomes an error status)
    bool ready = landed && mbar_wait_bounded(smem_u32(bar), 0);
    if (landed && !ready) {
        // report, give the tensor core one more bounded wait before the TMEM is freed, write nothing
        if (threadIdx.x == 0 && p.status) atomicOr(p.status, kStatusTimeout);
        mbar_wait_bounded(smem_u32(bar), 0);
    }
    asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");

    float nf = 0.f;
    if (ready) {
        const int quarter = warp & 3, half = warp >> 2;  // TMEM lanes 32*quarter.., chunks c = half + k*kChunkStep
        float* blk = stg + warp * 32 * kStgRow;
        const int rsub = lane >> 3, cq = (lane & 7) * 4;  // coalesced phase: 4 rows x 8 float4 per instruction
        const int64_t mrow = m0 + quarter * 32;
        // backward: the chunk's ddelta values are loaded one chunk ahead, before
        // any store of this thread (dpre may be ddelta: each element is read and
        // then written by the same thread)
        float4 gcur[8], gnext[8];
        auto load_g = [&](int c, float4 (&g)[8]) {
            const int64_t col = n0 + c * 32 + cq;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int64_t m = mrow + 4 * i + rsub;
                g[i] = (c < kTN / 32 && m < p.M && col < p.D)
                           ? *reinterpret_cast<const float4*>(p.dout + m * p.D + col)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        };
        if (BWD) load_g(half, gnext);
        for (int c = half; c < kTN / 32; c += kChunkStep) {
            if (n0 + c * 32 >= p.D) break;  // uniform across the warp
            if (BWD) {
#pragma unroll
                for (int i = 0; i < 8; ++i) gcur[i] = gnext[i];
                load_g(c + kChunkStep, gnext);
            }
            unsigned v[32];
            asm volatile(
                "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
                : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
                  "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]),
                  "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]),
                  "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]),
                  "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
                : "r"(tmem + ((unsigned)(quarter * 32) << 16) + (unsigned)(c * 32)));
            asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
            // lane = row: write the row's 32 accumulators into the transpose block
#pragma unroll
            for (int q = 0; q < 8; ++q)
                *reinterpret_cast<float4*>(blk + lane * kStgRow + 4 * q) =
                    make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
            __syncwarp();
            const int64_t col = n0 + c * 32 + cq;
            const bool cv = col < p.D;
            const float4 b4 = (p.bias && cv) ? __ldg(reinterpret_cast<const float4*>(p.bias + col))
                                             : make_float4(0.f, 0.f, 0.f, 0.f);
            float4 db = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int r = 4 * i + rsub;
                const int64_t m = mrow + r;
                const float4 acc = *reinterpret_cast<const float4*>(blk + r * kStgRow + cq);
                if (m < p.M && cv) {
                    const float4 pre = make_float4(acc.x + b4.x, acc.y + b4.y, acc.z + b4.z, acc.w + b4.w);
                    float4 o;
                    if (!BWD) {
                        o = p.softplus ? softplus4(pre) : pre;
                    } else {
                        o = p.softplus ? dsoftplus4(gcur[i], pre) : gcur[i];
                        db.x += o.x; db.y += o.y; db.z += o.z; db.w += o.w;
                    }
                    *reinterpret_cast<float4*>(p.out + m * p.D + col) = o;
                    nf = __fmaf_rn(o.x + o.y + o.z + o.w, 0.0f, nf);
                }
            }
            if (BWD) {  // the 4 lanes holding these 4 columns (lane % 8 equal) sum their rows
#pragma unroll
                for (int s = 8; s < 32; s <<= 1) {
                    db.x += __shfl_xor_sync(0xffffffffu, db.x, s);
                    db.y += __shfl_xor_sync(0xffffffffu, db.y, s);
                    db.z += __shfl_xor_sync(0xffffffffu, db.z, s);
                    db.w += __shfl_xor_sync(0xffffffffu, db.w, s);
                }
                if (lane < 8) {
                    float* d = sDB + c * 32 + cq;
                    atomicAdd(d, db.x); atomicAdd(d + 1, db.y); atomicAdd(d + 2, db.z); atomicAdd(d + 3, db.w);
                }
            }
            __syncwarp();  // the block is rewritten by the next chunk
        }
    }
    flag_nonfinite(p.status, nf);
    asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
    __syncthreads();
    if (BWD && ready && p.dbias)
        for (int i = threadIdx.x; i < kTN; i += kDPThreads)
            if (n0 + i < p.D) atomicAdd(p.dbias + n0 + i, sDB[i]);
    if (warp == 0) {
        asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(kTN) : "memory");
    }
}

}  // namespace

int dtproj_smem_bytes(int64_t R) { return dtproj_smem(R); }

namespace {
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            f = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }();
    return fn;
}

// A [rows, R] bf16 matrix with rows `stride` elements apart, copied in boxes
// of 8 elements (16 bytes) x box_rows rows; rows past the end read as zero.
bool encode_rows(CUtensorMap* map, const void* base, int64_t R, int64_t rows, int64_t stride, int box_rows) {
    const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)R, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)(stride * 2)};
    const cuuint32_t box[2] = {8, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

int launch_dtproj(bool bwd, int64_t M, int64_t D, int64_t R, int64_t a_stride, const void* a, const void* w,
                  const float* bias, float* out, const float* dout, float* dbias, int softplus, unsigned* status,
                  cudaStream_t s) {
    if (M == 0 || D == 0) return 0;
    DtProjParams p{};
    p.M = M; p.D = D; p.R = R; p.a_stride = a_stride;
    p.tiles_n = (D + kTN - 1) / kTN;
    p.a = reinterpret_cast<const __nv_bfloat16*>(a);
    p.w = reinterpret_cast<const __nv_bfloat16*>(w);
    p.bias = bias; p.out = out; p.dout = dout; p.dbias = dbias; p.softplus = softplus; p.status = status;
    const int64_t tiles = ((M + kTM - 1) / kTM) * p.tiles_n;
    const int smem = dtproj_smem(R);
    CUtensorMap ta, tb;
    if (!encode_rows(&ta, a, R, M, a_stride, kTM) || !encode_rows(&tb, w, R, D, R, kTN)) return -1;
    // the limit is set once per device, so it is set for the largest R (256)
    static unsigned long long mask_f = 0, mask_b = 0;
    if (bwd) {
        if (!ensure_smem(ssm_dtproj_kernel<true>, dtproj_smem(256), mask_b)) return -1;
        ssm_dtproj_kernel<true><<<(unsigned)tiles, kDPThreads, smem, s>>>(p, ta, tb);
    } else {
        if (!ensure_smem(ssm_dtproj_kernel<false>, dtproj_smem(256), mask_f)) return -1;
        ssm_dtproj_kernel<false><<<(unsigned)tiles, kDPThreads, smem, s>>>(p, ta, tb);
    }
    return cudaGetLastError() == cudaSuccess ? 1 : -1;
}

}  // namespace ssm
