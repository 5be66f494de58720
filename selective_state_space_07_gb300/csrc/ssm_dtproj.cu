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
// A tile is 128 tokens x TN = 256 channels (128 when R = 256). One CTA per SM
// walks the tiles with three roles: one lane of warp 0 loads a tile's a rows
// and w rows (bf16, K-major) with TMA -- per 64-wide atom of K one 2D box of
// [64 elements x 128 or TN rows] with 128-byte swizzle, which is the tensor
// core's 128-byte-swizzled K-major layout (8-row x 128-byte atoms, SBO 1024
// bytes); rows and columns past M, D or R are zero-filled by the copy -- and
// issues the R/16 `tcgen05.mma ...
// kind::f16` (M 128, N TN, K 16 each) into one of two TMEM accumulators;
// the epilogue warps meanwhile drain the other accumulator: each reads 32
// TMEM lanes (rows; 4 or 2 warps per lane quarter, interleaved 32-column chunks) with
// `tcgen05.ld`, transposes 32x32 blocks through shared memory so that each
// store instruction writes whole 128-byte row segments, and applies the
// epilogue. The op is bound by writing the fp32 [M, D] result (K = R is
// small: 2*R flops per 4 output bytes), so the design keeps the epilogue's
// stores going while the next tile is loaded and multiplied.
#include "ssm_common.cuh"
#include "ssm_internal.h"

namespace ssm {

namespace {

constexpr int kTM = 128;           // tokens per tile: MMA M, TMEM lanes
// Epilogue warps: 16 in the forward, 8 in the backward (its prefetched
// ddelta and dbias sums take 168 registers; 12 warps would cap it at 128 and
// spill). Warp w >= 1 reads TMEM lanes 32(w%4) .. +31 and every (EW/4)-th
// 32-column chunk starting at (w-1)/4.
template <bool BWD> __host__ __device__ constexpr int epi_warps() { return BWD ? 8 : 16; }
// + warp 0 (operand TMA, MMA issue) and, in the backward, a last warp that streams ddelta with TMA
template <bool BWD> __host__ __device__ constexpr int dp_threads() { return 32 * (1 + epi_warps<BWD>() + (BWD ? 1 : 0)); }
constexpr int kChunkBytes = kTM * 32 * 4;  // one ddelta chunk: 128 rows x 32 fp32 columns
constexpr int kStgRow = 36;        // floats per row of a warp's 32x32 transpose block (padded)
constexpr int kStgWarpBytes = 32 * kStgRow * 4;
constexpr int kMaxSmem = 227 * 1024;
// The shared-memory request is above half an SM's 228 KB: one CTA per SM,
// so the two accumulators (2*TN of the SM's 512 TMEM columns) are always free.
constexpr int kMinSmem = 116 * 1024;

// Tile geometry for TN channels per tile (MMA N), EW epilogue warps and RS
// ddelta ring slots (backward). Shared memory: operands (A then B) | ddelta
// ring | transpose blocks | mbarriers + the TMEM address.
template <int TN, int EW, int RS> struct DpGeom {
    static_assert(TN == 128 || TN == 256, "N of the MMA");
    // kind::f16 instruction descriptor: fp32 accumulator, bf16 A and B, both K-major, N = TN, M = kTM
    static constexpr uint32_t idesc =
        (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(TN >> 3) << 17) | ((uint32_t)(kTM >> 4) << 24);
    // K in atoms of 64 bf16 (one 128-byte swizzled row per token or channel)
    __host__ __device__ static constexpr int atoms(int64_t R) { return (int)((R + 63) / 64); }
    __host__ __device__ static constexpr int operand_bytes(int64_t R) { return atoms(R) * (kTM + TN) * 128; }
    static constexpr int stg_bytes = EW * kStgWarpBytes;
    static constexpr int ring_bytes = RS * kChunkBytes;
    static constexpr int nbars = 5 + 2 * RS;  // op_full, tmem_full[2], tmem_empty[2], ring full[RS], ring empty[RS]
    // + 1 KB: the operand atoms start on a 1024-byte boundary (the swizzle's period)
    __host__ __device__ static constexpr int need(int64_t R) {
        return operand_bytes(R) + ring_bytes + stg_bytes + 8 * nbars + 16 + 1024;
    }
    __host__ __device__ static constexpr int smem(int64_t R) { return need(R) > kMinSmem ? need(R) : kMinSmem; }
    __host__ __device__ static constexpr bool fits(int64_t R) { return need(R) <= kMaxSmem; }
};
static_assert(kStgWarpBytes % 128 == 0 && (kTM + 128) * 16 * 2 % 128 == 0, "aligned mbarriers after the operands");

struct DtProjParams {
    int64_t M, D, R;
    int64_t tiles_m, tiles_n;
    const __nv_bfloat16* a;        // [M, R] (rows strided; read through the tensor map)
    const __nv_bfloat16* w;        // [D, R]
    const float* bias;             // [D] or null
    float* out;                    // forward: delta [M,D]; backward: dpre [M,D]
    const float* dout;             // backward: ddelta [M,D] (may alias out)
    float* dbias;                  // backward: [D] (zeroed on the stream first) or null
    int softplus;
    unsigned* status;
};


// Shared-memory matrix descriptor of a K-major operand in the 128-byte
// swizzled canonical layout: atoms of 8 rows x 128 bytes (64 bf16 of K), the
// 16-byte chunks of row r XOR-permuted by r % 8 -- what a TMA copy with
// 128-byte swizzle writes. SBO = 1024 bytes between 8-row groups; LBO is not
// used by this layout (encoded 1); version 1; layout type 2 (128-byte swizzle).
// A K step of 16 elements inside an atom advances the start by 32 bytes.
__device__ __forceinline__ uint64_t smem_desc_sw128(unsigned addr) {
    return (uint64_t)((addr >> 4) & 0x3FFFu) | (1ull << 16) | ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) |
           (2ull << 61);
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

// Persistent, warp-specialised: one CTA per SM walks tiles t = blockIdx.x,
// blockIdx.x + gridDim.x, ... Warp 0 (one lane) loads a tile's operands with
// TMA and issues its MMAs into one of two TMEM accumulators; warps 1..EW run
// the epilogue of the previous tile from the other accumulator meanwhile.
// mbarriers: op_full (the operands landed; TMA transaction count),
// tmem_full[b] (the MMAs into accumulator b completed: its operands may be
// overwritten and its epilogue may start), tmem_empty[b] (the EW epilogue
// warps finished reading accumulator b). Every wait is bounded by the global
// timer; a wait that runs out sets the timeout status and ends that role's
// loop (the others run out the same way), and the TMEM is freed at the end.
template <int TN, bool BWD, int RS>
__global__ void __launch_bounds__(dp_threads<BWD>(), 1)
    ssm_dtproj_kernel(const DtProjParams p, const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmG) {
    extern __shared__ __align__(1024) char dp_smem_raw[];
    // the swizzled atoms need 1024-byte alignment; the request has 1 KB of slack for it
    char* dp_smem = dp_smem_raw + ((1024u - (smem_u32(dp_smem_raw) & 1023u)) & 1023u);
    constexpr int EW = epi_warps<BWD>();
    using G = DpGeom<TN, EW, RS>;
    const int64_t R = p.R;
    char* sA = dp_smem;
    char* sB = dp_smem + G::atoms(R) * kTM * 128;
    char* ring = dp_smem + G::operand_bytes(R);  // ddelta chunks, row-major [128][32] fp32 each
    float* stg = reinterpret_cast<float*>(ring + G::ring_bytes);
    uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<char*>(stg) + G::stg_bytes);
    const unsigned op_full = smem_u32(bars), tfull0 = smem_u32(bars + 1), tempty0 = smem_u32(bars + 3);
    const unsigned rfull0 = smem_u32(bars + 5), rempty0 = smem_u32(bars + 5 + RS);
    unsigned* tslot = reinterpret_cast<unsigned*>(bars + G::nbars);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t tiles = p.tiles_m * p.tiles_n;

    if (warp == 0) {  // two accumulators: 2*TN TMEM columns x 128 lanes of fp32
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_u32(tslot)),
                     "r"(2 * TN)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    }
    if (threadIdx.x == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(op_full) : "memory");
        for (int b = 0; b < 2; ++b) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(tfull0 + 8 * b) : "memory");
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(tempty0 + 8 * b), "r"(EW)
                         : "memory");
        }
        for (int b = 0; b < RS; ++b) {  // a ddelta chunk is read by one epilogue warp per TMEM lane quarter
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(rfull0 + 8 * b) : "memory");
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 4;\n" ::"r"(rempty0 + 8 * b) : "memory");
        }
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
    const unsigned tmem = *tslot;
    float nf = 0.f;

    if (warp == 0) {
        if (lane == 0) {
            const unsigned a0 = smem_u32(sA), b0 = smem_u32(sB);
            int64_t it = 0;
            for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x, ++it) {
                const int64_t m0 = (t / p.tiles_n) * kTM, n0 = (t % p.tiles_n) * TN;
                const int buf = (int)(it & 1);
                // the operand buffer is free once the previous tile's MMAs completed
                if (it > 0 && !mbar_wait_bounded(tfull0 + 8 * ((it - 1) & 1), (unsigned)(((it - 1) >> 1) & 1))) {
                    if (p.status) atomicOr(p.status, kStatusTimeout);
                    break;
                }
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(op_full),
                             "r"((unsigned)G::operand_bytes(R))
                             : "memory");
                for (int at = 0; at < G::atoms(R); ++at) {  // one box per 64-wide atom of K (x = 64*at)
                    tma_load_2d(sA + at * kTM * 128, &tmA, at * 64, (int)m0, op_full);
                    tma_load_2d(sB + at * TN * 128, &tmB, at * 64, (int)n0, op_full);
                }
                if (!mbar_wait_bounded(op_full, (unsigned)(it & 1))) {
                    if (p.status) atomicOr(p.status, kStatusTimeout);
                    break;
                }
                // the accumulator is free once the epilogue of tile it-2 read it
                if (it >= 2 && !mbar_wait_bounded(tempty0 + 8 * buf, (unsigned)(((it >> 1) - 1) & 1))) {
                    if (p.status) atomicOr(p.status, kStatusTimeout);
                    break;
                }
                asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
                const unsigned d_tmem = tmem + (unsigned)(buf * TN);
                for (int j = 0; j < (int)(R / 16); ++j) {  // K = 16 per instruction: atom j/4, 32-byte step j%4
                    const uint64_t ad = smem_desc_sw128(a0 + (j >> 2) * kTM * 128 + (j & 3) * 32);
                    const uint64_t bd = smem_desc_sw128(b0 + (j >> 2) * TN * 128 + (j & 3) * 32);
                    const unsigned acc = j > 0;
                    asm volatile(
                        "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
                        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
                        "l"(ad), "l"(bd), "r"(G::idesc), "r"(acc)
                        : "memory");
                }
                asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
                                 tfull0 + 8 * buf)
                             : "memory");
            }
        }
        __syncwarp();
    } else if (BWD && warp == EW + 1) {
        // ddelta producer: the chunks of every tile in order, through the RS-slot ring
        if (lane == 0) {
            int64_t q = 0;
            bool ok = true;
            for (int64_t t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
                const int64_t m0 = (t / p.tiles_n) * kTM, n0 = (t % p.tiles_n) * TN;
                for (int c = 0; c < TN / 32 && n0 + c * 32 < p.D; ++c, ++q) {
                    const int slot = (int)(q % RS);
                    const int64_t k = q / RS;
                    if (k > 0 && !mbar_wait_bounded(rempty0 + 8 * slot, (unsigned)((k - 1) & 1))) {
                        if (p.status) atomicOr(p.status, kStatusTimeout);
                        ok = false;
                        break;
                    }
                    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(rfull0 + 8 * slot),
                                 "r"((unsigned)kChunkBytes)
                                 : "memory");
                    // x = a column multiple of 32 (128 bytes); rows past M read as zero
                    tma_load_2d(ring + slot * kChunkBytes, &tmG, (int)(n0 + c * 32), (int)m0, rfull0 + 8 * slot);
                }
            }
        }
        __syncwarp();
    } else {
        constexpr int step = EW / 4;  // warps per TMEM lane quarter
        const int ew = warp - 1, quarter = warp & 3, first = ew >> 2;  // TMEM lanes 32*quarter.., chunks first, first+step, ..
        float* blk = stg + ew * 32 * kStgRow;
        const int rsub = lane >> 3, cq = (lane & 7) * 4;  // coalesced phase: 4 rows x 8 float4 per instruction
        int64_t it = 0, qbase = 0;  // qbase: ddelta chunks of the earlier tiles (the producer's count)
        bool ok = true;
        for (int64_t t = blockIdx.x; t < tiles && ok; t += gridDim.x, ++it) {
            const int64_t m0 = (t / p.tiles_n) * kTM, n0 = (t % p.tiles_n) * TN;
            const int buf = (int)(it & 1);
            const int64_t mrow = m0 + quarter * 32;
            const int nch = (int)min64(TN / 32, (p.D - n0 + 31) / 32);
            if (!mbar_wait_bounded(tfull0 + 8 * buf, (unsigned)((it >> 1) & 1))) {
                if (lane == 0 && p.status) atomicOr(p.status, kStatusTimeout);
                break;
            }
            asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
            for (int c = first; c < nch; c += step) {
                // backward: this chunk's ddelta, 128 rows x 32 columns, in ring slot q % RS
                const int64_t q = qbase + c;
                const float* gch = reinterpret_cast<const float*>(ring + (int)(q % (RS > 0 ? RS : 1)) * kChunkBytes);
                if (BWD && !mbar_wait_bounded(rfull0 + 8 * (int)(q % (RS > 0 ? RS : 1)),
                                              (unsigned)((q / (RS > 0 ? RS : 1)) & 1))) {
                    if (lane == 0 && p.status) atomicOr(p.status, kStatusTimeout);
                    ok = false;
                    break;
                }
                unsigned v[32];
                asm volatile(
                    "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                    "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
                    : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
                      "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
                      "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]),
                      "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]),
                      "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
                    : "r"(tmem + ((unsigned)(quarter * 32) << 16) + (unsigned)(buf * TN + c * 32)));
                asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
                // lane = row: the row's 32 accumulators into the transpose block
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
                            const float4 g = *reinterpret_cast<const float4*>(gch + (quarter * 32 + r) * 32 + cq);
                            o = p.softplus ? dsoftplus4(g, pre) : g;
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
                    if (lane < 8 && cv && p.dbias) red_add_v4(p.dbias + col, db);
                }
                __syncwarp();  // the block is rewritten by the next chunk; the ring slot is read
                if (BWD && lane == 0)
                    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(rempty0 + 8 * (int)(q % (RS > 0 ? RS : 1)))
                                 : "memory");
            }
            qbase += nch;
            asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
            __syncwarp();
            if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(tempty0 + 8 * buf) : "memory");
        }
    }
    flag_nonfinite(p.status, nf);
    asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
    __syncthreads();
    if (warp == 0) {
        asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(2 * TN) : "memory");
    }
}

}  // namespace

int dtproj_smem_bytes(int64_t R) {
    return DpGeom<256, 16, 0>::fits(R) ? DpGeom<256, 16, 0>::smem(R) : DpGeom<128, 16, 0>::smem(R);
}

namespace {
// a bf16 operand [rows, R]: boxes of one 64-wide K atom (128 bytes, 128-byte swizzle) x box_rows
bool encode_operand(CUtensorMap* map, const void* base, int64_t R, int64_t rows, int64_t stride, int box_rows) {
    return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, R, rows, stride * 2, 64, box_rows,
                     CU_TENSOR_MAP_SWIZZLE_128B);
}

template <int TN, bool BWD, int RS> int launch_dtproj_t(const DtProjParams& p0, int64_t a_stride, cudaStream_t s) {
    DtProjParams p = p0;
    p.tiles_m = (p.M + kTM - 1) / kTM;
    p.tiles_n = (p.D + TN - 1) / TN;
    const int64_t tiles = p.tiles_m * p.tiles_n;
    const int smem = DpGeom<TN, epi_warps<BWD>(), RS>::smem(p.R);
    CUtensorMap ta, tb, tg;
    if (!encode_operand(&ta, p.a, p.R, p.M, a_stride, kTM) || !encode_operand(&tb, p.w, p.R, p.D, p.R, TN))
        return -1;
    if (BWD) {  // ddelta [M, D] fp32 in chunks of 32 columns (128 bytes) x 128 rows
        if (!encode_2d(&tg, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, p.dout, p.D, p.M, p.D * 4, 32, kTM,
                       CU_TENSOR_MAP_SWIZZLE_NONE))
            return -1;
    } else {
        tg = ta;  // not read by the forward
    }
    const unsigned grid = (unsigned)min64(tiles, (int64_t)sm_count());  // persistent: one CTA per SM
    // the limit is set once per device, so it is set to the largest request
    static unsigned long long mask = 0;
    if (!ensure_smem(ssm_dtproj_kernel<TN, BWD, RS>, kMaxSmem, mask)) return -1;
    ssm_dtproj_kernel<TN, BWD, RS><<<grid, dp_threads<BWD>(), smem, s>>>(p, ta, tb, tg);
    return cudaGetLastError() == cudaSuccess ? 1 : -1;
}

int launch_dtproj_fwd(const DtProjParams& p, int64_t a_stride, cudaStream_t s) {
    // 256-channel tiles while their operands fit next to the transpose blocks, else 128
    return DpGeom<256, epi_warps<false>(), 0>::fits(p.R) ? launch_dtproj_t<256, false, 0>(p, a_stride, s)
                                                         : launch_dtproj_t<128, false, 0>(p, a_stride, s);
}
int launch_dtproj_bwd(const DtProjParams& p, int64_t a_stride, cudaStream_t s) {
    // the widest tile, then the deepest ddelta ring, that fit
    constexpr int EW = epi_warps<true>();
    if (DpGeom<256, EW, 4>::fits(p.R)) return launch_dtproj_t<256, true, 4>(p, a_stride, s);
    if (DpGeom<128, EW, 4>::fits(p.R)) return launch_dtproj_t<128, true, 4>(p, a_stride, s);
    return launch_dtproj_t<128, true, 2>(p, a_stride, s);
}

}  // namespace

int launch_dtproj(bool bwd, int64_t M, int64_t D, int64_t R, int64_t a_stride, const void* a, const void* w,
                  const float* bias, float* out, const float* dout, float* dbias, int softplus, unsigned* status,
                  cudaStream_t s) {
    if (M == 0 || D == 0) return 0;
    DtProjParams p{};
    p.M = M; p.D = D; p.R = R;
    p.a = reinterpret_cast<const __nv_bfloat16*>(a);
    p.w = reinterpret_cast<const __nv_bfloat16*>(w);
    p.bias = bias; p.out = out; p.dout = dout; p.dbias = dbias; p.softplus = softplus; p.status = status;
    return bwd ? launch_dtproj_bwd(p, a_stride, s) : launch_dtproj_fwd(p, a_stride, s);
}

}  // namespace ssm
