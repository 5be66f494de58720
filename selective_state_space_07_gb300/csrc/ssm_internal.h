// Internal declarations shared by the translation units of libssmscan.so:
// kernel parameter blocks and the launchers ssm_api.cu calls.
#pragma once
#include <cuda.h>  // CUtensorMap (built through the runtime's driver entry point; no libcuda link)
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/ssm_scan.h"

namespace ssm {

constexpr unsigned kStatusNonFinite = 1u;  // workspace status bit: an output was Inf/NaN
constexpr unsigned kStatusTimeout = 2u;    // workspace status bit: a bounded wait inside a kernel ran out
constexpr int kFwdThreads = 128;  // ssm_step_kernel
#ifndef SSM_FWD_LPC
#define SSM_FWD_LPC 2
#endif
constexpr int kFwdLPC = SSM_FWD_LPC;  // forward: lanes sharing one channel (16/kFwdLPC states each)
#ifndef SSM_READ_BLOCK
#define SSM_READ_BLOCK 8
#endif
// Readout order shared by the forward and ssm_step: sequential fused
// multiply-add chains over blocks of kReadBlock consecutive states, the
// blocks summed as a balanced binary tree in state order.
constexpr int kReadBlock = SSM_READ_BLOCK;
#ifndef SSM_FWD_WARPS
#define SSM_FWD_WARPS 4
#endif
constexpr int kFwdCtaThreads = 32 * SSM_FWD_WARPS;  // threads of a forward / aggregate CTA
constexpr int kBwdThreads = 128;
constexpr int kConvThreads = 128;

struct FwdParams {
    int64_t B, L, D;
    int G;          // number of L-segments ("groups") scanned in parallel
    int64_t Lg;     // tokens per group, a multiple of 16
    int has_z, sp;  // gate present; Delta = softplus(dt + dt_bias)
    const void *x, *z, *Bm, *Cm;
    int64_t bcs;    // elements between consecutive tokens' Bm (and Cm) rows
    const float *dt, *dt_bias, *A, *Dskip;
    const float* hstart;  // G == 1: h0 [B,D,16] (nullable); G > 1: carries [B,G,D,16]
    void* y;
    float *h_last, *ckpt;
    float *aggH, *aggS;   // chunk aggregates [B,G,D,16] and [B,G,D]
    unsigned* status;
    // Bounded waits give up after wait_ns (0: one second). fault_tile1 > 0
    // (tests only) makes the staging of tile fault_tile1 - 1 (counted per
    // warp from its group's start) arm its barrier without issuing the
    // copies, so that its wait runs out.
    unsigned long long wait_ns;
    int64_t fault_tile1;
};

struct BwdParams {
    int64_t B, L, D;
    int G;
    int64_t Lg;
    int has_z, sp;
    const void *x, *z, *Bm, *Cm, *dy;
    int64_t bcs;    // elements between consecutive tokens' Bm (and Cm) rows
    const float *dt, *dt_bias, *A, *Dskip;
    const float* ckpt;    // [B, ceil(L/8), 8, D, 2]: state before every 8th token, pairs of states per channel
    const float* gstart;  // G == 1: dh_last [B,D,16] (nullable); G > 1: carries [B,G,D,16]
    void *dx, *dz;
    float *ddt, *dA, *dD, *ddt_bias, *dB, *dC, *dh0;
    float *aggQ, *aggS;
    unsigned* status;
};

struct StepParams {
    int64_t B, D;
    int has_z, sp;
    const void *x, *z, *Bm, *Cm;
    int64_t bcs;    // elements between consecutive batch rows of Bm_t (and Cm_t)
    const float *dt, *dt_bias, *A, *Dskip;
    float* state;
    void* y;
    unsigned* status;
};

// Set a kernel's dynamic shared-memory limit once per device (the attribute
// is per device; `mask` is one bit per device ordinal). It is set whatever
// the size, because static plus dynamic shared memory above 48 KB needs it
// even when the dynamic part alone is smaller.
template <typename K> inline bool ensure_smem(K kern, int bytes, unsigned long long& mask) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    const unsigned long long bit = 1ull << (dev & 63);
    if (mask & bit) return true;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
        return false;
    mask |= bit;
    return true;
}

// The row stride of Bm / Cm in elements: 0 means dense (N); otherwise at
// least N and a whole number of 16-byte units (the TMA tensor maps that stage
// the rows need a row pitch that is a multiple of 16 bytes). Returns an SSM_
// status code.
inline int check_bc_stride(int64_t s, int64_t N, int io_dtype) {
    if (s == 0) return SSM_OK;
    if (s < N || s > (int64_t(1) << 24)) return SSM_ERR_INVALID_ARG;
    const int64_t es = io_dtype == SSM_BF16 ? 2 : 4;
    return (s * es) % 16 == 0 ? SSM_OK : SSM_ERR_ALIGNMENT;
}

// Token shares per warp column of the conv: as many as one wave of
// resident warps can take (`warps`), each at least 16 tokens, and one when
// the call updates its state in place (the thread that reads the state at
// the start must be the one that writes it at the end).
inline int64_t conv_splits(int64_t cols, int64_t L, int64_t warps, bool in_place_state) {
    if (in_place_state || cols <= 0) return 1;
    int64_t s = warps / cols;
    const int64_t cap = (L + 15) / 16;
    if (s > cap) s = cap;
    return s < 1 ? 1 : s;
}

// L-groups when the caller leaves the choice. A pass over G groups runs
// G * ctas_per_group CTAs in waves of `capacity` (resident CTAs on the
// device); a wave that is partly empty wastes its share, and every group but
// the last costs an aggregate pass of relative price `alpha`. Returns the G
// in [1, gmax] that minimises 1/fill(G) + alpha*(G-1)/G, fill = waves /
// ceil(waves).
inline int choose_groups(int64_t ctas_per_group, int64_t capacity, double alpha, int64_t gmax) {
    if (ctas_per_group < 1) ctas_per_group = 1;
    if (capacity < 1) capacity = 1;
    int best = 1;
    double best_cost = 1e30;
    const int64_t top = gmax < 64 ? gmax : 64;
    for (int64_t G = 1; G <= top; ++G) {
        const double waves = (double)(G * ctas_per_group) / (double)capacity;
        const double full = (double)((G * ctas_per_group + capacity - 1) / capacity);
        const double cost = full / waves + alpha * (double)(G - 1) / (double)G;
        if (cost < best_cost - 1e-9) {
            best_cost = cost;
            best = (int)G;
        }
    }
    return best;
}

// Forward L-groups: one group when the grid already gives every SM more
// than one CTA (>= 1.5 per SM); otherwise as many groups as fill the resident
// CTA slots once. (The forward's aggregate pass costs about 0.6 of a main
// pass per token, and an SM that holds fewer CTAs finishes them sooner, so a
// partly filled single wave beats paying for aggregates; a grid far below
// one CTA per SM does not.)
inline int choose_groups_fwd(int64_t ctas_per_group, int64_t sms, int64_t blocks_per_sm, int64_t gmax) {
    if (ctas_per_group < 1) ctas_per_group = 1;
    if (2 * ctas_per_group >= 3 * sms) return 1;
    int64_t G = (sms * blocks_per_sm) / ctas_per_group;
    if (G > gmax) G = gmax;
    return G < 1 ? 1 : (int)G;
}

// Resident CTAs per SM of the forward / backward main kernels (occupancy
// query, cached per device), channels per CTA, and the SM count.
int fwd_blocks_per_sm(int io);
int bwd_blocks_per_sm(int io);
int fwd_channels_per_cta();
int bwd_channels_per_cta();
int sm_count();

// io: 0 = fp32, 1 = bf16. Each launcher returns the number of kernels it
// launched (>= 0) or -1 if a launch failed.
int launch_fwd(int io, const FwdParams& p, cudaStream_t s);
int launch_fwd_agg(int io, const FwdParams& p, cudaStream_t s);
int launch_carry(int64_t B, int64_t D, int G, bool reverse, const float* A, const float* start,
                 const float* aggV, const float* aggS, float* out, cudaStream_t s);
int launch_step(int io, int nsplit, const StepParams& p, cudaStream_t s);
int launch_conv(int io, bool bwd, int64_t B, int64_t L, int64_t D, int K, const void* xin, const float* w,
                const float* bias, const float* state_in, void* x, float* state_out, const void* dx, void* dxin,
                float* dw, float* dbias, float* dstate, unsigned* status, cudaStream_t s);
int launch_bwd(int io, const BwdParams& p, cudaStream_t s);
int dtproj_smem_bytes(int64_t R);
// A TMA descriptor of a 2D [rows, cols] tensor whose rows are stride_bytes
// apart, copied in boxes of box_cols x box_rows; elements past either end
// read as zero. False when the driver lacks the encoder or rejects the shape.
bool encode_2d(CUtensorMap* map, CUtensorMapDataType type, const void* base, int64_t cols, int64_t rows,
               int64_t stride_bytes, int box_cols, int box_rows, CUtensorMapSwizzle swizzle);
int launch_dtproj(bool bwd, int64_t M, int64_t D, int64_t R, int64_t a_stride, const void* a, const void* w,
                  const float* bias, float* out, const float* dout, float* dbias, int softplus, unsigned* status,
                  cudaStream_t s);
int launch_bwd_agg(int io, const BwdParams& p, cudaStream_t s);

// The per-thread launch count that ssm_last_launch_count reports: reset at
// the start of an entry point; count_launches adds a launcher's result and
// maps a failed launch (r < 0) to SSM_ERR_CUDA.
void reset_launches();
int count_launches(int r);

}  // namespace ssm
