// C entry points of libssmscan.so: argument validation (nothing is launched
// when an argument is wrong), launch-shape choice, and the sequence of
// kernels each call runs on the caller's stream. See include/ssm_scan.h.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include <cudaTypedefs.h>

#include "../../include/ssm_scan.h"
#include "ssm_common.cuh"
#include "ssm_internal.h"

namespace ssm {
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
}  // namespace

bool encode_2d(CUtensorMap* map, CUtensorMapDataType type, const void* base, int64_t cols, int64_t rows,
               int64_t stride_bytes, int box_cols, int box_rows, CUtensorMapSwizzle swizzle) {
    const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc || cols <= 0 || rows <= 0) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)stride_bytes};
    const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, type, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace ssm

namespace {

using ssm::BwdParams;
using ssm::FwdParams;
using ssm::StepParams;

constexpr int64_t kCK = 16;   // L-groups are whole forward tiles
constexpr int64_t kCkpt = 8;  // tokens between saved forward states
constexpr int64_t kGroupBudget = 131072;  // cap on B*D*groups held in the carry buffers
constexpr size_t kStatusBytes = 256;

thread_local int g_launches = 0;
// One-shot staging fault for the next ssm_scan_fwd of this thread (tests).
thread_local int64_t g_fault_tile1 = 0;
thread_local unsigned long long g_fault_wait_ns = 0;

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

int64_t max_groups(int64_t B, int64_t L, int64_t D) {
    const int64_t nck = std::max<int64_t>(1, ceil_div(L, kCK));
    const int64_t ch = std::max<int64_t>(1, B * D);
    return std::max<int64_t>(1, std::min<int64_t>(nck, std::max<int64_t>(1, kGroupBudget / ch)));
}

struct WsLayout {
    size_t aggV, aggS, carry, total;
};

WsLayout ws_layout(int64_t B, int64_t L, int64_t D) {
    const int64_t gm = max_groups(B, L, D);
    const size_t nv = (size_t)B * gm * D * 16 * sizeof(float);
    const size_t ns = (size_t)B * gm * D * sizeof(float);
    WsLayout w;
    w.aggV = kStatusBytes;
    w.aggS = w.aggV + nv;
    w.carry = w.aggS + ((ns + 255) / 256) * 256;
    w.total = w.carry + nv;
    return w;
}

bool misaligned(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

// Price of the backward's aggregate pass (one exponential per element, no
// outputs) relative to the backward main pass.
constexpr double kBwdAggCost = 0.15;

int auto_groups_fwd(int io, int64_t B, int64_t D, int64_t gmax) {
    const int64_t ctas = B * ceil_div(D, ssm::fwd_channels_per_cta());
    return ssm::choose_groups_fwd(ctas, ssm::sm_count(), ssm::fwd_blocks_per_sm(io), gmax);
}
int auto_groups_bwd(int io, int64_t B, int64_t D, int64_t gmax) {
    const int64_t ctas = B * ceil_div(D, ssm::bwd_channels_per_cta());
    return ssm::choose_groups(ctas, (int64_t)ssm::bwd_blocks_per_sm(io) * ssm::sm_count(), kBwdAggCost, gmax);
}

// Common checks of the forward-shaped arguments. Returns SSM_OK or an error.
int check_fwd(const ssm_fwd_args* a, bool need_y) {
    if (!a) return SSM_ERR_INVALID_ARG;
    if (a->B < 0 || a->L < 0 || a->D < 0 || a->N < 0) return SSM_ERR_INVALID_ARG;
    if (a->N != 16) return SSM_ERR_UNSUPPORTED;
    if (a->io_dtype != SSM_F32 && a->io_dtype != SSM_BF16) return SSM_ERR_UNSUPPORTED;
    if (a->delta_softplus != 0 && a->delta_softplus != 1) return SSM_ERR_INVALID_ARG;
    if (a->nsplit != 0 && a->nsplit != 1 && a->nsplit != 2 && a->nsplit != 4) return SSM_ERR_INVALID_ARG;
    if (a->groups < 0) return SSM_ERR_INVALID_ARG;
    if (a->D % 8 != 0) return SSM_ERR_ALIGNMENT;
    if (a->B > (int64_t(1) << 31) || a->D > (int64_t(1) << 31) || a->L > (int64_t(1) << 40))
        return SSM_ERR_INVALID_ARG;
    const int bc = ssm::check_bc_stride(a->bc_stride, a->N, a->io_dtype);
    if (bc != SSM_OK) return bc;
    // the tiles are addressed by 32-bit rows of the flattened [B*L] tensors and of the
    // checkpoints (2 rows per token: 16 states every 8 tokens)
    // (L is bounded first so that B * L stays inside int64)
    if (a->L > (int64_t(1) << 30) || a->B * a->L > (int64_t(1) << 30)) return SSM_ERR_UNSUPPORTED;
    const bool work = a->B > 0 && a->L > 0 && a->D > 0;
    if (work && (!a->x || !a->dt || !a->Bm || !a->Cm || !a->A || (need_y && !a->y))) return SSM_ERR_INVALID_ARG;
    const void* ptrs[] = {a->x, a->z, a->Bm, a->Cm, a->dt, a->dt_bias, a->A, a->Dskip, a->h0, a->y, a->h_last,
                          a->ckpt, a->workspace};
    for (const void* p : ptrs)
        if (misaligned(p)) return SSM_ERR_ALIGNMENT;
    if (!a->workspace || a->workspace_bytes < ssm_scan_workspace_bytes(a->B, a->L, a->D, a->N))
        return SSM_ERR_WORKSPACE;
    return SSM_OK;
}

__global__ void dA_log_kernel(const float* dA, const float* __restrict__ A, float* dA_log, int64_t n) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        dA_log[i] = dA[i] * A[i];
}

// The FMA-pipe 2^x applied to n values (tests and error-bound checks).
__global__ void exp2_fma_kernel(const float* __restrict__ x, float* __restrict__ y, int64_t n) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        y[i] = ssm::ex2_fma(x[i]);
}

int tally(int r) {
    if (r < 0) return SSM_ERR_CUDA;
    g_launches += r;
    return SSM_OK;
}

}  // namespace

namespace ssm {
void reset_launches() { g_launches = 0; }
int count_launches(int r) { return tally(r); }
}  // namespace ssm

extern "C" {

size_t ssm_scan_workspace_bytes(int64_t B, int64_t L, int64_t D, int64_t N) {
    (void)N;
    if (B < 0 || L < 0 || D < 0) return kStatusBytes;
    return ws_layout(B, L, D).total;
}

int64_t ssm_scan_ckpt_elems(int64_t B, int64_t L, int64_t D, int64_t N) {
    if (B < 0 || L < 0 || D < 0 || N < 0) return 0;
    return B * ceil_div(L, kCkpt) * D * N;
}

int ssm_scan_ckpt_interval(void) { return (int)kCkpt; }

int ssm_last_launch_count(void) { return g_launches; }

int ssm_debug_arm_wait_fault(int64_t tile, uint64_t wait_ns) {
    if (wait_ns > 10000000000ull) return SSM_ERR_INVALID_ARG;
    g_fault_tile1 = tile < 0 ? 0 : tile + 1;
    g_fault_wait_ns = tile < 0 ? 0 : wait_ns;
    return SSM_OK;
}

const char* ssm_status_string(int code) {
    switch (code) {
        case SSM_OK: return "ok";
        case SSM_ERR_INVALID_ARG: return "invalid argument (null required pointer, negative size or bad flag)";
        case SSM_ERR_UNSUPPORTED: return "unsupported (d_state must be 16; dtype must be fp32 or bf16)";
        case SSM_ERR_ALIGNMENT: return "alignment (D must be a multiple of 8 and pointers 16-byte aligned)";
        case SSM_ERR_WORKSPACE: return "workspace missing or smaller than ssm_scan_workspace_bytes()";
        case SSM_ERR_CUDA: return "a CUDA call or kernel launch failed";
        case SSM_ERR_NONFINITE: return "a kernel produced a non-finite value";
        case SSM_ERR_TIMEOUT: return "a bounded wait inside a kernel ran out (its results are not valid)";
        case SSM_ERR_SCRATCH_LIMIT:
            return "the requested L-groups need more scratch than the library's built-in 8 MiB array holds";
        default: return "unknown status";
    }
}

int ssm_clear_status(void* workspace, void* stream) {
    if (!workspace) return SSM_ERR_INVALID_ARG;
    return cudaMemsetAsync(workspace, 0, sizeof(unsigned), (cudaStream_t)stream) == cudaSuccess ? SSM_OK
                                                                                                : SSM_ERR_CUDA;
}

int ssm_poll_status(void* workspace, void* stream) {
    if (!workspace) return SSM_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    unsigned v = 0;
    if (cudaMemcpyAsync(&v, workspace, sizeof(unsigned), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return SSM_ERR_CUDA;
    if (cudaMemsetAsync(workspace, 0, sizeof(unsigned), s) != cudaSuccess) return SSM_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return SSM_ERR_CUDA;
    if (v & ssm::kStatusTimeout) return SSM_ERR_TIMEOUT;
    return (v & ssm::kStatusNonFinite) ? SSM_ERR_NONFINITE : SSM_OK;
}

int ssm_scan_fwd(const ssm_fwd_args* a, void* stream) {
    g_launches = 0;
    // a fault armed by ssm_debug_arm_wait_fault applies to this call only
    const int64_t fault_tile1 = g_fault_tile1;
    const unsigned long long fault_wait_ns = g_fault_wait_ns;
    g_fault_tile1 = 0;
    g_fault_wait_ns = 0;
    int rc = check_fwd(a, true);
    if (rc != SSM_OK) return rc;
    cudaStream_t s = (cudaStream_t)stream;
    const int64_t B = a->B, L = a->L, D = a->D;
    if (B == 0 || D == 0) return SSM_OK;
    if (L == 0) {
        if (a->h_last) {
            const size_t bytes = (size_t)B * D * 16 * sizeof(float);
            cudaError_t e = a->h0 ? cudaMemcpyAsync(a->h_last, a->h0, bytes, cudaMemcpyDeviceToDevice, s)
                                  : cudaMemsetAsync(a->h_last, 0, bytes, s);
            if (e != cudaSuccess) return SSM_ERR_CUDA;
        }
        return SSM_OK;
    }
    const int64_t nck = ceil_div(L, kCK), gmax = max_groups(B, L, D);
    const int64_t gcap = std::min<int64_t>(nck, gmax);
    int G = a->groups ? (int)std::min<int64_t>(a->groups, gcap) : auto_groups_fwd(a->io_dtype, B, D, gcap);
    const int64_t Lg = ceil_div(nck, G) * kCK;
    G = (int)ceil_div(L, Lg);
    const WsLayout w = ws_layout(B, L, D);
    char* ws = (char*)a->workspace;

    FwdParams p{};
    p.B = B; p.L = L; p.D = D; p.G = G; p.Lg = Lg;
    p.has_z = a->z != nullptr; p.sp = a->delta_softplus;
    p.x = a->x; p.z = a->z; p.Bm = a->Bm; p.Cm = a->Cm; p.bcs = a->bc_stride ? a->bc_stride : 16;
    p.dt = a->dt; p.dt_bias = a->dt_bias; p.A = a->A; p.Dskip = a->Dskip;
    p.hstart = a->h0; p.y = a->y; p.h_last = a->h_last; p.ckpt = a->ckpt;
    p.aggH = (float*)(ws + w.aggV); p.aggS = (float*)(ws + w.aggS);
    p.status = (unsigned*)ws;
    if (G > 1) {
        if ((rc = tally(ssm::launch_fwd_agg(a->io_dtype, p, s))) != SSM_OK) return rc;
        if ((rc = tally(ssm::launch_carry(B, D, G, false, a->A, a->h0, p.aggH, p.aggS, (float*)(ws + w.carry), s))) !=
            SSM_OK)
            return rc;
        p.hstart = (const float*)(ws + w.carry);
    }
    p.fault_tile1 = fault_tile1;
    p.wait_ns = fault_wait_ns;
    return tally(ssm::launch_fwd(a->io_dtype, p, s));
}

int ssm_scan_bwd(const ssm_bwd_args* a, void* stream) {
    g_launches = 0;
    if (!a) return SSM_ERR_INVALID_ARG;
    int rc = check_fwd(&a->f, false);
    if (rc != SSM_OK) return rc;
    const ssm_fwd_args& f = a->f;
    const int64_t B = f.B, L = f.L, D = f.D;
    const bool work = B > 0 && L > 0 && D > 0;
    if (work && (!a->dy || !a->dx || !a->d_dt || !f.ckpt || (f.z && !a->dz))) return SSM_ERR_INVALID_ARG;
    if (D > 0 && (!a->dA || !a->dD || !a->d_dt_bias)) return SSM_ERR_INVALID_ARG;
    if (B > 0 && L > 0 && (!a->dB || !a->dC)) return SSM_ERR_INVALID_ARG;
    const void* ptrs[] = {a->dy, a->dh_last, a->dx, a->dz, a->d_dt, a->dA, a->dD, a->d_dt_bias, a->dB, a->dC, a->dh0};
    for (const void* p : ptrs)
        if (misaligned(p)) return SSM_ERR_ALIGNMENT;
    cudaStream_t s = (cudaStream_t)stream;
    // The reductions are overwritten: zero them on the stream first.
    if (D > 0) {
        if (cudaMemsetAsync(a->dA, 0, (size_t)D * 16 * sizeof(float), s) != cudaSuccess ||
            cudaMemsetAsync(a->dD, 0, (size_t)D * sizeof(float), s) != cudaSuccess ||
            cudaMemsetAsync(a->d_dt_bias, 0, (size_t)D * sizeof(float), s) != cudaSuccess)
            return SSM_ERR_CUDA;
    }
    if (B > 0 && L > 0) {
        const size_t bl = (size_t)B * L * 16 * sizeof(float);
        if (cudaMemsetAsync(a->dB, 0, bl, s) != cudaSuccess || cudaMemsetAsync(a->dC, 0, bl, s) != cudaSuccess)
            return SSM_ERR_CUDA;
    }
    if (!work) {
        if (a->dh0 && B > 0 && D > 0) {
            const size_t bytes = (size_t)B * D * 16 * sizeof(float);
            cudaError_t e = a->dh_last ? cudaMemcpyAsync(a->dh0, a->dh_last, bytes, cudaMemcpyDeviceToDevice, s)
                                       : cudaMemsetAsync(a->dh0, 0, bytes, s);
            if (e != cudaSuccess) return SSM_ERR_CUDA;
        }
        return SSM_OK;
    }
    const int64_t nck = ceil_div(L, kCK), gmax = max_groups(B, L, D);
    const int64_t gcap = std::min<int64_t>(nck, gmax);
    int G = f.groups ? (int)std::min<int64_t>(f.groups, gcap) : auto_groups_bwd(f.io_dtype, B, D, gcap);
    const int64_t Lg = ceil_div(nck, G) * kCK;
    G = (int)ceil_div(L, Lg);
    const WsLayout w = ws_layout(B, L, D);
    char* ws = (char*)f.workspace;

    BwdParams p{};
    p.B = B; p.L = L; p.D = D; p.G = G; p.Lg = Lg;
    p.has_z = f.z != nullptr; p.sp = f.delta_softplus;
    p.x = f.x; p.z = f.z; p.Bm = f.Bm; p.Cm = f.Cm; p.dy = a->dy; p.bcs = f.bc_stride ? f.bc_stride : 16;
    p.dt = f.dt; p.dt_bias = f.dt_bias; p.A = f.A; p.Dskip = f.Dskip;
    p.ckpt = f.ckpt; p.gstart = a->dh_last;
    p.dx = a->dx; p.dz = a->dz; p.ddt = a->d_dt; p.dA = a->dA; p.dD = a->dD; p.ddt_bias = a->d_dt_bias;
    p.dB = a->dB; p.dC = a->dC; p.dh0 = a->dh0;
    p.aggQ = (float*)(ws + w.aggV); p.aggS = (float*)(ws + w.aggS);
    p.status = (unsigned*)ws;
    if (G > 1) {
        if ((rc = tally(ssm::launch_bwd_agg(f.io_dtype, p, s))) != SSM_OK) return rc;
        if ((rc = tally(ssm::launch_carry(B, D, G, true, f.A, a->dh_last, p.aggQ, p.aggS, (float*)(ws + w.carry), s))) !=
            SSM_OK)
            return rc;
        p.gstart = (const float*)(ws + w.carry);
    }
    return tally(ssm::launch_bwd(f.io_dtype, p, s));
}

int ssm_dA_log_grad(const float* dA, const float* A, float* dA_log, int64_t n, void* stream) {
    g_launches = 0;
    if (n < 0) return SSM_ERR_INVALID_ARG;
    if (n == 0) return SSM_OK;
    if (!dA || !A || !dA_log) return SSM_ERR_INVALID_ARG;
    const int64_t blocks = std::min<int64_t>(ceil_div(n, 256), 4096);
    dA_log_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(dA, A, dA_log, n);
    return tally(cudaGetLastError() == cudaSuccess ? 1 : -1);
}

int ssm_exp2_fma(const float* x, float* y, int64_t n, void* stream) {
    g_launches = 0;
    if (n < 0) return SSM_ERR_INVALID_ARG;
    if (n == 0) return SSM_OK;
    if (!x || !y) return SSM_ERR_INVALID_ARG;
    const int64_t blocks = std::min<int64_t>(ceil_div(n, 256), 4096);
    exp2_fma_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(x, y, n);
    return tally(cudaGetLastError() == cudaSuccess ? 1 : -1);
}

namespace {
int check_conv(const ssm_conv_args* a) {
    if (!a) return SSM_ERR_INVALID_ARG;
    if (a->B < 0 || a->L < 0 || a->D < 0) return SSM_ERR_INVALID_ARG;
    if (a->K < 1 || a->K > 4) return SSM_ERR_UNSUPPORTED;
    if (a->io_dtype != SSM_F32 && a->io_dtype != SSM_BF16) return SSM_ERR_UNSUPPORTED;
    if (a->D % 8 != 0) return SSM_ERR_ALIGNMENT;
    if (a->B > (int64_t(1) << 31) || a->D > (int64_t(1) << 31) || a->L > (int64_t(1) << 40)) return SSM_ERR_INVALID_ARG;
    const bool work = a->B > 0 && a->L > 0 && a->D > 0;
    if (work && (!a->xin || !a->w)) return SSM_ERR_INVALID_ARG;
    const void* ptrs[] = {a->xin, a->w, a->bias, a->state_in, a->x, a->state_out, a->workspace};
    for (const void* p : ptrs)
        if (misaligned(p)) return SSM_ERR_ALIGNMENT;
    return SSM_OK;
}
}  // namespace

int ssm_conv1d_fwd(const ssm_conv_args* a, void* stream) {
    g_launches = 0;
    int rc = check_conv(a);
    if (rc != SSM_OK) return rc;
    const bool work = a->B > 0 && a->L > 0 && a->D > 0;
    if (work && (!a->x || a->x == a->xin)) return SSM_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    if (!work) {
        if (a->state_out && a->B > 0 && a->D > 0 && a->K > 1 && a->state_out != a->state_in) {
            const size_t bytes = (size_t)a->B * a->D * (a->K - 1) * sizeof(float);
            cudaError_t e = a->state_in ? cudaMemcpyAsync(a->state_out, a->state_in, bytes, cudaMemcpyDeviceToDevice, s)
                                        : cudaMemsetAsync(a->state_out, 0, bytes, s);
            if (e != cudaSuccess) return SSM_ERR_CUDA;
        }
        return SSM_OK;
    }
    return tally(ssm::launch_conv(a->io_dtype, false, a->B, a->L, a->D, (int)a->K, a->xin, a->w, a->bias,
                                  a->state_in, a->x, a->state_out, nullptr, nullptr, nullptr, nullptr, nullptr,
                                  (unsigned*)a->workspace, s));
}

int ssm_conv1d_bwd(const ssm_conv_bwd_args* a, void* stream) {
    g_launches = 0;
    if (!a) return SSM_ERR_INVALID_ARG;
    int rc = check_conv(&a->f);
    if (rc != SSM_OK) return rc;
    const ssm_conv_args& f = a->f;
    const bool work = f.B > 0 && f.L > 0 && f.D > 0;
    if (work && (!a->dx || !a->dxin || a->dxin == a->dx || a->dxin == f.xin)) return SSM_ERR_INVALID_ARG;
    if (f.D > 0 && !a->dw) return SSM_ERR_INVALID_ARG;
    const void* ptrs[] = {a->dx, a->dxin, a->dw, a->dbias, a->dstate_in};
    for (const void* p : ptrs)
        if (misaligned(p)) return SSM_ERR_ALIGNMENT;
    cudaStream_t s = (cudaStream_t)stream;
    if (f.D > 0) {  // the reductions are overwritten: zero them on the stream first
        if (cudaMemsetAsync(a->dw, 0, (size_t)f.D * f.K * sizeof(float), s) != cudaSuccess) return SSM_ERR_CUDA;
        if (a->dbias && cudaMemsetAsync(a->dbias, 0, (size_t)f.D * sizeof(float), s) != cudaSuccess)
            return SSM_ERR_CUDA;
    }
    if (a->dstate_in && f.B > 0 && f.D > 0 && f.K > 1 && (!work))
        if (cudaMemsetAsync(a->dstate_in, 0, (size_t)f.B * f.D * (f.K - 1) * sizeof(float), s) != cudaSuccess)
            return SSM_ERR_CUDA;
    if (!work) return SSM_OK;
    return tally(ssm::launch_conv(f.io_dtype, true, f.B, f.L, f.D, (int)f.K, f.xin, f.w, f.bias, f.state_in,
                                  nullptr, nullptr, a->dx, a->dxin, a->dw, a->dbias, a->dstate_in,
                                  (unsigned*)f.workspace, s));
}

namespace {
int check_dtproj(const ssm_dtproj_args* a) {
    if (!a) return SSM_ERR_INVALID_ARG;
    if (a->M < 0 || a->D < 0 || a->R < 0 || a->a_stride < 0) return SSM_ERR_INVALID_ARG;
    if (a->softplus != 0 && a->softplus != 1) return SSM_ERR_INVALID_ARG;
    if (a->R < 16 || a->R > 256 || a->R % 16 != 0) return SSM_ERR_UNSUPPORTED;
    if (a->D % 8 != 0) return SSM_ERR_ALIGNMENT;
    const int64_t stride = a->a_stride ? a->a_stride : a->R;
    if (stride < a->R) return SSM_ERR_INVALID_ARG;
    if ((stride * 2) % 16 != 0) return SSM_ERR_ALIGNMENT;
    // the copies address rows with 32-bit coordinates
    if (a->M > 0x7fffffff || a->D > 0x7fffffff || stride > (int64_t(1) << 24)) return SSM_ERR_INVALID_ARG;
    if (((a->M + 127) / 128) * ((a->D + 255) / 256) > 0x7fffffff) return SSM_ERR_UNSUPPORTED;
    const bool work = a->M > 0 && a->D > 0;
    if (work && (!a->a || !a->w)) return SSM_ERR_INVALID_ARG;
    const void* ptrs[] = {a->a, a->w, a->bias, a->delta, a->workspace};
    for (const void* p : ptrs)
        if (misaligned(p)) return SSM_ERR_ALIGNMENT;
    return SSM_OK;
}
}  // namespace

int ssm_dtproj_fwd(const ssm_dtproj_args* a, void* stream) {
    g_launches = 0;
    int rc = check_dtproj(a);
    if (rc != SSM_OK) return rc;
    if (a->M == 0 || a->D == 0) return SSM_OK;
    if (!a->delta) return SSM_ERR_INVALID_ARG;
    return tally(ssm::launch_dtproj(false, a->M, a->D, a->R, a->a_stride ? a->a_stride : a->R, a->a, a->w, a->bias,
                                    a->delta, nullptr, nullptr, a->softplus, (unsigned*)a->workspace,
                                    (cudaStream_t)stream));
}

int ssm_dtproj_bwd(const ssm_dtproj_bwd_args* a, void* stream) {
    g_launches = 0;
    if (!a) return SSM_ERR_INVALID_ARG;
    int rc = check_dtproj(&a->f);
    if (rc != SSM_OK) return rc;
    const ssm_dtproj_args& f = a->f;
    const bool work = f.M > 0 && f.D > 0;
    if (work && (!a->ddelta || !a->dpre)) return SSM_ERR_INVALID_ARG;
    if (misaligned(a->ddelta) || misaligned(a->dpre) || misaligned(a->dbias)) return SSM_ERR_ALIGNMENT;
    cudaStream_t s = (cudaStream_t)stream;
    if (a->dbias && f.D > 0 && cudaMemsetAsync(a->dbias, 0, (size_t)f.D * sizeof(float), s) != cudaSuccess)
        return SSM_ERR_CUDA;
    if (!work) return SSM_OK;
    return tally(ssm::launch_dtproj(true, f.M, f.D, f.R, f.a_stride ? f.a_stride : f.R, f.a, f.w, f.bias, a->dpre,
                                    a->ddelta, a->dbias, f.softplus, (unsigned*)f.workspace, s));
}

int ssm_step(const ssm_step_args* a, void* stream) {
    g_launches = 0;
    if (!a) return SSM_ERR_INVALID_ARG;
    if (a->B < 0 || a->D < 0 || a->N < 0) return SSM_ERR_INVALID_ARG;
    if (a->N != 16) return SSM_ERR_UNSUPPORTED;
    if (a->io_dtype != SSM_F32 && a->io_dtype != SSM_BF16) return SSM_ERR_UNSUPPORTED;
    if (a->delta_softplus != 0 && a->delta_softplus != 1) return SSM_ERR_INVALID_ARG;
    if (a->nsplit != 0 && a->nsplit != 1 && a->nsplit != 2 && a->nsplit != 4) return SSM_ERR_INVALID_ARG;
    if (a->D % 8 != 0) return SSM_ERR_ALIGNMENT;
    const int bc = ssm::check_bc_stride(a->bc_stride, a->N, a->io_dtype);
    if (bc != SSM_OK) return bc;
    const bool work = a->B > 0 && a->D > 0;
    if (work && (!a->x_t || !a->dt_t || !a->Bm_t || !a->Cm_t || !a->A || !a->state || !a->y_t))
        return SSM_ERR_INVALID_ARG;
    const void* ptrs[] = {a->x_t, a->z_t, a->Bm_t, a->Cm_t, a->dt_t, a->dt_bias, a->A, a->Dskip, a->state, a->y_t,
                          a->workspace};
    for (const void* p : ptrs)
        if (misaligned(p)) return SSM_ERR_ALIGNMENT;
    if (!work) return SSM_OK;
    StepParams p{};
    p.B = a->B; p.D = a->D;
    p.has_z = a->z_t != nullptr; p.sp = a->delta_softplus;
    p.x = a->x_t; p.z = a->z_t; p.Bm = a->Bm_t; p.Cm = a->Cm_t; p.bcs = a->bc_stride ? a->bc_stride : 16;
    p.dt = a->dt_t; p.dt_bias = a->dt_bias; p.A = a->A; p.Dskip = a->Dskip;
    p.state = a->state; p.y = a->y_t; p.status = (unsigned*)a->workspace;
    // one lane per channel when the channels alone fill the GPU, else two
    // (the readout has two halves; nsplit = 4 runs as 2)
    const int nsplit = a->nsplit ? std::min(a->nsplit, 2) : (a->B * a->D >= 65536 ? 1 : 2);
    return tally(ssm::launch_step(a->io_dtype, nsplit, p, (cudaStream_t)stream));
}

}  // extern "C"
