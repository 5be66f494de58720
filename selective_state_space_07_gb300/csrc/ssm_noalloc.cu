// ssm_scan_fwd_noalloc: the sequence forward for callers that cannot
// allocate device memory.
//
// ssm_scan_fwd asks its caller for a workspace because, when it splits the
// sequence into several L-groups, it stores each group's aggregate and the
// carries between groups in global memory. Some callers cannot provide one:
// code that runs where cudaMalloc is off limits (inside an allocator or
// memory-pool callback, in a process whose device memory is fully planned
// ahead by another component, or in a plug-in that is handed only the
// tensors it reads and writes). This entry point keeps that scratch in one
// array compiled into the library instead, so it allocates nothing at all.
//
// Limits and rules:
// - The array holds kNoAllocScratchBytes (8 MiB). Every GPU that loads the
//   library reserves it until the process exits.
// - With groups == 0 the library picks the number of L-groups as
//   ssm_scan_fwd does, but never more than the array can hold; an explicit
//   groups whose carries do not fit is rejected with SSM_ERR_SCRATCH_LIMIT
//   before anything is launched.
// - The first call in each CUDA context (one per device for the runtime's
//   primary contexts) looks up the array's device address
//   (cudaGetSymbolAddress, with that device current) and caches it under
//   the context's unique ID; make that first call before any stream
//   capture. A context that is destroyed and created again (after
//   cudaDeviceReset, say) gets a new ID, so the address is looked up again
//   instead of reusing one from the old context.
// - All calls share the array and it keeps the last call's contents. The
//   kernels overwrite every carry they read, and the status word is zeroed
//   at the start of each call. Calls whose work overlaps on the GPU (other
//   streams, other host threads) race on the array: serialise them.
// - Non-finite outputs are latched in args->workspace when the caller
//   passes one (>= 256 bytes, read it with ssm_poll_status); otherwise they
//   are latched in the array, which the caller cannot read.
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "../../include/ssm_scan.h"
#include "ssm_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;
constexpr int64_t kChunk = 16;
constexpr size_t kStatus = 256;

// The scratch. In host code this name is only a stand-in for the symbol;
// kernels get the device address looked up below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;

// Unique ID of the calling thread's current CUDA context (the driver's
// cuCtxGetId, reached through the runtime's entry-point query so that the
// library needs no link to libcuda); false when it is not available.
bool current_context_id(unsigned long long* id) {
    static const auto fns = [] {
        void* get = nullptr;
        void* gid = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &get, 4000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            get = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &gid, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            gid = nullptr;
        return std::make_pair(reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(get),
                              reinterpret_cast<PFN_cuCtxGetId_v12000>(gid));
    }();
    if (!fns.first || !fns.second) return false;
    CUcontext ctx = nullptr;
    if (fns.first(&ctx) != CUDA_SUCCESS || !ctx) return false;
    return fns.second(ctx, id) == CUDA_SUCCESS;
}

// Looked-up addresses, keyed by context ID (or, when the driver gives no
// context IDs, by device ordinal + 1 with the top bit set).
struct ScratchEntry {
    unsigned long long key;
    void* addr;
};
ScratchEntry g_scratch_cache[64] = {};
int g_scratch_next = 0;

// Device address of g_noalloc_scratch in the current context (looked up
// once per context, with the device current). nullptr on failure.
void* scratch_on_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return nullptr;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    unsigned long long key = 0;
    bool have = current_context_id(&key);
    if (have)
        for (const ScratchEntry& e : g_scratch_cache)
            if (e.addr && e.key == key) return e.addr;
    void* p = nullptr;  // (the lookup also brings up the device's primary context when it has none yet)
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return nullptr;
    if (!have) have = current_context_id(&key);
    if (!have) key = (1ull << 63) | (unsigned long long)(dev + 1);
    g_scratch_cache[g_scratch_next] = ScratchEntry{key, p};
    g_scratch_next = (g_scratch_next + 1) % 64;
    return p;
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Bytes of scratch a forward with G groups needs (status word, aggregates,
// sums of Delta, carries).
size_t scratch_need(int64_t B, int64_t D, int G) {
    if (G <= 1) return kStatus;
    const size_t nv = (size_t)B * G * D * 16 * sizeof(float);
    const size_t ns = (((size_t)B * G * D * sizeof(float)) + 255) / 256 * 256;
    return kStatus + nv + ns + nv;
}

bool misaligned(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

}  // namespace

extern "C" int ssm_scan_fwd_noalloc(const ssm_fwd_args* a, void* stream) {
    ssm::reset_launches();
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
    if (a->B * a->L > (int64_t(1) << 30)) return SSM_ERR_UNSUPPORTED;
    const int64_t B = a->B, L = a->L, D = a->D;
    const bool work = B > 0 && L > 0 && D > 0;
    if (work && (!a->x || !a->dt || !a->Bm || !a->Cm || !a->A || !a->y)) return SSM_ERR_INVALID_ARG;
    const void* ptrs[] = {a->x, a->z, a->Bm, a->Cm, a->dt, a->dt_bias, a->A, a->Dskip, a->h0, a->y, a->h_last,
                          a->ckpt, a->workspace};
    for (const void* p : ptrs)
        if (misaligned(p)) return SSM_ERR_ALIGNMENT;
    if (a->workspace && a->workspace_bytes < kStatus) return SSM_ERR_WORKSPACE;

    // launch shape: as ssm_scan_fwd chooses it, within the array
    const int64_t nck = std::max<int64_t>(1, cdiv(L, kChunk));
    int G = 1;
    if (work) {
        if (a->groups) {
            G = (int)std::min<int64_t>(a->groups, nck);
            G = (int)cdiv(L, cdiv(nck, G) * kChunk);
            if (scratch_need(B, D, G) > kNoAllocScratchBytes) return SSM_ERR_SCRATCH_LIMIT;
        } else {
            int64_t want = ssm::choose_groups_fwd(B * cdiv(D, ssm::fwd_channels_per_cta()), ssm::sm_count(),
                                                  ssm::fwd_blocks_per_sm(a->io_dtype), nck);
            while (want > 1 && scratch_need(B, D, (int)want) > kNoAllocScratchBytes) --want;
            G = (int)cdiv(L, cdiv(nck, want) * kChunk);
        }
    }
    if (scratch_need(B, D, G) > kNoAllocScratchBytes) return SSM_ERR_SCRATCH_LIMIT;

    cudaStream_t s = (cudaStream_t)stream;
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

    char* scratch = (char*)scratch_on_current_device();
    if (!scratch) return SSM_ERR_CUDA;
    unsigned* status = a->workspace ? (unsigned*)a->workspace : (unsigned*)scratch;
    if (!a->workspace && cudaMemsetAsync(scratch, 0, sizeof(unsigned), s) != cudaSuccess) return SSM_ERR_CUDA;

    const int64_t Lg = cdiv(nck, G) * kChunk;
    const size_t nv = (size_t)B * G * D * 16 * sizeof(float);
    const size_t ns = (((size_t)B * G * D * sizeof(float)) + 255) / 256 * 256;
    ssm::FwdParams p{};
    p.B = B; p.L = L; p.D = D; p.G = G; p.Lg = Lg;
    p.has_z = a->z != nullptr; p.sp = a->delta_softplus;
    p.x = a->x; p.z = a->z; p.Bm = a->Bm; p.Cm = a->Cm; p.bcs = a->bc_stride ? a->bc_stride : 16;
    p.dt = a->dt; p.dt_bias = a->dt_bias; p.A = a->A; p.Dskip = a->Dskip;
    p.hstart = a->h0; p.y = a->y; p.h_last = a->h_last; p.ckpt = a->ckpt;
    p.aggH = (float*)(scratch + kStatus);
    p.aggS = (float*)(scratch + kStatus + nv);
    p.status = status;
    int rc;
    if (G > 1) {
        float* carry = (float*)(scratch + kStatus + nv + ns);
        if ((rc = ssm::count_launches(ssm::launch_fwd_agg(a->io_dtype, p, s))) != SSM_OK) return rc;
        if ((rc = ssm::count_launches(ssm::launch_carry(B, D, G, false, a->A, a->h0, p.aggH, p.aggS, carry, s))) !=
            SSM_OK)
            return rc;
        p.hstart = carry;
    }
    return ssm::count_launches(ssm::launch_fwd(a->io_dtype, p, s));
}
