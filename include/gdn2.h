/*
 * gdn2.h -- C ABI of the Gated DeltaNet-2 chunkwise forward in
 * libssmscan.so (sm_103a tensor cores).
 *
 * The operation (docs.rs, burn-gdn2 0.1.4, src/forward.rs, chunk_wy_forward:
 * "Gated DeltaNet 2 -- linear recurrent token mixer with channel-wise
 * erase/write gates"). Per (batch, head), the sequence is cut into chunks of
 * 64 tokens (the last one ragged); per chunk, with S the [K, V] state before
 * it:
 *   G       = cumulative sum of the log-gates g over the chunk's tokens
 *   decay   = mean over key channels of exp(G[i] - G[j])
 *   aqk     = (q k^T) * decay * scale          (j <= i)
 *   akk     = ((b * k) k^T) * decay            (j <  i)
 *   W, U    : (I + akk) W = b * k * exp(G),  (I + akk) U = w * v
 *   v_new   = U - W S
 *   out     = aqk v_new + (q * exp(G)) S * scale
 *   S       = S * exp(G[last]) (per key row) + (k * exp(G[last] - G))^T v_new
 *
 * Layout [batch, heads, time, dim], dense and contiguous:
 *   q, k, b           [B, H, T, K]  bf16      (b: per-key-channel erase gate)
 *   g                 [B, H, T, K]  fp32      (log-gates, <= 0)
 *   v, w              [B, H, T, V]  bf16      (w: per-value-channel write gate)
 *   state_in/out      [B, H, K, V]  fp32
 *   out               [B, H, T, V]  bf16
 * Products are formed on the tensor cores from bf16 operands with fp32
 * accumulation; the state is carried in fp32. K = V = 128 and chunk = 64
 * (0 means 64) are required (else SSM_ERR_UNSUPPORTED); every pointer must
 * be 16-byte aligned (else SSM_ERR_ALIGNMENT); q, k, v, g, b, w and out
 * must be non-null when B*H*T > 0, sizes non-negative, B*H below 2^31 and
 * scale finite (else SSM_ERR_INVALID_ARG); B*H*T must stay below
 * 2^31 - 128 token rows (else SSM_ERR_UNSUPPORTED: copies address rows with
 * 32-bit coordinates). state_in NULL means a zero
 * initial state; state_out NULL skips the final state. With T = 0 the
 * final state is the initial one (copied, or zeroed).
 *
 * The intra-chunk decay is evaluated as the product of exp(G[i] - G[m]) and
 * exp(G[m] - G[j]) about the chunk's middle token m, so each factor must
 * stay inside the float range: per key channel the log-gates of a
 * half-chunk (32 tokens) must sum to more than -80. Gates outside that
 * range give non-finite outputs, which are latched in the status word.
 *
 * Calls are asynchronous on `stream`; the caller owns every buffer;
 * workspace (nullable, >= 256 bytes) receives the status word read by
 * ssm_poll_status (non-finite outputs; SSM_ERR_TIMEOUT if a tensor-core
 * completion never arrived). Argument errors return a negative SSM_ code
 * before anything is launched.
 */
#ifndef GDN2_H
#define GDN2_H

#include <stddef.h>
#include <stdint.h>

#include "ssm_scan.h" /* the SSM_ status codes and ssm_poll_status */

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
    int64_t B, H, T, K, V;
    int32_t chunk;
    float scale;
    const void* q;
    const void* k;
    const void* v;
    const float* g;
    const void* b;
    const void* w;
    const float* state_in;
    void* out;
    float* state_out;
    void* workspace;
} gdn2_fwd_args;

int gdn2_chunk_fwd(const gdn2_fwd_args* args, void* stream);

/* One token of the mixer, the per-token form the chunked steps reduce to
 * with chunks of one token (the fused recurrent forward the page checks the
 * chunked one against; decoding): with S the state, updated in place,
 *   S     = S * exp(g) (per key row)
 *   v_new = w * v - (b * k)^T S
 *   S     = S + k v_new^T
 *   out   = scale * q^T S
 * Layout: q, k, b [B, H, K] bf16; g [B, H, K] fp32; v, w [B, H, V] bf16;
 * state [B, H, K, V] fp32 (in place); out [B, H, V] bf16. Everything in
 * fp32 (one token is a matrix-vector step: no tensor cores). With gates that
 * differ across key channels the chunked forward's key-mean decay makes it a
 * different evaluation from this one; with one gate per token they agree.
 * K = V = 128 (else SSM_ERR_UNSUPPORTED); q, k, b, g, v, w, state and out
 * 16-byte aligned (else SSM_ERR_ALIGNMENT) and non-null when B*H > 0, B*H
 * below 2^31, scale finite (else SSM_ERR_INVALID_ARG). Asynchronous on
 * `stream`; workspace (nullable) receives the status word. */
typedef struct {
    int64_t B, H, K, V;
    float scale;
    const void* q;
    const void* k;
    const void* v;
    const float* g;
    const void* b;
    const void* w;
    float* state;
    void* out;
    void* workspace;
} gdn2_step_args;

int gdn2_step(const gdn2_step_args* args, void* stream);

/* Test hook: arms a one-shot fault for this thread's next gdn2_chunk_fwd.
 * The copies of q, k and b for chunk `chunk` (0-based, in every CTA) are not
 * issued while the chunk's other copies are, and every bounded wait of that
 * call gives up after wait_ns (0 keeps the 1 s default): the wait for the
 * missing copies runs out, each CTA waits for the copies it did issue, frees
 * its tensor memory and stops; ssm_poll_status then returns SSM_ERR_TIMEOUT
 * and the outputs are not valid. chunk < 0 disarms. SSM_ERR_INVALID_ARG for
 * wait_ns above 10 s. */
int gdn2_debug_arm_wait_fault(int64_t chunk, uint64_t wait_ns);

#ifdef __cplusplus
}
#endif
#endif /* GDN2_H */
