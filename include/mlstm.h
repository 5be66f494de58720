/*
 * mlstm.h -- C ABI of the mLSTM stabilized chunkwise forward in
 * libssmscan.so (sm_103a tensor cores).
 *
 * The operation: the mLSTM cell whose two implementations the page
 * Evil-Inference-Code, README_FIX_RUST.md ("mLSTM Equivalence Fixes (Rust vs
 * Python)") makes agree -- matrix memory C [K, V], normaliser n [K] and
 * log-domain stabilizer m per (batch, head), exponential input gate and
 * sigmoid forget gate (section 2, "Stabilization Logic": the denominator is
 * the larger of |q . n| and exp(-m); section 3: m starts at 0). Per token t,
 * with q scaled by `scale`:
 *   log f = log sigmoid(fgate_t), log i = igate_t
 *   m_t   = max(log f + m_{t-1}, log i)
 *   C_t   = exp(log f + m_{t-1} - m_t) C_{t-1} + exp(log i - m_t) k_t v_t^T
 *   n_t   = exp(log f + m_{t-1} - m_t) n_{t-1} + exp(log i - m_t) k_t
 *   h_t   = (q_t^T C_t) / max(|q_t . n_t|, exp(-m_t))
 * evaluated chunkwise: per chunk of 64 tokens the intra-chunk terms are the
 * parallel (quadratic) form, with the chunk's log forget gates summed by
 * iteration (section 2, "Cumulative Sum"), and the state carries across
 * chunks. With norm_weight non-null, each output row is then normalised
 * over its V channels (mean and biased variance, eps = norm_eps) and
 * multiplied by norm_weight[head] -- no bias (section 3, "LayerNorm").
 *
 * Layout [batch, heads, time, dim], dense and contiguous:
 *   q, k              [B, H, T, K]  bf16
 *   v                 [B, H, T, V]  bf16
 *   igate, fgate      [B, H, T]     fp32   (gate pre-activations)
 *   C_in / C_out      [B, H, K, V]  fp32   (stabilized: the plain C times exp(-m))
 *   n_in / n_out      [B, H, K]     fp32   (likewise)
 *   m_in / m_out      [B, H]        fp32
 *   norm_weight       [H, V]        fp32
 *   h                 [B, H, T, V]  bf16
 * Products are formed on the tensor cores from bf16 operands with fp32
 * accumulation; gates, stabilizer, denominator, state and norm are fp32.
 * K = V = 128 and chunk = 64 (0 means 64) are required (else
 * SSM_ERR_UNSUPPORTED); every pointer must be 16-byte aligned except
 * igate, fgate, n_in/n_out and m_in/m_out, which need 4 bytes (else
 * SSM_ERR_ALIGNMENT); q, k, v, igate, fgate and h must be non-null
 * when B*H*T > 0, sizes non-negative, B*H below 2^31, scale finite and
 * norm_eps finite and non-negative (else SSM_ERR_INVALID_ARG); B*H*T must
 * stay below 2^31 - 128 token rows (else SSM_ERR_UNSUPPORTED: copies address
 * rows with 32-bit coordinates). C_in, n_in, m_in: all NULL for a zero state
 * with m = 0, or all non-null; C_out, n_out, m_out likewise (NULL skips the
 * final state). With T = 0 the final state is the initial one.
 *
 * Range: every exponential the kernel takes has an argument <= 0 (the
 * stabilizer is the running maximum), so no gate value overflows it; a
 * non-finite input or output is latched in the status word.
 *
 * Calls are asynchronous on `stream`; the caller owns every buffer;
 * workspace (nullable, >= 256 bytes) receives the status word read by
 * ssm_poll_status (non-finite outputs; SSM_ERR_TIMEOUT if a copy or a
 * tensor-core completion never arrived). Argument errors return a negative
 * SSM_ code before anything is launched.
 */
#ifndef MLSTM_H
#define MLSTM_H

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
    float norm_eps;
    const void* q;
    const void* k;
    const void* v;
    const float* igate;
    const float* fgate;
    const float* C_in;
    const float* n_in;
    const float* m_in;
    const float* norm_weight;
    void* h;
    float* C_out;
    float* n_out;
    float* m_out;
    void* workspace;
} mlstm_fwd_args;

int mlstm_chunk_fwd(const mlstm_fwd_args* args, void* stream);

/* One token of the cell (the recurrent step; decoding): with the state (C, n,
 * m) read and updated in place,
 *   m' = max(log sigmoid(fgate) + m, igate)
 *   C' = exp(log sigmoid(fgate) + m - m') C + exp(igate - m') k v^T,  n' likewise
 *   h  = (q^T C') / max(|q . n'|, exp(-m'))  (q scaled by `scale`), then the
 *        head-wise norm when norm_weight is non-null.
 * Layout: q, k [B, H, K] bf16; v [B, H, V] bf16; igate, fgate [B, H] fp32;
 * C [B, H, K, V], n [B, H, K], m [B, H] fp32 (stabilized, in place);
 * norm_weight [H, V] fp32 or NULL; h [B, H, V] bf16. Everything in fp32
 * (no tensor cores: one token is a matrix-vector step). K = V = 128 (else
 * SSM_ERR_UNSUPPORTED); q, k, v, C, norm_weight and h 16-byte aligned, the
 * gates, n and m 4-byte aligned (else SSM_ERR_ALIGNMENT); q, k, v, the
 * gates, C, n, m and h non-null when B*H > 0, B*H below 2^31, scale finite,
 * norm_eps finite and non-negative (else SSM_ERR_INVALID_ARG). A zero state
 * is C = n = 0 and m = 0. Asynchronous on `stream`; workspace (nullable)
 * receives the status word (non-finite outputs). */
typedef struct {
    int64_t B, H, K, V;
    float scale;
    float norm_eps;
    const void* q;
    const void* k;
    const void* v;
    const float* igate;
    const float* fgate;
    float* C;
    float* n;
    float* m;
    const float* norm_weight;
    void* h;
    void* workspace;
} mlstm_step_args;

int mlstm_step(const mlstm_step_args* args, void* stream);

/* Test hook: arms a one-shot fault for this thread's next mlstm_chunk_fwd.
 * The copy of q for chunk `chunk` (0-based, in every CTA) is not issued
 * while the chunk's other copies are, and every bounded wait of that call
 * gives up after wait_ns (0 keeps the 1 s default): the wait for the
 * missing copy runs out, each CTA waits for the copies it did issue, frees
 * its tensor memory and stops; ssm_poll_status then returns SSM_ERR_TIMEOUT
 * and the outputs are not valid. chunk < 0 disarms. SSM_ERR_INVALID_ARG for
 * wait_ns above 10 s. */
int mlstm_debug_arm_wait_fault(int64_t chunk, uint64_t wait_ns);

#ifdef __cplusplus
}
#endif
#endif /* MLSTM_H */
