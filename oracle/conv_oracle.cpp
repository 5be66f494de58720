// Oracle for the causal depthwise conv1d + SiLU in front of the S6 scan --
// TEST INFRASTRUCTURE ONLY (see ssm_oracle.cpp; same rules: the product path
// never loads it, and it shares no code with the GPU kernels).
//
// What it computes (rustytorch commit log, "MambaBlock" S6 forward commit:
// "in_proj -> causal depthwise conv1d -> SiLU -> x_proj -> ..."; the
// MambaRecurrence commit carries a "conv-ring" state between steps):
//
//   padded[p] = state[p]                  for p <  K-1   (state: the K-1 inputs before t = 0)
//             = xin[p - (K-1)]            for p >= K-1
//   pre[t]    = bias[d] + sum_k w[d,k] * padded[t + k]     (k = 0 .. K-1)
//   x[t]      = silu(pre[t]) = pre * sigmoid(pre)
//   state_out = the last K-1 entries of padded
//
// Backward, for loss = <dx, x>:
//   dpre[t]      = dx[t] * silu'(pre[t])
//   dpadded[p]   = sum over k with 0 <= p-k < L of w[d,k] * dpre[p-k]
//   dxin[s]      = dpadded[s + K-1];  dstate[j] = dpadded[j]
//   dw[d,k]      = sum over (b, t) of dpre[t] * padded[t+k];  dbias[d] = sum dpre
//
// Plain loops per (b, d) channel in t order and k order; nothing blocked or
// reordered. Double is the parity reference; float mirrors the pages' CPU
// f32 path.
#include <cmath>
#include <cstdint>
#include <vector>

namespace {

template <typename T> T c_sigmoid(T z) {
    if (z >= T(0)) return T(1) / (T(1) + std::exp(-z));
    T e = std::exp(z);
    return e / (T(1) + e);
}

struct ConvArgs {
    int64_t B, L, D, K;
    const void* xin;      // [B,L,D]
    const void* w;        // [D,K]
    const void* bias;     // [D] or null
    const void* state;    // [B,D,K-1] or null
    void* x;              // [B,L,D] out
    void* state_out;      // [B,D,K-1] out or null
    const void* dx;       // [B,L,D] (bwd)
    void* dxin;           // [B,L,D] (bwd out)
    void* dw;             // [D,K]   (bwd out)
    void* dbias;          // [D]     (bwd out, or null)
    void* dstate;         // [B,D,K-1] (bwd out, or null)
};

template <typename T> void padded_row(const ConvArgs* a, int64_t b, int64_t d, std::vector<T>& p) {
    const int64_t K = a->K, L = a->L, D = a->D;
    const T* xin = static_cast<const T*>(a->xin);
    const T* st = static_cast<const T*>(a->state);
    p.assign(L + K - 1, T(0));
    for (int64_t j = 0; j < K - 1; ++j) p[j] = st ? st[(b * D + d) * (K - 1) + j] : T(0);
    for (int64_t t = 0; t < L; ++t) p[K - 1 + t] = xin[(b * L + t) * D + d];
}

template <typename T> T pre_at(const ConvArgs* a, int64_t d, const std::vector<T>& p, int64_t t) {
    const T* w = static_cast<const T*>(a->w);
    const T* bias = static_cast<const T*>(a->bias);
    T s = bias ? bias[d] : T(0);
    for (int64_t k = 0; k < a->K; ++k) s = s + w[d * a->K + k] * p[t + k];
    return s;
}

template <typename T> int conv_fwd(const ConvArgs* a) {
    const int64_t B = a->B, L = a->L, D = a->D, K = a->K;
    if (K < 1) return -1;
    T* x = static_cast<T*>(a->x);
    T* so = static_cast<T*>(a->state_out);
    std::vector<T> p;
    for (int64_t b = 0; b < B; ++b)
        for (int64_t d = 0; d < D; ++d) {
            padded_row<T>(a, b, d, p);
            for (int64_t t = 0; t < L; ++t) {
                const T pre = pre_at<T>(a, d, p, t);
                x[(b * L + t) * D + d] = pre * c_sigmoid(pre);
            }
            if (so)
                for (int64_t j = 0; j < K - 1; ++j) so[(b * D + d) * (K - 1) + j] = p[L + j];
        }
    return 0;
}

template <typename T> int conv_bwd(const ConvArgs* a) {
    const int64_t B = a->B, L = a->L, D = a->D, K = a->K;
    if (K < 1) return -1;
    const T* w = static_cast<const T*>(a->w);
    const T* dx = static_cast<const T*>(a->dx);
    T* dxin = static_cast<T*>(a->dxin);
    T* dw = static_cast<T*>(a->dw);
    T* dbias = static_cast<T*>(a->dbias);
    T* dst = static_cast<T*>(a->dstate);
    for (int64_t i = 0; i < D * K; ++i) dw[i] = T(0);
    if (dbias)
        for (int64_t d = 0; d < D; ++d) dbias[d] = T(0);
    std::vector<T> p, dpre(L), dp;
    for (int64_t b = 0; b < B; ++b)
        for (int64_t d = 0; d < D; ++d) {
            padded_row<T>(a, b, d, p);
            for (int64_t t = 0; t < L; ++t) {
                const T pre = pre_at<T>(a, d, p, t);
                const T s = c_sigmoid(pre);
                dpre[t] = dx[(b * L + t) * D + d] * (s * (T(1) + pre * (T(1) - s)));
            }
            dp.assign(L + K - 1, T(0));
            for (int64_t q = 0; q < L + K - 1; ++q)
                for (int64_t k = 0; k < K; ++k) {
                    const int64_t t = q - k;
                    if (t >= 0 && t < L) dp[q] = dp[q] + w[d * K + k] * dpre[t];
                }
            for (int64_t t = 0; t < L; ++t) dxin[(b * L + t) * D + d] = dp[K - 1 + t];
            if (dst)
                for (int64_t j = 0; j < K - 1; ++j) dst[(b * D + d) * (K - 1) + j] = dp[j];
            for (int64_t k = 0; k < K; ++k) {
                T s = T(0);
                for (int64_t t = 0; t < L; ++t) s = s + dpre[t] * p[t + k];
                dw[d * K + k] = dw[d * K + k] + s;
            }
            if (dbias) {
                T s = T(0);
                for (int64_t t = 0; t < L; ++t) s = s + dpre[t];
                dbias[d] = dbias[d] + s;
            }
        }
    return 0;
}

}  // namespace

extern "C" {
int conv_oracle_fwd_f64(const ConvArgs* a) { return conv_fwd<double>(a); }
int conv_oracle_fwd_f32(const ConvArgs* a) { return conv_fwd<float>(a); }
int conv_oracle_bwd_f64(const ConvArgs* a) { return conv_bwd<double>(a); }
int conv_oracle_bwd_f32(const ConvArgs* a) { return conv_bwd<float>(a); }
}  // extern "C"
