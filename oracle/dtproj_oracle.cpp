// Oracle for the dt projection in front of the S6 scan -- TEST
// INFRASTRUCTURE ONLY (same rules as ssm_oracle.cpp: the product path never
// loads it, and it shares no code with the GPU kernels).
//
// What it computes (rustytorch commit log, "MambaBlock" S6 forward commit:
// "delta=softplus(dt.dt_proj+dt_bias)", where dt is the first dt_rank
// columns of the x_proj output):
//
//   pre[m,d]   = bias[d] + sum_{r<R} a[m,r] * w[d,r]     (r ascending)
//   delta[m,d] = softplus(pre[m,d])                       (or pre itself when softplus is off)
//
// a [M,R] (M = batch * tokens), w [D,R] (the projection's weight, one row per
// output channel), bias [D] (nullable = 0). Backward, given dDelta [M,D]:
//
//   dpre[m,d] = dDelta[m,d] * sigmoid(pre[m,d])           (dDelta itself when softplus is off)
//   dbias[d]  = sum_m dpre[m,d]                           (m ascending)
//
// The GEMMs of the backward (dpre @ w, dpre^T @ a) are plain matrix
// products; the tests take them from numpy. Double is the parity reference.
#include <cmath>
#include <cstdint>

namespace {

// softplus(v) = max(v,0) + log1p(exp(-|v|))
template <typename T> T d_softplus(T v) { return (v > T(0) ? v : T(0)) + std::log1p(std::exp(-std::fabs(v))); }
// logistic sigmoid on the side where exp cannot overflow
template <typename T> T d_sigmoid(T z) {
    if (z >= T(0)) return T(1) / (T(1) + std::exp(-z));
    const T e = std::exp(z);
    return e / (T(1) + e);
}

struct DtProjArgs {
    int64_t M, D, R;
    int32_t softplus;
    int32_t pad_;
    const void* a;      // [M,R]
    const void* w;      // [D,R]
    const void* bias;   // [D] or null
    void* delta;        // [M,D] out (fwd)
    const void* ddelta; // [M,D] (bwd)
    void* dpre;         // [M,D] out (bwd)
    void* dbias;        // [D] out (bwd) or null
};

template <typename T> T pre_at(const DtProjArgs* p, int64_t m, int64_t d) {
    const T* a = static_cast<const T*>(p->a);
    const T* w = static_cast<const T*>(p->w);
    const T* bias = static_cast<const T*>(p->bias);
    T s = bias ? bias[d] : T(0);
    for (int64_t r = 0; r < p->R; ++r) s = s + a[m * p->R + r] * w[d * p->R + r];
    return s;
}

template <typename T> int fwd(const DtProjArgs* p) {
    if (p->M < 0 || p->D < 0 || p->R < 0) return -1;
    T* out = static_cast<T*>(p->delta);
    for (int64_t m = 0; m < p->M; ++m)
        for (int64_t d = 0; d < p->D; ++d) {
            const T v = pre_at<T>(p, m, d);
            out[m * p->D + d] = p->softplus ? d_softplus(v) : v;
        }
    return 0;
}

template <typename T> int bwd(const DtProjArgs* p) {
    if (p->M < 0 || p->D < 0 || p->R < 0) return -1;
    const T* g = static_cast<const T*>(p->ddelta);
    T* dpre = static_cast<T*>(p->dpre);
    T* dbias = static_cast<T*>(p->dbias);
    for (int64_t m = 0; m < p->M; ++m)
        for (int64_t d = 0; d < p->D; ++d) {
            const T gd = g[m * p->D + d];
            dpre[m * p->D + d] = p->softplus ? gd * d_sigmoid(pre_at<T>(p, m, d)) : gd;
        }
    if (dbias)
        for (int64_t d = 0; d < p->D; ++d) {
            T s = T(0);
            for (int64_t m = 0; m < p->M; ++m) s = s + dpre[m * p->D + d];
            dbias[d] = s;
        }
    return 0;
}

}  // namespace

extern "C" {
int dtproj_oracle_fwd_f64(const DtProjArgs* p) { return fwd<double>(p); }
int dtproj_oracle_fwd_f32(const DtProjArgs* p) { return fwd<float>(p); }
int dtproj_oracle_bwd_f64(const DtProjArgs* p) { return bwd<double>(p); }
int dtproj_oracle_bwd_f32(const DtProjArgs* p) { return bwd<float>(p); }
}  // extern "C"
