// spec_estimator.cu -- one online step of the acceptance estimator
// ("Verificación Adaptativa sin una cabeza de confianza", "Ajuste de los
// Coeficientes"): the confidence of draft position i is
// sigmoid(omega * f_i + beta_{i+1}) with f_i = logit(q_max); only drafts up to
// and including the first rejection carry a label (1 before n_acc, 0 at
// n_acc < K). This kernel takes one gradient step of size lr on the mean
// log-loss of the batch's labels.
//
// One CTA; every sum runs in a fixed order (per-thread strided loop, then a
// fixed shuffle tree and a fixed cross-warp order), so the result is
// bit-reproducible. The work is O(B*K), negligible next to the logit pass.
#include <cuda_runtime.h>

#include <cstdint>

#include "spec_verify.h"

namespace sv_est {

constexpr int NT = 512;
constexpr int NWARP = NT / 32;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ int warp_sum_i(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// block sums of (a, n); results valid in thread 0
__device__ void block_sum(float &a, int &n, float *fs, int *is) {
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    a = warp_sum(a);
    n = warp_sum_i(n);
    if (l == 0) {
        fs[w] = a;
        is[w] = n;
    }
    __syncthreads();
    if (w == 0) {
        a = l < NWARP ? fs[l] : 0.f;
        n = l < NWARP ? is[l] : 0;
        a = warp_sum(a);
        n = warp_sum_i(n);
    }
    __syncthreads();
}

__global__ void __launch_bounds__(NT) estimator_kernel(int B, int K, const float *__restrict__ feature,
                                                       const int32_t *__restrict__ acc_len,
                                                       const int32_t *__restrict__ draft_len,
                                                       float *__restrict__ params, float lr,
                                                       float *__restrict__ grad_out,
                                                       int32_t *__restrict__ count_out) {
    __shared__ float fs[NWARP];
    __shared__ int is[NWARP];
    __shared__ float g_sh[1024 + 1];
    __shared__ int c_sh[1024 + 1];
    const int tid = threadIdx.x;
    const float omega = params[0];
    float gw = 0.f;
    int nw = 0;
    // position-major: the intercept gradients first, the slope's sum alongside
    for (int i = 0; i < K; ++i) {
        const float beta = params[1 + i];
        float gi = 0.f;
        int ni = 0;
        for (int b = tid; b < B; b += NT) {
            const int n = acc_len[b];
            const int kb = draft_len ? min(max(draft_len[b], 0), K) : K;
            if (i > n || i >= kb) continue;         // not labelled (or never verified)
            const float y = i < n ? 1.f : 0.f;
            const float f = feature[(size_t)b * K + i];
            const float e = 1.f / (1.f + expf(-(omega * f + beta))) - y;
            gi += e;
            ++ni;
            gw = fmaf(e, f, gw);
        }
        block_sum(gi, ni, fs, is);
        if (tid == 0) {
            g_sh[1 + i] = gi;
            c_sh[1 + i] = ni;
        }
    }
    nw = 0;
    block_sum(gw, nw, fs, is);
    if (tid == 0) {
        int N = 0;
        for (int i = 0; i < K; ++i) N += c_sh[1 + i];
        g_sh[0] = gw;
        c_sh[0] = N;
    }
    __syncthreads();
    const int N = c_sh[0];
    for (int k = tid; k <= K; k += NT) {
        const float g = N > 0 ? g_sh[k] / (float)N : 0.f;
        if (grad_out) grad_out[k] = g;
        if (count_out) count_out[k] = c_sh[k];
        if (N > 0) params[k] = params[k] - lr * g;
    }
}

// K <= kSmallK: every thread loads the K features of its sequences once and
// keeps the per-position partial sums in registers; one pass of reductions
// follows (a fixed shuffle tree per position, then the warps in order). The
// sums run in a fixed order, so the result is bit-reproducible; the general
// kernel above walks the positions one round at a time instead.
constexpr int kSmallK = 16;

__global__ void __launch_bounds__(NT) estimator_kernel_small(int B, int K, const float *__restrict__ feature,
                                                             const int32_t *__restrict__ acc_len,
                                                             const int32_t *__restrict__ draft_len,
                                                             float *__restrict__ params, float lr,
                                                             float *__restrict__ grad_out,
                                                             int32_t *__restrict__ count_out) {
    __shared__ float g_w[NWARP][kSmallK + 1];
    __shared__ int c_w[NWARP][kSmallK + 1];
    __shared__ int n_sh;
    const int tid = threadIdx.x, w = tid >> 5, l = tid & 31;
    const float omega = params[0];
    float gi[kSmallK], beta[kSmallK];
    int ni[kSmallK];
    float gw = 0.f;
#pragma unroll
    for (int i = 0; i < kSmallK; ++i) {
        gi[i] = 0.f;
        ni[i] = 0;
        beta[i] = i < K ? params[1 + i] : 0.f;
    }
    for (int b = tid; b < B; b += NT) {
        // every load of the sequence goes out before any of them is used
        float fv[kSmallK];
#pragma unroll
        for (int i = 0; i < kSmallK; ++i) fv[i] = i < K ? feature[(size_t)b * K + i] : 0.f;
        const int n = acc_len[b];
        const int kb = draft_len ? min(max(draft_len[b], 0), K) : K;
#pragma unroll
        for (int i = 0; i < kSmallK; ++i) {
            if (i >= K || i > n || i >= kb) continue;   // not labelled (or never verified)
            const float y = i < n ? 1.f : 0.f;
            const float f = fv[i];
            const float e = 1.f / (1.f + expf(-(omega * f + beta[i]))) - y;
            gi[i] += e;
            ++ni[i];
            gw = fmaf(e, f, gw);
        }
    }
#pragma unroll
    for (int i = 0; i < kSmallK; ++i) {
        if (i < K) {
            const float g = warp_sum(gi[i]);
            const int c = warp_sum_i(ni[i]);
            if (l == 0) {
                g_w[w][1 + i] = g;
                c_w[w][1 + i] = c;
            }
        }
    }
    gw = warp_sum(gw);
    if (l == 0) g_w[w][0] = gw;
    __syncthreads();
    // position k's totals over the warps in order (k = 0: the slope)
    float g = 0.f;
    int c = 0;
    if (tid <= K) {
        for (int q = 0; q < NWARP; ++q) {
            g += g_w[q][tid];
            if (tid > 0) c += c_w[q][tid];
        }
    }
    if (tid == 0) {
        int N = 0;
        for (int i = 1; i <= K; ++i) {
            int ci = 0;
            for (int q = 0; q < NWARP; ++q) ci += c_w[q][i];
            N += ci;
        }
        n_sh = N;
        c = N;
    }
    __syncthreads();
    const int N = n_sh;
    if (tid <= K) {
        const float gm = N > 0 ? g / (float)N : 0.f;
        if (grad_out) grad_out[tid] = gm;
        if (count_out) count_out[tid] = c;
        if (N > 0) params[tid] = params[tid] - lr * gm;
    }
}

}  // namespace sv_est

// defined in spec_verify.cu: sets the thread-local message read by spec_last_error
extern "C" int spec_internal_set_error(int code, const char *msg);

static int estimator_impl(int32_t B, int32_t K, const float *feature, const int32_t *accepted_len,
                          const int32_t *draft_len, float *est_params, float lr, float *grad_out,
                          int32_t *count_out, void *stream) {
    if (B < 0) return spec_internal_set_error(SPEC_ERR_INVALID_ARG, "B must be >= 0");
    if (K < 1 || K > 1024) return spec_internal_set_error(SPEC_ERR_UNSUPPORTED, "K must be in [1, 1024]");
    if (!est_params) return spec_internal_set_error(SPEC_ERR_INVALID_ARG, "est_params is NULL");
    if (B > 0 && (!feature || !accepted_len))
        return spec_internal_set_error(SPEC_ERR_INVALID_ARG, "feature / accepted_len is NULL");
    spec_internal_set_error(SPEC_OK, "");
    if (K <= sv_est::kSmallK)
        sv_est::estimator_kernel_small<<<1, sv_est::NT, 0, static_cast<cudaStream_t>(stream)>>>(
            B, K, feature, accepted_len, draft_len, est_params, lr, grad_out, count_out);
    else
        sv_est::estimator_kernel<<<1, sv_est::NT, 0, static_cast<cudaStream_t>(stream)>>>(
            B, K, feature, accepted_len, draft_len, est_params, lr, grad_out, count_out);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return spec_internal_set_error(SPEC_ERR_CUDA, cudaGetErrorString(e));
    return SPEC_OK;
}

extern "C" int spec_estimator_update(int32_t B, int32_t K, const float *feature, const int32_t *accepted_len,
                                     float *est_params, float lr, float *grad_out, int32_t *count_out,
                                     void *stream) {
    return estimator_impl(B, K, feature, accepted_len, nullptr, est_params, lr, grad_out, count_out, stream);
}

extern "C" int spec_estimator_update_ragged(int32_t B, int32_t K, const float *feature,
                                            const int32_t *accepted_len, const int32_t *draft_len,
                                            float *est_params, float lr, float *grad_out, int32_t *count_out,
                                            void *stream) {
    if (B > 0 && !draft_len) return spec_internal_set_error(SPEC_ERR_INVALID_ARG, "draft_len is NULL");
    return estimator_impl(B, K, feature, accepted_len, draft_len, est_params, lr, grad_out, count_out, stream);
}
