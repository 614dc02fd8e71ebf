// spec_irls.cu -- IRLS refit of the acceptance estimator ("Verificación
// Adaptativa sin una cabeza de confianza", "Ajuste de los Coeficientes").
//
// The coefficients theta = (omega, beta_1..beta_K) stay fixed over a round of
// decoding steps. Every step adds the gradient g and Hessian H of the summed
// log-loss of its eligible labels to the round's state; the refit at the end
// of the round solves H d = g and moves each coefficient by d damped by
// n / (n + c), n being the labels behind it.
//
// With one shared slope and an intercept per draft position, H is an arrow
// matrix: the slope row and column plus a diagonal (a label touches the
// slope and exactly one intercept). So the state is O(K) and the solve is a
// Schur complement on the slope, O(K), in fp64:
//   s   = H_ww - sum_k H_wk^2 / H_kk
//   d_w = (g_w - sum_k H_wk g_k / H_kk) / s
//   d_k = (g_k - H_wk d_w) / H_kk
//
// Both kernels are a single CTA with every sum in a fixed order, so results
// are bit-reproducible. Per label the sigmoid terms are fp32 (GB300's fp64
// rate is a small fraction of its fp32 rate, and one CTA runs on one SM);
// every sum across lanes, positions and steps, and the solve, are fp64.
#include <cuda_runtime.h>

#include <cstdint>

#include "spec_verify.h"

namespace sv_irls {

constexpr int NT = 512;
constexpr int NWARP = NT / 32;
constexpr int kMaxK = 1024;

// state layout, in doubles (spec_verify.h documents it for callers)
__host__ __device__ constexpr int off_g(int) { return 0; }
__host__ __device__ constexpr int off_hww(int K) { return K + 1; }
__host__ __device__ constexpr int off_hwb(int K) { return K + 2; }
__host__ __device__ constexpr int off_hbb(int K) { return 2 * K + 2; }
__host__ __device__ constexpr int off_n(int K) { return 3 * K + 2; }
__host__ __device__ constexpr int state_doubles(int K) { return 4 * K + 3; }

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// sigma(z) and sigma(-z) without cancellation: both from t = exp(-|z|)
__device__ __forceinline__ void sigmoid_pair(float z, float &s, float &sn) {
    const float t = expf(-fabsf(z));
    const float a = 1.f / (1.f + t);   // sigma(|z|)
    const float b = t * a;             // sigma(-|z|)
    s = z >= 0.f ? a : b;
    sn = z >= 0.f ? b : a;
}

// One decoding step of a round. Warp w takes draft positions w, w + NWARP, ...;
// its lanes visit sequences b = lane, lane + 32, ... in ascending order, in
// batches of 8: fp32 terms and batch sums, fp64 lane sums across batches
// (the fp32 error is bounded by 8 terms whatever B is), then an fp32
// butterfly merges the lanes. Then one thread per state entry adds this step
// to it in fp64; the slope's three entries sum the positions in ascending
// order. fp64 work stays a few operations per lane: GB300's fp64 rate is a
// small fraction of its fp32 rate.
__global__ void __launch_bounds__(NT) irls_accumulate_kernel(int B, int K, const float *__restrict__ feature,
                                                            const int32_t *__restrict__ acc_len,
                                                            const int32_t *__restrict__ draft_len,
                                                            const float *__restrict__ params,
                                                            double *__restrict__ state) {
    // per position: sum e, sum w, sum w f, count; and the slope's sum e f, sum w f^2
    __shared__ double sh[kMaxK][6];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float omega = params[0];
    for (int i = warp; i < K; i += NWARP) {
        const float beta = params[1 + i];
        double se = 0.0, sw = 0.0, swf = 0.0, sef = 0.0, swff = 0.0, cnt = 0.0;
        constexpr int kBatch = 8;                // loads of 8 sequences in flight per lane
        for (int b0 = lane; b0 < B; b0 += 32 * kBatch) {
            int nb[kBatch];
            float fb[kBatch];
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                const int b = b0 + 32 * j;
                nb[j] = b < B ? acc_len[b] : -1;
                fb[j] = b < B ? feature[(size_t)b * K + i] : 0.f;
                // a draft at or past the verified length carries no label
                if (draft_len && b < B && i >= min(max(draft_len[b], 0), K)) nb[j] = -1;
            }
            float be = 0.f, bw = 0.f, bwf = 0.f, bef = 0.f, bwff = 0.f, bc = 0.f;
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                if (i > nb[j]) continue;         // no label at this position (i < K)
                const float f = fb[j];
                float s, sn;
                sigmoid_pair(fmaf(omega, f, beta), s, sn);
                const float e = i < nb[j] ? -sn : s;   // sigma(z) - y
                const float w = s * sn;
                const float wf = w * f;
                be += e;
                bef = fmaf(e, f, bef);
                bw += w;
                bwf += wf;
                bwff = fmaf(wf, f, bwff);
                bc += 1.f;
            }
            se += (double)be;
            sef += (double)bef;
            sw += (double)bw;
            swf += (double)bwf;
            swff += (double)bwff;
            cnt += (double)bc;
        }
        const float le = warp_sum_f((float)se), lw = warp_sum_f((float)sw), lwf = warp_sum_f((float)swf);
        const float lef = warp_sum_f((float)sef), lwff = warp_sum_f((float)swff);
        const double lc = warp_sum_d(cnt);       // exact count
        if (lane == 0) {
            sh[i][0] = (double)le;
            sh[i][1] = (double)lw;
            sh[i][2] = (double)lwf;
            sh[i][3] = lc;
            sh[i][4] = (double)lef;
            sh[i][5] = (double)lwff;
        }
    }
    __syncthreads();
    for (int j = threadIdx.x; j < state_doubles(K); j += NT) {
        double v;
        if (j == off_g(K) || j == off_hww(K) || j == off_n(K)) {
            const int c = j == off_g(K) ? 4 : (j == off_hww(K) ? 5 : 3);
            v = 0.0;
            for (int i = 0; i < K; ++i) v += sh[i][c];
        } else if (j < off_hww(K)) {
            v = sh[j - off_g(K) - 1][0];
        } else if (j < off_hbb(K)) {
            v = sh[j - off_hwb(K)][2];
        } else if (j < off_n(K)) {
            v = sh[j - off_hbb(K)][1];
        } else {
            v = sh[j - off_n(K) - 1][3];
        }
        state[j] += v;
    }
}

// End of a round: the arrow solve, damping, the update of the fp32
// parameters, the applied step (optional), and a zeroed state for the next
// round. One warp: lane l takes coefficients l, l + 32, ...; the two sums of
// the Schur complement are lane sums in ascending k, then a butterfly.
__global__ void irls_refit_kernel(int K, double *__restrict__ state, float *__restrict__ params, double damping,
                                  double *__restrict__ step_out) {
    const int lane = threadIdx.x & 31;
    const double *g = state + off_g(K);
    const double *hwb = state + off_hwb(K);
    const double *hbb = state + off_hbb(K);
    const double *n = state + off_n(K);
    const double hww = state[off_hww(K)];
    const double n0 = n[0];
    // intercepts with labels and a positive curvature take part; the rest hold
    double t1 = 0.0, t2 = 0.0;
    for (int k = lane; k < K; k += 32) {
        if (n[1 + k] > 0.0 && hbb[k] > 0.0) {
            const double r = hwb[k] * (1.0 / hbb[k]);
            t1 += r * hwb[k];
            t2 += r * g[1 + k];
        }
    }
    t1 = warp_sum_d(t1);
    t2 = warp_sum_d(t2);
    const double sc = hww - t1;
    // the slope is held when this round does not determine it
    const double dw = (n0 > 0.0 && sc > 1e-12 * hww) ? (g[0] - t2) / sc : 0.0;
    if (lane == 0) {
        const double stepw = n0 > 0.0 ? dw * (n0 / (n0 + damping)) : 0.0;
        params[0] = (float)((double)params[0] - stepw);
        if (step_out) step_out[0] = stepw;
    }
    for (int k = lane; k < K; k += 32) {
        const double nk = n[1 + k];
        const double dk = (nk > 0.0 && hbb[k] > 0.0) ? (g[1 + k] - hwb[k] * dw) * (1.0 / hbb[k]) : 0.0;
        const double step = nk > 0.0 ? dk * (nk / (nk + damping)) : 0.0;
        params[1 + k] = (float)((double)params[1 + k] - step);
        if (step_out) step_out[1 + k] = step;
    }
    __syncwarp();
    for (int j = lane; j < state_doubles(K); j += 32) state[j] = 0.0;
}

}  // namespace sv_irls

// defined in spec_verify.cu: sets the thread-local message read by spec_last_error
extern "C" int spec_internal_set_error(int code, const char *msg);

namespace {

int irls_check_k(int32_t K) {
    if (K < 1 || K > sv_irls::kMaxK) return spec_internal_set_error(SPEC_ERR_UNSUPPORTED, "K must be in [1, 1024]");
    return SPEC_OK;
}

int launched() {
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return spec_internal_set_error(SPEC_ERR_CUDA, cudaGetErrorString(e));
    return SPEC_OK;
}

}  // namespace

extern "C" {

size_t spec_irls_state_size(int32_t K) {
    if (K < 1 || K > sv_irls::kMaxK) return 0;
    return (size_t)sv_irls::state_doubles(K) * sizeof(double);
}

int spec_irls_reset(int32_t K, void *state, void *stream) {
    int rc = irls_check_k(K);
    if (rc != SPEC_OK) return rc;
    if (!state) return spec_internal_set_error(SPEC_ERR_INVALID_ARG, "state is NULL");
    spec_internal_set_error(SPEC_OK, "");
    const cudaError_t e = cudaMemsetAsync(state, 0, spec_irls_state_size(K), static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return spec_internal_set_error(SPEC_ERR_CUDA, cudaGetErrorString(e));
    return SPEC_OK;
}

}  // extern "C"

static int irls_accumulate_impl(int32_t B, int32_t K, const float *feature, const int32_t *accepted_len,
                                const int32_t *draft_len, const float *est_params, void *state, void *stream) {
    if (B < 0) return spec_internal_set_error(SPEC_ERR_INVALID_ARG, "B must be >= 0");
    int rc = irls_check_k(K);
    if (rc != SPEC_OK) return rc;
    if (!est_params || !state) return spec_internal_set_error(SPEC_ERR_INVALID_ARG, "est_params / state is NULL");
    if (B > 0 && (!feature || !accepted_len))
        return spec_internal_set_error(SPEC_ERR_INVALID_ARG, "feature / accepted_len is NULL");
    if ((reinterpret_cast<uintptr_t>(state) & 7u) != 0)
        return spec_internal_set_error(SPEC_ERR_INVALID_ARG, "state must be 8-byte aligned");
    spec_internal_set_error(SPEC_OK, "");
    sv_irls::irls_accumulate_kernel<<<1, sv_irls::NT, 0, static_cast<cudaStream_t>(stream)>>>(
        B, K, feature, accepted_len, draft_len, est_params, static_cast<double *>(state));
    return launched();
}

extern "C" {

int spec_irls_accumulate(int32_t B, int32_t K, const float *feature, const int32_t *accepted_len,
                         const float *est_params, void *state, void *stream) {
    return irls_accumulate_impl(B, K, feature, accepted_len, nullptr, est_params, state, stream);
}

int spec_irls_accumulate_ragged(int32_t B, int32_t K, const float *feature, const int32_t *accepted_len,
                                const int32_t *draft_len, const float *est_params, void *state, void *stream) {
    if (B > 0 && !draft_len) return spec_internal_set_error(SPEC_ERR_INVALID_ARG, "draft_len is NULL");
    return irls_accumulate_impl(B, K, feature, accepted_len, draft_len, est_params, state, stream);
}

int spec_irls_refit(int32_t K, void *state, float *est_params, double damping, double *step_out, void *stream) {
    int rc = irls_check_k(K);
    if (rc != SPEC_OK) return rc;
    if (!est_params || !state) return spec_internal_set_error(SPEC_ERR_INVALID_ARG, "est_params / state is NULL");
    if (!(damping >= 0.0) || !(damping < 1e300))
        return spec_internal_set_error(SPEC_ERR_INVALID_ARG, "damping must be finite and >= 0");
    if ((reinterpret_cast<uintptr_t>(state) & 7u) != 0)
        return spec_internal_set_error(SPEC_ERR_INVALID_ARG, "state must be 8-byte aligned");
    spec_internal_set_error(SPEC_OK, "");
    sv_irls::irls_refit_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        K, static_cast<double *>(state), est_params, damping, step_out);
    return launched();
}

}  // extern "C"
