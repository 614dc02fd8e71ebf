// spec_ngram.cu -- n-gram (prompt-lookup) drafting ("Speculative Decoding: как
// черновая модель ускоряет генерацию LLM без потери качества", section
// "N-gram (prompt lookup)"; FLy's "Aceleração Multinível" drafts this way).
//
// The drafts are read from the context itself: the tokens that followed an
// earlier occurrence of the context's last n tokens. n runs from n_max down
// to n_min and the longest match wins; among its matches the most recent
// occurrence (the one that ends last, before the context does); up to K
// tokens that follow it are proposed.
//
// One warp per sequence. For a candidate end e (the occurrence is
// ctx[e-n .. e-1], the drafts start at ctx[e]) let m(e) be the number of
// tokens before e that agree with the context's final tokens, read
// backwards, capped at n_max. The rule above picks the lexicographic maximum
// of (m(e), e) over m(e) >= n_min: lanes sweep e from L-1 down, 256 at a
// time, and stop after the first block that holds a full-length (n_max)
// match, since no earlier e can beat it. Integer work only: exact.
#include <cuda_runtime.h>

#include <cstdint>

#include "spec_verify.h"

namespace sv_ngram {

constexpr int NT = 128;
constexpr int NWARP = NT / 32;
constexpr unsigned kFull = 0xffffffffu;

__global__ void __launch_bounds__(NT) ngram_kernel(int B, int ld, const int32_t *__restrict__ ctx,
                                                   const int32_t *__restrict__ len, int n_min, int n_max, int K,
                                                   int32_t *__restrict__ draft_tokens,
                                                   int32_t *__restrict__ draft_len) {
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.x * NWARP + (threadIdx.x >> 5);
    if (b >= B) return;
    const int32_t *c = ctx + (size_t)b * ld;
    const int L = min(max(len[b], 0), ld);
    int best_m = 0, best_e = -1;
    const int32_t last = L >= 1 ? __ldg(c + L - 1) : 0;
    // blocks of 32*kU candidates, all first-token loads of a block in flight
    // together; lane's candidates e = e0 - lane - 32u
    constexpr int kU = 8;
    for (int e0 = L - 1; e0 >= 1; e0 -= 32 * kU) {
        int32_t first[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int e = e0 - lane - 32 * u;
            first[u] = e >= 1 ? __ldg(c + e - 1) : 0;
        }
        bool full = false;
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int e = e0 - lane - 32 * u;
            int m = 0;
            if (e >= 1 && first[u] == last) {
                m = 1;
                while (m < n_max && m < e && __ldg(c + e - 1 - m) == __ldg(c + L - 1 - m)) ++m;
            }
            if (m >= n_min && (m > best_m || (m == best_m && e > best_e))) {
                best_m = m;
                best_e = e;
            }
            full |= m == n_max;
        }
        // a full-length match in this block cannot be beaten further down
        if (__any_sync(kFull, full)) break;
    }
    // lexicographic maximum of (m, e) over the warp
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const int om = __shfl_xor_sync(kFull, best_m, o);
        const int oe = __shfl_xor_sync(kFull, best_e, o);
        if (om > best_m || (om == best_m && oe > best_e)) {
            best_m = om;
            best_e = oe;
        }
    }
    const int start = best_e;   // -1: no match
    const int n = start >= 0 ? min(K, L - start) : 0;
    for (int k = lane; k < K; k += 32)
        draft_tokens[(size_t)b * K + k] = k < n ? __ldg(c + start + k) : -1;
    if (lane == 0) draft_len[b] = n;
}

}  // namespace sv_ngram

// defined in spec_verify.cu: sets the thread-local message read by spec_last_error
extern "C" int spec_internal_set_error(int code, const char *msg);

extern "C" int spec_ngram_draft(int32_t B, int32_t ld, const int32_t *ctx, const int32_t *len, int32_t n_min,
                                int32_t n_max, int32_t K, int32_t *draft_tokens, int32_t *draft_len, void *stream) {
    if (B < 0 || ld < 0) return spec_internal_set_error(SPEC_ERR_INVALID_ARG, "B and ld must be >= 0");
    if (K < 1) return spec_internal_set_error(SPEC_ERR_INVALID_ARG, "K must be >= 1");
    if (n_min < 1 || n_max < n_min) return spec_internal_set_error(SPEC_ERR_INVALID_ARG, "need 1 <= n_min <= n_max");
    if (B > 0 && (!ctx || !len || !draft_tokens || !draft_len))
        return spec_internal_set_error(SPEC_ERR_INVALID_ARG, "ctx / len / draft_tokens / draft_len is NULL");
    spec_internal_set_error(SPEC_OK, "");
    if (B == 0) return SPEC_OK;
    const int grid = (B + sv_ngram::NWARP - 1) / sv_ngram::NWARP;
    sv_ngram::ngram_kernel<<<grid, sv_ngram::NT, 0, static_cast<cudaStream_t>(stream)>>>(
        B, ld, ctx, len, n_min, n_max, K, draft_tokens, draft_len);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return spec_internal_set_error(SPEC_ERR_CUDA, cudaGetErrorString(e));
    return SPEC_OK;
}
