// spec_av.cu -- adaptive-verification (AV) pruning and budget ("Verificación
// Adaptativa sin una cabeza de confianza", "Antecedentes" and "Otras
// Características Consideradas").
//
// Before the target model runs, AV decides how many drafts of the batch to
// verify. Survival of draft i of sequence b is the running product of the
// acceptance confidences conf[b][0..i]; the drafts are ranked by survival over
// the whole batch; verifying the top k is expected to emit B + (sum of the top
// k survivals) tokens at a measured cost draft_cost[k] + verify_cost[k]; the
// budget is the k that maximises that ratio, and the top `budget` drafts are
// verified. Survival never grows along a sequence and ties rank by position,
// so each sequence's winners are a prefix of its drafts: draft_len[b] of them,
// which is what spec_verify_ragged takes.
//
// One CTA. Survival is an fp32 running product (the same precision ranks the
// drafts on every side); the ranking on (survival descending, flat index
// ascending) merges the B already-ranked per-sequence runs pairwise in
// shared memory, log2(B) rounds of merge path. The top-k sums are exact:
// each survival rounded to a multiple of 2^-32 and summed as 64-bit
// integers (a chunked scan, any order gives the same sums). The ratio is
// fp32 with every step correctly rounded: (float)(B*2^32 + S_k) divided by
// the fp32 cost, so the decision is reproducible bit for bit anywhere; the
// first maximum wins. (GB300's fp64 rate is a small fraction of fp32, and
// this kernel runs on one SM.)
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "spec_verify.h"

namespace sv_av {

constexpr int NT = 1024;
constexpr int NWARP = NT / 32;
constexpr int kMaxN = 16384;   // drafts per batch (B * K) one CTA ranks

// a ranks before b
__device__ __forceinline__ bool before(float ka, int ia, float kb, int ib) {
    return ka > kb || (ka == kb && ia < ib);
}

__device__ __forceinline__ unsigned long long warp_incl_scan_u64(unsigned long long v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
    }
    return v;
}

// survival s in (0, 1] in units of 2^-32, rounded to nearest (ties to even),
// with integer operations on the float's bits: s = m * 2^(e - 150) for the
// 24-bit significand m, so s * 2^32 = m * 2^(e - 118). Non-positive (and the
// NaN key -1) give 0; subnormals round to 0.
__device__ __forceinline__ unsigned long long fixed32(float s) {
    if (!(s > 0.f)) return 0ull;
    const unsigned bits = __float_as_uint(s);
    const int e = (int)(bits >> 23);
    if (e == 0) return 0ull;
    const unsigned long long m = (bits & 0x7fffffu) | 0x800000u;
    const int sh = e - 118;
    if (sh >= 0) return m << sh;
    if (sh < -25) return 0ull;                     // below half a unit
    const unsigned long long q = m >> -sh, rem = m & ((1ull << -sh) - 1), half = 1ull << (-sh - 1);
    return q + ((rem > half || (rem == half && (q & 1ull))) ? 1ull : 0ull);
}

__global__ void __launch_bounds__(NT) av_budget_kernel(int B, int K, const float *__restrict__ conf,
                                                       const float *__restrict__ draft_cost,
                                                       const float *__restrict__ verify_cost,
                                                       int32_t *__restrict__ draft_len, int32_t *__restrict__ budget,
                                                       float *__restrict__ survival, float *__restrict__ objective) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int N = B * K;
    // two (key, index) buffers for the merge rounds, then the reductions
    float *kbuf[2];
    unsigned short *ibuf[2];
    kbuf[0] = reinterpret_cast<float *>(smem);
    kbuf[1] = kbuf[0] + N;
    ibuf[0] = reinterpret_cast<unsigned short *>(kbuf[1] + N);
    ibuf[1] = ibuf[0] + N;
    unsigned long long *wtot =
        reinterpret_cast<unsigned long long *>(smem + (((size_t)N * 12 + 15) & ~(size_t)15));   // [NWARP]
    float *bestv = reinterpret_cast<float *>(wtot + NWARP);                                    // [NWARP]
    int *bestk = reinterpret_cast<int *>(bestv + NWARP);                                       // [NWARP]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    for (int b = tid; b < B; b += NT) draft_len[b] = 0;
    // survival: fp32 running product in ascending position (NaN ranks last).
    // Each sequence's run is already in rank order: survival never grows
    // along it and equal values rank by position.
    for (int b = tid; b < B; b += NT) {
        float sv = 1.f;
        for (int i = 0; i < K; ++i) {
            sv = __fmul_rn(sv, conf[(size_t)b * K + i]);
            if (survival) survival[(size_t)b * K + i] = sv;
            kbuf[0][b * K + i] = sv == sv ? sv : -1.f;
            ibuf[0][b * K + i] = (unsigned short)(b * K + i);
        }
    }
    __syncthreads();

    // merge the sorted runs pairwise (run length K, 2K, 4K, ...). Thread t
    // produces outputs [t*C, t*C + C) of each round: a co-rank binary search
    // (merge path) places its first output, then it merges sequentially.
    const int C = (N + NT - 1) / NT;
    int src = 0;
    for (int L = K; L < N; L <<= 1, src ^= 1) {
        const float *ka = kbuf[src];
        const unsigned short *ia = ibuf[src];
        float *kd = kbuf[src ^ 1];
        unsigned short *id = ibuf[src ^ 1];
        int o = tid * C;
        const int oend = min(o + C, N);
        while (o < oend) {
            const int base = (o / (2 * L)) * (2 * L);
            const int LA = min(L, N - base);
            const int LB = min(L, N - base - LA);
            const float *A = ka + base, *Bk = ka + base + LA;
            const unsigned short *Ai = ia + base, *Bi = ia + base + LA;
            const int q0 = o - base;
            const int q1 = min(oend - base, LA + LB);
            int lo = max(0, q0 - LB), hi = min(q0, LA);
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                const int jb = q0 - mid - 1;
                if (before(A[mid], Ai[mid], Bk[jb], Bi[jb])) lo = mid + 1;
                else hi = mid;
            }
            int i = lo, j = q0 - lo;
            for (int q = q0; q < q1; ++q) {
                const bool takeA = i < LA && (j >= LB || before(A[i], Ai[i], Bk[j], Bi[j]));
                kd[base + q] = takeA ? A[i] : Bk[j];
                id[base + q] = takeA ? Ai[i] : Bi[j];
                if (takeA) ++i;
                else ++j;
            }
            o = base + q1;
        }
        __syncthreads();
    }
    const float *key = kbuf[src];
    const unsigned short *idx = ibuf[src];

    // S_k = sum of the top k survivals (units of 2^-32): thread t owns ranks
    // [t*C, t*C + C)
    const int r0 = tid * C;
    unsigned long long own = 0ull;
    for (int r = r0; r < r0 + C && r < N; ++r) own += fixed32(key[r]);
    const unsigned long long wincl = warp_incl_scan_u64(own, lane);
    if (lane == 31) wtot[warp] = wincl;
    __syncthreads();
    if (warp == 0) {
        const unsigned long long v = lane < NWARP ? wtot[lane] : 0ull;
        const unsigned long long t = warp_incl_scan_u64(v, lane);
        __syncwarp();
        if (lane < NWARP) wtot[lane] = t - v;   // exclusive warp offsets
    }
    __syncthreads();
    unsigned long long S = wtot[warp] + wincl - own;   // the ranks before r0
    // objective_k = (float)(B*2^32 + S_k) / (draft_cost[k] + verify_cost[k])
    // for k = 0..N (thread t takes k = r + 1 for its ranks r, thread 0 also
    // k = 0); every step is correctly rounded
    const unsigned long long base = (unsigned long long)B << 32;
    float bv = -INFINITY;
    int bk = 0x7fffffff;
    auto consider = [&](int k, unsigned long long Sk) {
        const float c = __fadd_rn(draft_cost[k], verify_cost[k]);
        const float o = c > 0.f ? __fmul_rn(__fdiv_rn(__ull2float_rn(base + Sk), c), 0x1p-32f) : -INFINITY;
        if (objective) objective[k] = o;
        if (o > bv) {   // ascending k: the first maximum stays
            bv = o;
            bk = k;
        }
    };
    if (tid == 0) consider(0, 0ull);
    for (int r = r0; r < r0 + C && r < N; ++r) {
        S += fixed32(key[r]);
        consider(r + 1, S);
    }
    // first maximum over the block: larger value, then smaller k
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int ok = __shfl_xor_sync(0xffffffffu, bk, o);
        if (ov > bv || (ov == bv && ok < bk)) {
            bv = ov;
            bk = ok;
        }
    }
    if (lane == 0) {
        bestv[warp] = bv;
        bestk[warp] = bk;
    }
    __syncthreads();
    if (warp == 0) {
        float v = lane < NWARP ? bestv[lane] : -INFINITY;
        int kk = lane < NWARP ? bestk[lane] : 0x7fffffff;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, v, o);
            const int ok = __shfl_xor_sync(0xffffffffu, kk, o);
            if (ov > v || (ov == v && ok < kk)) {
                v = ov;
                kk = ok;
            }
        }
        if (lane == 0) bestk[0] = v > -INFINITY ? kk : 0;
    }
    __syncthreads();
    const int bud = bestk[0];
    if (tid == 0) *budget = bud;
    // the winners: each sequence's count (its winners are a prefix)
    for (int r = tid; r < bud; r += NT) atomicAdd(draft_len + idx[r] / K, 1);
}

}  // namespace sv_av

// defined in spec_verify.cu: sets the thread-local message read by spec_last_error
extern "C" int spec_internal_set_error(int code, const char *msg);

extern "C" int spec_av_budget(int32_t B, int32_t K, const float *conf, const float *draft_cost,
                              const float *verify_cost, int32_t *draft_len, int32_t *budget, float *survival,
                              float *objective, void *stream) {
    if (B < 1 || K < 1) return spec_internal_set_error(SPEC_ERR_INVALID_ARG, "B and K must be >= 1");
    if ((int64_t)B * K > sv_av::kMaxN)
        return spec_internal_set_error(SPEC_ERR_UNSUPPORTED, "B * K must be <= 16384");
    if (!conf || !draft_cost || !verify_cost || !draft_len || !budget)
        return spec_internal_set_error(SPEC_ERR_INVALID_ARG, "conf / cost tables / draft_len / budget is NULL");
    const size_t N = (size_t)B * K;
    const size_t smem = ((N * 12 + 15) & ~(size_t)15) + sv_av::NWARP * (8 + 4 + 4);
    // the largest dynamic shared size, set once per device
    static std::mutex mu;
    static bool done[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return spec_internal_set_error(SPEC_ERR_CUDA, cudaGetErrorString(e));
    {
        std::lock_guard<std::mutex> lk(mu);
        if (!done[dev & 63]) {
            e = cudaFuncSetAttribute(sv_av::av_budget_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)((size_t)sv_av::kMaxN * 12 + sv_av::NWARP * (8 + 4 + 4)));
            if (e != cudaSuccess) return spec_internal_set_error(SPEC_ERR_CUDA, cudaGetErrorString(e));
            done[dev & 63] = true;
        }
    }
    spec_internal_set_error(SPEC_OK, "");
    sv_av::av_budget_kernel<<<1, sv_av::NT, smem, static_cast<cudaStream_t>(stream)>>>(
        B, K, conf, draft_cost, verify_cost, draft_len, budget, survival, objective);
    e = cudaGetLastError();
    if (e != cudaSuccess) return spec_internal_set_error(SPEC_ERR_CUDA, cudaGetErrorString(e));
    return SPEC_OK;
}
