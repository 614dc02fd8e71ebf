// spec_verify.cu -- fused verification pass for GB300 (sm_103a) and its C ABI.
//
// One persistent kernel does the whole pass ("Speculative Decoding: как
// черновая модель ускоряет генерацию LLM без потери качества", "Алгоритм на
// каждом шаге", steps 3-4):
//
//  * Work is a queue of stream units (sequence b, row r, vocabulary tile t),
//    ordered sequence-major and claimed with one atomic each, so that a
//    sequence's rows are read close together in time. Every unit streams its
//    tile from HBM exactly once with 128-bit non-allocating loads and folds it
//    into an online softmax accumulator (max, complement mass, entropy moment,
//    argmax); the CTA's partial goes to the workspace.
//  * The CTA that completes the last unit of sequence b (atomic counter, no
//    waiting) finalises b: merges the partials of each row, applies the
//    verification rule of the call's mode, computes the per-position
//    statistics and confidences, and, in stochastic mode, draws the residual
//    or bonus token by inverse CDF, re-reading at most two rows of b while
//    they are still resident in L2.
//
// Nothing in the kernel waits on another CTA, so it cannot deadlock whatever
// the number of resident CTAs. All reductions run in a fixed order.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include "spec_device.cuh"
#include "spec_verify.h"

namespace sv {

constexpr int NT = 256;              // threads per CTA
constexpr int NWARP = NT / 32;
constexpr int kUnroll = 4;           // 16-byte loads in flight per thread
constexpr int kResBlk = NT * 8;      // elements per block of the residual scan
constexpr int kMaxRows = 2 * SPEC_MAX_K + 1;

enum { MODE_STOCHASTIC = 0, MODE_GREEDY = 1, MODE_FLY = 2, MODE_CONF = 3 };

// workspace header (zeroed before every launch)
enum { CTR_CLAIM = 0, CTR_STATUS = 1, kHeaderWords = 16 };

struct Args {
    const void *zt;
    const void *zd;
    long long ts;            // target row stride (elements)
    long long ds;            // draft row stride (elements)
    const int32_t *x;
    const float *u;
    const float *est;
    int32_t *out_tokens;
    int32_t *acc_len;
    float *pos_stats;
    float *feature;
    float *conf;
    int B, K, V, mode;
    float theta;
    int W;
    int nt_rows;             // target rows streamed per sequence (K+1 or 0)
    int nd_rows;             // draft rows streamed per sequence (K or 0)
    int rows;
    int nT;                  // tiles per row
    int TS;                  // tile size (elements, multiple of 8)
    unsigned units;          // B * rows * nT
    int t_vec_ok, d_vec_ok;  // rows start on 16-byte boundaries
    float inv_log_v;         // 1 / ln V
    unsigned *ctr;           // header words
    unsigned *seq_done;      // [B] completed units per sequence
    float4 *part;            // [B][rows][nT] tile partials
};

struct FinSmem {
    float M[kMaxRows + 1];
    float R[kMaxRows + 1];
    float T[kMaxRows + 1];
    int I[kMaxRows + 1];
    float lse_t, lse_d;
    double P, target;
    int n, token, entry, retry;
};

__device__ __forceinline__ void raise_status(const Args &a, unsigned code) {
    atomicMax(a.ctr + CTR_STATUS, code);
}

template <typename T>
__device__ __forceinline__ const T *trow_ptr(const Args &a, int b, int j) {
    return static_cast<const T *>(a.zt) + ((long long)b * (a.K + 1) + j) * a.ts;
}

template <typename T>
__device__ __forceinline__ const T *drow_ptr(const Args &a, int b, int i) {
    return static_cast<const T *>(a.zd) + ((long long)b * a.K + i) * a.ds;
}

// ---------------------------------------------------------------------------
// Stream one tile [v0, v1) of a row: per-thread accumulators, ascending index
// order inside each thread (head scalars, 16-byte vectors, tail scalars).
// ---------------------------------------------------------------------------
template <typename T>
__device__ __forceinline__ RowAcc tile_acc(const T *row, int v0, int v1) {
    constexpr int E = Elem<T>::kPerVec;
    const int tid = threadIdx.x;
    RowAcc s = acc_empty();
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(row + v0);
    int head = (int)(((16u - (unsigned)(a0 & 15u)) & 15u) / sizeof(T));
    if (head > v1 - v0) head = v1 - v0;
    const int vb = v0 + head;
    const int nvec = (v1 - vb) / E;
    const int ve = vb + nvec * E;
    const int tail = v1 - ve;
    if (tid < head) {
        float z[1] = {Elem<T>::load(row + v0 + tid)};
        acc_chunk<1>(s, z, v0 + tid);
    }
    const uint4 *vp = reinterpret_cast<const uint4 *>(row + vb);
    int k = tid;
    for (; k + (kUnroll - 1) * NT < nvec; k += kUnroll * NT) {
        uint4 w[kUnroll];
#pragma unroll
        for (int q = 0; q < kUnroll; ++q) w[q] = ldg_stream(vp + k + q * NT);
#pragma unroll
        for (int q = 0; q < kUnroll; ++q) {
            float z[E];
            Elem<T>::unpack(w[q], z);
            acc_chunk<E>(s, z, vb + (k + q * NT) * E);
        }
    }
    for (; k < nvec; k += NT) {
        float z[E];
        Elem<T>::unpack(ldg_stream(vp + k), z);
        acc_chunk<E>(s, z, vb + k * E);
    }
    if (tid < tail) {
        float z[1] = {Elem<T>::load(row + ve + tid)};
        acc_chunk<1>(s, z, ve + tid);
    }
    return s;
}

// Block-wide merge; the result is valid in every lane of warp 0.
__device__ __forceinline__ RowAcc block_merge(RowAcc s, float4 *red) {
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    s = warp_merge(s);
    if (l == 0) red[w] = acc_pack(s);
    __syncthreads();
    if (w == 0) {
        RowAcc t = l < NWARP ? acc_unpack(red[l]) : acc_empty();
        s = warp_merge(t);
    }
    return s;
}

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ double warp_incl_scan_d(double v) {
    const int l = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double t = __shfl_up_sync(0xffffffffu, v, o);
        if (l >= o) v += t;
    }
    return v;
}

// r_v = max(0, p_v - q_v) (or p_v without a draft row) for v..v+7, fp32.
template <typename T>
__device__ __forceinline__ void resid8(const T *trow, const T *drow, int v, int V, bool tv, bool dv,
                                       float lse_t, float lse_d, float (&r)[8]) {
    float zt[8];
    load8<T>(trow, v, V, tv, zt);
    if (drow) {
        float zd[8];
        load8<T>(drow, v, V, dv, zd);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float p = ex2((zt[j] - lse_t) * kLog2e);
            const float q = ex2((zd[j] - lse_d) * kLog2e);
            r[j] = fmaxf(p - q, 0.f);
        }
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) r[j] = ex2((zt[j] - lse_t) * kLog2e);
    }
}

__device__ __forceinline__ float sum8(const float (&r)[8]) {
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) s += r[j];
    return s;
}

// ---------------------------------------------------------------------------
// Inverse-CDF draw from norm(max(0, p - q)) (q absent: from p) with uniform u:
// the smallest v whose running sum (ascending v) exceeds u * Z
// ("Математика верификации"). Pass 1 (all warps) sums each warp's 256-element
// slice of every 2048-element block in fp32; warp 0 scans the slice totals in
// fp64, picks the slice holding u*Z and scans it lane by lane (fp64 prefix).
// If the residual mass is zero (only possible through rounding) the draw falls
// back to p. Returns the token (valid in every thread).
// ---------------------------------------------------------------------------
template <typename T>
__device__ int residual_draw(const Args &a, const T *trow, const T *drow, float lse_t, float lse_d,
                             float u, float *wsum, FinSmem &sm) {
    const int tid = threadIdx.x, w = tid >> 5, l = tid & 31;
    const int V = a.V;
    const int nblk = (V + kResBlk - 1) / kResBlk;
    const bool tv = a.t_vec_ok != 0, dv = a.d_vec_ok != 0;
    const T *dr = drow;
    bool ok = false;
    for (int attempt = 0; attempt < 2 && !ok; ++attempt) {
        if (attempt == 1) dr = nullptr;        // Z == 0: draw from p
        for (int k = 0; k < nblk; ++k) {
            float r[8];
            resid8<T>(trow, dr, k * kResBlk + tid * 8, V, tv, dv, lse_t, lse_d, r);
            const float s = warp_sum_f(sum8(r));
            if (l == 0) wsum[k * NWARP + w] = s;
        }
        __syncthreads();
        if (w == 0) {
            const int ne = nblk * NWARP;
            const int per = (ne + 31) / 32;
            const int e0 = min(ne, l * per), e1 = min(ne, e0 + per);
            double seg = 0.0;
            for (int e = e0; e < e1; ++e) seg += (double)wsum[e];
            const double incl = warp_incl_scan_d(seg);
            double excl = __shfl_up_sync(0xffffffffu, incl, 1);
            if (l == 0) excl = 0.0;
            const double Z = __shfl_sync(0xffffffffu, incl, 31);
            const double target = (double)u * Z;
            int found = -1;
            double P = 0.0, c = excl;
            for (int e = e0; e < e1; ++e) {
                const double prev = c;
                c += (double)wsum[e];
                if (c > target) {
                    found = e;
                    P = prev;
                    break;
                }
            }
            const unsigned m = __ballot_sync(0xffffffffu, found >= 0);
            int entry = -1;
            double Pe = 0.0;
            if (m) {
                const int L = __ffs(m) - 1;
                entry = __shfl_sync(0xffffffffu, found, L);
                Pe = __shfl_sync(0xffffffffu, P, L);
            } else {
                // rounding left u*Z at the total: the last slice with mass
                int last = -1;
                for (int e = e0; e < e1; ++e)
                    if (wsum[e] > 0.f) last = e;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
                entry = last;
                Pe = Z;   // nothing in the slice exceeds target: take its last mass
            }
            if (l == 0) {
                sm.retry = (Z > 0.0 && entry >= 0) ? 0 : 1;
                sm.entry = entry;
                sm.P = Pe;
                sm.target = target;
            }
        }
        __syncthreads();
        ok = sm.retry == 0;
        __syncthreads();
    }
    if (!ok) {
        if (tid == 0) raise_status(a, SPEC_ERR_BAD_ROW);
        return 0;
    }
    if (w == 0) {
        const int entry = sm.entry;
        const int v = (entry / NWARP) * kResBlk + (entry % NWARP) * 256 + l * 8;
        float r[8];
        resid8<T>(trow, dr, v, V, tv, dv, lse_t, lse_d, r);
        const float s = sum8(r);               // the same fp32 value pass 1 summed
        const double incl = warp_incl_scan_d((double)s);
        double excl = __shfl_up_sync(0xffffffffu, incl, 1);
        if (l == 0) excl = 0.0;
        const double P = sm.P, target = sm.target;
        const unsigned m = __ballot_sync(0xffffffffu, P + incl > target);
        int L;
        if (m) {
            L = __ffs(m) - 1;
        } else {
            const unsigned nz = __ballot_sync(0xffffffffu, s > 0.f);
            L = nz ? 31 - __clz(nz) : 0;
        }
        if (l == L) {
            int tok = -1, lastpos = -1;
            double c = P + excl;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (r[j] > 0.f) lastpos = j;
                c += (double)r[j];
                if (tok < 0 && c > target) tok = j;
            }
            if (tok < 0) tok = lastpos >= 0 ? lastpos : 0;
            sm.token = v + tok;
        }
    }
    __syncthreads();
    return sm.token;
}

// ---------------------------------------------------------------------------
// Finalise sequence b (whole CTA): merge tile partials per row, decide, write.
// ---------------------------------------------------------------------------
template <typename T>
__device__ void finalize(const Args &a, int b, FinSmem &sm, float *wsum) {
    const int tid = threadIdx.x, w = tid >> 5, l = tid & 31;
    const int K = a.K;
    for (int r = w; r < a.rows; r += NWARP) {
        const float4 *pp = a.part + ((size_t)b * a.rows + r) * a.nT;
        RowAcc s = acc_empty();
        for (int t = l; t < a.nT; t += 32) s = acc_merge(s, acc_unpack(__ldcg(pp + t)));
        s = warp_merge(s);
        if (l == 0) {
            sm.M[r] = s.M;
            sm.R[r] = s.R;
            sm.T[r] = s.T;
            sm.I[r] = s.I;
        }
    }
    __syncthreads();

    if (w == 0) {
        const float nan = __int_as_float(0x7fc00000);
        float lse_t = nan, h = nan, lse_d = nan, f = nan, lr = nan;
        int amax_t = -1;
        bool bad_row = false;
        if (l < a.nt_rows) {
            const float M = sm.M[l], R = sm.R[l];
            bad_row |= !(M > neg_inf());
            const float lp1 = log1pf(R);
            lse_t = M + lp1;
            h = (lp1 - sm.T[l] * kLn2 / (1.f + R)) * a.inv_log_v;
            amax_t = sm.I[l];
        }
        if (l < a.nd_rows) {
            const int r = a.nt_rows + l;
            const float M = sm.M[r], R = sm.R[r];
            bad_row |= !(M > neg_inf());
            lse_d = M + log1pf(R);
            f = R > 0.f ? -logf(R) : kFeatureClamp;
        }
        if (bad_row) raise_status(a, SPEC_ERR_BAD_ROW);
        int xi = -1;
        bool bad_tok = false;
        if (a.mode != MODE_CONF && l < K) {
            xi = a.x[(size_t)b * K + l];
            bad_tok = xi < 0 || xi >= a.V;
            if (bad_tok) raise_status(a, SPEC_ERR_BAD_TOKEN);
        }
        if (a.mode != MODE_CONF && l < K && a.nd_rows > 0) {
            if (!bad_tok) {
                const float zx = Elem<T>::load(trow_ptr<T>(a, b, l) + xi);
                const float qx = Elem<T>::load(drow_ptr<T>(a, b, l) + xi);
                lr = (zx - lse_t) - (qx - lse_d);
            } else {
                lr = neg_inf();
            }
        }
        int n = K;
        if (a.mode == MODE_STOCHASTIC) {
            // accept iff u < min(1, p/q); lr = +inf (q(x) = 0 < p(x)) accepts,
            // NaN (p(x) = q(x) = 0) rejects
            bool acc = false;
            if (l < K) {
                const float ui = a.u[(size_t)b * (K + 1) + l];
                acc = lr >= 0.f || ui < ex2(lr * kLog2e);
            }
            const unsigned m = __ballot_sync(0xffffffffu, acc);
            n = __ffs(~m) - 1;
            if (n > K) n = K;
        } else if (a.mode == MODE_GREEDY) {
            const bool acc = l < K && !bad_tok && xi == amax_t;
            const unsigned m = __ballot_sync(0xffffffffu, acc);
            n = __ffs(~m) - 1;
            if (n > K) n = K;
        } else if (a.mode == MODE_FLY) {
            // "Training-Free Loosely Speculative Decoding", 2.A: a deviation
            // is excused only if h >= theta, the W-window fits in the draft and
            // holds no further deviation; an invalid token is never excused
            const bool dev = l < K && (bad_tok || xi != amax_t);
            const bool open = l < K && !bad_tok && h >= a.theta;
            const unsigned dm = __ballot_sync(0xffffffffu, dev);
            const unsigned gm = __ballot_sync(0xffffffffu, open);
            n = K;
            for (int j = 0; j < K; ++j) {
                if (!((dm >> j) & 1u)) continue;
                bool excused = ((gm >> j) & 1u) && (j + a.W <= K - 1);
                if (excused) {
                    const unsigned win = (a.W >= 32) ? 0xffffffffu : ((1u << a.W) - 1u);
                    excused = ((dm >> (j + 1)) & win) == 0u;
                }
                if (!excused) {
                    n = j;
                    break;
                }
            }
        }
        // per-position outputs
        if (a.mode != MODE_CONF && a.pos_stats && l <= K) {
            float *ps = a.pos_stats + ((size_t)b * (K + 1) + l) * 4;
            ps[0] = lse_t;
            ps[1] = h;
            ps[2] = l < K ? lr : nan;
            ps[3] = l < K ? f : nan;
        }
        if (a.feature && l < a.nd_rows) a.feature[(size_t)b * K + l] = f;
        if (a.conf && a.est && l < a.nd_rows) {
            const float z = a.est[0] * f + a.est[1 + l];
            a.conf[(size_t)b * K + l] = 1.f / (1.f + expf(-z));
        }
        const float lt_n = __shfl_sync(0xffffffffu, lse_t, n);
        const float ld_n = __shfl_sync(0xffffffffu, lse_d, n);
        const int am_n = __shfl_sync(0xffffffffu, amax_t, n);
        if (l == 0) {
            sm.n = n;
            sm.lse_t = lt_n;
            sm.lse_d = ld_n;
            sm.token = am_n;
        }
    }
    __syncthreads();
    if (a.mode == MODE_CONF) return;
    const int n = sm.n;
    int token = sm.token;
    if (a.mode == MODE_STOCHASTIC) {
        const T *tr = trow_ptr<T>(a, b, n);
        const T *dr = n < K ? drow_ptr<T>(a, b, n) : nullptr;
        const float un = a.u[(size_t)b * (K + 1) + K];
        token = residual_draw<T>(a, tr, dr, sm.lse_t, sm.lse_d, un, wsum, sm);
    }
    for (int j = tid; j <= K; j += NT)
        a.out_tokens[(size_t)b * (K + 1) + j] =
            j < n ? a.x[(size_t)b * K + j] : (j == n ? token : -1);
    if (tid == 0) a.acc_len[b] = n;
}

// ---------------------------------------------------------------------------
// The persistent kernel.
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(NT, 3) verify_kernel(const Args a) {
    __shared__ FinSmem sm;
    __shared__ float4 red[NWARP];
    __shared__ unsigned s_unit, s_next;
    __shared__ int s_last;
    extern __shared__ float wsum[];
    const int tid = threadIdx.x;
    const unsigned per_seq = (unsigned)a.rows * (unsigned)a.nT;

    if (tid == 0) s_unit = atomicAdd(a.ctr + CTR_CLAIM, 1u);
    __syncthreads();
    unsigned unit = s_unit;
    while (unit < a.units) {
        if (tid == 0) s_next = atomicAdd(a.ctr + CTR_CLAIM, 1u);
        const int b = (int)(unit / per_seq);
        const unsigned rem = unit - (unsigned)b * per_seq;
        const int r = (int)(rem / (unsigned)a.nT);
        const int t = (int)(rem - (unsigned)r * (unsigned)a.nT);
        const T *row = r < a.nt_rows ? trow_ptr<T>(a, b, r) : drow_ptr<T>(a, b, r - a.nt_rows);
        const int v0 = t * a.TS;
        const int v1 = min(a.V, v0 + a.TS);
        RowAcc s = tile_acc<T>(row, v0, v1);
        s = block_merge(s, red);
        if (tid == 0) {
            a.part[unit] = acc_pack(s);
            __threadfence();
            const unsigned prev = atomicAdd(a.seq_done + b, 1u);
            s_last = prev == per_seq - 1;
        }
        __syncthreads();
        if (s_last) {
            __threadfence();
            finalize<T>(a, b, sm, wsum);
        }
        unit = s_next;
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------

thread_local std::string g_err;

static int fail(int code, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
static int fail(int code, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return code;
}

struct Plan {
    int nT, TS;
    unsigned long long units;
    size_t seq_off, part_off, bytes;
};

// Tiles hold at most 64 KiB of logits. Small batches split rows further, down
// to 2048 elements a tile, until there are about 8192 units, so that each of
// the resident CTAs claims many units and the queue's tail stays short.
static void plan_tiles(int B, int rows, int V, int esize, Plan &p) {
    const int ts_max = 65536 / esize;
    int nT = (V + ts_max - 1) / ts_max;
    const long long rows_total = (long long)B * rows;
    long long want = (8192 + rows_total - 1) / rows_total;
    const long long cap = V / 2048;
    if (want > cap) want = cap;
    if (want > nT) nT = (int)want;
    if (nT < 1) nT = 1;
    int TS = (V + nT - 1) / nT;
    TS = (TS + 7) & ~7;
    nT = (V + TS - 1) / TS;
    p.nT = nT;
    p.TS = TS;
}

static size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Workspace: [header words][seq_done: B words][partials: B * rows * nT float4]
static void plan_workspace(int B, int rows, int V, int esize, Plan &p) {
    plan_tiles(B, rows, V, esize, p);
    p.seq_off = kHeaderWords * sizeof(unsigned);
    p.part_off = align_up(p.seq_off + (size_t)B * sizeof(unsigned), 16);
    p.bytes = p.part_off + (size_t)B * rows * p.nT * sizeof(float4);
    p.units = (unsigned long long)B * rows * p.nT;
}

struct DevInfo {
    int sms = 0;
    int occ[2] = {0, 0};
};

static std::mutex g_dev_mu;
static DevInfo g_dev[64];

static size_t dyn_smem_bytes(int V) { return (size_t)((V + kResBlk - 1) / kResBlk) * NWARP * sizeof(float); }

template <typename T>
static int occupancy(size_t dyn) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, verify_kernel<T>, NT, dyn) != cudaSuccess) n = 1;
    return n < 1 ? 1 : n;
}

static int grid_for(int dtype, unsigned long long units, int *grid) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return fail(SPEC_ERR_CUDA, "cudaGetDevice failed");
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DevInfo &d = g_dev[dev & 63];
    if (d.sms == 0) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return fail(SPEC_ERR_CUDA, "cannot query the SM count");
        const size_t dmax = dyn_smem_bytes(SPEC_MAX_V);
        cudaFuncSetAttribute(verify_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dmax);
        cudaFuncSetAttribute(verify_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)dmax);
        d.occ[0] = occupancy<float>(dmax);
        d.occ[1] = occupancy<__nv_bfloat16>(dmax);
        d.sms = sms;
    }
    unsigned long long g = (unsigned long long)d.sms * (unsigned long long)d.occ[dtype];
    if (g > units) g = units;
    *grid = (int)(g < 1 ? 1 : g);
    return SPEC_OK;
}

static int launch(Args &a, const Plan &p, int dtype, void *ws, void *stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    char *base = static_cast<char *>(ws);
    a.ctr = reinterpret_cast<unsigned *>(base);
    a.seq_done = reinterpret_cast<unsigned *>(base + p.seq_off);
    a.part = reinterpret_cast<float4 *>(base + p.part_off);
    a.nT = p.nT;
    a.TS = p.TS;
    a.units = (unsigned)p.units;
    a.inv_log_v = (float)(1.0 / std::log((double)a.V));
    const size_t dyn = dyn_smem_bytes(a.V);
    int grid = 1;
    int rc = grid_for(dtype, p.units, &grid);
    if (rc != SPEC_OK) return rc;
    cudaError_t e = cudaMemsetAsync(ws, 0, p.part_off, st);
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "workspace reset failed: %s", cudaGetErrorString(e));
    if (dtype == SPEC_BF16)
        verify_kernel<__nv_bfloat16><<<grid, NT, dyn, st>>>(a);
    else
        verify_kernel<float><<<grid, NT, dyn, st>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(e));
    return SPEC_OK;
}

static int check_common(int B, int K, int V, int dtype) {
    if (B < 1) return fail(SPEC_ERR_INVALID_ARG, "B must be >= 1 (got %d)", B);
    if (K < 1 || K > SPEC_MAX_K) return fail(SPEC_ERR_UNSUPPORTED, "K must be in [1, %d] (got %d)", SPEC_MAX_K, K);
    if (V < 2 || V > SPEC_MAX_V) return fail(SPEC_ERR_UNSUPPORTED, "V must be in [2, %d] (got %d)", SPEC_MAX_V, V);
    if (dtype != SPEC_F32 && dtype != SPEC_BF16) return fail(SPEC_ERR_UNSUPPORTED, "unknown dtype %d", dtype);
    Plan pl;
    plan_tiles(B, 2 * K + 1, V, dtype == SPEC_BF16 ? 2 : 4, pl);
    if ((unsigned long long)B * (2 * K + 1) * (unsigned long long)pl.nT >= (1ull << 31))
        return fail(SPEC_ERR_UNSUPPORTED, "batch too large (B=%d)", B);
    return SPEC_OK;
}

static bool elem_aligned(const void *p, int esize) {
    return (reinterpret_cast<uintptr_t>(p) % (uintptr_t)esize) == 0;
}

static bool vec_ok(const void *p, long long stride, int esize) {
    return (reinterpret_cast<uintptr_t>(p) % 16u) == 0 && ((stride * esize) % 16) == 0;
}

}  // namespace sv

using namespace sv;

extern "C" {

// used by the other translation units of the library; not part of the ABI
__attribute__((visibility("hidden"))) int spec_internal_set_error(int code, const char *msg) {
    g_err = msg ? msg : "";
    return code;
}

const char *spec_last_error(void) { return g_err.c_str(); }

const char *spec_version(void) { return "specverify 0.1 (sm_103a)"; }

size_t spec_workspace_size(const spec_verify_params *p) {
    if (!p) return 0;
    if (check_common(p->B, p->K, p->V, p->dtype) != SPEC_OK) return 0;
    Plan pl;
    plan_workspace(p->B, 2 * p->K + 1, p->V, p->dtype == SPEC_BF16 ? 2 : 4, pl);
    return pl.bytes;
}

size_t spec_confidence_workspace_size(int32_t B, int32_t K, int32_t V, int32_t dtype) {
    if (check_common(B, K, V, dtype) != SPEC_OK) return 0;
    Plan pl;
    plan_workspace(B, K, V, dtype == SPEC_BF16 ? 2 : 4, pl);
    return pl.bytes;
}

int spec_verify(const spec_verify_params *p, const void *target_logits, const void *draft_logits,
                const int32_t *draft_tokens, const float *uniforms, int32_t *out_tokens,
                int32_t *accepted_len, float *pos_stats, const float *est_params, float *feature,
                float *conf, void *workspace, size_t workspace_bytes, void *stream) {
    g_err.clear();
    if (!p) return fail(SPEC_ERR_INVALID_ARG, "params is NULL");
    int rc = check_common(p->B, p->K, p->V, p->dtype);
    if (rc != SPEC_OK) return rc;
    if (p->mode != SPEC_STOCHASTIC && p->mode != SPEC_GREEDY && p->mode != SPEC_FLY)
        return fail(SPEC_ERR_UNSUPPORTED, "unknown mode %d", p->mode);
    if (p->reserved != 0) return fail(SPEC_ERR_INVALID_ARG, "params.reserved must be 0");
    const int es = p->dtype == SPEC_BF16 ? 2 : 4;
    const long long ts = p->t_row_stride ? p->t_row_stride : p->V;
    const long long ds = p->d_row_stride ? p->d_row_stride : p->V;
    if (ts < p->V || ds < p->V) return fail(SPEC_ERR_INVALID_ARG, "row strides must be >= V");
    if (!target_logits) return fail(SPEC_ERR_INVALID_ARG, "target_logits is NULL");
    if (!draft_tokens) return fail(SPEC_ERR_INVALID_ARG, "draft_tokens is NULL");
    if (!out_tokens || !accepted_len) return fail(SPEC_ERR_INVALID_ARG, "out_tokens / accepted_len is NULL");
    if (p->mode == SPEC_STOCHASTIC && (!draft_logits || !uniforms))
        return fail(SPEC_ERR_INVALID_ARG, "stochastic mode needs draft_logits and uniforms");
    if ((feature || conf) && !draft_logits)
        return fail(SPEC_ERR_INVALID_ARG, "feature / conf need draft_logits");
    if (conf && !est_params) return fail(SPEC_ERR_INVALID_ARG, "conf needs est_params");
    if (p->mode == SPEC_FLY && (p->fly_window < 1 || !std::isfinite(p->fly_theta)))
        return fail(SPEC_ERR_INVALID_ARG, "FLy needs fly_window >= 1 and a finite fly_theta");
    if (!elem_aligned(target_logits, es) || (draft_logits && !elem_aligned(draft_logits, es)))
        return fail(SPEC_ERR_INVALID_ARG, "logit pointers must be aligned to the element size");
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % 16u) != 0)
        return fail(SPEC_ERR_INVALID_ARG, "workspace must be a 16-byte aligned device pointer");
    Plan pl;
    plan_workspace(p->B, 2 * p->K + 1, p->V, es, pl);
    if (workspace_bytes < pl.bytes)
        return fail(SPEC_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes", workspace_bytes, pl.bytes);

    Args a;
    memset(&a, 0, sizeof a);
    a.zt = target_logits;
    a.zd = draft_logits;
    a.ts = ts;
    a.ds = ds;
    a.x = draft_tokens;
    a.u = uniforms;
    a.est = est_params;
    a.out_tokens = out_tokens;
    a.acc_len = accepted_len;
    a.pos_stats = pos_stats;
    a.feature = feature;
    a.conf = conf;
    a.B = p->B;
    a.K = p->K;
    a.V = p->V;
    a.mode = p->mode;
    a.theta = p->fly_theta;
    a.W = p->fly_window;
    a.nt_rows = p->K + 1;
    a.nd_rows = draft_logits ? p->K : 0;
    a.rows = a.nt_rows + a.nd_rows;
    a.t_vec_ok = vec_ok(target_logits, ts, es);
    a.d_vec_ok = draft_logits ? vec_ok(draft_logits, ds, es) : 0;
    // the tile plan is that of the workspace (2K+1 rows); the streamed row
    // count may be smaller (no draft rows), which only shortens the queue
    pl.units = (unsigned long long)p->B * a.rows * pl.nT;
    return launch(a, pl, p->dtype, workspace, stream);
}

int spec_confidence(int32_t B, int32_t K, int32_t V, int32_t dtype, const void *draft_logits,
                    int64_t d_row_stride, const float *est_params, float *feature, float *conf,
                    void *workspace, size_t workspace_bytes, void *stream) {
    g_err.clear();
    int rc = check_common(B, K, V, dtype);
    if (rc != SPEC_OK) return rc;
    const int es = dtype == SPEC_BF16 ? 2 : 4;
    const long long ds = d_row_stride ? d_row_stride : V;
    if (ds < V) return fail(SPEC_ERR_INVALID_ARG, "row stride must be >= V");
    if (!draft_logits || !feature) return fail(SPEC_ERR_INVALID_ARG, "draft_logits / feature is NULL");
    if ((conf == nullptr) != (est_params == nullptr))
        return fail(SPEC_ERR_INVALID_ARG, "conf and est_params go together");
    if (!elem_aligned(draft_logits, es))
        return fail(SPEC_ERR_INVALID_ARG, "draft_logits must be aligned to the element size");
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % 16u) != 0)
        return fail(SPEC_ERR_INVALID_ARG, "workspace must be a 16-byte aligned device pointer");
    Plan pl;
    plan_workspace(B, K, V, es, pl);
    if (workspace_bytes < pl.bytes)
        return fail(SPEC_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes", workspace_bytes, pl.bytes);
    Args a;
    memset(&a, 0, sizeof a);
    a.zt = draft_logits;   // no target rows are streamed
    a.zd = draft_logits;
    a.ts = ds;
    a.ds = ds;
    a.est = est_params;
    a.feature = feature;
    a.conf = conf;
    a.B = B;
    a.K = K;
    a.V = V;
    a.mode = MODE_CONF;
    a.nt_rows = 0;
    a.nd_rows = K;
    a.rows = K;
    a.d_vec_ok = vec_ok(draft_logits, ds, es);
    return launch(a, pl, dtype, workspace, stream);
}

int spec_get_device_status(const void *workspace, int32_t *status_out) {
    g_err.clear();
    if (!workspace || !status_out) return fail(SPEC_ERR_INVALID_ARG, "NULL argument");
    unsigned v = 0;
    cudaError_t e = cudaMemcpy(&v, static_cast<const unsigned *>(workspace) + CTR_STATUS, sizeof v,
                               cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "status read failed: %s", cudaGetErrorString(e));
    *status_out = (int32_t)v;
    return SPEC_OK;
}

}  // extern "C"
