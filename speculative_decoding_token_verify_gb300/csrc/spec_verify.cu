// spec_verify.cu -- fused verification pass for GB300 (sm_103a) and its C ABI.
//
// One persistent kernel does the whole pass ("Speculative Decoding: как
// черновая модель ускоряет генерацию LLM без потери качества", "Алгоритм на
// каждом шаге", steps 3-4). Every warp is an independent worker (no
// block-wide barrier) that pulls work from two queues:
//
//  * stream units (sequence b, row r, vocabulary tile t), ordered
//    sequence-major and claimed with one atomic each. A unit streams its tile
//    from HBM exactly once with 128-bit non-allocating loads and folds it into
//    an online softmax accumulator (max, complement mass, entropy moment,
//    argmax); the partial goes to the workspace. The warp that completes the
//    last unit of b (per-sequence counter) finalises b: it merges the row
//    partials, applies the mode's rule, writes the per-position outputs and,
//    in stochastic mode, publishes b's draw.
//  * residual units (published sequence, range of 256-element slices),
//    claimed first whenever one is published: they sum max(0, p - q) (or p for
//    the bonus draw) per slice of the stop rows while those rows are still in
//    L2. The warp that completes the last residual unit of b locates the token
//    by an inverse-CDF scan of the slice sums and one slice.
//
// A warp waits only when the stream queue is empty and residual work is still
// to be published; every unit in flight completes without waiting, so the
// wait ends, and it is bounded anyway (SPEC_ERR_TIMEOUT). All reductions run
// in a fixed order.
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

// Launch shape (compile-time; the defaults are the tuned ones)
#ifndef SV_THREADS
#define SV_THREADS 128
#endif
#ifndef SV_MIN_BLOCKS
#define SV_MIN_BLOCKS 8
#endif
#ifndef SV_TILE_BYTES
#define SV_TILE_BYTES 32768
#endif
#ifndef SV_RES_SLICES
#define SV_RES_SLICES 16
#endif
#ifndef SV_UNROLL
#define SV_UNROLL 4
#endif

constexpr int NT = SV_THREADS;         // threads per CTA (independent warps)
constexpr int NWARP = NT / 32;
constexpr int kUnroll = SV_UNROLL;     // 16-byte loads per lane in flight
constexpr int kSlice = 256;            // elements per scan slice (32 lanes x 8)
constexpr int kResSlices = SV_RES_SLICES;  // slices per residual unit
constexpr int kResBatch = 4;           // slices whose loads are in flight together
static_assert(kResSlices % kResBatch == 0, "residual units hold whole batches");
constexpr unsigned kSpinLimit = 1u << 20;  // polls before giving up (~2 s)
constexpr unsigned kFull = 0xffffffffu;
// lane that publishes results and counts completions: not lane 0, which issues
// the warp's bulk copies, so its release fences never wait behind them
constexpr int kSig = 1;
static_assert(NT % 32 == 0 && NT <= 1024, "CTA size must be a multiple of 32");

enum { MODE_STOCHASTIC = 0, MODE_GREEDY = 1, MODE_FLY = 2, MODE_CONF = 3 };

// workspace header words (zeroed before every launch); the busy counters sit
// on separate 128-byte lines so that their atomics and polls do not queue on
// one L2 slice
enum { CTR_CLAIM = 0, CTR_STATUS = 32, CTR_RES_ALLOC = 64, CTR_RES_CLAIM = 96, CTR_RES_PUB = 128,
       kHeaderWords = 160 };

// what finalise hands to the residual units of a sequence
struct Draw {
    float lse_t, lse_d, u;
    int n;
};

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
    unsigned res_units;      // B * nR in stochastic mode, else 0
    int nR;                  // residual units per sequence
    int nslice;              // scan slices per row
    unsigned *res_ready;     // [B] published flag per slot
    unsigned *res_done;      // [B] residual units completed per sequence
    float4 *slotrec;         // [B] per published slot: (lse_t, lse_d, u, 32*b + n)
    double *utot;            // [B][nR] residual mass per residual unit
    float *slices;           // [B][nslice] residual mass per slice
};

__device__ __forceinline__ unsigned ld_relaxed(const unsigned *p) {
    unsigned v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release(unsigned *p, unsigned v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// atomic add that also releases this thread's earlier writes
__device__ __forceinline__ unsigned atom_add_release(unsigned *p, unsigned v) {
    unsigned old;
    asm volatile("atom.release.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ void fence_acquire() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }


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

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}

__device__ __forceinline__ double warp_incl_scan_d(double v, int l) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double t = __shfl_up_sync(kFull, v, o);
        if (l >= o) v += t;
    }
    return v;
}

// ---------------------------------------------------------------------------
// Stream one unit (a tile of one row) with one warp. The tile's 16-byte
// aligned body is read with kUnroll non-allocating 16-byte loads per lane in
// flight and folded chunk by chunk; scalars before the first and after the
// last 16-byte boundary are read directly. Latency is hidden by many resident
// warps (the kernel keeps its register budget small for that), not by deep
// per-warp buffers.
// ---------------------------------------------------------------------------
template <typename T>
struct UnitGeo {
    const T *row;
    int v0, vb, head, ve, tail;
    unsigned bytes;   // body bytes (a multiple of 16)
    bool target;      // a target row (carries the entropy moment)
};

template <typename T>
__device__ __forceinline__ UnitGeo<T> unit_geo(const Args &a, unsigned unit, unsigned per_seq) {
    UnitGeo<T> g;
    const int b = (int)(unit / per_seq);
    const unsigned rem = unit - (unsigned)b * per_seq;
    const int r = (int)(rem / (unsigned)a.nT);
    const int t = (int)(rem - (unsigned)r * (unsigned)a.nT);
    g.target = r < a.nt_rows;
    g.row = g.target ? trow_ptr<T>(a, b, r) : drow_ptr<T>(a, b, r - a.nt_rows);
    g.v0 = t * a.TS;
    const int v1 = min(a.V, g.v0 + a.TS);
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(g.row + g.v0);
    int head = (int)(((16u - (unsigned)(a0 & 15u)) & 15u) / sizeof(T));
    if (head > v1 - g.v0) head = v1 - g.v0;
    g.head = head;
    g.vb = g.v0 + head;
    constexpr int E = 16 / (int)sizeof(T);
    const int nvec = (v1 - g.vb) / E;
    g.ve = g.vb + nvec * E;
    g.tail = v1 - g.ve;
    g.bytes = (unsigned)nvec * 16u;
    return g;
}

// Fold one unit. Returns the warp-merged accumulator (identical in every lane).
template <typename T, bool kEnt>
__device__ __forceinline__ RowAcc unit_consume(const UnitGeo<T> &g, int l) {
    RowAcc hs = acc_empty(), ts = acc_empty();
    if (l < g.head) {
        float z[1] = {Elem<T>::load(g.row + g.v0 + l)};
        acc_chunk<1>(hs, z, g.v0 + l);
    }
    if (l < g.tail) {
        float z[1] = {Elem<T>::load(g.row + g.ve + l)};
        acc_chunk<1>(ts, z, g.ve + l);
    }
    const uint4 *vp = reinterpret_cast<const uint4 *>(g.row + g.vb);
    const int nvec = (int)(g.bytes / 16u);
    StreamAcc s = stream_init();
    int k = l;
    for (; k + (kUnroll - 1) * 32 < nvec; k += kUnroll * 32) {
        uint4 w[kUnroll];
#pragma unroll
        for (int q = 0; q < kUnroll; ++q) w[q] = ldg_stream(vp + k + q * 32);
#pragma unroll
        for (int q = 0; q < kUnroll; ++q) {
            stream_chunk<T, kEnt>(s, w[q], k + q * 32);
            // keep the bits of the lane's best chunk (no reload when finishing)
            if (s.bk == k + q * 32) s.bw = w[q];
        }
    }
    for (; k < nvec; k += 32) {
        const uint4 w = ldg_stream(vp + k);
        stream_chunk<T, kEnt>(s, w, k);
        if (s.bk == k) s.bw = w;
    }
    const RowAcc vs = stream_finish<T>(s, g.vb);
    return warp_merge(acc_merge(acc_merge(hs, vs), ts));
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
// Finalise sequence b with one warp: lane j merges the tile partials of
// target row j and draft row j (ascending tiles), then the lanes apply the
// mode's rule, write the per-position outputs and, in stochastic mode, publish
// the draw of b for the residual units.
// ---------------------------------------------------------------------------
template <typename T>
__device__ __noinline__ void finalize(const Args &a, int b, int l) {
    const int K = a.K;
    const float nan = __int_as_float(0x7fc00000);
    // loads that do not depend on the row statistics go out first: the draft
    // token, its uniform and the two logits it indexes
    const bool conf_only = a.mode == MODE_CONF;
    int xi = -1;
    bool bad_tok = false;
    float ui = 0.f, zx = 0.f, qx = 0.f;
    if (!conf_only && l < K) {
        xi = a.x[(size_t)b * K + l];
        if (a.mode == MODE_STOCHASTIC) ui = a.u[(size_t)b * (K + 1) + l];
        bad_tok = xi < 0 || xi >= a.V;
        if (!bad_tok && a.nd_rows > 0) {
            zx = Elem<T>::load(trow_ptr<T>(a, b, l) + xi);
            qx = Elem<T>::load(drow_ptr<T>(a, b, l) + xi);
        }
    }
    RowAcc tr = acc_empty(), dr = acc_empty();
    {
        // eight partials of each row in flight at a time, merged in tile order
        const float4 *tp = a.part + ((size_t)b * a.rows + l) * a.nT;
        const float4 *dp = a.part + ((size_t)b * a.rows + a.nt_rows + l) * a.nT;
        const bool has_t = l < a.nt_rows, has_d = l < a.nd_rows;
        for (int t0 = 0; t0 < a.nT; t0 += 8) {
            float4 vt[8], vd[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const bool in = t0 + j < a.nT;
                vt[j] = (has_t && in) ? __ldcg(tp + t0 + j) : acc_pack(acc_empty());
                vd[j] = (has_d && in) ? __ldcg(dp + t0 + j) : acc_pack(acc_empty());
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                tr = acc_merge(tr, acc_unpack(vt[j]));
                dr = acc_merge(dr, acc_unpack(vd[j]));
            }
        }
    }
    float lse_t = nan, h = nan, lse_d = nan, f = nan, lr = nan;
    int amax_t = -1;
    bool bad_row = false;
    if (l < a.nt_rows) {
        bad_row |= !(tr.M > neg_inf());
        const float lp1 = log1pf(tr.R);
        lse_t = tr.M + lp1;
        h = (lp1 - tr.T * kLn2 / (1.f + tr.R)) * a.inv_log_v;
        amax_t = tr.I;
    }
    if (l < a.nd_rows) {
        bad_row |= !(dr.M > neg_inf());
        lse_d = dr.M + log1pf(dr.R);
        f = dr.R > 0.f ? -logf(dr.R) : kFeatureClamp;
    }
    if (bad_row) raise_status(a, SPEC_ERR_BAD_ROW);
    if (bad_tok) raise_status(a, SPEC_ERR_BAD_TOKEN);
    if (!conf_only && l < K && a.nd_rows > 0) lr = bad_tok ? neg_inf() : (zx - lse_t) - (qx - lse_d);
    int n = K;
    if (a.mode == MODE_STOCHASTIC) {
        // "Математика верификации": accept iff u < min(1, p/q); lr = +inf
        // (q(x) = 0 < p(x)) accepts, NaN (p(x) = q(x) = 0) rejects
        const bool acc = l < K && (lr >= 0.f || ui < ex2(lr * kLog2e));
        n = min(__ffs(~__ballot_sync(kFull, acc)) - 1, K);
    } else if (a.mode == MODE_GREEDY) {
        const bool acc = l < K && !bad_tok && xi == amax_t;
        n = min(__ffs(~__ballot_sync(kFull, acc)) - 1, K);
    } else if (a.mode == MODE_FLY) {
        // "Training-Free Loosely Speculative Decoding", 2.A: a deviation is
        // excused only if h >= theta, the W-window fits in the draft and holds
        // no further deviation; an invalid token is never excused
        const bool dev = l < K && (bad_tok || xi != amax_t);
        const bool open = l < K && !bad_tok && h >= a.theta;
        const unsigned dm = __ballot_sync(kFull, dev);
        const unsigned gm = __ballot_sync(kFull, open);
        n = K;
        for (int j = 0; j < K; ++j) {
            if (!((dm >> j) & 1u)) continue;
            bool excused = ((gm >> j) & 1u) && (j + a.W <= K - 1);
            if (excused) {
                const unsigned win = (a.W >= 32) ? kFull : ((1u << a.W) - 1u);
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
        // "Puntuar la Distribución": sigmoid(omega * logit(q_max) + beta_{i+1})
        const float z = a.est[0] * f + a.est[1 + l];
        a.conf[(size_t)b * K + l] = 1.f / (1.f + expf(-z));
    }
    if (a.mode == MODE_CONF) return;
    const float lt_n = __shfl_sync(kFull, lse_t, n);
    const float ld_n = __shfl_sync(kFull, lse_d, n);
    const int am_n = __shfl_sync(kFull, amax_t, n);
    const bool draw = a.mode == MODE_STOCHASTIC;   // the token at n comes from locate()
    for (int j = l; j <= K; j += 32) {
        if (draw && j == n) continue;
        a.out_tokens[(size_t)b * (K + 1) + j] = j < n ? a.x[(size_t)b * K + j] : (j == n ? am_n : -1);
    }
    if (l == kSig) {
        a.acc_len[b] = n;
        if (draw) {
            // hand the draw to the residual units of b and publish them
            const unsigned slot = atomicAdd(a.ctr + CTR_RES_ALLOC, 1u);
            a.slotrec[slot] = make_float4(lt_n, ld_n, a.u[(size_t)b * (K + 1) + K], __int_as_float(b * 32 + n));
            __threadfence();
            st_release(a.res_ready + slot, 1u);
            atomicAdd(a.ctr + CTR_RES_PUB, (unsigned)a.nR);
        }
    }
}

// ---------------------------------------------------------------------------
// Residual units and the final inverse-CDF scan ("Математика верификации":
// on a rejection the token is drawn from norm(max(0, p - q)); after K
// acceptances the bonus token is drawn from p_K). The draw takes the smallest
// v whose running sum in ascending v exceeds u * Z.
// ---------------------------------------------------------------------------

// Per-unit totals make the scan two-level: each residual unit stores its
// slice sums and, in fp64, their sum in slice order; locate() scans the unit
// totals, then the slices of one unit, then one slice.

// lane-parallel fp64 inclusive scan over n (<= 32*per) values held
// contiguously per lane; finds the first index whose running sum exceeds
// `target`. Returns that index (or -1) and the running sum before it in *P.
template <int kPer>
__device__ __forceinline__ int scan_find(const double (&v)[kPer], int n, int l, double target, double base,
                                         double *P) {
    double seg = 0.0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) seg += (l * kPer + j < n) ? v[j] : 0.0;
    const double incl = warp_incl_scan_d(seg, l) + base;
    double c = incl - seg;
    int found = -1;
    double Pf = 0.0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        if (found < 0 && l * kPer + j < n) {
            const double prev = c;
            c += v[j];
            if (c > target) {
                found = l * kPer + j;
                Pf = prev;
            }
        }
    }
    const unsigned m = __ballot_sync(kFull, found >= 0);
    if (!m) return -1;
    const int L = __ffs(m) - 1;
    *P = __shfl_sync(kFull, Pf, L);
    return __shfl_sync(kFull, found, L);
}

// the last index in [0, n) with a positive value, warp-wide (-1 if none)
template <int kPer>
__device__ __forceinline__ int last_positive(const double (&v)[kPer], int n, int l) {
    int lm = -1;
#pragma unroll
    for (int j = 0; j < kPer; ++j)
        if (l * kPer + j < n && v[j] > 0.0) lm = l * kPer + j;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lm = max(lm, __shfl_xor_sync(kFull, lm, o));
    return lm;
}

constexpr int kUnitsPerLane = ((SPEC_MAX_V / kSlice + kResSlices - 1) / kResSlices + 31) / 32;  // unit totals per lane
static_assert((SPEC_MAX_V / kSlice + kResSlices - 1) / kResSlices <= 32 * kUnitsPerLane,
              "residual units per row exceed the locate scan");
static_assert(kResSlices <= 32, "a residual unit's slices are scanned one per lane");

// Sum of slice s (elements 256s .. 256s+255) of the draw's weights, per lane
// (8 elements each), in the fixed order every consumer of slice sums uses.
template <typename T>
__device__ __forceinline__ float slice_lane_sum(const Args &a, const T *tr, const T *dr, int s, int l,
                                               float lse_t, float lse_d, float (&r)[8]) {
    resid8<T>(tr, dr, s * kSlice + l * 8, a.V, a.t_vec_ok != 0, a.d_vec_ok != 0, lse_t, lse_d, r);
    return sum8(r);
}

// Locate the token of sequence b's draw from its unit totals (fp64) and slice
// totals: Z is the sum of the unit totals; the scan picks the unit, then the
// slice whose running sum first exceeds u*Z, then rescans that slice lane by
// lane with an fp64 prefix. Returns the token, or -1 when Z is not positive
// (only possible through rounding, or a bad row).
template <typename T>
__device__ int locate_scan(const Args &a, int b, const T *tr, const T *dr, const Draw &d, int l) {
    const double *ut = a.utot + (size_t)b * a.nR;
    double v[kUnitsPerLane];
#pragma unroll
    for (int j = 0; j < kUnitsPerLane; ++j) {
        const int i = l * kUnitsPerLane + j;
        v[j] = i < a.nR ? __ldcg(ut + i) : 0.0;
    }
    double seg = 0.0;
#pragma unroll
    for (int j = 0; j < kUnitsPerLane; ++j) seg += v[j];
    const double Z = __shfl_sync(kFull, warp_incl_scan_d(seg, l), 31);
    if (!(Z > 0.0)) return -1;
    const double target = (double)d.u * Z;
    // nothing inside a fallback unit or slice may exceed the target: its last
    // mass is taken
    const double none = -2.0 * Z - 1.0;
    double P = 0.0;
    int unit = scan_find<kUnitsPerLane>(v, a.nR, l, target, 0.0, &P);
    if (unit < 0) {
        unit = last_positive<kUnitsPerLane>(v, a.nR, l);
        if (unit < 0) return -1;
        P = none;
    }
    const int s0 = unit * kResSlices;
    const int ns = min(kResSlices, a.nslice - s0);
    double sv[1];
    sv[0] = l < ns ? (double)__ldcg(a.slices + (size_t)b * a.nslice + s0 + l) : 0.0;
    double P2 = 0.0;
    int sl = scan_find<1>(sv, ns, l, target, P, &P2);
    if (sl < 0) {
        sl = last_positive<1>(sv, ns, l);
        if (sl < 0) return -1;
        P2 = none;
    }
    const int entry = s0 + sl;
    float r[8];
    const float s = slice_lane_sum<T>(a, tr, dr, entry, l, d.lse_t, d.lse_d, r);
    const double in = warp_incl_scan_d((double)s, l);
    const double ex = in - (double)s;
    const unsigned hit = __ballot_sync(kFull, P2 + in > target);
    int L;
    if (hit) {
        L = __ffs(hit) - 1;
    } else {
        const unsigned nz = __ballot_sync(kFull, s > 0.f);
        L = nz ? 31 - __clz(nz) : 0;
    }
    int tok = -1, lastpos = -1;
    double cc = P2 + ex;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        if (r[j] > 0.f) lastpos = j;
        cc += (double)r[j];
        if (tok < 0 && cc > target) tok = j;
    }
    if (tok < 0) tok = lastpos >= 0 ? lastpos : 0;
    return __shfl_sync(kFull, entry * kSlice + L * 8 + tok, L);
}

// Residual unit t of sequence b: the sums of its slices of the draw's weights
// (kResBatch slices' loads in flight at a time) and their fp64 total in slice
// order.
template <typename T>
__device__ __forceinline__ void unit_sums(const Args &a, int b, int t, const T *tr, const T *dr, const Draw &d,
                                          int l) {
    double tot = 0.0;
    for (int i0 = 0; i0 < kResSlices; i0 += kResBatch) {
        float part[kResBatch];
#pragma unroll
        for (int i = 0; i < kResBatch; ++i) {
            float r[8];
            part[i] = slice_lane_sum<T>(a, tr, dr, t * kResSlices + i0 + i, l, d.lse_t, d.lse_d, r);
        }
#pragma unroll
        for (int i = 0; i < kResBatch; ++i) {
            const int sidx = t * kResSlices + i0 + i;
            const float s = warp_sum_f(part[i]);
            if (sidx < a.nslice) {
                tot += (double)s;
                if (l == kSig) a.slices[(size_t)b * a.nslice + sidx] = s;
            }
        }
    }
    if (l == kSig) a.utot[(size_t)b * a.nR + t] = tot;
}

// The last residual unit of sequence b: locate its token. If the residual
// mass vanished (only possible through rounding) the warp redraws from p.
template <typename T>
__device__ __noinline__ void locate(const Args &a, int b, const Draw &d, int l) {
    const int K = a.K;
    const T *tr = trow_ptr<T>(a, b, d.n);
    const T *dr = d.n < K ? drow_ptr<T>(a, b, d.n) : nullptr;
    int token = locate_scan<T>(a, b, tr, dr, d, l);
    if (token < 0 && dr != nullptr) {
        for (int t = 0; t < a.nR; ++t) unit_sums<T>(a, b, t, tr, nullptr, d, l);
        __threadfence_block();
        __syncwarp();
        token = locate_scan<T>(a, b, tr, nullptr, d, l);
    }
    if (token < 0) {
        if (l == 0) raise_status(a, SPEC_ERR_BAD_ROW);
        token = 0;
    }
    if (l == 0) a.out_tokens[(size_t)b * (K + 1) + d.n] = token;
}

// One residual unit of the sequence published in `slot`. Its record holds
// (lse_t, lse_d, u, 32*b + n). The last unit of the sequence locates its token.
template <typename T>
__device__ __noinline__ void residual_unit(const Args &a, unsigned id, int l) {
    const int slot = (int)(id / (unsigned)a.nR);
    const int t = (int)(id - (unsigned)slot * (unsigned)a.nR);
    const float4 rec = __ldcg(a.slotrec + slot);
    const int bits = __float_as_int(rec.w);
    const int b = bits >> 5;
    Draw d;
    d.lse_t = rec.x;
    d.lse_d = rec.y;
    d.u = rec.z;
    d.n = bits & 31;
    const T *tr = trow_ptr<T>(a, b, d.n);
    const T *dr = d.n < a.K ? drow_ptr<T>(a, b, d.n) : nullptr;
    unit_sums<T>(a, b, t, tr, dr, d, l);
    bool last = false;
    if (l == kSig) last = atom_add_release(a.res_done + b, 1u) == (unsigned)a.nR - 1;
    last = __shfl_sync(kFull, last, kSig);
    if (last) {
        fence_acquire();
        locate<T>(a, b, d, l);
    }
}

// ---------------------------------------------------------------------------
// Scheduling, per warp (lane 0 keeps the state). Stream units come first, in
// sequence-major order, one atomicAdd each, prefetched one job ahead. Once the
// stream queue is empty the warp turns to residual units: claimed with
// atomicAdd in publication order (a CAS loop would serialise the GPU on one
// counter), each run once its sequence is published. A warp waits only when it
// holds no stream unit and has completed everything it streamed; every
// publication depends only on stream units held by running warps, which never
// wait, so each wait ends.
// ---------------------------------------------------------------------------
struct Sched {
    unsigned next_stream;   // prefetched stream unit (>= units: none left)
    unsigned pend;          // claimed residual unit not yet run (kNone: none)
};
constexpr unsigned kNone = 0xffffffffu;

enum { JOB_DONE = 0, JOB_STREAM = 1, JOB_RESIDUAL = 2, JOB_WAIT = 3 };

// lane 0: the next job that can start now; JOB_WAIT when the only work left
// is residual work that is not published yet (see wait_job).
__device__ __forceinline__ int next_job(const Args &a, Sched &q, unsigned &id) {
    if (q.next_stream < a.units) {
        id = q.next_stream;
        q.next_stream = atomicAdd(a.ctr + CTR_CLAIM, 1u);
        return JOB_STREAM;
    }
    return a.res_units ? JOB_WAIT : JOB_DONE;
}

// lane 0: wait for a residual unit. Called only when the warp holds no stream
// unit and has completed every unit it streamed, so the sequences it waits for
// depend only on other warps' units, none of which waits.
__device__ __forceinline__ int wait_job(const Args &a, Sched &q, unsigned &id) {
    unsigned ns = 64;
    for (unsigned it = 0; it < kSpinLimit; ++it) {
        if (q.pend == kNone) {
            if (ld_relaxed(a.ctr + CTR_RES_CLAIM) >= a.res_units) return JOB_DONE;
            const unsigned c = atomicAdd(a.ctr + CTR_RES_CLAIM, 1u);
            if (c >= a.res_units) return JOB_DONE;
            q.pend = c;
        }
        if (ld_relaxed(a.res_ready + q.pend / (unsigned)a.nR)) {
            id = q.pend;
            q.pend = kNone;
            fence_acquire();
            return JOB_RESIDUAL;
        }
        __nanosleep(ns);
        ns = min(ns * 2u, 2048u);
    }
    raise_status(a, SPEC_ERR_TIMEOUT);
    return JOB_DONE;
}

// ---------------------------------------------------------------------------
// The persistent kernel: every warp is an independent worker (no block-wide
// barrier anywhere, no shared memory).
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(NT, SV_MIN_BLOCKS) verify_kernel(const Args a) {
    const int l = threadIdx.x & 31;
    const unsigned per_seq = (unsigned)a.rows * (unsigned)a.nT;
    Sched q;
    q.pend = kNone;
    q.next_stream = 0u;
    if (l == 0) q.next_stream = atomicAdd(a.ctr + CTR_CLAIM, 1u);
    // Completion of a stream unit: its partial and a release-increment of the
    // sequence's counter go out at once, but the returned count (is this the
    // sequence's last unit?) is read only after the next unit, so the warp
    // does not stall on the atomic. The check is always made before the warp
    // waits or takes other work.
    int dprev_b = -1;            // sequence of the unit whose count is pending
    unsigned dprev_old = 0u;     // that count (lane kSig)
    for (;;) {
        int kind = 0;
        unsigned unit = 0;
        if (l == 0) kind = next_job(a, q, unit);
        kind = __shfl_sync(kFull, kind, 0);
        unit = __shfl_sync(kFull, unit, 0);
        if (kind != JOB_STREAM && dprev_b >= 0) {
            const bool last = __shfl_sync(kFull, dprev_old == per_seq - 1, kSig);
            if (last) {
                fence_acquire();
                finalize<T>(a, dprev_b, l);
            }
            dprev_b = -1;
        }
        if (kind == JOB_WAIT) {
            if (l == 0) kind = wait_job(a, q, unit);
            kind = __shfl_sync(kFull, kind, 0);
            unit = __shfl_sync(kFull, unit, 0);
        }
        if (kind == JOB_DONE) break;
        if (kind == JOB_RESIDUAL) {
            residual_unit<T>(a, unit, l);
            continue;
        }
        const UnitGeo<T> g = unit_geo<T>(a, unit, per_seq);
        // target rows also carry the entropy moment; draft rows do not need it
        const RowAcc s = g.target ? unit_consume<T, true>(g, l) : unit_consume<T, false>(g, l);
        if (dprev_b >= 0) {
            const bool last = __shfl_sync(kFull, dprev_old == per_seq - 1, kSig);
            if (last) {
                fence_acquire();
                finalize<T>(a, dprev_b, l);
            }
        }
        const int b = (int)(unit / per_seq);
        if (l == kSig) {
            a.part[unit] = acc_pack(s);
            dprev_old = atom_add_release(a.seq_done + b, 1u);
        }
        dprev_b = b;
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
    int nT, TS, nR, nslice;
    unsigned long long units;
    size_t seq_off, ready_off, done_off, rec_off, utot_off, part_off, slice_off;
    size_t zero_bytes, bytes;
};

#ifndef SV_MIN_TILE
#define SV_MIN_TILE 4096
#endif

// A stream unit is one warp's share: a tile of at most SV_TILE_BYTES of
// logits. Small batches split rows further, down to SV_MIN_TILE elements,
// aiming at ~32K units (about 7 per resident warp of a GB300) so that the
// queue's tail stays short.
static void plan_tiles(int B, int rows, int V, int esize, Plan &p) {
    const int ts_max = SV_TILE_BYTES / esize;
    int nT = (V + ts_max - 1) / ts_max;
    const long long rows_total = (long long)B * rows;
    long long want = (32768 + rows_total - 1) / rows_total;
    const long long cap = V / SV_MIN_TILE;
    if (want > cap) want = cap;
    if (want > nT) nT = (int)want;
    if (nT < 1) nT = 1;
    int TS = (V + nT - 1) / nT;
    TS = (TS + 7) & ~7;
    nT = (V + TS - 1) / TS;
    p.nT = nT;
    p.TS = TS;
    p.nslice = (V + kSlice - 1) / kSlice;
    p.nR = (p.nslice + kResSlices - 1) / kResSlices;
}

static size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Workspace: [header words | seq_done[B] | res_ready[B] | res_done[B]] (zeroed
// per call) [slot records B | unit totals B*nR | tile partials B*rows*nT |
// slices B*nslice]
static void plan_workspace(int B, int rows, int V, int esize, Plan &p) {
    plan_tiles(B, rows, V, esize, p);
    p.seq_off = kHeaderWords * sizeof(unsigned);
    p.ready_off = p.seq_off + (size_t)B * sizeof(unsigned);
    p.done_off = p.ready_off + (size_t)B * sizeof(unsigned);
    p.zero_bytes = p.done_off + (size_t)B * sizeof(unsigned);
    p.rec_off = align_up(p.zero_bytes, 16);
    p.utot_off = align_up(p.rec_off + (size_t)B * sizeof(float4), 16);
    p.part_off = align_up(p.utot_off + (size_t)B * p.nR * sizeof(double), 16);
    p.slice_off = align_up(p.part_off + (size_t)B * rows * p.nT * sizeof(float4), 16);
    p.bytes = align_up(p.slice_off + (size_t)B * p.nslice * sizeof(float), 16);
    p.units = (unsigned long long)B * rows * p.nT;
}

struct DevInfo {
    int sms = 0;
    int occ[2] = {0, 0};
};

static std::mutex g_dev_mu;
static DevInfo g_dev[64];

constexpr size_t kDynSmem = 0;

template <typename T>
static int occupancy() {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, verify_kernel<T>, NT, kDynSmem) != cudaSuccess) n = 0;
    return n;
}

// Grid = resident CTAs (SMs x occupancy), at most one warp per unit.
static int grid_for(int dtype, unsigned long long units, int *grid) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return fail(SPEC_ERR_CUDA, "cudaGetDevice failed");
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DevInfo &d = g_dev[dev & 63];
    if (d.sms == 0) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return fail(SPEC_ERR_CUDA, "cannot query the SM count");
        d.occ[0] = occupancy<float>();
        d.occ[1] = occupancy<__nv_bfloat16>();
        if (d.occ[0] < 1 || d.occ[1] < 1)
            return fail(SPEC_ERR_CUDA, "the verify kernel cannot be resident (shared memory %zu bytes)", kDynSmem);
        d.sms = sms;
    }
    unsigned long long g = (unsigned long long)d.sms * (unsigned long long)d.occ[dtype];
    const unsigned long long need = (units + NWARP - 1) / NWARP;
    if (g > need) g = need;
    *grid = (int)(g < 1 ? 1 : g);
    return SPEC_OK;
}

static int launch(Args &a, const Plan &p, int dtype, void *ws, void *stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    char *base = static_cast<char *>(ws);
    a.ctr = reinterpret_cast<unsigned *>(base);
    a.seq_done = reinterpret_cast<unsigned *>(base + p.seq_off);
    a.res_ready = reinterpret_cast<unsigned *>(base + p.ready_off);
    a.res_done = reinterpret_cast<unsigned *>(base + p.done_off);
    a.slotrec = reinterpret_cast<float4 *>(base + p.rec_off);
    a.utot = reinterpret_cast<double *>(base + p.utot_off);
    a.part = reinterpret_cast<float4 *>(base + p.part_off);
    a.slices = reinterpret_cast<float *>(base + p.slice_off);
    a.nT = p.nT;
    a.TS = p.TS;
    a.nR = p.nR;
    a.nslice = p.nslice;
    a.units = (unsigned)p.units;
    a.res_units = a.mode == MODE_STOCHASTIC ? (unsigned)a.B * (unsigned)p.nR : 0u;
    a.inv_log_v = (float)(1.0 / std::log((double)a.V));
    int grid = 1;
    int rc = grid_for(dtype, p.units, &grid);
    if (rc != SPEC_OK) return rc;
    cudaError_t e = cudaMemsetAsync(ws, 0, p.zero_bytes, st);
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "workspace reset failed: %s", cudaGetErrorString(e));
    if (dtype == SPEC_BF16)
        verify_kernel<__nv_bfloat16><<<grid, NT, kDynSmem, st>>>(a);
    else
        verify_kernel<float><<<grid, NT, kDynSmem, st>>>(a);
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

// ---------------------------------------------------------------------------
// Scratch for spec_verify_static: a fixed device array in this library's own
// module, so that the call needs no device allocation. Every GPU that loads
// the library holds it until the process exits.
// ---------------------------------------------------------------------------
constexpr size_t kStaticScratchBytes = (size_t)SPEC_STATIC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

static std::mutex g_static_mu;
static void *g_static_ptr[64];   // device address of g_static_scratch, per device

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


// Allocation-free variant of spec_verify: the workspace is the library's
// static scratch array instead of caller memory. The host-side name of that
// array is not a device address, so its address is looked up once per device
// (cudaGetSymbolAddress, with that device current) on the first call there.
int spec_verify_static(const spec_verify_params *p, const void *target_logits, const void *draft_logits,
                       const int32_t *draft_tokens, const float *uniforms, int32_t *out_tokens,
                       int32_t *accepted_len, float *pos_stats, const float *est_params, float *feature,
                       float *conf, void *stream) {
    g_err.clear();
    if (!p) return fail(SPEC_ERR_INVALID_ARG, "params is NULL");
    const size_t need = spec_workspace_size(p);
    if (need == 0) return check_common(p->B, p->K, p->V, p->dtype);   // sets the message
    if (need > kStaticScratchBytes)
        return fail(SPEC_ERR_UNSUPPORTED,
                    "spec_verify_static: this call needs %zu bytes of scratch, more than the %zu-byte static "
                    "array; use spec_verify with a caller workspace",
                    need, kStaticScratchBytes);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "cudaGetDevice failed: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return fail(SPEC_ERR_UNSUPPORTED, "device index %d out of range", dev);
    void *ws = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_static_mu);
        if (!g_static_ptr[dev]) {
            void *ptr = nullptr;
            e = cudaGetSymbolAddress(&ptr, g_static_scratch);
            if (e != cudaSuccess || !ptr)
                return fail(SPEC_ERR_CUDA, "cudaGetSymbolAddress of the static scratch failed: %s",
                            cudaGetErrorString(e));
            g_static_ptr[dev] = ptr;
        }
        ws = g_static_ptr[dev];
    }
    // spec_verify zeroes the counters it needs (cudaMemsetAsync, no allocation)
    return spec_verify(p, target_logits, draft_logits, draft_tokens, uniforms, out_tokens, accepted_len,
                       pos_stats, est_params, feature, conf, ws, kStaticScratchBytes, stream);
}

}  // extern "C"
