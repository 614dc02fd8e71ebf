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
#define SV_MIN_BLOCKS 4
#endif
#ifndef SV_TILE_BYTES
#define SV_TILE_BYTES 16384
#endif
#ifndef SV_RES_SLICES
#define SV_RES_SLICES 8
#endif
#ifndef SV_STAGES
#define SV_STAGES 3
#endif
#ifndef SV_STAGE_BYTES
#define SV_STAGE_BYTES 4096
#endif

constexpr int NT = SV_THREADS;         // threads per CTA (independent warps)
constexpr int NWARP = NT / 32;
constexpr int kStages = SV_STAGES;     // bulk-copy ring depth per warp
constexpr int kStageBytes = SV_STAGE_BYTES;  // bytes per ring stage
constexpr int kStageVecs = kStageBytes / 16;
constexpr int kSlice = 256;            // elements per scan slice (32 lanes x 8)
constexpr int kResSlices = SV_RES_SLICES;  // slices per residual unit
constexpr int kStage = 256;            // slice totals staged per warp in shared memory
constexpr unsigned kSpinLimit = 1u << 20;  // polls before giving up (~2 s)
constexpr unsigned kWaitLimit = 1u << 22;  // mbarrier polls before giving up
constexpr unsigned kFull = 0xffffffffu;
// lane that publishes results and counts completions: not lane 0, which issues
// the warp's bulk copies, so its release fences never wait behind them
constexpr int kSig = 1;
static_assert(NT % 32 == 0 && NT <= 1024, "CTA size must be a multiple of 32");
static_assert(kStageBytes % 512 == 0, "a stage must hold a whole number of warp vectors");

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
    int *res_seq;            // [B] slot -> sequence
    Draw *draw;              // [B]
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

// ---- bulk copies (TMA) into a warp's shared-memory ring -------------------

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// arm the barrier for `bytes` and copy them from global to shared memory
__device__ __forceinline__ void bulk_load(void *dst, const void *src, unsigned bytes, uint64_t *bar) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, unsigned parity) {
    unsigned ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0u;
}

__device__ __forceinline__ uint4 lds128(const void *p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(smem_addr(p)));
    return v;
}

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
// Stream units through a per-warp ring of bulk copies. The body of a unit
// (its 16-byte aligned part) is copied stage by stage into the warp's ring in
// shared memory by lane 0 (cp.async.bulk, completion counted on one mbarrier
// per stage); the lanes fold each landed stage and lane 0 refills it. The
// producer runs up to one stream unit ahead of the consumer, so copies keep
// flowing across unit boundaries and while the warp finalises or does
// residual work. Scalars before the first and after the last 16-byte boundary
// of a tile are read directly.
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

// Ring state: fi (fills issued) and the producer cursor matter in lane 0; ci
// (stages consumed) is the same in every lane.
struct Ring {
    unsigned char *buf;   // kStages * kStageBytes
    uint64_t *bar;        // kStages mbarriers
    unsigned fi, ci;
    unsigned pf_unit;     // unit whose body is being issued
    const char *pf_src;
    unsigned pf_bytes, pf_off;
    bool ahead;           // pf_unit is the warp's next stream unit, not the current one
    bool dead;            // a copy never landed (SPEC_ERR_TIMEOUT raised)
};

// lane 0: issue copies until the ring is full or nothing is left to prefetch
template <typename T>
__device__ __forceinline__ void ring_fill(const Args &a, Ring &rg, unsigned next_stream, unsigned per_seq) {
    while (rg.fi - rg.ci < (unsigned)kStages) {
        if (rg.pf_off >= rg.pf_bytes) {
            if (rg.ahead || next_stream >= a.units) return;
            const UnitGeo<T> g = unit_geo<T>(a, next_stream, per_seq);
            rg.pf_unit = next_stream;
            rg.pf_src = reinterpret_cast<const char *>(g.row + g.vb);
            rg.pf_bytes = g.bytes;
            rg.pf_off = 0;
            rg.ahead = true;
            continue;
        }
        const unsigned n = min((unsigned)kStageBytes, rg.pf_bytes - rg.pf_off);
        const unsigned slot = rg.fi % (unsigned)kStages;
        // the warp's reads of this slot (ordered before by __syncwarp) come
        // before the bulk copy that overwrites it
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        bulk_load(rg.buf + slot * kStageBytes, rg.pf_src + rg.pf_off, n, rg.bar + slot);
        rg.pf_off += n;
        ++rg.fi;
    }
}

// lane 0: point the producer at the stream unit the warp starts now
template <typename T>
__device__ __forceinline__ void ring_start(const Args &a, Ring &rg, unsigned unit, unsigned next_stream,
                                           unsigned per_seq) {
    if (rg.ahead && rg.pf_unit == unit) {
        rg.ahead = false;     // already being prefetched
    } else {
        const UnitGeo<T> g = unit_geo<T>(a, unit, per_seq);
        rg.pf_unit = unit;
        rg.pf_src = reinterpret_cast<const char *>(g.row + g.vb);
        rg.pf_bytes = g.bytes;
        rg.pf_off = 0;
        rg.ahead = false;
    }
    ring_fill<T>(a, rg, next_stream, per_seq);
}

// Fold one unit: head/tail scalars directly, the body stage by stage from the
// ring. Returns the warp-merged accumulator (identical in every lane).
template <typename T, bool kEnt>
__device__ __forceinline__ RowAcc unit_consume(const Args &a, const UnitGeo<T> &g, Ring &rg, unsigned next_stream,
                                               unsigned per_seq, int l) {
    RowAcc hs = acc_empty(), ts = acc_empty();
    if (l < g.head) {
        float z[1] = {Elem<T>::load(g.row + g.v0 + l)};
        acc_chunk<1>(hs, z, g.v0 + l);
    }
    if (l < g.tail) {
        float z[1] = {Elem<T>::load(g.row + g.ve + l)};
        acc_chunk<1>(ts, z, g.ve + l);
    }
    StreamAcc s = stream_init();
    const unsigned nstage = (g.bytes + kStageBytes - 1) / kStageBytes;
    for (unsigned c = 0; c < nstage; ++c) {
        const unsigned slot = rg.ci % (unsigned)kStages;
        const unsigned par = (rg.ci / (unsigned)kStages) & 1u;
        if (!rg.dead) {
            unsigned it = 0;
            while (!mbar_try_wait(rg.bar + slot, par)) {
                if (++it >= kWaitLimit) {
                    rg.dead = true;
                    break;
                }
            }
            rg.dead = __any_sync(kFull, rg.dead);   // the warp decides as one
            if (rg.dead && l == 0) raise_status(a, SPEC_ERR_TIMEOUT);
        }
        const int nv = (int)(min((unsigned)kStageBytes, g.bytes - c * kStageBytes) / 16u);
        const unsigned char *st = rg.buf + slot * kStageBytes;
        uint4 w[kStageVecs / 32];
#pragma unroll
        for (int j = 0; j < kStageVecs / 32; ++j) {
            const int v = j * 32 + l;
            w[j] = v < nv ? lds128(st + v * 16) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int j = 0; j < kStageVecs / 32; ++j) {
            const int v = j * 32 + l;
            if (v < nv) stream_chunk<T, kEnt>(s, w[j], (int)c * kStageVecs + v);
        }
        // keep the bits of this lane's best chunk if it lies in this stage; the
        // load must have landed before the stage is handed back for a refill
        if (s.bk >= (int)c * kStageVecs) {
            s.bw = lds128(st + (s.bk - (int)c * kStageVecs) * 16);
            asm volatile("mov.b32 %0, %0;\n\tmov.b32 %1, %1;\n\tmov.b32 %2, %2;\n\tmov.b32 %3, %3;"
                         : "+r"(s.bw.x), "+r"(s.bw.y), "+r"(s.bw.z), "+r"(s.bw.w));
        }
        __syncwarp();
        ++rg.ci;
        if (l == 0 && !rg.dead) ring_fill<T>(a, rg, next_stream, per_seq);
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
        // "Математика верификации": accept iff u < min(1, p/q); lr = +inf
        // (q(x) = 0 < p(x)) accepts, NaN (p(x) = q(x) = 0) rejects
        bool acc = false;
        if (l < K) {
            const float ui = a.u[(size_t)b * (K + 1) + l];
            acc = lr >= 0.f || ui < ex2(lr * kLog2e);
        }
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
            Draw d;
            d.lse_t = lt_n;
            d.lse_d = ld_n;
            d.u = a.u[(size_t)b * (K + 1) + K];
            d.n = n;
            a.draw[b] = d;
            const unsigned slot = atomicAdd(a.ctr + CTR_RES_ALLOC, 1u);
            a.res_seq[slot] = b;
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

// Sum of slice s (elements 256s .. 256s+255) of the draw's weights, per lane
// (8 elements each), in the fixed order every consumer of slice sums uses.
template <typename T>
__device__ __forceinline__ float slice_lane_sum(const Args &a, const T *tr, const T *dr, int s, int l,
                                               float lse_t, float lse_d, float (&r)[8]) {
    resid8<T>(tr, dr, s * kSlice + l * 8, a.V, a.t_vec_ok != 0, a.d_vec_ok != 0, lse_t, lse_d, r);
    return sum8(r);
}

// Locate the token of a draw whose slice totals are in `sl` (global): the
// warp sums them in fp64 (Z), then scans them page by page through shared
// memory to find the slice whose running sum first exceeds u*Z, and rescans
// that slice lane by lane with an fp64 prefix. Returns the token, or -1 when
// Z is not positive (only possible through rounding, or a bad row).
template <typename T>
__device__ int locate_scan(const Args &a, const float *sl, const T *tr, const T *dr, const Draw &d,
                           float *stage, int l) {
    const int ne = a.nslice;
    double z = 0.0;
    for (int e0 = 0; e0 < ne; e0 += 256) {
        float v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int e = e0 + j * 32 + l;
            v[j] = e < ne ? __ldcg(sl + e) : 0.f;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) z += (double)v[j];
    }
    const double Z = warp_sum_d(z);
    if (!(Z > 0.0)) return -1;
    const double target = (double)d.u * Z;
    double run = 0.0;
    int entry = -1, last_mass = -1;
    double P = 0.0;
    for (int p0 = 0; p0 < ne && entry < 0; p0 += kStage) {
        const int np = min(kStage, ne - p0);
        for (int e0 = 0; e0 < np; e0 += 256) {
            float v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int e = e0 + j * 32 + l;
                v[j] = e < np ? __ldcg(sl + p0 + e) : 0.f;
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int e = e0 + j * 32 + l;
                if (e < np) stage[e] = v[j];
            }
        }
        __syncwarp();
        const int per = (np + 31) / 32;
        const int e0 = min(np, l * per), e1 = min(np, e0 + per);
        double seg = 0.0;
        int lm = -1;
        for (int e = e0; e < e1; ++e) {
            seg += (double)stage[e];
            if (stage[e] > 0.f) lm = p0 + e;
        }
        const double incl = warp_incl_scan_d(seg, l) + run;
        double c = incl - seg;
        int found = -1;
        double Pf = 0.0;
        for (int e = e0; e < e1 && found < 0; ++e) {
            const double prev = c;
            c += (double)stage[e];
            if (c > target) {
                found = p0 + e;
                Pf = prev;
            }
        }
        const unsigned m = __ballot_sync(kFull, found >= 0);
        if (m) {
            const int L = __ffs(m) - 1;
            entry = __shfl_sync(kFull, found, L);
            P = __shfl_sync(kFull, Pf, L);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lm = max(lm, __shfl_xor_sync(kFull, lm, o));
        last_mass = max(last_mass, lm);
        run = __shfl_sync(kFull, incl, 31);
        __syncwarp();
    }
    if (entry < 0) {
        // rounding left u*Z at the total: the last slice with mass
        if (last_mass < 0) return -1;
        entry = last_mass;
        P = -2.0 * Z - 1.0;  // nothing inside exceeds target: take its last mass
    }
    float r[8];
    const float s = slice_lane_sum<T>(a, tr, dr, entry, l, d.lse_t, d.lse_d, r);
    const double in = warp_incl_scan_d((double)s, l);
    const double ex = in - (double)s;
    const unsigned hit = __ballot_sync(kFull, P + in > target);
    int L;
    if (hit) {
        L = __ffs(hit) - 1;
    } else {
        const unsigned nz = __ballot_sync(kFull, s > 0.f);
        L = nz ? 31 - __clz(nz) : 0;
    }
    int tok = -1, lastpos = -1;
    double cc = P + ex;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        if (r[j] > 0.f) lastpos = j;
        cc += (double)r[j];
        if (tok < 0 && cc > target) tok = j;
    }
    if (tok < 0) tok = lastpos >= 0 ? lastpos : 0;
    return __shfl_sync(kFull, entry * kSlice + L * 8 + tok, L);
}

// The last residual unit of sequence b: locate its token. If the residual
// mass vanished (only possible through rounding) the warp redraws from p.
template <typename T>
__device__ __noinline__ void locate(const Args &a, int b, const Draw &d, float *stage, int l) {
    const int K = a.K;
    const T *tr = trow_ptr<T>(a, b, d.n);
    const T *dr = d.n < K ? drow_ptr<T>(a, b, d.n) : nullptr;
    float *sl = a.slices + (size_t)b * a.nslice;
    int token = locate_scan<T>(a, sl, tr, dr, d, stage, l);
    if (token < 0 && dr != nullptr) {
        // recompute the slice totals of p alone and scan again
        for (int s = 0; s < a.nslice; ++s) {
            float r[8];
            const float t = warp_sum_f(slice_lane_sum<T>(a, tr, nullptr, s, l, d.lse_t, d.lse_d, r));
            if (l == 0) sl[s] = t;
        }
        __threadfence_block();
        __syncwarp();
        token = locate_scan<T>(a, sl, tr, nullptr, d, stage, l);
    }
    if (token < 0) {
        if (l == 0) raise_status(a, SPEC_ERR_BAD_ROW);
        token = 0;
    }
    if (l == 0) a.out_tokens[(size_t)b * (K + 1) + d.n] = token;
}

// One residual unit: slices [kResSlices*t, kResSlices*(t+1)) of the stop rows
// of the sequence in `slot`. The last unit of the sequence locates its token.
template <typename T>
__device__ __noinline__ void residual_unit(const Args &a, unsigned id, float *stage, int l) {
    const int slot = (int)(id / (unsigned)a.nR);
    const int t = (int)(id - (unsigned)slot * (unsigned)a.nR);
    int b = 0;
    float4 dv = make_float4(0.f, 0.f, 0.f, 0.f);
    if (l == 0) {
        b = __ldcg(a.res_seq + slot);
        dv = __ldcg(reinterpret_cast<const float4 *>(a.draw + b));
    }
    b = __shfl_sync(kFull, b, 0);
    Draw d;
    d.lse_t = __shfl_sync(kFull, dv.x, 0);
    d.lse_d = __shfl_sync(kFull, dv.y, 0);
    d.u = __shfl_sync(kFull, dv.z, 0);
    d.n = __shfl_sync(kFull, __float_as_int(dv.w), 0);
    const T *tr = trow_ptr<T>(a, b, d.n);
    const T *dr = d.n < a.K ? drow_ptr<T>(a, b, d.n) : nullptr;
    float part[kResSlices];
#pragma unroll
    for (int i = 0; i < kResSlices; ++i) {
        float r[8];
        part[i] = slice_lane_sum<T>(a, tr, dr, t * kResSlices + i, l, d.lse_t, d.lse_d, r);
    }
#pragma unroll
    for (int i = 0; i < kResSlices; ++i) {
        const int sidx = t * kResSlices + i;
        const float s = warp_sum_f(part[i]);
        if (l == kSig && sidx < a.nslice) a.slices[(size_t)b * a.nslice + sidx] = s;
    }
    bool last = false;
    if (l == kSig) last = atom_add_release(a.res_done + b, 1u) == (unsigned)a.nR - 1;
    last = __shfl_sync(kFull, last, kSig);
    if (last) {
        fence_acquire();
        locate<T>(a, b, d, stage, l);
    }
}

// ---------------------------------------------------------------------------
// Scheduling, per warp (lane 0 keeps the state). Residual units are claimed
// with atomicAdd (a CAS loop would serialise the GPU on one counter) and only
// when the published count suggests one is free; a unit claimed before its
// sequence is published stays pending while the warp keeps streaming. A warp
// waits only when it holds no stream unit; every publication depends only on
// stream units held by running warps, which never wait, so each wait ends.
// ---------------------------------------------------------------------------
struct Sched {
    unsigned next_stream;   // prefetched stream unit (>= units: none left)
    unsigned pend;          // claimed residual unit not yet run (kNone: none)
    unsigned res_claim, res_pub, pend_ready;   // loads issued one job ahead
};
constexpr unsigned kNone = 0xffffffffu;

__device__ __forceinline__ void sched_prefetch(const Args &a, Sched &q) {
    if (!a.res_units) return;
    q.res_claim = ld_relaxed(a.ctr + CTR_RES_CLAIM);
    q.res_pub = ld_relaxed(a.ctr + CTR_RES_PUB);
    q.pend_ready = q.pend != kNone ? ld_relaxed(a.res_ready + q.pend / (unsigned)a.nR) : 0u;
}

enum { JOB_DONE = 0, JOB_STREAM = 1, JOB_RESIDUAL = 2, JOB_WAIT = 3 };

// lane 0: the next job that can start now; JOB_WAIT when the only work left
// is residual work that is not published yet (see wait_job).
__device__ __forceinline__ int next_job(const Args &a, Sched &q, unsigned &id) {
    if (a.res_units) {
        if (q.pend == kNone && q.res_claim < q.res_pub && q.res_claim < a.res_units) {
            const unsigned c = atomicAdd(a.ctr + CTR_RES_CLAIM, 1u);
            if (c < a.res_units) {
                q.pend = c;
                q.pend_ready = ld_relaxed(a.res_ready + c / (unsigned)a.nR);
            }
        }
        if (q.pend != kNone && q.pend_ready) {
            id = q.pend;
            q.pend = kNone;
            fence_acquire();           // the slot's data after its flag
            return JOB_RESIDUAL;
        }
    }
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
// barrier anywhere). Dynamic shared memory per warp: the bulk-copy ring, its
// mbarriers and a page of slice totals for the final scan.
// ---------------------------------------------------------------------------
constexpr int kWarpSmem = kStages * kStageBytes + ((kStages * 8 + 127) / 128) * 128 + kStage * 4;

template <typename T>
__global__ void __launch_bounds__(NT, SV_MIN_BLOCKS) verify_kernel(const Args a) {
    extern __shared__ __align__(128) unsigned char dsm[];
    const int l = threadIdx.x & 31;
    unsigned char *base = dsm + (threadIdx.x >> 5) * kWarpSmem;
    Ring rg;
    rg.buf = base;
    rg.bar = reinterpret_cast<uint64_t *>(base + kStages * kStageBytes);
    float *stage = reinterpret_cast<float *>(base + kStages * kStageBytes + ((kStages * 8 + 127) / 128) * 128);
    rg.fi = rg.ci = 0u;
    rg.pf_unit = kNone;
    rg.pf_src = nullptr;
    rg.pf_bytes = rg.pf_off = 0u;
    rg.ahead = false;
    rg.dead = false;
    if (l == 0) {
        for (int i = 0; i < kStages; ++i) mbar_init(rg.bar + i, 1u);
        mbar_init_fence();
    }
    __syncwarp();
    const unsigned per_seq = (unsigned)a.rows * (unsigned)a.nT;
    Sched q;
    q.pend = kNone;
    q.res_claim = q.res_pub = q.pend_ready = 0u;
    q.next_stream = 0u;
    if (l == 0) {
        q.next_stream = atomicAdd(a.ctr + CTR_CLAIM, 1u);
        sched_prefetch(a, q);
    }
    for (;;) {
        int kind = 0;
        unsigned unit = 0;
        if (l == 0) {
            kind = next_job(a, q, unit);
            if (kind == JOB_WAIT) kind = wait_job(a, q, unit);
            if (kind == JOB_STREAM) ring_start<T>(a, rg, unit, q.next_stream, per_seq);
            sched_prefetch(a, q);      // consumed at the next job
        }
        kind = __shfl_sync(kFull, kind, 0);
        unit = __shfl_sync(kFull, unit, 0);
        if (kind == JOB_DONE || rg.dead) break;
        if (kind == JOB_RESIDUAL) {
            residual_unit<T>(a, unit, stage, l);
            continue;
        }
        const unsigned nxt = __shfl_sync(kFull, q.next_stream, 0);
        const UnitGeo<T> g = unit_geo<T>(a, unit, per_seq);
        // target rows also carry the entropy moment; draft rows do not need it
        const RowAcc s = g.target ? unit_consume<T, true>(a, g, rg, nxt, per_seq, l)
                                  : unit_consume<T, false>(a, g, rg, nxt, per_seq, l);
        const int b = (int)(unit / per_seq);
        bool last = false;
        if (l == kSig) {
            a.part[unit] = acc_pack(s);
            last = atom_add_release(a.seq_done + b, 1u) == per_seq - 1;
        }
        last = __shfl_sync(kFull, last, kSig);
        if (last) {
            fence_acquire();
            finalize<T>(a, b, l);
        }
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
    size_t seq_off, ready_off, done_off, resseq_off, draw_off, part_off, slice_off;
    size_t zero_bytes, bytes;
};

#ifndef SV_MIN_TILE
#define SV_MIN_TILE 4096
#endif

// A stream unit is one warp's share: a tile of at most SV_TILE_BYTES of
// logits. Small batches split rows further, down to SV_MIN_TILE elements,
// aiming at ~64K units (about 16 per warp of a full GB300) so that the
// queue's tail stays short.
static void plan_tiles(int B, int rows, int V, int esize, Plan &p) {
    const int ts_max = SV_TILE_BYTES / esize;
    int nT = (V + ts_max - 1) / ts_max;
    const long long rows_total = (long long)B * rows;
    long long want = (65536 + rows_total - 1) / rows_total;
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
// per call) [res_seq[B] | draw[B] | tile partials B*rows*nT | slices B*nslice]
static void plan_workspace(int B, int rows, int V, int esize, Plan &p) {
    plan_tiles(B, rows, V, esize, p);
    p.seq_off = kHeaderWords * sizeof(unsigned);
    p.ready_off = p.seq_off + (size_t)B * sizeof(unsigned);
    p.done_off = p.ready_off + (size_t)B * sizeof(unsigned);
    p.zero_bytes = p.done_off + (size_t)B * sizeof(unsigned);
    p.resseq_off = p.zero_bytes;
    p.draw_off = align_up(p.resseq_off + (size_t)B * sizeof(int), 16);
    p.part_off = align_up(p.draw_off + (size_t)B * sizeof(Draw), 16);
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

constexpr size_t kDynSmem = (size_t)NWARP * kWarpSmem;

template <typename T>
static int occupancy() {
    int n = 0;
    if (cudaFuncSetAttribute(verify_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDynSmem) !=
        cudaSuccess)
        return 0;
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
    a.res_seq = reinterpret_cast<int *>(base + p.resseq_off);
    a.draw = reinterpret_cast<Draw *>(base + p.draw_off);
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
