// spec_verify.cu -- fused verification pass for GB300 (sm_103a) and its C ABI.
//
// One persistent kernel does the whole pass ("Speculative Decoding: как
// черновая модель ускоряет генерацию LLM без потери качества", "Алгоритм на
// каждом шаге", steps 3-4). Every warp is an independent worker (no
// block-wide barrier) that pulls work from two queues:
//
//  * stream units (sequence b, row r, vocabulary tile t), ordered
//    sequence-major and claimed with one atomic each (one unit ahead, except
//    at the end of the queue, where a unit is claimed only when a warp is
//    free to start it). A unit streams its tile from HBM exactly once with
//    128-bit loads (direct, or through a cp.async ring in the warp's staging
//    buffer in the modes with no draw) and folds it into an online softmax
//    accumulator (max, complement mass, entropy moment, argmax); the partial
//    goes to the workspace. A sequence's first unit also gathers the logits
//    at its draft tokens. The warp that completes the last unit of b
//    (per-sequence counter) finalises b: it merges the row partials, applies
//    the mode's rule, publishes b's draw (stochastic mode) and writes the
//    per-position outputs. In stochastic mode the queue's last sequences
//    stream in smaller tiles, so that the draw chain ending the launch
//    starts sooner.
//  * residual units (published sequence, a run of 256-element slices),
//    taken once the stream queue is empty and claimed one ahead: each sums
//    max(0, p - q) (or p for the bonus draw) per slice of the stop rows in
//    one memory round trip. The warp that completes the last residual unit
//    of b locates the token by an inverse-CDF scan of the slice sums and one
//    slice.
//
// A warp waits only when the stream queue is empty and residual work is still
// to be published; every unit in flight completes without waiting, so the
// wait ends, and it is bounded anyway (SPEC_ERR_TIMEOUT). All reductions run
// in a fixed order.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include "spec_device.cuh"
#include "spec_nucleus.cuh"
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
#define SV_TILE_BYTES 65536
#endif
// slices per residual unit: 8 KB (bf16) or 32 KB (fp32) of the two rows
#ifndef SV_RES_SLICES_BF16
#define SV_RES_SLICES_BF16 8
#endif
#ifndef SV_RES_SLICES_F32
#define SV_RES_SLICES_F32 16
#endif
#ifndef SV_UNROLL
#define SV_UNROLL 4
#endif
// launches with no draw (greedy, FLy, confidences; temperature 1) stream
// through a two-chunk cp.async ring in the warp's staging buffer, so that
// the next chunks' loads stay in flight while a chunk is folded (FLy B=128,
// K=15: 0.1154 against 0.1224 ms). The ring cost stochastic launches 2-7%,
// whether on all rows or on target rows only, so they keep direct loads and
// a kernel without the ring's code. 0 turns the ring off.
#ifndef SV_STREAM_RING
#define SV_STREAM_RING 1
#endif
// the last SV_LAZY_ROUNDS x (resident warps) stream units are claimed when
// due instead of one unit ahead
#ifndef SV_LAZY_ROUNDS
#define SV_LAZY_ROUNDS 4
#endif
// likewise the last SV_RES_LAZY x (resident warps) residual units, in 1/4
// rounds (a unit held ahead by a warp still busy with another would wait
// while idle warps run dry; at the queue's end those units carry the draw
// chain of the last sequences)
#ifndef SV_RES_LAZY
#define SV_RES_LAZY 0
#endif
// words between consecutive published-draw flags (polled by waiting warps)
#ifndef SV_READY_STRIDE
#define SV_READY_STRIDE 1
#endif
// longest sleep between polls of a waiting warp (ns)
#ifndef SV_POLL_NS_MAX
#define SV_POLL_NS_MAX 256
#endif

constexpr int NT = SV_THREADS;         // threads per CTA (independent warps)
constexpr int NWARP = NT / 32;
constexpr int kUnroll = SV_UNROLL;     // 16-byte loads per lane in flight
constexpr int kSlice = 256;            // elements per scan slice (32 lanes x 8)
template <typename T>
__host__ __device__ constexpr int res_slices() { return sizeof(T) == 2 ? SV_RES_SLICES_BF16 : SV_RES_SLICES_F32; }
// slices whose loads are in flight together: 8 16-byte vectors per lane
// (two rows) for bf16, 16 for fp32
constexpr int kResBatch = 4;
static_assert(SV_RES_SLICES_BF16 % kResBatch == 0 && SV_RES_SLICES_F32 % kResBatch == 0,
              "residual units hold whole batches");
constexpr int kStage = 256;            // 16-byte entries of a warp's shared staging buffer (4 KB)
constexpr int kScanPer = 4 * kStage / 32;  // slice sums per lane in one pass of the locate scan
constexpr unsigned kSpinLimit = 1u << 20;  // default polls before giving up (< 1 s)
constexpr unsigned kFull = 0xffffffffu;
// lane that publishes results and counts completions (lane 0 keeps the
// scheduling state, so the two sets of long-latency operations stay apart)
constexpr int kSig = 1;
static_assert(NT % 32 == 0 && NT <= 1024, "CTA size must be a multiple of 32");

enum { MODE_STOCHASTIC = 0, MODE_GREEDY = 1, MODE_FLY = 2, MODE_CONF = 3 };

// workspace header words (zeroed before every launch); the busy counters sit
// on separate 128-byte lines so that their atomics and polls do not queue on
// one L2 slice
enum { CTR_CLAIM = 0, CTR_NUC_ROW = 16, CTR_STATUS = 32, CTR_RES_ALLOC = 64, CTR_RES_CLAIM = 96, kHeaderWords = 128 };

// what finalise hands to the residual units of a sequence. At temperature 1
// the weights are p_v = e^{z_v - lse}. With an inverse temperature s they are
// p_v = 2^{(z_v - M) sL - A}, sL = s log2e, A = log2(1 + R): z - M is exact
// where p_v matters (Sterbenz), so p keeps fp32 accuracy at any s, which
// s z - lse would not once |s M| is large.
struct Draw {
    float lse_t, lse_d;   // temperature variant: A_t, A_d
    float m_t, m_d, sL;   // temperature variant only
    float th_t, th_d;     // temperature variant: nucleus thresholds (top-p), else -inf
    float u;
    int n;
    bool bonus;   // all verified drafts accepted: the draw is from p_n alone
};


struct Args {
    const void *zt;
    const void *zd;
    long long ts;            // target row stride (elements)
    long long ds;            // draft row stride (elements)
    const int32_t *x;
    const int32_t *draft_len; // [B] drafts verified per sequence (pruned batch), or null: all K
    const float *inv_temp;    // [B] inverse temperature s per sequence, or null: s = 1 (temperature variant)
    const float *zth;         // [B][rows] nucleus thresholds (top-p), or null (temperature variant)
    int pre;                  // row statistics precomputed in `part` (one record per row; top-p)
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
    unsigned per_seq;        // stream units per sequence (rows * nT)
    unsigned units;          // head_units + (B - B1) * per_seq2
    // the queue's last sequences (b >= B1) stream in smaller tiles (nT2 of
    // TS2 elements per row), so that the last units of the launch are short
    int B1, nT2, TS2;
    unsigned per_seq2;       // rows * nT2
    unsigned head_units;     // B1 * per_seq
    unsigned lazy_from;      // stream units from here on are claimed when due, not one ahead
    int t_vec_ok, d_vec_ok;  // rows start on 16-byte boundaries
    float inv_log_v;         // 1 / ln V
    unsigned *ctr;           // header words
    unsigned *seq_done;      // [B] completed units per sequence
    float4 *part;            // [B][rows][nT] tile partials, one per stream unit
    unsigned res_units;      // B * nR in stochastic mode, else 0
    unsigned res_lazy_from;  // residual units from here on are claimed when due, not one ahead
    int nR;                  // residual units per sequence
    int nslice;              // scan slices per row
    int sstride;             // slice sums per sequence in `slices` (nslice rounded up to 4)
    unsigned *res_ready;     // [B] published flag per slot
    unsigned *res_done;      // [B] residual units completed per sequence
    float4 *slotrec;         // per published slot: (lse_t, lse_d, u, 64*b + 2*n + bonus); the
                             // temperature variant uses two entries per slot, (A_t, A_d, u, bits)
                             // and (M_t, M_d, sL, 0)
    float *slices;           // [B][sstride] residual mass per slice
    float *gx;               // [B][2K] logits at the draft tokens: target rows, then draft rows
    unsigned spin_limit;     // polls of a residual wait before SPEC_ERR_TIMEOUT
    int need_ent;            // target rows carry the entropy moment (pos_stats requested, or FLy)
    unsigned part_cap;       // tile-partial slots in the workspace
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

// 16-byte global -> shared copies that hold no registers while in flight
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    const unsigned sa = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }


// drafts verified for sequence b: draft_len[b] clamped to [0, K], or K
__device__ __forceinline__ int verified(const Args &a, int b) {
    return a.draft_len ? min(max(__ldg(a.draft_len + b), 0), a.K) : a.K;
}

__device__ __forceinline__ void raise_status(const Args &a, unsigned code) {
    atomicMax(a.ctr + CTR_STATUS, code);
}

// Checked builds (SPEC_CHECKED): structural index checks before the accesses
// they guard; a failed check raises SPEC_ERR_INDEX and the access is
// skipped. Other builds compile the checks away.
#ifdef SPEC_CHECKED
__device__ __forceinline__ bool sv_ok(const Args &a, bool cond) {
    if (!cond) raise_status(a, SPEC_ERR_INDEX);
    return cond;
}
#define SV_OK(a, cond) sv_ok((a), (cond))
#else
#define SV_OK(a, cond) true
#endif

// inverse temperature of sequence b; outside [SPEC_MIN_INV_TEMPERATURE,
// SPEC_MAX_INV_TEMPERATURE] (or NaN) the sequence runs at s = 1, and its
// finalize raises SPEC_ERR_BAD_TEMPERATURE
__device__ __forceinline__ bool temp_ok(float s) {
    return s >= SPEC_MIN_INV_TEMPERATURE && s <= SPEC_MAX_INV_TEMPERATURE;
}
__device__ __forceinline__ float seq_inv_temp(const Args &a, int b) {
    if (!a.inv_temp) return 1.f;
    const float s = __ldg(a.inv_temp + b);
    return temp_ok(s) ? s : 1.f;
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
    int b;            // sequence
    int r;            // row within the sequence (target rows first)
    int v0, vb, head, ve, tail;
    unsigned bytes;   // body bytes (a multiple of 16)
    bool target;      // a target row (carries the entropy moment)
};

// first stream unit (= partial slot) of sequence b, and its unit count
__device__ __forceinline__ unsigned seq_base(const Args &a, int b) {
    return b < a.B1 ? (unsigned)b * a.per_seq : a.head_units + (unsigned)(b - a.B1) * a.per_seq2;
}
__device__ __forceinline__ unsigned seq_units(const Args &a, int b) { return b < a.B1 ? a.per_seq : a.per_seq2; }

template <typename T>
__device__ __forceinline__ UnitGeo<T> unit_geo(const Args &a, unsigned unit) {
    UnitGeo<T> g;
    int b, nT, TS;
    unsigned rem;
    if (unit < a.head_units) {
        b = (int)(unit / a.per_seq);
        rem = unit - (unsigned)b * a.per_seq;
        nT = a.nT;
        TS = a.TS;
    } else {
        const unsigned u = unit - a.head_units;
        const int bt = (int)(u / a.per_seq2);
        b = a.B1 + bt;
        rem = u - (unsigned)bt * a.per_seq2;
        nT = a.nT2;
        TS = a.TS2;
    }
    const int r = (int)(rem / (unsigned)nT);
    const int t = (int)(rem - (unsigned)r * (unsigned)nT);
    g.b = b;
    g.r = r;
    g.target = r < a.nt_rows;
    g.row = g.target ? trow_ptr<T>(a, b, r) : drow_ptr<T>(a, b, r - a.nt_rows);
    g.v0 = t * TS;
    const int v1 = min(a.V, g.v0 + TS);
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
// sL, rs: exponent scale and rescale margin (log2e and kRescale at s = 1);
// kSub: difference-first exponents in the scalar head and tail folds (the
// temperature variant).
template <typename T, bool kEnt, bool kSub = false, bool kRing = false>
__device__ __forceinline__ RowAcc unit_consume(const UnitGeo<T> &g, int l, float4 *ring, float sL = kLog2e,
                                               float rs = kRescale) {
    RowAcc hs = acc_empty(), ts = acc_empty();
    if (l < g.head) {
        float z[1] = {Elem<T>::load(g.row + g.v0 + l)};
        acc_chunk<1, kSub>(hs, z, g.v0 + l, sL);
    }
    if (l < g.tail) {
        float z[1] = {Elem<T>::load(g.row + g.ve + l)};
        acc_chunk<1, kSub>(ts, z, g.ve + l, sL);
    }
    const uint4 *vp = reinterpret_cast<const uint4 *>(g.row + g.vb);
    const int nvec = (int)(g.bytes / 16u);
    StreamAcc s = stream_init(sL, rs);
    int k = l;
    if constexpr (kRing) {
        // Where the ring is used (kRing), chunks of kUnroll vectors per
        // lane go through two chunk slots in the warp's staging buffer (slot
        // c & 1, entry q*32 + l): while chunk c is folded from registers, chunks
        // c+1 and c+2 are in flight, with no registers held. Each lane reads back
        // only what it copied, so no barrier is needed; the ring is empty again
        // when the loop ends. Otherwise (and for the last partial chunk) lanes
        // load directly, kUnroll vectors in flight.
        static_assert(2 * kUnroll * 32 <= kStage, "two ring slots fit the staging buffer");
        const int nfull = (nvec - l + kUnroll * 32 - 1 - (kUnroll - 1) * 32) / (kUnroll * 32);   // full chunks of this lane
        if (nfull > 0) {
    #pragma unroll
            for (int q = 0; q < kUnroll; ++q) cp_async16(ring + q * 32 + l, vp + k + q * 32);
            cp_async_commit();
            if (nfull > 1) {
    #pragma unroll
                for (int q = 0; q < kUnroll; ++q) cp_async16(ring + kUnroll * 32 + q * 32 + l, vp + k + kUnroll * 32 + q * 32);
            }
            cp_async_commit();
            for (int c = 0; c < nfull; ++c, k += kUnroll * 32) {
                asm volatile("cp.async.wait_group 1;" ::: "memory");
                float4 *slot = ring + (c & 1) * (kUnroll * 32);
                uint4 w[kUnroll];
    #pragma unroll
                for (int q = 0; q < kUnroll; ++q) {
                    const float4 f = slot[q * 32 + l];
                    w[q] = make_uint4(__float_as_uint(f.x), __float_as_uint(f.y), __float_as_uint(f.z), __float_as_uint(f.w));
                }
                if (c + 2 < nfull) {
    #pragma unroll
                    for (int q = 0; q < kUnroll; ++q) cp_async16(slot + q * 32 + l, vp + k + 2 * kUnroll * 32 + q * 32);
                }
                cp_async_commit();
    #pragma unroll
                for (int q = 0; q < kUnroll; ++q) {
                    stream_chunk<T, kEnt>(s, w[q], k + q * 32, sL, rs);
                    if (s.bk == k + q * 32) s.bw = w[q];
                }
            }
            cp_async_wait();
        }
    }
    for (; k + (kUnroll - 1) * 32 < nvec; k += kUnroll * 32) {
        uint4 w[kUnroll];
#pragma unroll
        for (int q = 0; q < kUnroll; ++q) w[q] = ldg_stream(vp + k + q * 32);
#pragma unroll
        for (int q = 0; q < kUnroll; ++q) {
            stream_chunk<T, kEnt>(s, w[q], k + q * 32, sL, rs);
            // keep the bits of the lane's best chunk (no reload when finishing)
            if (s.bk == k + q * 32) s.bw = w[q];
        }
    }
    for (; k < nvec; k += 32) {
        const uint4 w = ldg_stream(vp + k);
        stream_chunk<T, kEnt>(s, w, k, sL, rs);
        if (s.bk == k) s.bw = w;
    }
    const RowAcc vs = stream_finish<T>(s, g.vb, sL);
    return warp_merge(acc_merge(acc_merge(hs, vs, sL), ts, sL), sL);
}

// one probability of the draw's distributions (see Draw). kTemp: 0 default,
// 1 per-sequence temperatures, 2 temperatures and top-p (zero outside the
// row's nucleus)
template <int kTemp>
__device__ __forceinline__ float prob_t(const Draw &d, float z) {
    if constexpr (kTemp == 2) return z >= d.th_t ? ex2(fmaf(z - d.m_t, d.sL, -d.lse_t)) : 0.f;
    else if constexpr (kTemp) return ex2(fmaf(z - d.m_t, d.sL, -d.lse_t));
    else return ex2((z - d.lse_t) * kLog2e);
}
template <int kTemp>
__device__ __forceinline__ float prob_d(const Draw &d, float z) {
    if constexpr (kTemp == 2) return z >= d.th_d ? ex2(fmaf(z - d.m_d, d.sL, -d.lse_d)) : 0.f;
    else if constexpr (kTemp) return ex2(fmaf(z - d.m_d, d.sL, -d.lse_d));
    else return ex2((z - d.lse_d) * kLog2e);
}

// r_v = max(0, p_v - q_v) (or p_v without a draft row) for v..v+7, fp32.
template <typename T, int kTemp>
__device__ __forceinline__ void resid8(const T *trow, const T *drow, int v, int V, bool tv, bool dv,
                                       const Draw &d, float (&r)[8]) {
    float zt[8];
    load8<T>(trow, v, V, tv, zt);
    if (drow) {
        float zd[8];
        load8<T>(drow, v, V, dv, zd);
#pragma unroll
        for (int j = 0; j < 8; ++j) r[j] = fmaxf(prob_t<kTemp>(d, zt[j]) - prob_d<kTemp>(d, zd[j]), 0.f);
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) r[j] = prob_t<kTemp>(d, zt[j]);
    }
}

__device__ __forceinline__ float sum8(const float (&r)[8]) {
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) s += r[j];
    return s;
}

__device__ __forceinline__ RowAcc shfl_acc(const RowAcc &a, int src) {
    RowAcc b;
    b.M = __shfl_sync(kFull, a.M, src);
    b.R = __shfl_sync(kFull, a.R, src);
    b.T = __shfl_sync(kFull, a.T, src);
    b.I = __shfl_sync(kFull, a.I, src);
    return b;
}

// Merge the tile partials of every row of sequence b: whole rows at a time
// are staged in the warp's shared buffer with asynchronous copies (all in
// flight together, no registers held). Each staged row gets L lanes (the
// largest power of two that fits): lane i of a row folds a contiguous run of
// its tiles in order, then the L lanes merge by butterfly, a fixed tree. Lane
// j ends with target row j in tr and draft row j in dr. nT <= kStage always
// (tiles hold >= 4096 of at most 2^20 elements).
__device__ __forceinline__ void merge_rows(const Args &a, int b, int l, float4 *buf, RowAcc &tr, RowAcc &dr,
                                           float sL) {
    const int nT = b < a.B1 ? a.nT : a.nT2;
    const int rc = min(kStage / nT, 32);       // whole rows per staging pass, one lane each at least
    const float4 *base = a.part + seq_base(a, b);
    tr = acc_empty();
    dr = acc_empty();
    if (!SV_OK(a, nT >= 1 && nT <= kStage && seq_base(a, b) + (unsigned)(a.rows * nT) <= a.part_cap)) return;
    const int drow = a.nt_rows + l;            // row index of lane l's draft row
    for (int r0 = 0; r0 < a.rows; r0 += rc) {
        const int rn = min(rc, a.rows - r0);
        const int cnt = rn * nT;
        for (int i = l; i < cnt; i += 32) cp_async16(buf + i, base + (size_t)r0 * nT + i);
        cp_async_wait_all();
        __syncwarp();
        int lsh = 0;
        while (lsh < 5 && (rn << (lsh + 1)) <= 32) ++lsh;
        const int ri = l >> lsh, sub = l & ((1 << lsh) - 1);
        const int run = (nT + (1 << lsh) - 1) >> lsh;
        RowAcc acc = acc_empty();
        if (ri < rn) {
            const float4 *pr = buf + ri * nT;
            const int t1 = min(nT, (sub + 1) * run);
            for (int t = sub * run; t < t1; ++t) acc = acc_merge(acc, acc_unpack(pr[t]), sL);
        }
        for (int o = 1; o < (1 << lsh); o <<= 1) acc = acc_merge(acc, shfl_xor_acc(acc, o), sL);
        // row r0 + i now sits in lane i * L
        const RowAcc st = shfl_acc(acc, (int)(((unsigned)(l - r0) << lsh) & 31u));
        const RowAcc sd = shfl_acc(acc, (int)(((unsigned)(drow - r0) << lsh) & 31u));
        if (l < a.nt_rows && l >= r0 && l < r0 + rn) tr = st;
        if (l < a.nd_rows && drow >= r0 && drow < r0 + rn) dr = sd;
        __syncwarp();
    }
}

// The logits at sequence b's draft tokens, zt[b, i, x_i] and zd[b, i, x_i]
// for the verified positions i, gathered by the warp that streams b's first
// unit and published with that unit's completion, so that the finalize of b
// has no load that waits on another (the token, then the logit it indexes).
template <typename T>
__device__ __noinline__ void gather_tokens(const Args &a, int b, int l) {
    const int K = a.K;
    if (SV_OK(a, b >= 0 && b < a.B) && l < verified(a, b)) {
        const int xv = __ldg(a.x + (size_t)b * K + l);
        if (xv >= 0 && xv < a.V) {
            const float zt = Elem<T>::load(trow_ptr<T>(a, b, l) + xv);
            const float zd = Elem<T>::load(drow_ptr<T>(a, b, l) + xv);
            a.gx[(size_t)b * 2 * K + l] = zt;
            a.gx[(size_t)b * 2 * K + K + l] = zd;
        }
    }
    // orders the lanes' stores before lane kSig's release of the unit
    __syncwarp();
}

// ---------------------------------------------------------------------------
// Finalise sequence b with one warp: the lanes merge the row partials (lane j
// ends with target row j and draft row j), apply the mode's rule, write the
// per-position outputs and, in stochastic mode, publish the draw of b for the
// residual units. kTemp: the rows are processed at sequence b's inverse
// temperature s (lse = s M + ln(1+R); the log-ratio is formed from z - M).
// ---------------------------------------------------------------------------
template <typename T, int kTemp>
__device__ __noinline__ void finalize(const Args &a, int b, int l, float4 *buf) {
    const int K = a.K;
    if (!SV_OK(a, b >= 0 && b < a.B)) return;
    float sc = 1.f;
    if constexpr (kTemp) {
        if (a.inv_temp) {
            const float s_raw = __ldg(a.inv_temp + b);
            if (l == 0 && !temp_ok(s_raw)) raise_status(a, SPEC_ERR_BAD_TEMPERATURE);
            sc = temp_ok(s_raw) ? s_raw : 1.f;
        }
    }
    const float sL = kTemp ? sc * kLog2e : kLog2e;
    // a pruned batch verifies drafts 0..kb-1 against target rows 0..kb
    // ("Verificación Adaptativa sin una cabeza de confianza", "Antecedentes")
    const int kb = verified(a, b);
    const float nan = __int_as_float(0x7fc00000);
    // loads that do not depend on the row statistics go out first: the draft
    // token, its uniform and the two logits it indexes
    const bool conf_only = a.mode == MODE_CONF;
    const bool draw = a.mode == MODE_STOCHASTIC;   // the token at n comes from locate()
    // the draw's slot is taken first; its value is needed only at the end
    unsigned slot = 0u;
    if (draw && l == kSig) slot = atomicAdd(a.ctr + CTR_RES_ALLOC, 1u);
    int xi = -1;
    bool bad_tok = false;
    float ui = 0.f, zx = 0.f, qx = 0.f;
    if (draw && l <= K) ui = a.u[(size_t)b * (K + 1) + l];   // lane K: the residual / bonus uniform
    if (!conf_only && l < kb) {
        xi = a.x[(size_t)b * K + l];
        // gathered by the sequence's first stream unit (gather_tokens); the
        // entries of an invalid token are never written, nor used
        if (a.gx) {
            zx = __ldcg(a.gx + (size_t)b * 2 * K + l);
            qx = __ldcg(a.gx + (size_t)b * 2 * K + K + l);
        }
        bad_tok = xi < 0 || xi >= a.V;
    }
    // the estimator parameters too (read after the outputs are stored, they
    // would cost a round trip of their own: the compiler cannot move a load
    // across stores that may alias it)
    float e_omega = 0.f, e_beta = 0.f;
    if (a.conf && a.est && l < a.nd_rows) {
        e_omega = __ldg(a.est);
        e_beta = __ldg(a.est + 1 + l);
    }
    RowAcc tr, dr;
    merge_rows(a, b, l, buf, tr, dr, sL);
    float lse_t = nan, h = nan, lse_d = nan, f = nan, lr = nan;
    float lp1_t = nan, lp1_d = nan;   // ln(1 + R) (temperature variant)
    int amax_t = -1;
    bool bad_row = false;
    if (l < a.nt_rows && l <= kb) {
        bad_row |= !(tr.M > neg_inf());
        const float lp1 = log1pf(tr.R);
        lp1_t = lp1;
        lse_t = kTemp ? fmaf(sc, tr.M, lp1) : tr.M + lp1;
        h = (lp1 - tr.T * kLn2 / (1.f + tr.R)) * a.inv_log_v;
        amax_t = tr.I;
    }
    if (l < a.nd_rows && l < kb) {
        bad_row |= !(dr.M > neg_inf());
        lp1_d = log1pf(dr.R);
        lse_d = kTemp ? fmaf(sc, dr.M, lp1_d) : dr.M + lp1_d;
        f = fminf(-logf(dr.R), kFeatureClamp);   // capped at 30 (R = 0: +inf -> 30)
    }
    if (bad_row) raise_status(a, SPEC_ERR_BAD_ROW);
    if (bad_tok) raise_status(a, SPEC_ERR_BAD_TOKEN);
    if (!conf_only && l < kb && a.nd_rows > 0) {
        if (bad_tok) {
            lr = neg_inf();
        } else if constexpr (kTemp) {
            // a token outside a row's nucleus has probability 0 there
            const bool in_t = !a.zth || zx >= a.zth[(size_t)b * a.rows + l];
            const bool in_d = !a.zth || qx >= a.zth[(size_t)b * a.rows + a.nt_rows + l];
            lr = (in_t ? fmaf(sc, zx - tr.M, -lp1_t) : neg_inf()) - (in_d ? fmaf(sc, qx - dr.M, -lp1_d) : neg_inf());
        } else {
            lr = (zx - lse_t) - (qx - lse_d);
        }
    }
    int n = kb;
    if (a.mode == MODE_STOCHASTIC) {
        // "Математика верификации": accept iff u < min(1, p/q); lr = +inf
        // (q(x) = 0 < p(x)) accepts, NaN (p(x) = q(x) = 0) rejects
        const bool acc = l < kb && (lr >= 0.f || ui < ex2(lr * kLog2e));
        n = min(__ffs(~__ballot_sync(kFull, acc)) - 1, kb);
    } else if (a.mode == MODE_GREEDY) {
        const bool acc = l < kb && !bad_tok && xi == amax_t;
        n = min(__ffs(~__ballot_sync(kFull, acc)) - 1, kb);
    } else if (a.mode == MODE_FLY) {
        // "Training-Free Loosely Speculative Decoding", 2.A: a deviation is
        // excused only if h >= theta, the W-window fits in the draft and holds
        // no further deviation; an invalid token is never excused
        const bool dev = l < kb && (bad_tok || xi != amax_t);
        const bool open = l < kb && !bad_tok && h >= a.theta;
        const unsigned dm = __ballot_sync(kFull, dev);
        const unsigned gm = __ballot_sync(kFull, open);
        n = kb;
        for (int j = 0; j < kb; ++j) {
            if (!((dm >> j) & 1u)) continue;
            bool excused = ((gm >> j) & 1u) && (j + a.W <= kb - 1);
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
    if (a.mode != MODE_CONF) {
        // the draw's weights: lse (s = 1), or M and A = log2(1 + R) (see Draw)
        const float lt_n = __shfl_sync(kFull, kTemp ? lp1_t * kLog2e : lse_t, n);
        const float ld_n = __shfl_sync(kFull, kTemp ? lp1_d * kLog2e : lse_d, n);
        float mt_n = 0.f, md_n = 0.f;
        if constexpr (kTemp) {
            mt_n = __shfl_sync(kFull, tr.M, n);
            md_n = __shfl_sync(kFull, dr.M, n);
        }
        const int am_n = __shfl_sync(kFull, amax_t, n);
        const float u_draw = __shfl_sync(kFull, ui, K);
        if (draw && l == kSig && SV_OK(a, slot < (unsigned)a.B)) {
            // hand the draw to the residual units of b before any other
            // output goes out, so that the release waits on the record
            // alone; the release store orders the record before the flag
            const float4 rec = make_float4(lt_n, ld_n, u_draw, __int_as_float((b << 6) | (n << 1) | (n == kb ? 1 : 0)));
            if constexpr (kTemp) {
                a.slotrec[2 * slot] = rec;
                a.slotrec[2 * slot + 1] = make_float4(mt_n, md_n, sL, 0.f);
            } else {
                a.slotrec[slot] = rec;
            }
            st_release(a.res_ready + (size_t)slot * SV_READY_STRIDE, 1u);
        }
        // K <= 31: lane j writes position j (lane j holds draft token j)
        if (l <= K && !(draw && l == n)) a.out_tokens[(size_t)b * (K + 1) + l] = l < n ? xi : (l == n ? am_n : -1);
        if (l == kSig) a.acc_len[b] = n;
    }
    if (a.mode != MODE_CONF && a.pos_stats && l <= K) {
        float *ps = a.pos_stats + ((size_t)b * (K + 1) + l) * 4;
        ps[0] = lse_t;
        ps[1] = h;
        ps[2] = l < kb ? lr : nan;
        ps[3] = l < kb ? f : nan;
    }
    if (a.feature && l < a.nd_rows) a.feature[(size_t)b * K + l] = f;
    if (a.conf && a.est && l < a.nd_rows) {
        // "Puntuar la Distribución": sigmoid(omega * logit(q_max) + beta_{i+1})
        const float z = e_omega * f + e_beta;
        a.conf[(size_t)b * K + l] = l < kb ? 1.f / (1.f + expf(-z)) : nan;
    }
}

// ---------------------------------------------------------------------------
// Residual units and the final inverse-CDF scan ("Математика верификации":
// on a rejection the token is drawn from norm(max(0, p - q)); after K
// acceptances the bonus token is drawn from p_K). The draw takes the smallest
// v whose running sum in ascending v exceeds u * Z.
// ---------------------------------------------------------------------------

// Each residual unit stores the fp32 sums of its slices; locate() scans all
// slice sums of the sequence, then rescans one slice lane by lane.

// Sum of slice s (elements 256s .. 256s+255) of the draw's weights, per lane
// (8 elements each), in the fixed order every consumer of slice sums uses.
template <typename T, int kTemp>
__device__ __forceinline__ float slice_lane_sum(const Args &a, const T *tr, const T *dr, int s, int l,
                                               const Draw &d, float (&r)[8]) {
    resid8<T, kTemp>(tr, dr, s * kSlice + l * 8, a.V, a.t_vec_ok != 0, a.d_vec_ok != 0, d, r);
    return sum8(r);
}

// Stage slice sums c0 .. c0 + 32*kScanPer - 1 of one sequence (the row of
// slice sums starts 16-byte aligned and is padded to a multiple of 4) in the
// warp's buffer, with copies that hold no registers; lane l then owns the
// contiguous run l*kScanPer .. of the chunk. Nothing past the row's padding
// is read; entries at or past n read back as 0 (run_get).
__device__ __forceinline__ void stage_issue(const float *ss, int n, int c0, int l, float4 *buf) {
    const int cn = min(4 * kStage, n - c0);
    const float4 *src = reinterpret_cast<const float4 *>(ss + c0);
    for (int i = l; i < (cn + 3) / 4; i += 32) cp_async16(buf + i, src + i);
}
__device__ __forceinline__ void stage_slices(const float *ss, int n, int c0, int l, float4 *buf) {
    stage_issue(ss, n, c0, l, buf);
    cp_async_wait_all();
    __syncwarp();
}

// group j (4 values) of lane l's staged run, entries at or past cn as 0
__device__ __forceinline__ float4 run_get(const float4 *buf, int l, int j, int cn) {
    const int i = l * kScanPer + 4 * j;
    float4 v = i < cn ? buf[i / 4] : make_float4(0.f, 0.f, 0.f, 0.f);
    if (i + 1 >= cn) v.y = 0.f;
    if (i + 2 >= cn) v.z = 0.f;
    if (i + 3 >= cn) v.w = 0.f;
    return v;
}

// fp32 sum of lane l's run of the staged chunk, in ascending order (at most
// kScanPer terms: relative error below 2e-6 of the run, so below 2e-6 of Z);
// read 16 bytes at a time
__device__ __forceinline__ float run_sum(const float4 *buf, int l, int cn) {
    float seg = 0.f;
#pragma unroll 2
    for (int j = 0; j < kScanPer / 4; ++j) {
        const float4 v = run_get(buf, l, j, cn);
        seg += v.x;
        seg += v.y;
        seg += v.z;
        seg += v.w;
    }
    return seg;
}

// Locate the token of sequence b's draw from its slice sums: Z is their total
// (a lane sums its run of slice sums in order, the runs are added across
// lanes by a butterfly); the scan picks the slice whose running sum first
// exceeds u*Z, then rescans that slice lane by lane with a prefix across
// lanes. Returns the token, or -1 when Z is not positive (only possible
// through rounding, or a bad row).
//
// All of it runs in fp32 (GB300's fp64 rate is a small fraction of fp32,
// and this scan is on the launch's critical path). Error budget, relative
// to Z: a slice sum (8 terms per lane, then a 32-lane butterfly) is off by
// under 12 ulp of itself; a lane's run of at most 32 slice sums, summed in
// order, by under 31 ulp of the run; a sum or a prefix across 32 lanes by
// under 5 ulp of the total; u*Z and the differences by 1 ulp each. That is
// under 60 * 2^-24 = 3.6e-6 in all, within the 1e-5 margin inside which a
// draw is flagged, so an unflagged token is the exact-arithmetic one.
__device__ __forceinline__ float warp_incl_scan_f(float v, int l) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float t = __shfl_up_sync(kFull, v, o);
        if (l >= o) v += t;
    }
    return v;
}

template <typename T, int kTemp>
__device__ int locate_scan(const Args &a, int b, const T *tr, const T *dr, const Draw &d, int l, float4 *buf,
                           bool prestaged = false) {
    const float *ss = a.slices + (size_t)b * a.sstride;
    const int n = a.nslice;
    constexpr int kChunk = 32 * kScanPer;
    // pass 1: Z (the first chunk's copies may already be in flight)
    float Z = 0.f;
    for (int c0 = 0; c0 < n; c0 += kChunk) {
        if (c0 == 0 && prestaged) {
            cp_async_wait_all();
            __syncwarp();
        } else {
            stage_slices(ss, n, c0, l, buf);
        }
        Z += warp_sum_f(run_sum(buf, l, n - c0));
        if (n > kChunk) __syncwarp();
    }
    if (!(Z > 0.f)) return -1;
    const float target = d.u * Z;
    // pass 2: the first slice whose running sum exceeds the target (a single
    // chunk is still staged)
    float P = 0.f;    // running sum before the current chunk
    int entry = -1;
    float P2 = 0.f;   // running sum before slice `entry`
    for (int c0 = 0; c0 < n; c0 += kChunk) {
        if (n > kChunk) stage_slices(ss, n, c0, l, buf);
        const int cn = n - c0;
        const float segf = run_sum(buf, l, cn);
        const float incl = warp_incl_scan_f(segf, l) + P;
        const float excl = incl - segf;
        // walk the run, relative to its start
        const float rel = target - excl;
        float c = 0.f;
        int found = -1;
        float Pf = 0.f;
#pragma unroll 1
        for (int j = 0; j < kScanPer / 4; ++j) {
            const float4 v = run_get(buf, l, j, cn);
            const float e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float prev = c;
                c += e[i];
                if (found < 0 && c > rel) {
                    found = c0 + l * kScanPer + 4 * j + i;
                    Pf = excl + prev;
                }
            }
        }
        const unsigned m = __ballot_sync(kFull, found >= 0);
        if (n > kChunk) __syncwarp();
        if (m) {
            const int L = __ffs(m) - 1;
            entry = __shfl_sync(kFull, found, L);
            P2 = __shfl_sync(kFull, Pf, L);
            break;
        }
        P = __shfl_sync(kFull, incl, 31);
    }
    if (entry < 0) {
        // rounding left the target at or above the total: the last positive
        // mass is taken (nothing inside that slice may exceed the target)
        for (int c0 = ((n - 1) / kChunk) * kChunk; c0 >= 0 && entry < 0; c0 -= kChunk) {
            __syncwarp();
            stage_slices(ss, n, c0, l, buf);
            int lm = -1;
#pragma unroll
            for (int j = 0; j < kScanPer / 4; ++j) {
                const float4 v = run_get(buf, l, j, n - c0);
                if (v.x > 0.f) lm = l * kScanPer + 4 * j;
                if (v.y > 0.f) lm = l * kScanPer + 4 * j + 1;
                if (v.z > 0.f) lm = l * kScanPer + 4 * j + 2;
                if (v.w > 0.f) lm = l * kScanPer + 4 * j + 3;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) lm = max(lm, __shfl_xor_sync(kFull, lm, o));
            if (lm >= 0) entry = c0 + lm;
        }
        if (entry < 0) return -1;
        P2 = -2.f * Z - 1.f;
    }
    float r[8];
    const float s = slice_lane_sum<T, kTemp>(a, tr, dr, entry, l, d, r);
    const float in = warp_incl_scan_f(s, l);
    const float ex = in - s;
    const unsigned hit = __ballot_sync(kFull, P2 + in > target);
    int L;
    if (hit) {
        L = __ffs(hit) - 1;
    } else {
        const unsigned nz = __ballot_sync(kFull, s > 0.f);
        L = nz ? 31 - __clz(nz) : 0;
    }
    int tok = -1, lastpos = -1;
    const float rel = target - (P2 + ex);
    float cc = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        if (r[j] > 0.f) lastpos = j;
        cc += r[j];
        if (tok < 0 && cc > rel) tok = j;
    }
    if (tok < 0) tok = lastpos >= 0 ? lastpos : 0;
    return __shfl_sync(kFull, entry * kSlice + L * 8 + tok, L);
}

// Lane sums of kResBatch whole slices s0 .. of 16-byte aligned rows: every
// load of the batch is issued before any arithmetic. Same per-lane order as
// slice_lane_sum.
template <typename T, bool kDraft, int kTemp>
__device__ __forceinline__ void batch_fast(const T *tr, const T *dr, int s0, int l, const Draw &d,
                                           float (&part)[kResBatch]) {
    constexpr int E = Elem<T>::kPerVec;
    constexpr int NV = 8 / E;   // 16-byte vectors per lane per slice per row
    uint4 wt[kResBatch][NV], wd[kResBatch][kDraft ? NV : 1];
#pragma unroll
    for (int i = 0; i < kResBatch; ++i)
#pragma unroll
        for (int k = 0; k < NV; ++k) wt[i][k] = ldg_stream(tr + (s0 + i) * kSlice + l * 8 + k * E);
    if constexpr (kDraft) {
#pragma unroll
        for (int i = 0; i < kResBatch; ++i)
#pragma unroll
            for (int k = 0; k < NV; ++k) wd[i][k] = ldg_stream(dr + (s0 + i) * kSlice + l * 8 + k * E);
    }
#pragma unroll
    for (int i = 0; i < kResBatch; ++i) {
        float r[8];
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            float zt[E];
            Elem<T>::unpack(wt[i][k], zt);
            if constexpr (kDraft) {
                float zd[E];
                Elem<T>::unpack(wd[i][k], zd);
#pragma unroll
                for (int j = 0; j < E; ++j)
                    r[k * E + j] = fmaxf(prob_t<kTemp>(d, zt[j]) - prob_d<kTemp>(d, zd[j]), 0.f);
            } else {
#pragma unroll
                for (int j = 0; j < E; ++j) r[k * E + j] = prob_t<kTemp>(d, zt[j]);
            }
        }
        part[i] = sum8(r);
    }
}

// Lane sums of kResBatch whole slices s0 .. that lane l staged in the warp's
// buffer (entry 64 i + l: target row, 64 i + 32 + l: draft row; each lane
// reads only what it copied). Same per-lane order as slice_lane_sum.
template <bool kDraft, int kTemp>
__device__ __forceinline__ void batch_staged_bf16(const float4 *buf, int l, const Draw &d,
                                                  float (&part)[kResBatch]) {
#pragma unroll
    for (int i = 0; i < kResBatch; ++i) {
        const float4 vt = buf[64 * i + l];
        float zt[8], r[8];
        Elem<__nv_bfloat16>::unpack(*reinterpret_cast<const uint4 *>(&vt), zt);
        if constexpr (kDraft) {
            const float4 vd = buf[64 * i + 32 + l];
            float zd[8];
            Elem<__nv_bfloat16>::unpack(*reinterpret_cast<const uint4 *>(&vd), zd);
#pragma unroll
            for (int j = 0; j < 8; ++j) r[j] = fmaxf(prob_t<kTemp>(d, zt[j]) - prob_d<kTemp>(d, zd[j]), 0.f);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) r[j] = prob_t<kTemp>(d, zt[j]);
        }
        part[i] = sum8(r);
    }
}

// Slices s0 .. s0 + res_slices<T>() - 1 of the draw's weights (kResBatch slices'
// loads in flight at a time); lane kSig stores their sums. For bf16 rows
// holding a whole unit of two batches, the second batch is copied to the
// warp's staging buffer while the first is loaded to registers, so the
// unit costs one memory round trip, not two.
template <typename T, int kTemp>
__device__ __forceinline__ void unit_sums(const Args &a, int b, int s0, const T *tr, const T *dr, const Draw &d,
                                          int l, float4 *buf) {
    if constexpr (sizeof(T) == 2 && res_slices<T>() == 2 * kResBatch) {
        const bool fast = a.t_vec_ok && (dr == nullptr || a.d_vec_ok) && (s0 + 2 * kResBatch) * kSlice <= a.V;
        if (fast) {
            const int s1 = s0 + kResBatch;
#pragma unroll
            for (int i = 0; i < kResBatch; ++i) {
                cp_async16(buf + 64 * i + l, tr + (s1 + i) * kSlice + l * 8);
                if (dr) cp_async16(buf + 64 * i + 32 + l, dr + (s1 + i) * kSlice + l * 8);
            }
            cp_async_commit();
            float part[kResBatch];
            if (dr) batch_fast<T, true, kTemp>(tr, dr, s0, l, d, part);
            else batch_fast<T, false, kTemp>(tr, dr, s0, l, d, part);
#pragma unroll
            for (int i = 0; i < kResBatch; ++i) {
                const float sm = warp_sum_f(part[i]);
                if (l == kSig && SV_OK(a, s0 + i < a.nslice)) a.slices[(size_t)b * a.sstride + s0 + i] = sm;
            }
            cp_async_wait();
            if (dr) batch_staged_bf16<true, kTemp>(buf, l, d, part);
            else batch_staged_bf16<false, kTemp>(buf, l, d, part);
#pragma unroll
            for (int i = 0; i < kResBatch; ++i) {
                const float sm = warp_sum_f(part[i]);
                if (l == kSig && SV_OK(a, s1 + i < a.nslice)) a.slices[(size_t)b * a.sstride + s1 + i] = sm;
            }
            __syncwarp();   // the buffer is reused by the next staged job
            return;
        }
    }
#pragma unroll
    for (int i0 = 0; i0 < res_slices<T>(); i0 += kResBatch) {
        float part[kResBatch];
        const bool fast = a.t_vec_ok && (dr == nullptr || a.d_vec_ok) && (s0 + i0 + kResBatch) * kSlice <= a.V;
        if (fast && dr) {
            batch_fast<T, true, kTemp>(tr, dr, s0 + i0, l, d, part);
        } else if (fast) {
            batch_fast<T, false, kTemp>(tr, dr, s0 + i0, l, d, part);
        } else {
#pragma unroll
            for (int i = 0; i < kResBatch; ++i) {
                float r[8];
                part[i] = slice_lane_sum<T, kTemp>(a, tr, dr, s0 + i0 + i, l, d, r);
            }
        }
#pragma unroll
        for (int i = 0; i < kResBatch; ++i) {
            const int sidx = s0 + i0 + i;
            const float s = warp_sum_f(part[i]);
            if (l == kSig && sidx < a.nslice) a.slices[(size_t)b * a.sstride + sidx] = s;
        }
    }
}

template <int kTemp>
__device__ __forceinline__ Draw decode_slot(const Args &a, int slot, int &b) {
    const float4 rec = __ldcg(a.slotrec + (kTemp ? 2 * slot : slot));
    const int bits = __float_as_int(rec.w);
    b = bits >> 6;
    Draw d;
    d.lse_t = rec.x;
    d.lse_d = rec.y;
    d.u = rec.z;
    d.m_t = d.m_d = 0.f;
    d.sL = kLog2e;
    d.th_t = d.th_d = neg_inf();
    if constexpr (kTemp) {
        const float4 r2 = __ldcg(a.slotrec + 2 * slot + 1);
        d.m_t = r2.x;
        d.m_d = r2.y;
        d.sL = r2.z;
    }
    d.n = (bits >> 1) & 31;
    d.bonus = (bits & 1) != 0;
    if constexpr (kTemp) {
        if (a.zth) {
            d.th_t = __ldg(a.zth + (size_t)b * a.rows + d.n);
            if (!d.bonus) d.th_d = __ldg(a.zth + (size_t)b * a.rows + a.nt_rows + d.n);
        }
    }
    return d;
}

// The last residual unit of the sequence in `slot` completed: locate its
// token. If the residual mass vanished (only possible through rounding) the
// warp redraws from p.
template <typename T, int kTemp>
__device__ __noinline__ void locate(const Args &a, int slot, int b_known, int l, float4 *buf) {
    // the sequence is known, so its slice sums are staged while the draw
    // record is read
    stage_issue(a.slices + (size_t)b_known * a.sstride, a.nslice, 0, l, buf);
    int b;
    const Draw d = decode_slot<kTemp>(a, slot, b);
    const int K = a.K;
    const T *tr = trow_ptr<T>(a, b, d.n);
    const T *dr = d.bonus ? nullptr : drow_ptr<T>(a, b, d.n);
    if (b != b_known) cp_async_wait_all();   // never (a slot names one sequence): restage safely
    if (!SV_OK(a, b >= 0 && b < a.B && b == b_known && d.n >= 0 && d.n <= a.K)) {
        cp_async_wait_all();
        return;
    }
    int token = locate_scan<T, kTemp>(a, b, tr, dr, d, l, buf, b == b_known);
    if (token < 0 && dr != nullptr) {
        for (int s0 = 0; s0 < a.nslice; s0 += res_slices<T>()) unit_sums<T, kTemp>(a, b, s0, tr, nullptr, d, l, buf);
        __threadfence();
        __syncwarp();
        token = locate_scan<T, kTemp>(a, b, tr, nullptr, d, l, buf);
    }
    if (token < 0) {
        if (l == 0) raise_status(a, SPEC_ERR_BAD_ROW);
        token = 0;
    }
    if (l == 0 && SV_OK(a, token >= 0 && token < a.V)) a.out_tokens[(size_t)b * (K + 1) + d.n] = token;
}

// One residual unit: part t of the sequence published in slot id / nR. Lane
// kSig stores the slice sums and release-increments the sequence's residual
// counter; the returned count (lane kSig) says whether this was its last unit.
struct ResDone {
    int slot;
    int b;
    unsigned old;
};

template <typename T, int kTemp>
__device__ __noinline__ ResDone residual_unit(const Args &a, unsigned id, int l, float4 *buf) {
    const int slot = (int)(id / (unsigned)a.nR);
    const int t = (int)(id - (unsigned)slot * (unsigned)a.nR);
    int b;
    const Draw d = decode_slot<kTemp>(a, slot, b);
    if (!SV_OK(a, slot >= 0 && slot < a.B && b >= 0 && b < a.B && d.n >= 0 && d.n <= a.K &&
                      t * res_slices<T>() < a.nslice)) {
        ResDone bad;
        bad.slot = slot;
        bad.b = 0;
        bad.old = 0xffffffffu;   // never the last unit: nothing follows
        return bad;
    }
    const T *tr = trow_ptr<T>(a, b, d.n);
    const T *dr = d.bonus ? nullptr : drow_ptr<T>(a, b, d.n);
    unit_sums<T, kTemp>(a, b, t * res_slices<T>(), tr, dr, d, l, buf);
    ResDone r;
    r.slot = slot;
    r.b = b;
    r.old = 0u;
    if (l == kSig) r.old = atom_add_release(a.res_done + b, 1u);
    return r;
}

// ---------------------------------------------------------------------------
// Scheduling, per warp (lane 0 keeps the state):
//
//  * Stream units come in sequence-major order, one atomicAdd each, claimed
//    one unit ahead, so that the claim's reply is never waited for; the last
//    units of the queue are claimed when due instead (see next_job).
//  * Residual units are taken once the stream queue is empty: claimed with
//    atomicAdd in slot order, one ahead, and run when their sequence's draw
//    is published, polled with a short backoff (bounded; SPEC_ERR_TIMEOUT).
//    Run together at the end, next to the stream's last units; mixed into
//    the stream phase they cost more than they save.
//
// A warp waits only when it holds no stream unit and has resolved every
// completion it owes; each publication depends only on stream units held by
// running warps, which never wait, so every wait ends.
// ---------------------------------------------------------------------------
struct Sched {
    unsigned ns;       // claimed next stream unit (kLazy: claim when due; >= units: none left)
    unsigned pend;     // claimed residual unit (kNone: none claimed; >= res_units: none left)
};
constexpr unsigned kNone = 0xffffffffu;
constexpr unsigned kLazy = 0xfffffffeu;

enum { JOB_DONE = 0, JOB_STREAM = 1, JOB_RESIDUAL = 2, JOB_WAIT = 3 };

// lane 0: the next job that can start now; JOB_WAIT when no stream unit is
// left and residual work remains (see wait_job). Units are claimed one ahead,
// which hides the claim's latency, except at the end of the queue: there a
// unit held by a warp that is still busy (streaming, or finalising a
// sequence) would wait while other warps run dry, so the last units are
// claimed only when a warp is free to start one.
__device__ __forceinline__ int next_job(const Args &a, Sched &q, unsigned &id) {
    unsigned c = q.ns;
    if (c == kLazy) c = atomicAdd(a.ctr + CTR_CLAIM, 1u);
    if (c < a.units) {
        id = c;
        q.ns = c < a.lazy_from ? atomicAdd(a.ctr + CTR_CLAIM, 1u) : kLazy;
        return JOB_STREAM;
    }
    q.ns = c;
    return a.res_units ? JOB_WAIT : JOB_DONE;
}

// lane 0: wait for a residual unit that can run. Called only when no stream
// unit is left and the warp has resolved every completion it owes.
__device__ __forceinline__ int wait_job(const Args &a, Sched &q, unsigned &id) {
    unsigned ns = 32;
    for (unsigned it = 0; it < a.spin_limit; ++it) {
        if (q.pend == kNone) {
            if (ld_relaxed(a.ctr + CTR_RES_CLAIM) >= a.res_units) return JOB_DONE;
            q.pend = atomicAdd(a.ctr + CTR_RES_CLAIM, 1u);
        }
        if (q.pend >= a.res_units) return JOB_DONE;
        if (ld_relaxed(a.res_ready + (size_t)(q.pend / (unsigned)a.nR) * SV_READY_STRIDE)) {
            fence_acquire();
            id = q.pend;
            // the next unit is claimed now (its reply is read only when this
            // unit is done), except by the warp running a draw's last unit
            // (usually the one that completes it, and then locates the token:
            // a unit held meanwhile would wait while idle warps run dry), and
            // at the queue's end, where units are claimed when a warp is free
            const bool last_part = id % (unsigned)a.nR == (unsigned)a.nR - 1u;
            q.pend = !last_part && id + 1u < a.res_lazy_from ? atomicAdd(a.ctr + CTR_RES_CLAIM, 1u) : kNone;
            return JOB_RESIDUAL;
        }
        __nanosleep(ns);
        ns = min(ns * 2u, (unsigned)SV_POLL_NS_MAX);
    }
    raise_status(a, SPEC_ERR_TIMEOUT);
    return JOB_DONE;
}

// ---------------------------------------------------------------------------
// The persistent kernel: every warp is an independent worker (no block-wide
// barrier anywhere; shared memory only as each warp's own staging buffer).
// ---------------------------------------------------------------------------
enum { DUE_NONE = 0, DUE_STREAM = 1, DUE_RESIDUAL = 2 };

template <typename T, int kTemp, bool kRing = false>
__global__ void __launch_bounds__(NT, SV_MIN_BLOCKS) verify_kernel(const Args a) {
    if constexpr (kTemp == 2) {
        // top-p: the nucleus pass's records are read below, and this launch
        // may begin as that kernel ends (a programmatic dependent launch):
        // wait for its completion and its writes
        asm volatile("griddepcontrol.wait;" ::: "memory");
    }
    const int l = threadIdx.x & 31;
    __shared__ float4 s_stage[NWARP][kStage];   // per-warp staging for finalize and locate
    float4 *const wbuf = s_stage[threadIdx.x >> 5];
    Sched q;
    q.pend = kNone;
    q.ns = 0u;
    if (l == 0) q.ns = atomicAdd(a.ctr + CTR_CLAIM, 1u);
    // A completed unit's result and a release-increment of its sequence's
    // counter go out at once, but the returned count (was this the last
    // unit?) is read only at the next boundary, or after the next stream unit
    // has published its own completion, so the warp neither stalls on the
    // atomic nor holds back its next unit's completion behind a finalize. The
    // finalize or locate it may owe is always done before the warp waits.
    int due = DUE_NONE;
    int due_id = 0;           // sequence (stream) or slot (residual)
    int due_b = 0;            // the slot's sequence (residual)
    unsigned due_old = 0u;    // the count returned to lane kSig
    for (;;) {
        int kind = 0;
        unsigned unit = 0;
        if (l == 0) kind = next_job(a, q, unit);
        kind = __shfl_sync(kFull, kind, 0);
        unit = __shfl_sync(kFull, unit, 0);
        if (kind != JOB_STREAM && due != DUE_NONE) {
            const unsigned need = due == DUE_STREAM ? seq_units(a, due_id) - 1u : (unsigned)a.nR - 1u;
            if (__shfl_sync(kFull, due_old == need, kSig)) {
                fence_acquire();
                if (due == DUE_STREAM) finalize<T, kTemp>(a, due_id, l, wbuf);
                else locate<T, kTemp>(a, due_id, due_b, l, wbuf);
            }
            due = DUE_NONE;
        }
        if (kind == JOB_WAIT) {
            if (l == 0) kind = wait_job(a, q, unit);
            kind = __shfl_sync(kFull, kind, 0);
            unit = __shfl_sync(kFull, unit, 0);
        }
        if (kind == JOB_DONE) break;
        if (kind == JOB_RESIDUAL) {
            if (!SV_OK(a, unit < a.res_units)) continue;
            const ResDone r = residual_unit<T, kTemp>(a, unit, l, wbuf);
            due = DUE_RESIDUAL;
            due_id = r.slot;
            due_b = r.b;
            due_old = r.old;
            continue;
        }
        const UnitGeo<T> g = unit_geo<T>(a, unit);
        if (!SV_OK(a, unit < a.units && unit < a.part_cap && g.b >= 0 && g.b < a.B && g.r >= 0 && g.r < a.rows &&
                          g.v0 >= 0 && g.head >= 0 && g.tail >= 0 && g.ve + g.tail <= a.V))
            continue;
        if (a.gx && unit == seq_base(a, g.b)) gather_tokens<T>(a, g.b, l);
        // rows a pruned batch never verified are not read (their partial is
        // empty; the unit still counts toward its sequence's completion)
        bool skip = false;
        if (a.draft_len) {
            const int kb = verified(a, g.b);
            skip = g.target ? g.r > kb : g.r - a.nt_rows >= kb;
        }
        // target rows carry the entropy moment when something reads it
        // (pos_stats, or FLy's gate); draft rows never need it
        const bool ent = g.target && a.need_ent;
        RowAcc s = acc_empty();
        if constexpr (kTemp) {
          if (!a.pre) {
            // the sequence's inverse temperature scales every exponent
            const float sc = seq_inv_temp(a, g.b);
            const float sL = sc * kLog2e, rs = __fdiv_rn(kRescale, sc);   // exact for powers of two
            s = skip ? acc_empty()
                     : (ent ? unit_consume<T, true, true>(g, l, wbuf, sL, rs) : unit_consume<T, false, true>(g, l, wbuf, sL, rs));
          }
        } else {
            s = skip ? acc_empty()
                     : (ent ? unit_consume<T, true, false, kRing>(g, l, wbuf) : unit_consume<T, false, false, kRing>(g, l, wbuf));
        }
        const int b = g.b;
        unsigned old = 0u;
        if (l == kSig) {
            if (!(kTemp && a.pre)) a.part[unit] = acc_pack(s);   // a precomputed record stays
            old = atom_add_release(a.seq_done + b, 1u);
        }
        // this unit's completion is out; now the previous one, whose count
        // has had a whole unit to come back
        if (due != DUE_NONE) {
            const unsigned need = due == DUE_STREAM ? seq_units(a, due_id) - 1u : (unsigned)a.nR - 1u;
            if (__shfl_sync(kFull, due_old == need, kSig)) {
                fence_acquire();
                if (due == DUE_STREAM) finalize<T, kTemp>(a, due_id, l, wbuf);
                else locate<T, kTemp>(a, due_id, due_b, l, wbuf);
            }
        }
        due = DUE_STREAM;
        due_id = b;
        due_old = old;
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
    int nT, TS, nR, nslice, sstride;
    int B1, nT2, TS2;               // the tail: sequences B1.. stream nT2 tiles of TS2 per row
    unsigned long long head_units;  // B1 * rows * nT
    unsigned long long units;       // stream units: head_units + (B - B1) * rows * nT2
    size_t seq_off, ready_off, done_off, rec_off, part_off, slice_off, zth_off, gx_off;
    size_t zero_bytes, bytes;
};

#ifndef SV_MIN_TILE
#define SV_MIN_TILE 4096
#endif
// stream units aimed at: stochastic mode (a draw chain follows the stream),
// and the other modes (the stream ends the launch)
#ifndef SV_TARGET_UNITS_DRAW
#define SV_TARGET_UNITS_DRAW 3072
#endif
#ifndef SV_TARGET_UNITS
#define SV_TARGET_UNITS 16384
#endif
// in stochastic mode the queue's last 1/SV_TAIL_DIV of the logits, kept
// within [SV_TAIL_MIN, SV_TAIL_BYTES] (whole sequences, at most half the
// batch), stream in tiles of SV_TAIL_TILE_BYTES; SV_TAIL_BYTES 0 turns the
// tail off
#ifndef SV_TAIL_BYTES
#define SV_TAIL_BYTES (80ll << 20)
#endif
#ifndef SV_TAIL_MIN
#define SV_TAIL_MIN (32ll << 20)
#endif
#ifndef SV_TAIL_DIV
#define SV_TAIL_DIV 14
#endif
#ifndef SV_TAIL_TILE_BYTES
#define SV_TAIL_TILE_BYTES 32768
#endif
// nT tiles of a row of V elements, rounded to a tile size that is a multiple of 8
static void split_row(int V, long long want, int &nT, int &TS) {
    if (want < 1) want = 1;
    TS = (int)((V + want - 1) / want);
    TS = (TS + 7) & ~7;
    nT = (V + TS - 1) / TS;
}

// A stream unit is one warp's share: a tile of at most SV_TILE_BYTES of
// logits. Small batches split rows further, down to SV_MIN_TILE elements,
// aiming at ~`target` units. Every unit boundary costs a warp a few
// microseconds without loads in flight (the partial's release, then the
// first loads of the next tile), so fewer, larger units stream faster.
// Where the stream ends the launch (greedy, FLy, confidences) the target is
// ~SV_TARGET_UNITS (about 3.4 per resident warp of a GB300), which keeps the
// last units short. In stochastic mode it is ~SV_TARGET_UNITS_DRAW (about
// one per warp): there the finalize merges fewer partials per row, and the
// end of the queue is kept short by its tail (the last sequences stream in
// smaller tiles, so that their draw chain of finalize, residual pass and
// locate starts sooner). In every mode the last units are claimed only when
// a warp is free (see next_job).
static void plan_tiles(int B, int rows, int V, int esize, bool draw, Plan &p) {
    const int ts_max = SV_TILE_BYTES / esize;
    const long long rows_total = (long long)B * rows;
    long long cap = V / SV_MIN_TILE;
    if (cap < 1) cap = 1;
    long long n = (V + ts_max - 1) / ts_max;
    const long long target = draw ? SV_TARGET_UNITS_DRAW : SV_TARGET_UNITS;
    long long want = (target + rows_total - 1) / rows_total;
    if (want > cap) want = cap;
    if (want > n) n = want;
    split_row(V, n, p.nT, p.TS);
    p.B1 = B;
    p.nT2 = p.nT;
    p.TS2 = p.TS;
    const int ts2 = SV_TAIL_TILE_BYTES / esize;
    if (draw && SV_TAIL_BYTES > 0 && ts2 >= SV_MIN_TILE && ts2 < p.TS) {
        const long long seq_bytes = (long long)rows * V * esize;
        long long tail = (long long)B * seq_bytes / SV_TAIL_DIV;
        if (tail < (long long)SV_TAIL_MIN) tail = SV_TAIL_MIN;
        if (tail > (long long)SV_TAIL_BYTES) tail = SV_TAIL_BYTES;
        long long nt = (tail + seq_bytes - 1) / seq_bytes;
        if (nt > B / 2) nt = B / 2;
        if (nt > 0) {
            split_row(V, (V + ts2 - 1) / ts2, p.nT2, p.TS2);
            p.B1 = B - (int)nt;
        }
    }
    p.head_units = (unsigned long long)p.B1 * rows * p.nT;
    p.units = p.head_units + (unsigned long long)(B - p.B1) * rows * p.nT2;
    p.nslice = (V + kSlice - 1) / kSlice;
    p.sstride = (p.nslice + 3) & ~3;
    const int rs = esize == 2 ? res_slices<__nv_bfloat16>() : res_slices<float>();
    p.nR = (p.nslice + rs - 1) / rs;
}

static size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Workspace: [header words | seq_done[B] | res_ready[B] | res_done[B]] (zeroed
// per call) [slot records 2B | tile partials | slices B*sstride | nucleus
// thresholds B*(2K+1) | draft-token logits B*2K (sized B*2*(2K+1))]. The
// partials hold one slot per stream unit of the largest plan among the row
// counts the call may stream (`rows_a`, `rows_b`), in either mode class.
// The plan returned tiles `rows_a` rows for the mode class `draw`.
static void plan_workspace(int B, int rows_a, int rows_b, int V, int esize, bool draw, Plan &p) {
    unsigned long long cap = 0;
    for (int r : {rows_a, rows_b})
        for (bool d : {false, true}) {
            Plan q;
            plan_tiles(B, r, V, esize, d, q);
            if (q.units > cap) cap = q.units;
        }
    plan_tiles(B, rows_a, V, esize, draw, p);
    p.seq_off = kHeaderWords * sizeof(unsigned);
    p.ready_off = p.seq_off + (size_t)B * sizeof(unsigned);
    p.done_off = p.ready_off + (size_t)B * SV_READY_STRIDE * sizeof(unsigned);
    p.zero_bytes = p.done_off + (size_t)B * sizeof(unsigned);
    p.rec_off = align_up(p.zero_bytes, 16);
    p.part_off = align_up(p.rec_off + (size_t)2 * B * sizeof(float4), 16);
    p.slice_off = align_up(p.part_off + (size_t)cap * sizeof(float4), 16);
    p.zth_off = align_up(p.slice_off + (size_t)B * p.sstride * sizeof(float), 16);
    const size_t rmax = (size_t)(rows_a > rows_b ? rows_a : rows_b);   // >= K
    p.gx_off = align_up(p.zth_off + (size_t)B * rmax * sizeof(float), 16);
    p.bytes = align_up(p.gx_off + (size_t)B * 2 * rmax * sizeof(float), 16);
}

// kernel variants: 0 the default, 1 temperature, 2 the staging-buffer ring
struct DevInfo {
    int sms = 0;
    int occ[2][3] = {{0, 0, 0}, {0, 0, 0}};   // [dtype][variant]
};

static std::mutex g_dev_mu;
static DevInfo g_dev[64];

// polls of a residual wait before it gives up (spec_debug_set_wait_limit)
static std::atomic<unsigned> g_wait_limit{kSpinLimit};

constexpr size_t kDynSmem = 0;

template <typename T, int kTemp, bool kRing>
static int occupancy() {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, verify_kernel<T, kTemp, kRing>, NT, kDynSmem) != cudaSuccess)
        n = 0;
    return n;
}

// Grid = resident CTAs (SMs x occupancy), at most one warp per unit.
static int grid_for(int dtype, int variant, unsigned long long units, int *grid) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return fail(SPEC_ERR_CUDA, "cudaGetDevice failed");
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DevInfo &d = g_dev[dev & 63];
    if (d.sms == 0) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return fail(SPEC_ERR_CUDA, "cannot query the SM count");
        d.occ[0][0] = occupancy<float, 0, false>();
        d.occ[1][0] = occupancy<__nv_bfloat16, 0, false>();
        d.occ[0][1] = occupancy<float, 1, false>();
        d.occ[1][1] = occupancy<__nv_bfloat16, 1, false>();
        d.occ[0][2] = occupancy<float, 0, true>();
        d.occ[1][2] = occupancy<__nv_bfloat16, 0, true>();
        for (int i = 0; i < 2; ++i)
            for (int v = 0; v < 3; ++v)
                if (d.occ[i][v] < 1)
                    return fail(SPEC_ERR_CUDA, "the verify kernel cannot be resident (shared memory %zu bytes)",
                                kDynSmem);
        d.sms = sms;
    }
    unsigned long long g = (unsigned long long)d.sms * (unsigned long long)d.occ[dtype][variant];
    const unsigned long long need = (units + NWARP - 1) / NWARP;
    if (g > need) g = need;
    *grid = (int)(g < 1 ? 1 : g);
    return SPEC_OK;
}

static int launch(Args &a, const Plan &p_in, int dtype, void *ws, void *stream, float top_p = 1.f) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    char *base = static_cast<char *>(ws);
    Plan p = p_in;
    if (a.pre) {
        // one unit per row: its statistics come from the nucleus pass
        p.nT = 1;
        p.TS = a.V;
        p.units = (unsigned long long)a.B * (unsigned long long)a.rows;
        p.B1 = a.B;
        p.nT2 = 1;
        p.TS2 = a.V;
        p.head_units = p.units;
        a.zth = reinterpret_cast<float *>(base + p.zth_off);
    }
    a.ctr = reinterpret_cast<unsigned *>(base);
    a.seq_done = reinterpret_cast<unsigned *>(base + p.seq_off);
    a.res_ready = reinterpret_cast<unsigned *>(base + p.ready_off);
    a.res_done = reinterpret_cast<unsigned *>(base + p.done_off);
    a.slotrec = reinterpret_cast<float4 *>(base + p.rec_off);
    a.part = reinterpret_cast<float4 *>(base + p.part_off);
    a.part_cap = (unsigned)((p.slice_off - p.part_off) / sizeof(float4));
    a.slices = reinterpret_cast<float *>(base + p.slice_off);
    // draft-token logits are gathered wherever the finalize forms log-ratios
    a.gx = (a.mode != MODE_CONF && a.nd_rows > 0) ? reinterpret_cast<float *>(base + p.gx_off) : nullptr;
    if (a.mode != MODE_STOCHASTIC && !a.pre) {
        // no draw follows the stream: the tiling of that mode class (more,
        // smaller units, no tail; the workspace has room for either)
        Plan q;
        plan_tiles(a.B, a.rows, a.V, dtype == SPEC_BF16 ? 2 : 4, false, q);
        p.nT = q.nT;
        p.TS = q.TS;
        p.B1 = q.B1;
        p.nT2 = q.nT2;
        p.TS2 = q.TS2;
        p.head_units = q.head_units;
        p.units = q.units;
    }
    a.nT = p.nT;
    a.TS = p.TS;
    a.per_seq = (unsigned)a.rows * (unsigned)p.nT;
    a.B1 = p.B1;
    a.nT2 = p.nT2;
    a.TS2 = p.TS2;
    a.per_seq2 = (unsigned)a.rows * (unsigned)p.nT2;
    a.head_units = (unsigned)p.head_units;
    a.nR = p.nR;
    a.nslice = p.nslice;
    a.sstride = p.sstride;
    a.units = (unsigned)p.units;
    a.res_units = a.mode == MODE_STOCHASTIC ? (unsigned)a.B * (unsigned)p.nR : 0u;
    a.inv_log_v = (float)(1.0 / std::log((double)a.V));
    a.spin_limit = g_wait_limit.load();
    // the entropy moment of target rows feeds pos_stats and FLy's gate only
    a.need_ent = (a.pos_stats != nullptr || a.mode == MODE_FLY) ? 1 : 0;
    int grid = 1;
    const bool temp = a.inv_temp != nullptr || a.pre;
    // the staging-buffer ring streams the launches with no draw
    const bool ring = SV_STREAM_RING && !temp && a.mode != MODE_STOCHASTIC;
    const int variant = temp ? 1 : (ring ? 2 : 0);
    int rc = grid_for(dtype, variant, p.units, &grid);
    if (rc != SPEC_OK) return rc;
    const unsigned long long lazy = (unsigned long long)SV_LAZY_ROUNDS * (unsigned long long)grid * NWARP;
    a.lazy_from = p.units > lazy ? (unsigned)(p.units - lazy) : 0u;
    const unsigned long long res_lazy = (unsigned long long)SV_RES_LAZY * (unsigned long long)grid * NWARP / 4ull;
    a.res_lazy_from = a.res_units > res_lazy ? (unsigned)(a.res_units - res_lazy) : 0u;
    cudaError_t e = cudaMemsetAsync(ws, 0, p.zero_bytes, st);
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "workspace reset failed: %s", cudaGetErrorString(e));
    if (a.pre) {
        NucleusArgs n;
        n.zt = a.zt;
        n.zd = a.zd;
        n.ts = a.ts;
        n.ds = a.ds;
        n.B = a.B;
        n.K = a.K;
        n.V = a.V;
        n.nt_rows = a.nt_rows;
        n.nd_rows = a.nd_rows;
        n.t_vec_ok = a.t_vec_ok;
        n.d_vec_ok = a.d_vec_ok;
        n.bf16 = dtype == SPEC_BF16 ? 1 : 0;
        n.draft_len = a.draft_len;
        n.inv_temp = a.inv_temp;
        n.top_p = top_p;
        n.need_ent = a.need_ent;
        n.rec = a.part;
        n.zth = const_cast<float *>(a.zth);
        n.status = a.ctr + CTR_STATUS;
        n.row_ctr = a.ctr + CTR_NUC_ROW;
        e = launch_nucleus(n, st);
        if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "nucleus launch failed: %s", cudaGetErrorString(e));
    }
    if (a.pre) {
        // after the nucleus pass, as a programmatic dependent launch: its
        // blocks are scheduled as that kernel's end (0.5% of a top-p call)
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)grid);
        cfg.blockDim = dim3(NT);
        cfg.dynamicSmemBytes = kDynSmem;
        cfg.stream = st;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        at[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        e = dtype == SPEC_BF16 ? cudaLaunchKernelEx(&cfg, verify_kernel<__nv_bfloat16, 2>, a)
                               : cudaLaunchKernelEx(&cfg, verify_kernel<float, 2>, a);
        if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(e));
        return SPEC_OK;
    }
    if (dtype == SPEC_BF16) {
        if (temp)
            a.zth ? verify_kernel<__nv_bfloat16, 2><<<grid, NT, kDynSmem, st>>>(a)
                  : verify_kernel<__nv_bfloat16, 1><<<grid, NT, kDynSmem, st>>>(a);
        else if (ring)
            verify_kernel<__nv_bfloat16, 0, true><<<grid, NT, kDynSmem, st>>>(a);
        else
            verify_kernel<__nv_bfloat16, 0><<<grid, NT, kDynSmem, st>>>(a);
    } else {
        if (temp)
            a.zth ? verify_kernel<float, 2><<<grid, NT, kDynSmem, st>>>(a)
                  : verify_kernel<float, 1><<<grid, NT, kDynSmem, st>>>(a);
        else if (ring)
            verify_kernel<float, 0, true><<<grid, NT, kDynSmem, st>>>(a);
        else
            verify_kernel<float, 0><<<grid, NT, kDynSmem, st>>>(a);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(e));
    return SPEC_OK;
}

static int check_common(int B, int K, int V, int dtype) {
    if (B < 1) return fail(SPEC_ERR_INVALID_ARG, "B must be >= 1 (got %d)", B);
    // the draw record packs the sequence index as 64 b + 2 n + bonus in an int
    if (B > SPEC_MAX_B) return fail(SPEC_ERR_UNSUPPORTED, "B must be <= %d (got %d)", SPEC_MAX_B, B);
    if (K < 1 || K > SPEC_MAX_K) return fail(SPEC_ERR_UNSUPPORTED, "K must be in [1, %d] (got %d)", SPEC_MAX_K, K);
    if (V < 2 || V > SPEC_MAX_V) return fail(SPEC_ERR_UNSUPPORTED, "V must be in [2, %d] (got %d)", SPEC_MAX_V, V);
    if (dtype != SPEC_F32 && dtype != SPEC_BF16) return fail(SPEC_ERR_UNSUPPORTED, "unknown dtype %d", dtype);
    for (int rows : {K, K + 1, 2 * K + 1})
        for (bool draw : {false, true}) {
            Plan pl;
            plan_tiles(B, rows, V, dtype == SPEC_BF16 ? 2 : 4, draw, pl);
            if (pl.units >= (1ull << 31)) return fail(SPEC_ERR_UNSUPPORTED, "batch too large (B=%d)", B);
        }
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
    plan_workspace(p->B, 2 * p->K + 1, p->K + 1, p->V, p->dtype == SPEC_BF16 ? 2 : 4, true, pl);
    return pl.bytes;
}

size_t spec_confidence_workspace_size(int32_t B, int32_t K, int32_t V, int32_t dtype) {
    if (check_common(B, K, V, dtype) != SPEC_OK) return 0;
    Plan pl;
    plan_workspace(B, K, K, V, dtype == SPEC_BF16 ? 2 : 4, false, pl);
    return pl.bytes;
}

}  // extern "C"

static int verify_impl(const spec_verify_params *p, const void *target_logits, const void *draft_logits,
                       const int32_t *draft_tokens, const int32_t *draft_len, const float *inv_temp,
                       float top_p, const float *uniforms,
                       int32_t *out_tokens, int32_t *accepted_len, float *pos_stats, const float *est_params,
                       float *feature, float *conf, void *workspace, size_t workspace_bytes, void *stream) {
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
    // the tiling follows the rows actually streamed; the layout has room for
    // either row count, so spec_workspace_size covers both
    const int rows = draft_logits ? 2 * p->K + 1 : p->K + 1;
    Plan pl;
    plan_workspace(p->B, rows, draft_logits ? p->K + 1 : 2 * p->K + 1, p->V, es, p->mode == SPEC_STOCHASTIC, pl);
    if (workspace_bytes < pl.bytes)
        return fail(SPEC_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes", workspace_bytes, pl.bytes);

    Args a;
    memset(&a, 0, sizeof a);
    a.zt = target_logits;
    a.zd = draft_logits;
    a.ts = ts;
    a.ds = ds;
    a.x = draft_tokens;
    a.draft_len = draft_len;
    a.inv_temp = inv_temp;
    a.pre = top_p < 1.f ? 1 : 0;
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
    return launch(a, pl, p->dtype, workspace, stream, top_p);
}

extern "C" {

int spec_verify(const spec_verify_params *p, const void *target_logits, const void *draft_logits,
                const int32_t *draft_tokens, const float *uniforms, int32_t *out_tokens,
                int32_t *accepted_len, float *pos_stats, const float *est_params, float *feature,
                float *conf, void *workspace, size_t workspace_bytes, void *stream) {
    return verify_impl(p, target_logits, draft_logits, draft_tokens, nullptr, nullptr, 1.f, uniforms, out_tokens,
                       accepted_len, pos_stats, est_params, feature, conf, workspace, workspace_bytes, stream);
}

int spec_verify_ragged(const spec_verify_params *p, const void *target_logits, const void *draft_logits,
                       const int32_t *draft_tokens, const int32_t *draft_len, const float *uniforms,
                       int32_t *out_tokens, int32_t *accepted_len, float *pos_stats, const float *est_params,
                       float *feature, float *conf, void *workspace, size_t workspace_bytes, void *stream) {
    if (!draft_len) {
        g_err = "draft_len is NULL";
        return SPEC_ERR_INVALID_ARG;
    }
    return verify_impl(p, target_logits, draft_logits, draft_tokens, draft_len, nullptr, 1.f, uniforms, out_tokens,
                       accepted_len, pos_stats, est_params, feature, conf, workspace, workspace_bytes, stream);
}

int spec_verify_temperature(const spec_verify_params *p, const void *target_logits, const void *draft_logits,
                            const int32_t *draft_tokens, const int32_t *draft_len, const float *inv_temperature,
                            const float *uniforms, int32_t *out_tokens, int32_t *accepted_len, float *pos_stats,
                            const float *est_params, float *feature, float *conf, void *workspace,
                            size_t workspace_bytes, void *stream) {
    if (!inv_temperature) {
        g_err = "inv_temperature is NULL";
        return SPEC_ERR_INVALID_ARG;
    }
    return verify_impl(p, target_logits, draft_logits, draft_tokens, draft_len, inv_temperature, 1.f, uniforms,
                       out_tokens, accepted_len, pos_stats, est_params, feature, conf, workspace, workspace_bytes,
                       stream);
}

int spec_verify_top_p(const spec_verify_params *p, const void *target_logits, const void *draft_logits,
                      const int32_t *draft_tokens, const int32_t *draft_len, const float *inv_temperature,
                      float top_p, const float *uniforms, int32_t *out_tokens, int32_t *accepted_len,
                      float *pos_stats, const float *est_params, float *feature, float *conf, void *workspace,
                      size_t workspace_bytes, void *stream) {
    if (!(top_p > 0.f && top_p <= 1.f)) {
        g_err = "top_p must be in (0, 1]";
        return SPEC_ERR_INVALID_ARG;
    }
    return verify_impl(p, target_logits, draft_logits, draft_tokens, draft_len, inv_temperature, top_p, uniforms,
                       out_tokens, accepted_len, pos_stats, est_params, feature, conf, workspace, workspace_bytes,
                       stream);
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
    plan_workspace(B, K, K, V, es, false, pl);
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


uint32_t spec_debug_set_wait_limit(uint32_t polls) { return g_wait_limit.exchange(polls); }

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

// Status word of the last static call on the current device: read straight
// from the static array through its looked-up device address (no allocation).
int spec_static_device_status(int32_t *status_out) {
    g_err.clear();
    if (!status_out) return fail(SPEC_ERR_INVALID_ARG, "NULL argument");
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "cudaGetDevice failed: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return fail(SPEC_ERR_UNSUPPORTED, "device index %d out of range", dev);
    void *ws = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_static_mu);
        ws = g_static_ptr[dev];
    }
    if (!ws) {
        *status_out = SPEC_OK;   // no static call on this device yet
        return SPEC_OK;
    }
    return spec_get_device_status(ws, status_out);
}

}  // extern "C"
