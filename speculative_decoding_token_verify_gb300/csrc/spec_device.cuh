// spec_device.cuh -- device building blocks of the verification pass (sm_103a).
//
// Row statistics are kept as an online "softmax accumulator" over a set of
// logits z_v of one vocabulary row ("Speculative Decoding: как черновая
// модель ускоряет генерацию LLM без потери качества", "Математика
// верификации": p(x) and q(x) are softmaxes of the target's and the draft's
// logits):
//
//   M  running max of z                      (fp32)
//   I  lowest index attaining M              (argmax, ties -> lowest index)
//   R  sum over v != I of 2^{(z_v - M) log2e} (the complement mass; the argmax
//      term is exactly 1 and kept out so that 1 - q_max = R/(1+R) never
//      cancels)
//   T  sum over v of 2^{y_v} y_v, y_v = (z_v - M) log2e  (entropy moment)
//
// From these: lse = M + ln(1 + R); normalised entropy
// h = (ln(1+R) - T ln2 / (1+R)) / ln V ("Training-Free Loosely Speculative
// Decoding", 2.A.1); logit(q_max) = -ln R ("Verificación Adaptativa sin una
// cabeza de confianza", "Puntuar la Distribución").
//
// Two accumulators merge associatively (winner = larger M, then lower I);
// every reduction in this library runs in a fixed order, so results are
// bit-reproducible.
//
// Temperature. With an inverse temperature s > 0 the distributions are
// softmax(s z) ("Speculative Decoding: ...", "Математика верификации" holds
// for any pair of distributions the two models sample from). M and I stay in
// raw logit units (s does not move the argmax); R and T are sums over the
// processed exponents y_v = (z_v - M) s log2e. Every function below takes the
// exponent scale sL = s log2e (default log2e, s = 1); then lse = s M + ln(1+R)
// and h and logit(q_max) keep their formulas.
//
// Exponents in the streaming loop are one fused multiply-add each,
// fma(z, sL, -fl(ref sL)): the product z sL is exact inside the FMA, so the
// only error beyond the final rounding is the rounding of ref sL itself,
// eps = ref sL - fl(ref sL), an offset shared by every term taken against
// that reference (it grows with |s ref|: 6e-5 at s = 100 and logits near
// 10). eps is exact by another FMA, fma(ref, sL, -fl(ref sL)), and the
// accumulator folds it into the exponent of each change of reference and of
// the final scale, so the sums come out as if every exponent had been exact:
// the same accuracy as forming z - ref first, at one instruction per pair of
// logits instead of two. With kSub the scalar folds (acc_chunk) form
// differences first.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace sv {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// lower clamp of exponents (log2 units): 2^-200 is 0 in fp32 and keeps
// 0 * y finite for masked (-inf) logits
constexpr float kYMin = -200.0f;
// cap of logit(q_max) = -ln R (q_max within 1e-13 of 1; also R = 0). Every
// term of a complement R >= e^-30 over at most 2^20 tokens that matters is
// a normal fp32 number, so the cap is exact under flush-to-zero arithmetic.
constexpr float kFeatureClamp = 30.0f;

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000u); }

// 2^x with the hardware approximation (ex2.approx.ftz.f32)
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

struct RowAcc {
    float M;
    float R;
    float T;
    int I;
};

__device__ __forceinline__ RowAcc acc_empty() {
    RowAcc a;
    a.M = neg_inf();
    a.R = 0.f;
    a.T = 0.f;
    a.I = 0x7fffffff;
    return a;
}

// a (+) b. Symmetric: merge(a, b) and merge(b, a) give identical bits.
__device__ __forceinline__ RowAcc acc_merge(const RowAcc &a, const RowAcc &b, float sL = kLog2e) {
    if (b.M == neg_inf()) return a;
    if (a.M == neg_inf()) return b;
    const bool aw = (a.M > b.M) || (a.M == b.M && a.I < b.I);
    RowAcc w = aw ? a : b;
    const RowAcc &l = aw ? b : a;
    const float d = (l.M - w.M) * sL;       // <= 0
    const float al = ex2(d);
    const float sl = 1.f + l.R;             // loser's total mass incl. its max
    w.R = fmaf(al, sl, w.R);
    w.T = fmaf(al, fmaf(d, sl, l.T), w.T);
    return w;
}

// Fold E logits z[0..E) with global indices base..base+E-1 (ascending) into s.
// Entries equal to -inf contribute nothing.
template <int E, bool kSub = false>
__device__ __forceinline__ void acc_chunk(RowAcc &s, const float (&z)[E], int base, float sL = kLog2e) {
    float c = z[0];
#pragma unroll
    for (int j = 1; j < E; ++j) c = fmaxf(c, z[j]);
    if (c > s.M) {
        // new running maximum: the old maximum joins the complement
        if (s.M != neg_inf()) {
            const float d = (s.M - c) * sL;
            const float al = ex2(d);
            const float st = 1.f + s.R;
            s.T = al * fmaf(d, st, s.T);
            s.R = al * st;
        }
        s.M = c;
        int jf = E - 1;
#pragma unroll
        for (int j = E - 1; j >= 0; --j)
            if (z[j] == c) jf = j;
        s.I = base + jf;
        const float ml = c * sL;
        float r = 0.f, t = 0.f;
#pragma unroll
        for (int j = 0; j < E; ++j) {
            const float y = fmaxf(kSub ? (z[j] - c) * sL : fmaf(z[j], sL, -ml), kYMin);
            const float e = ex2(y);
            if (j != jf) {
                r += e;
                t = fmaf(e, y, t);
            }
        }
        s.R += r;
        s.T += t;
    } else if (s.M != neg_inf()) {
        const float ml = s.M * sL;
        float r = 0.f, t = 0.f;
#pragma unroll
        for (int j = 0; j < E; ++j) {
            const float y = fmaxf(kSub ? (z[j] - s.M) * sL : fmaf(z[j], sL, -ml), kYMin);
            const float e = ex2(y);
            r += e;
            t = fmaf(e, y, t);
        }
        s.R += r;
        s.T += t;
    }
}

__device__ __forceinline__ RowAcc shfl_xor_acc(const RowAcc &a, int o) {
    RowAcc b;
    b.M = __shfl_xor_sync(0xffffffffu, a.M, o);
    b.R = __shfl_xor_sync(0xffffffffu, a.R, o);
    b.T = __shfl_xor_sync(0xffffffffu, a.T, o);
    b.I = __shfl_xor_sync(0xffffffffu, a.I, o);
    return b;
}

// butterfly: every lane ends with the same merged value
__device__ __forceinline__ RowAcc warp_merge(RowAcc a, float sL = kLog2e) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = acc_merge(a, shfl_xor_acc(a, o), sL);
    return a;
}

__device__ __forceinline__ float4 acc_pack(const RowAcc &a) {
    return make_float4(a.M, a.R, a.T, __int_as_float(a.I));
}

__device__ __forceinline__ RowAcc acc_unpack(const float4 &v) {
    RowAcc a;
    a.M = v.x;
    a.R = v.y;
    a.T = v.z;
    a.I = __float_as_int(v.w);
    return a;
}

// ---- packed arithmetic (sm_100+ f32x2 and bf16x2 forms) -------------------

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2,%3};\n\tmov.b64 rb, {%4,%5};\n\tmov.b64 rc, {%6,%7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0,%1}, rd;}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
    float2 d;
    asm("{.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2,%3};\n\tmov.b64 rb, {%4,%5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0,%1}, rd;}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// pair arithmetic used by the hot loop: f32x2 instructions, or two scalar
// ones when SV_PACKED is 0
#ifndef SV_PACKED
#define SV_PACKED 1
#endif
__device__ __forceinline__ float2 pfma(float2 a, float2 b, float2 c) {
#if SV_PACKED
    return ffma2(a, b, c);
#else
    return make_float2(fmaf(a.x, b.x, c.x), fmaf(a.y, b.y, c.y));
#endif
}

__device__ __forceinline__ float2 padd(float2 a, float2 b) {
#if SV_PACKED
    return fadd2(a, b);
#else
    return make_float2(a.x + b.x, a.y + b.y);
#endif
}

// elementwise max of two bf16 pairs
__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// ---- streaming accumulator (the hot loop) ---------------------------------
//
// Per thread, over the 16-byte chunks of one tile, with a lazy reference mr:
// exponents are taken relative to mr, which only moves when a chunk max
// exceeds it by more than kRescale processed nats, i.e. kRescale / s logit
// units (so terms stay below e^8 and the rescale branch is rare after the
// first chunk). The running max bv and the
// chunk holding it (bk) are tracked per chunk; the mass of that chunk (C) is
// kept apart from the rest (S), so that the complement mass R never has to be
// formed as a difference; its bits are kept too, so that stream_finish() can
// locate the argmax and sum its other elements without a reload, and return
// the canonical RowAcc. Logits below kMaskFloor count as masked (zero mass).

constexpr float kMaskFloor = -1.0e29f;
constexpr float kRescale = 8.0f;
constexpr uint32_t kMaskBf16x2 = 0xF149F149u;   // bf16 pair (-9.95e29, -9.95e29)
constexpr float kMaskF32 = -1.0e30f;

struct StreamAcc {
    float mr;    // reference logit
    float mrL;   // fl(mr * sL)
    float eps;   // mr * sL - mrL, exact (the offset every exponent against mr carries)
    float mrh;   // mr + rs, rs = kRescale / s (a chunk max above it moves the reference)
    float S;     // sum of 2^{(z - mr) log2e} over chunks other than the best one
    float C;     // the same sum over the best chunk
    float2 T;    // sum of 2^y * y, y = (z - mr) log2e (entropy moment, pairwise)
    float bv;    // running max
    int bk;      // chunk (vector) index holding bv
    uint4 bw;    // that chunk's bits, captured by the caller (so finishing needs no reload)
};

__device__ __forceinline__ StreamAcc stream_init(float sL = kLog2e, float rs = kRescale) {
    StreamAcc s;
    s.mr = kMaskFloor;
    s.mrL = kMaskFloor * sL;
    s.eps = fmaf(kMaskFloor, sL, -s.mrL);
    s.mrh = kMaskFloor + rs;
    s.S = 0.f;
    s.C = 0.f;
    s.T = make_float2(0.f, 0.f);
    s.bv = neg_inf();
    s.bk = 0;
    s.bw = make_uint4(0u, 0u, 0u, 0u);
    return s;
}

// Move the reference to c. The sums carry 2^eps_old (and T also eps_old S);
// rescaled with the exponent d = (mr - c) sL + eps_c - eps_old they carry
// 2^eps_c, like the terms taken against c from now on.
__device__ __forceinline__ void stream_rescale(StreamAcc &s, float c, float sL, float rs) {
    const float cL = c * sL;
    const float ce = fmaf(c, sL, -cL);
    const float d = fmaf(s.mr - c, sL, ce - s.eps);
    const float al = ex2(d);
    const float t = al * fmaf(d, s.S + s.C, s.T.x + s.T.y);
    s.T = make_float2(t, 0.f);
    s.S *= al;
    s.C *= al;
    s.mr = c;
    s.mrL = cL;
    s.eps = ce;
    s.mrh = c + rs;
}

// fold the exponentials of one chunk given as fp32 pairs
template <int NP, bool kEnt>
__device__ __forceinline__ void stream_fold(StreamAcc &s, const float2 (&z)[NP], float c, int k, float sL,
                                            float rs) {
    if (c > s.mrh) stream_rescale(s, c, sL, rs);
    const bool nb = c > s.bv;
    s.bv = nb ? c : s.bv;
    s.bk = nb ? k : s.bk;
    const float2 L2 = make_float2(sL, sL);
    const float2 ml = make_float2(-s.mrL, -s.mrL);
    float2 e[NP];
    float2 y[NP];
#pragma unroll
    for (int p = 0; p < NP; ++p) {
        y[p] = pfma(z[p], L2, ml);
        e[p] = make_float2(ex2(y[p].x), ex2(y[p].y));
    }
    float2 a = e[0];
#pragma unroll
    for (int p = 1; p < NP; ++p) a = padd(a, e[p]);
    const float cs = a.x + a.y;
    if constexpr (kEnt) {
#pragma unroll
        for (int p = 0; p < NP; ++p) s.T = pfma(e[p], y[p], s.T);
    }
    s.S += nb ? s.C : cs;
    s.C = nb ? cs : s.C;
}

template <typename T, bool kEnt>
__device__ __forceinline__ void stream_chunk(StreamAcc &s, uint4 w, int k, float sL = kLog2e,
                                             float rs = kRescale) {
    if constexpr (sizeof(T) == 2) {
        if constexpr (kEnt) {
            w.x = bmax2(w.x, kMaskBf16x2);
            w.y = bmax2(w.y, kMaskBf16x2);
            w.z = bmax2(w.z, kMaskBf16x2);
            w.w = bmax2(w.w, kMaskBf16x2);
        }
        const uint32_t m = bmax2(bmax2(w.x, w.y), bmax2(w.z, w.w));
        const float c = fmaxf(bf16_lo(m), bf16_hi(m));
        float2 z[4];
        z[0] = make_float2(bf16_lo(w.x), bf16_hi(w.x));
        z[1] = make_float2(bf16_lo(w.y), bf16_hi(w.y));
        z[2] = make_float2(bf16_lo(w.z), bf16_hi(w.z));
        z[3] = make_float2(bf16_lo(w.w), bf16_hi(w.w));
        stream_fold<4, kEnt>(s, z, c, k, sL, rs);
    } else {
        float2 z[2];
        z[0] = make_float2(__uint_as_float(w.x), __uint_as_float(w.y));
        z[1] = make_float2(__uint_as_float(w.z), __uint_as_float(w.w));
        if constexpr (kEnt) {
            z[0].x = fmaxf(z[0].x, kMaskF32);
            z[0].y = fmaxf(z[0].y, kMaskF32);
            z[1].x = fmaxf(z[1].x, kMaskF32);
            z[1].y = fmaxf(z[1].y, kMaskF32);
        }
        const float c = fmaxf(fmaxf(z[0].x, z[0].y), fmaxf(z[1].x, z[1].y));
        stream_fold<2, kEnt>(s, z, c, k, sL, rs);
    }
}

// ---- element access -------------------------------------------------------

template <typename T> struct Elem;

template <> struct Elem<float> {
    static constexpr int kPerVec = 4;   // elements per 16-byte vector
    __device__ __forceinline__ static float load(const float *p) { return __ldg(p); }
    __device__ __forceinline__ static void unpack(const uint4 &w, float (&z)[4]) {
        z[0] = __uint_as_float(w.x);
        z[1] = __uint_as_float(w.y);
        z[2] = __uint_as_float(w.z);
        z[3] = __uint_as_float(w.w);
    }
};

template <> struct Elem<__nv_bfloat16> {
    static constexpr int kPerVec = 8;
    __device__ __forceinline__ static float load(const __nv_bfloat16 *p) {
        const unsigned short h = __ldg(reinterpret_cast<const unsigned short *>(p));
        return __uint_as_float(static_cast<uint32_t>(h) << 16);
    }
    // bf16 -> fp32 is exact: the bf16 bits are the high half of the fp32 bits
    __device__ __forceinline__ static void unpack(const uint4 &w, float (&z)[8]) {
        z[0] = __uint_as_float(w.x << 16);
        z[1] = __uint_as_float(w.x & 0xffff0000u);
        z[2] = __uint_as_float(w.y << 16);
        z[3] = __uint_as_float(w.y & 0xffff0000u);
        z[4] = __uint_as_float(w.z << 16);
        z[5] = __uint_as_float(w.z & 0xffff0000u);
        z[6] = __uint_as_float(w.w << 16);
        z[7] = __uint_as_float(w.w & 0xffff0000u);
    }
};

__device__ __forceinline__ uint4 ldg_stream(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// 8 consecutive logits v..v+7 of a row as fp32; entries >= V read as -inf.
// `vec_ok`: the row start is 16-byte aligned (then v, a multiple of 8, is too).
template <typename T>
__device__ __forceinline__ void load8(const T *row, int v, int V, bool vec_ok, float (&z)[8]) {
    if (vec_ok && v + 8 <= V) {
        if constexpr (Elem<T>::kPerVec == 8) {
            Elem<T>::unpack(__ldg(reinterpret_cast<const uint4 *>(row + v)), z);
        } else {
            float a[4], b[4];
            Elem<T>::unpack(__ldg(reinterpret_cast<const uint4 *>(row + v)), a);
            Elem<T>::unpack(__ldg(reinterpret_cast<const uint4 *>(row + v + 4)), b);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                z[j] = a[j];
                z[4 + j] = b[j];
            }
        }
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) z[j] = (v + j < V) ? Elem<T>::load(row + v + j) : neg_inf();
    }
}

// Canonical RowAcc of one thread's streamed chunks; vector 0 of the tile has
// row index `vb`.
// The final scale's exponent d = (mr - bv) sL - eps takes the offset out.
template <typename T>
__device__ __forceinline__ RowAcc stream_finish(const StreamAcc &s, int vb, float sL = kLog2e) {
    constexpr int E = Elem<T>::kPerVec;
    RowAcc a = acc_empty();
    if (!(s.bv > kMaskFloor)) return a;          // nothing unmasked seen
    float z[E];
    Elem<T>::unpack(s.bw, z);
    int jf = E - 1;
#pragma unroll
    for (int j = E - 1; j >= 0; --j)
        if (z[j] == s.bv) jf = j;
    float crest = 0.f;
#pragma unroll
    for (int j = 0; j < E; ++j)
        if (j != jf) crest += ex2(fmaf(z[j], sL, -s.mrL));
    const float d = fmaf(s.mr - s.bv, sL, -s.eps);   // <= 0 (up to eps): mr is some chunk max <= bv
    const float al = ex2(d);
    a.M = s.bv;
    a.R = al * (s.S + crest);
    a.T = al * fmaf(d, s.S + s.C, s.T.x + s.T.y);
    a.I = vb + s.bk * E + jf;
    return a;
}

}  // namespace sv
