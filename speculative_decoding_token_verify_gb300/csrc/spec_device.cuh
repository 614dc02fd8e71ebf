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
// logit(q_max) when the complement mass R is exactly zero
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
__device__ __forceinline__ RowAcc acc_merge(const RowAcc &a, const RowAcc &b) {
    if (b.M == neg_inf()) return a;
    if (a.M == neg_inf()) return b;
    const bool aw = (a.M > b.M) || (a.M == b.M && a.I < b.I);
    RowAcc w = aw ? a : b;
    const RowAcc &l = aw ? b : a;
    const float d = (l.M - w.M) * kLog2e;   // <= 0
    const float al = ex2(d);
    const float sl = 1.f + l.R;             // loser's total mass incl. its max
    w.R = fmaf(al, sl, w.R);
    w.T = fmaf(al, fmaf(d, sl, l.T), w.T);
    return w;
}

// Fold E logits z[0..E) with global indices base..base+E-1 (ascending) into s.
// Entries equal to -inf contribute nothing.
template <int E>
__device__ __forceinline__ void acc_chunk(RowAcc &s, const float (&z)[E], int base) {
    float c = z[0];
#pragma unroll
    for (int j = 1; j < E; ++j) c = fmaxf(c, z[j]);
    if (c > s.M) {
        // new running maximum: the old maximum joins the complement
        if (s.M != neg_inf()) {
            const float d = (s.M - c) * kLog2e;
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
        const float ml = c * kLog2e;
        float r = 0.f, t = 0.f;
#pragma unroll
        for (int j = 0; j < E; ++j) {
            const float y = fmaxf(fmaf(z[j], kLog2e, -ml), kYMin);
            const float e = ex2(y);
            if (j != jf) {
                r += e;
                t = fmaf(e, y, t);
            }
        }
        s.R += r;
        s.T += t;
    } else if (s.M != neg_inf()) {
        const float ml = s.M * kLog2e;
        float r = 0.f, t = 0.f;
#pragma unroll
        for (int j = 0; j < E; ++j) {
            const float y = fmaxf(fmaf(z[j], kLog2e, -ml), kYMin);
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
__device__ __forceinline__ RowAcc warp_merge(RowAcc a) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = acc_merge(a, shfl_xor_acc(a, o));
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

}  // namespace sv
