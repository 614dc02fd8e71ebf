// spec_nucleus.cu -- per-row nucleus (top-p) statistics for verification at a
// sampling top-p ("Verificación Adaptativa sin una cabeza de confianza",
// "Benchmarks": serving samples with top-p; "Speculative Decoding: как
// черновая модель ускоряет генерацию LLM без потери качества",
// "Математика верификации": the rule is lossless for the processed p, q).
//
// The nucleus of a row is every token whose logit is at least z*, the largest
// logit value whose upper mass (the tokens with logit >= z*) reaches top_p of
// the row's mass under p = softmax(s z); tokens tied at z* are all kept.
//
// Two kernels find z*. Both take one row per CTA at a time (persistent over
// rows) and re-read the row from L2 between passes, with two CTAs per SM so
// that the rows in flight stay L2-resident:
//  * nucleus_row_kernel (V up to 256 K): bins the weights by their float
//    encoding (see the comments above it);
//  * nucleus_kernel (larger V, where 32-bit bin counters would lose
//    precision): the passes below.
//
// The passes of one row:
//
//  A. max M, its lowest index I, and the smallest finite logit;
//  B. weights e_v = 2^((z_v - M) s log2e), in 2^-40 fixed point, summed for
//     the total and, for the tokens within ln(V / (1 - top_p)) + 1 nats of
//     M (the boundary cannot lie farther), binned over the processed
//     distance into 256 bins with per-warp 64-bit shared atomics (integer
//     sums: exact, order-independent); the first bin (from d = 0) whose
//     running mass reaches top_p of the total holds z*;
//  C. that bin's tokens (d is monotone in z, so they form a contiguous key
//     range): their key range, and the tokens copied to shared memory;
//  D. while the range holds more than one key: a 256-way histogram over the
//     key range (of the copied tokens; of the row if they did not fit), the
//     first sub-range whose running mass reaches the target;
//  E. the nucleus statistics in the RowAcc form of spec_device.cuh: R = the
//     mass of nucleus tokens other than I, T = the entropy moment, fp32 in a
//     fixed order.
//
// The record (M, R, T, I) and z* go to the caller's workspace, where the
// verification kernel reads them in place of its streamed row statistics.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <type_traits>

#include "spec_device.cuh"
#include "spec_nucleus.cuh"
#include "spec_verify.h"

namespace sv {
namespace nuc {

#ifndef SV_NUC_CTAS
#define SV_NUC_CTAS 2   // CTAs per SM: rows in flight stay L2-resident
#endif

constexpr int NT = 256;
constexpr int NW = NT / 32;
constexpr int kBins = 256;
constexpr int kMaxRefine = 6;   // key-range passes (<= 4 needed for 32-bit keys)
constexpr unsigned kFull = 0xffffffffu;
typedef unsigned long long u64;

// Order-preserving integer key of a logit, in the element's own precision
// (consecutive representable values get consecutive keys; -0 and +0 share one).
template <typename T> struct Key;
template <> struct Key<float> {
    __device__ static uint32_t of(float z) {
        const uint32_t u = __float_as_uint(z == 0.f ? 0.f : z);
        return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    }
    __device__ static float value(uint32_t k) {
        return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
    }
};
template <> struct Key<__nv_bfloat16> {
    __device__ static uint32_t of(float z) {   // z holds a bf16 value exactly
        const uint32_t u = __float_as_uint(z == 0.f ? 0.f : z) >> 16;
        return (u & 0x8000u) ? (~u & 0xffffu) : (u | 0x8000u);
    }
    __device__ static float value(uint32_t k) {
        const uint32_t u = (k & 0x8000u) ? (k & 0x7fffu) : (~k & 0xffffu);
        return __uint_as_float(u << 16);
    }
};

// Visit every element (v, z) of a row: each thread takes 8-element groups
// tid, tid + NT, ..., with 4 groups' loads in flight; entries past V read
// as -inf (zero mass, lowest key) and are visited too. The loop is
// warp-uniform (every lane of a warp makes the same calls), so f may use
// warp-collective operations.
template <typename T, typename F>
__device__ __forceinline__ void for_row(const T *row, int V, bool vec_ok, F &&f) {
    const int ng = (V + 7) >> 3;
    const int lane = threadIdx.x & 31;
    for (int g0 = threadIdx.x - lane; g0 < ng; g0 += 4 * NT) {
        float z[4][8];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int g = g0 + lane + u * NT;
            if (g < ng) {
                load8<T>(row, g * 8, V, vec_ok, z[u]);
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) z[u][j] = neg_inf();
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int j = 0; j < 8; ++j) f((g0 + lane + u * NT) * 8 + j, z[u][j]);
    }
}

constexpr int kCandW = 160;     // boundary-bin tokens kept in shared memory, per warp

struct Shared {
    u64 hist[NW][kBins];          // per-warp histograms
    u64 cfix[NW][kCandW];         // boundary-bin tokens: fixed-point mass
    uint32_t ckey[NW][kCandW];    // ... logit key
    int cv[NW][kCandW];           // ... vocabulary index
    int cnt[NW];                  // tokens each warp found in the boundary bin
    float4 acc[NW];               // per-warp row statistics
    u64 wsum[NW];                 // per-warp scan totals
    float fw[NW][2];              // per-warp float partials
    uint32_t kw[NW][2];
    int sel;                      // selected bin
    u64 sel_above;                // mass above the selected bin
};

__device__ __forceinline__ u64 shfl_up_u64(u64 v, int o) { return __shfl_up_sync(kFull, v, o); }

// Block-wide inclusive scan of one u64 per thread (thread order); also
// returns the block total. SH: a shared-memory struct with u64 wsum[NW].
template <typename SH>
__device__ __forceinline__ u64 block_scan(u64 v, SH &sh, u64 &total) {
    const int l = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const u64 t = shfl_up_u64(v, o);
        if (l >= o) v += t;
    }
    if (l == 31) sh.wsum[w] = v;
    __syncthreads();
    u64 pre = 0, tot = 0;
#pragma unroll
    for (int i = 0; i < NW; ++i) {
        const u64 s = sh.wsum[i];
        if (i < w) pre += s;
        tot += s;
    }
    total = tot;
    return v + pre;
}

// Thread t holds the mass h of bin t: scan the bins in order and select the
// first whose running mass, plus `above`, reaches `tgt`. Returns the bin;
// `above` becomes the mass before it. tgt is lowered to the mass available
// when the bins hold less (only possible through rounding of the total).
template <typename SH>
__device__ __forceinline__ int select_from(SH &sh, u64 h, u64 &tgt, u64 &above) {
    const int t = threadIdx.x;
    u64 tot;
    const u64 incl = block_scan(h, sh, tot) + above;
    if (above + tot < tgt) tgt = above + tot;
    // exactly one thread hits: running sums only grow, `above` stays below
    // tgt and the bins reach it
    const bool hit = incl >= tgt && incl - h < tgt;
    if (t == 0) {
        sh.sel = kBins - 1;
        sh.sel_above = above;
    }
    __syncthreads();
    if (hit) {
        sh.sel = t;
        sh.sel_above = incl - h;
    }
    __syncthreads();
    const int j = sh.sel;
    above = sh.sel_above;
    return j;
}

// Sum the per-warp histograms (thread t owns bin t; they are cleared) and
// select as select_from does.
template <typename SH>
__device__ __forceinline__ int select_bin(SH &sh, u64 &tgt, u64 &above) {
    const int t = threadIdx.x;
    __syncthreads();
    u64 h = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
        h += sh.hist[w][t];
        sh.hist[w][t] = 0ull;
    }
    return select_from(sh, h, tgt, above);
}

__device__ __forceinline__ uint32_t bmin2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("min.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// smallest element of a 16-byte chunk
template <typename T>
__device__ __forceinline__ float chunk_min(const uint4 &w) {
    if constexpr (sizeof(T) == 2) {
        const uint32_t m = bmin2(bmin2(w.x, w.y), bmin2(w.z, w.w));
        return fminf(bf16_lo(m), bf16_hi(m));
    } else {
        return fminf(fminf(__uint_as_float(w.x), __uint_as_float(w.y)),
                     fminf(__uint_as_float(w.z), __uint_as_float(w.w)));
    }
}

template <typename T>
__global__ void __launch_bounds__(NT, SV_NUC_CTAS) nucleus_kernel(const NucleusArgs a) {
    __shared__ Shared sh;
    const int t = threadIdx.x, l = t & 31, w = t >> 5;
    for (int i = t; i < NW * kBins; i += NT) (&sh.hist[0][0])[i] = 0ull;
    const int rows = a.nt_rows + a.nd_rows;
    const int nrow = a.B * rows;
    // tokens farther than this many nats below the maximum hold less than
    // (1 - top_p)/e of a total >= 1, so the boundary is never there
    const float Drel = logf((float)a.V / (1.f - a.top_p)) + 1.f;
    for (int row = blockIdx.x; row < nrow; row += gridDim.x) {
        const int b = row / rows, r = row - b * rows;
        const bool target = r < a.nt_rows;
        const int kb = a.draft_len ? min(max(__ldg(a.draft_len + b), 0), a.K) : a.K;
        const bool verified = target ? r <= kb : r - a.nt_rows < kb;
        if (!verified) {
            if (t == 0) {
                a.rec[row] = acc_pack(acc_empty());
                a.zth[row] = __int_as_float(0x7f800000);
            }
            continue;
        }
        const T *p = target ? static_cast<const T *>(a.zt) + ((long long)b * (a.K + 1) + r) * a.ts
                            : static_cast<const T *>(a.zd) + ((long long)b * a.K + (r - a.nt_rows)) * a.ds;
        const bool vok = target ? a.t_vec_ok != 0 : a.d_vec_ok != 0;
        float s = 1.f;
        if (a.inv_temp) {
            const float si = __ldg(a.inv_temp + b);
            s = (si >= SPEC_MIN_INV_TEMPERATURE && si <= SPEC_MAX_INV_TEMPERATURE) ? si : 1.f;
        }
        const float sL = s * kLog2e;

        // ---- A: the row's statistics (max M, its lowest index I, complement
        // mass R relative to M) with the streaming accumulator, and the
        // smallest logit
        constexpr int E = Elem<T>::kPerVec;
        RowAcc ra = acc_empty();
        float cmin = __int_as_float(0x7f800000);
        if (vok && a.V % E == 0) {
            const uint4 *vp = reinterpret_cast<const uint4 *>(p);
            const int nvec = a.V / E;
            StreamAcc acc = stream_init(sL, __fdiv_rn(kRescale, s));
            for (int k0 = t; k0 < nvec; k0 += 4 * NT) {
                uint4 wv[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int k = k0 + u * NT;
                    if (k < nvec) wv[u] = ldg_stream(vp + k);
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int k = k0 + u * NT;
                    if (k < nvec) {
                        stream_chunk<T, false>(acc, wv[u], k, sL, __fdiv_rn(kRescale, s));
                        if (acc.bk == k) acc.bw = wv[u];
                        cmin = fminf(cmin, chunk_min<T>(wv[u]));
                    }
                }
            }
            ra = stream_finish<T>(acc, 0, sL);
        } else {
            for (int v = t; v < a.V; v += NT) {
                float z[1] = {Elem<T>::load(p + v)};
                acc_chunk<1, true>(ra, z, v, sL);
                cmin = fminf(cmin, z[0]);
            }
        }
        ra = warp_merge(ra, sL);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) cmin = fminf(cmin, __shfl_xor_sync(kFull, cmin, o));
        if (l == 0) {
            sh.acc[w] = acc_pack(ra);
            sh.fw[w][0] = cmin;
        }
        __syncthreads();
        ra = acc_unpack(sh.acc[0]);
        cmin = sh.fw[0][0];
#pragma unroll
        for (int i = 1; i < NW; ++i) {
            ra = acc_merge(ra, acc_unpack(sh.acc[i]), sL);
            cmin = fminf(cmin, sh.fw[i][0]);
        }
        __syncthreads();
        const float M = ra.M;
        const int I = ra.I;
        if (!(M > neg_inf()) || M == __int_as_float(0x7f800000)) {
            // no finite logit: the verification kernel reports the bad row
            if (t == 0) {
                a.rec[row] = acc_pack(acc_empty());
                a.zth[row] = __int_as_float(0x7f800000);
            }
            continue;
        }

        // ---- B: mass histogram of the tokens within Dr = min(s (M - min),
        // Drel) nats of M, over y = (z - M) s log2e (bins of Dr/256 nats)
        const float Dr = fminf((M - cmin) * s, Drel);   // -inf logits: Dr = Drel
        const float ylim = -Dr * kLog2e;                 // y >= ylim <=> binned
        const float ybin = Dr > 0.f ? -(float)kBins * kLn2 / Dr : 0.f;
        auto bin_of = [&](float y) -> int { return min(kBins - 1, (int)(y * ybin)); };
        for_row<T>(p, a.V, vok, [&](int v, float z) {
            const float y = (z - M) * sL;
            if (y >= ylim) atomicAdd(&sh.hist[w][bin_of(y)], __float2ull_rn(ex2(y) * 0x1p40f));
        });
        u64 tgt = (u64)ceil((double)a.top_p * ((double)(1.f + ra.R) * 0x1p40));
        u64 above = 0;
        const int j1 = select_bin(sh, tgt, above);

        // ---- C: the tokens above bin j1 are in the nucleus: their mass
        // (other than I) and entropy moment accumulate per thread; bin j1's
        // tokens (a contiguous key range: y is monotone in z) go to this
        // warp's region of shared memory, in a fixed order
        uint32_t klo = 0xffffffffu, khi = 0u;
        float Ra = 0.f, Ta = 0.f;
        int wc = 0;   // warp-uniform count of bin-j1 tokens seen by this warp
        for_row<T>(p, a.V, vok, [&](int v, float z) {
            const float y = (z - M) * sL;
            const int bn = (v < a.V && y >= ylim) ? bin_of(y) : kBins;
            if (bn < j1) {
                const float e = ex2(y);
                if (v != I) Ra += e;
                Ta = fmaf(e, y, Ta);
            }
            const bool cand = bn == j1;
            const unsigned m = __ballot_sync(kFull, cand);
            if (m) {
                if (cand) {
                    const uint32_t k = Key<T>::of(z);
                    klo = min(klo, k);
                    khi = max(khi, k);
                    const int slot = wc + __popc(m & ((1u << l) - 1u));
                    if (slot < kCandW) {
                        sh.ckey[w][slot] = k;
                        sh.cfix[w][slot] = __float2ull_rn(ex2(y) * 0x1p40f);
                        sh.cv[w][slot] = v;
                    }
                }
                wc += __popc(m);
            }
        });
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            klo = min(klo, __shfl_xor_sync(kFull, klo, o));
            khi = max(khi, __shfl_xor_sync(kFull, khi, o));
        }
        if (l == 0) {
            sh.kw[w][0] = klo;
            sh.kw[w][1] = khi;
            sh.cnt[w] = wc;
        }
        __syncthreads();
        klo = sh.kw[0][0];
        khi = sh.kw[0][1];
        bool fits = true;
#pragma unroll
        for (int i = 0; i < NW; ++i) {
            klo = min(klo, sh.kw[i][0]);
            khi = max(khi, sh.kw[i][1]);
            fits &= sh.cnt[i] <= kCandW;
        }

        // ---- D: refine the key range to one key, 256 sub-ranges a round,
        // over the kept tokens (over the row when they did not fit)
        int it = 0;
        while (klo < khi && it < kMaxRefine) {
            const u64 W = (u64)(khi - klo) + 1ull;
            if (fits) {
                for (int i = t; i < NW * kCandW; i += NT) {
                    const int wi = i / kCandW, si = i - wi * kCandW;
                    if (si < sh.cnt[wi]) {
                        const uint32_t k = sh.ckey[wi][si];
                        if (k >= klo && k <= khi)
                            atomicAdd(&sh.hist[w][(int)(((u64)(khi - k) << 8) / W)], sh.cfix[wi][si]);
                    }
                }
            } else {
                const float zlo = Key<T>::value(klo), zhi = Key<T>::value(khi);
                for_row<T>(p, a.V, vok, [&](int v, float z) {
                    if (v < a.V && z >= zlo && z <= zhi) {
                        const uint32_t k = Key<T>::of(z);
                        const u64 f = __float2ull_rn(ex2((z - M) * sL) * 0x1p40f);
                        atomicAdd(&sh.hist[w][(int)(((u64)(khi - k) << 8) / W)], f);
                    }
                });
            }
            const int j = select_bin(sh, tgt, above);
            // keys of sub-range j: khi - k in [ceil(j W / 256), ceil((j + 1) W / 256) - 1]
            const u64 lo_off = ((u64)j * W + 255ull) >> 8;
            const u64 hi_off = (((u64)(j + 1) * W + 255ull) >> 8) - 1ull;
            const uint32_t nkhi = khi - (uint32_t)lo_off;
            const uint32_t nklo = khi - (uint32_t)hi_off;
            khi = nkhi;
            klo = nklo;
            ++it;
        }
        if (klo < khi && t == 0) atomicMax(a.status, (unsigned)SPEC_ERR_BAD_ROW);   // not reached
        const uint32_t kstar = khi;
        const float zstar = Key<T>::value(kstar);

        // ---- E: nucleus statistics (fixed order): the tokens above bin j1
        // (per thread, from pass C) plus the kept bin-j1 tokens at or above
        // z* (each warp its own, lane-strided in slot order); or, when the
        // bin's tokens did not fit, one more pass over the row
        float R = 0.f, Tm = 0.f;
        if (fits) {
            R = Ra;
            Tm = Ta;
            const int n = sh.cnt[w];
            for (int i = l; i < n; i += 32) {
                if (sh.ckey[w][i] >= kstar) {
                    const float y = (Key<T>::value(sh.ckey[w][i]) - M) * sL;
                    const float e = ex2(y);
                    if (sh.cv[w][i] != I) R += e;
                    Tm = fmaf(e, y, Tm);
                }
            }
        } else {
            for_row<T>(p, a.V, vok, [&](int v, float z) {
                if (v < a.V && z >= zstar) {
                    const float y = (z - M) * sL;
                    const float e = ex2(y);
                    if (v != I) R += e;
                    Tm = fmaf(e, y, Tm);
                }
            });
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            R += __shfl_xor_sync(kFull, R, o);
            Tm += __shfl_xor_sync(kFull, Tm, o);
        }
        if (l == 0) {
            sh.fw[w][0] = R;
            sh.fw[w][1] = Tm;
        }
        __syncthreads();
        if (t == 0) {
            float Rs = 0.f, Ts = 0.f;
            for (int i = 0; i < NW; ++i) {
                Rs += sh.fw[i][0];
                Ts += sh.fw[i][1];
            }
            RowAcc acc;
            acc.M = M;
            acc.R = Rs;
            acc.T = Ts;
            acc.I = I;
            a.rec[row] = acc_pack(acc);
            a.zth[row] = zstar;
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// Mass bins. A token's weight e = 2^(z s log2e - R), R = ceil(M s log2e) an
// integer reference (e <= 1 up to rounding), is binned by the top bits of its
// float encoding -- the exponent and 3 mantissa bits: 8 bins a binade over
// [2^-47, 2) -- and its bin adds the token's 24-bit significand shifted right
// by `ushift`. The sums are integers (exact, independent of order), and a
// bin's mass is its sum times a power of two. Weights below 2^-47 go to bin 0
// (at most V 2^-46 of mass, which only enters the total).
// ---------------------------------------------------------------------------
constexpr int kSub = 3;                                               // mantissa bits in a bin index
constexpr int kBinades = 64;
constexpr int NB = kBinades << kSub;                                  // 512 bins
constexpr uint32_t kLoBits = (uint32_t)(127 - (kBinades - 1)) << 23; // 2^-63
constexpr uint32_t kHiBits = (128u << 23) - 1u;                       // the largest float below 2
constexpr int kBinBase = (int)(kLoBits >> (23 - kSub));
constexpr int kKeyBins = 256;

__device__ __forceinline__ float pow2i(int k) { return __int_as_float((k + 127) << 23); }   // k in [-126, 127]

__device__ __forceinline__ int bin_of(uint32_t b) { return (int)(b >> (23 - kSub)) - kBinBase; }
// The same bin counted from the top (position 0: just below 2, NB - 1: bin 0),
// from the unclamped encoding of a weight: one unsigned min sends weights
// below 2^-63, zero and NaN to the bottom position. A weight of 2 or more
// (only in a row whose bins are taken again) lands on some position.
__device__ __forceinline__ uint32_t pos_of(uint32_t b) {
    return min((kHiBits >> (23 - kSub)) - (b >> (23 - kSub)), (uint32_t)(NB - 1));
}
// mass of one significand unit in bin g: 2^(E - 150 + ushift), E = the bin's
// biased exponent, 128 - kBinades + g / 8
__device__ __forceinline__ float bin_scale(int g, int ushift) { return pow2i((g >> kSub) - kBinades - 22 + ushift); }
// log2 of bin g's lower edge; g = NB gives the top edge
__device__ __forceinline__ float bin_edge(int g) {
    return (float)((g >> kSub) - (kBinades - 1)) + log2f(1.f + (float)(g & ((1 << kSub) - 1)) * (1.f / (1 << kSub)));
}

// Does one of a vector's elements lie in [zl, zh] (exact element values)?
template <typename T>
__device__ __forceinline__ bool vec_in_range(const uint4 &x, float zl, float zh) {
    if constexpr (sizeof(T) == 2) {
        // per-half masks: 0xFFFF where the comparison holds
        const __nv_bfloat162 lo2 = __bfloat162bfloat162(__float2bfloat16_rn(zl));
        const __nv_bfloat162 hi2 = __bfloat162bfloat162(__float2bfloat16_rn(zh));
        const uint32_t wv[4] = {x.x, x.y, x.z, x.w};
        uint32_t any = 0u;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162 *>(&wv[i]);
            any |= __hge2_mask(v, lo2) & __hle2_mask(v, hi2);
        }
        return any != 0u;
    } else {
        const float z[4] = {__uint_as_float(x.x), __uint_as_float(x.y), __uint_as_float(x.z), __uint_as_float(x.w)};
        bool any = false;
#pragma unroll
        for (int i = 0; i < 4; ++i) any |= (z[i] >= zl) & (z[i] <= zh);
        return any;
    }
}

// The same question for a bf16 vector, answered with a superset (pass C's
// exact test follows): with c a bf16 value, rb >= max(zh - c, c - zl) and
// rr > rb^2, take d = v - c rounded to bf16 and q = d d - rr rounded once.
// Rounding is monotone and rb is a bf16 value, so v in [zl, zh] gives
// |d| <= rb, d^2 < rr and q < 0: the sign bit is set. The test is two packed
// FMA-pipe operations a word, against two packed compares and a merge.
struct NearBf16 {
    __nv_bfloat162 c2, nrr2;   // (c, c) and (-rr, -rr)
    __device__ NearBf16(float zl, float zh) {
        const __nv_bfloat16 cb = __float2bfloat16_rn(0.5f * zl + 0.5f * zh);
        const float c = __bfloat162float(cb);
        const float rb = __bfloat162float(__float2bfloat16_ru(fmaxf(__fsub_ru(zh, c), __fsub_ru(c, zl))));
        // rr: above rb^2 by a margin, a bf16 value, and positive (rb = 0)
        float rr = __fmul_ru(__fmul_ru(rb, rb), 1.f + 0x1p-7f);
        rr = fmaxf(__bfloat162float(__float2bfloat16_ru(rr)), 0x1p-100f);
        c2 = __bfloat162bfloat162(cb);
        nrr2 = __bfloat162bfloat162(__float2bfloat16_rn(-rr));
    }
    __device__ __forceinline__ bool operator()(const uint4 &x) const {
        const uint32_t wv[4] = {x.x, x.y, x.z, x.w};
        uint32_t any = 0u;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162 *>(&wv[i]);
            const __nv_bfloat162 d = __hsub2(v, c2);
            const __nv_bfloat162 q = __hfma2(d, d, nrr2);
            any |= *reinterpret_cast<const uint32_t *>(&q);
        }
        return (any & 0x80008000u) != 0u;
    }
};

// Positions in order, thread t holding positions P t .. P t + P - 1 (the
// first n valid) with masses a[] and r[]: the first position with mass whose
// running a-mass, on top of base_a, reaches tgt; when none does (rounding),
// the last position with mass, else 0. Sets the running a- and r-masses
// before it (on top of base_a, base_r) and its own r-mass. Sums in a fixed
// association.
template <int P, int NWARP, typename SH>
__device__ __forceinline__ int select_pos(SH &sh, const float (&a)[P], const float (&r)[P], int n, float tgt,
                                          float base_a, float base_r, float &above_a, float &above_r, float &r_sel) {
    const int t = threadIdx.x, l = t & 31, w = t >> 5;
    float sa = 0.f, sr = 0.f;
#pragma unroll
    for (int p = 0; p < P; ++p) {
        sa += a[p];
        sr += r[p];
    }
    float ia = sa, ir = sr;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float ua = __shfl_up_sync(kFull, ia, o), ur = __shfl_up_sync(kFull, ir, o);
        if (l >= o) {
            ia += ua;
            ir += ur;
        }
    }
    float ea = __shfl_up_sync(kFull, ia, 1), er = __shfl_up_sync(kFull, ir, 1);
    if (l == 0) ea = er = 0.f;
    if (l == 31) {
        sh.wa[w] = ia;
        sh.wr[w] = ir;
    }
    if (t == 0) {
        sh.sel = 0x7fffffff;
        sh.sel_last = -1;
    }
    __syncthreads();
    float pa = base_a, pr = base_r;
    for (int i = 0; i < w; ++i) {
        pa += sh.wa[i];
        pr += sh.wr[i];
    }
    pa += ea;
    pr += er;
    int first = 0x7fffffff, last = -1;
    {
        float x = pa;
#pragma unroll
        for (int p = 0; p < P; ++p) {
            const int pos = P * t + p;
            x += a[p];
            if (pos < n && a[p] > 0.f) {
                if (x >= tgt && first == 0x7fffffff) first = pos;
                last = pos;
            }
        }
    }
    if (first != 0x7fffffff) atomicMin(&sh.sel, first);
    if (last >= 0) atomicMax(&sh.sel_last, last);
    __syncthreads();
    const int s = sh.sel != 0x7fffffff ? sh.sel : max(sh.sel_last, 0);
    if (s / P == t) {
        float xa = pa, xr = pr;
#pragma unroll
        for (int p = 0; p < P; ++p)
            if (p < s - P * t) {
                xa += a[p];
                xr += r[p];
            }
        float rs = 0.f;
#pragma unroll
        for (int p = 0; p < P; ++p)
            if (p == s - P * t) rs = r[p];
        sh.sel_a = xa;
        sh.sel_r = xr;
        sh.sel_rs = rs;
    }
    __syncthreads();
    above_a = sh.sel_a;
    above_r = sh.sel_r;
    r_sel = sh.sel_rs;
    __syncthreads();
    return s;
}

// Block sum of one float per thread (warp order, then warp sums in order);
// the result in every thread.
template <int NWARP, typename SH>
__device__ __forceinline__ float block_sum(SH &sh, float v) {
    const int l = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    if (l == 0) sh.wa[w] = v;
    __syncthreads();
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < NWARP; ++i) s += sh.wa[i];
    __syncthreads();
    return s;
}

// ---------------------------------------------------------------------------
// Row variant (nucleus_row_kernel): one CTA of 512 threads per row,
// persistent over rows (claimed from a counter as CTAs finish), two CTAs per
// SM. One pass reads the row from HBM; the later passes re-read it from L2
// (two rows per SM in flight: under 80 MB at V = 128256 bf16). The passes of
// one row:
//
//  AB. one read: the max M and its lowest index I, and the weights'
//     significands into the mass bins above (a column of counters per lane)
//     against a provisional reference R, kHead binades above the largest
//     element of the row's first 512 units. When M lies above what R covers
//     (rare), the bins are taken again from L2 against R = ceil(M s log2e).
//     The first bin j1, from the top, whose running mass reaches top_p of
//     the total holds z*;
//  C. the tokens of bin j1 -- a prefilter on the logit range the bin can hold
//     (bf16: the sign of (v - c)^2 - rr in packed FMAs; fp32: compares;
//     units with a hit queued per warp), then pass AB's exact bin test --
//     add their significands to a histogram over their keys: one bin per key
//     while the range holds at most 256 keys, else 256 sub-ranges, of which
//     the selected one narrows the range for another round (bf16: at most
//     two rounds; fp32: at most five). The first key whose running mass, on
//     top of the bins above j1, reaches the target is z*;
//  -- R, the nucleus mass other than I's, comes from the same integer sums;
//     when the entropy moment is wanted, one more pass sums e y over the
//     tokens with z >= z*.
// ---------------------------------------------------------------------------
#ifndef SV_NUC_RT
#define SV_NUC_RT 512
#endif
#ifndef SV_NUC_UF
#define SV_NUC_UF 2    // 16-byte vectors in flight per thread (aligned rows): 2 beats 4 by 3.5%, 1 is 13% slower
#endif
constexpr int RT = SV_NUC_RT;
constexpr int kRowCtas = RT >= 1024 ? 1 : 2;   // CTAs per SM
constexpr int RW = RT / 32;
constexpr int kRQueue = 256;    // units a warp queues before it processes them
constexpr int kHead = 12;       // binades of headroom of the provisional reference

struct RShared {
    union {
        uint32_t hist[NB][32];              // pass B: bins, a column per lane (no bank conflicts)
        struct {
            uint32_t key[RW][kKeyBins];     // pass C: per-warp key histograms
            uint4 qv[RW][kRQueue];          // ... units holding a candidate (aligned rows: their data)
            uint32_t qk[RW][kRQueue];       // ... and their unit index
        } c;
    } u;
    float wa[RW], wr[RW];
    int wi[RW];
    int sel, sel_last;
    float sel_a, sel_r, sel_rs;
    int next_row[2];                        // the CTA's next row, by iteration parity
};
constexpr int kRUnionWords = (int)(sizeof(RShared::u) / 4);

// the largest element of a 16-byte vector
template <typename T>
__device__ __forceinline__ float vec_max(const uint4 &x) {
    if constexpr (sizeof(T) == 2) {
        const uint32_t m = bmax2(bmax2(x.x, x.y), bmax2(x.z, x.w));
        return fmaxf(bf16_lo(m), bf16_hi(m));
    } else {
        return fmaxf(fmaxf(__uint_as_float(x.x), __uint_as_float(x.y)),
                     fmaxf(__uint_as_float(x.z), __uint_as_float(x.w)));
    }
}

// kAl: rows start on 16-byte boundaries; a unit is then one 16-byte vector
// (EU = 8 bf16 or 4 fp32 elements, SV_NUC_UF in flight per thread), else a group
// of 8 elements read one by one. Units k = t, t + 512, ... go to thread t;
// the V mod EU last elements to the last warp.
template <typename T, bool kAl>
__global__ void __launch_bounds__(RT, kRowCtas) nucleus_row_kernel(const NucleusArgs a, int ushift) {
    extern __shared__ __align__(16) unsigned char rsm[];
    RShared &sh = *reinterpret_cast<RShared *>(rsm);
    const int t = threadIdx.x, l = t & 31, w = t >> 5;
    constexpr int EU = kAl ? Elem<T>::kPerVec : 8;   // elements of a unit
    constexpr int UF = kAl ? SV_NUC_UF : 1;          // units in flight per thread
    for (int i = t; i < kRUnionWords; i += RT) (&sh.u.hist[0][0])[i] = 0u;
    __syncthreads();
    const int rows = a.nt_rows + a.nd_rows;
    const int nrow = a.B * rows;
    const int V = a.V, nu = V / EU, ut = V - nu * EU;
    const uint32_t umask = (1u << (23 - ushift)) - 1u, uimpl = 1u << (23 - ushift);
    auto unit = [&](uint32_t b) -> uint32_t { return ((b >> ushift) & umask) | uimpl; };
    const uint32_t colbase = (uint32_t)__cvta_generic_to_shared(&sh.u.hist[0][l]);   // this lane's bin column
    // the grid's first rows are the CTAs' own; the rest are claimed as CTAs
    // finish (rows differ in cost), one claim a row, read after a barrier
    // from a slot of that iteration's parity
    int it_row = 0;
    bool ahead = false;   // CTA-uniform: the next row was claimed during this one
    auto next_row = [&]() -> int {
        const int q = (++it_row) & 1;
        if (!ahead && t == 0) sh.next_row[q] = (int)gridDim.x + (int)atomicAdd(a.row_ctr, 1u);
        ahead = false;
        __syncthreads();
        return sh.next_row[q];
    };
    for (int row = blockIdx.x; row < nrow; row = next_row()) {
        const int b = row / rows, r = row - b * rows;
        const bool target = r < a.nt_rows;
        const int kb = a.draft_len ? min(max(__ldg(a.draft_len + b), 0), a.K) : a.K;
        const bool verified = target ? r <= kb : r - a.nt_rows < kb;
        if (!verified) {
            if (t == 0) {
                a.rec[row] = acc_pack(acc_empty());
                a.zth[row] = __int_as_float(0x7f800000);
            }
            continue;
        }
        const T *p = target ? static_cast<const T *>(a.zt) + ((long long)b * (a.K + 1) + r) * a.ts
                            : static_cast<const T *>(a.zd) + ((long long)b * a.K + (r - a.nt_rows)) * a.ds;
        const uint4 *vp = reinterpret_cast<const uint4 *>(p);
        auto load_unit = [&](int k, float (&z)[EU]) {
            if constexpr (kAl) Elem<T>::unpack(__ldg(vp + k), z);
            else load8<T>(p, 8 * k, V, false, z);
        };
        float s = 1.f;
        if (a.inv_temp) {
            const float si = __ldg(a.inv_temp + b);
            s = (si >= SPEC_MIN_INV_TEMPERATURE && si <= SPEC_MAX_INV_TEMPERATURE) ? si : 1.f;
        }
        const float sL = s * kLog2e;

        // ---- AB: one read of the row for the max, its lowest index (the first
        // unit holding a thread's max is read again for it) and the mass bins.
        // The weights are taken against a provisional reference, kHead
        // binades above the largest element of the first RT units (one per
        // thread); the bins reach 63 binades below 1, so the window that
        // counts (47 binades below the max) fits unless the max lies more
        // than kHead binades above that sample's -- then pass B takes the
        // bins again against the max.
        float Ms = neg_inf();
        if (t < nu) {
            float z[EU];
            load_unit(t, z);
#pragma unroll
            for (int j = 0; j < EU; ++j) Ms = fmaxf(Ms, z[j]);
        }
        if (t < ut) Ms = fmaxf(Ms, Elem<T>::load(p + nu * EU + t));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) Ms = fmaxf(Ms, __shfl_xor_sync(kFull, Ms, o));
        if (l == 0) sh.wa[w] = Ms;
        __syncthreads();
        Ms = sh.wa[0];
#pragma unroll
        for (int q = 1; q < RW; ++q) Ms = fmaxf(Ms, sh.wa[q]);
        __syncthreads();
        const bool fused = Ms > neg_inf() && Ms < __int_as_float(0x7f800000);
        float Rf = fused ? ceilf(Ms * sL) + (float)kHead : 0.f;
        float nR = -Rf;
        // a token's significand into its bin, counted from the top
        auto bin_add = [&](float z) {
            const uint32_t bb = __float_as_uint(ex2(fmaf(z, sL, nR)));
            atomicAdd(&sh.u.hist[pos_of(bb)][l], unit(bb));
        };
        // two tokens as bin_add takes one: their exponents by one packed FMA
        // (rounded as the scalar one), the position and the unit from each
        // weight's bits exactly as pos_of and unit take them, and the adds as
        // reductions on this lane's column (the old value is not wanted). With
        // pass C's squared prefilter, this one asm block measured about 3%
        // faster per call than the same steps written in C++.
        auto bin_add2 = [&](float z0, float z1) {
            asm volatile(
                "{\n\t"
                ".reg .f32 y0, y1;\n\t"
                ".reg .b64 zz, ss, rr, yy;\n\t"
                ".reg .b32 b0, b1, p0, p1, u0, u1;\n\t"
                "mov.b64 zz, {%1, %2};\n\t"
                "mov.b64 ss, {%3, %3};\n\t"
                "mov.b64 rr, {%4, %4};\n\t"
                "fma.rn.f32x2 yy, zz, ss, rr;\n\t"
                "mov.b64 {y0, y1}, yy;\n\t"
                "ex2.approx.ftz.f32 y0, y0;\n\t"
                "ex2.approx.ftz.f32 y1, y1;\n\t"
                "mov.b32 b0, y0;\n\t"
                "mov.b32 b1, y1;\n\t"
                "shr.u32 p0, b0, %9;\n\t"
                "shr.u32 p1, b1, %9;\n\t"
                "sub.u32 p0, %8, p0;\n\t"
                "sub.u32 p1, %8, p1;\n\t"
                "min.u32 p0, p0, %10;\n\t"
                "min.u32 p1, p1, %10;\n\t"
                "shr.u32 u0, b0, %5;\n\t"
                "shr.u32 u1, b1, %5;\n\t"
                "and.b32 u0, u0, %6;\n\t"
                "and.b32 u1, u1, %6;\n\t"
                "or.b32 u0, u0, %7;\n\t"
                "or.b32 u1, u1, %7;\n\t"
                "mad.lo.u32 p0, p0, %11, %0;\n\t"
                "mad.lo.u32 p1, p1, %11, %0;\n\t"
                "red.shared.add.u32 [p0], u0;\n\t"
                "red.shared.add.u32 [p1], u1;\n\t"
                "}" ::"r"(colbase),
                "f"(z0), "f"(z1), "f"(sL), "f"(nR), "r"(ushift), "r"(umask), "r"(uimpl),
                "r"(kHiBits >> (23 - kSub)), "n"(23 - kSub), "n"(NB - 1), "n"((int)sizeof(sh.u.hist[0]))
                : "memory");
        };
        float M = neg_inf();
        int I = 0x7fffffff;
        {
            int bk = -1;
            if constexpr (kAl) {
                // one vector: its max (strict: the first unit holding the
                // maximum), and its weights into the bins when fused
                auto vec_body = [&](auto with_bins, const uint4 &xv, int k) {
                    const float c = vec_max<T>(xv);
                    if (c > M) {
                        M = c;
                        bk = k;
                    }
                    if constexpr (decltype(with_bins)::value) {
                        float z[EU];
                        Elem<T>::unpack(xv, z);
#pragma unroll
                        for (int j = 0; j < EU; j += 2) bin_add2(z[j], z[j + 1]);
                    }
                };
                // whole rounds of UF vectors unguarded, then the thread's rest
                auto run = [&](auto with_bins) {
                    int k0 = t;
                    for (; k0 + (UF - 1) * RT < nu; k0 += UF * RT) {
                        uint4 x[UF];
#pragma unroll
                        for (int u = 0; u < UF; ++u) x[u] = __ldg(vp + k0 + u * RT);
#pragma unroll
                        for (int u = 0; u < UF; ++u) vec_body(with_bins, x[u], k0 + u * RT);
                    }
                    for (; k0 < nu; k0 += RT) vec_body(with_bins, __ldg(vp + k0), k0);
                };
                if (fused) run(std::true_type{});
                else run(std::false_type{});
            } else {
                for (int k0 = t; k0 < nu; k0 += RT) {
                    float z[8];
                    load_unit(k0, z);
                    float c = neg_inf();
#pragma unroll
                    for (int j = 0; j < 8; ++j) c = fmaxf(c, z[j]);
                    if (c > M) {
                        M = c;
                        bk = k0;
                    }
                    if (fused)
#pragma unroll
                        for (int j = 0; j < 8; j += 2) bin_add2(z[j], z[j + 1]);
                }
            }
            if (bk >= 0) {
                float z[EU];
                load_unit(bk, z);
                int jf = EU - 1;
#pragma unroll
                for (int j = EU - 1; j >= 0; --j)
                    if (z[j] == M) jf = j;
                I = bk * EU + jf;
            }
            if (t < ut) {
                const float z = Elem<T>::load(p + nu * EU + t);
                if (z > M) {
                    M = z;
                    I = nu * EU + t;
                }
            }
            if (fused && w == RW - 1 && l < ut) bin_add(Elem<T>::load(p + nu * EU + l));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float om = __shfl_xor_sync(kFull, M, o);
            const int oi = __shfl_xor_sync(kFull, I, o);
            if (om > M || (om == M && oi < I)) {
                M = om;
                I = oi;
            }
        }
        if (l == 0) {
            sh.wa[w] = M;
            sh.wi[w] = I;
        }
        __syncthreads();
        M = sh.wa[0];
        I = sh.wi[0];
#pragma unroll
        for (int q = 1; q < RW; ++q)
            if (sh.wa[q] > M || (sh.wa[q] == M && sh.wi[q] < I)) {
                M = sh.wa[q];
                I = sh.wi[q];
            }
        __syncthreads();
        if (!(M > neg_inf()) || M == __int_as_float(0x7f800000)) {
            // no finite logit, or an infinite one: the verification kernel
            // reports the bad row (the bins are cleared for the next row)
            for (int i = t; i < NB * 32; i += RT) (&sh.u.hist[0][0])[i] = 0u;
            if (t == 0) {
                a.rec[row] = acc_pack(acc_empty());
                a.zth[row] = __int_as_float(0x7f800000);
            }
            __syncthreads();
            continue;
        }

        // ---- B (only when the sample's reference does not hold): the bins
        // again, against R = ceil(M s log2e)
        if (!fused || ceilf(M * sL) > Rf) {
            if (fused) {
                for (int i = t; i < NB * 32; i += RT) (&sh.u.hist[0][0])[i] = 0u;
                __syncthreads();
            }
            Rf = ceilf(M * sL);
            nR = -Rf;
            for (int k0 = t; k0 < nu; k0 += UF * RT) {
                if constexpr (kAl) {
                    uint4 x[UF];
#pragma unroll
                    for (int u = 0; u < UF; ++u)
                        if (k0 + u * RT < nu) x[u] = __ldg(vp + k0 + u * RT);
#pragma unroll
                    for (int u = 0; u < UF; ++u)
                        if (k0 + u * RT < nu) {
                            float z[EU];
                            Elem<T>::unpack(x[u], z);
#pragma unroll
                            for (int j = 0; j < EU; j += 2) bin_add2(z[j], z[j + 1]);
                        }
                } else {
                    float z[8];
                    load_unit(k0, z);
#pragma unroll
                    for (int j = 0; j < 8; j += 2) bin_add2(z[j], z[j + 1]);
                }
            }
            if (w == RW - 1 && l < ut) bin_add(Elem<T>::load(p + nu * EU + l));
        }
        __syncthreads();
        // thread t takes position t from the top: bin NB - 1 - t
        const int g = NB - 1 - t;
        float m = 0.f;
        if (g >= 0) {
            u64 h = 0;
#pragma unroll 8
            for (int q = 0; q < 32; ++q) {
                const int c = (q + l) & 31;
                h += sh.u.hist[t][c];
                sh.u.hist[t][c] = 0u;
            }
            m = (float)h * bin_scale(g, ushift);
        }
        const float Z = block_sum<RW>(sh, m);
        const uint32_t bI = __float_as_uint(ex2(fmaf(M, sL, nR)));   // I, binned as pass B binned it
        const int gI = NB - 1 - (int)pos_of(bI);
        const float mI = (float)unit(bI) * bin_scale(gI, ushift);
        const float tgt = a.top_p * Z;
        float above_a, above_r, rsel;
        const float ma[1] = {g >= 1 ? m : 0.f};
        const float mr[1] = {g >= 1 ? (g == gI ? m - mI : m) : 0.f};
        const int j1 = NB - 1 - select_pos<1, RW>(sh, ma, mr, NB - 1, tgt, 0.f, 0.f, above_a, above_r, rsel);

        // ---- the logit range bin j1 can hold (its weight range, widened past
        // the exponential's and the roundings' errors), as keys
        uint32_t klo, khi;
        {
            float zlo = (bin_edge(j1) - 0x1p-12f + Rf) / sL, zhi = (bin_edge(j1 + 1) + 0x1p-12f + Rf) / sL;
            zlo -= fabsf(zlo) * 0x1p-16f + 0x1p-120f;
            zhi = fminf(zhi + fabsf(zhi) * 0x1p-16f + 0x1p-120f, M);
            if constexpr (sizeof(T) == 2) {
                zlo = __bfloat162float(__float2bfloat16_rd(zlo));
                zhi = __bfloat162float(__float2bfloat16_ru(zhi));
            }
            klo = Key<T>::of(zlo);
            khi = Key<T>::of(zhi);
            klo = min(klo, khi);   // an empty bin (only when no bin holds mass)
        }

        // ---- C (rounds): the candidates' significands by key
        const uint32_t jsel = (uint32_t)(j1 + kBinBase);
        const float scj = bin_scale(j1, ushift);
        uint32_t kstar = khi;
        float Rn = 0.f;   // nucleus mass other than I, relative to 2^R
        for (int it = 0;; ++it) {
            const u64 W = (u64)(khi - klo) + 1ull;
            const bool exact = W <= (u64)kKeyBins;
            const float zl = Key<T>::value(klo), zh = Key<T>::value(khi);
            const NearBf16 near(zl, zh);   // the scan's prefilter (bf16 rows)
            // a candidate in the logit range: pass B's exact bin test, then
            // its key (exact rounds) or sub-range (the 64-bit division only in
            // the rare rounds that need it)
            auto candidate = [&](auto ex, int idx, float z) {
                if (idx == I) return;
                const uint32_t bb = __float_as_uint(ex2(fmaf(z, sL, nR)));
                if ((bb >> (23 - kSub)) == jsel) {
                    const uint32_t d = khi - Key<T>::of(z);
                    int sub;
                    if constexpr (decltype(ex)::value) sub = (int)d;
                    else sub = (int)(((u64)d << 8) / W);
                    atomicAdd(&sh.u.c.key[w][sub], unit(bb));
                }
            };
            // a queued unit: the mask of its elements in the logit range, then
            // one candidate per set bit (usually one)
            const __nv_bfloat162 lo2 = __bfloat162bfloat162(__float2bfloat16_rn(zl));
            const __nv_bfloat162 hi2 = __bfloat162bfloat162(__float2bfloat16_rn(zh));
            auto flush_as = [&](auto ex, int qn) {
                if constexpr (kAl && sizeof(T) == 2) {
                    // bf16: the in-range mask by packed compares (zl and zh are
                    // bf16 values, so they are exact), bit q for the low element
                    // of word q and bit 16 + q for its high one; a candidate's
                    // element is read back from the queue
                    for (int i = l; i < qn; i += 32) {
                        const int k = (int)sh.u.c.qk[w][i];
                        const uint4 xv = sh.u.c.qv[w][i];
                        const uint32_t wv[4] = {xv.x, xv.y, xv.z, xv.w};
                        unsigned m = 0u;
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162 *>(&wv[q]);
                            m |= (__hge2_mask(v, lo2) & __hle2_mask(v, hi2) & 0x00010001u) << q;
                        }
                        const __nv_bfloat16 *qe = reinterpret_cast<const __nv_bfloat16 *>(&sh.u.c.qv[w][i]);
                        while (m) {
                            const int bit = __ffs(m) - 1;
                            m &= m - 1u;
                            const int j = bit < 16 ? 2 * bit : 2 * (bit - 16) + 1;
                            candidate(ex, k * EU + j, __bfloat162float(qe[j]));
                        }
                    }
                } else {
                    for (int i = l; i < qn; i += 32) {
                        const int k = (int)sh.u.c.qk[w][i];
                        float z[EU];
                        if constexpr (kAl) Elem<T>::unpack(sh.u.c.qv[w][i], z);
                        else load_unit(k, z);
                        unsigned m = 0u;
#pragma unroll
                        for (int j = 0; j < EU; ++j) m |= (unsigned)((z[j] >= zl) & (z[j] <= zh)) << j;
                        while (m) {
                            const int j = __ffs(m) - 1;
                            m &= m - 1u;
                            float zj = z[0];
#pragma unroll
                            for (int q = 1; q < EU; ++q) zj = q == j ? z[q] : zj;
                            candidate(ex, k * EU + j, zj);
                        }
                    }
                }
            };
            auto flush = [&](int qn) {
                __syncwarp();
                if (exact) flush_as(std::true_type{}, qn);
                else flush_as(std::false_type{}, qn);
                __syncwarp();
            };
            int qn = 0;   // warp-uniform
            // a unit with a hit goes to the warp's queue (warp-collective)
            const unsigned lanes_below = (1u << l) - 1u;
            auto enqueue = [&](bool hit, int k, const uint4 &xv) {
                const unsigned mk = __ballot_sync(kFull, hit);
                const int slot = qn + __popc(mk & lanes_below);
                if (hit) {
                    sh.u.c.qk[w][slot] = (uint32_t)k;
                    if constexpr (kAl) sh.u.c.qv[w][slot] = xv;
                }
                qn += __popc(mk);
            };
            if constexpr (kAl) {
                int k0 = t - l;
                // whole rounds (every lane's UF vectors exist), unguarded
                for (; k0 + 31 + (UF - 1) * RT < nu; k0 += UF * RT) {
                    uint4 x[UF];
#pragma unroll
                    for (int u = 0; u < UF; ++u) x[u] = __ldg(vp + k0 + l + u * RT);
                    if constexpr (sizeof(T) == 2) {
#pragma unroll
                        for (int u = 0; u < UF; ++u) enqueue(near(x[u]), k0 + l + u * RT, x[u]);
                    } else {
#pragma unroll
                        for (int u = 0; u < UF; ++u) enqueue(vec_in_range<T>(x[u], zl, zh), k0 + l + u * RT, x[u]);
                    }
                    if (qn > kRQueue - UF * 32) {
                        flush(qn);
                        qn = 0;
                    }
                }
                // the rest, one vector a lane at a time
                for (; k0 < nu; k0 += RT) {
                    const int k = k0 + l;
                    uint4 xv = make_uint4(0u, 0u, 0u, 0u);
                    if (k < nu) xv = __ldg(vp + k);
                    enqueue(k < nu && vec_in_range<T>(xv, zl, zh), k, xv);
                    if (qn > kRQueue - 32) {
                        flush(qn);
                        qn = 0;
                    }
                }
            } else {
                for (int k0 = t - l; k0 < nu; k0 += RT) {
                    bool any = false;
                    if (k0 + l < nu) {
                        float z[8];
                        load_unit(k0 + l, z);
#pragma unroll
                        for (int j = 0; j < 8; ++j) any |= (z[j] >= zl) & (z[j] <= zh);
                    }
                    enqueue(any, k0 + l, make_uint4(0u, 0u, 0u, 0u));
                    if (qn > kRQueue - 32) {
                        flush(qn);
                        qn = 0;
                    }
                }
            }
            flush(qn);
            if (w == RW - 1 && l < ut) {
                const float z = Elem<T>::load(p + nu * EU + l);
                if (z >= zl && z <= zh) {
                    if (exact) candidate(std::true_type{}, nu * EU + l, z);
                    else candidate(std::false_type{}, nu * EU + l, z);
                }
            }
            // I, left out above, with its key
            float uI = 0.f;
            int sI = -1;
            if (M >= zl && M <= zh && (bI >> (23 - kSub)) == jsel) {
                const uint32_t d = khi - Key<T>::of(M);
                uI = (float)unit(bI);
                sI = exact ? (int)d : (int)(((u64)d << 8) / W);
            }
            // the CTA's next row, claimed now: after the barrier each thread
            // asks L2 for its first unit of it (the next row's first loads)
            const bool claim = !ahead;
            if (claim && t == 0) sh.next_row[(it_row + 1) & 1] = (int)gridDim.x + (int)atomicAdd(a.row_ctr, 1u);
            ahead = true;
            __syncthreads();
            if constexpr (kAl) {
                const int nx = sh.next_row[(it_row + 1) & 1];
                if (claim && nx < nrow && t < nu) {
                    const int b2 = nx / rows, r2 = nx - b2 * rows;
                    const T *q = r2 < a.nt_rows
                                     ? static_cast<const T *>(a.zt) + ((long long)b2 * (a.K + 1) + r2) * a.ts
                                     : static_cast<const T *>(a.zd) + ((long long)b2 * a.K + (r2 - a.nt_rows)) * a.ds;
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const uint4 *>(q) + t));
                }
            }
            float us = 0.f;
            if (t < kKeyBins) {
                u64 h = 0;
#pragma unroll
                for (int q = 0; q < RW; ++q) {
                    h += sh.u.c.key[q][t];
                    sh.u.c.key[q][t] = 0u;
                }
                us = (float)h;
            }
            const float ka[1] = {(t == sI ? us + uI : us) * scj};
            const float kr[1] = {us * scj};
            float aa, ar, rs;
            const int sk = select_pos<1, RW>(sh, ka, kr, kKeyBins, tgt, above_a, above_r, aa, ar, rs);
            if (exact) {
                kstar = khi - (uint32_t)sk;
                Rn = ar + rs;
                break;
            }
            // keys of sub-range sk: khi - k in [ceil(sk W / 256), ceil((sk + 1) W / 256) - 1]
            const u64 lo_off = ((u64)sk * W + 255ull) >> 8;
            const u64 hi_off = (((u64)(sk + 1) * W + 255ull) >> 8) - 1ull;
            const uint32_t nkhi = khi - (uint32_t)lo_off;
            klo = khi - (uint32_t)hi_off;
            khi = nkhi;
            above_a = aa;
            above_r = ar;
            if (it + 1 >= kMaxRefine) {   // not reached: 32-bit keys need at most five rounds
                if (t == 0) atomicMax(a.status, (unsigned)SPEC_ERR_BAD_ROW);
                kstar = khi;
                Rn = ar;
                break;
            }
        }
        // the queue overlapped pass B's bins: clear it for the next row
        for (int i = RW * kKeyBins + t; i < NB * 32; i += RT) (&sh.u.hist[0][0])[i] = 0u;
        const float zstar = Key<T>::value(kstar);

        // ---- the entropy moment over the nucleus, when wanted: exponents
        // taken against the max itself (the reference R may lie binades above
        // it, and converting would cancel)
        float Tn = 0.f;
        if (a.need_ent) {
            float tc = 0.f;
            const float nM = -(M * sL);
            auto add = [&](float z) {
                if (z >= zstar) {
                    const float y = fmaf(z, sL, nM);
                    tc = fmaf(ex2(y), y, tc);
                }
            };
            int k0 = t;
            if constexpr (kAl) {
                for (; k0 + (UF - 1) * RT < nu; k0 += UF * RT) {
                    uint4 x[UF];
#pragma unroll
                    for (int u = 0; u < UF; ++u) x[u] = __ldg(vp + k0 + u * RT);
#pragma unroll
                    for (int u = 0; u < UF; ++u) {
                        float z[EU];
                        Elem<T>::unpack(x[u], z);
#pragma unroll
                        for (int j = 0; j < EU; ++j) add(z[j]);
                    }
                }
            }
            for (; k0 < nu; k0 += RT) {
                float z[EU];
                load_unit(k0, z);
#pragma unroll
                for (int j = 0; j < EU; ++j) add(z[j]);
            }
            if (t < ut) add(Elem<T>::load(p + nu * EU + t));
            Tn = block_sum<RW>(sh, tc);
        }
        if (t == 0) {
            // from the reference 2^R to the max: weights times 2^dl
            const float dl = Rf - M * sL;
            const float f = ex2(dl);
            RowAcc acc;
            acc.M = M;
            acc.R = Rn * f;
            acc.T = Tn;
            acc.I = I;
            a.rec[row] = acc_pack(acc);
            a.zth[row] = zstar;
        }
        __syncthreads();
    }
}

}  // namespace nuc

namespace {

// The row variant (every row layout, V up to 256 K elements); `launched`
// says whether it ran.
template <typename T>
cudaError_t launch_row(const NucleusArgs &a, cudaStream_t stream, int sms, long long nrow, bool &launched) {
    launched = false;
    // the most tokens one 32-bit counter can receive -- a lane's column of
    // pass B's bins (that lane of every warp), a warp's key histogram in
    // pass C -- with the scalar tail on the last warp: significands are
    // shifted so that no counter overflows, by at most 6 bits (2^-18
    // relative)
    const bool al = a.t_vec_ok && (a.nd_rows == 0 || a.d_vec_ok);
    const int eu = al ? 16 / (int)sizeof(T) : 8;   // elements of a unit
    const int nu = a.V / eu, tail = a.V % eu;
    auto units = [&](int t) -> long long { return t < nu ? (nu - 1 - t) / nuc::RT + 1 : 0; };
    long long tw = 0;
    for (int i = 0; i < 32; ++i) {
        long long col = 0;
        for (int w = 0; w < nuc::RW; ++w) col += units(32 * w + i);
        tw = std::max(tw, col * eu + (i < tail ? 1 : 0));
    }
    for (int w = 0; w < nuc::RW; ++w) {
        long long gw = 0;
        for (int i = 0; i < 32; ++i) gw += units(32 * w + i);
        tw = std::max(tw, gw * eu + (w == nuc::RW - 1 ? tail : 0));
    }
    int ushift = 3;
    while (ushift <= 6 && tw * (long long)((1u << (24 - ushift)) - 1u) > 0xffffffffLL) ++ushift;
    if (ushift > 6) return cudaSuccess;
    void (*kern)(const NucleusArgs, int) = al ? nuc::nucleus_row_kernel<T, true> : nuc::nucleus_row_kernel<T, false>;
    const int smem = (int)sizeof(nuc::RShared);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    long long grid = (long long)nuc::kRowCtas * sms;
    if (grid > nrow) grid = nrow;
    if (grid < 1) grid = 1;
    kern<<<(unsigned)grid, nuc::RT, smem, stream>>>(a, ushift);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    launched = true;
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_nucleus(const NucleusArgs &a, cudaStream_t stream) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const long long nrow = (long long)a.B * (a.nt_rows + a.nd_rows);
    bool launched = false;
    e = a.bf16 ? launch_row<__nv_bfloat16>(a, stream, sms, nrow, launched)
               : launch_row<float>(a, stream, sms, nrow, launched);
    if (e != cudaSuccess || launched) return e;
    // rows not 16-byte aligned, or larger than 8 slices: one CTA per row, the
    // row re-read from L2 between passes
    long long grid = (long long)sms * SV_NUC_CTAS;
    if (grid > nrow) grid = nrow;
    if (grid < 1) grid = 1;
    if (a.bf16)
        nuc::nucleus_kernel<__nv_bfloat16><<<(unsigned)grid, nuc::NT, 0, stream>>>(a);
    else
        nuc::nucleus_kernel<float><<<(unsigned)grid, nuc::NT, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace sv
