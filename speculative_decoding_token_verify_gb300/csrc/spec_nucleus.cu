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
// Two kernels find z* by the same mass-weighted radix select:
//  * nucleus_cluster_kernel (used when rows are 16-byte aligned and a
//    cluster of at most 8 CTAs holds one in 32 or 64 KB slices): the row is
//    read from HBM once into the cluster's distributed shared memory, and
//    every pass below reads shared memory; see the comment above it.
//  * nucleus_kernel (every other row): one CTA takes one row at a time
//    (persistent over rows), re-reading the row between passes (L2-resident:
//    two CTAs per SM keep under 100 MB of rows in flight).
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

#include <cooperative_groups.h>
#include <cstdint>

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
// Cluster variant. A thread-block cluster of C CTAs holds one row in its
// distributed shared memory: CTA c keeps elements [c S, (c + 1) S), loaded
// once from HBM by the bulk-copy engine (cp.async.bulk, completion on an
// mbarrier). Every pass then reads shared memory, and the per-row merges
// (row statistics, histograms, key ranges, nucleus sums) go through DSMEM:
// each CTA publishes its part in an exchange slot, one cluster barrier, and
// every CTA reads all parts in rank order, so all of them hold identical
// results. Exchange slots alternate between two buffers: a slot is written
// again only after the cluster barrier that follows every read of it.
// ---------------------------------------------------------------------------
constexpr int kSliceBytes = 65536;        // row bytes a CTA holds, at most
constexpr int kSliceSmall = 32768;        // ... preferred: four CTAs per SM
constexpr int kMaxCluster = 8;            // portable cluster size
constexpr unsigned kWaitLimit = 1u << 20; // mbarrier polls before giving up
constexpr int kX = kBins + 8;             // u64 words per exchange slot

constexpr int kCandC = 64;                // boundary-bin tokens kept per warp
constexpr float kBinUnit = 0x1p19f;       // histogram unit: 2^-19 of a bin's top weight

struct CShared {
    unsigned long long bar;       // mbarrier of the slice load
    uint32_t hist[NW][kBins];     // per-warp histograms (kBinUnit units, <= 4096 tokens a warp)
    u64 xbuf[2][kX];              // exchange slots, read by the peers
    uint32_t ckey[NW][kCandC];    // boundary-bin tokens: logit key,
    uint32_t cfix[NW][kCandC];    // ... mass in kBinUnit units of the bin's top weight,
    int cv[NW][kCandC];           // ... vocabulary index
    int cnt[NW];
    float bscale[kBins];          // 2^-y_hi(j): a bin-j weight in units of its top weight
    float dsum[NW];
    float4 acc[NW];
    float fw[NW][2];
    uint32_t kw[NW][2];
    int sel;
    float sel_above;
};
constexpr int kCSharedBytes = (int)((sizeof(CShared) + 127) & ~(size_t)127);

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(unsigned long long *bar) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(bar)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(unsigned long long *bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

// Wait, with a bounded number of polls, for the phase of parity `par` to
// complete. Returns false when the limit ran out.
__device__ __forceinline__ bool mbar_wait(unsigned long long *bar, unsigned par) {
    unsigned ns = 32;
    for (unsigned it = 0; it < kWaitLimit; ++it) {
        unsigned done;
        asm volatile("{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                     "selp.u32 %0, 1, 0, p;\n\t}"
                     : "=r"(done)
                     : "r"(smem_u32(bar)), "r"(par)
                     : "memory");
        if (done) return true;
        __nanosleep(ns);
        ns = min(ns * 2u, 256u);
    }
    return false;
}

// bytes (a multiple of 16; both addresses 16-byte aligned) from global to
// this CTA's shared memory, completing on `bar`
__device__ __forceinline__ void bulk_load(void *dst, const void *src, unsigned bytes, unsigned long long *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// order this CTA's earlier generic-proxy accesses of shared memory before
// later async-proxy (bulk copy) writes
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

namespace cg = cooperative_groups;

__device__ __forceinline__ float elem_f(float x) { return x; }
__device__ __forceinline__ float elem_f(__nv_bfloat16 x) { return __bfloat162float(x); }

__device__ __forceinline__ u64 pack2(float x, float y) {
    return (u64)__float_as_uint(x) | ((u64)__float_as_uint(y) << 32);
}
__device__ __forceinline__ float lo_f(u64 v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float hi_f(u64 v) { return __uint_as_float((uint32_t)(v >> 32)); }

__device__ __forceinline__ u64 fixed40(float y) { return __float2ull_rn(ex2(y) * 0x1p40f); }

// Sum the per-warp histograms of every CTA of the cluster (thread t owns bin
// t; CTAs added in rank order, exact 64-bit integers); this CTA's histograms
// are cleared.
// With `ztot`, the per-warp partial sums in sh.fw[.][0] travel along: the
// CTA's sum (warp order), then the cluster's (rank order) lands in *ztot.
__device__ __forceinline__ u64 cluster_bins(CShared &sh, cg::cluster_group &cl, int C, int &par,
                                            float *ztot = nullptr) {
    const int t = threadIdx.x;
    __syncthreads();
    u64 h = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
        h += sh.hist[w][t];
        sh.hist[w][t] = 0u;
    }
    sh.xbuf[par][t] = h;
    if (ztot && t == 0) {
        float zs = 0.f;
        for (int i = 0; i < NW; ++i) zs += sh.fw[i][0];
        sh.xbuf[par][kBins] = pack2(zs, 0.f);
    }
    cl.sync();
    u64 H = 0;
    float Z = 0.f;
    for (int c = 0; c < C; ++c) {
        const u64 *x = cl.map_shared_rank(&sh.xbuf[par][0], c);
        H += x[t];
        if (ztot) Z += lo_f(x[kBins]);
    }
    if (ztot) *ztot = Z;
    par ^= 1;
    return H;
}

// Thread t holds the mass h >= 0 of bin t (fp32): the running sums in bin
// order, in a fixed association; the selected bin is the lowest whose
// running sum plus `above` reaches tgt (the last bin with mass if rounding
// leaves all short). `above` becomes the running sum before it.
__device__ __forceinline__ int select_f(CShared &sh, float h, float tgt, float &above) {
    const int t = threadIdx.x, l = t & 31, w = t >> 5;
    float v = h;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float u = __shfl_up_sync(kFull, v, o);
        if (l >= o) v += u;
    }
    if (l == 31) sh.dsum[w] = v;
    if (t == 0) sh.sel = kBins;
    __syncthreads();
    float pre = above;
    for (int i = 0; i < w; ++i) pre += sh.dsum[i];
    const float incl = pre + v;
    if (incl >= tgt) atomicMin(&sh.sel, t);
    __syncthreads();
    if (sh.sel == kBins) {   // only through rounding: the last bin with mass
        if (h > 0.f) atomicMax(&sh.sel, kBins + 1 + t);
        __syncthreads();
        if (t == 0) sh.sel = sh.sel > kBins ? sh.sel - kBins - 1 : kBins - 1;
        __syncthreads();
    }
    const int j = sh.sel;
    if (t == j) sh.sel_above = incl - h;
    __syncthreads();
    above = sh.sel_above;
    __syncthreads();
    return j;
}

// Visit the slice in shared memory: vectors k = t, t + NT, ... (element
// v0 + k E + j), then the tail scalars (warp 0, lane < tail); the same fixed
// order every pass. Warp-uniform: every lane of a warp makes the same calls
// (past the slice, z is -inf), so f may use warp-collective operations.
template <typename T, typename F>
__device__ __forceinline__ void for_slice(const T *slice, int nvec, int tail, int v0, F &&f) {
    constexpr int E = Elem<T>::kPerVec;
    const uint4 *sv = reinterpret_cast<const uint4 *>(slice);
    const int lane = threadIdx.x & 31;
    for (int k0 = (int)threadIdx.x - lane; k0 < nvec; k0 += NT) {
        const int k = k0 + lane;
        float z[E];
        if (k < nvec) {
            Elem<T>::unpack(sv[k], z);
        } else {
#pragma unroll
            for (int j = 0; j < E; ++j) z[j] = neg_inf();
        }
#pragma unroll
        for (int j = 0; j < E; ++j) f(v0 + k * E + j, z[j]);
    }
    if (threadIdx.x < 32) f(v0 + nvec * E + lane, lane < tail ? elem_f(slice[nvec * E + lane]) : neg_inf());
}

template <typename T>
__global__ void __launch_bounds__(NT, 4) nucleus_cluster_kernel(const NucleusArgs a, int S) {
    extern __shared__ __align__(128) unsigned char dsm[];
    CShared &sh = *reinterpret_cast<CShared *>(dsm);
    T *slice = reinterpret_cast<T *>(dsm + kCSharedBytes);
    cg::cluster_group cl = cg::this_cluster();
    const int C = (int)cl.num_blocks();
    const int rank = (int)cl.block_rank();
    const int t = threadIdx.x, l = t & 31, w = t >> 5;
    constexpr int E = Elem<T>::kPerVec;
    for (int i = t; i < NW * kBins; i += NT) (&sh.hist[0][0])[i] = 0ull;
    if (t == 0) mbar_init(&sh.bar);
    __syncthreads();
    unsigned phase = 0;
    bool pending = false;   // a slice load whose wait gave up
    int par = 0;
    const int rows = a.nt_rows + a.nd_rows;
    const int nrow = a.B * rows;
    const int ncl = (int)(gridDim.x / (unsigned)C), cid = (int)(blockIdx.x / (unsigned)C);
    const int v0 = rank * S;
    const int len = max(0, min(a.V, v0 + S) - v0);
    const int nvec = len / E, tail = len - nvec * E;
    const float Drel = logf((float)a.V / (1.f - a.top_p)) + 1.f;
    for (int row = cid; row < nrow; row += ncl) {
        const int b = row / rows, r = row - b * rows;
        const bool target = r < a.nt_rows;
        const int kb = a.draft_len ? min(max(__ldg(a.draft_len + b), 0), a.K) : a.K;
        const bool verified = target ? r <= kb : r - a.nt_rows < kb;
        if (!verified) {   // uniform over the cluster: no barrier is skipped unevenly
            if (rank == 0 && t == 0) {
                a.rec[row] = acc_pack(acc_empty());
                a.zth[row] = __int_as_float(0x7f800000);
            }
            continue;
        }
        const T *p = target ? static_cast<const T *>(a.zt) + ((long long)b * (a.K + 1) + r) * a.ts
                            : static_cast<const T *>(a.zd) + ((long long)b * a.K + (r - a.nt_rows)) * a.ds;
        float s = 1.f;
        if (a.inv_temp) {
            const float si = __ldg(a.inv_temp + b);
            s = (si >= SPEC_MIN_INV_TEMPERATURE && si <= SPEC_MAX_INV_TEMPERATURE) ? si : 1.f;
        }
        const float sL = s * kLog2e;
        const float rs = __fdiv_rn(kRescale, s);

        // ---- load this CTA's slice once (the previous row's reads are done)
        __syncthreads();
        if (t == 0 && nvec > 0) {
            fence_proxy_async();
            mbar_expect_tx(&sh.bar, (unsigned)nvec * 16u);
            bulk_load(slice, p + v0, (unsigned)nvec * 16u, &sh.bar);
        }
        if (t < tail) slice[nvec * E + t] = p[v0 + nvec * E + t];
        if (nvec > 0) {
            pending = !mbar_wait(&sh.bar, phase);
            if (pending && t == 0) atomicMax(a.status, (unsigned)SPEC_ERR_TIMEOUT);
            phase ^= 1u;
        }
        __syncthreads();

        // ---- A: max M, its lowest index I and the smallest logit (chunk
        // maxima on packed bf16 / fp32 compares), merged over the cluster in
        // rank order
        float M = neg_inf(), cmin = __int_as_float(0x7f800000);
        int I = 0x7fffffff;
        {
            const uint4 *sv = reinterpret_cast<const uint4 *>(slice);
            int bk = -1;
            uint4 bw = make_uint4(0u, 0u, 0u, 0u);
            for (int k = t; k < nvec; k += NT) {
                const uint4 wv = sv[k];
                float c;
                if constexpr (sizeof(T) == 2) {
                    const uint32_t m = bmax2(bmax2(wv.x, wv.y), bmax2(wv.z, wv.w));
                    c = fmaxf(bf16_lo(m), bf16_hi(m));
                } else {
                    c = fmaxf(fmaxf(__uint_as_float(wv.x), __uint_as_float(wv.y)),
                              fmaxf(__uint_as_float(wv.z), __uint_as_float(wv.w)));
                }
                if (c > M) {   // strict: the first chunk holding the maximum
                    M = c;
                    bk = k;
                    bw = wv;
                }
                cmin = fminf(cmin, chunk_min<T>(wv));
            }
            if (bk >= 0) {
                float z[E];
                Elem<T>::unpack(bw, z);
                int jf = E - 1;
#pragma unroll
                for (int q = E - 1; q >= 0; --q)
                    if (z[q] == M) jf = q;
                I = v0 + bk * E + jf;
            }
            if (t < tail) {
                const float z = elem_f(slice[nvec * E + t]);
                if (z > M) {
                    M = z;
                    I = v0 + nvec * E + t;
                }
                cmin = fminf(cmin, z);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float om = __shfl_xor_sync(kFull, M, o);
            const int oi = __shfl_xor_sync(kFull, I, o);
            if (om > M || (om == M && oi < I)) {
                M = om;
                I = oi;
            }
            cmin = fminf(cmin, __shfl_xor_sync(kFull, cmin, o));
        }
        if (l == 0) {
            sh.fw[w][0] = M;
            sh.fw[w][1] = cmin;
            sh.kw[w][0] = (uint32_t)I;
        }
        __syncthreads();
        if (t == 0) {
            float m = sh.fw[0][0], cm = sh.fw[0][1];
            int ii = (int)sh.kw[0][0];
            for (int q = 1; q < NW; ++q) {
                if (sh.fw[q][0] > m || (sh.fw[q][0] == m && (int)sh.kw[q][0] < ii)) {
                    m = sh.fw[q][0];
                    ii = (int)sh.kw[q][0];
                }
                cm = fminf(cm, sh.fw[q][1]);
            }
            sh.xbuf[par][0] = pack2(m, __int_as_float(ii));
            sh.xbuf[par][1] = pack2(cm, 0.f);
        }
        cl.sync();
        M = neg_inf();
        I = 0x7fffffff;
        cmin = __int_as_float(0x7f800000);
        for (int c = 0; c < C; ++c) {
            const u64 *xc = cl.map_shared_rank(&sh.xbuf[par][0], c);
            const float om = lo_f(xc[0]);
            const int oi = __float_as_int(hi_f(xc[0]));
            if (om > M || (om == M && oi < I)) {
                M = om;
                I = oi;
            }
            cmin = fminf(cmin, lo_f(xc[1]));
        }
        par ^= 1;
        if (!(M > neg_inf()) || M == __int_as_float(0x7f800000)) {
            // no finite logit (the verification kernel reports the bad row);
            // M is the cluster's, so every CTA leaves the row here
            if (rank == 0 && t == 0) {
                a.rec[row] = acc_pack(acc_empty());
                a.zth[row] = __int_as_float(0x7f800000);
            }
            continue;
        }

        // ---- B: every token's weight e = 2^y, y = (z - M) s log2e, summed
        // (fixed order) into the total Z; those within Dr nats of M also go
        // to a histogram of Dr/256-nat bins, a token of bin j counting
        // ex2(y - y_hi(j)) in kBinUnit units of the bin's top weight 2^y_hi(j)
        // (32 bits keep ~2^-20 relative precision); bin masses in fp32
        // (bin and unit conversions by the 2^23 magic-number rounding on the
        // FMA pipe: bin j holds y * ybin in [j - 1/2, j + 1/2), its top is
        // y_hi(j) = (j - 1/2) ystep; rounding keeps the bin monotone in z,
        // which is all the search needs)
        const float Dr = fminf((M - cmin) * s, Drel);
        const float ylim = -Dr * kLog2e;                                   // y >= ylim <=> binned
        const float ybin = Dr > 0.f ? -(float)kBins * kLn2 / Dr : 0.f;
        const float ystep = Dr > 0.f ? 1.f / ybin : 0.f;
        auto bin_of = [&](float y) -> int {
            return min(kBins - 1, __float_as_int(fmaf(y, ybin, 0x1p23f)) - 0x4B000000);
        };
        auto unit_of = [&](float e, int j) -> uint32_t {   // e = 2^y of a bin-j token
            return (uint32_t)(__float_as_int(fmaf(e * sh.bscale[j], kBinUnit, 0x1p23f)) - 0x4B000000);
        };
        sh.bscale[t] = ex2(-((float)t - 0.5f) * ystep);
        const float tmass = ex2(((float)t - 0.5f) * ystep) * (1.f / kBinUnit);   // thread t: bin t's unit mass
        __syncthreads();
        float Zs = 0.f;
        for_slice<T>(slice, nvec, tail, v0, [&](int v, float z) {
            const float y = (z - M) * sL;
            const float e = ex2(y);
            Zs += e;
            if (y >= ylim) {
                const int j = bin_of(y);
                atomicAdd(&sh.hist[w][j], unit_of(e, j));
            }
        });
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) Zs += __shfl_xor_sync(kFull, Zs, o);
        if (l == 0) sh.fw[w][0] = Zs;
        float Z = 0.f;
        const u64 H1 = cluster_bins(sh, cl, C, par, &Z);
        const float tgt = a.top_p * Z;
        float above = 0.f;
        const int j1 = select_f(sh, (float)H1 * tmass, tgt, above);
        const float j1mass = ex2(((float)j1 - 0.5f) * ystep) * (1.f / kBinUnit);   // unit mass of bin j1

        // ---- C: tokens above bin j1 are in the nucleus: their mass (other
        // than I) and entropy moment accumulate per thread; bin j1's tokens
        // (a contiguous key range: y is monotone in z) are copied to this
        // warp's list in a fixed order, and their key range is merged over
        // the cluster
        float Ra = 0.f, Ta = 0.f;
        uint32_t klo = 0xffffffffu, khi = 0u;
        int wc = 0;   // warp-uniform count of bin-j1 tokens this warp met
        for_slice<T>(slice, nvec, tail, v0, [&](int v, float z) {
            const float y = (z - M) * sL;
            const int bn = y >= ylim ? bin_of(y) : kBins;
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
                    if (slot < kCandC) {
                        sh.ckey[w][slot] = k;
                        sh.cfix[w][slot] = unit_of(ex2(y), j1);
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
        bool fits = true;   // this CTA's bin-j1 tokens are all in the lists
        if (t == 0) {
            uint32_t lo = sh.kw[0][0], hi = sh.kw[0][1];
            for (int i = 1; i < NW; ++i) {
                lo = min(lo, sh.kw[i][0]);
                hi = max(hi, sh.kw[i][1]);
            }
            sh.xbuf[par][0] = (u64)lo | ((u64)hi << 32);
        }
#pragma unroll
        for (int i = 0; i < NW; ++i) fits &= sh.cnt[i] <= kCandC;
        cl.sync();
        klo = 0xffffffffu;
        khi = 0u;
        for (int c = 0; c < C; ++c) {
            const u64 xv = cl.map_shared_rank(&sh.xbuf[par][0], c)[0];
            klo = min(klo, (uint32_t)xv);
            khi = max(khi, (uint32_t)(xv >> 32));
        }
        par ^= 1;

        // ---- D: refine the key range to one key, 256 sub-ranges a round
        // (over the lists; over the slice where a list overflowed)
        int it = 0;
        while (klo < khi && it < kMaxRefine) {
            const u64 W = (u64)(khi - klo) + 1ull;
            if (fits) {
                for (int i = t; i < NW * kCandC; i += NT) {
                    const int wi = i / kCandC, si = i - wi * kCandC;
                    if (si < sh.cnt[wi]) {
                        const uint32_t k = sh.ckey[wi][si];
                        if (k >= klo && k <= khi) atomicAdd(&sh.hist[w][(int)(((u64)(khi - k) << 8) / W)], sh.cfix[wi][si]);
                    }
                }
            } else {
                const float zlo = Key<T>::value(klo), zhi = Key<T>::value(khi);
                for_slice<T>(slice, nvec, tail, v0, [&](int v, float z) {
                    if (z >= zlo && z <= zhi) {
                        const uint32_t k = Key<T>::of(z);
                        atomicAdd(&sh.hist[w][(int)(((u64)(khi - k) << 8) / W)], unit_of(ex2((z - M) * sL), j1));
                    }
                });
            }
            const int j = select_f(sh, (float)cluster_bins(sh, cl, C, par) * j1mass, tgt, above);
            // keys of sub-range j: khi - k in [ceil(j W / 256), ceil((j + 1) W / 256) - 1]
            const u64 lo_off = ((u64)j * W + 255ull) >> 8;
            const u64 hi_off = (((u64)(j + 1) * W + 255ull) >> 8) - 1ull;
            const uint32_t nkhi = khi - (uint32_t)lo_off;
            const uint32_t nklo = khi - (uint32_t)hi_off;
            khi = nkhi;
            klo = nklo;
            ++it;
        }
        if (klo < khi && rank == 0 && t == 0) atomicMax(a.status, (unsigned)SPEC_ERR_BAD_ROW);   // not reached
        const uint32_t kstar = khi;
        const float zstar = Key<T>::value(kstar);

        // ---- E: nucleus statistics in a fixed order: the tokens above bin j1
        // (per thread) and this warp's listed tokens at or above z*
        // (lane-strided, slot order); where a list overflowed, a pass over
        // the slice instead
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
            for_slice<T>(slice, nvec, tail, v0, [&](int v, float z) {
                if (z >= zstar) {
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
            sh.xbuf[par][0] = pack2(Rs, Ts);
        }
        cl.sync();
        if (rank == 0 && t == 0) {
            float Rc = 0.f, Tc = 0.f;
            for (int c = 0; c < C; ++c) {
                const u64 xv = cl.map_shared_rank(&sh.xbuf[par][0], c)[0];
                Rc += lo_f(xv);
                Tc += hi_f(xv);
            }
            RowAcc acc;
            acc.M = M;
            acc.R = Rc;
            acc.T = Tc;
            acc.I = I;
            a.rec[row] = acc_pack(acc);
            a.zth[row] = zstar;
        }
        par ^= 1;
    }
    // a load whose wait gave up is waited for again (bounded) before the CTA
    // leaves; and no CTA leaves while a peer may still read its exchange slots
    if (pending) (void)mbar_wait(&sh.bar, phase ^ 1u);
    cl.sync();
}

}  // namespace nuc

namespace {

// The cluster variant when the rows are 16-byte aligned and a cluster of at
// most 8 CTAs holds one in 64 KB slices; `launched` says whether it ran.
template <typename T>
cudaError_t launch_cluster(const NucleusArgs &a, cudaStream_t stream, int sms, long long nrow, bool &launched) {
    launched = false;
    constexpr int es = (int)sizeof(T), E = 16 / es;
    if (!a.t_vec_ok || (a.nd_rows > 0 && !a.d_vec_ok)) return cudaSuccess;
    // the smallest cluster whose slices fit 32 KB (four CTAs per SM), else
    // 64 KB (two per SM)
    int C = 1, S = 0, per_sm = 4;
    for (int lim : {nuc::kSliceSmall, nuc::kSliceBytes}) {
        for (C = 1; C <= nuc::kMaxCluster; C *= 2) {
            S = ((a.V + C - 1) / C + E - 1) / E * E;
            if (S * es <= lim) break;
        }
        if (C <= nuc::kMaxCluster) break;
        per_sm = 2;
    }
    if (C > nuc::kMaxCluster) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(nuc::nucleus_cluster_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         nuc::kCSharedBytes + nuc::kSliceBytes);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)C);
    cfg.blockDim = dim3(nuc::NT);
    cfg.dynamicSmemBytes = (size_t)(nuc::kCSharedBytes + S * es);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int ncl = 0;
    if (cudaOccupancyMaxActiveClusters(&ncl, nuc::nucleus_cluster_kernel<T>, &cfg) != cudaSuccess || ncl < 1) {
        (void)cudaGetLastError();   // not schedulable here: the caller takes the other variant
        return cudaSuccess;
    }
    long long want = (long long)per_sm * sms / C;
    if (want > ncl) want = ncl;
    if (want > nrow) want = nrow;
    if (want < 1) want = 1;
    cfg.gridDim = dim3((unsigned)(want * C));
    e = cudaLaunchKernelEx(&cfg, nuc::nucleus_cluster_kernel<T>, a, S);
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
    e = a.bf16 ? launch_cluster<__nv_bfloat16>(a, stream, sms, nrow, launched)
               : launch_cluster<float>(a, stream, sms, nrow, launched);
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
