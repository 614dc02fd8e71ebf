// spec_nucleus.cuh -- launch interface of the nucleus (top-p) row pass,
// shared by spec_verify.cu (the caller) and spec_nucleus.cu (the kernel).
// Internal to the library: not part of the C ABI.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace sv {

struct NucleusArgs {
    const void *zt;            // [B][K+1] target rows, row stride ts elements
    const void *zd;            // [B][K] draft rows (nd_rows > 0), row stride ds
    long long ts, ds;
    int B, K, V;
    int nt_rows, nd_rows;      // rows per sequence: target rows first, then draft rows
    int t_vec_ok, d_vec_ok;    // rows start on 16-byte boundaries
    int bf16;                  // element type: 1 bf16, 0 fp32
    const int32_t *draft_len;  // [B] or null (all K verified)
    const float *inv_temp;     // [B] or null (s = 1)
    float top_p;               // in (0, 1)
    int need_ent;              // the entropy moment T is wanted (else recorded as 0)
    float4 *rec;               // [B][rows] out: (M, R, T, I) of each row's nucleus
    float *zth;                // [B][rows] out: the nucleus threshold z* (raw logit)
    unsigned *status;          // device status word (atomicMax)
    unsigned *row_ctr;         // zeroed counter: rows past the grid's first are claimed from it
};

// Enqueue the nucleus pass on `stream`. Returns a cudaError_t.
cudaError_t launch_nucleus(const NucleusArgs &a, cudaStream_t stream);

}  // namespace sv
