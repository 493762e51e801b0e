// Launchers of the HBM-bound kernels (elementwise.cu).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace gns {

// A set of G matrices: either contiguous (base + g * stride) or a device
// array of per-matrix pointers (ptrs != nullptr).
struct MatrixSet {
    const void* base;
    long long stride;       // elements between matrices when contiguous
    const void* const* ptrs;
};

// Number of partial sums per matrix for the deterministic norm (depends on
// the matrix size only, so results never depend on the bucket size G).
int norm_blocks(long long numel);

// partial[g * nblk + b] = sum of squares of chunk b of fp32 matrix g.
int launch_sumsq(const MatrixSet& in, long long numel, int G, float* partial, int* err,
                 cudaStream_t s);

// Scale and cast an fp32 R x C matrix set to fp16 in the same layout:
//   scale_g = 2^k / (1.05 * (sqrt(sum_b partial[g][b]) + 1e-7)),
//   out[g] (R x C, row stride ld_out, a multiple of 8) = fp16(scale_g * x).
// A non-finite norm raises the non-finite error word.
int launch_scale_cast(const MatrixSet& in, int G, int R, int C, const float* partial, int nblk, int k_exp, void* out,
                      long long ld_out, long long stride_out, int* err, cudaStream_t s);

// out[g] (R x C, contiguous) = in[g] (R x C, row stride ld_in), fp32.
int launch_copy_rows_f32(const float* in, long long ld_in, long long stride_in, float* out, int G,
                         int R, int C, cudaStream_t s);

// M[g] <- mu * M[g] + float(G[g]); optionally per-matrix sum-of-squares
// partials of the new M (same chunking as launch_sumsq).
int launch_momentum(const MatrixSet& M, const MatrixSet& Gr, long long numel, int count, float mu,
                    float* partial, cudaStream_t s);

// W[g] <- SR_bf16((1 - lr wd) W[g] - (lr scale) O[g]) with Philox keyed by
// (seed, step, base + i), base = base_dev[g] when base_dev is not null, else
// base_scalar. O[g] is fp16 R x C with row stride ld_o.
int launch_muon_update(const MatrixSet& W, const MatrixSet& O, long long ld_o,
                       const long long* base_dev, long long base_scalar, int count, int R, int C,
                       float lr, float wd, float scale, uint64_t seed, uint64_t step,
                       cudaStream_t s);

}  // namespace gns
