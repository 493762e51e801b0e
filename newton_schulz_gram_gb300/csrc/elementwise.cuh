// Launchers of the HBM-bound kernels (elementwise.cu).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "ptx.cuh"

namespace gns {

// A set of G matrices: either contiguous (base + g * stride) or a device
// array of per-matrix pointers (ptrs != nullptr).
struct MatrixSet {
    const void* base;
    long long stride;       // elements between matrices when contiguous
    const void* const* ptrs;
};

// The Frobenius norm is summed in parts of norm_part_len(numel) elements
// (the last one shorter), norm_parts(numel) per matrix: a function of the
// matrix size only, so a matrix's scale never depends on its bucket.
constexpr long long kNormPartElems = 16384;
constexpr int kMaxNormParts = 8192;

__host__ __device__ inline long long norm_part_len(long long numel) {
    const long long even = (numel + kMaxNormParts - 1) / kMaxNormParts;
    const long long len = (even + 3) & ~3LL;
    return len > kNormPartElems ? len : kNormPartElems;
}

__host__ __device__ inline int norm_parts(long long numel) {
    const long long len = norm_part_len(numel);
    const long long p = (numel + len - 1) / len;
    return static_cast<int>(p < 1 ? 1 : p);
}

// Norm, scale and cast of a bucket of G fp32 R x C matrices in one pass:
//   [momentum only] M[g] <- mu M[g] + float(grads[g]) (in place, fp32),
//   scale_g = 2^k_exp / (1.05 (||x_g||_F + 1e-7)),
//   out[g] (R x C, row stride ld_out, a multiple of 8) = fp16(scale_g x_g).
// partial holds G * norm_parts(R C) floats and queue 1 + G ints, which the
// caller zeroes (stream-ordered) before the launch. A non-finite norm raises
// the non-finite error word.
struct NormCastJob {
    MatrixSet in;     // fp32 input matrices, or the momentum M (updated in place)
    MatrixSet grads;  // bf16 gradients; base and ptrs both null: no momentum update
    float mu;
    int G, R, C;
    int k_exp;
    void* out;
    long long ld_out, stride_out;
    float* partial;
    int* queue;
    DevStatus st;
};

int launch_norm_cast(const NormCastJob& job, int num_sms, cudaStream_t s);

// out[g] (R x C, contiguous) = in[g] (R x C, row stride ld_in), fp32.
int launch_copy_rows_f32(const float* in, long long ld_in, long long stride_in, float* out, int G,
                         int R, int C, cudaStream_t s);

// M[g] <- mu * M[g] + float(G[g]), fp32 with two roundings.
int launch_momentum(const MatrixSet& M, const MatrixSet& Gr, long long numel, int count, float mu,
                    cudaStream_t s);

// W[g] <- SR_bf16((1 - lr wd) W[g] - (lr scale) O[g]) with Philox keyed by
// (seed, step, base + i), base = base_dev[g] when base_dev is not null, else
// base_scalar. O[g] is fp16 R x C with row stride ld_o. With row_step
// (NorMuon), row r of matrix g uses the step row_step[g R + r] in place of
// lr scale.
int launch_muon_update(const MatrixSet& W, const MatrixSet& O, long long ld_o,
                       const long long* base_dev, long long base_scalar, int count, int R, int C,
                       float lr, float wd, float scale, uint64_t seed, uint64_t step, int num_sms,
                       cudaStream_t s, const float* row_step = nullptr);

// NorMuon statistics (Dion3 Eq. 2), fp32: per row r of O[g] (fp16 R x C,
// row stride ld_o, a multiple of 8), v_r <- beta2 v_r + (1 - beta2) mean_j
// O_rj^2 into V[g] (fp32 length R, in place), inv_r = 1 / (sqrt(v_r) + eps),
// and row_sq / row_hat = sum_j O_rj^2 and its scaled counterpart
// ([count][R] each). Then launch_normuon_factor turns them into the per-row
// steps row_step = lr scale (||O|| / ||O^||) inv_r, [count][R].
int launch_normuon_rows(const MatrixSet& O, long long ld_o, const MatrixSet& V, int count, int R, int C, float beta2,
                        float eps, float* row_sq, float* row_hat, float* inv, cudaStream_t s);
int launch_normuon_factor(const float* row_sq, const float* row_hat, const float* inv, int count, int R,
                          float lr_scale, float* row_step, cudaStream_t s);

// The bounded-wait check: one block of kBoundedWaitThreads threads waits on
// an mbarrier phase (kind 0) or a counter `never` (kind 1, stays zero) that
// nothing completes; thread 0 with `first`'s bound, the others with `rest`'s.
// Adds one to *gave_up for every wait that gave up.
constexpr int kBoundedWaitThreads = 256;
int launch_bounded_wait_test(const DevStatus& first, const DevStatus& rest, int kind, const int* never,
                             int* gave_up, cudaStream_t s);

}  // namespace gns
