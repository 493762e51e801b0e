// Launchers of the Dion3 update-rule kernels (dion3.cu).
#pragma once

#include <cmath>
#include <cstdint>
#include <cuda_runtime.h>

#include "elementwise.cuh"

namespace gns {

// Largest selection dimension the one-block selection handles (its norms sit
// in shared memory).
constexpr int kDion3MaxSelect = 16384;

// k = ceil(f n), clamped to [1, n].
int dion3_selection_count(int n, float f);

// M[g] <- M[g] + float(G[g]) (fp32 R x C, in place) and the l1 norms of its
// rows (cols = false, l1 [count][R]) or columns (cols = true, l1 [count][C]),
// each summed in a fixed order.
int launch_dion3_accumulate(const MatrixSet& M, const MatrixSet& G, int count, int R, int C, bool cols, float* l1,
                            cudaStream_t s);

// Per matrix: sel[g][0 .. k) = the indices of the k largest of its n norms,
// largest first, equal norms by lower index; pos[g][i] = rank of i, or -1
// when i is not selected. n <= kDion3MaxSelect.
int launch_dion3_select(const float* l1, int count, int n, int k, int* sel, int* pos, cudaStream_t s);

// X[g] (fp32 k x m, contiguous) = the selected rows of M[g] (m = C), or its
// selected columns as rows (cols, m = R).
int launch_dion3_gather(const MatrixSet& M, int count, int R, int C, bool cols, const int* sel, int k, float* X,
                        cudaStream_t s);

// W[g] <- SR_bf16((1 - lr wd) W - lr scale o) for every element, o the
// element's entry of O[g] (fp16 k x m, row stride ld_o, matrix stride
// stride_o) when its row (column) is selected, else 0; M[g] <- mu M[g] on the
// selected rows (columns). pos as from launch_dion3_select (nsel entries per
// matrix), base_dev[g] the global index of W[g]'s first element.
int launch_dion3_update(const MatrixSet& W, const MatrixSet& M, const void* O, long long ld_o, long long stride_o,
                        const int* pos, int nsel, const long long* base_dev, int count, int R, int C, bool cols,
                        float lr, float wd, float scale, float mu, uint64_t seed, uint64_t step, cudaStream_t s);

}  // namespace gns
