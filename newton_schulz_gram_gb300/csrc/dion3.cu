// Kernels of the Dion3 update rule ("Dion3: Full-stack orthogonal updates",
// §6 and Algorithm 4, Muon flavor) around the Gram Newton-Schulz core:
// momentum accumulation with l1 norms along the selection dimension, top-k
// selection, gather of the selected rows (or columns), and the update with
// error feedback.
//
// Arithmetic contracts (restated from the pages):
// * M <- M + G: fp32, one rounding, G promoted from bf16 (Algorithm 4 line 2).
// * Selection: the k rows (or columns) with the largest l1 norm, largest
//   first, equal norms by lower index; NaN norms count as +infinity so the
//   ranks always form a permutation.
// * Update, every element: w' = decay w - step o with o = 0 outside the
//   selection (decay = 1 - lr wd, step = lr scale, single fp32 roundings),
//   then the Muon flavor's stochastic rounding keyed by the global index.
//   Error feedback: M <- mu M (fp32) on the selected rows only.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "dion3.cuh"
#include "philox.cuh"
#include "ptx.cuh"

namespace gns {
namespace {

constexpr int kThreads = 256;

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

template <typename T>
__device__ __forceinline__ T* ptr_of(const MatrixSet& s, int g) {
    return s.ptrs ? static_cast<T*>(const_cast<void*>(s.ptrs[g]))
                  : static_cast<T*>(const_cast<void*>(s.base)) + static_cast<long long>(g) * s.stride;
}

__device__ __forceinline__ float l1_key(float v) { return isnan(v) ? __int_as_float(0x7f800000) : v; }

// Row mode: one warp per row; lane l takes columns l, l + 32, ... in order,
// then a fixed butterfly.
__global__ void __launch_bounds__(kThreads) accumulate_rows_kernel(MatrixSet Ms, MatrixSet Gs, int R, int C,
                                                                   float* l1) {
    grid_dependency_wait();
    grid_launch_dependents();
    const int g = blockIdx.y;
    const int r = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= R) return;
    float* m = ptr_of<float>(Ms, g) + static_cast<long long>(r) * C;
    const __nv_bfloat16* gr = ptr_of<const __nv_bfloat16>(Gs, g) + static_cast<long long>(r) * C;
    float s = 0.0f;
    for (int j = lane; j < C; j += 32) {
        const float v = __fadd_rn(m[j], __bfloat162float(gr[j]));
        m[j] = v;
        s = __fadd_rn(s, fabsf(v));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, o));
    if (lane == 0) l1[static_cast<long long>(g) * R + r] = s;
}

// Column mode: a block owns 32 columns; warp w takes rows w, w + 8, ... in
// order for its lane's column; the 8 warp partials are added in order.
__global__ void __launch_bounds__(kThreads) accumulate_cols_kernel(MatrixSet Ms, MatrixSet Gs, int R, int C,
                                                                   float* l1) {
    __shared__ float part[kThreads / 32][32];
    grid_dependency_wait();
    grid_launch_dependents();
    const int g = blockIdx.y;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int c = blockIdx.x * 32 + lane;
    float* m = ptr_of<float>(Ms, g);
    const __nv_bfloat16* gr = ptr_of<const __nv_bfloat16>(Gs, g);
    float s = 0.0f;
    if (c < C) {
        for (int r = warp; r < R; r += kThreads / 32) {
            const long long i = static_cast<long long>(r) * C + c;
            const float v = __fadd_rn(m[i], __bfloat162float(gr[i]));
            m[i] = v;
            s = __fadd_rn(s, fabsf(v));
        }
    }
    part[warp][lane] = s;
    __syncthreads();
    if (warp == 0 && c < C) {
        float t = part[0][lane];
        for (int w = 1; w < kThreads / 32; ++w) t = __fadd_rn(t, part[w][lane]);
        l1[static_cast<long long>(g) * C + c] = t;
    }
}

// One block per matrix: the rank of every candidate among the n norms (in
// shared memory); ranks below k are selected.
__global__ void __launch_bounds__(1024) select_kernel(const float* l1, int n, int k, int* sel, int* pos) {
    extern __shared__ float key[];
    grid_dependency_wait();
    grid_launch_dependents();
    const int g = blockIdx.x;
    const float* x = l1 + static_cast<long long>(g) * n;
    for (int i = threadIdx.x; i < n; i += blockDim.x) key[i] = l1_key(x[i]);
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const float v = key[i];
        int rank = 0;
        for (int j = 0; j < n; ++j) {
            const float u = key[j];
            rank += (u > v || (u == v && j < i)) ? 1 : 0;
        }
        if (rank < k) sel[static_cast<long long>(g) * k + rank] = i;
        pos[static_cast<long long>(g) * n + i] = rank < k ? rank : -1;
    }
}

// X[g][p][:] = row sel[p] of M[g] (row mode), one warp per output row.
__global__ void __launch_bounds__(kThreads) gather_rows_kernel(MatrixSet Ms, int C, const int* sel, int k,
                                                               float* X) {
    grid_dependency_wait();
    grid_launch_dependents();
    const int g = blockIdx.y;
    const int p = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (p >= k) return;
    const float* src = ptr_of<const float>(Ms, g) + static_cast<long long>(sel[static_cast<long long>(g) * k + p]) * C;
    float* dst = X + (static_cast<long long>(g) * k + p) * C;
    for (int j = lane; j < C; j += 32) dst[j] = src[j];
}

// X[g][p][i] = M[g][i][sel[p]] (column mode): 32 x 32 tiles through shared
// memory, so the stores are coalesced.
__global__ void __launch_bounds__(1024) gather_cols_kernel(MatrixSet Ms, int R, int C, const int* sel, int k,
                                                           float* X) {
    __shared__ float tile[32][33];
    grid_dependency_wait();
    grid_launch_dependents();
    const int g = blockIdx.z;
    const int i0 = blockIdx.x * 32, p0 = blockIdx.y * 32;
    const int tx = threadIdx.x, ty = threadIdx.y;
    const float* m = ptr_of<const float>(Ms, g);
    if (i0 + ty < R && p0 + tx < k) {
        const int col = sel[static_cast<long long>(g) * k + p0 + tx];
        tile[ty][tx] = m[static_cast<long long>(i0 + ty) * C + col];
    }
    __syncthreads();
    if (p0 + ty < k && i0 + tx < R) X[(static_cast<long long>(g) * k + p0 + ty) * R + i0 + tx] = tile[tx][ty];
}

// Every element of W[g] (R x C): o from O (row or column p of the selection,
// or 0), the fused update with stochastic rounding, and error feedback on
// the selected part of M. One thread per block of 8 global indices (one
// Philox output).
__global__ void __launch_bounds__(kThreads) update_kernel(MatrixSet Ws, MatrixSet Ms, const __half* O, long long ld_o,
                                                          long long stride_o, const int* pos, int nsel,
                                                          const long long* base_dev, int R, int C, int cols,
                                                          float lr, float wd, float scale, float mu, uint32_t k0,
                                                          uint32_t k1, uint32_t s0, uint32_t s1) {
    grid_dependency_wait();
    grid_launch_dependents();
    const int g = blockIdx.y;
    uint16_t* W = ptr_of<uint16_t>(Ws, g);
    float* M = ptr_of<float>(Ms, g);
    const __half* Og = O + static_cast<long long>(g) * stride_o;
    const int* pg = pos + static_cast<long long>(g) * nsel;
    const long long base = base_dev[g];
    const long long numel = static_cast<long long>(R) * C;
    const float decay = __fsub_rn(1.0f, __fmul_rn(lr, wd));
    const float stepv = __fmul_rn(lr, scale);
    const long long blk_first = base >> 3;
    const long long nblk = ((base + numel - 1) >> 3) - blk_first + 1;
    for (long long t = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; t < nblk;
         t += static_cast<long long>(gridDim.x) * kThreads) {
        const long long blk = blk_first + t;
        uint32_t c[4] = {static_cast<uint32_t>(blk), static_cast<uint32_t>(static_cast<unsigned long long>(blk) >> 32),
                         s0, s1};
        philox4x32_10(c, k0, k1);
        const long long i0 = blk * 8 - base;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const long long i = i0 + e;
            if (i < 0 || i >= numel) continue;
            const int r = static_cast<int>(i / C), col = static_cast<int>(i - static_cast<long long>(r) * C);
            const int p = cols ? pg[col] : pg[r];
            float o = 0.0f;
            if (p >= 0) {
                o = __half2float(cols ? Og[static_cast<long long>(p) * ld_o + r] : Og[static_cast<long long>(p) * ld_o + col]);
                M[i] = __fmul_rn(mu, M[i]);
            }
            const float w = __uint_as_float(static_cast<uint32_t>(W[i]) << 16);
            const float wn = __fsub_rn(__fmul_rn(decay, w), __fmul_rn(stepv, o));
            W[i] = sr_bf16(wn, sr_draw(c, e));
        }
    }
}

int blocks_for(long long work, int per_block) {
    long long b = (work + per_block - 1) / per_block;
    return static_cast<int>(b < 1 ? 1 : (b > 65535 ? 65535 : b));
}

}  // namespace

int dion3_selection_count(int n, float f) {
    const double x = std::ceil(static_cast<double>(f) * n - 1e-9);
    int k = static_cast<int>(x);
    if (k < 1) k = 1;
    if (k > n) k = n;
    return k;
}

int launch_dion3_accumulate(const MatrixSet& M, const MatrixSet& G, int count, int R, int C, bool cols, float* l1,
                            cudaStream_t s) {
    if (count <= 0) return cudaSuccess;
    if (!cols)
        return launch_pdl(accumulate_rows_kernel, dim3((R + 7) / 8, count), dim3(kThreads), 0, s, M, G, R, C, l1);
    return launch_pdl(accumulate_cols_kernel, dim3((C + 31) / 32, count), dim3(kThreads), 0, s, M, G, R, C, l1);
}

int launch_dion3_select(const float* l1, int count, int n, int k, int* sel, int* pos, cudaStream_t s) {
    if (count <= 0) return cudaSuccess;
    if (n > kDion3MaxSelect) return cudaErrorInvalidValue;
    const size_t smem = sizeof(float) * static_cast<size_t>(n);
    if (smem > 48 * 1024) {
        const cudaError_t e =
            cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    return launch_pdl(select_kernel, dim3(count), dim3(1024), smem, s, l1, n, k, sel, pos);
}

int launch_dion3_gather(const MatrixSet& M, int count, int R, int C, bool cols, const int* sel, int k, float* X,
                        cudaStream_t s) {
    if (count <= 0) return cudaSuccess;
    if (!cols) return launch_pdl(gather_rows_kernel, dim3((k + 7) / 8, count), dim3(kThreads), 0, s, M, C, sel, k, X);
    return launch_pdl(gather_cols_kernel, dim3((R + 31) / 32, (k + 31) / 32, count), dim3(32, 32), 0, s, M, R, C, sel,
                      k, X);
}

int launch_dion3_update(const MatrixSet& W, const MatrixSet& M, const void* O, long long ld_o, long long stride_o,
                        const int* pos, int nsel, const long long* base_dev, int count, int R, int C, bool cols,
                        float lr, float wd, float scale, float mu, uint64_t seed, uint64_t step, cudaStream_t s) {
    if (count <= 0) return cudaSuccess;
    const long long groups = static_cast<long long>(R) * C / 8 + 2;
    return launch_pdl(update_kernel, dim3(blocks_for(groups, kThreads * 2), count), dim3(kThreads), 0, s, W, M,
                      static_cast<const __half*>(O), ld_o, stride_o, pos, nsel, base_dev, R, C, cols ? 1 : 0, lr, wd,
                      scale, mu, static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32),
                      static_cast<uint32_t>(step), static_cast<uint32_t>(step >> 32));
}

}  // namespace gns
