// HBM-bound kernels around the GEMM core: the Frobenius norm, the
// scale / cast / transpose to fp16, and the two Muon elementwise passes.
//
// Arithmetic contracts (shared with nothing else; restated from the pages):
// * Norm (Dion3 Algorithm 3, line 2, with the App. B.2.2 safety factor):
//   s = 2^k / (1.05 (||X||_F + 1e-7)). The 2^k is an exact power-of-two
//   prescale of the fp16 copy, undone by the GEMM epilogues.
//   The sum of squares is deterministic: each matrix is cut into a number of
//   chunks that depends only on its size, each chunk summed in a fixed order.
// * Momentum (Dion3 Eq. 1): M <- mu M + G, fp32, two roundings.
// * Update (Dion3 §6 "Weight Update"; Muon kernel card): decay = 1 - lr wd,
//   step = lr s, w' = decay w - step o, each fp32 operation rounded once,
//   then stochastic rounding to bf16 with Philox4x32-10 (Salmon et al.,
//   SC'11) keyed by (seed, step) and counter (g >> 2, step), g = base + i;
//   element g uses the low 16 bits of output word g & 3.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "elementwise.cuh"
#include "ptx.cuh"

namespace gns {
namespace {

constexpr int kThreads = 256;

// Launch with the programmatic-dependent-launch attribute; every kernel here
// starts with grid_dependency_wait(), so it reads nothing the previous grid
// writes before that grid has completed.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

__device__ __forceinline__ const float* mat_f32(const MatrixSet& s, int g) {
    return s.ptrs ? static_cast<const float*>(s.ptrs[g])
                  : static_cast<const float*>(s.base) + static_cast<long long>(g) * s.stride;
}

template <typename T>
__device__ __forceinline__ T* mat_ptr(const MatrixSet& s, int g) {
    return s.ptrs ? static_cast<T*>(const_cast<void*>(s.ptrs[g]))
                  : static_cast<T*>(const_cast<void*>(s.base)) + static_cast<long long>(g) * s.stride;
}

__device__ __forceinline__ long long chunk_len(long long numel, int nblk) {
    return (((numel + nblk - 1) / nblk) + 3) & ~3LL;
}

// Fixed-order block reduction of one float per thread.
__device__ __forceinline__ float block_sum(float v) {
    __shared__ float red[kThreads / 32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float t = 0.0f;
    if (threadIdx.x == 0) {
        for (int w = 0; w < kThreads / 32; ++w) t += red[w];
    }
    __syncthreads();
    return t;  // valid in thread 0
}

// Sum of x^2 over [beg, end) of x, each thread over a fixed stride.
__device__ __forceinline__ float chunk_sumsq(const float* x, long long beg, long long end) {
    float s = 0.0f;
    const bool vec = (reinterpret_cast<uintptr_t>(x) & 15) == 0;
    long long i = beg + 4LL * threadIdx.x;
    if (vec) {
        for (; i + 3 < end; i += 4LL * kThreads) {
            const float4 f = *reinterpret_cast<const float4*>(x + i);
            s = fmaf(f.x, f.x, s);
            s = fmaf(f.y, f.y, s);
            s = fmaf(f.z, f.z, s);
            s = fmaf(f.w, f.w, s);
        }
        for (int e = 0; e < 4; ++e)
            if (i + e < end) s = fmaf(x[i + e], x[i + e], s);
    } else {
        for (; i < end; i += 4LL * kThreads)
            for (int e = 0; e < 4; ++e)
                if (i + e < end) s = fmaf(x[i + e], x[i + e], s);
    }
    return s;
}

__global__ void __launch_bounds__(kThreads) sumsq_kernel(MatrixSet in, long long numel, int nblk,
                                                         float* partial) {
    grid_dependency_wait();
    grid_launch_dependents();
    const float* x = mat_f32(in, blockIdx.y);
    const long long chunk = chunk_len(numel, nblk);
    const long long beg = static_cast<long long>(blockIdx.x) * chunk;
    const long long end = beg + chunk < numel ? beg + chunk : numel;
    const float t = block_sum(beg < end ? chunk_sumsq(x, beg, end) : 0.0f);
    if (threadIdx.x == 0) partial[static_cast<long long>(blockIdx.y) * nblk + blockIdx.x] = t;
}

// Scale and cast, in the input's own layout: 4 consecutive elements per
// thread (vector load and store when aligned), grid-stride over the matrix.
__global__ void __launch_bounds__(kThreads) scale_cast_kernel(MatrixSet in, int R, int C, const float* partial,
                                                              int nblk, int k_exp, __half* out, long long ld_o,
                                                              long long stride_o, int* err) {
    __shared__ float s_scale;
    grid_dependency_wait();
    grid_launch_dependents();
    const int g = blockIdx.y;
    if (threadIdx.x == 0) {
        float t = 0.0f;
        const float* p = partial + static_cast<long long>(g) * nblk;
        for (int b = 0; b < nblk; ++b) t += p[b];
        const float norm = sqrtf(t);
        if (!isfinite(norm)) raise_error(err, kDevErrNonFinite);
        s_scale = ldexpf(1.0f, k_exp) / (1.05f * (norm + 1e-7f));
    }
    __syncthreads();
    const float scale = s_scale;
    const float* x = mat_f32(in, g);
    __half* og = out + static_cast<long long>(g) * stride_o;
    const bool vec = ((reinterpret_cast<uintptr_t>(x) & 15) == 0) && (C % 4 == 0);
    const long long groups_per_row = (C + 3) / 4;
    const long long groups = static_cast<long long>(R) * groups_per_row;
    for (long long q = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; q < groups;
         q += static_cast<long long>(gridDim.x) * kThreads) {
        const long long r = q / groups_per_row;
        const int c = static_cast<int>(q - r * groups_per_row) * 4;
        const float* src = x + r * C + c;
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        if (vec) {
            const float4 f = *reinterpret_cast<const float4*>(src);
            v[0] = f.x;
            v[1] = f.y;
            v[2] = f.z;
            v[3] = f.w;
        } else {
            for (int e = 0; e < 4; ++e)
                if (c + e < C) v[e] = src[e];
        }
        __half* dst = og + r * ld_o + c;
        // ld_o is a multiple of 8 halves and c of 4: 8-byte aligned; columns
        // past C land in the row padding.
        __half2 h01 = __floats2half2_rn(v[0] * scale, v[1] * scale);
        __half2 h23 = __floats2half2_rn(v[2] * scale, v[3] * scale);
        uint2 packed;
        packed.x = *reinterpret_cast<uint32_t*>(&h01);
        packed.y = *reinterpret_cast<uint32_t*>(&h23);
        *reinterpret_cast<uint2*>(dst) = packed;
    }
}

__global__ void __launch_bounds__(kThreads) copy_rows_kernel(const float* in, long long ld_in, long long stride_in,
                                                             float* out, int R, int C) {
    grid_dependency_wait();
    grid_launch_dependents();
    const int g = blockIdx.y;
    const long long numel = static_cast<long long>(R) * C;
    for (long long i = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; i < numel;
         i += static_cast<long long>(gridDim.x) * kThreads) {
        const long long r = i / C, c = i - r * C;
        out[static_cast<long long>(g) * numel + i] = in[static_cast<long long>(g) * stride_in + r * ld_in + c];
    }
}

__global__ void __launch_bounds__(kThreads) momentum_kernel(MatrixSet Ms, MatrixSet Gs, long long numel, int nblk,
                                                            float mu, float* partial) {
    grid_dependency_wait();
    grid_launch_dependents();
    const int g = blockIdx.y;
    float* M = mat_ptr<float>(Ms, g);
    const __nv_bfloat16* Gr = mat_ptr<const __nv_bfloat16>(Gs, g);
    const long long chunk = chunk_len(numel, nblk);
    const long long beg = static_cast<long long>(blockIdx.x) * chunk;
    const long long end = beg + chunk < numel ? beg + chunk : numel;
    float s = 0.0f;
    const bool vec = ((reinterpret_cast<uintptr_t>(M) & 15) == 0) && ((reinterpret_cast<uintptr_t>(Gr) & 7) == 0);
    long long i = beg + 4LL * threadIdx.x;
    if (vec) {
        for (; i + 3 < end; i += 4LL * kThreads) {
            float4 m = *reinterpret_cast<const float4*>(M + i);
            const uint2 graw = *reinterpret_cast<const uint2*>(Gr + i);
            const __nv_bfloat162* gb = reinterpret_cast<const __nv_bfloat162*>(&graw);
            const float2 g01 = __bfloat1622float2(gb[0]);
            const float2 g23 = __bfloat1622float2(gb[1]);
            m.x = __fadd_rn(__fmul_rn(mu, m.x), g01.x);
            m.y = __fadd_rn(__fmul_rn(mu, m.y), g01.y);
            m.z = __fadd_rn(__fmul_rn(mu, m.z), g23.x);
            m.w = __fadd_rn(__fmul_rn(mu, m.w), g23.y);
            *reinterpret_cast<float4*>(M + i) = m;
            s = fmaf(m.x, m.x, s);
            s = fmaf(m.y, m.y, s);
            s = fmaf(m.z, m.z, s);
            s = fmaf(m.w, m.w, s);
        }
    }
    for (; i < end; i += 4LL * kThreads) {
        for (int e = 0; e < 4; ++e) {
            if (i + e < end) {
                const float m = __fadd_rn(__fmul_rn(mu, M[i + e]), __bfloat162float(Gr[i + e]));
                M[i + e] = m;
                s = fmaf(m, m, s);
            }
        }
    }
    if (partial) {
        const float t = block_sum(s);
        if (threadIdx.x == 0) partial[static_cast<long long>(g) * nblk + blockIdx.x] = t;
    }
}

__device__ __forceinline__ void philox4x32_10(uint32_t (&c)[4], uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        const uint32_t hi0 = __umulhi(0xD2511F53u, c[0]);
        const uint32_t lo0 = 0xD2511F53u * c[0];
        const uint32_t hi1 = __umulhi(0xCD9E8D57u, c[2]);
        const uint32_t lo1 = 0xCD9E8D57u * c[2];
        const uint32_t n0 = hi1 ^ c[1] ^ k0;
        const uint32_t n2 = hi0 ^ c[3] ^ k1;
        c[0] = n0;
        c[1] = lo1;
        c[2] = n2;
        c[3] = lo0;
    }
}

__device__ __forceinline__ uint16_t sr_bf16(float w, uint32_t u16) {
    const uint32_t b = __float_as_uint(w);
    if ((b & 0x7F800000u) == 0x7F800000u)
        return static_cast<uint16_t>((b & 0x007FFFFFu) ? ((b >> 16) | 0x40u) : (b >> 16));
    return static_cast<uint16_t>((b + u16) >> 16);
}

// One thread per group of 4 global indices g = 4 blk .. 4 blk + 3.
__global__ void __launch_bounds__(kThreads) muon_update_kernel(MatrixSet Ws, MatrixSet Os, long long ld_o,
                                                               const long long* base_dev, long long base_scalar,
                                                               int R, int C, float lr, float wd, float scale,
                                                               uint32_t k0, uint32_t k1, uint32_t s0, uint32_t s1) {
    grid_dependency_wait();
    grid_launch_dependents();
    const int g = blockIdx.y;
    uint16_t* W = mat_ptr<uint16_t>(Ws, g);
    const __half* O = mat_ptr<const __half>(Os, g);
    const long long base = base_dev ? base_dev[g] : base_scalar;
    const long long numel = static_cast<long long>(R) * C;
    const float decay = __fsub_rn(1.0f, __fmul_rn(lr, wd));
    const float stepv = __fmul_rn(lr, scale);
    // Blocks of the global index space that overlap [base, base + numel).
    const long long blk_first = base >> 2;
    const long long blk_last = (base + numel - 1) >> 2;
    const long long nblk = blk_last - blk_first + 1;
    const bool fast = ((base & 3) == 0) && (C % 4 == 0) && (ld_o % 4 == 0) &&
                      ((reinterpret_cast<uintptr_t>(W) & 7) == 0) && ((reinterpret_cast<uintptr_t>(O) & 7) == 0);
    for (long long t = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; t < nblk;
         t += static_cast<long long>(gridDim.x) * kThreads) {
        const long long blk = blk_first + t;
        uint32_t c[4] = {static_cast<uint32_t>(blk), static_cast<uint32_t>(static_cast<unsigned long long>(blk) >> 32),
                         s0, s1};
        philox4x32_10(c, k0, k1);
        const long long i0 = blk * 4 - base;  // local index of global index 4 blk
        if (fast) {
            const long long r = i0 / C, col = i0 - r * C;
            const uint2 wraw = *reinterpret_cast<const uint2*>(W + i0);
            const uint2 oraw = *reinterpret_cast<const uint2*>(O + r * ld_o + col);
            const uint16_t* wv = reinterpret_cast<const uint16_t*>(&wraw);
            const __half* ov = reinterpret_cast<const __half*>(&oraw);
            uint16_t outv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float w = __uint_as_float(static_cast<uint32_t>(wv[e]) << 16);
                const float o = __half2float(ov[e]);
                const float wn = __fsub_rn(__fmul_rn(decay, w), __fmul_rn(stepv, o));
                outv[e] = sr_bf16(wn, c[e] & 0xFFFFu);
            }
            uint2 packed;
            packed.x = static_cast<uint32_t>(outv[0]) | (static_cast<uint32_t>(outv[1]) << 16);
            packed.y = static_cast<uint32_t>(outv[2]) | (static_cast<uint32_t>(outv[3]) << 16);
            *reinterpret_cast<uint2*>(W + i0) = packed;
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const long long i = i0 + e;
                if (i < 0 || i >= numel) continue;
                const long long r = i / C, col = i - r * C;
                const float w = __uint_as_float(static_cast<uint32_t>(W[i]) << 16);
                const float o = __half2float(O[r * ld_o + col]);
                const float wn = __fsub_rn(__fmul_rn(decay, w), __fmul_rn(stepv, o));
                W[i] = sr_bf16(wn, c[e] & 0xFFFFu);
            }
        }
    }
}

int grid_for(long long work, int per_block_items) {
    long long b = (work + per_block_items - 1) / per_block_items;
    if (b < 1) b = 1;
    if (b > 65535) b = 65535;
    return static_cast<int>(b);
}

}  // namespace

int norm_blocks(long long numel) {
    long long b = numel / (1 << 16);
    if (b < 1) b = 1;
    if (b > 64) b = 64;
    return static_cast<int>(b);
}

int launch_sumsq(const MatrixSet& in, long long numel, int G, float* partial, int* err, cudaStream_t s) {
    (void)err;
    if (G <= 0 || numel <= 0) return cudaSuccess;
    const int nblk = norm_blocks(numel);
    return launch_pdl(sumsq_kernel, dim3(nblk, G), dim3(kThreads), s, in, numel, nblk, partial);
}

int launch_scale_cast(const MatrixSet& in, int G, int R, int C, const float* partial, int nblk, int k_exp, void* out,
                      long long ld_out, long long stride_out, int* err, cudaStream_t s) {
    if (G <= 0) return cudaSuccess;
    const long long groups = static_cast<long long>(R) * ((C + 3) / 4);
    return launch_pdl(scale_cast_kernel, dim3(grid_for(groups, kThreads * 8), G), dim3(kThreads), s, in, R, C, partial,
                      nblk, k_exp, static_cast<__half*>(out), ld_out, stride_out, err);
}

int launch_copy_rows_f32(const float* in, long long ld_in, long long stride_in, float* out, int G, int R, int C,
                         cudaStream_t s) {
    if (G <= 0) return cudaSuccess;
    const long long numel = static_cast<long long>(R) * C;
    return launch_pdl(copy_rows_kernel, dim3(grid_for(numel, kThreads * 8), G), dim3(kThreads), s, in, ld_in,
                      stride_in, out, R, C);
}

int launch_momentum(const MatrixSet& M, const MatrixSet& Gr, long long numel, int count, float mu, float* partial,
                    cudaStream_t s) {
    if (count <= 0 || numel <= 0) return cudaSuccess;
    const int nblk = partial ? norm_blocks(numel) : grid_for(numel, kThreads * 16);
    return launch_pdl(momentum_kernel, dim3(nblk, count), dim3(kThreads), s, M, Gr, numel, nblk, mu, partial);
}

int launch_muon_update(const MatrixSet& W, const MatrixSet& O, long long ld_o, const long long* base_dev,
                       long long base_scalar, int count, int R, int C, float lr, float wd, float scale,
                       uint64_t seed, uint64_t step, cudaStream_t s) {
    if (count <= 0 || static_cast<long long>(R) * C <= 0) return cudaSuccess;
    const long long groups = static_cast<long long>(R) * C / 4 + 2;
    return launch_pdl(muon_update_kernel, dim3(grid_for(groups, kThreads * 4), count), dim3(kThreads), s, W, O,
                      ld_o, base_dev, base_scalar, R, C, lr, wd, scale, static_cast<uint32_t>(seed),
                      static_cast<uint32_t>(seed >> 32), static_cast<uint32_t>(step),
                      static_cast<uint32_t>(step >> 32));
}

}  // namespace gns
