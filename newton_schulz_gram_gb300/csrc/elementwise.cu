// HBM-bound kernels around the GEMM core: the norm, scale and fp16 cast of
// the inputs (with the Muon momentum update first, for the Muon step), the
// Muon elementwise passes (the standalone momentum and update kernels), the
// NorMuon statistics, the copy of unaligned outputs and the bounded-wait
// check.
//
// Arithmetic contracts (shared with nothing else; restated from the pages):
// * Momentum (Dion3 Eq. 1): M <- mu M + G, fp32, two roundings.
// * Update (Dion3 §6 "Weight Update"; Muon kernel card): decay = 1 - lr wd,
//   step = lr s, w' = decay w - step o, each fp32 operation rounded once,
//   then stochastic rounding to bf16 with Philox4x32-10 (Salmon et al.,
//   SC'11) keyed by (seed, step) and counter (g >> 3, step), g = base + i;
//   element g uses 16-bit half (g & 1) of output word (g & 7) >> 1.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <cstdlib>

#include "elementwise.cuh"
#include "philox.cuh"
#include "ptx.cuh"

namespace gns {
namespace {

constexpr int kThreads = 256;
static_assert(kBoundedWaitThreads == kThreads, "the bounded-wait check runs one block of kThreads");

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

// M <- mu M + G over [beg, end) (beg a multiple of 4), fp32 with two
// roundings, by a worker of NT threads (t its thread index); returns the sum of
// squares of this thread's new M values.
template <int NT>
__device__ __forceinline__ float momentum_range(float* M, const __nv_bfloat16* Gr, long long beg, long long end,
                                                float mu, int t) {
    constexpr long long kStep = 4LL * NT;
    float s = 0.0f;
    long long i = beg + 4LL * t;
    auto upd = [&](float4& m, uint2 graw) {
        const __nv_bfloat162* gb = reinterpret_cast<const __nv_bfloat162*>(&graw);
        const float2 g01 = __bfloat1622float2(gb[0]);
        const float2 g23 = __bfloat1622float2(gb[1]);
        m.x = __fadd_rn(__fmul_rn(mu, m.x), g01.x);
        m.y = __fadd_rn(__fmul_rn(mu, m.y), g01.y);
        m.z = __fadd_rn(__fmul_rn(mu, m.z), g23.x);
        m.w = __fadd_rn(__fmul_rn(mu, m.w), g23.y);
        s = fmaf(m.x, m.x, s);
        s = fmaf(m.y, m.y, s);
        s = fmaf(m.z, m.z, s);
        s = fmaf(m.w, m.w, s);
    };
    const bool vec = ((reinterpret_cast<uintptr_t>(M) & 15) == 0) && ((reinterpret_cast<uintptr_t>(Gr) & 7) == 0);
    if (vec) {
        for (; i + 3 * kStep + 3 < end; i += 4 * kStep) {
            float4 m[4];
            uint2 gr[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                m[u] = __ldcg(reinterpret_cast<const float4*>(M + i + u * kStep));
                gr[u] = __ldcg(reinterpret_cast<const uint2*>(Gr + i + u * kStep));
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                upd(m[u], gr[u]);
                *reinterpret_cast<float4*>(M + i + u * kStep) = m[u];
            }
        }
        for (; i + 3 < end; i += kStep) {
            float4 m = __ldcg(reinterpret_cast<const float4*>(M + i));
            upd(m, __ldcg(reinterpret_cast<const uint2*>(Gr + i)));
            *reinterpret_cast<float4*>(M + i) = m;
        }
    }
    for (; i < end; i += kStep) {
        for (int e = 0; e < 4; ++e) {
            if (i + e < end) {
                const float m = __fadd_rn(__fmul_rn(mu, M[i + e]), __bfloat162float(Gr[i + e]));
                M[i + e] = m;
                s = fmaf(m, m, s);
            }
        }
    }
    return s;
}

// ---------------------------------------------------- norm + cast items
//
// An item is elements [beg, end) of one matrix, flattened row-major; a full
// item has kNormPartElems = 4 kItemVec kThreads elements (64 KB of fp32), and
// thread t owns its groups of 4 at beg + 4 (t + kThreads u), u = 0 ..
// kItemVec - 1. All kItemVec loads of a thread are issued before the first
// is used.
constexpr int kItemVec = 16;
static_assert(kNormPartElems == 4LL * kThreads * kItemVec, "a full norm part is one item");

__device__ __forceinline__ bool item_full(const void* x, long long beg, long long end) {
    return end - beg == kNormPartElems && (reinterpret_cast<uintptr_t>(x) & 15) == 0;
}

// The kItemVec float4 of a full item owned by this thread.
struct ItemRegs {
    float4 f[kItemVec];
};

__device__ __forceinline__ void item_load(ItemRegs& r, const float* x, long long beg, long long end) {
    if (item_full(x, beg, end)) {
        const float4* v = reinterpret_cast<const float4*>(x + beg) + threadIdx.x;
#pragma unroll
        for (int u = 0; u < kItemVec; ++u) r.f[u] = __ldcg(v + kThreads * u);
    }
}

// This thread's sum of squares over its groups of the item, u ascending
// (from the registers item_load filled, for a full item).
__device__ __forceinline__ float item_sumsq(const ItemRegs& r, const float* x, long long beg, long long end) {
    float s = 0.0f;
    if (item_full(x, beg, end)) {
#pragma unroll
        for (int u = 0; u < kItemVec; ++u) {
            s = fmaf(r.f[u].x, r.f[u].x, s);
            s = fmaf(r.f[u].y, r.f[u].y, s);
            s = fmaf(r.f[u].z, r.f[u].z, s);
            s = fmaf(r.f[u].w, r.f[u].w, s);
        }
    } else {
        for (long long i = beg + 4LL * threadIdx.x; i < end; i += 4LL * kThreads)
            for (int e = 0; e < 4; ++e)
                if (i + e < end) s = fmaf(x[i + e], x[i + e], s);
    }
    return s;
}

__device__ __forceinline__ float4 momentum4(float4 m, uint2 graw, float mu) {
    const __nv_bfloat162* gb = reinterpret_cast<const __nv_bfloat162*>(&graw);
    const float2 g01 = __bfloat1622float2(gb[0]);
    const float2 g23 = __bfloat1622float2(gb[1]);
    m.x = __fadd_rn(__fmul_rn(mu, m.x), g01.x);
    m.y = __fadd_rn(__fmul_rn(mu, m.y), g01.y);
    m.z = __fadd_rn(__fmul_rn(mu, m.z), g23.x);
    m.w = __fadd_rn(__fmul_rn(mu, m.w), g23.y);
    return m;
}

// M <- mu M + G over the item; returns this thread's sum of squares of the
// new M (same element order as item_sumsq).
__device__ __forceinline__ float item_momentum(float* M, const __nv_bfloat16* Gr, long long beg, long long end,
                                               float mu) {
    float s = 0.0f;
    if (item_full(M, beg, end) && (reinterpret_cast<uintptr_t>(Gr) & 7) == 0) {
        float4* mv = reinterpret_cast<float4*>(M + beg) + threadIdx.x;
        const uint2* gv = reinterpret_cast<const uint2*>(Gr + beg) + threadIdx.x;
#pragma unroll
        for (int h = 0; h < kItemVec; h += kItemVec / 2) {
            float4 m[kItemVec / 2];
            uint2 gr[kItemVec / 2];
#pragma unroll
            for (int u = 0; u < kItemVec / 2; ++u) {
                m[u] = __ldcg(mv + kThreads * (h + u));
                gr[u] = __ldcg(gv + kThreads * (h + u));
            }
#pragma unroll
            for (int u = 0; u < kItemVec / 2; ++u) {
                const float4 n = momentum4(m[u], gr[u], mu);
                mv[kThreads * (h + u)] = n;
                s = fmaf(n.x, n.x, s);
                s = fmaf(n.y, n.y, s);
                s = fmaf(n.z, n.z, s);
                s = fmaf(n.w, n.w, s);
            }
        }
    } else {
        for (long long i = beg + 4LL * threadIdx.x; i < end; i += 4LL * kThreads) {
            for (int e = 0; e < 4; ++e) {
                if (i + e < end) {
                    const float m = __fadd_rn(__fmul_rn(mu, M[i + e]), __bfloat162float(Gr[i + e]));
                    M[i + e] = m;
                    s = fmaf(m, m, s);
                }
            }
        }
    }
    return s;
}

// The cast of one item: out = fp16(scale x); element i of the matrix goes
// to row i / C, column i % C of out (row stride ld_o, a multiple of 8
// halves). A full item with C % 4 == 0 casts the registers item_load filled.
__device__ __forceinline__ bool cast_fast(const float* x, long long beg, long long end, int C) {
    return item_full(x, beg, end) && C % 4 == 0;
}

__device__ __forceinline__ void item_cast_store(const ItemRegs& r, const float* x, long long beg, long long end, int C,
                                                float scale, __half* out, long long ld_o) {
    auto h4 = [&](float4 f) {
        __half2 h01 = __floats2half2_rn(f.x * scale, f.y * scale);
        __half2 h23 = __floats2half2_rn(f.z * scale, f.w * scale);
        uint2 packed;
        packed.x = *reinterpret_cast<uint32_t*>(&h01);
        packed.y = *reinterpret_cast<uint32_t*>(&h23);
        return packed;
    };
    if (cast_fast(x, beg, end, C)) {
        if (ld_o == C) {
            uint2* o = reinterpret_cast<uint2*>(out + beg) + threadIdx.x;
#pragma unroll
            for (int u = 0; u < kItemVec; ++u) o[kThreads * u] = h4(r.f[u]);
        } else {
#pragma unroll
            for (int u = 0; u < kItemVec; ++u) {
                const long long i = beg + 4LL * (threadIdx.x + kThreads * u);
                const long long row = i / C;
                *reinterpret_cast<uint2*>(out + row * ld_o + (i - row * C)) = h4(r.f[u]);
            }
        }
    } else {
        for (long long i = beg + threadIdx.x; i < end; i += kThreads) {
            const long long row = i / C;
            out[row * ld_o + (i - row * C)] = __float2half_rn(x[i] * scale);
        }
    }
}

// ------------------------------------------------------ norm + cast queue
//
// One pass over the bucket. Matrices are taken in chunks of `mpc`; the work
// items are the norm parts S_c of chunk c (sum of squares, optionally after
// the momentum update) and its cast items C_c (the same element ranges).
// Blocks draw items from a ticket counter in the order S_0 .. S_{L-1}, then
// S_{c+L}, C_c for c = 0, 1, ...: a chunk is cast L chunks after it was
// summed, while it is still in L2. A norm part stores its partial sum and
// counts itself done (release, no wait). A cast item issues its loads, waits
// until every part of its matrix is done, sums the partials in a fixed order
// (the same in every cast item, so every item gets the same scale) and
// stores. A block holds at most two tickets (the item it works on and the
// next one) and works through them in order; every part a cast item waits
// for has a smaller ticket, held by a running block, so by induction on the
// ticket every wait ends, whatever the grid size and residency.
struct NormCastArgs {
    NormCastJob j;
    long long numel, part_len;
    int nparts, mpc, nchunks, lag, total;
};

struct NcItem {
    int sum;  // 1 norm part, 0 cast item
    int g, part;
};

// Round r of the queue is S_r (if r < nchunks) followed by C_{r-L} (if
// r >= L). Chunks hold mpc matrices except possibly the last, so the first
// k chunks hold min(k mpc, G) matrices, and round r starts at ticket
// nparts (mats(min(r, n)) + mats(clamp(r - L, 0, n))).
__device__ __forceinline__ int nc_mats_before(const NormCastArgs& a, int k) {
    const long long m = static_cast<long long>(k) * a.mpc;
    return m < a.j.G ? static_cast<int>(m) : a.j.G;
}

__device__ __forceinline__ long long nc_round_start(const NormCastArgs& a, int r) {
    const int rs = r < a.nchunks ? r : a.nchunks;
    int rc = r - a.lag;
    rc = rc < 0 ? 0 : (rc > a.nchunks ? a.nchunks : rc);
    return static_cast<long long>(a.nparts) * (nc_mats_before(a, rs) + nc_mats_before(a, rc));
}

__device__ NcItem nc_decode(const NormCastArgs& a, int q) {
    // Largest round r with start(r) <= q (start is non-decreasing in r).
    int lo = 0, hi = a.nchunks + a.lag;  // start(hi) = total > q
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (nc_round_start(a, mid) <= q)
            lo = mid;
        else
            hi = mid;
    }
    const int r = lo;
    int o = static_cast<int>(q - nc_round_start(a, r));
    if (r < a.nchunks) {
        const int ssize = (nc_mats_before(a, r + 1) - nc_mats_before(a, r)) * a.nparts;
        if (o < ssize) return {1, r * a.mpc + o / a.nparts, o % a.nparts};
        o -= ssize;
    }
    const int c = r - a.lag;
    return {0, c * a.mpc + o / a.nparts, o % a.nparts};
}

template <bool kMomentum>
__global__ void __launch_bounds__(kThreads, 2) norm_cast_kernel(const __grid_constant__ NormCastArgs a) {
    // Per-item shared values, double-buffered by item parity: a block passes
    // one barrier per item, and a buffer is written again only two items
    // later, after every thread has passed the barrier in between.
    __shared__ float red[2][kThreads / 32];
    __shared__ int s_next[2];
    __shared__ float s_scale[2];
    grid_dependency_wait();
    grid_launch_dependents();
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    int* ticket = a.j.queue;
    int* ready = a.j.queue + 1;
    // Thread 0 releases a finished part's count at the start of its block's
    // next item, after that item's loads are issued, so the release latency
    // overlaps them; always before any wait of that item.
    int pending = -1;
    auto release_pending = [&]() {
        if (t == 0 && pending >= 0) {
            red_release_add(ready + pending, 1);
            pending = -1;
        }
    };
    if (t == 0) s_next[0] = atomicAdd(ticket, 1);
    __syncthreads();
    int q = s_next[0];
    for (int k = 0; q < a.total; ++k) {
        const int b = k & 1;
        // The next ticket is taken now; its value is needed only at the barrier.
        int nxt = 0;
        if (t == 0) nxt = atomicAdd(ticket, 1);
        const NcItem it = nc_decode(a, q);
        const long long beg = it.part * a.part_len;
        const long long end = beg + a.part_len < a.numel ? beg + a.part_len : a.numel;
        ItemRegs regs;
        if (it.sum) {
            float s;
            if constexpr (kMomentum) {
                release_pending();
                s = item_momentum(mat_ptr<float>(a.j.in, it.g), mat_ptr<const __nv_bfloat16>(a.j.grads, it.g), beg,
                                  end, a.j.mu);
            } else {
                const float* x = mat_f32(a.j.in, it.g);
                item_load(regs, x, beg, end);
                release_pending();
                s = item_sumsq(regs, x, beg, end);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            if (lane == 0) red[b][warp] = s;
            if (t == 0) s_next[b ^ 1] = nxt;
            // The item's one barrier; it also orders every thread's M stores
            // (momentum) before thread 0's release at its next item.
            __syncthreads();
            if (t == 0) {
                float v = 0.0f;
                for (int w = 0; w < kThreads / 32; ++w) v += red[b][w];
                a.j.partial[static_cast<long long>(it.g) * a.nparts + it.part] = v;
                pending = it.g;
            }
        } else {
            const float* x = mat_f32(a.j.in, it.g);
            // The input is read-only here, so its loads may start before the
            // wait; the momentum is written by this kernel and is read after.
            if constexpr (!kMomentum) item_load(regs, x, beg, end);
            release_pending();
            if (warp == 0) {
                // Every part of matrix g summed: fixed-order sum of its partials
                // (the same in every cast item of g).
                bool ok = true;
                if (lane == 0) ok = wait_counter(ready + it.g, a.nparts, a.j.st);
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                if (ok) (void)ld_acquire(ready + it.g);
                // Lane l adds partials l, l + 32, l + 64, ... in that order; the
                // loads of 8 of them are issued together.
                const float* p = a.j.partial + static_cast<long long>(it.g) * a.nparts;
                float v = 0.0f;
                if (ok) {
                    for (int b0 = 0; b0 < a.nparts; b0 += 32 * 8) {
                        float pv[8];
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            const int bb = b0 + lane + 32 * u;
                            pv[u] = bb < a.nparts ? __ldcg(p + bb) : 0.0f;
                        }
#pragma unroll
                        for (int u = 0; u < 8; ++u) v += pv[u];
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                if (lane == 0) {
                    const float norm = sqrtf(v);
                    if (ok && !isfinite(norm)) raise_error(a.j.st, kDevErrNonFinite);
                    s_scale[b] = ok ? ldexpf(1.0f, a.j.k_exp) / (1.05f * (norm + 1e-7f)) : 0.0f;
                }
            }
            if (t == 0) s_next[b ^ 1] = nxt;
            __syncthreads();  // the item's one barrier: the scale and the next ticket
            if constexpr (kMomentum) item_load(regs, x, beg, end);
            item_cast_store(regs, x, beg, end, a.j.C, s_scale[b],
                            static_cast<__half*>(a.j.out) + static_cast<long long>(it.g) * a.j.stride_out,
                            a.j.ld_out);
        }
        q = s_next[b ^ 1];
    }
    release_pending();
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

// Momentum alone (no norm): blocks over fixed chunks of each matrix.
__global__ void __launch_bounds__(kThreads) momentum_kernel(MatrixSet Ms, MatrixSet Gs, long long numel, int nblk,
                                                            float mu) {
    grid_dependency_wait();
    grid_launch_dependents();
    const int g = blockIdx.y;
    const long long chunk = chunk_len(numel, nblk);
    const long long beg = static_cast<long long>(blockIdx.x) * chunk;
    const long long end = beg + chunk < numel ? beg + chunk : numel;
    if (beg < end)
        momentum_range<kThreads>(mat_ptr<float>(Ms, g), mat_ptr<const __nv_bfloat16>(Gs, g), beg, end, mu,
                                 threadIdx.x);
}

// One thread per block of 8 global indices g = 8 blk .. 8 blk + 7 (one
// Philox output). With row_step (NorMuon), row r of matrix g takes the step
// row_step[g R + r] instead of lr * scale.
__global__ void __launch_bounds__(kThreads) muon_update_kernel(MatrixSet Ws, MatrixSet Os, long long ld_o,
                                                               const long long* base_dev, long long base_scalar,
                                                               int R, int C, float lr, float wd, float scale,
                                                               const float* row_step, uint32_t k0, uint32_t k1,
                                                               uint32_t s0, uint32_t s1) {
    grid_dependency_wait();
    grid_launch_dependents();
    const int g = blockIdx.y;
    uint16_t* W = mat_ptr<uint16_t>(Ws, g);
    const __half* O = mat_ptr<const __half>(Os, g);
    const long long base = base_dev ? base_dev[g] : base_scalar;
    const long long numel = static_cast<long long>(R) * C;
    const float decay = __fsub_rn(1.0f, __fmul_rn(lr, wd));
    const float step_all = __fmul_rn(lr, scale);
    const float* rs = row_step ? row_step + static_cast<long long>(g) * R : nullptr;
    // Blocks of the global index space that overlap [base, base + numel).
    const long long blk_first = base >> 3;
    const long long blk_last = (base + numel - 1) >> 3;
    const long long nblk = blk_last - blk_first + 1;
    const bool fast = ((base & 7) == 0) && (C % 8 == 0) && (ld_o % 8 == 0) &&
                      ((reinterpret_cast<uintptr_t>(W) & 15) == 0) && ((reinterpret_cast<uintptr_t>(O) & 15) == 0);
    const long long stride = static_cast<long long>(gridDim.x) * kThreads;  // blocks per grid stride
    long long t = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x;
    if (fast) {
        // Whole blocks of eight elements of one row (base and C are multiples
        // of 8): 16-byte loads and store. The row of O is needed only for a
        // strided O or per-row steps; it is then advanced by the stride's
        // (rows, columns) instead of dividing per block.
        const long long es = stride * 8;
        const bool track = rs != nullptr || ld_o != C;
        long long i0 = t * 8, r = 0, col = 0, dr = 0, dc = 0;
        if (track) {
            r = i0 / C;
            col = i0 - r * C;
            dr = es / C;
            dc = es - dr * C;
        }
        for (; t < nblk; t += stride, i0 += es) {
            const long long blk = blk_first + t;
            uint32_t c[4] = {static_cast<uint32_t>(blk),
                             static_cast<uint32_t>(static_cast<unsigned long long>(blk) >> 32), s0, s1};
            philox4x32_10(c, k0, k1);
            const float stepv = rs ? rs[r] : step_all;
            const uint4 wraw = *reinterpret_cast<const uint4*>(W + i0);
            const uint4 oraw = *reinterpret_cast<const uint4*>(O + (track ? r * ld_o + col : i0));
            const uint16_t* wv = reinterpret_cast<const uint16_t*>(&wraw);
            const __half* ov = reinterpret_cast<const __half*>(&oraw);
            uint32_t outv[4];
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
                uint32_t pair = 0;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float w = __uint_as_float(static_cast<uint32_t>(wv[e + h]) << 16);
                    const float o = __half2float(ov[e + h]);
                    const float wn = __fsub_rn(__fmul_rn(decay, w), __fmul_rn(stepv, o));
                    pair |= static_cast<uint32_t>(sr_bf16(wn, sr_draw(c, e + h))) << (16 * h);
                }
                outv[e >> 1] = pair;
            }
            *reinterpret_cast<uint4*>(W + i0) = make_uint4(outv[0], outv[1], outv[2], outv[3]);
            if (track) {
                col += dc;
                r += dr;
                if (col >= C) {
                    col -= C;
                    ++r;
                }
            }
        }
        return;
    }
    for (; t < nblk; t += stride) {
        const long long blk = blk_first + t;
        uint32_t c[4] = {static_cast<uint32_t>(blk), static_cast<uint32_t>(static_cast<unsigned long long>(blk) >> 32),
                         s0, s1};
        philox4x32_10(c, k0, k1);
        const long long i0 = blk * 8 - base;  // local index of global index 8 blk
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const long long i = i0 + e;
            if (i < 0 || i >= numel) continue;
            const long long r = i / C, col = i - r * C;
            const float stepv = rs ? rs[r] : step_all;
            const float w = __uint_as_float(static_cast<uint32_t>(W[i]) << 16);
            const float o = __half2float(O[r * ld_o + col]);
            const float wn = __fsub_rn(__fmul_rn(decay, w), __fmul_rn(stepv, o));
            W[i] = sr_bf16(wn, sr_draw(c, e));
        }
    }
}

// NorMuon (Dion3 Eq. 2), fp32 throughout. One warp per row r of matrix g:
// s = sum_j O_rj^2 (lane l takes the 8-column groups l, l + 32, ... in
// order, then a fixed butterfly), v_r <- beta2 v_r + (1 - beta2) s / C,
// inv_r = 1 / (sqrt(v_r) + eps); stores s and s inv_r^2 for the norms.
__global__ void __launch_bounds__(kThreads) normuon_rows_kernel(MatrixSet Os, long long ld_o, MatrixSet Vs, int R,
                                                                int C, float beta2, float eps, float* row_sq,
                                                                float* row_hat, float* inv) {
    grid_dependency_wait();
    grid_launch_dependents();
    const int g = blockIdx.y;
    const int r = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= R) return;
    const __half* o = mat_ptr<const __half>(Os, g) + static_cast<long long>(r) * ld_o;
    float s = 0.0f;
    const int groups = C / 8;
    for (int q = lane; q < groups; q += 32) {
        const uint4 raw = *reinterpret_cast<const uint4*>(o + 8 * q);
        const __half2* h = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = __half22float2(h[e]);
            s = fmaf(f.x, f.x, s);
            s = fmaf(f.y, f.y, s);
        }
    }
    for (int j = 8 * groups + lane; j < C; j += 32) {
        const float f = __half2float(o[j]);
        s = fmaf(f, f, s);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) {
        float* v = mat_ptr<float>(Vs, g) + r;
        const float vn = __fadd_rn(__fmul_rn(beta2, *v), __fmul_rn(__fsub_rn(1.0f, beta2), __fdiv_rn(s, static_cast<float>(C))));
        *v = vn;
        const float iv = __frcp_rn(__fadd_rn(__fsqrt_rn(vn), eps));
        const long long k = static_cast<long long>(g) * R + r;
        row_sq[k] = s;
        row_hat[k] = __fmul_rn(__fmul_rn(s, iv), iv);
        inv[k] = iv;
    }
}

// One block per matrix: ||O||^2 and ||O^||^2 summed over the rows in a fixed
// order, factor = lr scale ||O|| / ||O^|| (0 when O^ = 0), and the per-row
// steps row_step_r = factor inv_r.
__global__ void __launch_bounds__(kThreads) normuon_factor_kernel(const float* row_sq, const float* row_hat,
                                                                  const float* inv, int R, float lr_scale,
                                                                  float* row_step) {
    __shared__ float s_sq[kThreads], s_hat[kThreads];
    __shared__ float s_factor;
    grid_dependency_wait();
    grid_launch_dependents();
    const long long off = static_cast<long long>(blockIdx.x) * R;
    float a = 0.0f, b = 0.0f;
    for (int r = threadIdx.x; r < R; r += kThreads) {
        a += row_sq[off + r];
        b += row_hat[off + r];
    }
    s_sq[threadIdx.x] = a;
    s_hat[threadIdx.x] = b;
    __syncthreads();
    for (int w = kThreads / 2; w > 0; w >>= 1) {
        if (threadIdx.x < w) {
            s_sq[threadIdx.x] += s_sq[threadIdx.x + w];
            s_hat[threadIdx.x] += s_hat[threadIdx.x + w];
        }
        __syncthreads();
    }
    if (threadIdx.x == 0)
        s_factor = s_hat[0] > 0.0f ? __fmul_rn(lr_scale, __fsqrt_rn(__fdiv_rn(s_sq[0], s_hat[0]))) : 0.0f;
    __syncthreads();
    const float f = s_factor;
    for (int r = threadIdx.x; r < R; r += kThreads) row_step[off + r] = __fmul_rn(f, inv[off + r]);
}

// Check of the bounded waits (no part of the path): every thread of one
// block waits for something that never happens, an mbarrier phase that no
// thread completes (kind 0) or a counter that nothing releases (kind 1).
// Thread 0 waits with the bound of `first`; the other threads wait with the
// much longer bound of `rest` and must give up through the abort mark that
// thread 0 raises when its own bound runs out. gave_up counts the waits that
// returned false.
__global__ void __launch_bounds__(kThreads) bounded_wait_test_kernel(DevStatus first, DevStatus rest, int kind,
                                                                     const int* never, int* gave_up) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        fence_mbar_init();
    }
    __syncthreads();
    const DevStatus st = threadIdx.x == 0 ? first : rest;
    const bool ok = kind == 0 ? mbar_wait(smem_u32(&bar), 0, st) : wait_counter(never, 1, st);
    if (!ok) atomicAdd(gave_up, 1);
}

int grid_for(long long work, int per_block_items) {
    long long b = (work + per_block_items - 1) / per_block_items;
    if (b < 1) b = 1;
    if (b > 65535) b = 65535;
    return static_cast<int>(b);
}

}  // namespace

int launch_norm_cast(const NormCastJob& job, int num_sms, cudaStream_t s) {
    if (job.G <= 0) return cudaSuccess;
    NormCastArgs a{};
    a.j = job;
    a.numel = static_cast<long long>(job.R) * job.C;
    a.nparts = norm_parts(a.numel);
    a.part_len = norm_part_len(a.numel);
    const bool momentum = job.grads.base || job.grads.ptrs;
    // Between its sum and its cast a chunk stays in L2 while the next chunk
    // is summed and the items in flight (two per block, 64 KB each) complete, so
    // both the chunk and the number of blocks are kept small. GNS_NC_CHUNK_MB
    // and GNS_NC_BLOCKS_PER_SM override them (tuning).
    long long chunk_bytes = 16LL << 20;
    if (const char* e = std::getenv("GNS_NC_CHUNK_MB")) {
        if (std::atoll(e) > 0) chunk_bytes = std::atoll(e) << 20;
    }
    a.lag = 1;
    if (const char* e = std::getenv("GNS_NC_LAG")) {
        if (std::atoi(e) > 0) a.lag = std::atoi(e);
    }
    int blocks_per_sm = 2;
    if (const char* e = std::getenv("GNS_NC_BLOCKS_PER_SM")) {
        if (std::atoi(e) > 0) blocks_per_sm = std::atoi(e);
    }
    const long long per = a.numel * (momentum ? 6 : 4);
    a.mpc = static_cast<int>(std::max(1LL, std::min<long long>(job.G, chunk_bytes / std::max(per, 1LL))));
    a.nchunks = (job.G + a.mpc - 1) / a.mpc;
    const long long total = static_cast<long long>(job.G) * 2 * a.nparts;
    if (total > (1LL << 30)) return cudaErrorInvalidValue;
    a.total = static_cast<int>(total);
    cudaError_t e = cudaSuccess;
    static int per_sm[2] = {0, 0};
    int& occ = per_sm[momentum ? 1 : 0];
    if (occ == 0) {
        e = momentum ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, norm_cast_kernel<true>, kThreads, 0)
                     : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, norm_cast_kernel<false>, kThreads, 0);
        if (e != cudaSuccess) return e;
        if (occ < 1) occ = 1;
    }
    const long long grid = std::min<long long>(static_cast<long long>(num_sms) * std::min(occ, blocks_per_sm), a.total);
    if (momentum)
        return launch_pdl(norm_cast_kernel<true>, dim3(static_cast<unsigned>(grid)), dim3(kThreads), s, a);
    return launch_pdl(norm_cast_kernel<false>, dim3(static_cast<unsigned>(grid)), dim3(kThreads), s, a);
}

int launch_copy_rows_f32(const float* in, long long ld_in, long long stride_in, float* out, int G, int R, int C,
                         cudaStream_t s) {
    if (G <= 0) return cudaSuccess;
    const long long numel = static_cast<long long>(R) * C;
    return launch_pdl(copy_rows_kernel, dim3(grid_for(numel, kThreads * 8), G), dim3(kThreads), s, in, ld_in,
                      stride_in, out, R, C);
}

int launch_momentum(const MatrixSet& M, const MatrixSet& Gr, long long numel, int count, float mu, cudaStream_t s) {
    if (count <= 0 || numel <= 0) return cudaSuccess;
    const int nblk = grid_for(numel, kThreads * 16);
    return launch_pdl(momentum_kernel, dim3(nblk, count), dim3(kThreads), s, M, Gr, numel, nblk, mu);
}

int launch_normuon_rows(const MatrixSet& O, long long ld_o, const MatrixSet& V, int count, int R, int C, float beta2,
                        float eps, float* row_sq, float* row_hat, float* inv, cudaStream_t s) {
    if (count <= 0 || R <= 0) return cudaSuccess;
    const int rows_per_block = kThreads / 32;
    return launch_pdl(normuon_rows_kernel, dim3((R + rows_per_block - 1) / rows_per_block, count), dim3(kThreads), s,
                      O, ld_o, V, R, C, beta2, eps, row_sq, row_hat, inv);
}

int launch_normuon_factor(const float* row_sq, const float* row_hat, const float* inv, int count, int R,
                          float lr_scale, float* row_step, cudaStream_t s) {
    if (count <= 0 || R <= 0) return cudaSuccess;
    return launch_pdl(normuon_factor_kernel, dim3(count), dim3(kThreads), s, row_sq, row_hat, inv, R, lr_scale,
                      row_step);
}

int launch_bounded_wait_test(const DevStatus& first, const DevStatus& rest, int kind, const int* never,
                             int* gave_up, cudaStream_t s) {
    return launch_pdl(bounded_wait_test_kernel, dim3(1), dim3(kThreads), s, first, rest, kind, never, gave_up);
}

int launch_muon_update(const MatrixSet& W, const MatrixSet& O, long long ld_o, const long long* base_dev,
                       long long base_scalar, int count, int R, int C, float lr, float wd, float scale,
                       uint64_t seed, uint64_t step, int num_sms, cudaStream_t s, const float* row_step) {
    if (count <= 0 || static_cast<long long>(R) * C <= 0) return cudaSuccess;
    // One thread per block of eight elements up to one resident wave (eight
    // 256-thread blocks per SM) over all matrices; beyond that every thread
    // strides through the matrix.
    const long long groups = static_cast<long long>(R) * C / 8 + 2;
    const long long wave = std::max(1LL, (8LL * std::max(1, num_sms) + count - 1) / count);
    const int gx = static_cast<int>(std::max(1LL, std::min(std::min(wave, 65535LL), (groups + kThreads - 1) / kThreads)));
    return launch_pdl(muon_update_kernel, dim3(gx, count), dim3(kThreads), s, W, O,
                      ld_o, base_dev, base_scalar, R, C, lr, wd, scale, row_step, static_cast<uint32_t>(seed),
                      static_cast<uint32_t>(seed >> 32), static_cast<uint32_t>(step),
                      static_cast<uint32_t>(step >> 32));
}

}  // namespace gns
