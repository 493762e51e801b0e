// Grouped, persistent tcgen05 GEMM for sm_103a.
//
// One CTA per SM walks the phase's tile list with a static stride. Warp roles:
//   warp 0      TMA producer: A and B k-blocks (64 fp16 = 128 B wide, 128-byte
//               swizzle) into a STAGES-deep ring of shared-memory slots.
//   warp 1      TMEM owner and MMA issuer: one thread issues
//               tcgen05.mma.cta_group::1.kind::f16 (M = 128, N = BN, K = 16)
//               into one of two TMEM accumulators (2 x BN fp32 columns), so
//               the epilogue of tile i overlaps the MMAs of tile i + 1.
//   warps 2-5   epilogue: tcgen05.ld of 32 x 32 sub-blocks, the fp32 epilogue
//               alpha * acc + beta * C (+ the second output delta * v + gamma I),
//               then TMA stores of the sub-block and, when asked, of its
//               transpose (the mirror write of the symmetric product, Dion3 §5
//               "Epilogue: Writing to the Transposed Tile").
//
// Symmetric products (Dion3 §5 "Triangular Scheduler", App. C.1) visit only
// tiles (i, j) with i >= j. Off-diagonal tiles write D(i, j) and D(j, i) =
// D(i, j)^T. A diagonal tile writes its strictly-lower 32 x 32 sub-blocks
// twice (direct and mirrored), its diagonal sub-blocks once after copying
// their lower half onto their upper half, and skips its upper sub-blocks;
// every element is written exactly once and D is exactly symmetric.
#include <cstdio>

#include "gemm.cuh"
#include "ptx.cuh"

namespace gns {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int kThreads = 192;

// Staging layout inside one per-warp epilogue buffer (bytes).
constexpr int kOffD = 0;       // D sub-block: fp16 (2 KB, 64B swizzle) or fp32 (4 KB, 128B swizzle)
constexpr int kOffDt = 2048;   // D^T sub-block, fp16, unswizzled 64-byte rows
constexpr int kOffD2 = 4096;   // D2 sub-block
constexpr int kOffD2t = 6144;  // D2^T sub-block

template <int BN>
struct Cfg;
template <>
struct Cfg<128> {
    static constexpr int STAGES = 5;
    static constexpr int SBUF = 8192;  // D, D^T, D2, D2^T
};
template <>
struct Cfg<256> {
    static constexpr int STAGES = 4;
    static constexpr int SBUF = 4096;  // D (fp32) or D + D^T (fp16)
};

template <int BN>
constexpr int smem_bytes() {
    return 1024 + Cfg<BN>::STAGES * (BM * BK * 2 + BN * BK * 2) + 4 * 2 * Cfg<BN>::SBUF +
           (2 * Cfg<BN>::STAGES + 5) * 8 + 16;
}

struct TileInfo {
    int p, g, m0, n0;
};

template <int BN>
__device__ __forceinline__ TileInfo decode_tile(const GemmPhase& P, int tile) {
    const int p = (P.nprob > 1 && tile >= P.prob[1].tile_begin) ? 1 : 0;
    const GemmProblem& pr = P.prob[p];
    const int local = tile - pr.tile_begin;
    const int g = local / pr.tiles_per_matrix;
    const int t = local - g * pr.tiles_per_matrix;
    int i, j;
    if (pr.flags & kFlagSym) {
        // Row-major enumeration of the lower triangle: t = i (i + 1) / 2 + j.
        i = static_cast<int>((sqrtf(8.0f * static_cast<float>(t) + 1.0f) - 1.0f) * 0.5f);
        while ((i + 1) * (i + 2) / 2 <= t) ++i;
        while (i * (i + 1) / 2 > t) --i;
        j = t - i * (i + 1) / 2;
    } else {
        i = t / pr.tiles_n;
        j = t - i * pr.tiles_n;
    }
    return TileInfo{p, g, i * BM, j * BN};
}

// Address of element (row, col) of a 32 x 32 fp16 block staged with the
// 64-byte swizzle (16-byte chunk index XOR (row / 2) mod 4).
__device__ __forceinline__ uint32_t sw64_addr(uint32_t base, int row, int col) {
    return base + row * 64 + ((((col >> 3) ^ (row >> 1)) & 3) << 4) + (col & 7) * 2;
}

// fp16 sub-block row `lane` (32 values) into a 64B-swizzled staging block.
__device__ __forceinline__ void stage_row_f16(uint32_t base, int lane, const float (&v)[32]) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t addr = base + lane * 64 + (((k ^ (lane >> 1)) & 3) << 4);
        st_shared_v4(addr, pack_half2(v[8 * k + 0], v[8 * k + 1]), pack_half2(v[8 * k + 2], v[8 * k + 3]),
                     pack_half2(v[8 * k + 4], v[8 * k + 5]), pack_half2(v[8 * k + 6], v[8 * k + 7]));
    }
}

// fp32 sub-block row into a 128B-swizzled staging block.
__device__ __forceinline__ void stage_row_f32(uint32_t base, int lane, const float (&v)[32]) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t addr = base + lane * 128 + (((k ^ lane) & 7) << 4);
        st_shared_v4(addr, __float_as_uint(v[4 * k + 0]), __float_as_uint(v[4 * k + 1]),
                     __float_as_uint(v[4 * k + 2]), __float_as_uint(v[4 * k + 3]));
    }
}

// Column `lane` of the transposed block: element (j, lane) = v[j].
__device__ __forceinline__ void stage_col_f16(uint32_t base, int lane, const float (&v)[32]) {
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const __half h = __float2half_rn(v[j]);
        st_shared_u16(base + j * 64 + lane * 2, *reinterpret_cast<const uint16_t*>(&h));
    }
}

// Upper half of a diagonal 32 x 32 block := transpose of its lower half.
__device__ __forceinline__ void symmetrize_block(uint32_t base, int lane) {
    for (int j = lane + 1; j < 32; ++j)
        st_shared_u16(sw64_addr(base, lane, j), ld_shared_u16(sw64_addr(base, j, lane)));
}

// Waits for an mbarrier phase during teardown, ignoring the error word.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer() - t0 > kWaitLimitNs) break;
    }
}

template <int BN>
__global__ void __launch_bounds__(kThreads, 1) gemm_tc_kernel(const __grid_constant__ GemmPhase P) {
    constexpr int STAGES = Cfg<BN>::STAGES;
    constexpr int SBUF = Cfg<BN>::SBUF;
    constexpr uint32_t A_BYTES = BM * BK * 2;
    constexpr uint32_t B_BYTES = BN * BK * 2;
    constexpr uint32_t TMEM_COLS = 2 * BN;
    constexpr uint32_t IDESC = idesc_f16_f32(BM, BN);

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = sA + STAGES * A_BYTES;
    uint8_t* sEpi = sB + STAGES * B_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sEpi + 4 * 2 * SBUF);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5);

    const uint32_t full0 = smem_u32(bars);
    const uint32_t empty0 = smem_u32(bars + STAGES);
    const uint32_t accf0 = smem_u32(bars + 2 * STAGES);
    const uint32_t acce0 = smem_u32(bars + 2 * STAGES + 2);
    const uint32_t drain_bar = smem_u32(bars + 2 * STAGES + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    int* err = P.err;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf0 + 8 * b, 1);
            mbar_init(acce0 + 8 * b, 4);
        }
        mbar_init(drain_bar, 1);
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        for (int p = 0; p < P.nprob; ++p) {
            prefetch_tmap(&P.prob[p].tmA);
            prefetch_tmap(&P.prob[p].tmB);
        }
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            int issued = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < P.total_tiles && ok; tile += gridDim.x) {
                const TileInfo t = decode_tile<BN>(P, tile);
                const GemmProblem& pr = P.prob[t.p];
                const int kblocks = (pr.K + BK - 1) / BK;
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!mbar_wait(empty0 + 8 * stage, phase ^ 1, err)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = full0 + 8 * stage;
                    mbar_arrive_expect_tx(fb, A_BYTES + B_BYTES);
                    tma_load_3d(smem_u32(sA + stage * A_BYTES), &pr.tmA, fb, kb * BK, t.m0, t.g);
                    tma_load_3d(smem_u32(sB + stage * B_BYTES), &pr.tmB, fb, kb * BK, t.n0, t.g);
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            // The last min(issued, STAGES) loads may still be in flight; wait
            // for each before this CTA can exit.
            const int pending = issued < STAGES ? issued : STAGES;
            for (int i = 0; i < pending; ++i) {
                if (stage == 0) {
                    stage = STAGES;
                    phase ^= 1;
                }
                --stage;
                drain_wait(full0 + 8 * stage, phase);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // -------------------------------------------------------- MMA issuer
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            int iter = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < P.total_tiles && ok; tile += gridDim.x, ++iter) {
                const TileInfo t = decode_tile<BN>(P, tile);
                const GemmProblem& pr = P.prob[t.p];
                const int kblocks = (pr.K + BK - 1) / BK;
                const int buf = iter & 1;
                if (!mbar_wait(acce0 + 8 * buf, ((iter >> 1) & 1) ^ 1, err)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + buf * BN;
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!mbar_wait(full0 + 8 * stage, phase, err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t adesc = sw128_kmajor_desc(smem_u32(sA + stage * A_BYTES));
                    const uint64_t bdesc = sw128_kmajor_desc(smem_u32(sB + stage * B_BYTES));
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        tc_mma_f16(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, IDESC, (kb | kk) != 0 ? 1u : 0u);
                    }
                    tc_commit(empty0 + 8 * stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                tc_commit(accf0 + 8 * buf);
            }
            // All MMAs issued by this thread must finish before TMEM is freed.
            tc_commit(drain_bar);
            drain_wait(drain_bar, 0);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------- epilogue
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const int ew = warp - 2;
        int iter = 0;
        uint32_t groups = 0;
        for (int tile = blockIdx.x; tile < P.total_tiles; tile += gridDim.x, ++iter) {
            const TileInfo t = decode_tile<BN>(P, tile);
            const GemmProblem& pr = P.prob[t.p];
            const int buf = iter & 1;
            if (!mbar_wait(accf0 + 8 * buf, (iter >> 1) & 1, err)) break;
            tc_fence_after();

            const int flags = pr.flags;
            const bool sym = flags & kFlagSym;
            const bool diag_tile = sym && (t.m0 == t.n0);
            const int r0 = t.m0 + q * 32;
            const int grow = r0 + lane;
            const bool rows_live = r0 < pr.M;

#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                const int c0 = t.n0 + c * 32;
                if (!rows_live || c0 >= pr.N) continue;
                if (diag_tile && c > q) continue;
                const bool diag_block = diag_tile && (c == q);

                uint32_t acc[32];
                tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * BN + c * 32, acc);
                tmem_ld_wait();

                float v[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = pr.alpha * __uint_as_float(acc[j]);
                if ((flags & kFlagC) && grow < pr.M) {
                    const __half* crow = pr.C + static_cast<long long>(t.g) * pr.strideC +
                                         static_cast<long long>(grow) * pr.ldc + c0;
                    if (c0 + 32 <= pr.N) {
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const uint4 raw = *reinterpret_cast<const uint4*>(crow + 8 * k);
                            const __half2* h = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float2 f = __half22float2(h[e]);
                                v[8 * k + 2 * e] = fmaf(pr.beta, f.x, v[8 * k + 2 * e]);
                                v[8 * k + 2 * e + 1] = fmaf(pr.beta, f.y, v[8 * k + 2 * e + 1]);
                            }
                        }
                    } else {
                        for (int j = 0; j < 32; ++j)
                            if (c0 + j < pr.N) v[j] = fmaf(pr.beta, __half2float(crow[j]), v[j]);
                    }
                }

                uint8_t* st = sEpi + (ew * 2 + (groups & 1)) * SBUF;
                const uint32_t sbase = smem_u32(st);
                if (lane == 0) bulk_wait_read<1>();
                __syncwarp();

                if (flags & kFlagOutF32) {
                    stage_row_f32(sbase + kOffD, lane, v);
                } else {
                    stage_row_f16(sbase + kOffD, lane, v);
                    if ((flags & kFlagDt) && !diag_block) stage_col_f16(sbase + kOffDt, lane, v);
                }
                if (flags & kFlagD2) {
                    float v2[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        v2[j] = pr.delta * v[j] + ((grow == c0 + j) ? pr.gamma : 0.0f);
                    stage_row_f16(sbase + kOffD2, lane, v2);
                    if ((flags & kFlagDt) && !diag_block) stage_col_f16(sbase + kOffD2t, lane, v2);
                }
                if (diag_block) {
                    __syncwarp();
                    symmetrize_block(sbase + kOffD, lane);
                    if (flags & kFlagD2) symmetrize_block(sbase + kOffD2, lane);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_3d(&pr.tmD, sbase + kOffD, c0, r0, t.g);
                    if ((flags & kFlagDt) && !diag_block) tma_store_3d(&pr.tmDt, sbase + kOffDt, r0, c0, t.g);
                    if (flags & kFlagD2) {
                        tma_store_3d(&pr.tmD2, sbase + kOffD2, c0, r0, t.g);
                        if ((flags & kFlagDt) && !diag_block)
                            tma_store_3d(&pr.tmD2t, sbase + kOffD2t, r0, c0, t.g);
                    }
                    bulk_commit();
                }
                ++groups;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acce0 + 8 * buf);
        }
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

template <int BN>
int launch_impl(const GemmPhase& phase, int num_sms, cudaStream_t stream) {
    static bool configured = false;
    constexpr int bytes = smem_bytes<BN>();
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    if (phase.total_tiles <= 0) return cudaSuccess;
    const int grid = phase.total_tiles < num_sms ? phase.total_tiles : num_sms;
    gemm_tc_kernel<BN><<<grid, kThreads, bytes, stream>>>(phase);
    return cudaGetLastError();
}

}  // namespace

int gemm_smem_bytes(int bn) { return bn == 256 ? smem_bytes<256>() : smem_bytes<128>(); }

int launch_gemm_phase(const GemmPhase& phase, int bn, int num_sms, cudaStream_t stream) {
    if (bn == 256) return launch_impl<256>(phase, num_sms, stream);
    return launch_impl<128>(phase, num_sms, stream);
}

}  // namespace gns
