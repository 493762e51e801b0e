// Grouped, persistent tcgen05 GEMM for sm_103a.
//
// One CTA (or CTA pair) per SM (pair of SMs) walks the program's tile list
// with a static stride. Tiles of later phases wait, per matrix, for the
// earlier phases' tiles of the same matrix (see gemm.cuh). Warp roles:
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
// the 128 x BN tiles that touch the lower triangle (row block i holds the
// column blocks j with j * BN <= 128 i + 127). Each 32 x 32 sub-block is then
// classified by its global position: strictly lower sub-blocks are written
// directly and mirrored, diagonal sub-blocks are written once after their
// upper half is replaced by the transpose of their lower half, upper
// sub-blocks are skipped. Every element is written exactly once and the
// result is exactly symmetric.
//
// Transposed sub-blocks are built in shared memory with ldmatrix.trans /
// stmatrix; all fp16 staging uses the 64-byte swizzle of its TMA maps.
#include <cstdio>

#include "gemm.cuh"
#include "philox.cuh"
#include "ptx.cuh"

namespace gns {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;
static_assert(sizeof(GemmProgram) <= 32764, "kernel parameter block too large");
constexpr int kEpiWarps = 8;                 // two per TMEM lane quarter
constexpr int kThreads = 64 + 32 * kEpiWarps;  // producer, MMA, epilogue

// One per-warp epilogue staging buffer (bytes): a 32 x 32 fp16 block and its
// transpose, or one 32 x 32 fp32 block. A second output reuses it in a
// second pass.
constexpr int SBUF = 4096;
constexpr int kOffD = 0;
constexpr int kOffDt = 2048;

// Kernel variants: <BN, CG>. CG = 1: one CTA computes a 128 x BN tile.
// CG = 2: a cluster of two CTAs computes a 256 x BN tile with paired MMAs
// (tcgen05.mma.cta_group::2, M = 256); each CTA stages its 128 rows of A and
// BN / 2 rows of B, so a stage costs half the shared memory per MMA.
template <int BN, int CG>
struct Cfg;
template <>
struct Cfg<128, 1> {
    static constexpr int STAGES = 6;
};
template <>
struct Cfg<256, 1> {
    static constexpr int STAGES = 4;
};
template <>
struct Cfg<256, 2> {
    static constexpr int STAGES = 6;
};

template <int BN, int CG>
constexpr int smem_bytes() {
    return 1024 + Cfg<BN, CG>::STAGES * (BM * BK * 2 + (BN / CG) * BK * 2) + kEpiWarps * SBUF +
           (2 * Cfg<BN, CG>::STAGES + 5) * 8 + 16;
}

struct TileInfo {
    int p, g, m0, n0, s;  // problem, matrix, tile origin, phase
};

// Column blocks a symmetric row block of height tm touches: j * bn <= tm i + tm - 1
// (rounded up to even when two CTA pairs share the row's A).
__host__ __device__ __forceinline__ int sym_row_tiles(int i, int tm, int bn, int tiles_n, bool share) {
    int c = (tm * i + tm - 1) / bn + 1;
    c = c < tiles_n ? c : tiles_n;
    return share ? c + (c & 1) : c;
}

template <int BN, int CG>
__device__ __forceinline__ TileInfo decode_tile(const GemmProgram& P, int tile) {
    constexpr int TM = BM * CG;
    int s = 0;
    while (s + 1 < P.nphase && tile >= P.phase[s + 1].tile_begin) ++s;
    const GemmPhaseDesc& ph = P.phase[s];
    const int local = tile - ph.tile_begin;
    int g = local / ph.tiles_per_matrix;
    int t = local - g * ph.tiles_per_matrix;
    if (ph.reverse) g = P.G - 1 - g;
    int p = ph.prob_begin;
    while (t >= P.prob[p].tiles_per_matrix) {
        t -= P.prob[p].tiles_per_matrix;
        ++p;
    }
    const GemmProblem& pr = P.prob[p];
    int i, j;
    // Tiles past the real ones (padding) decode to out-of-range tiles: their
    // loads read zeros and their epilogue writes nothing.
    if (pr.flags & kFlagSym) {
        const bool share = pr.flags & kFlagShareA;
        int acc = 0;
        i = 0;
        while (true) {
            const int cnt = sym_row_tiles(i, TM, BN, pr.tiles_n, share);
            if (t < acc + cnt) break;
            acc += cnt;
            ++i;
        }
        j = t - acc;
    } else {
        i = t / pr.tiles_n_walk;
        j = t - i * pr.tiles_n_walk;
    }
    return TileInfo{p, g, i * TM, j * BN, s};
}

// An MN-major operand tile is staged as 64-wide M/N blocks of 64 K rows
// (one TMA box each), 8 KB apart.
constexpr uint32_t kMnBlockBytes = 64 * BK * 2;

// One k-block of one operand into shared memory: a K-major tile is one box
// {64 (K), rows}; an MN-major tile is rows / 64 boxes {64 (M or N), 64 (K)}.
// mode 0: this CTA's own barrier; 1: the pair leader's barrier (bar is a
// cluster address); 2: multicast to the CTAs in `mask`, completing on the
// pair leader's barrier of each destination.
__device__ __forceinline__ void load_operand(int mode, uint32_t dst, const CUtensorMap* map, uint32_t bar, bool mn,
                                             int row0, int rows, int kb, int g, uint16_t mask) {
    const int boxes = mn ? rows / 64 : 1;
    for (int h = 0; h < boxes; ++h) {
        const uint32_t d = dst + h * kMnBlockBytes;
        const int c0 = mn ? row0 + 64 * h : kb * BK;
        const int c1 = mn ? kb * BK : row0;
        if (mode == 0)
            tma_load_3d(d, map, bar, c0, c1, g);
        else if (mode == 1)
            tma_load_3d_pair(d, map, bar, c0, c1, g);
        else
            tma_load_3d_multicast_pair(d, map, bar, c0, c1, g, mask);
    }
}

// Address of element (row, col) of a 32 x 32 fp16 block staged with the
// 64-byte swizzle (16-byte chunk index XOR (row / 2) mod 4).
__device__ __forceinline__ uint32_t sw64_addr(uint32_t base, int row, int col) {
    return base + row * 64 + ((((col >> 3) ^ (row >> 1)) & 3) << 4) + (col & 7) * 2;
}

// Row `lane` (32 values) of a 64B-swizzled fp16 block.
__device__ __forceinline__ void stage_row_f16(uint32_t base, int lane, const float (&v)[32]) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t addr = base + lane * 64 + (((k ^ (lane >> 1)) & 3) << 4);
        st_shared_v4(addr, pack_half2(v[8 * k + 0], v[8 * k + 1]), pack_half2(v[8 * k + 2], v[8 * k + 3]),
                     pack_half2(v[8 * k + 4], v[8 * k + 5]), pack_half2(v[8 * k + 6], v[8 * k + 7]));
    }
}

// Row `lane` of a 128B-swizzled fp32 block.
__device__ __forceinline__ void stage_row_f32(uint32_t base, int lane, const float (&v)[32]) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t addr = base + lane * 128 + (((k ^ lane) & 7) << 4);
        st_shared_v4(addr, __float_as_uint(v[4 * k + 0]), __float_as_uint(v[4 * k + 1]),
                     __float_as_uint(v[4 * k + 2]), __float_as_uint(v[4 * k + 3]));
    }
}

// dst = src^T for a 32 x 32 fp16 block (both 64B-swizzled): 8 x 8 block (R, i)
// of src, loaded transposed, is stored as block (i, R) of dst.
__device__ __forceinline__ void transpose_block(uint32_t src, uint32_t dst, int lane) {
#pragma unroll
    for (int R = 0; R < 4; ++R) {
        uint32_t a0, a1, a2, a3;
        ldmatrix_x4_trans(sw64_addr(src, 8 * R + (lane & 7), 8 * (lane >> 3)), a0, a1, a2, a3);
        stmatrix_x4(sw64_addr(dst, lane, 8 * R), a0, a1, a2, a3);
    }
}

// Diagonal block: row `lane` keeps its lower part (col <= lane) and takes the
// upper part from the transposed copy, i.e. D(r, c) = D(c, r) for c > r.
__device__ __forceinline__ void merge_upper(uint32_t d, uint32_t dt, int lane) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int c0 = 8 * k;
        if (c0 > lane) {
            const uint4 v = ld_shared_v4(sw64_addr(dt, lane, c0));
            st_shared_v4(sw64_addr(d, lane, c0), v.x, v.y, v.z, v.w);
        } else if (c0 + 7 > lane) {
            for (int e = 0; e < 8; ++e)
                if (c0 + e > lane) st_shared_u16(sw64_addr(d, lane, c0 + e), ld_shared_u16(sw64_addr(dt, lane, c0 + e)));
        }
    }
}

// Row `grow` of C, columns c0 .. c0 + 31, as 16 packed fp16 pairs.
__device__ __forceinline__ void load_c(const GemmProblem& pr, int g, int grow, int c0, uint4 (&cb)[4]) {
    if (grow >= pr.M) {
#pragma unroll
        for (int k = 0; k < 4; ++k) cb[k] = make_uint4(0, 0, 0, 0);
        return;
    }
    const __half* crow = pr.C + static_cast<long long>(g) * pr.strideC + static_cast<long long>(grow) * pr.ldc + c0;
    if (c0 + 32 <= pr.N) {
#pragma unroll
        for (int k = 0; k < 4; ++k) cb[k] = *reinterpret_cast<const uint4*>(crow + 8 * k);
    } else {
        uint16_t h[32];
        for (int j = 0; j < 32; ++j) h[j] = (c0 + j < pr.N) ? reinterpret_cast<const uint16_t*>(crow)[j] : 0;
#pragma unroll
        for (int k = 0; k < 4; ++k)
            cb[k] = make_uint4(h[8 * k] | (uint32_t(h[8 * k + 1]) << 16), h[8 * k + 2] | (uint32_t(h[8 * k + 3]) << 16),
                               h[8 * k + 4] | (uint32_t(h[8 * k + 5]) << 16), h[8 * k + 6] | (uint32_t(h[8 * k + 7]) << 16));
    }
}

// Fused Muon update of one output row segment: columns c0 .. c0 + 31 of row
// `row` of matrix g, whose output values (alpha acc) are v. Each value is
// rounded to fp16 first (the value the unfused path stores and reads back),
// so the result equals the separate update kernel's bit for bit.
__device__ __forceinline__ void muon_update_row(const GemmProblem& pr, int g, int row, int c0, const float (&v)[32]) {
    if (row >= pr.M || c0 >= pr.N) return;
    const MuonFuse& mf = pr.muon;
    const float decay = __fsub_rn(1.0f, __fmul_rn(mf.lr, mf.wd));
    const float stepv = __fmul_rn(mf.lr, mf.scale);
    const long long i0 = static_cast<long long>(row) * pr.N + c0;
    const unsigned long long g0 = static_cast<unsigned long long>(mf.base[g] + i0);
    uint16_t* wp = mf.w[g] + i0;
    const int ncol = pr.N - c0 < 32 ? pr.N - c0 : 32;
    auto upd = [&](uint16_t wbits, float acc, uint32_t u) -> uint16_t {
        const float o = __half2float(__float2half_rn(acc));
        const float w = __uint_as_float(static_cast<uint32_t>(wbits) << 16);
        const float wn = __fsub_rn(__fmul_rn(decay, w), __fmul_rn(stepv, o));
        return sr_bf16(wn, u & 0xFFFFu);
    };
    // Register arrays only: every index below is a compile-time constant
    // (a runtime index would move v to local memory for every tile).
    if (ncol == 32 && (g0 & 3) == 0 && (reinterpret_cast<uintptr_t>(wp) & 15) == 0) {
        uint32_t wv[16];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint4 x = reinterpret_cast<const uint4*>(wp)[k];
            wv[4 * k + 0] = x.x;
            wv[4 * k + 1] = x.y;
            wv[4 * k + 2] = x.z;
            wv[4 * k + 3] = x.w;
        }
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            const unsigned long long blk = (g0 >> 2) + b;
            uint32_t c[4] = {static_cast<uint32_t>(blk), static_cast<uint32_t>(blk >> 32), mf.step_lo, mf.step_hi};
            philox4x32_10(c, mf.seed_lo, mf.seed_hi);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t pair = wv[2 * b + h];
                const uint32_t lo = upd(static_cast<uint16_t>(pair & 0xFFFFu), v[4 * b + 2 * h], c[2 * h]);
                const uint32_t hi = upd(static_cast<uint16_t>(pair >> 16), v[4 * b + 2 * h + 1], c[2 * h + 1]);
                wv[2 * b + h] = lo | (hi << 16);
            }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k)
            reinterpret_cast<uint4*>(wp)[k] = make_uint4(wv[4 * k + 0], wv[4 * k + 1], wv[4 * k + 2], wv[4 * k + 3]);
    } else {
        unsigned long long cur = ~0ULL;
        uint32_t c0 = 0, c1 = 0, c2 = 0, c3 = 0;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            if (j < ncol) {
                const unsigned long long gi = g0 + j;
                if ((gi >> 2) != cur) {
                    cur = gi >> 2;
                    uint32_t c[4] = {static_cast<uint32_t>(cur), static_cast<uint32_t>(cur >> 32), mf.step_lo,
                                     mf.step_hi};
                    philox4x32_10(c, mf.seed_lo, mf.seed_hi);
                    c0 = c[0];
                    c1 = c[1];
                    c2 = c[2];
                    c3 = c[3];
                }
                const uint32_t e = static_cast<uint32_t>(gi & 3);
                const uint32_t u = e == 0 ? c0 : (e == 1 ? c1 : (e == 2 ? c2 : c3));
                wp[j] = upd(wp[j], v[j], u);
            }
        }
    }
}

// Waits for an mbarrier phase during teardown, ignoring the error word.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer() - t0 > kWaitLimitNs) break;
    }
}

template <int BN, int CG, int NP>
__global__ void __launch_bounds__(kThreads, 1) gemm_tc_kernel(const __grid_constant__ GemmProgram P) {
    static_assert(NP == 1 || CG == 2, "pairs per cluster needs paired MMAs");
    constexpr int CL = CG * NP;  // CTAs per cluster
    constexpr int STAGES = Cfg<BN, CG>::STAGES;
    constexpr int NCH = BN / 32;
    constexpr int BNH = BN / CG;  // rows of B this CTA stages
    constexpr uint32_t A_BYTES = BM * BK * 2;
    constexpr uint32_t B_BYTES = BNH * BK * 2;
    constexpr uint32_t TMEM_COLS = 2 * BN;
    constexpr uint32_t IDESC = idesc_f16_f32(BM * CG, BN);  // K-major; MN-major bits added per k-block
    constexpr int TM = BM * CG;  // tile M edge; the storage tile of lower-only matrices

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = sA + STAGES * A_BYTES;
    uint8_t* sEpi = sB + STAGES * B_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sEpi + kEpiWarps * SBUF);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5);

    const uint32_t full0 = smem_u32(bars);
    const uint32_t empty0 = smem_u32(bars + STAGES);
    const uint32_t accf0 = smem_u32(bars + 2 * STAGES);
    const uint32_t acce0 = smem_u32(bars + 2 * STAGES + 2);
    const uint32_t drain_bar = smem_u32(bars + 2 * STAGES + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    int* err = P.err;
    const uint32_t crank = (CL > 1) ? cluster_ctarank() : 0;  // rank in the cluster
    const uint32_t rank = crank & (CG - 1);                  // rank in the pair: 0 = leader
    const uint32_t lead = crank & ~uint32_t(CG - 1);         // cluster rank of the pair leader
    const int pair = static_cast<int>(crank >> 1) & (NP - 1);  // pair within the cluster
    const int unit = blockIdx.x / CL;                        // this cluster's tile walker
    const int units = gridDim.x / CL;
    const int nwalk = P.total_tiles / NP;                    // super-tiles: NP consecutive tiles

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            // With two pairs per cluster every stage is released by both
            // pairs' MMAs (a shared A half lands in both pairs).
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, NP);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf0 + 8 * b, 1);
            mbar_init(acce0 + 8 * b, kEpiWarps * CG);
        }
        mbar_init(drain_bar, 1);
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        for (int m = 0; m < P.nmaps; ++m) prefetch_tmap(&P.maps[m]);
    }
    // Counter value at which every tile of the phases before phase s is done.
    auto dep_target = [&](int s) { return P.phase[s].wait_tiles * (kEpiWarps * CG); };
    if (warp == 1) {
        tmem_alloc<CG>(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish<CG>();
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (CL > 1) cluster_sync();  // all CTAs' barriers exist before any remote use
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // Everything above overlaps the previous kernel's tail; operands written
    // by it are read only after this point.
    grid_dependency_wait();
    grid_launch_dependents();

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            int issued = 0;
            bool ok = true;
            for (int w = unit; w < nwalk && ok; w += units) {
                const TileInfo t = decode_tile<BN, CG>(P, w * NP + pair);
                const GemmProblem& pr = P.prob[t.p];
                const CUtensorMap* mapA = &P.maps[pr.mA];
                const CUtensorMap* mapB = &P.maps[pr.mB];
                const bool a_mn0 = pr.flags & kFlagAmn;
                const bool b_mn0 = pr.flags & kFlagBmn;
                const bool a_sym = pr.flags & kFlagAsym;
                const bool b_sym = pr.flags & kFlagBsym;
                const CUtensorMap* mapAt = a_sym ? &P.maps[pr.mAt] : mapA;
                const CUtensorMap* mapBt = b_sym ? &P.maps[pr.mBt] : mapB;
                const int ti = t.m0 / TM, tj = t.n0 / TM;
                const bool share = (NP == 2) && (pr.flags & kFlagShareA);
                const int kblocks = (pr.K + BK - 1) / BK;
                if (P.counters && P.phase[t.s].wait_tiles > 0) {
                    // The operands of this phase are outputs of earlier phases on
                    // the same matrix, stored by other CTAs.
                    if (!wait_counter(P.counters + t.g, dep_target(t.s), err)) break;
                    fence_proxy_async_global();
                }
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!mbar_wait(empty0 + 8 * stage, phase ^ 1, err)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = full0 + 8 * stage;
                    const int arow = t.m0 + BM * static_cast<int>(rank);
                    const int brow = t.n0 + BNH * static_cast<int>(rank);
                    // Lower-only operands: a k-block right of the diagonal tile is
                    // read transposed from the tile below it.
                    const int kt = (kb * BK) / TM;
                    const bool a_t = a_sym && kt > ti;
                    const bool b_t = b_sym && kt > tj;
                    const bool a_mn = a_mn0 || a_t;
                    const bool b_mn = b_mn0 || b_t;
                    const CUtensorMap* mA_k = a_t ? mapAt : mapA;
                    const CUtensorMap* mB_k = b_t ? mapBt : mapB;
                    if constexpr (CG == 1) {
                        mbar_arrive_expect_tx(fb, A_BYTES + B_BYTES);
                        load_operand(0, smem_u32(sA + stage * A_BYTES), mA_k, fb, a_mn, arow, BM, kb, t.g, 0);
                        load_operand(0, smem_u32(sB + stage * B_BYTES), mB_k, fb, b_mn, brow, BNH, kb, t.g, 0);
                    } else {
                        // All halves complete on the pair leader's barrier. A
                        // shared A half is loaded once by the first pair and
                        // multicast to the same-rank CTA of both pairs.
                        if (rank == 0) mbar_arrive_expect_tx(fb, 2 * (A_BYTES + B_BYTES));
                        const uint32_t lead_fb = map_to_rank(fb, lead);
                        if (!share) {
                            load_operand(1, smem_u32(sA + stage * A_BYTES), mA_k, lead_fb, a_mn, arow, BM, kb, t.g, 0);
                        } else if (pair == 0) {
                            const uint16_t mask = static_cast<uint16_t>((1u << rank) | (1u << (2 + rank)));
                            load_operand(2, smem_u32(sA + stage * A_BYTES), mA_k, lead_fb, a_mn, arow, BM, kb, t.g,
                                         mask);
                        }
                        load_operand(1, smem_u32(sB + stage * B_BYTES), mB_k, lead_fb, b_mn, brow, BNH, kb, t.g, 0);
                    }
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            // The last min(issued, STAGES) loads may still be in flight; wait
            // for each (on the barrier that counts them) before exiting.
            if (CG == 1 || rank == 0) {
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
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------- MMA issuer (pair leader)
        if (lane == 0 && rank == 0) {
            uint32_t stage = 0, phase = 0;
            int iter = 0;
            bool ok = true;
            constexpr uint16_t kStageMask = (NP == 2) ? 0xF : 0x3;  // both pairs' CTAs
            const uint16_t pair_mask = static_cast<uint16_t>(0x3u << (2 * pair));
            for (int w = unit; w < nwalk && ok; w += units, ++iter) {
                const TileInfo t = decode_tile<BN, CG>(P, w * NP + pair);
                const GemmProblem& pr = P.prob[t.p];
                const int kblocks = (pr.K + BK - 1) / BK;
                const int buf = iter & 1;
                const bool a_mn0 = pr.flags & kFlagAmn;
                const bool b_mn0 = pr.flags & kFlagBmn;
                const bool a_sym = pr.flags & kFlagAsym;
                const bool b_sym = pr.flags & kFlagBsym;
                const int ti = t.m0 / TM, tj = t.n0 / TM;
                if (!mbar_wait(acce0 + 8 * buf, ((iter >> 1) & 1) ^ 1, err)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + buf * BN;
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!mbar_wait(full0 + 8 * stage, phase, err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // The operand layouts the producer chose for this k-block.
                    const int kt = (kb * BK) / TM;
                    const uint32_t a_mn = (a_mn0 || (a_sym && kt > ti)) ? 1u : 0u;
                    const uint32_t b_mn = (b_mn0 || (b_sym && kt > tj)) ? 1u : 0u;
                    const uint32_t idesc = IDESC | (a_mn << 15) | (b_mn << 16);
                    // Per 16-wide k step: 32 bytes along a K-major row, or two
                    // 8-row groups (2048 bytes) of an MN-major tile.
                    const uint32_t a_step = a_mn ? (2048 >> 4) : (32 >> 4);
                    const uint32_t b_step = b_mn ? (2048 >> 4) : (32 >> 4);
                    const uint32_t sa = smem_u32(sA + stage * A_BYTES);
                    const uint32_t sb = smem_u32(sB + stage * B_BYTES);
                    const uint64_t adesc = a_mn ? sw128_mnmajor_desc(sa, kMnBlockBytes) : sw128_kmajor_desc(sa);
                    const uint64_t bdesc = b_mn ? sw128_mnmajor_desc(sb, kMnBlockBytes) : sw128_kmajor_desc(sb);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        tc_mma_f16<CG>(d_tmem, adesc + a_step * kk, bdesc + b_step * kk, idesc,
                                       (kb | kk) != 0 ? 1u : 0u);
                    }
                    if constexpr (CG == 1)
                        tc_commit<1>(empty0 + 8 * stage);
                    else
                        tc_commit_pair(empty0 + 8 * stage, kStageMask);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                if constexpr (CG == 1)
                    tc_commit<1>(accf0 + 8 * buf);
                else
                    tc_commit_pair(accf0 + 8 * buf, pair_mask);
            }
            // All MMAs issued by this thread must finish before TMEM is freed.
            tc_commit<CG>(drain_bar);
            drain_wait(drain_bar, 0);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------- epilogue
        const int q = warp & 3;                 // TMEM lane quarter this warp may access
        const int ew = warp - 2;                // epilogue warp 0..7
        constexpr int CPW = NCH / 2;            // chunks per warp: two warps share a quarter
        const int cbeg = (ew >> 2) * CPW;       // this warp's first chunk
        const uint32_t stg = smem_u32(sEpi + ew * SBUF);
        const uint32_t acce_lead = (CG == 2) ? map_to_rank(acce0, lead) : acce0;
        int iter = 0;
        for (int w = unit; w < nwalk; w += units, ++iter) {
            const TileInfo t = decode_tile<BN, CG>(P, w * NP + pair);
            const GemmProblem& pr = P.prob[t.p];
            const int buf = iter & 1;
            const int flags = pr.flags;
            const bool sym = flags & kFlagSym;
            const bool hasC = flags & kFlagC;
            const bool f32 = flags & kFlagOutF32;
            const int r0 = t.m0 + BM * static_cast<int>(rank) + q * 32;
            const int grow = r0 + lane;
            const bool rows_live = r0 < pr.M;
            const int sr = r0 >> 5;
            auto active = [&](int c) {
                const int c0 = t.n0 + 32 * c;
                return rows_live && c0 < pr.N && !(sym && (c0 >> 5) > sr);
            };
            const int cend = cbeg + CPW;
            int c = cbeg;
            while (c < cend && !active(c)) ++c;
            if (hasC && P.counters && P.phase[t.s].wait_tiles > 0) {
                // C is an earlier phase's output: acquire it like the producer.
                if (!wait_counter(P.counters + t.g, dep_target(t.s), err)) break;
            }
            uint4 cb[4];
            if (hasC && c < cend) load_c(pr, t.g, grow, t.n0 + 32 * c, cb);

            if (!mbar_wait(accf0 + 8 * buf, (iter >> 1) & 1, err)) break;
            tc_fence_after();

#pragma unroll 1
            while (c < cend) {
                const int c0 = t.n0 + 32 * c;
                uint32_t acc[32];
                tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * BN + c * 32, acc);
                int cn = c + 1;
                while (cn < cend && !active(cn)) ++cn;
                uint4 cbn[4];
                if (hasC && cn < cend) load_c(pr, t.g, grow, t.n0 + 32 * cn, cbn);
                tmem_ld_wait();

                float v[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = pr.alpha * __uint_as_float(acc[j]);
                if (hasC) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint32_t w[4] = {cb[k].x, cb[k].y, cb[k].z, cb[k].w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
                            v[8 * k + 2 * e] = fmaf(pr.beta, f.x, v[8 * k + 2 * e]);
                            v[8 * k + 2 * e + 1] = fmaf(pr.beta, f.y, v[8 * k + 2 * e + 1]);
                        }
                    }
                }
                if (flags & kFlagMuon) {
                    muon_update_row(pr, t.g, grow, c0, v);
#pragma unroll
                    for (int k = 0; k < 4; ++k) cb[k] = cbn[k];
                    c = cn;
                    continue;
                }
                const bool diag_block = sym && ((c0 >> 5) == sr);
                // Lower-only outputs mirror only inside diagonal tiles.
                const bool mirror = (flags & kFlagDt) && !diag_block && (!(flags & kFlagLower) || t.m0 == t.n0);

                // Stage, transpose (mirror or diagonal fix-up) and store one
                // 32 x 32 block; the buffer is free once the previous stores
                // have read it.
                auto emit = [&](const float (&val)[32], int map_d, int map_dt) {
                    if (lane == 0) bulk_wait_read<0>();
                    __syncwarp();
                    if (f32) {
                        stage_row_f32(stg + kOffD, lane, val);
                    } else {
                        stage_row_f16(stg + kOffD, lane, val);
                        if (mirror || diag_block) {
                            __syncwarp();
                            transpose_block(stg + kOffD, stg + kOffDt, lane);
                            if (diag_block) {
                                __syncwarp();
                                merge_upper(stg + kOffD, stg + kOffDt, lane);
                            }
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_3d(&P.maps[map_d], stg + kOffD, c0, r0, t.g);
                        if (mirror) tma_store_3d(&P.maps[map_dt], stg + kOffDt, r0, c0, t.g);
                        bulk_commit();
                    }
                };
                emit(v, pr.mD, pr.mDt);
                if (flags & kFlagD2) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = pr.delta * v[j] + ((grow == c0 + j) ? pr.gamma : 0.0f);
                    emit(v, pr.mD2, pr.mD2t);
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) cb[k] = cbn[k];
                c = cn;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if constexpr (CG == 1)
                    mbar_arrive(acce0 + 8 * buf);
                else
                    mbar_arrive_cluster(acce_lead + 8 * buf);
                if (P.counters) {
                    // Publish this warp's part of the tile: stores complete,
                    // then a release on the matrix's counter.
                    bulk_wait_all();
                    fence_proxy_async_global();
                    red_release_add(P.counters + t.g, 1);
                }
            }
        }
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    // The leader's MMAs read the peer's shared memory, multicasts write into
    // other CTAs and epilogues arrive on the leader's barriers: no CTA of the
    // cluster leaves before all are done.
    if constexpr (CL > 1) cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<CG>(tmem_base, TMEM_COLS);
    }
}

// Clusters of CL CTAs that can be resident at once with this kernel's
// shared memory; the grid never exceeds it, so every cluster of a program
// runs concurrently (tiles wait on tiles of other clusters).
template <int BN, int CG, int NP>
int max_clusters(int num_sms) {
    static int cached = -1;
    if (cached < 0) {
        constexpr int CL = CG * NP;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(CL * (num_sms / CL));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = smem_bytes<BN, CG>();
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = CL;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, gemm_tc_kernel<BN, CG, NP>, &cfg) != cudaSuccess || n <= 0) {
            cudaGetLastError();
            n = num_sms / CL;
        }
        cached = n;
    }
    return cached < num_sms / (CG * NP) ? cached : num_sms / (CG * NP);
}

template <int BN, int CG, int NP>
int launch_impl(const GemmProgram& prog, int num_sms, cudaStream_t stream) {
    static bool configured = false;
    constexpr int bytes = smem_bytes<BN, CG>();
    constexpr int CL = CG * NP;
    if (!configured) {
        cudaError_t e =
            cudaFuncSetAttribute(gemm_tc_kernel<BN, CG, NP>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    if (prog.total_tiles <= 0) return cudaSuccess;
    if (prog.total_tiles % NP != 0) return cudaErrorInvalidValue;
    const int walks = prog.total_tiles / NP;
    const int clusters = max_clusters<BN, CG, NP>(num_sms);
    const int grid = CL * (walks < clusters ? walks : clusters);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = CL;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<BN, CG, NP>, prog);
}

}  // namespace

int gemm_smem_bytes(int bn, int cg) {
    if (cg == 2) return smem_bytes<256, 2>();
    return bn == 256 ? smem_bytes<256, 1>() : smem_bytes<128, 1>();
}

int gemm_tiles_per_matrix(int M, int N, int bn, int cg, bool sym, int np, bool share, int* walk_n) {
    const int tmh = BM * cg;
    const int tm = (M + tmh - 1) / tmh;
    const int tn = (N + bn - 1) / bn;
    const int wn = share ? tn + (tn & 1) : tn;
    if (walk_n) *walk_n = wn;
    int total = 0;
    if (!sym) {
        total = tm * wn;
    } else {
        for (int i = 0; i < tm; ++i) total += sym_row_tiles(i, tmh, bn, tn, share);
    }
    if (np == 2) total += total & 1;
    return total;
}

int gemm_signals_per_tile(int cg) { return kEpiWarps * cg; }

int launch_gemm_program(const GemmProgram& prog, int bn, int cg, int np, int num_sms, cudaStream_t stream) {
    if (cg == 2) {
        if (np == 2) return launch_impl<256, 2, 2>(prog, num_sms, stream);
        return launch_impl<256, 2, 1>(prog, num_sms, stream);
    }
    if (bn == 256) return launch_impl<256, 1, 1>(prog, num_sms, stream);
    return launch_impl<128, 1, 1>(prog, num_sms, stream);
}

}  // namespace gns
