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
//   warps 2-9   epilogue: tcgen05.ld of 32 x 32 sub-blocks, the fp32 epilogue
//               alpha * acc + beta * C (+ the second output delta * v + gamma I),
//               then the sub-block and, when asked, its transpose (the mirror
//               write of the symmetric product, Dion3 §5 "Epilogue: Writing to
//               the Transposed Tile") are staged in shared memory and written
//               to global memory by the warp's own coalesced stores (8 rows of
//               64 bytes per instruction), so the epilogue never waits on the
//               TMA unit, which the operand loads keep busy.
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
// stmatrix; all staging uses 64-byte rows with the 64-byte swizzle (fp32 blocks
// are staged as two 16-column halves).
#include <cstdio>

#include <cuda_bf16.h>

#include "gemm.cuh"
#include "philox.cuh"
#include "ptx.cuh"

namespace gns {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;
static_assert(sizeof(GemmProgram) <= 32764, "kernel parameter block too large");
constexpr int kSchedWarp = 2 + kEpiWarps;     // the scheduler warp follows the epilogue warps
constexpr int kThreads = 32 * (kSchedWarp + 1);  // producer, MMA, epilogue, scheduler
constexpr int kRing = 8;                         // ring slots of published tile records (claims are paced by the lookahead)

// Per-warp epilogue shared memory: three 2 KB slots of 32 rows x 64 bytes
// (64-byte swizzle). Slots 0 and 1 receive, by TMA, the C addend of the
// warp's next two 32 x 32 blocks; once a block's C has been read, its slot
// stages that block's output for the coalesced stores. Slot 2 holds the
// transposed block of a mirrored or diagonal sub-block.
constexpr int kSlot = 2048;
constexpr int SBUF = 3 * kSlot;

// Kernel variants: <BN, CG>. CG = 1: one CTA computes a 128 x BN tile.
// CG = 2: a cluster of two CTAs computes a 256 x BN tile with paired MMAs
// (tcgen05.mma.cta_group::2, M = 256); each CTA stages its 128 rows of A and
// BN / 2 rows of B, so a stage costs half the shared memory per MMA.
template <int BN, int CG>
struct Cfg;
template <>
struct Cfg<128, 1> {
    static constexpr int STAGES = 5;
};
template <>
struct Cfg<256, 1> {
    static constexpr int STAGES = 3;
};
template <>
struct Cfg<256, 2> {
    static constexpr int STAGES = 5;
};

// Tables copied from the kernel parameters into shared memory at start: the
// item-list builder decodes every item through them, and the roles read a
// problem's fields per tile (parameter-space loads with a tile-dependent
// index are slow under load).
struct CtlPhase {
    int item_begin, tiles_per_matrix, prob_begin, wait;
};
struct CtlProb {
    int tiles_per_matrix, tiles_n, flags, K, tiles_m;
    int mA, mB, mAt, mBt, mC;
};
constexpr int kCtlBytes = kMaxPhases * static_cast<int>(sizeof(CtlPhase)) + kMaxProblems * static_cast<int>(sizeof(CtlProb));
__host__ __device__ constexpr int kNumBars(int stages) { return 2 * stages + 5 + 2 * kEpiWarps + 3 * kRing; }

template <int BN, int CG>
constexpr int smem_bytes() {
    return 1024 + Cfg<BN, CG>::STAGES * (BM * BK * 2 + (BN / CG) * BK * 2) + kEpiWarps * SBUF +
           kNumBars(Cfg<BN, CG>::STAGES) * 8 + 16 + kCtlBytes + 16 + kRing * static_cast<int>(sizeof(ProgItem));
}
static_assert(smem_bytes<256, 2>() <= 232448, "shared memory budget");
static_assert(smem_bytes<128, 1>() <= 232448, "shared memory budget");
static_assert(smem_bytes<256, 1>() <= 232448, "shared memory budget");

// Column blocks a symmetric row block of height tm touches: j * bn <= tm i + tm - 1.
__host__ __device__ __forceinline__ int sym_row_tiles(int i, int tm, int bn, int tiles_n) {
    const int c = (tm * i + tm - 1) / bn + 1;
    return c < tiles_n ? c : tiles_n;
}

__host__ __device__ __forceinline__ int item_prob(const ProgItem& it) { return it.meta & 255; }
__host__ __device__ __forceinline__ int item_matrix(const ProgItem& it) { return static_cast<int>(static_cast<unsigned>(it.meta) >> 8); }
__host__ __device__ __forceinline__ ProgItem make_item(int p, int g, int wait, int m0, int n0) {
    return ProgItem{p | (g << 8), wait, m0, n0};
}

// Tile t (0-based, in walk order) of matrix g in phase `s`: the problem it
// belongs to and its origin. Symmetric products list the lower-triangle tiles
// row by row; other products walk row by row, or column by column with
// kFlagColWalk (the tiles that share a B column block run together).
template <int BN, int CG>
__host__ __device__ ProgItem decode_tile(const CtlPhase& ph, const CtlProb* cpb, int g, int t) {
    constexpr int TM = BM * CG;
    int p = ph.prob_begin;
    while (t >= cpb[p].tiles_per_matrix) {
        t -= cpb[p].tiles_per_matrix;
        ++p;
    }
    const int flags = cpb[p].flags;
    int i, j;
    if ((flags & kFlagSym) && TM == BN) {
        // Square tiles: row block i holds i + 1 tiles, i (i + 1) / 2 before it.
        i = static_cast<int>((sqrtf(8.0f * static_cast<float>(t) + 1.0f) - 1.0f) * 0.5f);
        while (i * (i + 1) / 2 > t) --i;
        while ((i + 1) * (i + 2) / 2 <= t) ++i;
        j = t - i * (i + 1) / 2;
    } else if (flags & kFlagSym) {
        int acc = 0;
        i = 0;
        while (true) {
            const int cnt = sym_row_tiles(i, TM, BN, cpb[p].tiles_n);
            if (t < acc + cnt) break;
            acc += cnt;
            ++i;
        }
        j = t - acc;
    } else if (flags & kFlagColWalk) {
        j = t / cpb[p].tiles_m;
        i = t - j * cpb[p].tiles_m;
    } else {
        i = t / cpb[p].tiles_n;
        j = t - i * cpb[p].tiles_n;
    }
    return make_item(p, g, ph.wait, i * TM, j * BN);
}

// Tile w of the program's list: phase by phase, matrix by matrix.
template <int BN, int CG>
__host__ __device__ ProgItem decode_item(const CtlPhase* cph, const CtlProb* cpb, int nphase, int w) {
    int s = 0;
    while (s + 1 < nphase && w >= cph[s + 1].item_begin) ++s;
    const int local = w - cph[s].item_begin;
    const int g = local / cph[s].tiles_per_matrix;
    return decode_tile<BN, CG>(cph[s], cpb, g, local - g * cph[s].tiles_per_matrix);
}

// An MN-major operand tile is staged as 64-wide M/N blocks of 64 K rows
// (one TMA box each), 8 KB apart.
constexpr uint32_t kMnBlockBytes = 64 * BK * 2;

// One k-block of one operand into shared memory: a K-major tile is one box
// {64 (K), rows}; an MN-major tile is rows / 64 boxes {64 (M or N), 64 (K)}.
// mode 0: this CTA's own barrier; 1: the pair leader's barrier (bar is a
// cluster address).
__device__ __forceinline__ void load_operand(int mode, uint32_t dst, const CUtensorMap* map, uint32_t bar, bool mn,
                                             int row0, int rows, int kb, int g) {
    const int boxes = mn ? rows / 64 : 1;
    for (int h = 0; h < boxes; ++h) {
        const uint32_t d = dst + h * kMnBlockBytes;
        const int c0 = mn ? row0 + 64 * h : kb * BK;
        const int c1 = mn ? kb * BK : row0;
        if (mode == 0)
            tma_load_3d(d, map, bar, c0, c1, g);
        else
            tma_load_3d_pair(d, map, bar, c0, c1, g);
    }
}

// Address of element (row, col) of a 32 x 32 fp16 block staged with the
// 64-byte swizzle (16-byte chunk index XOR (row / 2) mod 4).
__device__ __forceinline__ uint32_t sw64_addr(uint32_t base, int row, int col) {
    return base + row * 64 + ((((col >> 3) ^ (row >> 1)) & 3) << 4) + (col & 7) * 2;
}

// Address of 16-byte piece k of row r in a 64B-swizzled block of 64-byte rows.
__device__ __forceinline__ uint32_t sw64_piece(uint32_t base, int r, int k) {
    return base + r * 64 + (((k ^ (r >> 1)) & 3) << 4);
}

// Row `lane` (32 values) of a 64B-swizzled fp16 block.
__device__ __forceinline__ void stage_row_f16(uint32_t base, int lane, const float (&v)[32]) {
#pragma unroll
    for (int k = 0; k < 4; ++k)
        st_shared_v4(sw64_piece(base, lane, k), pack_half2(v[8 * k + 0], v[8 * k + 1]),
                     pack_half2(v[8 * k + 2], v[8 * k + 3]), pack_half2(v[8 * k + 4], v[8 * k + 5]),
                     pack_half2(v[8 * k + 6], v[8 * k + 7]));
}

// Columns 16 H .. 16 H + 15 of row `lane` as one 64-byte fp32 row of a
// 64B-swizzled block.
template <int H>
__device__ __forceinline__ void stage_row_f32_half(uint32_t base, int lane, const float (&v)[32]) {
#pragma unroll
    for (int k = 0; k < 4; ++k)
        st_shared_v4(sw64_piece(base, lane, k), __float_as_uint(v[16 * H + 4 * k + 0]),
                     __float_as_uint(v[16 * H + 4 * k + 1]), __float_as_uint(v[16 * H + 4 * k + 2]),
                     __float_as_uint(v[16 * H + 4 * k + 3]));
}

// dst = src^T for a 32 x 32 fp16 block (both 64B-swizzled): 8 x 8 block (R, i)
// of src, loaded transposed, is stored as block (i, R) of dst.
__device__ __forceinline__ void transpose_block(uint32_t src, uint32_t dst, int lane) {
    uint32_t a[4][4];  // all loads first, then all stores (one round trip, not four)
#pragma unroll
    for (int R = 0; R < 4; ++R)
        ldmatrix_x4_trans(sw64_addr(src, 8 * R + (lane & 7), 8 * (lane >> 3)), a[R][0], a[R][1], a[R][2], a[R][3]);
#pragma unroll
    for (int R = 0; R < 4; ++R) stmatrix_x4(sw64_addr(dst, lane, 8 * R), a[R][0], a[R][1], a[R][2], a[R][3]);
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

// Stores one 16-byte piece v of a staged row at p, clipped to the `left`
// elements still inside the matrix (the ragged right edge; out of line, it is
// rare and would otherwise bloat the epilogue's hot code).
template <int ES>
static __device__ __noinline__ void store_piece_clipped(uint8_t* p, uint4 v, int left) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    if constexpr (ES == 2) {
#pragma unroll
        for (int e = 0; e < 8; ++e)
            if (e < left) reinterpret_cast<uint16_t*>(p)[e] = static_cast<uint16_t>(w[e >> 1] >> (16 * (e & 1)));
    } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (e < left) reinterpret_cast<uint32_t*>(p)[e] = w[e];
    }
}

// Writes a staged block of 32 rows x 64 bytes (64B-swizzled, elements of ES
// bytes) to rows r0 .. r0 + 31 and the 64 / ES columns from c0 of matrix g
// of `o`, clipped to rows x cols. Instruction j stores rows 8 j .. 8 j + 7,
// four lanes per 64-byte row segment.
template <int ES>
__device__ __forceinline__ void store_rows64(uint32_t stg, const OutView& o, int g, int r0, int c0, int rows, int cols,
                                             int lane) {
    constexpr int EPP = 16 / ES;  // elements per 16-byte piece
    const int k = lane & 3;
    const int gc = c0 + EPP * k;
    // All four shared-memory reads first: under load each round trip costs
    // hundreds of cycles, so they are issued back to back, not one per store.
    uint4 vv[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) vv[j] = ld_shared_v4(sw64_piece(stg, 8 * j + (lane >> 2), k));
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int r = 8 * j + (lane >> 2);
        const uint4 v = vv[j];
        const int gr = r0 + r;
        if (gr >= rows || gc >= cols) continue;
        uint8_t* p = static_cast<uint8_t*>(o.p) +
                     (static_cast<long long>(g) * o.stride + static_cast<long long>(gr) * o.ld + gc) * ES;
        if (gc + EPP <= cols)
            *reinterpret_cast<uint4*>(p) = v;
        else
            store_piece_clipped<ES>(p, v, cols - gc);
    }
}

// 32 bytes to global memory in one store (sm_100 and later).
__device__ __forceinline__ void st_global_v8(void* p, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t a4,
                                             uint32_t a5, uint32_t a6, uint32_t a7) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(a0), "r"(a1), "r"(a2),
                 "r"(a3), "r"(a4), "r"(a5), "r"(a6), "r"(a7)
                 : "memory");
}

// An output whose rows (and matrices) start on 32-byte boundaries takes the
// direct path below for full-width blocks.
__device__ __forceinline__ bool out_direct(const OutView& o, int es) {
    return (reinterpret_cast<uintptr_t>(o.p) & 31) == 0 && ((o.ld * es) & 31) == 0 && ((o.stride * es) & 31) == 0;
}

// Row `row` of a 32 x 32 block, columns c0 .. c0 + 31, written straight from
// the lane's registers (no shared-memory staging): 32 fp16 values (64 bytes)
// as two 32-byte stores, or 32 fp32 values as four.
__device__ __forceinline__ void direct_row(const OutView& o, int g, int row, int c0, const float (&v)[32], bool f32) {
    const long long idx = static_cast<long long>(g) * o.stride + static_cast<long long>(row) * o.ld + c0;
    if (f32) {
        float* p = static_cast<float*>(o.p) + idx;
#pragma unroll
        for (int k = 0; k < 4; ++k)
            st_global_v8(p + 8 * k, __float_as_uint(v[8 * k + 0]), __float_as_uint(v[8 * k + 1]),
                         __float_as_uint(v[8 * k + 2]), __float_as_uint(v[8 * k + 3]), __float_as_uint(v[8 * k + 4]),
                         __float_as_uint(v[8 * k + 5]), __float_as_uint(v[8 * k + 6]), __float_as_uint(v[8 * k + 7]));
    } else {
        __half* p = static_cast<__half*>(o.p) + idx;
#pragma unroll
        for (int k = 0; k < 2; ++k)
            st_global_v8(p + 16 * k, pack_half2(v[16 * k + 0], v[16 * k + 1]), pack_half2(v[16 * k + 2], v[16 * k + 3]),
                         pack_half2(v[16 * k + 4], v[16 * k + 5]), pack_half2(v[16 * k + 6], v[16 * k + 7]),
                         pack_half2(v[16 * k + 8], v[16 * k + 9]), pack_half2(v[16 * k + 10], v[16 * k + 11]),
                         pack_half2(v[16 * k + 12], v[16 * k + 13]), pack_half2(v[16 * k + 14], v[16 * k + 15]));
    }
}

// The rarer epilogue paths.
// A 32 x 32 fp32 block, staged and stored as two 16-column halves (inline:
// the values are a register array, which a call would move to local memory).
__device__ __forceinline__ void emit_f32(uint32_t slot, const float (&val)[32], const OutView& od, int g, int r0,
                                             int c0, int M, int N, int lane) {
    stage_row_f32_half<0>(slot, lane, val);
    __syncwarp();
    store_rows64<4>(slot, od, g, r0, c0, M, N, lane);
    __syncwarp();
    stage_row_f32_half<1>(slot, lane, val);
    __syncwarp();
    store_rows64<4>(slot, od, g, r0, c0 + 16, M, N, lane);
}

// The transposed copy of a staged fp16 block in sT; for a diagonal block the
// staged block's upper half is then replaced from it.
static __device__ __noinline__ void stage_transpose(uint32_t slot, uint32_t sT, bool diag, int lane) {
    __syncwarp();
    transpose_block(slot, sT, lane);
    if (diag) {
        __syncwarp();
        merge_upper(slot, sT, lane);
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
    if (ncol == 32 && (g0 & 7) == 0 && (reinterpret_cast<uintptr_t>(wp) & 15) == 0) {
        uint32_t wv[16];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint4 x = reinterpret_cast<const uint4*>(wp)[k];
            wv[4 * k + 0] = x.x;
            wv[4 * k + 1] = x.y;
            wv[4 * k + 2] = x.z;
            wv[4 * k + 3] = x.w;
        }
        // Four blocks of eight global indices, one Philox output each.
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const unsigned long long blk = (g0 >> 3) + b;
            uint32_t c[4] = {static_cast<uint32_t>(blk), static_cast<uint32_t>(blk >> 32), mf.step_lo, mf.step_hi};
            philox4x32_10(c, mf.seed_lo, mf.seed_hi);
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const uint32_t pair = wv[4 * b + h];
                const uint32_t lo = upd(static_cast<uint16_t>(pair & 0xFFFFu), v[8 * b + 2 * h], sr_draw(c, 2 * h));
                const uint32_t hi = upd(static_cast<uint16_t>(pair >> 16), v[8 * b + 2 * h + 1], sr_draw(c, 2 * h + 1));
                wv[4 * b + h] = lo | (hi << 16);
            }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k)
            reinterpret_cast<uint4*>(wp)[k] = make_uint4(wv[4 * k + 0], wv[4 * k + 1], wv[4 * k + 2], wv[4 * k + 3]);
    } else {
        unsigned long long cur = ~0ULL;
        uint32_t c[4] = {0, 0, 0, 0};
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            if (j < ncol) {
                const unsigned long long gi = g0 + j;
                if ((gi >> 3) != cur) {
                    cur = gi >> 3;
                    c[0] = static_cast<uint32_t>(cur);
                    c[1] = static_cast<uint32_t>(cur >> 32);
                    c[2] = mf.step_lo;
                    c[3] = mf.step_hi;
                    philox4x32_10(c, mf.seed_lo, mf.seed_hi);
                }
                const int e = static_cast<int>(gi & 7);
                const uint32_t u = (e >> 1) == 0 ? c[0] : ((e >> 1) == 1 ? c[1] : ((e >> 1) == 2 ? c[2] : c[3]));
                wp[j] = upd(wp[j], v[j], (u >> (16 * (e & 1))) & 0xFFFFu);
            }
        }
    }
}

// Waits for an mbarrier phase during teardown, ignoring the abort mark.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer() - t0 > limit_ns) break;
    }
}

template <int BN, int CG>
__global__ void __launch_bounds__(kThreads, 1) gemm_tc_kernel(const __grid_constant__ GemmProgram P) {
    constexpr int CL = CG;  // CTAs per cluster: one pair, or one CTA
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
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars(STAGES));
    const uint32_t pub0 = smem_u32(tmem_slot + 2);  // per-buffer counts of finished epilogue warps
    CtlPhase* cph = reinterpret_cast<CtlPhase*>(tmem_slot + 4);
    CtlProb* cpb = reinterpret_cast<CtlProb*>(cph + kMaxPhases);
    // kRing tile records, 16-byte aligned (vector accesses, also from the peer CTA).
    ProgItem* ring =
        reinterpret_cast<ProgItem*>((reinterpret_cast<uintptr_t>(cpb + kMaxProblems) + 15) & ~uintptr_t(15));

    const uint32_t full0 = smem_u32(bars);
    const uint32_t empty0 = smem_u32(bars + STAGES);
    const uint32_t accf0 = smem_u32(bars + 2 * STAGES);
    const uint32_t acce0 = smem_u32(bars + 2 * STAGES + 2);
    const uint32_t drain_bar = smem_u32(bars + 2 * STAGES + 4);
    const uint32_t cbar0 = smem_u32(bars + 2 * STAGES + 5);  // two C-slot barriers per epilogue warp
    // Tile ring: slot j's "record ready" barrier (in every CTA) and "free"
    // barrier (the pair leader's, counting every consumer of both CTAs).
    const uint32_t ringf0 = smem_u32(bars + 2 * STAGES + 5 + 2 * kEpiWarps);
    const uint32_t ringe0 = ringf0 + 8 * kRing;
    // Slot j's "taken by the producer" barrier (the pair leader's producer):
    // paces the claims (the program's lookahead).
    const uint32_t taken0 = ringe0 + 8 * kRing;
    constexpr int kRingConsumers = CG * (1 + kEpiWarps) + 1;  // producers, epilogue warps, MMA issuer

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const DevStatus& err = P.st;
    const uint32_t crank = (CL > 1) ? cluster_ctarank() : 0;  // rank in the cluster
    const uint32_t rank = crank & (CG - 1);                  // rank in the pair: 0 = leader
    const uint32_t lead = crank & ~uint32_t(CG - 1);         // cluster rank of the pair leader
    const int nphase = P.nphase;
    const uint32_t ring_u32 = smem_u32(ring);
    const uint32_t ringe_lead = (CG == 2) ? map_to_rank(ringe0, lead) : ringe0;
    // Reads the record of ring slot j once its "ready" phase is complete and
    // hands the slot back; returns false when the wait gave up.
    auto take = [&](int j, ProgItem& out) -> bool {
        const int slot = j % kRing;
        if (!mbar_wait_cluster(ringf0 + 8 * slot, (j / kRing) & 1, err)) return false;
        out = ring[slot];
        if constexpr (CG == 2)
            mbar_arrive_cluster(ringe_lead + 8 * slot);
        else
            mbar_arrive(ringe0 + 8 * slot);
        return true;
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf0 + 8 * b, 1);
            mbar_init(acce0 + 8 * b, kEpiWarps * CG);
        }
        mbar_init(drain_bar, 1);
        for (int b = 0; b < 2 * kEpiWarps; ++b) mbar_init(cbar0 + 8 * b, 1);
        for (int b = 0; b < kRing; ++b) {
            mbar_init(ringf0 + 8 * b, 1);
            mbar_init(ringe0 + 8 * b, kRingConsumers);
            mbar_init(taken0 + 8 * b, 1);
        }
        tmem_slot[2] = 0;
        tmem_slot[3] = 0;
        fence_mbar_init();
    }
    for (int i = threadIdx.x; i < nphase; i += blockDim.x) {
        const GemmPhaseDesc& ph = P.phase[i];
        cph[i] = CtlPhase{ph.item_begin, ph.tiles_per_matrix, ph.prob_begin, ph.wait};
    }
    for (int i = threadIdx.x; i < P.nprob; i += blockDim.x) {
        const GemmProblem& pr = P.prob[i];
        cpb[i] = CtlProb{pr.tiles_per_matrix, pr.tiles_n, pr.flags, pr.K, pr.tiles_m,
                         pr.mA, pr.mB, pr.mAt, pr.mBt, pr.mC};
    }
    if (warp == 0 && lane == 0) {
        for (int m = 0; m < P.nmaps; ++m) prefetch_tmap(&P.maps[m]);
    }
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
            for (int k = 0; ok; ++k) {
                ProgItem it;
                if (!take(k, it) || it.meta < 0) break;
                if (rank == 0) mbar_arrive(taken0 + 8 * (k % kRing));
                const int g = item_matrix(it);
                const CtlProb& pr = cpb[item_prob(it)];
                const CUtensorMap* mapA = &P.maps[pr.mA];
                const CUtensorMap* mapB = &P.maps[pr.mB];
                const bool a_mn0 = pr.flags & kFlagAmn;
                const bool b_mn0 = pr.flags & kFlagBmn;
                const bool a_sym = pr.flags & kFlagAsym;
                const bool b_sym = pr.flags & kFlagBsym;
                const CUtensorMap* mapAt = a_sym ? &P.maps[pr.mAt] : mapA;
                const CUtensorMap* mapBt = b_sym ? &P.maps[pr.mBt] : mapB;
                const int ti = it.m0 / TM, tj = it.n0 / TM;
                const int kblocks = (pr.K + BK - 1) / BK;
                // The operands of this tile are outputs of earlier tiles on the
                // same matrix, stored by other CTAs: the scheduler acquired
                // them before it published the tile (its release on the ring
                // orders that acquire before these loads).
                if (it.wait > 0) fence_proxy_async_global();
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!mbar_wait(empty0 + 8 * stage, phase ^ 1, err)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = full0 + 8 * stage;
                    const int arow = it.m0 + BM * static_cast<int>(rank);
                    const int brow = it.n0 + BNH * static_cast<int>(rank);
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
                        load_operand(0, smem_u32(sA + stage * A_BYTES), mA_k, fb, a_mn, arow, BM, kb, g);
                        load_operand(0, smem_u32(sB + stage * B_BYTES), mB_k, fb, b_mn, brow, BNH, kb, g);
                    } else {
                        // All halves complete on the pair leader's barrier.
                        if (rank == 0) mbar_arrive_expect_tx(fb, 2 * (A_BYTES + B_BYTES));
                        const uint32_t lead_fb = map_to_rank(fb, lead);
                        load_operand(1, smem_u32(sA + stage * A_BYTES), mA_k, lead_fb, a_mn, arow, BM, kb, g);
                        load_operand(1, smem_u32(sB + stage * B_BYTES), mB_k, lead_fb, b_mn, brow, BNH, kb, g);
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
                    drain_wait(full0 + 8 * stage, phase, err.limit_ns);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------- MMA issuer (pair leader)
        if (lane == 0 && rank == 0) {
            uint32_t stage = 0, phase = 0;
            bool ok = true;
            constexpr uint16_t kPairMask = 0x3;  // both CTAs of the pair
            // Stage-0 descriptors of both operand layouts; a stage adds its
            // byte offset / 16 to the start-address field (addresses < 256 KB).
            const uint64_t ak0 = sw128_kmajor_desc(smem_u32(sA)), amn0 = sw128_mnmajor_desc(smem_u32(sA), kMnBlockBytes);
            const uint64_t bk0 = sw128_kmajor_desc(smem_u32(sB)), bmn0 = sw128_mnmajor_desc(smem_u32(sB), kMnBlockBytes);
            for (int k = 0; ok; ++k) {
                ProgItem it;
                if (!take(k, it) || it.meta < 0) break;
                const CtlProb& pr = cpb[item_prob(it)];
                const int pflags = pr.flags;
                const int kblocks = (pr.K + BK - 1) / BK;
                const int buf = k & 1;
                // First k-block read transposed (lower-only operands: the
                // k-blocks right of the diagonal tile); MN-major operands are
                // transposed from the first k-block on.
                const int a_tkb = (pflags & kFlagAmn) ? 0 : (pflags & kFlagAsym) ? (it.m0 + TM) / BK : 0x7fffffff;
                const int b_tkb = (pflags & kFlagBmn) ? 0 : (pflags & kFlagBsym) ? (it.n0 + TM) / BK : 0x7fffffff;
                if (!mbar_wait(acce0 + 8 * buf, ((k >> 1) & 1) ^ 1, err)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + buf * BN;
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!mbar_wait(full0 + 8 * stage, phase, err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // The operand layouts the producer chose for this k-block.
                    const bool a_mn = kb >= a_tkb, b_mn = kb >= b_tkb;
                    const uint32_t idesc = IDESC | (a_mn ? (1u << 15) : 0u) | (b_mn ? (1u << 16) : 0u);
                    // Per 16-wide k step: 32 bytes along a K-major row, or two
                    // 8-row groups (2048 bytes) of an MN-major tile.
                    const uint32_t a_step = a_mn ? (2048 >> 4) : (32 >> 4);
                    const uint32_t b_step = b_mn ? (2048 >> 4) : (32 >> 4);
                    const uint64_t adesc = (a_mn ? amn0 : ak0) + ((stage * A_BYTES) >> 4);
                    const uint64_t bdesc = (b_mn ? bmn0 : bk0) + ((stage * B_BYTES) >> 4);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        tc_mma_f16<CG>(d_tmem, adesc + a_step * kk, bdesc + b_step * kk, idesc,
                                       (kb | kk) != 0 ? 1u : 0u);
                    }
                    if constexpr (CG == 1)
                        tc_commit<1>(empty0 + 8 * stage);
                    else
                        tc_commit_pair(empty0 + 8 * stage, kPairMask);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                if constexpr (CG == 1)
                    tc_commit<1>(accf0 + 8 * buf);
                else
                    tc_commit_pair(accf0 + 8 * buf, kPairMask);
            }
            // All MMAs issued by this thread must finish before TMEM is freed.
            tc_commit<CG>(drain_bar);
            drain_wait(drain_bar, 0, err.limit_ns);
        }
        __syncwarp();
    } else if (warp == kSchedWarp) {
        // ------------------------------------------------------- scheduler
        // The pair leader's scheduler claims the pair's next tile from the
        // launch's ticket counter, decodes it, acquires its inputs (its
        // matrix's counter) and publishes the record in the ring slot of both
        // CTAs. A slot is reused once every role of both CTAs has read it; a
        // tile is claimed only `lookahead` tiles ahead of the producer, so a
        // pair never holds tiles (long ones of the first phase above all)
        // that another pair would start sooner. Claiming in ticket order
        // makes every wait end whatever the residency of the grid: a tile
        // waits only for tiles with smaller tickets, claimed by running CTAs.
        // A record with meta < 0 ends the walk.
        if (lane == 0 && rank == 0) {
            const uint32_t peer_ring = (CG == 2) ? map_to_rank(ring_u32, lead + 1) : 0;
            const uint32_t peer_ringf = (CG == 2) ? map_to_rank(ringf0, lead + 1) : 0;
            const int la = P.lookahead < 1 ? 1 : (P.lookahead > kRing ? kRing : P.lookahead);
            for (int j = 0;; ++j) {
                const int slot = j % kRing;
                if (!mbar_wait_cluster(ringe0 + 8 * slot, ((j / kRing) & 1) ^ 1, err)) break;
                // Tile j is claimed once the producer has taken tile j - la.
                // The producer has taken at most j - 1 tiles and la <= kRing,
                // so the slot's barrier is at most one phase ahead.
                if (j >= la && !mbar_wait(taken0 + 8 * ((j - la) % kRing), ((j - la) / kRing) & 1, err)) break;
                const int t = atomicAdd(P.ticket, 1);
                ProgItem rec{-1, 0, 0, 0};
                if (t < P.total_items) {
                    rec = decode_item<BN, CG>(cph, cpb, nphase, t);
                    if (P.counters && rec.wait > 0 &&
                        !wait_counter(P.counters + item_matrix(rec), rec.wait, err))
                        break;
                }
                ring[slot] = rec;
                mbar_arrive(ringf0 + 8 * slot);
                if constexpr (CG == 2) {
                    st_cluster_v4(peer_ring + slot * static_cast<uint32_t>(sizeof(ProgItem)), rec.meta, rec.wait,
                                  rec.m0, rec.n0);
                    mbar_arrive_cluster(peer_ringf + 8 * slot);
                }
                if (rec.meta < 0) break;
            }
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------- epilogue
        const int q = warp & 3;                 // TMEM lane quarter this warp may access
        const int ew = warp - 2;                // epilogue warp 0..7
        constexpr int CPW = NCH / 2;            // chunks per warp: two warps share a quarter
        const int cbeg = (ew >> 2) * CPW;       // this warp's first chunk
        const uint32_t wbase = smem_u32(sEpi + ew * SBUF);
        const uint32_t sT = wbase + 2 * kSlot;  // transposed block
        const uint32_t cbw = cbar0 + 16 * ew;   // barrier of C slot k: cbw + 8 k
        const uint32_t acce_lead = (CG == 2) ? map_to_rank(acce0, lead) : acce0;
        uint32_t cpar = 0;  // bit k: parity of C slot k's next completion
        uint32_t cpend = 0; // bit k: a C load into slot k is in flight
        int iter = 0;       // GEMM tiles done (accumulator buffer iter & 1)
        bool ok = true;
        for (int k = 0; ok; ++k) {
            // The tile record: lane 0 waits for the slot and hands it back
            // once every lane holds the record.
            ProgItem it{};
            int got = 0;
            const int slot = k % kRing;
            if (lane == 0) got = mbar_wait_cluster(ringf0 + 8 * slot, (k / kRing) & 1, err) ? 1 : 0;
            if (!__shfl_sync(0xffffffffu, got, 0)) break;
            __syncwarp();
            it = ring[slot];
            __syncwarp();
            if (lane == 0) {
                if constexpr (CG == 2)
                    mbar_arrive_cluster(ringe_lead + 8 * slot);
                else
                    mbar_arrive(ringe0 + 8 * slot);
            }
            if (it.meta < 0) break;
            const int g = item_matrix(it);
            const GemmProblem& pr = P.prob[item_prob(it)];
            const int buf = iter & 1;
            const int flags = cpb[item_prob(it)].flags;
            const bool sym = flags & kFlagSym;
            const bool hasC = flags & kFlagC;
            const bool f32 = flags & kFlagOutF32;
            const int M = pr.M, N = pr.N;
            const int r0 = it.m0 + BM * static_cast<int>(rank) + q * 32;
            const int grow = r0 + lane;
            const int sr = r0 >> 5;
            // A diagonal tile of a product of a matrix with itself: written
            // whole as computed (no upper blocks skipped, nothing mirrored).
            const bool whole = (flags & kFlagSelfSym) && TM == BN && it.m0 == it.n0;
            // This warp's live 32 x 32 blocks of the tile, in order (bit c - cbeg).
            uint32_t am = 0;
            if (r0 < M) {
#pragma unroll
                for (int c = 0; c < CPW; ++c) {
                    const int c0 = it.n0 + 32 * (cbeg + c);
                    if (c0 < N && !(sym && !whole && (c0 >> 5) > sr)) am |= 1u << c;
                }
            }
            const CUtensorMap* mapC = &P.maps[cpb[item_prob(it)].mC];
            // C of block k of the list into slot k & 1 (lane 0 issues).
            auto load_c = [&](int kk, int c) {
                const uint32_t bar = cbw + 8 * (kk & 1);
                mbar_arrive_expect_tx(bar, kSlot);
                tma_load_3d(wbase + (kk & 1) * kSlot, mapC, bar, it.n0 + 32 * c, r0, g);
            };
            if (hasC && am) {
                if (P.counters && it.wait > 0) {
                    // C is an earlier item's output: acquire it like the producer.
                    int okc = 1;
                    if (lane == 0) okc = wait_counter(P.counters + g, it.wait, err) ? 1 : 0;
                    if (!__shfl_sync(0xffffffffu, okc, 0)) break;
                }
                uint32_t m = am;
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {
                    if (m) {
                        if (lane == 0) {
                            if (kk == 0) fence_proxy_async_global();
                            load_c(kk, cbeg + __ffs(m) - 1);
                        }
                        cpend |= 1u << kk;
                        m &= m - 1;
                    }
                }
            }

            // Every lane waits; the warp goes on only if all saw the phase (a lane
            // that gave up on the bounded wait takes the warp out with it, so the
            // warp-wide tcgen05.ld below never runs divergent).
            if (!__all_sync(0xffffffffu, mbar_wait(accf0 + 8 * buf, (iter >> 1) & 1, err))) break;
            tc_fence_after();

            uint32_t m = am;
            int kq = 0;
#pragma unroll 1
            while (m) {
                const int c = cbeg + __ffs(m) - 1;
                m &= m - 1;
                const int c0 = it.n0 + 32 * c;
                const uint32_t slot = wbase + (kq & 1) * kSlot;
                uint32_t acc[32];
                tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * BN + c * 32, acc);
                uint4 cb[4];
                if (hasC) {
                    if (!__all_sync(0xffffffffu, mbar_wait(cbw + 8 * (kq & 1), (cpar >> (kq & 1)) & 1, err))) {
                        ok = false;
                        break;
                    }
                    cpar ^= 1u << (kq & 1);
                    cpend &= ~(1u << (kq & 1));
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) cb[kk] = ld_shared_v4(sw64_piece(slot, lane, kk));
                }
                tmem_ld_wait();

                float v[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = pr.alpha * __uint_as_float(acc[j]);
                if (hasC) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint32_t wv[4] = {cb[kk].x, cb[kk].y, cb[kk].z, cb[kk].w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&wv[e]));
                            v[8 * kk + 2 * e] = fmaf(pr.beta, f.x, v[8 * kk + 2 * e]);
                            v[8 * kk + 2 * e + 1] = fmaf(pr.beta, f.y, v[8 * kk + 2 * e + 1]);
                        }
                    }
                }
                // Every lane has read its C row: the slot may be overwritten.
                __syncwarp();
                if (flags & kFlagMuon) {
                    muon_update_row(pr, g, grow, c0, v);
                } else {
                    const bool diag_block = sym && !whole && ((c0 >> 5) == sr);
                    // Lower-only outputs mirror only inside diagonal tiles.
                    const bool mirror = (flags & kFlagDt) && !diag_block && !whole &&
                                        (!(flags & kFlagLower) || it.m0 == it.n0);
                    // Stage, transpose (mirror or diagonal fix-up) and store one
                    // 32 x 32 block; the slot is free again once the warp has
                    // read it back.
                    auto emit = [&](const float (&val)[32], const OutView& od, const OutView& odt) {
                        if (P.direct_store && !mirror && !diag_block && c0 + 32 <= N && out_direct(od, f32 ? 4 : 2)) {
                            if (grow < M) direct_row(od, g, grow, c0, val, f32);
                        } else if (f32) {
                            emit_f32(slot, val, od, g, r0, c0, M, N, lane);
                        } else {
                            stage_row_f16(slot, lane, val);
                            if (mirror || diag_block) stage_transpose(slot, sT, diag_block, lane);
                            __syncwarp();
                            store_rows64<2>(slot, od, g, r0, c0, M, N, lane);
                            if (mirror) store_rows64<2>(sT, odt, g, c0, r0, N, M, lane);
                        }
                        __syncwarp();
                    };
                    emit(v, pr.d, pr.dt);
                    if (flags & kFlagD2) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] = pr.delta * v[j] + ((grow == c0 + j) ? pr.gamma : 0.0f);
                        emit(v, pr.d2, pr.d2t);
                    }
                }
                // The C of the block two places further into the slot just freed.
                if (hasC && m && (m & (m - 1))) {
                    const uint32_t m2 = m & (m - 1);
                    if (lane == 0) load_c(kq, cbeg + __ffs(m2) - 1);
                    cpend |= 1u << (kq & 1);
                }
                ++kq;
            }
            if (!ok) break;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                // Publish the tile once per CTA: each warp counts itself done
                // (a CTA-scope release covering its lanes' stores, which the
                // warp barrier above ordered before it); the warp that
                // completes the count releases the CTA's part of the tile to
                // the matrix's counter, cumulatively over all eight warps'
                // stores, so only one warp per tile waits for its stores to
                // land. The count comes before the accumulator is handed
                // back, so a buffer's counts never mix two tiles.
                const uint32_t old = atom_add_acqrel_cta(pub0 + 4 * buf, 1);
                if constexpr (CG == 1)
                    mbar_arrive(acce0 + 8 * buf);
                else
                    mbar_arrive_cluster(acce_lead + 8 * buf);
                if (P.counters && old % kEpiWarps == kEpiWarps - 1) red_release_add(P.counters + g, kEpiWarps);
            }
            ++iter;
        }
        // C loads still in flight (only after a failed wait) land before exit.
        if (lane == 0) {
            for (int kk = 0; kk < 2; ++kk)
                if (cpend & (1u << kk)) drain_wait(cbw + 8 * kk, (cpar >> kk) & 1, err.limit_ns);
        }
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    // The leader's MMAs read the peer's shared memory and the peer's loads
    // and epilogues arrive on the leader's barriers: no CTA of the cluster
    // leaves before all are done.
    if constexpr (CL > 1) cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<CG>(tmem_base, TMEM_COLS);
    }
}

// Per-device launch state of one kernel variant: the dynamic shared-memory
// opt-in is a per-device function attribute, and the resident cluster count
// is a property of the device, so both are kept per device ordinal.
constexpr int kMaxDevices = 64;

struct VariantState {
    bool configured = false;
    int clusters = -1;
};

template <int BN, int CG>
VariantState& variant_state(int dev) {
    static VariantState st[kMaxDevices];
    return st[dev];
}

// Sets the variant's dynamic shared-memory opt-in on the current device once.
template <int BN, int CG>
cudaError_t configure(VariantState& vs) {
    if (!vs.configured) {
        const cudaError_t e =
            cudaFuncSetAttribute(gemm_tc_kernel<BN, CG>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes<BN, CG>());
        if (e != cudaSuccess) return e;
        vs.configured = true;
    }
    return cudaSuccess;
}

// Clusters of CG CTAs that can be resident at once with this kernel's
// shared memory on the current device; the grid never exceeds it, so every
// cluster of a program runs concurrently (tiles wait on tiles of other
// clusters).
template <int BN, int CG>
int max_clusters(VariantState& vs, int num_sms) {
    if (vs.clusters < 0 && configure<BN, CG>(vs) == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(CG * (num_sms / CG));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = smem_bytes<BN, CG>();
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = CG;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, gemm_tc_kernel<BN, CG>, &cfg) != cudaSuccess || n <= 0) {
            cudaGetLastError();
            n = num_sms / CG;
        }
        vs.clusters = n;
    }
    if (vs.clusters < 0) {
        cudaGetLastError();
        return num_sms / CG > 1 ? num_sms / CG : 1;
    }
    const int cap = num_sms / CG > 1 ? num_sms / CG : 1;  // at least one cluster, even under an SM cap of 1
    return vs.clusters < cap ? vs.clusters : cap;
}

template <int BN, int CG>
int launch_impl(const GemmProgram& prog, int num_sms, cudaStream_t stream) {
    constexpr int bytes = smem_bytes<BN, CG>();
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    VariantState& vs = variant_state<BN, CG>(dev);
    e = configure<BN, CG>(vs);
    if (e != cudaSuccess) return e;
    if (prog.total_items <= 0) return cudaSuccess;
    const int clusters = max_clusters<BN, CG>(vs, num_sms);
    const int grid = CG * (prog.total_items < clusters ? prog.total_items : clusters);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = CG;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<BN, CG>, prog);
}

}  // namespace

int gemm_smem_bytes(int bn, int cg) {
    if (cg == 2) return smem_bytes<256, 2>();
    return bn == 256 ? smem_bytes<256, 1>() : smem_bytes<128, 1>();
}

int gemm_tiles_per_matrix(int M, int N, int bn, int cg, bool sym, int* walk_n) {
    const int tmh = BM * cg;
    const int tm = (M + tmh - 1) / tmh;
    const int tn = (N + bn - 1) / bn;
    if (walk_n) *walk_n = tn;
    int total = 0;
    if (!sym) {
        total = tm * tn;
    } else {
        for (int i = 0; i < tm; ++i) total += sym_row_tiles(i, tmh, bn, tn);
    }
    return total;
}

int gemm_signals_per_tile(int cg) { return kEpiWarps * cg; }

int launch_gemm_program(const GemmProgram& prog, int bn, int cg, int num_sms, cudaStream_t stream) {
    if (cg == 2) return launch_impl<256, 2>(prog, num_sms, stream);
    if (bn == 256) return launch_impl<256, 1>(prog, num_sms, stream);
    return launch_impl<128, 1>(prog, num_sms, stream);
}

}  // namespace gns
