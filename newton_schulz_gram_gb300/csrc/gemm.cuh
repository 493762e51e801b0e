// Shared (host and device) description of one grouped GEMM launch.
//
// A launch runs a "program": a sequence of phases over a bucket of G
// matrices. Each phase holds one or more independent problems; a problem is
// a batch of G equal-shaped products D_g = alpha * A_g B_g^T (+ beta * C_g),
// fp16 operands, fp32 accumulation, A_g M x K and B_g N x K row-major (K
// contiguous). For a symmetric product (Dion3 §5) only the tiles touching the
// lower triangle are computed and each is also written transposed into the
// upper triangle.
//
// The work of a launch is a list of tiles, phase by phase, matrix by
// matrix. CTAs (pairs) claim the tiles in list order from a ticket counter.
// Every tile, once stored, adds kEpiWarps * CG to its matrix's counter in
// global memory (one release per CTA, cumulative over its epilogue warps'
// stores); a tile that needs the earlier phases of its matrix first waits
// until the counter reaches its target (acquire). Matrices thus pipeline
// through the phases without a grid-wide barrier. Every dependency points
// to a tile with a smaller ticket, claimed by a running CTA, so every wait
// ends whatever the residency of the grid.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace gns {

enum GemmFlags : int {
    kFlagSym = 1,     // lower-triangle tile list, mirrored epilogue (M == N)
    kFlagC = 2,       // add beta * C (fp16, row-major, same shape as D)
    kFlagDt = 4,      // also write D transposed into Dt ([G][N][M])
    kFlagD2 = 8,      // also write D2 = delta * D + gamma * I (fp16), and its mirror D2t
    kFlagOutF32 = 16, // D is fp32 (otherwise fp16)
    kFlagAmn = 32,    // A is MN-major: the stored matrix is K x M (A^T row-major)
    kFlagBmn = 64,    // B is MN-major: the stored matrix is K x N (B^T row-major)
    // Symmetric matrices stored lower-only: only tiles (I, J) with J <= I of
    // a square tiling (edge = the tile's M edge, which then equals BN) hold
    // data, diagonal tiles in full. An operand flagged so reads a k-block in
    // tile column J > I as the transpose of tile (J, I) (an MN-major load
    // through mAt / mBt); an output flagged kFlagLower is written that way
    // (mirrored blocks only inside diagonal tiles).
    kFlagAsym = 256,
    kFlagBsym = 512,
    kFlagLower = 1024,
    // Fused Muon update: D is not stored; each output element o = fp16(alpha
    // acc) updates the bf16 weight of the same (row, column) of matrix g,
    // W <- SR_bf16((1 - lr wd) W - (lr scale) o), with the stochastic
    // rounding counter of global index w_base[g] + row N + column.
    kFlagMuon = 2048,
    // Non-symmetric product walked column by column: the tiles sharing a B
    // column block run together, so B (for Q X, the large X) is read from
    // DRAM about once and hits L2 for the other tile rows.
    kFlagColWalk = 4096,
    // Symmetric product of one matrix with itself (A and B the same stored
    // operand, and C exactly symmetric): every element (i, j) and (j, i) is
    // the same sum of the same products in the same order, so the
    // accumulator of a diagonal tile is exactly symmetric and all of its
    // blocks, above the diagonal too, are written as computed, with no
    // mirrored copy (square tiles only).
    kFlagSelfSym = 8192
};

// Parameters of the fused Muon update (kFlagMuon).
struct MuonFuse {
    uint16_t* const* w;     // device array [G]: bf16 W, row-major M x N, contiguous
    const long long* base;  // device array [G]: global index of each W's first element
    float lr, wd, scale;
    uint32_t seed_lo, seed_hi, step_lo, step_hi;
};

constexpr int kMaxMaps = 64;
constexpr int kMaxProblems = 48;
constexpr int kMaxPhases = 40;

// Epilogue warps of a CTA of the GEMM program (two per TMEM lane quarter);
// each CTA adds kEpiWarps counter signals per tile.
constexpr int kEpiWarps = 8;

// One tile record (16 bytes): meta = problem | matrix g << 8 (negative: the
// end of the walk), the tile's origin (m0, n0), and `wait`, the matrix
// counter value the tile needs before it starts (0: none).
struct alignas(16) ProgItem {
    int meta;
    int wait;
    int m0;
    int n0;
};

// An output written by the epilogue: G row-major matrices, element (g, r, c)
// at p + g stride + r ld (fp16, or fp32 for kFlagOutF32). ld is a multiple of
// 16 bytes and p is 16-byte aligned, so rows are stored in 16-byte pieces.
struct OutView {
    void* p;
    long long ld, stride;
};

struct GemmProblem {
    const __half* C;  // addend, row-major [G][M][ldc]
    long long ldc;
    long long strideC;
    OutView d, dt, d2, d2t;  // D, its transpose, D2 and its transpose
    float alpha, beta, delta, gamma;
    int M, N, K;
    int tiles_n;           // tile columns of the matrix
    int tiles_n_walk;      // tile columns enumerated per row (= tiles_n)
    int tiles_m;           // tile rows of the matrix
    int tiles_per_matrix;  // tiles enumerated per matrix
    int flags;
    // Indices into GemmProgram::maps (-1 when unused). K-major operand maps:
    // box {64 (K), rows per CTA}; MN-major operand maps: box {64 (M or N),
    // 64 (K)}; both 128-byte swizzle. The addend's map (mC): box {32, 32},
    // 64-byte swizzle.
    int mA, mB, mC;
    int mAt, mBt;  // MN-major views (box {64, 64}) of lower-only A / B
    MuonFuse muon;
};

struct GemmPhaseDesc {
    int prob_begin, nprob;  // problems prob[prob_begin .. prob_begin + nprob)
    int tiles_per_matrix;   // over all its problems
    int item_begin;         // ticket of its first tile
    int wait;               // counter target of its tiles: signals of all earlier tiles of the matrix
};

struct alignas(128) GemmProgram {
    CUtensorMap maps[kMaxMaps];
    GemmProblem prob[kMaxProblems];
    GemmPhaseDesc phase[kMaxPhases];
    int* counters;       // [G] per-matrix signal counters, zero at launch; null when nothing waits
    int* ticket;         // the launch's ticket counter, zero at launch
    DevStatus st;
    int nmaps, nprob, nphase, G, total_items;
    int direct_store;    // full-width, 32-byte aligned output blocks go straight from registers to memory
    int lookahead;       // a CTA pair claims tile j once its producer has taken tile j - lookahead (1 .. 8)
};

// Host-side launcher (gemm_tc.cu). Tile shapes: cg = 1 and bn = 128 or 256
// (one CTA, 128 x bn tiles), or cg = 2 and bn = 256 (a CTA pair, 256 x 256
// tiles with paired MMAs). Launches carry the programmatic-dependent-launch
// attribute; the kernel waits for the previous grid before reading its
// operands. Returns a cudaError_t value.
int launch_gemm_program(const GemmProgram& prog, int bn, int cg, int num_sms, cudaStream_t stream);

int gemm_smem_bytes(int bn, int cg);
// Tile walk of one matrix of an M x N problem: lower-triangle tiles if sym.
// Returns tiles per matrix and sets *walk_n (tiles per row walked for
// non-symmetric problems).
int gemm_tiles_per_matrix(int M, int N, int bn, int cg, bool sym, int* walk_n);
// Counter increments one tile contributes (one per epilogue warp).
int gemm_signals_per_tile(int cg);

}  // namespace gns
