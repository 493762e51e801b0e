// Shared (host and device) description of one grouped GEMM launch.
//
// A launch ("phase") runs up to two independent problems. Each problem is a
// batch of G equal-shaped products D_g = alpha * A_g B_g^T (+ beta * C_g),
// fp16 operands, fp32 accumulation, where A_g is M x K and B_g is N x K, both
// row-major (K contiguous). For a symmetric product (Dion3 §5) only the
// lower-triangle 128 x 128 tiles are computed and each is also written
// transposed into the upper triangle.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>

namespace gns {

enum GemmFlags : int {
    kFlagSym = 1,     // triangular tile list, mirrored epilogue (M == N, BN == 128)
    kFlagC = 2,       // add beta * C (fp16, row-major, same shape as D)
    kFlagDt = 4,      // also write D transposed through tmDt
    kFlagD2 = 8,      // also write D2 = delta * D + gamma * I (fp16) through tmD2 (+ tmD2t)
    kFlagOutF32 = 16  // D is fp32 (otherwise fp16)
};

struct alignas(128) GemmProblem {
    CUtensorMap tmA;    // [G][M][K] fp16, box {64, 128}, 128-byte swizzle
    CUtensorMap tmB;    // [G][N][K] fp16, box {64, BN}, 128-byte swizzle
    CUtensorMap tmD;    // [G][M][N] fp16 (box {32,32}, 64B swizzle) or fp32 (box {32,32}, 128B swizzle)
    CUtensorMap tmDt;   // [G][N][M] fp16, box {32, 32}, no swizzle
    CUtensorMap tmD2;   // [G][M][N] fp16, as tmD
    CUtensorMap tmD2t;  // [G][N][M] fp16, as tmDt
    const __half* C;    // addend, row-major [G][M][ldc]
    long long ldc;
    long long strideC;
    float alpha, beta, delta, gamma;
    int M, N, K, G;
    int tiles_m, tiles_n, tiles_per_matrix, tile_begin;
    int flags;
    int pad_;
};

struct alignas(128) GemmPhase {
    GemmProblem prob[2];
    int* err;
    int nprob;
    int total_tiles;
};

// Host-side launchers (gemm_tc.cu). `bn` selects the tile width: 128 for
// symmetric phases (and those with a second output), 256 for the general
// products. Return a cudaError_t value.
int launch_gemm_phase(const GemmPhase& phase, int bn, int num_sms, cudaStream_t stream);
int gemm_smem_bytes(int bn);

}  // namespace gns
