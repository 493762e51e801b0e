/*
 * gns.h: C ABI of the GB300 (sm_103a) Gram Newton-Schulz / Muon library.
 *
 * Every entry point is plain C: device or host pointers, sizes, scalars and a
 * CUDA stream passed as void* (cudaStream_t; NULL means the legacy default
 * stream). No call allocates caller-visible memory. Calls that take device
 * pointers are asynchronous on `stream` unless stated otherwise.
 *
 * Ownership: the caller owns every buffer it passes. The library owns one
 * cached workspace per device (Gram state, fp16 copies of the inputs, norm
 * partials, a status word). It grows on demand and is freed by
 * gns_release(). Calls on different streams of one device must not overlap
 * in time, because they share that workspace.
 *
 * Errors: argument and shape errors, and failures of CUDA runtime calls, are
 * returned at once as a negative gns_status. Conditions found on the device
 * (a non-finite input norm, a bounded wait that ran out) set a per-device
 * status word that gns_get_status() reads.
 *
 * Notation: a matrix X of R x C is handled as n x m with n = min(R, C),
 * m = max(R, C); a matrix with R > C is transposed on the way in and back on
 * the way out. Citations are to "Dion3: Full-stack orthogonal updates"
 * (arXiv 2608.11612) and to the grouped Muon kernel card
 * (kernels/phanerozoic/muon).
 */
#ifndef GNS_H
#define GNS_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GNS_OK = 0,
    GNS_ERR_INVALID = -1,     /* bad argument (null pointer, size, steps, alignment) */
    GNS_ERR_CUDA = -2,        /* a CUDA runtime call failed; see gns_last_error() */
    GNS_ERR_NONFINITE = -3,   /* device: some input matrix had a non-finite norm */
    GNS_ERR_TIMEOUT = -4,     /* device: a bounded wait inside a kernel ran out */
    GNS_ERR_NOMEM = -5,       /* the workspace could not be allocated */
    GNS_ERR_UNSUPPORTED = -6  /* the current device is not an sm_103 (GB300) GPU */
} gns_status;

/* Default (and maximum) number of Newton-Schulz steps a call accepts. */
#define GNS_MAX_STEPS 64

/*
 * gns_orthogonalize_batched: approximate polar(X) for each of G matrices.
 *
 * Follows Dion3 §4.2 Algorithm 3 (stabilized Gram Newton-Schulz) with the
 * a-term distribution of App. B.2.3, and, for square matrices, the standard
 * iteration of §2.2 Algorithm 1 with symmetric products (App. C.3), as §4.1
 * prescribes for alpha = 1. Each matrix is scaled to Frobenius norm 1/1.05
 * (App. B.2.2 safety factor; X / (1.05 (||X||_F + 1e-7))), cast to fp16 and
 * iterated in fp16 storage with fp32 accumulation.
 *
 *   ptr        device fp32 [G][R][C], row-major, contiguous. Overwritten in
 *              place with the result (fp32, same shape).
 *   G, R, C    G >= 0 (G == 0 is a no-op), R >= 1, C >= 1.
 *   steps      1..GNS_MAX_STEPS (5 in the pages' setting).
 *   restart_at restart period p: restart after every step t with t % p == 0
 *              and steps - t >= p (p = 2, steps = 5 gives Algorithm 3's single
 *              restart after step 2; p <= 0 never restarts). Ignored for
 *              square matrices.
 *   coeffs     HOST float[3*steps], (a_t, b_t, c_t) for t = 1..steps, or
 *              NULL for the constant quintic (3.4445, -4.7750, 2.0315) of the
 *              Muon kernel card at every step. Non-finite values are rejected.
 *   stream     cudaStream_t.
 * Returns GNS_OK or a negative gns_status. Asynchronous.
 */
int gns_orthogonalize_batched(float* ptr, int G, int R, int C, int steps, int restart_at,
                              const float* coeffs, void* stream);

/*
 * gns_orthogonalize_batched_schedule: gns_orthogonalize_batched with any
 * restart schedule (Dion3 App. B.2.1 chooses one per coefficient schedule):
 * bit t of restart_mask set (1 <= t < steps) = restart after step t
 * (X <- Q X, R <- X X^T, Q <- I). Other bits set: GNS_ERR_INVALID. The
 * periodic restart_at of gns_orthogonalize_batched is the mask with the
 * multiples t of restart_at that leave at least restart_at steps.
 */
int gns_orthogonalize_batched_schedule(float* ptr, int G, int R, int C, int steps, uint64_t restart_mask,
                                       const float* coeffs, void* stream);

/*
 * gns_gram_ns_state: gns_orthogonalize_batched on a rectangular bucket that
 * also hands back the iteration's fp16 Gram state, to check the stability
 * bounds of Dion3 App. B.2.1 (Fig. 18: with a restart after step 2 the
 * eigenvalues of R_t stay above -0.4 and those of Q_t below about 100).
 *
 *   ptr, G, R, C, steps, restart_mask  as gns_orthogonalize_batched_schedule
 *              (bit t: restart after step t), with R != C (square matrices
 *              have no Gram state: GNS_ERR_INVALID) and the whole bucket in
 *              one workspace chunk (else GNS_ERR_INVALID). Default
 *              coefficients.
 *   r_state    device uint16 (fp16 bits) [G][n][n], n = min(R, C): the last
 *              Gram matrix R the run computed (R_{steps-1}, or X X^T when a
 *              restart follows the last update; R_0 for steps = 1), scaled:
 *              stored R = r_scale * R. Only the lower triangle (with the
 *              diagonal) is defined: the library stores symmetric
 *              intermediates lower-only.
 *   q_state    device uint16 (fp16 bits) [G][n][n]: the final Q_steps (the
 *              accumulated polynomial since the last restart), unscaled,
 *              lower triangle defined as for r_state.
 *   r_scale    HOST float: receives the power-of-two state scale.
 *   stream     cudaStream_t. The copies are stream-ordered after the run.
 * Returns GNS_OK or a negative gns_status. Diagnostic: it runs the same
 * program as gns_orthogonalize_batched plus two device copies.
 */
int gns_gram_ns_state(float* ptr, int G, int R, int C, int steps, uint64_t restart_mask, uint16_t* r_state,
                      uint16_t* q_state, float* r_scale, void* stream);

/*
 * gns_orthogonalize_batched_host: the same computation on a HOST buffer.
 * host_ptr is fp32 [G][R][C] in host memory (pinned memory gives full copy
 * speed); the library copies it to a device staging buffer it owns, runs
 * gns_orthogonalize_batched there, copies the result back and synchronizes
 * `stream` before returning. The bucket is pipelined in chunks of about
 * 64 MiB (GNS_HOST_CHUNK_MB overrides), the first and last half size: chunk
 * copies in and out run on two library-owned streams and overlap the
 * neighbouring chunks' orthogonalization on `stream`.
 */
int gns_orthogonalize_batched_host(float* host_ptr, int G, int R, int C, int steps,
                                   int restart_at, const float* coeffs, void* stream);

/*
 * gns_orthogonalize_batched_noalloc: gns_orthogonalize_batched without any
 * device allocation, for callers that cannot let a library call cudaMalloc
 * (their device memory is already held by their own allocator or pool, or
 * they cannot accept the device-wide synchronization that growing the cached
 * workspace costs). The paper has no counterpart; this is a library entry
 * point only.
 *
 * Arguments, layout and results are those of gns_orthogonalize_batched (the
 * results are bit-identical). The workspace is one fixed 64 MiB array in
 * device memory that every GPU which loads the library holds until the
 * process exits; the bucket is processed in as many sequential chunks as
 * that space requires. A matrix whose workspace alone exceeds it (for
 * example 4096 x 14336) is rejected with GNS_ERR_INVALID and a message in
 * gns_last_error(). The first call on a device looks up the array's device
 * address (cudaGetSymbolAddress); make that first call before any stream
 * capture. Every call shares the array, so calls that overlap on the GPU (on
 * different streams) race and must not be issued. Device-side conditions (a
 * non-finite input norm, a bounded wait that ran out) go to a status word
 * inside the array, which gns_get_status() reads and clears without
 * allocating. GNS_NUM_SMS caps the SMs used, as for the allocating entry
 * points.
 */
int gns_orthogonalize_batched_noalloc(float* ptr, int G, int R, int C, int steps, int restart_at,
                                      const float* coeffs, void* stream);

/* One 2D tensor of a Muon step. data is a device pointer; rows x cols,
 * row-major, contiguous. base_index is the global index of element (0, 0)
 * for the stochastic-rounding counter (the Muon kernel card: a parameter
 * updated whole or across shards rounds identically). */
typedef struct {
    void* data;
    int rows;
    int cols;
    int64_t base_index;
} gns_tensor;

/*
 * muon_step: one Muon step over n weight matrices (Dion3 §2.1 Eq. 1 with
 * decoupled weight decay, §6 "Weight Update"; the Muon kernel card):
 *   M <- mu M + G                              (fp32, M_0 = 0)
 *   O <- gns(M)                                (as gns_orthogonalize_batched,
 *                                               steps 5, restart_at 2, quintic)
 *   W <- SR_bf16((1 - lr*wd) W - lr*s*O),  s = 0.2 sqrt(max(rows, cols))
 * with the update in fp32 (decay = 1 - lr*wd, step = lr*s,
 * w' = decay*w - step*o, each rounded once) and a stochastically rounded
 * bf16 write-back keyed by (seed, step, base_index + element index)
 * (Philox4x32-10: one output serves the block g >> 3 of eight global indices,
 * element g = base_index + i taking the 16-bit half (g & 1), low first, of
 * output word (g & 7) >> 1).
 *
 *   params    n tensors, bf16 weights, updated in place.
 *   grads     n tensors, bf16 gradients (same shapes), read.
 *   momentum  n tensors, fp32 momentum (same shapes), updated in place.
 * Matrices are grouped into buckets of equal (rows, cols) and each bucket is
 * orthogonalized in one batched pass. Returns GNS_OK or a negative status.
 */
int muon_step(const gns_tensor* params, const gns_tensor* grads, const gns_tensor* momentum,
              int n, float lr, float wd, float mu, uint64_t seed, uint64_t step, void* stream);

/*
 * normuon_step: one NorMuon step (Dion3 §2.1 Eq. 2) over n weight matrices:
 * muon_step's momentum and orthogonalization, then, per row i of O (the
 * weight's own rows), in fp32:
 *   v_i <- beta2 v_i + (1 - beta2) (1/cols) sum_j O_ij^2
 *   U   =  (||O||_F / ||O^||_F) O^,   O^_ij = O_ij / (sqrt(v_i) + eps)
 *   W   <- SR_bf16((1 - lr*wd) W - lr*s*U),  s = 0.2 sqrt(max(rows, cols))
 * with the stochastic rounding of muon_step. The row statistics and the two
 * norms are summed in a fixed order, so results do not depend on the
 * bucketing.
 *   second_moments  n tensors, fp32 v, each rows x 1 (the weight's rows),
 *                   updated in place; start them at zero.
 * Other arguments as muon_step; beta2 in [0, 1], eps >= 0.
 */
int normuon_step(const gns_tensor* params, const gns_tensor* grads, const gns_tensor* momentum,
                 const gns_tensor* second_moments, int n, float lr, float wd, float mu, float beta2,
                 float eps, uint64_t seed, uint64_t step, void* stream);

/*
 * dion3_step: one step of the Dion3 update rule (Dion3 §6, Algorithm 4,
 * Muon flavor) over n weight matrices:
 *   M <- M + G                                        (fp32)
 *   S <- the k = ceil(fraction * d) rows of M with the largest l1 norm, d the
 *        row count, or the columns when they are fewer (d = cols); largest
 *        first, equal norms by lower index
 *   O <- gns(M[S])                                    (k x max(rows, cols))
 *   W <- SR_bf16((1 - lr*wd) W - lr*s*O~),  O~ = O on S and 0 elsewhere,
 *        s = 0.2 sqrt(max(rows, cols)), stochastic rounding as muon_step
 *   M[S] <- mu M[S]                                   (error feedback)
 * fraction in (0, 1]; min(rows, cols) <= 16384. Other arguments as muon_step.
 */
int dion3_step(const gns_tensor* params, const gns_tensor* grads, const gns_tensor* momentum, int n,
               float fraction, float lr, float wd, float mu, uint64_t seed, uint64_t step, void* stream);

/*
 * gns_muon_momentum: the first elementwise pass of muon_step on one tensor:
 * M <- mu*M + float(G), fp32, two roundings (Dion3 Eq. 1).
 *   M      device fp32 [numel], updated in place.
 *   G_bf16 device bf16 bits [numel].
 */
int gns_muon_momentum(float* M, const uint16_t* G_bf16, int64_t numel, float mu, void* stream);

/*
 * gns_muon_update: the last elementwise pass of muon_step on one tensor:
 * W <- SR_bf16(decay*W - step*O), decay = 1 - lr*wd, step = lr*scale, all in
 * fp32 with single roundings, SR keyed as in muon_step.
 *   W_bf16 device bf16 bits [rows][cols], updated in place.
 *   O_fp16 device fp16 bits [rows][cols], read.
 */
int gns_muon_update(uint16_t* W_bf16, const uint16_t* O_fp16, int rows, int cols, float lr,
                    float wd, float scale, uint64_t seed, uint64_t step, int64_t base_index,
                    void* stream);

/*
 * gns_symm_gemm: the symmetric product of Dion3 §5 (D = alpha A B + beta C
 * with A B and C symmetric), batched over G matrices. Only lower-triangle
 * tiles are computed; each is written to its own place and mirrored into the
 * upper triangle, so D is exactly symmetric.
 *   A  device fp16 [G][n][k] row-major.
 *   B  device fp16 [G][n][k] row-major; the product is A B^T (the Gram
 *      product X X^T when B == A; A B when B is symmetric and k == n).
 *   C  device fp16 [G][n][n] (exactly symmetric) or NULL (beta ignored).
 *   D  device fp16 [G][n][n], written.
 * n and k must be multiples of 8 (16-byte rows) and every pointer 16-byte
 * aligned. Asynchronous.
 */
int gns_symm_gemm(const void* A, const void* B, const void* C, void* D, int G, int n, int k,
                  float alpha, float beta, void* stream);

/* Synchronizes `stream`, returns the device status word of the current device
 * as a gns_status (GNS_OK, GNS_ERR_NONFINITE or GNS_ERR_TIMEOUT) and clears it.
 * It reads both the allocating entry points' word and, once the
 * allocation-free entry point has run on the device, that entry point's word
 * (the first nonzero one is returned, both are cleared); it allocates nothing.
 * A condition stays recorded until it is read: a non-finite input makes only
 * its own matrix's output non-finite, and a later call runs normally whether
 * or not the word has been read. */
int gns_get_status(void* stream);

/*
 * gns_test_bounded_wait: a check of the library's failure handling, not part
 * of the path (the pages have no counterpart; their only failure mode is the
 * numerical divergence that the restarts prevent). Launches one block of 256
 * threads on `stream` that wait for something that never happens: an
 * mbarrier phase no thread completes (kind 0) or a device counter nothing
 * releases (kind 1). Thread 0 waits at most limit_ns nanoseconds
 * (1000 .. 1e9); the others wait with a 1000 times longer bound and must give
 * up through the abort mark thread 0 raises. Synchronizes `stream` and
 * returns the number of waits that gave up (256 when every wait ended), or a
 * negative gns_status. Afterwards gns_get_status() reports GNS_ERR_TIMEOUT and
 * the device stays usable: no fault, no trap, no hang.
 */
int gns_test_bounded_wait(int kind, int64_t limit_ns, void* stream);

/* Static text for a gns_status value. */
const char* gns_status_string(int status);

/* Text of the last failing CUDA call on this thread ("" if none). */
const char* gns_last_error(void);

/* Number of kernel launches the library has issued since it was loaded
 * (all devices, all entry points). */
int64_t gns_launch_count(void);

/* Measurement support. With profiling on (on != 0), every kernel launch is
 * bracketed by two CUDA events recorded on its own stream. Off by default. */
void gns_profile_enable(int on);

/* Synchronizes the recorded events and returns, per kernel class, the number
 * of profiled launches (counts[k]) and their summed event durations in ms
 * (ms[k]) since the previous read; then forgets them. Classes: 0 tcgen05
 * GEMM, 1 norm + scale + cast to fp16 (with the momentum update inside
 * muon_step), 2 Muon elementwise (update / write-back, standalone momentum),
 * 3 output copy. Writes min(max_classes, 4) entries of each non-null array
 * and returns the number of classes (4), or a negative gns_status. */
int gns_profile_read(int64_t* counts, double* ms, int max_classes);

/* Workspace bytes currently held on the current device. */
int64_t gns_workspace_bytes(void);

/* Frees the cached workspace of the current device (synchronizes it first). */
void gns_release(void);

#ifdef __cplusplus
}
#endif

#endif /* GNS_H */
