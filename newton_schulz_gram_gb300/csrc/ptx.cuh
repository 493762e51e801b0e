// Inline-PTX primitives for sm_103a: mbarrier, TMA (cp.async.bulk.tensor),
// tcgen05 (TMEM allocation, MMA, commit, loads) and their descriptors.
//
// Every wait here is bounded: after DevStatus::limit_ns of %globaltimer time
// it gives up, records GNS_ERR_TIMEOUT in the status word, raises the abort
// mark of its call and returns false, so a kernel never spins forever. A
// wait also gives up as soon as another thread has raised the abort mark of
// the same call.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>

namespace gns {

constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;  // 2 s
constexpr int kDevErrTimeout = -4;                        // == GNS_ERR_TIMEOUT
constexpr int kDevErrNonFinite = -3;                      // == GNS_ERR_NONFINITE

// Device-side error reporting of one library call, passed to its kernels by
// value. word[0] is the status word: the first condition any kernel found
// (GNS_ERR_NONFINITE or GNS_ERR_TIMEOUT), kept until the host reads and
// clears it. word[1] is the abort mark: the number (epoch) of the call whose
// wait ran out. Waits give up early only when word[1] equals their own
// call's epoch, so neither a non-finite input nor an abort left over from an
// earlier call stops the waits of a later one.
struct DevStatus {
    int* word;
    int epoch;  // nonzero, different for consecutive calls on a device
    int pad;
    unsigned long long limit_ns;
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void raise_error(const DevStatus& st, int code) {
    if (st.word) atomicCAS(st.word, 0, code);
}

// A wait of this call ran out: record it and make the call's other waits give up.
__device__ __forceinline__ void raise_timeout(const DevStatus& st) {
    if (st.word) {
        atomicCAS(st.word, 0, kDevErrTimeout);
        atomicExch(st.word + 1, st.epoch);
    }
}

__device__ __forceinline__ bool call_aborted(const DevStatus& st) {
    return st.word && *reinterpret_cast<const volatile int*>(st.word + 1) == st.epoch;
}

// ----------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// try_wait with acquire semantics at cluster scope: for phases completed by
// arrivals from other CTAs of the cluster that publish data.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

static __device__ __noinline__ bool mbar_wait_cluster_slow(uint32_t bar, uint32_t parity, const DevStatus& st) {
    const uint64_t t0 = globaltimer();
    while (true) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait_cluster(bar, parity)) return true;
        if (call_aborted(st)) return false;
        if (globaltimer() - t0 > st.limit_ns) {
            raise_timeout(st);
            return false;
        }
    }
}

// Bounded wait with cluster-scope acquire.
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, const DevStatus& st) {
    return mbar_try_wait_cluster(bar, parity) || mbar_wait_cluster_slow(bar, parity, st);
}

// The bounded spin of mbar_wait, out of line.
static __device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, const DevStatus& st) {
    const uint64_t t0 = globaltimer();
    while (true) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (call_aborted(st)) return false;
        if (globaltimer() - t0 > st.limit_ns) {
            raise_timeout(st);
            return false;
        }
    }
}

// Waits for the phase with the given parity to complete. Bounded. The first
// test is inline: on the issue paths the phase is usually complete already,
// and a call per k-block costs the single issuing thread measurable time.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const DevStatus& st) {
    return mbar_try_wait(bar, parity) || mbar_wait_slow(bar, parity, st);
}

// -------------------------------------------------------------------- TMA

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* m) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* m, uint32_t bar,
                                            int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// ------------------------------------------------------------- clusters

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// All threads of every CTA in the cluster.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The shared::cluster address of the same variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t smem_addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
    return r;
}

// 16 bytes into the shared memory of a CTA of the cluster (a shared::cluster
// address).
__device__ __forceinline__ void st_cluster_v4(uint32_t cluster_addr, int a, int b, int c, int d) {
    asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(cluster_addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

// Arrive on an mbarrier that may live in another CTA of the cluster.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// TMA load into this CTA's shared memory whose completion is signalled on an
// mbarrier of either CTA of the pair (the leader's, for paired MMAs).
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* m, uint32_t cluster_bar, int c0,
                                                 int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(cluster_bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// ---------------------------------------------------------------- tcgen05

// TMEM allocation. With CG == 2 one warp of each CTA of the pair executes
// these together and both receive the same address.
template <int CG>
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    if constexpr (CG == 1)
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                     : "memory");
    else
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                     : "memory");
}

template <int CG>
__device__ __forceinline__ void tmem_relinquish() {
    if constexpr (CG == 1)
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    else
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

template <int CG>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    if constexpr (CG == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
    else
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrives once on `bar` (this CTA) when all earlier tcgen05 async ops of this
// thread end.
template <int CG>
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    if constexpr (CG == 1)
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                     : "memory");
    else
        asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                     : "memory");
}

// The same, arriving on the mbarrier at this offset in every CTA of `mask`
// (cluster ranks).
__device__ __forceinline__ void tc_commit_pair(uint32_t bar, uint16_t mask = 3) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
        "h"(mask)
        : "memory");
}

// D(tmem) (+)= A(smem) * B(smem)^T, fp16 inputs, fp32 accumulator. With CG == 2
// the leader CTA issues it for the pair: A and B halves come from both CTAs'
// shared memory at the same offsets, each CTA's TMEM receives its M/2 rows.
template <int CG>
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                           uint32_t accumulate) {
    if constexpr (CG == 1)
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
            : "memory");
}

// Each thread of the warp reads its TMEM lane (row), 32 consecutive columns.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05 format): K-major operand staged by
// a TMA load with 128-byte swizzle, rows of 128 bytes (64 fp16), 8-row groups
// 1024 bytes apart. The tile base must be 1024-byte aligned.
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t smem_addr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);  // start address
    d |= static_cast<uint64_t>(1) << 16;                       // leading byte offset (unused)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;               // stride byte offset
    d |= static_cast<uint64_t>(1) << 46;                       // descriptor version
    d |= static_cast<uint64_t>(2) << 61;                       // 128-byte swizzle
    return d;
}

// Shared-memory matrix descriptor for an MN-major operand staged by TMA loads
// of 64 (M or N) x 64 (K) boxes with 128-byte swizzle: each K row is 128
// bytes (64 fp16 along M/N), 8-row K groups are 1024 bytes apart (stride byte
// offset) and consecutive 64-wide M/N blocks are `mn_block_bytes` apart
// (leading byte offset). The tile base must be 1024-byte aligned.
__device__ __forceinline__ uint64_t sw128_mnmajor_desc(uint32_t smem_addr, uint32_t mn_block_bytes) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);        // start address
    d |= static_cast<uint64_t>((mn_block_bytes >> 4) & 0x3FFFu) << 16;  // leading byte offset
    d |= static_cast<uint64_t>(1024 >> 4) << 32;                     // stride byte offset
    d |= static_cast<uint64_t>(1) << 46;                             // descriptor version
    d |= static_cast<uint64_t>(2) << 61;                             // 128-byte swizzle
    return d;
}

// Instruction descriptor of tcgen05.mma kind::f16: fp16 A and B, fp32
// accumulator, M x N tile; a_mn / b_mn select MN-major (transposed) operands.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N, uint32_t a_mn = 0, uint32_t b_mn = 0) {
    return (1u << 4)                                 // D format: f32
           | (0u << 7) | (0u << 10)                  // A, B format: f16
           | (a_mn << 15) | (b_mn << 16)             // A, B major-ness (0 = K-major)
           | (static_cast<uint32_t>(N >> 3) << 17)   // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);  // M / 16
}

// ------------------------------------------- cross-CTA ordering through global memory

// Orders this thread's completed bulk (async-proxy) global writes before its
// subsequent generic operations, e.g. a release that publishes them.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ void red_release_add(int* addr, int v) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ int ld_acquire(const int* addr) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(addr) : "memory");
    return v;
}

// Shared-memory fetch-and-add with acquire-release semantics at CTA scope.
__device__ __forceinline__ uint32_t atom_add_acqrel_cta(uint32_t smem_addr, uint32_t v) {
    uint32_t old;
    asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(smem_addr), "r"(v) : "memory");
    return old;
}

// Spins until *addr >= target (acquire). Bounded like the mbarrier waits.
static __device__ __noinline__ bool wait_counter(const int* addr, int target, const DevStatus& st) {
    if (ld_acquire(addr) >= target) return true;
    const uint64_t t0 = globaltimer();
    while (true) {
        for (int i = 0; i < 32; ++i) {
            if (ld_acquire(addr) >= target) return true;
            __nanosleep(64);
        }
        if (call_aborted(st)) return false;
        if (globaltimer() - t0 > st.limit_ns) {
            raise_timeout(st);
            return false;
        }
    }
}

// ------------------------------------------------- programmatic dependent launch

// Blocks until the grids this one depends on have completed and their memory
// is visible (a no-op when the launch carried no programmatic dependency).
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Lets the next grid in the stream start launching (its CTAs still wait for
// this grid in grid_dependency_wait before touching dependent data).
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------ small helpers

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
    asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

// Four 8 x 8 b16 matrices from shared memory, transposed (one row address per thread).
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                                  uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}

// Four 8 x 8 b16 matrices to shared memory (one row address per thread).
__device__ __forceinline__ void stmatrix_x4(uint32_t addr, uint32_t r0, uint32_t r1, uint32_t r2, uint32_t r3) {
    asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(r0), "r"(r1),
                 "r"(r2), "r"(r3)
                 : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ uint16_t ld_shared_u16(uint32_t addr) {
    uint16_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr) : "memory");
    return v;
}

}  // namespace gns
