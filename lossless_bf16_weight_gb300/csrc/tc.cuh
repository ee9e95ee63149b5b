// Blackwell tensor-core plumbing (sm_100 family, inline PTX): mbarriers,
// tensor-memory allocation, shared-memory matrix descriptors, tcgen05.mma of
// kind::f16 with BF16 operands and an fp32 accumulator in tensor memory, and
// tcgen05.ld for the epilogue.
//
// Operand layout used throughout: K-major tiles of 64 BF16 (128 bytes) per
// row, stored in 8-row x 128-byte atoms (1024 bytes) with the 128-byte
// swizzle: the 16-byte chunk c of row r sits at chunk position c ^ (r % 8)
// of that row.  Consecutive 8-row atoms are 1024 bytes apart.
//
// Every wait is bounded: a wait that runs out sets a flag in the caller's
// status word and returns false, so a kernel never spins forever.
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

namespace uw {

constexpr uint32_t kWaitTries = 1u << 22;  // try_wait calls before a wait gives up

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}

// Make barrier initialisation visible to the other threads and to the
// asynchronous proxy (tensor-core commits); follow with a CTA barrier.
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}

// A waiting thread is suspended for at most kWaitHintNs per try_wait: with
// the system's own limit, hand-offs between the warps of the tensor-core
// kernel (producer -> MMA -> stage reuse) took measurably longer (batch 16
// on the 14336 x 4096 gate matrix: fused 49.0 -> 47.4 us, uncompressed
// 26.1 -> 24.9 us; any hint from 20 to 1000 ns did the same).
constexpr uint32_t kWaitHintNs = 20;

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(bar), "r"(parity), "n"(kWaitHintNs) : "memory");
    return ok != 0;
}

// Wait until the phase with the given parity has completed; false (and
// `flag` set in *status) if it did not within `tries` attempts.
__device__ __forceinline__ bool mbar_wait_tries(uint32_t bar, uint32_t parity, uint32_t *status, uint32_t flag,
                                                uint32_t tries) {
    for (uint32_t i = 0; i < tries; i++)
        if (mbar_try_wait(bar, parity))
            return true;
    atomicOr(status, flag);
    return false;
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t *status, uint32_t flag) {
    return mbar_wait_tries(bar, parity, status, flag, kWaitTries);
}

// Arrive on the mbarrier and add `bytes` to the transaction count its
// current phase waits for.
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(bar), "r"(bytes) : "memory");
}

// One box of a 2-D tensor map (kernel-parameter tensor map at `tmap`) into
// shared memory at `dst`, completion counted on the mbarrier; coordinate x0
// is the inner one (its byte offset must be a multiple of 16).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *tmap, int x0, int x1, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x0), "r"(x1), "r"(bar) : "memory");
}

// One box from shared memory at `src` to a 2-D tensor (kernel-parameter
// tensor map at `tmap`) at coordinates (x0, x1), in the calling thread's
// bulk group (x0's byte offset must be a multiple of 16; elements outside
// the tensor are not written).  Follow with tma_store_commit, and wait with
// tma_store_wait_read before the source is written again.
__device__ __forceinline__ void tma_store_2d(const void *tmap, int x0, int x1, uint32_t src) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];"
                 :: "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x0), "r"(x1), "r"(src) : "memory");
}
__device__ __forceinline__ void tma_store_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// The thread's committed stores have finished reading their shared sources.
__device__ __forceinline__ void tma_store_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// The thread's committed stores are complete.
__device__ __forceinline__ void tma_store_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Bulk copy global -> shared by the copy engine; completion is counted on
// the mbarrier.  Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 :: "r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

// Generic-proxy writes to shared memory (st.shared, cp.async) must be made
// visible to the tensor cores' asynchronous proxy before they read them.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// One full warp: allocate `ncols` tensor-memory columns (a power of two,
// 32..512); the base address is written to shared memory at `slot`.
__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" :: "r"(slot), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols) : "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row atoms
// 1024 bytes apart.  Fields: start address >> 4 (bits 0..13), leading
// byte offset >> 4 (16..29, unused for this layout: 1), stride byte offset
// >> 4 (32..45), the fixed value 1 at bits 46..48, swizzle mode 2 (128-byte)
// at bits 61..63.  `addr` is a shared address; its atom must be
// 1024-aligned, and it may be advanced by 32 bytes per 16-element K slice.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t addr) {
    return uint64_t((addr & 0x3FFFFu) >> 4) | (uint64_t(1) << 16) | (uint64_t(1024 >> 4) << 32) |
           (uint64_t(1) << 46) | (uint64_t(2) << 61);
}

// Instruction descriptor for kind::f16: fp32 accumulator (bits 4..5 = 1),
// A and B BF16 (bits 7..9 = 1, 10..12 = 1), both K-major (bits 15, 16 = 0),
// N >> 3 at bits 17..22, M >> 4 at bits 24..28.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T for one K slice of 16; issued by one thread.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        :: "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(uint32_t(accumulate)) : "memory");
}

// Arrive once on the mbarrier when every tcgen05.mma issued so far by this
// thread has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" :: "r"(bar)
                 : "memory");
}

// 32 lanes x 16 consecutive fp32 columns: thread t of the warp gets lane
// (taddr >> 16) + t.  The warp may only touch its own quarter of the lanes
// (warp index % 4).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 16-byte global -> shared copy; `bytes` = 0 fills the destination with
// zeros and reads nothing.
__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void *src, uint32_t bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" :: "r"(dst), "l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" :: "r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

// Byte offset of the 16-byte chunk c (elements 8c..8c+7) of row r inside a
// swizzled K-major tile of 64-element rows.
__host__ __device__ constexpr uint32_t sw128_offset(uint32_t r, uint32_t c) {
    return (r >> 3) * 1024u + (r & 7u) * 128u + ((c ^ (r & 7u)) << 4);
}

}  // namespace uw
