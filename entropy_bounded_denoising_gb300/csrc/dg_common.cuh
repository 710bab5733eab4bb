// dg_common.cuh -- device helpers shared by the libdg kernels (sm_103a only).
//
// Philox-4x32-10 follows Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as
// 1, 2, 3" (SC'11).  The PTX wrappers cover mbarriers, bulk / tensor copies (TMA) and the
// fifth-generation tensor core (tcgen05) with its tensor memory (TMEM).  Every wait is
// bounded: when a bound expires the caller sets DG_DEV_TIMEOUT in the status word and
// unwinds instead of spinning forever.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dg.h"

#define DG_DEVINL __device__ __forceinline__

// ------------------------------------------------------------------ status word
namespace dg {

DG_DEVINL void raise_status(unsigned* status, unsigned bits) {
    if (status) atomicOr(status, bits);
}

// Programmatic dependent launch.  Kernels of the library are launched so that they may start
// while the previous kernel on the stream drains; each calls pdl_wait() before its first
// global-memory access (and before any early exit, so that completion stays ordered along the
// stream), then pdl_release() to let the next kernel start in turn.  Without the launch
// attribute both are no-ops.
DG_DEVINL void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
DG_DEVINL void pdl_release() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Per-canvas parameters the acceptance kernel works with (else DG_DEV_BAD_PARAM, canvas skipped).
DG_DEVINL bool canvas_params_ok(const dg_canvas_params& p, int32_t L) {
    return p.temperature > 0.f && isfinite(p.temperature) && p.k >= 1 && p.max_steps >= 1 && p.min_accept >= 0 &&
           p.min_accept <= L;
}

// ------------------------------------------------------------------ Philox-4x32-10
struct u4 { uint32_t x, y, z, w; };

constexpr uint32_t kPhiloxM0 = 0xD2511F53u;
constexpr uint32_t kPhiloxM1 = 0xCD9E8D57u;
constexpr uint32_t kPhiloxW0 = 0x9E3779B9u;
constexpr uint32_t kPhiloxW1 = 0xBB67AE85u;

// Random-number streams (counter word 3, low byte).
constexpr uint32_t kStreamGumbel = 0u;
constexpr uint32_t kStreamRenoise = 1u;
constexpr uint32_t kStreamInit = 2u;

// 32 x 32 -> 64-bit product as (lo, hi).
DG_DEVINL void mul_wide(uint32_t a, uint32_t b, uint32_t& lo, uint32_t& hi) {
    asm("{\n\t.reg .b64 t;\n\tmul.wide.u32 t, %2, %3;\n\tmov.b64 {%0, %1}, t;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(a), "r"(b));
}

// Ten rounds: each multiplies the even words, swaps halves and mixes in the round key,
// the key advancing by the Weyl constants between rounds.
DG_DEVINL u4 philox10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        uint32_t lo0, hi0, lo1, hi1;
        mul_wide(c0, kPhiloxM0, lo0, hi0);
        mul_wide(c2, kPhiloxM1, lo1, hi1);
        const uint32_t n0 = hi1 ^ c1 ^ (k0 + (uint32_t)r * kPhiloxW0);
        const uint32_t n2 = hi0 ^ c3 ^ (k1 + (uint32_t)r * kPhiloxW1);
        c1 = lo1;
        c3 = lo0;
        c0 = n0;
        c2 = n2;
    }
    return u4{c0, c1, c2, c3};
}

// Philox-4x32-10 for many counters that differ only in word 0 (the Gumbel stream of one
// position): the parts of the first two rounds that do not depend on word 0 are computed
// once.  philox10_c0(c0, philox_pre(c1, c2, c3, k0, k1)) == philox10(c0, c1, c2, c3, k0, k1).
struct PhiloxPre {
    uint32_t c3k1;  // round 1: c3 ^ k1
    uint32_t u1;    // round 2: lo(c2 * M1) ^ (k0 + W0)
    uint32_t u2;    // round 2: hi(n0 * M0) ^ (k1 + W1), n0 = hi(c2 * M1) ^ c1 ^ k0
    uint32_t w3;    // round 2: lo(n0 * M0), word 3 after the round
    uint32_t k0, k1;
};

DG_DEVINL PhiloxPre philox_pre(uint32_t c1, uint32_t c2, uint32_t c3, uint32_t k0, uint32_t k1) {
    PhiloxPre p;
    uint32_t lo1, hi1, lo0, hi0;
    mul_wide(c2, kPhiloxM1, lo1, hi1);
    const uint32_t n0 = hi1 ^ c1 ^ k0;
    mul_wide(n0, kPhiloxM0, lo0, hi0);
    p.c3k1 = c3 ^ k1;
    p.u1 = lo1 ^ (k0 + kPhiloxW0);
    p.u2 = hi0 ^ (k1 + kPhiloxW1);
    p.w3 = lo0;
    p.k0 = k0;
    p.k1 = k1;
    return p;
}

DG_DEVINL u4 philox10_c0(uint32_t c0, const PhiloxPre& p) {
    uint32_t lo0, hi0, lo1, hi1;
    mul_wide(c0, kPhiloxM0, lo0, hi0);           // round 1, word 0 product
    const uint32_t n2 = hi0 ^ p.c3k1;            // round 1, new word 2 (word 3 = lo0)
    mul_wide(n2, kPhiloxM1, lo1, hi1);           // round 2, word 2 product
    uint32_t c0r = hi1 ^ p.u1, c1r = lo1, c2r = p.u2 ^ lo0, c3r = p.w3;
#pragma unroll
    for (int r = 2; r < 10; ++r) {
        mul_wide(c0r, kPhiloxM0, lo0, hi0);
        mul_wide(c2r, kPhiloxM1, lo1, hi1);
        const uint32_t n0 = hi1 ^ c1r ^ (p.k0 + (uint32_t)r * kPhiloxW0);
        const uint32_t m2 = hi0 ^ c3r ^ (p.k1 + (uint32_t)r * kPhiloxW1);
        c1r = lo1;
        c3r = lo0;
        c0r = n0;
        c2r = m2;
    }
    return u4{c0r, c1r, c2r, c3r};
}

// Counter word 3: stream id in the low byte, bits 32..55 of the seed above it.
DG_DEVINL uint32_t ctr_word3(uint64_t seed, uint32_t stream) {
    return stream | ((uint32_t)((seed >> 32) & 0xFFFFFFu) << 8);
}

// u = (floor(w / 2^9) + 1/2) / 2^23, exact in fp32, 2^-24 <= u <= 1 - 2^-24.
DG_DEVINL float uniform_from_word(uint32_t w) {
    return __uint2float_rn((w >> 9) * 2u + 1u) * 5.9604644775390625e-8f;  // (2k + 1) / 2^24
}

// Uniform token in [0, V): floor((w0 << 32 | w1) * V / 2^64).
DG_DEVINL uint32_t token_from_words(uint32_t w0, uint32_t w1, uint32_t V) {
    const uint64_t x = ((uint64_t)w0 << 32) | w1;
    return (uint32_t)__umul64hi(x, (uint64_t)V);
}

DG_DEVINL uint32_t random_token(uint64_t seed, uint32_t request_id, uint32_t step, uint32_t position,
                                uint32_t stream, uint32_t V) {
    const u4 w = philox10(0u, position, step, ctr_word3(seed, stream), (uint32_t)seed, request_id);
    return token_from_words(w.x, w.y, V);
}

// ------------------------------------------------------------------ bounded waits
// Roughly 2^22 polls with a ~1 us suspend hint each: a few seconds at most.
constexpr uint32_t kWaitPolls = 1u << 22;

DG_DEVINL uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

DG_DEVINL void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

DG_DEVINL void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

DG_DEVINL void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

DG_DEVINL void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

DG_DEVINL void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

DG_DEVINL bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(1000u)
        : "memory");
    return ok != 0;
}

// As mbar_try_wait, acquiring at cluster scope (for arrivals released by the peer CTA).
DG_DEVINL bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(1000u)
        : "memory");
    return ok != 0;
}

DG_DEVINL bool mbar_wait_cluster(uint64_t* bar, uint32_t parity) {
    for (uint32_t i = 0; i < kWaitPolls; ++i)
        if (mbar_try_wait_cluster(bar, parity)) return true;
    return false;
}

// Shared-memory address of `p`'s counterpart in CTA `rank` of the cluster.
DG_DEVINL uint32_t mapa_shared(const void* p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}

// Arrive on an mbarrier of another CTA of the cluster, given by its cluster shared address
// (default semantics, as for a local arrive: no cluster-wide fence on the way).
DG_DEVINL void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// Returns false when the bound expired (`polls` polls; the kernels use kWaitPolls).
DG_DEVINL bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t polls = kWaitPolls) {
    for (uint32_t i = 0; i < polls; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// Whole-warp wait: lane 0 polls, the warp then synchronises (which also orders the data the
// barrier guards for the other lanes).  Keeps 31 lanes from hammering shared memory.
// Must be called by all 32 lanes, converged.  `sleep_ns` > 0 backs off between polls for
// waits that are off the critical path.
DG_DEVINL bool mbar_wait_warp(uint64_t* bar, uint32_t parity, uint32_t sleep_ns = 0, uint32_t polls = kWaitPolls) {
    int ok = 1;
    if ((threadIdx.x & 31) == 0) {
        ok = 0;
        for (uint32_t i = 0; i < polls; ++i) {
            if (mbar_try_wait(bar, parity)) {
                ok = 1;
                break;
            }
            if (sleep_ns) __nanosleep(sleep_ns);
        }
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();
    return ok != 0;
}

// ------------------------------------------------------------------ bulk copies (TMA)
// Plain bulk copy global -> shared; both addresses 16-byte aligned, bytes % 16 == 0.
DG_DEVINL void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

DG_DEVINL void tma_load_2d(void* dst, const void* tmap, int32_t c0, int32_t c1, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_u32(dst)),
        "l"(tmap), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}

DG_DEVINL void tma_load_3d(void* dst, const void* tmap, int32_t c0, int32_t c1, int32_t c2, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, "
        "%4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}

DG_DEVINL void prefetch_tmap(const void* tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// ------------------------------------------------------------------ tcgen05 / TMEM
DG_DEVINL void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {  // whole warp
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

DG_DEVINL void tmem_relinquish() {  // whole warp
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

DG_DEVINL void tmem_dealloc(uint32_t taddr, uint32_t ncols) {  // whole warp
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// The same for a CTA pair (cta_group::2): one warp of each of the two CTAs executes them
// together, and the columns are allocated in both CTAs' tensor memory.
DG_DEVINL void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {  // whole warp, both CTAs
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

DG_DEVINL void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

DG_DEVINL void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

DG_DEVINL void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
DG_DEVINL void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem], kind::f16 (bf16 inputs, fp32 accumulate), one thread.
DG_DEVINL void tc_mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// As tc_mma_f16 with A read from tensor memory (row = lane, two bf16 per 32-bit column, the
// lower K index in the low half) at `a_tmem`; B from shared memory.
DG_DEVINL void tc_mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// CTA-pair MMA (cta_group::2, issued by one thread of the pair's first CTA): M = 256 rows,
// 128 from each CTA's shared memory; each CTA supplies N/2 columns of B; D lands in both
// CTAs' tensor memory (each its own 128 rows, all N columns).
DG_DEVINL void tc_mma_f16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                               uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on the mbarrier at `bar`'s offset in every CTA of `mask` once all previously issued
// pair MMAs of this thread completed.
DG_DEVINL void tc_commit_pair_mc(uint64_t* bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(mask)
        : "memory");
}

// Arrive on an mbarrier once all previously issued tcgen05.mma of this thread completed.
DG_DEVINL void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// tmem_ld32 without its wait: several loads can be in flight before one tmem_ld_wait (the
// registers are undefined until then).
DG_DEVINL void tmem_ld32_nowait(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

DG_DEVINL void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// The wait with the registers a tmem_ld32_nowait wrote passed through it: they are undefined
// until the wait, and an operand dependency is what keeps the compiler from scheduling a use of
// them before it (a plain volatile asm orders memory and other asm, not register arithmetic).
DG_DEVINL void tmem_ld_wait_dep(uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.wait::ld.sync.aligned;"
        : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
          "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]),
          "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
          "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
        :
        : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread t of the warp gets lane (base + t).
DG_DEVINL void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
    tmem_ld_wait_dep(r);
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// The same direction: 32 lanes x 32 consecutive columns from registers (whole warp); the
// caller waits with tmem_st_wait before anything reads the columns, and before the source
// registers can be written again (the store is asynchronous).
DG_DEVINL void tmem_st32(uint32_t taddr, const float (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
        "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
        "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15])),
        "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])), "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])),
        "r"(__float_as_uint(v[20])), "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])), "r"(__float_as_uint(v[27])),
        "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])), "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
        : "memory");
}

// Raw 32-bit words, as tmem_st32.
DG_DEVINL void tmem_st32u(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
        "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
        "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
        "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}

// 32 lanes x 16 columns of raw 32-bit words (whole warp).
DG_DEVINL void tmem_st16u(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
        "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}

DG_DEVINL void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ------------------------------------------------------------------ tcgen05 descriptors
// Shared-memory matrix descriptor (tcgen05): start >> 4 in bits 0..13, leading byte offset
// >> 4 in 16..29, stride byte offset >> 4 in 32..45, version 1 in 46..47, layout in 61..63
// (2 = 128-byte swizzle, 4 = 64-byte swizzle).
DG_DEVINL uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo, int swizzle_bytes) {
    const uint64_t layout = swizzle_bytes == 128 ? 2ull : 4ull;
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (layout << 61);
}

// Instruction descriptor, kind::f16: fp32 accumulator (bit 4), bf16 A (bits 7..9 = 1) and
// B (bits 10..12 = 1), A K-major (bit 15 = 0), B major in bit 16, N >> 3 in 17..22,
// M >> 4 in 24..28.
__host__ __device__ constexpr uint32_t instr_desc(int M, int N, bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

}  // namespace dg

// ------------------------------------------------------------------ host helpers
namespace dghost {
// Device address of the status word of the current device (set up on first use).
unsigned* status_word();
// Record one kernel launch made by the library (process-wide counter).
void count_launch();
// Streaming multiprocessor count of the current device.
int sm_count();
// Map a CUDA error to a dg_status (DG_OK when err == cudaSuccess).
inline dg_status cuda_status(cudaError_t err) { return err == cudaSuccess ? DG_OK : DG_ERR_CUDA; }
// Encode a tiled tensor map (driver entry point fetched once).  Returns false on failure.
bool encode_tmap(void* tmap, int dtype_code, int rank, void* base, const uint64_t* dims,
                 const uint64_t* strides_bytes, const uint32_t* box, int swizzle_bytes);
// LM head (dg_gemm.cu): logits = bf16(hidden . W^T) for the active canvases' rows, [n][L][ld]
// bf16; with `stats` non-null also each row's softmax state per kLmTileCols-column tile, as
// 5 arrays (max, count, r, t, first column of the max) of n * L floats per tile, tile after
// tile.  `plan` needs n + 1 ints.  Enqueues 2 kernels on `stream`.
constexpr int kLmTileCols = 256;
dg_status lm_head_gemm(const uint16_t* hidden, int64_t ldh, const uint16_t* W, int64_t ldw, int64_t n, int32_t L,
                       int64_t V, int32_t d, const dg_canvas_params* params, uint16_t* logits, int64_t ld,
                       int32_t* plan, float* stats, cudaStream_t stream);
// Programmatic dependent launch on (build with -DDG_NO_PDL for plain stream order).
#ifdef DG_NO_PDL
constexpr bool kPdl = false;
#else
constexpr bool kPdl = true;
#endif
// Launch with programmatic stream serialisation (the kernel calls dg::pdl_wait first).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = kPdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}
}  // namespace dghost
