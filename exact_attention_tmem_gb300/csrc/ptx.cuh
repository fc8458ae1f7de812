// ptx.cuh — inline-PTX building blocks for sm_103a kernels: mbarriers with bounded
// waits, tensor-memory-access (TMA) tile loads, and the tcgen05 family (tensor-memory
// allocation, MMA issue and commit, tensor-memory loads and stores).
//
// Encodings follow the PTX ISA for tcgen05 (shared-memory matrix descriptor and the
// kind::f16 / kind::tf32 instruction descriptor).  Every wait in this file is bounded:
// a wait that exceeds its time limit sets the CTA's abort flag and the device status
// word instead of spinning forever, and every role then winds down.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

namespace fa {

// ---------------------------------------------------------------------------------
// bounded waits
// ---------------------------------------------------------------------------------
// Device status word layout (the word itself lives in the host library's module and
// reaches kernels as a pointer): word 0 bit 0 = some wait timed out; word 1 = the
// site id of the first wait that gave up.
enum : unsigned int { kStatusTimeout = 1u };

// Upper bound for any single wait inside a kernel.  Legitimate waits last
// microseconds; one second means the pipeline is broken.
constexpr unsigned long long kWaitLimitNs = 1000000000ull;
// Longest sleep of one polling step inside a wait (the thread wakes when the phase
// completes); well below the limit so that the abort flag and clock are rechecked.
constexpr uint32_t kWaitSleepNs = 20000;

// Per-CTA context of the bounded waits: the shared abort flag that makes every role
// wind down once one wait has given up, and the device status word.
struct WaitCtx {
    volatile int *abort_flag;
    unsigned int *status;
};

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------------------------
// launch order of attention work items
// ---------------------------------------------------------------------------------
// A grid of num_heads x per_head CTAs, where rank 0 of a head is its longest walk
// (causal work) is taken in groups of heads, rank-major inside a group: rank 0 of every
// head of the group, then rank 1, ...  The longest walks of a group start first, so the
// last CTAs of the grid are short ones (no long tail on a few SMs), while the group's
// heads alone are in flight and their tiles stay in L2.  A group has 8 heads, or more
// when a head has few work items, so that it holds at least 128 CTAs.
__host__ __device__ __forceinline__ int heavy_first_group(int per_head) {
    const int g = (128 + per_head - 1) / per_head;
    return g > 8 ? g : 8;
}
__host__ __device__ __forceinline__ void heavy_first_item(int idx, int per_head, int num_heads, int &head,
                                                          int &rank) {
    const int group = heavy_first_group(per_head);
    const int per_group = group * per_head;
    const int g = idx / per_group;
    const int r = idx - g * per_group;
    const int rest = num_heads - g * group;
    const int heads_here = rest < group ? rest : group;
    rank = r / heads_here;
    head = g * group + r % heads_here;
}
// The same order for a grid of exactly num_heads x per_head CTAs, one item each.
__device__ __forceinline__ void heavy_first_order(int idx, int per_head, int &head, int &rank) {
    heavy_first_item(idx, per_head, static_cast<int>(gridDim.x) / per_head, head, rank);
}

// ---------------------------------------------------------------------------------
// programmatic dependent launch
// ---------------------------------------------------------------------------------
// Waits for the grids this one depends on (programmatic dependent launch); a no-op for
// a normal launch.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Lets a grid launched after this one with programmatic serialization start now.
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the async proxy (TMA, tcgen05.commit).
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

// try_wait with a suspend-time hint: the thread sleeps in the barrier unit (issuing
// nothing) until the phase completes or about `ns` nanoseconds pass.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}

// Slow path of mbar_wait: keeps polling until the phase completes, the CTA's abort
// flag is raised by another thread, or the time limit passes (then raises the flag
// and records `site` in the device status word).
// With `honour_abort` false the wait ignores the abort flag (used to drain copies
// still in flight before a CTA exits), but it is still time-limited.
static __device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, WaitCtx ctx, int site,
                                            bool honour_abort) {
    const unsigned long long t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait_sleep(bar, parity, kWaitSleepNs)) return true;
        if ((it & 31u) == 0) {
            if (honour_abort && *ctx.abort_flag) return false;
            if (globaltimer_ns() - t0 > kWaitLimitNs) {
                *ctx.abort_flag = 1;
                if (atomicOr(&ctx.status[0], kStatusTimeout) == 0u) ctx.status[1] = (unsigned)site;
                return false;
            }
        }
    }
}

// Waits until the barrier phase with parity `parity` has completed.  Returns false
// if the wait gave up: the CTA's abort flag was raised, or the time limit passed.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, WaitCtx ctx, int site) {
    if (mbar_try_wait(bar, parity)) return true;
    return mbar_wait_slow(bar, parity, ctx, site, true);
}

// Same, but not cut short by the abort flag (still time-limited).
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity, WaitCtx ctx, int site) {
    if (mbar_try_wait(bar, parity)) return true;
    return mbar_wait_slow(bar, parity, ctx, site, false);
}

// ---------------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor) and bulk copies
// ---------------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 3-D tiled load of one box into shared memory; completion is signalled on `bar`
// as transaction bytes.  Coordinates are element indices (x innermost).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, uint32_t bar, int x,
                                            int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
        : "memory");
}

// Plain bulk copy global -> shared (both 16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
        : "memory");
}

// 3-D tiled bulk reduction shared -> global: the box at (x, y, z) is added (fp32 add)
// element-wise into global memory; elements outside the tensor are skipped.  Completion
// is tracked with bulk async-groups (bulk_commit_group / bulk_wait_group*).
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap *map, uint32_t src, int x, int y, int z) {
    asm volatile(
        "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(src), "r"(x), "r"(y), "r"(z)
        : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until the sources of all but the most recently committed bulk group have been read.
__device__ __forceinline__ void bulk_wait_group_read1() {
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
// Waits until the sources of every committed bulk group have been read: the shared
// memory may then be reused or released.  The global writes complete on their own and
// are visible to any grid that waits for this one to finish.
__device__ __forceinline__ void bulk_wait_group_read0() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Barrier over `count` threads (a multiple of 32) with hardware barrier `id` (1..15).
__device__ __forceinline__ void named_barrier_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Barrier over `count` threads that also returns the AND of `pred` over them: used to
// make a give-up decision uniform before a group enters further named barriers.
__device__ __forceinline__ bool named_barrier_and(int id, int count, bool pred) {
    uint32_t out;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %3, 0;\n\t"
        "bar.red.and.pred p, %1, %2, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(out)
        : "r"(id), "r"(count), "r"(pred ? 1u : 0u)
        : "memory");
    return out != 0;
}

// Orders this thread's generic-proxy shared-memory writes before later async-proxy
// reads (tcgen05.mma operands written with st.shared).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------------
// tcgen05: tensor memory allocation
// ---------------------------------------------------------------------------------
// Whole-warp operations.  The allocated base address is written to shared memory.
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ---------------------------------------------------------------------------------
// tcgen05: descriptors
// ---------------------------------------------------------------------------------
// Shared-memory matrix descriptor, 128-byte swizzle.
//   bits  0-13  start address >> 4
//   bits 16-29  leading-dimension byte offset >> 4
//   bits 32-45  stride-dimension byte offset >> 4
//   bits 46-48  fixed 0b001
//   bits 49-51  base offset (0: every operand tile starts on a 1024-byte boundary)
//   bit  52     LBO mode (0: relative)
//   bits 61-63  swizzle mode (2: 128-byte)
// K-major operand: rows of 128 bytes, 8-row groups of 1024 bytes; SBO = 1024, LBO
// unused.  Stepping K inside the 128-byte row moves the start address.
// MN-major operand: 128-byte rows run along M (or N), one row per K index; SBO = 1024
// (next 8 K rows), LBO = distance between 64-element (128-byte) column blocks.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// Instruction descriptor for kind::f16 (ab_format 1 = bf16) and kind::tf32
// (ab_format 2), fp32 accumulator.
//   bits 4-5 D format (1 = f32); 7-9 A format; 10-12 B format; 15 A major (1 = MN);
//   16 B major (1 = MN); 17-22 N >> 3; 24-28 M >> 4.
__host__ __device__ constexpr uint32_t make_idesc(uint32_t ab_format, int M, int N, bool a_mn_major,
                                                  bool b_mn_major) {
    return (1u << 4) | (ab_format << 7) | (ab_format << 10) | ((a_mn_major ? 1u : 0u) << 15) |
           ((b_mn_major ? 1u : 0u) << 16) | ((static_cast<uint32_t>(N) >> 3) << 17) |
           ((static_cast<uint32_t>(M) >> 4) << 24);
}
constexpr uint32_t kFormatBF16 = 1;
constexpr uint32_t kFormatTF32 = 2;
constexpr uint32_t kFormatE4M3 = 0;   // kind::f8f6f4 operand format

// ---------------------------------------------------------------------------------
// tcgen05: MMA issue (lane 0 of the calling warp) and commit
// ---------------------------------------------------------------------------------
// Warp-collective forms: the whole warp executes the call (so descriptors and
// addresses stay warp-uniform and the issuing code stays short) and lane 0 alone
// issues the instruction.  The commit must come from the same lane as the MMAs.
template <bool kTF32 = false>
__device__ __forceinline__ void umma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
    if constexpr (kTF32) {
        asm volatile(
            "{\n\t.reg .pred p, e;\n\t.reg .b32 l;\n\tmov.u32 l, %%laneid;\n\tsetp.eq.u32 e, l, 0;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
            : "memory");
    } else {
        asm volatile(
            "{\n\t.reg .pred p, e;\n\t.reg .b32 l;\n\tmov.u32 l, %%laneid;\n\tsetp.eq.u32 e, l, 0;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
            : "memory");
    }
}
template <bool kTF32 = false>
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
    if constexpr (kTF32) {
        asm volatile(
            "{\n\t.reg .pred p, e;\n\t.reg .b32 l;\n\tmov.u32 l, %%laneid;\n\tsetp.eq.u32 e, l, 0;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
            "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
            : "memory");
    } else {
        asm volatile(
            "{\n\t.reg .pred p, e;\n\t.reg .b32 l;\n\tmov.u32 l, %%laneid;\n\tsetp.eq.u32 e, l, 0;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
            "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
            : "memory");
    }
}
// Whole bf16 products issued from one asm block (warp-collective, lane 0 issues): the
// K steps' descriptors come in as arrays (see sdesc_step), the first step accumulates
// only if `accumulate` is non-zero, the rest always do.  TS forms step the A operand by
// 8 tensor-memory columns (16 bf16 K elements) per step.  Fewer instructions per
// product than one call per step, which matters because the MMA warp shares its
// sub-partition with softmax warps.
__device__ __forceinline__ void umma_f16_ss_x4(uint32_t d_tmem, const uint64_t (&a)[4], const uint64_t (&b)[4],
                                                uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, t, e;\n\t.reg .b32 l;\n\tmov.u32 l, %%laneid;\n\tsetp.eq.u32 e, l, 0;\n\t"
        "setp.ne.b32 p, %2, 0;\n\tsetp.eq.u32 t, l, l;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %7, %1, p;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %4, %8, %1, t;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %5, %9, %1, t;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %6, %10, %1, t;\n\t"
        "}"
        ::"r"(d_tmem), "r"(idesc), "r"(accumulate), "l"(a[0]), "l"(a[1]), "l"(a[2]), "l"(a[3]), "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3])
        : "memory");
}
__device__ __forceinline__ void umma_f16_ss_x8(uint32_t d_tmem, const uint64_t (&a)[8], const uint64_t (&b)[8],
                                                uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, t, e;\n\t.reg .b32 l;\n\tmov.u32 l, %%laneid;\n\tsetp.eq.u32 e, l, 0;\n\t"
        "setp.ne.b32 p, %2, 0;\n\tsetp.eq.u32 t, l, l;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %11, %1, p;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %4, %12, %1, t;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %5, %13, %1, t;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %6, %14, %1, t;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %7, %15, %1, t;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %8, %16, %1, t;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %9, %17, %1, t;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %10, %18, %1, t;\n\t"
        "}"
        ::"r"(d_tmem), "r"(idesc), "r"(accumulate), "l"(a[0]), "l"(a[1]), "l"(a[2]), "l"(a[3]), "l"(a[4]), "l"(a[5]), "l"(a[6]), "l"(a[7]), "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]), "l"(b[4]), "l"(b[5]), "l"(b[6]), "l"(b[7])
        : "memory");
}
__device__ __forceinline__ void umma_f16_ts_x8(uint32_t d_tmem, uint32_t a_tmem, const uint64_t (&b)[8],
                                                uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, t, e;\n\t.reg .b32 l, ta;\n\tmov.u32 l, %%laneid;\n\tsetp.eq.u32 e, l, 0;\n\t"
        "setp.ne.b32 p, %3, 0;\n\tsetp.eq.u32 t, l, l;\n\t"
        "add.u32 ta, %1, 0;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], %4, %2, p;\n\t"
        "add.u32 ta, %1, 8;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], %5, %2, t;\n\t"
        "add.u32 ta, %1, 16;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], %6, %2, t;\n\t"
        "add.u32 ta, %1, 24;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], %7, %2, t;\n\t"
        "add.u32 ta, %1, 32;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], %8, %2, t;\n\t"
        "add.u32 ta, %1, 40;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], %9, %2, t;\n\t"
        "add.u32 ta, %1, 48;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], %10, %2, t;\n\t"
        "add.u32 ta, %1, 56;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], %11, %2, t;\n\t"
        "}"
        ::"r"(d_tmem), "r"(a_tmem), "r"(idesc), "r"(accumulate), "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]), "l"(b[4]), "l"(b[5]), "l"(b[6]), "l"(b[7])
        : "memory");
}

__device__ __forceinline__ void umma_f8_ss_x4(uint32_t d_tmem, const uint64_t (&a)[4], const uint64_t (&b)[4],
                                                uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, t, e;\n\t.reg .b32 l;\n\tmov.u32 l, %%laneid;\n\tsetp.eq.u32 e, l, 0;\n\t"
        "setp.ne.b32 p, %2, 0;\n\tsetp.eq.u32 t, l, l;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %3, %7, %1, p;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %4, %8, %1, t;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %5, %9, %1, t;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %6, %10, %1, t;\n\t"
        "}"
        ::"r"(d_tmem), "r"(idesc), "r"(accumulate), "l"(a[0]), "l"(a[1]), "l"(a[2]), "l"(a[3]), "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3])
        : "memory");
}
__device__ __forceinline__ void umma_f8_ts_x4(uint32_t d_tmem, uint32_t a_tmem, const uint64_t (&b)[4],
                                                uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, t, e;\n\t.reg .b32 l, ta;\n\tmov.u32 l, %%laneid;\n\tsetp.eq.u32 e, l, 0;\n\t"
        "setp.ne.b32 p, %3, 0;\n\tsetp.eq.u32 t, l, l;\n\t"
        "add.u32 ta, %1, 0;\n\t@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [ta], %4, %2, p;\n\t"
        "add.u32 ta, %1, 8;\n\t@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [ta], %5, %2, t;\n\t"
        "add.u32 ta, %1, 16;\n\t@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [ta], %6, %2, t;\n\t"
        "add.u32 ta, %1, 24;\n\t@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [ta], %7, %2, t;\n\t"
        "}"
        ::"r"(d_tmem), "r"(a_tmem), "r"(idesc), "r"(accumulate), "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3])
        : "memory");
}

// Descriptor `desc` with its start-address field (16-byte units, low 14 bits) advanced
// by `bytes`; shared addresses stay below 256 KB, so no carry leaves the field.
__device__ __forceinline__ uint64_t sdesc_step(uint64_t desc, uint32_t bytes) {
    return (desc & 0xFFFFFFFF00000000ull) | static_cast<uint32_t>(static_cast<uint32_t>(desc) + (bytes >> 4));
}

__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t.reg .b32 l;\n\tmov.u32 l, %%laneid;\n\tsetp.eq.u32 e, l, 0;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
        : "memory");
}

// Four fp32 values from shared memory (16-byte aligned shared-window address).  The asm
// is volatile so that it stays after the barrier wait that made the data visible.
__device__ __forceinline__ float4 lds_f4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
    return v;
}

// ---------------------------------------------------------------------------------
// small math helpers
// ---------------------------------------------------------------------------------
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Four fp32 values to e4m3 (round to nearest even, saturating at +-448), packed with
// a in the lowest byte: the element order of an 8-bit MMA operand row.
__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
    uint32_t lo, hi;
    asm("{\n\t.reg .b16 t;\n\tcvt.rn.satfinite.e4m3x2.f32 t, %2, %1;\n\tcvt.u32.u16 %0, t;\n\t}"
        : "=r"(lo) : "f"(a), "f"(b));
    asm("{\n\t.reg .b16 t;\n\tcvt.rn.satfinite.e4m3x2.f32 t, %2, %1;\n\tcvt.u32.u16 %0, t;\n\t}"
        : "=r"(hi) : "f"(c), "f"(d));
    return lo | (hi << 16);
}

// Packed fp32x2 arithmetic (one instruction for two lanes of work).
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mov.b64 rc, {%6, %7};\n\tfma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "sub.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
// Three-input maximum.
__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Two floats to packed bf16x2: `lo` in bits 0-15, `hi` in bits 16-31.
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// ---------------------------------------------------------------------------------
// tcgen05: tensor memory <-> registers (each thread owns one TMEM lane = one row)
// ---------------------------------------------------------------------------------
// tcgen05.ld, shape 32x32b, 32 repetitions: thread t of the warp receives 32 consecutive
// 32-bit columns of TMEM lane (warp's lane quarter base + t), starting at column taddr.
// The wait is in the same asm statement so the registers are valid when it returns.
__device__ __forceinline__ void tmem_ld_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// tcgen05.ld, shape 32x32b, 64 repetitions: thread t of the warp receives 64 consecutive
// 32-bit columns of TMEM lane (warp's lane quarter base + t), starting at column taddr.
// The wait is in the same asm statement so the registers are valid when it returns.
__device__ __forceinline__ void tmem_ld_x64(uint32_t taddr, uint32_t (&r)[64]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
        : "r"(taddr)
        : "memory");
}

// tcgen05.ld, shape 32x32b, 128 repetitions: thread t of the warp receives 128 consecutive
// 32-bit columns of TMEM lane (warp's lane quarter base + t), starting at column taddr.
// The wait is in the same asm statement so the registers are valid when it returns.
__device__ __forceinline__ void tmem_ld_x128(uint32_t taddr, uint32_t (&r)[128]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x128.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, %64, %65, %66, %67, %68, %69, %70, %71, %72, %73, %74, %75, %76, %77, %78, %79, %80, %81, %82, %83, %84, %85, %86, %87, %88, %89, %90, %91, %92, %93, %94, %95, %96, %97, %98, %99, %100, %101, %102, %103, %104, %105, %106, %107, %108, %109, %110, %111, %112, %113, %114, %115, %116, %117, %118, %119, %120, %121, %122, %123, %124, %125, %126, %127}, [%128];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]), "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]), "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]), "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]), "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]), "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]), "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]), "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]), "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
        : "r"(taddr)
        : "memory");
}

// tcgen05.st, shape 32x32b, 32 repetitions (the mirror of tmem_ld_x32); waits for completion.
__device__ __forceinline__ void tmem_st_x32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};\n\t"
        "tcgen05.wait::st.sync.aligned;"
        :
        : "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

// tcgen05.st, shape 32x32b, 64 repetitions (the mirror of tmem_ld_x64); waits for completion.
__device__ __forceinline__ void tmem_st_x64(uint32_t taddr, const uint32_t (&r)[64]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, %64};\n\t"
        "tcgen05.wait::st.sync.aligned;"
        :
        : "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]), "r"(r[32]), "r"(r[33]), "r"(r[34]), "r"(r[35]), "r"(r[36]), "r"(r[37]), "r"(r[38]), "r"(r[39]), "r"(r[40]), "r"(r[41]), "r"(r[42]), "r"(r[43]), "r"(r[44]), "r"(r[45]), "r"(r[46]), "r"(r[47]), "r"(r[48]), "r"(r[49]), "r"(r[50]), "r"(r[51]), "r"(r[52]), "r"(r[53]), "r"(r[54]), "r"(r[55]), "r"(r[56]), "r"(r[57]), "r"(r[58]), "r"(r[59]), "r"(r[60]), "r"(r[61]), "r"(r[62]), "r"(r[63])
        : "memory");
}

// tcgen05.st, shape 32x32b, 128 repetitions (the mirror of tmem_ld_x128); waits for completion.
__device__ __forceinline__ void tmem_st_x128(uint32_t taddr, const uint32_t (&r)[128]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x128.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, %64, %65, %66, %67, %68, %69, %70, %71, %72, %73, %74, %75, %76, %77, %78, %79, %80, %81, %82, %83, %84, %85, %86, %87, %88, %89, %90, %91, %92, %93, %94, %95, %96, %97, %98, %99, %100, %101, %102, %103, %104, %105, %106, %107, %108, %109, %110, %111, %112, %113, %114, %115, %116, %117, %118, %119, %120, %121, %122, %123, %124, %125, %126, %127, %128};\n\t"
        "tcgen05.wait::st.sync.aligned;"
        :
        : "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]), "r"(r[32]), "r"(r[33]), "r"(r[34]), "r"(r[35]), "r"(r[36]), "r"(r[37]), "r"(r[38]), "r"(r[39]), "r"(r[40]), "r"(r[41]), "r"(r[42]), "r"(r[43]), "r"(r[44]), "r"(r[45]), "r"(r[46]), "r"(r[47]), "r"(r[48]), "r"(r[49]), "r"(r[50]), "r"(r[51]), "r"(r[52]), "r"(r[53]), "r"(r[54]), "r"(r[55]), "r"(r[56]), "r"(r[57]), "r"(r[58]), "r"(r[59]), "r"(r[60]), "r"(r[61]), "r"(r[62]), "r"(r[63]), "r"(r[64]), "r"(r[65]), "r"(r[66]), "r"(r[67]), "r"(r[68]), "r"(r[69]), "r"(r[70]), "r"(r[71]), "r"(r[72]), "r"(r[73]), "r"(r[74]), "r"(r[75]), "r"(r[76]), "r"(r[77]), "r"(r[78]), "r"(r[79]), "r"(r[80]), "r"(r[81]), "r"(r[82]), "r"(r[83]), "r"(r[84]), "r"(r[85]), "r"(r[86]), "r"(r[87]), "r"(r[88]), "r"(r[89]), "r"(r[90]), "r"(r[91]), "r"(r[92]), "r"(r[93]), "r"(r[94]), "r"(r[95]), "r"(r[96]), "r"(r[97]), "r"(r[98]), "r"(r[99]), "r"(r[100]), "r"(r[101]), "r"(r[102]), "r"(r[103]), "r"(r[104]), "r"(r[105]), "r"(r[106]), "r"(r[107]), "r"(r[108]), "r"(r[109]), "r"(r[110]), "r"(r[111]), "r"(r[112]), "r"(r[113]), "r"(r[114]), "r"(r[115]), "r"(r[116]), "r"(r[117]), "r"(r[118]), "r"(r[119]), "r"(r[120]), "r"(r[121]), "r"(r[122]), "r"(r[123]), "r"(r[124]), "r"(r[125]), "r"(r[126]), "r"(r[127])
        : "memory");
}

// tcgen05.ld (32x32b, 32 repetitions) without waiting.  The registers are not valid
// until tmem_wait_ld_fence() has run on the same array: that wait takes them as in-out
// operands, so no use of them can be scheduled before it.
__device__ __forceinline__ void tmem_ld_x32_nowait(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr)
                 : "memory");
}
__device__ __forceinline__ void tmem_wait_ld_fence(uint32_t (&r)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]) : : "memory");
}

}  // namespace fa
