// Device-side building blocks shared by the GEMM kernels: inline-PTX wrappers for
// mbarriers, the tensor memory accelerator (TMA), tcgen05 MMAs and tensor memory, and
// the bounded waits. Every wait gives up after the call's timeout, records
// UB_ERR_TIMEOUT and publishes the call's epoch in the abort word; nothing traps.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "ub_internal.h"

namespace ubk {
namespace {

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
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

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int x, int y)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
        : "memory");
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, uint32_t src, int x, int y)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(x), "r"(y)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void bulk_wait_read()
{
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void fence_proxy_async_shared()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Programmatic dependent launch. `pdl_wait` blocks until the grid before this one has
// completed and its memory is visible; `pdl_trigger` lets the next kernel on the stream
// start launching once every CTA of this grid has reached it (all of them resident, so
// the next grid's CTAs can only take SMs that are free). Without the launch attribute
// both are no-ops. Every kernel here runs its prologue (barriers, TMEM, tensor-map
// prefetch), waits, and only then triggers: a grid launched on the trigger finds every
// earlier grid on the stream complete, which a bulk collective launched beside a GEMM
// (ub_bulk.cu, no wait of its own at entry) relies on for its inputs. Two kinds of
// launch skip the entry wait and trigger at once, each waiting for the grid before it
// at exit instead (so that it still completes after that grid): a bulk collective in
// beside mode, and an AG-GEMM launched behind its own gather kernel (p.after_gather),
// whose reads of the gathered buffer the chunk flags order.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

// fp32 pair -> packed bf16x2 (round to nearest even); `lo` lands at the lower address.
__device__ __forceinline__ uint32_t pack_bf16x2(uint32_t lo, uint32_t hi)
{
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(__uint_as_float(hi)), "f"(__uint_as_float(lo)));
    return d;
}

// ---- tcgen05

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Shared-memory matrix descriptor of a K-major operand tile written by TMA with the
// 128-byte swizzle: rows of 128 bytes (64 bf16 of K), 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);  // start address      [0,14)
    d |= static_cast<uint64_t>(16u >> 4) << 16;           // leading offset     [16,30) (unused: K fits one row)
    d |= static_cast<uint64_t>(1024u >> 4) << 32;         // stride offset      [32,46)
    d |= static_cast<uint64_t>(1u) << 46;                 // descriptor version [46,48)
    d |= static_cast<uint64_t>(2u) << 61;                 // swizzle: 128 B     [61,64)
    return d;
}

// Shared-memory matrix descriptor of an MN-major operand tile (MN contiguous in global
// memory, e.g. a weight stored K x N) written by TMA with the 128-byte swizzle in boxes
// of 64 MN elements x 64 K rows: each 8 K-rows x 64 MN group is one 1024-byte swizzle
// atom; atoms follow each other along K every 1024 bytes (stride offset) and the second
// box of 64 MN elements starts 8 KiB later (leading offset).
__device__ __forceinline__ uint64_t smem_desc_mn_sw128(uint32_t saddr)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);  // start address      [0,14)
    d |= static_cast<uint64_t>(8192u >> 4) << 16;         // leading offset: next 64 MN
    d |= static_cast<uint64_t>(1024u >> 4) << 32;         // stride offset: next 8 K rows
    d |= static_cast<uint64_t>(1u) << 46;                 // descriptor version
    d |= static_cast<uint64_t>(2u) << 61;                 // swizzle: 128 B
    return d;
}
constexpr uint32_t MN_BOX_BYTES = 64 * BK * 2;           // one 64 (MN) x 64 (K) box

// Arrive on `bar` once every tcgen05 operation this thread issued so far has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t *v)
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]),
          "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]),
          "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]),
          "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 16 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t *v)
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr));
}

// Contiguous global -> shared copy (the tensor memory accelerator's untiled form) that
// completes `bytes` on an mbarrier; both addresses 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}



// Bounded pause used on the abort path so that copies already issued land first.
__device__ void settle(uint64_t ns)
{
    const uint64_t t0 = global_timer();
    while (global_timer() - t0 < ns) __nanosleep(1000);
}

// ------------------------------------------------------------------ bounded waits

struct WaitCtx {
    uint32_t *abort_word;
    int32_t *status;
    uint64_t timeout_ns;
    uint32_t epoch;
};

__device__ __forceinline__ bool call_aborted(const WaitCtx &w)
{
    return *reinterpret_cast<volatile uint32_t *>(w.abort_word) == w.epoch;
}

__device__ void raise_error(const WaitCtx &w, int code)
{
    atomicCAS(reinterpret_cast<int *>(w.status), 0, code);
    __threadfence();
    atomicExch(w.abort_word, w.epoch);
}

// A waiting thread reads the abort word at most once per this many ns. Every waiting
// thread of every CTA polls the same word, so frequent reads would queue on the one L2
// slice that holds it, in front of the operand loads that the waits are waiting for.
constexpr uint64_t kAbortPollNs = 16000;

// Timeout and abort checks of a spinning wait, made every few spins: false when the
// wait must give up (the call was aborted, or the timeout ran out: UB_ERR_TIMEOUT).
struct WaitClock {
    uint64_t t0, next_poll;
    __device__ __forceinline__ WaitClock() : t0(global_timer()), next_poll(t0 + kAbortPollNs) {}
    __device__ __forceinline__ bool ok(const WaitCtx &w)
    {
        const uint64_t now = global_timer();
        if (now - t0 > w.timeout_ns) {
            raise_error(w, UB_ERR_TIMEOUT);
            return false;
        }
        if (now >= next_poll) {
            if (call_aborted(w)) return false;
            next_poll = now + kAbortPollNs;
        }
        return true;
    }
};

// Wait for phase `parity` of an mbarrier. False when this call was aborted or the
// wait ran past the timeout (which then raises UB_ERR_TIMEOUT).
__device__ bool mbar_wait(uint32_t bar, uint32_t parity, const WaitCtx &w)
{
    if (mbar_try_wait(bar, parity)) return true;
    WaitClock clk;
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((n & 15u) == 0 && !clk.ok(w)) return false;
    }
}

// Wait used while draining at exit: ignores the abort word, still bounded in time.
__device__ bool mbar_wait_drain(uint32_t bar, uint32_t parity, uint64_t timeout_ns)
{
    const uint64_t t0 = global_timer();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer() - t0 > timeout_ns) return false;
    }
    return true;
}

// Wait until the readiness flag of every chunk in `mask` holds this call's epoch, then
// order the tensor-memory-accelerator reads that follow after them. Epochs are unique per
// handle (a call captured into a graph clears the flags in stream order before it
// starts), so a flag left by any other call never matches. Every flag still pending is
// read with an acquire load on each pass, the passes 512 ns apart: every producer thread
// of the grid polls the same few words, and faster polling queues on the L2 slice that
// holds them, in front of the operand loads (measured on GB300: polling every 128 ns made
// the AG-GEMM 1-2 % slower at T = 1024-4096). Once all are set, one proxy fence orders the
// async-proxy (TMA) reads of the chunks after the acquires.
__device__ bool wait_flags(const uint32_t *flags, uint32_t mask, const WaitCtx &w)
{
    WaitClock clk;
    for (uint32_t n = 0;; ++n) {
        for (uint32_t m = mask; m != 0u; m &= m - 1u) {
            const int r = __ffs(static_cast<int>(m)) - 1;
            uint32_t v;
            asm volatile("ld.acquire.sys.global.u32 %0, [%1];" : "=r"(v) : "l"(flags + r) : "memory");
            if (v == w.epoch) mask &= ~(1u << r);
        }
        if (mask == 0u) {
            asm volatile("fence.proxy.async.global;" ::: "memory");
            return true;
        }
        if ((n & 7u) == 7u && !clk.ok(w)) return false;
        __nanosleep(512);
    }
}

// The same for one chunk's flag.
__device__ __forceinline__ bool wait_flag(const uint32_t *flag, const WaitCtx &w) { return wait_flags(flag, 1u, w); }

// One look, without waiting, at the readiness flags in `mask` (at most UB_MAX_TP): the
// loads are relaxed and issued together, so they are in flight at once; only when every
// flag holds `epoch` does an acquire fence (with the proxy fence for the TMA reads that
// follow) make the chunks' contents visible, as wait_flags' acquire loads do.
__device__ __forceinline__ bool try_flags(const uint32_t *flags, uint32_t mask, uint32_t epoch)
{
    uint32_t v[UB_MAX_TP];
#pragma unroll
    for (int r = 0; r < UB_MAX_TP; ++r)
        if ((mask >> r) & 1u) asm volatile("ld.relaxed.sys.global.u32 %0, [%1];" : "=r"(v[r]) : "l"(flags + r) : "memory");
    bool all = true;
#pragma unroll
    for (int r = 0; r < UB_MAX_TP; ++r)
        if ((mask >> r) & 1u) all = all && v[r] == epoch;
    if (all) {
        asm volatile("fence.acq_rel.sys;" ::: "memory");
        asm volatile("fence.proxy.async.global;" ::: "memory");
    }
    return all;
}

__device__ __forceinline__ void st_release_u32(uint32_t *ptr, uint32_t v)
{
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(ptr), "r"(v) : "memory");
}

// All-gather done by the GEMM's own epilogue warps (128 threads, named barrier 1) before
// their first tile, while the producer already loads the self chunk's tiles. The parts
// to copy, in issue order (gather_part): the self chunk's rows from g_self_head_vecs on
// (the rows past its whole 256-row tiles, which the CTA-pair kernel reads from the
// buffer), the other chunks in ring order after the self rank, then the self chunk's
// first rows (read in place, so they need no flag unless they are the whole chunk).
// Two orders, chosen per call by the host:
//  - part by part (p.fused_gather == 1): every CTA copies its 1/gridDim.x share of each
//    part in turn, so the chunks land in ring order, the first soonest: for calls of
//    several waves of tiles, whose first wave needs only the first chunks;
//  - end to end (p.fused_gather == 2): the parts laid end to end and every CTA copies one
//    contiguous 1/gridDim.x of the whole, two batches of loads in flight per thread, so
//    a CTA pays the memory latency a few times instead of once per part and every chunk
//    lands sooner on average, but all at about the same time: for one wave of tiles,
//    which all start together (QKV at T = 1024 on GB300: 45.8 against 51.7 us a call).
// 16-byte loads bypass L1. A flagged part is complete when every CTA whose share meets it
// has counted it (after a CTA barrier and a fence); the CTA that completes the count
// resets the chunk's counter and publishes its readiness flag with the call's epoch (no
// flag for chunk p.g_drop). A chunk's counter serves one flagged part per call.
struct GatherPart {
    int r;           // chunk
    int64_t lo, hi;  // its vectors [lo, hi)
    bool flag;       // publishes the chunk's readiness flag once complete
};
__device__ __forceinline__ int gather_n_parts(const GemmParams &p)
{
    return (p.g_self_head_vecs < p.g_chunk_vecs) + (p.tp - 1) + (p.g_self_head_vecs > 0);
}
__device__ __forceinline__ GatherPart gather_part(const GemmParams &p, int i)
{
    const int64_t head = p.g_self_head_vecs, cv = p.g_chunk_vecs;
    const int k0 = head < cv ? 1 : 0;
    if (i < k0) return GatherPart{p.self_rank, head, cv, true};
    if (i < k0 + p.tp - 1) {
        int r = p.self_rank + 1 + (i - k0);
        if (r >= p.tp) r -= p.tp;
        return GatherPart{r, 0, cv, true};
    }
    return GatherPart{p.self_rank, 0, head, head >= cv};
}

__device__ __forceinline__ uint4 ld_nc_v4(const uint4 *p)
{
    uint4 x;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(x.x), "=r"(x.y), "=r"(x.z), "=r"(x.w)
                 : "l"(p));
    return x;
}

// Copy n 16-byte vectors src -> dst with the 128 threads et = 0..127 (vector i to thread
// i % 128): two batches of 8 loads per thread in flight, the next batch's loads issued
// before the current batch is stored.
__device__ __forceinline__ void copy_vecs(const uint4 *__restrict__ src, uint4 *__restrict__ dst, int64_t n, int et)
{
    constexpr int U = 8;
    constexpr int64_t STEP = U * 128;
    uint4 a[U], b[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
        if (et + u * 128 < n) a[u] = ld_nc_v4(src + et + u * 128);
    for (int64_t v = et; v < n; v += 2 * STEP) {
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (v + STEP + u * 128 < n) b[u] = ld_nc_v4(src + v + STEP + u * 128);
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (v + u * 128 < n) dst[v + u * 128] = a[u];
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (v + 2 * STEP + u * 128 < n) a[u] = ld_nc_v4(src + v + 2 * STEP + u * 128);
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (v + STEP + u * 128 < n) dst[v + STEP + u * 128] = b[u];
    }
}

// The end-to-end order (p.fused_gather == 2).
__device__ void fused_gather_end_to_end(const GemmParams &p, int et)
{
    const int64_t G = gridDim.x;
    const int np = gather_n_parts(p);
    int64_t total = 0;
    for (int i = 0; i < np; ++i) {
        const GatherPart g = gather_part(p, i);
        total += g.hi - g.lo;
    }
    const int64_t per = (total + G - 1) / G;
    const int64_t a = static_cast<int64_t>(blockIdx.x) * per;
    const int64_t b = a + per < total ? a + per : total;
    int64_t s0 = 0;
    for (int i = 0; i < np; ++i) {
        const GatherPart g = gather_part(p, i);
        const int64_t s1 = s0 + g.hi - g.lo;
        const int64_t lo = a > s0 ? a : s0, hi = b < s1 ? b : s1;
        if (lo < hi) {
            const int64_t v0 = g.lo + (lo - s0);
            copy_vecs(static_cast<const uint4 *>(p.g_src[g.r]) + v0,
                      static_cast<uint4 *>(p.g_ub) + static_cast<int64_t>(g.r) * p.g_chunk_vecs + v0, hi - lo, et);
        }
        s0 = s1;
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");  // this CTA's share is written
    if (et != 0) return;
    __threadfence();
    s0 = 0;
    for (int i = 0; i < np; ++i) {
        const GatherPart g = gather_part(p, i);
        const int64_t s1 = s0 + g.hi - g.lo;
        // the CTAs whose shares meet part [s0, s1): s0 / per .. (s1 - 1) / per
        if (g.flag && s1 > s0 && blockIdx.x >= s0 / per && blockIdx.x <= (s1 - 1) / per) {
            const uint32_t done = atomicAdd(p.g_counters + g.r, 1u) + 1u;
            if (done == static_cast<uint32_t>((s1 - 1) / per - s0 / per + 1)) {
                p.g_counters[g.r] = 0u;  // zero again for the next call
                __threadfence();
                if (g.r != p.g_drop) st_release_u32(const_cast<uint32_t *>(p.flags) + g.r, p.epoch);
            }
        }
        s0 = s1;
    }
}

// The part-by-part order (p.fused_gather == 1).
__device__ void fused_gather(const GemmParams &p, int et)
{
    if (p.fused_gather == 2) {
        fused_gather_end_to_end(p, et);
        return;
    }
    const int G = static_cast<int>(gridDim.x);
    const int64_t head = p.g_self_head_vecs;
    for (int q = 0; q <= p.tp; ++q) {
        int r = p.self_rank;
        int64_t lo = 0, hi = p.g_chunk_vecs;
        bool publish = true;
        if (q == 0) {
            lo = head;                  // the self chunk's last rows
            if (lo >= hi) continue;
        } else if (q < p.tp) {
            r += q;                     // the other chunks
            if (r >= p.tp) r -= p.tp;
        } else {
            hi = head;                  // the self chunk's first rows
            publish = head >= p.g_chunk_vecs;
            if (hi <= 0) continue;
        }
        const int64_t per = (hi - lo + G - 1) / G;
        const int64_t v0 = lo + static_cast<int64_t>(blockIdx.x) * per;
        const int64_t v1 = v0 + per < hi ? v0 + per : hi;
        const uint4 *src = static_cast<const uint4 *>(p.g_src[r]);
        uint4 *dst = static_cast<uint4 *>(p.g_ub) + static_cast<int64_t>(r) * p.g_chunk_vecs;
        constexpr int U = 16;
        for (int64_t v = v0 + et; v < v1; v += U * 128) {
            uint4 x[U];
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (v + u * 128 < v1)
                    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(x[u].x), "=r"(x[u].y), "=r"(x[u].z), "=r"(x[u].w)
                                 : "l"(src + v + u * 128));
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (v + u * 128 < v1) dst[v + u * 128] = x[u];
        }
        if (!publish) continue;
        asm volatile("bar.sync 1, 128;" ::: "memory");  // this CTA's share of the part is written
        if (et == 0) {
            __threadfence();
            const uint32_t done = atomicAdd(p.g_counters + r, 1u) + 1u;
            if (done == static_cast<uint32_t>(G)) {
                p.g_counters[r] = 0u;  // zero again for the next call
                __threadfence();
                if (r != p.g_drop) st_release_u32(const_cast<uint32_t *>(p.flags) + r, p.epoch);
            }
        }
    }
}

// Wait until a partial tile of this call is published (bounded, abort-aware).
__device__ bool wait_partial(const uint32_t *flag, const WaitCtx &w)
{
    WaitClock clk;
    for (uint32_t n = 0;; ++n) {
        uint32_t v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
        if (v == w.epoch) return true;
        if ((n & 15u) == 15u && !clk.ok(w)) return false;
        __nanosleep(64);
    }
}

}  // namespace
}  // namespace ubk
