// Standalone reduce-scatter of tp partial results: the independent reduce-scatter of
// the "bulk" overlap method in "How to setup TP Overlap configs" (TransformerEngine
// issue #1344), run beside an unrelated GEMM (for example the input-gradient partials
// of a column-parallel layer reduced while its weight-gradient GEMM runs).
//
//   Y_shards[r][i][n] = bf16( sum_{j<tp} P_j[r*c + i][n] ),  c = T / tp, fp32 sum in j order
//
// The work is HBM-bound: (tp + 1) * T * hidden * 2 bytes for tp * T * hidden adds. Each
// thread owns 8 consecutive columns of one row (16-byte loads and stores, coalesced
// across the warp); a grid-stride loop covers the active rows only. The CTAs are small
// (256 threads, no shared memory, under 88 registers a thread), four per SM alone, so
// that together they keep enough loads in flight to stream HBM. One fits on an SM beside
// a persistent GEMM CTA of the pair kernel: that CTA leaves about 1 KB of the SM's shared
// memory, and in each of the SM's four register files room for two more warps of at
// most 88 registers (a reduce-scatter of more loads in flight per thread, 98 registers
// and up, ran only after the GEMM).
//
// Beside a GEMM on a second stream, which grid the GPU places first decides the overlap
// (GB300, beside the weight-gradient GEMM: per run either about a third hidden or none,
// the collective's four CTAs per SM then keeping the GEMM's out). Beside mode (`beside`)
// removes the choice: the host launches the kernel on the GEMM's stream as its
// programmatic dependent, one CTA per SM, so it starts only once every GEMM CTA holds
// its SM. What it then hides is bounded by HBM: its 168 MB (T = 4096, tp 4, hidden 4096)
// beside the GEMM's own traffic slow the GEMM by some microseconds.
#include <cuda_bf16.h>

#include "ub_internal.h"

namespace ubk {
namespace {

// Programmatic dependent launch (see ub_device.cuh). A plain launch waits for the grid
// before it, then lets the next kernel launch. Beside mode (`beside`, the host launches
// the kernel as a programmatic dependent of the GEMM issued just before it): no wait at
// entry -- the kernel launches once every CTA of the GEMM holds its SM (the GEMM triggers
// only after its own wait, so every grid before the GEMM is complete and the inputs are
// in memory), runs in the room the GEMM's CTAs leave, and waits for the GEMM at exit, so
// that it completes only after the GEMM and work behind it on the stream sees both. It
// lets the next kernel launch at once: that kernel's CTAs take SMs as the GEMM's leave
// and wait for this one (so for the GEMM too) before touching memory, so its launch and
// prologue overlap the GEMM's end instead of following this kernel's exit.
__device__ __forceinline__ void pdl_enter(int beside)
{
    if (!beside) asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void pdl_leave(int beside)
{
    if (beside) asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ uint4 ld_stream(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// bf16 -> fp32 is exact: the bf16 pattern is the top half of the fp32 pattern.
__device__ __forceinline__ void add_bf16x2(uint32_t w, float &lo, float &hi)
{
    lo += __uint_as_float(w << 16);
    hi += __uint_as_float(w & 0xFFFF0000u);
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi)
{
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// TP partials, U vectors of 8 columns per thread per iteration: all TP * U 16-byte loads
// are issued before the first add, so enough bytes are in flight to cover HBM latency.
template <int TP, int U>
__global__ void __launch_bounds__(256) bulk_rs_kernel(const __grid_constant__ BulkRsParams p)
{
    pdl_enter(p.beside);
    const int64_t vecs_per_row = p.H / 8;
    const int64_t total = p.T * vecs_per_row;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; base < total;
         base += stride * U) {
        uint4 q[U][TP];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t v = base + u * stride;
            if (v < total) {
                const int64_t t = v / vecs_per_row;
                const int64_t col = (v - t * vecs_per_row) * 8;
#pragma unroll
                for (int j = 0; j < TP; ++j)
                    q[u][j] = ld_stream(static_cast<const __nv_bfloat16 *>(p.P[j]) + t * p.H + col);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t v = base + u * stride;
            if (v >= total) break;
            const int64_t t = v / vecs_per_row;
            const int64_t col = (v - t * vecs_per_row) * 8;
            float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int j = 0; j < TP; ++j) {
                add_bf16x2(q[u][j].x, a[0], a[1]);
                add_bf16x2(q[u][j].y, a[2], a[3]);
                add_bf16x2(q[u][j].z, a[4], a[5]);
                add_bf16x2(q[u][j].w, a[6], a[7]);
            }
            const int64_t r = t / p.c;
            const int64_t i = t - r * p.c;
            uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.Y[r]) + i * p.H + col);
            *dst = make_uint4(pack2(a[0], a[1]), pack2(a[2], a[3]), pack2(a[4], a[5]), pack2(a[6], a[7]));
        }
    }
    pdl_leave(p.beside);
}

// One CTA group per chunk, ring order: block b copies part (b % ctas_per_chunk) of chunk
// self_rank + b / ctas_per_chunk (mod tp), the self chunk first.
__global__ void __launch_bounds__(256) gather_kernel(const __grid_constant__ GatherParams p)
{
    pdl_enter(p.beside);
    const int q = blockIdx.x / p.ctas_per_chunk;  // 0..tp-1
    const int part = blockIdx.x - q * p.ctas_per_chunk;
    const int r = (p.self_rank + q) % p.tp;
    const uint4 *src = static_cast<const uint4 *>(p.src[r]);
    uint4 *dst = static_cast<uint4 *>(p.ub) + static_cast<int64_t>(r) * p.chunk_vecs;
    const int64_t stride = static_cast<int64_t>(p.ctas_per_chunk) * blockDim.x;
    // eight 16-byte loads in flight per thread before the first store
    constexpr int U = 8;
    for (int64_t v = static_cast<int64_t>(part) * blockDim.x + threadIdx.x; v < p.chunk_vecs; v += U * stride) {
        uint4 x[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (v + u * stride < p.chunk_vecs) x[u] = ld_stream(src + v + u * stride);
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (v + u * stride < p.chunk_vecs) dst[v + u * stride] = x[u];
    }
    __syncthreads();
    if (threadIdx.x == 0 && p.ctas_per_chunk == 1) {
        // the whole chunk is this CTA's: its release store publishes every thread's
        // copies (ordered before it by the CTA barrier), no count needed
        if (r != p.drop)
            asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p.flags + r), "r"(p.epoch) : "memory");
    } else if (threadIdx.x == 0) {
        __threadfence();
        const uint32_t done = atomicAdd(p.counters + r, 1u) + 1u;
        if (done == static_cast<uint32_t>(p.ctas_per_chunk)) {
            // last CTA of this chunk: every part is written (each CTA fenced before
            // counting); reset the counter for the next call, then publish the flag
            p.counters[r] = 0u;
            __threadfence();
            if (r != p.drop)
                asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p.flags + r), "r"(p.epoch) : "memory");
        }
    }
    pdl_leave(p.beside);
}

}  // namespace

cudaError_t launch_gather(const GatherParams &p, cudaStream_t stream)
{
    cudaError_t e = launch_ex(gather_kernel, p, p.tp * p.ctas_per_chunk, 256, 0, 0, p.pdl != 0, stream);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_bulk_rs(const BulkRsParams &p, int grid, cudaStream_t stream)
{
    cudaError_t e;
    switch (p.tp) {
    case 1: e = launch_ex(bulk_rs_kernel<1, 4>, p, grid, 256, 0, 0, p.pdl != 0, stream); break;
    case 2: e = launch_ex(bulk_rs_kernel<2, 4>, p, grid, 256, 0, 0, p.pdl != 0, stream); break;
    case 3: e = launch_ex(bulk_rs_kernel<3, 2>, p, grid, 256, 0, 0, p.pdl != 0, stream); break;
    case 4: e = launch_ex(bulk_rs_kernel<4, 2>, p, grid, 256, 0, 0, p.pdl != 0, stream); break;
    case 5: e = launch_ex(bulk_rs_kernel<5, 2>, p, grid, 256, 0, 0, p.pdl != 0, stream); break;
    case 6: e = launch_ex(bulk_rs_kernel<6, 2>, p, grid, 256, 0, 0, p.pdl != 0, stream); break;
    case 7: e = launch_ex(bulk_rs_kernel<7, 1>, p, grid, 256, 0, 0, p.pdl != 0, stream); break;
    default: e = launch_ex(bulk_rs_kernel<8, 1>, p, grid, 256, 0, 0, p.pdl != 0, stream); break;
    }
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace ubk
