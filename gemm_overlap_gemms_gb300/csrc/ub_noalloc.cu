// ag_gemm_noalloc: the AG-GEMM for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at all: code that runs inside another
// framework's memory pool or a custom allocator that owns the whole device, plugins
// loaded into a process whose allocations are audited, or code that must not grow
// the device footprint after start-up. They cannot create a handle (ub_create
// allocates the user buffer and the control block). This entry point keeps the same
// kernel but takes its scratch -- the gathered input (user buffer), the readiness
// flags, the abort word and the status word -- from one file-scope device array of a
// fixed size that lives as long as the library is loaded. It makes no cudaMalloc,
// no cudaFree and no other allocating call; it also creates no streams or events.
//
// The paper has no counterpart to this entry point; it is an addition of this
// library.
#include <cuda.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "ub_internal.h"

namespace {

// Scratch layout: [UB_NOALLOC_MAX_ELEMS bf16 of user buffer][256-byte control block:
// UB_MAX_TP flags | abort word | status word]. Zero-initialised when the module loads.
constexpr size_t kUbBytes = static_cast<size_t>(UB_NOALLOC_MAX_ELEMS) * 2;
constexpr size_t kCtrlBytes = 256;
static __device__ __align__(256) unsigned char g_scratch[kUbBytes + kCtrlBytes];

constexpr int kMaxDevices = 64;

struct DeviceScratch {
    char *base = nullptr;  // device address of g_scratch on this device
    uint32_t epoch = 0;    // last epoch written into this device's flags
    bool ready = false;
};

std::mutex g_mu;
DeviceScratch g_dev[kMaxDevices];

int fail(int code, const char *fmt, ...)
{
    char msg[256];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(msg, sizeof msg, fmt, ap);
    va_end(ap);
    ubk::set_last_error(msg);
    return code;
}

typedef CUresult (*PFN_encode)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                               const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                               CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
typedef CUresult (*PFN_write32)(CUstream, CUdeviceptr, cuuint32_t, unsigned int);

struct Fns {
    PFN_encode encode = nullptr;
    PFN_write32 write32 = nullptr;
};

const Fns *fns()
{
    static Fns f;
    static bool ok = false;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q1, q2;
        void *a = nullptr, *b = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &a, 12000, cudaEnableDefault, &q1) ==
                cudaSuccess &&
            cudaGetDriverEntryPointByVersion("cuStreamWriteValue32", &b, 12000, cudaEnableDefault, &q2) ==
                cudaSuccess &&
            q1 == cudaDriverEntryPointSuccess && q2 == cudaDriverEntryPointSuccess && a && b) {
            f.encode = reinterpret_cast<PFN_encode>(a);
            f.write32 = reinterpret_cast<PFN_write32>(b);
            ok = true;
        }
    });
    return ok ? &f : nullptr;
}

int encode(const Fns *f, CUtensorMap *map, const void *ptr, uint64_t inner, uint64_t outer, uint64_t pitch,
           uint32_t box_inner, uint32_t box_outer)
{
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {pitch};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = f->encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box,
                           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? UB_OK : fail(UB_ERR_CUDA, "ag_gemm_noalloc: cuTensorMapEncodeTiled failed (%d)", (int)r);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int ag_gemm_noalloc(const void *const *shards, int tp, int64_t T, int64_t hidden, const void *Wt,
                               int64_t N, void *Y, void *stream)
{
    // Host-side checks first: nothing below runs for a call that is rejected here.
    if (!shards || !Wt || !Y) return fail(UB_ERR_ARG, "ag_gemm_noalloc: null pointer argument");
    if (tp < 1 || tp > UB_MAX_TP) return fail(UB_ERR_ARG, "ag_gemm_noalloc: tp %d outside [1, %d]", tp, UB_MAX_TP);
    if (T <= 0 || hidden <= 0 || N <= 0)
        return fail(UB_ERR_ZERO, "ag_gemm_noalloc: zero extent (T=%lld hidden=%lld N=%lld)", (long long)T,
                    (long long)hidden, (long long)N);
    if (hidden % 8 != 0 || N % 8 != 0)
        return fail(UB_ERR_ALIGN, "ag_gemm_noalloc: hidden and N must be multiples of 8");
    if (T % tp != 0) return fail(UB_ERR_DIVISIBLE, "ag_gemm_noalloc: T=%lld not divisible by tp=%d", (long long)T, tp);
    if (T > (int64_t(1) << 31) - 1 || N > (int64_t(1) << 24) || hidden > (int64_t(1) << 24) ||
        T * hidden > static_cast<int64_t>(UB_NOALLOC_MAX_ELEMS))
        return fail(UB_ERR_CAPACITY,
                    "ag_gemm_noalloc: T*hidden = %lld exceeds the fixed scratch of %lld elements (32 MiB)",
                    (long long)(T * hidden), (long long)UB_NOALLOC_MAX_ELEMS);
    if (!aligned16(Wt) || !aligned16(Y)) return fail(UB_ERR_ALIGN, "ag_gemm_noalloc: Wt / Y not 16-byte aligned");
    for (int r = 0; r < tp; ++r) {
        if (!shards[r]) return fail(UB_ERR_ARG, "ag_gemm_noalloc: shard %d is null", r);
        if (!aligned16(shards[r])) return fail(UB_ERR_ALIGN, "ag_gemm_noalloc: shard %d not 16-byte aligned", r);
    }
    const Fns *f = fns();
    if (!f) return fail(UB_ERR_CUDA, "ag_gemm_noalloc: driver entry points unavailable");

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(UB_ERR_CUDA, "ag_gemm_noalloc: cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return fail(UB_ERR_ARG, "ag_gemm_noalloc: device %d unsupported", dev);
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return fail(UB_ERR_CUDA, "ag_gemm_noalloc: cudaDeviceGetAttribute: %s", cudaGetErrorString(e));

    std::lock_guard<std::mutex> lock(g_mu);
    nvtxRangePushA("ag_gemm_noalloc");
    struct Pop {
        ~Pop() { nvtxRangePop(); }
    } pop;
    DeviceScratch &ds = g_dev[dev];
    if (!ds.ready) {
        // Set-up, once per device, with that device current: the host-side name of
        // g_scratch is only a stand-in, so ask the runtime for its device address.
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_scratch);
        if (e != cudaSuccess || !p)
            return fail(UB_ERR_CUDA, "ag_gemm_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
        ds.base = static_cast<char *>(p);
        ds.ready = true;
    }
    char *ub = ds.base;
    uint32_t *ctrl = reinterpret_cast<uint32_t *>(ds.base + kUbBytes);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t H = hidden, c = T / tp;

    ubk::GemmParams p;
    memset(&p, 0, sizeof p);
    for (int r = 0; r < tp; ++r) {
        // self rank 0: its chunk is read in place; the others from the scratch buffer
        const void *src = r == 0 ? shards[0] : static_cast<const void *>(ub + r * c * H * 2);
        if (int rc = encode(f, &p.tmA[r], src, H, c, H * 2, ubk::BK, ubk::BM)) return rc;
        if (int rc = encode(f, &p.tmY[r], static_cast<char *>(Y) + r * c * N * 2, N, c, N * 2, ubk::STORE_COLS, 32))
            return rc;
    }
    if (int rc = encode(f, &p.tmB[0], Wt, H, N, H * 2, ubk::BK, ubk::BN)) return rc;
    p.flags = ctrl;
    p.abort_word = ctrl + UB_MAX_TP;
    p.status = reinterpret_cast<int32_t *>(ctrl + UB_MAX_TP + 1);
    p.timeout_ns = 1000000000ull;
    p.tp = tp;
    p.c = static_cast<int>(c);
    p.n_out = static_cast<int>(N);
    p.k_blocks = static_cast<int>((H + ubk::BK - 1) / ubk::BK);
    p.k_blocks_per_shard = p.k_blocks;
    p.m_tiles = static_cast<int>((c + ubk::BM - 1) / ubk::BM);
    p.n_tiles = static_cast<int>((N + ubk::BN - 1) / ubk::BN);
    p.num_tiles = tp * p.m_tiles * p.n_tiles;
    p.self_rank = 0;
    uint32_t epoch = ++ds.epoch;  // flags are never reset: epochs only grow
    if (epoch == 0) epoch = ++ds.epoch;  // 0 is what a cleared flag holds
    p.epoch = epoch;

    // The status word keeps the previous call's value: clear it for this call.
    e = cudaMemsetAsync(p.status, 0, sizeof(int32_t), s);
    if (e != cudaSuccess) return fail(UB_ERR_CUDA, "ag_gemm_noalloc: clearing status: %s", cudaGetErrorString(e));
    // Chunk copies and their flags on the caller's stream (no side stream is created
    // here), in ring order after rank 0; they therefore complete before the kernel.
    // Chunk 0 is not copied: the kernel reads it in place from its shard and never
    // waits for its flag, and nothing else reads the scratch.
    for (int r = 1; r < tp; ++r) {
        e = cudaMemcpyAsync(ub + r * c * H * 2, shards[r], static_cast<size_t>(c * H * 2), cudaMemcpyDeviceToDevice,
                            s);
        if (e != cudaSuccess) return fail(UB_ERR_CUDA, "ag_gemm_noalloc: cudaMemcpyAsync: %s", cudaGetErrorString(e));
        CUresult cr = f->write32(reinterpret_cast<CUstream>(s), reinterpret_cast<CUdeviceptr>(ctrl + r), epoch,
                                 CU_STREAM_WRITE_VALUE_DEFAULT);
        if (cr != CUDA_SUCCESS) return fail(UB_ERR_CUDA, "ag_gemm_noalloc: cuStreamWriteValue32 failed (%d)", (int)cr);
    }
    const int grid = p.num_tiles < sms ? p.num_tiles : sms;
    e = ubk::launch_gemm(p, ubk::MODE_AG, grid, s);
    if (e != cudaSuccess) return fail(UB_ERR_CUDA, "ag_gemm_noalloc: launch: %s", cudaGetErrorString(e));
    return UB_OK;
}
