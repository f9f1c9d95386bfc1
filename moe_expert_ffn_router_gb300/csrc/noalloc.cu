// rvq_gemv for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: a plug-in that runs inside a host
// framework which owns all device memory and forbids allocations from
// extensions, or a latency-critical loop where an allocation (and its implicit
// device synchronisation) is not allowed.  rvq_gemv needs a caller-provided
// workspace for its split-K partial sums; this entry point instead uses a
// fixed array compiled into the library, so it performs no allocation at all.
//
// The array is a file-scope __device__ variable: every GPU that loads this
// library holds RVQ_NOALLOC_SCRATCH_BYTES of it until the process exits.  In
// host code its name is only a host-side stand-in, so its device address is
// looked up with cudaGetSymbolAddress, once per device and context (the first
// call made with that device current, and again if the device's context was
// replaced, e.g. after cudaDeviceReset), and passed to the kernels.
#include <mutex>

#include "internal.cuh"

static __device__ __align__(256) uint8_t rvq_noalloc_scratch[RVQ_NOALLOC_SCRATCH_BYTES];

namespace {

// CUresult cuCtxGetCurrent(CUcontext *), CUresult cuCtxGetId(CUcontext, unsigned long long *),
// reached through the runtime's driver entry points (the library does not
// link the driver library itself).
using CtxGetCurrentFn = int (*)(void **);
using CtxGetIdFn = int (*)(void *, unsigned long long *);

template <class F>
F driver_fn(const char *name) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<F>(p);
}

// Process-unique id of the calling thread's current context (0 if unknown).
unsigned long long current_context_id() {
    static const CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
    static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
    void *ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != 0 || !ctx || get_id(ctx, &id) != 0)
        return 0;
    return id;
}

struct Site {
    unsigned long long ctx_id;
    void *addr;
};
std::mutex g_mu;
Site g_site[64] = {};

// Device address of the scratch array for the current device and context.
rvq_status scratch_address(void **out) {
    int dev = 0;
    RVQ_CUDA(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) {
        rvq::set_error("rvq_gemv_noalloc: device ordinal %d out of range", dev);
        return RVQ_EINVAL;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    const unsigned long long id = current_context_id();
    if (g_site[dev].addr && id != 0 && g_site[dev].ctx_id == id) {
        *out = g_site[dev].addr;
        return RVQ_OK;
    }
    void *p = nullptr;
    RVQ_CUDA(cudaGetSymbolAddress(&p, rvq_noalloc_scratch));
    // the lookup makes the device's context current if nothing had yet; an
    // unknown id (0) is never cached, so such a caller looks the address up
    // on every call
    const unsigned long long id_after = id ? id : current_context_id();
    g_site[dev] = Site{id_after, id_after ? p : nullptr};
    *out = p;
    return RVQ_OK;
}

}  // namespace

extern "C" rvq_status rvq_gemv_noalloc(const uint8_t *packed_codes_dev,
                                       const float *packed_cb_dev, int32_t rows, int32_t cols,
                                       const void *x_dev, rvq_dtype xdt, int32_t n, float *y_dev,
                                       rvq_stream_t stream) {
    // every argument check comes first: a rejected call launches nothing and
    // leaves the array (and its status block) as the last call left them
    RVQ_TRY(rvq::check_gemv_args("rvq_gemv_noalloc", packed_codes_dev, packed_cb_dev, rows, cols,
                                 x_dev, xdt, n, y_dev));
    const size_t need = rvq_gemv_workspace_bytes(rows, cols, n);
    if (need > RVQ_NOALLOC_SCRATCH_BYTES) {
        rvq::set_error("rvq_gemv_noalloc: %d x %d matrix with n = %d needs %zu bytes of scratch, "
                       "more than the fixed %u; use rvq_gemv with a workspace",
                       rows, cols, n, need, (unsigned)RVQ_NOALLOC_SCRATCH_BYTES);
        return RVQ_ENOMEM;
    }
    void *scratch = nullptr;
    RVQ_TRY(scratch_address(&scratch));
    // The array keeps the previous call's contents: the status block must
    // start at zero (the partial sums are fully overwritten by every call).
    RVQ_CUDA(cudaMemsetAsync(scratch, 0, RVQ_WS_STATUS_BYTES, (cudaStream_t)stream));
    return rvq_gemv(packed_codes_dev, packed_cb_dev, rows, cols, x_dev, xdt, n, y_dev, scratch,
                    RVQ_NOALLOC_SCRATCH_BYTES, stream);
}

extern "C" rvq_status rvq_gemv_noalloc_status(uint32_t *bits_out, rvq_stream_t stream) {
    void *scratch = nullptr;
    RVQ_TRY(scratch_address(&scratch));
    return rvq::read_status_word(scratch, bits_out, (cudaStream_t)stream);
}
