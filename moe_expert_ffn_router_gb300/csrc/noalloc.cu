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
// looked up once per device with cudaGetSymbolAddress (on the first call made
// with that device current) and passed to the kernels.
#include <mutex>

#include "internal.cuh"

static __device__ __align__(256) uint8_t rvq_noalloc_scratch[RVQ_NOALLOC_SCRATCH_BYTES];

namespace {
std::mutex g_noalloc_mu;
void *g_noalloc_addr[64] = {nullptr};
}  // namespace

extern "C" rvq_status rvq_gemv_noalloc(const uint8_t *packed_codes_dev,
                                       const float *packed_cb_dev, int32_t rows, int32_t cols,
                                       const void *x_dev, rvq_dtype xdt, int32_t n, float *y_dev,
                                       rvq_stream_t stream) {
    if (!rvq::packable(rows, cols) || n < 1) {
        rvq::set_error("rvq_gemv_noalloc: rows %d must be a multiple of 32, cols %d of 512, n %d >= 1",
                       rows, cols, n);
        return RVQ_EINVAL;
    }
    const size_t need = rvq_gemv_workspace_bytes(rows, cols, n);
    if (need > RVQ_NOALLOC_SCRATCH_BYTES) {
        rvq::set_error("rvq_gemv_noalloc: %d x %d matrix with n = %d needs %zu bytes of scratch, "
                       "more than the fixed %u; use rvq_gemv with a workspace",
                       rows, cols, n, need, (unsigned)RVQ_NOALLOC_SCRATCH_BYTES);
        return RVQ_ENOMEM;
    }
    int dev = 0;
    RVQ_CUDA(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) {
        rvq::set_error("rvq_gemv_noalloc: device ordinal %d out of range", dev);
        return RVQ_EINVAL;
    }
    void *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_noalloc_mu);
        if (!g_noalloc_addr[dev]) {
            void *p = nullptr;
            RVQ_CUDA(cudaGetSymbolAddress(&p, rvq_noalloc_scratch));
            g_noalloc_addr[dev] = p;
        }
        scratch = g_noalloc_addr[dev];
    }
    // The array keeps the previous call's contents: the status block must
    // start at zero (the partial sums are fully overwritten by every call).
    RVQ_CUDA(cudaMemsetAsync(scratch, 0, RVQ_WS_STATUS_BYTES, (cudaStream_t)stream));
    return rvq_gemv(packed_codes_dev, packed_cb_dev, rows, cols, x_dev, xdt, n, y_dev, scratch,
                    RVQ_NOALLOC_SCRATCH_BYTES, stream);
}
