// Weighted combine + residual, and the packing kernels for the code layout,
// the codebook layout and the expert-record header.
#include "internal.cuh"

namespace rvq {
namespace {

// out[t][c] = res[t][c] + sum_slot w[t][slot] * sum_s ypart[(t*k+slot)*nslot + s][c]
// (reading: the pages do not describe the combine; this is the standard MoE
// output with the routing weights).  Block = 16 column quads x k slots: each
// thread reduces one slot's split-K partials for four columns (128-bit
// loads), then the slot products are added to the residual in slot order.
constexpr int CB_Q = 16;  // column quads per block

__global__ void combine_kernel(const float *__restrict__ ypart, int nslot,
                               const float *__restrict__ w, int n, int k, int d,
                               const void *res, int rdt, float *out, float *out2) {
    __shared__ float4 prod[32][CB_Q];
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    const int d4 = d >> 2;
    const int qx = threadIdx.x, slot = threadIdx.y;
    const int t = blockIdx.y;
    const int c4 = blockIdx.x * CB_Q + qx;
    if (c4 < d4) {
        const float wv = w[(int64_t)t * k + slot];
        const float4 *yp = reinterpret_cast<const float4 *>(
            ypart + ((int64_t)(t * k + slot) * nslot) * d) + c4;
        float4 y = __ldg(yp);
#pragma unroll 4
        for (int q = 1; q < nslot; ++q) {
            const float4 v = __ldg(yp + (int64_t)q * d4);
            y.x += v.x; y.y += v.y; y.z += v.z; y.w += v.w;
        }
        prod[slot][qx] = make_float4(wv * y.x, wv * y.y, wv * y.z, wv * y.w);
    }
    __syncthreads();
    if (slot != 0 || c4 >= d4) return;
    const int c = c4 * 4;
    float4 acc;
    if (rdt == RVQ_BF16) {
        const uint2 r = *reinterpret_cast<const uint2 *>(
            reinterpret_cast<const uint16_t *>(res) + (int64_t)t * d + c);
        acc.x = __uint_as_float(r.x << 16);
        acc.y = __uint_as_float(r.x & 0xFFFF0000u);
        acc.z = __uint_as_float(r.y << 16);
        acc.w = __uint_as_float(r.y & 0xFFFF0000u);
    } else {
        acc = *reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(res) +
                                                (int64_t)t * d + c);
    }
    for (int s = 0; s < k; ++s) {
        const float4 v = prod[s][qx];
        acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    *reinterpret_cast<float4 *>(out + (int64_t)t * d + c) = acc;
    if (out2) *reinterpret_cast<float4 *>(out2 + (int64_t)t * d + c) = acc;
}

// A layer call's input or output moved between a host buffer the GPU maps
// (pinned) and device memory by the GPU itself, 16 bytes per thread and
// step: as a kernel of the call's launch chain, programmatic dependent launch
// carries through it (a cudaMemcpyAsync node would end the overlap).
__global__ void __launch_bounds__(256) io_copy_kernel(const uint4 *__restrict__ src,
                                                      uint4 *__restrict__ dst, int64_t n16) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16;
         i += (int64_t)gridDim.x * blockDim.x)
        dst[i] = src[i];
}

// nslot == 1 (outputs already reduced, e.g. by the tensor-core path): one
// thread per (token, column quad) with all k slot loads in flight at once.
__global__ void __launch_bounds__(256) combine1_kernel(const float *__restrict__ y,
                                                       const float *__restrict__ w, int n, int k,
                                                       int d, const void *res, int rdt,
                                                       float *out, float *out2) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    const int d4 = d >> 2;
    const int c4 = blockIdx.x * blockDim.x + threadIdx.x;
    const int t = blockIdx.y;
    if (c4 >= d4) return;
    const int c = c4 * 4;
    float4 acc;
    if (rdt == RVQ_BF16) {
        const uint2 r = __ldg(reinterpret_cast<const uint2 *>(
            reinterpret_cast<const uint16_t *>(res) + (int64_t)t * d + c));
        acc.x = __uint_as_float(r.x << 16);
        acc.y = __uint_as_float(r.x & 0xFFFF0000u);
        acc.z = __uint_as_float(r.y << 16);
        acc.w = __uint_as_float(r.y & 0xFFFF0000u);
    } else {
        acc = __ldg(reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(res) +
                                                     (int64_t)t * d + c));
    }
    const float4 *yp = reinterpret_cast<const float4 *>(y + (int64_t)t * k * d) + c4;
    for (int s0 = 0; s0 < k; s0 += 8) {
        float4 v[8];
        float ws[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const bool on = s0 + i < k;
            v[i] = on ? __ldg(yp + (int64_t)(s0 + i) * d4) : make_float4(0.f, 0.f, 0.f, 0.f);
            ws[i] = on ? __ldg(w + (int64_t)t * k + s0 + i) : 0.f;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            acc.x += ws[i] * v[i].x;
            acc.y += ws[i] * v[i].y;
            acc.z += ws[i] * v[i].z;
            acc.w += ws[i] * v[i].w;
        }
    }
    *reinterpret_cast<float4 *>(out + (int64_t)t * d + c) = acc;
    if (out2) *reinterpret_cast<float4 *>(out2 + (int64_t)t * d + c) = acc;
}

// Row-wise RMS normalisation without a gain (the layer stack's pre-norm):
// out = x / sqrt(mean(x^2) + eps), sums in fp32, one block per row.
__global__ void __launch_bounds__(256) rms_norm_kernel(const void *__restrict__ x, int xdt, int d,
                                                       float eps, void *__restrict__ out,
                                                       int odt) {
    __shared__ float red[8];
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    const int64_t row = (int64_t)blockIdx.x * d;
    const int d4 = d >> 2;
    const float inv = block_rms_inv(x, xdt, row, d, eps, red);
    for (int c4 = threadIdx.x; c4 < d4; c4 += blockDim.x) {
        const float4 v = load4(x, xdt, row + c4 * 4);
        const float4 y = make_float4(v.x * inv, v.y * inv, v.z * inv, v.w * inv);
        if (odt == RVQ_BF16) {
            uint2 b;
            b.x = bf16x2_bits(y.x, y.y);
            b.y = bf16x2_bits(y.z, y.w);
            *reinterpret_cast<uint2 *>(reinterpret_cast<uint16_t *>(out) + row + c4 * 4) = b;
        } else {
            *reinterpret_cast<float4 *>(reinterpret_cast<float *>(out) + row + c4 * 4) = y;
        }
    }
}

// One thread per 16-byte packed word.  Packed word (tile g,b; stage s; half h;
// lane l) byte i <-> canonical code (row 32b+l, chunk 32g+((16h+i+l) mod 32), s).
__global__ void pack_kernel(const uint8_t *__restrict__ src, int rows, int cols,
                            uint8_t *__restrict__ dst, int unpack) {
    const int64_t words = (int64_t)rows * cols * 3 / 128;
    const int64_t wi = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (wi >= words) return;
    const int RB = rows / 32;
    const int64_t tile = wi / 192;
    const int within = (int)(wi % 192);
    const int sh = within / 32, l = within % 32;
    const int s = sh >> 1, h = sh & 1;
    const int g = (int)(tile / RB), b = (int)(tile % RB);
    const int row = 32 * b + l;
    const int64_t rowbase = (int64_t)row * (cols / 8);
    if (!unpack) {
        uint8_t v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int chunk = 32 * g + ((16 * h + i + l) & 31);
            v[i] = src[(rowbase + chunk) * 3 + s];
        }
        uint4 o;
        o.x = v[0] | (v[1] << 8) | (v[2] << 16) | ((uint32_t)v[3] << 24);
        o.y = v[4] | (v[5] << 8) | (v[6] << 16) | ((uint32_t)v[7] << 24);
        o.z = v[8] | (v[9] << 8) | (v[10] << 16) | ((uint32_t)v[11] << 24);
        o.w = v[12] | (v[13] << 8) | (v[14] << 16) | ((uint32_t)v[15] << 24);
        *reinterpret_cast<uint4 *>(dst + wi * 16) = o;
    } else {
        const uint8_t *p = src + wi * 16;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int chunk = 32 * g + ((16 * h + i + l) & 31);
            dst[(rowbase + chunk) * 3 + s] = p[i];
        }
    }
}

// canonical fp32 [count][3][256][8] -> pair-interleaved [count][3][128][8][2]
__global__ void pack_codebooks_kernel(const float *__restrict__ src, float *__restrict__ dst,
                                      int count) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= count * 6144) return;
    const int mat = i / 6144, r = i % 6144;
    const int s = r / 2048, k = (r / 8) % 256, dim = r % 8;
    dst[mat * 6144 + ((s * 128 + k / 2) * 8 + dim) * 2 + (k & 1)] = src[i];
}

__global__ void write_header_kernel(uint8_t *record, rvq_expert_header h) {
    if (threadIdx.x == 0) *reinterpret_cast<rvq_expert_header *>(record) = h;
}

}  // namespace

rvq_status launch_rms_norm(const void *x, int xdt, int n, int d, float eps, void *out, int odt,
                           cudaStream_t stream, bool pdl) {
    if (n == 0) return RVQ_OK;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)n);
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    RVQ_CUDA(cudaLaunchKernelEx(&cfg, rms_norm_kernel, x, xdt, d, eps, out, odt));
    return RVQ_OK;
}

rvq_status launch_io_copy(const void *src, void *dst, size_t bytes, cudaStream_t stream,
                          bool pdl) {
    if (bytes == 0) return RVQ_OK;
    if ((bytes & 15u) != 0 || ((uintptr_t)src & 15u) != 0 || ((uintptr_t)dst & 15u) != 0) {
        set_error("io copy: %zu bytes between %p and %p are not 16-byte aligned", bytes, src, dst);
        return RVQ_EALIGN;
    }
    const int64_t n16 = (int64_t)(bytes / 16);
    const int64_t want = (n16 + 255) / 256;
    const int blocks = (int)(want < 4 * num_sms() ? want : 4 * num_sms());
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    RVQ_CUDA(cudaLaunchKernelEx(&cfg, io_copy_kernel, reinterpret_cast<const uint4 *>(src),
                                reinterpret_cast<uint4 *>(dst), n16));
    return RVQ_OK;
}

rvq_status launch_combine(const float *ypart, int nslot, const float *w, int n, int k, int d,
                          const void *res, int rdt, float *out, cudaStream_t stream, bool pdl,
                          float *out2) {
    if (n == 0) return RVQ_OK;
    if (k > 32) {
        set_error("combine: k %d > 32", k);
        return RVQ_EINVAL;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    cfg.stream = stream;
    if (nslot == 1 && n > 64) {
        cfg.gridDim = dim3((unsigned)((d / 4 + 255) / 256), (unsigned)n);
        cfg.blockDim = dim3(256);
        RVQ_CUDA(cudaLaunchKernelEx(&cfg, combine1_kernel, ypart, w, n, k, d, res, rdt, out, out2));
        return RVQ_OK;
    }
    cfg.gridDim = dim3((unsigned)((d / 4 + CB_Q - 1) / CB_Q), (unsigned)n);
    cfg.blockDim = dim3(CB_Q, (unsigned)k);
    RVQ_CUDA(cudaLaunchKernelEx(&cfg, combine_kernel, ypart, nslot, w, n, k, d, res, rdt, out,
                                out2));
    return RVQ_OK;
}

rvq_status launch_pack(const uint8_t *src, int rows, int cols, uint8_t *dst, bool unpack,
                       cudaStream_t stream) {
    const int64_t words = (int64_t)rows * cols * 3 / 128;
    const int bs = 256;
    pack_kernel<<<(unsigned)((words + bs - 1) / bs), bs, 0, stream>>>(src, rows, cols, dst,
                                                                       unpack ? 1 : 0);
    RVQ_LAUNCHED("pack");
    return RVQ_OK;
}

rvq_status launch_pack_codebooks(const float *src, float *dst, int count, cudaStream_t stream) {
    const int total = count * 6144;
    pack_codebooks_kernel<<<(total + 255) / 256, 256, 0, stream>>>(src, dst, count);
    RVQ_LAUNCHED("pack_codebooks");
    return RVQ_OK;
}

rvq_status launch_write_header(uint8_t *record, const rvq_expert_header &h, cudaStream_t stream) {
    write_header_kernel<<<1, 32, 0, stream>>>(record, h);
    RVQ_LAUNCHED("write_header");
    return RVQ_OK;
}

}  // namespace rvq
