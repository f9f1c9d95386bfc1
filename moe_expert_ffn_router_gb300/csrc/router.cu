// Router: logits, top-k selection with renormalised softmax weights, and the
// token -> expert grouping.
//
// The pages say only that a resident router picks 16 expert IDs per layer and
// that no low-probability expert is dropped [GeekNews topic 32035, section
// "Read-ahead and router prediction"; "Running a 2.78-Trillion-Parameter
// Model on a Laptop", section "Technical Insight"].  Readings used here: a
// linear router, the k largest fp32 logits with equal logits ordered by the
// lower expert index, weights softmax renormalised over the selected k, and
// pairs grouped by (expert, token).
#include "internal.cuh"

namespace rvq {
namespace {

// ------------------------------------------------------------------ logits
// Block = EB experts x TB tokens; 256 threads split the hidden dimension in
// 8-element pieces (128-bit loads of Wr, 64/128-bit loads of x).
constexpr int LG_EB = 2;
constexpr int LG_TB = 8;
constexpr int LG_NT = 256;

__global__ void __launch_bounds__(LG_NT) router_logits_kernel(
    const float *__restrict__ wr, const float *__restrict__ bias, const void *__restrict__ x,
    int xdt, int n, int E, int d, float *__restrict__ logits) {
    const int e0 = blockIdx.x * LG_EB;
    const int t0 = blockIdx.y * LG_TB;
    float acc[LG_EB][LG_TB];
#pragma unroll
    for (int a = 0; a < LG_EB; ++a)
#pragma unroll
        for (int b = 0; b < LG_TB; ++b) acc[a][b] = 0.f;
    for (int c = threadIdx.x * 8; c < d; c += LG_NT * 8) {
        float w[LG_EB][8];
#pragma unroll
        for (int a = 0; a < LG_EB; ++a) {
            if (e0 + a < E) {
                const float4 *p = reinterpret_cast<const float4 *>(wr + (int64_t)(e0 + a) * d + c);
                float4 u = __ldg(p), v = __ldg(p + 1);
                w[a][0] = u.x; w[a][1] = u.y; w[a][2] = u.z; w[a][3] = u.w;
                w[a][4] = v.x; w[a][5] = v.y; w[a][6] = v.z; w[a][7] = v.w;
            } else {
#pragma unroll
                for (int q = 0; q < 8; ++q) w[a][q] = 0.f;
            }
        }
#pragma unroll
        for (int b = 0; b < LG_TB; ++b) {
            if (t0 + b < n) {
                float xv[8];
                load8(x, xdt, (int64_t)(t0 + b) * d + c, xv);
#pragma unroll
                for (int a = 0; a < LG_EB; ++a)
#pragma unroll
                    for (int q = 0; q < 8; ++q) acc[a][b] = fmaf(w[a][q], xv[q], acc[a][b]);
            }
        }
    }
    __shared__ float red[LG_NT / 32][LG_EB * LG_TB];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int a = 0; a < LG_EB; ++a)
#pragma unroll
        for (int b = 0; b < LG_TB; ++b) {
            float v = acc[a][b];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            if (lane == 0) red[warp][a * LG_TB + b] = v;
        }
    __syncthreads();
    if (threadIdx.x < LG_EB * LG_TB) {
        const int a = threadIdx.x / LG_TB, b = threadIdx.x % LG_TB;
        if (e0 + a < E && t0 + b < n) {
            float v = 0.f;
            for (int q = 0; q < LG_NT / 32; ++q) v += red[q][threadIdx.x];
            if (bias) v += bias[e0 + a];
            logits[(int64_t)(t0 + b) * E + e0 + a] = v;
        }
    }
}

// ------------------------------------------------------------------- route
constexpr int RT_NT = 1024;
constexpr int RT_NW = RT_NT / 32;
constexpr size_t RT_SMEM_MAX = 200 * 1024;

// Order-preserving key for fp32 (after -0 -> +0): larger float, larger key.
__device__ __forceinline__ uint32_t float_key(float f) {
    uint32_t u = __float_as_uint(f + 0.0f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__global__ void __launch_bounds__(RT_NT, 1) route_kernel(const float *__restrict__ logits, int n,
                                                          int E, int k, int32_t *__restrict__ idx,
                                                          float *__restrict__ wout,
                                                          int32_t *__restrict__ offsets,
                                                          int32_t *__restrict__ pairs,
                                                          uint32_t *status) {
    extern __shared__ __align__(16) uint32_t rsm[];
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    const int W = (n + 31) >> 5;
    uint32_t *mask = rsm;                                   // [E][W]
    int32_t *cnt = reinterpret_cast<int32_t *>(mask + (size_t)E * W);  // [E+1]
    uint16_t *pre = reinterpret_cast<uint16_t *>(cnt + E + 1);          // [E][W]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

    for (int i = threadIdx.x; i < E * W; i += RT_NT) mask[i] = 0u;
    __syncthreads();

    // Phase 1: one warp per token; lane holds experts lane, lane+32, ...
    const int EP = (E + 31) >> 5;  // <= 8
    for (int t = warp; t < n; t += RT_NW) {
        uint32_t key[8];
        float val[8];
        bool bad = false;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int e = lane + 32 * q;
            if (q < EP && e < E) {
                val[q] = logits[(int64_t)t * E + e];
                bad |= !isfinite(val[q]);
                key[q] = float_key(val[q]);
            } else {
                val[q] = 0.f;
                key[q] = 0u;  // below every real key
            }
        }
        if (__any_sync(0xffffffffu, bad) && lane == 0) set_dev_error(status, RVQ_DEV_ERR_NONFINITE);
        uint32_t taken = 0u;
        float my_logit = 0.f;
        int my_idx = 0;
        for (int s = 0; s < k; ++s) {
            uint32_t bk = 0u;
            int bi = 0x7fffffff;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int e = lane + 32 * q;
                if (q < EP && e < E && !((taken >> q) & 1u) && key[q] > bk) {
                    bk = key[q];
                    bi = e;
                }
            }
            if (bi == 0x7fffffff) bk = 0u;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const uint32_t ok = __shfl_xor_sync(0xffffffffu, bk, o);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                if (ok > bk || (ok == bk && oi < bi)) {
                    bk = ok;
                    bi = oi;
                }
            }
            if (bi == 0x7fffffff) bi = 0;  // only with invalid inputs
            if ((bi & 31) == lane && bi < E) taken |= 1u << (bi >> 5);
            // fetch the winner's logit from the owner lane
            float wl = 0.f;
#pragma unroll
            for (int q = 0; q < 8; ++q)
                if ((bi >> 5) == q) wl = val[q];
            wl = __shfl_sync(0xffffffffu, wl, bi & 31);
            if (lane == s) {
                my_logit = wl;
                my_idx = bi;
            }
        }
        // weights: exp(l - l_max) / sum over the selection (l_max = first pick)
        const float lmax = __shfl_sync(0xffffffffu, my_logit, 0);
        float ex = (lane < k) ? expf(my_logit - lmax) : 0.f;
        float sum = ex;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        sum = __shfl_sync(0xffffffffu, sum, 0);  // one denominator for every slot
        if (lane < k) {
            idx[(int64_t)t * k + lane] = my_idx;
            wout[(int64_t)t * k + lane] = ex / sum;
            atomicOr(&mask[(size_t)my_idx * W + (t >> 5)], 1u << (t & 31));
        }
    }
    __syncthreads();

    // Phase 2: per-expert running counts over token words.
    for (int e = threadIdx.x; e < E; e += RT_NT) {
        int run = 0;
        for (int w = 0; w < W; ++w) {
            pre[(size_t)e * W + w] = (uint16_t)run;
            run += __popc(mask[(size_t)e * W + w]);
        }
        cnt[e] = run;
    }
    __syncthreads();
    // Exclusive scan of counts (E <= 256) by warp 0: 8 experts per lane.
    if (warp == 0) {
        int v[8];
        int s = 0;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int e = lane * 8 + q;
            v[q] = (e < E) ? cnt[e] : 0;
            s += v[q];
        }
        int incl = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        int run = incl - s;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int e = lane * 8 + q;
            if (e < E) {
                cnt[e] = run;  // now the exclusive offset
                offsets[e] = run;
            }
            run += v[q];
        }
        if (lane == 31) offsets[E] = run;
    }
    __syncthreads();

    // Phase 3: each (token, slot) lands at offset[e] + rank of t among e's tokens.
    for (int t = warp; t < n; t += RT_NW) {
        if (lane < k) {
            const int e = idx[(int64_t)t * k + lane];
            const size_t wi = (size_t)e * W + (t >> 5);
            const int pos = cnt[e] + pre[wi] + __popc(mask[wi] & ((1u << (t & 31)) - 1u));
            pairs[pos] = t * k + lane;
        }
    }
}

size_t route_smem(int n, int E) {
    const size_t W = (size_t)(n + 31) / 32;
    return (size_t)E * W * 4 + (size_t)(E + 1) * 4 + (size_t)E * W * 2 + 16;
}

}  // namespace

int route_max_tokens(int E) {
    if (E <= 0) return 0;
    const size_t per_w = (size_t)E * 6;
    const size_t avail = RT_SMEM_MAX - (size_t)(E + 1) * 4 - 16;
    size_t W = avail / per_w;
    if (W > 2047) W = 2047;  // keep counts inside uint16
    return (int)(W * 32);
}

rvq_status launch_router_logits(const float *wr, const float *bias, const void *x, int xdt, int n,
                                int E, int d, float *logits, cudaStream_t stream) {
    dim3 grid((E + LG_EB - 1) / LG_EB, (n + LG_TB - 1) / LG_TB);
    router_logits_kernel<<<grid, LG_NT, 0, stream>>>(wr, bias, x, xdt, n, E, d, logits);
    RVQ_LAUNCHED("router_logits");
    return RVQ_OK;
}

rvq_status launch_route(const float *logits, int n, int E, int k, int32_t *idx, float *w,
                        int32_t *offsets, int32_t *pairs, uint32_t *status, cudaStream_t stream,
                        bool pdl) {
    static int attr_done[64] = {0};
    int dev = 0;
    RVQ_CUDA(cudaGetDevice(&dev));
    if (dev < 64 && !attr_done[dev]) {
        RVQ_CUDA(cudaFuncSetAttribute(route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)RT_SMEM_MAX));
        attr_done[dev] = 1;
    }
    const size_t smem = route_smem(n, E);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(RT_NT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    RVQ_CUDA(cudaLaunchKernelEx(&cfg, route_kernel, logits, n, E, k, idx, w, offsets, pairs,
                                status));
    return RVQ_OK;
}

}  // namespace rvq
