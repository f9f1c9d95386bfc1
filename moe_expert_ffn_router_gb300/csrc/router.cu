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

#include <cooperative_groups.h>

namespace rvq {
namespace {

// ------------------------------------------------------------------ logits
// One block per (expert, tile of TB tokens); 256 threads stride the hidden
// dimension four elements at a time (128-bit loads of the router row).
constexpr int LG_NT = 256;

template <int TB>
__global__ void __launch_bounds__(LG_NT) router_logits_kernel(
    const float *__restrict__ wr, const float *__restrict__ bias, const void *__restrict__ x,
    int xdt, int n, int E, int d, float *__restrict__ logits) {
    const int e = blockIdx.x;
    const int t0 = blockIdx.y * TB;
    const int nt = min(TB, n - t0);
    // Launched early behind the preceding kernel: the block's router row is
    // requested into L2 before the dependency wait (a hint only: every load
    // below comes after the wait, so a row written by that kernel is still
    // read as it left it), hiding its DRAM time behind the preceding kernel.
    if (threadIdx.x == 0 && blockIdx.y == 0) {
        const float *row = wr + (int64_t)e * d;
        if (((uintptr_t)row & 15u) == 0 && (d & 3) == 0)
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(row), "r"((uint32_t)d * 4u)
                         : "memory");
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    float acc[TB];
#pragma unroll
    for (int b = 0; b < TB; ++b) acc[b] = 0.f;
    const float4 *w4 = reinterpret_cast<const float4 *>(wr + (int64_t)e * d);
    const int d4 = d >> 2;
    // every load of a thread in flight at once (d = 7168: 7 per thread)
#pragma unroll 8
    for (int c4 = threadIdx.x; c4 < d4; c4 += LG_NT) {
        const float4 wv = __ldg(w4 + c4);
#pragma unroll
        for (int b = 0; b < TB; ++b) {
            if (b < nt) {
                const int64_t base = (int64_t)(t0 + b) * d + c4 * 4;
                float4 xv;
                if (xdt == RVQ_BF16) {
                    const uint2 q = __ldg(reinterpret_cast<const uint2 *>(
                        reinterpret_cast<const uint16_t *>(x) + base));
                    xv = make_float4(__uint_as_float(q.x << 16), __uint_as_float(q.x & 0xFFFF0000u),
                                     __uint_as_float(q.y << 16), __uint_as_float(q.y & 0xFFFF0000u));
                } else {
                    xv = __ldg(reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(x) + base));
                }
                acc[b] = fmaf(wv.x, xv.x, acc[b]);
                acc[b] = fmaf(wv.y, xv.y, acc[b]);
                acc[b] = fmaf(wv.z, xv.z, acc[b]);
                acc[b] = fmaf(wv.w, xv.w, acc[b]);
            }
        }
    }
    __shared__ float red[LG_NT / 32][TB];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int b = 0; b < TB; ++b) {
        float v = acc[b];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) red[warp][b] = v;
    }
    __syncthreads();
    if (threadIdx.x < nt) {
        float v = 0.f;
#pragma unroll
        for (int q = 0; q < LG_NT / 32; ++q) v += red[q][threadIdx.x];
        if (bias) v += bias[e];
        logits[(int64_t)(t0 + threadIdx.x) * E + e] = v;
    }
}

// One token of a pre-norm layer: every block derives the RMS factor of h
// itself (the 28 KB row is read from L2 by all of them), rounds h / rms to
// bf16 exactly as the RMS norm kernel does and takes the dot product with its
// router row in the order router_logits_kernel<1> uses; block 0 also writes
// the normalised row for the expert FFN.  One launch instead of two on the
// decode critical path.
__global__ void __launch_bounds__(LG_NT) router_norm_logits_kernel(
    const float *__restrict__ wr, const float *__restrict__ bias, const void *__restrict__ h,
    int hdt, int E, int d, float eps, uint16_t *__restrict__ xn, float *__restrict__ logits) {
    __shared__ float red[LG_NT / 32];
    const int e = blockIdx.x;
    if (threadIdx.x == 0) {
        const float *row = wr + (int64_t)e * d;
        if (((uintptr_t)row & 15u) == 0 && (d & 3) == 0)
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(row), "r"((uint32_t)d * 4u)
                         : "memory");
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    const float inv = block_rms_inv(h, hdt, 0, d, eps, red);
    const float4 *w4 = reinterpret_cast<const float4 *>(wr + (int64_t)e * d);
    const int d4 = d >> 2;
    float acc = 0.f;
#pragma unroll 8
    for (int c4 = threadIdx.x; c4 < d4; c4 += LG_NT) {
        const float4 wv = __ldg(w4 + c4);
        const float4 v = load4(h, hdt, (int64_t)c4 * 4);
        uint2 q;
        q.x = bf16x2_bits(v.x * inv, v.y * inv);
        q.y = bf16x2_bits(v.z * inv, v.w * inv);
        if (e == 0) *reinterpret_cast<uint2 *>(xn + (int64_t)c4 * 4) = q;
        acc = fmaf(wv.x, __uint_as_float(q.x << 16), acc);
        acc = fmaf(wv.y, __uint_as_float(q.x & 0xFFFF0000u), acc);
        acc = fmaf(wv.z, __uint_as_float(q.y << 16), acc);
        acc = fmaf(wv.w, __uint_as_float(q.y & 0xFFFF0000u), acc);
    }
    __syncthreads();  // every warp has read red[] (the RMS sum) before it is reused
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) red[warp] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        float v = 0.f;
#pragma unroll
        for (int q = 0; q < LG_NT / 32; ++q) v += red[q];
        if (bias) v += bias[e];
        logits[e] = v;
    }
}

// Prefill-sized batches: a tiled fp32 GEMM, logits[n][E] = x Wr^T.  Each
// output tile of 64 tokens x 64 experts belongs to a cluster of LT_S blocks
// that split the hidden dimension; in a block 256 threads hold 4 x 4 outputs
// each, and K runs in slices of 32 staged (k-major, fp32) in shared memory
// with the next slice prefetched into registers.  (One block per tile over
// the whole of K leaves 2048 x 256 logits at 128 blocks: most of the GPU
// idle.)  The cluster's rank-0 block adds the partial tiles from its peers'
// shared memory in rank order, so sums run in a fixed order and the result
// does not depend on the launch.
constexpr int LT_T = 64, LT_E = 64, LT_K = 32, LT_PAD = 4, LT_S = 4;

__global__ void __launch_bounds__(256) router_logits_tiled_kernel(
    const float *__restrict__ wr, const float *__restrict__ bias, const void *__restrict__ x,
    int xdt, int n, int E, int d, float *__restrict__ logits) {
    // staging for the K slices; afterwards this block's partial tile
    __shared__ __align__(16) float stage[2 * LT_K * (LT_T + LT_PAD)];
    static_assert(LT_E + LT_PAD == LT_T + LT_PAD && LT_T * LT_E <= 2 * LT_K * (LT_T + LT_PAD),
                  "partial tile fits the staging area");
    float (*xs)[LT_T + LT_PAD] = reinterpret_cast<float (*)[LT_T + LT_PAD]>(stage);
    float (*ws)[LT_E + LT_PAD] =
        reinterpret_cast<float (*)[LT_E + LT_PAD]>(stage + LT_K * (LT_T + LT_PAD));
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int e0 = blockIdx.x * LT_E, t0 = blockIdx.y * LT_T;
    // this block's share of K (gridDim.z = blocks of the cluster)
    const int dk = d / (int)gridDim.z;
    const int kb = (int)blockIdx.z * dk, ke = kb + dk;
    // loader: row = tid / 4 (token or expert), 8 consecutive k at (tid % 4) * 8
    const int lr = tid >> 2, lk = (tid & 3) * 8;
    const bool xin = t0 + lr < n, win = e0 + lr < E;
    const int64_t xrow = (int64_t)(t0 + lr) * d, wrow = (int64_t)(e0 + lr) * d;
    float xv[8], wv[8];
    auto load = [&](int k0) {
        if (xin) {
            if (xdt == RVQ_BF16) {
                const uint4 q = __ldg(reinterpret_cast<const uint4 *>(
                    reinterpret_cast<const uint16_t *>(x) + xrow + k0 + lk));
                const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    xv[2 * i] = __uint_as_float(w[i] << 16);
                    xv[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
                }
            } else {
                const float4 *p = reinterpret_cast<const float4 *>(
                    reinterpret_cast<const float *>(x) + xrow + k0 + lk);
                const float4 a = __ldg(p), b = __ldg(p + 1);
                xv[0] = a.x; xv[1] = a.y; xv[2] = a.z; xv[3] = a.w;
                xv[4] = b.x; xv[5] = b.y; xv[6] = b.z; xv[7] = b.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) xv[i] = 0.f;
        }
        if (win) {
            const float4 *p = reinterpret_cast<const float4 *>(wr + wrow + k0 + lk);
            const float4 a = __ldg(p), b = __ldg(p + 1);
            wv[0] = a.x; wv[1] = a.y; wv[2] = a.z; wv[3] = a.w;
            wv[4] = b.x; wv[5] = b.y; wv[6] = b.z; wv[7] = b.w;
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) wv[i] = 0.f;
        }
    };
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    load(kb);
    for (int k0 = kb; k0 < ke; k0 += LT_K) {
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            xs[lk + i][lr] = xv[i];
            ws[lk + i][lr] = wv[i];
        }
        __syncthreads();
        if (k0 + LT_K < ke) load(k0 + LT_K);
        // two-level sums (a slice of 32 products, then across slices) keep the
        // rounding error of the 7168-term dot products near the tree-sum level
        float part[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) part[i][j] = 0.f;
#pragma unroll
        for (int kk = 0; kk < LT_K; ++kk) {
            const float4 a = *reinterpret_cast<const float4 *>(&xs[kk][ty * 4]);
            const float4 b = *reinterpret_cast<const float4 *>(&ws[kk][tx * 4]);
            const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) part[i][j] = fmaf(av[i], bv[j], part[i][j]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] += part[i][j];
    }
    // partial tile -> shared memory; rank 0 adds the peers' tiles in rank order
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    float *part = stage;  // [LT_T][LT_E]
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) part[(ty * 4 + i) * LT_E + tx * 4 + j] = acc[i][j];
    cluster.sync();
    if (cluster.block_rank() == 0) {
        for (unsigned r = 1; r < cluster.num_blocks(); ++r) {
            const float *peer = cluster.map_shared_rank(part, r);
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] += peer[(ty * 4 + i) * LT_E + tx * 4 + j];
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int t = t0 + ty * 4 + i;
            if (t >= n) continue;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int e = e0 + tx * 4 + j;
                if (e < E) logits[(int64_t)t * E + e] = acc[i][j] + (bias ? bias[e] : 0.f);
            }
        }
    }
    // the peers' tiles stay in place until rank 0 has read them
    cluster.sync();
}

// ------------------------------------------------------------------- route
constexpr size_t RT_SMEM_MAX = 200 * 1024;
constexpr int RT_KEEP = 4;  // tokens per warp whose selection stays in registers

// Order-preserving key for fp32 (after -0 -> +0): larger float, larger key.
__device__ __forceinline__ uint32_t float_key(float f) {
    uint32_t u = __float_as_uint(f + 0.0f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_float(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// One warp selects the k largest keys of one token's logits with warp-wide
// max/min reductions (one redux.sync each per pick); lane s < k returns the
// s-th pick and its renormalised softmax weight.
__device__ __forceinline__ void warp_topk(const float *__restrict__ row, int E, int k, int lane,
                                          uint32_t *status, int &my_idx, float &my_w) {
    const int EP = (E + 31) >> 5;  // <= 8
    uint32_t key[8];
    bool bad = false;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const int e = lane + 32 * q;
        if (q < EP && e < E) {
            const float v = row[e];
            bad |= !isfinite(v);
            key[q] = float_key(v);
        } else {
            key[q] = 0u;  // below every real key
        }
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) set_dev_error(status, RVQ_DEV_ERR_NONFINITE);
    // lane-local best (ties: lower q = lower expert index)
    uint32_t taken = 0u, lk = 0u;
    int lq = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q)
        if (key[q] > lk) { lk = key[q]; lq = q; }
    uint32_t kmax0 = 0u, my_key = 0u;
    my_idx = 0;
    for (int s = 0; s < k; ++s) {
        const uint32_t kmax = __reduce_max_sync(0xffffffffu, lk);
        const uint32_t cand = (lk == kmax) ? (uint32_t)(lane + 32 * lq) : 0xffffffffu;
        uint32_t emin = __reduce_min_sync(0xffffffffu, cand);
        if (emin >= (uint32_t)E) emin = 0;  // only with invalid inputs
        if (s == 0) kmax0 = kmax;
        if (lane == s) {
            my_idx = (int)emin;
            my_key = kmax;
        }
        if ((int)(emin & 31) == lane) {
            taken |= 1u << (emin >> 5);
            lk = 0u;
            lq = 0;
#pragma unroll
            for (int q = 0; q < 8; ++q)
                if (!((taken >> q) & 1u) && key[q] > lk) { lk = key[q]; lq = q; }
        }
    }
    // w = exp(l - l_max) / sum over the selection (l_max = first pick)
    const float lmax = key_float(kmax0);
    const float ex = (lane < k) ? expf(key_float(my_key) - lmax) : 0.f;
    float sum = ex;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    sum = __shfl_sync(0xffffffffu, sum, 0);  // one denominator for every slot
    my_w = ex / sum;
}

// Selection only, one warp per token over the whole grid (prefill batches);
// the grouping follows in route_kernel<NT, false>.
__global__ void __launch_bounds__(256) route_select_kernel(const float *__restrict__ logits, int n,
                                                           int E, int k, int32_t *__restrict__ idx,
                                                           float *__restrict__ wout,
                                                           uint32_t *status) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t >= n) return;
    int my_idx;
    float my_w;
    warp_topk(logits + (int64_t)t * E, E, k, lane, status, my_idx, my_w);
    if (lane < k) {
        idx[(int64_t)t * k + lane] = my_idx;
        wout[(int64_t)t * k + lane] = my_w;
    }
}

// One block.  Phase 1: one warp per token selects its k experts (SELECT), or
// the selection is read back from idx.  Phase 2: per-expert token bitmaps give
// counts and running ranks; phase 3 scatters each (token, slot) to
// offsets[e] + rank, i.e. pairs sorted by (expert, token).
template <int NT, bool SELECT>
__global__ void __launch_bounds__(NT, 1) route_kernel(const float *__restrict__ logits, int n,
                                                      int E, int k, int32_t *idx,
                                                      float *__restrict__ wout,
                                                      int32_t *__restrict__ offsets,
                                                      int32_t *__restrict__ pairs,
                                                      uint32_t *status, const LutJob plan,
                                                      int4 *__restrict__ pd) {
    constexpr int NWARP = NT / 32;
    extern __shared__ __align__(16) uint32_t rsm[];
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    const int W = (n + 31) >> 5;
    uint32_t *mask = rsm;                                               // [E][W]
    int32_t *cnt = reinterpret_cast<int32_t *>(mask + (size_t)E * W);   // [E+1]
    uint16_t *pre = reinterpret_cast<uint16_t *>(cnt + E + 1);          // [E][W]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

    for (int i = threadIdx.x; i < E * W; i += NT) mask[i] = 0u;
    __syncthreads();

    int keep[RT_KEEP];
#pragma unroll
    for (int r = 0; r < RT_KEEP; ++r) keep[r] = 0;
    int r = 0;
    if (SELECT) {
        for (int t = warp; t < n; t += NWARP, ++r) {
            int my_idx;
            float my_w;
            warp_topk(logits + (int64_t)t * E, E, k, lane, status, my_idx, my_w);
            if (lane < k) {
                idx[(int64_t)t * k + lane] = my_idx;
                wout[(int64_t)t * k + lane] = my_w;
                atomicOr(&mask[(size_t)my_idx * W + (t >> 5)], 1u << (t & 31));
            }
#pragma unroll
            for (int q = 0; q < RT_KEEP; ++q)
                if (q == r) keep[q] = my_idx;
        }
    } else {
        for (int i = threadIdx.x; i < n * k; i += NT) {
            const int t = i / k;
            const int e = idx[i];
            atomicOr(&mask[(size_t)e * W + (t >> 5)], 1u << (t & 31));
        }
    }
    __syncthreads();

    // Phase 2: per-expert running counts over token words.
    for (int e = threadIdx.x; e < E; e += NT) {
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
    r = 0;
    for (int t = warp; t < n; t += NWARP, ++r) {
        if (lane < k) {
            int e = 0;
            if (SELECT && r < RT_KEEP) {
#pragma unroll
                for (int q = 0; q < RT_KEEP; ++q)
                    if (q == r) e = keep[q];
            } else {
                e = idx[(int64_t)t * k + lane];
            }
            const size_t wi = (size_t)e * W + (t >> 5);
            const int pos = cnt[e] + pre[wi] + __popc(mask[wi] & ((1u << (t & 31)) - 1u));
            pairs[pos] = t * k + lane;
            // the decode plan's descriptor of this position (group sizes are
            // not needed: the plan's tc_min_tokens is <= 0)
            if (pd) pd[pos] = pair_desc(plan, e, 0, t * k + lane);
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
    // the small-batch kernels may start behind the preceding kernel
    // (programmatic dependent launch; they wait before reading anything)
    cudaLaunchConfig_t pcfg = {};
    cudaLaunchAttribute pattr[1];
    pattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pattr[0].val.programmaticStreamSerializationAllowed = 1;
    pcfg.attrs = pattr;
    pcfg.numAttrs = 1;
    pcfg.blockDim = dim3(LG_NT);
    pcfg.stream = stream;
    if (n == 1) {
        pcfg.gridDim = dim3((unsigned)E, 1);
        RVQ_CUDA(cudaLaunchKernelEx(&pcfg, router_logits_kernel<1>, wr, bias, x, xdt, n, E, d,
                                    logits));
    } else if (n > 64 && d % LT_K == 0) {
        // a cluster of LT_S blocks per output tile when K splits evenly
        const int S = d % (LT_S * LT_K) == 0 ? LT_S : 1;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)((E + LT_E - 1) / LT_E), (unsigned)((n + LT_T - 1) / LT_T),
                           (unsigned)S);
        cfg.blockDim = dim3(256);
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 1;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = (unsigned)S;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        RVQ_CUDA(cudaLaunchKernelEx(&cfg, router_logits_tiled_kernel, wr, bias, x, xdt, n, E, d,
                                    logits));
    } else {
        pcfg.gridDim = dim3((unsigned)E, (unsigned)((n + 7) / 8));
        RVQ_CUDA(cudaLaunchKernelEx(&pcfg, router_logits_kernel<8>, wr, bias, x, xdt, n, E, d,
                                    logits));
    }
    RVQ_LAUNCHED("router_logits");
    return RVQ_OK;
}

rvq_status launch_router_norm_logits(const float *wr, const float *bias, const void *h, int hdt,
                                     int E, int d, float eps, uint16_t *xn, float *logits,
                                     cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3((unsigned)E);
    cfg.blockDim = dim3(LG_NT);
    cfg.stream = stream;
    RVQ_CUDA(cudaLaunchKernelEx(&cfg, router_norm_logits_kernel, wr, bias, h, hdt, E, d, eps, xn,
                                logits));
    RVQ_LAUNCHED("router_norm_logits");
    return RVQ_OK;
}

template <int NT, bool SELECT>
rvq_status launch_route_nt(const float *logits, int n, int E, int k, int32_t *idx, float *w,
                           int32_t *offsets, int32_t *pairs, uint32_t *status,
                           cudaStream_t stream, bool pdl, const LutJob *plan, int4 *pd) {
    static std::atomic<int> attr_done[64];  // per device; setting twice is harmless
    int dev = 0;
    RVQ_CUDA(cudaGetDevice(&dev));
    if (dev < 64 && !attr_done[dev]) {
        RVQ_CUDA(cudaFuncSetAttribute(route_kernel<NT, SELECT>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)RT_SMEM_MAX));
        attr_done[dev] = 1;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = route_smem(n, E);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    const LutJob none = {};
    RVQ_CUDA(cudaLaunchKernelEx(&cfg, route_kernel<NT, SELECT>, logits, n, E, k, idx, w, offsets,
                                pairs, status, plan ? *plan : none, plan ? pd : nullptr));
    return RVQ_OK;
}

rvq_status launch_route(const float *logits, int n, int E, int k, int32_t *idx, float *w,
                        int32_t *offsets, int32_t *pairs, uint32_t *status, cudaStream_t stream,
                        bool pdl, const LutJob *plan, int4 *pd) {
    if (plan && (n > kRouteSingleBlockTokens || !pd || plan->tc_min_tokens > 0)) {
        set_error("route: the fused pair plan needs n <= %d, pd and no tensor-core dispatch",
                  kRouteSingleBlockTokens);
        return RVQ_EINVAL;
    }
    if (n <= kRouteSingleBlockTokens)
        return launch_route_nt<256, true>(logits, n, E, k, idx, w, offsets, pairs, status, stream,
                                          pdl, plan, pd);
    // larger batches: the selection spreads over the grid, the grouping stays in one block
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((n + 7) / 8));
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    RVQ_CUDA(cudaLaunchKernelEx(&cfg, route_select_kernel, logits, n, E, k, idx, w, status));
    return launch_route_nt<1024, false>(logits, n, E, k, idx, w, offsets, pairs, status, stream,
                                        pdl, nullptr, nullptr);
}

}  // namespace rvq
