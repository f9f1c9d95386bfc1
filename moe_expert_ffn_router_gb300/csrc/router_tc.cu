// Router logits on the tensor cores, for prefill-sized batches of bf16 tokens:
// logits[n][E] = x Wr^T (+ bias).
//
// The router is the linear map of the pages' resident router (it picks the
// experts of each layer) [GeekNews topic 32035, section "Read-ahead and router
// prediction"]; the readings of the rest (fp32 logits, the k largest) are
// those of the SIMT kernels in router.cu.
//
// At 2048 tokens x 256 experts x 7168 the product is a real contraction
// (3.8 GFLOP), so it runs as a tcgen05 GEMM.  fp32 accuracy with bf16
// operands: the bf16 tokens are exact, and Wr is split into three bf16 terms
// (w1 = bf16(w), w2 = bf16(w - w1), w3 = bf16(w - w1 - w2), 24 significant
// bits together), so x.w1 + x.w2 + x.w3 has exact products and fp32
// accumulation.
//  * A tile is 128 tokens (TMEM lanes) x 128 experts (fp32 accumulator
//    columns).  A cluster of 4 CTAs splits K; each CTA streams 64-column
//    slices of x and of the three Wr terms by TMA (128-byte swizzle, three
//    stages) and issues 12 MMAs (K=16 each) per slice from one thread.
//  * Slice ks accumulates into accumulator ks mod 4 (all 512 TMEM columns):
//    the tensor pipe's fp32 accumulation error grows with the length of a
//    chain, and one chain over a CTA's 336 MMAs measured 5e-5 against logits
//    of RMS 2.5, twice the 1e-5 x RMS bound.  The epilogue adds the four in a
//    fixed order.
//  * The partial tiles go to shared memory; rank r of the cluster adds the 4
//    partials of its 32 tokens in rank order (distributed shared memory) and
//    the bias, so the sums run in a fixed order.
//  * Every wait is bounded (1 s, then RVQ_DEV_ERR_TIMEOUT and an orderly
//    exit with the TMEM columns released).
#include "internal.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cooperative_groups.h>
#include <string.h>

namespace rvq {
namespace {

constexpr int RC_M = 128;   // tokens per tile
constexpr int RC_N = 128;   // experts per tile
constexpr int RC_KC = 64;   // K per stage: one 128-byte swizzled bf16 row
constexpr int RC_ST = 3;    // pipeline stages
constexpr int RC_S = 4;     // CTAs of a cluster (K split)
constexpr int RC_ABYTES = RC_M * RC_KC * 2;          // 16 KiB of tokens
constexpr int RC_BBYTES = RC_N * RC_KC * 2;          // 16 KiB per Wr term
constexpr int RC_STAGE = RC_ABYTES + 3 * RC_BBYTES;  // 64 KiB
constexpr int RC_PP = RC_N + 4;  // partial tile pitch in floats (16-byte store phases conflict-free)
constexpr int RC_SMEM = RC_ST * RC_STAGE + 256;
constexpr int RC_THREADS = 128;
constexpr int RC_NACC = 4;  // accumulators (TMEM columns RC_N each)
constexpr unsigned long long kRcWaitNs = 1000000000ull;
static_assert(RC_M * RC_PP * 4 <= RC_ST * RC_STAGE, "the partial tile fits the stages");
static_assert(RC_M % RC_S == 0 && RC_THREADS == RC_N, "reduction shape");

__device__ __forceinline__ uint32_t rc_smem(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ unsigned long long rc_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ bool rc_try(uint32_t mbar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.b32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(mbar), "r"(parity)
        : "memory");
    return done != 0;
}

// Bounded wait; false once another role has aborted or after kRcWaitNs
// (then this thread raises the abort flag and records the timeout).
__device__ __forceinline__ bool rc_wait(uint32_t mbar, uint32_t parity, volatile int *abort_flag,
                                        uint32_t *status) {
    if (rc_try(mbar, parity)) return true;
    const unsigned long long t0 = rc_ns();
    for (;;) {
        if (rc_try(mbar, parity)) return true;
        if (*abort_flag) return false;
        if (rc_ns() - t0 > kRcWaitNs) {
            *abort_flag = 1;
            if (status) set_dev_error(status, RVQ_DEV_ERR_TIMEOUT);
            return false;
        }
    }
}

// K-major operand, 128-byte swizzle: 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t rc_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)1u << 16;            // leading offset (unused for swizzled K-major)
    d |= (uint64_t)(1024u >> 4) << 32;  // stride offset
    d |= (uint64_t)1u << 46;            // descriptor version (sm_100 family)
    d |= (uint64_t)2u << 61;            // SWIZZLE_128B
    return d;
}

// kind::f16: D fp32, A and B bf16, both K-major.
constexpr uint32_t kRcIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(RC_N >> 3) << 17) |
                              ((uint32_t)(RC_M >> 4) << 24);

__device__ __forceinline__ void rc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t acc) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %3, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %4, p;\n}\n" ::"r"(d),
        "l"(a), "l"(b), "r"(acc), "r"(kRcIdesc));
}

__device__ __forceinline__ void rc_commit(uint32_t mbar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     mbar)
                 : "memory");
}

__device__ __forceinline__ void rc_tma(uint32_t dst, const CUtensorMap *tm, int col, int row,
                                       uint32_t mbar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(col), "r"(row), "r"(mbar)
        : "memory");
}

// w -> three bf16 terms, term t of element i at w3[t * count + i].
__global__ void __launch_bounds__(256) router_split_kernel(const float4 *__restrict__ wr,
                                                           int64_t count4, uint2 *__restrict__ w3) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count4;
         i += (int64_t)gridDim.x * blockDim.x) {
        const float4 v = __ldg(wr + i);
        const float a[4] = {v.x, v.y, v.z, v.w};
        uint32_t t[3][2];
#pragma unroll
        for (int j = 0; j < 4; j += 2) {
            uint32_t h[3][2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const __nv_bfloat16 b1 = __float2bfloat16_rn(a[j + u]);
                const float r1 = a[j + u] - __bfloat162float(b1);
                const __nv_bfloat16 b2 = __float2bfloat16_rn(r1);
                const __nv_bfloat16 b3 = __float2bfloat16_rn(r1 - __bfloat162float(b2));
                h[0][u] = __bfloat16_as_ushort(b1);
                h[1][u] = __bfloat16_as_ushort(b2);
                h[2][u] = __bfloat16_as_ushort(b3);
            }
#pragma unroll
            for (int s = 0; s < 3; ++s) t[s][j >> 1] = h[s][0] | (h[s][1] << 16);
        }
#pragma unroll
        for (int s = 0; s < 3; ++s) w3[s * count4 + i] = make_uint2(t[s][0], t[s][1]);
    }
}

__global__ void __launch_bounds__(RC_THREADS, 1) router_logits_tc_kernel(
    const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
    const float *__restrict__ bias, int n, int E, int d, float *__restrict__ logits,
    uint32_t *status) {
    extern __shared__ __align__(1024) uint8_t smem[];
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * RC_M, e0 = blockIdx.y * RC_N;
    const int dk = d / RC_S, kb = (int)blockIdx.z * dk, nk = dk / RC_KC;
    uint8_t *bars = smem + RC_ST * RC_STAGE;
    const uint32_t full0 = rc_smem(bars), empty0 = full0 + 8 * RC_ST, accb = empty0 + 8 * RC_ST;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bars + 8 * (2 * RC_ST + 1));
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 8 * (2 * RC_ST + 1) + 4);
    if (threadIdx.x == 0) {
        for (int s = 0; s < RC_ST; ++s) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(full0 + 8 * s));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(empty0 + 8 * s));
        }
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(accb));
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        // one CTA per SM (shared memory), so the allocation never waits
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         rc_smem(tslot)),
                     "r"((uint32_t)(RC_NACC * RC_N)));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tslot;

    if (warp == 0 && lane == 0) {
        // TMA producer: the token slice and the three Wr-term slices per stage
        for (int ks = 0; ks < nk; ++ks) {
            const int s = ks % RC_ST;
            if (ks >= RC_ST && !rc_wait(empty0 + 8 * s, ((ks / RC_ST) - 1) & 1, abort_flag, status))
                break;
            const uint32_t st = rc_smem(smem + s * RC_STAGE);
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(full0 + 8 * s),
                         "r"((uint32_t)RC_STAGE)
                         : "memory");
            const int kx = kb + ks * RC_KC;
            rc_tma(st, &tm_x, kx, m0, full0 + 8 * s);
#pragma unroll
            for (int t = 0; t < 3; ++t)
                rc_tma(st + RC_ABYTES + t * RC_BBYTES, &tm_w, kx, t * E + e0, full0 + 8 * s);
        }
    } else if (warp == 1 && lane == 0) {
        // MMA issuer: 4 K=16 steps x 3 Wr terms per slice, one commit per slice
        for (int ks = 0; ks < nk; ++ks) {
            const int s = ks % RC_ST;
            if (!rc_wait(full0 + 8 * s, (ks / RC_ST) & 1, abort_flag, status)) break;
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const uint32_t st = rc_smem(smem + s * RC_STAGE);
            const uint64_t ad = rc_desc(st);
            const uint32_t dacc = tmem + (uint32_t)((ks % RC_NACC) * RC_N);
#pragma unroll
            for (int kk = 0; kk < RC_KC / 16; ++kk)
#pragma unroll
                for (int t = 0; t < 3; ++t)
                    rc_mma(dacc, ad + 2 * kk, rc_desc(st + RC_ABYTES + t * RC_BBYTES) + 2 * kk,
                           (ks >= RC_NACC || kk > 0 || t > 0) ? 1u : 0u);
            rc_commit(empty0 + 8 * s);
        }
        rc_commit(accb);  // also after an abort, so the epilogue's wait ends
    }
    __syncwarp();

    // epilogue: warp w holds tokens 32 w .. 32 w + 31 (its TMEM lane quarter)
    float *part = reinterpret_cast<float *>(smem);  // the stages are free once accb completes
    const bool ok = rc_wait(accb, 0, abort_flag, status) && !*abort_flag;
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (ok) {
        float *row = part + (32 * warp + lane) * RC_PP;
        const int nacc = nk < RC_NACC ? nk : RC_NACC;
#pragma unroll 1
        for (int c = 0; c < RC_N / 32; ++c) {
            float v[32];
#pragma unroll 1
            for (int a = 0; a < nacc; ++a) {
                uint32_t r[32];
                asm volatile(
                    "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,"
                    "%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,"
                    "%31}, [%32];"
                    : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                      "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                      "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
                      "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
                      "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]),
                      "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                    : "r"(tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)(a * RC_N + 32 * c)));
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    v[j] = a == 0 ? __uint_as_float(r[j]) : v[j] + __uint_as_float(r[j]);
            }
#pragma unroll
            for (int j = 0; j < 32; j += 4)
                *reinterpret_cast<float4 *>(row + 32 * c + j) =
                    make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    cluster.sync();  // every partial tile of the cluster is in place
    if (ok) {
        // rank r: tokens 32 r .. 32 r + 31; thread j: expert e0 + j
        const unsigned r = cluster.block_rank();
        const int j = threadIdx.x;
        const float b = bias ? bias[e0 + j] : 0.f;
        const float *peer[RC_S];
#pragma unroll
        for (int q = 0; q < RC_S; ++q) peer[q] = cluster.map_shared_rank(part, q);
        for (int i = 0; i < RC_M / RC_S; ++i) {
            const int t = (int)r * (RC_M / RC_S) + i;
            float v = peer[0][t * RC_PP + j];
#pragma unroll
            for (int q = 1; q < RC_S; ++q) v += peer[q][t * RC_PP + j];
            if (m0 + t < n) logits[(int64_t)(m0 + t) * E + e0 + j] = v + b;
        }
    }
    cluster.sync();  // the peers' tiles stay in place until read
    if (warp == 0) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"((uint32_t)(RC_NACC * RC_N)));
    }
}

}  // namespace

bool router_tc_supported(int n, int E, int d) {
    return n >= RC_M && E % RC_N == 0 && d % (RC_S * RC_KC) == 0;
}

size_t router_tc_split_bytes(int E, int d) { return (size_t)3 * E * d * 2; }

rvq_status launch_router_logits_tc(const float *wr, const float *bias, const void *x, int n,
                                   int E, int d, float *logits, void *wsplit, uint32_t *status,
                                   cudaStream_t stream) {
    if (!router_tc_supported(n, E, d) || ((uintptr_t)x & 15u) || ((uintptr_t)wsplit & 15u) ||
        ((uintptr_t)wr & 15u)) {
        set_error("router (tensor cores): n %d / E %d / d %d or alignment not supported", n, E, d);
        return RVQ_EINVAL;
    }
    static std::atomic<int> attr_done[64];  // per device; setting twice is harmless
    int dev = 0;
    RVQ_CUDA(cudaGetDevice(&dev));
    if (dev < 64 && !attr_done[dev]) {
        RVQ_CUDA(cudaFuncSetAttribute(router_logits_tc_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, RC_SMEM));
        attr_done[dev] = 1;
    }
    const int64_t count4 = (int64_t)E * d / 4;
    router_split_kernel<<<(unsigned)(2 * num_sms()), 256, 0, stream>>>(
        reinterpret_cast<const float4 *>(wr), count4, reinterpret_cast<uint2 *>(wsplit));
    RVQ_LAUNCHED("router_split");
    const PFN_cuTensorMapEncodeTiled_v12000 encode =
        reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encoder_entry());
    if (encode == nullptr) {
        set_error("router (tensor cores): cuTensorMapEncodeTiled is not available");
        return RVQ_ECUDA;
    }
    // tokens: d x n bf16 (rows past n read as zero); Wr terms: d x 3E bf16
    CUtensorMap tm_x, tm_w;
    memset(&tm_x, 0, sizeof(tm_x));
    memset(&tm_w, 0, sizeof(tm_w));
    const cuuint32_t box[2] = {(cuuint32_t)RC_KC, (cuuint32_t)RC_M};
    const cuuint32_t estr[2] = {1u, 1u};
    const cuuint64_t dx[2] = {(cuuint64_t)d, (cuuint64_t)n};
    const cuuint64_t dw[2] = {(cuuint64_t)d, (cuuint64_t)3 * E};
    const cuuint64_t pitch[1] = {(cuuint64_t)d * 2u};
    CUresult r = encode(&tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(x), dx,
                        pitch, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r == CUDA_SUCCESS)
        r = encode(&tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, wsplit, dw, pitch, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        set_error("router (tensor cores): cuTensorMapEncodeTiled failed (%d)", (int)r);
        return RVQ_ECUDA;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((n + RC_M - 1) / RC_M), (unsigned)(E / RC_N), (unsigned)RC_S);
    cfg.blockDim = dim3(RC_THREADS);
    cfg.dynamicSmemBytes = RC_SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = (unsigned)RC_S;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    RVQ_CUDA(cudaLaunchKernelEx(&cfg, router_logits_tc_kernel, tm_x, tm_w, bias, n, E, d, logits,
                                status));
    RVQ_LAUNCHED("router_logits_tc");
    return RVQ_OK;
}

}  // namespace rvq
