// Prefill path of the expert FFN: RVQ code tiles dequantised to bf16 in
// shared memory feed tcgen05 tensor-core GEMMs (fp32 accumulators in TMEM).
//
// For prefill-sized groups (tens to hundreds of tokens per expert) the FFN is
// a real dense contraction, so the weights are decoded once per tile --
// W[r][8j+i] = C1[c(r,j,1)][i] + C2[c(r,j,2)][i] + C3[c(r,j,3)][i], the residual
// decode of the pages ("WASTE Inference Engine", section "Residual Vector
// Quantization (RVQ)") -- rounded to bf16 and multiplied on the tensor cores.
//
// GEMM orientation (swap-AB): A = 128 rows of W x 64 K-columns (K-major), B =
// up to 256 tokens of the expert's group x 64 K-columns (K-major), D = W x^T
// (128 rows x N tokens, fp32, in TMEM).  One RVQ chunk (8 weights) is exactly
// one 16-byte unit of the 128-byte swizzle row, so a decoded chunk is stored
// with one 128-bit shared-memory store at its swizzled position.
//  * gate/up launch: two accumulators (gate at TMEM column 0, up at 256); the
//    epilogue computes h = silu(g) * u and writes it as bf16 [pair][f].
//  * down launch: one accumulator; the epilogue writes y fp32 [pair][d].
// Every mbarrier wait is bounded; on expiry the block records
// RVQ_DEV_ERR_TIMEOUT, frees its TMEM and returns.
#include "internal.cuh"

namespace rvq {
namespace {

constexpr int PF_NT = 128;                      // 4 warps <-> TMEM lanes 0..127 (rows of the tile)
constexpr int PF_M = 128;                       // rows of W per tile
constexpr int PF_NMAX = 256;                    // tokens per pass (MMA N)
constexpr int PF_KC = 64;                       // K columns per step: one 128-byte swizzle row
constexpr int kTileA = PF_M * PF_KC * 2;        // 16 KiB
constexpr int kTileB = PF_NMAX * PF_KC * 2;     // 32 KiB
constexpr int kCbF32 = 3 * 256 * 8 * 4;         // 24 KiB: one matrix's codebooks, fp32 [s][k][8]
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s: a bounded wait, never a hang

// shared memory layout (dynamic, 1024-byte aligned)
constexpr int OFF_A = 0;                        // 2 A tiles
constexpr int OFF_B = 2 * kTileA;               // B tile
constexpr int OFF_CB = OFF_B + kTileB;          // 2 fp32 codebooks
constexpr int OFF_ENT = OFF_CB + 2 * kCbF32;    // pair entries of the pass [256] int32
constexpr int OFF_Q = OFF_ENT + PF_NMAX * 4;    // per-expert pass prefix [257] int32
constexpr int OFF_MISC = OFF_Q + 260 * 4;       // mbarrier, tmem slot, flags
constexpr int kPfSmem = OFF_MISC + 64 + 1024;  // + slack to align the tile base to 1024 B

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

// tcgen05 shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row
// groups 1024 bytes apart (SBO), leading offset unused for swizzled K-major.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);        // start address
    d |= (uint64_t)1u << 16;                         // LBO (16 B, unused)
    d |= (uint64_t)(1024u >> 4) << 32;               // SBO = 1024 B
    d |= (uint64_t)1u << 46;                         // descriptor version (sm_100 family)
    d |= (uint64_t)2u << 61;                         // SWIZZLE_128B
    return d;
}

// Instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void mma_commit(uint32_t mbar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     mbar)
                 : "memory");
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait on an mbarrier phase; returns false after kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint32_t mbar, uint32_t parity) {
    const unsigned long long t0 = global_ns();
    for (;;) {
        uint32_t done;
        asm volatile(
            "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
            "selp.b32 %0, 1, 0, p;\n}\n"
            : "=r"(done)
            : "r"(mbar), "r"(parity)
            : "memory");
        if (done) return true;
        if (global_ns() - t0 > kWaitLimitNs) return false;
    }
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ uint32_t bf16_bits(float f) {
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// Code byte of (row r, chunk j, stage s) in the packed tile layout.
__device__ __forceinline__ uint8_t code_at(const uint8_t *codes, int RB, int r, int j, int s) {
    const int l = r & 31, g = j >> 5;
    const int t = ((j & 31) - l) & 31;
    return codes[((size_t)g * RB + (r >> 5)) * kTileBytes + ((s * 2 + (t >> 4)) * 32 + l) * 16 +
                 (t & 15)];
}

struct PfItem {
    int valid, e, o, n, npad, mt, j0;
};

__global__ void __launch_bounds__(PF_NT, 1) prefill_gemm_kernel(const PfJob job) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // the 128-byte swizzle is a function of shared-address bits 4..9: tiles
    // must start on 1024-byte boundaries of the shared window
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    int32_t *ent = reinterpret_cast<int32_t *>(smem + OFF_ENT);
    int32_t *Q = reinterpret_cast<int32_t *>(smem + OFF_Q);
    uint64_t *mbar = reinterpret_cast<uint64_t *>(smem + OFF_MISC);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_MISC + 8);
    int *flag = reinterpret_cast<int *>(smem + OFF_MISC + 12);
    PfItem *itp = reinterpret_cast<PfItem *>(smem + OFF_MISC + 16);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int MT = job.rows / PF_M;
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // ---- item: (expert e, pass of <= 256 tokens, M tile) ----------------
    if (tid == 0) {
        PfItem it = {0, 0, 0, 0, 0, 0, 0};
        int acc = 0;
        bool ok = job.offsets[0] == 0 && job.offsets[job.E] == job.n_pairs;
        for (int e = 0; e < job.E && ok; ++e) {
            const int ne = job.offsets[e + 1] - job.offsets[e];
            if (ne < 0) ok = false;
            Q[e] = acc;
            acc += job.min_tokens <= ne ? (ne + PF_NMAX - 1) / PF_NMAX : 0;
        }
        Q[job.E] = acc;
        const int pi = blockIdx.x / MT;
        if (!ok) {
            set_dev_error(job.status, RVQ_DEV_ERR_INDEX);
        } else if (pi < acc) {
            int lo = 0, hi = job.E;  // largest e with Q[e] <= pi (and a pass there)
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (Q[mid] <= pi) lo = mid; else hi = mid;
            }
            const int e = lo;
            const int ne = job.offsets[e + 1] - job.offsets[e];
            const int np = pi - Q[e];
            it.e = e;
            it.o = job.offsets[e];
            it.j0 = np * PF_NMAX;
            it.n = min(PF_NMAX, ne - it.j0);
            it.npad = (it.n + 15) & ~15;
            it.mt = blockIdx.x % MT;
            it.valid = it.n > 0;
            const rvq_expert_header *h =
                reinterpret_cast<const rvq_expert_header *>(job.base + (uint64_t)e * job.record_bytes);
            if (h->magic != RVQ_BANK_MAGIC || h->expert != e || h->layer != job.layer ||
                h->d != job.d || h->f != job.f || h->record_bytes != job.record_bytes) {
                set_dev_error(job.status, RVQ_DEV_ERR_CORRUPT);
                it.valid = 0;
            }
        }
        *itp = it;
        *flag = 0;
    }
    __syncthreads();
    const PfItem it = *itp;
    if (!it.valid) return;
    asm volatile("griddepcontrol.launch_dependents;");

    const uint8_t *rec = job.base + (uint64_t)it.e * job.record_bytes;
    // pair entries of this pass; codebooks -> fp32 [s][k][8] (each weight is
    // rounded to bf16 once, after the three codewords are summed)
    for (int j = tid; j < it.n; j += PF_NT) {
        const int p = job.pairs[it.o + it.j0 + j];
        ent[j] = (p >= 0 && p < job.n_pairs) ? p : -1;
        if (p < 0 || p >= job.n_pairs) set_dev_error(job.status, RVQ_DEV_ERR_INDEX);
    }
    for (int m = 0; m < job.n_mat; ++m) {
        const float *cbp = reinterpret_cast<const float *>(rec + job.cb_off[m]);
        float *cbs = reinterpret_cast<float *>(smem + OFF_CB + m * kCbF32);
        for (int x = tid; x < 3 * 256 * 8; x += PF_NT) {
            const int s = x / 2048, k = (x / 8) % 256, i = x % 8;
            cbs[x] = cbp[((s * 128 + k / 2) * 8 + i) * 2 + (k & 1)];
        }
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(job.n_mat == 2 ? 512 : 256));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(mbar)), "r"(1));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tmem_slot;

    const int RB = job.rows / 32;
    const int row = tid;                           // this thread's row within the tile
    const int R = it.mt * PF_M + row;              // row of W
    const uint32_t idesc = idesc_bf16(PF_M, it.npad);
    const int ksteps = job.cols / PF_KC;
    const int esz = job.x_dtype == RVQ_BF16 ? 2 : 4;
    bool ok = true;

    for (int ks = 0; ks < ksteps && ok; ++ks) {
        // (a) decode this thread's row: 8 chunks per matrix, one 16-byte
        //     swizzle unit each
        for (int m = 0; m < job.n_mat; ++m) {
            const uint8_t *codes = rec + job.codes_off[m];
            const float4 *cbs = reinterpret_cast<const float4 *>(smem + OFF_CB + m * kCbF32);
            uint8_t *tile = smem + OFF_A + m * kTileA;
#pragma unroll 2
            for (int cc = 0; cc < 8; ++cc) {
                const int j = ks * 8 + cc;
                const int k0 = code_at(codes, RB, R, j, 0);
                const int k1 = code_at(codes, RB, R, j, 1);
                const int k2 = code_at(codes, RB, R, j, 2);
                const float4 a0 = cbs[(0 * 256 + k0) * 2], b0 = cbs[(0 * 256 + k0) * 2 + 1];
                const float4 a1 = cbs[(1 * 256 + k1) * 2], b1 = cbs[(1 * 256 + k1) * 2 + 1];
                const float4 a2 = cbs[(2 * 256 + k2) * 2], b2 = cbs[(2 * 256 + k2) * 2 + 1];
                uint32_t o[4];
                o[0] = bf16_bits(a0.x + a1.x + a2.x) | (bf16_bits(a0.y + a1.y + a2.y) << 16);
                o[1] = bf16_bits(a0.z + a1.z + a2.z) | (bf16_bits(a0.w + a1.w + a2.w) << 16);
                o[2] = bf16_bits(b0.x + b1.x + b2.x) | (bf16_bits(b0.y + b1.y + b2.y) << 16);
                o[3] = bf16_bits(b0.z + b1.z + b2.z) | (bf16_bits(b0.w + b1.w + b2.w) << 16);
                *reinterpret_cast<uint4 *>(tile + row * 128 + ((cc ^ (row & 7)) * 16)) =
                    make_uint4(o[0], o[1], o[2], o[3]);
            }
        }
        // (b) B tile: the pass's tokens (rows beyond n are zero)
        for (int x = tid; x < it.npad * 8; x += PF_NT) {
            const int j = x >> 3, cc = x & 7;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (j < it.n && ent[j] >= 0) {
                const int64_t rowi = (int64_t)(ent[j] / job.x_div) * job.x_stride + ks * PF_KC + cc * 8;
                if (esz == 2) {
                    v = *reinterpret_cast<const uint4 *>(reinterpret_cast<const uint8_t *>(job.x) +
                                                         rowi * 2);
                } else {
                    const float4 *f = reinterpret_cast<const float4 *>(
                        reinterpret_cast<const float *>(job.x) + rowi);
                    const float4 f0 = f[0], f1 = f[1];
                    v.x = bf16_bits(f0.x) | (bf16_bits(f0.y) << 16);
                    v.y = bf16_bits(f0.z) | (bf16_bits(f0.w) << 16);
                    v.z = bf16_bits(f1.x) | (bf16_bits(f1.y) << 16);
                    v.w = bf16_bits(f1.z) | (bf16_bits(f1.w) << 16);
                }
            }
            *reinterpret_cast<uint4 *>(smem + OFF_B + j * 128 + ((cc ^ (j & 7)) * 16)) = v;
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();
        // (c) one thread issues the MMAs: 4 x K=16 per matrix
        if (tid == 0) {
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            for (int m = 0; m < job.n_mat; ++m) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t ad = smem_desc(smem_u32(smem + OFF_A + m * kTileA) + kk * 32);
                    const uint64_t bd = smem_desc(smem_u32(smem + OFF_B) + kk * 32);
                    mma_bf16(tmem + m * 256, ad, bd, idesc, (ks > 0 || kk > 0) ? 1u : 0u);
                }
            }
            mma_commit(smem_u32(mbar));
        }
        // (d) the tiles may be overwritten once the MMAs have read them
        if (!mbar_wait(smem_u32(mbar), (uint32_t)(ks & 1))) *flag = 1;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        __syncthreads();
        ok = *flag == 0;
    }

    if (ok) {
        // epilogue: lane <-> row; 32 token columns per TMEM load
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        for (int c0 = 0; c0 < it.npad; c0 += 32) {
            float g[32], u[32];
            tmem_ld32(tmem + lane_base + c0, g);
            if (job.n_mat == 2) tmem_ld32(tmem + lane_base + 256 + c0, u);
#pragma unroll
            for (int q = 0; q < 32; ++q) {
                const int j = c0 + q;
                if (j < it.n && ent[j] >= 0) {
                    if (job.n_mat == 2) {
                        const float hv = g[q] / (1.0f + expf(-g[q])) * u[q];
                        reinterpret_cast<uint16_t *>(job.out)[(size_t)ent[j] * job.rows + R] =
                            (uint16_t)bf16_bits(hv);
                    } else {
                        reinterpret_cast<float *>(job.out)[(size_t)ent[j] * job.rows + R] = g[q];
                    }
                }
            }
        }
    } else if (tid == 0) {
        set_dev_error(job.status, RVQ_DEV_ERR_TIMEOUT);
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(job.n_mat == 2 ? 512 : 256));
}

}  // namespace

int prefill_max_items(const PfJob &job) {
    // sum over experts of ceil(n_e / 256) <= E + n_pairs / 256, times the M tiles
    return (job.E + job.n_pairs / PF_NMAX + 1) * (job.rows / PF_M);
}

rvq_status launch_prefill_gemm(const PfJob &job, cudaStream_t stream, bool pdl) {
    static int attr_done[64] = {0};
    int dev = 0;
    RVQ_CUDA(cudaGetDevice(&dev));
    if (dev < 64 && !attr_done[dev]) {
        RVQ_CUDA(cudaFuncSetAttribute(prefill_gemm_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, kPfSmem));
        attr_done[dev] = 1;
    }
    if (job.rows % PF_M || job.cols % PF_KC || job.n_mat < 1 || job.n_mat > 2) {
        set_error("prefill: rows %d / cols %d not tileable", job.rows, job.cols);
        return RVQ_EINVAL;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)prefill_max_items(job));
    cfg.blockDim = dim3(PF_NT);
    cfg.dynamicSmemBytes = kPfSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    RVQ_CUDA(cudaLaunchKernelEx(&cfg, prefill_gemm_kernel, job));
    return RVQ_OK;
}

}  // namespace rvq
