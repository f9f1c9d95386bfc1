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
// up to 256 tokens of one expert's group x 64 K-columns (K-major), D = W x^T
// (128 rows x N tokens, fp32, in TMEM).  One RVQ chunk (8 weights) is exactly
// one 16-byte unit of the 128-byte swizzle row, so a decoded chunk is stored
// with one 128-bit shared-memory store at its swizzled position.
//
// A work item is (expert, pass of <= 256 tokens, M tile) and carries two A
// tiles that share the B tile:
//  * gate/up launch: tile 0 = 128 rows of gate, tile 1 = the same rows of up;
//    the epilogue computes h = silu(g) * u and writes bf16 h [pair][f].
//  * down launch: tiles 0 and 1 = rows [256 m, 256 m + 128) and the next 128
//    rows of down; the epilogue writes fp32 y [pair][d].
// Items are split into contiguous ranges over a persistent grid (one CTA per
// SM), so consecutive items of a CTA mostly share the expert and its codebooks.
//
// Warp roles (512 threads):
//  warp 0      TMEM owner; lane 0 issues the MMAs (8 per K step) and commits
//  warps 1-3   B producers: cp.async gathers of token rows into the B stage
//  warps 4-7   epilogue: TMEM -> registers -> global (lane quarter = warp % 4)
//  warps 8-15  A producers: decode code bytes into the two bf16 A tiles
// The stages (A0, A1, B) form a two-deep ring guarded by full/empty mbarriers;
// the accumulators (512 TMEM columns: tile 0 at 0, tile 1 at 256) by acc_full
// and acc_empty.
//
// Decoding is bound by shared-memory gathers of codewords, so the codebooks
// sit in shared memory as fp16 (summed in fp16, then rounded once to bf16) in
// a bank-private layout: line (stage s, codeword k) is 128 bytes, and 16-byte
// group q of every line serves lane q of each quarter-warp.  Groups 0-3 hold
// tile 0's codebook, groups 4-7 tile 1's.  A quarter-warp thus reads eight
// codewords from eight distinct bank groups whatever the codes are, and the
// eight rows it decodes have distinct (row mod 8), so its swizzled stores are
// conflict-free as well.
//
// Every wait is bounded (1 s); on expiry the CTA records RVQ_DEV_ERR_TIMEOUT,
// every role leaves its loop, the MMAs in flight are drained and TMEM is freed.
#include "internal.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace rvq {
namespace {

constexpr int PF_THREADS = 512;
constexpr int PF_NMAX = 256;                     // tokens per pass (MMA N)
constexpr int PF_KC = 64;                        // K columns per stage (one 128-byte swizzle row)
constexpr int PF_NST = 2;                        // ring depth
constexpr int kTileA = 128 * PF_KC * 2;          // 16 KiB
constexpr int kTileB = PF_NMAX * PF_KC * 2;      // 32 KiB
constexpr int kStage = 2 * kTileA + kTileB;      // 64 KiB
constexpr int kCbLine = 128;                     // one (stage, codeword) line
constexpr int kCbBytes = 3 * 256 * kCbLine;      // 96 KiB
constexpr int OFF_CB = 0;
constexpr int OFF_ST = kCbBytes;
constexpr int OFF_BAR = OFF_ST + PF_NST * kStage;
// mbarriers, 8 bytes each from OFF_BAR
constexpr int BAR_FULL = 0;                      // [PF_NST]
constexpr int BAR_EMPTY = PF_NST;                // [PF_NST]
constexpr int BAR_ACC_FULL = 2 * PF_NST;
constexpr int BAR_ACC_EMPTY = 2 * PF_NST + 1;
constexpr int BAR_DONE = 2 * PF_NST + 2;
constexpr int BAR_CB = 2 * PF_NST + 3;           // A producers: codebook swap rendezvous
constexpr int BAR_NEVER = 2 * PF_NST + 4;        // self-test: a phase nothing completes
constexpr int kNumBars = 2 * PF_NST + 5;
constexpr int OFF_TMEM = OFF_BAR + 8 * kNumBars;
constexpr int OFF_FLAG = OFF_TMEM + 4;
constexpr int OFF_Q = OFF_BAR + 128;             // pass prefix [E + 1]
constexpr int kMaxE = 256;
constexpr int kPfSmem = OFF_Q + 4 * (kMaxE + 1) + 1024;  // + slack to align the base to 1 KiB
static_assert(OFF_FLAG + 4 <= OFF_Q, "control block overlaps the pass prefix");
static_assert(kPfSmem <= 232448, "shared memory per CTA");

constexpr int kLoaders = 96;                     // B producer threads (warps 1-3)
constexpr int kDecoders = 256;                   // A producer threads (warps 8-15)
constexpr uint32_t kFullCount = kLoaders + kDecoders / 32;
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s: a bounded wait, never a hang

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

__device__ __forceinline__ void mbar_init(uint32_t mbar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(mbar), "r"(count));
}

__device__ __forceinline__ void mbar_arrive(uint32_t mbar) {
    asm volatile("{\n.reg .b64 st;\nmbarrier.arrive.shared::cta.b64 st, [%0];\n}\n" ::"r"(mbar)
                 : "memory");
}

// try_wait with a suspend hint: a waiting warp sleeps (up to 20 us) instead
// of spinning, leaving issue slots to the decoding warps; it wakes when the
// phase completes.
__device__ __forceinline__ bool mbar_try(uint32_t mbar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        "selp.b32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(mbar), "r"(parity), "r"(20000u)
        : "memory");
    return done != 0;
}

// Bounded wait on an mbarrier phase.  Returns false once another role has
// aborted, or after kWaitLimitNs (then this thread raises the abort flag and
// records the timeout).
__device__ __forceinline__ bool mbar_wait(uint32_t mbar, uint32_t parity, volatile int *abort_flag,
                                          uint32_t *status) {
    if (mbar_try(mbar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (;;) {
        if (mbar_try(mbar, parity)) return true;
        if (*abort_flag) return false;
        if (global_ns() - t0 > kWaitLimitNs) {
            *abort_flag = 1;
            set_dev_error(status, RVQ_DEV_ERR_TIMEOUT);
            return false;
        }
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

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&b);
}

// Three fp16x2 codeword words summed in fp16, rounded once to bf16x2.
__device__ __forceinline__ uint32_t sum3_bf16x2(uint32_t a, uint32_t b, uint32_t c) {
    const __half2 s = __hadd2(__hadd2(*reinterpret_cast<const __half2 *>(&a),
                                      *reinterpret_cast<const __half2 *>(&b)),
                              *reinterpret_cast<const __half2 *>(&c));
    const float2 f = __half22float2(s);
    return pack_bf16x2(f.x, f.y);
}

// Rotate a 32-byte vector left by l bytes (l in 0..31).  The packed code
// layout stores chunk j of a row with lane l = row mod 32 at byte
// (j - l) mod 32 of its stage plane; the rotation puts chunk j at byte j.
__device__ __forceinline__ void derotate(uint32_t (&w)[8], int l) {
    const int wl = l >> 2;
    const uint32_t bl = (uint32_t)(l & 3) * 8u;
    uint32_t a[8], b[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = (wl & 1) ? w[(i + 7) & 7] : w[i];
#pragma unroll
    for (int i = 0; i < 8; ++i) b[i] = (wl & 2) ? a[(i + 6) & 7] : a[i];
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = (wl & 4) ? b[(i + 4) & 7] : b[i];
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = __funnelshift_l(a[(i + 7) & 7], a[i], bl);
}

// 128-bit shared store issued as volatile asm without a memory clobber: the
// compiler keeps it in order with the fences and barrier arrivals (also
// volatile asm) but may schedule the codebook loads of later chunks ahead of
// it -- the A tiles and the codebooks never overlap.
__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w));
}

// 128-bit shared load through a 32-bit shared address (no generic address
// arithmetic).  Not volatile: its address depends on code bytes loaded after
// every codebook swap, which keeps it behind the swap's barrier.
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "r"(addr));
    return v;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

struct PfItem {
    int e, o, j0, n, npad, mt;
    bool valid;
};

// Work item `it` -> (expert, pass, M tile).  Q[e] = passes before expert e.
__device__ __forceinline__ PfItem pf_item(const PfJob &job, const int32_t *Q, int MT, int it) {
    PfItem I;
    const int pi = it / MT;
    I.mt = it - pi * MT;
    int lo = 0, hi = job.E;  // largest e < E with Q[e] <= pi (it has a pass there)
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (Q[mid] <= pi) lo = mid; else hi = mid;
    }
    I.e = lo;
    I.o = job.offsets[lo];
    const int ne = job.offsets[lo + 1] - I.o;
    I.j0 = (pi - Q[lo]) * PF_NMAX;
    I.n = min(PF_NMAX, ne - I.j0);
    I.npad = (I.n + 15) & ~15;
    const rvq_expert_header *h =
        reinterpret_cast<const rvq_expert_header *>(job.base + (uint64_t)lo * job.record_bytes);
    I.valid = I.n > 0 && h->magic == RVQ_BANK_MAGIC && h->expert == lo && h->layer == job.layer &&
              h->d == job.d && h->f == job.f && h->record_bytes == job.record_bytes;
    return I;
}

__global__ void __launch_bounds__(PF_THREADS, 1) prefill_gemm_kernel(const PfJob job) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // the 128-byte swizzle is a function of shared-address bits 4..9: tiles
    // must start on 1024-byte boundaries of the shared window
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + OFF_BAR;
    auto bar = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + OFF_FLAG);
    int32_t *Q = reinterpret_cast<int32_t *>(smem + OFF_Q);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int MT = job.rows / job.tile_rows;
    const int KS = job.cols / PF_KC;

    asm volatile("griddepcontrol.wait;" ::: "memory");

    // ---- setup: pass prefix (warp 1), barriers + TMEM (warp 0) ----------
    if (warp == 1) {
        const int E = job.E;
        const int per = (E + 31) / 32;
        const int e0 = min(E, lane * per), e1 = min(E, e0 + per);
        int cnt = 0;
        bool ok = true;
        for (int e = e0; e < e1; ++e) {
            const int ne = job.offsets[e + 1] - job.offsets[e];
            ok = ok && ne >= 0;
            cnt += (ne >= job.min_tokens) ? (ne + PF_NMAX - 1) / PF_NMAX : 0;
        }
        int incl = cnt;
#pragma unroll
        for (int s = 1; s < 32; s <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, s);
            if (lane >= s) incl += v;
        }
        int pre = incl - cnt;
        for (int e = e0; e < e1; ++e) {
            Q[e] = pre;
            const int ne = job.offsets[e + 1] - job.offsets[e];
            pre += (ne >= job.min_tokens) ? (ne + PF_NMAX - 1) / PF_NMAX : 0;
        }
        ok = __all_sync(0xffffffffu, ok) && job.offsets[0] == 0 && job.offsets[E] == job.n_pairs;
        if (lane == 31) Q[E] = ok ? incl : 0;
        if (!ok && lane == 0) set_dev_error(job.status, RVQ_DEV_ERR_INDEX);
    } else if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         sbase + OFF_TMEM),
                     "r"(512));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
        if (lane == 0) {
            for (int s = 0; s < PF_NST; ++s) {
                mbar_init(bar(BAR_FULL + s), kFullCount);
                mbar_init(bar(BAR_EMPTY + s), 1);
            }
            mbar_init(bar(BAR_ACC_FULL), 1);
            mbar_init(bar(BAR_ACC_EMPTY), 4);
            mbar_init(bar(BAR_DONE), 1);
            mbar_init(bar(BAR_CB), kDecoders / 32);
            mbar_init(bar(BAR_NEVER), 1);
            *abort_flag = 0;
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + OFF_TMEM);

    const int total = Q[job.E] * MT;
    const int it0 = (int)((int64_t)blockIdx.x * total / gridDim.x);
    const int it1 = (int)((int64_t)(blockIdx.x + 1) * total / gridDim.x);

    if (warp == 0) {
        // ================= MMA issuer =================
        if (lane == 0) {
            uint32_t st = 0, ph = 0, nacc = 0;
            // self-test of the failure path: wait for an arrival nothing makes,
            // so the bounded wait expires and every role gives up
            if (job.selftest_stall) mbar_wait(bar(BAR_NEVER), 0, abort_flag, job.status);
            for (int it = it0; it < it1 && !*abort_flag; ++it) {
                const PfItem I = pf_item(job, Q, MT, it);
                if (!I.valid) continue;
                if (!mbar_wait(bar(BAR_ACC_EMPTY), (nacc & 1u) ^ 1u, abort_flag, job.status)) break;
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t idesc = idesc_bf16(128, I.npad);
                bool ok = true;
                for (int ks = 0; ks < KS; ++ks) {
                    if (!mbar_wait(bar(BAR_FULL + st), ph, abort_flag, job.status)) {
                        ok = false;
                        break;
                    }
                    // the B stage was written through the generic proxy (cp.async)
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    const uint32_t sa = sbase + OFF_ST + st * kStage;
#pragma unroll
                    for (int t = 0; t < 2; ++t) {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            mma_bf16(tmem + t * 256, smem_desc(sa + t * kTileA + kk * 32),
                                     smem_desc(sa + 2 * kTileA + kk * 32), idesc,
                                     (ks > 0 || kk > 0) ? 1u : 0u);
                        }
                    }
                    mma_commit(bar(BAR_EMPTY + st));
                    if (++st == PF_NST) {
                        st = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit(bar(BAR_ACC_FULL));
                ++nacc;
            }
            // drain: every MMA issued has completed before TMEM is released
            mma_commit(bar(BAR_DONE));
            int no_abort = 0;
            mbar_wait(bar(BAR_DONE), 0, &no_abort, job.status);
        }
        __syncwarp();
    } else if (warp < 4) {
        // ================= B producers =================
        const int lt = tid - 32;
        const int esz = job.x_dtype == RVQ_BF16 ? 2 : 4;
        uint32_t st = 0, ph = 0;
        for (int it = it0; it < it1 && !*abort_flag; ++it) {
            const PfItem I = pf_item(job, Q, MT, it);
            if (!I.valid) continue;
            const uint8_t *src[3];
#pragma unroll
            for (int r = 0; r < 3; ++r) {
                const int j = lt + kLoaders * r;
                src[r] = nullptr;
                if (j < I.n) {
                    const int p = job.pairs[I.o + I.j0 + j];
                    if (p >= 0 && p < job.n_pairs)
                        src[r] = reinterpret_cast<const uint8_t *>(job.x) +
                                 ((int64_t)(p / job.x_div) * job.x_stride) * esz;
                    else
                        set_dev_error(job.status, RVQ_DEV_ERR_INDEX);
                }
            }
            bool ok = true;
            for (int ks = 0; ks < KS; ++ks) {
                if (!mbar_wait(bar(BAR_EMPTY + st), ph ^ 1u, abort_flag, job.status)) {
                    ok = false;
                    break;
                }
                const uint32_t sb = sbase + OFF_ST + st * kStage + 2 * kTileA;
                const uint32_t full = bar(BAR_FULL + st);
                if (esz == 2) {
#pragma unroll
                    for (int r = 0; r < 3; ++r) {
                        const int j = lt + kLoaders * r;
                        if (src[r] != nullptr) {
                            const uint8_t *s = src[r] + ks * PF_KC * 2;
#pragma unroll
                            for (int c = 0; c < 8; ++c)
                                cp_async16(sb + j * 128 + ((c ^ (j & 7)) << 4), s + c * 16);
                        }
                    }
                    // arrives once this thread's copies have landed
                    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(full)
                                 : "memory");
                } else {
                    uint8_t *bt = smem + OFF_ST + st * kStage + 2 * kTileA;
#pragma unroll
                    for (int r = 0; r < 3; ++r) {
                        const int j = lt + kLoaders * r;
                        if (src[r] != nullptr) {
                            const float4 *s =
                                reinterpret_cast<const float4 *>(src[r] + ks * PF_KC * 4);
                            for (int c = 0; c < 8; ++c) {
                                const float4 f0 = s[2 * c], f1 = s[2 * c + 1];
                                *reinterpret_cast<uint4 *>(bt + j * 128 + ((c ^ (j & 7)) << 4)) =
                                    make_uint4(pack_bf16x2(f0.x, f0.y), pack_bf16x2(f0.z, f0.w),
                                               pack_bf16x2(f1.x, f1.y), pack_bf16x2(f1.z, f1.w));
                            }
                        }
                    }
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    mbar_arrive(full);
                }
                if (++st == PF_NST) {
                    st = 0;
                    ph ^= 1u;
                }
            }
            if (!ok) break;
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
    } else if (warp < 8) {
        // ================= epilogue =================
        const int ew = warp - 4;                 // TMEM lanes 32 ew .. 32 ew + 31
        const int rit = ew * 32 + lane;          // row within the tile
        const uint32_t tl = tmem + ((uint32_t)(ew * 32) << 16);
        uint32_t nacc = 0;
        for (int it = it0; it < it1; ++it) {
            const PfItem I = pf_item(job, Q, MT, it);
            if (!I.valid) continue;
            if (!mbar_wait(bar(BAR_ACC_FULL), nacc & 1u, abort_flag, job.status)) break;
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const int R0 = I.mt * job.tile_rows;
            for (int c0 = 0; c0 < I.n; c0 += 32) {
                const int jl = c0 + lane;
                const int pl = jl < I.n ? job.pairs[I.o + I.j0 + jl] : -1;
                float a0[32], a1[32];
                tmem_ld32(tl + c0, a0);
                tmem_ld32(tl + 256 + c0, a1);
#pragma unroll
                for (int q = 0; q < 32; ++q) {
                    const int p = __shfl_sync(0xffffffffu, pl, q);
                    if (c0 + q < I.n && p >= 0 && p < job.n_pairs) {
                        if (job.mode == PF_MODE_SWIGLU) {
                            const float g = a0[q];
                            const float hv = g / (1.0f + expf(-g)) * a1[q];
                            reinterpret_cast<uint16_t *>(job.out)[(size_t)p * job.rows + R0 + rit] =
                                (uint16_t)bf16_bits(hv);
                        } else {
                            float *y = reinterpret_cast<float *>(job.out) + (size_t)p * job.rows + R0;
                            y[job.row_off[0] + rit] = a0[q];
                            y[job.row_off[1] + rit] = a1[q];
                        }
                    }
                }
            }
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(BAR_ACC_EMPTY));
            ++nacc;
        }
    } else {
        // ================= A producers (decode) =================
        const int dt = tid - 256;
        const int dw = dt >> 5, qw = lane >> 3, q = lane & 7;
        const int b8 = dw * 4 + qw;              // quarter-warp 0..31
        const int r0 = (b8 >> 1) * 8;
        const int tile = q >> 2;
        // quarter-warps of type 0 decode tile-0 rows r0..r0+3 and tile-1 rows
        // r0+4..r0+7, type 1 the other halves: (row mod 8) differs per lane
        const int rit = (b8 & 1) == 0 ? r0 + q : (tile == 0 ? r0 + 4 + q : r0 + q - 4);
        const int sw = rit & 7;
        const uint32_t cbl = sbase + OFF_CB + q * 16;  // this lane's bank group
        const int RB = job.rows / 32;
        const int G = KS / 4;                    // 32-chunk groups along K
        int cur_e = -1;
        uint32_t st = 0, ph = 0, ncb = 0;
        for (int it = it0; it < it1 && !*abort_flag; ++it) {
            const PfItem I = pf_item(job, Q, MT, it);
            if (!I.valid) continue;
            const uint8_t *rec = job.base + (uint64_t)I.e * job.record_bytes;
            if (I.e != cur_e) {
                // every A producer is done with the previous codebooks
                if (cur_e >= 0) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(BAR_CB));
                    if (!mbar_wait(bar(BAR_CB), ncb & 1u, abort_flag, job.status)) break;
                    ++ncb;
                }
                // record fp32 [s][k/2][i][k&1] -> fp16 lines, one 16-byte group per unit
                for (int u = dt; u < 3 * 256 * 8; u += kDecoders) {
                    const int L = u >> 3, g = u & 7;
                    const int s = L >> 8, k = L & 255;
                    const float *cb = reinterpret_cast<const float *>(rec + job.cb_off[g >> 2]) +
                                      ((s * 128 + (k >> 1)) * 8) * 2 + (k & 1);
                    uint32_t w[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const __half2 h2 = __floats2half2_rn(cb[(2 * i) * 2], cb[(2 * i + 1) * 2]);
                        w[i] = *reinterpret_cast<const uint32_t *>(&h2);
                    }
                    *reinterpret_cast<uint4 *>(smem + OFF_CB + L * kCbLine + g * 16) =
                        make_uint4(w[0], w[1], w[2], w[3]);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(BAR_CB));
                if (!mbar_wait(bar(BAR_CB), ncb & 1u, abort_flag, job.status)) break;
                ++ncb;
                cur_e = I.e;
            }
            const int R = I.mt * job.tile_rows + job.row_off[tile] + rit;
            const int l = R & 31;
            // this row's code planes of 32-chunk group g: 6 x 16 bytes (stage s, half h)
            const uint8_t *cp = rec + job.codes_off[tile] + (size_t)(R >> 5) * kTileBytes + l * 16;
            uint4 nxt[6];
#pragma unroll
            for (int v = 0; v < 6; ++v) nxt[v] = *reinterpret_cast<const uint4 *>(cp + v * 512);
            bool ok = true;
            for (int g = 0; g < G && ok; ++g) {
                uint32_t U[3][8];
#pragma unroll
                for (int s = 0; s < 3; ++s) {
                    U[s][0] = nxt[2 * s].x;
                    U[s][1] = nxt[2 * s].y;
                    U[s][2] = nxt[2 * s].z;
                    U[s][3] = nxt[2 * s].w;
                    U[s][4] = nxt[2 * s + 1].x;
                    U[s][5] = nxt[2 * s + 1].y;
                    U[s][6] = nxt[2 * s + 1].z;
                    U[s][7] = nxt[2 * s + 1].w;
                }
                if (g + 1 < G) {
                    const uint8_t *cpn = cp + (size_t)(g + 1) * RB * kTileBytes;
#pragma unroll
                    for (int v = 0; v < 6; ++v)
                        nxt[v] = *reinterpret_cast<const uint4 *>(cpn + v * 512);
                }
#pragma unroll
                for (int s = 0; s < 3; ++s) derotate(U[s], l);
#pragma unroll
                for (int k4 = 0; k4 < 4; ++k4) {
                    if (!mbar_wait(bar(BAR_EMPTY + st), ph ^ 1u, abort_flag, job.status)) {
                        ok = false;
                        break;
                    }
                    const uint32_t A = sbase + OFF_ST + st * kStage + tile * kTileA + rit * 128;
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const int cg = k4 * 8 + c;
                        const uint32_t k0 = (U[0][cg >> 2] >> (8 * (cg & 3))) & 0xFFu;
                        const uint32_t k1 = (U[1][cg >> 2] >> (8 * (cg & 3))) & 0xFFu;
                        const uint32_t k2 = (U[2][cg >> 2] >> (8 * (cg & 3))) & 0xFFu;
                        const uint4 w0 = lds128(cbl + k0 * kCbLine);
                        const uint4 w1 = lds128(cbl + (256 + k1) * kCbLine);
                        const uint4 w2 = lds128(cbl + (512 + k2) * kCbLine);
                        uint4 o;
                        o.x = sum3_bf16x2(w0.x, w1.x, w2.x);
                        o.y = sum3_bf16x2(w0.y, w1.y, w2.y);
                        o.z = sum3_bf16x2(w0.z, w1.z, w2.z);
                        o.w = sum3_bf16x2(w0.w, w1.w, w2.w);
                        sts128(A + ((c ^ sw) << 4), o);
                    }
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(BAR_FULL + st));
                    if (++st == PF_NST) {
                        st = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok) break;
        }
    }

    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512));
    }
}

}  // namespace

rvq_status launch_prefill_gemm(const PfJob &job, cudaStream_t stream, bool pdl) {
    static int attr_done[64] = {0};
    int dev = 0;
    RVQ_CUDA(cudaGetDevice(&dev));
    if (dev < 64 && !attr_done[dev]) {
        RVQ_CUDA(cudaFuncSetAttribute(prefill_gemm_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, kPfSmem));
        attr_done[dev] = 1;
    }
    if ((job.tile_rows != 128 && job.tile_rows != 256) || job.rows % job.tile_rows ||
        job.cols % (4 * PF_KC) || job.E < 1 || job.E > kMaxE || job.min_tokens < 1 ||
        (job.mode != PF_MODE_SWIGLU && job.mode != PF_MODE_PLAIN)) {
        set_error("prefill: rows %d / cols %d / tile %d / E %d not supported", job.rows, job.cols,
                  job.tile_rows, job.E);
        return RVQ_EINVAL;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)num_sms());
    cfg.blockDim = dim3(PF_THREADS);
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
