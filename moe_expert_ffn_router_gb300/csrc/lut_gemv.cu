// Lookup-table GEMV on RVQ codes (decode path of the expert FFN).
//
// Method: for each input vector x and chunk j (8 input columns) a table
// T_s[j][k] = <x[8j..8j+7], C_s[k]> is built for the three stages s and 256
// entries k; an output row is then sum_j sum_s T_s[j][code(r,j,s)], i.e. three
// table reads per chunk and row, and the weight matrix is never formed
// ["Running a 2.78-Trillion-Parameter Model on a Laptop: Inside WASTE's
// NVMe-Streaming Engine", section "Technical Insight"; "WASTE Inference
// Engine: Running Kimi K3 2.78T on Consumer Hardware", section "Residual
// Vector Quantization (RVQ)"].
//
// GB300 design (not the pages' CPU loop):
//  * A block owns one "item": one expert matrix, up to two (token, 32-chunk
//    group) units, a range of C steps over chunk groups and a range of rows.
//    Its table for one step (2 units x 3 stages x 256 entries x 32 chunks,
//    192 KiB) lives in shared memory and is built exactly once per (token,
//    chunk group, row range); it is never written to HBM.
//  * Lane l of a warp owns row 32b + l.  The packed code layout rotates each
//    row's chunk order by l, so at every unrolled step t the 32 lanes read 32
//    different table columns (bank = column): the lookups are conflict-free
//    for any code values, and each lane accumulates its own row with no
//    cross-lane reduction.
//  * A code byte becomes a shared-memory address with one byte permute
//    (code -> bits 8..15, column offset -> bits 0..7), one LDS and half of a
//    packed fp32x2 add.  Code tiles (3 KiB per 32 rows x 32 chunks) are
//    streamed with 128-bit non-allocating loads, one row block ahead.
//  * Items of the same (expert, chunk group) for different token pairs are
//    adjacent in launch order, so a second token pair re-reads codes from L2.
//  * Split-K partials (one slot per item column range) are reduced by the
//    next kernel (SwiGLU for gate/up, the combine for down).
#include "internal.cuh"

namespace rvq {
namespace {

constexpr int NT = 256;
constexpr int NW = NT / 32;
constexpr int kMaxSplitRows = 2048;  // shared accumulator: 2048 x float2 = 16 KiB

struct Item {
    int valid;
    int type;  // 0: two tokens, one chunk group per step; 1: one token, two groups per step
    int entryA, entryB;
    int g0;
    int slotA, slotB;
    int rb0, nrb;
    const uint8_t *codes;
    const float *cb;
    const void *xA, *xB;
};

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

__device__ __forceinline__ uint64_t pk2(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1,%2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ float2 upk2(uint64_t v) {
    float2 r;
    asm("mov.b64 {%0,%1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t ffma2(uint64_t x, uint64_t y, uint64_t acc) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(x), "l"(y), "l"(acc));
    return r;
}

__device__ int segment_of(const int32_t *offsets, int E, int p) {
    int lo = 0, hi = E;
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (offsets[mid] <= p) lo = mid; else hi = mid;
    }
    return lo;
}

// Decode blockIdx into an item (thread 0 only).
__device__ void decode_item(const LutJob &job, int m, Item &it) {
    it.valid = 0;
    const int per_pair = job.G / (2 * job.C);
    const int i = blockIdx.x / job.S;
    const int split = blockIdx.x % job.S;
    const int p = i / per_pair;
    if (p >= job.n_pairs) return;
    int e = 0, o = 0, ne = job.n_pairs;
    if (job.offsets) {
        if (job.offsets[0] != 0 || job.offsets[job.E] != job.n_pairs) {
            set_dev_error(job.status, RVQ_DEV_ERR_INDEX);
            return;
        }
        e = segment_of(job.offsets, job.E, p);
        o = job.offsets[e];
        ne = job.offsets[e + 1] - o;
        if (!(0 <= o && o <= p && p < o + ne && o + ne <= job.n_pairs)) {
            set_dev_error(job.status, RVQ_DEV_ERR_INDEX);
            return;
        }
    }
    const uint8_t *rec = job.base ? job.base + (uint64_t)e * job.record_bytes : nullptr;
    if (job.check_header && rec) {
        const rvq_expert_header *h = reinterpret_cast<const rvq_expert_header *>(rec);
        if (h->magic != RVQ_BANK_MAGIC || h->expert != e || h->layer != job.layer ||
            h->d != job.d || h->f != job.f || h->record_bytes != job.record_bytes) {
            set_dev_error(job.status, RVQ_DEV_ERR_CORRUPT);
            return;
        }
    }
    const int li = i - per_pair * o;
    const int Q = ne >> 1;
    const int runs = job.G / job.C;  // chunk-group runs of the two-token items
    int tauA, tauB;
    if (li < Q * runs) {
        const int gr = li / Q, q = li % Q;
        it.type = 0;
        tauA = 2 * q;
        tauB = 2 * q + 1;
        it.g0 = gr * job.C;
        it.slotA = it.slotB = gr;
    } else {
        const int l2 = li - Q * runs;
        it.type = 1;
        tauA = tauB = ne - 1;
        it.g0 = l2 * 2 * job.C;
        it.slotA = 2 * l2;
        it.slotB = 2 * l2 + 1;
    }
    int eA = o + tauA, eB = o + tauB;
    if (job.pairs) {
        eA = job.pairs[eA];
        eB = job.pairs[eB];
    }
    if (eA < 0 || eA >= job.n_pairs || eB < 0 || eB >= job.n_pairs) {
        set_dev_error(job.status, RVQ_DEV_ERR_INDEX);
        return;
    }
    it.entryA = eA;
    it.entryB = eB;
    if (job.record_bytes) {
        it.codes = rec + job.codes_off[m];
        it.cb = reinterpret_cast<const float *>(rec + job.cb_off[m]);
    } else {
        it.codes = job.codes_ptr;
        it.cb = job.cb_ptr;
    }
    it.xA = reinterpret_cast<const uint8_t *>(job.x) +
            (int64_t)(eA / job.x_div) * job.x_stride * (job.x_dtype == RVQ_BF16 ? 2 : 4);
    it.xB = reinterpret_cast<const uint8_t *>(job.x) +
            (int64_t)(eB / job.x_div) * job.x_stride * (job.x_dtype == RVQ_BF16 ? 2 : 4);
    const int RB = job.rows / 32;
    it.nrb = RB / job.S;
    it.rb0 = split * it.nrb;
    it.valid = 1;
}

// Build the step's table.  Column c = lane.  Type 0 interleaves the two
// tokens (T[s][k][c][u], 8-byte pairs); type 1 keeps the two chunk groups in
// separate 128-byte halves (T[s][k][u][c]).  Two entries (k, k+1) per packed
// FMA, using the pair-interleaved codebook.
__device__ __forceinline__ void build_table(uint8_t *lut, const float *cb, const float xa[8],
                                            const float xb[8], int type, int lane, int warp) {
    uint64_t xa2[8], xb2[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        xa2[i] = pk2(xa[i], xa[i]);
        xb2[i] = pk2(xb[i], xb[i]);
    }
    const ulonglong2 *cb2 = reinterpret_cast<const ulonglong2 *>(cb);
#pragma unroll 2
    for (int kp = warp; kp < 3 * 128; kp += NW) {
        const int s = kp >> 7, k = (kp & 127) * 2;
        // 16 floats: (k, k+1) interleaved for dims 0..7
        ulonglong2 c0 = __ldg(cb2 + kp * 4 + 0);
        ulonglong2 c1 = __ldg(cb2 + kp * 4 + 1);
        ulonglong2 c2 = __ldg(cb2 + kp * 4 + 2);
        ulonglong2 c3 = __ldg(cb2 + kp * 4 + 3);
        const uint64_t cw[8] = {c0.x, c0.y, c1.x, c1.y, c2.x, c2.y, c3.x, c3.y};
        uint64_t ta = 0, tb = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            ta = ffma2(xa2[i], cw[i], ta);
            tb = ffma2(xb2[i], cw[i], tb);
        }
        const float2 a = upk2(ta), b = upk2(tb);  // (entry k, entry k+1)
        uint8_t *row0 = lut + s * kLutStageBytes + k * 256;
        uint8_t *row1 = row0 + 256;
        if (type == 0) {
            *reinterpret_cast<float2 *>(row0 + lane * 8) = make_float2(a.x, b.x);
            *reinterpret_cast<float2 *>(row1 + lane * 8) = make_float2(a.y, b.y);
        } else {
            *reinterpret_cast<float *>(row0 + lane * 4) = a.x;
            *reinterpret_cast<float *>(row1 + lane * 4) = a.y;
            *reinterpret_cast<float *>(row0 + 128 + lane * 4) = b.x;
            *reinterpret_cast<float *>(row1 + 128 + lane * 4) = b.y;
        }
    }
}

__device__ __forceinline__ void load_tile(uint4 (&c)[6], const uint8_t *tile) {
#pragma unroll
    for (int q = 0; q < 6; ++q) c[q] = ldg_stream(tile + q * 512);
}

__device__ __forceinline__ uint32_t word_of(const uint4 &v, int q) {
    return q == 0 ? v.x : q == 1 ? v.y : q == 2 ? v.z : v.w;
}

// Two tokens, one chunk group: one permute + one 8-byte LDS per code byte.
__device__ __forceinline__ uint64_t rows_pair(const uint4 (&c)[6], const uint32_t (&aux)[32],
                                              const uint8_t *lut) {
    uint64_t acc = 0;
#pragma unroll
    for (int s = 0; s < 3; ++s)
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t w = word_of(c[s * 2 + h], q);
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    const uint32_t idx = prmt(w, aux[h * 16 + q * 4 + b], 0x7604u | (b << 4));
                    const uint64_t v =
                        *reinterpret_cast<const uint64_t *>(lut + s * kLutStageBytes + idx);
                    acc = fadd2(acc, v);
                }
            }
    return acc;
}

// One token, two chunk groups: two permutes + two 4-byte LDS per code pair.
__device__ __forceinline__ uint64_t rows_single(const uint4 (&ca)[6], const uint4 (&cb)[6],
                                                const uint32_t (&aux)[32], const uint8_t *lut) {
    uint64_t acc = 0;
#pragma unroll
    for (int s = 0; s < 3; ++s)
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t wa = word_of(ca[s * 2 + h], q);
                const uint32_t wb = word_of(cb[s * 2 + h], q);
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    const uint32_t a = aux[h * 16 + q * 4 + b];
                    const uint32_t ia = prmt(wa, a, 0x7604u | (b << 4));
                    const uint32_t ib = prmt(wb, a, 0x7604u | (b << 4));
                    const float va =
                        *reinterpret_cast<const float *>(lut + s * kLutStageBytes + ia);
                    const float vb =
                        *reinterpret_cast<const float *>(lut + s * kLutStageBytes + 128 + ib);
                    acc = fadd2(acc, pk2(va, vb));
                }
            }
    return acc;
}

template <int TYPE>
__device__ __forceinline__ void run_item(const LutJob &job, const Item &it, int m, uint8_t *lut,
                                         float2 *sacc) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int RB = job.rows / 32;
    const int C = job.C;
    const int nrb_w = (it.nrb - warp + NW - 1) / NW;  // may be 0
    const int nslot = job.G / C;
    float *part = job.part[m];

    uint32_t aux[32];
#pragma unroll
    for (int t = 0; t < 32; ++t) aux[t] = ((lane + t) & 31) << (TYPE == 0 ? 3 : 2);

    auto tile_ptr = [&](int g, int rb) {
        return it.codes + ((size_t)g * RB + rb) * kTileBytes + lane * 16;
    };
    const int gstep = TYPE == 0 ? 1 : 2;

    uint4 curA[6], curB[6], nxtA[6], nxtB[6];
    if (nrb_w > 0) {
        load_tile(curA, tile_ptr(it.g0, it.rb0 + warp));
        if (TYPE == 1) load_tile(curB, tile_ptr(it.g0 + 1, it.rb0 + warp));
    }
    for (int j = 0; j < C; ++j) {
        const int gA = it.g0 + j * gstep, gB = gA + (TYPE == 0 ? 0 : 1);
        float xa[8], xb[8];
        load8(it.xA, job.x_dtype, (int64_t)(gA * 32 + lane) * 8, xa);
        load8(it.xB, job.x_dtype, (int64_t)(gB * 32 + lane) * 8, xb);
        if (j > 0) __syncthreads();
        build_table(lut, it.cb, xa, xb, TYPE, lane, warp);
        __syncthreads();
        for (int i = 0; i < nrb_w; ++i) {
            const int rb = it.rb0 + warp + NW * i;
            // prefetch the next row block (possibly of the next step)
            int jn = j, in = i + 1;
            if (in >= nrb_w) { jn = j + 1; in = 0; }
            if (jn < C) {
                const int gnA = it.g0 + jn * gstep;
                const int rbn = it.rb0 + warp + NW * in;
                load_tile(nxtA, tile_ptr(gnA, rbn));
                if (TYPE == 1) load_tile(nxtB, tile_ptr(gnA + 1, rbn));
            }
            uint64_t acc = TYPE == 0 ? rows_pair(curA, aux, lut) : rows_single(curA, curB, aux, lut);
            float2 a = upk2(acc);
            const int rl = (rb - it.rb0) * 32 + lane;
            if (C > 1) {
                if (j > 0) {
                    const float2 prev = sacc[rl];
                    a.x += prev.x;
                    a.y += prev.y;
                }
                if (j < C - 1) sacc[rl] = a;
            }
            if (j == C - 1) {
                const int row = rb * 32 + lane;
                part[((size_t)it.entryA * nslot + it.slotA) * job.rows + row] = a.x;
                part[((size_t)it.entryB * nslot + it.slotB) * job.rows + row] = a.y;
            }
#pragma unroll
            for (int q = 0; q < 6; ++q) {
                curA[q] = nxtA[q];
                if (TYPE == 1) curB[q] = nxtB[q];
            }
        }
    }
}

__global__ void __launch_bounds__(NT, 1) lut_gemv_kernel(const LutJob job) {
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ Item it;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int m = blockIdx.y;
    if (threadIdx.x == 0) decode_item(job, m, it);
    __syncthreads();
    if (!it.valid) return;
    asm volatile("griddepcontrol.launch_dependents;");
    float2 *sacc = reinterpret_cast<float2 *>(smem + kLutBytes);
    if (it.type == 0)
        run_item<0>(job, it, m, smem, sacc);
    else
        run_item<1>(job, it, m, smem, sacc);
}

// ---------------------------------------------------------------- reductions

__global__ void swiglu_reduce_kernel(const float *__restrict__ gpart,
                                     const float *__restrict__ upart, int n_pairs, int nslot,
                                     int rows, float *__restrict__ h) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)n_pairs * rows) return;
    const int64_t p = i / rows, r = i % rows;
    const float *gp = gpart + p * nslot * rows + r;
    const float *up = upart + p * nslot * rows + r;
    float g = 0.f, u = 0.f;
    for (int s = 0; s < nslot; ++s) {
        g += gp[(int64_t)s * rows];
        u += up[(int64_t)s * rows];
    }
    h[i] = g / (1.0f + expf(-g)) * u;
}

__global__ void slot_reduce_kernel(const float *__restrict__ part, int64_t n_entries, int nslot,
                                   int rows, float *__restrict__ y) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n_entries * rows) return;
    const int64_t p = i / rows, r = i % rows;
    const float *pp = part + p * nslot * rows + r;
    float acc = 0.f;
    for (int s = 0; s < nslot; ++s) acc += pp[(int64_t)s * rows];
    y[i] = acc;
}

// Standalone table build: lut[t][j][s][k] for canonical codebooks.
__global__ void lut_build_kernel(const float *__restrict__ cb, const void *__restrict__ x, int xdt,
                                 int n, int cols, float *__restrict__ lut) {
    const int chunks = cols / 8;
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t total = (int64_t)n * chunks * 768;
    if (i >= total) return;
    const int sk = (int)(i % 768);
    const int64_t tj = i / 768;
    const int j = (int)(tj % chunks);
    const int t = (int)(tj / chunks);
    float xv[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) xv[q] = load1(x, xdt, (int64_t)t * cols + j * 8 + q);
    const float *c = cb + (int64_t)sk * 8;
    float acc = 0.f;
#pragma unroll
    for (int q = 0; q < 8; ++q) acc = fmaf(xv[q], c[q], acc);
    lut[i] = acc;
}

template <typename K, typename... Args>
cudaError_t launch_ex(K kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl,
                      Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace

rvq_status launch_lut_gemv(const LutJob &job, cudaStream_t stream, bool pdl) {
    static int attr_done[64] = {0};
    int dev = 0;
    RVQ_CUDA(cudaGetDevice(&dev));
    const size_t smem = kLutBytes + (size_t)kMaxSplitRows * sizeof(float2);
    if (dev < 64 && !attr_done[dev]) {
        RVQ_CUDA(cudaFuncSetAttribute(lut_gemv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)smem));
        attr_done[dev] = 1;
    }
    if (job.rows / job.S > kMaxSplitRows || (job.rows / 32) % job.S != 0 ||
        job.G % (2 * job.C) != 0) {
        set_error("lut_gemv: bad split (rows %d, S %d, G %d, C %d)", job.rows, job.S, job.G,
                  job.C);
        return RVQ_EINVAL;
    }
    const int items = lut_items(job);
    if (items == 0) return RVQ_OK;
    dim3 grid(items, job.n_mat);
    RVQ_CUDA(launch_ex(lut_gemv_kernel, grid, dim3(NT), smem, stream, pdl, job));
    return RVQ_OK;
}

rvq_status launch_swiglu_reduce(const float *gpart, const float *upart, int n_pairs, int nslot,
                                int rows, float *h, cudaStream_t stream, bool pdl) {
    const int64_t total = (int64_t)n_pairs * rows;
    if (total == 0) return RVQ_OK;
    const int bs = 256;
    RVQ_CUDA(launch_ex(swiglu_reduce_kernel, dim3((unsigned)((total + bs - 1) / bs)), dim3(bs), 0,
                       stream, pdl, gpart, upart, n_pairs, nslot, rows, h));
    return RVQ_OK;
}

rvq_status launch_slot_reduce(const float *part, int n_entries, int nslot, int rows, float *y,
                              cudaStream_t stream, bool pdl) {
    const int64_t total = (int64_t)n_entries * rows;
    if (total == 0) return RVQ_OK;
    const int bs = 256;
    RVQ_CUDA(launch_ex(slot_reduce_kernel, dim3((unsigned)((total + bs - 1) / bs)), dim3(bs), 0,
                       stream, pdl, part, (int64_t)n_entries, nslot, rows, y));
    return RVQ_OK;
}

rvq_status launch_lut_build(const float *cb, const void *x, int xdt, int n, int cols, float *lut,
                            cudaStream_t stream) {
    const int64_t total = (int64_t)n * (cols / 8) * 768;
    if (total == 0) return RVQ_OK;
    const int bs = 256;
    lut_build_kernel<<<(unsigned)((total + bs - 1) / bs), bs, 0, stream>>>(cb, x, xdt, n, cols, lut);
    RVQ_LAUNCHED("lut_build");
    return RVQ_OK;
}

}  // namespace rvq
