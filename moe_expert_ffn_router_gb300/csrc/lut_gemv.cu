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

constexpr int NT = 512;
constexpr int NW = NT / 32;
constexpr int kMaxSplitRows = 2048;  // rows per item: at most 8 row blocks per warp
constexpr int kMaxAccRows = 1024;    // rows per item when C > 1 (shared accumulator)
constexpr int kCbBytes = 3 * 128 * 8 * 2 * 4;  // packed codebook of one matrix, 24 KiB

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

// Decode blockIdx into an item, with the whole of warp 0 (all 32 lanes call
// it; lane 0 writes `it`).  The expert segment holding pair position p is
// found with one parallel read of offsets[0..E] (9 per lane) and a ballot;
// the two pair entries and the record header are then read in parallel: two
// dependent memory round trips per item.
__device__ void decode_item(const LutJob &job, int m, Item &it) {
    const int lane = threadIdx.x & 31;
    const int per_pair = job.G / (2 * job.C);
    const int i = blockIdx.x / job.S;
    const int split = blockIdx.x % job.S;
    const int p = i / per_pair;
    bool ok = p < job.n_pairs;
    int e = 0, o = 0, ne = job.n_pairs;
    if (ok && job.offsets) {
        int off[9];
#pragma unroll
        for (int q = 0; q < 9; ++q) {
            const int x = lane * 9 + q;
            off[q] = x <= job.E ? job.offsets[x] : 0x7fffffff;
        }
        const int next_first = __shfl_down_sync(0xffffffffu, off[0], 1);
        int found = -1, fo = 0, fhi = 0;
#pragma unroll
        for (int q = 0; q < 9; ++q) {
            const int x = lane * 9 + q;
            const int hi = q < 8 ? off[q + 1] : (lane < 31 ? next_first : 0x7fffffff);
            if (found < 0 && x < job.E && off[q] <= p && p < hi) {
                found = x;
                fo = off[q];
                fhi = hi;
            }
        }
        // offsets[0] sits in lane 0, offsets[E] in lane E / 9
        const int o0 = __shfl_sync(0xffffffffu, off[0], 0);
        int oE = 0;
#pragma unroll
        for (int q = 0; q < 9; ++q)
            if (lane * 9 + q == job.E) oE = off[q];
        oE = __shfl_sync(0xffffffffu, oE, job.E / 9);
        const unsigned hit = __ballot_sync(0xffffffffu, found >= 0);
        if (o0 != 0 || oE != job.n_pairs || hit == 0) {
            ok = false;
        } else {
            const int src = __ffs(hit) - 1;
            e = __shfl_sync(0xffffffffu, found, src);
            o = __shfl_sync(0xffffffffu, fo, src);
            ne = __shfl_sync(0xffffffffu, fhi, src) - o;
            ok = 0 <= o && o <= p && p < o + ne && o + ne <= job.n_pairs;
        }
        if (!ok && lane == 0) set_dev_error(job.status, RVQ_DEV_ERR_INDEX);
    }
    if (!ok) {
        if (lane == 0) it.valid = 0;
        return;
    }
    const int li = i - per_pair * o;
    const int Q = ne >> 1;
    const int runs = job.G / job.C;  // chunk-group runs of the two-token items
    int type, tauA, tauB, g0, slotA, slotB;
    if (li < Q * runs) {
        const int gr = li / Q, q = li % Q;
        type = 0;
        tauA = 2 * q;
        tauB = 2 * q + 1;
        g0 = gr * job.C;
        slotA = slotB = gr;
    } else {
        const int l2 = li - Q * runs;
        type = 1;
        tauA = tauB = ne - 1;
        g0 = l2 * 2 * job.C;
        slotA = 2 * l2;
        slotB = 2 * l2 + 1;
    }
    const uint8_t *rec = job.base ? job.base + (uint64_t)e * job.record_bytes : nullptr;
    // parallel reads: lane 0 / 1 the pair entries, lane 2 the header words
    int v = 0;
    if (lane == 0) v = job.pairs ? job.pairs[o + tauA] : o + tauA;
    if (lane == 1) v = job.pairs ? job.pairs[o + tauB] : o + tauB;
    bool hdr_ok = true;
    if (lane == 2 && job.check_header && rec) {
        const rvq_expert_header *h = reinterpret_cast<const rvq_expert_header *>(rec);
        hdr_ok = h->magic == RVQ_BANK_MAGIC && h->expert == e && h->layer == job.layer &&
                 h->d == job.d && h->f == job.f && h->record_bytes == job.record_bytes;
    }
    const int eA = __shfl_sync(0xffffffffu, v, 0);
    const int eB = __shfl_sync(0xffffffffu, v, 1);
    hdr_ok = __shfl_sync(0xffffffffu, hdr_ok ? 1 : 0, 2) != 0;
    if (lane != 0) return;
    it.valid = 0;
    if (!hdr_ok) {
        set_dev_error(job.status, RVQ_DEV_ERR_CORRUPT);
        return;
    }
    if (eA < 0 || eA >= job.n_pairs || eB < 0 || eB >= job.n_pairs) {
        set_dev_error(job.status, RVQ_DEV_ERR_INDEX);
        return;
    }
    it.type = type;
    it.g0 = g0;
    it.slotA = slotA;
    it.slotB = slotB;
    it.entryA = eA;
    it.entryB = eB;
    if (job.record_bytes) {
        it.codes = rec + job.codes_off[m];
        it.cb = reinterpret_cast<const float *>(rec + job.cb_off[m]);
    } else {
        it.codes = job.codes_ptr;
        it.cb = job.cb_ptr;
    }
    const int esz = job.x_dtype == RVQ_BF16 ? 2 : 4;
    it.xA = reinterpret_cast<const uint8_t *>(job.x) + (int64_t)(eA / job.x_div) * job.x_stride * esz;
    it.xB = reinterpret_cast<const uint8_t *>(job.x) + (int64_t)(eB / job.x_div) * job.x_stride * esz;
    const int RB = job.rows / 32;
    it.nrb = RB / job.S;
    it.rb0 = split * it.nrb;
    it.valid = 1;
}

// Build the step's table.  Column c = lane.  Type 0 interleaves the two
// tokens (T[s][k][c][u], 8-byte pairs); type 1 keeps the two chunk groups in
// separate 128-byte halves (T[s][k][u][c]).  Two entries (k, k+1) per packed
// FMA, using the pair-interleaved codebook.
__device__ __forceinline__ void build_table(uint8_t *lut, const uint8_t *cb_s, const float xa[8],
                                            const float xb[8], int type, int lane, int warp) {
    uint64_t xa2[8], xb2[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        xa2[i] = pk2(xa[i], xa[i]);
        xb2[i] = pk2(xb[i], xb[i]);
    }
    const ulonglong2 *cb2 = reinterpret_cast<const ulonglong2 *>(cb_s);
#pragma unroll 4
    for (int kp = warp; kp < 3 * 128; kp += NW) {
        const int s = kp >> 7, k = (kp & 127) * 2;
        // 16 floats: (k, k+1) interleaved for dims 0..7 (same address in every
        // lane: shared-memory broadcast)
        const ulonglong2 c0 = cb2[kp * 4 + 0];
        const ulonglong2 c1 = cb2[kp * 4 + 1];
        const ulonglong2 c2 = cb2[kp * 4 + 2];
        const ulonglong2 c3 = cb2[kp * 4 + 3];
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

__device__ __forceinline__ uint32_t word_of(const uint4 &v, int q) {
    return q == 0 ? v.x : q == 1 ? v.y : q == 2 ? v.z : v.w;
}

// One 32-row x 32-chunk code tile (6 words of 16 B per lane) against the
// table.  Two tokens (TYPE 0): one permute + one 8-byte LDS per code byte
// gives both tokens' entries.  One token (TYPE 1): one permute + one 4-byte LDS
// per code byte, two lookups per packed add.  aux[t] carries the lane's
// rotated column offset (and, for TYPE 1, the table half) in bits 0..7.
template <int TYPE>
__device__ __forceinline__ uint64_t tile_lookups(const uint4 (&c)[6], const uint32_t (&aux)[32],
                                                 const uint8_t *lut) {
    uint64_t acc = 0;
#pragma unroll
    for (int s = 0; s < 3; ++s)
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t w = word_of(c[s * 2 + h], q);
                if constexpr (TYPE == 0) {
#pragma unroll
                    for (int b = 0; b < 4; ++b) {
                        const uint32_t idx = prmt(w, aux[h * 16 + q * 4 + b], 0x7604u | (b << 4));
                        acc = fadd2(acc, *reinterpret_cast<const uint64_t *>(
                                             lut + s * kLutStageBytes + idx));
                    }
                } else {
#pragma unroll
                    for (int b = 0; b < 4; b += 2) {
                        const uint32_t i0 = prmt(w, aux[h * 16 + q * 4 + b], 0x7604u | (b << 4));
                        const uint32_t i1 =
                            prmt(w, aux[h * 16 + q * 4 + b + 1], 0x7604u | ((b + 1) << 4));
                        const float v0 = *reinterpret_cast<const float *>(lut + s * kLutStageBytes + i0);
                        const float v1 = *reinterpret_cast<const float *>(lut + s * kLutStageBytes + i1);
                        acc = fadd2(acc, pk2(v0, v1));
                    }
                }
            }
    return acc;
}

// Streams the item's code tiles through a 2-deep register ring.  Work unit =
// one code tile: TYPE 0 has one tile per row block (both tokens), TYPE 1 two
// (groups A and B, each against its own table half).  With 16 warps a warp's
// tiles are q = warp + 16 i; for TYPE 1 the table half is warp & 1.  The first
// tiles of a step are requested before its table is built, so the build
// overlaps HBM traffic; tile i + D is requested once tile i is consumed.
template <int TYPE>
__device__ __forceinline__ void run_item(const LutJob &job, const Item &it, int m, uint8_t *lut,
                                         uint8_t *cb_s, float *sacc) {
    constexpr int D = 2;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int RB = job.rows / 32;
    const int C = job.C;
    const int ntiles = TYPE == 0 ? it.nrb : 2 * it.nrb;
    const int nt_w = (ntiles - warp + NW - 1) / NW;  // tiles of this warp (may be 0)
    const int nslot = job.G / C;
    const int rows_split = it.nrb * 32;
    float *part = job.part[m];
    const int gstep = TYPE == 0 ? 1 : 2;
    const int u = TYPE == 0 ? 0 : (warp & 1);  // table half / unit of this warp (TYPE 1)

    uint32_t aux[32];
#pragma unroll
    for (int t = 0; t < 32; ++t)
        aux[t] = TYPE == 0 ? (((lane + t) & 31) << 3) : ((((lane + t) & 31) << 2) | (u << 7));

    auto tile_rb = [&](int i) {  // row block of this warp's i-th tile
        const int q = warp + NW * i;
        return it.rb0 + (TYPE == 0 ? q : (q >> 1));
    };
    uint4 buf[D][6];
    auto load_tile = [&](uint4 (&b)[6], int gA, int i) {
        const int g = gA + u;
        const uint8_t *p = it.codes + ((size_t)g * RB + tile_rb(i)) * kTileBytes + lane * 16;
#pragma unroll
        for (int q = 0; q < 6; ++q) b[q] = ldg_stream(p + q * 512);
    };

    // item prologue: first tiles in flight, then the matrix's codebook into
    // shared memory (one coalesced 24 KiB copy per item)
#pragma unroll
    for (int d = 0; d < D; ++d)
        if (d < nt_w) load_tile(buf[d], it.g0, d);
    {
        const uint4 *src = reinterpret_cast<const uint4 *>(it.cb);
        uint4 *dst = reinterpret_cast<uint4 *>(cb_s);
        uint4 v[kCbBytes / 16 / NT];
#pragma unroll
        for (int q = 0; q < kCbBytes / 16 / NT; ++q) v[q] = __ldg(src + threadIdx.x + NT * q);
#pragma unroll
        for (int q = 0; q < kCbBytes / 16 / NT; ++q) dst[threadIdx.x + NT * q] = v[q];
    }
    for (int j = 0; j < C; ++j) {
        const int gA = it.g0 + j * gstep, gB = gA + (TYPE == 0 ? 0 : 1);
        if (j > 0) {
#pragma unroll
            for (int d = 0; d < D; ++d)
                if (d < nt_w) load_tile(buf[d], gA, d);
        }
        float xa[8], xb[8];
        load8(it.xA, job.x_dtype, (int64_t)(gA * 32 + lane) * 8, xa);
        load8(it.xB, job.x_dtype, (int64_t)(gB * 32 + lane) * 8, xb);
        __syncthreads();  // codebook stored (j = 0) / previous step's lookups done (j > 0)
        build_table(lut, cb_s, xa, xb, TYPE, lane, warp);
        __syncthreads();
        for (int i0 = 0; i0 < nt_w; i0 += D) {
#pragma unroll
            for (int d = 0; d < D; ++d) {
                const int i = i0 + d;
                if (i < nt_w) {
                    const uint64_t acc = tile_lookups<TYPE>(buf[d], aux, lut);
                    if (i + D < nt_w) load_tile(buf[d], gA, i + D);
                    const int rb = tile_rb(i);
                    const int rl = (rb - it.rb0) * 32 + lane;
                    const int row = rb * 32 + lane;
                    float2 a = upk2(acc);
                    if constexpr (TYPE == 1) {
                        // one token: both halves of the packed sum belong to this unit
                        float v = a.x + a.y;
                        if (C > 1) {
                            if (j > 0) v += sacc[u * rows_split + rl];
                            if (j < C - 1) sacc[u * rows_split + rl] = v;
                        }
                        if (j == C - 1) {
                            const int e = u ? it.entryB : it.entryA;
                            const int sl = u ? it.slotB : it.slotA;
                            part[((size_t)e * nslot + sl) * job.rows + row] = v;
                        }
                    } else {
                        if (C > 1) {
                            if (j > 0) {
                                a.x += sacc[rl];
                                a.y += sacc[rows_split + rl];
                            }
                            if (j < C - 1) {
                                sacc[rl] = a.x;
                                sacc[rows_split + rl] = a.y;
                            }
                        }
                        if (j == C - 1) {
                            part[((size_t)it.entryA * nslot + it.slotA) * job.rows + row] = a.x;
                            part[((size_t)it.entryB * nslot + it.slotB) * job.rows + row] = a.y;
                        }
                    }
                }
            }
        }
    }
}

__global__ void __launch_bounds__(NT, 1) lut_gemv_kernel(const LutJob job) {
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ Item it;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int m = blockIdx.y;
    if (threadIdx.x < 32) decode_item(job, m, it);
    __syncthreads();
    if (!it.valid) return;
    asm volatile("griddepcontrol.launch_dependents;");
    uint8_t *cb_s = smem + kLutBytes;
    float *sacc = reinterpret_cast<float *>(cb_s + kCbBytes);
    if (it.type == 0)
        run_item<0>(job, it, m, smem, cb_s, sacc);
    else
        run_item<1>(job, it, m, smem, cb_s, sacc);
}

// ---------------------------------------------------------------- reductions

// h[p][r..r+3] = silu(sum_s g) * sum_s u over the split-K slots.  Four
// adjacent lanes share one float4 of rows and take every fourth slot; two
// xor-shuffles combine their sums (a fixed order, so results are repeatable).
__global__ void __launch_bounds__(256) swiglu_reduce_kernel(const float *__restrict__ gpart,
                                                            const float *__restrict__ upart,
                                                            int n_pairs, int nslot, int rows,
                                                            float *__restrict__ h) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    const int r4 = rows >> 2;
    const int64_t gi = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int j = (int)(gi & 3);
    const int64_t i = gi >> 2;
    const bool valid = i < (int64_t)n_pairs * r4;
    float4 g = make_float4(0.f, 0.f, 0.f, 0.f), u = g;
    if (valid) {
        const int64_t p = i / r4, r = (i % r4) * 4;
        const float4 *gp = reinterpret_cast<const float4 *>(gpart + p * nslot * rows + r);
        const float4 *up = reinterpret_cast<const float4 *>(upart + p * nslot * rows + r);
#pragma unroll 4
        for (int s = j; s < nslot; s += 4) {
            const float4 a = __ldg(gp + (int64_t)s * r4), b = __ldg(up + (int64_t)s * r4);
            g.x += a.x; g.y += a.y; g.z += a.z; g.w += a.w;
            u.x += b.x; u.y += b.y; u.z += b.z; u.w += b.w;
        }
    }
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
        g.x += __shfl_xor_sync(0xffffffffu, g.x, o);
        g.y += __shfl_xor_sync(0xffffffffu, g.y, o);
        g.z += __shfl_xor_sync(0xffffffffu, g.z, o);
        g.w += __shfl_xor_sync(0xffffffffu, g.w, o);
        u.x += __shfl_xor_sync(0xffffffffu, u.x, o);
        u.y += __shfl_xor_sync(0xffffffffu, u.y, o);
        u.z += __shfl_xor_sync(0xffffffffu, u.z, o);
        u.w += __shfl_xor_sync(0xffffffffu, u.w, o);
    }
    if (!valid || j != 0) return;
    float4 o;
    o.x = g.x / (1.0f + expf(-g.x)) * u.x;
    o.y = g.y / (1.0f + expf(-g.y)) * u.y;
    o.z = g.z / (1.0f + expf(-g.z)) * u.z;
    o.w = g.w / (1.0f + expf(-g.w)) * u.w;
    reinterpret_cast<float4 *>(h)[i] = o;
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
    const size_t smem = kLutBytes + kCbBytes + (size_t)kMaxAccRows * 2 * sizeof(float);
    if (dev < 64 && !attr_done[dev]) {
        RVQ_CUDA(cudaFuncSetAttribute(lut_gemv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)smem));
        attr_done[dev] = 1;
    }
    if (job.rows / job.S > kMaxSplitRows || (job.C > 1 && job.rows / job.S > kMaxAccRows) ||
        (job.rows / 32) % job.S != 0 ||
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
    const int64_t total = (int64_t)n_pairs * (rows / 4) * 4;
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
