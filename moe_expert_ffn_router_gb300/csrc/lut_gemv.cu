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
//  * Work is split into "items": one expert matrix, two (token, 32-chunk
//    group) units, a run of C steps over chunk groups and a range of rows.  A
//    step's table (2 units x 3 stages x 256 entries x 32 chunks, 192 KiB)
//    lives in shared memory, built once per (token, chunk group, row range)
//    and never written to HBM.
//  * A small plan kernel turns the grouping (offsets, pairs) into one 16-byte
//    descriptor per item and checks each expert record's header.
//  * The GEMV kernel is persistent: one block per SM walks its items.  While
//    it streams the codes of one item it already fetches the next item's
//    codebook and inputs (cp.async into shared memory) and its first code
//    tiles (register ring), so HBM keeps streaming across item boundaries.
//  * Lane l of a warp owns row 32b + l.  The packed code layout rotates each
//    row's chunk order by l, so at every unrolled step t the 32 lanes read 32
//    different table columns (bank = column): the lookups are conflict-free
//    for any code values, and each lane accumulates its own row with no
//    cross-lane reduction.
//  * A code byte becomes a shared-memory address with one byte permute
//    (code -> bits 8..15, column offset -> bits 0..7), one LDS and half of a
//    packed fp32x2 add.  Code tiles (3 KiB per 32 rows x 32 chunks) are
//    streamed with 128-bit non-allocating loads.
//  * Items of the same (expert, chunk group) for different token pairs are
//    adjacent in the item order, so a second token pair re-reads codes from L2.
//  * Split-K partials (one slot per item column range) are reduced by the
//    next kernel (SwiGLU for gate/up, the combine for down); the decode
//    kernel's down launch reduces the gate/up partials itself.
#include "internal.cuh"
#include "lut_common.cuh"

#include <type_traits>

namespace rvq {
namespace {

constexpr int NT = 512;
constexpr int NW = NT / 32;
constexpr int kMaxSplitRows = 2048;  // rows per item: at most 8 row blocks per warp
constexpr int kMaxAccRows = 512;     // rows per item when C > 1 (shared accumulator)
constexpr int kCbBytes = 3 * 128 * 8 * 2 * 4;  // packed codebook of one matrix, 24 KiB
constexpr int kXsBytes = 2 * 32 * 8 * 4;        // inputs of one step: 2 units x 32 chunks x 8 fp32
constexpr int kSmemBytes = kLutBytes + kCbBytes + kXsBytes + kMaxAccRows * 2 * 4;

__device__ __forceinline__ uint64_t ffma2(uint64_t x, uint64_t y, uint64_t acc) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(x), "l"(y), "l"(acc));
    return r;
}
__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gmem_src) {
    const uint32_t d = (uint32_t)__cvta_generic_to_shared(smem_dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// ----------------------------------------------------------------- plan
// Item i of a launch (before the row split) -> descriptor.  Item order
// within expert e (n_e tokens, Q = n_e / 2 token pairs, G/C runs of C chunk
// groups): two-token items li = run * Q + q, then (n_e odd) the one-token
// items of the last token, each covering 2C groups.
__device__ ItemDesc plan_one(const LutJob &job, const int32_t *soff, int i) {
    ItemDesc d;
    d.expert = -1;
    d.entryA = d.entryB = 0;
    d.g0 = 0;
    d.type = 0;
    d.pad = 0;
    const int per_pair = job.G / (2 * job.C);
    const int p = i / per_pair;
    int e = 0, o = 0, ne = job.n_pairs;
    if (job.offsets) {
        if (soff[0] != 0 || soff[job.E] != job.n_pairs) {
            set_dev_error(job.status, RVQ_DEV_ERR_INDEX);
            return d;
        }
        int lo = 0, hi = job.E;  // largest e with offsets[e] <= p
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (soff[mid] <= p) lo = mid; else hi = mid;
        }
        e = lo;
        o = soff[e];
        ne = soff[e + 1] - o;
        if (!(0 <= o && o <= p && p < o + ne && o + ne <= job.n_pairs)) {
            set_dev_error(job.status, RVQ_DEV_ERR_INDEX);
            return d;
        }
        if (job.tc_min_tokens > 0 && ne >= job.tc_min_tokens) {
            d.expert = -2;  // the tensor-core path takes this expert
            return d;
        }
    }
    const int li = i - per_pair * o;
    const int Q = ne >> 1;
    const int runs = job.G / job.C;
    int tauA, tauB;
    if (li < Q * runs) {
        d.type = 0;
        tauA = 2 * (li % Q);
        tauB = tauA + 1;
        d.g0 = (int16_t)((li / Q) * job.C);
    } else {
        d.type = 1;
        tauA = tauB = ne - 1;
        d.g0 = (int16_t)((li - Q * runs) * 2 * job.C);
    }
    const int eA = job.pairs ? job.pairs[o + tauA] : o + tauA;
    const int eB = job.pairs ? job.pairs[o + tauB] : o + tauB;
    if (eA < 0 || eA >= job.n_pairs || eB < 0 || eB >= job.n_pairs) {
        set_dev_error(job.status, RVQ_DEV_ERR_INDEX);
        return d;
    }
    // the walkers address the record by this index (an expert cache's slot)
    const int rec = job.base ? record_of(job, e) : e;
    if (rec < 0) {
        set_dev_error(job.status, RVQ_DEV_ERR_CORRUPT);
        return d;
    }
    if (job.check_header && job.base) {
        // the pages check magic, expert id and offset range on every read
        const rvq_expert_header *h = reinterpret_cast<const rvq_expert_header *>(
            job.base + (uint64_t)rec * job.record_bytes);
        if (h->magic != RVQ_BANK_MAGIC || h->expert != e || h->layer != job.layer ||
            h->d != job.d || h->f != job.f || h->record_bytes != job.record_bytes) {
            set_dev_error(job.status, RVQ_DEV_ERR_CORRUPT);
            return d;
        }
    }
    d.expert = rec;
    d.entryA = eA;
    d.entryB = eB;
    return d;
}

__global__ void __launch_bounds__(256) plan_kernel(const LutJob ja, const LutJob jb) {
    __shared__ int32_t soff[257];
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    const int32_t *offsets = ja.offsets;
    const int E = ja.E;
    if (offsets)
        for (int x = threadIdx.x; x <= E; x += blockDim.x) soff[x] = offsets[x];
    __syncthreads();
    const int na = lut_items(ja) / ja.S;
    const int nb = jb.n_pairs ? lut_items(jb) / jb.S : 0;
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t < na)
        ja.desc[t] = plan_one(ja, soff, t);
    else if (t < na + nb)
        jb.desc[t - na] = plan_one(jb, soff, t - na);
}

// ----------------------------------------------------------------- table build
// Two entries (k, k+1) per packed FMA from the pair-interleaved codebook in
// shared memory.  Half-warp h takes entry pair 2w' + h (w' = warp's step), so
// one 128-bit broadcast load serves two entry pairs; lane r of a half handles
// columns r and r + 16 (in swapped order in the upper half so the 4-byte
// stores of the two halves fall in different banks).  Type 0 interleaves the
// two tokens (T[s][k][c][u], 8-byte pairs); type 1 keeps the two chunk groups
// in separate 128-byte halves (T[s][k][u][c]).
__device__ __forceinline__ void build_table(uint8_t *lut, const uint8_t *cb_s, const uint8_t *xs_s,
                                            int xdt, int type, int lane, int warp) {
    const int hf = lane >> 4, r = lane & 15;
    const int c0 = hf ? r + 16 : r, c1 = hf ? r : r + 16;
    uint64_t x2[4][8];  // (unit A col c0, A c1, B c0, B c1) x dims, duplicated pairs
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        const int u = v >> 1, c = (v & 1) ? c1 : c0;
        float xv[8];
        if (xdt == RVQ_BF16) {
            const uint4 q = *reinterpret_cast<const uint4 *>(xs_s + (u * 32 + c) * 16);
            const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                xv[2 * i] = __uint_as_float(w[i] << 16);
                xv[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
            }
        } else {
            const float4 a = *reinterpret_cast<const float4 *>(xs_s + (u * 32 + c) * 32);
            const float4 b = *reinterpret_cast<const float4 *>(xs_s + (u * 32 + c) * 32 + 16);
            xv[0] = a.x; xv[1] = a.y; xv[2] = a.z; xv[3] = a.w;
            xv[4] = b.x; xv[5] = b.y; xv[6] = b.z; xv[7] = b.w;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) x2[v][i] = pk2(xv[i], xv[i]);
    }
    const ulonglong2 *cb2 = reinterpret_cast<const ulonglong2 *>(cb_s);
#pragma unroll 2
    for (int kq = warp; kq < 3 * 64; kq += NW) {
        const int kp = 2 * kq + hf;  // entry pair index over all stages
        const int s = kp >> 7, k = (kp & 127) * 2;
        const ulonglong2 q0 = cb2[kp * 4 + 0];
        const ulonglong2 q1 = cb2[kp * 4 + 1];
        const ulonglong2 q2 = cb2[kp * 4 + 2];
        const ulonglong2 q3 = cb2[kp * 4 + 3];
        const uint64_t cw[8] = {q0.x, q0.y, q1.x, q1.y, q2.x, q2.y, q3.x, q3.y};
        uint64_t t[4] = {0, 0, 0, 0};
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int v = 0; v < 4; ++v) t[v] = ffma2(x2[v][i], cw[i], t[v]);
        const float2 a0 = upk2(t[0]), a1 = upk2(t[1]), b0 = upk2(t[2]), b1 = upk2(t[3]);
        uint8_t *row0 = lut + s * kLutStageBytes + k * 256;
        uint8_t *row1 = row0 + 256;
        if (type == 0) {
            *reinterpret_cast<float2 *>(row0 + c0 * 8) = make_float2(a0.x, b0.x);
            *reinterpret_cast<float2 *>(row1 + c0 * 8) = make_float2(a0.y, b0.y);
            *reinterpret_cast<float2 *>(row0 + c1 * 8) = make_float2(a1.x, b1.x);
            *reinterpret_cast<float2 *>(row1 + c1 * 8) = make_float2(a1.y, b1.y);
        } else {
            *reinterpret_cast<float *>(row0 + c0 * 4) = a0.x;
            *reinterpret_cast<float *>(row1 + c0 * 4) = a0.y;
            *reinterpret_cast<float *>(row0 + c1 * 4) = a1.x;
            *reinterpret_cast<float *>(row1 + c1 * 4) = a1.y;
            *reinterpret_cast<float *>(row0 + 128 + c0 * 4) = b0.x;
            *reinterpret_cast<float *>(row1 + 128 + c0 * 4) = b0.y;
            *reinterpret_cast<float *>(row0 + 128 + c1 * 4) = b1.x;
            *reinterpret_cast<float *>(row1 + 128 + c1 * 4) = b1.y;
        }
    }
}

// One 32-row x 32-chunk code tile (6 words of 16 B per lane) against the
// table.  Two tokens (type 0): one permute + one 8-byte LDS per code byte
// gives both tokens' entries.  One token (type 1): one permute + one 4-byte
// LDS per code byte, two lookups per packed add.  The lane's rotated column
// offset for step t (and, for type 1, the table half) is byte (t & 1) of
// aux2[t >> 1]; bytes 2..3 of aux2 are zero, so a single byte permute
// assembles the shared-memory address (code << 8) | offset.
template <int TYPE>
__device__ __forceinline__ uint64_t tile_lookups(const uint4 (&c)[6], const uint32_t (&aux2)[16],
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
                        const int t = h * 16 + q * 4 + b;
                        const uint32_t idx =
                            prmt(w, aux2[t >> 1], 0x7600u | (b << 4) | (4 + (t & 1)));
                        acc = fadd2(acc, *reinterpret_cast<const uint64_t *>(
                                             lut + s * kLutStageBytes + idx));
                    }
                } else {
#pragma unroll
                    for (int b = 0; b < 4; b += 2) {
                        const int t = h * 16 + q * 4 + b;  // even: t and t + 1 share aux2
                        const uint32_t i0 = prmt(w, aux2[t >> 1], 0x7604u | (b << 4));
                        const uint32_t i1 = prmt(w, aux2[t >> 1], 0x7605u | ((b + 1) << 4));
                        const float v0 = *reinterpret_cast<const float *>(lut + s * kLutStageBytes + i0);
                        const float v1 = *reinterpret_cast<const float *>(lut + s * kLutStageBytes + i1);
                        acc = fadd2(acc, pk2(v0, v1));
                    }
                }
            }
    return acc;
}

// ------------------------------------------------------------ persistent GEMV
// A phase = (matrix, item, step).  The block's work index w runs over
// matrix-major (item * S + split), so the items of both matrices of a
// gate/up launch share one set of persistent blocks.  valid: 1 usable,
// -1 skipped item (error flagged by the plan), 0 past the end.
struct Phase {
    ItemDesc d;
    int w, step, valid, m, wl;  // wl = item * S + split within matrix m
};

// What one warp needs to stream a phase, derived once per phase so that a
// tile costs one pointer increment.
struct WarpPlan {
    const uint8_t *tile;  // this warp's first code tile (lane offset included)
    int tstride;          // bytes between this warp's consecutive tiles
    int nt;               // tiles of this warp in the phase
};

__device__ __forceinline__ Phase load_phase(const LutJob &job, int w, int step) {
    Phase P;
    P.w = w;
    P.step = step;
    P.valid = 0;
    const int per_m = lut_items(job);
    P.m = w / per_m;
    P.wl = w - P.m * per_m;
    P.d.expert = 0;
    P.d.entryA = P.d.entryB = 0;
    P.d.g0 = 0;
    P.d.type = 0;
    P.d.pad = 0;
    if (P.m >= job.n_mat) return P;
    const int4 raw = __ldg(reinterpret_cast<const int4 *>(job.desc) + P.wl / job.S);
    *reinterpret_cast<int4 *>(&P.d) = raw;
    P.valid = P.d.expert < 0 ? -1 : 1;
    return P;
}

__device__ __forceinline__ int ph_gA(const Phase &P) {
    return P.d.g0 + P.step * (P.d.type == 0 ? 1 : 2);
}
__device__ __forceinline__ const uint8_t *ph_record(const LutJob &job, const Phase &P) {
    return job.base + (uint64_t)P.d.expert * job.record_bytes;
}
__device__ __forceinline__ const uint8_t *ph_cb(const LutJob &job, const Phase &P) {
    return job.record_bytes ? ph_record(job, P) + job.cb_off[P.m]
                            : reinterpret_cast<const uint8_t *>(job.cb_ptr);
}

__device__ __forceinline__ WarpPlan warp_plan(const LutJob &job, const Phase &P, int lane,
                                              int warp) {
    WarpPlan W;
    const int RB = job.rows / 32;
    const int nrb = RB / job.S;
    const int rb0 = (P.wl % job.S) * nrb;
    const uint8_t *codes =
        job.record_bytes ? ph_record(job, P) + job.codes_off[P.m] : job.codes_ptr;
    if (P.d.type == 0) {  // tile q = warp + NW i -> row block q
        W.tile = codes + ((size_t)ph_gA(P) * RB + rb0 + warp) * kTileBytes + lane * 16;
        W.tstride = NW * kTileBytes;
        W.nt = (nrb - warp + NW - 1) / NW;
    } else {              // tile q -> row block q >> 1, chunk group gA + (q & 1)
        const int u = warp & 1;
        W.tile = codes + ((size_t)(ph_gA(P) + u) * RB + rb0 + (warp >> 1)) * kTileBytes + lane * 16;
        W.tstride = (NW / 2) * kTileBytes;
        W.nt = (2 * nrb - warp + NW - 1) / NW;
    }
    return W;
}

// cp.async of one step's inputs: 2 units x 32 chunks x 8 values.
__device__ __forceinline__ void issue_x(const LutJob &job, const Phase &P, uint8_t *xs_s) {
    const int esz = job.x_dtype == RVQ_BF16 ? 2 : 4;
    const int per_unit = 32 * 8 * esz / 16;  // 16-byte pieces per unit
    const int tid = threadIdx.x;
    if (tid < 2 * per_unit) {
        const int u = tid / per_unit, q = tid % per_unit;
        const int entry = u ? P.d.entryB : P.d.entryA;
        const int g = ph_gA(P) + (u ? P.d.type : 0);
        const uint8_t *src = reinterpret_cast<const uint8_t *>(job.x) +
                             ((int64_t)(entry / job.x_div) * job.x_stride + (int64_t)g * 256) * esz +
                             q * 16;
        cp_async16(xs_s + u * 32 * 8 * esz + q * 16, src);
    }
}

__device__ __forceinline__ void issue_cb(const uint8_t *cb, uint8_t *cb_s) {
#pragma unroll
    for (int q = 0; q < kCbBytes / 16 / NT; ++q) {
        const int o = (threadIdx.x + NT * q) * 16;
        cp_async16(cb_s + o, cb + o);
    }
}

__device__ __forceinline__ void load_tile(uint4 (&b)[6], const uint8_t *p) {
#pragma unroll
    for (int q = 0; q < 6; ++q) b[q] = ldg_stream(p + q * 512);
}

__device__ __forceinline__ void load_first(const WarpPlan &W, uint4 (&buf)[2][6]) {
    if (W.nt > 0) load_tile(buf[0], W.tile);
    if (W.nt > 1) load_tile(buf[1], W.tile + W.tstride);
}

// Stream one phase's tiles (type TYPE) through the 2-deep ring.  Once the
// phase's own tiles are all requested, the freed ring slots take the first
// tiles of the next phase (plan Wn; nt_next = 0 disables that).
template <int TYPE>
__device__ __forceinline__ void stream_phase(const LutJob &job, const Phase &P,
                                             const WarpPlan &W, const WarpPlan &Wn, int nt_next,
                                             uint4 (&buf)[2][6], const uint8_t *lut, float *sacc,
                                             int lane, int warp) {
    const int u = TYPE == 0 ? 0 : (warp & 1);
    const int C = job.C, j = P.step;
    const int nslot = job.G / C;
    const int nrb = job.rows / 32 / job.S;
    const int rows_split = nrb * 32;
    const int row0 = (P.wl % job.S) * rows_split;
    const int slotA = P.d.g0 / C;
    // partial rows: row = row0 + rbl * 32 + lane, rbl = this tile's row block in the split
    const int rbl0 = TYPE == 0 ? warp : (warp >> 1);
    const int rbl_step = TYPE == 0 ? NW : NW / 2;
    float *part = job.part[P.m];
    float *pA, *pB;
    if (TYPE == 0) {
        pA = part + ((size_t)P.d.entryA * nslot + slotA) * job.rows + row0 + lane;
        pB = part + ((size_t)P.d.entryB * nslot + slotA) * job.rows + row0 + lane;
    } else {
        const int e = u ? P.d.entryB : P.d.entryA;
        pA = part + ((size_t)e * nslot + slotA + u) * job.rows + row0 + lane;
        pB = pA;
    }
    uint32_t aux2[16];
#pragma unroll
    for (int p = 0; p < 16; ++p) {
        const uint32_t c0 = TYPE == 0 ? (((lane + 2 * p) & 31) << 3)
                                      : ((((lane + 2 * p) & 31) << 2) | (u << 7));
        const uint32_t c1 = TYPE == 0 ? (((lane + 2 * p + 1) & 31) << 3)
                                      : ((((lane + 2 * p + 1) & 31) << 2) | (u << 7));
        aux2[p] = c0 | (c1 << 8);
    }
    const uint8_t *next = W.tile + 2 * W.tstride;  // tile i + 2 of this phase
    const uint8_t *next_n = Wn.tile;               // then tiles of the next phase
    int left_n = nt_next;
    for (int i0 = 0; i0 < W.nt; i0 += 2) {
#pragma unroll
        for (int dd = 0; dd < 2; ++dd) {
            const int i = i0 + dd;
            if (i < W.nt) {
                const uint64_t acc = tile_lookups<TYPE>(buf[dd], aux2, lut);
                if (i + 2 < W.nt) {
                    load_tile(buf[dd], next);
                    next += W.tstride;
                } else if (left_n > 0) {
                    load_tile(buf[dd], next_n);
                    next_n += Wn.tstride;
                    --left_n;
                }
                const int rl = (rbl0 + i * rbl_step) * 32 + lane;  // row within the split
                float2 a = upk2(acc);
                if constexpr (TYPE == 1) {
                    float v = a.x + a.y;
                    if (C > 1) {
                        if (j > 0) v += sacc[u * rows_split + rl];
                        if (j < C - 1) sacc[u * rows_split + rl] = v;
                    }
                    if (j == C - 1) pA[rl - lane] = v;
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
                        pA[rl - lane] = a.x;
                        pB[rl - lane] = a.y;
                    }
                }
            }
        }
    }
}

__global__ void __launch_bounds__(NT, 1) lut_gemv_kernel(const LutJob job) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t *lut = smem;
    uint8_t *cb_s = smem + kLutBytes;
    uint8_t *xs_s = cb_s + kCbBytes;
    float *sacc = reinterpret_cast<float *>(xs_s + kXsBytes);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");

    Phase P = load_phase(job, blockIdx.x, 0);
    uint4 buf[2][6];
    const uint8_t *cb_loaded = nullptr;
    if (P.valid > 0) {
        // codebook and inputs first (the build waits for them), then tiles
        cb_loaded = ph_cb(job, P);
        issue_cb(cb_loaded, cb_s);
        issue_x(job, P, xs_s);
        cp_async_commit();
        load_first(warp_plan(job, P, lane, warp), buf);
    } else {
        cp_async_commit();
    }

    while (P.valid != 0) {
        // the phase after this one: the next step of this item, or this
        // block's next item (descriptor read now, used after the build)
        const Phase N = P.step + 1 < job.C ? load_phase(job, P.w, P.step + 1)
                                           : load_phase(job, P.w + gridDim.x, 0);
        cp_async_wait_all();
        __syncthreads();  // codebook + inputs landed; previous lookups done
        if (P.valid > 0) build_table(lut, cb_s, xs_s, job.x_dtype, P.d.type, lane, warp);
        __syncthreads();
        if (N.valid > 0) {
            issue_x(job, N, xs_s);
            const uint8_t *ncb = ph_cb(job, N);
            if (ncb != cb_loaded) {
                issue_cb(ncb, cb_s);
                cb_loaded = ncb;
            }
        }
        cp_async_commit();
        WarpPlan Wn;
        Wn.tile = nullptr;
        Wn.tstride = 0;
        Wn.nt = 0;
        if (N.valid > 0) Wn = warp_plan(job, N, lane, warp);
        if (P.valid > 0) {
            const WarpPlan W = warp_plan(job, P, lane, warp);
            // tile i of the next phase must land in ring slot i % 2: the
            // hand-over works when this warp's tile count is even
            const int nt_next = (W.nt > 0 && (W.nt % 2) == 0) ? min(Wn.nt, 2) : 0;
            if (P.d.type == 0)
                stream_phase<0>(job, P, W, Wn, nt_next, buf, lut, sacc, lane, warp);
            else
                stream_phase<1>(job, P, W, Wn, nt_next, buf, lut, sacc, lane, warp);
            if (nt_next == 0) load_first(Wn, buf);
        } else {
            load_first(Wn, buf);
        }
        P = N;
    }
    cp_async_wait_all();
}

// ------------------------------------------- interleaved build-and-stream GEMV
// For one token per expert (decode) the table build of the next unit is
// interleaved with the streaming of the current one inside each block: the
// shared table holds two halves (column block h of the one-token layout
// T[s][k][h][c], the type-1 layout), every warp streams code tiles against
// the current half and, after its last tile of a phase, builds its share of
// the next table into the other half.  A block barrier per table swaps them.
// A unit is (matrix, token-expert pair, 32-chunk group, 512-row slice): one
// 32-row tile per warp.  A table serves all units of one (matrix, pair,
// group) in the block's contiguous unit range.  The next table's inputs (its
// 256 input values and, when the expert or matrix changes, its codebook) are
// fetched by one bulk copy onto an mbarrier while the warps stream.  In the
// down launch the 256 values are h = silu(g) u of the gate/up launch: every
// warp reduces a share of them from the split-K partials at the start of the
// phase (il_swiglu_x) and arrives on the same mbarrier, so no separate SwiGLU
// launch (and its two kernel boundaries) sits between the two GEMVs.
constexpr int IL_ROWS = 512;                   // rows per unit = 16 warps x 32
constexpr int IL_XS = 32 * 8 * 4;              // one table's inputs, fp32 or bf16
constexpr int kIlSmemBytes = kLutBytes + kCbBytes + IL_XS + 64;
constexpr unsigned long long kIlWaitNs = 1000000000ull;  // bounded waits: 1 s

__device__ __forceinline__ unsigned long long il_now() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Per sorted pair position p: {expert or -1 (skip), entry, 0, 0}.
__global__ void __launch_bounds__(256) plan_pairs_kernel(const LutJob job, int4 *pd) {
    __shared__ int32_t soff[257];
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    const int E = job.E;
    for (int x = threadIdx.x; x <= E; x += blockDim.x) soff[x] = job.offsets[x];
    __syncthreads();
    const int p = blockIdx.x * blockDim.x + threadIdx.x;
    if (p >= job.n_pairs) return;
    int4 d = make_int4(-1, 0, 0, 0);
    if (soff[0] != 0 || soff[E] != job.n_pairs) {
        set_dev_error(job.status, RVQ_DEV_ERR_INDEX);
        pd[p] = d;
        return;
    }
    int lo = 0, hi = E;  // largest e with offsets[e] <= p
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (soff[mid] <= p) lo = mid; else hi = mid;
    }
    const int e = lo, ne = soff[e + 1] - soff[e];
    const int entry = job.pairs[p];
    // {record index (an expert cache's slot), entry}: the walkers address the
    // record by it
    if (!(soff[e] <= p && p < soff[e + 1]))
        set_dev_error(job.status, RVQ_DEV_ERR_INDEX);
    else
        d = pair_desc(job, e, ne, entry);
    pd[p] = d;
}

__device__ __forceinline__ bool il_try(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        "selp.b32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity), "r"(20000u)
        : "memory");
    return done != 0;
}

// Bounded phase wait; false after the limit (the thread then records the
// timeout).
__device__ __forceinline__ bool il_wait(uint32_t bar, uint32_t parity, uint32_t *status) {
    if (il_try(bar, parity)) return true;
    const unsigned long long t0 = il_now();
    for (;;) {
        if (il_try(bar, parity)) return true;
        if (il_now() - t0 > kIlWaitNs) {
            set_dev_error(status, RVQ_DEV_ERR_TIMEOUT);
            return false;
        }
    }
}

// One table: (matrix, pair position, chunk group), first row slice and the
// number of consecutive row-slice units of the block's range it serves.
struct IlTab {
    int m, p, g, r0, nr;
    int2 d;  // {expert, entry}
};

// Walk over the block's unit range [w, w1): units (m, p, g, r) in that order
// with S row slices; positions whose pair descriptor says skip are passed
// over whole.  Fills the next table and advances past it.
struct IlWalk {
    int w, m, p, g, r;
    int pc;   // pair position whose descriptor is cached in dc
    int2 dc;
};
__device__ __forceinline__ IlWalk il_start(const LutJob &job, int S, int w) {
    const int per_m = job.n_pairs * job.G * S, gs = job.G * S;
    IlWalk k;
    k.w = w;
    k.pc = -1;
    k.dc = make_int2(-1, 0);
    k.m = w / per_m;
    int rem = w - k.m * per_m;
    k.p = rem / gs;
    rem -= k.p * gs;
    k.g = rem / S;
    k.r = rem - k.g * S;
    return k;
}
__device__ __forceinline__ bool il_next(const LutJob &job, int S, int w1, const int4 *pd,
                                        IlWalk &k, IlTab &t) {
    for (;;) {
        if (k.w >= w1) return false;
        if (k.p != k.pc) {
            const int4 v = __ldg(pd + k.p);
            k.dc = make_int2(v.x, v.y);
            k.pc = k.p;
        }
        const int2 d = k.dc;
        if (d.x >= 0) {
            t.m = k.m;
            t.p = k.p;
            t.g = k.g;
            t.r0 = k.r;
            t.nr = min(S - k.r, w1 - k.w);
            t.d = d;
            k.w += t.nr;
            k.r = 0;
            if (++k.g == job.G) {
                k.g = 0;
                if (++k.p == job.n_pairs) {
                    k.p = 0;
                    ++k.m;
                }
            }
            return true;
        }
        k.w += (job.G - k.g) * S - k.r;  // rest of this pair position
        k.g = 0;
        k.r = 0;
        if (++k.p == job.n_pairs) {
            k.p = 0;
            ++k.m;
        }
    }
}

// This warp's share of one table (16 warps x 6 iterations of four entry
// pairs).  Quarter q of the warp takes entry pair 4 it + q (a 64-byte
// codeword pair, broadcast to its 8 lanes); lane r of the quarter computes
// columns r, r + 8, r + 16, r + 24 for both entries.  Stores rotate the
// column order by the quarter, so every 4-byte store instruction writes 32
// distinct banks.
__device__ __forceinline__ void il_build(uint8_t *lut, int h, const uint8_t *cb_s,
                                         const uint8_t *xs_s, int xdt, int warp, int lane) {
    const int q = lane >> 3, r = lane & 7;
    // slot jj of this lane holds column r + 8 ((jj + q) mod 4): the quarters
    // rotate their column blocks, so each store instruction writes 32 banks
    float x[4][8];
    int coff[4];
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
        const int c = r + 8 * ((jj + q) & 3);
        coff[jj] = c * 4;
        float(&xj)[8] = x[jj];
        if (xdt == RVQ_BF16) {
            const uint4 v = *reinterpret_cast<const uint4 *>(xs_s + c * 16);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                xj[2 * i] = __uint_as_float(w[i] << 16);
                xj[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
            }
        } else {
            const float4 a = *reinterpret_cast<const float4 *>(xs_s + c * 32);
            const float4 b = *reinterpret_cast<const float4 *>(xs_s + c * 32 + 16);
            xj[0] = a.x; xj[1] = a.y; xj[2] = a.z; xj[3] = a.w;
            xj[4] = b.x; xj[5] = b.y; xj[6] = b.z; xj[7] = b.w;
        }
    }
    const float4 *cb4 = reinterpret_cast<const float4 *>(cb_s);
#pragma unroll 1
    for (int it = warp; it < 96; it += NW) {
        const int kp = 4 * it + q;  // entry pair over the three stages
        const int s = kp >> 7, k = (kp & 127) * 2;
        // pair layout: (C_k[i], C_k+1[i]) for i = 0..7
        const float4 c0 = cb4[kp * 4 + 0], c1 = cb4[kp * 4 + 1];
        const float4 c2 = cb4[kp * 4 + 2], c3 = cb4[kp * 4 + 3];
        const float ca[8] = {c0.x, c0.z, c1.x, c1.z, c2.x, c2.z, c3.x, c3.z};
        const float cbv[8] = {c0.y, c0.w, c1.y, c1.w, c2.y, c2.w, c3.y, c3.w};
        float ta[4], tb[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            ta[j] = 0.f;
            tb[j] = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                ta[j] = fmaf(x[j][i], ca[i], ta[j]);
                tb[j] = fmaf(x[j][i], cbv[i], tb[j]);
            }
        }
        uint8_t *row0 = lut + s * kLutStageBytes + k * 256 + h * 128;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            *reinterpret_cast<float *>(row0 + coff[jj]) = ta[jj];
            *reinterpret_cast<float *>(row0 + 256 + coff[jj]) = tb[jj];
        }
    }
}

// One thread fetches a table's inputs onto the mbarrier: the pair's 256
// input values of chunk group g and, unless `same_cb`, the codebook.  The
// two halves can be issued apart (the codebook first, the inputs once the
// kernel that writes them has completed): il_fetch_cb announces both.
__device__ __forceinline__ void il_fetch_cb(const LutJob &job, const IlTab &t, bool same_cb,
                                            uint8_t *cb_s, uint32_t bar) {
    const int esz = job.x_dtype == RVQ_BF16 ? 2 : 4;
    // (with the SwiGLU reduction fused, the inputs are written by the block)
    const uint32_t bytes =
        (job.sw_g ? 0u : 256u * esz) + (same_cb ? 0u : (uint32_t)kCbBytes);
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
    if (!same_cb) {
        const uint8_t *cb = job.base + (uint64_t)t.d.x * job.record_bytes + job.cb_off[t.m];
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                (uint32_t)__cvta_generic_to_shared(cb_s)),
            "l"(cb), "r"((uint32_t)kCbBytes), "r"(bar)
            : "memory");
    }
}
__device__ __forceinline__ void il_fetch_x(const LutJob &job, const IlTab &t, uint8_t *xs_s,
                                           uint32_t bar) {
    const int esz = job.x_dtype == RVQ_BF16 ? 2 : 4;
    const uint8_t *xsrc = reinterpret_cast<const uint8_t *>(job.x) +
                          ((int64_t)(t.d.y / job.x_div) * job.x_stride + (int64_t)t.g * 256) * esz;
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            (uint32_t)__cvta_generic_to_shared(xs_s)),
        "l"(xsrc), "r"((uint32_t)(256 * esz)), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void il_fetch(const LutJob &job, const IlTab &t, bool same_cb,
                                         uint8_t *cb_s, uint8_t *xs_s, uint32_t bar) {
    il_fetch_cb(job, t, same_cb, cb_s, bar);
    if (!job.sw_g) il_fetch_x(job, t, xs_s, bar);
}

// Down launch with the SwiGLU reduction fused: table t's 256 inputs
// h[r] = silu(g[r]) u[r] for rows r = 256 g .. 256 g + 255 of pair entry
// t.d.y, g and u summed over the gate/up launch's split-K slots (at most 32):
// eight adjacent lanes per four rows, lane j taking slots j, j + 8, ... (all
// its loads in flight at once), then three xor-shuffles, a fixed order.
// Called by all 512 threads; each warp then arrives on `bar`.
__device__ __forceinline__ void il_swiglu_x(const LutJob &job, const IlTab &t, uint8_t *xs_s,
                                            int tid, uint32_t bar) {
    const int j = tid & 7, i4 = tid >> 3;  // slot residue, float4 of rows
    const int f4 = job.cols / 4, nslot = job.sw_nslot;
    const int64_t off = (int64_t)t.d.y * nslot * f4 + t.g * 64 + i4;
    const float4 *gp = reinterpret_cast<const float4 *>(job.sw_g) + off;
    const float4 *up = reinterpret_cast<const float4 *>(job.sw_u) + off;
    static_assert(kIlSwigluMaxSlots <= 4 * 8, "four slots per lane of eight");
    float4 a[4], b[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int s = j + 8 * q;
        a[q] = s < nslot ? __ldg(gp + (int64_t)s * f4) : make_float4(0.f, 0.f, 0.f, 0.f);
        b[q] = s < nslot ? __ldg(up + (int64_t)s * f4) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float4 g = a[0], u = b[0];
#pragma unroll
    for (int q = 1; q < 4; ++q) {
        g.x += a[q].x; g.y += a[q].y; g.z += a[q].z; g.w += a[q].w;
        u.x += b[q].x; u.y += b[q].y; u.z += b[q].z; u.w += b[q].w;
    }
#pragma unroll
    for (int o = 1; o <= 4; o <<= 1) {
        g.x += __shfl_xor_sync(0xffffffffu, g.x, o);
        g.y += __shfl_xor_sync(0xffffffffu, g.y, o);
        g.z += __shfl_xor_sync(0xffffffffu, g.z, o);
        g.w += __shfl_xor_sync(0xffffffffu, g.w, o);
        u.x += __shfl_xor_sync(0xffffffffu, u.x, o);
        u.y += __shfl_xor_sync(0xffffffffu, u.y, o);
        u.z += __shfl_xor_sync(0xffffffffu, u.z, o);
        u.w += __shfl_xor_sync(0xffffffffu, u.w, o);
    }
    if (j == 0) {
        float4 o;
        o.x = g.x / (1.0f + expf(-g.x)) * u.x;
        o.y = g.y / (1.0f + expf(-g.y)) * u.y;
        o.z = g.z / (1.0f + expf(-g.z)) * u.z;
        o.w = g.w / (1.0f + expf(-g.w)) * u.w;
        reinterpret_cast<float4 *>(xs_s)[i4] = o;
    }
    __syncwarp();
    if ((tid & 31) == 0)
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__global__ void __launch_bounds__(NT, 1) lut_gemv_il_kernel(const LutJob job, const int4 *pd) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t *lut = smem;
    uint8_t *cb_s = smem + kLutBytes;
    uint8_t *xs_s = cb_s + kCbBytes;
    const uint32_t inbar = (uint32_t)__cvta_generic_to_shared(xs_s + IL_XS);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int S = job.rows / IL_ROWS;
    const int U = job.n_mat * job.n_pairs * job.G * S;
    const int w0 = (int)((int64_t)blockIdx.x * U / gridDim.x);
    const int w1 = (int)((int64_t)(blockIdx.x + 1) * U / gridDim.x);
    const int RB = job.rows / 32;
    const int nslot = job.G;
    // arrivals per table: the fetching thread, and with the SwiGLU reduction
    // fused every warp (each computes a share of the inputs)
    const bool fused = job.sw_g != nullptr;
    if (threadIdx.x == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(inbar), "r"(fused ? 1u + NW : 1u));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // The table walk reads the pair plan; with early_start it was written
    // by an earlier kernel that the preceding one waited for before it let
    // this launch start, so the walk, the first code tiles and the first
    // codebook need not wait for the preceding kernel (which writes only this
    // launch's inputs: x, or the gate/up partials of a fused SwiGLU).
    const bool early = job.early_start != 0;
    if (!early) {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        asm volatile("griddepcontrol.launch_dependents;");
    }

    // table walk (identical in every thread) and this warp's tile walk
    IlWalk tw = il_start(job, S, w0), gw = tw;
    IlTab cur, nxt;
    bool has_cur = il_next(job, S, w1, pd, tw, cur);
    bool has_nxt = has_cur && il_next(job, S, w1, pd, tw, nxt);
    int gi = 0, gn = 0;  // tile walk: index within table gt, its unit count
    // this warp's next tile and output of table gt: set when the walk enters
    // a table, then advanced by one unit (IL_ROWS rows) per tile
    const uint8_t *gtile = nullptr;
    float *gout = nullptr;
    auto gen = [&](const uint8_t *&tile, float *&out) -> bool {
        if (gi == gn) {
            IlTab gt;
            if (!il_next(job, S, w1, pd, gw, gt)) return false;
            gi = 0;
            gn = gt.nr;
            const int rb = gt.r0 * (IL_ROWS / 32) + warp;
            const uint8_t *rec = job.base + (uint64_t)gt.d.x * job.record_bytes;
            gtile = rec + job.codes_off[gt.m] + ((size_t)gt.g * RB + rb) * kTileBytes + lane * 16;
            gout = job.part[gt.m] + ((size_t)gt.d.y * nslot + gt.g) * job.rows + rb * 32 + lane;
        }
        ++gi;
        tile = gtile;
        out = gout;
        gtile += (IL_ROWS / 32) * kTileBytes;
        gout += IL_ROWS;
        return true;
    };
    uint4 buf[2][6];
    float *outp[2] = {nullptr, nullptr};
    bool have[2] = {false, false};
#pragma unroll
    for (int dd = 0; dd < 2; ++dd) {
        const uint8_t *t;
        if (gen(t, outp[dd])) {
            load_tile(buf[dd], t);
            have[dd] = true;
        }
    }

    uint32_t inph = 0;  // phase of the input barrier
    bool alive = true;  // false after a timed-out wait: no more reads, barriers still met
    int cb_m = -1, cb_e = -1;
    if (has_cur && threadIdx.x == 0) {
        // the first table's codebook and code tiles (bank data)
        il_fetch_cb(job, cur, false, cb_s, inbar);
        const uint8_t *t0 = job.base + (uint64_t)cur.d.x * job.record_bytes +
                            job.codes_off[cur.m] +
                            ((size_t)cur.g * RB + cur.r0 * (IL_ROWS / 32)) * kTileBytes;
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(t0),
                     "r"((uint32_t)(cur.nr * (IL_ROWS / 32) * kTileBytes))
                     : "memory");
    }
    if (early) {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        asm volatile("griddepcontrol.launch_dependents;");
    }
    if (has_cur) {
        // the first table: its inputs, then built by all warps before streaming
        if (fused) {
            il_swiglu_x(job, cur, xs_s, threadIdx.x, inbar);
        } else if (threadIdx.x == 0) {
            il_fetch_x(job, cur, xs_s, inbar);
        }
        cb_m = cur.m;
        cb_e = cur.d.x;
        alive = il_wait(inbar, inph, job.status);
        ++inph;
        if (alive) il_build(lut, 0, cb_s, xs_s, job.x_dtype, warp, lane);
    }
    __syncthreads();

    uint32_t aux2[16];
    int sp = 0;  // ring slot holding this warp's next tile
    for (int b = 0; has_cur; ++b) {
        const int h = b & 1;
        if (has_nxt && threadIdx.x == 0) {
            const bool same = nxt.m == cb_m && nxt.d.x == cb_e;
            il_fetch(job, nxt, same, cb_s, xs_s, inbar);
            // the next table's code tiles (its units are adjacent row slices,
            // one contiguous range) into L2 while this table streams
            const uint8_t *t0 = job.base + (uint64_t)nxt.d.x * job.record_bytes +
                                job.codes_off[nxt.m] +
                                ((size_t)nxt.g * RB + nxt.r0 * (IL_ROWS / 32)) * kTileBytes;
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(t0),
                         "r"((uint32_t)(nxt.nr * (IL_ROWS / 32) * kTileBytes))
                         : "memory");
        }
        if (has_nxt) {
            cb_m = nxt.m;
            cb_e = nxt.d.x;
            // the previous table's build is done with the inputs' buffer
            if (fused) il_swiglu_x(job, nxt, xs_s, threadIdx.x, inbar);
        }
#pragma unroll
        for (int p2 = 0; p2 < 16; ++p2) {
            const uint32_t c0 = (((lane + 2 * p2) & 31) << 2) | ((uint32_t)h << 7);
            const uint32_t c1 = (((lane + 2 * p2 + 1) & 31) << 2) | ((uint32_t)h << 7);
            aux2[p2] = c0 | (c1 << 8);
        }
        // this warp's tiles of the current table (one per unit); the ring
        // slots alternate along the warp's whole tile sequence
        auto step = [&](auto slot, int i) {
            constexpr int dd = decltype(slot)::value;
            if (!have[dd]) return;
            if (alive) *outp[dd] = tile_lookups1_ilp(buf[dd], aux2, lut);
            if (i == cur.nr - 1 && has_nxt) {
                // build this warp's share of the next table into the other
                // half after its last tile of this one (the inputs were
                // fetched at phase start, so the fetch hides behind the tiles)
                if (alive) alive = il_wait(inbar, inph, job.status);
                if (alive) il_build(lut, h ^ 1, cb_s, xs_s, job.x_dtype, warp, lane);
            }
            const uint8_t *t;
            have[dd] = gen(t, outp[dd]);
            if (have[dd]) load_tile(buf[dd], t);
        };
        for (int i = 0; i < cur.nr; ++i) {
            if (sp == 0)
                step(std::integral_constant<int, 0>{}, i);
            else
                step(std::integral_constant<int, 1>{}, i);
            sp ^= 1;
        }
        if (has_nxt) ++inph;
        __syncthreads();  // the next table is complete; this half is free
        cur = nxt;
        has_cur = has_nxt;
        has_nxt = has_cur && il_next(job, S, w1, pd, tw, nxt);
    }
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

rvq_status launch_lut_plan(const LutJob &ja, const LutJob *jb, cudaStream_t stream, bool pdl) {
    const int na = lut_items(ja) / ja.S;
    const int nb = jb ? lut_items(*jb) / jb->S : 0;
    if (na + nb == 0) return RVQ_OK;
    LutJob b = jb ? *jb : LutJob{};
    if (!jb) b.n_pairs = 0;
    RVQ_CUDA(launch_ex(plan_kernel, dim3((na + nb + 255) / 256), dim3(256), 0, stream, pdl, ja, b));
    return RVQ_OK;
}

rvq_status launch_lut_gemv(const LutJob &job, cudaStream_t stream, bool pdl) {
    static std::atomic<int> attr_done[64];  // per device; setting twice is harmless
    int dev = 0;
    RVQ_CUDA(cudaGetDevice(&dev));
    if (dev < 64 && !attr_done[dev]) {
        RVQ_CUDA(cudaFuncSetAttribute(lut_gemv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      kSmemBytes));
        attr_done[dev] = 1;
    }
    if (job.rows / job.S > kMaxSplitRows || (job.C > 1 && job.rows / job.S > kMaxAccRows) ||
        (job.rows / 32) % job.S != 0 || job.G % (2 * job.C) != 0 || !job.desc) {
        set_error("lut_gemv: bad split (rows %d, S %d, G %d, C %d)", job.rows, job.S, job.G,
                  job.C);
        return RVQ_EINVAL;
    }
    const int work = lut_items(job) * job.n_mat;
    if (work == 0) return RVQ_OK;
    const int grid = work < num_sms() ? work : num_sms();
    RVQ_CUDA(launch_ex(lut_gemv_kernel, dim3(grid), dim3(NT), (size_t)kSmemBytes, stream, pdl,
                       job));
    return RVQ_OK;
}

rvq_status launch_lut_plan_pairs(const LutJob &job, int4 *pd, cudaStream_t stream, bool pdl) {
    if (job.n_pairs == 0) return RVQ_OK;
    if (!job.offsets || !job.pairs || !job.base || job.E > 256) {
        set_error("lut_plan_pairs: needs a bank, offsets and pairs (E %d)", job.E);
        return RVQ_EINVAL;
    }
    RVQ_CUDA(launch_ex(plan_pairs_kernel, dim3((job.n_pairs + 255) / 256), dim3(256), 0, stream,
                       pdl, job, pd));
    return RVQ_OK;
}

rvq_status launch_lut_gemv_il(const LutJob &job, const int4 *pd, cudaStream_t stream, bool pdl) {
    static std::atomic<int> attr_done[64];  // per device; setting twice is harmless
    int dev = 0;
    RVQ_CUDA(cudaGetDevice(&dev));
    if (dev < 64 && !attr_done[dev]) {
        RVQ_CUDA(cudaFuncSetAttribute(lut_gemv_il_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, kIlSmemBytes));
        attr_done[dev] = 1;
    }
    if (job.rows % IL_ROWS || job.cols % 256 || job.G != job.cols / 256 || !job.base || !pd) {
        set_error("lut_gemv_il: rows %d / cols %d not supported", job.rows, job.cols);
        return RVQ_EINVAL;
    }
    const int64_t units = (int64_t)job.n_mat * job.n_pairs * job.G * (job.rows / IL_ROWS);
    if (units == 0) return RVQ_OK;
    const int grid = units < num_sms() ? (int)units : num_sms();
    RVQ_CUDA(launch_ex(lut_gemv_il_kernel, dim3(grid), dim3(NT), (size_t)kIlSmemBytes, stream, pdl,
                       job, pd));
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
