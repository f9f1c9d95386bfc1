// Decode lookup-table GEMV with the tables built on the tensor cores.
//
// Method: for an input vector x and chunk j (8 input columns) the table
// T_s[j][k] = <x[8j..8j+7], C_s[k]> holds the partial dot product of every
// codeword k of stage s; an output row is sum_j sum_s T_s[j][code(r,j,s)],
// three table reads per chunk and row, and the weight matrix is never formed
// ["Running a 2.78-Trillion-Parameter Model on a Laptop: Inside WASTE's
// NVMe-Streaming Engine", section "Technical Insight"; "WASTE Inference
// Engine: Running Kimi K3 2.78T on Consumer Hardware", section "Residual
// Vector Quantization (RVQ)"].
//
// GB300 design.
//  * Work: a unit is (matrix, token-expert pair, 32-chunk group, 512-row
//    slice); a table (3 stages x 256 entries x 32 chunk columns, 96 KiB of
//    fp32) serves every unit of its (matrix, pair, group) in the block's
//    range.  Persistent blocks, one per SM, take contiguous unit ranges, cut
//    on table boundaries when there are at least as many tables as blocks.
//  * A table is the product C X^T of the 768 x 8 codebook (all three stages)
//    and the group's 32 x 8 inputs, computed by tcgen05.mma (kind::f16, fp32
//    accumulators in TMEM): M = 128 codewords per MMA (6 M tiles), N = 32
//    chunk columns, K = 48.  The fp32 codebook is split exactly into three
//    bf16 terms C = C1 + C2 + C3 and the inputs into x = x1 + x2 + x3 (x2 = x3
//    = 0 for bf16 inputs); K holds x1C1 + x1C2 + x1C3 + x2C1 + x2C2 + x3C1.
//    Every bf16 x bf16 product is exact in fp32 and the sums are fp32, so the
//    table matches the fp32 dot products to rounding (the two terms left out,
//    x2C3 and x3C2, are below 2^-24 of the product).  A (the codebook terms)
//    lives in TMEM and is rewritten only when the expert or matrix changes;
//    B (the input terms) is 4 KiB of shared memory per table.
//  * Warp roles (640 threads): warps 0-3 build (warp w owns TMEM lane
//    quarter w): codebook -> A, inputs -> B, MMAs (warp 0 lane 0, which also
//    issues the bulk copies and L2 prefetches), then each thread moves its
//    codeword rows of D out of TMEM into the table half.  A codeword row is
//    32 consecutive fp32 columns, while the lookups need column c in bank c;
//    each lane rotates its eight 16-byte chunks by lane % 8 before storing,
//    so every quarter-warp store covers all 32 banks.  Warps 4-19 stream the
//    code tiles (a 2-deep register ring per warp) and look them up.
//  * Two table halves interleaved in one 192 KiB array (T[s][k][h][c]); a
//    pair of mbarriers per half hands a table from the builders (full, 4
//    arrivals) to the lookup warps and back (empty, 16 arrivals), so the
//    next table is built while the current one is read; no block-wide
//    barrier in the main loop.
//  * Lookups: lane l owns row 32b + l of a 32-row x 32-chunk code tile; the
//    packed layout rotates each row's chunk order by l, so the 32 lanes read
//    32 different table columns (banks) at every step for any code values.
//  * Every wait is bounded (1 s); on expiry the block records
//    RVQ_DEV_ERR_TIMEOUT, every role leaves its loop, outstanding copies and
//    MMAs are drained and TMEM is freed.
#include "internal.cuh"
#include "lut_common.cuh"
#include "tc_util.cuh"

namespace rvq {
namespace {

constexpr int TB_THREADS = 640;
constexpr int TB_BUILD_WARPS = 4;              // warps 0-3
constexpr int TB_LOOK_WARPS = 16;              // warps 4-19
constexpr int TB_ROWS = 512;                   // rows per unit (16 row blocks of 32)
constexpr int TB_RB = TB_ROWS / 32;
constexpr int TB_RING = 2;                     // code tiles in flight per lookup warp
constexpr int TB_CB = 24576;                   // packed fp32 codebook of one matrix
constexpr int TB_OFF_LUT = 0;                  // [s][k][h][c] fp32, 192 KiB
constexpr int TB_OFF_CB = kLutBytes;           // codebook staging (bulk copy)
constexpr int TB_OFF_B = TB_OFF_CB + TB_CB;    // MMA B: 32 rows x 128 B, 128-byte swizzle
constexpr int TB_OFF_XS = TB_OFF_B + 32 * 128; // one table's 256 inputs (<= 1 KiB)
constexpr int TB_OFF_BAR = TB_OFF_XS + 1024;
enum { BAR_FULL = 0, BAR_EMPTY = 2, BAR_MMA = 4, BAR_CB = 5, BAR_X = 6, BAR_DONE = 7,
       BAR_NEVER = 8, TB_NBAR = 9 };
constexpr int TB_OFF_TMEM = TB_OFF_BAR + 8 * TB_NBAR;
constexpr int TB_OFF_FLAG = TB_OFF_TMEM + 4;
constexpr int TB_SMEM = TB_OFF_FLAG + 4 + 1024;  // + slack to align the base to 1 KiB
static_assert(TB_OFF_B % 1024 == 0, "the swizzled B operand starts on 1 KiB");
static_assert(TB_SMEM <= 232448, "shared memory per CTA");
constexpr uint32_t TB_TMEM_COLS = 512;
constexpr uint32_t TB_TMEM_D = 0;              // D: M tile i at columns 32 i (6 x 32)
constexpr uint32_t TB_TMEM_A = 256;            // A: M tile i at columns 256 + 24 i (6 x 24)
static_assert(TB_TMEM_A + 6 * 24 <= TB_TMEM_COLS && 6 * 32 <= TB_TMEM_A, "TMEM columns");
// registers: every warp keeps the 96 the block is launched with (640 threads
// x 96 = 61,440; checked on the host before the first launch)
constexpr uint32_t TB_REG_BUILD = 96, TB_REG_LOOK = 96;
constexpr int TB_REG_LAUNCH = 96;
static_assert(TB_BUILD_WARPS * 32 * TB_REG_BUILD + TB_LOOK_WARPS * 32 * TB_REG_LOOK <=
                  TB_THREADS * TB_REG_LAUNCH,
              "register split");

// One table of the block's sequence.
struct TbTab {
    int m, p, g, r0, nr;  // matrix, pair position, chunk group, first row slice, slices
    int rec, entry;       // record index (cache slot), pair entry (input row = entry / x_div)
};

// Walk over the block's unit range [w, w1): units (m, p, g, r) in that order
// with S row slices; pair positions whose descriptor is -1 (the tensor-core
// path's, or unusable) are passed over whole.
struct TbWalk {
    int w, m, p, g, r;
    int pc;  // pair position whose descriptor is cached in dc
    int2 dc;
};

__device__ __forceinline__ TbWalk tb_start(const LutJob &job, int S, int w) {
    const int per_m = job.n_pairs * job.G * S, gs = job.G * S;
    TbWalk k;
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

__device__ __forceinline__ bool tb_next(const LutJob &job, int S, int w1, const int4 *pd,
                                        TbWalk &k, TbTab &t) {
    for (;;) {
        if (k.w >= w1) return false;
        if (k.p != k.pc) {
            if (pd) {
                const int4 v = __ldg(pd + k.p);
                k.dc = make_int2(v.x, v.y);
            } else {
                k.dc = make_int2(0, k.p);  // single matrix: pair p is input row p
            }
            k.pc = k.p;
        }
        if (k.dc.x >= 0) {
            t.m = k.m;
            t.p = k.p;
            t.g = k.g;
            t.r0 = k.r;
            t.nr = min(S - k.r, w1 - k.w);
            t.rec = k.dc.x;
            t.entry = k.dc.y;
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

__device__ __forceinline__ const uint8_t *tb_codes(const LutJob &job, const TbTab &t) {
    return job.base ? job.base + (uint64_t)t.rec * job.record_bytes + job.codes_off[t.m]
                    : job.codes_ptr;
}
__device__ __forceinline__ const uint8_t *tb_cb(const LutJob &job, const TbTab &t) {
    return job.base ? job.base + (uint64_t)t.rec * job.record_bytes + job.cb_off[t.m]
                    : reinterpret_cast<const uint8_t *>(job.cb_ptr);
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void prefetch_l2(const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
// Barrier of the builder warps (named barrier 1) that also ORs a flag over
// them, so every builder takes the same exit decision.
__device__ __forceinline__ bool builders_sync_any(bool v) {
    uint32_t r;
    asm volatile(
        "{\n.reg .pred pi, po;\nsetp.ne.u32 pi, %1, 0;\nbar.red.or.pred po, 1, %2, pi;\n"
        "selp.u32 %0, 1, 0, po;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)v), "n"(TB_BUILD_WARPS * 32)
        : "memory");
    return r != 0;
}
// A bounded wait whose result is the same in every lane of the warp (the
// warp-collective tcgen05 and shuffle steps after it need all lanes).
__device__ __forceinline__ bool warp_wait(uint32_t mbar, uint32_t parity, volatile int *abort_flag,
                                          uint32_t *status) {
    const bool ok = mbar_wait(mbar, parity, abort_flag, status);
    return __all_sync(0xffffffffu, ok);
}

// Issuer: one table's 256 inputs (chunk group g of its input row) into xs.
__device__ __forceinline__ void fetch_x(const LutJob &job, const TbTab &t, uint32_t xs,
                                        uint32_t bar) {
    const int esz = job.x_dtype == RVQ_BF16 ? 2 : 4;
    const uint8_t *src = reinterpret_cast<const uint8_t *>(job.x) +
                         ((int64_t)(t.entry / job.x_div) * job.x_stride + (int64_t)t.g * 256) * esz;
    mbar_arrive_expect_tx(bar, 256u * esz);
    bulk_g2s(xs, src, 256u * esz, bar);
}

// Issuer: a matrix's packed codebook into the staging buffer.
__device__ __forceinline__ void fetch_cb(const LutJob &job, const TbTab &t, uint32_t cbs,
                                         uint32_t bar) {
    mbar_arrive_expect_tx(bar, (uint32_t)TB_CB);
    bulk_g2s(cbs, tb_cb(job, t), (uint32_t)TB_CB, bar);
}

// Issuer: the table's code tiles (adjacent row slices of one chunk group, one
// contiguous range) into L2.
__device__ __forceinline__ void prefetch_table(const LutJob &job, const TbTab &t) {
    const int RB = job.rows / 32;
    const uint8_t *t0 = tb_codes(job, t) + ((size_t)t.g * RB + (size_t)t.r0 * TB_RB) * kTileBytes;
    prefetch_l2(t0, (uint32_t)(t.nr * TB_RB * kTileBytes));
}

__device__ __forceinline__ uint16_t bf16_rn_bits(float f) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}
__device__ __forceinline__ float bf16_val(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// Exact split of fp32 v into three bf16 terms, v = t1 + t2 + t3.
__device__ __forceinline__ void split3(float v, uint16_t &t1, uint16_t &t2, uint16_t &t3) {
    t1 = bf16_rn_bits(v);
    const float r1 = v - bf16_val(t1);
    t2 = bf16_rn_bits(r1);
    const float r2 = r1 - bf16_val(t2);
    t3 = bf16_rn_bits(r2);
}

// Builders: the staged fp32 codebook -> A (TMEM).  Thread (quarter q, lane l)
// writes codeword rows e = 128 i + 32 q + l of M tiles i < 6: 24 columns of
// bf16 pairs, K chunks [C1 | C2 | C3 | C1 | C2 | C1] (8 dimensions each).
__device__ __forceinline__ void codebook_to_tmem(const uint8_t *cbs, uint32_t tmem_a_q, int q,
                                                 int lane) {
    const float4 *cb4 = reinterpret_cast<const float4 *>(cbs);
#pragma unroll 1
    for (int i = 0; i < 6; ++i) {
        const int e = 128 * i + 32 * q + lane;
        // packed layout: (C_2j[d], C_2j+1[d]) pairs, 16 floats per entry pair
        const int base = (e >> 1) * 4, odd = e & 1;
        float c[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float4 v = cb4[base + j];
            c[2 * j] = odd ? v.y : v.x;
            c[2 * j + 1] = odd ? v.w : v.z;
        }
        uint32_t w1[4], w2[4], w3[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint16_t a1, a2, a3, b1, b2, b3;
            split3(c[2 * j], a1, a2, a3);
            split3(c[2 * j + 1], b1, b2, b3);
            w1[j] = (uint32_t)a1 | ((uint32_t)b1 << 16);
            w2[j] = (uint32_t)a2 | ((uint32_t)b2 << 16);
            w3[j] = (uint32_t)a3 | ((uint32_t)b3 << 16);
        }
        const uint32_t ta = tmem_a_q + 24u * i;
        const uint32_t v0[8] = {w1[0], w1[1], w1[2], w1[3], w2[0], w2[1], w2[2], w2[3]};
        const uint32_t v1[8] = {w3[0], w3[1], w3[2], w3[3], w1[0], w1[1], w1[2], w1[3]};
        const uint32_t v2[8] = {w2[0], w2[1], w2[2], w2[3], w1[0], w1[1], w1[2], w1[3]};
        tmem_st8(ta, v0);
        tmem_st8(ta + 8, v1);
        tmem_st8(ta + 16, v2);
    }
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Warp 0: the table's inputs (xs) -> B rows, K chunks [x1 | x1 | x1 | x2 | x2 |
// x3] of column c = lane, 128-byte swizzled (chunk j of row c at 16-byte slot
// j ^ (c % 8)).
__device__ __forceinline__ void inputs_to_b(const uint8_t *xs, int xdt, uint8_t *bsm, int lane) {
    float x[8];
    if (xdt == RVQ_BF16) {
        const uint4 v = *reinterpret_cast<const uint4 *>(xs + lane * 16);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[2 * i] = __uint_as_float(w[i] << 16);
            x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    } else {
        const float4 a = *reinterpret_cast<const float4 *>(xs + lane * 32);
        const float4 b = *reinterpret_cast<const float4 *>(xs + lane * 32 + 16);
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
        x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    }
    uint32_t w1[4], w2[4], w3[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint16_t a1, a2, a3, b1, b2, b3;
        split3(x[2 * j], a1, a2, a3);
        split3(x[2 * j + 1], b1, b2, b3);
        w1[j] = (uint32_t)a1 | ((uint32_t)b1 << 16);
        w2[j] = (uint32_t)a2 | ((uint32_t)b2 << 16);
        w3[j] = (uint32_t)a3 | ((uint32_t)b3 << 16);
    }
    uint8_t *row = bsm + lane * 128;
    const int sw = lane & 7;
    const uint4 c1 = make_uint4(w1[0], w1[1], w1[2], w1[3]);
    const uint4 c2 = make_uint4(w2[0], w2[1], w2[2], w2[3]);
    const uint4 c3 = make_uint4(w3[0], w3[1], w3[2], w3[3]);
    *reinterpret_cast<uint4 *>(row + ((0 ^ sw) << 4)) = c1;
    *reinterpret_cast<uint4 *>(row + ((1 ^ sw) << 4)) = c1;
    *reinterpret_cast<uint4 *>(row + ((2 ^ sw) << 4)) = c1;
    *reinterpret_cast<uint4 *>(row + ((3 ^ sw) << 4)) = c2;
    *reinterpret_cast<uint4 *>(row + ((4 ^ sw) << 4)) = c2;
    *reinterpret_cast<uint4 *>(row + ((5 ^ sw) << 4)) = c3;
}

// Rotate eight 16-byte chunks (4 words each) left by `by` chunks when `on`.
template <int BY>
__device__ __forceinline__ void rot_chunks(uint32_t (&r)[32], bool on) {
    uint32_t t[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) t[i] = r[(i + 4 * BY) & 31];
#pragma unroll
    for (int i = 0; i < 32; ++i) r[i] = on ? t[i] : r[i];
}

// Builders: M tile i's D rows of this warp's lane quarter -> table half h.
// Row e = 128 i + 32 q + l holds T[e / 256][e % 256][h][0..31] (byte e * 256 +
// h * 128); chunk j goes to slot (j + l) % 8.
__device__ __forceinline__ void d_to_table(uint32_t tmem_d_q, uint8_t *lut, int h, int q,
                                           int lane) {
    const int rot = lane & 7;
#pragma unroll 1
    for (int i = 0; i < 6; ++i) {
        float v[32];
        tmem_ld32(tmem_d_q + 32u * i, v);
        uint32_t r[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) r[c] = __float_as_uint(v[c]);
        rot_chunks<1>(r, rot & 1);
        rot_chunks<2>(r, rot & 2);
        rot_chunks<4>(r, rot & 4);
        const int e = 128 * i + 32 * q + lane;
        uint8_t *row = lut + (size_t)e * 256 + h * 128;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            *reinterpret_cast<uint4 *>(row + (((j + rot) & 7) << 4)) =
                make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
    }
}

// A lookup warp's walk over its tiles: block tile index j (over the block's
// tables in order, 16 nr tiles per table) with j = warp index mod 16.
struct TileGen {
    TbWalk w;
    TbTab t;
    int ti;   // table index in the block's sequence
    int jl;   // this warp's next tile index within table ti
    bool has;
};

__device__ __forceinline__ bool tile_next(const LutJob &job, int S, int w1, const int4 *pd, int wl,
                                          TileGen &G, int lane, const uint8_t *&tile, float *&out,
                                          int &ti) {
    while (G.has) {
        if (G.jl < TB_RB * G.t.nr) {
            const int RB = job.rows / 32;
            const int rb = (G.t.r0 + (G.jl >> 4)) * TB_RB + (G.jl & 15);
            tile = tb_codes(job, G.t) + ((size_t)G.t.g * RB + rb) * kTileBytes + lane * 16;
            out = job.part[G.t.m] + ((size_t)G.t.entry * job.G + G.t.g) * job.rows + rb * 32 + lane;
            ti = G.ti;
            G.jl += TB_LOOK_WARPS;
            return true;
        }
        // next table: its first block tile index is this one's end
        G.jl -= TB_RB * G.t.nr;
        ++G.ti;
        G.has = tb_next(job, S, w1, pd, G.w, G.t);
    }
    return false;
}

__device__ __forceinline__ void load_tile6(uint4 (&b)[6], const uint8_t *p) {
#pragma unroll
    for (int w = 0; w < 6; ++w) b[w] = ldg_stream(p + w * 512);
}

__global__ void __launch_bounds__(TB_THREADS, 1) lut_gemv_tc_kernel(const LutJob job,
                                                                    const int4 *pd) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    uint8_t *lut = smem + TB_OFF_LUT;
    const uint32_t bar0 = sbase + TB_OFF_BAR;
    auto bar = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + TB_OFF_FLAG);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // this block's unit range: whole tables when there are enough of them
    const int S = job.rows / TB_ROWS;
    const int tables = job.n_mat * job.n_pairs * job.G;
    int w0, w1;
    if (tables >= (int)gridDim.x) {
        w0 = (int)((int64_t)blockIdx.x * tables / gridDim.x) * S;
        w1 = (int)((int64_t)(blockIdx.x + 1) * tables / gridDim.x) * S;
    } else {
        const int64_t U = (int64_t)tables * S;
        w0 = (int)((int64_t)blockIdx.x * U / gridDim.x);
        w1 = (int)((int64_t)(blockIdx.x + 1) * U / gridDim.x);
    }

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         sbase + TB_OFF_TMEM),
                     "r"(TB_TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
        if (lane == 0) {
            mbar_init(bar(BAR_FULL + 0), TB_BUILD_WARPS);
            mbar_init(bar(BAR_FULL + 1), TB_BUILD_WARPS);
            mbar_init(bar(BAR_EMPTY + 0), TB_LOOK_WARPS);
            mbar_init(bar(BAR_EMPTY + 1), TB_LOOK_WARPS);
            mbar_init(bar(BAR_MMA), 1);
            mbar_init(bar(BAR_CB), 1);
            mbar_init(bar(BAR_X), 1);
            mbar_init(bar(BAR_DONE), 1);
            mbar_init(bar(BAR_NEVER), 1);
            *abort_flag = 0;
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + TB_OFF_TMEM);
    // early_start: the pair plan was written two or more launches back, so the
    // walk, the code tiles and the codebooks need not wait for the preceding
    // kernel (which writes only the inputs x)
    const bool early = job.early_start != 0;
    if (!early) {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        asm volatile("griddepcontrol.launch_dependents;");
    }

    if (warp < TB_BUILD_WARPS) {
        // ======================= builders =======================
        if (TB_REG_BUILD != TB_REG_LAUNCH)
            asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(TB_REG_BUILD));
        const bool issuer = tid == 0;
        const int q = warp;
        const uint32_t tq = tmem + ((uint32_t)(32 * q) << 16);
        const uint32_t cbs = sbase + TB_OFF_CB, xs = sbase + TB_OFF_XS;
        TbWalk bw = tb_start(job, S, w0);
        TbTab cur;
        bool has = tb_next(job, S, w1, pd, bw, cur);
        uint32_t ph_cb = 0, ph_x = 0, ph_mma = 0;
        bool cb_pending = false, x_pending = false;  // bulk copies issued, not yet waited
        int a_m = -1, a_rec = -1;                    // codebook held in A
        bool cb_free = true;                         // staging holds nothing still needed
        if (has) {
            if (issuer) {
                fetch_cb(job, cur, cbs, bar(BAR_CB));
                prefetch_table(job, cur);
            }
            cb_pending = true;
            cb_free = false;
        }
        if (early) {
            asm volatile("griddepcontrol.wait;" ::: "memory");
            asm volatile("griddepcontrol.launch_dependents;");
        }
        if (has) {
            if (issuer) fetch_x(job, cur, xs, bar(BAR_X));
            x_pending = true;
        }
        if (issuer && job.selftest_stall) mbar_wait(bar(BAR_NEVER), 0, abort_flag, job.status);
        const uint64_t bdesc = smem_desc(sbase + TB_OFF_B);
        const uint32_t idesc = idesc_bf16(128, 32);
        const int nk = job.x_dtype == RVQ_BF16 ? 2 : 3;  // K steps: bf16 inputs have x2 = x3 = 0
        int t = 0;
        for (;;) {
            // every builder runs the same iterations: failures are ORed at the
            // barrier below, and all builders leave together
            bool fail = *abort_flag != 0;
            TbWalk bw2 = bw;
            TbTab nxt;
            const bool has_n = has && tb_next(job, S, w1, pd, bw2, nxt);
            const int h = t & 1;
            // 1. the table's codebook into A (only when the expert or matrix changes)
            if (has && !fail && (cur.m != a_m || cur.rec != a_rec)) {
                if (warp_wait(bar(BAR_CB), ph_cb, abort_flag, job.status)) {
                    ph_cb ^= 1;
                    cb_pending = false;
                    cb_free = true;
                    codebook_to_tmem(smem + TB_OFF_CB, tq + TB_TMEM_A, q, lane);
                    a_m = cur.m;
                    a_rec = cur.rec;
                } else {
                    fail = true;  // the copy stays pending: drained below
                }
            }
            // 2. the inputs into B (warp 0)
            if (has && !fail && warp == 0) {
                if (warp_wait(bar(BAR_X), ph_x, abort_flag, job.status)) {
                    inputs_to_b(smem + TB_OFF_XS, job.x_dtype, smem + TB_OFF_B, lane);
                    // generic-proxy stores -> visible to the MMA (async proxy)
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                } else {
                    fail = true;
                }
            }
            // (only warp 0 waits on the inputs; the issuer's copy of these
            // flags is the one the drain reads)
            if (has && !fail) {
                ph_x ^= 1;
                x_pending = false;
            }
            __syncwarp();
            // A complete, the previous table's D read out, B written
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            const bool stop = builders_sync_any(fail || !has);
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            if (stop) break;
            const bool new_cb = has_n && cb_free && (nxt.m != cur.m || nxt.rec != cur.rec);
            if (issuer) {
#pragma unroll 1
                for (int i = 0; i < 6; ++i)
                    for (int kk = 0; kk < nk; ++kk)
                        mma_bf16_ts(tmem + TB_TMEM_D + 32u * i, tmem + TB_TMEM_A + 24u * i + 8u * kk,
                                    bdesc + 2u * kk, idesc, kk > 0 ? 1u : 0u);
                mma_commit(bar(BAR_MMA));
                // the next table's inputs, code tiles and (if it changes) codebook
                if (has_n) {
                    fetch_x(job, nxt, xs, bar(BAR_X));
                    prefetch_table(job, nxt);
                    if (new_cb) fetch_cb(job, nxt, cbs, bar(BAR_CB));
                }
            }
            if (has_n) x_pending = true;
            if (new_cb) {
                cb_free = false;
                cb_pending = true;
            }
            // 3. D -> table half h once that half's previous table (t - 2) is read
            bool ok = warp_wait(bar(BAR_MMA), ph_mma, abort_flag, job.status);
            ph_mma ^= 1;
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            if (ok && t >= 2)
                ok = warp_wait(bar(BAR_EMPTY + h), ((t - 2) >> 1) & 1, abort_flag, job.status);
            if (ok) d_to_table(tq + TB_TMEM_D, lut, h, q, lane);
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (ok && lane == 0) mbar_arrive(bar(BAR_FULL + h));
            cur = nxt;
            bw = bw2;
            has = has_n;
            ++t;
        }
        // drain: copies and MMAs in flight complete before the block exits
        if (issuer) {
            int no_abort = 0;
            if (cb_pending) mbar_wait(bar(BAR_CB), ph_cb, &no_abort, job.status);
            if (x_pending) mbar_wait(bar(BAR_X), ph_x, &no_abort, job.status);
            mma_commit(bar(BAR_DONE));
            mbar_wait(bar(BAR_DONE), 0, &no_abort, job.status);
        }
    } else {
        // ======================= lookups =======================
        if (TB_REG_LOOK != TB_REG_LAUNCH)
            asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(TB_REG_LOOK));
        const int wl = warp - TB_BUILD_WARPS;
        TileGen G;
        G.w = tb_start(job, S, w0);
        G.ti = 0;
        G.jl = wl;
        G.has = tb_next(job, S, w1, pd, G.w, G.t);
        // the block's table count (every table gets one arrival per warp)
        int n_tab = 0;
        {
            TbWalk cw = tb_start(job, S, w0);
            TbTab ct;
            while (tb_next(job, S, w1, pd, cw, ct)) ++n_tab;
        }
        uint4 buf[TB_RING][6];
        float *outp[TB_RING];
        int tix[TB_RING];
        bool have[TB_RING];
#pragma unroll
        for (int d = 0; d < TB_RING; ++d) {
            const uint8_t *tp;
            have[d] = tile_next(job, S, w1, pd, wl, G, lane, tp, outp[d], tix[d]);
            if (have[d]) load_tile6(buf[d], tp);
        }
        if (early) {
            asm volatile("griddepcontrol.wait;" ::: "memory");
            asm volatile("griddepcontrol.launch_dependents;");
        }
        uint32_t aux2[16];
        int tc = 0;       // tables this warp has released (arrived empty on)
        int waited = -1;  // table whose full phase this warp has seen
        bool alive = true;
        // release every table before ti (each is waited for first, so that an
        // arrival never counts toward an earlier phase of its half)
        auto release_upto = [&](int ti) -> bool {
            while (tc < ti) {
                if (waited < tc) {
                    if (!warp_wait(bar(BAR_FULL + (tc & 1)), (tc >> 1) & 1, abort_flag, job.status))
                        return false;
                    waited = tc;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(BAR_EMPTY + (tc & 1)));
                ++tc;
            }
            return true;
        };
        // release the tables before ti, then wait until ti is built
        auto enter = [&](int ti) -> bool {
            if (!release_upto(ti)) return false;
            if (waited < ti) {
                if (!warp_wait(bar(BAR_FULL + (ti & 1)), (ti >> 1) & 1, abort_flag, job.status))
                    return false;
                waited = ti;
                const uint32_t hb = (uint32_t)(ti & 1) << 7;
#pragma unroll
                for (int p2 = 0; p2 < 16; ++p2) {
                    const uint32_t c0 = (((lane + 2 * p2) & 31) << 2) | hb;
                    const uint32_t c1 = (((lane + 2 * p2 + 1) & 31) << 2) | hb;
                    aux2[p2] = c0 | (c1 << 8);
                }
            }
            return true;
        };
        int d = 0;
        for (;;) {
            bool any = false;
            // the ring is consumed in order: slot d holds the warp's oldest tile
            auto step = [&](auto slot) {
                constexpr int dd = decltype(slot)::value;
                if (!have[dd]) return;
                any = true;
                if (alive) alive = enter(tix[dd]);
                if (alive) *outp[dd] = tile_lookups1_g8(buf[dd], aux2, lut);
                const uint8_t *tp;
                have[dd] = alive && tile_next(job, S, w1, pd, wl, G, lane, tp, outp[dd], tix[dd]);
                if (have[dd]) load_tile6(buf[dd], tp);
            };
            static_assert(TB_RING == 2, "the ring steps below");
            if (d == 0) step(std::integral_constant<int, 0>{});
            else step(std::integral_constant<int, 1>{});
            if (!any) break;
            d = d == TB_RING - 1 ? 0 : d + 1;
        }
        // release the remaining tables (the builders wait on them)
        if (alive) release_upto(n_tab);
    }

    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(TB_TMEM_COLS));
    }
}

}  // namespace

rvq_status launch_lut_gemv_tc(const LutJob &job, const int4 *pd, cudaStream_t stream, bool pdl) {
    static std::atomic<int> attr_done[64];  // per device; setting twice is harmless
    int dev = 0;
    RVQ_CUDA(cudaGetDevice(&dev));
    if (dev < 64 && !attr_done[dev]) {
        RVQ_CUDA(cudaFuncSetAttribute(lut_gemv_tc_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, TB_SMEM));
        // the warp groups' setmaxnreg shares must fit the registers the block
        // is launched with, or the increase would wait forever
        cudaFuncAttributes fa;
        RVQ_CUDA(cudaFuncGetAttributes(&fa, lut_gemv_tc_kernel));
        if (fa.numRegs < TB_REG_LAUNCH) {
            set_error("lut_gemv_tc: kernel built with %d registers per thread, needs %d",
                      fa.numRegs, TB_REG_LAUNCH);
            return RVQ_ECUDA;
        }
        attr_done[dev] = 1;
    }
    if (job.rows % TB_ROWS || job.cols % 256 || job.G != job.cols / 256 || job.n_mat < 1 ||
        job.n_mat > 2 || (job.base == nullptr && (job.n_mat != 1 || pd != nullptr || !job.codes_ptr ||
                                                  !job.cb_ptr)) ||
        (job.base != nullptr && !pd) || (job.x_dtype != RVQ_F32 && job.x_dtype != RVQ_BF16)) {
        set_error("lut_gemv_tc: rows %d / cols %d / matrices %d not supported", job.rows, job.cols,
                  job.n_mat);
        return RVQ_EINVAL;
    }
    const int64_t tables = (int64_t)job.n_mat * job.n_pairs * job.G;
    const int64_t units = tables * (job.rows / TB_ROWS);
    if (units == 0) return RVQ_OK;
    if (units > (int64_t)1 << 30) {
        set_error("lut_gemv_tc: %lld units exceed the index range", (long long)units);
        return RVQ_EINVAL;
    }
    const int grid = units < num_sms() ? (int)units : num_sms();
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(TB_THREADS);
    cfg.dynamicSmemBytes = TB_SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    RVQ_CUDA(cudaLaunchKernelEx(&cfg, lut_gemv_tc_kernel, job, pd));
    return RVQ_OK;
}

}  // namespace rvq
