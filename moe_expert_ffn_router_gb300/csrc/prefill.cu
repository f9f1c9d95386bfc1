// Prefill path of the expert FFN: RVQ code tiles dequantised to 16-bit floats
// feed tcgen05 tensor-core GEMMs (fp32 accumulators in TMEM).
//
// For prefill-sized groups (tens to hundreds of tokens per expert) the FFN is
// a real dense contraction, so the weights are decoded once per tile --
// W[r][8j+i] = C1[c(r,j,1)][i] + C2[c(r,j,2)][i] + C3[c(r,j,3)][i], the residual
// decode of the pages ("WASTE Inference Engine", section "Residual Vector
// Quantization (RVQ)") -- and multiplied on the tensor cores.
//
// Precision: both GEMMs run on fp16 operands with fp32 accumulation.  The
// codewords are staged as fp16 and each weight is their fp16 sum; the tokens
// are converted to fp16 once per launch pair (tokens_f16_kernel), and
// h = silu(g) u is rounded to fp16.  fp16 keeps three more mantissa bits than
// bf16: with bf16 down operands (the weight sum rounded twice, h to 8 bits)
// one pair in about two thousand exceeded 2e-2 x RMS of the fp64 oracle, and
// a weight summed in fp16 needs no conversion before the MMA.  Values beyond
// the fp16 range (|x| or |h| > 65504) saturate and are reported as
// RVQ_DEV_ERR_NONFINITE.
//
// GEMM orientation (swap-AB): A = 128 weight rows x 64 K (16-bit, in tensor
// memory: row = TMEM lane, two K values per 32-bit column), B = up to NMAX
// tokens of one expert's group x 64 K (K-major, 128-byte swizzle, shared
// memory), D = W x^T (128 rows x N tokens, fp32, TMEM).  The decode warps
// write their rows of A straight into tensor memory (tcgen05.st), so A costs
// no shared-memory stores or operand reads, and every MMA reads B once.
//
// A work item is (expert, pass of <= NMAX tokens, M tiles of 128 A rows):
//  * gate/up launch (NMAX 160): an M tile holds 64 weight rows of gate and the
//    same 64 rows of up, interleaved in fours (A row r holds weight row
//    64 m + 4 (r / 8) + r % 4, of gate if r % 8 < 4, of up otherwise), so a
//    row's gate and up accumulators sit four TMEM lanes apart and the epilogue
//    pairs them with one shuffle: h = silu(g) * u -> fp16, row = the token's
//    position in the expert-grouped order, so each pass's rows are contiguous.
//    An item takes two M tiles (2 m, 2 m + 1) that share every K step's
//    gathered token rows (8 MMAs per B slot).
//  * down launch (NMAX 192): the A rows are down rows [128 m, 128 m + 128); B
//    is the pass's contiguous h rows, loaded by TMA; the epilogue writes fp32
//    y [pair][d].
// Items are split into contiguous ranges of equal estimated cost over a
// persistent grid (one CTA per SM), so consecutive items of a CTA mostly share
// the expert and its codebooks.  The first 256 items of a CTA are described
// once, in shared memory, by all threads at the start: walking the offsets
// and record headers between items (dependent global loads) cost each role
// ~3,500 cycles per item.
//
// Warp roles (512 threads):
//  warp 0      TMEM owner; lane 0 issues the MMAs (4 per M tile and K step)
//              and commits; gate/up: M tile 0 only
//  warps 1-2   gate/up B producers: cp.async gathers of fp16 token rows into
//              the B slot, eight threads per 128-byte row (a warp instruction
//              touches four lines, not 32)
//  warp 3      gate/up B relay (lane 0): once a slot's rows have landed,
//              fences them into the async proxy and signals the K step (the
//              fence costs the MMA thread nothing)
//  warp 1 l.0  down B producer: tiled TMA loads of the pass's h rows (async
//              proxy, completion counted on the K step's full barrier)
//  warps 4-7   epilogue: TMEM -> registers -> global (lane quarter = warp % 4);
//              gate/up: warp 7 lane 0 issues M tile 1's MMAs of an item before
//              the warp drains it (a second issuing thread: one thread issues
//              a tcgen05.mma only about every 115 cycles)
//  warps 8-15  A producers: decode code bytes into TMEM (lane quarter =
//              warp % 4); down: warps 8-11 take the even K steps, 12-15 the
//              odd ones; gate/up: warps 8-11 the item's first M tile, 12-15
//              its second, every K step.  Each warp loads its rows' code
//              planes one 32-chunk group ahead, across items too.
// K step t of the CTA's sequence uses an A stage (down: t % 4, TMEM columns
// 384 + 32 s; gate/up: t % 3, columns 320 + 64 s + 32 u for M tile u), B slot
// t % 5 (shared memory; five slots keep the token rows in flight against the
// L2 latency of the row gathers) and the full/empty mbarrier pair t % 8.
// full[t % 8] completes once the decode warps of the K step and the B side
// (the relay, or the TMA producer's expect_tx arrival and its bytes) have
// arrived, so each MMA-issuing thread waits once and commits once per K step
// (gate/up: empty[] takes both issuers' commits).  A decode warp reuses a
// stage after empty[t - stages], a B producer a slot after
// empty[(t - 5) % 8].  Down: two accumulators (TMEM columns 0 and 192,
// guarded by acc_full / acc_empty) let the epilogue of one item overlap the
// main loop of the next.  Gate/up: the item's M tiles use both (columns 0 and
// 160), each released by the epilogue as soon as it is drained (the next
// item's first M tile starts while the second still drains).
// Measured limits (per-warp clock traces of the 2048-token chunk): a decode
// warp takes ~700-780 cycles per gate/up K step, and issuing a tcgen05.mma
// occupies the issuing thread's sub-partition for ~85-115 cycles.  The decode
// warps on the sub-partitions that also run an issuer or the loaders start
// each step late, so the K step settles at ~1,150 cycles (~750 with the
// decode switched off).  Down is bound by its single issuer (4 MMAs and one
// wait, fence and commit per K step, ~650 cycles), its decode running ahead.
//
// Decoding is bound by shared-memory gathers of codewords, so the codebooks
// sit in shared memory as fp16 in a bank-private layout: line (stage s,
// codeword k) is 128 bytes, and 16-byte group q of every line serves lane q
// of each quarter-warp.  For gate/up, groups 0-3 hold gate's codebook and 4-7
// up's (lanes with r % 8 < 4 decode gate rows); for down all eight hold
// down's.  A quarter-warp thus reads eight codewords from eight distinct bank
// groups whatever the codes are.
//
// Every wait is bounded (1 s); on expiry the CTA records RVQ_DEV_ERR_TIMEOUT,
// every role leaves its loop, the MMAs in flight are drained and TMEM is freed.
#include "internal.cuh"
#include "tc_util.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <string.h>

namespace rvq {
namespace {

constexpr int PF_THREADS = 512;
constexpr int PF_NMAX = 192;                     // tokens per pass (MMA N), down
constexpr int PF_NMAX_PAIR = 160;                // gate/up: two accumulators of 160 columns leave
                                                 // TMEM room for three A stages
constexpr int PF_KC = 64;                        // K columns per stage (one 128-byte swizzle row)
constexpr int PF_NST = 4;                        // A stages (TMEM)
constexpr int PF_NSLOT = 5;                      // B slots (shared memory)
constexpr int PF_NBAR = 8;                       // full/empty barrier pairs (K steps in flight)
constexpr int PF_MROWS = 128;                    // A rows per item (MMA M)
constexpr int kSlotB = PF_NMAX * PF_KC * 2;      // 24 KiB of B per slot
constexpr int kCbLine = 128;                     // one (stage, codeword) line
constexpr int kCbBytes = 3 * 256 * kCbLine;      // 96 KiB
constexpr int OFF_CB = 0;
constexpr int OFF_ST = kCbBytes;
constexpr int OFF_BAR = OFF_ST + PF_NSLOT * kSlotB;
// mbarriers, 8 bytes each from OFF_BAR
constexpr int BAR_FULL = 0;                      // [PF_NBAR]
constexpr int BAR_EMPTY = BAR_FULL + PF_NBAR;    // [PF_NBAR]
constexpr int BAR_LANDED = BAR_EMPTY + PF_NBAR;  // [PF_NBAR] B rows of the K step in shared memory
constexpr int BAR_ACC_FULL = BAR_LANDED + PF_NBAR;    // [2]
constexpr int BAR_ACC_EMPTY = BAR_ACC_FULL + 2;       // [2]
constexpr int BAR_DONE = BAR_ACC_EMPTY + 2;      // [2]: each MMA issuer's final drain
constexpr int BAR_CB = BAR_DONE + 2;             // A producers: codebook swap rendezvous
constexpr int BAR_NEVER = BAR_CB + 1;            // self-test: a phase nothing completes
constexpr int kNumBars = BAR_NEVER + 1;
constexpr int OFF_TMEM = OFF_BAR + 8 * kNumBars;
constexpr int OFF_FLAG = OFF_TMEM + 4;
constexpr int OFF_Q = OFF_BAR + 512;             // pass prefix [E + 1]
constexpr int kMaxE = 256;
constexpr int OFF_W = OFF_Q + 4 * (kMaxE + 2);   // cost prefix [E + 1] (int64)
constexpr int kItemTable = 256;                  // items of a CTA described in shared memory
constexpr int OFF_IT = (OFF_W + 8 * (kMaxE + 1) + 15) & ~15;  // item table [kItemTable] (int4)
constexpr int OFF_EPI = OFF_IT + 16 * kItemTable;     // down epilogue: pair ids of a chunk [4][32]
constexpr int kPfSmem = OFF_EPI + 4 * 32 * 4 + 1024;  // + slack to align the base to 1 KiB
static_assert(OFF_IT % 16 == 0 && OFF_EPI % 16 == 0, "item table alignment");
static_assert(OFF_FLAG + 4 <= OFF_Q, "control block overlaps the pass prefix");
static_assert(kPfSmem <= 232448, "shared memory per CTA");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemD = 0;                   // accumulator b: columns [NMAX b, + NMAX)
// down: A stage s at columns [2 PF_NMAX + 32 s, + 32)
static_assert(2 * PF_NMAX + PF_NST * (PF_KC / 2) <= kTmemCols, "TMEM columns");
// gate/up items pair two M tiles on one B slot: accumulator of M tile u at
// columns [PF_NMAX_PAIR u, + PF_NMAX_PAIR), A stage s of M tile u at
// 2 PF_NMAX_PAIR + 64 s + 32 u
constexpr int PF_NST_PAIR = 3;
static_assert(2 * PF_NMAX_PAIR + PF_NST_PAIR * PF_KC <= kTmemCols, "TMEM columns (paired M tiles)");
static_assert(PF_NBAR >= PF_NSLOT + 1 && PF_NBAR >= PF_NST + 1, "a barrier pair outlives its stage");
static_assert(kSlotB % 1024 == 0 && OFF_ST % 1024 == 0, "swizzled slots start on 1 KiB");

constexpr int kLoaders = 64;                     // gate/up B producer threads (warps 1-2)
constexpr int kTmaRows = 32;                     // token rows per down B TMA box
constexpr int kLoaderRows = PF_NMAX_PAIR / 8;    // token rows per producer thread (8 threads a row)
constexpr int kDecodeWarps = 8;                  // A producer warps (8-15)
// full[] arrivals: the decode warps of the K step (down: one half of them;
// gate/up: all eight, four per M tile) + the B side (the relay, or the TMA
// producer's expect_tx arrival)
constexpr uint32_t kFullCount = kDecodeWarps / 2 + 1;
constexpr uint32_t kFullCountPair = kDecodeWarps + 1;

// Three fp16x2 codeword words summed in fp16: two fp16 weights.
__device__ __forceinline__ uint32_t sum3_f16x2(uint32_t a, uint32_t b, uint32_t c) {
    const __half2 s = __hadd2(__hadd2(*reinterpret_cast<const __half2 *>(&a),
                                      *reinterpret_cast<const __half2 *>(&b)),
                              *reinterpret_cast<const __half2 *>(&c));
    return *reinterpret_cast<const uint32_t *>(&s);
}

// A value as fp16 bits for the GEMMs (h = silu(g) u, or a token); beyond the
// fp16 range it saturates to +-65504 and is reported (*over = true); NaN
// stays NaN.
__device__ __forceinline__ uint16_t h_to_f16(float hv, bool &over) {
    if (fabsf(hv) > 65504.0f) {
        over = true;
        hv = copysignf(65504.0f, hv);
    }
    return __half_as_ushort(__float2half_rn(hv));
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

// Tiled TMA load of one box (64 bf16 columns from col x kTmaRows rows from
// row) to dst, 128-byte swizzled by shared-address bits (the layout the MMA's
// B descriptor reads); completes its bytes on mbar.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *tm, int col, int row,
                                            uint32_t mbar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(col), "r"(row), "r"(mbar)
        : "memory");
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

struct PfItem {
    int e, o, j0, n, npad, mt;
    int rec;  // record index of expert e (its cache slot, or e)
    bool valid;
};

// Cost of one item per K step, in units of ~7.7 cycles, fitted to timestamp
// traces of the 2048-token chunk:
//  * gate/up (two M tiles, token rows gathered by cp.async): ~1,600 cycles
//    of decoding plus ~3.9 per row, the epilogue between items included;
//  * down (rows by TMA): ~800 cycles + ~1 per row, plus a start of ~3,000
//    cycles spread over its 32 K steps.
// CTAs get contiguous item ranges of equal total cost: item costs differ by
// 2x or more across a Zipf-skewed chunk, and equal item counts left the
// slowest CTA 1.5x behind the median.
__device__ __forceinline__ int64_t pf_cost(const PfJob &job, int npad) {
    return job.mode == PF_MODE_SWIGLU ? (int64_t)210 + npad / 2 : (int64_t)116 + npad / 8;
}

// Tokens per pass of the launch.
__device__ __forceinline__ int pf_nmax(const PfJob &job) {
    return job.mode == PF_MODE_SWIGLU ? PF_NMAX_PAIR : PF_NMAX;
}

// Passes of expert e (0 when its group is below min_tokens) and their cost.
__device__ __forceinline__ void pf_expert_cost(const PfJob &job, int ne, int MT, int &passes,
                                               int64_t &cost) {
    const int NM = pf_nmax(job);
    passes = ne >= job.min_tokens && ne > 0 ? (ne + NM - 1) / NM : 0;
    cost = 0;
    if (passes > 0) {
        const int last = ne - (passes - 1) * NM;
        cost = (int64_t)MT * ((passes - 1) * pf_cost(job, NM) + pf_cost(job, (last + 15) & ~15));
    }
}

// First item whose cumulative cost start is >= t (W[e] = cost before expert e).
__device__ int pf_first_item(const PfJob &job, const int32_t *Q, const int64_t *W, int MT,
                             int64_t t) {
    const int E = job.E;
    if (t >= W[E]) return Q[E] * MT;
    int lo = 0, hi = E;  // largest e with W[e] <= t: W[e + 1] > t, so e has work
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (W[mid] <= t) lo = mid; else hi = mid;
    }
    const int ne = job.offsets[lo + 1] - job.offsets[lo];
    const int NM = pf_nmax(job);
    const int P = (ne + NM - 1) / NM;
    const int64_t cf = pf_cost(job, NM);
    const int64_t cl = pf_cost(job, (ne - (P - 1) * NM + 15) & ~15);
    int64_t rem = t - W[lo];
    const int64_t pq = rem / ((int64_t)MT * cf);
    const int pi = (int)(pq < (int64_t)P - 1 ? pq : (int64_t)P - 1);
    rem -= (int64_t)pi * MT * cf;
    const int64_t c = pi < P - 1 ? cf : cl;
    // mt may equal MT: the first item of the next pass
    return (Q[lo] + pi) * MT + (int)((rem + c - 1) / c);
}

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
    const int NM = pf_nmax(job);
    I.j0 = (pi - Q[lo]) * NM;
    I.n = min(NM, ne - I.j0);
    I.npad = (I.n + 15) & ~15;
    I.rec = record_of(job, lo);
    const rvq_expert_header *h = I.rec < 0 ? nullptr :
        reinterpret_cast<const rvq_expert_header *>(job.base + (uint64_t)I.rec * job.record_bytes);
    I.valid = I.n > 0 && h && h->magic == RVQ_BANK_MAGIC && h->expert == lo &&
              h->layer == job.layer && h->d == job.d && h->f == job.f &&
              h->record_bytes == job.record_bytes;
    return I;
}

// An item as one table entry: {o, rec, j0, e | n << 12 | mt << 21 | valid << 31}.
__device__ __forceinline__ int4 pf_pack(const PfItem &I) {
    return make_int4(I.o, I.rec, I.j0,
                     (int)((uint32_t)I.e | ((uint32_t)I.n << 12) | ((uint32_t)I.mt << 21) |
                           ((uint32_t)I.valid << 31)));
}
__device__ __forceinline__ PfItem pf_unpack(int4 v) {
    PfItem I;
    I.o = v.x;
    I.rec = v.y;
    I.j0 = v.z;
    const uint32_t w = (uint32_t)v.w;
    I.e = (int)(w & 0xFFFu);
    I.n = (int)((w >> 12) & 0x1FFu);
    I.mt = (int)((w >> 21) & 0x3FFu);
    I.valid = (w >> 31) != 0;
    I.npad = (I.n + 15) & ~15;
    return I;
}

// kPair: gate/up launch (two M tiles per item, SwiGLU epilogue); otherwise down.
template <bool kPair>
__global__ void __launch_bounds__(PF_THREADS, 1)
    prefill_gemm_kernel(const PfJob job, const __grid_constant__ CUtensorMap tmap_b) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // the 128-byte swizzle is a function of shared-address bits 4..9: B stages
    // must start on 1024-byte boundaries of the shared window
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + OFF_BAR;
    auto bar = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + OFF_FLAG);
    int32_t *Q = reinterpret_cast<int32_t *>(smem + OFF_Q);
    int64_t *W = reinterpret_cast<int64_t *>(smem + OFF_W);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // gate/up: an item is a pair of M tiles sharing each K step's B slot
    constexpr bool pair = kPair;
    constexpr bool swiglu = kPair;
    const int MT = job.rows / job.tile_rows / (pair ? 2 : 1);  // items per pass
    constexpr int NST = pair ? PF_NST_PAIR : PF_NST;           // A stages: K step t uses t % NST
    constexpr int NMAX = pair ? PF_NMAX_PAIR : PF_NMAX;        // tokens per pass
    constexpr uint32_t kTmemA = 2 * NMAX;                      // first A stage column
    const int KS = job.cols / PF_KC;             // a multiple of 4

    asm volatile("griddepcontrol.wait;" ::: "memory");

    // ---- setup: pass prefix (warp 1), barriers + TMEM (warp 0) ----------
    if (warp == 1) {
        // pass prefix Q and cost prefix W over the experts (lane: a run of them)
        const int E = job.E;
        const int per = (E + 31) / 32;
        const int e0 = min(E, lane * per), e1 = min(E, e0 + per);
        int cnt = 0;
        int64_t cst = 0;
        bool ok = true;
        for (int e = e0; e < e1; ++e) {
            const int ne = job.offsets[e + 1] - job.offsets[e];
            ok = ok && ne >= 0;
            int P;
            int64_t c;
            pf_expert_cost(job, ne, MT, P, c);
            cnt += P;
            cst += c;
        }
        int incl = cnt;
        int64_t cincl = cst;
#pragma unroll
        for (int s = 1; s < 32; s <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, s);
            const int64_t cv = __shfl_up_sync(0xffffffffu, cincl, s);
            if (lane >= s) {
                incl += v;
                cincl += cv;
            }
        }
        int pre = incl - cnt;
        int64_t cpre = cincl - cst;
        for (int e = e0; e < e1; ++e) {
            Q[e] = pre;
            W[e] = cpre;
            const int ne = job.offsets[e + 1] - job.offsets[e];
            int P;
            int64_t c;
            pf_expert_cost(job, ne, MT, P, c);
            pre += P;
            cpre += c;
        }
        ok = __all_sync(0xffffffffu, ok) && job.offsets[0] == 0 && job.offsets[E] == job.n_pairs;
        if (lane == 31) {
            Q[E] = ok ? incl : 0;
            W[E] = ok ? cincl : 0;
        }
        if (!ok && lane == 0) set_dev_error(job.status, RVQ_DEV_ERR_INDEX);
    } else if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         sbase + OFF_TMEM),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
        if (lane == 0) {
            for (int s = 0; s < PF_NBAR; ++s) {
                mbar_init(bar(BAR_FULL + s), pair ? kFullCountPair : kFullCount);
                // gate/up: each M tile's MMA issuer commits (two arrivals)
                mbar_init(bar(BAR_EMPTY + s), pair ? 2 : 1);
                mbar_init(bar(BAR_LANDED + s), kLoaders);
            }
            for (int b = 0; b < 2; ++b) {
                mbar_init(bar(BAR_ACC_FULL + b), 1);
                mbar_init(bar(BAR_ACC_EMPTY + b), 4);
            }
            mbar_init(bar(BAR_DONE), 1);
            mbar_init(bar(BAR_DONE + 1), 1);
            mbar_init(bar(BAR_CB), kDecodeWarps);
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

    // this CTA's items: an equal share of the total cost
    const int64_t T = W[job.E];
    const int it0 = pf_first_item(job, Q, W, MT, (int64_t)blockIdx.x * T / gridDim.x);
    const int it1 = pf_first_item(job, Q, W, MT, (int64_t)(blockIdx.x + 1) * T / gridDim.x);
    // the first kItemTable items described once, one per thread, so that no
    // role walks the offsets and record headers (dependent global loads)
    // between items
    int4 *itab = reinterpret_cast<int4 *>(smem + OFF_IT);
    if (tid < kItemTable && it0 + tid < it1) itab[tid] = pf_pack(pf_item(job, Q, MT, it0 + tid));
    __syncthreads();
    auto item = [&](int it) -> PfItem {
        return it - it0 < kItemTable ? pf_unpack(itab[it - it0]) : pf_item(job, Q, MT, it);
    };

    // The MMAs of one item on accumulator `acc` (TMEM columns acc * NMAX),
    // issued by one thread: gate/up M tile u == acc (its A stage columns
    // + 32 u), down the item's alternating accumulator.  One thread issues a
    // tcgen05.mma about every 115 cycles whatever N <= 192 (a microbenchmark;
    // two threads on separate accumulators issue twice as many), so gate/up
    // gives each M tile its own issuing thread: warp 0 lane 0 (tile 0) and
    // warp 7 lane 0 (tile 1, between its epilogue drains).  Returns false once
    // the kernel aborts.
    const uint64_t bdesc0 = smem_desc(sbase + OFF_ST);
    auto issue_item = [&](const PfItem &I, uint32_t &kg, uint32_t &slot, uint32_t acc,
                          uint32_t acc_use, uint32_t u) -> bool {
        if (!mbar_wait(bar(BAR_ACC_EMPTY + acc), (acc_use & 1u) ^ 1u, abort_flag, job.status))
            return false;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t idesc = idesc_f16(PF_MROWS, I.npad);
        const uint32_t td = tmem + kTmemD + acc * NMAX;
        for (int ks = 0; ks < KS; ++ks, ++kg) {
            if (!mbar_wait(bar(BAR_FULL + (kg & (PF_NBAR - 1))), (kg / PF_NBAR) & 1u, abort_flag,
                           job.status))
                return false;
            // (the B producers fenced their slot writes into the async proxy)
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            // start-address field: +1 per 16 bytes (32 bytes per 16 K)
            const uint64_t bd = bdesc0 + slot * (uint32_t)(kSlotB >> 4);
            const uint32_t ta = pair ? tmem + kTmemA + (kg % NST) * PF_KC + 32 * u
                                     : tmem + kTmemA + (kg % NST) * (PF_KC / 2);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16_ts(td, ta + kk * 8, bd + 2 * kk, idesc, (ks > 0 || kk > 0) ? 1u : 0u);
            mma_commit(bar(BAR_EMPTY + (kg & (PF_NBAR - 1))));
            slot = slot == PF_NSLOT - 1 ? 0 : slot + 1;
        }
        mma_commit(bar(BAR_ACC_FULL + acc));
        return true;
    };
    // every MMA an issuer queued has completed before TMEM is released
    auto issuer_drain = [&](int which) {
        mma_commit(bar(BAR_DONE + which));
        int no_abort = 0;
        mbar_wait(bar(BAR_DONE + which), 0, &no_abort, job.status);
    };

    if (warp == 0) {
        // ================= MMA issuer =================
        if (lane == 0) {
            uint32_t kg = 0, slot = 0, nacc = 0;  // K steps, B slot, items consumed
            // self-test of the failure path: wait for an arrival nothing makes,
            // so the bounded wait expires and every role gives up
            if (job.selftest_stall) mbar_wait(bar(BAR_NEVER), 0, abort_flag, job.status);
            for (int it = it0; it < it1 && !*abort_flag; ++it) {
                const PfItem I = item(it);
                if (!I.valid) {
                    // a bad or missing record (header mismatch, no cache slot):
                    // every role skips the item; the MMA thread reports it
                    if (I.n > 0) set_dev_error(job.status, RVQ_DEV_ERR_CORRUPT);
                    continue;
                }
                // down: two accumulators alternate over items; gate/up: this
                // thread issues M tile 0 on accumulator 0 (warp 7 issues M
                // tile 1 on accumulator 1), each released by the epilogue on
                // its own
                const uint32_t ab = pair ? 0u : (nacc & 1u), use = pair ? nacc : (nacc >> 1);
                if (!issue_item(I, kg, slot, ab, use, 0)) break;
                ++nacc;
            }
            issuer_drain(0);
        }
        __syncwarp();
    } else if (warp < 4) {
        // ================= B producers and relay =================
        uint32_t kg = 0, slot = 0;
        if (!swiglu) {
            // down: the pass's h rows are contiguous (grouped order); one
            // thread loads kTmaRows-row boxes per K step
            if (warp == 1 && lane == 0) {
                for (int it = it0; it < it1 && !*abort_flag; ++it) {
                    const PfItem I = item(it);
                    if (!I.valid) continue;
                    const int nbox = (I.npad + kTmaRows - 1) / kTmaRows;
                    const uint32_t bytes = (uint32_t)nbox * kTmaRows * (PF_KC * 2);
                    const int q0 = I.o + I.j0;
                    bool ok = true;
                    for (int ks = 0; ks < KS; ++ks, ++kg) {
                        if (kg >= (uint32_t)PF_NSLOT) {
                            const uint32_t kp = kg - PF_NSLOT;
                            if (!mbar_wait(bar(BAR_EMPTY + (kp & (PF_NBAR - 1))),
                                           (kp / PF_NBAR) & 1u, abort_flag, job.status)) {
                                ok = false;
                                break;
                            }
                        }
                        const uint32_t sb = sbase + OFF_ST + slot * kSlotB;
                        const uint32_t full = bar(BAR_FULL + (kg & (PF_NBAR - 1)));
                        mbar_arrive_expect_tx(full, bytes);
                        for (int i = 0; i < nbox; ++i)
                            tma_load_2d(sb + i * kTmaRows * (PF_KC * 2), &tmap_b, ks * PF_KC,
                                        q0 + i * kTmaRows, full);
                        slot = slot == PF_NSLOT - 1 ? 0 : slot + 1;
                    }
                    if (!ok) break;
                }
            }
        } else if (warp < 3) {
            // gate/up: fp16 token rows x16[entry / x_div], gathered by cp.async.
            // Eight consecutive threads copy the eight 16-byte chunks of one row,
            // so a warp instruction touches four 128-byte lines (one L1 tag
            // lookup each) instead of 32.
            const int lt = tid - 32;
            const int c = lt & 7;                 // the 16-byte chunk this thread copies
            const int r0 = lt >> 3;               // rows r0, r0 + 8, ...
            const uint32_t sw = (uint32_t)((c ^ r0) << 4);  // 128-byte swizzle (row & 7 = r0)
            for (int it = it0; it < it1 && !*abort_flag; ++it) {
                const PfItem I = item(it);
                if (!I.valid) continue;
                // token row of each of this thread's rows (-1: none)
                int row[kLoaderRows];
#pragma unroll
                for (int r = 0; r < kLoaderRows; ++r) {
                    const int j = r0 + 8 * r;
                    row[r] = -1;
                    if (j < I.n) {
                        const int p = job.pairs[I.o + I.j0 + j];
                        if (p >= 0 && p < job.n_pairs)
                            row[r] = p / job.x_div;
                        else
                            set_dev_error(job.status, RVQ_DEV_ERR_INDEX);
                    }
                }
                const uint8_t *xb = reinterpret_cast<const uint8_t *>(job.x) + c * 16;
                bool ok = true;
                for (int ks = 0; ks < KS; ++ks, ++kg) {
                    // the slot's previous K step (5 back) has been consumed
                    if (kg >= (uint32_t)PF_NSLOT) {
                        const uint32_t kp = kg - PF_NSLOT;
                        if (!mbar_wait(bar(BAR_EMPTY + (kp & (PF_NBAR - 1))), (kp / PF_NBAR) & 1u,
                                       abort_flag, job.status)) {
                            ok = false;
                            break;
                        }
                    }
                    const uint32_t sb = sbase + OFF_ST + slot * kSlotB + r0 * 128 + sw;
                    const uint32_t landed = bar(BAR_LANDED + (kg & (PF_NBAR - 1)));
                    const uint8_t *xk = xb + ks * PF_KC * 2;
#pragma unroll
                    for (int r = 0; r < kLoaderRows; ++r)
                        if (row[r] >= 0)
                            cp_async16(sb + r * 8 * 128, xk + (int64_t)row[r] * job.x_stride * 2);
                    // arrives once this thread's copies have landed
                    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(landed)
                                 : "memory");
                    slot = slot == PF_NSLOT - 1 ? 0 : slot + 1;
                }
                if (!ok) break;
            }
            asm volatile("cp.async.wait_all;" ::: "memory");
        } else if (lane == 0) {
            // relay: every producer's rows of the K step are in shared memory
            // (their arrivals release them); the fence orders them before the
            // MMA's async-proxy reads, which acquire through full[]
            for (int it = it0; it < it1 && !*abort_flag; ++it) {
                const PfItem I = item(it);
                if (!I.valid) continue;
                bool ok = true;
                for (int ks = 0; ks < KS; ++ks, ++kg) {
                    if (!mbar_wait_spin(bar(BAR_LANDED + (kg & (PF_NBAR - 1))),
                                        (kg / PF_NBAR) & 1u, abort_flag, job.status)) {
                        ok = false;
                        break;
                    }
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    mbar_arrive(bar(BAR_FULL + (kg & (PF_NBAR - 1))));
                }
                if (!ok) break;
            }
        }
    } else if (warp < 8) {
        // ================= epilogue =================
        // Compact on purpose: it runs once per item, and a fully unrolled
        // epilogue (~45 KB of code) stalled the next item on instruction fetch.
        const int ew = warp - 4;                 // TMEM lanes 32 ew .. 32 ew + 31
        const int ar = ew * 32 + lane;           // A row
        const int q = lane & 7;
        const bool up = swiglu && q >= 4;        // gate/up: this lane holds up's accumulator
        // weight row of this lane within the M tile (gate/up: gate lanes q < 4)
        const int rin = swiglu ? (ar >> 3) * 4 + (q & 3) : ar;
        const uint32_t tl = tmem + ((uint32_t)(ew * 32) << 16) + kTmemD;
        uint32_t nacc = 0;
        bool over = false;
        // gate/up: warp 7 lane 0 also issues M tile 1's MMAs of each item
        // (between draining the previous item and draining this one)
        const bool issuer = pair && warp == 7;
        uint32_t kg1 = 0, slot1 = 0;
        bool issue_ok = true;
        for (int it = it0; it < it1; ++it) {
            const PfItem I = item(it);
            if (!I.valid) continue;
            if (issuer) {
                if (lane == 0 && issue_ok && !*abort_flag)
                    issue_ok = issue_item(I, kg1, slot1, 1, nacc, 1);
                __syncwarp();
            }
            const int32_t *pp = job.pairs + I.o + I.j0;
            // the pair id of the item's token j (-1: none)
            auto pair_at = [&](int j) -> int {
                const int p = j < I.n ? pp[j] : -1;
                return (p >= 0 && p < job.n_pairs) ? p : -1;
            };
            const int nch = (I.n + 31) / 32;     // 32-token chunks of the accumulator
            // down: the pair id of each token (its y row), fetched before the
            // accumulator is ready (gate/up writes h by grouped position)
            int p0 = swiglu ? -1 : pair_at(lane);
            const uint32_t ab = pair ? 0u : (nacc & 1u), use = pair ? nacc : (nacc >> 1);
            // gate/up: the item's two M tiles, accumulators 0 and 1, each
            // drained once its own issuer's MMAs are done and released as soon
            // as it is drained
            bool acc_ok = true;
#pragma unroll 1
            for (int mu = 0; mu < (pair ? 2 : 1); ++mu) {
                const uint32_t acc = pair ? (uint32_t)mu : ab;
                if (!mbar_wait(bar(BAR_ACC_FULL + acc), use & 1u, abort_flag, job.status)) {
                    acc_ok = false;
                    break;
                }
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const int R = ((pair ? 2 * I.mt + mu : I.mt)) * job.tile_rows + rin;
                int pc = p0;
#pragma unroll 1
                for (int c = 0; c < nch; ++c) {
                    const int pn = !swiglu && c + 1 < nch ? pair_at(32 * (c + 1) + lane) : -1;
                    float a[32];
                    tmem_ld32(tl + acc * NMAX + 32 * c, a);
                    if (swiglu) {
                        // h rows in the grouped order; a gate lane and its up
                        // partner (lane ^ 4) hold g and u of the same weight row:
                        // the gate lane takes token t, the up lane token t + 1
                        uint16_t *hrow = reinterpret_cast<uint16_t *>(job.out) +
                                         (size_t)(I.o + I.j0 + 32 * c) * job.rows + R;
                        const int nt = I.n - 32 * c;     // tokens of this chunk
                        // two phases, so that the 16 exchanges and SwiGLUs overlap
                        // instead of forming one chain per token pair
                        float oth[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            oth[i] = __shfl_xor_sync(0xffffffffu, up ? a[2 * i] : a[2 * i + 1], 4);
                        // columns past the chunk's tokens hold padding: not converted
                        const int t0 = up ? 1 : 0;
                        uint16_t hb[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const float g = up ? oth[i] : a[2 * i];
                            const float u = up ? a[2 * i + 1] : oth[i];
                            const float hv = __fdividef(g * u, 1.0f + __expf(-g));
                            hb[i] = h_to_f16(2 * i + t0 < nt ? hv : 0.0f, over);
                        }
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            if (2 * i + t0 < nt) hrow[(size_t)(2 * i + t0) * job.rows] = hb[i];
                    } else {
                        // the chunk's 32 pair ids to every lane through a per-warp
                        // scratch (broadcast reads) rather than 32 shuffles
                        int *pw = reinterpret_cast<int *>(smem + OFF_EPI) + 32 * ew;
                        pw[lane] = pc;
                        __syncwarp();
                        int pv[32];
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int4 v = reinterpret_cast<const int4 *>(pw)[i];
                            pv[4 * i] = v.x;
                            pv[4 * i + 1] = v.y;
                            pv[4 * i + 2] = v.z;
                            pv[4 * i + 3] = v.w;
                        }
                        __syncwarp();
                        float *yrow = reinterpret_cast<float *>(job.out) + R;
#pragma unroll
                        for (int t = 0; t < 32; ++t)
                            if (pv[t] >= 0) yrow[(size_t)pv[t] * job.rows] = a[t];
                    }
                    pc = pn;
                }
                asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(BAR_ACC_EMPTY + acc));
            }
            if (!acc_ok) break;
            ++nacc;
        }
        if (__any_sync(0xffffffffu, over) && lane == 0) set_dev_error(job.status, RVQ_DEV_ERR_NONFINITE);
        if (issuer && lane == 0) issuer_drain(1);
        __syncwarp();
    } else {
        // ================= A producers (decode into TMEM) =================
        const int dt = tid - 256;
        const int quarter = warp & 3;            // TMEM lanes 32 quarter .. + 31
        // down: warps 8-11 take the even K steps, 12-15 the odd ones; gate/up:
        // warps 8-11 decode the item's first M tile, 12-15 its second, every K step
        const int half = pair ? 0 : (warp - 8) >> 2;
        const int u = pair ? (warp - 8) >> 2 : 0;
        constexpr int nj = pair ? 4 : 2;         // K steps of a 4-step group decoded here
        const int ar = quarter * 32 + lane;      // A row
        const int q = lane & 7;
        const int mat = swiglu ? (q >> 2) : 0;   // gate / up (down: both slots hold down)
        const int rin = swiglu ? (ar >> 3) * 4 + (q & 3) : ar;
        const uint32_t cbl = sbase + OFF_CB + q * 16;  // this lane's bank group
        const uint32_t ta = tmem + ((uint32_t)(quarter * 32) << 16) + kTmemA;
        const int RB = job.rows / 32;
        const int G = KS / 4;                    // 32-chunk groups along K
        // this row's code planes of 32-chunk group 0 of an item: 6 x 16 bytes
        // (stage s, half h) at cp + (2 s + h) * 512; group g adds g * RB tiles
        auto planes_of = [&](const PfItem &J) -> const uint8_t * {
            const int R = (pair ? 2 * J.mt + u : J.mt) * job.tile_rows + rin;
            return job.base + (uint64_t)J.rec * job.record_bytes + job.codes_off[mat] +
                   (size_t)(R >> 5) * kTileBytes + (R & 31) * 16;
        };
        // the first valid item at or after `from` (it1: none)
        auto next_valid = [&](int from, PfItem &J) -> int {
            for (; from < it1; ++from) {
                J = item(from);
                if (J.valid) break;
            }
            return from;
        };
        int cur_e = -1;
        uint32_t kg = 0, ncb = 0;
        PfItem I;
        int it = next_valid(it0, I);
        // the planes of the item's first group, loaded one group ahead (across
        // items too: the next item's first group loads during this item's last)
        uint4 nxt[6];
        if (it < it1) {
            const uint8_t *cp0 = planes_of(I);
#pragma unroll
            for (int v = 0; v < 6; ++v) nxt[v] = *reinterpret_cast<const uint4 *>(cp0 + v * 512);
        }
        while (it < it1 && !*abort_flag) {
            PfItem In;
            const int itn = next_valid(it + 1, In);
            const uint8_t *rec = job.base + (uint64_t)I.rec * job.record_bytes;
            if (I.e != cur_e) {
                // every A producer is done with the previous codebooks
                if (cur_e >= 0) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(BAR_CB));
                    if (!mbar_wait(bar(BAR_CB), ncb & 1u, abort_flag, job.status)) break;
                    ++ncb;
                }
                // record fp32 [s][k/2][i][k&1] -> fp16 lines, one 16-byte group per unit
                for (int u = dt; u < 3 * 256 * 8; u += kDecodeWarps * 32) {
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
            const int R = (pair ? 2 * I.mt + u : I.mt) * job.tile_rows + rin;
            const int l = R & 31;
            // Chunk j of this row sits at byte (j - l) mod 32 of each stage
            // plane; rotating by l - 8 half puts chunks 8 half .. 8 half + 7 (K
            // step 4 g + half) in bytes 0..7 and chunks 8 half + 16 .. + 23 (K
            // step 4 g + half + 2) in bytes 16..23 (gate/up: half 0, every
            // chunk j at byte j).
            const int rot = (l - 8 * half) & 31;
            const uint8_t *cp = planes_of(I);
            const uint8_t *cpn = itn < it1 ? planes_of(In) : nullptr;
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
#pragma unroll
                for (int s = 0; s < 3; ++s) derotate(U[s], rot);
                // the next group's planes (or the next item's first) load while
                // this one decodes
                const uint8_t *cg = g + 1 < G ? cp + (size_t)(g + 1) * RB * kTileBytes : cpn;
                if (cg != nullptr) {
#pragma unroll
                    for (int v = 0; v < 6; ++v)
                        nxt[v] = *reinterpret_cast<const uint4 *>(cg + v * 512);
                }
#pragma unroll
                for (int j = 0; j < nj; ++j) {
                    // this K step, its A stage and its first code word
                    const uint32_t kt = pair ? kg + 4 * g + j : kg + 4 * g + 2 * j + half;
                    const uint32_t st = kt % (uint32_t)NST;
                    const int w0 = pair ? 2 * j : 4 * j;
                    const uint32_t tst = pair ? st * PF_KC + 32 * u : st * (PF_KC / 2);
                    // the stage's previous K step (NST back) has been consumed
                    if (kt >= (uint32_t)NST) {
                        const uint32_t kp = kt - NST;
                        if (!mbar_wait(bar(BAR_EMPTY + (kp & (PF_NBAR - 1))),
                                       (kp / PF_NBAR) & 1u, abort_flag, job.status)) {
                            ok = false;
                            break;
                        }
                    }
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
#pragma unroll
                    for (int hq = 0; hq < 4; ++hq) {
                        uint32_t o[8];
#pragma unroll
                        for (int c = 0; c < 2; ++c) {
                            // chunk 2 hq + c of the K step: word w0 + hq / 2, byte 2 (hq % 2) + c
                            const int w = w0 + (hq >> 1), b = 8 * (2 * (hq & 1) + c);
                            const uint32_t k0 = (U[0][w] >> b) & 0xFFu;
                            const uint32_t k1 = (U[1][w] >> b) & 0xFFu;
                            const uint32_t k2 = (U[2][w] >> b) & 0xFFu;
                            const uint4 w0 = lds128(cbl + k0 * kCbLine);
                            const uint4 w1 = lds128(cbl + (256 + k1) * kCbLine);
                            const uint4 w2 = lds128(cbl + (512 + k2) * kCbLine);
                            o[4 * c + 0] = sum3_f16x2(w0.x, w1.x, w2.x);
                            o[4 * c + 1] = sum3_f16x2(w0.y, w1.y, w2.y);
                            o[4 * c + 2] = sum3_f16x2(w0.z, w1.z, w2.z);
                            o[4 * c + 3] = sum3_f16x2(w0.w, w1.w, w2.w);
                        }
                        tmem_st8(ta + tst + 8 * hq, o);
                    }
                    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(BAR_FULL + (kt & (PF_NBAR - 1))));
                }
            }
            if (!ok) break;
            kg += KS;
            it = itn;
            I = In;
        }
    }

    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols));
    }
}

// x [n][d] (fp32 or bf16) -> fp16, eight values per thread and step.
__global__ void __launch_bounds__(256) tokens_f16_kernel(const void *x, int xdt, int64_t n8,
                                                          uint4 *x16, uint32_t *status) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    bool over = false;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8;
         i += (int64_t)gridDim.x * blockDim.x) {
        float v[8];
        if (xdt == RVQ_BF16) {
            const uint4 w = reinterpret_cast<const uint4 *>(x)[i];
            const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                v[2 * j] = __uint_as_float(u[j] << 16);
                v[2 * j + 1] = __uint_as_float(u[j] & 0xFFFF0000u);
            }
        } else {
            const float4 a = reinterpret_cast<const float4 *>(x)[2 * i];
            const float4 b = reinterpret_cast<const float4 *>(x)[2 * i + 1];
            v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
            v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
        }
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            o[j] = (uint32_t)h_to_f16(v[2 * j], over) |
                   ((uint32_t)h_to_f16(v[2 * j + 1], over) << 16);
        x16[i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (over) set_dev_error(status, RVQ_DEV_ERR_NONFINITE);
    asm volatile("griddepcontrol.launch_dependents;");
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (the
// library does not link the driver library itself).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (fn == nullptr) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

}  // namespace

void *tensor_map_encoder_entry() { return reinterpret_cast<void *>(tensor_map_encoder()); }

rvq_status launch_tokens_f16(const void *x, int xdt, int n, int d, uint16_t *x16,
                             uint32_t *status, cudaStream_t stream, bool pdl) {
    if ((xdt != RVQ_F32 && xdt != RVQ_BF16) || n < 1 || d < 8 || d % 8 != 0 ||
        ((uintptr_t)x & 15u) != 0 || ((uintptr_t)x16 & 15u) != 0) {
        set_error("tokens to fp16: dtype %d, n %d, d %d not supported", xdt, n, d);
        return RVQ_EINVAL;
    }
    const int64_t n8 = (int64_t)n * d / 8;
    const int64_t want = (n8 + 255) / 256;
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
    RVQ_CUDA(cudaLaunchKernelEx(&cfg, tokens_f16_kernel, x, xdt, n8,
                                reinterpret_cast<uint4 *>(x16), status));
    return RVQ_OK;
}

rvq_status launch_prefill_gemm(const PfJob &job, cudaStream_t stream, bool pdl) {
    static std::atomic<int> attr_done[64];  // per device; setting twice is harmless
    int dev = 0;
    RVQ_CUDA(cudaGetDevice(&dev));
    if (dev < 64 && !attr_done[dev]) {
        RVQ_CUDA(cudaFuncSetAttribute(prefill_gemm_kernel<true>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, kPfSmem));
        RVQ_CUDA(cudaFuncSetAttribute(prefill_gemm_kernel<false>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, kPfSmem));
        attr_done[dev] = 1;
    }
    // gate/up items cover 64 weight rows of each matrix, down items 128 rows
    const int want_rows = job.mode == PF_MODE_SWIGLU ? PF_MROWS / 2 : PF_MROWS;
    // gate/up items take two M tiles
    const int tile_mult = job.mode == PF_MODE_SWIGLU ? 2 * job.tile_rows : job.tile_rows;
    if ((job.mode != PF_MODE_SWIGLU && job.mode != PF_MODE_PLAIN) || job.tile_rows != want_rows ||
        job.rows % tile_mult || job.rows / tile_mult > 1023 || job.cols % (4 * PF_KC) ||
        job.E < 1 || job.E > kMaxE || job.min_tokens < 1) {
        set_error("prefill: rows %d / cols %d / tile %d / E %d not supported", job.rows, job.cols,
                  job.tile_rows, job.E);
        return RVQ_EINVAL;
    }
    if (job.x_dtype != PF_H_F16 || ((uintptr_t)job.x & 15u) != 0 || (job.x_stride * 2) % 16 != 0 ||
        job.x_stride < job.cols || job.x_div < 1 || job.n_pairs < 1) {
        set_error("prefill: B input must be fp16 rows of pitch >= %d (16-byte multiple), "
                  "16-byte aligned", job.cols);
        return RVQ_EINVAL;
    }
    // down: B = the pass's contiguous fp16 h rows, loaded by TMA (a 2D map
    // over h: cols x n_pairs rows, pitch x_stride, boxes of 64 columns x
    // kTmaRows rows, 128-byte swizzle; rows past the end read as zero)
    CUtensorMap tmap;
    memset(&tmap, 0, sizeof(tmap));
    if (job.mode == PF_MODE_PLAIN) {
        if (job.x_div != 1) {
            set_error("prefill: down input must be h rows in grouped order");
            return RVQ_EINVAL;
        }
        const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
        if (encode == nullptr) {
            set_error("prefill: cuTensorMapEncodeTiled is not available");
            return RVQ_ECUDA;
        }
        const cuuint64_t dims[2] = {(cuuint64_t)job.cols, (cuuint64_t)job.n_pairs};
        const cuuint64_t strides[1] = {(cuuint64_t)job.x_stride * 2u};
        const cuuint32_t box[2] = {(cuuint32_t)PF_KC, (cuuint32_t)kTmaRows};
        const cuuint32_t estr[2] = {1u, 1u};
        const CUresult r = encode(&tmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                                  const_cast<void *>(job.x), dims, strides, box, estr,
                                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) {
            set_error("prefill: cuTensorMapEncodeTiled failed (%d)", (int)r);
            return RVQ_ECUDA;
        }
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
    if (job.mode == PF_MODE_SWIGLU)
        RVQ_CUDA(cudaLaunchKernelEx(&cfg, prefill_gemm_kernel<true>, job, tmap));
    else
        RVQ_CUDA(cudaLaunchKernelEx(&cfg, prefill_gemm_kernel<false>, job, tmap));
    return RVQ_OK;
}

}  // namespace rvq
