// Internal declarations shared by the rvqmoe CUDA translation units.
// Nothing here is part of the public C ABI (include/rvqmoe.h).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <atomic>

#include "../../include/rvqmoe.h"

namespace rvq {

// ------------------------------------------------------------------ errors
void set_error(const char *fmt, ...);
rvq_status cuda_status(cudaError_t e, const char *what);
#define RVQ_TRY(expr)                              \
    do {                                           \
        rvq_status _s = (expr);                    \
        if (_s != RVQ_OK) return _s;               \
    } while (0)
#define RVQ_CUDA(expr)                                             \
    do {                                                           \
        cudaError_t _e = (expr);                                   \
        if (_e != cudaSuccess) return ::rvq::cuda_status(_e, #expr); \
    } while (0)
#define RVQ_LAUNCHED(what) RVQ_CUDA(cudaGetLastError())
rvq_status check_gemv_args(const char *who, const uint8_t *packed_codes_dev,
                           const float *packed_cb_dev, int32_t rows, int32_t cols,
                           const void *x_dev, rvq_dtype xdt, int32_t n, const float *y_dev);
rvq_status read_status_word(void *status_dev, uint32_t *bits_out, cudaStream_t st);

// ------------------------------------------------------------------ layout
constexpr int kTileRows = 32;          // rows per tile (one per lane)
constexpr int kTileChunks = 32;        // chunks per tile (rotation period)
constexpr int kTileBytes = 3 * 2 * 32 * 16;  // 3072
constexpr int kLutStageBytes = 65536;  // 256 entries x 256 B per stage
constexpr int kLutBytes = 3 * kLutStageBytes;

inline bool packable(int32_t rows, int32_t cols) {
    return rows > 0 && cols > 0 && rows % 32 == 0 && cols % 512 == 0;
}

// Bank record part offsets (bytes from record start).
struct RecordLayout {
    uint64_t cb_off, gate_off, up_off, down_off, record_bytes;
};
RecordLayout record_layout(int32_t d, int32_t f);

// ------------------------------------------------------------- device utils
__device__ __forceinline__ void set_dev_error(uint32_t *status, uint32_t bit) {
    if (status) atomicOr(status, bit);
}

__device__ __forceinline__ uint4 ldg_stream(const void *p) {
    // Code bytes are read once per step: skip L1.
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ float4 ldg_f4(const void *p) {
    return __ldg(reinterpret_cast<const float4 *>(p));
}

// Load 8 consecutive inputs (bf16 or fp32) as fp32.
__device__ __forceinline__ void load8(const void *base, int dtype, int64_t idx, float v[8]) {
    if (dtype == RVQ_BF16) {
        uint4 q = __ldg(reinterpret_cast<const uint4 *>(
            reinterpret_cast<const __nv_bfloat16 *>(base) + idx));
        uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    } else {
        const float *f = reinterpret_cast<const float *>(base) + idx;
        float4 a = __ldg(reinterpret_cast<const float4 *>(f));
        float4 b = __ldg(reinterpret_cast<const float4 *>(f) + 1);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
}

// Four consecutive inputs (fp32 or bf16) at element idx (idx % 4 == 0) as fp32.
__device__ __forceinline__ float4 load4(const void *base, int dtype, int64_t idx) {
    if (dtype == RVQ_BF16) {
        const uint2 q = *reinterpret_cast<const uint2 *>(reinterpret_cast<const uint16_t *>(base) + idx);
        return make_float4(__uint_as_float(q.x << 16), __uint_as_float(q.x & 0xFFFF0000u),
                           __uint_as_float(q.y << 16), __uint_as_float(q.y & 0xFFFF0000u));
    }
    return *reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(base) + idx);
}

// 1 / sqrt(mean(x[row .. row + d)^2) + eps) for a block of 256 threads (red:
// 8 floats of shared memory).  The RMS norm and the router that normalises
// its own input both use it, so they derive the same factor bit for bit.
__device__ __forceinline__ float block_rms_inv(const void *x, int xdt, int64_t row, int d, float eps,
                                               float *red) {
    const int d4 = d >> 2;
    float ss = 0.f;
    for (int c4 = threadIdx.x; c4 < d4; c4 += 256) {
        const float4 v = load4(x, xdt, row + c4 * 4);
        ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) tot += red[w];
    return 1.0f / sqrtf(tot / (float)d + eps);
}

__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(lo)) |
           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(hi)) << 16);
}

__device__ __forceinline__ float load1(const void *base, int dtype, int64_t idx) {
    if (dtype == RVQ_BF16)
        return __uint_as_float(
            (uint32_t)reinterpret_cast<const uint16_t *>(base)[idx] << 16);
    return reinterpret_cast<const float *>(base)[idx];
}

// ------------------------------------------------------- LUT-GEMV job (host)
// One work item of a LUT-GEMV launch, written by the plan kernel.
struct ItemDesc {
    int32_t expert;   // -1: skip (the plan flagged an error)
    int32_t entryA;   // pair entries of the two units
    int32_t entryB;
    int16_t g0;       // first chunk group
    int8_t type;      // 0: two tokens, one group per step; 1: one token, two groups per step
    int8_t pad;
};
static_assert(sizeof(ItemDesc) == 16, "ItemDesc is one 16-byte load");

// One launch of the fused lookup-table GEMV over grouped (token, expert)
// pairs.  See lut_gemv.cu for the item decomposition.
struct LutJob {
    const uint8_t *base;       // bank base (NULL for a single matrix)
    uint64_t record_bytes;     // 0 for a single matrix
    const uint8_t *codes_ptr;  // single matrix: packed codes
    const float *cb_ptr;       // single matrix: packed codebooks
    uint64_t codes_off[2];     // per matrix slot (blockIdx.y)
    uint64_t cb_off[2];
    float *part[2];            // partial outputs [entry][nslot][rows]
    int32_t n_mat;             // 1 or 2 (gate+up)
    int32_t rows, cols;
    int32_t G;                 // cols / 256
    int32_t C;                 // chunk groups per item step run (divides G/2)
    int32_t S;                 // row splits
    int32_t E;                 // experts (1 for single matrix)
    int32_t n_pairs;           // n * k (or n)
    const void *x;             // input rows
    int32_t x_dtype;
    int64_t x_stride;          // elements between input rows
    int32_t x_div;             // input row = entry / x_div
    const int32_t *offsets;    // [E+1] (NULL: single group of n_pairs)
    const int32_t *pairs;      // [n_pairs] (NULL: identity)
    uint32_t *status;
    ItemDesc *desc;            // [items before the row split], from the plan kernel
    int32_t tc_min_tokens;     // > 0: experts with at least this many tokens are left to the
                               // tensor-core path (their items are skipped here)
    // record header check
    int32_t check_header;
    int32_t layer, d, f;
    // interleaved GEMV: 1 when only the inputs (x, or the gate/up partials of
    // a fused SwiGLU) come from the immediately preceding kernel (the pair
    // plan was written two or more launches back),
    // so the first table's codebook and code tiles are requested before the
    // dependency wait
    int32_t early_start;
    // expert cache: record index of expert e = slot_of[e] (< n_records), or
    // -1 when not resident; NULL: record e
    const int32_t *slot_of;
    int32_t n_records;
    // interleaved down GEMV with the SwiGLU reduction fused (sw_g != NULL):
    // a table's inputs h = silu(sum of sw_g) * sum of sw_u over the gate/up
    // launch's sw_nslot split-K slots ([entry][slot][f] each) are computed by
    // the block instead of read from x
    const float *sw_g, *sw_u;
    int32_t sw_nslot;
};
// split-K slots (d / 256) up to which the down GEMV can fuse the reduction
constexpr int kIlSwigluMaxSlots = 32;
// tokens up to which it does: the fused reduction costs every table of the
// down launch a round trip to L2, which outweighs the separate launch it
// saves from 8 tokens on (K3-shaped layer: batch 1 -5 %, batch 8 +1 %,
// batch 16 +2 % per step)
constexpr int kIlSwigluMaxTokens = 4;

__host__ __device__ inline int lut_items(const LutJob &j) { return (j.G / (2 * j.C)) * j.n_pairs * j.S; }

rvq_status launch_lut_gemv(const LutJob &job, cudaStream_t stream, bool pdl);
// One token per unit, table build interleaved with streaming (C == 1 layout:
// one partial slot per chunk group).  pd: per sorted pair {expert | -1, entry}.
rvq_status launch_lut_plan_pairs(const LutJob &job, int4 *pd, cudaStream_t stream, bool pdl);
rvq_status launch_lut_gemv_il(const LutJob &job, const int4 *pd, cudaStream_t stream, bool pdl);
// Descriptors for one or two LUT-GEMV jobs sharing the same grouping.
rvq_status launch_lut_plan(const LutJob &ja, const LutJob *jb, cudaStream_t stream, bool pdl);
rvq_status launch_lut_build(const float *cb, const void *x, int xdt, int n, int cols,
                            float *lut, cudaStream_t stream);
// h[entry][r] = silu(sum_slot gate_part) * sum_slot up_part
rvq_status launch_swiglu_reduce(const float *gpart, const float *upart, int n_pairs, int nslot,
                                int rows, float *h, cudaStream_t stream, bool pdl);
// y[entry][r] = sum_slot part[entry][slot][r]
rvq_status launch_slot_reduce(const float *part, int n_entries, int nslot, int rows, float *y,
                              cudaStream_t stream, bool pdl);
rvq_status launch_rms_norm(const void *x, int xdt, int n, int d, float eps, void *out, int odt,
                           cudaStream_t stream, bool pdl);
// out2 (optional): a second copy of out, e.g. a host buffer the GPU maps
rvq_status launch_combine(const float *ypart, int nslot, const float *w, int n, int k, int d,
                          const void *res, int rdt, float *out, cudaStream_t stream, bool pdl,
                          float *out2 = nullptr);
// bytes (a multiple of 16, both ends 16-byte aligned) copied by a kernel,
// for a host buffer the GPU maps; waits for the preceding kernel of the stream
rvq_status launch_io_copy(const void *src, void *dst, size_t bytes, cudaStream_t stream,
                          bool pdl);
rvq_status launch_router_logits(const float *wr, const float *bias, const void *x, int xdt,
                                int n, int E, int d, float *logits, cudaStream_t stream);
// One token: xn = bf16(h / rms(h)) (written by block 0) and its logits, in one
// launch; the same values as launch_rms_norm followed by launch_router_logits.
rvq_status launch_router_norm_logits(const float *wr, const float *bias, const void *h, int hdt,
                                     int E, int d, float eps, uint16_t *xn, float *logits,
                                     cudaStream_t stream);
// With `plan` (n <= 64 only), the routing block also writes the decode
// GEMV's pair descriptors pd[position] = pair_desc(plan, ...) (the plan's
// tc_min_tokens must be <= 0), so no separate plan launch is needed.
rvq_status launch_route(const float *logits, int n, int E, int k, int32_t *idx, float *w,
                        int32_t *offsets, int32_t *pairs, uint32_t *status,
                        cudaStream_t stream, bool pdl, const LutJob *plan = nullptr,
                        int4 *pd = nullptr);
int route_max_tokens(int E);
rvq_status launch_pack(const uint8_t *src, int rows, int cols, uint8_t *dst, bool unpack,
                       cudaStream_t stream);
rvq_status launch_pack_codebooks(const float *src, float *dst, int count, cudaStream_t stream);
rvq_status launch_write_header(uint8_t *record, const rvq_expert_header &h, cudaStream_t stream);

// ------------------------------------------------- tensor-core (prefill) job
constexpr int PF_MODE_SWIGLU = 0;  // gate/up: A rows interleave gate and up; out = h fp16
constexpr int PF_MODE_PLAIN = 1;   // down: out = y fp32
constexpr int PF_H_F16 = 2;        // PfJob x_dtype: fp16 B rows (tokens for gate/up, h for down)
struct PfJob {
    const uint8_t *base;       // bank
    uint64_t record_bytes;
    uint64_t codes_off[2];     // per matrix slot: gate, up (SWIGLU) or down, down (PLAIN)
    uint64_t cb_off[2];
    int32_t tile_rows;         // weight rows per M tile and matrix: 64 (SWIGLU) or 128 (PLAIN)
    int32_t mode;
    int32_t rows, cols;        // of each matrix
    int32_t E, n_pairs;
    int32_t min_tokens;        // experts with fewer tokens are not this launch's work
    const int32_t *offsets, *pairs;
    const void *x;             // fp16 B rows: x16[entry / x_div] (gate/up) or h[grouped position] (down)
    int32_t x_dtype;
    int64_t x_stride;
    int32_t x_div;
    void *out;                 // gate/up: h bf16 [grouped position][rows]; down: y fp32 [entry][rows]
    uint32_t *status;
    int32_t layer, d, f;       // record header check
    int32_t selftest_stall;    // 1: the MMA role first waits for an arrival nothing makes
    const int32_t *slot_of;    // expert cache (as in LutJob); NULL: record e
    int32_t n_records;
};

// Record index of expert e in the job's bank: its cache slot, or e itself;
// -1 when a cached expert has no valid slot (the caller flags the record).
template <class J>
__device__ __forceinline__ int record_of(const J &job, int e) {
    if (!job.slot_of) return e;
    const int s = job.slot_of[e];
    return (s >= 0 && s < job.n_records) ? s : -1;
}
// The decode GEMV's descriptor of one sorted (expert e, group size ne) pair
// entry: {record index, entry, 0, 0}, or {-1, ...} for a pair the tensor-core
// path takes or one that cannot be used (a bad entry sets RVQ_DEV_ERR_INDEX; a
// missing record or a header that does not match sets RVQ_DEV_ERR_CORRUPT).
__device__ __forceinline__ int4 pair_desc(const LutJob &job, int e, int ne, int entry) {
    int4 d = make_int4(-1, 0, 0, 0);
    if (entry < 0 || entry >= job.n_pairs) {
        set_dev_error(job.status, RVQ_DEV_ERR_INDEX);
        return d;
    }
    if (job.tc_min_tokens > 0 && ne >= job.tc_min_tokens) return d;
    const int rec = record_of(job, e);
    const rvq_expert_header *h = rec < 0 ? nullptr :
        reinterpret_cast<const rvq_expert_header *>(job.base + (uint64_t)rec * job.record_bytes);
    if (rec < 0 ||
        (job.check_header &&
         (h->magic != RVQ_BANK_MAGIC || h->expert != e || h->layer != job.layer || h->d != job.d ||
          h->f != job.f || h->record_bytes != job.record_bytes)))
        set_dev_error(job.status, RVQ_DEV_ERR_CORRUPT);
    else
        d = make_int4(rec, entry, 0, 0);
    return d;
}
rvq_status launch_prefill_gemm(const PfJob &job, cudaStream_t stream, bool pdl);
// tokens x [n][d] (RVQ_F32 or RVQ_BF16) -> fp16 x16 [n][d] for the prefill
// GEMMs; |x| beyond the fp16 range saturates and sets RVQ_DEV_ERR_NONFINITE
rvq_status launch_tokens_f16(const void *x, int xdt, int n, int d, uint16_t *x16,
                             uint32_t *status, cudaStream_t stream, bool pdl);
// offline residual k-means encoder (encode.cu)
size_t encode_workspace_bytes(int rows, int cols);
rvq_status launch_rvq_encode(const float *w, int rows, int cols, int iters, uint8_t *codes,
                             float *codebooks, void *ws, cudaStream_t stream);
// CRC-32 of each record's payload: mode 1 seals the headers, mode 0 verifies
rvq_status launch_record_crc(uint8_t *base, uint64_t record_bytes, int n_records, int mode,
                             uint32_t *crc_out, uint32_t *status, cudaStream_t stream);
// cuTensorMapEncodeTiled (PFN_cuTensorMapEncodeTiled_v12000) or null
void *tensor_map_encoder_entry();
// tensor-core router logits (bf16 tokens, n >= 128, E % 128 == 0, d % 256 == 0):
// splits Wr into three bf16 terms in wsplit (router_tc_split_bytes), then the GEMM
bool router_tc_supported(int n, int E, int d);
size_t router_tc_split_bytes(int E, int d);
rvq_status launch_router_logits_tc(const float *wr, const float *bias, const void *x, int n,
                                   int E, int d, float *logits, void *wsplit, uint32_t *status,
                                   cudaStream_t stream);

// FFN plan: how moe_expert_ffn splits its work (host side, deterministic).
struct FfnPlan {
    int C_gu, S_gu;   // gate/up: chunk groups per item step run, row splits
    int C_d, S_d;     // down
    int nslot_gu, nslot_d;
    size_t off_gpart, off_upart, off_h, off_dpart, off_desc_gu, off_desc_d;
    size_t off_h16, off_ypair;  // tensor-core path: h fp16, y fp32 [pair][d]
    size_t off_x16;             // tensor-core path: the tokens as fp16 [n_tokens][d]
    int n_tokens;               // tokens the x16 region holds
    size_t off_wsplit;          // tensor-core router: Wr as three bf16 terms (0 bytes if unused)
    size_t total;
};
FfnPlan plan_ffn(int d, int f, int n_pairs, int E, int n_tokens = 0);
// The FFN launches of one layer (api.cu): lookup tables (run_ffn) and tensor
// cores (run_ffn_tc).  slot_of / n_records: an expert cache's slot map and
// slot count (NULL: the bank holds record e at index e).
rvq_status run_ffn(const rvq_moe_bank *bank, const void *x_dev, rvq_dtype xdt, int32_t n,
                   int32_t k, const int32_t *offsets_dev, const int32_t *pairs_dev, void *ws_dev,
                   const FfnPlan &P, cudaStream_t st, void **marks, bool pdl,
                   int32_t tc_min_tokens = 0, const int32_t *slot_of = nullptr,
                   int32_t n_records = 0, bool pairs_planned = false);
// Tokens route_kernel takes in one block; only that path can also write the
// decode GEMV's pair plan.
constexpr int kRouteSingleBlockTokens = 64;
// run_ffn takes the interleaved decode GEMV with a per-pair plan for these
// shapes; pairs_planned = the routing launch already wrote that plan.
constexpr int kDecodePairPlanMaxTokens = 16;
static_assert(kDecodePairPlanMaxTokens <= kRouteSingleBlockTokens,
              "every batch with a pair plan must fit the single-block routing launch");
inline bool decode_pair_plan(const FfnPlan &P, int n) {
    return P.C_gu == 1 && P.C_d == 1 && n <= kDecodePairPlanMaxTokens;
}
rvq_status run_ffn_tc(const rvq_moe_bank *bank, const void *x_dev, rvq_dtype xdt, int32_t n,
                      int32_t k, const int32_t *offsets_dev, const int32_t *pairs_dev,
                      void *ws_dev, const FfnPlan &P, float *y_pair, int32_t tc_min_tokens,
                      cudaStream_t st, bool pdl, void *mid_event = nullptr,
                      const int32_t *slot_of = nullptr, int32_t n_records = 0);
int num_sms();

}  // namespace rvq
