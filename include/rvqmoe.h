/*
 * rvqmoe -- Mixture-of-Experts expert FFN on 3-stage residual-vector-quantised
 * (RVQ) weights, for NVIDIA GB300 (sm_103a).  C ABI.
 *
 * Method (sources are public web pages on the WASTE inference engine):
 *  - Expert weights are coded by 3-stage residual vector quantisation of
 *    8-dimensional sub-vectors with 256-entry codebooks: one uint8 code per
 *    stage per sub-vector, 3.00 bits per weight, no entropy coding
 *    ["WASTE Inference Engine: Running Kimi K3 2.78T on Consumer Hardware",
 *    section "Residual Vector Quantization (RVQ)"; GeekNews topic 32035,
 *    section "Quantization and accuracy"].
 *  - The weight matrix is never materialised: a partial-dot lookup table is
 *    built per codebook and position, T_s[j][k] = <x[8j..8j+7], C_s[k]>, and
 *    each output row is a sum over positions j of three table reads
 *    ["Running a 2.78-Trillion-Parameter Model on a Laptop: Inside WASTE's
 *    NVMe-Streaming Engine", section "Technical Insight"].
 *  - An expert is gate, up and down projection matrices stored together in
 *    one record with its codebooks and a checked header [same page, section
 *    "Technical Insight"; GeekNews topic 32035, section "Disk streaming
 *    structure"]; the router picks 16 experts per layer [GeekNews topic
 *    32035, section "Read-ahead and router prediction"].
 *  Readings where the pages are silent (sub-vectors along the input
 *  dimension, one codebook set per matrix, top-k softmax renormalised over
 *  the selected experts with ties to the lower index, SwiGLU, weighted
 *  combine plus residual) are stated at the calls below.
 *
 * Conventions for every call:
 *  - Pointers marked (dev) are device memory, (host) host memory.  The caller
 *    owns every buffer; the library allocates no device or host buffers (the
 *    tiered expert store's handle and its copy streams, created by
 *    moe_cache_create and released by moe_cache_destroy, are the exception).
 *  - Batch sizes (n tokens) are at least 1: an empty batch is an argument
 *    error (RVQ_EINVAL), so a caller with no tokens skips the call.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream), except where "synchronous" is stated.
 *  - Arguments are checked on the host before anything is launched; a bad
 *    argument returns RVQ_EINVAL (shape, null pointer, range) or RVQ_EALIGN
 *    (a pointer that is not 16-byte aligned) and launches nothing.
 *  - Conditions only the device can see (an expert index outside the bank, a
 *    corrupted record header, a non-finite router logit) set bits of the
 *    status word at the start of the caller's workspace; rvq_ws_status()
 *    reads them.  No call traps, aborts or exits.
 *  - rvq_last_error() returns a thread-local message for the last failure.
 *  - Calls on different streams with different buffers are thread-safe.
 */
#ifndef RVQMOE_H
#define RVQMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *rvq_stream_t; /* identical to cudaStream_t */

typedef enum rvq_status {
    RVQ_OK = 0,
    RVQ_EINVAL = 1,   /* invalid argument (shape, range, null pointer)          */
    RVQ_EALIGN = 2,   /* pointer not 16-byte aligned                             */
    RVQ_ENOMEM = 3,   /* caller-provided workspace or buffer too small           */
    RVQ_ECORRUPT = 4, /* bank record header failed validation                    */
    RVQ_EDEVICE = 5,  /* a kernel flagged a bad index or non-finite input        */
    RVQ_ETIMEOUT = 6, /* a bounded device-side wait gave up                      */
    RVQ_ECUDA = 7,    /* a CUDA runtime call failed (message in rvq_last_error)  */
    RVQ_ENOTIMPL = 8  /* configuration not supported by this build               */
} rvq_status;

typedef enum rvq_dtype { RVQ_F32 = 0, RVQ_BF16 = 1 } rvq_dtype;

/* Bits of the device status word (first 4 bytes of every workspace). */
#define RVQ_DEV_ERR_INDEX 0x1u    /* expert index / offsets outside range      */
#define RVQ_DEV_ERR_NONFINITE 0x2u /* router logit NaN or infinite             */
#define RVQ_DEV_ERR_CORRUPT 0x4u  /* expert record header mismatch             */
#define RVQ_DEV_ERR_TIMEOUT 0x8u  /* bounded spin-wait expired                 */

/* Bytes at the start of every workspace reserved for the status block. */
#define RVQ_WS_STATUS_BYTES 256u

const char *rvq_status_string(rvq_status s);
const char *rvq_last_error(void);
/* Library version, e.g. 0x000100 for 0.1.0. */
uint32_t rvq_version(void);

/* --------------------------------------------------------------------------
 * Packed code layout ("RVQ tile layout").  A matrix of `rows` x `cols`
 * weights has cols/8 sub-vectors ("chunks") per row and 3 codes per chunk.
 * Requirements: rows % 32 == 0, cols % 512 == 0.  Size: exactly
 * 3 * rows * cols / 8 bytes (3.00 bits per weight).
 *   tile (g, b), g < cols/256 (32-chunk group), b < rows/32 (32-row block),
 *   starts at byte ((g * rows/32) + b) * 3072.  Inside a tile, byte
 *   ((s*2 + h)*32 + l)*16 + i  (stage s < 3, half h < 2, lane l < 32, i < 16)
 *   holds the stage-s code of row 32b + l, chunk 32g + ((16h + i + l) mod 32).
 * The per-row rotation (l) makes the 32 lanes of a warp read 32 different
 * table columns at every step, so shared-memory lookups never conflict.
 *
 * Packed codebook layout: fp32 [3][128][8][2]; element (stage s, entry k,
 * dimension i) sits at ((s*128 + k/2)*8 + i)*2 + (k & 1), i.e. entries are
 * interleaved in pairs so that two table entries are built per packed
 * fp32x2 FMA.  Size RVQ_CODEBOOK_BYTES.
 * ------------------------------------------------------------------------ */
#define RVQ_CODEBOOK_BYTES 24576u

/* 3 * rows * cols / 8; 0 if rows/cols do not satisfy the layout rules. */
size_t rvq_code_bytes(int32_t rows, int32_t cols);

/* Canonical codes (dev) uint8 [rows][cols/8][3] -> packed codes (dev).
 * dst_bytes must be >= rvq_code_bytes(rows, cols).  src and dst must not
 * overlap.  EINVAL on shape, ENOMEM if dst_bytes is short. */
rvq_status rvq_pack(const uint8_t *codes_dev, int32_t rows, int32_t cols,
                    uint8_t *packed_dev, size_t dst_bytes, rvq_stream_t stream);

/* Inverse of rvq_pack (used by round-trip tests). */
rvq_status rvq_unpack(const uint8_t *packed_dev, int32_t rows, int32_t cols,
                      uint8_t *codes_dev, size_t dst_bytes, rvq_stream_t stream);

/* Canonical codebooks (dev) fp32 [3][256][8] -> packed codebooks (dev). */
rvq_status rvq_pack_codebooks(const float *cb_dev, float *cb_packed_dev, rvq_stream_t stream);

/* --------------------------------------------------------------------------
 * Partial-dot lookup table, "per codebook and position" [starlog page,
 * "Technical Insight"]: lut[t][j][s][k] = sum_{i<8} x[t][8j+i] * C_s[k][i]
 * for every token t < n, chunk j < cols/8, stage s < 3, entry k < 256, fp32.
 * codebooks: canonical fp32 [3][256][8] (dev); x: [n][cols] of xdt (dev);
 * lut: fp32 [n][cols/8][3][256] (dev).  cols % 8 == 0.  The fused GEMV and
 * FFN calls build the same table tile by tile in shared memory and never
 * write it out; this call exists to expose and test that step on its own.
 * ------------------------------------------------------------------------ */
rvq_status rvq_lut_build(const float *codebooks_dev, const void *x_dev, rvq_dtype xdt,
                         int32_t n, int32_t cols, float *lut_dev, rvq_stream_t stream);

/* --------------------------------------------------------------------------
 * One RVQ matrix times n input vectors, on the codes directly:
 * y[t][r] = sum_j sum_s T^t_s[j][code(r,j,s)] (== W x with W the residual
 * decode) [agentlenshq page, "Residual Vector Quantization (RVQ)"].
 * packed codes + packed codebooks (dev); x [n][cols] of xdt (dev); y fp32
 * [n][rows] (dev).  Workspace (dev) of at least
 * rvq_gemv_workspace_bytes(rows, cols, n) bytes, 256-byte aligned; its
 * status block must have been cleared once with rvq_ws_clear().
 * ------------------------------------------------------------------------ */
size_t rvq_gemv_workspace_bytes(int32_t rows, int32_t cols, int32_t n);
rvq_status rvq_gemv(const uint8_t *packed_codes_dev, const float *packed_cb_dev,
                    int32_t rows, int32_t cols, const void *x_dev, rvq_dtype xdt, int32_t n,
                    float *y_dev, void *ws_dev, size_t ws_bytes, rvq_stream_t stream);

/* --------------------------------------------------------------------------
 * rvq_gemv for callers that cannot allocate device memory (for example a
 * plug-in inside a framework that owns all device memory, or a loop where an
 * allocation and its implicit synchronisation are not allowed).  The source
 * pages have no counterpart to this call; it is an addition of this library.
 * Same operation, arguments, layouts and results as rvq_gemv, without the
 * workspace: the split-K scratch is a fixed RVQ_NOALLOC_SCRATCH_BYTES device
 * array inside the library, held by every GPU that loads the library until
 * the process exits.  Calls no cudaMalloc/cudaFree or allocating routine.
 *  - Argument checks as rvq_gemv (EINVAL / EALIGN), then RVQ_ENOMEM when
 *    rows x cols x n would need more scratch than the fixed maximum
 *    (rvq_gemv_workspace_bytes > max).  A rejected call launches nothing.
 *  - The first call on a device (and the first after the device's context
 *    was replaced, e.g. by cudaDeviceReset) looks up the array's device
 *    address with that device current; make that first call before any
 *    stream capture.
 *  - Every call shares the one array: calls whose work overlaps on the GPU
 *    (other streams, other threads) race and give wrong results; serialise
 *    them.  Each call clears the status block it needs at the start, so a
 *    call's device status must be read before the next call.
 * rvq_gemv_noalloc_status: synchronous; waits for `stream`, then reads the
 * device status word of the array (what rvq_ws_status reads from a
 * workspace) and returns RVQ_OK, RVQ_EDEVICE, RVQ_ECORRUPT or RVQ_ETIMEOUT,
 * storing the raw bits in *bits_out if not NULL and clearing them.  The
 * single-matrix GEMV reads no expert records, offsets or pair lists and has
 * no bounded waits, so its launches detect no device-side error and the word
 * reads 0 after them; the call is there so that a caller never has to assume
 * that (and reads any bit a later kernel of the path might set).
 * ------------------------------------------------------------------------ */
#define RVQ_NOALLOC_SCRATCH_BYTES 4194304u /* 4 MiB */
rvq_status rvq_gemv_noalloc(const uint8_t *packed_codes_dev, const float *packed_cb_dev,
                            int32_t rows, int32_t cols, const void *x_dev, rvq_dtype xdt,
                            int32_t n, float *y_dev, rvq_stream_t stream);
rvq_status rvq_gemv_noalloc_status(uint32_t *bits_out, rvq_stream_t stream);

/* --------------------------------------------------------------------------
 * Offline RVQ encoder: the pages' conversion step (GeekNews topic 32035,
 * "Quantization and accuracy", "Conversion": every expert matrix is encoded
 * once, offline, into 3 x 256 codewords of 8 dimensions).  Residual k-means,
 * one stage at a time: codebook = the residual sub-vectors at indices
 * floor(k N / 256) (N = rows * cols / 8, sub-vector i = W[i / (cols/8)]
 * [8 (i % (cols/8)) ..]), then `iters` rounds of nearest codeword (fp32
 * distance, fused multiply-adds in dimension order, ties to the lower index)
 * and mean of each codeword's members (int64 fixed point x 2^32 summed, then
 * divided by the count in double, rounded to fp32), a last assignment for the
 * stage's codes, and the residual minus the chosen codewords.  Reproducible:
 * bit-identical from run to run and to the same steps on the CPU.
 * w fp32 [rows][cols] (dev), |w| < 128, cols % 8 == 0, 256 <= N <= 2^21
 * (N = rows * cols / 8 sub-vectors; the bounds keep the fixed-point member
 * sums inside int64, and a 7168 x 2048 expert matrix is N = 1,835,008);
 * codes uint8 [rows][cols/8][3] and codebooks fp32 [3][256][8] (dev) in the
 * canonical layout rvq_pack / moe_bank_write_expert take; ws of
 * rvq_encode_workspace_bytes(rows, cols) bytes, 256-byte aligned. */
size_t rvq_encode_workspace_bytes(int32_t rows, int32_t cols);
rvq_status rvq_encode(const float *w_dev, int32_t rows, int32_t cols, int32_t iters,
                      uint8_t *codes_dev, float *codebooks_dev, void *ws_dev, size_t ws_bytes,
                      rvq_stream_t stream);

/* --------------------------------------------------------------------------
 * Expert bank: n_experts records of record_bytes each, contiguous in HBM.
 * Record = [rvq_expert_header, 128 B][packed codebooks gate, up, down]
 *          [packed codes gate f x d][up f x d][down d x f]; every part starts
 * on a 128-byte boundary, records on a 256-byte boundary.  gate, up and down
 * of one expert are adjacent, as in the pages' one-read expert record.
 * ------------------------------------------------------------------------ */
#define RVQ_BANK_MAGIC 0x31515652u /* "RVQ1" little-endian */
#define RVQ_HDR_FLAG_CRC32 0x1u    /* header crc32 holds the payload checksum  */

typedef struct rvq_expert_header {
    uint32_t magic;        /* RVQ_BANK_MAGIC                                  */
    uint32_t version;      /* 1                                               */
    int32_t layer;         /* layer id given to moe_bank_init                 */
    int32_t expert;        /* expert id == record index                       */
    int32_t d, f;          /* hidden and intermediate size                    */
    uint32_t flags;        /* RVQ_HDR_FLAG_CRC32 once sealed, else 0          */
    uint32_t crc32;        /* payload checksum once sealed (moe_bank_seal)    */
    uint64_t cb_off;       /* byte offsets from the record start             */
    uint64_t gate_off, up_off, down_off;
    uint64_t record_bytes;
    uint8_t pad[56];
} rvq_expert_header;       /* 128 bytes */

typedef struct rvq_moe_bank {
    uint8_t *base;         /* (dev) first record, 256-byte aligned            */
    uint64_t record_bytes; /* moe_bank_record_bytes(d, f)                     */
    int32_t n_experts, d, f, layer;
} rvq_moe_bank;

uint64_t moe_bank_record_bytes(int32_t d, int32_t f);

/* Fill *bank for a device buffer of `bytes` bytes (host-side only, launches
 * nothing).  d % 512 == 0, f % 512 == 0, 1 <= n_experts <= 256.  ENOMEM if
 * bytes < n_experts * record_bytes. */
rvq_status moe_bank_init(rvq_moe_bank *bank, uint8_t *base_dev, uint64_t bytes,
                         int32_t n_experts, int32_t d, int32_t f, int32_t layer);

/* Write one expert record: packs canonical codes (dev) gate/up [f][d/8][3],
 * down [d][f/8][3] and canonical codebooks (dev) fp32 [3 matrices][3][256][8]
 * (gate, up, down), and writes the header. */
rvq_status moe_bank_write_expert(const rvq_moe_bank *bank, int32_t expert,
                                 const uint8_t *gate_codes_dev, const uint8_t *up_codes_dev,
                                 const uint8_t *down_codes_dev, const float *codebooks_dev,
                                 rvq_stream_t stream);

/* Synchronous: copies every record header to the host and checks magic,
 * version, layer, expert id, shape and offset ranges.  ECORRUPT on mismatch
 * (message names the first bad record). */
rvq_status moe_bank_validate(const rvq_moe_bank *bank, rvq_stream_t stream);

/* Payload checksums: the pages' opt-in CRC check of each expert record
 * (GeekNews topic 32035, "Disk streaming structure").  CRC-32 (ISO-HDLC:
 * reflected polynomial 0xEDB88320, register preset to all ones, result
 * complemented) over each record's bytes [128, record_bytes), computed on the
 * device, one block per record.  Both calls are asynchronous on `stream`.
 *  - moe_bank_seal writes the value to every header (crc32) and sets
 *    RVQ_HDR_FLAG_CRC32.  Seal after the last moe_bank_write_expert (a write
 *    replaces the header and so clears the seal of that record).
 *  - moe_bank_verify recomputes it.  crc_dev (uint32 [n_experts], dev, or
 *    NULL) receives the computed values; a sealed record whose value differs
 *    sets RVQ_DEV_ERR_CORRUPT in the status word of ws_dev (ws_bytes >=
 *    RVQ_WS_STATUS_BYTES; read it with rvq_ws_status; the call does not clear
 *    it).  Unsealed records are only reported in crc_dev.
 * One pass reads the whole bank (4.2 GB for 256 K3-shaped experts), so the
 * check is an explicit pass, not part of the layer call. */
rvq_status moe_bank_seal(const rvq_moe_bank *bank, rvq_stream_t stream);
rvq_status moe_bank_verify(const rvq_moe_bank *bank, uint32_t *crc_dev, void *ws_dev,
                           size_t ws_bytes, rvq_stream_t stream);

/* --------------------------------------------------------------------------
 * Tiered expert store: the pages' streaming engine with host memory in place
 * of NVMe ("Running a 2.78-Trillion-Parameter Model on a Laptop", "Technical
 * Insight"; GeekNews topic 32035, "Read-ahead and router prediction").  A
 * host-resident bank holds every layer's expert records; an HBM cache of
 * record slots holds recently used ones, keyed by (layer, expert), least
 * recently used replaced first.
 *  - host_bank: pinned host memory (cudaHostAlloc or registered), records
 *    [layer][expert], moe_bank_record_bytes(d, f) each, byte-identical to a
 *    device bank written by moe_bank_write_expert (copy one over).
 *  - slots_dev: device buffer (256-byte aligned) of slots_bytes; it holds
 *    slots_bytes / record_bytes slots.
 *  - slot_map_dev: int32 [n_layers][n_experts] (dev), kept by the cache: the
 *    slot of each resident record, -1 otherwise.  The kernels address records
 *    through it and still check every header (expert id, layer), so a record
 *    that is not resident is reported (RVQ_DEV_ERR_CORRUPT), never used.
 * The cache owns host-side state; calls on one cache must not overlap.
 * ------------------------------------------------------------------------ */
typedef struct rvq_expert_cache rvq_expert_cache;
typedef struct rvq_cache_stats {
    uint64_t hits;          /* routed experts found resident                  */
    uint64_t misses;        /* routed experts copied in on demand             */
    uint64_t prefetched;    /* records copied in by router lookahead          */
    uint64_t prefetch_used; /* of those, later routed while still resident    */
    uint64_t bytes_copied;  /* host -> HBM record bytes                       */
    int32_t slots;
    int32_t pad;
} rvq_cache_stats;
rvq_status moe_cache_create(rvq_expert_cache **cache, const uint8_t *host_bank, int32_t n_layers,
                            int32_t n_experts, int32_t d, int32_t f, uint8_t *slots_dev,
                            uint64_t slots_bytes, int32_t *slot_map_dev);
rvq_status moe_cache_destroy(rvq_expert_cache *cache);
rvq_status moe_cache_stats(const rvq_expert_cache *cache, rvq_cache_stats *stats);
/* The bank view of layer `layer` (base = the slots), e.g. for
 * moe_workspace_bytes. */
rvq_status moe_cache_bank(const rvq_expert_cache *cache, int32_t layer, rvq_moe_bank *bank);
/* One MoE layer on cached records.  Synchronous on the host: after routing it
 * reads the expert counts back to decide the copies.  Router logits -> top-k
 * and grouping -> the routed experts made resident (misses copied
 * host -> HBM on the cache's own copy streams (four, one per slot residue,
 * so several copy engines run at once); `stream` waits for the slots it
 * needs) ->
 * expert FFN on the cached records (lookup tables; tensor cores for groups of
 * >= tc_min_tokens when > 0) -> combine + residual.  Other arguments as in
 * moe_layer_forward_ex, with ws_bytes >= moe_workspace_bytes of the cache's
 * bank view.  Router lookahead: with next_wr_dev non-NULL and lookahead > 0,
 * the next layer's router (next_wr_dev, next_bias_dev) runs on this layer's
 * input (next_logits_dev: fp32 [n][n_experts] scratch, dev), and each
 * token's `lookahead` highest-scoring experts of the next layer are copied in
 * while this layer's FFN runs (never replacing this layer's records; skipped
 * when no slot is free).  ENOMEM when this layer's experts do not fit. */
rvq_status moe_layer_forward_streamed(rvq_expert_cache *cache, int32_t layer,
                                      const float *wr_dev, const float *bias_dev,
                                      const void *x_dev, rvq_dtype xdt, int32_t n, int32_t k,
                                      float *logits_dev, int32_t *topk_idx_dev, float *topk_w_dev,
                                      int32_t *offsets_dev, int32_t *pairs_dev, float *out_dev,
                                      void *ws_dev, size_t ws_bytes, const void *residual_dev,
                                      rvq_dtype rdt, int32_t tc_min_tokens,
                                      const float *next_wr_dev, const float *next_bias_dev,
                                      int32_t lookahead, float *next_logits_dev,
                                      rvq_stream_t stream);

/* --------------------------------------------------------------------------
 * Router.  logits[t][e] = sum_c Wr[e][c] * x[t][c] (+ bias[e]), fp32
 * accumulate.  Wr fp32 [E][d] (dev); bias fp32 [E] (dev) or NULL; x [n][d]
 * of xdt (dev); logits fp32 [n][E] (dev).  1 <= E <= 256, d % 8 == 0.
 * ------------------------------------------------------------------------ */
rvq_status moe_router_logits(const float *wr_dev, const float *bias_dev, const void *x_dev,
                             rvq_dtype xdt, int32_t n, int32_t E, int32_t d,
                             float *logits_dev, rvq_stream_t stream);

/* Top-k selection, weights and token grouping.
 * Selection: the k largest fp32 logits of each token, equal logits ordered by
 * the lower expert index; slots are written in that order.  Weights:
 * w = exp(l - l_max) / sum over the k selected (softmax renormalised over
 * the selection).  Grouping: offsets[E+1] = exclusive prefix of per-expert
 * counts; pairs[n*k] sorted by (expert, token), entry = t*k + slot.
 * topk_idx int32 [n][k], topk_w fp32 [n][k], offsets int32 [E+1], pairs int32
 * [n*k] (all dev).  1 <= k <= min(E, 32), E <= 256, 1 <= n <= moe_route_max_tokens(E).
 * A non-finite logit sets RVQ_DEV_ERR_NONFINITE in the workspace status word
 * (ws >= RVQ_WS_STATUS_BYTES); outputs are then unspecified but in range. */
int32_t moe_route_max_tokens(int32_t E);
rvq_status moe_route(const float *logits_dev, int32_t n, int32_t E, int32_t k,
                     int32_t *topk_idx_dev, float *topk_w_dev, int32_t *offsets_dev,
                     int32_t *pairs_dev, void *ws_dev, size_t ws_bytes, rvq_stream_t stream);

/* --------------------------------------------------------------------------
 * Expert FFN on the grouped pairs: for every pair entry p = t*k + slot with
 * expert e, y_pair[p] = Wd_e (silu(Wg_e x_t) * (Wu_e x_t)), silu(g) =
 * g / (1 + exp(-g)), all matrices evaluated on their RVQ codes through
 * shared-memory lookup tables with fp32 accumulation.  Reads offsets [E+1]
 * and pairs [n*k] from moe_route (dev); x [n][d] of xdt (dev); y_pair fp32
 * [n*k][d] (dev).  Each block checks its expert's record header on read and
 * sets RVQ_DEV_ERR_CORRUPT / RVQ_DEV_ERR_INDEX instead of computing with a bad
 * record.  ws >= moe_workspace_bytes(bank, n, k), 256-byte aligned.
 * ------------------------------------------------------------------------ */
size_t moe_workspace_bytes(const rvq_moe_bank *bank, int32_t n, int32_t k);
rvq_status moe_expert_ffn(const rvq_moe_bank *bank, const void *x_dev, rvq_dtype xdt,
                          int32_t n, int32_t k, const int32_t *offsets_dev,
                          const int32_t *pairs_dev, float *y_pair_dev, void *ws_dev,
                          size_t ws_bytes, rvq_stream_t stream);

/* A starting point for tc_min_tokens, measured on GB300 with K3-shaped
 * experts (d = 7168, f = 2048): at 64 tokens per step a threshold of 6 was
 * the fastest tried (4 and 8 within 4 %), while at 32 tokens the lookup
 * tables alone were fastest; a 2048-token prefill chunk is fastest with every
 * expert on the tensor cores (1).  The crossover depends on the shapes and
 * on the group sizes of the step. */
#define RVQMOE_PREFILL_MIN_TOKENS 6

/* As moe_expert_ffn, with per-expert dispatch to the tensor-core path.
 * Experts whose group holds at least tc_min_tokens tokens are computed by
 * the prefill path: their codes are decoded tile by tile to fp16 on chip
 * (W = C1[c1] + C2[c2] + C3[c3] from fp16 shared-memory codebooks, summed in
 * fp16, held in tensor memory as the MMA's A operand) and multiplied with the
 * tokens converted to fp16 on the tensor cores (tcgen05, fp32 accumulators in
 * TMEM): gate and up GEMMs, h = silu(g) * u rounded to fp16, down GEMM.
 * Results of those experts carry 16-bit rounding (the tests hold them to
 * 2e-2 x RMS).  A token or h value beyond the fp16 range (65504) saturates
 * and sets RVQ_DEV_ERR_NONFINITE.
 * tc_min_tokens <= 0: every expert takes the lookup-table path (identical to
 * moe_expert_ffn); 1: every expert takes the tensor-core path.  A bounded
 * device wait that expires sets RVQ_DEV_ERR_TIMEOUT. */
rvq_status moe_expert_ffn_ex(const rvq_moe_bank *bank, const void *x_dev, rvq_dtype xdt,
                             int32_t n, int32_t k, const int32_t *offsets_dev,
                             const int32_t *pairs_dev, float *y_pair_dev, void *ws_dev,
                             size_t ws_bytes, int32_t tc_min_tokens, rvq_stream_t stream);

/* Weighted combine plus residual: out[t][c] = residual[t][c] +
 * sum_slot topk_w[t][slot] * y_pair[t*k + slot][c], fp32.  residual [n][d]
 * of rdt (dev), out fp32 [n][d] (dev); out may alias residual only if rdt is
 * RVQ_F32. */
rvq_status moe_combine(const float *y_pair_dev, const float *topk_w_dev, int32_t n, int32_t k,
                       int32_t d, const void *residual_dev, rvq_dtype rdt, float *out_dev,
                       rvq_stream_t stream);

/* One whole MoE layer: router logits, routing and grouping, expert FFN and
 * combine, with the last reduction of the FFN fused into the combine.
 * Outputs as the separate calls (logits, topk_idx, topk_w, offsets, pairs,
 * out; all dev).  x is also the residual.  bias may be NULL.
 * ws >= moe_workspace_bytes(bank, n, k).  If `events` is not NULL it must
 * hold MOE_LAYER_EVENTS cudaEvent_t handles, recorded on `stream` before
 * the first kernel and after each kernel (for per-kernel timing). */
#define MOE_LAYER_EVENTS 8
rvq_status moe_layer_forward(const rvq_moe_bank *bank, const float *wr_dev, const float *bias_dev,
                             const void *x_dev, rvq_dtype xdt, int32_t n, int32_t k,
                             float *logits_dev, int32_t *topk_idx_dev, float *topk_w_dev,
                             int32_t *offsets_dev, int32_t *pairs_dev, float *out_dev,
                             void *ws_dev, size_t ws_bytes, void **events,
                             rvq_stream_t stream);

/* As moe_layer_forward, with two additions.
 *  - residual_dev (dtype rdt, [n][d], 16-byte aligned; NULL: x itself) is the
 *    stream the combine adds to: out = residual + sum_slot w * expert(x).  A
 *    layer stack passes the normalised stream as x and the raw stream here.
 *    A bf16 residual must not alias out (EINVAL).
 *  - the per-expert tensor-core dispatch of moe_expert_ffn_ex (tc_min_tokens
 *    <= 0: lookup tables only).  With dispatch the event marks are: 0 start,
 *    1 router logits, 2 routing, 3 lookup-table experts done, 4 tensor-core
 *    gate/up GEMM, 5 tensor-core down GEMM, 6 = 5, 7 combine. */
rvq_status moe_layer_forward_ex(const rvq_moe_bank *bank, const float *wr_dev,
                                const float *bias_dev, const void *x_dev, rvq_dtype xdt, int32_t n,
                                int32_t k, float *logits_dev, int32_t *topk_idx_dev,
                                float *topk_w_dev, int32_t *offsets_dev, int32_t *pairs_dev,
                                float *out_dev, void *ws_dev, size_t ws_bytes,
                                const void *residual_dev, rvq_dtype rdt, int32_t tc_min_tokens,
                                void **events, rvq_stream_t stream);

/* One whole MoE layer with its input and output in host memory, for callers
 * whose tokens arrive from and leave to the host.  The call queues, all on
 * `stream` and asynchronous (synchronise the stream before reading out_host):
 *  - a copy of x_host (n x d of xdt) into x_dev;
 *  - the layer of moe_layer_forward_ex (x is also the residual; no event
 *    marks);
 *  - a copy of out (fp32 n x d) from out_dev back to out_host.
 * A transfer of up to 1 MiB whose host buffer the device maps (pinned memory,
 * which is mapped on systems with unified addressing) at a 16-byte aligned
 * address is made by the call's own kernels: the input by a copy kernel that
 * waits for the preceding kernel on the stream like the layer's kernels, the
 * output by the combine, which writes it to out_host beside out_dev.  The
 * step thus stays one chain of dependent launches.  Larger transfers, and any
 * other host buffer, go through cudaMemcpyAsync: pageable memory works, with
 * the driver's staging.
 * x_dev (dev, >= n x d x sizeof(xdt) bytes, 16-byte aligned) and the other
 * device buffers are the caller's, as in moe_layer_forward_ex.  Every
 * argument is checked before the first copy (EINVAL / EALIGN / ENOMEM,
 * nothing queued). */
rvq_status moe_layer_forward_host(const rvq_moe_bank *bank, const float *wr_dev,
                                  const float *bias_dev, const void *x_host, rvq_dtype xdt,
                                  int32_t n, int32_t k, void *x_dev, float *logits_dev,
                                  int32_t *topk_idx_dev, float *topk_w_dev, int32_t *offsets_dev,
                                  int32_t *pairs_dev, float *out_dev, float *out_host, void *ws_dev,
                                  size_t ws_bytes, int32_t tc_min_tokens, rvq_stream_t stream);

/* A CUDA graph of one layer call, for loops that run the same layer on the
 * same buffers step after step (decode).  moe_layer_graph_create records the
 * launches of moe_layer_forward_ex (x is also the residual; no event marks)
 * once, by stream capture on `stream`, and instantiates them; each
 * moe_layer_graph_launch then runs the whole layer as one graph launch on the
 * stream it is given, without the per-kernel host launch cost.
 *  - x_host and out_host both non-NULL: the graph also holds the copy of
 *    x_host (n x d of xdt) into x_dev before the layer and of out_dev (fp32
 *    n x d) into out_host after it, as moe_layer_forward_host; both NULL: the
 *    layer reads x_dev as it is when the graph runs.  One of them NULL: EINVAL.
 *  - The graph records pointers, not contents: every buffer must outlive the
 *    graph, and each launch reads what they hold when it runs.
 *  - Creating queues no work.  `stream` must be a stream that can be captured
 *    (not the legacy default stream): otherwise RVQ_ECUDA, nothing recorded.
 *  - Arguments are checked as in moe_layer_forward_host before the capture
 *    starts (EINVAL / EALIGN / ENOMEM; *graph_out is set to NULL on error).
 * moe_layer_graph_destroy frees the graph (NULL: no-op); it must not run
 * while a launch of it is pending on a stream that has not been synchronised.
 * The pages have no counterpart: this is how the library replays its launch
 * sequence on the GPU. */
typedef struct rvq_layer_graph rvq_layer_graph;
rvq_status moe_layer_graph_create(const rvq_moe_bank *bank, const float *wr_dev,
                                  const float *bias_dev, const void *x_host, rvq_dtype xdt,
                                  int32_t n, int32_t k, void *x_dev, float *logits_dev,
                                  int32_t *topk_idx_dev, float *topk_w_dev, int32_t *offsets_dev,
                                  int32_t *pairs_dev, float *out_dev, float *out_host, void *ws_dev,
                                  size_t ws_bytes, int32_t tc_min_tokens, rvq_stream_t stream,
                                  rvq_layer_graph **graph_out);
rvq_status moe_layer_graph_launch(const rvq_layer_graph *graph, rvq_stream_t stream);
rvq_status moe_layer_graph_destroy(rvq_layer_graph *graph);

/* A pre-norm layer of a stack in one call: xn = bf16(h / sqrt(mean(h^2) +
 * eps)) row by row (the values moe_rms_norm gives), then moe_layer_forward_ex
 * with x = xn (bf16) and residual = h: out = h + sum_slot w * expert(xn).
 * The stack's reading of the pages' per-layer input (they show no
 * normalisation; the stream grows without bound otherwise).
 *  - h_dev: dtype hdt (fp32 or bf16) [n][d], 16-byte aligned; out may alias an
 *    fp32 h (each element is read before it is written), not a bf16 one.
 *  - xn_dev: bf16 [n][d] (dev, 16-byte aligned), written; must not alias h or
 *    out.
 *  - eps > 0.  Other arguments as in moe_layer_forward_ex (no event marks).
 * For one token the norm runs inside the router launch (every router block
 * derives the same factor; block 0 writes xn), one launch less on the decode
 * critical path; larger batches launch the norm first. */
rvq_status moe_layer_forward_prenorm(const rvq_moe_bank *bank, const float *wr_dev,
                                     const float *bias_dev, const void *h_dev, rvq_dtype hdt,
                                     int32_t n, int32_t k, float eps, uint16_t *xn_dev,
                                     float *logits_dev, int32_t *topk_idx_dev, float *topk_w_dev,
                                     int32_t *offsets_dev, int32_t *pairs_dev, float *out_dev,
                                     void *ws_dev, size_t ws_bytes, int32_t tc_min_tokens,
                                     rvq_stream_t stream);

/* Row-wise RMS normalisation without a gain, the pre-norm of a layer stack:
 * out[t][c] = x[t][c] / sqrt(mean_c x[t][c]^2 + eps), sums in fp32.
 * The pages describe no normalisation: a stack of their layers (router,
 * top-k, RVQ SwiGLU experts, combine + residual) without one grows without
 * bound (the expert FFN is quadratic in its input), so the stack applies
 * this before each layer, as pre-norm transformer blocks do.
 * x: dtype xdt [n][d]; out: dtype odt [n][d]; d % 4 == 0; both 16-byte
 * aligned (EALIGN); eps >= 0; x may alias out only when both are fp32. */
rvq_status moe_rms_norm(const void *x_dev, rvq_dtype xdt, int32_t n, int32_t d, float eps,
                        void *out_dev, rvq_dtype odt, rvq_stream_t stream);

/* Self-test of the failure path of the tensor-core kernel (no counterpart in
 * the pages): launches the prefill GEMM on one zero token routed to expert 0
 * with its MMA role first waiting for an mbarrier arrival that nothing makes.
 * The bounded wait (1 s) expires, every role of every block gives up, the
 * kernel frees its tensor memory and returns; afterwards rvq_ws_status()
 * reports RVQ_ETIMEOUT (bit RVQ_DEV_ERR_TIMEOUT) and the context stays usable.
 * No GPU fault, trap or hang is involved.  ws: as for moe_layer_forward with
 * n = 1, k = 1 (its contents are overwritten).  Synchronises the stream once
 * before the launch. */
rvq_status rvq_selftest_prefill_timeout(const rvq_moe_bank *bank, void *ws_dev, size_t ws_bytes,
                                        rvq_stream_t stream);

/* --------------------------------------------------------------------------
 * Workspace status block.
 * rvq_ws_clear: zero the status block (async).  Call once per workspace.
 * rvq_ws_status: synchronous; waits for `stream`, reads the status word,
 * returns RVQ_OK, RVQ_EDEVICE (index / non-finite), RVQ_ECORRUPT or
 * RVQ_ETIMEOUT, stores the raw bits in *bits_out if not NULL, and clears it.
 * ------------------------------------------------------------------------ */
rvq_status rvq_ws_clear(void *ws_dev, rvq_stream_t stream);
rvq_status rvq_ws_status(void *ws_dev, uint32_t *bits_out, rvq_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* RVQMOE_H */
