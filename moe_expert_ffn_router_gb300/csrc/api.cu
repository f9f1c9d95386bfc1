// extern "C" entry points of librvqmoe (declared in include/rvqmoe.h):
// argument checks, work planning, kernel dispatch.  Host code only.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <vector>

#include <new>

#include "internal.cuh"

namespace rvq {

static thread_local char g_err[512] = "";

void set_error(const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
}

rvq_status cuda_status(cudaError_t e, const char *what) {
    set_error("%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
    return RVQ_ECUDA;
}

RecordLayout record_layout(int32_t d, int32_t f) {
    RecordLayout L;
    const uint64_t code = (uint64_t)3 * (uint64_t)d * (uint64_t)f / 8;  // per matrix
    L.cb_off = sizeof(rvq_expert_header);
    L.gate_off = L.cb_off + 3 * (uint64_t)RVQ_CODEBOOK_BYTES;
    L.up_off = L.gate_off + code;
    L.down_off = L.up_off + code;
    const uint64_t end = L.down_off + code;
    L.record_bytes = (end + 255) / 256 * 256;
    return L;
}

int num_sms() {
    static std::atomic<int> cached[64];  // per device
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 152;
    if (dev < 64 && cached[dev]) return cached[dev];
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
        v = 152;
    if (dev < 64) cached[dev] = v;
    return v;
}

static size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// Choose (C, S) for one LUT-GEMV launch: C chunk groups per step run (G must
// be divisible by 2C), S row splits (rows/32 divisible by S, rows/S <= 2048).
// Cost model: waves x item time, item time = C x (table build + streaming of
// the item's rows), plus the split-K partial traffic.  Deterministic.
static void choose_split(int rows, int cols, int n_pairs, int n_mat, int E, int &C_out,
                         int &S_out) {
    const int G = cols / 256, RB = rows / 32;
    const int sms = num_sms();
    const double build_us = 1.3, sm_bw = 45000.0;  // bytes per microsecond per SM
    // rows streamed per step: one-token items read two groups (192 B/row),
    // two-token items read one (96 B/row).
    const double bytes_row = n_pairs <= E ? 192.0 : 96.0;
    double best = 1e300;
    int bc = 1, bs = 1;
    for (int C = 1; 2 * C <= G; ++C) {
        if (G % (2 * C)) continue;
        for (int S = 1; S <= RB; ++S) {
            if (RB % S) continue;
            const int rs = rows / S;
            if (rs > 2048) continue;
            if (C > 1 && rs > 512) continue;  // shared accumulator limit
            if (rs < 256 && S > 1) continue;
            const double items = (double)(G / (2 * C)) * n_pairs * S * n_mat;
            const double waves = ceil(items / sms);
            const double item_us = C * (build_us + rs * bytes_row / sm_bw);
            const double part_bytes = (double)n_pairs * (G / C) * rows * 4.0 * 2.0 * n_mat;
            const double t = waves * item_us + part_bytes / (sms * sm_bw);
            if (t < best * 0.999) {
                best = t;
                bc = C;
                bs = S;
            }
        }
    }
    C_out = bc;
    S_out = bs;
}

FfnPlan plan_ffn(int d, int f, int n_pairs, int E, int n_tokens) {
    FfnPlan P;
    choose_split(f, d, n_pairs, 2, E, P.C_gu, P.S_gu);
    choose_split(d, f, n_pairs, 1, E, P.C_d, P.S_d);
    P.nslot_gu = (d / 256) / P.C_gu;
    P.nslot_d = (f / 256) / P.C_d;
    size_t off = RVQ_WS_STATUS_BYTES;
    P.off_gpart = off;
    off = align256(off + (size_t)n_pairs * P.nslot_gu * f * 4);
    P.off_upart = off;
    off = align256(off + (size_t)n_pairs * P.nslot_gu * f * 4);
    P.off_h = off;
    off = align256(off + (size_t)n_pairs * f * 4);
    P.off_dpart = off;
    off = align256(off + (size_t)n_pairs * P.nslot_d * d * 4);
    P.off_desc_gu = off;
    off = align256(off + (size_t)((d / 256) / (2 * P.C_gu)) * n_pairs * sizeof(ItemDesc));
    P.off_desc_d = off;
    off = align256(off + (size_t)((f / 256) / (2 * P.C_d)) * n_pairs * sizeof(ItemDesc));
    P.off_h16 = off;
    off = align256(off + (size_t)n_pairs * f * 2);
    P.off_ypair = off;
    off = align256(off + (size_t)n_pairs * d * 4);
    P.off_x16 = off;
    P.n_tokens = n_tokens;
    off = align256(off + (size_t)n_tokens * d * 2);
    P.off_wsplit = off;
    if (router_tc_supported(n_tokens, E, d)) off = align256(off + router_tc_split_bytes(E, d));
    P.total = off;
    return P;
}

static bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace rvq

using namespace rvq;

#define CHECK_ARG(cond, ...)          \
    do {                              \
        if (!(cond)) {                \
            set_error(__VA_ARGS__);   \
            return RVQ_EINVAL;        \
        }                             \
    } while (0)
#define CHECK_ALIGN(p, name)                                               \
    do {                                                                   \
        if (!aligned16(p)) {                                               \
            set_error("%s: pointer %p is not 16-byte aligned", name, (const void *)(p)); \
            return RVQ_EALIGN;                                             \
        }                                                                  \
    } while (0)

extern "C" {

const char *rvq_status_string(rvq_status s) {
    switch (s) {
        case RVQ_OK: return "ok";
        case RVQ_EINVAL: return "invalid argument";
        case RVQ_EALIGN: return "misaligned pointer";
        case RVQ_ENOMEM: return "buffer or workspace too small";
        case RVQ_ECORRUPT: return "corrupt expert record";
        case RVQ_EDEVICE: return "device-detected input error";
        case RVQ_ETIMEOUT: return "device wait timed out";
        case RVQ_ECUDA: return "CUDA error";
        case RVQ_ENOTIMPL: return "not implemented";
    }
    return "unknown status";
}

const char *rvq_last_error(void) { return g_err; }

uint32_t rvq_version(void) { return 0x000100u; }

size_t rvq_code_bytes(int32_t rows, int32_t cols) {
    if (!packable(rows, cols)) return 0;
    return (size_t)3 * (size_t)rows * (size_t)cols / 8;
}

rvq_status rvq_pack(const uint8_t *codes_dev, int32_t rows, int32_t cols, uint8_t *packed_dev,
                    size_t dst_bytes, rvq_stream_t stream) {
    CHECK_ARG(packable(rows, cols), "rvq_pack: rows %d must be a multiple of 32 and cols %d of 512",
              rows, cols);
    CHECK_ARG(codes_dev && packed_dev, "rvq_pack: null pointer");
    CHECK_ALIGN(packed_dev, "rvq_pack: packed");
    if (dst_bytes < rvq_code_bytes(rows, cols)) {
        set_error("rvq_pack: dst_bytes %zu < %zu", dst_bytes, rvq_code_bytes(rows, cols));
        return RVQ_ENOMEM;
    }
    return launch_pack(codes_dev, rows, cols, packed_dev, false, (cudaStream_t)stream);
}

rvq_status rvq_unpack(const uint8_t *packed_dev, int32_t rows, int32_t cols, uint8_t *codes_dev,
                      size_t dst_bytes, rvq_stream_t stream) {
    CHECK_ARG(packable(rows, cols), "rvq_unpack: rows %d must be a multiple of 32 and cols %d of 512",
              rows, cols);
    CHECK_ARG(codes_dev && packed_dev, "rvq_unpack: null pointer");
    CHECK_ALIGN(packed_dev, "rvq_unpack: packed");
    if (dst_bytes < rvq_code_bytes(rows, cols)) {
        set_error("rvq_unpack: dst_bytes %zu < %zu", dst_bytes, rvq_code_bytes(rows, cols));
        return RVQ_ENOMEM;
    }
    return launch_pack(packed_dev, rows, cols, codes_dev, true, (cudaStream_t)stream);
}

rvq_status rvq_pack_codebooks(const float *cb_dev, float *cb_packed_dev, rvq_stream_t stream) {
    CHECK_ARG(cb_dev && cb_packed_dev, "rvq_pack_codebooks: null pointer");
    CHECK_ALIGN(cb_packed_dev, "rvq_pack_codebooks: dst");
    return launch_pack_codebooks(cb_dev, cb_packed_dev, 1, (cudaStream_t)stream);
}

rvq_status rvq_lut_build(const float *codebooks_dev, const void *x_dev, rvq_dtype xdt, int32_t n,
                         int32_t cols, float *lut_dev, rvq_stream_t stream) {
    CHECK_ARG(codebooks_dev && x_dev && lut_dev, "rvq_lut_build: null pointer");
    CHECK_ARG(n >= 1 && cols >= 8 && cols % 8 == 0, "rvq_lut_build: n %d, cols %d", n, cols);
    CHECK_ARG(xdt == RVQ_F32 || xdt == RVQ_BF16, "rvq_lut_build: dtype %d", (int)xdt);
    return launch_lut_build(codebooks_dev, x_dev, (int)xdt, n, cols, lut_dev, (cudaStream_t)stream);
}

size_t rvq_gemv_workspace_bytes(int32_t rows, int32_t cols, int32_t n) {
    if (!packable(rows, cols) || n < 1) return 0;
    int C, S;
    choose_split(rows, cols, n, 1, 1 << 30, C, S);
    const int nslot = (cols / 256) / C;
    const size_t items = (size_t)((cols / 256) / (2 * C)) * n;
    return RVQ_WS_STATUS_BYTES + align256((size_t)n * nslot * rows * 4) +
           align256(items * sizeof(ItemDesc));
}

}  // extern "C"

// Host-side argument checks of rvq_gemv (every one runs before any launch);
// also used by rvq_gemv_noalloc, which has no workspace argument.
rvq_status rvq::check_gemv_args(const char *who, const uint8_t *packed_codes_dev,
                                const float *packed_cb_dev, int32_t rows, int32_t cols,
                                const void *x_dev, rvq_dtype xdt, int32_t n, const float *y_dev) {
    CHECK_ARG(packable(rows, cols), "%s: rows %d must be a multiple of 32 and cols %d of 512", who,
              rows, cols);
    CHECK_ARG(n >= 1, "%s: n %d", who, n);
    CHECK_ARG(packed_codes_dev && packed_cb_dev && x_dev && y_dev, "%s: null pointer", who);
    CHECK_ARG(xdt == RVQ_F32 || xdt == RVQ_BF16, "%s: dtype %d", who, (int)xdt);
    const void *ptrs[3] = {packed_codes_dev, packed_cb_dev, x_dev};
    const char *names[3] = {"codes", "codebooks", "x"};
    for (int i = 0; i < 3; ++i)
        if (!aligned16(ptrs[i])) {
            set_error("%s: %s pointer %p is not 16-byte aligned", who, names[i], ptrs[i]);
            return RVQ_EALIGN;
        }
    return RVQ_OK;
}

// Reads (and, when nonzero, clears) a device status word after the stream's
// work: RVQ_OK, RVQ_ECORRUPT, RVQ_ETIMEOUT or RVQ_EDEVICE.
rvq_status rvq::read_status_word(void *status_dev, uint32_t *bits_out, cudaStream_t st) {
    uint32_t bits = 0;
    RVQ_CUDA(cudaMemcpyAsync(&bits, status_dev, 4, cudaMemcpyDeviceToHost, st));
    RVQ_CUDA(cudaStreamSynchronize(st));
    if (bits_out) *bits_out = bits;
    if (bits) {
        RVQ_CUDA(cudaMemsetAsync(status_dev, 0, 4, st));
        RVQ_CUDA(cudaStreamSynchronize(st));
        set_error("device status bits 0x%x", bits);
        if (bits & RVQ_DEV_ERR_CORRUPT) return RVQ_ECORRUPT;
        if (bits & RVQ_DEV_ERR_TIMEOUT) return RVQ_ETIMEOUT;
        return RVQ_EDEVICE;
    }
    return RVQ_OK;
}

extern "C" {

rvq_status rvq_gemv(const uint8_t *packed_codes_dev, const float *packed_cb_dev, int32_t rows,
                    int32_t cols, const void *x_dev, rvq_dtype xdt, int32_t n, float *y_dev,
                    void *ws_dev, size_t ws_bytes, rvq_stream_t stream) {
    RVQ_TRY(check_gemv_args("rvq_gemv", packed_codes_dev, packed_cb_dev, rows, cols, x_dev, xdt, n,
                            y_dev));
    CHECK_ARG(ws_dev, "rvq_gemv: null workspace");
    CHECK_ALIGN(ws_dev, "rvq_gemv: workspace");
    const size_t need = rvq_gemv_workspace_bytes(rows, cols, n);
    if (ws_bytes < need) {
        set_error("rvq_gemv: workspace %zu < %zu", ws_bytes, need);
        return RVQ_ENOMEM;
    }
    LutJob job = {};
    job.codes_ptr = packed_codes_dev;
    job.cb_ptr = packed_cb_dev;
    job.n_mat = 1;
    job.rows = rows;
    job.cols = cols;
    job.G = cols / 256;
    choose_split(rows, cols, n, 1, 1 << 30, job.C, job.S);
    job.E = 1;
    job.n_pairs = n;
    job.x = x_dev;
    job.x_dtype = (int)xdt;
    job.x_stride = cols;
    job.x_div = 1;
    job.status = (uint32_t *)ws_dev;
    float *part = (float *)((uint8_t *)ws_dev + RVQ_WS_STATUS_BYTES);
    job.part[0] = part;
    job.desc = (ItemDesc *)((uint8_t *)part + align256((size_t)n * (job.G / job.C) * rows * 4));
    cudaStream_t st = (cudaStream_t)stream;
    RVQ_TRY(launch_lut_plan(job, nullptr, st, false));
    RVQ_TRY(launch_lut_gemv(job, st, true));
    return launch_slot_reduce(part, n, job.G / job.C, rows, y_dev, st, true);
}

uint64_t moe_bank_record_bytes(int32_t d, int32_t f) {
    if (d <= 0 || f <= 0 || d % 512 || f % 512) return 0;
    return record_layout(d, f).record_bytes;
}

rvq_status moe_bank_init(rvq_moe_bank *bank, uint8_t *base_dev, uint64_t bytes, int32_t n_experts,
                         int32_t d, int32_t f, int32_t layer) {
    CHECK_ARG(bank && base_dev, "moe_bank_init: null pointer");
    CHECK_ARG(d > 0 && f > 0 && d % 512 == 0 && f % 512 == 0,
              "moe_bank_init: d %d and f %d must be multiples of 512", d, f);
    CHECK_ARG(n_experts >= 1 && n_experts <= 256, "moe_bank_init: n_experts %d", n_experts);
    if (((uintptr_t)base_dev & 255u) != 0) {
        set_error("moe_bank_init: base %p is not 256-byte aligned", (void *)base_dev);
        return RVQ_EALIGN;
    }
    const uint64_t rb = moe_bank_record_bytes(d, f);
    if (bytes < rb * (uint64_t)n_experts) {
        set_error("moe_bank_init: %llu bytes < %d records x %llu", (unsigned long long)bytes,
                  n_experts, (unsigned long long)rb);
        return RVQ_ENOMEM;
    }
    bank->base = base_dev;
    bank->record_bytes = rb;
    bank->n_experts = n_experts;
    bank->d = d;
    bank->f = f;
    bank->layer = layer;
    return RVQ_OK;
}

static rvq_status check_bank(const rvq_moe_bank *bank, const char *who) {
    CHECK_ARG(bank && bank->base, "%s: null bank", who);
    CHECK_ARG(bank->d > 0 && bank->f > 0 && bank->d % 512 == 0 && bank->f % 512 == 0 &&
                  bank->n_experts >= 1 && bank->n_experts <= 256,
              "%s: bad bank shape", who);
    CHECK_ARG(bank->record_bytes == record_layout(bank->d, bank->f).record_bytes,
              "%s: record_bytes %llu does not match d %d, f %d", who,
              (unsigned long long)bank->record_bytes, bank->d, bank->f);
    return RVQ_OK;
}

rvq_status moe_bank_write_expert(const rvq_moe_bank *bank, int32_t expert,
                                 const uint8_t *gate_codes_dev, const uint8_t *up_codes_dev,
                                 const uint8_t *down_codes_dev, const float *codebooks_dev,
                                 rvq_stream_t stream) {
    RVQ_TRY(check_bank(bank, "moe_bank_write_expert"));
    CHECK_ARG(expert >= 0 && expert < bank->n_experts, "moe_bank_write_expert: expert %d", expert);
    CHECK_ARG(gate_codes_dev && up_codes_dev && down_codes_dev && codebooks_dev,
              "moe_bank_write_expert: null pointer");
    const RecordLayout L = record_layout(bank->d, bank->f);
    uint8_t *rec = bank->base + (uint64_t)expert * bank->record_bytes;
    cudaStream_t st = (cudaStream_t)stream;
    RVQ_TRY(launch_pack(gate_codes_dev, bank->f, bank->d, rec + L.gate_off, false, st));
    RVQ_TRY(launch_pack(up_codes_dev, bank->f, bank->d, rec + L.up_off, false, st));
    RVQ_TRY(launch_pack(down_codes_dev, bank->d, bank->f, rec + L.down_off, false, st));
    RVQ_TRY(launch_pack_codebooks(codebooks_dev, (float *)(rec + L.cb_off), 3, st));
    rvq_expert_header h;
    memset(&h, 0, sizeof(h));
    h.magic = RVQ_BANK_MAGIC;
    h.version = 1;
    h.layer = bank->layer;
    h.expert = expert;
    h.d = bank->d;
    h.f = bank->f;
    h.cb_off = L.cb_off;
    h.gate_off = L.gate_off;
    h.up_off = L.up_off;
    h.down_off = L.down_off;
    h.record_bytes = L.record_bytes;
    return launch_write_header(rec, h, st);
}

rvq_status moe_bank_validate(const rvq_moe_bank *bank, rvq_stream_t stream) {
    RVQ_TRY(check_bank(bank, "moe_bank_validate"));
    const RecordLayout L = record_layout(bank->d, bank->f);
    std::vector<rvq_expert_header> hs((size_t)bank->n_experts);
    cudaStream_t st = (cudaStream_t)stream;
    RVQ_CUDA(cudaMemcpy2DAsync(hs.data(), sizeof(rvq_expert_header), bank->base,
                               bank->record_bytes, sizeof(rvq_expert_header), bank->n_experts,
                               cudaMemcpyDeviceToHost, st));
    RVQ_CUDA(cudaStreamSynchronize(st));
    for (int e = 0; e < bank->n_experts; ++e) {
        const rvq_expert_header &h = hs[(size_t)e];
        const char *bad = nullptr;
        if (h.magic != RVQ_BANK_MAGIC) bad = "magic";
        else if (h.version != 1) bad = "version";
        else if (h.expert != e) bad = "expert id";
        else if (h.layer != bank->layer) bad = "layer";
        else if (h.d != bank->d || h.f != bank->f) bad = "shape";
        else if (h.cb_off != L.cb_off || h.gate_off != L.gate_off || h.up_off != L.up_off ||
                 h.down_off != L.down_off || h.record_bytes != L.record_bytes)
            bad = "offset range";
        if (bad) {
            set_error("moe_bank_validate: record %d: bad %s", e, bad);
            return RVQ_ECORRUPT;
        }
    }
    return RVQ_OK;
}

size_t rvq_encode_workspace_bytes(int32_t rows, int32_t cols) {
    if (rows < 1 || cols < 8 || cols % 8 || (int64_t)rows * (cols / 8) < 256 ||
        (int64_t)rows * (cols / 8) > (int64_t(1) << 21))
        return 0;
    return encode_workspace_bytes(rows, cols);
}

rvq_status rvq_encode(const float *w_dev, int32_t rows, int32_t cols, int32_t iters,
                      uint8_t *codes_dev, float *codebooks_dev, void *ws_dev, size_t ws_bytes,
                      rvq_stream_t stream) {
    CHECK_ARG(w_dev && codes_dev && codebooks_dev && ws_dev, "rvq_encode: null pointer");
    CHECK_ARG(rows >= 1 && cols >= 8 && cols % 8 == 0 && (int64_t)rows * (cols / 8) >= 256 &&
                  (int64_t)rows * (cols / 8) <= (int64_t(1) << 21) && iters >= 0 && iters <= 1000,
              "rvq_encode: rows %d, cols %d, iters %d", rows, cols, iters);
    CHECK_ALIGN(w_dev, "rvq_encode: w");
    CHECK_ALIGN(codebooks_dev, "rvq_encode: codebooks");
    CHECK_ARG(((uintptr_t)ws_dev & 255u) == 0, "rvq_encode: workspace is not 256-byte aligned");
    if (ws_bytes < encode_workspace_bytes(rows, cols)) {
        set_error("rvq_encode: workspace %zu < %zu", ws_bytes, encode_workspace_bytes(rows, cols));
        return RVQ_ENOMEM;
    }
    return launch_rvq_encode(w_dev, rows, cols, iters, codes_dev, codebooks_dev, ws_dev,
                             (cudaStream_t)stream);
}

rvq_status moe_bank_seal(const rvq_moe_bank *bank, rvq_stream_t stream) {
    RVQ_TRY(check_bank(bank, "moe_bank_seal"));
    return launch_record_crc(bank->base, bank->record_bytes, bank->n_experts, 1, nullptr, nullptr,
                             (cudaStream_t)stream);
}

rvq_status moe_bank_verify(const rvq_moe_bank *bank, uint32_t *crc_dev, void *ws_dev,
                           size_t ws_bytes, rvq_stream_t stream) {
    RVQ_TRY(check_bank(bank, "moe_bank_verify"));
    CHECK_ARG(ws_dev, "moe_bank_verify: null workspace");
    if (ws_bytes < RVQ_WS_STATUS_BYTES) {
        set_error("moe_bank_verify: workspace %zu < %u", ws_bytes, RVQ_WS_STATUS_BYTES);
        return RVQ_ENOMEM;
    }
    return launch_record_crc(bank->base, bank->record_bytes, bank->n_experts, 0, crc_dev,
                             (uint32_t *)ws_dev, (cudaStream_t)stream);
}

rvq_status moe_router_logits(const float *wr_dev, const float *bias_dev, const void *x_dev,
                             rvq_dtype xdt, int32_t n, int32_t E, int32_t d, float *logits_dev,
                             rvq_stream_t stream) {
    CHECK_ARG(wr_dev && x_dev && logits_dev, "moe_router_logits: null pointer");
    CHECK_ARG(n >= 1 && E >= 1 && E <= 256 && d >= 8 && d % 8 == 0,
              "moe_router_logits: n %d, E %d, d %d", n, E, d);
    CHECK_ARG(xdt == RVQ_F32 || xdt == RVQ_BF16, "moe_router_logits: dtype %d", (int)xdt);
    CHECK_ALIGN(wr_dev, "moe_router_logits: Wr");
    CHECK_ALIGN(x_dev, "moe_router_logits: x");
    return launch_router_logits(wr_dev, bias_dev, x_dev, (int)xdt, n, E, d, logits_dev,
                                (cudaStream_t)stream);
}

int32_t moe_route_max_tokens(int32_t E) { return route_max_tokens(E); }

static rvq_status check_route(int32_t n, int32_t E, int32_t k, const char *who) {
    CHECK_ARG(E >= 1 && E <= 256, "%s: E %d", who, E);
    CHECK_ARG(k >= 1 && k <= E && k <= 32, "%s: k %d (E %d)", who, k, E);
    CHECK_ARG(n >= 1 && n <= route_max_tokens(E), "%s: n %d (max %d)", who, n,
              route_max_tokens(E));
    return RVQ_OK;
}

rvq_status moe_route(const float *logits_dev, int32_t n, int32_t E, int32_t k,
                     int32_t *topk_idx_dev, float *topk_w_dev, int32_t *offsets_dev,
                     int32_t *pairs_dev, void *ws_dev, size_t ws_bytes, rvq_stream_t stream) {
    RVQ_TRY(check_route(n, E, k, "moe_route"));
    CHECK_ARG(logits_dev && topk_idx_dev && topk_w_dev && offsets_dev && pairs_dev && ws_dev,
              "moe_route: null pointer");
    if (ws_bytes < RVQ_WS_STATUS_BYTES) {
        set_error("moe_route: workspace %zu < %u", ws_bytes, RVQ_WS_STATUS_BYTES);
        return RVQ_ENOMEM;
    }
    return launch_route(logits_dev, n, E, k, topk_idx_dev, topk_w_dev, offsets_dev, pairs_dev,
                        (uint32_t *)ws_dev, (cudaStream_t)stream, false);
}

size_t moe_workspace_bytes(const rvq_moe_bank *bank, int32_t n, int32_t k) {
    if (!bank || n < 1 || k < 1) return 0;
    if (bank->d <= 0 || bank->f <= 0 || bank->d % 512 || bank->f % 512) return 0;
    return plan_ffn(bank->d, bank->f, n * k, bank->n_experts, n).total;
}

static LutJob ffn_job(const rvq_moe_bank *bank, const RecordLayout &L, int n_pairs, void *ws,
                      const int32_t *slot_of, int32_t n_records) {
    LutJob j = {};
    j.slot_of = slot_of;
    j.n_records = n_records;
    j.base = bank->base;
    j.record_bytes = bank->record_bytes;
    j.E = bank->n_experts;
    j.n_pairs = n_pairs;
    j.status = (uint32_t *)ws;
    j.check_header = 1;
    j.layer = bank->layer;
    j.d = bank->d;
    j.f = bank->f;
    (void)L;
    return j;
}

}  // extern "C"

// item plan -> gate/up LUT-GEMV -> SwiGLU reduction -> down LUT-GEMV; `marks`
// (4 events or NULL) are recorded after each kernel.
rvq_status rvq::run_ffn(const rvq_moe_bank *bank, const void *x_dev, rvq_dtype xdt, int32_t n,
                   int32_t k, const int32_t *offsets_dev, const int32_t *pairs_dev, void *ws_dev,
                   const FfnPlan &P, cudaStream_t st, void **marks, bool pdl,
                   int32_t tc_min_tokens, const int32_t *slot_of, int32_t n_records,
                   bool pairs_planned) {
    auto mark = [&](int i) -> rvq_status {
        if (marks) RVQ_CUDA(cudaEventRecord((cudaEvent_t)marks[i], st));
        return RVQ_OK;
    };
    const RecordLayout L = record_layout(bank->d, bank->f);
    const int np = n * k;
    uint8_t *ws = (uint8_t *)ws_dev;
    float *gpart = (float *)(ws + P.off_gpart);
    float *upart = (float *)(ws + P.off_upart);
    float *h = (float *)(ws + P.off_h);
    float *dpart = (float *)(ws + P.off_dpart);

    LutJob gu = ffn_job(bank, L, np, ws_dev, slot_of, n_records);
    gu.codes_off[0] = L.gate_off;
    gu.codes_off[1] = L.up_off;
    gu.cb_off[0] = L.cb_off;
    gu.cb_off[1] = L.cb_off + RVQ_CODEBOOK_BYTES;
    gu.part[0] = gpart;
    gu.part[1] = upart;
    gu.n_mat = 2;
    gu.rows = bank->f;
    gu.cols = bank->d;
    gu.G = bank->d / 256;
    gu.C = P.C_gu;
    gu.S = P.S_gu;
    gu.x = x_dev;
    gu.x_dtype = (int)xdt;
    gu.x_stride = bank->d;
    gu.x_div = k;
    gu.offsets = offsets_dev;
    gu.pairs = pairs_dev;
    gu.desc = (ItemDesc *)(ws + P.off_desc_gu);

    LutJob dn = ffn_job(bank, L, np, ws_dev, slot_of, n_records);
    dn.codes_off[0] = L.down_off;
    dn.cb_off[0] = L.cb_off + 2 * RVQ_CODEBOOK_BYTES;
    dn.part[0] = dpart;
    dn.n_mat = 1;
    dn.rows = bank->d;
    dn.cols = bank->f;
    dn.G = bank->f / 256;
    dn.C = P.C_d;
    dn.S = P.S_d;
    dn.x = h;
    dn.x_dtype = RVQ_F32;
    dn.x_stride = bank->f;
    dn.x_div = 1;
    dn.offsets = offsets_dev;
    dn.pairs = pairs_dev;
    dn.desc = (ItemDesc *)(ws + P.off_desc_d);
    gu.tc_min_tokens = dn.tc_min_tokens = tc_min_tokens;
    if (decode_pair_plan(P, n)) {
        // decode batches up to 16 tokens: one-token units with the table build
        // interleaved into the streaming (measured faster than two-token items
        // up to 16 tokens, slower from 32); the pair plan reuses the gate/up
        // descriptor space (>= n_pairs x 16 bytes)
        int4 *pd = (int4 *)(ws + P.off_desc_gu);
        if (!pairs_planned) RVQ_TRY(launch_lut_plan_pairs(gu, pd, st, pdl));
        RVQ_TRY(mark(0));
        RVQ_TRY(launch_lut_gemv_il(gu, pd, st, pdl));
        RVQ_TRY(mark(1));
        if (P.nslot_gu <= kIlSwigluMaxSlots && n <= kIlSwigluMaxTokens) {
            // the down launch reduces its tables' inputs h from the gate/up
            // partials itself (no separate SwiGLU launch)
            dn.sw_g = gpart;
            dn.sw_u = upart;
            dn.sw_nslot = P.nslot_gu;
        } else {
            RVQ_TRY(launch_swiglu_reduce(gpart, upart, np, P.nslot_gu, bank->f, h, st, pdl));
        }
        RVQ_TRY(mark(2));
        dn.early_start = 1;  // the plan is two or more launches back; only the inputs are new
        RVQ_TRY(launch_lut_gemv_il(dn, pd, st, pdl));
        return mark(3);
    }
    RVQ_TRY(launch_lut_plan(gu, &dn, st, pdl));
    RVQ_TRY(mark(0));
    RVQ_TRY(launch_lut_gemv(gu, st, pdl));
    RVQ_TRY(mark(1));
    RVQ_TRY(launch_swiglu_reduce(gpart, upart, np, P.nslot_gu, bank->f, h, st, pdl));
    RVQ_TRY(mark(2));
    RVQ_TRY(launch_lut_gemv(dn, st, pdl));
    return mark(3);
}

// Tensor-core (prefill) path for experts with at least tc_min_tokens tokens:
// the tokens to fp16, gate/up GEMMs with the SwiGLU epilogue into h (fp16),
// then the down GEMM writing y fp32 [pair][d] for those experts' pairs.
rvq_status rvq::run_ffn_tc(const rvq_moe_bank *bank, const void *x_dev, rvq_dtype xdt, int32_t n,
                      int32_t k, const int32_t *offsets_dev, const int32_t *pairs_dev,
                      void *ws_dev, const FfnPlan &P, float *y_pair, int32_t tc_min_tokens,
                      cudaStream_t st, bool pdl, void *mid_event, const int32_t *slot_of,
                      int32_t n_records) {
    const RecordLayout L = record_layout(bank->d, bank->f);
    uint8_t *ws = (uint8_t *)ws_dev;
    if (P.n_tokens < n) {
        set_error("tensor-core FFN: workspace plan for %d tokens, called with %d", P.n_tokens, n);
        return RVQ_EINVAL;
    }
    // both GEMMs run on fp16 operands: the tokens are converted once
    uint16_t *x16 = (uint16_t *)(ws + P.off_x16);
    RVQ_TRY(launch_tokens_f16(x_dev, (int)xdt, n, bank->d, x16, (uint32_t *)ws_dev, st, pdl));
    PfJob g = {};
    g.base = bank->base;
    g.slot_of = slot_of;
    g.n_records = n_records;
    g.record_bytes = bank->record_bytes;
    g.codes_off[0] = L.gate_off;
    g.codes_off[1] = L.up_off;
    g.cb_off[0] = L.cb_off;
    g.cb_off[1] = L.cb_off + RVQ_CODEBOOK_BYTES;
    g.tile_rows = 64;
    g.mode = PF_MODE_SWIGLU;
    g.rows = bank->f;
    g.cols = bank->d;
    g.E = bank->n_experts;
    g.n_pairs = n * k;
    g.min_tokens = tc_min_tokens;
    g.offsets = offsets_dev;
    g.pairs = pairs_dev;
    g.x = x16;
    g.x_dtype = PF_H_F16;
    g.x_stride = bank->d;
    g.x_div = k;
    g.out = ws + P.off_h16;
    g.status = (uint32_t *)ws_dev;
    g.layer = bank->layer;
    g.d = bank->d;
    g.f = bank->f;
    RVQ_TRY(launch_prefill_gemm(g, st, pdl));
    if (mid_event) RVQ_CUDA(cudaEventRecord((cudaEvent_t)mid_event, st));
    PfJob dn = g;
    dn.codes_off[0] = dn.codes_off[1] = L.down_off;
    dn.cb_off[0] = dn.cb_off[1] = L.cb_off + 2 * RVQ_CODEBOOK_BYTES;
    dn.tile_rows = 128;
    dn.mode = PF_MODE_PLAIN;
    dn.rows = bank->d;
    dn.cols = bank->f;
    dn.x = ws + P.off_h16;
    dn.x_dtype = PF_H_F16;
    dn.x_stride = bank->f;
    dn.x_div = 1;
    dn.out = y_pair;
    return launch_prefill_gemm(dn, st, pdl);
}

extern "C" {

static rvq_status check_ffn_args(const rvq_moe_bank *bank, const void *x_dev, rvq_dtype xdt,
                                 int32_t n, int32_t k, void *ws_dev, size_t ws_bytes,
                                 const char *who) {
    RVQ_TRY(check_bank(bank, who));
    RVQ_TRY(check_route(n, bank->n_experts, k, who));
    CHECK_ARG(x_dev && ws_dev, "%s: null pointer", who);
    CHECK_ARG(xdt == RVQ_F32 || xdt == RVQ_BF16, "%s: dtype %d", who, (int)xdt);
    CHECK_ALIGN(x_dev, who);
    if (((uintptr_t)ws_dev & 255u) != 0) {
        set_error("%s: workspace %p is not 256-byte aligned", who, ws_dev);
        return RVQ_EALIGN;
    }
    const size_t need = moe_workspace_bytes(bank, n, k);
    if (ws_bytes < need) {
        set_error("%s: workspace %zu < %zu", who, ws_bytes, need);
        return RVQ_ENOMEM;
    }
    return RVQ_OK;
}

rvq_status moe_expert_ffn_ex(const rvq_moe_bank *bank, const void *x_dev, rvq_dtype xdt,
                             int32_t n, int32_t k, const int32_t *offsets_dev,
                             const int32_t *pairs_dev, float *y_pair_dev, void *ws_dev,
                             size_t ws_bytes, int32_t tc_min_tokens, rvq_stream_t stream) {
    RVQ_TRY(check_ffn_args(bank, x_dev, xdt, n, k, ws_dev, ws_bytes, "moe_expert_ffn"));
    CHECK_ARG(offsets_dev && pairs_dev && y_pair_dev, "moe_expert_ffn: null pointer");
    CHECK_ALIGN(y_pair_dev, "moe_expert_ffn: y_pair");
    const FfnPlan P = plan_ffn(bank->d, bank->f, n * k, bank->n_experts, n);
    cudaStream_t st = (cudaStream_t)stream;
    if (tc_min_tokens != 1) {  // some experts take the lookup-table path
        RVQ_TRY(run_ffn(bank, x_dev, xdt, n, k, offsets_dev, pairs_dev, ws_dev, P, st, nullptr,
                        true, tc_min_tokens > 0 ? tc_min_tokens : 0));
        RVQ_TRY(launch_slot_reduce((float *)((uint8_t *)ws_dev + P.off_dpart), n * k, P.nslot_d,
                                   bank->d, y_pair_dev, st, true));
    }
    if (tc_min_tokens > 0)  // and the rest the tensor-core path (overwrites their y_pair rows)
        RVQ_TRY(run_ffn_tc(bank, x_dev, xdt, n, k, offsets_dev, pairs_dev, ws_dev, P, y_pair_dev,
                           tc_min_tokens, st, true));
    return RVQ_OK;
}

rvq_status moe_expert_ffn(const rvq_moe_bank *bank, const void *x_dev, rvq_dtype xdt, int32_t n,
                          int32_t k, const int32_t *offsets_dev, const int32_t *pairs_dev,
                          float *y_pair_dev, void *ws_dev, size_t ws_bytes, rvq_stream_t stream) {
    return moe_expert_ffn_ex(bank, x_dev, xdt, n, k, offsets_dev, pairs_dev, y_pair_dev, ws_dev,
                             ws_bytes, 0, stream);
}

rvq_status moe_combine(const float *y_pair_dev, const float *topk_w_dev, int32_t n, int32_t k,
                       int32_t d, const void *residual_dev, rvq_dtype rdt, float *out_dev,
                       rvq_stream_t stream) {
    CHECK_ARG(y_pair_dev && topk_w_dev && residual_dev && out_dev, "moe_combine: null pointer");
    CHECK_ARG(n >= 1 && k >= 1 && d >= 4 && d % 4 == 0, "moe_combine: n %d, k %d, d %d", n, k, d);
    CHECK_ARG(rdt == RVQ_F32 || rdt == RVQ_BF16, "moe_combine: dtype %d", (int)rdt);
    CHECK_ALIGN(y_pair_dev, "moe_combine: y_pair");
    CHECK_ALIGN(residual_dev, "moe_combine: residual");
    CHECK_ALIGN(out_dev, "moe_combine: out");
    if (rdt == RVQ_BF16)
        CHECK_ARG((const void *)out_dev != residual_dev, "moe_combine: bf16 residual cannot alias out");
    return launch_combine(y_pair_dev, 1, topk_w_dev, n, k, d, residual_dev, (int)rdt, out_dev,
                          (cudaStream_t)stream, false);
}

rvq_status moe_rms_norm(const void *x_dev, rvq_dtype xdt, int32_t n, int32_t d, float eps,
                        void *out_dev, rvq_dtype odt, rvq_stream_t stream) {
    CHECK_ARG(x_dev && out_dev, "moe_rms_norm: null pointer");
    CHECK_ARG(n >= 1 && d >= 4 && d % 4 == 0, "moe_rms_norm: n %d, d %d", n, d);
    CHECK_ARG((xdt == RVQ_F32 || xdt == RVQ_BF16) && (odt == RVQ_F32 || odt == RVQ_BF16),
              "moe_rms_norm: dtypes %d, %d", (int)xdt, (int)odt);
    CHECK_ARG(eps >= 0.f, "moe_rms_norm: eps %g", (double)eps);
    CHECK_ALIGN(x_dev, "moe_rms_norm: x");
    CHECK_ALIGN(out_dev, "moe_rms_norm: out");
    return launch_rms_norm(x_dev, (int)xdt, n, d, eps, out_dev, (int)odt, (cudaStream_t)stream,
                           false);
}

static rvq_status layer_after_router(const rvq_moe_bank *bank, const void *x_dev, rvq_dtype xdt,
                                     int32_t n, int32_t k, float *logits_dev,
                                     int32_t *topk_idx_dev, float *topk_w_dev,
                                     int32_t *offsets_dev, int32_t *pairs_dev, float *out_dev,
                                     void *ws_dev, const void *residual_dev, rvq_dtype rdt,
                                     int32_t tc_min_tokens, void **events, cudaStream_t st,
                                     const FfnPlan &P, float *out2 = nullptr);

// moe_layer_forward_ex, with out2 (optional) a second copy of the output that
// the combine writes (a host buffer the GPU maps).
static rvq_status layer_forward(const rvq_moe_bank *bank, const float *wr_dev,
                                const float *bias_dev, const void *x_dev, rvq_dtype xdt, int32_t n,
                                int32_t k, float *logits_dev, int32_t *topk_idx_dev,
                                float *topk_w_dev, int32_t *offsets_dev, int32_t *pairs_dev,
                                float *out_dev, void *ws_dev, size_t ws_bytes,
                                const void *residual_dev, rvq_dtype rdt, int32_t tc_min_tokens,
                                void **events, rvq_stream_t stream, float *out2) {
    RVQ_TRY(check_ffn_args(bank, x_dev, xdt, n, k, ws_dev, ws_bytes, "moe_layer_forward"));
    if (!residual_dev) {
        residual_dev = x_dev;
        rdt = xdt;
    }
    CHECK_ARG(rdt == RVQ_F32 || rdt == RVQ_BF16, "moe_layer_forward: residual dtype %d", (int)rdt);
    CHECK_ALIGN(residual_dev, "moe_layer_forward: residual");
    if (rdt == RVQ_BF16)
        CHECK_ARG((const void *)out_dev != residual_dev,
                  "moe_layer_forward: bf16 residual cannot alias out");
    CHECK_ARG(wr_dev && logits_dev && topk_idx_dev && topk_w_dev && offsets_dev && pairs_dev &&
                  out_dev,
              "moe_layer_forward: null pointer");
    CHECK_ALIGN(wr_dev, "moe_layer_forward: Wr");
    CHECK_ALIGN(out_dev, "moe_layer_forward: out");
    if (xdt == RVQ_BF16)
        CHECK_ARG((const void *)out_dev != x_dev, "moe_layer_forward: bf16 x cannot alias out");
    const FfnPlan P = plan_ffn(bank->d, bank->f, n * k, bank->n_experts, n);
    cudaStream_t st = (cudaStream_t)stream;
    const bool pdl = events == nullptr;
    auto mark = [&](int i) -> rvq_status {
        if (events) RVQ_CUDA(cudaEventRecord((cudaEvent_t)events[i], st));
        return RVQ_OK;
    };
    (void)pdl;
    RVQ_TRY(mark(0));
    if (xdt == RVQ_BF16 && router_tc_supported(n, bank->n_experts, bank->d))
        // prefill-sized bf16 batch: the logits GEMM on the tensor cores
        RVQ_TRY(launch_router_logits_tc(wr_dev, bias_dev, x_dev, n, bank->n_experts, bank->d,
                                        logits_dev, (uint8_t *)ws_dev + P.off_wsplit,
                                        (uint32_t *)ws_dev, st));
    else
        RVQ_TRY(launch_router_logits(wr_dev, bias_dev, x_dev, (int)xdt, n, bank->n_experts,
                                     bank->d, logits_dev, st));
    RVQ_TRY(mark(1));
    return layer_after_router(bank, x_dev, xdt, n, k, logits_dev, topk_idx_dev, topk_w_dev,
                              offsets_dev, pairs_dev, out_dev, ws_dev, residual_dev, rdt,
                              tc_min_tokens, events, st, P, out2);
}

rvq_status moe_layer_forward_ex(const rvq_moe_bank *bank, const float *wr_dev,
                                const float *bias_dev, const void *x_dev, rvq_dtype xdt, int32_t n,
                                int32_t k, float *logits_dev, int32_t *topk_idx_dev,
                                float *topk_w_dev, int32_t *offsets_dev, int32_t *pairs_dev,
                                float *out_dev, void *ws_dev, size_t ws_bytes,
                                const void *residual_dev, rvq_dtype rdt, int32_t tc_min_tokens,
                                void **events, rvq_stream_t stream) {
    return layer_forward(bank, wr_dev, bias_dev, x_dev, xdt, n, k, logits_dev, topk_idx_dev,
                         topk_w_dev, offsets_dev, pairs_dev, out_dev, ws_dev, ws_bytes,
                         residual_dev, rdt, tc_min_tokens, events, stream, nullptr);
}

// Routing, expert FFN and combine of a layer whose logits are computed.
static rvq_status layer_after_router(const rvq_moe_bank *bank, const void *x_dev, rvq_dtype xdt,
                                     int32_t n, int32_t k, float *logits_dev,
                                     int32_t *topk_idx_dev, float *topk_w_dev,
                                     int32_t *offsets_dev, int32_t *pairs_dev, float *out_dev,
                                     void *ws_dev, const void *residual_dev, rvq_dtype rdt,
                                     int32_t tc_min_tokens, void **events, cudaStream_t st,
                                     const FfnPlan &P, float *out2) {
    const bool pdl = events == nullptr;
    auto mark = [&](int i) -> rvq_status {
        if (events) RVQ_CUDA(cudaEventRecord((cudaEvent_t)events[i], st));
        return RVQ_OK;
    };
    // decode batches on the lookup-table path: the routing block also writes
    // the GEMV's pair plan (one launch less on the critical path)
    const bool fuse_plan = tc_min_tokens <= 0 && decode_pair_plan(P, n);
    LutJob plan = {};
    if (fuse_plan)
        plan = ffn_job(bank, record_layout(bank->d, bank->f), n * k, ws_dev, nullptr, 0);
    RVQ_TRY(launch_route(logits_dev, n, bank->n_experts, k, topk_idx_dev, topk_w_dev, offsets_dev,
                         pairs_dev, (uint32_t *)ws_dev, st, pdl, fuse_plan ? &plan : nullptr,
                         fuse_plan ? (int4 *)((uint8_t *)ws_dev + P.off_desc_gu) : nullptr));
    RVQ_TRY(mark(2));
    if (tc_min_tokens <= 0) {
        // lookup-table path only; the down partials are reduced inside the combine
        RVQ_TRY(run_ffn(bank, x_dev, xdt, n, k, offsets_dev, pairs_dev, ws_dev, P, st,
                        events ? events + 3 : nullptr, pdl, 0, nullptr, 0, fuse_plan));
        float *dpart = (float *)((uint8_t *)ws_dev + P.off_dpart);
        RVQ_TRY(launch_combine(dpart, P.nslot_d, topk_w_dev, n, k, bank->d, residual_dev,
                               (int)rdt, out_dev, st, pdl, out2));
        return mark(7);
    }
    // with tensor-core dispatch: marks 3 = lookup-table experts done, 4 = after the
    // tensor-core gate/up GEMM, 5 = after the tensor-core down GEMM, 7 = after the combine
    float *ypair = (float *)((uint8_t *)ws_dev + P.off_ypair);
    if (tc_min_tokens != 1) {
        RVQ_TRY(run_ffn(bank, x_dev, xdt, n, k, offsets_dev, pairs_dev, ws_dev, P, st, nullptr,
                        pdl, tc_min_tokens));
        RVQ_TRY(launch_slot_reduce((float *)((uint8_t *)ws_dev + P.off_dpart), n * k, P.nslot_d,
                                   bank->d, ypair, st, pdl));
    }
    RVQ_TRY(mark(3));
    RVQ_TRY(run_ffn_tc(bank, x_dev, xdt, n, k, offsets_dev, pairs_dev, ws_dev, P, ypair,
                       tc_min_tokens, st, pdl, events ? events[4] : nullptr));
    RVQ_TRY(mark(5));
    RVQ_TRY(mark(6));
    RVQ_TRY(launch_combine(ypair, 1, topk_w_dev, n, k, bank->d, residual_dev, (int)rdt, out_dev,
                           st, pdl, out2));
    return mark(7);
}

// The checks of a layer call whose input and output may live in host memory
// (both host pointers or neither, per `host_needed`), before anything is queued.
static rvq_status check_layer_io(const rvq_moe_bank *bank, const float *wr_dev, const void *x_host,
                                 rvq_dtype xdt, int32_t n, int32_t k, const void *x_dev,
                                 const float *logits_dev, const int32_t *topk_idx_dev,
                                 const float *topk_w_dev, const int32_t *offsets_dev,
                                 const int32_t *pairs_dev, const float *out_dev,
                                 const float *out_host, void *ws_dev, size_t ws_bytes,
                                 bool host_needed, const char *who) {
    CHECK_ARG(bank && x_dev && out_dev, "%s: null pointer", who);
    if (host_needed)
        CHECK_ARG(x_host && out_host, "%s: null host pointer", who);
    else
        CHECK_ARG((x_host == nullptr) == (out_host == nullptr),
                  "%s: x_host and out_host must be given together", who);
    CHECK_ARG(n >= 1 && bank->d > 0, "%s: n %d", who, n);
    CHECK_ARG(xdt == RVQ_F32 || xdt == RVQ_BF16, "%s: dtype %d", who, (int)xdt);
    CHECK_ALIGN(x_dev, who);
    RVQ_TRY(check_ffn_args(bank, x_dev, xdt, n, k, ws_dev, ws_bytes, who));
    CHECK_ARG(wr_dev && logits_dev && topk_idx_dev && topk_w_dev && offsets_dev && pairs_dev,
              "%s: null pointer", who);
    CHECK_ALIGN(out_dev, who);
    if (xdt == RVQ_BF16)
        CHECK_ARG((const void *)out_dev != x_dev, "%s: bf16 x cannot alias out", who);
    return RVQ_OK;
}

// The address at which kernels of this device reach host buffer p, when p is
// pinned memory the device maps (16-byte aligned); NULL otherwise (pageable
// memory, or a mapping the device cannot use).
static void *mapped_host(const void *p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        (void)cudaGetLastError();  // an unknown pointer is not an error here
        return nullptr;
    }
    if (a.type != cudaMemoryTypeHost || !a.devicePointer || ((uintptr_t)a.devicePointer & 15u))
        return nullptr;
    return a.devicePointer;
}

// Largest host transfer a copy kernel makes; larger ones go to the copy engines
// (measured alike for a prefill chunk's tens of MB).
constexpr size_t kIoKernelMaxBytes = size_t(1) << 20;

// x_host -> x_dev, the layer, out_dev -> out_host (the copies only when the
// host pointers are given), all queued on st.
static rvq_status queue_layer_io(const rvq_moe_bank *bank, const float *wr_dev,
                                 const float *bias_dev, const void *x_host, rvq_dtype xdt,
                                 int32_t n, int32_t k, void *x_dev, float *logits_dev,
                                 int32_t *topk_idx_dev, float *topk_w_dev, int32_t *offsets_dev,
                                 int32_t *pairs_dev, float *out_dev, float *out_host, void *ws_dev,
                                 size_t ws_bytes, int32_t tc_min_tokens, cudaStream_t st) {
    const size_t esz = xdt == RVQ_BF16 ? 2 : 4;
    const size_t xbytes = (size_t)n * bank->d * esz, obytes = (size_t)n * bank->d * 4;
    // up to kIoKernelMaxBytes, a host buffer the GPU maps (pinned) is read by
    // a copy kernel, or written by the combine, inside the call's launch
    // chain; otherwise the copy is a cudaMemcpyAsync
    if (x_host) {
        if (void *xm = xbytes <= kIoKernelMaxBytes ? mapped_host(x_host) : nullptr)
            RVQ_TRY(launch_io_copy(xm, x_dev, xbytes, st, true));
        else
            RVQ_CUDA(cudaMemcpyAsync(x_dev, x_host, xbytes, cudaMemcpyHostToDevice, st));
    }
    // a mapped output is written by the combine itself, beside out_dev
    float *om = out_host && obytes <= kIoKernelMaxBytes ? (float *)mapped_host(out_host) : nullptr;
    RVQ_TRY(layer_forward(bank, wr_dev, bias_dev, x_dev, xdt, n, k, logits_dev, topk_idx_dev,
                          topk_w_dev, offsets_dev, pairs_dev, out_dev, ws_dev, ws_bytes, nullptr,
                          xdt, tc_min_tokens, nullptr, (rvq_stream_t)st, om));
    if (out_host && !om)
        RVQ_CUDA(cudaMemcpyAsync(out_host, out_dev, obytes, cudaMemcpyDeviceToHost, st));
    return RVQ_OK;
}

rvq_status moe_layer_forward_host(const rvq_moe_bank *bank, const float *wr_dev,
                                  const float *bias_dev, const void *x_host, rvq_dtype xdt,
                                  int32_t n, int32_t k, void *x_dev, float *logits_dev,
                                  int32_t *topk_idx_dev, float *topk_w_dev, int32_t *offsets_dev,
                                  int32_t *pairs_dev, float *out_dev, float *out_host, void *ws_dev,
                                  size_t ws_bytes, int32_t tc_min_tokens, rvq_stream_t stream) {
    // every argument of the layer call is checked before the first copy
    RVQ_TRY(check_layer_io(bank, wr_dev, x_host, xdt, n, k, x_dev, logits_dev, topk_idx_dev,
                           topk_w_dev, offsets_dev, pairs_dev, out_dev, out_host, ws_dev, ws_bytes,
                           true, "moe_layer_forward_host"));
    return queue_layer_io(bank, wr_dev, bias_dev, x_host, xdt, n, k, x_dev, logits_dev,
                          topk_idx_dev, topk_w_dev, offsets_dev, pairs_dev, out_dev, out_host,
                          ws_dev, ws_bytes, tc_min_tokens, (cudaStream_t)stream);
}

}  // extern "C"

// An instantiated graph of one layer call (moe_layer_graph_create).
struct rvq_layer_graph {
    cudaGraph_t graph;
    cudaGraphExec_t exec;
};

extern "C" {

rvq_status moe_layer_graph_create(const rvq_moe_bank *bank, const float *wr_dev,
                                  const float *bias_dev, const void *x_host, rvq_dtype xdt,
                                  int32_t n, int32_t k, void *x_dev, float *logits_dev,
                                  int32_t *topk_idx_dev, float *topk_w_dev, int32_t *offsets_dev,
                                  int32_t *pairs_dev, float *out_dev, float *out_host, void *ws_dev,
                                  size_t ws_bytes, int32_t tc_min_tokens, rvq_stream_t stream,
                                  rvq_layer_graph **graph_out) {
    CHECK_ARG(graph_out, "moe_layer_graph_create: null graph_out");
    *graph_out = nullptr;
    RVQ_TRY(check_layer_io(bank, wr_dev, x_host, xdt, n, k, x_dev, logits_dev, topk_idx_dev,
                           topk_w_dev, offsets_dev, pairs_dev, out_dev, out_host, ws_dev, ws_bytes,
                           false, "moe_layer_graph_create"));
    cudaStream_t st = (cudaStream_t)stream;
    // relaxed: the launch helpers may set function attributes on first use
    RVQ_CUDA(cudaStreamBeginCapture(st, cudaStreamCaptureModeRelaxed));
    const rvq_status rc = queue_layer_io(bank, wr_dev, bias_dev, x_host, xdt, n, k, x_dev,
                                         logits_dev, topk_idx_dev, topk_w_dev, offsets_dev,
                                         pairs_dev, out_dev, out_host, ws_dev, ws_bytes,
                                         tc_min_tokens, st);
    cudaGraph_t g = nullptr;
    const cudaError_t ce = cudaStreamEndCapture(st, &g);  // the capture always ends here
    if (rc != RVQ_OK || ce != cudaSuccess) {
        if (g) cudaGraphDestroy(g);
        if (rc != RVQ_OK) return rc;
        set_error("moe_layer_graph_create: stream capture failed: %s", cudaGetErrorString(ce));
        return RVQ_ECUDA;
    }
    cudaGraphExec_t ex = nullptr;
    const cudaError_t ie = cudaGraphInstantiate(&ex, g, 0);
    if (ie != cudaSuccess) {
        cudaGraphDestroy(g);
        set_error("moe_layer_graph_create: cudaGraphInstantiate: %s", cudaGetErrorString(ie));
        return RVQ_ECUDA;
    }
    rvq_layer_graph *lg = new (std::nothrow) rvq_layer_graph{g, ex};
    if (!lg) {
        cudaGraphExecDestroy(ex);
        cudaGraphDestroy(g);
        set_error("moe_layer_graph_create: out of host memory");
        return RVQ_ENOMEM;
    }
    *graph_out = lg;
    return RVQ_OK;
}

rvq_status moe_layer_graph_launch(const rvq_layer_graph *graph, rvq_stream_t stream) {
    CHECK_ARG(graph, "moe_layer_graph_launch: null graph");
    RVQ_CUDA(cudaGraphLaunch(graph->exec, (cudaStream_t)stream));
    return RVQ_OK;
}

rvq_status moe_layer_graph_destroy(rvq_layer_graph *graph) {
    if (!graph) return RVQ_OK;
    const cudaError_t a = cudaGraphExecDestroy(graph->exec);
    const cudaError_t b = cudaGraphDestroy(graph->graph);
    delete graph;
    if (a != cudaSuccess || b != cudaSuccess) {
        set_error("moe_layer_graph_destroy: %s", cudaGetErrorString(a != cudaSuccess ? a : b));
        return RVQ_ECUDA;
    }
    return RVQ_OK;
}

rvq_status moe_layer_forward(const rvq_moe_bank *bank, const float *wr_dev, const float *bias_dev,
                             const void *x_dev, rvq_dtype xdt, int32_t n, int32_t k,
                             float *logits_dev, int32_t *topk_idx_dev, float *topk_w_dev,
                             int32_t *offsets_dev, int32_t *pairs_dev, float *out_dev,
                             void *ws_dev, size_t ws_bytes, void **events, rvq_stream_t stream) {
    return moe_layer_forward_ex(bank, wr_dev, bias_dev, x_dev, xdt, n, k, logits_dev, topk_idx_dev,
                                topk_w_dev, offsets_dev, pairs_dev, out_dev, ws_dev, ws_bytes,
                                nullptr, xdt, 0, events, stream);
}

rvq_status moe_layer_forward_prenorm(const rvq_moe_bank *bank, const float *wr_dev,
                                     const float *bias_dev, const void *h_dev, rvq_dtype hdt,
                                     int32_t n, int32_t k, float eps, uint16_t *xn_dev,
                                     float *logits_dev, int32_t *topk_idx_dev, float *topk_w_dev,
                                     int32_t *offsets_dev, int32_t *pairs_dev, float *out_dev,
                                     void *ws_dev, size_t ws_bytes, int32_t tc_min_tokens,
                                     rvq_stream_t stream) {
    CHECK_ARG(h_dev && xn_dev && wr_dev && logits_dev && topk_idx_dev && topk_w_dev &&
                  offsets_dev && pairs_dev && out_dev,
              "moe_layer_forward_prenorm: null pointer");
    CHECK_ARG(hdt == RVQ_F32 || hdt == RVQ_BF16, "moe_layer_forward_prenorm: h dtype %d", (int)hdt);
    CHECK_ARG(eps > 0.f, "moe_layer_forward_prenorm: eps must be positive");
    CHECK_ALIGN(h_dev, "moe_layer_forward_prenorm: h");
    CHECK_ALIGN(xn_dev, "moe_layer_forward_prenorm: xn");
    CHECK_ARG((const void *)xn_dev != h_dev && (void *)xn_dev != (void *)out_dev,
              "moe_layer_forward_prenorm: xn aliases h or out");
    if (hdt == RVQ_BF16)
        CHECK_ARG((const void *)out_dev != h_dev, "moe_layer_forward_prenorm: bf16 h cannot alias out");
    RVQ_TRY(check_ffn_args(bank, xn_dev, RVQ_BF16, n, k, ws_dev, ws_bytes,
                           "moe_layer_forward_prenorm"));
    CHECK_ALIGN(wr_dev, "moe_layer_forward_prenorm: Wr");
    CHECK_ALIGN(out_dev, "moe_layer_forward_prenorm: out");
    const int d = bank->d;
    const FfnPlan P = plan_ffn(d, bank->f, n * k, bank->n_experts, n);
    cudaStream_t st = (cudaStream_t)stream;
    if (n == 1) {
        // one token: the norm inside the router launch
        RVQ_TRY(launch_router_norm_logits(wr_dev, bias_dev, h_dev, (int)hdt, bank->n_experts, d,
                                          eps, xn_dev, logits_dev, st));
    } else {
        RVQ_TRY(launch_rms_norm(h_dev, (int)hdt, n, d, eps, xn_dev, (int)RVQ_BF16, st, true));
        if (router_tc_supported(n, bank->n_experts, d))
            RVQ_TRY(launch_router_logits_tc(wr_dev, bias_dev, xn_dev, n, bank->n_experts, d,
                                            logits_dev, (uint8_t *)ws_dev + P.off_wsplit,
                                            (uint32_t *)ws_dev, st));
        else
            RVQ_TRY(launch_router_logits(wr_dev, bias_dev, xn_dev, (int)RVQ_BF16, n,
                                         bank->n_experts, d, logits_dev, st));
    }
    return layer_after_router(bank, xn_dev, RVQ_BF16, n, k, logits_dev, topk_idx_dev, topk_w_dev,
                              offsets_dev, pairs_dev, out_dev, ws_dev, h_dev, hdt, tc_min_tokens,
                              nullptr, st, P);
}

rvq_status rvq_selftest_prefill_timeout(const rvq_moe_bank *bank, void *ws_dev, size_t ws_bytes,
                                        rvq_stream_t stream) {
    RVQ_TRY(check_bank(bank, "rvq_selftest_prefill_timeout"));
    CHECK_ARG(ws_dev && ((uintptr_t)ws_dev & 255u) == 0,
              "rvq_selftest_prefill_timeout: workspace must be 256-byte aligned");
    CHECK_ARG(ws_bytes >= moe_workspace_bytes(bank, 1, 1),
              "rvq_selftest_prefill_timeout: workspace %zu < %zu", ws_bytes,
              moe_workspace_bytes(bank, 1, 1));
    const int E = bank->n_experts;
    const FfnPlan P = plan_ffn(bank->d, bank->f, 1, E, 1);
    uint8_t *ws = (uint8_t *)ws_dev;
    cudaStream_t st = (cudaStream_t)stream;
    // one token routed to expert 0: offsets and pairs in the gate partial
    // region, a zero input row in the y region, h16 as the output
    int32_t host[258];
    host[0] = 0;
    for (int e = 1; e <= E; ++e) host[e] = 1;
    host[E + 1] = 0;  // pairs[0]
    int32_t *offsets = (int32_t *)(ws + P.off_gpart);
    RVQ_CUDA(cudaMemcpyAsync(offsets, host, sizeof(int32_t) * (E + 2), cudaMemcpyHostToDevice, st));
    void *x = ws + P.off_ypair;
    RVQ_CUDA(cudaMemsetAsync(x, 0, (size_t)bank->d * 2, st));
    const RecordLayout L = record_layout(bank->d, bank->f);
    PfJob g = {};
    g.base = bank->base;
    g.record_bytes = bank->record_bytes;
    g.codes_off[0] = L.gate_off;
    g.codes_off[1] = L.up_off;
    g.cb_off[0] = L.cb_off;
    g.cb_off[1] = L.cb_off + RVQ_CODEBOOK_BYTES;
    g.tile_rows = 64;
    g.mode = PF_MODE_SWIGLU;
    g.rows = bank->f;
    g.cols = bank->d;
    g.E = E;
    g.n_pairs = 1;
    g.min_tokens = 1;
    g.offsets = offsets;
    g.pairs = offsets + E + 1;
    g.x = x;
    g.x_dtype = PF_H_F16;
    g.x_stride = bank->d;
    g.x_div = 1;
    g.out = ws + P.off_h16;
    g.status = (uint32_t *)ws_dev;
    g.layer = bank->layer;
    g.d = bank->d;
    g.f = bank->f;
    g.selftest_stall = 1;
    // the host array must outlive the copy
    RVQ_CUDA(cudaStreamSynchronize(st));
    return launch_prefill_gemm(g, st, false);
}

rvq_status rvq_ws_clear(void *ws_dev, rvq_stream_t stream) {
    CHECK_ARG(ws_dev, "rvq_ws_clear: null workspace");
    RVQ_CUDA(cudaMemsetAsync(ws_dev, 0, RVQ_WS_STATUS_BYTES, (cudaStream_t)stream));
    return RVQ_OK;
}

rvq_status rvq_ws_status(void *ws_dev, uint32_t *bits_out, rvq_stream_t stream) {
    CHECK_ARG(ws_dev, "rvq_ws_status: null workspace");
    return read_status_word(ws_dev, bits_out, (cudaStream_t)stream);
}

}  // extern "C"
