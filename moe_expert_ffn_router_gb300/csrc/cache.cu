// Tiered expert store: a host-resident bank of every layer's expert records
// and an HBM cache of record slots, least recently used replaced first, with
// the next layer's router run early to prefetch its experts.
//
// This is the pages' streaming engine with host memory in place of NVMe: the
// whole model does not fit the fast memory, so a bounded cache keyed by
// (layer, expert) holds recently used expert records, a miss reads the
// record in one piece (gate, up and down are adjacent), and the router of the
// next layer evaluated on the current hidden state predicts which experts to
// fetch ahead ["Running a 2.78-Trillion-Parameter Model on a Laptop",
// section "Technical Insight"; GeekNews topic 32035, section "Read-ahead and
// router prediction"].  GB300 form:
//  * host records are pinned; a miss is one cudaMemcpyAsync of the record,
//    the misses spread round-robin over the cache's own copy streams (one
//    stream moved ~176 GB/s of 16.6 MB records over NVLink-C2C; several keep
//    more copy engines busy), and the compute stream waits on the slot's
//    event only when it needs the slot;
//  * the kernels address records through a device slot map
//    (expert -> slot, -1 when absent), and still check each record's header
//    (expert id, layer), so a stale or missing slot is reported as a corrupt
//    record instead of being computed with;
//  * the host reads the layer's routing back once (the expert counts) to
//    decide the copies, as the pages' engine reads the router's choice before
//    issuing its reads.
#include "internal.cuh"

#include <algorithm>
#include <vector>

struct rvq_expert_cache {
    const uint8_t *host;   // [layers][experts][record_bytes], pinned
    int32_t layers, experts, d, f;
    uint64_t rb;
    uint8_t *slots;        // device, n_slots records
    int32_t n_slots;
    int32_t *map_dev;      // device [layers][experts]
    std::vector<int32_t> map;        // host copy: slot of (layer, expert) or -1
    std::vector<int64_t> key;        // slot -> layer * experts + expert, or -1
    std::vector<uint64_t> used;      // slot -> last use (tick)
    std::vector<uint8_t> prefetched; // slot filled by a prefetch and not used since
    std::vector<cudaEvent_t> ready;  // slot -> its last copy
    int32_t *stage = nullptr;        // pinned [layers][experts]: map rows for the device
    int32_t *h_off = nullptr;        // pinned [experts + 1]
    float *h_next = nullptr;         // pinned next-layer logits
    size_t h_next_cap = 0;
    uint64_t tick = 0;
    std::vector<cudaStream_t> copy;  // the cache's copy streams
    int next_copy = 0;
    rvq_cache_stats st = {};
};

namespace rvq {
namespace {

constexpr int kCopyStreams = 4;

// Makes the listed experts of `layer` resident.  pinned: slots that must not
// be replaced (this call's and, for a prefetch, the current layer's); a slot
// this call uses is added.  Misses are copied on the copy stream of their
// slot.  ENOMEM when no slot is
// free to replace (the caller's working set exceeds the cache).
rvq_status cache_acquire(rvq_expert_cache *c, int layer, const std::vector<int> &experts,
                         std::vector<uint8_t> &pinned, bool prefetch,
                         std::vector<int> *slots_out) {
    for (int e : experts) {
        const int64_t k = (int64_t)layer * c->experts + e;
        int s = c->map[(size_t)k];
        if (s >= 0) {
            c->used[(size_t)s] = ++c->tick;
            if (!prefetch) {
                ++c->st.hits;
                if (c->prefetched[(size_t)s]) {
                    ++c->st.prefetch_used;
                    c->prefetched[(size_t)s] = 0;
                }
            }
        } else {
            // an empty slot, else the least recently used one not pinned
            int victim = -1;
            for (int v = 0; v < c->n_slots; ++v) {
                if (pinned[(size_t)v]) continue;
                if (c->key[(size_t)v] < 0) {
                    victim = v;
                    break;
                }
                if (victim < 0 || c->used[(size_t)v] < c->used[(size_t)victim]) victim = v;
            }
            if (victim < 0) {
                if (prefetch) return RVQ_OK;  // a hint: no room, nothing fetched
                set_error("moe_layer_forward_streamed: %d slots cannot hold layer %d's experts",
                          c->n_slots, layer);
                return RVQ_ENOMEM;
            }
            if (c->key[(size_t)victim] >= 0) c->map[(size_t)c->key[(size_t)victim]] = -1;
            // a slot's copies stay on one stream, so a refill is ordered after
            // the slot's previous copy
            const cudaStream_t cp = c->copy[(size_t)victim % c->copy.size()];
            RVQ_CUDA(cudaMemcpyAsync(c->slots + (uint64_t)victim * c->rb,
                                     c->host + (uint64_t)k * c->rb, c->rb,
                                     cudaMemcpyHostToDevice, cp));
            RVQ_CUDA(cudaEventRecord(c->ready[(size_t)victim], cp));
            c->key[(size_t)victim] = k;
            c->map[(size_t)k] = victim;
            c->used[(size_t)victim] = ++c->tick;
            c->prefetched[(size_t)victim] = prefetch ? 1 : 0;
            c->st.bytes_copied += c->rb;
            if (prefetch) ++c->st.prefetched; else ++c->st.misses;
            s = victim;
        }
        pinned[(size_t)s] = 1;
        if (slots_out) slots_out->push_back(s);
    }
    return RVQ_OK;
}

}  // namespace
}  // namespace rvq

using namespace rvq;

extern "C" {

rvq_status moe_cache_create(rvq_expert_cache **out, const uint8_t *host_bank, int32_t n_layers,
                            int32_t n_experts, int32_t d, int32_t f, uint8_t *slots_dev,
                            uint64_t slots_bytes, int32_t *slot_map_dev) {
    if (!out || !host_bank || !slots_dev || !slot_map_dev || n_layers < 1 || n_experts < 1 ||
        n_experts > 256 || d <= 0 || f <= 0 || d % 512 || f % 512) {
        set_error("moe_cache_create: bad arguments (layers %d, experts %d, d %d, f %d)", n_layers,
                  n_experts, d, f);
        return RVQ_EINVAL;
    }
    if (((uintptr_t)slots_dev & 255u) || ((uintptr_t)slot_map_dev & 3u)) {
        set_error("moe_cache_create: slots must be 256-byte aligned");
        return RVQ_EALIGN;
    }
    const uint64_t rb = moe_bank_record_bytes(d, f);
    const uint64_t ns = slots_bytes / rb;
    if (ns < 1 || ns > (1u << 30)) {
        set_error("moe_cache_create: %llu bytes hold no record of %llu bytes",
                  (unsigned long long)slots_bytes, (unsigned long long)rb);
        return RVQ_ENOMEM;
    }
    rvq_expert_cache *c = new rvq_expert_cache();
    c->host = host_bank;
    c->layers = n_layers;
    c->experts = n_experts;
    c->d = d;
    c->f = f;
    c->rb = rb;
    c->slots = slots_dev;
    c->n_slots = (int32_t)ns;
    c->map_dev = slot_map_dev;
    c->map.assign((size_t)n_layers * n_experts, -1);
    c->key.assign((size_t)ns, -1);
    c->used.assign((size_t)ns, 0);
    c->prefetched.assign((size_t)ns, 0);
    c->ready.assign((size_t)ns, nullptr);
    c->st.slots = (int32_t)ns;
    cudaError_t err = cudaSuccess;
    for (size_t s = 0; s < ns && err == cudaSuccess; ++s)
        err = cudaEventCreateWithFlags(&c->ready[s], cudaEventDisableTiming);
    c->copy.assign(kCopyStreams, nullptr);
    for (int i = 0; i < kCopyStreams && err == cudaSuccess; ++i)
        err = cudaStreamCreateWithFlags(&c->copy[(size_t)i], cudaStreamNonBlocking);
    if (err == cudaSuccess)
        err = cudaHostAlloc(&c->stage, sizeof(int32_t) * (size_t)n_layers * n_experts,
                            cudaHostAllocDefault);
    if (err == cudaSuccess)
        err = cudaHostAlloc(&c->h_off, sizeof(int32_t) * (size_t)(n_experts + 1),
                            cudaHostAllocDefault);
    if (err == cudaSuccess) {
        for (size_t i = 0; i < c->map.size(); ++i) c->stage[i] = -1;
        err = cudaMemcpy(slot_map_dev, c->stage, sizeof(int32_t) * c->map.size(),
                         cudaMemcpyHostToDevice);
    }
    if (err != cudaSuccess) {
        set_error("moe_cache_create: %s", cudaGetErrorString(err));
        moe_cache_destroy(c);
        return RVQ_ECUDA;
    }
    *out = c;
    return RVQ_OK;
}

rvq_status moe_cache_destroy(rvq_expert_cache *c) {
    if (!c) return RVQ_OK;
    for (cudaStream_t q : c->copy)
        if (q) cudaStreamSynchronize(q);
    for (cudaEvent_t e : c->ready)
        if (e) cudaEventDestroy(e);
    for (cudaStream_t q : c->copy)
        if (q) cudaStreamDestroy(q);
    if (c->stage) cudaFreeHost(c->stage);
    if (c->h_off) cudaFreeHost(c->h_off);
    if (c->h_next) cudaFreeHost(c->h_next);
    delete c;
    return RVQ_OK;
}

rvq_status moe_cache_stats(const rvq_expert_cache *c, rvq_cache_stats *stats) {
    if (!c || !stats) {
        set_error("moe_cache_stats: null pointer");
        return RVQ_EINVAL;
    }
    *stats = c->st;
    return RVQ_OK;
}

rvq_status moe_cache_bank(const rvq_expert_cache *c, int32_t layer, rvq_moe_bank *bank) {
    if (!c || !bank || layer < 0 || layer >= c->layers) {
        set_error("moe_cache_bank: bad arguments (layer %d)", layer);
        return RVQ_EINVAL;
    }
    bank->base = c->slots;
    bank->record_bytes = c->rb;
    bank->n_experts = c->experts;
    bank->d = c->d;
    bank->f = c->f;
    bank->layer = layer;
    return RVQ_OK;
}

rvq_status moe_layer_forward_streamed(rvq_expert_cache *c, int32_t layer, const float *wr_dev,
                                      const float *bias_dev, const void *x_dev, rvq_dtype xdt,
                                      int32_t n, int32_t k, float *logits_dev,
                                      int32_t *topk_idx_dev, float *topk_w_dev,
                                      int32_t *offsets_dev, int32_t *pairs_dev, float *out_dev,
                                      void *ws_dev, size_t ws_bytes, const void *residual_dev,
                                      rvq_dtype rdt, int32_t tc_min_tokens,
                                      const float *next_wr_dev, const float *next_bias_dev,
                                      int32_t lookahead, float *next_logits_dev,
                                      rvq_stream_t stream) {
    if (!c || layer < 0 || layer >= c->layers || !wr_dev || !x_dev || !logits_dev ||
        !topk_idx_dev || !topk_w_dev || !offsets_dev || !pairs_dev || !out_dev || !ws_dev) {
        set_error("moe_layer_forward_streamed: bad arguments (layer %d)", layer);
        return RVQ_EINVAL;
    }
    const int E = c->experts;
    if (n < 1 || k < 1 || k > E || k > 32 || n > route_max_tokens(E) ||
        (xdt != RVQ_F32 && xdt != RVQ_BF16)) {
        set_error("moe_layer_forward_streamed: n %d, k %d, dtype %d", n, k, (int)xdt);
        return RVQ_EINVAL;
    }
    if (!residual_dev) {
        residual_dev = x_dev;
        rdt = xdt;
    }
    const bool la = next_wr_dev && lookahead > 0 && next_logits_dev && layer + 1 < c->layers;
    rvq_moe_bank B;
    moe_cache_bank(c, layer, &B);
    const FfnPlan P = plan_ffn(B.d, B.f, n * k, E, n);
    if (ws_bytes < P.total || ((uintptr_t)ws_dev & 255u)) {
        set_error("moe_layer_forward_streamed: workspace %zu < %zu or unaligned", ws_bytes,
                  P.total);
        return RVQ_ENOMEM;
    }
    cudaStream_t st = (cudaStream_t)stream;
    uint32_t *status = (uint32_t *)ws_dev;
    // routing
    if (xdt == RVQ_BF16 && router_tc_supported(n, E, B.d))
        RVQ_TRY(launch_router_logits_tc(wr_dev, bias_dev, x_dev, n, E, B.d, logits_dev,
                                        (uint8_t *)ws_dev + P.off_wsplit, status, st));
    else
        RVQ_TRY(launch_router_logits(wr_dev, bias_dev, x_dev, (int)xdt, n, E, B.d, logits_dev,
                                     st));
    RVQ_TRY(launch_route(logits_dev, n, E, k, topk_idx_dev, topk_w_dev, offsets_dev, pairs_dev,
                         status, st, false));
    if (la) {
        // lookahead: the next layer's router on this layer's input
        RVQ_TRY(launch_router_logits(next_wr_dev, next_bias_dev, x_dev, (int)xdt, n, E, B.d,
                                     next_logits_dev, st));
        const size_t need = (size_t)n * E;
        if (c->h_next_cap < need) {
            if (c->h_next) cudaFreeHost(c->h_next);
            c->h_next = nullptr;
            c->h_next_cap = 0;
            RVQ_CUDA(cudaHostAlloc(&c->h_next, sizeof(float) * need, cudaHostAllocDefault));
            c->h_next_cap = need;
        }
        RVQ_CUDA(cudaMemcpyAsync(c->h_next, next_logits_dev, sizeof(float) * need,
                                 cudaMemcpyDeviceToHost, st));
    }
    RVQ_CUDA(cudaMemcpyAsync(c->h_off, offsets_dev, sizeof(int32_t) * (E + 1),
                             cudaMemcpyDeviceToHost, st));
    RVQ_CUDA(cudaStreamSynchronize(st));
    // this layer's experts resident; the compute stream waits for their copies
    std::vector<int> ex, slots;
    for (int e = 0; e < E; ++e)
        if (c->h_off[e + 1] > c->h_off[e]) ex.push_back(e);
    std::vector<uint8_t> pinned((size_t)c->n_slots, 0);
    RVQ_TRY(cache_acquire(c, layer, ex, pinned, false, &slots));
    for (int s : slots) RVQ_CUDA(cudaStreamWaitEvent(st, c->ready[(size_t)s], 0));
    int32_t *row = c->stage + (size_t)layer * E;
    for (int e = 0; e < E; ++e) row[e] = c->map[(size_t)layer * E + e];
    int32_t *map_row = c->map_dev + (size_t)layer * E;
    RVQ_CUDA(cudaMemcpyAsync(map_row, row, sizeof(int32_t) * E, cudaMemcpyHostToDevice, st));
    // the expert FFN on the cached records, then the combine
    if (tc_min_tokens <= 0) {
        RVQ_TRY(run_ffn(&B, x_dev, xdt, n, k, offsets_dev, pairs_dev, ws_dev, P, st, nullptr,
                        false, 0, map_row, c->n_slots));
        float *dpart = (float *)((uint8_t *)ws_dev + P.off_dpart);
        RVQ_TRY(launch_combine(dpart, P.nslot_d, topk_w_dev, n, k, B.d, residual_dev, (int)rdt,
                               out_dev, st, false));
    } else {
        float *ypair = (float *)((uint8_t *)ws_dev + P.off_ypair);
        if (tc_min_tokens != 1) {
            RVQ_TRY(run_ffn(&B, x_dev, xdt, n, k, offsets_dev, pairs_dev, ws_dev, P, st,
                            nullptr, false, tc_min_tokens, map_row, c->n_slots));
            RVQ_TRY(launch_slot_reduce((float *)((uint8_t *)ws_dev + P.off_dpart), n * k,
                                       P.nslot_d, B.d, ypair, st, false));
        }
        RVQ_TRY(run_ffn_tc(&B, x_dev, xdt, n, k, offsets_dev, pairs_dev, ws_dev, P, ypair,
                           tc_min_tokens, st, false, nullptr, map_row, c->n_slots));
        RVQ_TRY(launch_combine(ypair, 1, topk_w_dev, n, k, B.d, residual_dev, (int)rdt, out_dev,
                               st, false));
    }
    if (la) {
        // prefetch the predicted experts of the next layer while this one computes
        std::vector<int> pred;
        std::vector<uint8_t> want((size_t)E, 0);
        const int m = std::min<int>(lookahead, E);
        std::vector<int> order((size_t)E);
        for (int t = 0; t < n; ++t) {
            const float *lg = c->h_next + (size_t)t * E;
            for (int e = 0; e < E; ++e) order[(size_t)e] = e;
            std::partial_sort(order.begin(), order.begin() + m, order.end(), [&](int a, int b) {
                return lg[a] > lg[b] || (lg[a] == lg[b] && a < b);
            });
            for (int i = 0; i < m; ++i) want[(size_t)order[(size_t)i]] = 1;
        }
        for (int e = 0; e < E; ++e)
            if (want[(size_t)e]) pred.push_back(e);
        RVQ_TRY(cache_acquire(c, layer + 1, pred, pinned, true, nullptr));
    }
    return RVQ_OK;
}

}  // extern "C"
