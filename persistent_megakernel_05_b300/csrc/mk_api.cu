// mk_api.cu -- host runtime behind include/mk.h: validation, scratch and KV-pool
// allocation, the KV tensor map, RoPE table, and the cooperative launch of the
// persistent decode-step kernel (mk_kernel.cuh).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "mk.h"
#include "mk_kernel.cuh"

using mk::bf16;

struct mk_handle {
    int device = 0;
    mk_model_desc desc{};
    std::vector<uint8_t> sliding;
    mk::Plan plan{};
    void* block = nullptr;          // scratch arena
    size_t block_bytes = 0;
    mk::LayerPlan* d_layers = nullptr;
    float* d_gains = nullptr;
    float2* d_rope = nullptr;
    CUtensorMap kv_tmap;            // KV pool tensor map, copied into every launch's parameters
    void* kv = nullptr;
    mk_kv_pool pool{};
    uint32_t epoch = 0;             // tag epoch of the last step (1 .. 2^20 - 1, cycling)
    uint32_t cnt_epoch = 0;         // steps since the counters were last zeroed
    int last_batch = 0;             // batch of the last step (selects the activation format)
    float temperature = 0.f;        // next-token rule: 0 greedy, > 0 Gumbel-max sampling
    int top_k = 0;                  // sampling over the top_k largest logits (0: all)
    uint64_t seed = 0;
    long long timeout_ns = 1000000000LL;
    int skip_publish = -1;
    int prefetch_slots = mk::kDefaultPrefetchSlots;
    int pf_batch = 0;               // batch the shared-prefix groups were declared for (0: none)
    int pf_lead[mk::kMaxBatch] = {};
    int pf_pages[mk::kMaxBatch] = {};
    int num_ctas = 0;
    int hd = 0;
    int64_t weight_bytes = 0;
    size_t counters_words = 0, arrivals_words = 0;
    // mk_decode_step_host: pinned host staging and its device twin, grown on demand
    void* host_stage = nullptr;     // [tokens | positions | seq_lens | page_table], then the outputs
    void* dev_stage = nullptr;      // the same inputs on the device
    size_t stage_bytes = 0;         // capacity of both input areas
    float* dev_logits = nullptr;    // [max_batch][vocab] fp32, allocated on first use
};

namespace {

struct DeviceGuard {  // restores the caller's current device
    int prev = -1;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
        cudaSetDevice(dev);
    }
    ~DeviceGuard() {
        if (prev >= 0) cudaSetDevice(prev);
    }
};

inline int perm_col_host(int k) {
    return (k & ~63) | (((k & 7) >> 1) << 4) | (((k & 63) >> 3) << 1) | (k & 1);
}

mk_status validate_desc(const mk_model_desc* d) {
    if (!d) return MK_ERR_INVALID_ARG;
    if (d->n_layers < 1 || d->n_layers > mk::kMaxLayers) return MK_ERR_INVALID_ARG;
    if (d->d_model < 64 || d->d_model % 64) return MK_ERR_INVALID_ARG;
    if (d->head_dim != 64 && d->head_dim != 128) return MK_ERR_INVALID_ARG;
    if (d->n_q_heads < 1 || d->n_kv_heads < 1 || d->n_q_heads % d->n_kv_heads)
        return MK_ERR_INVALID_ARG;
    const int G = d->n_q_heads / d->n_kv_heads;
    if (G > 8 || G * d->head_dim > 512) return MK_ERR_INVALID_ARG;
    if ((d->n_q_heads * d->head_dim) % 64) return MK_ERR_INVALID_ARG;
    if (d->vocab < 1) return MK_ERR_INVALID_ARG;
    // GEMV rows are split over CTAs in 32-bit arithmetic (rows * CTAs < 2^32, CTAs <= 1024)
    if (d->vocab > (1 << 22) || d->ffn_dim > (1 << 22) || d->d_model > (1 << 22)) return MK_ERR_INVALID_ARG;
    if (d->n_experts < 0 || d->n_experts > mk::kMaxExperts) return MK_ERR_INVALID_ARG;
    if (d->n_experts > 0) {
        // MoE: top-k of E experts, each a SwiGLU of width expert_ffn_dim (one k-chunk)
        if (d->top_k < 1 || d->top_k > d->n_experts || d->top_k > mk::kMaxTopK) return MK_ERR_INVALID_ARG;
        if (d->expert_ffn_dim < 64 || d->expert_ffn_dim % 64 || d->expert_ffn_dim > mk::KCW)
            return MK_ERR_INVALID_ARG;
    } else if (d->ffn_dim < 64 || d->ffn_dim % 64) {
        return MK_ERR_INVALID_ARG;
    }
    if (!(d->rms_eps > 0.f) || !(d->rope_theta > 0.f)) return MK_ERR_INVALID_ARG;
    if (d->sliding_window < 0) return MK_ERR_INVALID_ARG;
    if (d->max_batch < 1 || d->max_batch > mk::kMaxBatch) return MK_ERR_INVALID_ARG;
    if (d->page_size != mk::kPage) return MK_ERR_INVALID_ARG;
    if (d->max_positions < 1) return MK_ERR_INVALID_ARG;
    return MK_OK;
}

mk_status validate_weights(const mk_model_desc* d, const mk_weights* w) {
    if (!w || !w->embed || !w->final_norm || !w->lm_head || !w->layers) return MK_ERR_INVALID_ARG;
    for (int l = 0; l < d->n_layers; ++l) {
        const mk_layer_weights& L = w->layers[l];
        if (!L.attn_norm || !L.wq || !L.wk || !L.wv || !L.wo || !L.mlp_norm) return MK_ERR_INVALID_ARG;
        if (d->n_experts > 0 ? (!L.router || !L.exp_gate || !L.exp_up || !L.exp_down)
                             : (!L.w_gate || !L.w_up || !L.w_down))
            return MK_ERR_INVALID_ARG;
    }
    return MK_OK;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

template <int HD>
cudaError_t set_kernel_attrs() {
    cudaError_t e = cudaFuncSetAttribute(mk::decode_step_kernel<HD, false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, mk::kSmemBytes);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(mk::decode_step_kernel<HD, true>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, mk::kSmemBytes);
}

// resident CTAs per SM of both instances (single- and multi-step launches)
template <int HD>
cudaError_t occupancy(int* blocks) {
    int b1 = 0, b2 = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b1, mk::decode_step_kernel<HD, false>,
                                                                  mk::kThreads, mk::kSmemBytes);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b2, mk::decode_step_kernel<HD, true>,
                                                          mk::kThreads, mk::kSmemBytes);
    *blocks = b1 < b2 ? b1 : b2;
    return e;
}

void free_handle(mk_handle* h) {
    if (!h) return;
    if (h->kv) cudaFree(h->kv);
    if (h->block) cudaFree(h->block);
    if (h->d_layers) cudaFree(h->d_layers);
    if (h->d_gains) cudaFree(h->d_gains);
    if (h->d_rope) cudaFree(h->d_rope);
    if (h->host_stage) cudaFreeHost(h->host_stage);
    if (h->dev_stage) cudaFree(h->dev_stage);
    if (h->dev_logits) cudaFree(h->dev_logits);
    delete h;
}

// BF16 gain vector on the device -> fp32, permuted column order, into host vector
bool fetch_gain(const void* dptr, int d, float* out) {
    std::vector<uint16_t> tmp(d);
    if (cudaMemcpy(tmp.data(), dptr, sizeof(uint16_t) * d, cudaMemcpyDeviceToHost) != cudaSuccess)
        return false;
    for (int k = 0; k < d; ++k) {
        uint32_t u = (uint32_t)tmp[k] << 16;
        float f;
        std::memcpy(&f, &u, 4);
        out[perm_col_host(k)] = f;
    }
    return true;
}

}  // namespace

extern "C" {

const char* mk_status_string(mk_status s) {
    switch (s) {
        case MK_OK: return "ok";
        case MK_ERR_INVALID_ARG: return "invalid argument";
        case MK_ERR_UNSUPPORTED_DEVICE: return "unsupported device (need sm_103 with cooperative launch)";
        case MK_ERR_OOM: return "out of device memory";
        case MK_ERR_LAUNCH: return "kernel launch failed";
        case MK_ERR_BAD_PAGE: return "page-table entry out of range";
        case MK_ERR_TIMEOUT: return "device-side dependency wait timed out";
        case MK_ERR_INTERNAL: return "internal / CUDA runtime error";
        case MK_ERR_NO_DEVICE: return "no CUDA device";
    }
    return "unknown status";
}

mk_status mk_create(const mk_model_desc* desc, const mk_weights* weights, int device,
                    mk_handle** out) {
    if (!out) return MK_ERR_INVALID_ARG;
    *out = nullptr;
    mk_status st = validate_desc(desc);
    if (st != MK_OK) return st;
    st = validate_weights(desc, weights);
    if (st != MK_OK) return st;
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || ndev == 0) {
        cudaGetLastError();
        return MK_ERR_NO_DEVICE;
    }
    if (device < 0 || device >= ndev) return MK_ERR_INVALID_ARG;
    DeviceGuard guard(device);
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return MK_ERR_INTERNAL;
    if (prop.major != 10 || prop.minor != 3 || !prop.cooperativeLaunch)
        return MK_ERR_UNSUPPORTED_DEVICE;
    const int hd = desc->head_dim;
    int blocks = 0;
    cudaError_t e = hd == 128 ? set_kernel_attrs<128>() : set_kernel_attrs<64>();
    if (e == cudaSuccess) e = hd == 128 ? occupancy<128>(&blocks) : occupancy<64>(&blocks);
    if (e != cudaSuccess || blocks < 1) {
        cudaGetLastError();
        return MK_ERR_UNSUPPORTED_DEVICE;
    }

    // each CTA keeps its ceil(d / CTAs) residual rows in shared memory
    if ((desc->d_model + prop.multiProcessorCount - 1) / prop.multiProcessorCount > mk::kMaxOwnRows)
        return MK_ERR_INVALID_ARG;
    mk_handle* h = new (std::nothrow) mk_handle();
    if (!h) return MK_ERR_OOM;
    h->device = device;
    h->desc = *desc;
    h->sliding.assign(desc->n_layers, 0);
    if (desc->layer_is_sliding)
        for (int l = 0; l < desc->n_layers; ++l) h->sliding[l] = desc->layer_is_sliding[l] ? 1 : 0;
    h->desc.layer_is_sliding = nullptr;
    h->num_ctas = prop.multiProcessorCount;
    h->hd = hd;

    const int L = desc->n_layers, d = desc->d_model, Hq = desc->n_q_heads, Hkv = desc->n_kv_heads;
    const int G = Hq / Hkv, F = desc->ffn_dim, V = desc->vocab, maxB = desc->max_batch;
    const int C = h->num_ctas;
    const int qkv_rows = (Hq + 2 * Hkv) * hd;
    const int E = desc->n_experts, Fe = desc->expert_ffn_dim;
    const int hrow = E > 0 ? E * Fe : F;  // SwiGLU row: dense width, or every expert's slot

    // ---- scratch arena
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes, 256); return o; };
    // activations and attention partials are tagged 64-bit words
    const size_t o_x = take(8 * (size_t)maxB * d);
    const size_t o_qkv = take(8 * (size_t)maxB * qkv_rows);
    const size_t o_attn = take(8 * (size_t)maxB * Hq * hd);
    const size_t o_h = take(8 * (size_t)maxB * hrow);
    const size_t o_part = take(8 * (size_t)maxB * Hkv * C * (G * hd + 2 * G));
    const size_t o_route = take(8 * (size_t)maxB * (E > 0 ? E : 1));
    const size_t o_union = take(sizeof(int) * (size_t)L);
    const size_t o_xf = take(sizeof(float) * (size_t)maxB * d);
    const size_t o_attnf = take(sizeof(float) * (size_t)maxB * Hq * hd);
    const size_t o_hf = take(sizeof(float) * (size_t)maxB * hrow);
    const size_t o_am = take(16 * (size_t)C * maxB);  // tagged (value, index) pairs
    const size_t o_cand = take(16 * (size_t)C * maxB * mk::kMaxSampleTopK);  // top-k sampling lists
    h->counters_words = (size_t)(1 + L * mk::kStagesPerLayer) * mk::kCounterStride;
    h->arrivals_words = (size_t)mk::kCounterStride;
    const size_t o_cnt = take(sizeof(uint32_t) * h->counters_words);
    const size_t o_arr = take(sizeof(uint32_t) * h->arrivals_words);
    // status word (2 ints, 2 spare), then the next tokens of mk_decode_step_host, so that
    // one device-to-host copy returns both
    const size_t o_status = take(sizeof(int) * (4 + mk::kMaxBatch));
    h->block_bytes = off;
    if (cudaMalloc(&h->block, h->block_bytes) != cudaSuccess) {
        cudaGetLastError();
        free_handle(h);
        return MK_ERR_OOM;
    }
    uint8_t* base = static_cast<uint8_t*>(h->block);
    if (cudaMemset(h->block, 0, h->block_bytes) != cudaSuccess) { free_handle(h); return MK_ERR_INTERNAL; }

    // ---- norm gains (fp32, permuted), RoPE table, layer table
    std::vector<float> gains((size_t)(2 * L + 1) * d);
    for (int l = 0; l < L; ++l) {
        if (!fetch_gain(weights->layers[l].attn_norm, d, &gains[(size_t)(2 * l) * d]) ||
            !fetch_gain(weights->layers[l].mlp_norm, d, &gains[(size_t)(2 * l + 1) * d])) {
            cudaGetLastError();
            free_handle(h);
            return MK_ERR_INVALID_ARG;
        }
    }
    if (!fetch_gain(weights->final_norm, d, &gains[(size_t)(2 * L) * d])) {
        cudaGetLastError();
        free_handle(h);
        return MK_ERR_INVALID_ARG;
    }
    const int half = hd / 2;
    std::vector<float2> rope((size_t)desc->max_positions * half);
    for (int pos = 0; pos < desc->max_positions; ++pos)
        for (int i = 0; i < half; ++i) {
            const double inv_freq = std::pow((double)desc->rope_theta, -2.0 * i / (double)hd);
            const double ang = (double)pos * inv_freq;
            rope[(size_t)pos * half + i] = make_float2((float)std::cos(ang), (float)std::sin(ang));
        }
    if (cudaMalloc(&h->d_gains, sizeof(float) * gains.size()) != cudaSuccess ||
        cudaMalloc(&h->d_rope, sizeof(float2) * rope.size()) != cudaSuccess ||
        cudaMalloc(&h->d_layers, sizeof(mk::LayerPlan) * L) != cudaSuccess) {
        cudaGetLastError();
        free_handle(h);
        return MK_ERR_OOM;
    }
    std::vector<mk::LayerPlan> lp(L);
    int64_t wbytes = 0;
    for (int l = 0; l < L; ++l) {
        const mk_layer_weights& W = weights->layers[l];
        lp[l].wq = (const bf16*)W.wq; lp[l].wk = (const bf16*)W.wk; lp[l].wv = (const bf16*)W.wv;
        lp[l].wo = (const bf16*)W.wo; lp[l].w_gate = (const bf16*)W.w_gate;
        lp[l].w_up = (const bf16*)W.w_up; lp[l].w_down = (const bf16*)W.w_down;
        lp[l].router = (const bf16*)W.router; lp[l].exp_gate = (const bf16*)W.exp_gate;
        lp[l].exp_up = (const bf16*)W.exp_up; lp[l].exp_down = (const bf16*)W.exp_down;
        lp[l].attn_gain = h->d_gains + (size_t)(2 * l) * d;
        lp[l].mlp_gain = h->d_gains + (size_t)(2 * l + 1) * d;
        lp[l].sliding = h->sliding[l];
        const int64_t mlp = E > 0 ? (int64_t)E * d + 3LL * E * Fe * d : 3LL * F * d;
        wbytes += 2LL * ((int64_t)qkv_rows * d + (int64_t)d * Hq * hd + mlp + 2LL * d);
    }
    wbytes += 2LL * ((int64_t)V * d + d);
    h->weight_bytes = wbytes;
    if (cudaMemcpy(h->d_gains, gains.data(), sizeof(float) * gains.size(), cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemcpy(h->d_rope, rope.data(), sizeof(float2) * rope.size(), cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemcpy(h->d_layers, lp.data(), sizeof(mk::LayerPlan) * L, cudaMemcpyHostToDevice) != cudaSuccess) {
        cudaGetLastError();
        free_handle(h);
        return MK_ERR_INTERNAL;
    }

    mk::Plan& p = h->plan;
    p.L = L; p.d = d; p.Hq = Hq; p.Hkv = Hkv; p.hd = hd; p.G = G; p.F = F; p.V = V;
    p.E = E; p.topk = desc->top_k; p.Fe = Fe; p.hrow = hrow;
    p.window = desc->sliding_window; p.max_pos = desc->max_positions; p.maxB = maxB;
    p.num_pages = 0;
    p.eps = desc->rms_eps;
    p.scale = (float)(1.0 / std::sqrt((double)hd));
    p.C = C;
    p.qkv_rows = qkv_rows;
    for (int l = 0; l < L; ++l)
        if (h->sliding[l]) p.sliding_mask[l >> 5] |= 1u << (l & 31);
    p.layers = h->d_layers;
    p.embed = (const bf16*)weights->embed;
    p.lm_head = (const bf16*)weights->lm_head;
    p.final_gain = h->d_gains + (size_t)(2 * L) * d;
    p.rope = h->d_rope;
    p.x = (uint64_t*)(base + o_x);
    p.qkv = (uint64_t*)(base + o_qkv);
    p.attn = (uint64_t*)(base + o_attn);
    p.h = (uint64_t*)(base + o_h);
    p.part = (uint64_t*)(base + o_part);
    p.route = (uint64_t*)(base + o_route);
    p.moe_union = (int*)(base + o_union);
    p.xf = (float*)(base + o_xf);
    p.attnf = (float*)(base + o_attnf);
    p.hf = (float*)(base + o_hf);
    p.counters = (uint32_t*)(base + o_cnt);
    p.amax = (uint64_t*)(base + o_am);
    p.cand = (uint64_t*)(base + o_cand);
    p.arrivals = (uint32_t*)(base + o_arr);
    p.status = (int*)(base + o_status);
    p.kv = nullptr;
    *out = h;
    return MK_OK;
}

mk_status mk_kv_alloc(mk_handle* h, int32_t num_pages, mk_kv_pool* out) {
    if (!h || !out || num_pages < 1) return MK_ERR_INVALID_ARG;
    if (h->kv) return MK_ERR_INVALID_ARG;
    DeviceGuard guard(h->device);
    const mk_model_desc& d = h->desc;
    const int64_t rows = (int64_t)d.n_layers * num_pages * 2 * d.n_kv_heads * mk::kPage;
    if (rows >= (1LL << 31)) return MK_ERR_OOM;
    const int64_t elems = rows * h->hd;
    const int64_t bytes = elems * 2;
    if (cudaMalloc(&h->kv, (size_t)bytes) != cudaSuccess) {
        cudaGetLastError();
        h->kv = nullptr;
        return MK_ERR_OOM;
    }
    // tensor map: the pool as a 2D [rows][head_dim] BF16 tensor, box 64 x 16, 128B swizzle
    PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", (void**)&encode, 12000,
                                         cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !encode) {
        cudaGetLastError();
        cudaFree(h->kv);
        h->kv = nullptr;
        return MK_ERR_INTERNAL;
    }
    CUtensorMap map;
    cuuint64_t gdim[2] = {(cuuint64_t)h->hd, (cuuint64_t)rows};
    cuuint64_t gstride[1] = {(cuuint64_t)h->hd * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)mk::kPage};
    cuuint32_t estride[2] = {1, 1};
    CUresult r = encode(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, h->kv, gdim, gstride, box,
                        estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        cudaFree(h->kv);
        h->kv = nullptr;
        return MK_ERR_INTERNAL;
    }
    h->kv_tmap = map;
    h->plan.kv = (bf16*)h->kv;
    h->plan.num_pages = num_pages;
    mk_kv_pool& P = h->pool;
    P.base = h->kv;
    P.num_pages = num_pages;
    P.slot_stride = h->hd;
    P.head_stride = (int64_t)mk::kPage * h->hd;
    P.kv_stride = P.head_stride * d.n_kv_heads;
    P.page_stride = 2 * P.kv_stride;
    P.layer_stride = P.page_stride * num_pages;
    P.bytes = bytes;
    *out = P;
    return MK_OK;
}

mk_status mk_kv_free(mk_handle* h, mk_kv_pool* pool) {
    if (!h || !h->kv) return MK_ERR_INVALID_ARG;
    if (pool && pool->base != h->kv) return MK_ERR_INVALID_ARG;
    DeviceGuard guard(h->device);
    cudaDeviceSynchronize();
    cudaFree(h->kv);
    h->kv = nullptr;
    h->plan.kv = nullptr;
    h->plan.num_pages = 0;
    h->pool = mk_kv_pool{};
    if (pool) *pool = mk_kv_pool{};
    return MK_OK;
}

}  // extern "C"

namespace {

// decode steps one launch may run (the loader's MoE readiness words encode step * 128)
constexpr int32_t kMaxStepsPerLaunch = 1 << 16;

// One launch of the decode kernel for n_steps consecutive steps (see mk_decode_steps).
mk_status launch_steps(mk_handle* h, int32_t n_steps, const int32_t* tokens, const int32_t* positions,
                       const int32_t* page_table, int32_t max_pages_per_seq, const int32_t* seq_lens,
                       int32_t batch, int32_t* next_tokens, float* logits, void* stream) {
    if (!h || !tokens || !positions || !page_table || !seq_lens || !next_tokens)
        return MK_ERR_INVALID_ARG;
    if (batch < 1 || batch > h->desc.max_batch || max_pages_per_seq < 1) return MK_ERR_INVALID_ARG;
    if (n_steps < 1 || n_steps > kMaxStepsPerLaunch) return MK_ERR_INVALID_ARG;
    // the kernel partitions attention units in 32-bit arithmetic
    if ((uint64_t)batch * h->desc.n_kv_heads * max_pages_per_seq * h->num_ctas >= (1ull << 31))
        return MK_ERR_INVALID_ARG;
    if (!h->kv) return MK_ERR_INVALID_ARG;
    // declared shared-prefix groups describe the rows of one batch size
    if (h->pf_batch != 0 && h->pf_batch != batch) return MK_ERR_INVALID_ARG;
    DeviceGuard guard(h->device);
    mk::StepArgs a;
    a.kv_tmap = h->kv_tmap;
    a.p = h->plan;
    a.tokens = tokens;
    a.positions = positions;
    a.page_table = page_table;
    a.seq_lens = seq_lens;
    a.next_tokens = next_tokens;
    a.n_steps = n_steps;
    a.logits_last = logits;
    a.logits = n_steps == 1 ? logits : nullptr;  // the kernel sets it for the last step
    a.max_pages = max_pages_per_seq;
    a.B = batch;
    // 20-bit epochs, never 0 (zeroed memory never carries a valid tag); step s of the
    // launch uses the s-th epoch after the first
    const uint32_t epoch = h->epoch % 0xFFFFFu + 1u;
    a.epoch = epoch;
    // the stage counters only advance in steps whose batch exceeds the tagged-word limit
    const bool counted = batch > mk::kMaxTaggedBatch;
    const uint32_t cnt_epoch = h->cnt_epoch + (counted ? 1u : 0u);
    a.stage_target = cnt_epoch * (uint32_t)h->num_ctas;
    a.skip_publish = h->skip_publish;
    a.prefetch_slots = h->prefetch_slots;
    a.timeout_ns = h->timeout_ns;
    a.temperature = h->temperature;
    a.top_k = h->top_k;
    a.seed_lo = (uint32_t)h->seed;
    a.seed_hi = (uint32_t)(h->seed >> 32);
    a.pf_on = h->pf_batch != 0;
    for (int b = 0; b < mk::kMaxBatch; ++b) {
        a.pf_lead[b] = h->pf_batch ? h->pf_lead[b] : -1;
        a.pf_pages[b] = h->pf_batch ? h->pf_pages[b] : 0;
    }
    void* args[] = {&a};
    const bool multi = n_steps > 1;
    const void* fn = h->hd == 128
        ? (multi ? (const void*)mk::decode_step_kernel<128, true> : (const void*)mk::decode_step_kernel<128, false>)
        : (multi ? (const void*)mk::decode_step_kernel<64, true> : (const void*)mk::decode_step_kernel<64, false>);
    cudaError_t e = cudaLaunchCooperativeKernel(fn, dim3(h->num_ctas), dim3(mk::kThreads), args,
                                                mk::kSmemBytes, (cudaStream_t)stream);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return MK_ERR_LAUNCH;
    }
    h->epoch = (uint32_t)((epoch - 1u + (uint32_t)(n_steps - 1)) % 0xFFFFFu) + 1u;
    h->cnt_epoch = cnt_epoch + (counted ? (uint32_t)(n_steps - 1) : 0u);
    h->last_batch = batch;
    return MK_OK;
}

}  // namespace

extern "C" {

mk_status mk_decode_step(mk_handle* h, const int32_t* tokens, const int32_t* positions,
                         const int32_t* page_table, int32_t max_pages_per_seq,
                         const int32_t* seq_lens, int32_t batch, int32_t* next_tokens,
                         float* logits, void* stream) {
    return launch_steps(h, 1, tokens, positions, page_table, max_pages_per_seq, seq_lens, batch,
                        next_tokens, logits, stream);
}

mk_status mk_decode_steps(mk_handle* h, int32_t n_steps, const int32_t* tokens,
                          const int32_t* positions, const int32_t* page_table,
                          int32_t max_pages_per_seq, const int32_t* seq_lens, int32_t batch,
                          int32_t* next_tokens, float* logits, void* stream) {
    return launch_steps(h, n_steps, tokens, positions, page_table, max_pages_per_seq, seq_lens,
                        batch, next_tokens, logits, stream);
}


mk_status mk_decode_step_host(mk_handle* h, const int32_t* tokens, const int32_t* positions,
                              const int32_t* page_table, int32_t max_pages_per_seq,
                              const int32_t* seq_lens, int32_t batch, int32_t* next_tokens,
                              float* logits, void* stream) {
    if (!h || !tokens || !positions || !page_table || !seq_lens || !next_tokens)
        return MK_ERR_INVALID_ARG;
    if (batch < 1 || batch > h->desc.max_batch || max_pages_per_seq < 1) return MK_ERR_INVALID_ARG;
    DeviceGuard guard(h->device);
    const size_t nb = (size_t)batch;
    const size_t in_bytes = sizeof(int32_t) * (3 * nb + nb * (size_t)max_pages_per_seq);
    const size_t out_bytes = sizeof(int32_t) * (4 + mk::kMaxBatch);
    if (in_bytes > h->stage_bytes) {
        if (h->host_stage) cudaFreeHost(h->host_stage);
        if (h->dev_stage) cudaFree(h->dev_stage);
        h->host_stage = h->dev_stage = nullptr;
        h->stage_bytes = 0;
        if (cudaHostAlloc(&h->host_stage, in_bytes + out_bytes, cudaHostAllocDefault) != cudaSuccess ||
            cudaMalloc(&h->dev_stage, in_bytes) != cudaSuccess) {
            cudaGetLastError();
            if (h->host_stage) cudaFreeHost(h->host_stage);
            if (h->dev_stage) cudaFree(h->dev_stage);
            h->host_stage = h->dev_stage = nullptr;
            return MK_ERR_OOM;
        }
        h->stage_bytes = in_bytes;
    }
    if (logits && !h->dev_logits &&
        cudaMalloc(&h->dev_logits, sizeof(float) * (size_t)h->desc.max_batch * h->desc.vocab) != cudaSuccess) {
        cudaGetLastError();
        h->dev_logits = nullptr;
        return MK_ERR_OOM;
    }
    // pack the inputs; one host-to-device copy
    int32_t* hs = static_cast<int32_t*>(h->host_stage);
    std::memcpy(hs, tokens, sizeof(int32_t) * nb);
    std::memcpy(hs + nb, positions, sizeof(int32_t) * nb);
    std::memcpy(hs + 2 * nb, seq_lens, sizeof(int32_t) * nb);
    std::memcpy(hs + 3 * nb, page_table, sizeof(int32_t) * nb * (size_t)max_pages_per_seq);
    cudaStream_t st = (cudaStream_t)stream;
    if (cudaMemcpyAsync(h->dev_stage, hs, in_bytes, cudaMemcpyHostToDevice, st) != cudaSuccess) {
        cudaGetLastError();
        return MK_ERR_INTERNAL;
    }
    const int32_t* ds = static_cast<const int32_t*>(h->dev_stage);
    const mk_status ls = launch_steps(h, 1, ds, ds + nb, ds + 3 * nb, max_pages_per_seq, ds + 2 * nb, batch,
                                      h->plan.status + 4, logits ? h->dev_logits : nullptr, stream);
    if (ls != MK_OK) {
        cudaStreamSynchronize(st);  // the copy must finish before the staging is reused
        return ls;
    }
    // the status word and the next tokens in one device-to-host copy
    int32_t* ho = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(h->host_stage) + h->stage_bytes);
    if (cudaMemcpyAsync(ho, h->plan.status, sizeof(int32_t) * (4 + nb), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        (logits && cudaMemcpyAsync(logits, h->dev_logits, sizeof(float) * nb * (size_t)h->desc.vocab,
                                   cudaMemcpyDeviceToHost, st) != cudaSuccess) ||
        cudaStreamSynchronize(st) != cudaSuccess) {
        cudaGetLastError();
        return MK_ERR_INTERNAL;
    }
    std::memcpy(next_tokens, ho + 4, sizeof(int32_t) * nb);
    return (mk_status)ho[0];
}

mk_status mk_status_sync(mk_handle* h, void* stream, int32_t* failing_task) {
    if (!h) return MK_ERR_INVALID_ARG;
    DeviceGuard guard(h->device);
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) {
        cudaGetLastError();
        return MK_ERR_INTERNAL;
    }
    int st[2] = {0, -1};
    if (cudaMemcpy(st, h->plan.status, sizeof(st), cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return MK_ERR_INTERNAL;
    }
    if (failing_task) *failing_task = st[0] ? st[1] : -1;
    return (mk_status)st[0];
}

mk_status mk_status_reset(mk_handle* h) {
    if (!h) return MK_ERR_INVALID_ARG;
    DeviceGuard guard(h->device);
    if (cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        return MK_ERR_INTERNAL;
    }
    if (cudaMemset(h->plan.counters, 0, sizeof(uint32_t) * h->counters_words) != cudaSuccess ||
        cudaMemset(h->plan.arrivals, 0, sizeof(uint32_t) * h->arrivals_words) != cudaSuccess ||
        cudaMemset(h->plan.status, 0, sizeof(int) * 4) != cudaSuccess) {
        cudaGetLastError();
        return MK_ERR_INTERNAL;
    }
    h->cnt_epoch = 0;
    // the tag epoch keeps advancing: words written before the reset never match a later tag
    return MK_OK;
}

mk_status mk_set_option(mk_handle* h, mk_option opt, int64_t value) {
    if (!h) return MK_ERR_INVALID_ARG;
    switch (opt) {
        case MK_OPT_TIMEOUT_NS:
            if (value < 1000) return MK_ERR_INVALID_ARG;
            h->timeout_ns = value;
            return MK_OK;
        case MK_OPT_SKIP_PUBLISH:
            h->skip_publish = (int)value;
            return MK_OK;
        case MK_OPT_PREFETCH_SLOTS:
            if (value < 0 || value > 64) return MK_ERR_INVALID_ARG;
            h->prefetch_slots = (int)value;
            return MK_OK;
    }
    return MK_ERR_INVALID_ARG;
}

mk_status mk_set_sampling(mk_handle* h, float temperature, int32_t top_k, uint64_t seed) {
    if (!h || !std::isfinite(temperature) || temperature < 0.f) return MK_ERR_INVALID_ARG;
    if (top_k < 0 || top_k > mk::kMaxSampleTopK) return MK_ERR_INVALID_ARG;
    h->temperature = temperature;
    h->top_k = top_k;
    h->seed = seed;
    return MK_OK;
}

mk_status mk_set_shared_prefix(mk_handle* h, int32_t batch, const int32_t* leader,
                               const int32_t* shared_pages) {
    if (!h) return MK_ERR_INVALID_ARG;
    if (batch == 0) {
        h->pf_batch = 0;
        return MK_OK;
    }
    if (batch < 1 || batch > h->desc.max_batch || !leader || !shared_pages) return MK_ERR_INVALID_ARG;
    int lead[mk::kMaxBatch], pages[mk::kMaxBatch], size[mk::kMaxBatch] = {};
    for (int b = 0; b < batch; ++b) {
        const int L = leader[b];
        // a row joins the group of an earlier (or the same) row that leads its own group
        if (L < 0 || L > b || leader[L] != L) return MK_ERR_INVALID_ARG;
        if (shared_pages[b] < 0 || shared_pages[b] != shared_pages[L]) return MK_ERR_INVALID_ARG;
        lead[b] = L;
        pages[b] = shared_pages[b];
        ++size[L];
    }
    const int G = h->desc.n_q_heads / h->desc.n_kv_heads;
    for (int b = 0; b < batch; ++b)
        if (size[b] * G > 16) return MK_ERR_INVALID_ARG;  // two 8-wide query column tiles
    h->pf_batch = batch;
    for (int b = 0; b < mk::kMaxBatch; ++b) {
        h->pf_lead[b] = b < batch ? lead[b] : -1;
        h->pf_pages[b] = b < batch ? pages[b] : 0;
    }
    return MK_OK;
}

mk_status mk_get_info(const mk_handle* h, mk_info* out) {
    if (!h || !out) return MK_ERR_INVALID_ARG;
    out->num_ctas = h->num_ctas;
    out->threads_per_cta = mk::kThreads;
    out->smem_bytes = mk::kSmemBytes;
    out->ring_stages = mk::kStages;
    out->weight_bytes = h->weight_bytes;
    out->scratch_bytes = (int64_t)h->block_bytes;
    return MK_OK;
}

mk_status mk_debug_buffer(const mk_handle* h, int32_t which, void** dev_ptr, int64_t* bytes) {
    if (!h || !dev_ptr || !bytes) return MK_ERR_INVALID_ARG;
    const mk::Plan& p = h->plan;
    const int64_t B = p.maxB;
    const bool tg = h->last_batch <= mk::kMaxTaggedBatch;
    switch (which) {
        case MK_BUF_X:
            *dev_ptr = tg ? (void*)p.x : (void*)p.xf;
            *bytes = (tg ? 8 : 4) * B * p.d;
            return MK_OK;
        case MK_BUF_QKV: *dev_ptr = p.qkv; *bytes = 8 * B * p.qkv_rows; return MK_OK;
        case MK_BUF_ATTN:
            *dev_ptr = tg ? (void*)p.attn : (void*)p.attnf;
            *bytes = (tg ? 8 : 4) * B * p.Hq * p.hd;
            return MK_OK;
        case MK_BUF_H:
            *dev_ptr = tg ? (void*)p.h : (void*)p.hf;
            *bytes = (tg ? 8 : 4) * B * p.hrow;
            return MK_OK;
        case MK_BUF_ROUTE:
            if (p.E == 0) return MK_ERR_INVALID_ARG;
            *dev_ptr = p.route;
            *bytes = 8 * B * p.E;
            return MK_OK;
        case MK_BUF_MOE_UNION:
            if (p.E == 0) return MK_ERR_INVALID_ARG;
            *dev_ptr = p.moe_union;
            *bytes = 4 * (int64_t)p.L;
            return MK_OK;
    }
    return MK_ERR_INVALID_ARG;
}

void mk_destroy(mk_handle* h) {
    if (!h) return;
    DeviceGuard guard(h->device);
    cudaDeviceSynchronize();
    free_handle(h);
}

}  // extern "C"

// ===========================================================================
// mk_decode_step_noalloc: the same decode-step kernel, with every byte of its
// scratch (plan tables, norm gains, RoPE table, activations, attention partials,
// counters, status word) carved out of one file-scope static device
// array instead of memory from cudaMalloc. It exists for callers that must not
// allocate device memory: code running where an allocation would synchronise the
// device or is forbidden (allocator-free runtimes, memory-capped sandboxes, hosts
// that pre-plan every byte of HBM).
// ===========================================================================
namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)8 << 20;  // 8 MiB, held on every GPU
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kNoAllocMaxDevices = 64;
struct NoAllocDevice {
    bool ready;
    int num_sms;
    unsigned char* base;  // device address of g_noalloc_scratch on this device
    // the RoPE table the array holds (written by the last call on this device): it is
    // rewritten only when the next call needs another one (theta, head dim, positions
    // or its place in the array differ)
    bool rope_valid;
    float rope_theta;
    int rope_hd, rope_max_pos;
    size_t rope_off;
};
NoAllocDevice g_noalloc_dev[kNoAllocMaxDevices];
std::mutex g_noalloc_mutex;

// Parameters of the set-up kernel: the layer table and gain sources travel as kernel
// parameters, so nothing is staged through allocated memory.
struct NoAllocSetup {
    mk::LayerPlan layers[mk::kMaxLayers];
    const uint16_t* gain_src[2 * mk::kMaxLayers + 1];
    mk::LayerPlan* layers_dst;
    float* gains_dst;
    float2* rope_dst;
    uint32_t* zero_dst;
    long long zero_words;
    int L, d, hd, max_pos;
    float theta;
};

__global__ void noalloc_setup_kernel(const __grid_constant__ NoAllocSetup s) {
    const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long n = (long long)gridDim.x * blockDim.x;
    for (long long i = tid; i < s.L; i += n) s.layers_dst[i] = s.layers[i];
    const long long ng = (long long)(2 * s.L + 1) * s.d;
    for (long long i = tid; i < ng; i += n) {
        const int v = (int)(i / s.d), k = (int)(i % s.d);
        const uint32_t u = (uint32_t)s.gain_src[v][k] << 16;
        s.gains_dst[(size_t)v * s.d + mk::perm_col(k)] = __uint_as_float(u);
    }
    const int half = s.hd / 2;
    const long long nr = (long long)s.max_pos * half;
    for (long long i = tid; i < nr; i += n) {
        const int pos = (int)(i / half), j = (int)(i % half);
        const double inv_freq = pow((double)s.theta, -2.0 * j / (double)s.hd);
        const double ang = (double)pos * inv_freq;
        s.rope_dst[i] = make_float2((float)cos(ang), (float)sin(ang));
    }
    for (long long i = tid; i < s.zero_words; i += n) s.zero_dst[i] = 0u;
}

// Once per device, with that device current: check it, set the kernel attributes and
// look up the device address of the static array.
mk_status noalloc_device_setup(int dev, NoAllocDevice** out) {
    if (dev < 0 || dev >= kNoAllocMaxDevices) return MK_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    NoAllocDevice& D = g_noalloc_dev[dev];
    if (!D.ready) {
        cudaDeviceProp prop;
        if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) {
            cudaGetLastError();
            return MK_ERR_INTERNAL;
        }
        if (prop.major != 10 || prop.minor != 3 || !prop.cooperativeLaunch)
            return MK_ERR_UNSUPPORTED_DEVICE;
        if (set_kernel_attrs<128>() != cudaSuccess || set_kernel_attrs<64>() != cudaSuccess) {
            cudaGetLastError();
            return MK_ERR_UNSUPPORTED_DEVICE;
        }
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
            cudaGetLastError();
            return MK_ERR_INTERNAL;
        }
        D.base = static_cast<unsigned char*>(ptr);
        D.num_sms = prop.multiProcessorCount;
        D.ready = true;
    }
    *out = &D;
    return MK_OK;
}

}  // namespace

extern "C" mk_status mk_decode_step_noalloc(
    const mk_model_desc* desc, const mk_weights* weights, void* kv_pool, int32_t num_pages,
    const int32_t* tokens, const int32_t* positions, const int32_t* page_table,
    int32_t max_pages_per_seq, const int32_t* seq_lens, int32_t batch, int32_t* next_tokens,
    float* logits, int32_t* status_out, void* stream) {
    mk_status st = validate_desc(desc);
    if (st != MK_OK) return st;
    st = validate_weights(desc, weights);
    if (st != MK_OK) return st;
    if (!kv_pool || num_pages < 1 || !tokens || !positions || !page_table || !seq_lens ||
        !next_tokens || !status_out || max_pages_per_seq < 1)
        return MK_ERR_INVALID_ARG;
    if (batch < 1 || batch > desc->max_batch) return MK_ERR_INVALID_ARG;
    if ((uint64_t)batch * desc->n_kv_heads * max_pages_per_seq * 1024u >= (1ull << 31))
        return MK_ERR_INVALID_ARG;  // 32-bit attention-unit arithmetic (any CTA count <= 1024)
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return MK_ERR_NO_DEVICE;
    }
    NoAllocDevice* D = nullptr;
    st = noalloc_device_setup(dev, &D);
    if (st != MK_OK) return st;

    const int L = desc->n_layers, d = desc->d_model, Hq = desc->n_q_heads, Hkv = desc->n_kv_heads;
    const int hd = desc->head_dim, G = Hq / Hkv, F = desc->ffn_dim, V = desc->vocab;
    const int maxB = desc->max_batch, C = D->num_sms;
    if ((d + C - 1) / C > mk::kMaxOwnRows) return MK_ERR_INVALID_ARG;
    const int qkv_rows = (Hq + 2 * Hkv) * hd;
    const int E = desc->n_experts, Fe = desc->expert_ffn_dim;
    const int hrow = E > 0 ? E * Fe : F;
    const int64_t rows = (int64_t)L * num_pages * 2 * Hkv * mk::kPage;
    if (rows >= (1LL << 31)) return MK_ERR_INVALID_ARG;

    // carve the static array
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes, 256); return o; };
    const size_t o_layers = take(sizeof(mk::LayerPlan) * L);
    const size_t o_gains = take(sizeof(float) * (size_t)(2 * L + 1) * d);
    const size_t o_rope = take(sizeof(float2) * (size_t)desc->max_positions * (hd / 2));
    const size_t o_xf = take(sizeof(float) * (size_t)maxB * d);
    const size_t o_attnf = take(sizeof(float) * (size_t)maxB * Hq * hd);
    const size_t o_hf = take(sizeof(float) * (size_t)maxB * hrow);
    const size_t o_union = take(sizeof(int) * (size_t)L);
    // cleared every call (every call runs with tag epoch 1 and counter epoch 1): the
    // tagged activations, attention partials and argmax pairs, the counters and the
    // status word
    const size_t o_zero = off;
    const size_t o_x = take(8 * (size_t)maxB * d);
    const size_t o_qkv = take(8 * (size_t)maxB * qkv_rows);
    const size_t o_attn = take(8 * (size_t)maxB * Hq * hd);
    const size_t o_h = take(8 * (size_t)maxB * hrow);
    const size_t o_part = take(8 * (size_t)maxB * Hkv * C * (G * hd + 2 * G));
    const size_t o_route = take(8 * (size_t)maxB * (E > 0 ? E : 1));
    const size_t o_am = take(16 * (size_t)C * maxB);  // tagged (value, index) pairs
    const size_t o_cnt = take(sizeof(uint32_t) * (size_t)(1 + L * mk::kStagesPerLayer) * mk::kCounterStride);
    const size_t o_arr = take(sizeof(uint32_t) * mk::kCounterStride);
    const size_t o_status = take(sizeof(int) * 4);
    if (off > kNoAllocScratchBytes) return MK_ERR_INVALID_ARG;  // model/batch too large
    unsigned char* base = D->base;

    // KV tensor map, encoded on the host; it travels in the kernel parameters
    PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", (void**)&encode, 12000,
                                         cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !encode) {
        cudaGetLastError();
        return MK_ERR_INTERNAL;
    }
    CUtensorMap map;
    cuuint64_t gdim[2] = {(cuuint64_t)hd, (cuuint64_t)rows};
    cuuint64_t gstride[1] = {(cuuint64_t)hd * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)mk::kPage};
    cuuint32_t estride[2] = {1, 1};
    if (encode(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, kv_pool, gdim, gstride, box, estride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return MK_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;

    NoAllocSetup su;
    std::memset(&su, 0, sizeof(su));
    float* gains = reinterpret_cast<float*>(base + o_gains);
    for (int l = 0; l < L; ++l) {
        const mk_layer_weights& W = weights->layers[l];
        mk::LayerPlan& lp = su.layers[l];
        lp.wq = (const bf16*)W.wq; lp.wk = (const bf16*)W.wk; lp.wv = (const bf16*)W.wv;
        lp.wo = (const bf16*)W.wo; lp.w_gate = (const bf16*)W.w_gate;
        lp.w_up = (const bf16*)W.w_up; lp.w_down = (const bf16*)W.w_down;
        lp.router = (const bf16*)W.router; lp.exp_gate = (const bf16*)W.exp_gate;
        lp.exp_up = (const bf16*)W.exp_up; lp.exp_down = (const bf16*)W.exp_down;
        lp.attn_gain = gains + (size_t)(2 * l) * d;
        lp.mlp_gain = gains + (size_t)(2 * l + 1) * d;
        lp.sliding = (desc->layer_is_sliding && desc->layer_is_sliding[l]) ? 1 : 0;
        su.gain_src[2 * l] = (const uint16_t*)W.attn_norm;
        su.gain_src[2 * l + 1] = (const uint16_t*)W.mlp_norm;
    }
    su.gain_src[2 * L] = (const uint16_t*)weights->final_norm;
    su.layers_dst = reinterpret_cast<mk::LayerPlan*>(base + o_layers);
    su.gains_dst = gains;
    su.rope_dst = reinterpret_cast<float2*>(base + o_rope);
    su.zero_dst = reinterpret_cast<uint32_t*>(base + o_zero);
    su.zero_words = (long long)((o_status + sizeof(int) * 4 - o_zero) / sizeof(uint32_t));
    su.L = L; su.d = d; su.hd = hd; su.max_pos = desc->max_positions; su.theta = desc->rope_theta;
    {
        // The RoPE table (max_positions x head_dim / 2 angles in double) is the costly
        // part of the set-up: skip it when the array already holds this very table.
        std::lock_guard<std::mutex> lock(g_noalloc_mutex);
        const bool same = D->rope_valid && D->rope_theta == desc->rope_theta && D->rope_hd == hd &&
                          D->rope_max_pos == desc->max_positions && D->rope_off == o_rope;
        if (same) su.max_pos = 0;
        // from here on the array holds this call's table (the set-up kernel writes it
        // before anything else on the stream reads it)
        D->rope_valid = false;
        noalloc_setup_kernel<<<C, 256, 0, s>>>(su);
        if (cudaGetLastError() != cudaSuccess) return MK_ERR_LAUNCH;
        D->rope_valid = true;
        D->rope_theta = desc->rope_theta;
        D->rope_hd = hd;
        D->rope_max_pos = desc->max_positions;
        D->rope_off = o_rope;
    }

    mk::StepArgs a;
    mk::Plan& p = a.p;
    p.L = L; p.d = d; p.Hq = Hq; p.Hkv = Hkv; p.hd = hd; p.G = G; p.F = F; p.V = V;
    p.E = E; p.topk = desc->top_k; p.Fe = Fe; p.hrow = hrow;
    p.window = desc->sliding_window; p.max_pos = desc->max_positions; p.maxB = maxB;
    p.num_pages = num_pages;
    p.eps = desc->rms_eps;
    p.scale = (float)(1.0 / std::sqrt((double)hd));
    p.C = C;
    p.qkv_rows = qkv_rows;
    std::memset(p.sliding_mask, 0, sizeof(p.sliding_mask));
    for (int l = 0; l < L; ++l)
        if (desc->layer_is_sliding && desc->layer_is_sliding[l]) p.sliding_mask[l >> 5] |= 1u << (l & 31);
    p.layers = su.layers_dst;
    p.embed = (const bf16*)weights->embed;
    p.lm_head = (const bf16*)weights->lm_head;
    p.final_gain = gains + (size_t)(2 * L) * d;
    p.rope = su.rope_dst;
    p.x = (uint64_t*)(base + o_x);
    p.qkv = (uint64_t*)(base + o_qkv);
    p.attn = (uint64_t*)(base + o_attn);
    p.h = (uint64_t*)(base + o_h);
    p.part = (uint64_t*)(base + o_part);
    p.route = (uint64_t*)(base + o_route);
    p.moe_union = (int*)(base + o_union);
    p.xf = (float*)(base + o_xf);
    p.attnf = (float*)(base + o_attnf);
    p.hf = (float*)(base + o_hf);
    p.counters = (uint32_t*)(base + o_cnt);
    p.amax = (uint64_t*)(base + o_am);
    p.cand = nullptr;  // always greedy here
    p.arrivals = (uint32_t*)(base + o_arr);
    p.status = (int*)(base + o_status);
    p.kv = (bf16*)kv_pool;
    a.kv_tmap = map;
    a.tokens = tokens;
    a.positions = positions;
    a.page_table = page_table;
    a.seq_lens = seq_lens;
    a.next_tokens = next_tokens;
    a.logits = logits;
    a.max_pages = max_pages_per_seq;
    a.B = batch;
    a.epoch = 1;  // every tagged word and counter was cleared above
    a.stage_target = (uint32_t)C;
    a.skip_publish = -1;
    a.prefetch_slots = mk::kDefaultPrefetchSlots;
    a.timeout_ns = 1000000000LL;
    a.temperature = 0.f;  // greedy
    a.top_k = 0;
    a.seed_lo = a.seed_hi = 0;
    a.n_steps = 1;
    a.logits_last = logits;
    a.pf_on = 0;  // no shared-prefix groups
    for (int b = 0; b < mk::kMaxBatch; ++b) {
        a.pf_lead[b] = -1;
        a.pf_pages[b] = 0;
    }
    void* args[] = {&a};
    const void* fn = hd == 128 ? (const void*)mk::decode_step_kernel<128, false>
                               : (const void*)mk::decode_step_kernel<64, false>;
    if (cudaLaunchCooperativeKernel(fn, dim3(C), dim3(mk::kThreads), args, mk::kSmemBytes, s) !=
        cudaSuccess) {
        cudaGetLastError();
        return MK_ERR_LAUNCH;
    }
    if (cudaMemcpyAsync(status_out, base + o_status, 2 * sizeof(int), cudaMemcpyDeviceToDevice, s) !=
        cudaSuccess) {
        cudaGetLastError();
        return MK_ERR_INTERNAL;
    }
    return MK_OK;
}

#ifdef MK_PROF
// Profile builds only: the per-CTA section cycle sums, and clearing them.
extern "C" __attribute__((visibility("default"))) int mk_prof_read(void* dst, size_t bytes) {
    if (bytes > sizeof(mk::g_mk_prof)) bytes = sizeof(mk::g_mk_prof);
    return (int)cudaMemcpyFromSymbol(dst, mk::g_mk_prof, bytes);
}
extern "C" __attribute__((visibility("default"))) int mk_prof_clear() {
    static unsigned long long zero[mk::kProfCtas][mk::kProfSections];
    return (int)cudaMemcpyToSymbol(mk::g_mk_prof, zero, sizeof(zero));
}
#endif
#ifdef MK_TRACE
// Trace builds only: copy the per-CTA timeline of the last step to host memory.
extern "C" __attribute__((visibility("default"))) int mk_trace_read(void* dst, size_t bytes) {
    if (bytes > sizeof(mk::g_mk_trace)) bytes = sizeof(mk::g_mk_trace);
    return (int)cudaMemcpyFromSymbol(dst, mk::g_mk_trace, bytes);
}
extern "C" __attribute__((visibility("default"))) int mk_trace_clear() {
    static ulonglong2 zero[mk::kTraceEvents];
    for (int c = 0; c < mk::kTraceCtas; ++c)
        if (cudaMemcpyToSymbol(mk::g_mk_trace, zero, sizeof(zero), sizeof(zero) * c) != cudaSuccess) return 1;
    return 0;
}
#endif
