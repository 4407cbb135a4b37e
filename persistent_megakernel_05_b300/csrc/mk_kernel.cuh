// mk_kernel.cuh -- the persistent decode-step kernel (one launch = one decode step).
//
// Design (pages: "Cohere Megakernel", section "Megakernel ne demek"; "Kog Inference
// Engine", sections on memory bandwidth and the monokernel):
//   * one CTA per SM, launched cooperatively so every CTA is resident;
//   * the step is a fixed list of stages per layer -- QKV tiles, attention key splits
//     (+ a merge of the splits' partial softmax states), O-projection tiles, gate/up
//     tiles, down tiles -- then LM-head tiles and the greedy argmax. Each stage's work
//     is cut into row tiles (GEMV) or page ranges (attention) statically assigned to CTAs;
//   * stages are ordered by the data itself, never by a grid-wide barrier: up to
//     kMaxTaggedBatch rows every activation word carries the tag of the write that
//     produced it (one 64-bit store, no fence), and a reader polls the words it needs;
//     above that, fp32 activations sit behind per-stage counters (release / acquire);
//   * warp 0 of every CTA is the loader: it walks the CTA's own task list and streams
//     every weight row and every KV page the CTA will need into a ring of shared-memory
//     slots with TMA, without waiting on any dependency (weights and old KV rows never
//     depend on this step's activations), so HBM keeps streaming while the consumers
//     wait. It has the SM's scheduler 0 to itself (warps 4 and 8 only exit), so busy
//     consumer warps never starve it of issue slots;
//   * eight consumer warps (warps 1-3, 5-7, 9-10 on schedulers 1-3) compute: exact fp32
//     CUDA-core GEMV for batches up to 2, BF16 mma.sync GEMV tiles above (activations
//     split hi + lo), flash-decode attention on mma.sync with keys in the M dimension and
//     online softmax, fused epilogues (RoPE + KV append, residual add, SwiGLU, partial
//     argmax); warp 11 optionally prefetches the loader's future reads into L2.
// Every wait is bounded; on an error the kernel latches a status word and winds down
// (waits become no-ops, in-flight TMA copies are drained) instead of hanging.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>
#include "mk_ptx.cuh"

namespace mk {

typedef __nv_bfloat16 bf16;

constexpr int kConsumerWarps = 8;
constexpr int kConsumerThreads = 32 * kConsumerWarps;
// Warp roles. An SM schedules warp w on scheduler w mod 4: the loader (warp 0) keeps
// scheduler 0 to itself (warps 4 and 8 exit at once), the consumers are warps 1-3, 5-7,
// 9 and 10, warp 11 is the optional L2 prefetcher.
constexpr int kWarps = 12;
constexpr int kThreads = 32 * kWarps;
constexpr int kPrefetchWarp = 11;
__device__ __forceinline__ bool idle_warp(int w) { return w == 4 || w == 8; }
__device__ __forceinline__ int consumer_index(int w) { return w - 1 - (w > 4) - (w > 8); }
constexpr int kDefaultPrefetchSlots = 0;          // L2 prefetch lead (slots); 0 = off

// Shared-memory ring depth. Five 33 KB slots (165 KB in flight per SM) with the scratch
// and the shared state fit the 196 KB carveout, which leaves ~60 KB of the SM's unified
// L1/shared array to L1 for the consumers' saved registers and the norm-gain reads.
// Measured (alternating runs on one box), ms/step: 2B batch 1: 4 slots 1.033, 5 slots
// 1.019, 6 slots 1.095; 2B batch 8: 2.667, 2.582, 2.602; MoE batch 1: 1.228, 1.225, 1.267.
constexpr int kStages = 5;
constexpr int KCW = 2048;                          // GEMV k-chunk: columns of a weight slot
constexpr int kGroupRows = 8;                      // weight rows per ring slot
constexpr int kSlotBytes = 33 * 1024;              // >= 8 * (2 * KCW + 16), multiple of 1024
constexpr int kScratchBytes = 20 * 1024;
constexpr int kMaxBatch = 8;
constexpr int kPage = 16;
constexpr int kTaskRows = 128;                     // <= 16 row groups of 8 per GEMV task
constexpr int kMaxLayers = 128;
constexpr int kMaxExperts = 64;                    // MoE: experts per layer (one warp routes a row)
constexpr int kMaxTopK = 16;                       // MoE: experts routed per row
constexpr int kMaxSampleTopK = 32;                 // sampling: largest top-k cut (one warp lane each)
constexpr int kCounterStride = 32;                 // u32 words per counter (128 B apart)
constexpr int kStagesPerLayer = 8;                 // counter slots per layer
constexpr int kMaxOwnRows = 32;                    // residual rows a CTA owns: ceil(d / CTAs) <= 32
constexpr int kMaxSplitsG = 1184;                  // splits (<= CTAs) x G (<= 8): merge staging
constexpr int kPieceCache = 4;                     // attention pieces a CTA caches per layer class
constexpr int kPieceWords = 16;                    // 32-bit words of one cached piece (>= sizeof(Piece) / 4)

// ---- optional timeline trace (compile with -DMK_TRACE; no code otherwise) ----
#ifdef MK_TRACE
constexpr int kTraceCtas = 160, kTraceEvents = 2048;  // [cta][consumer 0..1023 | producer 1024..]
__device__ ulonglong2 g_mk_trace[kTraceCtas][kTraceEvents];
__device__ __forceinline__ void trace_event(int cta, int& n, int base, uint32_t code, uint32_t arg) {
    if (cta < kTraceCtas && n < kTraceEvents / 2)
        g_mk_trace[cta][base + n++] = make_ulonglong2(globaltimer(), ((unsigned long long)code << 32) | arg);
}
#define MK_TRACE_C(c, code, arg) do { if ((c).tid == 0) trace_event(blockIdx.x, (c).sm->trace_n, 0, code, arg); } while (0)
#define MK_TRACE_P(pr, code, arg) do { if ((pr).lane == 0 && !(pr).pf) trace_event(blockIdx.x, (pr).tn, kTraceEvents / 2, code, arg); } while (0)
#else
#define MK_TRACE_C(c, code, arg) do { } while (0)
#define MK_TRACE_P(pr, code, arg) do { } while (0)
#endif
// ---- optional section profile (compile with -DMK_PROF; no code otherwise) ----
// Consumer thread 0 of every CTA adds the SM cycles since its previous mark to the
// section named by each mark: a cheap (clock64, no memory traffic) breakdown of where a
// step's time goes, summed over steps until cleared.
#ifdef MK_PROF
constexpr int kProfCtas = 160, kProfSections = 64;
__device__ unsigned long long g_mk_prof[kProfCtas][kProfSections];
// sums accumulate in shared memory (no global round trip inside a section) and are
// flushed to g_mk_prof once at the end of the step
#define MK_PROF_MARK(c, sec) do { if ((c).tid == 0) { \
    const long long t_ = clock64(); (c).sm->prof[sec] += t_ - (c).sm->prof_pt; (c).sm->prof_pt = t_; } } while (0)
#else
#define MK_PROF_MARK(c, sec) do { } while (0)
#endif
// profile sections: GEMV kind k (QKV, O, GU, DOWN, LM, ROUTE) uses 1 + 4k .. 4 + 4k
enum ProfSection { PS_OTHER = 0, PS_G_DATA = 1, PS_G_SLOTS = 2, PS_G_EPI = 3, PS_G_END = 4,
                   PS_A_ENTRY = 25, PS_A_QPOLL = 26, PS_A_QSYNC = 27, PS_A_FRAG = 28, PS_A_LOOP = 29,
                   PS_A_POST = 30, PS_A_FINISH = 31, PS_M_ML = 32, PS_M_W = 33, PS_M_O = 34,
                   PS_A_END = 35, PS_EMBED = 36, PS_ARGMAX = 37, PS_A_LWAIT = 38, PS_G_SWAIT = 39,
                   PS_MOE_ROUTE = 40, PS_L_ISSUE = 41, PS_L_BLOCK = 42, PS_L_DEP = 43,
                   PS_L_SLOTS = 44, PS_L_NBLOCK = 45, PS_T_RET = 46, PS_T_CALL = 47,
                   PS_TOTAL_NS = 62, PS_TOTAL = 63 };
// loader sections (lane 0 of the loader; MK_PROF builds): cycles issuing, cycles waiting
// for a free ring slot, cycles waiting on a routing / step dependency, slots issued,
// slots that found the ring full
#ifdef MK_PROF
#define MK_PROF_L(pr, sec) do { if ((pr).lane == 0 && !(pr).pf) { \
    const long long t_ = clock64(); (pr).sm->prof[sec] += t_ - (pr).ppt; (pr).ppt = t_; } } while (0)
#define MK_PROF_LCOUNT(pr, sec) do { if ((pr).lane == 0 && !(pr).pf) (pr).sm->prof[sec] += 1; } while (0)
#else
#define MK_PROF_L(pr, sec) do { } while (0)
#define MK_PROF_LCOUNT(pr, sec) do { } while (0)
#endif

enum TraceCode { TR_WAIT = 1, TR_READY = 2, TR_DONE = 3, TR_PIECE = 4, TR_MERGE = 5, TR_END = 6,
                 TR_P_STAGE = 11, TR_P_BLOCK = 12, TR_P_GO = 13,
                 TR_S_WAIT = 20, TR_S_FULL = 21, TR_S_REL = 22, TR_S_ISSUE = 23,
                 TR_A_Q = 30, TR_A_LOOP = 31, TR_A_PART = 32, TR_A_ARRIVED = 33, TR_A_MERGED = 34,
                 TR_G_NORM = 40, TR_G_X = 41, TR_G_SUM = 42, TR_G_EPI = 43,
                 TR_Q_LOADED = 50, TR_Q_SYNCED = 51, TR_Q_FRAG = 52, TR_M_ML = 53, TR_M_W = 54, TR_M_O = 55,
                 TR_R_POLLED = 60, TR_R_DONE = 61 };

// error codes (same values as mk_status)
constexpr int kErrInvalid = 1, kErrBadPage = 5, kErrTimeout = 6, kErrInternal = 7;

// stage ids (task id = layer * 16 + stage id)
enum StageId { ST_QKV = 0, ST_ATTN = 1, ST_O = 2, ST_GU = 3, ST_DOWN = 4, ST_ROUTE = 5 };
enum GemvKind { G_QKV = 0, G_O = 1, G_GU = 2, G_DOWN = 3, G_LM = 4, G_ROUTE = 5 };

struct LayerPlan {
    const bf16 *wq, *wk, *wv, *wo, *w_gate, *w_up, *w_down;
    const bf16 *router, *exp_gate, *exp_up, *exp_down;  // MoE layers: [E][d], [E][Fe][d] x2, [E][d][Fe]
    const float *attn_gain, *mlp_gain;  // fp32, permuted column order
    int sliding;
    int pad_;
};

struct Plan {
    int L, d, Hq, Hkv, hd, G, F, V, window, max_pos, maxB, num_pages;
    int E, topk, Fe;                    // MoE: experts, routed per row, expert width (E = 0: dense)
    int hrow;                           // row stride of the SwiGLU activations: max(F, E * Fe)
    float eps, scale;                   // scale = 1/sqrt(hd)
    int C;                              // CTAs in the launch
    int qkv_rows;                       // (Hq + 2 Hkv) * hd
    uint32_t sliding_mask[kMaxLayers / 32];  // bit l: layer l slides (kept with the step
                                        // arguments in shared memory: no global read per use)
    const LayerPlan* layers;            // [L]
    const bf16* embed;
    const bf16* lm_head;
    const float* final_gain;            // fp32, permuted
    const float2* rope;                 // [max_pos][hd/2] (cos, sin)
    // activations between stages, as tagged words (fp32 value | write tag)
    uint64_t* x;                        // [maxB][d]  residual stream, permuted
    uint64_t* qkv;                      // [maxB][qkv_rows] natural order, pre-RoPE
    uint64_t* attn;                     // [maxB][Hq*hd] permuted
    uint64_t* h;                        // [maxB][hrow] permuted (MoE: routed-weighted, by union slot)
    uint64_t* route;                    // [maxB][E] router logits (MoE)
    int* moe_union;                     // [L] experts in each layer's routed union, last step
    uint64_t* part;                     // [maxB*Hkv][C] records: o [G][hd], then (m, l) [G]
    // batches above kMaxTaggedBatch: x, attn, h as plain fp32 (same layouts), published
    // by per-stage counters with release / acquire ordering instead of tags
    float* xf;
    float* attnf;
    float* hf;
    uint32_t* counters;                 // stage counters, kCounterStride apart
    uint64_t* amax;                     // [C][maxB][2] tagged (value, index as float bits)
    uint64_t* cand;                     // [C][maxB][kMaxSampleTopK][2] top-k sampling candidates
    uint32_t* arrivals;                 // (unused by the kernel; zeroed with the counters)
    int* status;                        // [0] code, [1] task
    bf16* kv;                           // paged pool base
};

struct StepArgs {
    // CUtensorMap of the KV pool as [rows][hd] (box 64 x 16, 128B swizzle). It travels in
    // the kernel parameters (grid-constant), so a TMA copy finds its descriptor in the
    // parameter space instead of fetching it from global memory.
    alignas(64) CUtensorMap kv_tmap;
    Plan p;
    const int* tokens;
    const int* positions;
    const int* page_table;
    const int* seq_lens;
    int* next_tokens;
    float* logits;                      // may be null
    int max_pages;
    int B;
    uint32_t epoch;                     // step number mod 2^20, never 0: high bits of every tag
    uint32_t stage_target;              // counter target of every stage: steps since reset * C
    float temperature;                  // 0: greedy; > 0: Gumbel-max sampling
    int top_k;                          // sampling over the top_k largest logits (0: all)
    uint32_t seed_lo, seed_hi;          // Philox key of the sampling draws
    int skip_publish;                   // task id whose outputs are never written, or -1
    int prefetch_slots;                 // L2 prefetch lead over the loader, in slots (0 = off)
    long long timeout_ns;
    // shared prefixes: row b shares its logical pages [0, pf_pages[b]) with the rows of
    // the same leader pf_lead[b] (-1: none); pf_on = 0 when no group is declared
    int pf_on;
    int pf_lead[kMaxBatch];
    int pf_pages[kMaxBatch];
    // decode steps in this launch: step s > 0 takes step s-1's tokens as input, at
    // positions + s; next_tokens is [n_steps][B]; logits (if any) are the last step's
    int n_steps;
    float* logits_last;
};

// Up to this batch size the activations between stages travel as tagged words (one
// read latency per hand-off, no fence) and the GEMVs run on the CUDA cores; above it the
// activations travel as fp32 behind counters (a tagged word doubles the bytes every CTA
// reads and the registers a poll holds) and the GEMVs run on mma.sync tiles, which read
// those fp32 rows. From 3 rows on that pair is faster: 8B shapes at 4 rows 1.845 -> 1.447
// ms per step for 8 layers, 2B shapes at 4 rows -1.4 %, 3 rows unchanged; at 2 rows the
// tensor-core GEMV is a third slower.
constexpr int kMaxTaggedBatch = 2;
__device__ __forceinline__ bool tagged(const StepArgs& a) { return a.B <= kMaxTaggedBatch; }

// counter slots (batches above kMaxTaggedBatch)
__device__ __forceinline__ int cnt_embed() { return 0; }
__device__ __forceinline__ int cnt_stage(int l, int s) { return 1 + l * kStagesPerLayer + s; }

// Tags of the tagged-word writes: (epoch, layer, producer). Two consecutive writes of a
// word never carry the same tag, so a stale word is never taken for the awaited one.
enum TagCode { TAG_EMBED = 0, TAG_QKV = 1, TAG_PART = 2, TAG_ATTN = 3, TAG_O = 4, TAG_GU = 5,
               TAG_DOWN = 6, TAG_ROUTE = 7 };
__device__ __forceinline__ uint32_t tag_of(const StepArgs& a, int l, int code) {
    return (a.epoch << 12) | ((uint32_t)l << 3) | (uint32_t)code;
}

// column permutation of fp32 activation rows: within each 64-column block, thread t of
// an mma quad finds its 16 B-operand values (8 column pairs) in 4 consecutive float4s
__device__ __forceinline__ int perm_col(int k) {
    return (k & ~63) | (((k & 7) >> 1) << 4) | (((k & 63) >> 3) << 1) | (k & 1);
}

struct Smem {
    float rstd[kMaxBatch];
    float amax_v[kMaxBatch];
    int amax_i[kMaxBatch];
    float tk_v[kMaxBatch][kMaxSampleTopK];  // top-k sampling: each row's running top-k logits
    int tk_i[kMaxBatch][kMaxSampleTopK];
    int pos[kMaxBatch];                    // consumers' positions of their current step
    int ppos[kMaxBatch];                   // the loader's positions of its current step
    int tok[kMaxBatch];                    // the next step's input tokens
    volatile int step_ready;               // steps whose K/V appends the loader may read
    int cstep;                             // the consumers' step of this launch
    float ssq[kConsumerWarps][kMaxBatch];  // per-warp sums of squares (fused RMSNorm)
    float xown[kMaxBatch][kMaxOwnRows];    // this CTA's rows of the residual stream
    volatile int abort;
    int bcast;
    volatile uint32_t lseq;  // ring slots the loader has started filling
    int pad_[5];
    // The step arguments, copied from the kernel parameters at entry: every field read
    // during the step is then a shared-memory read. Reads of the parameters through a
    // pointer were served from a cache the instruction stream of this large kernel keeps
    // evicting, and cost a global round trip each (a routing pass of ~2 us took ~12 us).
    StepArgs args;
    __align__(16) LayerPlan lp[2];  // consumers' copies of the plans of layers l (l & 1) and l + 1
    __align__(16) LayerPlan lpl[2]; // the loader's copies (it runs ahead of the consumers)
    // the consumers' attention pieces of the current step, per layer class (full / sliding
    // window): computed at the first layer of each class, reused by the others
    int pc_tag[2];                     // cstep * 2 + class + 1 the pieces below belong to; 0: none
    int pc_n[2];                       // pieces (-1: more than the cache holds)
    __align__(16) int pc_words[2][kPieceCache * kPieceWords];
    // MoE routing of the current layer, written by the consumers, read by the loader too
    volatile int moe_ready;            // step * kMaxLayers + layer + 1 whose routing is below
    int moe_nu;                        // experts in the union of the batch rows' routes
    int moe_uni[kMaxExperts];          // that union, ascending expert id
    float moe_w[kMaxBatch][kMaxExperts];  // routing weight of union slot j for row b (0: not routed)
#ifdef MK_PROF
    unsigned long long prof[64];
    long long prof_pt;                 // cycle count at the last profile mark
#endif
#ifdef MK_TRACE
    int trace_n;                       // consumer trace events recorded
#endif
    uint64_t full[kStages];
    uint64_t empty[kStages];
    __align__(16) bf16 knew[128];
    __align__(16) bf16 vnew[128];
};

constexpr int kSmemBytes = 1024 + kStages * kSlotBytes + kScratchBytes + (int)sizeof(Smem);
// The SM's unified L1 / shared array is split in fixed carveouts; staying within the
// 196 KB one (with the 1 KB the runtime reserves per block) leaves ~60 KB to L1, which
// the consumers' saved registers and gain reads depend on.
static_assert(kSmemBytes + 1024 <= 196 * 1024, "shared memory beyond the 196 KB carveout shrinks L1");

struct Ctx {
    const StepArgs* a;
    Smem* sm;
    uint8_t* ring;       // generic pointer, 1024-aligned
    float* scratch;
    uint32_t ring_s;     // shared address of the ring
    uint32_t seq;        // ring sequence number (slot = seq % kStages)
    int cw, lane, tid;   // consumer warp (0..7), lane, consumer thread id (0..255)
};

// The dynamic shared memory of the kernel: [pad to 1024][ring][scratch][Smem].
extern __shared__ __align__(1024) uint8_t mk_smem[];

// A consumer thread's context, rebuilt from the thread index and the shared-memory base
// wherever it is needed. Functions that are not inlined take the ring sequence number
// and return the advanced one instead of taking the context by reference: a context
// whose address is taken lives in local memory, and its reloads after every call missed
// L1 and waited on L2 in the middle of the step.
__device__ __forceinline__ Ctx make_ctx(uint32_t seq) {
    Ctx c;
    const uint32_t raw_s = smem_u32(mk_smem);
    const uint32_t pad = (1024u - (raw_s & 1023u)) & 1023u;
    c.ring = mk_smem + pad;
    c.ring_s = raw_s + pad;
    c.scratch = reinterpret_cast<float*>(c.ring + kStages * kSlotBytes);
    c.sm = reinterpret_cast<Smem*>(c.ring + kStages * kSlotBytes + kScratchBytes);
    c.a = &c.sm->args;
    c.seq = seq;
    const int warp = (int)(threadIdx.x >> 5);
    c.cw = consumer_index(warp);
    c.lane = (int)(threadIdx.x & 31);
    c.tid = c.cw * 32 + c.lane;
    return c;
}

// ------------------------------------------------------------------ errors / waits
__device__ __forceinline__ void set_error(const Plan& p, Smem* sm, int code, int task) {
    if (atomicCAS(p.status, 0, code) == 0) p.status[1] = task;
    sm->abort = 1;
}

__device__ __forceinline__ bool status_bad(const Plan& p) { return ld_volatile_int(p.status) != 0; }

// wait until counter - target >= 0 (wrapping u32); one thread; false on abort/timeout
__device__ bool poll_counter(const StepArgs& a, Smem* sm, const uint32_t* c, uint32_t target,
                             int task) {
    if (sm->abort) return false;
    uint64_t t0 = 0;
    for (int it = 0;; ++it) {
        uint32_t v = ld_acquire(c);
        if ((int)(v - target) >= 0) return true;
        if (sm->abort) return false;
        if ((it & 7) == 7) {
            if (status_bad(a.p)) { sm->abort = 1; return false; }
            uint64_t t = globaltimer();
            if (t0 == 0) t0 = t;
            else if ((long long)(t - t0) > a.timeout_ns) {
                set_error(a.p, sm, kErrTimeout, task);
                return false;
            }
        }
        if (it > 32) __nanosleep(64);
    }
}

// all consumer threads: wait for a stage counter
__device__ __forceinline__ bool consumer_wait(Ctx& c, int slot, int task) {
    if (c.tid == 0) poll_counter(*c.a, c.sm, c.a->p.counters + slot * kCounterStride, c.a->stage_target, task);
    consumer_sync();
    return !c.sm->abort;
}

// all consumer threads: count this CTA's completion of a stage
__device__ __forceinline__ void publish(Ctx& c, int slot, int task) {
    consumer_sync();
    // bar.sync orders every consumer thread's stores before thread 0's release add
    if (c.tid == 0 && !c.sm->abort && c.a->skip_publish != task)
        red_release_add(c.a->p.counters + slot * kCounterStride, 1u);
}

// Back-off step of a thread polling tagged words: false once the wait must end (the CTA
// aborts, another CTA latched an error, or the time limit passes: kErrTimeout for `task`).
__device__ __noinline__ bool spin_check(const StepArgs& a, Smem* sm, int task, uint64_t* t0) {
    if (status_bad(a.p)) { sm->abort = 1; return false; }
    const uint64_t now = globaltimer();
    if (*t0 == 0) { *t0 = now; return true; }
    if ((long long)(now - *t0) > a.timeout_ns) {
        set_error(a.p, sm, kErrTimeout, task);
        return false;
    }
    return true;
}
struct Spin {
    uint64_t t0 = 0;
    int it = 0;
    __device__ __forceinline__ bool again(const StepArgs& a, Smem* sm, int task) {
        if (sm->abort) return false;
        if ((++it & 63) == 0 && !spin_check(a, sm, task, &t0)) return false;
        if (it > 64) __nanosleep(32);
        return true;
    }
};

// Spin on ONE pair of tagged words until both carry `tag` (false when the wait ends).
// A thread that needs several words and found one missing waits here on that word, so
// that a stalled hand-off costs one read per round instead of one per word; then it
// re-reads the whole set.
__device__ __forceinline__ bool ll_wait_pair(const uint64_t* p, uint32_t tag, Spin& sp, const StepArgs& a,
                                             Smem* sm, int task) {
    for (;;) {
        if (!sp.again(a, sm, task)) return false;
        uint64_t w0, w1;
        ll_ld2(p, w0, w1);
        if (ll_tag(w0) == tag && ll_tag(w1) == tag) return true;
    }
}

// Slow path of every ring wait (one lane): sleep on the barrier phase until it completes
// (true), the CTA aborts, another CTA latches an error, or `limit_ns` passes, which
// latches kErrTimeout for `task` (false). Out of line: it is cold code.
__device__ __noinline__ bool ring_wait_slow(const StepArgs* a, Smem* sm, uint32_t bar, uint32_t parity,
                                            long long limit_ns, int task) {
    const uint64_t t0 = globaltimer();
    for (int it = 0;; ++it) {
        if (mbar_wait_sleep(bar, parity, 20000u)) return true;
        if (sm->abort) return false;
        if ((it & 7) == 7) {
            if (status_bad(a->p)) { sm->abort = 1; return false; }
            if ((long long)(globaltimer() - t0) > limit_ns) {
                set_error(a->p, sm, kErrTimeout, task);
                return false;
            }
        }
    }
}

// a consumer warp waits for ring slot `seq` to be full; warp-uniform result
__device__ __forceinline__ bool wait_full(Ctx& c, int task) {
    const uint32_t slot = c.seq % kStages, parity = (c.seq / kStages) & 1;
    const uint32_t bar = smem_u32(&c.sm->full[slot]);
    int ok = 1;
    if (c.lane == 0) {
        if (c.sm->abort) ok = 0;
        else if (!mbar_try_wait(bar, parity))
            ok = ring_wait_slow(c.a, c.sm, bar, parity, c.a->timeout_ns, task);
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) mbar_try_wait(bar, parity);  // every lane acquires the completed phase
    return ok != 0;
}

__device__ __forceinline__ void release_slot(Ctx& c) {
    __syncwarp();
    if (c.lane == 0 && !c.sm->abort) mbar_arrive(smem_u32(&c.sm->empty[c.seq % kStages]));
    c.seq++;
}

// ------------------------------------------------------------------ schedule
__device__ __forceinline__ void cta_rows(int R, int cta, int C, int& r0, int& r1) {
    // 32-bit unsigned products: R * C < 2^32 for every stage (checked on the host)
    r0 = (int)((uint32_t)cta * (uint32_t)R / (uint32_t)C);
    r1 = (int)((uint32_t)(cta + 1) * (uint32_t)R / (uint32_t)C);
}

struct GemvStage {
    int kind, layer, R, K, task_id;
    int ldw;                     // elements between consecutive weight rows
    int kcw;                     // columns per k-chunk (one ring slot holds 8 rows of a chunk)
    int lds;                     // elements between source rows
    int moe;                     // 0 dense; 1 MoE gate/up over the routed union; 2 MoE down
    int Fe;                      // MoE expert width
    const int* uni;              // MoE: the routed union (ascending expert id), in shared memory
    uint32_t src_tag, out_tag;   // tag awaited on every source word / written on the outputs
    const bf16 *w0, *w1, *w2;
    int split1, split2;          // QKV: row boundaries between wq / wk / wv
    const uint64_t* src;         // B operand source rows [b][K] (tagged words), permuted
    const float* srcf;           // the same rows as fp32 (batches above kMaxTaggedBatch)
    int cnt_wait, cnt_pub;       // counter slots (batches above kMaxTaggedBatch)
    const float* gain;           // permuted fp32 gain or null (no norm)
};

// `lp` is layer l's plan (the consumers keep a copy in shared memory); `sm` supplies the
// routed union of a MoE layer (read only for its gate/up and down stages)
__device__ GemvStage make_gemv(const StepArgs& a, int kind, int l, const LayerPlan& lp, const Smem* sm) {
    const Plan& p = a.p;
    GemvStage s;
    s.kind = kind;
    s.layer = l;
    s.w1 = s.w2 = nullptr;
    s.split1 = s.split2 = 0;
    s.gain = nullptr;
    s.out_tag = 0;
    s.kcw = KCW;
    s.moe = 0;
    s.Fe = p.Fe;
    s.uni = nullptr;
    if (kind == G_LM) {
        s.R = p.V; s.K = p.d; s.w0 = p.lm_head; s.src = p.x; s.srcf = p.xf; s.gain = p.final_gain;
        s.task_id = p.L * 16; s.src_tag = tag_of(a, p.L - 1, TAG_DOWN);
        s.cnt_wait = cnt_stage(p.L - 1, ST_DOWN); s.cnt_pub = -1;
        s.ldw = s.lds = s.K;
        return s;
    }
    switch (kind) {
        case G_QKV:
            s.R = p.qkv_rows; s.K = p.d; s.w0 = lp.wq; s.w1 = lp.wk; s.w2 = lp.wv;
            s.split1 = p.Hq * p.hd; s.split2 = (p.Hq + p.Hkv) * p.hd;
            s.src = p.x; s.srcf = p.xf; s.gain = lp.attn_gain; s.task_id = l * 16 + ST_QKV;
            s.src_tag = l == 0 ? tag_of(a, 0, TAG_EMBED) : tag_of(a, l - 1, TAG_DOWN);
            s.out_tag = tag_of(a, l, TAG_QKV);
            s.cnt_wait = l == 0 ? cnt_embed() : cnt_stage(l - 1, ST_DOWN);
            s.cnt_pub = -1;  // q|k|v always travel as tagged words
            break;
        case G_O:
            s.R = p.d; s.K = p.Hq * p.hd; s.w0 = lp.wo; s.src = p.attn; s.srcf = p.attnf;
            s.task_id = l * 16 + ST_O;
            s.src_tag = tag_of(a, l, TAG_ATTN);
            s.out_tag = tag_of(a, l, TAG_O);
            s.cnt_wait = cnt_stage(l, ST_ATTN); s.cnt_pub = cnt_stage(l, ST_O);
            break;
        case G_ROUTE:  // router logits of a MoE layer (always tagged words)
            s.R = p.E; s.K = p.d; s.w0 = lp.router; s.src = p.x; s.srcf = p.xf;
            s.gain = lp.mlp_gain; s.task_id = l * 16 + ST_ROUTE;
            s.src_tag = tag_of(a, l, TAG_O);
            s.out_tag = tag_of(a, l, TAG_ROUTE);
            s.cnt_wait = cnt_stage(l, ST_O); s.cnt_pub = -1;
            break;
        case G_GU:
            s.K = p.d; s.src = p.x; s.srcf = p.xf;
            s.gain = lp.mlp_gain; s.task_id = l * 16 + ST_GU;
            s.src_tag = tag_of(a, l, TAG_O);
            s.out_tag = tag_of(a, l, TAG_GU);
            s.cnt_wait = cnt_stage(l, ST_O); s.cnt_pub = cnt_stage(l, ST_GU);
            if (p.E > 0) {  // rows = (union slot, expert row) pairs
                s.moe = 1; s.uni = sm->moe_uni; s.R = sm->moe_nu * p.Fe;
                s.w0 = lp.exp_gate; s.w1 = lp.exp_up;
            } else {
                s.R = p.F; s.w0 = lp.w_gate; s.w1 = lp.w_up;
            }
            break;
        default:  // G_DOWN
            s.R = p.d; s.src = p.h; s.srcf = p.hf;
            s.task_id = l * 16 + ST_DOWN;
            s.src_tag = tag_of(a, l, TAG_GU);
            s.out_tag = tag_of(a, l, TAG_DOWN);
            s.cnt_wait = cnt_stage(l, ST_GU); s.cnt_pub = cnt_stage(l, ST_DOWN);
            if (p.E > 0) {
                // one dense GEMV over the union's columns side by side (union slot j holds
                // columns [j Fe, (j + 1) Fe)): row r of the virtual matrix is the
                // concatenation of row r of each union expert's [d][Fe] down matrix. The
                // loader gathers each 2048-column chunk of a row from those matrices.
                s.moe = 2; s.uni = sm->moe_uni; s.K = sm->moe_nu * p.Fe;
                s.w0 = lp.exp_down; s.kcw = KCW; s.ldw = 0; s.lds = p.hrow;
                return s;
            }
            s.K = p.F; s.w0 = lp.w_down;
            s.ldw = s.K; s.lds = p.hrow;
            return s;
    }
    s.ldw = s.lds = s.K;
    return s;
}
__device__ __forceinline__ GemvStage make_gemv(const StepArgs& a, int kind, int l, const Smem* sm) {
    return make_gemv(a, kind, l, a.p.layers[kind == G_LM ? 0 : l], sm);
}

// stages whose individual ring slots are traced in MK_TRACE builds
__device__ __forceinline__ bool trace_slots(const GemvStage& s) {
    return s.kind == G_LM || (s.layer == 1 && s.kind == G_GU);
}

// rows per task: GU tasks count gate/up row PAIRS (<= 64 pairs = 8 + 8 row groups)
__device__ __forceinline__ int task_rows(int kind) { return kind == G_GU ? kTaskRows / 2 : kTaskRows; }

// Row groups of 8 weight rows; GU tasks list their gate groups first, then up groups.
__device__ __forceinline__ int num_groups(const GemvStage& s, int n) {
    const int g = (n + kGroupRows - 1) / kGroupRows;
    return s.kind == G_GU ? 2 * g : g;
}
__device__ __forceinline__ int group_rows(const GemvStage& s, int n, int gi, int ngate) {
    const int base = kGroupRows * (s.kind == G_GU && gi >= ngate ? gi - ngate : gi);
    return min(kGroupRows, n - base);
}
// weight row i of row group gi, as a pointer to its first column (of k-chunk 0)
__device__ __forceinline__ const bf16* gemv_row(const GemvStage& s, int r0, int gi, int ngate, int i) {
    if (s.kind == G_GU) {
        const bool up = gi >= ngate;
        int r = r0 + kGroupRows * (up ? gi - ngate : gi) + i;
        if (s.moe) r = s.uni[r / s.Fe] * s.Fe + r % s.Fe;  // (union slot, row) -> expert row
        return (up ? s.w1 : s.w0) + (size_t)r * s.ldw;
    }
    const int r = r0 + kGroupRows * gi + i;
    if (s.kind == G_QKV) {
        if (r < s.split1) return s.w0 + (size_t)r * s.ldw;
        if (r < s.split2) return s.w1 + (size_t)(r - s.split1) * s.ldw;
        return s.w2 + (size_t)(r - s.split2) * s.ldw;
    }
    return s.w0 + (size_t)r * s.ldw;
}
// element offset of k-chunk k0 within a weight row (not used for the MoE down
// projection, whose chunks are gathered from several expert matrices)
__device__ __forceinline__ size_t chunk_base(const GemvStage& s, int k0) {
    return (size_t)k0;
}

// Shared-memory geometry of one weight slot (8 rows x kc columns of k-chunk k0). Each
// row segment travels in its own copy; rows are kc * 2 + 16 bytes apart, so the 8 rows
// that one ldmatrix reads at the same column start in 8 different 16-byte bank groups
// (kc is a multiple of 64, so the pitch is 16 modulo 128).
struct SlotGeom {
    int kc, pitch;
    __device__ __forceinline__ int row_off(int r) const { return r * pitch; }
};
__device__ __forceinline__ SlotGeom slot_geom(const GemvStage& s, int k0) {
    SlotGeom g;
    g.kc = min(s.kcw, s.K - k0);
    g.pitch = g.kc * 2 + 16;
    return g;
}

// ---- attention work partition (identical in producer and consumers) ----
struct SeqSpan { int lo, pos, p0, np; };  // attended keys [lo, pos], logical pages [p0, p0+np)

__device__ __forceinline__ SeqSpan seq_span(const Plan& p, const int* posv, int l, int b) {
    SeqSpan s;
    s.pos = posv[b];
    const bool slides = (p.sliding_mask[l >> 5] >> (l & 31)) & 1u;
    s.lo = (p.window > 0 && slides) ? max(0, s.pos - p.window + 1) : 0;
    s.p0 = s.lo / kPage;
    s.np = s.pos / kPage - s.p0 + 1;
    return s;
}

// ---- shared prefixes (cascade attention) ----
// Rows whose leading logical pages are the same physical pages form a group (declared by
// the caller). In a layer where every row of a group attends its whole prefix (lo = 0)
// and keeps its current page to itself, the group's prefix pages are read once for all
// its rows: one item whose query columns are the rows' G heads side by side (at most 16
// columns, two 8-wide MMA column tiles), whose partial records go to every row's merge.
// Packed per row: lead (4 bits, leader + 1, 0 = none); rows of a leader (8 bits).
struct Groups {
    uint32_t lead;
    uint64_t rows;
    __device__ __forceinline__ int leader(int b) const { return (int)((lead >> (4 * b)) & 15u) - 1; }
    __device__ __forceinline__ uint32_t members(int L) const { return (uint32_t)(rows >> (8 * L)) & 0xffu; }
};

__device__ __forceinline__ Groups prefix_groups(const StepArgs& a, const int* posv, int l) {
    Groups gr{0u, 0ull};
    if (!a.pf_on) return gr;
    uint64_t rows = 0;
    for (int b = 0; b < a.B; ++b) {
        const int L = a.pf_lead[b];
        if (L >= 0 && L < a.B && a.pf_pages[L] > 0) rows |= 1ull << (8 * L + b);
    }
    for (int L = 0; L < a.B; ++L) {
        const uint32_t m = (uint32_t)(rows >> (8 * L)) & 0xffu;
        if (__popc(m) < 2) continue;
        bool ok = true;
        for (int r = 0; r < a.B; ++r)
            if ((m >> r) & 1u) {
                const SeqSpan sp = seq_span(a.p, posv, l, r);
                ok = ok && sp.lo == 0 && a.pf_pages[L] <= sp.pos / kPage;
            }
        if (!ok) continue;
        gr.rows |= (uint64_t)m << (8 * L);
        for (int r = 0; r < a.B; ++r)
            if ((m >> r) & 1u) gr.lead |= (uint32_t)(L + 1) << (4 * r);
    }
    return gr;
}

// One attention piece: pages [sp.p0 + u, sp.p0 + u + n) of an item (a row's pages, a
// row's private pages after its group's prefix, or a group's shared prefix).
struct Piece {
    SeqSpan sp;      // the item's pages [p0, p0 + np), keys [lo, pos]
    int b, g;        // row whose page table the item walks (a prefix: the leader), kv head
    uint32_t rows;   // rows whose queries the piece serves (bit mask)
    int u, n;        // the piece within the item
    int split, nsplit;
    int slot0;       // partial-record slot of split 0 (after the records of the row's prefix)
    int nrec;        // records the row's merge reads (prefix pieces + its own)
    bool prefix;     // a shared-prefix piece: writes records for every row, merges nothing
};
static_assert(sizeof(Piece) <= 4 * kPieceWords && alignof(Piece) <= 4, "a cached piece fits its words");

// Calls f(piece) for each attention piece of this CTA. Work items are (row b, kv head g)
// with np(b) pages each, plus one item per (active prefix group, g). When there are no
// more items than CTAs, every item gets CTAs of its own, in proportion to its pages and
// at least one: with C' = C - W spare CTAs and S_i the pages of the items before item i,
// item i takes CTAs [i + C' S_i / U, i + 1 + C' S_(i+1) / U) and splits its pages evenly
// over min(CTAs, pages) of them. No CTA then carries the fixed cost of two pieces (those
// CTAs would finish last and every merge would wait for them). With more items than
// CTAs (no prefix groups then), (b, g, page) units are dealt out in contiguous ranges.
// Items of one row each (no prefix groups): (b, g) in row-major order.
template <typename F>
__device__ __forceinline__ void for_each_row_piece(const StepArgs& a, const int* posv, int l, int cta, F&& f) {
    const Plan& p = a.p;
    uint32_t U = 0;
    for (int b = 0; b < a.B; ++b) U += (uint32_t)(p.Hkv * seq_span(p, posv, l, b).np);
    const uint32_t C = (uint32_t)p.C;
    const uint32_t W = (uint32_t)(a.B * p.Hkv);
    Piece pc;
    pc.slot0 = 0;
    pc.prefix = false;
    if (W <= C) {
        const uint32_t Cp = C - W;
        uint32_t S = 0, i = 0;
        for (int b = 0; b < a.B; ++b) {
            const SeqSpan sp = seq_span(p, posv, l, b);
            for (int g = 0; g < p.Hkv; ++g, ++i) {
                const uint32_t c0 = i + Cp * S / U;
                S += (uint32_t)sp.np;
                const uint32_t c1 = i + 1 + Cp * S / U;
                if ((uint32_t)cta < c1) {
                    const int nsplit = min((int)(c1 - c0), sp.np), k = cta - (int)c0;
                    if (k < nsplit) {
                        pc.sp = sp;
                        pc.b = b; pc.g = g; pc.rows = 1u << b;
                        pc.u = (int)((uint32_t)k * sp.np / nsplit);
                        pc.n = (int)((uint32_t)(k + 1) * sp.np / nsplit) - pc.u;
                        pc.split = k; pc.nsplit = nsplit; pc.nrec = nsplit;
                        f(pc);
                    }
                    return;
                }
            }
        }
        return;
    }
    const uint32_t u0 = (uint32_t)cta * U / C, u1 = (uint32_t)(cta + 1) * U / C;
    if (u0 >= u1) return;
    auto first_cta = [&](uint32_t s) -> int { return (int)(((s + 1) * C - 1) / U); };
    uint32_t s = 0;
    for (int b = 0; b < a.B; ++b) {
        const SeqSpan sp = seq_span(p, posv, l, b);
        for (int g = 0; g < p.Hkv; ++g) {
            const uint32_t e = s + (uint32_t)sp.np;
            const uint32_t lo = max(s, u0), hi = min(e, u1);
            if (lo < hi) {
                const int c0 = first_cta(s);
                pc.sp = sp;
                pc.b = b; pc.g = g; pc.rows = 1u << b;
                pc.u = (int)(lo - s); pc.n = (int)(hi - lo);
                pc.split = cta - c0; pc.nsplit = first_cta(e - 1) - c0 + 1;
                pc.nrec = pc.nsplit;
                f(pc);
            }
            s = e;
            if (s >= u1) return;
        }
    }
}

template <typename F>
__device__ __forceinline__ void for_each_group_piece(const StepArgs& a, const int* posv, int l, int cta, F& f);

template <typename F>
__device__ __forceinline__ void for_each_piece(const StepArgs& a, const int* posv, int l, int cta, F&& f) {
    if (!a.pf_on) for_each_row_piece(a, posv, l, cta, f);
    else for_each_group_piece(a, posv, l, cta, f);
}

// for_each_piece with shared-prefix groups declared (inlined like the rest: a call would
// put the callers' captured state in local memory)
template <typename F>
__device__ __forceinline__ void for_each_group_piece(const StepArgs& a, const int* posv, int l, int cta, F& f) {
    const Plan& p = a.p;
    // 32-bit unsigned unit arithmetic: U * C < 2^31 (checked on the host)
    const uint32_t C = (uint32_t)p.C;
    const Groups gr = prefix_groups(a, posv, l);
    int ng = 0;
    for (int L = 0; L < a.B; ++L) ng += gr.members(L) != 0u;
    const uint32_t W = (uint32_t)((a.B + ng) * p.Hkv);
    // no active group in this layer, or more items than CTAs: every row on its own
    if (ng == 0 || W > C) {
        for_each_row_piece(a, posv, l, cta, f);
        return;
    }
    {
        uint32_t U = 0;
        for (int b = 0; b < a.B; ++b) {
            const SeqSpan sp = seq_span(p, posv, l, b);
            const int L = gr.leader(b);
            if (L == b) U += (uint32_t)a.pf_pages[L];
            U += (uint32_t)(L >= 0 ? sp.pos / kPage - a.pf_pages[L] + 1 : sp.np);
        }
        U *= (uint32_t)p.Hkv;
        const uint32_t Cp = C - W;
        uint32_t S = 0, i = 0;
        int ncs[kMaxBatch];  // splits of each group's prefix item (this kv head)
        for (int g = 0; g < p.Hkv; ++g) {
            for (int b = 0; b < a.B; ++b) {
                const SeqSpan full = seq_span(p, posv, l, b);
                const int L = gr.leader(b);
                if (L == b) {  // the group's shared prefix, ahead of its rows' own pages
                    const int P = a.pf_pages[L];
                    const uint32_t c0 = i + Cp * S / U;
                    S += (uint32_t)P;
                    const uint32_t c1 = i + 1 + Cp * S / U;
                    ++i;
                    const int ns = min((int)(c1 - c0), P);
                    ncs[b] = ns;
                    if ((uint32_t)cta < c1) {
                        const int k = cta - (int)c0;
                        if (k < ns) {
                            Piece pc;
                            pc.sp = SeqSpan{0, full.pos, 0, P};
                            pc.b = b; pc.g = g; pc.rows = gr.members(L);
                            pc.u = (int)((uint32_t)k * P / ns);
                            pc.n = (int)((uint32_t)(k + 1) * P / ns) - pc.u;
                            pc.split = k; pc.nsplit = ns; pc.slot0 = 0; pc.nrec = ns; pc.prefix = true;
                            f(pc);
                        }
                        return;
                    }
                }
                SeqSpan sp = full;
                int slot0 = 0;
                if (L >= 0) {  // the row's pages after its group's prefix
                    sp.p0 = a.pf_pages[L];
                    sp.np = full.pos / kPage - sp.p0 + 1;
                    slot0 = ncs[L];
                }
                const uint32_t c0 = i + Cp * S / U;
                S += (uint32_t)sp.np;
                const uint32_t c1 = i + 1 + Cp * S / U;
                ++i;
                if ((uint32_t)cta < c1) {
                    const int ns = min((int)(c1 - c0), sp.np), k = cta - (int)c0;
                    if (k < ns) {
                        Piece pc;
                        pc.sp = sp;
                        pc.b = b; pc.g = g; pc.rows = 1u << b;
                        pc.u = (int)((uint32_t)k * sp.np / ns);
                        pc.n = (int)((uint32_t)(k + 1) * sp.np / ns) - pc.u;
                        pc.split = k; pc.nsplit = ns; pc.slot0 = slot0; pc.nrec = slot0 + ns;
                        pc.prefix = false;
                        f(pc);
                    }
                    return;
                }
            }
        }
    }
}

// ------------------------------------------------------------------ producer (warp 0)
// All 32 lanes walk the same schedule (warp-uniform control flow); lane 0 owns the
// ring barriers and up to 16 lanes issue the row / page copies of a slot in parallel.
struct Producer {
    const StepArgs* a;
    Smem* sm;
    uint32_t ring_s;
    uint32_t seq = 0;
    uint64_t policy;
    int lane;
    int tn = 0;  // trace events recorded (MK_TRACE builds)
    const CUtensorMap* tmap;  // the KV tensor map, in the kernel parameters
    // Prefetch mode: the same schedule walked ahead of the loader, each copy replaced by
    // an L2 prefetch of its source, so that HBM keeps streaming while the consumers wait
    // on a dependency and the loader on a full ring. It never blocks anyone and never
    // reports errors: when anything goes wrong it simply stops.
    bool pf = false;
    // page-table batch cache: ids of logical pages [pt_lp0, pt_lp0 + 32) of sequence pt_b
    int pt_b = -1, pt_lp0 = 0, pt_ids = -1;
#ifdef MK_PROF
    long long ppt = 0;  // cycle count at the loader's last profile mark
#endif

    __device__ __forceinline__ bool acquire_slot(int task) {
        if (pf) {
            int ok = 1;
            if (lane == 0) {
                const uint32_t lead = (uint32_t)a->prefetch_slots;
                uint64_t t0 = 0;
                for (int it = 0; seq >= sm->lseq + lead; ++it) {
                    if (sm->abort) { ok = 0; break; }
                    __nanosleep(128);
                    if ((it & 63) == 63) {
                        const uint64_t now = globaltimer();
                        if (t0 == 0) t0 = now;
                        else if ((long long)(now - t0) > a->timeout_ns) { ok = 0; break; }
                    }
                }
            }
            return __shfl_sync(0xffffffffu, ok, 0) != 0;
        }
        if (lane == 0) sm->lseq = seq;
        int ok = 1;
        MK_PROF_L(*this, PS_L_ISSUE);
        MK_PROF_LCOUNT(*this, PS_L_SLOTS);
        if (lane == 0) {
            if (sm->abort) ok = 0;
            else if (seq >= (uint32_t)kStages) {
                const uint32_t bar = smem_u32(&sm->empty[seq % kStages]);
                const uint32_t parity = ((seq / kStages) - 1) & 1;
                if (!mbar_try_wait(bar, parity)) {
                    MK_PROF_LCOUNT(*this, PS_L_NBLOCK);
                    MK_TRACE_P(*this, TR_P_BLOCK, task);
                    // a full ring only stalls when a consumer stalls; let the consumer's
                    // own (shorter) wait report the cause first
                    ok = ring_wait_slow(a, sm, bar, parity, 4 * a->timeout_ns, task);
                    MK_TRACE_P(*this, TR_P_GO, task);
                }
            }
        }
        MK_PROF_L(*this, PS_L_BLOCK);
        return __shfl_sync(0xffffffffu, ok, 0) != 0;
    }
    __device__ __forceinline__ void copy(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
        if (pf) l2_prefetch_1d(src, bytes);
        else tma_load_1d(dst, src, bytes, bar, policy);
    }
    __device__ __forceinline__ uint32_t slot_addr() const { return ring_s + (seq % kStages) * kSlotBytes; }
    __device__ __forceinline__ uint32_t full_bar() const { return smem_u32(&sm->full[seq % kStages]); }

    __device__ __forceinline__ bool gemv(const GemvStage& s, int cta) {
        MK_TRACE_P(*this, TR_P_STAGE, s.task_id);
        int a0, a1;
        cta_rows(s.R, cta, a->p.C, a0, a1);
        const int tr = task_rows(s.kind);
        for (int r0 = a0; r0 < a1; r0 += tr) {
            const int r1 = min(a1, r0 + tr);
            const int n = r1 - r0;
            const int ng = num_groups(s, n), ngate = s.kind == G_GU ? ng / 2 : ng;
            for (int k0 = 0; k0 < s.K; k0 += s.kcw) {
                const SlotGeom geo = slot_geom(s, k0);
                const size_t cb = chunk_base(s, k0);
                for (int gi = 0; gi < ng; ++gi) {
                    if (!acquire_slot(s.task_id)) return false;
                    const int nr = group_rows(s, n, gi, ngate);
                    const uint32_t dst = slot_addr(), bar = full_bar();
                    if (lane == 0 && !pf) mbar_arrive_expect_tx(bar, (uint32_t)(nr * geo.kc * 2));
                    __syncwarp();
                    if (s.moe == 2) {
                        // MoE down projection: row i's columns [k0, k0 + kc) come from the
                        // union experts they belong to; lane (i, segment) copies one piece
                        const int i = lane >> 2;
                        if (i < nr) {
                            const int r = r0 + kGroupRows * gi + i;
                            for (int j = k0 / s.Fe + (lane & 3); j * s.Fe < k0 + geo.kc; j += 4) {
                                const int c0 = max(k0, j * s.Fe), c1 = min(k0 + geo.kc, (j + 1) * s.Fe);
                                const bf16* src = s.w0 + ((size_t)s.uni[j] * s.R + r) * s.Fe + (c0 - j * s.Fe);
                                copy(dst + i * geo.pitch + (c0 - k0) * 2, src, (uint32_t)((c1 - c0) * 2), bar);
                            }
                        }
                    } else if (lane < nr) {
                        copy(dst + lane * geo.pitch, gemv_row(s, r0, gi, ngate, lane) + cb,
                             (uint32_t)(geo.kc * 2), bar);
                    }
                    if (trace_slots(s) && !pf) MK_TRACE_P(*this, TR_S_ISSUE, seq);
                    ++seq;
                }
            }
        }
        return true;
    }

    bool last_ok = true;  // result of the out-of-line shared-prefix walk

    // The attention stage: without shared-prefix groups inline; with them out of line
    // (a rare path whose code would otherwise sit in the loader's hot loop).
    template <int HD>
    __device__ __forceinline__ bool attention(int l, int cta);

    template <int HD, bool GROUPS>
    __device__ __forceinline__ bool attention_walk(int l, int cta) {
        const Plan& p = a->p;
        constexpr int PPS = 512 / HD;   // pages per ring slot (K + V of one kv head)
        constexpr int NB = HD / 64;     // 64-wide boxes per page row
        MK_TRACE_P(*this, TR_P_STAGE, l * 16 + ST_ATTN);
        bool ok = true;
        auto walk = [&](const Piece& pc) {
            if (!ok) return;
            const int b = pc.b, g = pc.g, u = pc.u, n = pc.n;
            const SeqSpan& sp = pc.sp;
            const int* pt = a->page_table + (size_t)b * a->max_pages;
            for (int st = 0; st < n; st += PPS) {
                const int np = min(PPS, n - st);
                // page ids travel in batches of 32 (lane i holds logical page lp0 + i), kept
                // across pieces and layers: one page-table read serves every layer that
                // walks the same pages
                const int want = sp.p0 + u + st;
                if (b != pt_b || want < pt_lp0 || want + np > pt_lp0 + 32) {
                    pt_b = b;
                    pt_lp0 = want;
                    pt_ids = want + lane < a->max_pages ? __ldg(pt + want + lane) : -1;
                }
                if (!acquire_slot(l * 16 + ST_ATTN)) { ok = false; return; }
                const int nbox = np * 2 * NB;  // <= 16
                const int i = lane / (2 * NB), kv = (lane / NB) & 1, bx = lane % NB;
                const int page = __shfl_sync(0xffffffffu, pt_ids, (want - pt_lp0 + i) & 31);
                bool bad = false;
                if (lane < nbox) bad = page < 0 || page >= p.num_pages;
                if (__any_sync(0xffffffffu, bad)) {
                    if (lane == 0 && !pf) set_error(p, sm, kErrBadPage, l * 16 + ST_ATTN);
                    ok = false;
                    return;
                }
                const uint32_t dst = slot_addr(), bar = full_bar();
                if (lane == 0 && !pf) mbar_arrive_expect_tx(bar, (uint32_t)(np * 2 * 2 * kPage * HD));
                __syncwarp();
                if (lane < nbox) {
                    const int row = (((l * p.num_pages + page) * 2 + kv) * p.Hkv + g) * kPage;
                    if (pf) l2_prefetch_2d(tmap, bx * 64, row);
                    else tma_load_2d(dst + i * 64 * HD + kv * 32 * HD + bx * 2048, tmap, bx * 64, row,
                                     bar, policy);
                }
                if (l == 1 && !pf) MK_TRACE_P(*this, TR_S_ISSUE, seq);
                ++seq;
            }
        };
        if (GROUPS) for_each_group_piece(*a, sm->ppos, l, cta, walk);
        else for_each_row_piece(*a, sm->ppos, l, cta, walk);
        return ok;
    }

    // A MoE layer's expert rows depend on its routing, which this CTA's consumers compute
    // from the router logits: wait until they publish it (bounded; on abort or time-out
    // the loader stops, and the consumers report the cause).
    __device__ __forceinline__ bool wait_route(int step, int l) {
        int ok = 1;
        if (lane == 0) {
            uint64_t t0 = 0;
            for (int it = 0; sm->moe_ready != step * kMaxLayers + l + 1; ++it) {
                if (sm->abort) { ok = 0; break; }
                __nanosleep(64);
                if ((it & 63) == 63) {
                    const uint64_t now = globaltimer();
                    if (t0 == 0) t0 = now;
                    else if ((long long)(now - t0) > 4 * a->timeout_ns) {
                        if (!pf) set_error(a->p, sm, kErrTimeout, l * 16 + ST_ROUTE);
                        ok = 0;
                        break;
                    }
                }
            }
            __threadfence_block();
        }
        __syncwarp();
        return __shfl_sync(0xffffffffu, ok, 0) != 0;
    }

    // Step `step` of a multi-step launch reads pages that the previous step appended to
    // (in other CTAs, by generic stores): wait until this CTA's consumers have seen every
    // CTA finish that step (each released its stores before its argmax record), then
    // order the coming TMA reads after that (bounded; on abort or time-out: stop).
    __device__ __forceinline__ bool wait_step(int step) {
        int ok = 1;
        if (lane == 0) {
            uint64_t t0 = 0;
            for (int it = 0; sm->step_ready < step; ++it) {
                if (sm->abort) { ok = 0; break; }
                __nanosleep(64);
                if ((it & 63) == 63) {
                    const uint64_t now = globaltimer();
                    if (t0 == 0) t0 = now;
                    else if ((long long)(now - t0) > 4 * a->timeout_ns) { ok = 0; break; }
                }
            }
            __threadfence_block();
        }
        __syncwarp();
        fence_proxy_async_global();
        return __shfl_sync(0xffffffffu, ok, 0) != 0;
    }

    template <int HD, bool MULTI>
    __device__ __forceinline__ void run(int cta) {
        policy = policy_evict_first();
        if (lane == 0) prefetch_tmap(tmap);
#ifdef MK_PROF
        ppt = clock64();
#endif
        const Plan& p = a->p;
        bool ok = !sm->abort;
        const int nsteps = MULTI ? a->n_steps : 1;
        // The loader keeps its own double-buffered copy of the layer plans in shared
        // memory: layer l + 1's plan is fetched while layer l streams, so a stage start
        // never waits on a global read. (The L2 prefetch walker reads them from global
        // memory: it must not touch the loader's buffers.)
        static_assert(sizeof(LayerPlan) / 16 <= 32, "a layer plan copies in one warp pass");
        auto fetch_plan = [&](int l) {
            if (!pf && lane < (int)(sizeof(LayerPlan) / 16))
                cp_async_16(smem_u32(&sm->lpl[l & 1]) + 16 * lane,
                            reinterpret_cast<const uint8_t*>(p.layers + l) + 16 * lane);
        };
        auto plan = [&](int l) -> const LayerPlan& { return pf ? p.layers[l] : sm->lpl[l & 1]; };
        for (int step = 0; step < nsteps && ok; ++step) {
            if (MULTI && step > 0 && lane < a->B) sm->ppos[lane] += 1;
            fetch_plan(0);
            __syncwarp();
            // the stages in order, as one loop with a single copy of the GEMV walker (a
            // compact loader keeps the step's instruction working set small): (layer l,
            // stage st) = QKV, attention, O, [router], gate/up, down; then the LM head
            for (int l = 0, st = 0; ok;) {
                if (st == 0 && l < p.L) {
                    cp_async_wait_all();  // layer l's plan is in place
                    __syncwarp();
                    if (l + 1 < p.L) fetch_plan(l + 1);  // slot (l + 1) & 1 held layer l - 1
                }
                int kind;
                if (l == p.L) kind = G_LM;
                else if (st == 0) kind = G_QKV;
                else if (st == 1) kind = -1;  // attention
                else if (st == 2) kind = G_O;
                else if (st == 3) kind = G_ROUTE;
                else kind = st == 4 ? G_GU : G_DOWN;
                if (kind == -1) {
                    if (MULTI && step > 0 && l == 0) ok = wait_step(step);
                    ok = ok && attention<HD>(l, cta);
                } else {
                    if (kind == G_GU && p.E > 0) {
                        MK_PROF_L(*this, PS_L_ISSUE);
                        ok = wait_route(step, l);
                        MK_PROF_L(*this, PS_L_DEP);
                    }
                    const LayerPlan& lp = kind == G_LM ? p.layers[0] : plan(l);
                    ok = ok && gemv(make_gemv(*a, kind, kind == G_LM ? 0 : l, lp, sm), cta);
                }
                if (kind == G_LM) break;
                st += (st == 2 && p.E == 0) ? 2 : 1;  // dense layers have no router stage
                if (st == 6) { st = 0; ++l; }
            }
        }
        MK_PROF_L(*this, PS_L_ISSUE);
        // drain: never leave a copy in flight into shared memory
        if (lane == 0 && !pf) {
            const uint32_t first = seq > (uint32_t)kStages ? seq - kStages : 0;
            for (uint32_t k = first; k < seq; ++k) {
                const uint32_t bar = smem_u32(&sm->full[k % kStages]);
                const uint32_t parity = (k / kStages) & 1;
                uint64_t t0 = globaltimer();
                while (!mbar_wait_sleep(bar, parity, 20000u))
                    if ((long long)(globaltimer() - t0) > a->timeout_ns) {
                        set_error(p, sm, kErrInternal, -3);
                        break;
                    }
            }
        }
        __syncwarp();
    }
};

// The loader's attention walk with shared-prefix groups, out of line: it works on a copy
// of the loader state (passed and returned by value), so the inline hot path keeps its
// state in registers.
template <int HD>
__device__ __noinline__ Producer producer_attention_groups(Producer pr, int l, int cta) {
    pr.last_ok = pr.attention_walk<HD, true>(l, cta);
    return pr;
}
template <int HD>
__device__ __forceinline__ bool Producer::attention(int l, int cta) {
    if (!a->pf_on) return attention_walk<HD, false>(l, cta);
    const Producer t = producer_attention_groups<HD>(*this, l, cta);
    seq = t.seq;
    pt_b = t.pt_b;
    pt_lp0 = t.pt_lp0;
    pt_ids = t.pt_ids;
    tn = t.tn;
#ifdef MK_PROF
    ppt = t.ppt;
#endif
    return t.last_ok;
}

// ------------------------------------------------------------------ consumer pieces
// rstd[b] = 1 / sqrt(mean(src[b]^2) + eps); fixed summation order. Every k-step reads
// all the batch rows at once, so the whole pass costs K / 1024 read latencies, not one
// per row and k-step. Small batches read the tagged rows, larger ones the fp32 rows.
__device__ __noinline__ void rms_scale(int kind, int layer) {
    Ctx c = make_ctx(0);
    const StepArgs& a = *c.a;
    const GemvStage s = make_gemv(a, kind, layer, c.sm->lp[kind == G_LM ? 0 : (layer & 1)], c.sm);
    const int K = s.K, B = a.B;
    float* red = c.scratch;
    float ss[kMaxBatch];
#pragma unroll
    for (int b = 0; b < kMaxBatch; ++b) ss[b] = 0.f;
    if (tagged(a)) {  // B <= kMaxTaggedBatch: pairs of tagged words
        for (int k = c.tid * 2; k < K; k += kConsumerThreads * 2) {
            uint64_t w[kMaxTaggedBatch][2];
            Spin sp;
            for (;;) {
#pragma unroll
                for (int b = 0; b < kMaxTaggedBatch; ++b) {
                    w[b][0] = w[b][1] = (uint64_t)s.src_tag << 32;
                    if (b < B) ll_ld2(s.src + (size_t)b * s.lds + k, w[b][0], w[b][1]);
                }
                int miss = -1;
#pragma unroll
                for (int b = kMaxTaggedBatch - 1; b >= 0; --b)
                    if (ll_tag(w[b][0]) != s.src_tag || ll_tag(w[b][1]) != s.src_tag) miss = b;
                if (miss < 0 || !ll_wait_pair(s.src + (size_t)miss * s.lds + k, s.src_tag, sp, a, c.sm, s.task_id))
                    break;
            }
#pragma unroll
            for (int b = 0; b < kMaxTaggedBatch; ++b) {
                const float v0 = ll_val(w[b][0]), v1 = ll_val(w[b][1]);
                if (b < B) ss[b] += v0 * v0 + v1 * v1;
            }
        }
    } else {
        for (int k = c.tid * 4; k < K; k += kConsumerThreads * 4) {
            float4 v[kMaxBatch];
#pragma unroll
            for (int b = 0; b < kMaxBatch; ++b)
                v[b] = b < B ? __ldcg(reinterpret_cast<const float4*>(s.srcf + (size_t)b * s.lds + k))
                             : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int b = 0; b < kMaxBatch; ++b) ss[b] += v[b].x * v[b].x + v[b].y * v[b].y + v[b].z * v[b].z + v[b].w * v[b].w;
        }
    }
#pragma unroll
    for (int b = 0; b < kMaxBatch; ++b) {
        if (b >= B) break;
        float t = ss[b];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
        if (c.lane == 0) red[b * kConsumerWarps + c.cw] = t;
    }
    consumer_sync();
    if (c.tid < B) {
        float t = 0.f;
        for (int w = 0; w < kConsumerWarps; ++w) t += red[c.tid * kConsumerWarps + w];
        c.sm->rstd[c.tid] = rsqrtf(t / (float)K + a.p.eps);
    }
    consumer_sync();
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC 2011), word 0 of the output block: the
// counter-based generator of the sampling draws (no state; the same value for the same
// (key, counter) on any thread, CTA or step).
__device__ __forceinline__ uint32_t philox4x32_10_w0(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                                     uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        const uint32_t hi0 = __umulhi(0xD2511F53u, c0), lo0 = 0xD2511F53u * c0;
        const uint32_t hi1 = __umulhi(0xCD9E8D57u, c2), lo1 = 0xCD9E8D57u * c2;
        const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
    }
    return c0;
}
// logit / T + standard Gumbel draw for (token, position, row): the value whose argmax
// is a draw from softmax(logits / T)
__device__ __forceinline__ float gumbel_score(const StepArgs& a, float logit, int token, int pos, int row) {
    const uint32_t x = philox4x32_10_w0((uint32_t)token, (uint32_t)pos, (uint32_t)row, 0u, a.seed_lo, a.seed_hi);
    const float u = ((float)(x >> 8) + 0.5f) * (1.0f / 16777216.0f);
    return logit / a.temperature - logf(-logf(u));
}
__device__ __forceinline__ int cta_of(const Ctx&) { return blockIdx.x; }

// ---- top-k sampling (the largest top_k logits of a row, then a Gumbel-max draw) ----
// Order of the candidates: the larger logit first, the lower index first among equal ones.
__device__ __forceinline__ bool tk_before(float v1, int i1, float v2, int i2) {
    return v1 > v2 || (v1 == v2 && i1 < i2);
}
__device__ __forceinline__ bool topk_sampling(const StepArgs& a) { return a.temperature > 0.f && a.top_k > 0; }
// A warp's running top-K list (K <= 32): lane j holds entry j, in the order above; unused
// entries are (-inf, INT_MAX). Every lane offers a candidate (cv, ci) (ignored when
// !valid); the survivors of the cut by the current K-th entry are inserted one by one.
__device__ __forceinline__ void tk_offer(float& lv, int& li, int K, float cv, int ci, bool valid) {
    const int lane = (int)(threadIdx.x & 31);
    float mv = __shfl_sync(0xffffffffu, lv, K - 1);
    int mi = __shfl_sync(0xffffffffu, li, K - 1);
    uint32_t m = __ballot_sync(0xffffffffu, valid && tk_before(cv, ci, mv, mi));
    while (m) {
        const int src = __ffs(m) - 1;
        m &= m - 1;
        const float v = __shfl_sync(0xffffffffu, cv, src);
        const int i = __shfl_sync(0xffffffffu, ci, src);
        if (!tk_before(v, i, mv, mi)) continue;  // (uniform) the cut rose since the vote
        const int pos = __popc(__ballot_sync(0xffffffffu, lane < K && tk_before(lv, li, v, i)));
        const float pv = __shfl_up_sync(0xffffffffu, lv, 1);
        const int pi = __shfl_up_sync(0xffffffffu, li, 1);
        if (lane < K) {
            if (lane > pos) { lv = pv; li = pi; }
            else if (lane == pos) { lv = v; li = i; }
        }
        mv = __shfl_sync(0xffffffffu, lv, K - 1);
        mi = __shfl_sync(0xffffffffu, li, K - 1);
    }
}
// LM-head epilogue of a top-k sampling step: warp b offers the task's logits of row b to
// the row's running list (kept in shared memory between tasks).
__device__ __noinline__ void tk_lm_task(int b, int r0, int n, const float* yout) {
    const Ctx c = make_ctx(0);
    const int K = c.a->top_k;
    float lv = c.lane < K ? c.sm->tk_v[b][c.lane] : -INFINITY;
    int li = c.lane < K ? c.sm->tk_i[b][c.lane] : 0x7fffffff;
    for (int r = c.lane; r - c.lane < n; r += 32)
        tk_offer(lv, li, K, r < n ? yout[r * 8 + b] : -INFINITY, r0 + r, r < n);
    if (c.lane < K) {
        c.sm->tk_v[b][c.lane] = lv;
        c.sm->tk_i[b][c.lane] = li;
    }
}
// The step's draw for row b from every CTA's list (tagged pairs, written after the LM
// head): warp-wide merge into the row's top-K, then argmax of logit / T + Gumbel noise
// over it (lowest index on equal scores). Returns the token (lane-uniform).
__device__ __noinline__ int tk_draw(int b, uint32_t tag, int task) {
    const Ctx c = make_ctx(0);
    const StepArgs& a = *c.a;
    const Plan& p = a.p;
    const int K = a.top_k;
    float lv = -INFINITY;
    int li = 0x7fffffff;
    // lane j takes entry j of 8 CTAs at a time (one read round per 8 CTAs)
    for (int ct0 = 0; ct0 < p.C; ct0 += 8) {
        uint64_t w[8][2];
        Spin sp;
        for (;;) {
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                w[q][0] = w[q][1] = (uint64_t)tag << 32;
                if (ct0 + q < p.C && c.lane < K)
                    ll_ld2(p.cand + (((size_t)(ct0 + q) * p.maxB + b) * kMaxSampleTopK + c.lane) * 2, w[q][0], w[q][1]);
            }
            int miss = -1;
#pragma unroll
            for (int q = 7; q >= 0; --q)
                if (ll_tag(w[q][0]) != tag || ll_tag(w[q][1]) != tag) miss = q;
            if (!__any_sync(0xffffffffu, miss >= 0)) break;
            // each lane waits on its first missing pair alone, then the batch is re-read
            bool ok = true;
            if (miss >= 0)
                ok = ll_wait_pair(p.cand + (((size_t)(ct0 + miss) * p.maxB + b) * kMaxSampleTopK + c.lane) * 2,
                                  tag, sp, a, c.sm, task);
            if (!__all_sync(0xffffffffu, ok)) break;
        }
#pragma unroll
        for (int q = 0; q < 8; ++q)
            tk_offer(lv, li, K, ll_val(w[q][0]), __float_as_int(ll_val(w[q][1])),
                     ct0 + q < p.C && c.lane < K);
    }
    const int pos = c.sm->pos[b];
    float bz = -INFINITY;
    int bi = 0x7fffffff;
    if (c.lane < K && li != 0x7fffffff) {
        bz = gumbel_score(a, lv, li, pos, b);
        bi = li;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float oz = __shfl_xor_sync(0xffffffffu, bz, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (oz > bz || (oz == bz && oi < bi)) { bz = oz; bi = oi; }
    }
    return bi == 0x7fffffff ? 0 : bi;
}

// the small-batch path computes the RMSNorm statistics from its own activation loads
// when the whole input row is one k-chunk
__device__ __forceinline__ bool fused_norm_stage(const StepArgs& a, const GemvStage& s) {
    return a.B <= kMaxTaggedBatch && s.K <= KCW;
}

// a consumer warp waits for ring slot `q` to be full; warp-uniform result. Fast path:
// every lane tests the barrier once (an acquire for each lane) and the warp votes.
__device__ __forceinline__ bool wait_full_at(Ctx& c, uint32_t q, int task) {
    const uint32_t slot = q % kStages, parity = (q / kStages) & 1;
    const uint32_t bar = smem_u32(&c.sm->full[slot]);
    if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
    int ok = 1;
    if (c.lane == 0) ok = ring_wait_slow(c.a, c.sm, bar, parity, c.a->timeout_ns, task);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) mbar_try_wait(bar, parity);  // every lane acquires the completed phase
    return ok != 0;
}
__device__ __forceinline__ void release_at(Ctx& c, uint32_t q) {
    __syncwarp();
    if (c.lane == 0) mbar_arrive(smem_u32(&c.sm->empty[q % kStages]));
}

// Sum of V = 8 * BP per-lane values over the 32 lanes of a warp, transposed: after the
// halving steps lane L holds the total of value index idx(L) (returned through `idx`).
template <int BP>
__device__ __forceinline__ float warp_transpose_reduce(float (&v)[8 * BP], int lane, int& idx) {
    constexpr int V = 8 * BP;
    idx = 0;
    int o = 16;
#pragma unroll
    for (int h = V / 2; h >= 1; h >>= 1, o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < h; ++i) {
            const float send = up ? v[i] : v[i + h];
            const float keep = up ? v[i + h] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
        if (up) idx += h;
    }
    for (; o >= 1; o >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
    return v[0];
}

// Small batches (B <= kMaxTaggedBatch): exact fp32 CUDA-core dot products. Each lane owns one 8-column
// piece of the k-chunk (a 16 B read of every row), with the piece's activations in
// registers. Each slot's 8 x BP partial sums are reduced across the warp at once (one
// value per lane, or per group of lanes, at the end) and added to this warp's partials
// in shared memory, which the epilogue sums over warps in a fixed order. The slot loop
// is not unrolled: at small batch most stages run only a few slots per CTA, so the code
// is executed once per layer, and a compact loop keeps the step's instruction working
// set small. When the whole input row is one chunk the RMSNorm statistics come from
// the same loads. Writes yout[vrow][8] when yout is given.
template <int BP>
__device__ __forceinline__ void gemv_fma(Ctx& c, const GemvStage& s, int r0, int r1, float* yout,
                                         bool fused_norm) {
    constexpr int V = 8 * BP;   // values one slot leaves per lane before the reduction
    constexpr int LPV = 32 / V;  // lanes holding each reduced value
    const StepArgs& a = *c.a;
    const int B = a.B;
    const int n = r1 - r0, ng = num_groups(s, n), ngate = s.kind == G_GU ? ng / 2 : ng;
    float* red = c.scratch;  // [8 warps][128 vrows][BP]
    for (int i = c.lane; i < kTaskRows * BP; i += 32) red[c.cw * kTaskRows * BP + i] = 0.f;
    __syncwarp();
    const int piece = 32 * c.cw + c.lane;
    // This lane's tagged activation words of chunk k0: BP rows x 8 columns (4 pairs).
    auto issue = [&](int k0, uint64_t (&w)[BP][8]) {
        const int col = k0 + 8 * piece;
        const int base = (col & ~63) + 2 * ((col >> 3) & 7);  // permuted pair (t = 0)
        const bool has = piece < (min(s.kcw, s.K - k0) >> 3);
#pragma unroll
        for (int b = 0; b < BP; ++b)
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                w[b][2 * t] = w[b][2 * t + 1] = (uint64_t)s.src_tag << 32;
                if (b < B && has) ll_ld2(s.src + (size_t)b * s.lds + base + 16 * t, w[b][2 * t], w[b][2 * t + 1]);
            }
    };
    auto tags_ok = [&](const uint64_t (&w)[BP][8]) {
        bool ok = true;
#pragma unroll
        for (int b = 0; b < BP; ++b)
#pragma unroll
            for (int i = 0; i < 8; ++i) ok = ok && ll_tag(w[b][i]) == s.src_tag;
        return ok;
    };
    // With BP == 1 the next chunk's words are requested before this chunk's slots are
    // processed, so a multi-chunk row (K > KCW) pays one read latency, not one per chunk.
    constexpr bool kAhead = BP == 1;
    uint64_t wn[BP][8];
    issue(0, wn);
#pragma unroll 1
    for (int k0 = 0; k0 < s.K; k0 += s.kcw) {
        const SlotGeom geo = slot_geom(s, k0);
        const bool has_p = piece < (geo.kc >> 3);
        float xv[BP][8];
        if (!kAhead && k0 > 0) issue(k0, wn);
        const int col = k0 + 8 * piece;
        const int base = (col & ~63) + 2 * ((col >> 3) & 7);  // permuted pair (t = 0)
        // the norm gains do not depend on the step: request them before the activations
        // are awaited, so the two reads overlap
        float2 gg[4];
#pragma unroll
        for (int t = 0; t < 4; ++t)
            gg[t] = (s.gain && has_p) ? ldg_na_f2(reinterpret_cast<const float2*>(s.gain + base + 16 * t))
                                      : make_float2(0.f, 0.f);
        if (!c.sm->abort) {  // poll until every word carries the awaited tag
            Spin sp;
            while (!tags_ok(wn)) {
                int miss = 0;  // first pair (b * 4 + t) that is not there yet
#pragma unroll
                for (int q = 4 * BP - 1; q >= 0; --q)
                    if (ll_tag(wn[q >> 2][2 * (q & 3)]) != s.src_tag || ll_tag(wn[q >> 2][2 * (q & 3) + 1]) != s.src_tag)
                        miss = q;
                if (!ll_wait_pair(s.src + (size_t)(miss >> 2) * s.lds + base + 16 * (miss & 3), s.src_tag, sp, a,
                                  c.sm, s.task_id))
                    break;
                issue(k0, wn);
            }
        }
#pragma unroll
        for (int b = 0; b < BP; ++b)
#pragma unroll
            for (int i = 0; i < 8; ++i) xv[b][i] = (b < B && has_p) ? ll_val(wn[b][i]) : 0.f;
        if (kAhead && k0 + s.kcw < s.K) issue(k0 + s.kcw, wn);
        if (s.gain) {
            if (fused_norm) {  // this chunk is the whole row: sum of squares from registers
#pragma unroll
                for (int b = 0; b < BP; ++b) {
                    float ss = 0.f;
#pragma unroll
                    for (int i = 0; i < 8; ++i) ss += xv[b][i] * xv[b][i];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
                    if (c.lane == 0) c.sm->ssq[c.cw][b] = ss;
                }
                consumer_sync();
            }
            float rs[BP];
#pragma unroll
            for (int b = 0; b < BP; ++b) {
                if (fused_norm) {  // every thread folds the 8 warp sums itself: no second barrier
                    float ss = 0.f;
#pragma unroll
                    for (int w = 0; w < kConsumerWarps; ++w) ss += c.sm->ssq[w][b];
                    rs[b] = b < B ? rsqrtf(ss / (float)s.K + a.p.eps) : 0.f;
                } else {
                    rs[b] = b < B ? c.sm->rstd[b] : 0.f;
                }
            }
            if (has_p) {
#pragma unroll
                for (int t = 0; t < 4; ++t) {
#pragma unroll
                    for (int b = 0; b < BP; ++b) {
                        xv[b][2 * t] *= rs[b] * gg[t].x;
                        xv[b][2 * t + 1] *= rs[b] * gg[t].y;
                    }
                }
            }
        }
        if (trace_slots(s)) MK_TRACE_C(c, TR_G_X, 0);
        if (k0 == 0) MK_PROF_MARK(c, PS_G_DATA + 4 * s.kind);
        uint32_t roff[8];  // byte offset of row r (this lane's piece) inside a slot
#pragma unroll
        for (int r = 0; r < 8; ++r) roff[r] = (uint32_t)(geo.row_off(r) + 16 * piece);
#pragma unroll 1
        for (int gi = 0; gi < ng; ++gi) {
            const int nr = group_rows(s, n, gi, ngate);
            if (trace_slots(s)) MK_TRACE_C(c, TR_S_WAIT, c.seq);
            MK_PROF_MARK(c, PS_G_SLOTS + 4 * s.kind);
            const bool ok = wait_full_at(c, c.seq, s.task_id);
            MK_PROF_MARK(c, PS_G_SWAIT);
            if (trace_slots(s)) MK_TRACE_C(c, TR_S_FULL, c.seq);
            uint4 wr[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) wr[r] = make_uint4(0u, 0u, 0u, 0u);
            if (ok && has_p) {
                const uint32_t slot = c.ring_s + (c.seq % kStages) * kSlotBytes;
#pragma unroll
                for (int r = 0; r < 8; ++r)
                    if (r < nr)
                        asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                                     : "=r"(wr[r].x), "=r"(wr[r].y), "=r"(wr[r].z), "=r"(wr[r].w)
                                     : "r"(slot + roff[r]));
            }
            release_at(c, c.seq);  // the rows are in registers: hand the slot back
            if (trace_slots(s)) MK_TRACE_C(c, TR_S_REL, c.seq);
            c.seq++;
            float acc[V];
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const uint32_t w[4] = {wr[r].x, wr[r].y, wr[r].z, wr[r].w};
#pragma unroll
                for (int b = 0; b < BP; ++b) {
                    float sacc = 0.f;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        sacc = fmaf(__uint_as_float(w[q] << 16), xv[b][2 * q], sacc);
                        sacc = fmaf(__uint_as_float(w[q] & 0xffff0000u), xv[b][2 * q + 1], sacc);
                    }
                    acc[r * BP + b] = sacc;
                }
            }
            int idx;  // (row r, batch b) = (idx / BP, idx % BP); LPV lanes hold each total
            const float v = warp_transpose_reduce<BP>(acc, c.lane, idx);
            if ((c.lane & (LPV - 1)) == 0) red[(c.cw * kTaskRows + gi * kGroupRows + idx / BP) * BP + idx % BP] += v;
        }
    }
    MK_PROF_MARK(c, PS_G_SLOTS + 4 * s.kind);
    consumer_sync();
    if (trace_slots(s)) MK_TRACE_C(c, TR_G_SUM, 0);
    if (yout)
        for (int e = c.tid; e < ng * kGroupRows * 8; e += kConsumerThreads) {
            const int vr = e >> 3, b = e & 7;
            float y = 0.f;
            if (b < BP) {
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w) y += red[(w * kTaskRows + vr) * BP + b];
            }
            yout[e] = y;
        }
}

// Epilogues of the small-batch path straight from the per-warp partials (no staging,
// no extra barrier): store q|k|v, residual add into the owned rows, or SiLU(gate) * up.
template <int BP>
__device__ __forceinline__ void fma_epilogue(Ctx& c, const GemvStage& s, int r0, int r1, int cta) {
    const StepArgs& a = *c.a;
    const Plan& p = a.p;
    // BP 1 and 2 serve exactly that batch; BP 4 serves batches 3 and 4
    const int B = BP < 4 ? BP : a.B, n = r1 - r0;
    const float* red = c.scratch;
    auto ysum = [&](int vr, int b) {
        float y = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) y += red[(w * kTaskRows + vr) * BP + b];
        return y;
    };
    if (a.skip_publish == s.task_id) return;
    int a0 = 0, a1;
    if (s.kind == G_O || s.kind == G_DOWN) cta_rows(p.d, cta, p.C, a0, a1);
    const int up0 = s.kind == G_GU ? kGroupRows * (num_groups(s, n) >> 1) : 0;
    // one loop for every stage kind (a uniform switch per element): at small batch each
    // thread stores at most a couple of outputs, so compact code matters more here
#pragma unroll 1
    for (int e = c.tid; e < n * B; e += kConsumerThreads) {
        const int r = BP == 1 ? e : e / B, b = BP == 1 ? 0 : e - r * B;
        const float y = ysum(r, b);
        switch (s.kind) {
            case G_QKV:
                ll_st(p.qkv + (size_t)b * p.qkv_rows + r0 + r, y, s.out_tag);
                break;
            case G_ROUTE:
                ll_st(p.route + (size_t)b * p.E + r0 + r, y, s.out_tag);
                break;
            case G_GU: {  // MoE: scaled by the row's routing weight of the union slot
                float h = silu(y) * ysum(up0 + r, b);
                if (s.moe) h *= c.sm->moe_w[b][(r0 + r) / s.Fe];
                ll_st(p.h + (size_t)b * p.hrow + perm_col(r0 + r), h, s.out_tag);
                break;
            }
            default: {  // G_O, G_DOWN: residual add into the owned rows
                const float xn = c.sm->xown[b][r0 + r - a0] + y;
                c.sm->xown[b][r0 + r - a0] = xn;
                ll_st(p.x + (size_t)b * p.d + perm_col(r0 + r), xn, s.out_tag);
                break;
            }
        }
    }
}

// Larger batches: BF16 mma.sync tiles of 16 weight rows (two consecutive slots) as the
// A operand and the batch rows as the 8 B columns, activations split hi + lo.
__device__ __forceinline__ void gemv_mma(Ctx& c, const GemvStage& s, int r0, int r1, float* yout) {
    const StepArgs& a = *c.a;
    const int n = r1 - r0, ng = num_groups(s, n);
    const int nt = (ng + 1) >> 1;  // 16-row tiles
    const int g = c.lane >> 2, t = c.lane & 3;
    const bool has_b = g < a.B;
    float acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    const float rs = has_b ? c.sm->rstd[g] : 0.f;
    // ldmatrix lane -> (tile row, chunk): lanes 0-7 rows 0-7 chunk X, 8-15 rows 8-15
    // chunk X (second slot), 16-23 rows 0-7 chunk X+1, 24-31 rows 8-15 chunk X+1
    const int lrow = c.lane & 7, lhalf = (c.lane >> 3) & 1, lch = c.lane >> 4;

    for (int k0 = 0; k0 < s.K; k0 += s.kcw) {
        const SlotGeom geo = slot_geom(s, k0);
        const int nblk = geo.kc >> 6;
        uint32_t bfr[4][4][4];  // [block][k-step][hi b0b1, hi b2b3, lo b0b1, lo b2b3]
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const int j = c.cw + 8 * jj;
#pragma unroll
            for (int i = 0; i < 4; ++i) bfr[jj][i][0] = bfr[jj][i][1] = bfr[jj][i][2] = bfr[jj][i][3] = 0u;
            if (j < nblk && has_b && !c.sm->abort) {
                const int col = k0 + 64 * j + 16 * t;
                const float4* src = reinterpret_cast<const float4*>(s.srcf + (size_t)g * s.lds + col);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float4 v = __ldcg(src + i);
                    if (s.gain) {
                        const float4 gg = __ldg(reinterpret_cast<const float4*>(s.gain + col) + i);
                        v.x *= rs * gg.x; v.y *= rs * gg.y; v.z *= rs * gg.z; v.w *= rs * gg.w;
                    }
                    split_bf16x2(v.x, v.y, bfr[jj][i][0], bfr[jj][i][2]);
                    split_bf16x2(v.z, v.w, bfr[jj][i][1], bfr[jj][i][3]);
                }
            }
        }
        if (k0 == 0) MK_PROF_MARK(c, PS_G_DATA + 4 * s.kind);
#pragma unroll
        for (int ti = 0; ti < 8; ++ti) {
            if (ti < nt) {
                const bool two = 2 * ti + 1 < ng;
                const uint32_t qa = c.seq, qb = c.seq + 1;
                bool ok = wait_full_at(c, qa, s.task_id);
                if (two) ok = wait_full_at(c, qb, s.task_id) && ok;
                if (ok) {
                    const uint32_t sa = c.ring_s + (qa % kStages) * kSlotBytes;
                    const uint32_t sb = two ? c.ring_s + (qb % kStages) * kSlotBytes : sa;
                    const uint32_t rowaddr = (lhalf ? sb : sa) + geo.row_off(lrow);
                    // four independent accumulator chains (hi/lo x even/odd k-step) keep
                    // the tensor pipe busy instead of waiting on one serial chain
                    float ct[4][4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) ct[q][0] = ct[q][1] = ct[q][2] = ct[q][3] = 0.f;
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        const int j = c.cw + 8 * jj;
                        if (j < nblk) {
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const int chunk = 8 * j + 2 * i + lch;
                                uint32_t a0, a1, a2, a3;
                                ldmatrix_x4(rowaddr + chunk * 16, a0, a1, a2, a3);
                                mma_16816(ct[(i & 1) * 2], a0, a1, a2, a3, bfr[jj][i][0], bfr[jj][i][1]);
                                mma_16816(ct[(i & 1) * 2 + 1], a0, a1, a2, a3, bfr[jj][i][2], bfr[jj][i][3]);
                            }
                        }
                    }
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[ti][e] += (ct[0][e] + ct[1][e]) + (ct[2][e] + ct[3][e]);
                }
                release_at(c, qa);
                if (two) release_at(c, qb);
                c.seq += two ? 2 : 1;
            }
        }
    }
    MK_PROF_MARK(c, PS_G_SLOTS + 4 * s.kind);
    // cross-warp reduction: red[w][tile][16 rows][8 cols] in rounds of 4 tiles
    float* red = c.scratch;
#pragma unroll
    for (int round = 0; round < 2; ++round) {
        if (round * 4 < nt) {
            consumer_sync();
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) {
                const int ti = round * 4 + rr;
                if (ti < nt) {
                    float* base = red + ((c.cw * 4 + rr) * 16) * 8;
                    *reinterpret_cast<float2*>(base + g * 8 + 2 * t) = make_float2(acc[ti][0], acc[ti][1]);
                    *reinterpret_cast<float2*>(base + (g + 8) * 8 + 2 * t) = make_float2(acc[ti][2], acc[ti][3]);
                }
            }
            consumer_sync();
            for (int e = c.tid; e < 4 * 16 * 8; e += kConsumerThreads) {
                const int rr = e >> 7, rem = e & 127;
                const int ti = round * 4 + rr;
                if (ti < nt) {
                    float y = 0.f;
#pragma unroll
                    for (int w = 0; w < kConsumerWarps; ++w) y += red[(w * 4 + rr) * 128 + rem];
                    yout[ti * 128 + rem] = y;  // vrow = 16 ti + row = 8 * group + row
                }
            }
        }
    }
}

// Epilogues from the staged outputs yout[vrow][8] (vrow = 8 * group + row; GU: up rows
// start at vrow 8 * ngate): the LM head at every batch, every stage above kMaxTaggedBatch rows.
__device__ __forceinline__ void yout_epilogue(Ctx& c, const GemvStage& s, int r0, int r1,
                                              const float* yout) {
    const StepArgs& a = *c.a;
    const Plan& p = a.p;
    const int n = r1 - r0;
    const int B = a.B;
    const bool pub = a.skip_publish != s.task_id;
    switch (s.kind) {
        case G_QKV:
            for (int e = c.tid; e < n * B; e += kConsumerThreads) {
                const int r = e / B, b = e % B;
                if (pub) ll_st(p.qkv + (size_t)b * p.qkv_rows + r0 + r, yout[r * 8 + b], s.out_tag);
            }
            break;
        case G_O:
        case G_DOWN: {
            int a0, a1;
            cta_rows(p.d, cta_of(c), p.C, a0, a1);
            for (int e = c.tid; e < n * B; e += kConsumerThreads) {
                const int r = e / B, b = e % B;
                const float xn = c.sm->xown[b][r0 + r - a0] + yout[r * 8 + b];
                c.sm->xown[b][r0 + r - a0] = xn;
                const size_t o = (size_t)b * p.d + perm_col(r0 + r);
                if (!tagged(a)) p.xf[o] = xn;
                else if (pub) ll_st(p.x + o, xn, s.out_tag);
            }
            break;
        }
        case G_GU: {
            const int up0 = kGroupRows * (num_groups(s, n) >> 1);
            for (int e = c.tid; e < n * B; e += kConsumerThreads) {
                const int r = e / B, b = e % B;
                const float yg = yout[r * 8 + b];
                const float yu = yout[(up0 + r) * 8 + b];
                float y = silu(yg) * yu;
                if (s.moe) y *= c.sm->moe_w[b][(r0 + r) / s.Fe];
                const size_t o = (size_t)b * p.hrow + perm_col(r0 + r);
                if (!tagged(a)) p.hf[o] = y;
                else if (pub) ll_st(p.h + o, y, s.out_tag);
            }
            break;
        }
        case G_ROUTE:
            for (int e = c.tid; e < n * B; e += kConsumerThreads) {
                const int r = e / B, b = e % B;
                if (pub) ll_st(p.route + (size_t)b * p.E + r0 + r, yout[r * 8 + b], s.out_tag);
            }
            break;
        default: {  // G_LM: logits + running argmax (warp w handles batch row w)
            if (a.logits)
                for (int e = c.tid; e < n * B; e += kConsumerThreads) {
                    const int r = e / B, b = e % B;
                    a.logits[(size_t)b * p.V + r0 + r] = yout[r * 8 + b];
                }
            if (c.cw < B && topk_sampling(a)) {
                tk_lm_task(c.cw, r0, n, yout);
            } else if (c.cw < B) {
                const int b = c.cw;
                const bool sample = a.temperature > 0.f;
                const int pos = c.sm->pos[b];
                float bv = -INFINITY;
                int bi = 0x7fffffff;
                for (int r = c.lane; r < n; r += 32) {
                    float v = yout[r * 8 + b];
                    if (sample) v = gumbel_score(a, v, r0 + r, pos, b);
                    if (v > bv) { bv = v; bi = r0 + r; }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                    if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
                }
                if (c.lane == 0) {
                    const float cv = c.sm->amax_v[b];
                    const int ci = c.sm->amax_i[b];
                    if (bv > cv || (bv == cv && bi < ci)) { c.sm->amax_v[b] = bv; c.sm->amax_i[b] = bi; }
                }
            }
            break;
        }
    }
}

// Non-inlined, one function per arithmetic path, so that each gets its own register
// budget. They work on register copies of the context and of the stage description;
// only the ring sequence number (and the trace count) go back to the caller.
template <int BP>
__device__ __noinline__ uint32_t gemv_task_fma(uint32_t seq, int kind, int layer, int r0, int r1) {
    Ctx c = make_ctx(seq);
    const StepArgs& a = *c.a;
    const GemvStage s = make_gemv(a, kind, layer, c.sm->lp[layer & 1], c.sm);
    gemv_fma<BP>(c, s, r0, r1, nullptr, fused_norm_stage(a, s));
    if (!c.sm->abort) fma_epilogue<BP>(c, s, r0, r1, cta_of(c));
    MK_PROF_MARK(c, PS_G_EPI + 4 * s.kind);
    if (trace_slots(s)) MK_TRACE_C(c, TR_G_EPI, 0);
    return c.seq;
}
// The LM head (once per step): outputs staged for the logits and argmax epilogue.
template <int BP>
__device__ __noinline__ uint32_t gemv_task_fma_lm(uint32_t seq, int r0, int r1) {
    Ctx c = make_ctx(seq);
    const StepArgs& a = *c.a;
    const GemvStage s = make_gemv(a, G_LM, 0, c.sm->lp[0], c.sm);
    float* yout = c.scratch + kConsumerWarps * kTaskRows * 4;  // [128 vrows][8]
    gemv_fma<BP>(c, s, r0, r1, yout, fused_norm_stage(a, s));
    consumer_sync();
    if (!c.sm->abort) yout_epilogue(c, s, r0, r1, yout);
    MK_PROF_MARK(c, PS_G_EPI + 4 * s.kind);
    if (trace_slots(s)) MK_TRACE_C(c, TR_G_EPI, 0);
    return c.seq;
}
__device__ __noinline__ uint32_t gemv_task_mma(uint32_t seq, int kind, int layer, int r0, int r1) {
    Ctx c = make_ctx(seq);
    const StepArgs& a = *c.a;
    const GemvStage s = make_gemv(a, kind, layer, c.sm->lp[layer & 1], c.sm);
    float* yout = c.scratch + kConsumerWarps * kTaskRows * 4;  // [128 vrows][8]
    gemv_mma(c, s, r0, r1, yout);
    consumer_sync();
    if (!c.sm->abort) yout_epilogue(c, s, r0, r1, yout);
    MK_PROF_MARK(c, PS_G_EPI + 4 * s.kind);
    if (trace_slots(s)) MK_TRACE_C(c, TR_G_EPI, 0);
    return c.seq;
}
__device__ __forceinline__ uint32_t gemv_task_call(uint32_t seq, int kind, int layer, int r0, int r1) {
    const int B = make_ctx(seq).a->B;
    static_assert(kMaxTaggedBatch == 2, "the CUDA-core GEMV is instantiated for 1 and 2 rows");
    if (B > kMaxTaggedBatch) return gemv_task_mma(seq, kind, layer, r0, r1);
    if (kind == G_LM) return B == 1 ? gemv_task_fma_lm<1>(seq, r0, r1) : gemv_task_fma_lm<2>(seq, r0, r1);
    return B == 1 ? gemv_task_fma<1>(seq, kind, layer, r0, r1) : gemv_task_fma<2>(seq, kind, layer, r0, r1);
}


// One GEMV stage of layer `layer` (kind G_*), out of line with its own registers; takes
// and returns the ring sequence number.
// Only a few scalars stay live across the calls it makes (the context and the stage
// description are rebuilt where needed), so it saves and restores nothing around them.
__device__ __noinline__ uint32_t gemv_stage_call(uint32_t seq, int kind, int layer, int cta) {
    int a0, a1, task, cnt_wait, cnt_pub;
    bool norm, tg;
    {
        const Ctx c = make_ctx(seq);
        MK_PROF_MARK(c, PS_T_CALL);
        const GemvStage s = make_gemv(*c.a, kind, layer, c.sm->lp[kind == G_LM ? 0 : (layer & 1)], c.sm);
        cta_rows(s.R, cta, c.a->p.C, a0, a1);
        task = s.task_id;
        cnt_wait = s.cnt_wait;
        cnt_pub = s.cnt_pub;
        norm = s.gain && !fused_norm_stage(*c.a, s);
        tg = tagged(*c.a);
        MK_PROF_MARK(c, PS_OTHER);
        MK_TRACE_C(c, TR_WAIT, task);
    }
    if (a0 < a1) {
        if (!tg) {
            Ctx c = make_ctx(seq);
            consumer_wait(c, cnt_wait, task);
        }
        if (norm) rms_scale(kind, layer);
        const int tr = task_rows(kind);
        for (int r0 = a0; r0 < a1; r0 += tr) {
            // a task's epilogue reads every warp's partials; the next task clears them
            if (r0 > a0) consumer_sync();
            seq = gemv_task_call(seq, kind, layer, r0, min(a1, r0 + tr));
        }
    }
    Ctx c = make_ctx(seq);
    if (!tg && cnt_pub >= 0) publish(c, cnt_pub, task);
    else consumer_sync();  // every warp is done with the shared scratch of this stage
    MK_PROF_MARK(c, PS_G_END + 4 * kind);
    MK_TRACE_C(c, TR_DONE, task);
    return c.seq;
}

__device__ __forceinline__ int bg_id(const Plan& p, int b, int g) { return b * p.Hkv + g; }

// ---- attention: one piece (a CTA's share of one item) ----
// Query columns of a piece: row r of the piece's rows (ascending) holds columns
// r*G .. r*G + G-1 (its G heads of kv head g). Columns go in 8-wide MMA tiles; with two
// tiles, warps 0-3 serve tile 0 and warps 4-7 tile 1 on the same pages.
__device__ __forceinline__ int piece_row(uint32_t rows, int r) { return (int)__fns(rows, 0u, r + 1); }

// Local columns (of a tile) whose per-warp softmax states fit the scratch at once.
template <int HD>
struct FinishCols {
    static constexpr int fit = (kScratchBytes - 512) / (kConsumerWarps * (HD + 8) * 4);
    static constexpr int value = fit < 8 ? fit : 8;
};

// After the key loop of a piece: merge the warps' partial softmax states of local
// columns [ch0, ch0 + FinishCols) (left in shared memory by the piece) and write them as
// this split's partial records, one per row, as tagged words. MULTI: a shared-prefix
// piece (several rows, one or two column tiles); otherwise one row, one tile, one pass.
template <int HD, bool MULTI>
__device__ __forceinline__ void attention_finish(int l, Piece pc, int ch0, int NC, int wpt_in) {
    Ctx c = make_ctx(0);
    const StepArgs& a = *c.a;
    const Plan& p = a.p;
    const int G = p.G;
    const int task = l * 16 + ST_ATTN;
    constexpr int OS = HD + 8;
    constexpr int kFC = FinishCols<HD>::value;
    float* ws_o = c.scratch;                                  // [8][kFC][OS]
    float* ws_m = c.scratch + kConsumerWarps * kFC * OS;      // [8][8]
    float* ws_l = ws_m + 64;                                  // [8][8]
    consumer_sync();
    const int GHD = G * HD, RS = GHD + 2 * G;
    const int wpt = MULTI ? wpt_in : kConsumerWarps;
    const int CT = MULTI ? (NC + 7) >> 3 : 1, nct = MULTI ? min(kFC, min(8, NC) - ch0) : G;
    const int tot = CT * nct * HD;
    const int slot = pc.slot0 + pc.split;
    const uint32_t tag = tag_of(a, l, TAG_PART);
    if (!c.sm->abort && a.skip_publish != task) {
        for (int e = 2 * c.tid; e < tot; e += 2 * kConsumerThreads) {
            const int T = MULTI ? e / (nct * HD) : 0, rem = e - T * nct * HD;
            const int hl = rem / HD, d = rem - hl * HD;
            const int h = MULTI ? ch0 + hl : hl, col = T * 8 + h;
            if (MULTI && col >= NC) continue;
            const int w0 = T * wpt;
            float M = -INFINITY;
#pragma unroll
            for (int k = 0; k < kConsumerWarps; ++k)
                if (k < wpt) M = fmaxf(M, ws_m[(w0 + k) * 8 + h]);
            float o0 = 0.f, o1 = 0.f, L = 0.f;
#pragma unroll
            for (int k = 0; k < kConsumerWarps; ++k) {
                if (k >= wpt) continue;
                const int w = w0 + k;
                const float mw = ws_m[w * 8 + h];
                const float f = mw == -INFINITY ? 0.f : expf(mw - M);
                const float2 ov = *reinterpret_cast<const float2*>(ws_o + (w * kFC + hl) * OS + d);
                o0 += f * ov.x;
                o1 += f * ov.y;
                L += f * ws_l[w * 8 + h];
            }
            const int r = MULTI ? col / G : 0, hh = col - r * G;
            const int b = MULTI ? piece_row(pc.rows, r) : pc.b;
            uint64_t* rec = p.part + ((size_t)(b * p.Hkv + pc.g) * p.C + slot) * RS;
            ll_st2(rec + hh * HD + d, o0, o1, tag);
            if (d == 0) ll_st2(rec + GHD + 2 * hh, M, L, tag);
        }
    }
    consumer_sync();  // the scratch is free for the next piece
    MK_PROF_MARK(c, PS_A_FINISH);
    if (l == 0 || l == 1) MK_TRACE_C(c, TR_A_PART, (uint32_t)pc.split);
}

// The split-`split` of the nsplit CTAs of a (sequence, kv head) item merges output dims
// [j0, j1) of the G heads (flattened h * HD + d) from all nrec partial records of that
// row (its shared prefix's pieces, if any, then its own): per head M = max m_s,
// w_s = exp(m_s - M), L = sum w_s l_s, O = sum w_s o_s / L. Every split takes an equal
// slice, so the merge is spread over all the item's CTAs instead of one CTA merging
// every split.
template <int HD>
__device__ __noinline__ void attention_merge(int l, int b, int g, int split, int nsplit_in, int nrec) {
    Ctx c = make_ctx(0);
    const StepArgs& a = *c.a;
    const Plan& p = a.p;
    const int G = p.G, GHD = G * HD, RS = GHD + 2 * G;
    const int task = l * 16 + ST_ATTN;
    const uint32_t tp = tag_of(a, l, TAG_PART);
    const int j0 = (int)((uint32_t)split * GHD / (uint32_t)nsplit_in);
    const int j1 = (int)((uint32_t)(split + 1) * GHD / (uint32_t)nsplit_in);
    const int nsplit = nrec;  // records merged
    if (j0 >= j1 || c.sm->abort) return;  // uniform over the CTA
    const int h0 = j0 / HD, nh = (j1 - 1) / HD - h0 + 1;
    const uint64_t* rec0 = p.part + (size_t)(b * p.Hkv + g) * p.C * RS;
    float2* mls = reinterpret_cast<float2*>(c.scratch);     // [nsplit][nh] (m, l)
    float* fw = c.scratch + 2 * kMaxSplitsG;                // [nsplit][nh] weights
    float* Ls = fw + kMaxSplitsG;                           // [nh]
    consumer_sync();
    // 1) (m, l) of every split for the heads of the slice
    for (int i = c.tid; i < nsplit * nh; i += kConsumerThreads) {
        const int si = i / nh, hh = i % nh;
        uint64_t w0, w1;
        Spin sp;
        for (;;) {
            ll_ld2(rec0 + (size_t)si * RS + GHD + 2 * (h0 + hh), w0, w1);
            if ((ll_tag(w0) == tp && ll_tag(w1) == tp) || !sp.again(a, c.sm, task)) break;
        }
        mls[i] = make_float2(ll_val(w0), ll_val(w1));
    }
    consumer_sync();
    MK_PROF_MARK(c, PS_M_ML);
    if (l == 1) MK_TRACE_C(c, TR_M_ML, 0);
    // 2) per head (one warp each): M, the weights w_s and L
    if (c.cw < nh) {
        const int hh = c.cw;
        float M = -INFINITY;
        for (int i = c.lane; i < nsplit; i += 32) M = fmaxf(M, mls[i * nh + hh].x);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        float L = 0.f;
        for (int i = c.lane; i < nsplit; i += 32) {
            const float2 ml = mls[i * nh + hh];
            const float f = ml.x == -INFINITY ? 0.f : expf(ml.x - M);
            fw[i * nh + hh] = f;
            L += f * ml.y;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
        if (c.lane == 0) Ls[hh] = L;
    }
    consumer_sync();
    MK_PROF_MARK(c, PS_M_W);
    if (l == 1) MK_TRACE_C(c, TR_M_W, 0);
    // 3) the slice of O: `rep` consecutive lanes per output dim share the splits
    //    round-robin (8 tagged reads in flight each) and combine them with shuffles
    const int len = j1 - j0;
    int rep = 32;
    while (rep > 1 && rep * len > kConsumerThreads) rep >>= 1;
    const uint32_t tattn = tag_of(a, l, TAG_ATTN);
    const bool pub = a.skip_publish != task;
    for (int jb = 0; jb < len; jb += kConsumerThreads / rep) {
        const int jj = jb + c.tid / rep, sub = c.tid % rep;
        float acc = 0.f;
        int hh = 0;
        if (jj < len) {
            const int j = j0 + jj;
            hh = j / HD - h0;
            for (int s0 = sub; s0 < nsplit; s0 += 8 * rep) {
                uint64_t w[8];
                Spin sp;
                for (;;) {
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const int si = s0 + k * rep;
                        w[k] = si < nsplit ? ll_ld(rec0 + (size_t)si * RS + j) : (uint64_t)tp << 32;
                    }
                    int miss = -1;
#pragma unroll
                    for (int k = 7; k >= 0; --k)
                        if (ll_tag(w[k]) != tp) miss = k;
                    if (miss < 0) break;
                    // wait on the missing word alone, then re-read the batch
                    const uint64_t* pm = rec0 + (size_t)(s0 + miss * rep) * RS + j;
                    bool got = false;
                    while (sp.again(a, c.sm, task))
                        if (ll_tag(ll_ld(pm)) == tp) { got = true; break; }
                    if (!got) break;
                }
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int si = s0 + k * rep;
                    if (si < nsplit) acc += fw[si * nh + hh] * ll_val(w[k]);
                }
            }
        }
        for (int off = 1; off < rep; off <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (jj < len && sub == 0) {
            const size_t o = (size_t)b * p.Hq * HD + perm_col(g * G * HD + j0 + jj);
            if (!tagged(a)) p.attnf[o] = acc / Ls[hh];
            else if (pub) ll_st(p.attn + o, acc / Ls[hh], tattn);
        }
    }
    consumer_sync();  // the scratch is free again
    MK_PROF_MARK(c, PS_M_O);
    if (l == 0 || l == 1) MK_TRACE_C(c, TR_A_MERGED, 0);
}

// PK (one row, G <= 4): the B columns are n = 2 h + part, the BF16 hi (part 0) and lo
// (part 1) halves of head h's q (and P) side by side, so one MMA covers both halves where
// the general path issues one per half; each lane then owns one head (t) instead of two.
template <int HD, bool MULTI, bool PK>
__device__ __noinline__ uint32_t attention_piece(uint32_t seq, int l, Piece pc) {
    static_assert(!(MULTI && PK), "packed columns hold one row's heads");
    Ctx c = make_ctx(seq);
    const SeqSpan sp = pc.sp;
    const int b = pc.b, g = pc.g, u = pc.u, n = pc.n;
    const StepArgs& a = *c.a;
    const Plan& p = a.p;
    constexpr int NKS = HD / 16;   // k16 steps over the head dim
    constexpr int NCH = HD / 8;    // 8-dim chunks
    constexpr int PPS = 512 / HD;  // pages per slot
    const int G = p.G;
    const int gq = c.lane >> 2, t = c.lane & 3;
    const int task = l * 16 + ST_ATTN;
    const int pos = sp.pos, lo = sp.lo;
    // query columns: the G heads of each row of the piece; 8-wide column tiles (1 or 2,
    // MULTI only: a shared prefix's rows side by side)
    const int nrows = MULTI ? __popc(pc.rows) : 1, NC = nrows * G;
    const int CT = MULTI ? (NC + 7) >> 3 : 1, wpt = MULTI ? kConsumerWarps / CT : kConsumerWarps;
    const int tile = MULTI ? c.cw / wpt : 0, wl = c.cw - tile * wpt;
    const bool has_last = !MULTI && (sp.p0 + u + n - 1) == pos / kPage;
    // page of the new token's K/V (appending piece): read now, used in the key loop
    const int last_page = has_last ? __ldg(a.page_table + (size_t)b * a.max_pages + pos / kPage) : -1;
    MK_PROF_MARK(c, PS_A_ENTRY);

    // Stage q of the columns (and the new token's k, v when this piece appends), plus the
    // rows' RoPE rows, through shared memory with coalesced loads: one L2 round trip.
    // Rows of q are padded to HD + 8 floats so the fragment reads below are conflict-free.
    constexpr int QS = HD + 8;
    float* qs = c.scratch;                         // [16][QS] (one row: [8][QS])
    float* ks = qs + (MULTI ? 16 : 8) * QS;        // [HD]
    float* vs = ks + HD;                           // [HD]
    float2* rs = reinterpret_cast<float2*>(vs + HD);  // [nrows][HD / 2]
    if (!c.sm->abort) {
        if (MULTI) {
            for (int i = c.tid; i < nrows * (HD / 2); i += kConsumerThreads) {
                const int r = i / (HD / 2);
                const int pr = r == 0 ? pos : c.sm->pos[piece_row(pc.rows, r)];
                rs[i] = ldg_na_f2(p.rope + (size_t)pr * (HD / 2) + (i - r * (HD / 2)));
            }
        } else {
            const float2* rope = p.rope + (size_t)pos * (HD / 2);
            for (int i = c.tid; i < HD / 2; i += kConsumerThreads) rs[i] = ldg_na_f2(rope + i);
        }
        // q of the columns, then (appending piece) k and v: pairs of tagged words, all of
        // a thread's pairs in flight at once, polled until they carry the QKV tag
        const uint64_t* row = p.qkv + (size_t)b * p.qkv_rows;
        const uint32_t tq = tag_of(a, l, TAG_QKV);
        const int nq = NC * HD / 2, nt = nq + (has_last ? HD : 0);
        constexpr int kPairs = ((MULTI ? 16 : 8) * HD / 2 + HD + kConsumerThreads - 1) / kConsumerThreads;
        auto src_of = [&](int i) -> const uint64_t* {
            if (i < nq) {
                if (!MULTI) return row + (size_t)g * G * HD + 2 * i;
                const int col = (2 * i) / HD, r = col / G;
                return p.qkv + (size_t)piece_row(pc.rows, r) * p.qkv_rows +
                       (size_t)(g * G + col - r * G) * HD + (2 * i - col * HD);
            }
            const int j = i - nq;
            return j < HD / 2 ? row + (size_t)(p.Hq + g) * HD + 2 * j
                              : row + (size_t)(p.Hq + p.Hkv + g) * HD + 2 * (j - HD / 2);
        };
        uint64_t w[kPairs][2];
        Spin sp;
        for (;;) {
#pragma unroll
            for (int k = 0; k < kPairs; ++k) {
                const int i = c.tid + k * kConsumerThreads;
                w[k][0] = w[k][1] = (uint64_t)tq << 32;
                if (i < nt) ll_ld2(src_of(i), w[k][0], w[k][1]);
            }
            int miss = -1;
#pragma unroll
            for (int k = kPairs - 1; k >= 0; --k)
                if (ll_tag(w[k][0]) != tq || ll_tag(w[k][1]) != tq) miss = k;
            if (miss < 0 || !ll_wait_pair(src_of(c.tid + miss * kConsumerThreads), tq, sp, a, c.sm, task)) break;
        }
#pragma unroll
        for (int k = 0; k < kPairs; ++k) {
            const int i = c.tid + k * kConsumerThreads;
            if (i >= nt) continue;
            const float2 v = make_float2(ll_val(w[k][0]), ll_val(w[k][1]));
            float* dst;
            if (i < nq) {
                dst = qs + ((2 * i) / HD) * QS + (2 * i) % HD;
            } else {
                const int j = i - nq;
                dst = j < HD / 2 ? ks + 2 * j : vs + 2 * (j - HD / 2);
            }
            *reinterpret_cast<float2*>(dst) = v;
        }
    }
    if (l == 1) MK_TRACE_C(c, TR_Q_LOADED, 0);
    MK_PROF_MARK(c, PS_A_QPOLL);
    consumer_sync();
    MK_PROF_MARK(c, PS_A_QSYNC);
    if (l == 1) MK_TRACE_C(c, TR_Q_SYNCED, 0);
    // q^T (after RoPE) as the B operand: column gq of this warp's tile, k = head dims;
    // hi/lo split. b0b1 of k-step s holds dims 16s + 2t, +1; b2b3 holds 16s + 8 + 2t, +1.
    const int qcol = PK ? (gq >> 1) : tile * 8 + gq;
    const float2* rq = MULTI ? rs + (qcol < NC ? qcol / G : 0) * (HD / 2) : rs;
    uint32_t qa[NKS][2], ql[NKS][2];
#pragma unroll
    for (int s = 0; s < NKS; ++s)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            float v0 = 0.f, v1 = 0.f;
            if (qcol < NC) {
                const int d = 16 * s + 8 * hh + 2 * t;
                const int dp = d < HD / 2 ? d + HD / 2 : d - HD / 2;
                const float4 cs = *reinterpret_cast<const float4*>(rq + (d % (HD / 2)));
                const float2 x0 = *reinterpret_cast<const float2*>(qs + qcol * QS + d);
                const float2 xp = *reinterpret_cast<const float2*>(qs + qcol * QS + dp);
                if (d < HD / 2) {
                    v0 = x0.x * cs.x - xp.x * cs.y;
                    v1 = x0.y * cs.z - xp.y * cs.w;
                } else {
                    v0 = x0.x * cs.x + xp.x * cs.y;
                    v1 = x0.y * cs.z + xp.y * cs.w;
                }
            }
            split_bf16x2(v0, v1, qa[s][hh], ql[s][hh]);
            if (PK && (gq & 1)) qa[s][hh] = ql[s][hh];  // column 2 h + 1: the lo half
        }
    // the new token's K (after RoPE) and V, rounded to BF16 (warp 0 also splices them)
    if (has_last && c.cw == 0) {
        for (int i = c.lane; i < HD / 2; i += 32) {
            const float2 cs = rs[i];
            const float k0 = ks[i], k1 = ks[i + HD / 2];
            c.sm->knew[i] = __float2bfloat16_rn(k0 * cs.x - k1 * cs.y);
            c.sm->knew[i + HD / 2] = __float2bfloat16_rn(k1 * cs.x + k0 * cs.y);
        }
        for (int i = c.lane; i < HD; i += 32) c.sm->vnew[i] = __float2bfloat16_rn(vs[i]);
        __syncwarp();
    }
    if (l == 0 || l == 1) MK_TRACE_C(c, TR_A_Q, (uint32_t)bg_id(p, b, g));
    consumer_sync();  // the staging area becomes the per-warp P buffers below
    MK_PROF_MARK(c, PS_A_FRAG);

    // Keys in the MMA M dimension: S^T = K q^T (16 keys x 8 head columns) and
    // O^T += V^T P^T (16 dims x 8 head columns), two MMAs (hi/lo) per 16x16 step.
    // This thread owns heads 2t, 2t+1 (real when < G) and, in O^T, dims 16 mt + g (+8).
    constexpr int NMT = HD / 16;
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    float oacc[NMT][4];
#pragma unroll
    for (int i = 0; i < NMT; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
    float* pbuf = c.scratch + c.cw * 32 * 9;  // P[32 keys][9] for this warp (fp32)
    // Windows of 2 * wpt pages (16, or 8 with two column tiles): warp w of a tile takes
    // pages 2w and 2w + 1 (one ring slot holds PPS pages) and processes the two together,
    // so two independent MMA chains hide each other's latency. Every warp waits for and
    // releases every slot of the window in order (a slot is handed back only after its
    // data has arrived).
    const int WIN = MULTI ? 2 * wpt : 2 * kConsumerWarps;
    const int lrow8 = c.lane & 7, lmi = c.lane >> 3;
    const int pa = 2 * wl, mys = pa / PPS;

    for (int w0 = 0; w0 < n; w0 += WIN) {
        const int nw = min(WIN, n - w0), nsl = (nw + PPS - 1) / PPS;
        for (int j = 0; j < nsl; ++j) {
            MK_PROF_MARK(c, PS_A_LOOP);
            const bool ok = wait_full_at(c, c.seq + j, task);
            MK_PROF_MARK(c, PS_A_LWAIT);
            if (j == mys && pa < nw && ok && !c.sm->abort) {
                const uint32_t slot = c.ring_s + ((c.seq + j) % kStages) * kSlotBytes;
                const uint32_t kbA = slot + (pa % PPS) * 64 * HD, kbB = kbA + 64 * HD;
                const int keyA = (sp.p0 + u + w0 + pa) * kPage, keyB = keyA + kPage;
                const bool hasB = pa + 1 < nw;
                if (has_last && (w0 + pa == n - 1 || (hasB && w0 + pa + 1 == n - 1))) {
                    // splice the new row into the last page and append it to the pool
                    const uint32_t kb = w0 + pa == n - 1 ? kbA : kbB;
                    const int row = pos % kPage;
                    const int page = MULTI ? 0 : last_page;  // (MULTI pieces never append)
                    if (page >= 0 && page < p.num_pages) {
                        if (c.lane < 2 * NCH) {
                            const int kv = c.lane / NCH, ch = c.lane % NCH;
                            const uint4 val = *reinterpret_cast<const uint4*>((kv ? c.sm->vnew : c.sm->knew) + ch * 8);
                            const uint32_t box = kb + kv * 32 * HD + (ch >> 3) * 2048;
                            const uint32_t dst = box + row * 128 + (((ch & 7) ^ (row & 7)) << 4);
                            asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(val.x),
                                         "r"(val.y), "r"(val.z), "r"(val.w) : "memory");
                            bf16* gdst = p.kv + ((((size_t)l * p.num_pages + page) * 2 + kv) * p.Hkv + g) *
                                                    kPage * HD + (size_t)row * HD + ch * 8;
                            *reinterpret_cast<uint4*>(gdst) = val;
                        }
                    } else {
                        set_error(p, c.sm, kErrBadPage, task);
                    }
                    fence_proxy_async_smem();  // generic writes before the slot's next TMA fill
                    __syncwarp();
                }
                // S^T = K q^T for both pages: A = K rows (keys) via ldmatrix, B = q^T; four
                // accumulator chains (page A / B x hi / lo; PK: page A / B x even / odd k-step)
                float shA[4] = {0.f, 0.f, 0.f, 0.f}, slA[4] = {0.f, 0.f, 0.f, 0.f};
                float shB[4] = {0.f, 0.f, 0.f, 0.f}, slB[4] = {0.f, 0.f, 0.f, 0.f};
                {
                    const int krow = lrow8 + (lmi & 1) * 8;
#pragma unroll
                    for (int s = 0; s < NKS; ++s) {
                        const int ch = 2 * s + (lmi >> 1);
                        const uint32_t off = (ch >> 3) * 2048 + krow * 128 + (((ch & 7) ^ (krow & 7)) << 4);
                        uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
                        ldmatrix_x4(kbA + off, a0, a1, a2, a3);
                        ldmatrix_x4(kbB + off, b0, b1, b2, b3);  // (page B may be past the piece: masked)
                        if (PK) {
                            mma_16816(s & 1 ? slA : shA, a0, a1, a2, a3, qa[s][0], qa[s][1]);
                            mma_16816(s & 1 ? slB : shB, b0, b1, b2, b3, qa[s][0], qa[s][1]);
                        } else {
                            mma_16816(shA, a0, a1, a2, a3, qa[s][0], qa[s][1]);
                            mma_16816(shB, b0, b1, b2, b3, qa[s][0], qa[s][1]);
                            mma_16816(slA, a0, a1, a2, a3, ql[s][0], ql[s][1]);
                            mma_16816(slB, b0, b1, b2, b3, ql[s][0], ql[s][1]);
                        }
                    }
                }
                // scores of keys A+g, A+g+8, B+g, B+g+8 (index 4 * page + 2 * (g + 8) + head)
                auto valid = [&](int key) { return key >= lo && key <= pos; };
                const bool okB = hasB;
                uint32_t ph[2][2], pl[2][2];  // [page][b0b1 | b2b3]
                if (PK) {
                    // this lane's head t: D columns 2t (hi) and 2t + 1 (lo), both k-step chains
                    float sc[4];
                    sc[0] = valid(keyA + gq) ? ((shA[0] + slA[0]) + (shA[1] + slA[1])) * p.scale : -INFINITY;
                    sc[1] = valid(keyA + gq + 8) ? ((shA[2] + slA[2]) + (shA[3] + slA[3])) * p.scale : -INFINITY;
                    sc[2] = okB && valid(keyB + gq) ? ((shB[0] + slB[0]) + (shB[1] + slB[1])) * p.scale : -INFINITY;
                    sc[3] = okB && valid(keyB + gq + 8) ? ((shB[2] + slB[2]) + (shB[3] + slB[3])) * p.scale : -INFINITY;
                    float mb = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
                    mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 4));
                    mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 8));
                    mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 16));
                    const float m_new = fmaxf(m_run[0], mb);
                    float corr = 1.f, pv[4] = {0.f, 0.f, 0.f, 0.f};
                    if (m_new != -INFINITY) {
                        corr = expf(m_run[0] - m_new);
#pragma unroll
                        for (int k = 0; k < 4; ++k) pv[k] = expf(sc[k] - m_new);
                    }
                    m_run[0] = m_new;
                    l_run[0] = l_run[0] * corr + ((pv[0] + pv[1]) + (pv[2] + pv[3]));
#pragma unroll
                    for (int mt = 0; mt < NMT; ++mt) {
                        oacc[mt][0] *= corr; oacc[mt][1] *= corr; oacc[mt][2] *= corr; oacc[mt][3] *= corr;
                    }
                    // P^T as the B operand: column gq = (head gq / 2, half gq % 2)
#pragma unroll
                    for (int k = 0; k < 4; ++k) pbuf[(gq + 8 * k) * 5 + t] = pv[k];
                    __syncwarp();
                    const int hq = gq >> 1;
#pragma unroll
                    for (int pg = 0; pg < 2; ++pg) {
                        uint32_t h0, l0, h1, l1;
                        split_bf16x2(pbuf[(16 * pg + 2 * t) * 5 + hq], pbuf[(16 * pg + 2 * t + 1) * 5 + hq], h0, l0);
                        split_bf16x2(pbuf[(16 * pg + 2 * t + 8) * 5 + hq], pbuf[(16 * pg + 2 * t + 9) * 5 + hq], h1, l1);
                        ph[pg][0] = (gq & 1) ? l0 : h0;
                        ph[pg][1] = (gq & 1) ? l1 : h1;
                    }
                    __syncwarp();
                } else {
                float sc[8];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    sc[e] = valid(keyA + gq + (e >> 1) * 8) ? (shA[e] + slA[e]) * p.scale : -INFINITY;
                    sc[4 + e] = okB && valid(keyB + gq + (e >> 1) * 8) ? (shB[e] + slB[e]) * p.scale : -INFINITY;
                }
                float pv[8];
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    float mb = fmaxf(fmaxf(sc[hh], sc[2 + hh]), fmaxf(sc[4 + hh], sc[6 + hh]));
                    mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 4));
                    mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 8));
                    mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 16));
                    const float m_new = fmaxf(m_run[hh], mb);
                    float corr = 1.f;
#pragma unroll
                    for (int k = 0; k < 4; ++k) pv[2 * k + hh] = 0.f;
                    if (m_new != -INFINITY) {
                        corr = expf(m_run[hh] - m_new);
#pragma unroll
                        for (int k = 0; k < 4; ++k) pv[2 * k + hh] = expf(sc[2 * k + hh] - m_new);
                    }
                    m_run[hh] = m_new;
                    l_run[hh] = l_run[hh] * corr + ((pv[hh] + pv[2 + hh]) + (pv[4 + hh] + pv[6 + hh]));
#pragma unroll
                    for (int mt = 0; mt < NMT; ++mt) { oacc[mt][hh] *= corr; oacc[mt][2 + hh] *= corr; }
                }
                // P^T as the B operand (32 keys x heads): transpose through this warp's buffer
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int key = gq + 8 * k;  // A: g, g+8; B: 16+g, 24+g
                    pbuf[key * 9 + 2 * t] = pv[2 * k];
                    pbuf[key * 9 + 2 * t + 1] = pv[2 * k + 1];
                }
                __syncwarp();
#pragma unroll
                for (int pg = 0; pg < 2; ++pg) {
                    split_bf16x2(pbuf[(16 * pg + 2 * t) * 9 + gq], pbuf[(16 * pg + 2 * t + 1) * 9 + gq], ph[pg][0], pl[pg][0]);
                    split_bf16x2(pbuf[(16 * pg + 2 * t + 8) * 9 + gq], pbuf[(16 * pg + 2 * t + 9) * 9 + gq], ph[pg][1], pl[pg][1]);
                }
                __syncwarp();
                }
                // keys 2t, 2t+1 / 2t+8, 2t+9 of each page's V^T: zero the invalid ones
                auto vmask = [&](int k0) {
                    return (valid(k0) ? 0x0000ffffu : 0u) | (valid(k0 + 1) ? 0xffff0000u : 0u);
                };
                const uint32_t mloA = vmask(keyA + 2 * t), mhiA = vmask(keyA + 2 * t + 8);
                const uint32_t mloB = okB ? vmask(keyB + 2 * t) : 0u, mhiB = okB ? vmask(keyB + 2 * t + 8) : 0u;
                // O^T += V^T P^T: A = V^T (dims x keys) via ldmatrix.trans of the V rows
                const int vrow = lrow8 + (lmi >> 1) * 8;
#pragma unroll
                for (int mt = 0; mt < NMT; ++mt) {
                    const int ch = 2 * mt + (lmi & 1);
                    const uint32_t off = 32 * HD + (ch >> 3) * 2048 + vrow * 128 + (((ch & 7) ^ (vrow & 7)) << 4);
                    uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
                    ldmatrix_x4_trans(kbA + off, a0, a1, a2, a3);
                    ldmatrix_x4_trans(kbB + off, b0, b1, b2, b3);
                    a0 &= mloA; a1 &= mloA; a2 &= mhiA; a3 &= mhiA;
                    b0 &= mloB; b1 &= mloB; b2 &= mhiB; b3 &= mhiB;
                    mma_16816(oacc[mt], a0, a1, a2, a3, ph[0][0], ph[0][1]);
                    if (!PK) mma_16816(oacc[mt], a0, a1, a2, a3, pl[0][0], pl[0][1]);
                    mma_16816(oacc[mt], b0, b1, b2, b3, ph[1][0], ph[1][1]);
                    if (!PK) mma_16816(oacc[mt], b0, b1, b2, b3, pl[1][0], pl[1][1]);
                }
            }
            release_at(c, c.seq + j);
        }
        c.seq += nsl;
    }

    MK_PROF_MARK(c, PS_A_LOOP);
    if (l == 0) MK_TRACE_C(c, TR_A_LOOP, (uint32_t)n);
    // this warp's softmax state for local columns 2t, 2t+1 -> shared memory (rows padded
    // to HD + 8), as many columns at a time as the scratch holds
    constexpr int OS = HD + 8;
    constexpr int kFC = FinishCols<HD>::value;
    float* ws_o = c.scratch;                                  // [8][kFC][OS]
    float* ws_m = c.scratch + kConsumerWarps * kFC * OS;      // [8][8]
    float* ws_l = ws_m + 64;                                  // [8][8]
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        l_run[hh] += __shfl_xor_sync(0xffffffffu, l_run[hh], 4);
        l_run[hh] += __shfl_xor_sync(0xffffffffu, l_run[hh], 8);
        l_run[hh] += __shfl_xor_sync(0xffffffffu, l_run[hh], 16);
    }
    const int ncl = MULTI ? min(8, NC) : 1;  // one pass for one row (G columns <= kFC)
    for (int ch0 = 0; ch0 < ncl; ch0 += kFC) {
        consumer_sync();  // the key loop's P buffers / the previous pass are done with it
        if (PK) {  // head t: the hi and lo columns of its D summed
            if (t < G) {
                if (gq == 0) { ws_m[c.cw * 8 + t] = m_run[0]; ws_l[c.cw * 8 + t] = l_run[0]; }
#pragma unroll
                for (int mt = 0; mt < NMT; ++mt) {
                    ws_o[(c.cw * kFC + t) * OS + 16 * mt + gq] = oacc[mt][0] + oacc[mt][1];
                    ws_o[(c.cw * kFC + t) * OS + 16 * mt + gq + 8] = oacc[mt][2] + oacc[mt][3];
                }
            }
        } else {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int h = 2 * t + hh;
            if (MULTI ? (h >= ch0 && h < ch0 + kFC && tile * 8 + h < NC) : h < G) {
                if (gq == 0) { ws_m[c.cw * 8 + h] = m_run[hh]; ws_l[c.cw * 8 + h] = l_run[hh]; }
#pragma unroll
                for (int mt = 0; mt < NMT; ++mt) {
                    ws_o[(c.cw * kFC + h - ch0) * OS + 16 * mt + gq] = oacc[mt][hh];
                    ws_o[(c.cw * kFC + h - ch0) * OS + 16 * mt + gq + 8] = oacc[mt][2 + hh];
                }
            }
        }
        }
        MK_PROF_MARK(c, PS_A_POST);
        attention_finish<HD, MULTI>(l, pc, ch0, NC, wpt);
    }
    return c.seq;
}

// The attention stage of layer l; GROUPS: with shared-prefix groups declared (a separate
// function, so the common path carries none of the group partition's code).
template <int HD, bool GROUPS>
__device__ __noinline__ uint32_t attention_stage(uint32_t seq, int l, int cta) {
    Ctx c = make_ctx(seq);
    MK_PROF_MARK(c, PS_OTHER);
    MK_TRACE_C(c, TR_WAIT, l * 16 + ST_ATTN);
    // every piece first writes its partial record; then each split merges its slice
    auto piece = [&](const Piece& pc) {
        MK_TRACE_C(c, TR_PIECE, (uint32_t)(pc.b * 256 + pc.g));
        if (pc.prefix) c.seq = attention_piece<HD, true, false>(c.seq, l, pc);
        else if (c.a->p.G <= 4) c.seq = attention_piece<HD, false, true>(c.seq, l, pc);
        else c.seq = attention_piece<HD, false, false>(c.seq, l, pc);
    };
    auto merge = [&](const Piece& pc) {
        if (pc.prefix) return;  // a shared prefix's records are merged by each row's own CTAs
        attention_merge<HD>(l, pc.b, pc.g, pc.split, pc.nsplit, pc.nrec);
        MK_TRACE_C(c, TR_MERGE, (uint32_t)(pc.b * 256 + pc.g));
    };
    if (GROUPS) {
        for_each_group_piece(*c.a, c.sm->pos, l, cta, piece);
        for_each_group_piece(*c.a, c.sm->pos, l, cta, merge);
    } else {
        // The partition depends only on the step's positions and on whether the layer
        // slides, so it is computed once per step and layer class and kept in shared memory.
        const Plan& p = c.a->p;
        const int cls = (p.window > 0 && ((p.sliding_mask[l >> 5] >> (l & 31)) & 1u)) ? 1 : 0;
        const int want = c.sm->cstep * 2 + cls + 1;
        Piece* cached = reinterpret_cast<Piece*>(c.sm->pc_words[cls]);
        if (c.sm->pc_tag[cls] != want) {
            int k = 0;
            for_each_row_piece(*c.a, c.sm->pos, l, cta, [&](const Piece& pc) {
                if (k < kPieceCache && c.tid == 0) cached[k] = pc;
                ++k;
            });
            consumer_sync();  // (every thread has read the previous tag)
            if (c.tid == 0) {
                c.sm->pc_n[cls] = k <= kPieceCache ? k : -1;
                c.sm->pc_tag[cls] = want;
            }
            consumer_sync();
        }
        const int np = c.sm->pc_n[cls];
        if (np < 0) {
            for_each_row_piece(*c.a, c.sm->pos, l, cta, piece);
            for_each_row_piece(*c.a, c.sm->pos, l, cta, merge);
        } else {
#pragma unroll 1
            for (int i = 0; i < np; ++i) piece(cached[i]);
#pragma unroll 1
            for (int i = 0; i < np; ++i) merge(cached[i]);
        }
    }
    // larger batches: every CTA counts its (possibly empty) share of the merges
    if (!tagged(*c.a)) publish(c, cnt_stage(l, ST_ATTN), l * 16 + ST_ATTN);
    MK_PROF_MARK(c, PS_A_END);
    return c.seq;
}

// x[b] = E[token b]. Each CTA writes the residual rows it owns (the same rows its O and
// down tiles update) and keeps them in shared memory for those residual adds.
__device__ __forceinline__ void embed_stage(Ctx& c, int cta) {
    const StepArgs& a = *c.a;
    const Plan& p = a.p;
    int a0, a1;
    cta_rows(p.d, cta, p.C, a0, a1);
    const int nr = a1 - a0;
    if (!c.sm->abort)
        for (int e = c.tid; e < a.B * nr; e += kConsumerThreads) {
            const int b = e / nr, k = a0 + e % nr;
            const int tok = c.sm->cstep == 0 ? __ldg(a.tokens + b) : c.sm->tok[b];
            const float v = __bfloat162float(p.embed[(size_t)tok * p.d + k]);
            const size_t o = (size_t)b * p.d + perm_col(k);
            if (!tagged(a)) p.xf[o] = v;
            else if (a.skip_publish != -2) ll_st(p.x + o, v, tag_of(a, 0, TAG_EMBED));
            c.sm->xown[b][k - a0] = v;
        }
    if (!tagged(a)) publish(c, cnt_embed(), -2);
}

// After the LM head: every CTA writes its running argmax of each row as a tagged pair
// (value, index); CTA 0 reads every CTA's pairs and reduces them (largest value, lowest
// index on ties) into next_tokens. When another step of the launch follows, every CTA
// reduces them itself (its next embedding needs the tokens), and each first releases the
// step's K/V appends, which the next step's TMA page loads in other CTAs will read.
template <bool MULTI>
__device__ __forceinline__ void argmax_finish(Ctx& c, int cta) {
    const StepArgs& a = *c.a;
    const Plan& p = a.p;
    const int step = MULTI ? c.sm->cstep : 0;
    const bool more = MULTI && step + 1 < a.n_steps;
    const int task = p.L * 16;
    const uint32_t tag = tag_of(a, p.L, TAG_EMBED);  // layer index L: no other write uses it
    consumer_sync();  // every warp's LM-head epilogue has updated amax_v / amax_i
    const bool tk = topk_sampling(a);
    if (c.tid == 0 && !c.sm->abort && a.skip_publish != task) {
        if (more) {
            fence_proxy_async_global();
            __threadfence();
        }
        for (int b = 0; b < a.B; ++b)
            ll_st2(p.amax + ((size_t)cta * p.maxB + b) * 2, c.sm->amax_v[b],
                   __int_as_float(c.sm->amax_i[b]), tag);
    }
    if (tk && c.cw < a.B && c.lane < a.top_k && !c.sm->abort && a.skip_publish != task) {
        // top-k sampling: this CTA's list of each row (each writer releases the step's
        // K/V appends first, as thread 0 does above)
        if (more) {
            fence_proxy_async_global();
            __threadfence();
        }
        const int b = c.cw;
        ll_st2(p.cand + (((size_t)cta * p.maxB + b) * kMaxSampleTopK + c.lane) * 2, c.sm->tk_v[b][c.lane],
               __int_as_float(c.sm->tk_i[b][c.lane]), tag);
    }
    if (!more && cta != 0) return;
    if (tk && c.cw < a.B) {
        const int b = c.cw;
        const int tok = tk_draw(b, tag, task);
        if (c.lane == 0) {
            c.sm->tok[b] = tok;
            if (cta == 0) a.next_tokens[(size_t)step * a.B + b] = tok;
        }
    } else if (c.cw < a.B) {
        const int b = c.cw;
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        // up to 8 CTAs' pairs per lane in flight at once; a missing pair is then awaited
        // alone and the batch re-read
        for (int k0 = c.lane; k0 < p.C; k0 += 8 * 32) {
            uint64_t w[8][2];
            Spin sp;
            for (;;) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int k = k0 + 32 * j;
                    w[j][0] = w[j][1] = (uint64_t)tag << 32;
                    if (k < p.C) ll_ld2(p.amax + ((size_t)k * p.maxB + b) * 2, w[j][0], w[j][1]);
                }
                int miss = -1;
#pragma unroll
                for (int j = 7; j >= 0; --j)
                    if (ll_tag(w[j][0]) != tag || ll_tag(w[j][1]) != tag) miss = j;
                if (miss < 0 || !ll_wait_pair(p.amax + ((size_t)(k0 + 32 * miss) * p.maxB + b) * 2, tag,
                                              sp, a, c.sm, task))
                    break;
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (k0 + 32 * j >= p.C) continue;
                const float v = ll_val(w[j][0]);
                const int vi = __float_as_int(ll_val(w[j][1]));
                if (v > bv || (v == bv && vi < bi)) { bv = v; bi = vi; }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
        }
        const int tok = bi == 0x7fffffff ? 0 : bi;
        if (c.lane == 0) {
            c.sm->tok[b] = tok;
            if (cta == 0) a.next_tokens[(size_t)step * a.B + b] = tok;
        }
    }
    if (!more) return;
    consumer_sync();  // the tokens are in shared memory; every warp is past this step's reads
    if (c.tid == 0) {
        __threadfence();  // the pairs read above: acquire the step's K/V appends they released
        fence_proxy_async_global();
        c.sm->step_ready = step + 1;
        c.sm->cstep = step + 1;
        // the consumers' step arguments for the next step (the loader reads none of these)
        StepArgs& m = *const_cast<StepArgs*>(c.a);
        m.epoch = m.epoch % 0xFFFFFu + 1u;
        if (!tagged(m)) m.stage_target += (uint32_t)p.C;
        if (step + 2 == m.n_steps) m.logits = m.logits_last;
        for (int b = 0; b < m.B; ++b) {
            c.sm->pos[b] += 1;
            c.sm->amax_v[b] = -INFINITY;
            c.sm->amax_i[b] = 0x7fffffff;
        }
    }
    for (int i = c.tid; i < kMaxBatch * kMaxSampleTopK; i += kConsumerThreads) {
        c.sm->tk_v[i / kMaxSampleTopK][i % kMaxSampleTopK] = -INFINITY;
        c.sm->tk_i[i / kMaxSampleTopK][i % kMaxSampleTopK] = 0x7fffffff;
    }
    consumer_sync();
}

// MoE routing of layer l (every CTA, identically): warp b polls row b's E router logits,
// takes softmax probabilities p (max-subtracted), picks the top-k by p (lowest expert id
// on ties) with weights p / sum of the picked p; then the union over the batch rows, in
// ascending expert id, goes to shared memory for the consumers' and the loader's stages.
// ("Kog Inference Engine", MoE paragraphs; the softmax-top-k reading of the router.)
__device__ __noinline__ void moe_route(int l) {
    Ctx c = make_ctx(0);
    const StepArgs& a = *c.a;
    const Plan& p = a.p;
    const int E = p.E, B = a.B, task = l * 16 + ST_ROUTE;
    float* sel = c.scratch;  // [B][64]: routing weight by expert id, -1 = not routed (B > 1)
    // Warp b routes row b; the other warps go straight to the barrier. (Routing the rows
    // redundantly on every warp tripled the issue load of the three schedulers the
    // consumers share: MoE batch 1 took 1.228 ms per step that way, 1.126 ms this way.)
    // The code is kept compact (loops not unrolled): it runs once per layer, so its
    // instructions are fetched cold each time.
    if (!c.sm->abort && c.cw < B) {
        const int b = c.cw;
        const uint32_t tag = tag_of(a, l, TAG_ROUTE);
        const uint64_t* row = p.route + (size_t)b * E;
        float v0 = -INFINITY, v1 = -INFINITY;
        {
            const int e0 = c.lane, e1 = c.lane + 32;
            uint64_t w0 = (uint64_t)tag << 32, w1 = (uint64_t)tag << 32;
            Spin sp;
            for (;;) {
                if (e0 < E) w0 = ll_ld(row + e0);
                if (e1 < E) w1 = ll_ld(row + e1);
                if ((ll_tag(w0) == tag && ll_tag(w1) == tag) || !sp.again(a, c.sm, task)) break;
            }
            if (e0 < E) v0 = ll_val(w0);
            if (e1 < E) v1 = ll_val(w1);
        }
        if (l == 1) MK_TRACE_C(c, TR_R_POLLED, 0);
        float m = fmaxf(v0, v1);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float p0 = c.lane < E ? expf(v0 - m) : 0.f, p1 = c.lane + 32 < E ? expf(v1 - m) : 0.f;
        float z = p0 + p1;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
        p0 /= z;
        p1 /= z;
        float* pw = c.scratch + 8 * 64 + c.cw * 64;             // this warp's p, by expert
        int* ids = reinterpret_cast<int*>(c.scratch + 16 * 64) + c.cw * kMaxTopK;
        // Top-k by rank: an expert's rank is the number of experts ahead of it (larger p,
        // or equal p and a lower id); it is picked when its rank is below k. The picked
        // p are then summed in rank order, the order in which a greedy selection takes them.
        pw[c.lane] = c.lane < E ? p0 : -1.f;
        pw[c.lane + 32] = c.lane + 32 < E ? p1 : -1.f;
        __syncwarp();
        int r0 = 0, r1 = 0;
#pragma unroll 1
        for (int e = 0; e < E; e += 4) {
            const float4 v = *reinterpret_cast<const float4*>(pw + e);
            const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                r0 += (vv[q] > p0 || (vv[q] == p0 && e + q < c.lane)) ? 1 : 0;
                r1 += (vv[q] > p1 || (vv[q] == p1 && e + q < c.lane + 32)) ? 1 : 0;
            }
        }
        const int topk = p.topk;
        const bool t0 = c.lane < E && r0 < topk, t1 = c.lane + 32 < E && r1 < topk;
        if (t0) ids[r0] = c.lane;
        if (t1) ids[r1] = c.lane + 32;
        __syncwarp();
        float picked = 0.f;
#pragma unroll 1
        for (int r = 0; r < topk; ++r) picked += pw[ids[r]];
        const float w0 = t0 ? p0 / picked : -1.f, w1 = t1 ? p1 / picked : -1.f;
        if (B == 1) {  // the union is this row's route, in ascending expert id
            const uint32_t m0 = __ballot_sync(0xffffffffu, t0), m1 = __ballot_sync(0xffffffffu, t1);
            const uint32_t below = (1u << c.lane) - 1u;
            const int s0 = __popc(m0 & below), s1 = __popc(m0) + __popc(m1 & below);
            if (t0) { c.sm->moe_uni[s0] = c.lane; c.sm->moe_w[0][s0] = w0; }
            if (t1) { c.sm->moe_uni[s1] = c.lane + 32; c.sm->moe_w[0][s1] = w1; }
            if (c.lane == 0) {
                c.sm->moe_nu = __popc(m0) + __popc(m1);
                if (blockIdx.x == 0) p.moe_union[l] = __popc(m0) + __popc(m1);
            }
        } else {
            sel[b * 64 + c.lane] = w0;
            sel[b * 64 + c.lane + 32] = w1;
        }
    }
    consumer_sync();
    if (B > 1) {
        if (c.cw == 0) {
            // union over the rows, ascending expert id: slot = rank among the routed ids
            bool in0 = false, in1 = false;
#pragma unroll 1
            for (int b = 0; b < B; ++b) {
                in0 = in0 || sel[b * 64 + c.lane] >= 0.f;
                in1 = in1 || sel[b * 64 + c.lane + 32] >= 0.f;
            }
            const uint32_t m0 = __ballot_sync(0xffffffffu, in0), m1 = __ballot_sync(0xffffffffu, in1);
            const uint32_t below = (1u << c.lane) - 1u;
            const int s0 = __popc(m0 & below), s1 = __popc(m0) + __popc(m1 & below);
            if (in0) c.sm->moe_uni[s0] = c.lane;
            if (in1) c.sm->moe_uni[s1] = c.lane + 32;
#pragma unroll 1
            for (int b = 0; b < B; ++b) {  // (rows b >= B are never read)
                if (in0) c.sm->moe_w[b][s0] = fmaxf(sel[b * 64 + c.lane], 0.f);
                if (in1) c.sm->moe_w[b][s1] = fmaxf(sel[b * 64 + c.lane + 32], 0.f);
            }
            if (c.lane == 0) {
                c.sm->moe_nu = __popc(m0) + __popc(m1);
                if (blockIdx.x == 0) p.moe_union[l] = __popc(m0) + __popc(m1);
            }
        }
        consumer_sync();
    }
    MK_PROF_MARK(c, PS_MOE_ROUTE);
    if (l == 1) MK_TRACE_C(c, TR_R_DONE, 0);
    if (c.tid == 0) {
        __threadfence_block();  // the routing above before the flag the loader waits on
        c.sm->moe_ready = c.sm->cstep * kMaxLayers + l + 1;
    }
}

template <int HD, bool MULTI>
__device__ __forceinline__ void consumer_run(Ctx& c, int cta) {
    const Plan& p = c.a->p;
    if (c.sm->abort) return;  // step inputs rejected (uniform: set before the first barrier)
    static_assert(sizeof(LayerPlan) % 16 == 0, "layer plans copy in 16-byte pieces");
    constexpr int kPlanChunks = (int)(sizeof(LayerPlan) / 16);
    // layer l's plan into shared memory (slot l & 1) without stalling the issuing thread;
    // it waits for its piece just before the barrier that precedes the first read
    auto fetch_plan = [&](int l) {
        if (c.tid < kPlanChunks)
            cp_async_16(smem_u32(&c.sm->lp[l & 1]) + 16 * c.tid,
                        reinterpret_cast<const uint8_t*>(p.layers + l) + 16 * c.tid);
    };
#ifdef MK_PROF
    if (c.tid < 64) c.sm->prof[c.tid] = 0;
    consumer_sync();
    const long long t_start = clock64();
    const uint64_t ns_start = globaltimer();  // with the cycle count: the SM clock of the run
    if (c.tid == 0) c.sm->prof_pt = t_start;
#endif
    const int nsteps = MULTI ? c.a->n_steps : 1;
    for (int step = 0; step < nsteps; ++step) {  // (sm->cstep advances in argmax_finish)
        fetch_plan(0);
        embed_stage(c, cta);
        MK_PROF_MARK(c, PS_EMBED);
        for (int l = 0; l < p.L; ++l) {
            if (c.tid < kPlanChunks) cp_async_wait_all();
            consumer_sync();  // layer l's plan is in place; slot (l + 1) & 1 is free
            c.seq = gemv_stage_call(c.seq, G_QKV, l, cta);
            MK_PROF_MARK(c, PS_T_RET);
            if (l + 1 < p.L) fetch_plan(l + 1);  // read at the next layer, after a barrier
            c.seq = c.a->pf_on ? attention_stage<HD, true>(c.seq, l, cta) : attention_stage<HD, false>(c.seq, l, cta);
            MK_PROF_MARK(c, PS_T_RET);
            c.seq = gemv_stage_call(c.seq, G_O, l, cta);
            MK_PROF_MARK(c, PS_T_RET);
            if (p.E > 0) {
                c.seq = gemv_stage_call(c.seq, G_ROUTE, l, cta);
                moe_route(l);
            }
            c.seq = gemv_stage_call(c.seq, G_GU, l, cta);
            MK_PROF_MARK(c, PS_T_RET);
            c.seq = gemv_stage_call(c.seq, G_DOWN, l, cta);
            MK_PROF_MARK(c, PS_T_RET);
        }
        c.seq = gemv_stage_call(c.seq, G_LM, 0, cta);
        argmax_finish<MULTI>(c, cta);
        MK_PROF_MARK(c, PS_ARGMAX);
        if (c.sm->abort) break;
    }
#ifdef MK_PROF
    if (c.tid == 0) {
        c.sm->prof[PS_TOTAL] += clock64() - t_start;
        c.sm->prof[PS_TOTAL_NS] += globaltimer() - ns_start;
    }
    consumer_sync();
    if (c.tid < 64 && cta < kProfCtas) g_mk_prof[cta][c.tid] += c.sm->prof[c.tid];
#endif
    MK_TRACE_C(c, TR_END, 0);
}

// The two roles as functions of their own (each with its own register allocation, and
// no state whose address escapes: every member the loader walks with stays in registers).
template <int HD, bool MULTI>
__device__ __noinline__ void loader_main(int cta, bool prefetch, const CUtensorMap* tmap) {
    const Ctx c = make_ctx(0);
    Producer pr;
    pr.a = c.a;
    pr.tmap = tmap;
    pr.sm = c.sm;
    pr.ring_s = c.ring_s;
    pr.lane = c.lane;
    pr.pf = prefetch;
    pr.run<HD, MULTI>(cta);
}
template <int HD, bool MULTI>
__device__ __noinline__ void consumer_main(int cta) {
    Ctx c = make_ctx(0);
    consumer_run<HD, MULTI>(c, cta);
}

// MULTI: a launch of several steps (mk_decode_steps); single-step launches run the
// instance without the step loop and its cross-step hand-off.
template <int HD, bool MULTI = false>
__global__ void __launch_bounds__(kThreads, 1) decode_step_kernel(const __grid_constant__ StepArgs a_param) {
    const uint32_t raw_s = smem_u32(mk_smem);
    const uint32_t pad = (1024u - (raw_s & 1023u)) & 1023u;
    uint8_t* ring = mk_smem + pad;
    Smem* sm = reinterpret_cast<Smem*>(ring + kStages * kSlotBytes + kScratchBytes);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    {
        static_assert(sizeof(StepArgs) % 16 == 0, "step arguments copy in 16-byte pieces");
        const uint4* src = reinterpret_cast<const uint4*>(&a_param);
        uint4* dst = reinterpret_cast<uint4*>(&sm->args);
        for (int i = threadIdx.x; i < (int)(sizeof(StepArgs) / 16); i += kThreads) dst[i] = src[i];
    }
    __syncthreads();
    const StepArgs& a = sm->args;

    if (threadIdx.x == 0) {
#ifdef MK_TRACE
        sm->trace_n = 0;
#endif
        sm->abort = 0;
        sm->lseq = 0;
        sm->moe_ready = 0;
        sm->step_ready = 0;
        sm->cstep = 0;
        sm->pc_tag[0] = sm->pc_tag[1] = 0;
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&sm->full[s]), 1);
            mbar_init(smem_u32(&sm->empty[s]), kConsumerWarps);
        }
        fence_barrier_init();
        // step-input checks (every CTA reads the same values)
        bool bad = a.B < 1 || a.B > a.p.maxB;
        for (int b = 0; b < kMaxBatch; ++b) sm->pos[b] = sm->ppos[b] = 0;
        bad = bad || a.n_steps < 1;
        for (int b = 0; b < a.B && !bad; ++b) {
            const int tok = __ldg(a.tokens + b), pos = __ldg(a.positions + b);
            const int sl = __ldg(a.seq_lens + b);
            const int last = pos + a.n_steps - 1;  // position of the launch's last step
            bad = tok < 0 || tok >= a.p.V || pos < 0 || last >= a.p.max_pos || last < pos ||
                  sl != pos + 1 || last / kPage >= a.max_pages;
            sm->pos[b] = sm->ppos[b] = pos;
        }
        if (bad) set_error(a.p, sm, kErrInvalid, -1);
        if (status_bad(a.p)) sm->abort = 1;
    }
    if (threadIdx.x < kMaxBatch) {
        sm->amax_v[threadIdx.x] = -INFINITY;
        sm->amax_i[threadIdx.x] = 0x7fffffff;
    }
    for (int i = threadIdx.x; i < kMaxBatch * kMaxSampleTopK; i += kThreads) {
        sm->tk_v[i / kMaxSampleTopK][i % kMaxSampleTopK] = -INFINITY;
        sm->tk_i[i / kMaxSampleTopK][i % kMaxSampleTopK] = 0x7fffffff;
    }
    __syncthreads();

    if (idle_warp(warp)) return;
    if (warp == 0 || warp == kPrefetchWarp) {
        // (the prefetching walker shares the loader's positions: single-step launches only)
        if (warp == 0 || (!MULTI && a.prefetch_slots > 0)) loader_main<HD, MULTI>(cta, warp != 0, &a_param.kv_tmap);
        return;
    }
    consumer_main<HD, MULTI>(cta);
}

}  // namespace mk
