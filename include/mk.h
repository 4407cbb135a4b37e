/*
 * mk.h -- C ABI of the persistent decode megakernel (sm_103a).
 *
 * One call, mk_decode_step, runs one autoregressive decode step of a pre-norm
 * transformer LM for 1..8 sequences as ONE persistent CUDA kernel: RMSNorm, QKV
 * projection, RoPE, paged-KV GQA attention (optionally sliding-window), output
 * projection + residual, SwiGLU MLP or softmax-top-k MoE, final norm, LM head and
 * greedy argmax (or temperature sampling, mk_set_sampling). Work is a task graph of
 * GEMV row tiles and attention key splits, ordered by the data instead of grid-wide
 * barriers: up to batch 4 every stage output is a tagged word its readers poll; above
 * that, per-stage dependency counters.
 *
 * Source of the operation (pages, by title and section):
 *   "Cohere, Megakernel sunum sistemini acik kaynak yapti", section
 *     "Megakernel ne demek": the whole decode pass in a single persistent CUDA
 *     kernel; work split into a graph of GEMM pieces and attention sections; no
 *     full-grid synchronisation barriers between operations.
 *   same page, section "Sinirlar acikca yazilmis": decode only, BF16 only, batch
 *     1..8, greedy sampling; continuous batching, ragged lengths, paged KV cache,
 *     sliding-window attention, prefix cache.
 *   "Kog AI: standart GPU'larda 3,000 token/s", sections on memory bandwidth and on
 *     the monokernel: decode at low batch is bound by HBM bandwidth; LM-head
 *     sampling stays on the GPU; prefetch overlaps the non-GEMM sections.
 *
 * Conventions
 *   - Every pointer passed to mk_decode_step and stored in mk_weights is CUDA
 *     device memory on the handle's device (PyTorch may allocate it). Host
 *     pointers are accepted only where a comment says "host".
 *   - All weights are BF16, row-major [out][in] (the nn.Linear convention); MoE
 *     experts are stacked [E][out][in]. Weights are BORROWED: they must stay
 *     valid and unchanged for the life of the handle.
 *   - The KV pool is OWNED by the handle (mk_kv_alloc / mk_kv_free).
 *   - Everything is asynchronous on the caller's stream (a cudaStream_t passed
 *     as void*; NULL = the legacy default stream). A handle is not thread-safe,
 *     and only one mk_decode_step may be in flight per handle at a time (its
 *     counters and scratch are per handle).
 *   - Errors found on the host return at once. Errors found on the device (a bad
 *     page id, a step input out of range, a dependency wait that timed out) are
 *     latched in a device status word and reported by mk_status_sync; the kernel
 *     then winds down without faulting the GPU. After such an error, call
 *     mk_status_reset before the next step.
 */
#ifndef MK_H_
#define MK_H_

#include <stdint.h>

#if defined(__GNUC__)
#define MK_API __attribute__((visibility("default")))
#else
#define MK_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum mk_status {
    MK_OK = 0,
    MK_ERR_INVALID_ARG = 1,        /* bad argument (host check) or bad step input (device) */
    MK_ERR_UNSUPPORTED_DEVICE = 2, /* not an sm_103 GPU, or no cooperative launch */
    MK_ERR_OOM = 3,                /* device allocation failed / KV pool too large */
    MK_ERR_LAUNCH = 4,             /* kernel launch refused (e.g. CTAs not co-resident) */
    MK_ERR_BAD_PAGE = 5,           /* a page-table entry used by the step is out of range */
    MK_ERR_TIMEOUT = 6,            /* a dependency wait passed its time limit */
    MK_ERR_INTERNAL = 7,           /* CUDA runtime error or broken invariant */
    MK_ERR_NO_DEVICE = 8           /* no CUDA device visible */
} mk_status;

/* Model descriptor (copied by mk_create). */
typedef struct mk_model_desc {
    int32_t n_layers;
    int32_t d_model;        /* multiple of 64 */
    int32_t n_q_heads;
    int32_t n_kv_heads;     /* n_q_heads / n_kv_heads <= 8 */
    int32_t head_dim;       /* 64 or 128 */
    int32_t ffn_dim;        /* dense SwiGLU width (multiple of 64); unused when n_experts > 0 */
    int32_t vocab;
    int32_t n_experts;      /* 0 = dense SwiGLU MLP; else softmax-top-k MoE */
    int32_t top_k;
    int32_t expert_ffn_dim; /* multiple of 64 */
    float rms_eps;          /* RMSNorm epsilon, e.g. 1e-5 */
    float rope_theta;       /* rotate-half RoPE base, e.g. 1e4 */
    int32_t sliding_window; /* 0 = none; else a sliding layer attends to the last W keys */
    const uint8_t *layer_is_sliding; /* host, [n_layers], nonzero = sliding; may be NULL */
    int32_t max_batch;      /* 1..8 */
    int32_t page_size;      /* must be 16 */
    int32_t max_positions;  /* positions[b] must stay below this (RoPE table size) */
} mk_model_desc;

typedef struct mk_layer_weights {
    const void *attn_norm;  /* [d] */
    const void *wq;         /* [n_q_heads*head_dim][d] */
    const void *wk;         /* [n_kv_heads*head_dim][d] */
    const void *wv;         /* [n_kv_heads*head_dim][d] */
    const void *wo;         /* [d][n_q_heads*head_dim] */
    const void *mlp_norm;   /* [d] */
    const void *w_gate;     /* dense: [ffn][d] */
    const void *w_up;       /* dense: [ffn][d] */
    const void *w_down;     /* dense: [d][ffn] */
    const void *router;     /* MoE: [E][d] */
    const void *exp_gate;   /* MoE: [E][expert_ffn][d] */
    const void *exp_up;     /* MoE: [E][expert_ffn][d] */
    const void *exp_down;   /* MoE: [E][d][expert_ffn] */
} mk_layer_weights;

typedef struct mk_weights {
    const void *embed;      /* [vocab][d] */
    const void *final_norm; /* [d] */
    const void *lm_head;    /* [vocab][d] (untied) */
    const mk_layer_weights *layers; /* host array [n_layers] of device pointers */
} mk_weights;

typedef struct mk_handle mk_handle;

/* Paged KV pool, BF16, layout [n_layers][num_pages][2 (K=0,V=1)][n_kv_heads][16][head_dim].
 * Strides are in elements. Page ids are global across layers: page p of layer l
 * starts at base + l*layer_stride + p*page_stride. K rows are stored after RoPE. */
typedef struct mk_kv_pool {
    void *base;             /* device; owned by the handle */
    int32_t num_pages;
    int64_t layer_stride, page_stride, kv_stride, head_stride, slot_stride;
    int64_t bytes;
} mk_kv_pool;

/* Creates a handle on `device` for one model (a descriptor plus borrowed weight
 * pointers). Source: "Cohere, Megakernel sunum sistemini acik kaynak yapti", section
 * "Sinirlar acikca yazilmis" (one model, BF16 weights, batch 1..8). Checks the GPU
 * (sm_103, cooperative launch),
 * copies the descriptor, records the weight pointers, uploads the RoPE table
 * (cos/sin computed on the host in double), and allocates the step scratch
 * (activations, attention partials, dependency counters, status word; the KV tensor
 * map is made by mk_kv_alloc).
 * Returns MK_ERR_INVALID_ARG for an unsupported shape, MK_ERR_NO_DEVICE /
 * MK_ERR_UNSUPPORTED_DEVICE for the GPU checks, MK_ERR_OOM if scratch cannot be
 * allocated. On error *out is NULL and nothing is leaked. */
MK_API mk_status mk_create(const mk_model_desc *desc, const mk_weights *weights, int device,
                    mk_handle **out);

/* Allocates the handle's paged KV pool of num_pages pages. Source: the paged KV cache
 * of "Cohere, Megakernel sunum sistemini acik kaynak yapti", section "Sinirlar acikca
 * yazilmis" (pages of 16 tokens here). One pool per handle; a
 * second call fails with MK_ERR_INVALID_ARG until mk_kv_free). The memory is not
 * initialised. Returns MK_ERR_OOM if the allocation fails. */
MK_API mk_status mk_kv_alloc(mk_handle *h, int32_t num_pages, mk_kv_pool *out);
MK_API mk_status mk_kv_free(mk_handle *h, mk_kv_pool *pool);

/* One decode step for `batch` sequences (1 <= batch <= max_batch), enqueued on
 * `stream` as a single cooperative kernel launch. Source: "Cohere, Megakernel sunum
 * sistemini acik kaynak yapti", sections "Megakernel ne demek" (the whole decode pass in
 * one persistent kernel) and "Sinirlar acikca yazilmis" (decode only, batch 1..8,
 * continuous batching, ragged lengths, paged KV, sliding window); "Kog AI: standart
 * GPU'larda 3,000 token/s", on LM-head sampling kept on the GPU.
 *   tokens[batch]       input token of each sequence (0 <= token < vocab)
 *   positions[batch]    tokens already cached = position of the input token
 *   page_table[batch][max_pages_per_seq]  entry i = page holding positions
 *                       [16i, 16i+16); every entry the step reads (the attended
 *                       range and the page of positions[b]) must be a valid page
 *   seq_lens[batch]     must equal positions[b] + 1 (keys attended incl. self)
 *   next_tokens[batch]  out: greedy argmax (lowest index on ties)
 *   logits              out: [batch][vocab] fp32, or NULL to skip
 * The step appends K/V of the input token at positions[b] of every layer, then
 * attends over keys [lo, positions[b]] (lo = 0, or positions[b]-W+1 clamped at 0
 * on sliding layers). Output buffers must not overlap the inputs. Page ids may
 * repeat across rows only for read-only shared prefixes (no row may append into
 * a page another row reads in the same step).
 * Returns host-side argument errors directly; device-side errors are latched
 * (see mk_status_sync). */
MK_API mk_status mk_decode_step(mk_handle *h, const int32_t *tokens, const int32_t *positions,
                         const int32_t *page_table, int32_t max_pages_per_seq,
                         const int32_t *seq_lens, int32_t batch, int32_t *next_tokens,
                         float *logits, void *stream);

/* One decode step from and to HOST memory, synchronous: the call a serving loop makes
 * when its tokens live on the host. The arguments mean what they mean for
 * mk_decode_step, with every pointer in host memory (pageable or pinned). The inputs
 * are packed into a pinned staging buffer the handle owns and reach the device in ONE
 * host-to-device copy; the step runs on `stream`; the device status word and the next
 * tokens come back in ONE device-to-host copy (the logits, when `logits` is not NULL,
 * in a second one); the call returns once they are in the caller's arrays.
 * The handle grows its staging buffers on the first call that needs more room (the
 * logits buffer, max_batch * vocab fp32, on the first call that asks for logits);
 * mk_destroy frees them. Calls on one handle must not overlap (the staging is shared).
 * Returns host-side argument errors, MK_ERR_OOM if staging cannot be allocated, else
 * the step's device status (MK_OK or the latched error, as mk_status_sync reports). */
MK_API mk_status mk_decode_step_host(mk_handle *h, const int32_t *tokens,
                                     const int32_t *positions, const int32_t *page_table,
                                     int32_t max_pages_per_seq, const int32_t *seq_lens,
                                     int32_t batch, int32_t *next_tokens, float *logits,
                                     void *stream);

/* n_steps consecutive decode steps of the same rows as ONE launch (the token of each
 * step is fed back on the device). Source: "Kog AI: standart GPU'larda 3,000 token/s",
 * on kernel boundaries and on sampling kept on the GPU.
 *   tokens, positions, page_table, seq_lens, batch: as for mk_decode_step, for step 0.
 *   Step s (0 <= s < n_steps) decodes at positions[b] + s; its input token is
 *   tokens[b] for s = 0, else the token step s-1 chose. Every row's page table must
 *   already map the pages of positions[b] + n_steps - 1.
 *   next_tokens[n_steps][batch]  out: the token each step chose (greedy, or sampled as
 *                       set by mk_set_sampling, with the step's own position)
 *   logits              out: the LAST step's [batch][vocab] fp32, or NULL
 * 1 <= n_steps <= 65536. The result equals n_steps calls of mk_decode_step that feed
 * each step's next_tokens back as the next tokens. Inside the launch, each CTA's loader
 * streams the next step's weights while the step's argmax is still being reduced.
 * Errors as for mk_decode_step; the device check of positions covers the last step. */
MK_API mk_status mk_decode_steps(mk_handle *h, int32_t n_steps, const int32_t *tokens,
                                 const int32_t *positions, const int32_t *page_table,
                                 int32_t max_pages_per_seq, const int32_t *seq_lens,
                                 int32_t batch, int32_t *next_tokens, float *logits,
                                 void *stream);

/* Waits for `stream`, then reads the device status word (the pages describe no error
 * mechanism; here device-side failures are latched and the kernel winds down instead of
 * faulting). Returns MK_OK or the
 * latched device error; *failing_task (may be NULL) receives the id of the task
 * that latched it (layer*16 + stage, or -1). */
MK_API mk_status mk_status_sync(mk_handle *h, void *stream, int32_t *failing_task);

/* Clears a latched device error and re-zeroes the stage counters (synchronous). */
MK_API mk_status mk_status_reset(mk_handle *h);

/* Options (host-side; take effect from the next step):
 *   MK_OPT_TIMEOUT_NS   limit for every device-side wait, in ns (default 1e9)
 *   MK_OPT_SKIP_PUBLISH test hook: the task with this id never publishes its
 *                       completion, so its waiters time out (-1 = off)
 *   MK_OPT_PREFETCH_SLOTS how many ring slots (32 KB each) a second producer warp
 *                       runs ahead of the loading warp, prefetching weights and KV
 *                       pages into L2 so that HBM streams across dependency waits;
 *                       0..64, 0 = off (the default). Results do not depend on it. */
typedef enum mk_option {
    MK_OPT_TIMEOUT_NS = 1,
    MK_OPT_SKIP_PUBLISH = 2,
    MK_OPT_PREFETCH_SLOTS = 3
} mk_option;
MK_API mk_status mk_set_option(mk_handle *h, mk_option opt, int64_t value);

/* Next-token rule from the next step on. Source: the sampling modes of "Cohere,
 * Megakernel sunum sistemini acik kaynak yapti", section "Sinirlar acikca yazilmis"
 * (greedy, temperature, a limited top_k; no top_p).
 *   temperature == 0 (the default): greedy argmax (lowest index on ties); top_k ignored.
 *   temperature > 0: a draw from softmax(logits / temperature), taken as
 *     argmax_i (logits_i / temperature + g_i) with g_i = -log(-log u_i) standard Gumbel
 *     noise; u_i comes from Philox4x32-10 with key = seed (low word first) and counter
 *     (token i, positions[b], row b, 0), u = (top 24 bits of word 0 + 0.5) / 2^24.
 *   top_k in 1..32: the draw is limited to the top_k largest logits of the row (the
 *     larger logit first, the lower index first among equal logits), i.e. softmax
 *     renormalised over them; top_k 1 is the greedy token. top_k 0: no cut.
 * The draw is a function of (seed, position, row, token) only, so a step can be replayed
 * exactly. The logits written by mk_decode_step stay the raw logits. Negative or
 * non-finite temperatures, or top_k outside 0..32: MK_ERR_INVALID_ARG.
 * mk_decode_step_noalloc is always greedy. */
MK_API mk_status mk_set_sampling(mk_handle *h, float temperature, int32_t top_k, uint64_t seed);

/* Shared prefixes (cascade attention) for the next steps of batch `batch`. Source: the
 * prefix cache of "Cohere, Megakernel sunum sistemini acik kaynak yapti", section
 * "Sinirlar acikca yazilmis", and the shared prefix caches of concurrent sessions in
 * "Magnitude: Donanimiza Gore Kernel Ayarlayan Kendi Kendini Derleyen Bir Cikarim
 * Motoru", section "Bellek ve eszamanlilik icin ne anlama geliyor?".
 *   leader[batch]        (host) row b shares its prefix with row leader[b]: leader[b] <= b
 *                        and leader[leader[b]] == leader[b]; a row with leader[b] == b and
 *                        no other member is a group of one (no sharing)
 *   shared_pages[batch]  (host) the caller guarantees that logical pages
 *                        [0, shared_pages[b]) of row b's page table hold the same page ids
 *                        as those of row leader[b]; equal within a group
 * At most 16 / (n_q_heads / n_kv_heads) rows per group (two 8-wide query column tiles).
 * In every layer where all rows of a group attend the whole prefix (no sliding window
 * cuts into it) and each row's current page lies after it, the prefix K/V pages are
 * read once per kv head for the whole group (through the leader's page table) instead
 * of once per row; elsewhere the rows attend on their own. Results do not depend on it
 * beyond fp32 summation order. batch == 0 clears the groups (leader and shared_pages
 * may be NULL). While groups are declared, mk_decode_step with another batch size
 * returns MK_ERR_INVALID_ARG. Errors: MK_ERR_INVALID_ARG for any violated rule above. */
MK_API mk_status mk_set_shared_prefix(mk_handle *h, int32_t batch, const int32_t *leader,
                                      const int32_t *shared_pages);

/* Read-only facts about a handle (for schedulers and benchmarks). */
typedef struct mk_info {
    int32_t num_ctas;          /* persistent CTAs per launch (one per SM) */
    int32_t threads_per_cta;
    int32_t smem_bytes;        /* dynamic shared memory per CTA */
    int32_t ring_stages;       /* shared-memory ring depth */
    int64_t weight_bytes;      /* bytes of weights one dense step streams (all layers + head) */
    int64_t scratch_bytes;     /* device scratch owned by the handle */
} mk_info;
MK_API mk_status mk_get_info(const mk_handle *h, mk_info *out);

/* The decode step for callers that cannot allocate device memory. It has no
 * counterpart in the pages: it is the same kernel as mk_decode_step, but it needs no
 * handle and allocates nothing. Callers that cannot call cudaMalloc -- code running
 * under a memory plan that owns every byte of HBM, allocator-free or sandboxed
 * runtimes, paths where an allocation would synchronise the device -- pass every
 * input and output themselves, including the KV pool.
 *
 * All scratch (norm gains, RoPE table, layer table, activations, attention partials,
 * dependency counters, status word) lives in one file-scope static
 * device array of MK_NOALLOC_SCRATCH_BYTES (8 MiB), which every GPU that loads this
 * library holds until the process exits. Descriptors whose scratch does not fit
 * (roughly: max_batch * n_kv_heads * 148 * (n_q_heads/n_kv_heads) * head_dim * 4 bytes
 * of attention partials, plus max_positions * head_dim * 4 bytes of RoPE table, plus
 * small terms) are rejected with MK_ERR_INVALID_ARG before anything is enqueued.
 *   desc, weights        as for mk_create (host structs; weights on the current device)
 *   kv_pool, num_pages   caller-owned device pool in the mk_kv_pool layout (BF16,
 *                        [n_layers][num_pages][2][n_kv_heads][16][head_dim], dense)
 *   tokens .. logits     as for mk_decode_step
 *   status_out           device int32[2], out: {status, failing task} of the step,
 *                        written on `stream` after the kernel (read it after a sync)
 * Runs on the CURRENT device. The first call on a device does a one-time set-up
 * (device checks, kernel attributes, and cudaGetSymbolAddress of the static array);
 * make that first call before any stream capture. Every call re-initialises the parts
 * of the array that must start from zero (counters, status) and rewrites the tables;
 * the array keeps the last call's contents otherwise. All calls share the one array,
 * so calls whose work overlaps on the GPU (different streams, or threads) race: run
 * them one after another. Host-side errors return at once; device-side errors are
 * reported through status_out. */
#define MK_NOALLOC_SCRATCH_BYTES (8u << 20)
MK_API mk_status mk_decode_step_noalloc(const mk_model_desc *desc, const mk_weights *weights,
                                        void *kv_pool, int32_t num_pages,
                                        const int32_t *tokens, const int32_t *positions,
                                        const int32_t *page_table, int32_t max_pages_per_seq,
                                        const int32_t *seq_lens, int32_t batch,
                                        int32_t *next_tokens, float *logits,
                                        int32_t *status_out, void *stream);

/* Introspection for stage-by-stage verification. After a step has completed (sync
 * the stream first), these device buffers hold the activations of the LAST layer the
 * step ran; they are overwritten by the next step. The element size is
 * *bytes / (max_batch * width): 8 bytes when the element is a tagged word (low 32 bits
 * the fp32 value, high 32 bits the tag of the write that produced it; QKV always, the
 * others after a step with batch <= 2), else 4 bytes of plain fp32.
 * Layouts (row b at b*width elements):
 *   MK_BUF_X     residual stream after the last layer (input of the final norm),
 *                [max_batch][d_model], permuted columns (below)
 *   MK_BUF_QKV   q|k|v projections of the last layer, BEFORE RoPE, natural order,
 *                [max_batch][(n_q_heads + 2 n_kv_heads) * head_dim]
 *   MK_BUF_ATTN  attention output of the last layer (input of the O projection),
 *                [max_batch][n_q_heads * head_dim], permuted columns
 *   MK_BUF_H     SwiGLU activations of the last layer (input of the down projection),
 *                [max_batch][ffn_dim], permuted columns; for a MoE model
 *                [max_batch][n_experts * expert_ffn_dim], where slot j of the routed
 *                union (ascending expert id) holds columns [j*Fe, (j+1)*Fe), already
 *                multiplied by the row's routing weight (0 for an expert it did not pick)
 *   MK_BUF_ROUTE router logits of the last layer, [max_batch][n_experts], tagged words
 *   MK_BUF_MOE_UNION  int32 [n_layers]: experts in each layer's routed union (last step)
 * Permuted columns: logical column k is stored at
 *   (k & ~63) | ((k & 7) >> 1) << 4 | ((k & 63) >> 3) << 1 | (k & 1).
 * *dev_ptr receives the device address (read-only use), *bytes its size. */
typedef enum mk_buffer {
    MK_BUF_X = 1,
    MK_BUF_QKV = 2,
    MK_BUF_ATTN = 3,
    MK_BUF_H = 4,
    MK_BUF_ROUTE = 5,
    MK_BUF_MOE_UNION = 6
} mk_buffer;
MK_API mk_status mk_debug_buffer(const mk_handle *h, int32_t which, void **dev_ptr,
                                 int64_t *bytes);

MK_API const char *mk_status_string(mk_status s);

/* Frees everything the handle owns (scratch, KV pool, RoPE table). Synchronises
 * the device first. NULL is allowed. */
MK_API void mk_destroy(mk_handle *h);

#ifdef __cplusplus
}
#endif
#endif /* MK_H_ */
