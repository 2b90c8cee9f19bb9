/*
 * libpagedattn -- decode-phase attention over a paged KV cache (GB300, sm_103a).
 *
 * The operation: during decode every sequence of the batch adds one token.
 * Its keys/values are appended to the sequence's KV cache, and each query
 * head attends over all cached tokens:
 *
 *     out[b][h] = softmax(scale * K_b q[b][h]) V_b
 *
 * K_b and V_b are the sequence's cached rows of KV head h / G (G = Hq / Hkv,
 * consecutive query heads share a KV head).  They are gathered through the
 * sequence's block table of fixed-size pages.
 *
 * Sources (web pages, by title and section):
 *  - "Eine LLM-Inferenz-Engine von Grund auf mit C++ und CUDA bauen",
 *    section 1.1: the KV cache, prefill vs. one-token-at-a-time decode.
 *    Section 3.4: long-context attention reads contiguous blocks and merges
 *    without atomics.
 *  - swiftLLM, feature list: PagedAttention (block-table paging) and paged
 *    attention v2 (Flash-Decoding: split the sequence, merge with
 *    log-sum-exp).
 *  - MonadKai/xLLM, introduction: KV cache with GQA; online-normaliser
 *    softmax.
 *
 * Conventions shared by every call:
 *  - Types: q, K, V, k_new, v_new and out are IEEE fp16.  Accumulation is
 *    fp32.  Indices are int32.
 *  - Layouts, all dense row-major:
 *      q, out           [batch][num_q_heads][head_dim]
 *      k_new, v_new     [batch][num_kv_heads][head_dim]
 *      k_pages, v_pages [num_pages][num_kv_heads][page_size][head_dim]
 *                       (each (page, kv head) slice is one contiguous run of
 *                       page_size * head_dim halves)
 *      block_table      [batch][max_pages_per_seq]; entry j is the physical
 *                       page holding tokens j*S .. j*S+S-1 of the sequence
 *      seq_lens         [batch]; counts the token being decoded
 *  - Logical token t of sequence b sits in page block_table[b][t / S], slot
 *    t % S.
 *  - Supported shapes: head_dim 64 or 128, page_size 16, G = Hq / Hkv in
 *    {1, 2, 4, 8}.  Anything else returns PA_ERR_UNSUPPORTED.
 *  - Pointers named "device" are CUDA device pointers; "host" pointers are
 *    ordinary host memory.  Device buffers must be 16-byte aligned.  The
 *    caller owns every buffer.  The library allocates no device memory.
 *  - stream is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Every device call is asynchronous and stream-ordered.  It returns after
 *    launching.
 *  - Errors: bad arguments are detected on the host before any launch and
 *    return a non-zero pa_status_t.  A launch failure returns PA_ERR_CUDA.
 *    Problems seen only on the device do not trap.  The kernel skips the
 *    access and ORs a PA_DEV_* bit into *dev_status (device int32, caller
 *    zeroes it; read it after the stream is synchronised).  Such problems
 *    are a block-table entry outside [0, num_pages), a seq_len outside
 *    [0, max_pages_per_seq * S], or a workspace not holding the plan.
 */
#ifndef PAGEDATTN_H
#define PAGEDATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1,  /* null pointer, misaligned buffer, bad size, bad seq_len */
  PA_ERR_UNSUPPORTED = 2,  /* head_dim / page_size / group size not built */
  PA_ERR_WORKSPACE = 3,    /* workspace smaller than the plan needs */
  PA_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
  PA_ERR_DEVICE_OOB = 5,   /* (reported through dev_status, see below) */
  PA_ERR_TIMEOUT = 6,      /* (reported through dev_status, see below) */
  PA_ERR_NO_MEMORY = 7,    /* host allocation in pa_plan failed */
  PA_ERR_PLAN = 8          /* plan does not match the shape */
} pa_status_t;

/* Bits ORed into *dev_status by the kernels. */
#define PA_DEV_BAD_PAGE 0x1       /* block-table entry outside [0, num_pages): page skipped */
#define PA_DEV_BAD_SEQ_LEN 0x2    /* seq_len < 0 or > max_pages_per_seq * page_size: clamped */
#define PA_DEV_PLAN_MISMATCH 0x4  /* workspace does not hold this plan, or seq_lens differ from it */
#define PA_DEV_TIMEOUT 0x8        /* a bounded wait gave up: the outputs it feeds are not written */

typedef struct {
  int32_t batch;             /* B, >= 0 */
  int32_t num_q_heads;       /* Hq */
  int32_t num_kv_heads;      /* Hkv, divides Hq */
  int32_t head_dim;          /* D: 64 or 128 */
  int32_t page_size;         /* S: 16 */
  int32_t max_pages_per_seq; /* row length of block_table */
  int32_t num_pages;         /* P: pages in each pool */
  int32_t dtype;             /* element type of q, k_new, v_new, the pools and out:
                                PA_DTYPE_F16 (0, the default of a zeroed struct) or
                                PA_DTYPE_BF16 (1); the INT8- and FP8-cache calls take F16 only */
} pa_shape_t;

#define PA_DTYPE_F16 0
#define PA_DTYPE_BF16 1

/*
 * A plan: how one decode call splits the batch into warp tasks.
 *
 * Each task is one (sequence, KV head, page range).  A sequence is cut into
 * several page-aligned ranges (Flash-Decoding splits) when that balances the
 * GPU.  pa_plan fills the struct.  host_blob (the task list, owned by the
 * plan) is released by pa_plan_free.
 */
typedef struct {
  pa_shape_t shape;          /* the shape the plan was made for */
  int32_t num_work_items;    /* warp tasks: one per (sequence, KV head, split) */
  int32_t num_groups;        /* (sequence, KV head) pairs with more than one split */
  int32_t num_split_items;   /* tasks that write partial results */
  int32_t max_splits;        /* largest split count of any sequence */
  int32_t chunk_pages;       /* target pages per split chosen by the planner */
  int32_t num_ctas;          /* grid of the split kernel */
  int32_t num_shared_ctas;   /* the first num_shared_ctas CTAs share one task among their warps */
  int32_t warps_per_cta;
  int32_t owns_blob;         /* 1 if host_blob was allocated by pa_plan */
  uint64_t plan_id;          /* stamp written into the workspace by pa_plan_upload */
  size_t blob_bytes;         /* bytes pa_plan_upload copies into the workspace */
  size_t workspace_bytes;    /* minimum workspace for pa_decode_attention */
  void* host_blob;           /* task list in host memory, owned by the plan */
  /* How the decode calls made with this plan run (copied from the options
   * of pa_plan_ex; pa_plan and pa_plan_in leave them 0, and every 0 is the
   * default), and the 8-bit kernels' page stages (set by every planner). */
  int32_t merge;             /* PA_MERGE_IN_SPLIT_KERNEL or PA_MERGE_COMBINE_KERNEL */
  int32_t l2_prefetch_pages; /* see pa_plan_options_t */
  int32_t l2_prefetch_ctas;  /* see pa_plan_options_t */
  int32_t q8_stages;         /* page stages per warp of the 8-bit-cache calls at head_dim 128:
                                2 or 3, set by every planner (see pa_plan_options_t) */
  uint64_t wait_limit_ns;    /* see pa_plan_options_t */
  int32_t early_kv;          /* see pa_plan_options_t */
} pa_plan_t;

/* How the split partials of a sequence are merged (paged attention v2's
 * log-sum-exp reduce). */
#define PA_MERGE_IN_SPLIT_KERNEL 0 /* the last split task of each (sequence, KV head) to
                                      finish merges them inside the split kernel: one launch */
#define PA_MERGE_COMBINE_KERNEL 1  /* split tasks only write partials; a separate combine
                                      kernel launched after the split kernel merges them */

/*
 * Options of a decode plan.  A zeroed struct, or a NULL pointer, gives the
 * defaults: every field's 0 is its default.  The planner fields change the
 * task list; the others are copied into the plan and read by each decode
 * call made with it.
 */
typedef struct {
  int32_t min_chunk_pages;   /* automatic plan: no split shorter than this many pages (0: 48) */
  int32_t waves;             /* automatic plan: about waves x resident CTAs tasks (0: 1) */
  int32_t bundle_max_pages;  /* when the GPU runs several waves of tasks, tasks of at most
                                this many pages run one per warp, four to a CTA
                                (0: 8; negative: never) */
  int32_t bundle_waves;      /* "several": more tasks than bundle_waves x the CTAs the GPU
                                holds at once (0: 3; negative: bundle at any task count) */
  int32_t merge;             /* PA_MERGE_IN_SPLIT_KERNEL (0) or PA_MERGE_COMBINE_KERNEL */
  int32_t l2_prefetch_pages; /* pages per warp that the split kernel's first CTAs ask L2 for
                                while the previous kernel still runs (0: 2; negative:
                                none; at most 32) */
  int32_t l2_prefetch_ctas;  /* CTAs that prefetch (0: the first wave, the CTAs the GPU
                                holds at once; negative: none) */
  int32_t q8_stages;         /* page stages per warp of the INT8 and FP8 split kernel at
                                head_dim 128: 2 or 3 (0: the planner's choice, 3 when all
                                the plan's CTAs are resident at once, else 2 when the
                                tasks average at most 12 pages per warp, else 3).  Head_dim
                                64 always takes 6. */
  uint64_t wait_limit_ns;    /* how long a warp waits for one page copy before it gives up,
                                sets PA_DEV_TIMEOUT and writes nothing (0: 1 s).  A copy
                                that was issued always lands before the kernel exits. */
  int32_t early_kv;          /* 1: the split kernel reads seq_lens and the block table and
                                starts its first page copies (K/V pages, and scales of an
                                8-bit cache) before it waits for the kernel ahead of it in
                                the stream, which with programmatic dependent launch may
                                still be running; q and the new token's rows are read after
                                the wait.  Set it only when no kernel queued ahead of the
                                call that may still be running writes the caches, their
                                scales, the block table, seq_lens or dev_status: a chain of
                                layer calls, each over its own layer's cache, with seq_lens
                                and the block table copied in before the chain, qualifies;
                                pa_kv_append followed by pa_decode_attention on the same
                                cache does not.  0 (default): everything after the wait. */
} pa_plan_options_t;

/*
 * Append the new token's K and V (decode-phase cache update; from-scratch
 * engine article, section 1.1; swiftLLM PagedAttention).
 *
 * For every b with seq_lens[b] = L > 0, row k_new[b][h] is copied to
 * k_pages[block_table[b][(L-1)/S]][h][(L-1)%S], and likewise for V.  The
 * copy is bit for bit.  Sequences with L == 0 are skipped.
 * Device: k_new, v_new, k_pages, v_pages, block_table, seq_lens, dev_status.
 */
pa_status_t pa_kv_append(const pa_shape_t* shape, const void* k_new, const void* v_new,
                         void* k_pages, void* v_pages, const int32_t* block_table,
                         const int32_t* seq_lens, int32_t* dev_status, void* stream);

/*
 * Plan the split-K decomposition (swiftLLM paged attention v2 /
 * Flash-Decoding; "Eine LLM-Inferenz-Engine ...", section 3.4 on long
 * contexts).  Host-only; touches no GPU.
 *
 * seq_lens_host: host int32[batch], the lengths the next decode calls will
 * see.  num_sms: SM count of the target GPU (152 on GB300).
 * forced_splits > 0 cuts every sequence into min(forced_splits, pages)
 * near-equal page ranges.  0 lets the planner choose from the total work
 * and num_sms.
 * Returns PA_ERR_INVALID_ARG for a bad seq_len, PA_ERR_UNSUPPORTED for an
 * unsupported shape, and PA_ERR_NO_MEMORY on host allocation failure.  On
 * success *plan_out owns host memory; release it with pa_plan_free.
 */
pa_status_t pa_plan(const pa_shape_t* shape, const int32_t* seq_lens_host, int32_t num_sms,
                    int32_t forced_splits, pa_plan_t* plan_out);

/*
 * Same as pa_plan, but the task list is written into caller-owned host
 * memory (for example pinned memory, so that pa_plan_upload is a true
 * asynchronous copy and can be captured in a CUDA graph).  The plan does not
 * own host_buffer; pa_plan_free leaves it alone.  If host_buffer_bytes is
 * too small, returns PA_ERR_WORKSPACE and sets plan_out->blob_bytes to the
 * size needed.  The buffer must stay unchanged until every upload that reads
 * it has completed on its stream.
 */
pa_status_t pa_plan_in(const pa_shape_t* shape, const int32_t* seq_lens_host, int32_t num_sms,
                       int32_t forced_splits, void* host_buffer, size_t host_buffer_bytes,
                       pa_plan_t* plan_out);

/*
 * pa_plan and pa_plan_in with options (NULL: the defaults).  host_buffer
 * NULL: the plan allocates and owns its task list (as pa_plan); otherwise
 * the list goes into host_buffer (as pa_plan_in).  A field out of range
 * (merge not a PA_MERGE_* value, l2_prefetch_pages > 32, early_kv
 * not 0 or 1) returns PA_ERR_INVALID_ARG.
 */
pa_status_t pa_plan_ex(const pa_shape_t* shape, const int32_t* seq_lens_host, int32_t num_sms,
                       int32_t forced_splits, const pa_plan_options_t* options,
                       void* host_buffer, size_t host_buffer_bytes, pa_plan_t* plan_out);

/* Release the plan's host memory (safe on a zeroed or already freed plan). */
void pa_plan_free(pa_plan_t* plan);

/*
 * Copy the plan's task list into the head of a device workspace
 * (cudaMemcpyAsync on stream).  The list starts with a header giving its
 * task, group and index counts.  pa_decode_attention checks those counts on
 * the device against the plan it is called with and sets
 * PA_DEV_PLAN_MISMATCH if they differ.  One upload serves any number of
 * decode calls that use the same plan and workspace.  A plan of the same
 * structure uploaded later (the next decode step's plan, for example) also
 * serves a call or a captured CUDA graph made with the earlier one.
 * The list ends with one counter per split group, zero in the plan.  A
 * decode call counts the finished splits of each group there and leaves
 * every counter at zero again; a call that set PA_DEV_PLAN_MISMATCH or
 * PA_DEV_TIMEOUT may not, so upload the plan again before the next call.
 * Returns PA_ERR_WORKSPACE if workspace_bytes < plan->workspace_bytes.
 */
pa_status_t pa_plan_upload(const pa_plan_t* plan, void* workspace, size_t workspace_bytes,
                           void* stream);

/*
 * Decode attention (the operation at the top of this header), computed with
 * an online softmax normaliser (xLLM introduction, SoftMax: online
 * normalizer).  Splits follow the plan; their (output, log-sum-exp) partials
 * go to the workspace, and the last split of each (sequence, KV head) to
 * finish merges them into out within the same kernel (swiftLLM paged
 * attention v2).  One kernel launch per call.  With a plan made with
 * merge = PA_MERGE_COMBINE_KERNEL (pa_plan_ex) the partials are instead
 * merged by a separate combine kernel launched after the split kernel on the
 * same stream (two launches when a sequence is split).  The two forms agree
 * to rounding; each gives the same bits on every call.
 *
 * Device: q, k_pages, v_pages, block_table, seq_lens, out [B][Hq][D] fp16,
 * workspace (holding the uploaded plan), dev_status.
 * A workspace serves one call at a time: the call writes its split partials
 * and group counters there, so calls in flight at once (on two streams, say)
 * each need their own workspace.
 * scale: the logit scale, normally 1/sqrt(head_dim).
 * out receives fp16 rounded to nearest even from the fp32 result.  A
 * sequence of length 0 gets zeros.
 * Returns PA_ERR_PLAN if plan->shape differs from *shape in batch, heads,
 * head_dim, page_size or max_pages_per_seq (the fields the task list depends
 * on) or a field a planner sets is out of range (task and CTA counts, merge,
 * l2_prefetch_pages, q8_stages, early_kv), and PA_ERR_WORKSPACE if workspace_bytes <
 * plan->workspace_bytes.
 */
pa_status_t pa_decode_attention(const pa_shape_t* shape, const pa_plan_t* plan, const void* q,
                                const void* k_pages, const void* v_pages,
                                const int32_t* block_table, const int32_t* seq_lens, float scale,
                                void* out, void* workspace, size_t workspace_bytes,
                                int32_t* dev_status, void* stream);

/*
 * pa_kv_append and pa_decode_attention in one launch: the decode step of
 * one layer.  The results are those of the two calls in sequence.  The new
 * token's K/V rows (k_new, v_new: device [B][Hkv][D] fp16) are written
 * bit for bit at position seq_lens[b] - 1 of the pools, and attention runs
 * over all seq_lens[b] tokens, the new one included.
 *
 * The task that owns the page of position L-1 patches that row of the tiles
 * it has staged, then writes the row to the pool after its own reads of the
 * page are done.  The separate append kernel, its launch and its dependent
 * load chain are saved.  Arguments and errors are those of the two calls;
 * k_pages/v_pages are written.
 */
pa_status_t pa_append_decode_attention(const pa_shape_t* shape, const pa_plan_t* plan,
                                       const void* q, const void* k_new, const void* v_new,
                                       void* k_pages, void* v_pages, const int32_t* block_table,
                                       const int32_t* seq_lens, float scale, void* out,
                                       void* workspace, size_t workspace_bytes,
                                       int32_t* dev_status, void* stream);

/* ---- INT8 KV cache ---------------------------------------------------
 *
 * The same paged cache held as INT8 codes with one fp32 scale per row
 * (MonadKai/xLLM, introduction: KV-cache quantisation, per-row INT8).  A row
 * is one token's D-vector of one KV head, and its value is code * scale.
 *
 * Layout (device):
 *   k_codes, v_codes: [num_pages][Hkv][16][D] int8 (a row is D bytes, a
 *                     (page, head) tile is 16 * D contiguous bytes)
 *   k_scales, v_scales: [num_pages][Hkv][16] fp32 (16-byte aligned)
 * A decode reads D + 4 bytes per row and tensor where the fp16 cache reads
 * 2 D.  The plan, workspace, q, out, block table, seq_lens and status are
 * those of the fp16 calls, and one plan serves both caches.
 *
 * Quantisation of a new row (append): scale = max|x| / 127 and
 * code = x / scale rounded to nearest, ties to even, clamped to
 * [-127, 127], both divisions in IEEE fp32 round-to-nearest; an all-zero
 * row gets scale 0 and zero codes.  Non-finite inputs give unspecified codes.
 *
 * Errors are those of the fp16 calls.  Scale pointers that are null or not
 * 16-byte aligned give PA_ERR_INVALID_ARG.
 */

/* pa_kv_append into the INT8 cache: quantise k_new/v_new ([B][Hkv][D] fp16)
 * and write codes and scales at position seq_lens[b] - 1. */
pa_status_t pa_kv_append_q8(const pa_shape_t* shape, const void* k_new, const void* v_new,
                            void* k_codes, void* v_codes, float* k_scales, float* v_scales,
                            const int32_t* block_table, const int32_t* seq_lens,
                            int32_t* dev_status, void* stream);

/* pa_decode_attention over the INT8 cache: attention over the dequantised
 * rows, fp32 accumulation, fp16 output. */
pa_status_t pa_decode_attention_q8(const pa_shape_t* shape, const pa_plan_t* plan, const void* q,
                                   const void* k_codes, const void* v_codes,
                                   const float* k_scales, const float* v_scales,
                                   const int32_t* block_table, const int32_t* seq_lens,
                                   float scale, void* out, void* workspace, size_t workspace_bytes,
                                   int32_t* dev_status, void* stream);

/* pa_kv_append_q8 and pa_decode_attention_q8 in one launch, with the same
 * results as the two calls in sequence. */
pa_status_t pa_append_decode_attention_q8(const pa_shape_t* shape, const pa_plan_t* plan,
                                          const void* q, const void* k_new, const void* v_new,
                                          void* k_codes, void* v_codes, float* k_scales,
                                          float* v_scales, const int32_t* block_table,
                                          const int32_t* seq_lens, float scale, void* out,
                                          void* workspace, size_t workspace_bytes,
                                          int32_t* dev_status, void* stream);

/* ---- FP8 (E4M3) KV cache ---------------------------------------------
 *
 * The same paged cache held as FP8 bytes with one fp32 scale per row
 * ("Eine LLM-Inferenz-Engine von Grund auf mit C++ und CUDA bauen", section 4:
 * FP8 quantisation of the cache; MonadKai/xLLM, introduction: KV-cache
 * quantisation).  The byte format is E4M3 of the OCP 8-bit floating-point
 * specification: sign, 4 exponent bits with bias 7, 3 mantissa bits,
 * subnormals m/8 * 2^-6, no infinities, S.1111.111 NaN, largest finite 448.
 * A row's value is value(code) * scale.
 *
 * Layout (device): as the INT8 cache, with k_codes, v_codes holding E4M3
 * bytes: [num_pages][Hkv][16][D] uint8 and [num_pages][Hkv][16] fp32 scales
 * (16-byte aligned).  The plan, workspace and the other buffers are those of
 * the fp16 calls.
 *
 * Quantisation of a new row (append): scale = max|x| / 448 and code = the
 * E4M3 value nearest x / scale, ties to the even mantissa, magnitudes above
 * 448 saturated, the sign of a zero kept; both divisions in IEEE fp32
 * round-to-nearest; an all-zero row gets scale 0 and zero codes.  Non-finite
 * inputs give unspecified codes.  A decode never uses the bytes of rows past
 * a sequence's end, so those may hold anything (NaN patterns too).
 *
 * Errors are those of the INT8 calls.
 */

/* pa_kv_append into the FP8 cache: quantise k_new/v_new ([B][Hkv][D] fp16)
 * and write codes and scales at position seq_lens[b] - 1. */
pa_status_t pa_kv_append_fp8(const pa_shape_t* shape, const void* k_new, const void* v_new,
                             void* k_codes, void* v_codes, float* k_scales, float* v_scales,
                             const int32_t* block_table, const int32_t* seq_lens,
                             int32_t* dev_status, void* stream);

/* pa_decode_attention over the FP8 cache: attention over the dequantised
 * rows, fp32 accumulation, fp16 output. */
pa_status_t pa_decode_attention_fp8(const pa_shape_t* shape, const pa_plan_t* plan, const void* q,
                                    const void* k_codes, const void* v_codes,
                                    const float* k_scales, const float* v_scales,
                                    const int32_t* block_table, const int32_t* seq_lens,
                                    float scale, void* out, void* workspace,
                                    size_t workspace_bytes, int32_t* dev_status, void* stream);

/* pa_kv_append_fp8 and pa_decode_attention_fp8 in one launch, with the same
 * results as the two calls in sequence. */
pa_status_t pa_append_decode_attention_fp8(const pa_shape_t* shape, const pa_plan_t* plan,
                                           const void* q, const void* k_new, const void* v_new,
                                           void* k_codes, void* v_codes, float* k_scales,
                                           float* v_scales, const int32_t* block_table,
                                           const int32_t* seq_lens, float scale, void* out,
                                           void* workspace, size_t workspace_bytes,
                                           int32_t* dev_status, void* stream);

/* Size of the library-owned scratch array used by pa_decode_attention_static. */
#define PA_STATIC_WORKSPACE_BYTES ((size_t)16 << 20)

/*
 * pa_decode_attention without a caller workspace: an entry point that
 * allocates nothing.  It has no counterpart in the pages; it exists for
 * callers that cannot allocate device memory.  Examples are code embedded in
 * another runtime that receives only its input and output buffers and must
 * not call cudaMalloc (the host runtime owns all device memory and its
 * accounting), and latency-critical loops where a cudaMalloc could stall on
 * device synchronisation.
 *
 * Same arguments, checks and result as pa_decode_attention, minus the
 * workspace.  The task list and the split partials live in one file-scope
 * __device__ array of PA_STATIC_WORKSPACE_BYTES (16 MiB).  Every GPU that
 * loads the library holds the array until the process exits.  Each call
 * uploads the plan's task list into it (host_blob must still be valid), then
 * launches the same kernels.  No cudaMalloc, cudaFree or allocating library
 * routine is called.
 *  - Each call looks up the array's device address on the current device
 *    (cudaGetSymbolAddress), so a context rebuilt after cudaDeviceReset is
 *    found anew.  The first call on a device may load the library's device
 *    code there: make that first call before any stream capture.
 *  - Every argument check of pa_decode_attention runs before anything is
 *    queued; a rejected call (a plan whose workspace_bytes exceeds
 *    PA_STATIC_WORKSPACE_BYTES gives PA_ERR_WORKSPACE) leaves the array as
 *    it was.
 *  - All calls on a device share the array, which keeps the previous call's
 *    contents.  What must start at zero (the split groups' counters) comes
 *    zeroed in each call's upload.  Calls that overlap on the GPU (other
 *    streams, other host threads) race on it: serialise them.
 */
pa_status_t pa_decode_attention_static(const pa_shape_t* shape, const pa_plan_t* plan,
                                       const void* q, const void* k_pages, const void* v_pages,
                                       const int32_t* block_table, const int32_t* seq_lens,
                                       float scale, void* out, int32_t* dev_status, void* stream);

/* ---- Several query tokens per sequence (chunked prefill, piggybacked
 * prefill and decode) ------------------------------------------------------
 *
 * The from-scratch engine article (section 4) names processing several
 * prompt tokens at once with a FlashAttention-style fused kernel as the next
 * step after decode; swiftLLM's feature list has piggybacked prefill and
 * decode and Flash Attention over PagedAttention.
 *
 * Sequence b has L = seq_lens[b] cached tokens, the newest q_lens[b] of
 * which are this step's queries: query i sits at position
 * L - q_lens[b] + i and attends positions 0 .. that position (causal):
 *   out[r][h] = softmax(scale * K[0..p] q[r][h]) V[0..p],  p = L - q_lens[b] + i.
 * q, out: device [T][Hq][D], and k_new, v_new: [T][Hkv][D], packed by
 * sequence (row r = cu[b] + i, cu = prefix sums of q_lens, T = cu[B]), in
 * the shape's dtype.  A decode token is q_lens[b] = 1.
 */
typedef struct {
  pa_shape_t shape;     /* the shape the plan was made for */
  int32_t num_tiles;    /* CTAs: rows_per_tile query rows (tokens x heads of one KV head) each */
  int32_t total_q;      /* T */
  int32_t owns_blob;    /* 1: host_blob is released by pa_prefill_plan_free */
  int32_t rows_per_tile; /* 128: the tcgen05 kernel; 64: the mma.sync kernel */
  uint64_t plan_id;
  size_t blob_bytes;    /* bytes pa_prefill_plan_upload copies */
  size_t workspace_bytes;
  void* host_blob;
  uint64_t wait_limit_ns; /* bound of each wait in the kernel (see pa_prefill_options_t) */
} pa_prefill_plan_t;

/* Options of a multi-token plan; a zeroed struct or NULL gives the
 * defaults. */
typedef struct {
  int32_t rows_per_tile;  /* 0 or 128: the tcgen05 kernel (TMEM accumulators, 128 rows per
                             CTA); 64: the mma.sync kernel (64 rows per CTA) */
  int32_t reserved;       /* 0 */
  uint64_t wait_limit_ns; /* how long a warp waits on one barrier (a copy, an MMA, another
                             warp) before it gives up, sets PA_DEV_TIMEOUT and leaves its
                             rows unwritten (0: 1 s).  Copies and MMAs that were issued
                             finish before the kernel exits. */
} pa_prefill_options_t;

/* Host: the tile list (longest work first) and the row offsets cu.
 * q_lens_host[b] must satisfy 0 <= q_lens[b] <= seq_lens[b]. */
pa_status_t pa_prefill_plan(const pa_shape_t* shape, const int32_t* seq_lens_host,
                            const int32_t* q_lens_host, pa_prefill_plan_t* plan_out);

/* pa_prefill_plan with options (NULL: the defaults).  rows_per_tile other
 * than 0, 64 or 128 returns PA_ERR_INVALID_ARG. */
pa_status_t pa_prefill_plan_ex(const pa_shape_t* shape, const int32_t* seq_lens_host,
                               const int32_t* q_lens_host, const pa_prefill_options_t* options,
                               pa_prefill_plan_t* plan_out);
void pa_prefill_plan_free(pa_prefill_plan_t* plan);
pa_status_t pa_prefill_plan_upload(const pa_prefill_plan_t* plan, void* workspace,
                                   size_t workspace_bytes, void* stream);

/* Write the T new rows: row cu[b] + i of k_new/v_new goes to position
 * seq_lens[b] - q_lens[b] + i of sequence b, bit for bit.  Needs the plan in
 * the workspace (for cu). */
pa_status_t pa_kv_append_tokens(const pa_shape_t* shape, const pa_prefill_plan_t* plan,
                                const void* k_new, const void* v_new, void* k_pages,
                                void* v_pages, const int32_t* block_table,
                                const int32_t* seq_lens, const void* workspace,
                                size_t workspace_bytes, int32_t* dev_status, void* stream);

/* The attention above, for every query row of the plan, on tensor cores
 * (FlashAttention-style: one CTA per tile of query rows of one KV head
 * streams the causal part of the sequence's pages once; tcgen05 MMAs into
 * tensor memory, or mma.sync when the plan was cut for it).  Errors as
 * pa_decode_attention's; device seq_lens shorter than the plan's q_lens
 * set PA_DEV_PLAN_MISMATCH. */
pa_status_t pa_prefill_attention(const pa_shape_t* shape, const pa_prefill_plan_t* plan,
                                 const void* q, const void* k_pages, const void* v_pages,
                                 const int32_t* block_table, const int32_t* seq_lens, float scale,
                                 void* out, void* workspace, size_t workspace_bytes,
                                 int32_t* dev_status, void* stream);

/* ---- KV blocks: how many, which are free, and moving them ------------
 *
 * swiftLLM's engine (architecture section) profiles the number of GPU
 * blocks, allocates the KV cache and a KV swap space, and swaps blocks in
 * and out before each step's compute.  A block is one page: 16 tokens of
 * every KV head of a pool.
 */

#define PA_KV_16BIT 0 /* fp16 or bf16 pools */
#define PA_KV_INT8 1  /* INT8 code pools plus fp32 row scales */
#define PA_KV_FP8 2   /* E4M3 code pools plus fp32 row scales */

/* Pages of num_layers layers' K and V pools (kv_kind: PA_KV_16BIT,
 * PA_KV_INT8 or PA_KV_FP8) that fit in free_bytes - reserve_bytes:
 *   floor((free - reserve) / (2 * Hkv * page_size * row_bytes * num_layers)),
 * row_bytes = 2 * head_dim (16-bit) or head_dim + 4 (8-bit codes + scale).
 * Host only.  Returns 0 when free <= reserve and -1 on a bad argument. */
int64_t pa_profile_num_blocks(const pa_shape_t* shape, int32_t num_layers, int32_t kv_kind,
                              size_t free_bytes, size_t reserve_bytes);

/* Free list of num_blocks pages (host, thread-safe).  Pages come out of a
 * LIFO stack: a fresh allocator hands out 0, 1, 2, ...; a freed page is the
 * next one handed out. */
typedef struct pa_block_allocator pa_block_allocator_t;
pa_status_t pa_block_allocator_create(int32_t num_blocks, pa_block_allocator_t** out);
void pa_block_allocator_destroy(pa_block_allocator_t* allocator);
int32_t pa_block_num_free(pa_block_allocator_t* allocator);  /* -1 for a null allocator */

/* Take n pages into blocks_out[0..n), all or nothing: PA_ERR_NO_MEMORY when
 * fewer than n are free (nothing taken). */
pa_status_t pa_block_alloc(pa_block_allocator_t* allocator, int32_t n, int32_t* blocks_out);

/* Return n pages.  A page out of range, not handed out, or listed twice
 * gives PA_ERR_INVALID_ARG, and then nothing is freed. */
pa_status_t pa_block_free(pa_block_allocator_t* allocator, const int32_t* blocks, int32_t n);

/* Grow one sequence's block-table row (host, max_pages entries) from old_len
 * to new_len tokens: entries [ceil(old_len/S), ceil(new_len/S)) get fresh
 * pages, S = page_size.  PA_ERR_NO_MEMORY (nothing taken) when the pool is
 * short; PA_ERR_INVALID_ARG when new_len < old_len or the row is too short. */
pa_status_t pa_block_table_grow(pa_block_allocator_t* allocator, int32_t* row, int32_t max_pages,
                                int32_t page_size, int32_t old_len, int32_t new_len);

/* Copy whole blocks between two pools of blocks of block_bytes bytes each:
 * for i < n, block pairs[2i+1] of dst_pool becomes block pairs[2i] of
 * src_pool, byte for byte.  One kernel moves them all.  Either pool may be
 * device memory or page-locked host memory mapped into the device's address
 * space (cudaHostAlloc), so one call is a swap-in (host to device), a
 * swap-out (device to host) or a block copy within the GPU.
 *
 * pairs: device (or mapped) int32 [n][2] = (src block, dst block), 8-byte
 * aligned.  Pools 16-byte aligned; block_bytes a positive multiple of 16
 * (a 16-bit pool's block is Hkv * 16 * D * 2 bytes; an INT8 or E4M3 code
 * pool's Hkv * 16 * D; a scale pool's Hkv * 16 * 4).  No block may be both read
 * and written by one call, and destinations must be distinct.  A pair with
 * an index outside [0, src_blocks) or [0, dst_blocks) is skipped and sets
 * PA_DEV_BAD_PAGE in *dev_status.  n = 0 launches nothing. */
pa_status_t pa_copy_blocks(void* dst_pool, int32_t dst_blocks, const void* src_pool,
                           int32_t src_blocks, size_t block_bytes, const int32_t* pairs,
                           int32_t n, int32_t* dev_status, void* stream);

/*
 * Export the physical slot of every logical token, for exact comparison
 * with the oracle: out_slots[b][t] = block_table[b][t/S]*S + t%S for
 * t < seq_lens[b], else -1.  A bad page index gives -2 and sets
 * PA_DEV_BAD_PAGE.  Device: block_table, seq_lens,
 * out_slots int32 [batch][max_pages_per_seq * page_size].
 */
pa_status_t pa_debug_gather_indices(const pa_shape_t* shape, const int32_t* block_table,
                                    const int32_t* seq_lens, int32_t* out_slots,
                                    int32_t* dev_status, void* stream);

/* Static description of a status code. */
const char* pa_status_string(pa_status_t status);

/* Library version string. */
const char* pa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_H */
