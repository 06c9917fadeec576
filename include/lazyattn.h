/*
 * lazyattn.h - C ABI of a GB300 (sm_103a) implementation of LazyAttention's
 * hot path: attention over a paged KV pool whose keys are stored WITHOUT rotary
 * position encoding; RoPE is applied inside the prefill and decode kernels at
 * each request's logical positions.
 *
 * Source: "LazyAttention: Efficient Retrieval-Augmented Generation with
 * Deferred Positional Encoding".
 *   - §3 "Problem statement": reuse a document's KV at any global offset, with
 *     several requests of one batch reading one document at different offsets.
 *   - §3.1 "Deferred encoding": Q, K, V are produced without positions; the cache
 *     is content-only; positions are applied during attention.
 *   - §3.1 Eq. 4: softmax(f(Q,m) f(K,n)^T / sqrt(d_k)) V, d_k = head_dim.
 *   - §3.2 "Prefilling": rotation of the half-dimension pair (k[i], k[i+D/2]) by
 *     angle a: k1' = k1 cos a - k2 sin a, k2' = k1 sin a + k2 cos a; cos/sin are
 *     table-driven.
 *   - §3.2 "Decoding": bit-packed 64-bit per-block metadata (block, offset, mask).
 *   - §3.5 "GQA/MQA compatibility": query head h reads KV head h / (Hq/Hkv).
 *   - Appendix C.4: angles from absolute indices m * theta_i.
 *
 * Conventions for every entry point
 *   - Every device buffer (pools, position table, q/k/v/out, tables, workspace,
 *     status word) is allocated and owned by the caller. The library never calls
 *     cudaMalloc/cudaFree; it owns only host-side metadata (free-page list).
 *   - Calls taking a stream enqueue work on it and return without synchronising,
 *     except lazyattn_pool_create and lazyattn_get_device_status (documented).
 *   - Argument errors are detected on the host, return a negative status and
 *     launch nothing. Index errors found on the device (page id out of range,
 *     position outside the table, no free decode slot) skip the offending work
 *     and record the first error code in the caller's device status word; they
 *     never trap or hang.
 *   - Not thread-safe per pool: serialise calls that share a pool handle.
 *   - Entry points that launch work (store_doc, prefill, decode, materialize,
 *     resolve, decode_noalloc) need the pool's device to be the current one and
 *     return LAZYATTN_EINVAL, launching nothing, when it is not.
 *
 * Input range (bf16 pools)
 *   The bf16 kernels multiply rotated keys and the rotated, scaled query as
 *   fp16 operands (fp32 accumulation). A rotation keeps the norm of every
 *   rotate-half pair (x_i, x_{i+D/2}), so the library accepts any input whose
 *   pairs satisfy
 *       keys  : sqrt(k_i^2 + k_{i+D/2}^2)                          <= 65024
 *       query : sqrt(q_i^2 + q_{i+D/2}^2) * logit_scale * log2(e)  <= 65024
 *   (logit_scale = 1/sqrt(head_dim), times YaRN's temperature; for head_dim
 *   128 the query bound is a pair norm of about 509,900). Such pairs stay
 *   below fp16's maximum (65504) at any angle and through every bf16 rounding
 *   on the way (materialised or document-local keys). The check runs in fp32 where the values
 *   enter: keys in lazyattn_store_doc and in the decode append, queries in
 *   lazyattn_prefill and lazyattn_decode; a pair outside the range (or a NaN)
 *   records LAZYATTN_ERANGE in the status word, and the outputs that depend on
 *   it are undefined. V is not checked; its components must stay below 2^90 in
 *   magnitude for the fp32 accumulators (sums of up to 2^26 keys with weights
 *   up to 2^8). fp32 pools compute in fp32 and have no such bound.
 *   The kernels read whole pages and give the empty slots of a page (past its
 *   entry's valid count) zero weight, so those slots must hold finite values:
 *   lazyattn_store_doc and lazyattn_materialize zero them, and the decode
 *   append zeroes a page's other slots when it writes the page's first token;
 *   pages filled by the caller directly must keep them finite too. Pages whose
 *   entry has no valid slot are not read.
 *
 * Data layout in device memory (row-major, innermost last)
 *   K pool, V pool : [num_pages][n_kv_heads][16][head_dim], element type dtype,
 *                    pre-RoPE. A (page, kv-head) tile is contiguous.
 *   position table : float2 [max_position][head_dim/2] = (cos, sin) of
 *                    pos * theta^(-2i/head_dim), computed in fp64, stored fp32.
 *   block table    : uint64 entries, see lazyattn_pack_entry.
 */
#ifndef LAZYATTN_H
#define LAZYATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LAZYATTN_PAGE_SIZE 16
#define LAZYATTN_MAX_START ((1 << 26) - 1)

typedef enum lazyattn_status {
    LAZYATTN_OK = 0,
    LAZYATTN_EINVAL = -1,     /* bad argument: null pointer, inconsistent or unsupported size */
    LAZYATTN_ENOSPC = -2,     /* not enough free pages in the pool */
    LAZYATTN_ERANGE = -3,     /* page id or logical position outside the pool / table */
    LAZYATTN_EDTYPE = -4,     /* dtype not supported by this entry point */
    LAZYATTN_ECUDA = -5,      /* a CUDA runtime call or kernel launch failed */
    LAZYATTN_EDEVICE = -6,    /* device-side check failed (see lazyattn_get_device_status) */
    LAZYATTN_EWORKSPACE = -7, /* workspace smaller than lazyattn_workspace_size() */
    LAZYATTN_ENODECODE = -8   /* device status only: a request had no writable free slot */
} lazyattn_status;

typedef enum lazyattn_dtype { LAZYATTN_F32 = 0, LAZYATTN_BF16 = 1 } lazyattn_dtype;

/* batch flags */
#define LAZYATTN_KEYS_PREROTATED 1  /* K pages already hold RoPE at their logical positions
                                       (the materialising baseline); kernels rotate q only */

/* Pool description. All pointers are device pointers owned by the caller.
 *   num_pages     pages in each of k_pool / v_pool (>= 1)
 *   page_size     must be LAZYATTN_PAGE_SIZE (16)
 *   n_q_heads     Hq; n_kv_heads Hkv; Hq % Hkv == 0; for LAZYATTN_BF16 also Hq / Hkv <= 8
 *                 (decode packs the query heads of one KV head into one 8-wide MMA tile)
 *   head_dim      D: 64 or 128 for LAZYATTN_F32; 128 for LAZYATTN_BF16
 *   dtype         element type of the pools, q, k_new, v_new and out
 *   rope_theta    RoPE base (> 0), frequencies theta^(-2i/D), i < D/2
 *   max_position  the position table covers logical positions [0, max_position)
 *   k_pool/v_pool [num_pages][n_kv_heads][16][head_dim]
 *   rope_table    lazyattn_rope_table_bytes(head_dim, max_position) bytes, filled by
 *                 lazyattn_pool_create: float2 [max_position][head_dim/2] (cos, sin) of
 *                 each frequency, then the same values as float4 [max_position][head_dim/4]
 *                 (cos f, cos f+1, sin f, sin f+1) for even f (the per-page rows the
 *                 bf16 kernels stage in shared memory, paired for two-lane arithmetic)
 *   status_word   one int32 in device memory, zeroed by lazyattn_pool_create; kernels
 *                 record the first device-side error there
 *   rope_scaling  LAZYATTN_ROPE_* below (0: plain RoPE; the fields after it are then ignored)
 *   rope_original_max_position   context length the model was trained for (YaRN, Llama 3.1)
 *   rope_factor   scale factor s >= 1 (all scaled kinds)
 *   rope_low, rope_high          YaRN: beta_slow, beta_fast (rotations within the original
 *                 context below which frequencies are interpolated / above which they are
 *                 kept); Llama 3.1: low_freq_factor, high_freq_factor. rope_low < rope_high.
 *   key_storage   LAZYATTN_KEYS_POSITION_FREE (0): K is stored with no position and rotated
 *                 in the kernels at each key's logical position. LAZYATTN_KEYS_DOC_LOCAL
 *                 (bf16 pools only): the paper's own layout (§3.2): lazyattn_store_doc
 *                 stores K rotated at document-local positions (token i of the call at i),
 *                 prefill applies one relative rotation by the document's offset, decode
 *                 rotates q instead of the keys; batches must then carry entry_delta.
 *   rope_interleaved  0: rotate-half pairs (i, i + D/2); 1 (bf16 pools only): interleaved pairs
 *                 (2i, 2i+1) with the same frequencies, as in the original RoPE / Llama layout.
 *                 q and k are then given and stored in their natural order; the library
 *                 de-interleaves them where they enter (store, append, q loads): a score is a
 *                 dot product over the head dimension, so one permutation applied to both q
 *                 and k leaves it unchanged, and v is never permuted.
 *   position_encoding  LAZYATTN_POS_ROPE (0) or LAZYATTN_POS_ALIBI (bf16 pools; §3.5 "Score-space
 *                 positional methods"): no rotation at all; every score q.k / sqrt(D) gets the
 *                 bias -slope_h * (m - n) for query head h at position m and key position n,
 *                 with the ALiBi slopes of Hq heads (2^(-8 (h+1) / Hq) for a power of two;
 *                 otherwise those of the power of two below Hq, then every other slope of
 *                 twice that). Requires plain RoPE fields, position-free keys, no interleaving.
 * A zero-initialised descriptor tail means plain RoPE and position-free keys.
 */
typedef struct lazyattn_pool_desc {
    int32_t num_pages;
    int32_t page_size;
    int32_t n_q_heads;
    int32_t n_kv_heads;
    int32_t head_dim;
    int32_t dtype;
    double rope_theta;
    int32_t max_position;
    void* k_pool;
    void* v_pool;
    void* rope_table;
    int32_t* status_word;
    int32_t rope_scaling;
    int32_t rope_original_max_position;
    double rope_factor;
    double rope_low;
    double rope_high;
    int32_t key_storage;
    int32_t rope_interleaved;
    int32_t position_encoding;
} lazyattn_pool_desc;

#define LAZYATTN_POS_ROPE 0
#define LAZYATTN_POS_ALIBI 1

#define LAZYATTN_KEYS_POSITION_FREE 0
#define LAZYATTN_KEYS_DOC_LOCAL 1

/* RoPE-family variants (§3.5 "Generalization Beyond Standard RoPE": scaled/NTK
 * variants and YaRN keep the score q^T R_{n-m} k, with variant-specific scaling
 * metadata). Each changes only the frequencies theta_i of the position table,
 * plus, for YaRN, an attention temperature on the logits:
 *   LINEAR  position interpolation: theta_i / s
 *   NTK     NTK-aware base change: base' = base * s^(D/(D-2))
 *   YARN    per-frequency ramp between theta_i / s and theta_i by the number r_i
 *           of rotations within the original context (interpolated for r < low,
 *           kept for r > high, linear in between); logits times (0.1 ln s + 1)^2
 *   LLAMA3  the Llama 3.1 rule: wavelength 2 pi / theta_i below orig/high kept,
 *           above orig/low divided by s, smooth blend in between */
#define LAZYATTN_ROPE_DEFAULT 0
#define LAZYATTN_ROPE_LINEAR 1
#define LAZYATTN_ROPE_NTK 2
#define LAZYATTN_ROPE_YARN 3
#define LAZYATTN_ROPE_LLAMA3 4

typedef struct lazyattn_pool* lazyattn_pool_t;
typedef struct lazyattn_plan* lazyattn_plan_t;

/* A batch of requests. Device arrays unless stated otherwise.
 *   num_requests   1 <= R <= 65535 (host value; requests index a grid dimension)
 *   max_entries    host upper bound on entries per request (grid sizing)
 *   max_q_len      prefill: host upper bound on query tokens per request; decode: unused
 *   total_q        prefill: number of rows of q / out (host value); decode: unused
 *   entries        packed entries of all requests back to back; lazyattn_decode
 *                  updates the entry it appends into, so this must be writable
 *   entry_offsets  int32 [R+1]: request r owns entries [entry_offsets[r], entry_offsets[r+1])
 *   q_offsets      prefill: int32 [R+1], request r owns rows [q_offsets[r], q_offsets[r+1]) of q/out
 *   q_start        prefill: int32 [R], logical position of request r's first query row;
 *                  row i of the request sits at q_start[r] + i
 *   flags          0 or LAZYATTN_KEYS_PREROTATED (not with doc-local pools)
 *   entry_delta    doc-local pools only (else ignored, may be NULL): int32 per entry, the
 *                  logical position of local position 0 of the entry's document, so the
 *                  entry's slot j sits at logical start + j and local start - delta + j;
 *                  0 <= delta <= start. Decode-appended tokens take the local position of
 *                  their slot in the entry they go into.
 *   decode_plan    lazyattn_decode only (else ignored; may be NULL): a plan built by
 *                  lazyattn_decode_plan_create from this batch's table and uploaded with
 *                  lazyattn_decode_plan_upload. With a plan, decode reads each page run that
 *                  several requests share once per group of requests (see there); without
 *                  one, every request reads its own pages.
 */
typedef struct lazyattn_batch {
    int32_t num_requests;
    int32_t max_entries;
    int32_t max_q_len;
    int32_t total_q;
    uint64_t* entries;
    const int32_t* entry_offsets;
    const int32_t* q_offsets;
    const int32_t* q_start;
    int32_t flags;
    const int32_t* entry_delta;
    lazyattn_plan_t decode_plan;
} lazyattn_batch;

#define LAZYATTN_OP_PREFILL 0
#define LAZYATTN_OP_DECODE 1

/* Human-readable name of a status code. Never NULL. */
const char* lazyattn_status_string(int status);

/* Pack one block-table entry (§3.2 "Decoding": block id, offset and mask in one
 * 64-bit word). Field layout:
 *   bits  0..31  physical page id
 *   bits 32..57  logical position of slot 0 of the page (<= LAZYATTN_MAX_START)
 *   bits 58..62  number of valid slots, 0..16 (slots [0, nvalid) hold tokens)
 *   bit  63      writable: lazyattn_decode may append into this page
 * Token at slot s of the page has logical position start + s. Out-of-range
 * fields are masked to their width (host helper; no validation). */
uint64_t lazyattn_pack_entry(int32_t page, int32_t start, int32_t nvalid, int32_t writable);

/* Bytes of the position table for head_dim and max_position (host helper):
 * both layouts described under lazyattn_pool_desc.rope_table. */
size_t lazyattn_rope_table_bytes(int32_t head_dim, int32_t max_position);

/* Create a pool over caller-owned buffers (§3 "Problem statement": one store of
 * documents whose KV is reused at any global offset; §3.1 "Deferred encoding":
 * the cache holds content only, positions come from the table filled here, as
 * §3.2 "Prefilling" table-drives cos/sin). Validates desc, fills the position
 * table (fp64 on the host, stored fp32) and zeroes the status word on `stream`,
 * then synchronises that stream before returning. All pages start free.
 * Returns LAZYATTN_OK and *out_pool, or EINVAL/EDTYPE/ECUDA, or ENOSPC when the host
 * memory for the pool's metadata or the position table cannot be had (nothing created). */
int lazyattn_pool_create(const lazyattn_pool_desc* desc, void* stream, lazyattn_pool_t* out_pool);

/* Release the host metadata of a pool (device buffers stay with the caller). */
int lazyattn_pool_destroy(lazyattn_pool_t pool);

/* Number of free pages (host). */
int lazyattn_pool_free_count(lazyattn_pool_t pool, int32_t* out_count);

/* (§3.2 "Decoding": a request's KV grows by one token per step into pages of
 * its own, while the shared document pages stay read-only.)
 * Take n free pages (lowest ids first) for caller-managed contents, e.g. the
 * private pages a request reserves for generated tokens. out_pages: host array
 * of n ids. ENOSPC (nothing taken) if fewer than n are free. */
int lazyattn_alloc_pages(lazyattn_pool_t pool, int32_t n, int32_t* out_pages);

/* Return pages to the free list. ERANGE for an id outside the pool, EINVAL for
 * a page that is already free (nothing freed in either case). The caller must
 * not free pages that queued kernels still read. */
int lazyattn_free_pages(lazyattn_pool_t pool, const int32_t* pages, int32_t n);

/* Store a document's (or a query segment's) pre-RoPE K/V in fresh pages
 * (§3.2: a document's KV is computed once, indexed from position 0, and reused
 * by every request; §4.3 phase 1, documents are prefilled independently and
 * cached without positions; §3.1 "Deferred encoding").
 * k, v: device [n_tokens][n_kv_heads][head_dim] in the pool dtype, unrotated.
 * Allocates ceil(n_tokens/16) pages, enqueues the copy on `stream`, writes the
 * page ids (in token order) to the host array out_pages (capacity out_cap) and
 * their number to *out_npages. Page j holds tokens [16j, 16j+16); the caller
 * builds entries (page_j, doc_start + 16j, nvalid_j, writable) from them.
 * EINVAL if n_tokens < 1 or out_cap too small; ENOSPC if the pool is full. */
int lazyattn_store_doc(lazyattn_pool_t pool, const void* k, const void* v, int32_t n_tokens,
                       void* stream, int32_t* out_pages, int32_t out_cap, int32_t* out_npages);

/* Bytes of workspace that lazyattn_prefill (op = LAZYATTN_OP_PREFILL) or
 * lazyattn_decode (op = LAZYATTN_OP_DECODE) needs for this batch shape. The
 * workspace is caller-allocated device memory, 256-byte aligned, and must be
 * ZERO-FILLED before its first use; every completed call leaves the parts that
 * must start at zero back at zero. Calls sharing one workspace must not
 * overlap in time. Returns 0 on invalid arguments. */
size_t lazyattn_workspace_size(lazyattn_pool_t pool, int32_t op, const lazyattn_batch* batch);

/* Prefill attention (§3.2 "Prefilling"; §3.4 TTFT).
 * q   : device [total_q][n_q_heads][head_dim], pre-RoPE, pool dtype.
 * out : device [total_q][n_q_heads][head_dim], pool dtype, caller-allocated.
 * Row i of request r (logical position m = q_start[r] + i), head h, reads KV head
 * h / (Hq/Hkv) and attends over every token of the request's entries whose
 * logical position n <= m, with q rotated at m and each key rotated at its own n
 * (unless LAZYATTN_KEYS_PREROTATED), scale 1/sqrt(head_dim). The query
 * segment's own K/V must already be stored and listed in the entries. Entries
 * with nvalid = 0 contribute nothing. A row that sees no key gets zeros.
 * Pool pages are only read.
 * workspace (optional, device, 256-byte aligned, no zero-fill needed): with at
 * least lazyattn_workspace_size(pool, LAZYATTN_OP_PREFILL, batch) bytes, bf16
 * pools may split each (request, KV head, query pair)'s KV tiles over 2..4 CTAs
 * when the batch fills few waves of the GPU, and merge their partial outputs
 * (per row: reference maximum, sum, unnormalised O) in a second kernel on the
 * same stream; NULL or fewer bytes: one CTA per item. Both give results within
 * the same error bounds. */
int lazyattn_prefill(lazyattn_pool_t pool, const lazyattn_batch* batch, const void* q, void* out,
                     void* workspace, size_t workspace_bytes, void* stream);

/* One decode step for every request (§3.2 "Decoding"; §3.4 decoding latency).
 * q     : device [R][n_q_heads][head_dim], pre-RoPE.
 * k_new, v_new : device [R][n_kv_heads][head_dim], pre-RoPE K and V of the new token.
 * out   : device [R][n_q_heads][head_dim].
 * For request r the new token is appended into the first entry with nvalid < 16
 * within the trailing run of writable entries of the request; it lands in slot
 * nvalid of that page (logical position m = start + nvalid) and the entry's
 * nvalid is incremented in place. Then q (rotated at m) attends over all the
 * request's tokens, including the new one. With LAZYATTN_KEYS_PREROTATED the new
 * key is stored rotated at m. If a request has no writable free slot its output
 * is zeros and LAZYATTN_ENODECODE is recorded in the status word.
 * Only the appended slot of a writable page is written; other pages are read. */
int lazyattn_decode(lazyattn_pool_t pool, const lazyattn_batch* batch, const void* q,
                    const void* k_new, const void* v_new, void* out,
                    void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------- decode plan
 * Document-major decode (§3 "Problem statement": requests of one batch read one
 * document at different global offsets; Fact 3.2: q^T R_{n-m} k depends on
 * positions only through n - m). A plan groups the pages of a batch's tables
 * into runs: maximal stretches of consecutive page ids at consecutive logical
 * positions, cut wherever any request's run starts or ends, so that every
 * request that reads a run reads all of it, with the same token counts per
 * page. With the plan, lazyattn_decode gives each run one pass per KV head over
 * its pages for all the requests that read it (up to 128 query rows, i.e.
 * 128 / (Hq/Hkv) requests per pass): the keys are rotated once at run-local
 * positions t, each request's q at m - delta (delta = the request's logical
 * position of the run's t = 0), and q^T R_{(delta + t) - m} k is the score the
 * method defines. Each (request, run) pass leaves a partial softmax result that
 * a combine merges per request. A request's trailing run of writable entries
 * (its query segment and generated tokens) is its own run, read after the
 * append. Results equal lazyattn_decode without a plan up to rounding order.
 *
 * A plan stays valid while the batch's table changes only by lazyattn_decode's
 * appends; build a new one after any other change (entries, offsets, pages or
 * their contents' layout). entries / entry_offsets / entry_delta are HOST copies
 * of the batch's arrays (entry_delta: doc-local pools only, else NULL).
 * Host memory only; ENOSPC if it cannot be had; ERANGE / EINVAL for a table
 * lazyattn_check_batch_host rejects; EDTYPE for fp32 pools (their decode needs no
 * plan). */
typedef struct lazyattn_decode_plan_stats {
    int32_t units;           /* passes per KV head (CTAs per KV head) */
    int32_t runs;            /* distinct page runs */
    int32_t partials;        /* partial results per KV head */
    int32_t max_readers;     /* most (request, occurrence) pairs reading one run */
    int64_t logical_pages;   /* pages the requests' tables name (with repeats) */
    int64_t pass_pages;      /* pages the passes read (a run once per pass) */
} lazyattn_decode_plan_stats;

int lazyattn_decode_plan_create(lazyattn_pool_t pool, const uint64_t* entries, const int32_t* entry_offsets,
                                const int32_t* entry_delta, int32_t num_requests, lazyattn_plan_t* out_plan);

/* Bytes of device memory the plan's image needs (256-byte aligned buffer). */
size_t lazyattn_decode_plan_device_bytes(lazyattn_plan_t plan);

/* Copy the plan's image into caller-owned device memory (bytes >= the size
 * above, 256-byte aligned) on `stream` and remember it; the buffer must stay
 * valid while batches use the plan. The host image is staged by the runtime
 * before the call returns. Not for use inside stream capture. */
int lazyattn_decode_plan_upload(lazyattn_plan_t plan, void* device_buffer, size_t bytes, void* stream);

int lazyattn_decode_plan_get_stats(lazyattn_plan_t plan, lazyattn_decode_plan_stats* out);

/* Release the plan's host memory (its device image stays with the caller). */
int lazyattn_decode_plan_destroy(lazyattn_plan_t plan);

/* Materialising baseline (what re-encoding systems such as Block-Attention do,
 * §4 "Baselines" and Appendix B): for every entry of `batch`, copy page
 * src -> dst_entries[i].page, rotating K at the entry's logical positions (RoPE
 * applied eagerly and stored in the pool dtype) and copying V unchanged. Entry
 * i of dst_entries must carry the same start and nvalid as entry i of the batch
 * and a distinct page per entry (its own private copy). dst_entries is a device
 * array parallel to batch->entries. Run prefill/decode on the destination
 * entries with LAZYATTN_KEYS_PREROTATED afterwards. */
int lazyattn_materialize(lazyattn_pool_t pool, const lazyattn_batch* batch,
                         const uint64_t* dst_entries, void* stream);

/* Debug view of block-table decoding: for every valid token of every request,
 * in table order, write (page, slot, logical position) as three int32 to
 * out_triples (device, capacity out_cap triples). Tokens of request r start at
 * row out_offsets[r] (device int32 [R+1], exclusive prefix sum of valid-token
 * counts, computed by the caller). Used to check indexing bit-exactly. */
int lazyattn_resolve(lazyattn_pool_t pool, const lazyattn_batch* batch, const int32_t* out_offsets,
                     int32_t* out_triples, int32_t out_cap, void* stream);

/* Host-side check of a block table before it is uploaded (a debug aid: the
 * kernels only range-check entries, on the device, and skip what fails).
 * entries / entry_offsets: HOST copies of a batch's arrays (int32 [R+1] offsets).
 * For every request r, every entry with nvalid > 0 must name a page below
 * num_pages, hold at most 16 valid slots and end at or below max_position
 * (else LAZYATTN_ERANGE), and no two tokens of the request may share a logical
 * position (else LAZYATTN_EINVAL): the request's entries describe one logical
 * sequence, one token per position (§3.2). Entries may come in any order.
 * Returns LAZYATTN_OK, or the failure with *out_request (if not NULL) set to the
 * first failing request (-1 for malformed arguments: EINVAL). ENOSPC if host
 * memory for the check cannot be had. Needs no GPU. */
int lazyattn_check_batch_host(const uint64_t* entries, const int32_t* entry_offsets, int32_t num_requests,
                              int32_t num_pages, int32_t max_position, int32_t* out_request);

/* Copy the device status word to *out_status (synchronises `stream`), then
 * reset it to zero if reset != 0. 0 means no device-side error since the last
 * reset; otherwise a negative lazyattn_status. */
int lazyattn_get_device_status(lazyattn_pool_t pool, int32_t* out_status, int32_t reset, void* stream);

/* Decode step that allocates nothing (no counterpart in the paper).
 * For callers that cannot obtain device memory for lazyattn_decode's workspace:
 * code whose host owns every device allocation, allocator-less runtimes, or
 * contexts that must not grow after start-up. Same arguments, semantics and
 * results as lazyattn_decode, without the workspace: scratch comes from a
 * fixed array of LAZYATTN_NOALLOC_SCRATCH_BYTES inside the library (device
 * global memory; every GPU that loads the library holds one until the process
 * exits). The call makes no cudaMalloc/cudaFree and no allocating library call.
 *   - A decode plan in the batch is ignored: this entry point reads each
 *     request's pages itself (the plan's image would need device memory).
 *   - Returns LAZYATTN_EWORKSPACE, launching nothing, if the batch needs more
 *     scratch than that (lazyattn_workspace_size(pool, LAZYATTN_OP_DECODE, b)
 *     tells how much it needs).
 *   - The pool's device must be current. The first call on a device looks up
 *     the array's device address (cudaGetSymbolAddress) and keeps it for the
 *     life of the process; make that first call before any stream capture, and
 *     do not use this entry point on a device after cudaDeviceReset (the array
 *     may then sit elsewhere).
 *   - Every call shares the one array, which keeps the previous call's
 *     contents (the call clears what must start at zero). Calls that overlap
 *     on the GPU - on different streams, or from different threads - race on
 *     it: serialise them. */
#define LAZYATTN_NOALLOC_SCRATCH_BYTES (16u << 20)
int lazyattn_decode_noalloc(lazyattn_pool_t pool, const lazyattn_batch* batch, const void* q,
                            const void* k_new, const void* v_new, void* out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* LAZYATTN_H */
