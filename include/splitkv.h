/*
 * splitkv.h -- split-KV (flash-decoding) attention for the decode step over a
 * paged KV cache, for NVIDIA GB300 (sm_103a).
 *
 * What the library computes.  For every sequence b, query token t and query
 * head h (KV head h / G, G = num_q_heads / num_kv_heads), with L = seq_lens[b]
 * and the keys 0 .. L-T+t visible to token t:
 *
 *     s_j  = scale * sum_d q[b][t][h][d] * K_j[d]
 *     lse  = ln sum_j exp(s_j)                                  (fp32 output)
 *     out  = sum_j exp(s_j - lse) * V_j                        (bf16 output)
 *
 * where K_j / V_j are row j % P of page block_table[b][j / P] (HND or NHD
 * layout, see splitkv_kv_layout), dequantised as code * kv_scale when the cache is FP8-e4m3.  The KV range of
 * each sequence is cut into num_splits page ranges, each handled by its own
 * CTA, and the per-split results are merged by their log-sum-exp.  This is the
 * split-KV scheme of "vLLM 0.30.0 FA4 SplitKV Bug: H100 Decode Can Be 48%
 * Slower", section "What SplitKV is trying to do" (one query token, few KV
 * heads, long KV history: split the KV range so more SMs work), with a
 * partial result per split and a combine step that gives empty splits zero
 * weight (section "Why the result is still correct").  Unlike the bug that
 * page dissects ("The actual bug is one missing constructor argument"), the
 * requested split count is honoured and every launched split CTA owns a
 * non-empty KV range.  FP8 KV with BF16 queries follows "Xqa decode kernels"
 * (vLLM pull request #43232), section "Purpose"; the multi-token MLA case
 * follows "Shipped: 484.5 tok/s on one GB300 ...", table "What shipped".
 *
 * Conventions for every entry point.
 *   - Pointers named *_host are host memory; every other data pointer is
 *     device memory owned by the caller.  The library never allocates device
 *     memory and never frees caller memory.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Device work is enqueued asynchronously on it; only
 *     splitkv_read_stats synchronises (that stream only).
 *   - Arguments are validated on the host before anything is enqueued; on an
 *     error nothing is written.  splitkv_last_error() then describes it.
 *   - Device data pointers must be 16-byte aligned.
 */
#ifndef SPLITKV_H
#define SPLITKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum splitkv_status {
  SPLITKV_OK = 0,
  SPLITKV_EINVAL = 1,        /* bad argument (null, shape, alignment, range)   */
  SPLITKV_EUNSUPPORTED = 2,  /* valid shape this build has no kernel for       */
  SPLITKV_ECUDA = 3,         /* a CUDA runtime call or launch failed           */
  SPLITKV_EWORKSPACE = 4,    /* workspace missing or too small                 */
  SPLITKV_EDEVICE = 5        /* a kernel reported an error in the status word  */
} splitkv_status;

typedef enum splitkv_dtype {
  SPLITKV_BF16 = 0,          /* K/V pages hold bf16                            */
  SPLITKV_FP8_E4M3 = 1       /* K/V pages hold OCP e4m3fn codes, x kv_scale    */
} splitkv_dtype;

typedef enum splitkv_combine_mode {
  SPLITKV_COMBINE_FUSED = 0,    /* the split kernel merges: the last CTA of each
                                   (b, h_kv) group, or with more than 8 splits the
                                   last CTA of each bundle of 8 and then the last
                                   bundle of the group (GQA; MLA always merges
                                   with the combine kernel)                    */
  SPLITKV_COMBINE_SEPARATE = 1  /* a second kernel merges all partials          */
} splitkv_combine_mode;

/* Order of the dimensions inside the K and V page pools.  "Xqa decode
 * kernels" (vLLM pull request #43232), section "Test Plan", runs its decode
 * path with the cache layout set to HND; NHD is the other value of that
 * setting.  Both hold the same rows; only the strides differ.  The MLA
 * family has one KV head, where the two orders coincide. */
typedef enum splitkv_kv_layout {
  SPLITKV_LAYOUT_HND = 0,    /* pages[num_pages][Hkv][P][dim]: one head's page rows
                                are contiguous                                 */
  SPLITKV_LAYOUT_NHD = 1     /* pages[num_pages][P][Hkv][dim]: the heads of one
                                key are contiguous                             */
} splitkv_kv_layout;

/* Shapes and element types of one decode-attention call (no pointers). */
typedef struct splitkv_desc {
  int32_t batch;              /* B, >= 1                                        */
  int32_t q_tokens;           /* T query tokens per sequence, causal among them;
                                 GQA: T * (Hq / Hkv) <= 32; MLA: T <= 16       */
  int32_t num_q_heads;        /* Hq                                             */
  int32_t num_kv_heads;       /* Hkv, divides Hq                                */
  int32_t qk_dim;             /* Dk: 128 (GQA) or 576 (MLA latent + rope)       */
  int32_t v_dim;              /* Dv: 128 (GQA) or 512 (MLA)                     */
  int32_t page_size;          /* P tokens per page, multiple of 16; MLA: 16, 32
                                 or a multiple of 64                           */
  int32_t max_pages_per_seq;  /* row length of block_table                     */
  int32_t num_pages_total;    /* pages in k_pages / v_pages                     */
  int32_t kv_dtype;           /* splitkv_dtype; q and out are always bf16       */
  int32_t v_shares_k;         /* 1: V_j = first v_dim columns of K_j (the MLA
                                 latent cache); MLA also serves 0 (V its own
                                 [N][1][P][512] tensor)                        */
  int32_t combine_mode;       /* splitkv_combine_mode                           */
  int32_t kv_layout;          /* splitkv_kv_layout of k_pages and v_pages       */
} splitkv_desc_t;

/* Opaque host object holding the split table of one set of sequence lengths. */
typedef struct splitkv_plan_s splitkv_plan_t;

/* Fields of one work item as returned by splitkv_plan_get_items (int32 each). */
enum {
  SPLITKV_ITEM_B = 0,         /* sequence                                        */
  SPLITKV_ITEM_HKV = 1,       /* first KV head; the item covers heads [HKV,
                                 HKV + splitkv_plan_heads_per_item)              */
  SPLITKV_ITEM_SPLIT = 2,     /* split index s in [0, S_b)                       */
  SPLITKV_ITEM_NSPLIT = 3,    /* S_b, splits of this sequence                    */
  SPLITKV_ITEM_PAGE0 = 4,     /* first page (logical, within the sequence)       */
  SPLITKV_ITEM_PAGE1 = 5,     /* one past the last page                          */
  SPLITKV_ITEM_SLOT = 6,      /* partial-result slot, -1 when S_b == 1           */
  SPLITKV_ITEM_GROUP = 7,     /* combine group of (b, HKV), -1 when S_b == 1     */
  SPLITKV_ITEM_FIELDS = 8
};

/*
 * splitkv_plan -- split planning (host only; no CUDA call unless num_sms == 0).
 *
 * For each sequence, n_b = ceil(seq_lens_host[b] / P) pages.  With
 * num_splits > 0, S_b = min(num_splits, n_b): the request is honoured
 * whenever the sequence has that many pages.  With num_splits == 0 the
 * planner picks one chunk size for all sequences by a load-balance cost model
 * (largest-first list scheduling of the work items over the kernel's resident
 * slots -- 3 CTAs per SM for GQA, one CTA pair per query token for MLA --
 * plus a fixed cost per item and a per-split merge cost) and S_b = n_b / chunk
 * rounded up or down, clamped to [1, min(n_b, 64)].  Split s covers pages
 * [floor(s*n_b/S_b), floor((s+1)*n_b/S_b)), which is never empty.  One work
 * item covers splitkv_plan_heads_per_item consecutive KV heads of one split.
 * Items are ordered longest first.  A sequence with no keys gets one empty
 * item per head group that writes out = 0, lse = -inf.
 *
 *   desc           shapes; copied into the plan
 *   seq_lens_host  [B] int32, 0 <= L <= max_pages_per_seq * P, L >= T or L == 0
 *   num_splits     requested splits per sequence, 0 = planner's choice, <= 64
 *   num_sms        SMs to plan for; 0 = query the current device
 *   plan_out       receives a new plan; free with splitkv_plan_destroy
 */
splitkv_status splitkv_plan(const splitkv_desc_t* desc, const int32_t* seq_lens_host,
                            int32_t num_splits, int32_t num_sms, splitkv_plan_t** plan_out);

/*
 * splitkv_plan_fixed -- a capacity plan for CUDA-graph-captured serving, where
 * the sequence lengths change from step to step while every launch's grid is
 * fixed ("Shipped: 484.5 tok/s on one GB300 ...", table "What shipped":
 * split attention was enabled for one captured shape only).  The plan holds
 * num_splits work items for every (sequence, KV-head group) -- B * Hkv /
 * heads_per_item * num_splits items, in (b, head group, s) order -- and one
 * combine group per (sequence, head group) when num_splits > 1.  Each decode
 * derives every item from the device lengths it is given (after its
 * dependency wait, so a preceding kernel may write them): with S_b =
 * min(num_splits, ceil(L_b / P)) (1 for L_b == 0), items s < S_b get the page
 * ranges splitkv_plan gives for this num_splits, and the others are unused:
 * their CTAs are launched and exit at once, logging 0 keys.  A length outside
 * [0, max_pages_per_seq * P] or below q_tokens (and not 0) sets
 * SPLITKV_DEVERR_SEQLEN in the status word and the sequence is served as
 * empty (out = 0, lse = -inf).  splitkv_plan_get_items returns the all-unused
 * template; splitkv_plan_refresh + splitkv_read_items show the live list.
 *   num_splits  1..64
 * EINVAL for bad arguments; EUNSUPPORTED for shapes no kernel serves.
 */
splitkv_status splitkv_plan_fixed(const splitkv_desc_t* desc, int32_t num_splits,
                                  splitkv_plan_t** plan_out);

/*
 * splitkv_plan_refresh -- one small kernel on `stream` that writes into
 * `workspace` (uploaded once with splitkv_plan_upload) the work list and the
 * combine-group table a decode of this capacity plan derives from seq_lens
 * (device, int32 [B]), for inspection with splitkv_read_items.  A decode does
 * not need it: the kernels derive the same items themselves.  Invalid
 * lengths are reported as splitkv_plan_fixed describes.  EINVAL if the plan
 * was not made by splitkv_plan_fixed or for NULL or misaligned pointers.
 */
splitkv_status splitkv_plan_refresh(const splitkv_plan_t* plan, void* workspace,
                                    const int32_t* seq_lens, void* stream);

/*
 * splitkv_read_items -- synchronises `stream` and copies the work list held in
 * `workspace` (splitkv_plan_num_items items, SPLITKV_ITEM_FIELDS int32 each,
 * launch order) to items_host.  EINVAL if capacity (items) is too small.
 */
splitkv_status splitkv_read_items(const splitkv_plan_t* plan, const void* workspace,
                                  int32_t* items_host, int32_t capacity, void* stream);

/* Frees a plan (NULL is ignored). */
void splitkv_plan_destroy(splitkv_plan_t* plan);

/*
 * Copies the work list out: items_host receives n * SPLITKV_ITEM_FIELDS int32
 * in launch order (fields above); capacity is in items.  *n_items always
 * receives the item count; EINVAL if capacity is smaller (nothing copied).
 */
splitkv_status splitkv_plan_get_items(const splitkv_plan_t* plan, int32_t* items_host,
                                      int32_t capacity, int32_t* n_items);

/*
 * splitkv_plan_get_ranges -- the split table per KV head: one row of
 * SPLITKV_RANGE_FIELDS int32 (b, h_kv, s, page_begin, page_end) for every
 * sequence b, KV head h_kv and split s < S_b, in launch order (the KV heads of
 * one work item consecutively).  Split s of sequence b covers pages
 * [floor(s * n_b / S_b), floor((s + 1) * n_b / S_b)) of n_b = ceil(L_b / P),
 * never empty unless L_b == 0.  capacity is in rows; *n_ranges always
 * receives the row count (items * heads_per_item); EINVAL if capacity is
 * smaller (nothing copied).  For a capacity plan these are the template's
 * rows, all empty until splitkv_plan_refresh fills the device list.
 */
enum { SPLITKV_RANGE_FIELDS = 5 };
splitkv_status splitkv_plan_get_ranges(const splitkv_plan_t* plan, int32_t* ranges_host,
                                       int32_t capacity, int32_t* n_ranges);

/* Number of work items. */
int32_t splitkv_plan_num_items(const splitkv_plan_t* plan);

/* CTAs the split-KV kernel launches for this plan (one per item for GQA; a
 * CTA pair per query token and item for MLA): the rows of the per-CTA log. */
int32_t splitkv_plan_num_ctas(const splitkv_plan_t* plan);

/* KV heads one work item covers: 2 when Hkv is even for the e4m3 GQA path
 * with at most 16 query rows (T * G) per KV head, where one TMA box then
 * brings a 16-key tile of both; 1 otherwise.  Partial-result rows of an item
 * are numbered head_slot * T * G + t * G + g. */
int32_t splitkv_plan_heads_per_item(const splitkv_plan_t* plan);

/* Kernel launches one splitkv_decode of this plan makes (1 or 2: the split
 * kernel, plus the combine kernel when splits must be merged and the merge
 * does not run inside the split kernel). */
int32_t splitkv_plan_launches_per_call(const splitkv_plan_t* plan);

/* Bytes of device workspace the plan needs (work list, tickets, per-CTA log,
 * partial outputs).  0 if plan is NULL. */
size_t splitkv_workspace_size(const splitkv_plan_t* plan);

/*
 * splitkv_plan_upload -- writes the plan's work list into `workspace` and
 * zeroes its merge tickets and status word (one host->device copy on
 * `stream`).  Must be called once per (plan, workspace) pair before
 * splitkv_decode; the kernels leave the tickets zeroed, so repeated decodes
 * (including CUDA-graph replays) need no further upload.
 */
splitkv_status splitkv_plan_upload(const splitkv_plan_t* plan, void* workspace,
                                   size_t workspace_bytes, void* stream);

/*
 * splitkv_decode -- one split-KV decode-attention call.
 *
 *   q            bf16 [B][T][Hq][Dk]
 *   k_pages      [num_pages_total][Hkv][P][Dk] of bf16 or e4m3 codes (HND;
 *                [num_pages_total][P][Hkv][Dk] with SPLITKV_LAYOUT_NHD)
 *   v_pages      the same with Dv; ignored (may be NULL) when v_shares_k
 *   block_table  int32 [B][max_pages_per_seq] physical page ids; entries past
 *                ceil(L/P) are never read
 *   seq_lens     int32 [B] device copy of the lengths the plan was built from
 *                (a mismatch is recorded in the status word)
 *   num_splits   the plan's num_splits, or 0 (= whatever the plan holds)
 *   scale        softmax scale applied to q.K (e.g. 1/sqrt(Dk))
 *   kv_scale     dequantisation scale of FP8 K and V (ignored for bf16)
 *   out          bf16 [B][T][Hq][Dv]
 *   lse          fp32 [B][T][Hq], natural-log LSE of the scaled scores; may be
 *                NULL
 *   workspace    uploaded with splitkv_plan_upload for this plan
 * Launches one kernel (FUSED) or two (SEPARATE, second with programmatic
 * dependent launch).
 */
splitkv_status splitkv_decode(const splitkv_plan_t* plan, void* workspace,
                              const void* q, const void* k_pages, const void* v_pages,
                              const int32_t* block_table, const int32_t* seq_lens,
                              int32_t num_splits, float scale, float kv_scale,
                              void* out, float* lse, void* stream);

/*
 * splitkv_decode_kv_scales -- splitkv_decode over an e4m3 cache whose K and V
 * carry their own dequantisation scale per KV head: K_j = code * k_scale[h],
 * V_j = code * v_scale[h] for KV head h (a separate per-tensor K and V scale
 * is the case of all-equal entries).  "Xqa decode kernels", section
 * "Purpose", names an FP8 KV cache with a scale; the per-head, per-tensor
 * split of that scale is this library's extension.
 *   k_scale, v_scale  fp32 [Hkv] device arrays, positive and finite (not
 *                     checked: they are read by the kernel after the
 *                     dependency wait, so a preceding kernel may write them)
 *   other arguments   as splitkv_decode (there is no kv_scale)
 * EUNSUPPORTED for bf16 caches and the MLA shape; EINVAL for NULL or
 * misaligned (< 4 bytes) scale arrays.
 */
splitkv_status splitkv_decode_kv_scales(const splitkv_plan_t* plan, void* workspace,
                                        const void* q, const void* k_pages, const void* v_pages,
                                        const int32_t* block_table, const int32_t* seq_lens,
                                        int32_t num_splits, float scale, const float* k_scale,
                                        const float* v_scale, void* out, float* lse,
                                        void* stream);

/*
 * splitkv_decode_partials / splitkv_combine_workspace -- splitkv_decode in
 * its two steps: the per-split partial attention pass, then the log-sum-exp
 * merge ("vLLM 0.30.0 FA4 SplitKV Bug: H100 Decode Can Be 48% Slower",
 * sections "What SplitKV is trying to do" and "Why the result is still
 * correct").  splitkv_decode_partials launches only the split-KV kernel, in
 * the SEPARATE form whatever desc.combine_mode says: sequences with one
 * split write out / lse, the others leave their fp32 (O_s, lse_s) partials
 * in the workspace.  splitkv_combine_workspace then merges those partials
 * into out / lse (one kernel; it reads nothing else), so the pair writes
 * exactly what splitkv_decode writes in SPLITKV_COMBINE_SEPARATE mode.
 * Between the two a caller may run its own work on the stream (or read,
 * exchange and merge the partials itself), as long as it leaves the
 * workspace's partials intact.
 *   splitkv_decode_partials     arguments and errors as splitkv_decode
 *   splitkv_combine_workspace   plan, workspace (as passed to the partials
 *                               call), out bf16 [B][T][Hq][Dv] (16-byte
 *                               aligned), lse fp32 [B][T][Hq] or NULL
 * EINVAL for NULL or misaligned pointers; EWORKSPACE for a NULL workspace.
 */
splitkv_status splitkv_decode_partials(const splitkv_plan_t* plan, void* workspace,
                                       const void* q, const void* k_pages, const void* v_pages,
                                       const int32_t* block_table, const int32_t* seq_lens,
                                       int32_t num_splits, float scale, float kv_scale, void* out,
                                       float* lse, void* stream);
splitkv_status splitkv_combine_workspace(const splitkv_plan_t* plan, void* workspace, void* out,
                                         float* lse, void* stream);

/*
 * splitkv_decode_noalloc -- splitkv_decode for callers that cannot allocate
 * device memory (code running inside another framework's memory budget,
 * plugins whose host forbids device allocations after start-up, real-time
 * loops that must not risk an allocation stall).  Same arguments and result
 * as splitkv_decode, minus the workspace: the workspace lives in one 16 MiB
 * device array inside the library, which every GPU that loads the library
 * holds until the process exits.  This entry point has no counterpart on the
 * pages; it is a packaging convenience.
 *
 *   - Calls no cudaMalloc, cudaFree or other allocating routine.
 *   - A plan whose splitkv_workspace_size exceeds 16 MiB is rejected with
 *     SPLITKV_EWORKSPACE (use splitkv_decode with a caller workspace).
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture.
 *   - Each call uploads the plan into the array (zeroing its merge tickets and
 *     status word) and then decodes.  All calls share the one array and it
 *     keeps the last call's contents, so calls that overlap on the GPU (other
 *     streams, other threads) race; serialise them on one stream.
 *   - The call's status word and per-CTA log are read with
 *     splitkv_noalloc_read_stats.
 */
splitkv_status splitkv_decode_noalloc(const splitkv_plan_t* plan, const void* q,
                                      const void* k_pages, const void* v_pages,
                                      const int32_t* block_table, const int32_t* seq_lens,
                                      int32_t num_splits, float scale, float kv_scale,
                                      void* out, float* lse, void* stream);

/*
 * splitkv_noalloc_read_stats -- splitkv_read_stats for the decodes of
 * splitkv_decode_noalloc, whose status word and per-CTA log live in the
 * library's scratch array rather than a caller workspace.  It synchronises
 * `stream` and copies the log and status of the last splitkv_decode_noalloc
 * call on the current device (which should be a call with this plan: the
 * array holds whatever the last call left).  Arguments and fields as
 * splitkv_read_stats.  No counterpart on the pages.
 * EINVAL for a NULL plan or a too-small capacity; EWORKSPACE for a plan larger
 * than the array (it can never have run there).
 */
splitkv_status splitkv_noalloc_read_stats(const splitkv_plan_t* plan, int32_t* cta_log_host,
                                          int32_t capacity, int32_t* status_host, void* stream);

/*
 * splitkv_combine -- the log-sum-exp merge on its own, over caller buffers.
 * For each row r < rows: M = max_s lse_part[s][r]; lse = M + ln sum_s
 * exp(lse_part[s][r] - M); out[r][:] = sum_s exp(lse_part[s][r] - lse) *
 * o_part[s][r][:].  Partials with lse = -inf have weight 0; if every partial
 * of a row is -inf the row gets out = 0, lse = -inf.
 *   o_part    fp32 [n_parts][rows][dv]      lse_part  fp32 [n_parts][rows]
 *   out_bf16  bf16 [rows][dv] or NULL       out_f32   fp32 [rows][dv] or NULL
 *   lse_out   fp32 [rows] or NULL
 *   n_parts >= 1; dv a positive multiple of 4
 */
splitkv_status splitkv_combine(const float* o_part, const float* lse_part, int32_t n_parts,
                               int32_t rows, int32_t dv, void* out_bf16, float* out_f32,
                               float* lse_out, void* stream);

/*
 * splitkv_read_stats -- synchronises `stream`, then copies to the host the
 * per-CTA log of the last decode on `workspace` and the device status word.
 *   cta_log_host  int32 [capacity][4] or NULL: per launched CTA {first page,
 *                 one-past-last page it iterated, keys it scored, flag} in
 *                 launch order; flag (GQA, fused mode): bit 0 set if the CTA
 *                 wrote its group's merged output, bit 1 set if it merged a
 *                 bundle of up to 8 splits; flag (MLA): nonzero if the CTA
 *                 gave up on a timed-out wait, (role << 24) | (x << 12) | y
 *                 with role 1 the N-ring producer, 2 the V-ring producer, 3
 *                 the producer of a separate V tensor (y = block), 4 the MMA
 *                 issuer (bit 23: half of QK(x) issued; x = next QK block,
 *                 y = next PV block), 5 the softmax warps (x = 1 waiting for
 *                 S, 2 for PV before a rescale; y = block), 6 the epilogue
 *   capacity      rows of cta_log_host; EINVAL if below splitkv_plan_num_ctas
 *   status_host   int32 or NULL: 0, or a bit set of SPLITKV_DEVERR_* values
 */
splitkv_status splitkv_read_stats(const splitkv_plan_t* plan, const void* workspace,
                                  int32_t* cta_log_host, int32_t capacity, int32_t* status_host,
                                  void* stream);

enum {
  SPLITKV_DEVERR_TIMEOUT = 1,    /* a bounded wait on a shared-memory barrier gave up */
  SPLITKV_DEVERR_SEQLEN = 2,     /* device seq_lens differs from the plan's           */
  SPLITKV_DEVERR_PAGE = 4        /* a block-table entry was outside [0, num_pages)    */
};

/*
 * splitkv_debug_gather -- copies keys [0, n_keys) of sequence b, KV head h_kv
 * through the block table into device memory `dst` ([n_keys][row_elems] raw
 * elements), using the same TMA tensor-map loads and swizzled shared-memory
 * reads as the decode kernel.  For checking the paged gather bit for bit.
 *   GQA:  `pages` is k_pages or v_pages in desc->kv_layout; row_elems = 128.
 *   MLA:  `pages` is the latent cache (row_elems = qk_dim = 576) or, with
 *         v_shares_k = 0, the separate V tensor (row_elems = v_dim = 512);
 *         h_kv = 0; rows come in the decode kernel's 64-key blocks of 64-column
 *         boxes (one box per page for pages of 16 or 32 keys).
 * Page ids outside [0, num_pages_total) are read as page 0, as the decode
 * kernels do.  EINVAL for other row widths, ranges or misaligned buffers.
 */
splitkv_status splitkv_debug_gather(const splitkv_desc_t* desc, const void* pages,
                                    int32_t row_elems, const int32_t* block_table,
                                    int32_t b, int32_t h_kv, int32_t n_keys, void* dst,
                                    void* stream);

/* Thread-local description of the last error returned on this thread. */
const char* splitkv_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* SPLITKV_H */
