/*
 * hp.h -- C ABI of the shared-prefix (cascade) decode attention library for
 * NVIDIA GB300 (sm_103a).
 *
 * The problem.  B decoding sequences each hold one new query token per query
 * head.  Their keys and values form a prefix tree: a prefix shared by all or
 * some of the sequences, possibly further shared levels, and a private suffix
 * per sequence.  Attention over the concatenated keys is split at every tree
 * vertex; the parts are computed separately and merged exactly by their
 * log-sum-exp (Hydragen, "Attention Decomposition Across Subsequences", Eq. 5;
 * "Hierarchical Sharing").  The queries of all sequences below a shared node
 * are stacked into one matrix and attend to the node's keys in one
 * matrix-matrix pass, so the node's KV is read once per step (Hydragen,
 * "Inter-Sequence Batched Prefix Attention"; ChunkAttention, "The Chunk-First
 * Phase Kernel in Detail").  Private suffixes are a paged per-sequence decode
 * (ChunkAttention, "The Sequence-First Phase Kernel in Detail").
 *
 * Conventions shared by every call:
 *   - q: bf16, row (b, h) at q + b*q_sb + h*q_sh (element strides; the head
 *     dimension is contiguous).  Query head h reads KV head h / (Hq/Hkv).
 *   - paged KV pools: bf16 [num_pages][Hkv][page_size][d], contiguous.  Token t
 *     of a page list sits at page list[t / page_size], slot t % page_size.
 *   - scale: the softmax scale applied to q.k (1/sqrt(d) in the pages); must be
 *     positive for hp_prefix_attn and hp_cascade_decode (HP_ERR_ARG otherwise).
 *   - out: bf16 or f32, row (b, h) at out + b*o_sb + h*o_sh (elements).
 *   - lse: f32, natural log of the softmax denominator of the scaled scores
 *     (Hydragen's LSE(Q,K)), element (b, h) at lse + b*lse_sb + h.  A row with
 *     no visible key gets out = 0 and lse = -inf.
 *   - All device pointers are owned by the caller.  The library never
 *     allocates, frees or synchronises inside the compute calls; every launch
 *     is ordered on the given stream and can be captured in a CUDA graph.
 *   - ws: caller-owned device workspace of at least the size the matching
 *     *_workspace_bytes / plan call reports, 256-byte aligned.  Its first
 *     bytes hold a device status word that kernels set on a bounds violation
 *     or a wait that ran out; read it with hp_read_device_status.
 *   - Supported: d in {64, 128}; Hq % Hkv == 0; page_size a multiple of 16 up
 *     to 256; bf16 q/K/V.  Anything else returns HP_ERR_UNSUPPORTED.
 *   - Errors are return codes; argument errors return before any launch.
 */
#ifndef HP_H
#define HP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t (the runtime's stream handle); NULL is the legacy stream. */
typedef struct CUstream_st *hp_stream_t;

typedef enum {
    HP_OK = 0,
    HP_ERR_ARG = 1,             /* invalid argument (null pointer, bad size, bad tree) */
    HP_ERR_UNSUPPORTED = 2,     /* valid but outside the supported shapes */
    HP_ERR_WORKSPACE = 3,       /* workspace or plan buffer too small or misaligned */
    HP_ERR_CUDA = 4,            /* a CUDA runtime call failed */
    HP_ERR_BOUNDS = 5,          /* device: a page id or length was out of range */
    HP_ERR_DEVICE_TIMEOUT = 6   /* device: a bounded wait ran out */
} hp_status;

typedef enum { HP_BF16 = 0, HP_F32 = 1 } hp_dtype;

/* Storage of a level's (or a paged decode's) keys and values.
 * HP_KV_BF16: bf16 pools [num_pages][Hkv][page_size][d].
 * HP_KV_E4M3: reduced-precision pools for the memory-bound per-sequence pass
 * (Hydragen, "Implications and Future Directions": quantising the KV cache
 * is the complementary remedy for suffix attention, which stays bound by its
 * bytes).  One byte per element: an E4M3 code (the OCP 8-bit floating-point
 * format with 4 exponent bits, bias 7, 3 mantissa bits, no infinities;
 * S.1111.111 is not a number and must not be stored), laid out
 * [num_pages][Hkv][page_size][d]; plus one f32 scale per (page, KV head) for K
 * and one for V, device arrays [num_pages][Hkv].  The stored value of a code
 * is its E4M3 value times the scale of its page and KV head.  Only d = 128;
 * queries stay bf16 and must lie within f16's range (|q| < 65504): the kernels
 * use f16 tensor-core products for these levels. */
typedef enum { HP_KV_BF16 = 0, HP_KV_E4M3 = 1 } hp_kv_type;

const char *hp_status_str(hp_status s);

/* ---------------------------------------------------------------------------
 * hp_merge_states -- exact merge of two attention states over disjoint key
 * sets (Hydragen Eq. 5 in its max-subtracted combine_lse form):
 *   M = max(lse_a, lse_b); wa = e^(lse_a - M); wb = e^(lse_b - M)
 *   o = (wa o_a + wb o_b) / (wa + wb);  lse = M + ln(wa + wb)
 * o_a, o_b: f32 [rows][d] (contiguous); lse_a, lse_b: f32 [rows].
 * o_out: [rows][d] of out_dt; lse_out: f32 [rows] (may be NULL).  Outputs may
 * alias the inputs element for element (o_out == o_a with out_dt = HP_F32).
 * Both states empty (-inf) gives o = 0, lse = -inf.  Any d >= 1.
 * ------------------------------------------------------------------------- */
hp_status hp_merge_states(const float *o_a, const float *lse_a, const float *o_b,
                          const float *lse_b, void *o_out, hp_dtype out_dt, float *lse_out,
                          int64_t rows, int32_t d, hp_stream_t stream);

/* ---------------------------------------------------------------------------
 * hp_suffix_decode_paged -- per-sequence paged decode (ChunkAttention's
 * sequence-first phase over private chunks; Hydragen's suffix attention).
 * Sequence b attends over its first seq_lens[b] tokens, token t at page
 * page_table[b*pt_stride + t/page_size], slot t % page_size, of the pools.
 * The G = Hq/Hkv query heads of a KV head are processed together; the keys of
 * a sequence are split into chunks whose partial states are merged in the
 * same call.  page_table and seq_lens are device int32 arrays read on the
 * device (so lengths may change between replays of a captured graph); a page
 * id outside [0, num_pages) or a length above pt_stride*page_size sets
 * HP_ERR_BOUNDS in the workspace status word and the offending keys are
 * skipped.
 * ------------------------------------------------------------------------- */
size_t hp_suffix_workspace_bytes(int32_t B, int32_t Hq, int32_t d, int32_t pt_stride,
                                 int32_t page_size);
hp_status hp_suffix_decode_paged(const void *q, int64_t q_sb, int64_t q_sh, int32_t B,
                                 const void *k_pool, const void *v_pool, int32_t num_pages,
                                 int32_t page_size, const int32_t *page_table, int32_t pt_stride,
                                 const int32_t *seq_lens, int32_t Hq, int32_t Hkv, int32_t d,
                                 float scale, void *out, hp_dtype out_dt, int64_t o_sb,
                                 int64_t o_sh, float *lse, int64_t lse_sb, void *ws,
                                 size_t ws_bytes, hp_stream_t stream);

/* ---------------------------------------------------------------------------
 * hp_suffix_decode_paged_noalloc -- the same paged decode for callers that
 * cannot hand the library any device memory of their own: a host program or
 * plugin that reaches this library only through the C ABI and has no device
 * allocator, code running where a caching allocator already holds all device
 * memory so that cudaMalloc would fail, or a latency-critical path that must
 * not pay for cudaMalloc's implicit synchronisation.  (This entry point has
 * no counterpart in the papers; it is a deployment convenience.)
 *
 * Arguments and results are those of hp_suffix_decode_paged without the
 * workspace.  Scratch lives in one fixed 16 MiB device array inside the
 * library, resident on every GPU that loads the library until the process
 * exits; the call itself allocates and frees nothing.  Each key split of a
 * call needs B*Hq partial rows of 2*d + 4 bytes (a bf16 O row and its f32
 * LSE); the call picks the fewest splits of at least 64 keys that fit, and
 * returns HP_ERR_WORKSPACE when even one split does not: B*Hq above 64,525
 * rows at d = 128, 127,096 at d = 64.  The first call in each CUDA context
 * (the first on a device, and the first after cudaDeviceReset) looks up the
 * array's device address, a host call made with that device current; make
 * that first call before any stream capture.  All calls share the array and
 * it keeps the last call's contents: calls that run at the same time on the
 * GPU race with each other, so serialise them.  The kernels keep a status
 * word at the start of the array (cleared by each call), but it is not
 * returned to the caller: device bounds errors go unreported.
 * ------------------------------------------------------------------------- */
hp_status hp_suffix_decode_paged_noalloc(const void *q, int64_t q_sb, int64_t q_sh, int32_t B,
                                         const void *k_pool, const void *v_pool,
                                         int32_t num_pages, int32_t page_size,
                                         const int32_t *page_table, int32_t pt_stride,
                                         const int32_t *seq_lens, int32_t Hq, int32_t Hkv,
                                         int32_t d, float scale, void *out, hp_dtype out_dt,
                                         int64_t o_sb, int64_t o_sh, float *lse, int64_t lse_sb,
                                         hp_stream_t stream);

/* ---------------------------------------------------------------------------
 * hp_suffix_decode_paged_e4m3 -- hp_suffix_decode_paged over E4M3 pools
 * (hp_kv_type HP_KV_E4M3): k_pool / v_pool hold the codes, k_scale / v_scale
 * the f32 scales [num_pages][Hkv] (device, 4-byte aligned).  d = 128 only.
 * Workspace: hp_suffix_workspace_bytes.  Otherwise as hp_suffix_decode_paged.
 * ------------------------------------------------------------------------- */
hp_status hp_suffix_decode_paged_e4m3(const void *q, int64_t q_sb, int64_t q_sh, int32_t B,
                                      const void *k_pool, const void *v_pool, const float *k_scale,
                                      const float *v_scale, int32_t num_pages, int32_t page_size,
                                      const int32_t *page_table, int32_t pt_stride,
                                      const int32_t *seq_lens, int32_t Hq, int32_t Hkv, int32_t d,
                                      float scale, void *out, hp_dtype out_dt, int64_t o_sb,
                                      int64_t o_sh, float *lse, int64_t lse_sb, void *ws,
                                      size_t ws_bytes, hp_stream_t stream);

/* ---------------------------------------------------------------------------
 * hp_stream_decode -- a decode step of Parallel Prompting requests, each
 * request's KV row read in place with the stream mask applied inside the
 * kernel (Read Once, Answer Many, Section 3 "Parallel Prompting", Eq. 2, and
 * Figure 2's in-kernel mask; Section 4 for the two index tensors).
 *
 * Request r (0 <= r < R) decodes P streams; its query for stream s is query
 * sequence r*P + s: q rows (r*P + s, h) at q + (r*P + s)*q_sb + h*q_sh (bf16,
 * as in the conventions above, 16-byte aligned, strides multiples of 8).
 * Its KV row holds row_len[r] slots -- the document, then the streams'
 * question and answer tokens in any order -- slot t at page
 * row_pages[r*pt_stride + t/page_size], position t % page_size, of the bf16
 * pools [num_pages][Hkv][page_size][d].  Slot t carries a stream id
 * slot_sid[r*sid_stride + t] (-1 for the document) and a position
 * slot_pos[r*sid_stride + t]; query r*P + s carries q_sid[r*P + s] and
 * q_pos[r*P + s].  Slot t is visible to that query iff
 *     slot_pos <= q_pos  and  (slot_sid == -1 or slot_sid == q_sid)
 * (the causal condition on positions, which the streams share, and the
 * stream condition of Eq. 2).  All device int32 arrays; sid_stride a multiple
 * of 4 with sid_stride >= pt_stride*page_size, slot arrays 16-byte aligned.
 * The streams of a request share the pass over its row (up to 8 groups of
 * 16 / (Hq/Hkv) streams per pass; more streams take further passes).  Rows
 * with no visible slot get out = 0, lse = -inf.  A page id outside
 * [0, num_pages) or a row length above pt_stride*page_size sets HP_ERR_BOUNDS
 * in the workspace status word.  ws: >= hp_stream_workspace_bytes.
 * ------------------------------------------------------------------------- */
size_t hp_stream_workspace_bytes(int32_t R, int32_t P, int32_t Hq, int32_t Hkv, int32_t d,
                                 int32_t pt_stride, int32_t page_size);
hp_status hp_stream_decode(const void *q, int64_t q_sb, int64_t q_sh, int32_t R, int32_t P,
                           const void *k_pool, const void *v_pool, int32_t num_pages,
                           int32_t page_size, const int32_t *row_pages, int32_t pt_stride,
                           const int32_t *row_len, const int32_t *slot_sid, const int32_t *slot_pos,
                           int32_t sid_stride, const int32_t *q_sid, const int32_t *q_pos, int32_t Hq,
                           int32_t Hkv, int32_t d, float scale, void *out, hp_dtype out_dt,
                           int64_t o_sb, int64_t o_sh, float *lse, int64_t lse_sb, void *ws,
                           size_t ws_bytes, hp_stream_t stream);

/* ---------------------------------------------------------------------------
 * hp_prefix_attn -- inter-sequence batched attention against one contiguous
 * shared prefix (Hydragen, "Inter-Sequence Batched Prefix Attention": the
 * queries of sequences [row_begin, row_begin + rows) are stacked and attend
 * to the prefix in one matrix-matrix pass; the prefix is read once).
 * k, v: bf16, token t of KV head g at k + t*kv_st + g*kv_sh (elements; the
 * head dimension contiguous; kv_st and kv_sh multiples of 8; 16-byte aligned
 * base).  Outputs rows b in [row_begin, row_begin + rows) of out / lse.
 * prefix_len = 0 gives out = 0, lse = -inf.
 * ------------------------------------------------------------------------- */
size_t hp_prefix_workspace_bytes(int32_t rows, int32_t Hq, int32_t Hkv, int32_t d,
                                 int32_t prefix_len);
hp_status hp_prefix_attn(const void *q, int64_t q_sb, int64_t q_sh, int32_t row_begin,
                         int32_t rows, const void *k, const void *v, int64_t kv_st, int64_t kv_sh,
                         int32_t prefix_len, int32_t Hq, int32_t Hkv, int32_t d, float scale,
                         void *out, hp_dtype out_dt, int64_t o_sb, int64_t o_sh, float *lse,
                         int64_t lse_sb, void *ws, size_t ws_bytes, hp_stream_t stream);

/* ---------------------------------------------------------------------------
 * Cascade decode over a level-by-level prefix tree (Hydragen "Hierarchical
 * Sharing"; ChunkAttention prefix tree and its (C, i, j) kernel context).
 *
 * A level is a set of nodes with disjoint sequence ranges.  Node
 * (seq_begin, seq_end, kv_len, page_off) holds kv_len tokens, visible to the
 * contiguous sequences [seq_begin, seq_end), in pages
 * page_ids[page_off .. page_off + ceil(kv_len/page_size)) of the level's pools.
 * Sequence b attends over the tokens of the node covering it at each level
 * (a level may leave b uncovered).  A private suffix is a level whose nodes
 * cover one sequence each; kv_len = 0 is legal.
 *
 * The nodes and page ids are HOST arrays, read only during hp_cascade_plan.
 * The pools are device pointers; they must stay valid while the plan is used.
 *
 * E4M3 levels (kv_type = HP_KV_E4M3, d = 128) serve nodes that run the
 * per-sequence pass: every node of such a level covers at most 16 / (Hq/Hkv)
 * sequences.  A tree with an E4M3 level keeps its batched (shared) nodes in
 * bf16 levels, and every level it runs in the per-sequence pass must then be
 * E4M3 (HP_ERR_UNSUPPORTED otherwise); decode-loop plans take bf16 levels
 * only.
 * ------------------------------------------------------------------------- */
typedef struct {
    int32_t seq_begin, seq_end, kv_len, page_off;
} hp_tree_node;

typedef struct {
    const void *k_pool; /* device, [num_pages][Hkv][page_size][d] of kv_type, 16-byte aligned */
    const void *v_pool;
    int32_t num_pages;
    int32_t page_size;
    int32_t num_nodes;
    const hp_tree_node *nodes; /* host */
    const int32_t *page_ids;   /* host */
    int32_t num_page_ids;
    int32_t kv_type;           /* hp_kv_type; 0 (bf16) when the struct is zero-initialised */
    const float *k_scale;      /* HP_KV_E4M3: device f32 [num_pages][Hkv], 4-byte aligned; else NULL */
    const float *v_scale;
} hp_tree_level;

typedef struct {
    int32_t num_levels; /* 1 .. 64; at most 8 distinct pool sets (K pool, V pool,
                           num_pages, page_size) across the levels */
    int32_t B, Hq, Hkv, d;
    const hp_tree_level *levels; /* host */
    int32_t num_sms;             /* SMs to plan for; 0 = the current device's count */
} hp_tree_desc;

/* Host summary of a plan, filled by hp_cascade_plan and passed back to
 * hp_cascade_decode (plain data, caller-owned, copyable).  `tag` ties it to
 * the device plan it describes; the kernels check it and report HP_ERR_ARG
 * through the status word on a mismatch. */
typedef struct {
    int32_t B, Hq, Hkv, d;
    int32_t n_tc_items;    /* shared-node items (tensor-core role) */
    int32_t n_small_items; /* small-row items (private suffixes, narrow nodes) */
    int32_t grid;          /* CTAs of the step's persistent launch (one per SM) */
    int32_t rec_stride;    /* bytes of each CTA's schedule record in the plan */
    int32_t num_levels;    /* distinct pool sets of the tree (tensor-map slots) */
    int32_t merge_stride;  /* int32 per row of the plan's merge table */
    int64_t n_part_rows;   /* partial (O, LSE) rows in the workspace */
    int64_t plan_bytes;
    int64_t ws_bytes;      /* workspace hp_cascade_decode needs */
    uint64_t tag;
} hp_plan_info;

/* Bytes of the device plan buffer for this tree (host only, no CUDA calls
 * when desc->num_sms > 0).  0 on an invalid descriptor. */
size_t hp_cascade_plan_bytes(const hp_tree_desc *desc);

/* Validate the tree, flatten it into work items (the pages' context
 * generation: shared nodes become batched items split along the key axis,
 * private nodes become per-sequence items), encode the TMA descriptors of
 * the pools, and copy the plan into plan_dev (device, >= plan_bytes,
 * 256-byte aligned) on `stream`.  The call waits for that copy, so it is not
 * for use inside stream capture.  Re-run only when the tree changes; a plan
 * is reused across steps while the tree and the pools are unchanged.
 * A sequence's own nodes at several levels (nodes covering only that
 * sequence, at most 16 query rows, in the same pools) are planned as one
 * node when every one of them but the last ends on a page boundary: one
 * partial state for that sequence instead of one per node. */
hp_status hp_cascade_plan(const hp_tree_desc *desc, void *plan_dev, size_t plan_bytes,
                          hp_plan_info *info, hp_stream_t stream);

/* One cascade decode step: every sequence, every head, all levels, merged
 * (two launches: the persistent kernel of both passes, then the merge kernel
 * as its programmatic dependent).  The persistent kernel is itself launched
 * as a programmatic dependent of the kernel before it in the stream: it sets
 * up while that kernel drains and waits for it to complete before it reads
 * q, the pools or the workspace.
 * q, out, lse as in the conventions above, for all B sequences; q strides
 * multiples of 8 elements, positive, and q 16-byte aligned (q is read by TMA).
 * ws: >= info->ws_bytes; one workspace serves one call at a time.
 * plan_dev must hold the plan hp_cascade_plan last
 * wrote there in this process, and info must describe a plan no larger than
 * it (HP_ERR_ARG otherwise, before any launch); an info of another plan of the
 * same size is reported by the kernels through the status word.
 * No host synchronisation, no allocation; graph-capturable. */
hp_status hp_cascade_decode(const void *plan_dev, const hp_plan_info *info, const void *q,
                            int64_t q_sb, int64_t q_sh, float scale, void *out, hp_dtype out_dt,
                            int64_t o_sb, int64_t o_sh, float *lse, int64_t lse_sb, void *ws,
                            size_t ws_bytes, hp_stream_t stream);

/* The same step for a caller whose queries arrive in, and whose outputs go
 * to, page-locked host memory (a serving loop that receives the step's
 * query vectors on the host and returns the attention output there): a
 * copy-in kernel reads q from host memory over the host link into the
 * workspace, the step runs on that copy, and the merge kernel stores O and
 * LSE straight into the host buffers.  No copy engine is used, so the three
 * kernels chain as programmatic dependents like the device-resident step;
 * the copy-in kernel issues its host reads before it waits for the kernel
 * ahead of it.  Not from the pages: their kernels take device tensors.
 * q_host, out_host and lse_host (lse_host may be NULL) must be page-locked
 * host memory (cudaHostAlloc / cudaHostRegister; HP_ERR_ARG otherwise, before
 * any launch), laid out as in hp_cascade_decode.
 * ws: >= hp_cascade_host_workspace_bytes(info) bytes (the step's workspace
 * followed by a B x Hq x d bf16 copy of q).  The host buffers must not be
 * written by the host while the step runs.  No host synchronisation, no
 * allocation; graph-capturable. */
size_t hp_cascade_host_workspace_bytes(const hp_plan_info *info);
hp_status hp_cascade_decode_host(const void *plan_dev, const hp_plan_info *info, const void *q_host,
                                 int64_t q_sb, int64_t q_sh, float scale, void *out_host, hp_dtype out_dt,
                                 int64_t o_sb, int64_t o_sh, float *lse_host, int64_t lse_sb, void *ws,
                                 size_t ws_bytes, hp_stream_t stream);

/* The same step, recording caller-created CUDA events (cudaEvent_t handles;
 * any may be NULL) on `stream` -- as external event nodes when the stream is
 * being captured, so they time each replay: events[0] before the step's
 * persistent kernel (prefix and suffix passes), events[1] after it,
 * events[2] after the merge kernel (events[3] is not used) -- for timing each
 * kernel of the step on its own stream.  With events[1] given, the merge is
 * launched after it instead of overlapping the persistent kernel's tail. */
hp_status hp_cascade_decode_profiled(const void *plan_dev, const hp_plan_info *info, const void *q,
                                     int64_t q_sb, int64_t q_sh, float scale, void *out,
                                     hp_dtype out_dt, int64_t o_sb, int64_t o_sh, float *lse,
                                     int64_t lse_sb, void *ws, size_t ws_bytes, hp_stream_t stream,
                                     void *const *events);

/* ---------------------------------------------------------------------------
 * Decode loop: many steps over one tree whose private suffixes grow.
 *
 * Each decoding step appends one token per sequence to that sequence's
 * private suffix, and the next step attends over it (Hydragen, "Inter-Sequence
 * Batched Prefix Attention", on autoregressive decoding).  The shared nodes
 * do not change.  Hydragen's suffix kernel accepts suffix lengths that change
 * from step to step while the loop stays inside CUDA graphs ("Implementation
 * Details", attention primitives).  ChunkAttention keeps the kernel context
 * on the GPU and copies it again only when the tree's structure changes
 * ("Context Generation and GPU-CPU Coordination", lazy context copy).
 *
 * Here a loop plan is built once with a capacity per suffix.  Each
 * sequence's current suffix length lives in a device array,
 * suffix_len[B] (int32).  hp_cascade_append_kv writes one token and
 * increments the length; hp_cascade_decode_loop reads it.  Both are
 * graph-capturable, so a whole multi-step loop can be one CUDA graph.
 *
 * The tree's last level must hold exactly one node per sequence, the node
 * of sequence b covering only b: its suffix.  Its kv_len is the length at
 * plan time.  Its page list must hold ceil(capacity / page_size) valid page
 * ids, distinct from each other and from every page that another node of
 * the same pools uses.  hp_cascade_append_kv writes into those pages.
 * Hq / Hkv must be at most 16.
 * ------------------------------------------------------------------------- */

/* Bytes of the device plan buffer of a loop plan (host only, no CUDA calls
 * when desc->num_sms > 0); 0 on an invalid descriptor or capacity.
 * capacity: maximum suffix length, >= every suffix node's kv_len, >= 1. */
size_t hp_cascade_loop_plan_bytes(const hp_tree_desc *desc, int32_t capacity);

/* hp_cascade_plan for a decode loop: the same validation, work items and
 * upload, plus the suffixes' page lists for hp_cascade_append_kv.  The
 * suffix work items reach to `capacity`; at run time each one ends at the
 * sequence's current length.  A loop plan is used only through
 * hp_cascade_append_kv and hp_cascade_decode_loop (hp_cascade_decode returns
 * HP_ERR_ARG on it).  Waits for the upload, like hp_cascade_plan. */
hp_status hp_cascade_loop_plan(const hp_tree_desc *desc, int32_t capacity, void *plan_dev,
                               size_t plan_bytes, hp_plan_info *info, hp_stream_t stream);

/* Append one token per sequence: K and V rows k_new / v_new, bf16 [B][Hkv][d]
 * at k_new + b*kv_sb + h*kv_sh (element strides, multiples of 8; head
 * dimension contiguous; both 16-byte aligned).  Sequence b's token goes to
 * position suffix_len[b] of its suffix, in the page of that position.  Then
 * suffix_len[b] (device, int32 [B]) is incremented.
 * A length outside [0, capacity) writes nothing, leaves the length as it was
 * and sets HP_ERR_BOUNDS in the status word of ws (>= 256 bytes, the step's
 * workspace).  One launch, no allocation, graph-capturable. */
hp_status hp_cascade_append_kv(const void *plan_dev, const hp_plan_info *info, const void *k_new,
                               const void *v_new, int64_t kv_sb, int64_t kv_sh, int32_t *suffix_len,
                               void *ws, size_t ws_bytes, hp_stream_t stream);

/* hp_cascade_decode over a loop plan: sequence b's suffix is its first
 * suffix_len[b] tokens (device, int32 [B], read on the device after the
 * kernels before it in the stream have completed).  A length below the
 * suffix's plan-time kv_len (or 0), or above the capacity, sets HP_ERR_BOUNDS
 * in the status word; the step then still runs within the reserved pages,
 * but its results are not valid.  Otherwise as hp_cascade_decode. */
hp_status hp_cascade_decode_loop(const void *plan_dev, const hp_plan_info *info, const int32_t *suffix_len,
                                 const void *q, int64_t q_sb, int64_t q_sh, float scale, void *out,
                                 hp_dtype out_dt, int64_t o_sb, int64_t o_sh, float *lse, int64_t lse_sb,
                                 void *ws, size_t ws_bytes, hp_stream_t stream);

/* hp_cascade_append_kv followed by hp_cascade_decode_loop, in the two
 * launches of one step: the persistent kernel writes each sequence's new
 * token (k_new, v_new as in hp_cascade_append_kv) into its suffix pages just
 * before it loads that chunk, and attends over the first suffix_len[b] + 1
 * suffix tokens; the merge kernel then advances suffix_len[b] by one.  The
 * results, the pools and the lengths equal those of the two separate calls.
 * A length outside [0, capacity) sets HP_ERR_BOUNDS, writes nothing for
 * that sequence and keeps its length. */
hp_status hp_cascade_decode_append(const void *plan_dev, const hp_plan_info *info, int32_t *suffix_len,
                                   const void *k_new, const void *v_new, int64_t kv_sb, int64_t kv_sh,
                                   const void *q, int64_t q_sb, int64_t q_sh, float scale, void *out,
                                   hp_dtype out_dt, int64_t o_sb, int64_t o_sh, float *lse,
                                   int64_t lse_sb, void *ws, size_t ws_bytes, hp_stream_t stream);

/* Host-side description of a plan for inspection and tests: the (level, node,
 * seq_begin, seq_end, pass) context list in the order the pages list it --
 * shared nodes (more than one sequence; batched pass = 1) level by level,
 * then each sequence's private nodes in level order (pass = 0).  Writes at
 * most cap entries of 5 int32 each into out; returns the entry count, or -1
 * on an invalid descriptor. */
int32_t hp_cascade_contexts(const hp_tree_desc *desc, int32_t *out, int32_t cap);

/* Work-item counts of a plan for a descriptor: [0] tensor-core items,
 * [1] small-row items, [2] partial rows, [3] merge entries.  -1 on error. */
int32_t hp_cascade_plan_stats(const hp_tree_desc *desc, int64_t *stats4);

/* The work items of the plan for a descriptor (capacity 0: hp_cascade_plan's;
 * > 0: hp_cascade_loop_plan's), host only, for inspection and tests; no CUDA
 * calls when desc->num_sms > 0.  Each item is 11 int32: level, first
 * sequence, sequences, first KV head, KV heads, k0, k1 (node-relative keys
 * [k0, k1)), first partial row, CTA of the persistent kernel, tensor-core
 * role (1) or paged role (0), and the sequence whose length ends the item
 * in a loop plan (-1 otherwise).  Items are listed CTA by CTA, in the order
 * each CTA runs them.  Writes at most cap items into out (may be NULL);
 * returns the item count, or -1 on an invalid descriptor. */
int32_t hp_cascade_plan_items(const hp_tree_desc *desc, int32_t capacity, int32_t *out, int32_t cap);

/* The page ids each of those items carries in its CTA's record (host only,
 * as above), items in hp_cascade_plan_items' order: item i's key t (of its
 * level's node) is in page pages[offsets[i] + t / page_size - k0 / page_size].
 * offsets (n + 1 entries) and pages (at most cap written) may be NULL;
 * returns the total page count, or -1 on an invalid descriptor. */
int64_t hp_cascade_plan_item_pages(const hp_tree_desc *desc, int32_t capacity, int64_t *offsets,
                                   int32_t *pages, int64_t cap);

/* The merge table of the same plan (host only, as above): one row of
 * `stride` int32 per (sequence b, KV head), row b*Hkv + kvh, holding the
 * part count and then the partial row of each part for query head g = 0 of
 * the group (head g adds g).  Writes at most cap int32 into out (may be
 * NULL); returns the stride, or -1 on an invalid descriptor. */
int32_t hp_cascade_plan_merge_table(const hp_tree_desc *desc, int32_t capacity, int32_t *out, int64_t cap);

/* ---------------------------------------------------------------------------
 * Device status: reads and clears the status word of a workspace.  This call
 * synchronises `stream`.  Returns HP_OK, HP_ERR_BOUNDS, HP_ERR_DEVICE_TIMEOUT
 * or HP_ERR_CUDA.
 * ------------------------------------------------------------------------- */
hp_status hp_read_device_status(void *ws, hp_stream_t stream);

/* Failure detection tests only.  While enabled (non-zero), every
 * hp_cascade_decode* launch makes CTA 0 arm its first key tile's barrier
 * but issue no copy: its bounded waits (2 s each) run out, the CTA drains and
 * returns, and the step reports HP_ERR_DEVICE_TIMEOUT through the status word
 * (that step's results are not valid; later steps are correct).  A
 * process-wide switch, off by default; it never faults the GPU. */
void hp_test_withhold_first_tile(int32_t enable);

/* Library build information: the SM architecture compiled for (103 for
 * sm_103a) and the library ABI version. */
int32_t hp_build_arch(void);
int32_t hp_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* HP_H */
