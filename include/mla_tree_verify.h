/*
 * mla_tree_verify.h — C ABI of the GB300 (sm_103a) MLA tree-verify attention library.
 *
 * The operation is the speculative-decoding verify attention over a Multi-head Latent
 * Attention (MLA) KV cache, as described in
 *   "The Architecture of Capture Safety: Designing a CUDA Graph-Compatible Verify
 *    Kernel for SGLang" — section "The Design Emerges" (split-K flash decode with a
 *    fixed NSPLIT; prefix rows through kv_indices and draft rows through
 *    out_cache_loc; the raw custom_mask indexed inline through mask_indptr;
 *    prefix_len derived on the device from kv_indptr; a caller-preallocated
 *    workspace), section "Assumptions and Their Validity" (static buffers whose
 *    contents change between graph replays), section "Output Knowledge Created"
 *    (kv_indptr is int32, qo_indptr is int64);
 *   "The Plan Document: A Pivot Point in Custom CUDA Kernel Development" — section
 *    "Input Knowledge Required" (one compressed 512-dim latent shared by all heads).
 *
 * For request b (0 <= b < bs): P_b = kv_indptr[b+1]-kv_indptr[b] prefix keys,
 * T_b = qo_indptr[b+1]-qo_indptr[b] draft tokens, L_b = P_b + T_b key columns.
 * Key column c reads the 576-dim row kv_cache[slot(c)], where
 *   slot(c) = kv_indices[kv_indptr[b] + c]                for c <  P_b,
 *   slot(c) = out_cache_loc[qo_indptr[b] + c - P_b]       for c >= P_b.
 * Draft i of request b (query row r = qo_indptr[b] + i) sees every prefix column and
 * the draft column c >= P_b iff custom_mask[mask_indptr[b] + i*L_b + c] != 0.  For each
 * of the 64 heads h:
 *   s_c = sm_scale * <q[r,h,0:576], kv[slot(c),0:576]>
 *   out[r,h,0:512] = softmax over visible c of s_c, applied to kv[slot(c),0:512]
 *   lse[r,h] = ln sum over visible c of exp(s_c)
 * A row that sees no key gets out = 0 and lse = -inf.
 *
 * Every buffer is owned by the caller.  The library allocates nothing, never blocks
 * the host, never reads device memory from the host, and only enqueues kernels on the
 * given stream; the launch grids depend only on (bs, max_q_per_req) and on the
 * device's SM count.  A call can therefore be captured in a CUDA graph and replayed
 * after the caller rewrites the contents (not the addresses) of its buffers.
 */
#ifndef MLA_TREE_VERIFY_H_
#define MLA_TREE_VERIFY_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MLA_TV_HEADS 64   /* query heads (one shared latent KV head) */
#define MLA_TV_HEADS_TP8 8 /* the same call with 8 heads per token: a tensor-parallel shard
                              of 8 ranks ("The Plan Document", section "Assumptions and
                              Their Implications": the TP8 regime, 8 heads per rank) */
#define MLA_TV_D_QK 576   /* 512 latent + 64 rope dims per KV row and per query head */
#define MLA_TV_D_V 512    /* V is the first 512 dims of each KV row */
#define MLA_TV_NSPLIT 64  /* at most this many partial results per query token */
#define MLA_TV_MAX_Q_PER_REQ 4096

/* Return codes (0 = success; negative = nothing was enqueued unless stated). */
#define MLA_TV_OK 0
#define MLA_TV_ERR_NULL -1        /* a required pointer is NULL */
#define MLA_TV_ERR_HEADS -2       /* num_heads is neither 64 nor 8 */
#define MLA_TV_ERR_SHAPE -3       /* bs < 1, max_q_per_req outside [1, 4096], negative size,
                                     num_slots or total_q*64 above INT32_MAX */
#define MLA_TV_ERR_ALIGN -4       /* q/kv_cache/out not 16-byte, workspace not 256-byte aligned */
#define MLA_TV_ERR_WORKSPACE -5   /* workspace_bytes below mla_tree_verify_workspace_bytes() */
#define MLA_TV_ERR_LAUNCH -6      /* a kernel launch failed (cudaGetLastError); work may be
                                     partly enqueued */
#define MLA_TV_ERR_DEVICE -7      /* no current CUDA device, or it is not sm_103 */
#define MLA_TV_ERR_SCALE -8       /* sm_scale is not finite */
#define MLA_TV_ERR_STATIC_LIMIT -9 /* mla_tree_verify_static_ws(): the batch needs more
                                      than MLA_TV_STATIC_WS_BYTES of scratch */

/* Device-side error bits, written into the workspace header by the kernels instead of
 * trapping; read them with mla_tree_verify_read_device_status(). */
#define MLA_TV_DEV_BAD_SLOT 1u    /* a slot outside [0, num_slots): that key is skipped, as if
                                     masked */
#define MLA_TV_DEV_BAD_INDPTR 2u  /* kv_indptr/qo_indptr out of range, decreasing, or
                                     T_b > max_q_per_req: nothing is computed or written */
#define MLA_TV_DEV_BAD_MASK 4u    /* mask_indptr[b+1]-mask_indptr[b] != T_b*L_b or beyond
                                     mask_len: request b's rows get out = 0, lse = -inf */
#define MLA_TV_DEV_TIMEOUT 8u     /* a pipeline wait inside the split kernel gave up (bounded
                                     waits, never a hang): outputs are not valid */

/*
 * Bytes of workspace that mla_tree_verify() needs for a batch of at most bs requests
 * with at most max_q_per_req draft tokens each, on the current device.  The size
 * depends on the device's SM count (one partial slot per query token plus one per
 * split CTA, each holding 64 heads x (512 fp32 outputs + 1 fp32 lse), and a 4-byte
 * counter per query token), so query it on the device that will run the call.  Returns 0 for invalid arguments.
 */
size_t mla_tree_verify_workspace_bytes(int32_t bs, int32_t max_q_per_req, int32_t num_heads);

/*
 * Verify attention for one batch.
 *   q              bf16 [total_q, H, 576], contiguous, 16-byte aligned (device);
 *                  H = num_heads (64, or 8 for a tensor-parallel shard)
 *   kv_cache       bf16 [num_slots, 576], contiguous, 16-byte aligned (device); page size 1
 *   kv_indices     int32 [num_kv_indices] prefix slots, request after request (device)
 *   kv_indptr      int32 [bs+1] (device)
 *   out_cache_loc  int64 [total_q] slot of each draft token's own KV row (device)
 *   custom_mask    uint8 [mask_len] per-request row-major [T_b, L_b] blocks, nonzero =
 *                  visible; only the draft columns (c >= P_b) are read (device)
 *   mask_indptr    int64 [bs+1] offsets of those blocks (device)
 *   qo_indptr      int64 [bs+1] (device)
 *   sm_scale       softmax scale applied to q.k
 *   out            bf16 [total_q, H, 512], 16-byte aligned (device); rows
 *                  [qo_indptr[0], qo_indptr[bs]) are written, others are untouched
 *   lse            fp32 [total_q, H] natural-log log-sum-exp (device)
 *   workspace      device scratch of workspace_bytes bytes, 256-byte aligned, reused
 *                  across calls; calls that share one workspace must not overlap
 *   bs, max_q_per_req, num_heads (64, or 8: the kernel then fills its 64 columns with
 *                  the 8 heads of 8 consecutive draft tokens of a request), num_slots,
 *                  total_q (rows of q/out),
 *   num_kv_indices, mask_len: element counts of the arrays above, used by the device
 *                  to range-check every index it reads
 *   stream         the CUDA stream to enqueue on
 * Returns MLA_TV_OK or a negative MLA_TV_ERR_* code (checked on the host, before any
 * launch, except MLA_TV_ERR_LAUNCH).
 */
int mla_tree_verify(const void* q, const void* kv_cache, const int32_t* kv_indices,
                    const int32_t* kv_indptr, const int64_t* out_cache_loc,
                    const uint8_t* custom_mask, const int64_t* mask_indptr,
                    const int64_t* qo_indptr, float sm_scale, void* out, float* lse,
                    void* workspace, size_t workspace_bytes, int32_t bs, int32_t max_q_per_req,
                    int32_t num_heads, int64_t num_slots, int64_t total_q,
                    int64_t num_kv_indices, int64_t mask_len, cudaStream_t stream);

/*
 * Same computation as mla_tree_verify(), and in addition records the indices the
 * kernels used: slot_dump [sum_b L_b] int64 receives slot(c) of every key column
 * (request after request; -1 for a slot outside the pool) and vis_dump [mask_len]
 * uint8 receives, at the position of each mask entry, the visibility the kernel used
 * (1 for prefix columns).  For comparing gather and mask indexing bit for bit.
 */
int mla_tree_verify_debug(const void* q, const void* kv_cache, const int32_t* kv_indices,
                          const int32_t* kv_indptr, const int64_t* out_cache_loc,
                          const uint8_t* custom_mask, const int64_t* mask_indptr,
                          const int64_t* qo_indptr, float sm_scale, void* out, float* lse,
                          void* workspace, size_t workspace_bytes, int32_t bs,
                          int32_t max_q_per_req, int32_t num_heads, int64_t num_slots,
                          int64_t total_q, int64_t num_kv_indices, int64_t mask_len,
                          int64_t* slot_dump, uint8_t* vis_dump, cudaStream_t stream);

/*
 * Debug settings of mla_tree_verify_debug_ex().  (Not from the pages: test hooks for the
 * library's own failure handling and merge paths.)
 *   slot_dump, vis_dump  NULL, or the dumps of mla_tree_verify_debug() (both or neither)
 *   wait_limit_ns        limit of every bounded wait inside the split kernel; 0 means the
 *                        default of 2 s.  A wait that runs out sets MLA_TV_DEV_TIMEOUT, and
 *                        the kernel drains its copies and MMAs, frees TMEM and returns, so
 *                        the context stays usable (outputs of that call are not valid).
 *   merge_mode           which path merges a query token's partials.  MLA_TV_MERGE_AUTO:
 *                        as timing allows (the normal call).  MLA_TV_MERGE_NO_TMEM: always
 *                        the ticket path (every piece writes its partial; the last ticket
 *                        merges from the workspace).  MLA_TV_MERGE_PREFER_TMEM: the CTA
 *                        that computes a token's last piece waits up to 20 ms for the other
 *                        pieces and then merges its own piece straight from TMEM.  The
 *                        output bits are the same in every mode.  A token cut into more
 *                        than 16 pieces always merges through the workspace, in two levels
 *                        (groups of 8 pieces, then the group results).
 *   lanes                CTAs per lane group (0: the library's choice; else 1, 2, 4 or 8,
 *                        dividing the split grid, or MLA_TV_ERR_SHAPE).  The lanes of a
 *                        group work on different draft tokens of one request over the same
 *                        key tiles; the result is correct for any choice, and its bits
 *                        may differ between choices (the partials are cut differently).
 */
#define MLA_TV_MERGE_AUTO 0
#define MLA_TV_MERGE_NO_TMEM 1
#define MLA_TV_MERGE_PREFER_TMEM 2
typedef struct {
  int64_t* slot_dump;
  uint8_t* vis_dump;
  uint64_t wait_limit_ns;
  int32_t merge_mode;
  int32_t lanes;
} mla_tree_verify_debug_opts;

/* Same computation as mla_tree_verify() with the settings above; opts must not be NULL. */
int mla_tree_verify_debug_ex(const void* q, const void* kv_cache, const int32_t* kv_indices,
                             const int32_t* kv_indptr, const int64_t* out_cache_loc,
                             const uint8_t* custom_mask, const int64_t* mask_indptr,
                             const int64_t* qo_indptr, float sm_scale, void* out, float* lse,
                             void* workspace, size_t workspace_bytes, int32_t bs,
                             int32_t max_q_per_req, int32_t num_heads, int64_t num_slots,
                             int64_t total_q, int64_t num_kv_indices, int64_t mask_len,
                             const mla_tree_verify_debug_opts* opts, cudaStream_t stream);

/*
 * Same computation as mla_tree_verify(), and in addition records three caller-created
 * CUDA events on `stream`: events[0] before the planner kernel, events[1] between the
 * planner and the split kernel, events[2] after the split kernel (which also merges
 * the partials).  cudaEventElapsedTime over consecutive pairs gives each kernel's
 * device time.  The event between the two kernels keeps the split kernel's prologue
 * from overlapping the planner, so the sum can exceed the time of an unprofiled call.
 * The events are recorded as external events, so a captured call leaves event-record
 * nodes in the graph and the times can be read after each replay.  Returns
 * MLA_TV_ERR_NULL if an event is missing.
 */
int mla_tree_verify_profiled(const void* q, const void* kv_cache, const int32_t* kv_indices,
                             const int32_t* kv_indptr, const int64_t* out_cache_loc,
                             const uint8_t* custom_mask, const int64_t* mask_indptr,
                             const int64_t* qo_indptr, float sm_scale, void* out, float* lse,
                             void* workspace, size_t workspace_bytes, int32_t bs,
                             int32_t max_q_per_req, int32_t num_heads, int64_t num_slots,
                             int64_t total_q, int64_t num_kv_indices, int64_t mask_len,
                             cudaEvent_t* events, cudaStream_t stream);

/*
 * One-time per-device set-up (kernel attributes for large shared memory, and the device
 * address of the scratch array of mla_tree_verify_static_ws()).  Called automatically
 * by the first call on each device; call it yourself before capturing a graph.
 * Returns MLA_TV_OK or MLA_TV_ERR_DEVICE.
 */
int mla_tree_verify_prepare(void);

/*
 * Copies the device error bits (MLA_TV_DEV_*) of the last call that used `workspace`
 * into *flags.  Synchronises `stream`: a diagnostic, not for use inside a capture.
 */
int mla_tree_verify_read_device_status(const void* workspace, uint32_t* flags,
                                       cudaStream_t stream);

/* Number of CTAs of the split kernel on the current device (its SM count). */
int32_t mla_tree_verify_split_grid(void);

/*
 * mla_tree_verify_static_ws — the same computation as mla_tree_verify(), for callers
 * that cannot allocate device memory.  (The paper has no counterpart to this entry
 * point.)  Such callers have no device allocator of their own, or may not call one on
 * this path: an engine that passes raw tensor pointers but keeps its memory pool
 * private, or C code for which cudaMalloc is ruled out after start-up because it can
 * synchronise the device and is not permitted during CUDA graph capture.
 *
 * Instead of a caller-provided workspace, this call uses one scratch array of
 * MLA_TV_STATIC_WS_BYTES (64 MiB) built into the library as a device variable; every
 * GPU that loads the library holds it until the process exits.  Batches whose
 * scratch (mla_tree_verify_workspace_bytes(bs, max_q_per_req, 64)) exceeds that size
 * are rejected with MLA_TV_ERR_STATIC_LIMIT before anything is enqueued; on a
 * 152-SM GB300 this admits bs * (ceil(max_q_per_req / g) + 7) up to about 350, with
 * g = 1 at 64 heads and 8 at 8 heads (at 64 heads and 16 drafts, 15 requests).  The
 * call allocates nothing.  mla_tree_verify_prepare(), or else the first call on each
 * device, looks up the array's device address (once, with that device current); make
 * one of them before any stream capture.  All calls on a device share the array and it keeps the previous
 * call's contents (each call rewrites what it reads before reading it), so calls
 * that can overlap on the GPU race with each other: order them on one stream.
 * Arguments and return codes are those of mla_tree_verify(), without workspace and
 * workspace_bytes.
 */
#define MLA_TV_STATIC_WS_BYTES (64u << 20)
int mla_tree_verify_static_ws(const void* q, const void* kv_cache, const int32_t* kv_indices,
                              const int32_t* kv_indptr, const int64_t* out_cache_loc,
                              const uint8_t* custom_mask, const int64_t* mask_indptr,
                              const int64_t* qo_indptr, float sm_scale, void* out, float* lse,
                              int32_t bs, int32_t max_q_per_req, int32_t num_heads,
                              int64_t num_slots, int64_t total_q, int64_t num_kv_indices,
                              int64_t mask_len, cudaStream_t stream);

/*
 * mla_tree_verify_kv_gather — the KV defragmentation step: copies the batch's scattered
 * page_size=1 prefix rows into consecutive rows and rewrites their indices, so that a
 * later verify call reads contiguous memory.  ("The Plan Document: A Pivot Point in
 * Custom CUDA Kernel Development", sections "Context: The Bottleneck That Demanded a
 * Custom Kernel" (K/V defragmentation) and "Output Knowledge Created" (Phase 3); the
 * pages give no algorithm, and this is the plainest reading: a gather-copy in index
 * order.)
 *
 * For every index entry i in [kv_indptr[0], kv_indptr[bs]), with j = i - kv_indptr[0]:
 *   dst row j          = kv_cache row kv_indices[i]   (576 bf16, bit for bit)
 *   new_indices[i]     = dst_slot0 + j
 * Request b's rows land, in order, at dst rows [kv_indptr[b] - kv_indptr[0],
 * kv_indptr[b+1] - kv_indptr[0]).  With dst = the pool's row dst_slot0 (a free region of
 * the same pool) and kv_indices replaced by new_indices, mla_tree_verify() reads the
 * same rows in the same order and returns bit-identical results.
 *
 *   kv_cache     bf16 [num_slots][576], 16-byte aligned (read only)
 *   kv_indices   int32 [num_kv_indices] (read only); entries [kv_indptr[0], kv_indptr[bs])
 *                are copied, and kv_indptr[bs] > num_kv_indices is an argument error
 *                flagged on the device (MLA_TV_GATHER_BAD_ARGS, nothing copied)
 *   kv_indptr    int32 [bs + 1], device (read only; read on the device, so the call is
 *                capturable)
 *   dst          bf16 [dst_rows][576], 16-byte aligned; must not overlap any row it
 *                copies from (overlap is not detected and leaves the copied rows undefined)
 *   dst_slot0    the slot number that dst row 0 carries; dst_slot0 + dst_rows <= INT32_MAX
 *   new_indices  int32, kv_indptr[bs] entries; entries before kv_indptr[0] are untouched
 *   status       device uint32 the caller zeroes once; the kernel ORs in
 *                MLA_TV_GATHER_BAD_SLOT (a slot outside [0, num_slots): its row is
 *                written as zeros) and MLA_TV_GATHER_BAD_ARGS (kv_indptr[0] < 0,
 *                kv_indptr[bs] < kv_indptr[0], kv_indptr[bs] > num_kv_indices, or more rows
 *                than dst_rows: nothing is copied)
 *
 * The caller owns every buffer.  Nothing is allocated or synchronised; one kernel is
 * enqueued on `stream` (a fixed grid of 4 CTAs per SM).  Returns MLA_TV_OK, or before
 * enqueuing anything MLA_TV_ERR_NULL / _SHAPE (bs < 1, num_slots outside [1, INT32_MAX],
 * num_kv_indices < 0, dst_rows < 0, dst_slot0 < 0 or dst_slot0 + dst_rows > INT32_MAX) / _ALIGN / _DEVICE, or
 * MLA_TV_ERR_LAUNCH.
 */
#define MLA_TV_GATHER_BAD_SLOT 1u
#define MLA_TV_GATHER_BAD_ARGS 2u
int mla_tree_verify_kv_gather(const void* kv_cache, int64_t num_slots, const int32_t* kv_indices,
                              int64_t num_kv_indices, const int32_t* kv_indptr, int32_t bs, void* dst, int64_t dst_rows,
                              int32_t dst_slot0, int32_t* new_indices, uint32_t* status,
                              cudaStream_t stream);

/* Static description of a return code. */
const char* mla_tree_verify_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* MLA_TREE_VERIFY_H_ */
