/*
 * avsg.h -- C interface of the GB300 sparse-KV reuse decode step.
 *
 * The operation (AVSG page, arxivdaily 2609.37538, English abstract): dynamic
 * sparse attention selects, per decode step, a subset of token ids of each
 * (request, kv-head); the full KV cache lives in host memory.  This library
 * keeps a device (HBM) buffer of B slots per (request, kv-head) *unit* and, on
 * every step,
 *   1. matches the selected ids against the ids resident in the buffer,
 *   2. reserves victim slots for the ids that are not resident (bucketed LRU,
 *      Spin page "Unifying Sparse Attention with Hierarchical Memory for
 *      Scalable Long-Context LLM Serving", section 2B),
 *   3. copies only those missing KV rows from host memory into their slots,
 *      spreading the copy evenly over the GPU's SMs,
 *   4. runs decode attention of every query head over the selected rows.
 * Multi-token prediction: with n_tok > 1 query tokens per step, one shared
 * reservation covers the union of the tokens' selections (same abstract).
 *
 * Within a step the copy of the misses (bound by the host link) overlaps the
 * reservation and the attention over the selected rows that were already
 * resident: the library runs the gather (into a staging area), the
 * reservation, the hash-table update and the move of the previous step's
 * staged rows into their slots on three internal streams, forked from and
 * joined back into the caller's stream with events.  A step's missed rows
 * reach their slots during the next step (its hits on them read the staged
 * copy); avsg_read_state, avsg_set_budget and avsg_clear_error move them
 * first, so every entry point sees the buffer of the step-by-step order.
 *
 * Reservation order (the pages give no formula; this is the reading the
 * library implements): empty slots first, by ascending slot index; then the
 * slots not selected in this step, by bucket min(63, t - last_step) from 63
 * down to 1, ties by ascending slot index.  The i-th missing id in ascending
 * id order takes the i-th reserved slot.  Every selected id ends the step
 * with last_step = t.  The outcome is deterministic: slot maps, hit flags,
 * tags and buffer rows are identical run to run.
 *
 * Threading: a handle is used by one host thread and one CUDA stream at a
 * time.  All device work of a step is enqueued on the caller's stream with no
 * host synchronisation; avsg_get_stats and avsg_read_state synchronise.
 */
#ifndef AVSG_H_
#define AVSG_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define AVSG_VERSION 1

/* Return codes.  0 is success; every error is negative. */
#define AVSG_OK 0
#define AVSG_ERR_INVALID_ARG (-1)   /* null pointer, bad size or bad config field */
#define AVSG_ERR_CAPACITY (-2)      /* n_tok * k exceeds the buffer slots, or k > max_select */
#define AVSG_ERR_CUDA (-3)          /* a CUDA runtime call failed; see avsg_cuda_error */
#define AVSG_ERR_BAD_SELECTION (-4) /* device: id outside [0, num_entries), or repeated in one token */
#define AVSG_ERR_TIMEOUT (-5)       /* device: a bounded wait gave up */
#define AVSG_ERR_BAD_STEP (-6)      /* t is negative or not larger than the previous step's t */
#define AVSG_ERR_UNSUPPORTED (-7)   /* shape without a compiled attention kernel */
#define AVSG_ERR_LATCHED (-8)       /* a device error is pending; call avsg_clear_error */
#define AVSG_ERR_INTERNAL (-9)      /* device: an index check of the bounds-checked build failed */

/* avsg_config.flags */
#define AVSG_FLAG_NO_REUSE 1u /* no buffer reuse: copy every selected row every step */
/* The miss gather is assigned by request: one CTA copies all the misses of one
 * request (its kv-heads' units), the assignment the AVSG page measures its even
 * split against.  Default: the misses of all units are split evenly over the
 * gather's CTAs.  Results are identical either way; only the copy's speed
 * differs.  Needs a shape with a tensor-core attention (else
 * AVSG_ERR_UNSUPPORTED at create); ignored with AVSG_FLAG_NO_REUSE. */
#define AVSG_FLAG_REQUEST_GATHER 2u

typedef struct avsg_handle_s* avsg_handle;

/*
 * Shape of one handle.  Units are ordered request-major: unit = r * H + h.
 * Host K is laid out [R][H][num_entries][entry_tokens][head_dim] bf16, host V
 * [R][H][num_entries][entry_tokens][v_dim] bf16: one entry of a unit is a
 * contiguous row of entry_tokens tokens (a head-wise page when > 1, Spin page
 * section 2B "head-wise physical pages").  The first initial_entries entries
 * of every unit are live at create (all num_entries when 0); selected ids must
 * be below the live count, which avsg_append raises by one per call.
 */
typedef struct avsg_config {
  int32_t num_requests;        /* R >= 1 */
  int32_t num_kv_heads;        /* H >= 1 */
  int32_t q_per_kv;            /* G: query heads per kv-head (1, 2, 4, 8 or 16) */
  int32_t entry_tokens;        /* tokens per entry: 1 (token) .. 64 (page) */
  int32_t head_dim;            /* D: K row width, multiple of 8 */
  int32_t v_dim;               /* Dv: V row width (== head_dim when kv_shared) */
  int32_t kv_shared;           /* 1: V is the K row itself (latent cache) */
  int32_t reserved0;           /* must be 0 */
  int64_t num_entries;         /* entries per unit the host arrays hold, 1 .. 2^31 - 1 */
  int32_t buffer_slots;        /* B: device slots per unit */
  int32_t max_select;          /* largest k accepted by avsg_step */
  int32_t max_tokens_per_step; /* largest n_tok (1 .. 8) */
  float softmax_scale;         /* 0 selects 1/sqrt(head_dim) */
  uint32_t flags;              /* AVSG_FLAG_* */
  int32_t initial_entries;     /* entries live at create, 0 .. num_entries (0: all of
                                  them); avsg_append adds one per unit per call */
} avsg_config;

typedef struct avsg_stats {
  uint64_t steps;           /* steps enqueued (host count) */
  uint64_t selected;        /* selected ids, summed over units and tokens */
  uint64_t unique_selected; /* distinct ids per unit and step (the union), summed */
  uint64_t hits;            /* distinct selected ids that were resident */
  uint64_t misses;          /* distinct selected ids copied from host */
  uint64_t miss_bytes;      /* host bytes copied into the buffer */
  int32_t device_error;     /* 0, or the AVSG_ERR_* code latched on the device */
  int32_t error_unit;       /* unit of that error, or -1 */
  int32_t error_position;   /* flat position (token * k + j) of that error, or -1 */
  int32_t reserved;
} avsg_stats;

typedef struct avsg_info {
  uint64_t device_bytes;    /* device memory held by the handle */
  int32_t hash_capacity;    /* per-unit open-addressing table entries */
  int32_t miss_set_capacity;/* per-unit per-step miss-set entries */
  int32_t attn_splits;      /* split-K partitions per (unit, token) at max_select */
  int32_t gather_ctas;      /* CTAs of the miss gather */
  int32_t num_sms;          /* SMs of the device */
  int32_t host_registered;  /* 1 if create registered the host KV itself */
} avsg_info;

/*
 * Per-kernel device time (ms), accumulated over the steps enqueued while
 * profiling was on: CUDA events recorded just before and after each kernel on
 * the stream it runs on (the events themselves keep consecutive kernels from
 * overlapping their launches).  launches[i] counts the timed launches.
 */
#define AVSG_KERNEL_MATCH 0
#define AVSG_KERNEL_RESERVE 1
#define AVSG_KERNEL_GATHER 2
#define AVSG_KERNEL_ATTENTION 3      /* single pass, or the pass over hit rows */
#define AVSG_KERNEL_ATTENTION_MISS 4 /* pass over miss rows */
#define AVSG_KERNEL_COMMIT 5         /* hash-table update */
#define AVSG_KERNEL_FINISH 6         /* reserved (the miss pass merges the two passes) */
#define AVSG_KERNEL_PLACE 7          /* staged missed rows into their slots */
#define AVSG_NUM_KERNELS 8
typedef struct avsg_kernel_times {
  double ms[AVSG_NUM_KERNELS];
  uint64_t launches[AVSG_NUM_KERNELS];
} avsg_kernel_times;

/*
 * avsg_create -- build a handle.
 *   cfg     : shape (copied).
 *   host_k  : host K rows, layout above; owned by the caller, must outlive the
 *             handle and must not change while steps run.
 *   host_v  : host V rows, or NULL when cfg->kv_shared.
 *   out     : receives the handle.
 * Host memory already allocated mapped (cudaHostAlloc(Mapped) or
 * avsg_host_alloc) is used in place; any other memory is registered with
 * cudaHostRegister(Mapped | ReadOnly) and unregistered by avsg_destroy.
 * Device memory is allocated on the current device; the buffer starts empty.
 * Errors: INVALID_ARG, CAPACITY (max_tokens_per_step * max_select > buffer_slots),
 * UNSUPPORTED, CUDA.  On error *out is NULL and nothing is held.
 */
int avsg_create(const avsg_config* cfg, const void* host_k, const void* host_v,
                avsg_handle* out);

/* avsg_destroy -- synchronise, free device memory, unregister host memory if
 * create registered it.  NULL is accepted. */
int avsg_destroy(avsg_handle h);

/*
 * avsg_step -- one decode step (one MTP iteration when n_tok > 1).
 *   t          : step index, >= 0 and strictly larger than the previous call's.
 *   n_tok, k   : query tokens (1 .. max_tokens_per_step) and selected entries
 *                per token (0 .. max_select); n_tok * k <= buffer_slots.
 *   d_sel      : device int32 [R][H][n_tok][k], ids in [0, num_entries),
 *                distinct within one token's list (may repeat across tokens).
 *   d_q        : device fp32 [R][H][n_tok][G][D].
 *   d_out      : device fp32 [R][H][n_tok][G][Dv]; attention of each query
 *                head over the rows of its token's selected entries
 *                (softmax(scale * q.K) V, fp32 accumulation); zeros when k = 0.
 *   d_slot_map : device int32 [R][H][n_tok][k] or NULL: buffer slot of each
 *                selected id, input order.
 *   d_hit      : device uint8 [R][H][n_tok][k] or NULL: 1 if the id was
 *                resident before the step.
 *   stream     : cudaStream_t (NULL = legacy default stream).
 * Host-side errors (INVALID_ARG, CAPACITY, BAD_STEP, LATCHED) change nothing.
 * Device-detected errors (BAD_SELECTION) are latched before any buffer state
 * changes: the rest of the step, and every later step, does nothing on the
 * device until avsg_clear_error; avsg_get_stats reports them.
 * With AVSG_FLAG_NO_REUSE the buffer is bypassed: every selected row is copied
 * to a staging area and d_slot_map receives the staging index (tok * k + j),
 * d_hit zeros; ids are range-checked but repeats are not rejected.
 */
int avsg_step(avsg_handle h, int32_t t, int32_t n_tok, int32_t k, const int32_t* d_sel,
              const float* d_q, float* d_out, int32_t* d_slot_map, uint8_t* d_hit,
              void* stream);

/*
 * avsg_step_host -- avsg_step with HOST buffers (same shapes).  Copies the
 * selection and queries to device staging owned by the handle, runs the step,
 * and copies d_out (and the slot map / hit flags when non-NULL) back, all
 * enqueued on `stream`; the results are valid after the stream synchronises.
 * Pinned host buffers make the copies asynchronous.
 */
int avsg_step_host(avsg_handle h, int32_t t, int32_t n_tok, int32_t k, const int32_t* h_sel,
                   const float* h_q, float* h_out, int32_t* h_slot_map, uint8_t* h_hit,
                   void* stream);

/*
 * Offload of a decode step's new KV (Spin page, section 2A, the Offload
 * operation): writes one new entry per unit into the host arrays at entry
 * index `live` (the current live count) and makes it selectable from the next
 * step on.  d_k: device bf16 [R][H][entry_tokens * head_dim]; d_v: device bf16
 * [R][H][entry_tokens * v_dim], NULL when kv_shared.  One strided copy per
 * array, device to host, enqueued on `stream` (ordered before later steps on
 * that stream); the buffer is not touched (a new entry is a miss until it is
 * selected).  For paged entries, a page is appended once it is full.
 * Works the same with AVSG_FLAG_NO_REUSE (both paths read host rows by id).
 * Returns CAPACITY when all num_entries entries are live, INVALID_ARG for
 * NULL rows, CUDA if the copy cannot be enqueued.
 */
int avsg_append(avsg_handle h, const void* d_k, const void* d_v, void* stream);

/*
 * Buffer elasticity (Spin page, section 2B): the buffer of each unit is sized
 * per step, split into mandatory slots (the current step's selection) and
 * buffer slots kept for temporal locality, under a system-wide budget.
 * avsg_set_budget gives every unit u a budget of usable slots, slots_per_unit
 * (host int32 [R][H]), each in 1 .. buffer_slots; it applies from the next
 * step on (enqueued on `stream`).  Entries held in slots at or above a lowered
 * budget are dropped (a later selection of them is a miss); the reservation
 * takes only slots below the budget.  A step needs n_tok * k <= every unit's
 * budget (else CAPACITY).  At create every budget is buffer_slots; avsg_reset
 * keeps the budgets.  Not available with AVSG_FLAG_NO_REUSE (UNSUPPORTED).
 */
int avsg_set_budget(avsg_handle h, const int32_t* slots_per_unit, void* stream);

/*
 * A planner for avsg_set_budget (host only, no handle): splits total_slots over
 * num_units units, each first given `mandatory` slots (the largest n_tok * k
 * it will run), the rest in proportion to weights[u] >= 0 (equal shares when
 * weights is NULL or all zero; the remainder of an equal split goes to the
 * lowest units), each capped at max_slots (buffer_slots).  Slots above a cap
 * stay unassigned.  out: host int32 [num_units].  Returns CAPACITY when
 * total_slots < num_units * mandatory, INVALID_ARG for bad arguments.
 */
int avsg_plan_budget(int64_t total_slots, int32_t num_units, int32_t mandatory, int32_t max_slots,
                     const float* weights, int32_t* out);

/* avsg_get_stats -- synchronise the last stream used and read the counters. */
int avsg_get_stats(avsg_handle h, avsg_stats* out);

/* avsg_info -- static facts about the handle. */
int avsg_get_info(avsg_handle h, avsg_info* out);

/*
 * avsg_read_state -- synchronise and copy one unit's buffer state to host:
 *   tag [B] int32 (resident id or -1), last_step [B] int32 (-1 when never
 *   used), k_rows [B][entry_tokens * D] bf16, v_rows [B][entry_tokens * Dv]
 *   bf16 (NULL when kv_shared).  Any output may be NULL.
 */
int avsg_read_state(avsg_handle h, int32_t unit, int32_t* tag, int32_t* last_step,
                    void* k_rows, void* v_rows);

/* avsg_reset -- empty every buffer, forget the last t, zero the counters
 * (enqueued on `stream`). */
int avsg_reset(avsg_handle h, void* stream);

/* avsg_clear_error -- synchronise, drop a latched device error and the
 * per-step scratch it left; the buffer state is as before the failed step. */
int avsg_clear_error(avsg_handle h);

/* avsg_profile -- enable (1) / disable (0) per-kernel event timing; enabling
 * zeroes the accumulated times. avsg_profile_read synchronises and reads. */
int avsg_profile(avsg_handle h, int32_t enable);
int avsg_profile_read(avsg_handle h, avsg_kernel_times* out);

/*
 * avsg_attention_noalloc -- the attention of avsg_step over rows the caller
 * already holds on the device, allocating nothing.  The pages have no
 * counterpart: this exists for callers that cannot call cudaMalloc (code
 * running inside another framework's memory pool or allocator budget, or a
 * serving process that must not allocate once it runs).
 *   d_k_rows   : device bf16 [num_units][rows_per_unit][entry_tokens][head_dim].
 *   d_v_rows   : device bf16 [num_units][rows_per_unit][entry_tokens][v_dim],
 *                ignored (may be NULL) when kv_shared (V is the K row).
 *   d_index    : device int32 [num_units][n_tok][k], row of each selected
 *                entry, each in [0, rows_per_unit).  Repeats within one
 *                (unit, token) list are not detected: such a row counts once
 *                per occurrence (avsg_step rejects them).
 *   d_q, d_out : as in avsg_step.  softmax_scale 0 selects 1/sqrt(head_dim).
 * Shapes: those avsg_create accepts for attention; num_units <= 4096 and
 * k <= rows_per_unit (AVSG_ERR_CAPACITY beyond), n_tok <= 8.
 * Scratch: a fixed 8 MiB device array inside the library, held by every GPU
 * that loads it until the process exits.  The first call on a device looks
 * up that array's address (cudaGetSymbolAddress); make the first call before
 * any stream capture.  Every call shares the array and clears what must start
 * at zero; calls that overlap on the GPU race, so serialise them.
 * An index outside [0, rows_per_unit) makes the call fill d_out with NaN.
 * Returns after enqueueing on `stream`.  The argument errors (INVALID_ARG,
 * CAPACITY, UNSUPPORTED) are found before anything is enqueued and change
 * nothing; after AVSG_ERR_CUDA part of the work may have been enqueued and
 * d_out is undefined.
 */
int avsg_attention_noalloc(int32_t num_units, int32_t rows_per_unit, int32_t q_per_kv,
                           int32_t head_dim, int32_t v_dim, int32_t entry_tokens,
                           int32_t kv_shared, int32_t n_tok, int32_t k, const void* d_k_rows,
                           const void* d_v_rows, const int32_t* d_index, const float* d_q,
                           float* d_out, float softmax_scale, void* stream);

/* Pinned, mapped, portable host memory for the KV cache (cudaHostAlloc). */
int avsg_host_alloc(size_t bytes, void** out);
int avsg_host_free(void* p);

/*
 * avsg_read_rows -- a measurement aid: reads n rows at scattered positions and
 * discards them, to measure the ceiling of the step's row reads.  The
 * attention reads the selected entries' rows from slots scattered over the
 * device buffer, and the miss gather reads the missed entries' rows from ids
 * scattered over the host store (AVSG page, arxivdaily 2609.37538, English
 * abstract: only the selected entries are read; only the misses cross the
 * host link); the rate of this read alone, at the same row size, bounds both.
 *   src      : rows [num_rows][row_bytes], device memory or the device pointer
 *              of mapped host memory; 16-byte aligned.
 *   row_bytes: a multiple of 16.
 *   d_idx    : device int32 [n], the rows to read; an index outside
 *              [0, num_rows) is skipped.
 *   ctas     : grid size, 0 for 4 per SM.
 *   d_sink   : device uint32 the kernel may write (it practically never does).
 * Enqueued on `stream`; INVALID_ARG for bad arguments, CUDA if the launch fails.
 */
int avsg_read_rows(const void* src, int64_t num_rows, int64_t row_bytes, const int32_t* d_idx,
                   int64_t n, int32_t ctas, uint32_t* d_sink, void* stream);

/* Error text, and the cudaError_t behind the last AVSG_ERR_CUDA of a handle. */
const char* avsg_strerror(int code);
int avsg_cuda_error(avsg_handle h);

#ifdef __cplusplus
}
#endif

#endif /* AVSG_H_ */
