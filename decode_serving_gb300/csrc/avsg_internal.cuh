// Internal declarations shared by the kernels and the C interface.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "avsg.h"

namespace avsg {

constexpr int32_t kEmpty = -1;                 // tag / hash key of an empty cell
constexpr int32_t kTomb = -2;                  // hash key of an erased cell
constexpr unsigned long long kMissEmpty = ~0ull;
constexpr int kOrders = 64;                    // reservation classes 0..63
constexpr int kNotCandidate = 255;
constexpr int kMaxTokens = 8;
constexpr int kCountsPerPair = 8;              // arrival counters per (unit, token)
constexpr int kMatchCluster = 8;               // match: one cluster of CTAs per unit
constexpr int kMatchThreads = 256;             // threads per match CTA
constexpr int kMatchPerThread = 4;             // selected ids per match thread (n_tok * k <= 8192)
constexpr size_t kMatchSmemMax = 200 * 1024;   // match's part of the miss set + hit bitmaps

// First device error of a step; later kernels of the step (and later steps)
// see a non-zero code and return before touching any state.
struct DevErr {
  int32_t code, unit, pos, aux;
};

struct DevCounters {
  unsigned long long hits, misses;
};

// One miss to copy: host row `id` of `unit` into buffer slot `slot`, which
// held `old_id` (kEmpty if none) before this step; `cell` is the id's
// miss-set cell (and its row in the staging area); bit j of `tokens` is set
// when query token j selected the id.
struct GatherDesc {
  int32_t unit, id, slot, old_id, cell, tokens, pad1, pad2;
};

// Everything a kernel needs about a handle: sizes and device pointers.
// Per-step inputs and outputs.  The step's first kernel receives them by
// value and stores them at DeviceState::io; the kernels after it read them
// there (after their grid-dependency wait).  A step captured as a CUDA graph
// is thus re-pointed by updating the parameters of one kernel node.
struct StepIO {
  const int32_t* sel;
  const float* q;
  float* out;
  int32_t* slot_map;
  uint8_t* hit;
  int32_t t;
  int32_t live;                    // entries per unit selectable this step (ids below it)
  int32_t parity;                  // 0 / 1 alternating by step: which half of the per-step
                                   // staging and descriptor arrays this step writes
  uint32_t seq;                    // steps since create / reset (parity = seq & 1)
};

struct DeviceState {
  int32_t U, B, G, D, DV, ET;      // units, slots per unit, q/kv, widths, tokens/entry
  int64_t L;                       // entries per unit
  int32_t HS, hs_shift;            // hash capacity (pow2) and 32 - log2(HS)
  int32_t MS, ms_shift;            // miss-set capacity (pow2) and 32 - log2(MS)
  int32_t max_union;               // max_tokens_per_step * max_select
  int32_t HW, HT;                  // hit bitmaps: 32-slot words per token, token rows per unit
  int32_t kv_shared;
  StepIO* io;                      // this step's inputs and outputs (see StepIO)
  float* qbuf;                     // [U][n_tok][G][D] this step's q, copied by match
  int64_t ek, ev;                  // bytes of one entry's K row / V row (ev 0 if shared)
  const unsigned char* host_k;     // mapped host KV (device-visible pointers)
  const unsigned char* host_v;
  unsigned char* kbuf;             // [U][B][ek]
  unsigned char* vbuf;             // [U][B][ev]
  unsigned char* kstage;           // [2][U][MS][ek] missed rows by miss-set cell (staged
                                   // gather), one half per step parity
  unsigned char* vstage;           // [2][U][MS][ev]
  int32_t* tag;                    // [U][B] resident id or kEmpty
  int32_t* last;                   // [U][B] step of last selection, -1 never
  uint32_t* hitbits;               // [U][HT][HW] this step's hit slots per token (written by match)
  int4* htab;                      // [U][HS] {key, slot, seq, cell}: seq and cell as in pend
  int32_t* hused;                  // [U] non-empty hash cells (live + erased)
  unsigned long long* mset;        // [U][MS] {id | token bits << 32}: this step's miss set
                                   // (two sets alternate by step; each is empty when its step starts)
  int32_t* hslot;                  // [U][n_tok][k] slot of each selected id if it was a hit,
                                   // else -2 - its miss-set cell (-1 if it has none)
  int32_t* mslot;                  // [U][MS] slot reserved for the miss in that cell
  GatherDesc* desc;                // [2][U * max_union]     (halves by step parity)
  int32_t* desc_count;             // [2]
  int32_t* gather_next;            // [1] chunks of miss-set cells handed to the gather (zeroed by match)
  int32_t* dbase;                  // [2][U] first descriptor of the unit that step
  int32_t* dcount;                 // [2][U] descriptors of the unit that step (0: none)
  float* part;                     // split-K partials
  int32_t* part_count;             // [U][max_tokens][8] arrival counters, 0 between steps
  DevCounters* counters;           // [U] distinct hits / misses, summed over steps
  DevErr* err;
  int32_t* budget;                 // [U] usable slots per unit (buffer elasticity), <= B
  // Deferred place (two-pass pipeline): a step's missed rows reach their
  // slots during the next step, so that step's hits on them read the staged
  // copy.  pend[u][slot] = (seq of the step that reserved the slot) << 32 |
  // its miss-set cell; the hash-table update copies it into the id's cell,
  // where match finds it in the window it already read (pend itself is read
  // only to rebuild the table).  stage_entry0 = entry index, counted from
  // kbuf (and from vbuf: the staging area follows each buffer at the same
  // distance), of the first staged entry.  deferred = 0: no pend, and the
  // hash cells' seq stays -1 (the other pipelines).
  unsigned long long* pend;
  int64_t stage_entry0;
  int32_t deferred;
  // late_commit = 1 (the overlapped pipelines, where no kernel of the step
  // reads them before the hash-table update): the update, not the
  // reservation, writes the reserved slots' new tags and resolves the slot
  // map's miss entries, so the reservation that the miss pass waits for
  // keeps only what that pass and the place need.
  int32_t late_commit;
};

// The per-step arrays of one parity.
struct StepBufs {
  GatherDesc* desc;
  int32_t* desc_count;
  int32_t* dbase;
  int32_t* dcount;
  unsigned char* kstage;
  unsigned char* vstage;
};
__host__ __device__ __forceinline__ StepBufs step_bufs(const DeviceState& s, int parity) {
  const size_t half = (size_t)s.U * s.MS;
  StepBufs b;
  b.desc = s.desc + (size_t)parity * s.U * s.max_union;
  b.desc_count = s.desc_count + parity;
  b.dbase = s.dbase + (size_t)parity * s.U;
  b.dcount = s.dcount + (size_t)parity * s.U;
  b.kstage = s.kstage ? s.kstage + (size_t)parity * half * s.ek : nullptr;
  b.vstage = s.vstage ? s.vstage + (size_t)parity * half * (s.ev ? s.ev : s.ek) : nullptr;
  return b;
}

// The slot value the hit pass reads for a hit on `slot` at step `seq`, from
// the id's hash cell {key, slot, mseq, mcell}: the slot itself, or, when the
// previous step reserved it (mseq == seq - 1: its row is still in that
// step's half of the staging area until the deferred place), the staged
// entry expressed as a slot of unit u counted from kbuf.
__device__ __forceinline__ int32_t hit_row_slot(const DeviceState& s, int u, int32_t slot,
                                                int32_t mseq, int32_t mcell, uint32_t seq) {
  if (!s.deferred || seq == 0 || mseq != (int32_t)(seq - 1) || mcell < 0) return slot;
  const int64_t e = s.stage_entry0 + (int64_t)((seq - 1) & 1) * s.U * s.MS +
                    (int64_t)u * s.MS + (int64_t)mcell - (int64_t)u * s.B;
  return (int32_t)e;
}

// Two adjacent 16-byte hash cells in one 32-byte load, cached in L2 only (a
// window of the table; p is 32-byte aligned).
__device__ __forceinline__ void ldcg_cells2(const int4* p, int4& a, int4& b) {
  asm volatile("ld.global.cg.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z),
                 "=r"(b.w)
               : "l"(p));
}

__device__ __forceinline__ uint32_t fib_hash(int32_t id, int shift) {
  // Knuth's multiplicative (Fibonacci) hashing: top bits of id * 2^32/phi.
  return ((uint32_t)id * 2654435769u) >> shift;
}

// Bounds-checked build (a separate library compiled with -DAVSG_DEBUG_BOUNDS,
// the stand-in for a memory checker): an index a kernel takes from the step's
// data or the buffer state -- a slot, a selected id, a miss-set cell, a
// descriptor -- is checked against its array before the access; a failed
// check latches AVSG_ERR_INTERNAL with the unit and position in the device
// error word, and the access is skipped.  In the product build the check is
// the constant true and costs nothing.
#ifdef AVSG_DEBUG_BOUNDS
__device__ __forceinline__ bool bound_ok(bool ok, DevErr* e, int unit, int pos);
#define AVSG_IN_BOUNDS(cond, err, unit, pos) ::avsg::bound_ok((cond), (err), (unit), (pos))
#else
#define AVSG_IN_BOUNDS(cond, err, unit, pos) true
#endif

// Programmatic dependent launch: a kernel may be scheduled while the previous
// one in the stream drains; griddep_wait() blocks until that grid has finished
// and its memory is visible, so everything after it sees the previous kernel's
// results.  griddep_launch() lets the next kernel start its own prologue.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ int load_err(const DevErr* e) {
  return *(const volatile int32_t*)&e->code;
}

// This step's StepIO, written by the step's first kernel (L2 loads: it was
// written by another grid).
__device__ __forceinline__ StepIO load_io(const StepIO* p) {
  static_assert(sizeof(StepIO) % 8 == 0, "StepIO is loaded as 8-byte words");
  union {
    StepIO v;
    unsigned long long w[sizeof(StepIO) / 8];
  } u;
  const unsigned long long* src = reinterpret_cast<const unsigned long long*>(p);
#pragma unroll
  for (int i = 0; i < (int)(sizeof(StepIO) / 8); ++i) u.w[i] = __ldcg(src + i);
  return u.v;
}

__device__ __forceinline__ void raise_error(DevErr* e, int code, int unit, int pos) {
  if (atomicCAS(&e->code, 0, code) == 0) {
    e->unit = unit;
    e->pos = pos;
  }
}

#ifdef AVSG_DEBUG_BOUNDS
__device__ __forceinline__ bool bound_ok(bool ok, DevErr* e, int unit, int pos) {
  if (!ok) raise_error(e, AVSG_ERR_INTERNAL, unit, pos);
  return ok;
}
#endif

// Launch with programmatic stream serialization (see griddep_wait).
bool pdl_enabled();
template <typename... Params, typename... Args>
cudaError_t launch_ex(bool pdl, void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                      cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl && pdl_enabled() ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Params>(args)...);
}
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args... args) {
  return launch_ex(true, kernel, grid, block, smem, st, args...);
}
// The same with thread-block clusters of cluster_x CTAs along x.
template <typename... Params, typename... Args>
cudaError_t launch_pdl_cluster(int cluster_x, void (*kernel)(Params...), dim3 grid, dim3 block,
                               size_t smem, cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = (unsigned)cluster_x;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Params>(args)...);
}


// Raises a kernel's dynamic shared memory limit once per size, and asks for
// the largest shared-memory carveout so consecutive kernels of a step keep
// one L1/shared split.
cudaError_t ensure_smem(const void* kernel, size_t bytes, int* done_bytes);

// Kernel launchers (one per .cu file).
// Shared memory of one match CTA in a cluster of `cl`: its part of the miss
// set (MS cells) and of n_tok hit bitmaps.
size_t match_smem_bytes(int MS, int n_tok, int HW, int cl);
// CTAs per unit (a cluster) of a match over n selected ids per unit: about
// one id per thread, more where shared memory or the ids per thread need it.
int match_cluster_size(int MS, int n_tok, int HW, int n);
cudaError_t launch_match(const DeviceState& s, const StepIO& v, int n_tok, int k, cudaStream_t st);
size_t victims_smem_bytes(const DeviceState& s);
cudaError_t launch_victims(const DeviceState& s, int n_tok, int k, cudaStream_t st);
// New per-unit slot budgets (device [U]): evicts entries above lowered budgets.
cudaError_t launch_budget(const DeviceState& s, const int32_t* budget_new, cudaStream_t st);
// Hash-table update of a step (erase evicted ids, insert new ones, rebuild):
// needed only by the next step's match, so it may run beside the gather and
// the attention.
cudaError_t launch_commit(const DeviceState& s, int n_tok, int k, cudaStream_t st);
cudaError_t launch_gather(const DeviceState& s, int ctas, cudaStream_t st);
// Staged gather: right after match, the host row of every claimed miss-set
// cell is copied to kstage/vstage at that cell (no slot needed yet); chunks
// of cells handed out by a counter, or with by_request an equal range of
// cells per CTA (one CTA per request).
cudaError_t launch_gather_stage(const DeviceState& s, int ctas, bool by_request, cudaStream_t st);
// Staged rows -> their reserved slots.  which: 0 the rows the current (or
// last) step staged; 1 the rows the step before it staged (the deferred place
// of the two-pass pipeline, run early in the next step).  Runs whatever the
// error word says: a step whose reservation did not run has no descriptors
// (match zeroes the counts of its parity first).
cudaError_t launch_place(const DeviceState& s, int which, int ctas, cudaStream_t st);
// Warms the device's path to a mapped host range (reads it whole once; sink:
// a device word it may write), so the first steps do not pay for first accesses.
cudaError_t launch_host_touch(const unsigned char* p, size_t bytes, unsigned* sink, int num_sms,
                              cudaStream_t st);
cudaError_t launch_gather_all(const DeviceState& s, const StepIO& v, int n_tok, int k, int ctas,
                              cudaStream_t st);

struct AttnLaunch {
  int n_tok, k, splits;
  int identity_slots;              // 1: slot of (tok, j) is tok * k + j (no-reuse staging)
  float scale_log2;                // softmax scale * log2(e)
  const float* q;
  float* out;
  const int32_t* slot_map;
  const StepIO* io;                // when set, out and slot_map are read from here, and q too
                                   // when q is null
  int num_sms;                     // SMs of the device (persistent grid size)
  int staged_misses;               // 16-head kernel: a miss's row is read from the staging
                                   // area at its miss-set cell (hslot holds -2 - cell)
  int fused_merge;                 // 16-head kernel (set by its launcher): the last cluster
                                   // to finish a column slice merges it (no merge kernel)
  size_t count_capacity;           // arrival counters available at DeviceState::part_count
  size_t part_capacity;            // floats available at DeviceState::part
};
bool attention_supported(int D, int DV, int G, int kv_shared);
int attention_rows_per_tile(int D, int DV, int G, int kv_shared);
cudaError_t launch_attention(const DeviceState& s, const AttnLaunch& a, cudaStream_t st);
// Merge of the split partials of launch_attention's generic and 16-head paths.
cudaError_t launch_attention_merge(const DeviceState& s, const AttnLaunch& a, cudaStream_t st);
// Tensor-core attention for 16 heads per kv-head over shared K = V rows
// (avsg_attn_h16.cu), used by launch_attention where it applies.
bool attention_h16_enabled();
bool attention_h16_supported(int D, int DV, int G, int kv_shared);
int attention_h16_rows_per_tile();
cudaError_t launch_attention_h16(const DeviceState& s, const AttnLaunch& a, cudaStream_t st);
// Default attention CTAs per SM for a shape (the target of the split count).
int attention_ctas_per_sm(int D, int DV, int G, int kv_shared);
// Tensor-core attention (avsg_attn_tc.cu): K rows of 64 or 128, G <= 8, Dv == D.
bool attention_tc_supported(int D, int DV, int G, int kv_shared);
size_t attention_tc_part_floats(int U, int max_tokens, int G, int DV, int num_sms);
cudaError_t launch_attention_tc(const DeviceState& s, const AttnLaunch& a, int num_sms,
                                cudaStream_t st);
// pass 0: hit rows of every (unit, token), a persistent grid of 2 CTAs per
// SM, each an equal share of all pairs' tiles.  pass 1: miss rows from this
// step's half of the staging area, listed from the reservation's
// descriptors: one CTA per unit over the union of a 2- or 3-token step's
// misses, else one per (unit, token); launched after the gather, the
// reservation and the hit pass, it merges both passes into the output.
cudaError_t launch_attention_tc_pass(const DeviceState& s, const AttnLaunch& a, int pass,
                                     cudaStream_t st);
// Floats of partials a two-pass step over `pairs` (unit, token) pairs needs.
size_t attention_tc_two_pass_floats(int pairs, int k, int ET, int G, int DV, int num_sms);
bool attention_tc_enabled();

}  // namespace avsg
