// The C interface declared in avsg.h: handle life cycle, argument checks,
// device-state layout, and the order in which a step's kernels are enqueued.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "avsg_internal.cuh"

using namespace avsg;

struct avsg_handle_s {
  avsg_config cfg{};
  DeviceState ds{};
  int device = 0, num_sms = 0, gather_ctas = 0, splits_cap = 0, target_ctas = 0, tile_rows = 0;
  int stage_ctas = 0;  // CTAs of the staged gather (it shares the GPU with the reservation)
  void* dev_block = nullptr;
  size_t dev_bytes = 0;
  const void* host_k = nullptr;
  const void* host_v = nullptr;
  bool reg_k = false, reg_v = false;
  bool no_reuse = false;
  bool has_t = false;
  int32_t last_t = -1;
  bool latched = false;
  cudaStream_t last_stream = nullptr;
  cudaError_t cuda_err = cudaSuccess;
  uint64_t steps = 0, selected = 0, host_misses = 0;
  int64_t live = 0;  // entries per unit selectable (avsg_append adds one)
  std::vector<int32_t> budget;  // usable slots per unit (avsg_set_budget)
  int32_t min_budget = 0;
  int32_t* budget_new = nullptr;  // device [U]: the budgets a set_budget call brings
  float scale_log2 = 0.f;
  size_t part_floats = 0;
  int32_t* slot_scratch = nullptr;  // [U][max_union] when the caller passes no slot map
  uint8_t* hit_scratch = nullptr;   // [U][max_union]
  int32_t* stage_sel = nullptr;     // avsg_step_host staging
  float* stage_q = nullptr;
  float* stage_out = nullptr;
  // profiling
  bool prof = false;
  std::vector<cudaEvent_t> ev_pool;
  size_t ev_used = 0;
  struct Rec {
    int kernel;
    cudaEvent_t a, b;
  };
  std::vector<Rec> recs;
  double prof_ms[AVSG_NUM_KERNELS] = {};
  uint64_t prof_launches[AVSG_NUM_KERNELS] = {};
  // side stream: the miss gather and the table commit run there while the
  // caller's stream runs attention over the hit rows
  cudaStream_t side = nullptr, side2 = nullptr, side3 = nullptr;  // side3: lowest priority
  cudaEvent_t ev_fork = nullptr, ev_gather = nullptr, ev_reserve = nullptr, ev_commit = nullptr,
              ev_staged = nullptr, ev_place = nullptr, ev_hits = nullptr;
  bool staged = false;  // staging area allocated: the two-pass pipeline is available
  bool by_request = false;  // staged gather assigned by request (AVSG_FLAG_REQUEST_GATHER)
  uint64_t seq = 0;     // steps enqueued since create/reset (their parity alternates)
  bool pending_place = false;  // the last step's staged rows await the place its next step runs
  bool overlap = false;  // steps run the two-pass pipeline
  bool overlap_h16 = false;  // ... in its 16-head form (one attention launch after the staged gather)
  // Captured steps: one CUDA graph per (tokens, k), re-pointed at each step
  // by updating its first kernel node (see StepIO).
  struct StepGraph {
    int n_tok = 0, k = 0;
    DeviceState sc{};           // the state the first kernel was captured with
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    cudaGraphNode_t first = nullptr;
    cudaKernelNodeParams kp{};  // function and launch shape of the first node
    uint64_t used = 0;
  };
  std::vector<StepGraph> graphs;
  uint64_t graph_clock = 0;
  cudaStream_t cap = nullptr;  // capture origin
};

namespace {

constexpr size_t kAlign = 256;

int fail_cuda(avsg_handle h, cudaError_t e) {
  if (h) h->cuda_err = e;
  return AVSG_ERR_CUDA;
}

int pow2_at_least(int64_t x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

int log2_exact(int p) {
  int l = 0;
  while ((1 << l) < p) ++l;
  return l;
}

// Carves one device allocation into aligned arrays.
struct Carver {
  size_t off = 0;
  template <typename T>
  size_t take(T** slot, size_t count) {
    off = (off + kAlign - 1) / kAlign * kAlign;
    const size_t at = off;
    off += sizeof(T) * (count ? count : 1);
    *slot = reinterpret_cast<T*>(at);  // offset for now, rebased later
    return at;
  }
};

template <typename T>
void rebase(T** p, void* base) {
  *p = reinterpret_cast<T*>(static_cast<char*>(base) + reinterpret_cast<size_t>(*p));
}

// Maps caller host memory for device reads: mapped allocations are used in
// place, anything else is registered here (and unregistered on destroy),
// read-only unless entries can still be appended.
int map_host(avsg_handle h, const void* p, size_t bytes, bool read_only, const unsigned char** dptr,
             bool* registered) {
  cudaPointerAttributes attr;
  cudaError_t e = cudaPointerGetAttributes(&attr, p);
  if (e == cudaSuccess && attr.type == cudaMemoryTypeHost && attr.devicePointer) {
    *dptr = static_cast<const unsigned char*>(attr.devicePointer);
    *registered = false;
    return AVSG_OK;
  }
  cudaGetLastError();
  e = cudaHostRegister(const_cast<void*>(p), bytes,
                       cudaHostRegisterMapped | (read_only ? cudaHostRegisterReadOnly : 0u));
  if (e != cudaSuccess) {
    cudaGetLastError();
    e = cudaHostRegister(const_cast<void*>(p), bytes, cudaHostRegisterMapped);
  }
  if (e != cudaSuccess) return fail_cuda(h, e);
  *registered = true;
  void* d = nullptr;
  e = cudaHostGetDevicePointer(&d, const_cast<void*>(p), 0);
  if (e != cudaSuccess) {
    cudaHostUnregister(const_cast<void*>(p));
    *registered = false;
    return fail_cuda(h, e);
  }
  *dptr = static_cast<const unsigned char*>(d);
  return AVSG_OK;
}

void release(avsg_handle h) {
  if (!h) return;
  for (auto& g : h->graphs) {
    if (g.exec) cudaGraphExecDestroy(g.exec);
    if (g.graph) cudaGraphDestroy(g.graph);
  }
  if (h->cap) cudaStreamDestroy(h->cap);
  for (cudaEvent_t e : h->ev_pool) cudaEventDestroy(e);
  for (cudaEvent_t e : {h->ev_fork, h->ev_gather, h->ev_reserve, h->ev_commit, h->ev_staged, h->ev_place,
                        h->ev_hits})
    if (e) cudaEventDestroy(e);
  if (h->side) cudaStreamDestroy(h->side);
  if (h->side2) cudaStreamDestroy(h->side2);
  if (h->side3) cudaStreamDestroy(h->side3);
  if (h->dev_block) cudaFree(h->dev_block);
  if (h->reg_k && h->host_k) cudaHostUnregister(const_cast<void*>(h->host_k));
  if (h->reg_v && h->host_v) cudaHostUnregister(const_cast<void*>(h->host_v));
  delete h;
}

// Splits of a (unit, token)'s entries over CTAs: about target_ctas CTAs in all,
// each with at least one tile of rows.
int attn_splits(const avsg_handle h, int n_tok, int k) {
  const int64_t pairs = (int64_t)h->ds.U * n_tok;
  int64_t s = (h->target_ctas + pairs - 1) / pairs;
  const int64_t by_rows = ((int64_t)k * h->ds.ET + h->tile_rows - 1) / h->tile_rows;
  if (s > by_rows) s = by_rows;
  if (s > h->splits_cap) s = h->splits_cap;
  // the merge reads every split's partial: at most about 2 MiB of them per pair
  const int64_t part_bytes = (int64_t)h->ds.G * (h->ds.DV + 2) * 4;
  const int64_t by_merge = ((int64_t)2 << 20) / part_bytes;
  if (s > by_merge) s = by_merge > 4 ? by_merge : 4;
  return (int)(s < 1 ? 1 : s);
}

int env_int_any(const char* name, int dflt) {
  const char* v = getenv(name);
  return (v && *v) ? atoi(v) : dflt;
}

int env_int(const char* name, int dflt) {
  const char* v = getenv(name);
  if (!v || !*v) return dflt;
  const int x = atoi(v);
  return x > 0 ? x : dflt;
}

}  // namespace

namespace avsg {

bool pdl_enabled() {
  static const int on = env_int_any("AVSG_PDL", 1);
  return on != 0;
}

bool attention_tc_enabled() {
  static const int on = env_int_any("AVSG_ATTN_TC", 1);
  return on != 0;
}

bool overlap_enabled() {
  static const int on = env_int_any("AVSG_OVERLAP", 1);
  return on != 0;
}

bool graphs_enabled() {
  static const int on = env_int_any("AVSG_GRAPH", 1);
  return on != 0;
}

cudaError_t ensure_smem(const void* kernel, size_t bytes, int* done_bytes) {
  if (*done_bytes > 0 && (int)bytes <= *done_bytes - 1) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                       (int)cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess && bytes > 0)
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) *done_bytes = (int)bytes + 1;  // +1: 0 bytes also counts as done
  return e;
}

}  // namespace avsg

namespace {

int init_state(avsg_handle h, cudaStream_t st) {
  const DeviceState& s = h->ds;
  const size_t ub = (size_t)s.U * s.B;
  cudaError_t e = cudaSuccess;
#define AVSG_SET(ptr, val, bytes) \
  if (e == cudaSuccess) e = cudaMemsetAsync((ptr), (val), (bytes), st)
  AVSG_SET(s.kbuf, 0, (size_t)s.U * s.B * s.ek);
  if (s.ev) AVSG_SET(s.vbuf, 0, (size_t)s.U * s.B * s.ev);
  if (!h->no_reuse) {
    AVSG_SET(s.tag, 0xFF, ub * 4);
    AVSG_SET(s.pend, 0xFF, ub * 8);
    AVSG_SET(s.last, 0xFF, ub * 4);
    AVSG_SET(s.hitbits, 0, (size_t)s.U * s.HT * s.HW * 4);
    AVSG_SET(s.htab, 0xFF, (size_t)s.U * s.HS * sizeof(int4));
    AVSG_SET(s.hused, 0, (size_t)s.U * 4);
    if (e == cudaSuccess && !h->budget.empty())
      e = cudaMemcpyAsync(s.budget, h->budget.data(), (size_t)s.U * 4, cudaMemcpyHostToDevice, st);
    AVSG_SET(s.mset, 0xFF, (size_t)s.U * s.MS * 8);
  }
  AVSG_SET(s.desc_count, 0, 2 * 4);
  AVSG_SET(s.dcount, 0, 2 * (size_t)s.U * 4);
  AVSG_SET(s.part_count, 0, (size_t)s.U * kMaxTokens * kCountsPerPair * 4);
  AVSG_SET(s.counters, 0, (size_t)s.U * sizeof(DevCounters));
  AVSG_SET(s.err, 0, sizeof(DevErr));
#undef AVSG_SET
  if (e != cudaSuccess) return fail_cuda(h, e);
  h->has_t = false;
  h->last_t = -1;
  h->latched = false;
  h->steps = h->selected = h->host_misses = 0;
  h->seq = 0;
  h->pending_place = false;
  return AVSG_OK;
}

}  // namespace

extern "C" int avsg_create(const avsg_config* cfg, const void* host_k, const void* host_v,
                           avsg_handle* out) {
  if (!out) return AVSG_ERR_INVALID_ARG;
  *out = nullptr;
  if (!cfg || !host_k) return AVSG_ERR_INVALID_ARG;
  const avsg_config c = *cfg;
  const bool shared = c.kv_shared != 0;
  const bool no_reuse = (c.flags & AVSG_FLAG_NO_REUSE) != 0;
  if (c.num_requests < 1 || c.num_kv_heads < 1 || c.q_per_kv < 1 || c.entry_tokens < 1 ||
      c.entry_tokens > 64 || c.head_dim < 8 || c.v_dim < 8 || c.head_dim % 8 || c.v_dim % 8 ||
      c.num_entries < 1 || c.num_entries > 0x7FFFFFFF || c.buffer_slots < 1 || c.max_select < 1 ||
      c.max_tokens_per_step < 1 || c.max_tokens_per_step > kMaxTokens || c.reserved0 ||
      c.initial_entries < 0 || (int64_t)c.initial_entries > c.num_entries ||
      (c.flags & ~(AVSG_FLAG_NO_REUSE | AVSG_FLAG_REQUEST_GATHER)) || !(c.softmax_scale >= 0.f) ||
      isinf(c.softmax_scale) ||
      (shared && (c.v_dim != c.head_dim || (host_v && host_v != host_k))) || (!shared && !host_v))
    return AVSG_ERR_INVALID_ARG;
  const int64_t U = (int64_t)c.num_requests * c.num_kv_heads;
  if (U > 65535) return AVSG_ERR_INVALID_ARG;
  const int64_t max_union = (int64_t)c.max_tokens_per_step * c.max_select;
  if (!no_reuse && max_union > c.buffer_slots) return AVSG_ERR_CAPACITY;
  if (max_union > (1 << 24) || (!no_reuse && c.buffer_slots > (1 << 24))) return AVSG_ERR_INVALID_ARG;
  // match keeps a step's miss set and hit bitmaps in one CTA's shared memory
  if (!no_reuse && (max_union > (int64_t)kMatchCluster * kMatchThreads * kMatchPerThread ||
                    match_smem_bytes(pow2_at_least(2 * max_union), c.max_tokens_per_step,
                                     (c.buffer_slots + 31) / 32, kMatchCluster) > kMatchSmemMax))
    return AVSG_ERR_CAPACITY;
  if (!attention_supported(c.head_dim, c.v_dim, c.q_per_kv, c.kv_shared)) return AVSG_ERR_UNSUPPORTED;
  // shapes with a staging area: the tensor-core two-pass pipeline and the
  // 16-head kernel, which both read missed rows from it by miss-set cell
  const bool tc_shape = attention_tc_supported(c.head_dim, c.v_dim, c.q_per_kv, c.kv_shared);
  const bool h16_shape = attention_h16_enabled() &&
                         attention_h16_supported(c.head_dim, c.v_dim, c.q_per_kv, c.kv_shared);
  if ((c.flags & AVSG_FLAG_REQUEST_GATHER) && !no_reuse && !tc_shape && !h16_shape)
    return AVSG_ERR_UNSUPPORTED;  // request-level assignment exists in the staged gather only
  const int64_t ek = (int64_t)c.entry_tokens * c.head_dim * 2;
  const int64_t ev = shared ? 0 : (int64_t)c.entry_tokens * c.v_dim * 2;
  if ((double)U * max_union * ((ek + ev) / 16) >= 2147483647.0) return AVSG_ERR_INVALID_ARG;

  avsg_handle h = new avsg_handle_s();
  h->cfg = c;
  h->no_reuse = no_reuse;
  h->host_k = host_k;
  h->host_v = shared ? nullptr : host_v;
  h->live = c.initial_entries > 0 ? c.initial_entries : c.num_entries;
  cudaError_t e = cudaGetDevice(&h->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device);
  if (e != cudaSuccess) {
    release(h);
    return AVSG_ERR_CUDA;
  }
  DeviceState& s = h->ds;
  s.U = (int32_t)U;
  s.B = no_reuse ? (int32_t)max_union : c.buffer_slots;
  s.G = c.q_per_kv;
  s.D = c.head_dim;
  s.DV = c.v_dim;
  s.ET = c.entry_tokens;
  s.L = c.num_entries;
  s.kv_shared = shared ? 1 : 0;
  s.ek = ek;
  s.ev = ev;
  s.max_union = (int32_t)max_union;
  s.HS = pow2_at_least(8LL * (no_reuse ? 1 : c.buffer_slots));
  s.hs_shift = 32 - log2_exact(s.HS);
  s.HW = (s.B + 31) / 32;
  s.HT = c.max_tokens_per_step;
  s.MS = pow2_at_least(2 * max_union);
  if (s.MS < 2 * kMatchCluster) s.MS = 2 * kMatchCluster;  // every match CTA holds two cells or more
  s.MS = s.MS < 2 ? 2 : s.MS;
  s.ms_shift = 32 - log2_exact(s.MS);
  if (s.hs_shift >= 32) s.hs_shift = 31;
  if (s.ms_shift >= 32) s.ms_shift = 31;
  h->tile_rows = attention_rows_per_tile(s.D, s.DV, s.G, s.kv_shared);
  h->target_ctas = h->num_sms * env_int("AVSG_ATTN_CTAS_PER_SM",
                                         attention_ctas_per_sm(s.D, s.DV, s.G, s.kv_shared));
  h->gather_ctas = h->num_sms * env_int("AVSG_GATHER_CTAS_PER_SM", 4);
  // The staged gather splits all units' miss-set cells evenly over its CTAs;
  // with one CTA per request each CTA's range is exactly one request's units.
  h->by_request = (c.flags & AVSG_FLAG_REQUEST_GATHER) != 0;
  h->stage_ctas = h->by_request ? c.num_requests : env_int("AVSG_STAGE_CTAS", h->num_sms / 2);
  {
    int64_t cap = (h->target_ctas + U - 1) / U;
    const int64_t by_rows = ((int64_t)c.max_select * c.entry_tokens + h->tile_rows - 1) / h->tile_rows;
    if (cap > by_rows) cap = by_rows;
    h->splits_cap = (int)(cap < 1 ? 1 : cap);
  }
  const float scale = c.softmax_scale > 0.f ? c.softmax_scale : 1.0f / sqrtf((float)c.head_dim);
  h->scale_log2 = scale * 1.4426950408889634f;

  const bool read_only = h->live >= c.num_entries;  // nothing left to append
  int rc = map_host(h, host_k, (size_t)(U * c.num_entries * ek), read_only, &s.host_k, &h->reg_k);
  if (rc == AVSG_OK && !shared)
    rc = map_host(h, host_v, (size_t)(U * c.num_entries * ev), read_only, &s.host_v, &h->reg_v);
  if (shared) s.host_v = s.host_k;
  if (rc != AVSG_OK) {
    release(h);
    return rc;
  }

  const bool st_arrays = !no_reuse;
  const size_t ub = st_arrays ? (size_t)U * s.B : 0;
  // staging rows for the two-pass pipeline (one per miss-set cell, a half per
  // step parity), each right after its buffer: the buffer is padded to whole
  // entries and 256 bytes, so a staged entry is also an entry index counted
  // from kbuf (and from vbuf, at the same distance)
  h->staged = !no_reuse && (tc_shape || h16_shape);
  size_t unit = (size_t)ek;
  while (unit % kAlign) unit += (size_t)ek;
  const size_t kbuf_bytes = ((size_t)U * s.B * ek + unit - 1) / unit * unit;
  Carver cv;
  cv.take(&s.kbuf, kbuf_bytes);
  cv.take(&s.kstage, h->staged ? 2 * (size_t)U * s.MS * ek : 0);
  cv.take(&s.vbuf, ev ? kbuf_bytes : 0);
  cv.take(&s.vstage, h->staged ? 2 * (size_t)U * s.MS * ev : 0);
  s.stage_entry0 = (int64_t)(kbuf_bytes / (size_t)ek);
  s.deferred = 0;  // set below for the two-pass pipeline
  s.late_commit = 0;  // set below for the overlapped pipelines
  if ((double)U * s.B + 2.0 * U * s.MS >= 2147483647.0) {
    release(h);
    return AVSG_ERR_INVALID_ARG;
  }
  cv.take(&s.tag, ub);
  cv.take(&s.last, ub);
  cv.take(&s.hitbits, st_arrays ? (size_t)U * s.HT * s.HW : 0);
  cv.take(&s.htab, st_arrays ? (size_t)U * s.HS : 0);
  cv.take(&s.hused, (size_t)U);
  cv.take(&s.mset, st_arrays ? (size_t)U * s.MS : 0);
  cv.take(&s.hslot, (size_t)U * max_union);
  cv.take(&s.mslot, st_arrays ? (size_t)U * s.MS : 0);
  cv.take(&s.desc, 2 * (size_t)U * max_union);
  cv.take(&s.desc_count, 2);
  cv.take(&s.gather_next, 1);
  cv.take(&s.io, 1);
  cv.take(&s.qbuf, st_arrays ? (size_t)U * c.max_tokens_per_step * s.G * s.D : 0);
  cv.take(&s.dbase, 2 * (size_t)U);
  cv.take(&s.dcount, 2 * (size_t)U);

  {
    size_t part = (size_t)U * c.max_tokens_per_step * h->splits_cap * s.G * (s.DV + 2);
    const size_t tc = attention_tc_part_floats((int)U, c.max_tokens_per_step, s.G, s.DV, h->num_sms);
    size_t two = 0;  // two-pass attention (most at max_tokens_per_step * max_select)
    if (tc_shape)
      for (int nt = 1; nt <= c.max_tokens_per_step; ++nt) {
        const size_t need = attention_tc_two_pass_floats((int)U * nt, c.max_select, s.ET, s.G,
                                                         s.DV, h->num_sms);
        two = need > two ? need : two;
      }
    h->part_floats = part > tc ? part : tc;
    h->part_floats = h->part_floats > two ? h->part_floats : two;
    h->overlap = h->staged && overlap_enabled() && (h16_shape || attention_tc_enabled());
    h->overlap_h16 = h->overlap && !tc_shape;
    s.deferred = h->overlap && !h->overlap_h16 ? 1 : 0;
    s.late_commit = h->overlap ? 1 : 0;
    cv.take(&s.part, h->part_floats);
  }
  cv.take(&s.part_count, (size_t)U * kMaxTokens * kCountsPerPair);
  cv.take(&s.counters, (size_t)U);
  cv.take(&s.err, 1);
  cv.take(&s.budget, (size_t)U);
  cv.take(&s.pend, st_arrays ? (size_t)U * s.B : 0);
  cv.take(&h->budget_new, (size_t)U);
  cv.take(&h->slot_scratch, (size_t)U * max_union);
  cv.take(&h->hit_scratch, (size_t)U * max_union);
  cv.take(&h->stage_sel, (size_t)U * max_union);
  cv.take(&h->stage_q, (size_t)U * c.max_tokens_per_step * s.G * s.D);
  cv.take(&h->stage_out, (size_t)U * c.max_tokens_per_step * s.G * s.DV);
  h->dev_bytes = (cv.off + kAlign - 1) / kAlign * kAlign;
  e = cudaMalloc(&h->dev_block, h->dev_bytes);
  if (e != cudaSuccess) {
    release(h);
    return AVSG_ERR_CUDA;
  }
  void* b = h->dev_block;
  rebase(&s.kbuf, b); rebase(&s.vbuf, b); rebase(&s.tag, b); rebase(&s.last, b);
  rebase(&s.kstage, b); rebase(&s.vstage, b);
  rebase(&s.hitbits, b); rebase(&s.htab, b); rebase(&s.hused, b); rebase(&s.io, b); rebase(&s.qbuf, b);
  rebase(&s.mslot, b); rebase(&s.desc, b);
  rebase(&s.desc_count, b); rebase(&s.gather_next, b); rebase(&s.part, b);
  rebase(&s.dbase, b); rebase(&s.dcount, b); rebase(&s.mset, b); rebase(&s.hslot, b);
  rebase(&s.part_count, b);
  rebase(&s.counters, b); rebase(&s.err, b); rebase(&s.budget, b); rebase(&h->budget_new, b);
  rebase(&s.pend, b);
  rebase(&h->slot_scratch, b); rebase(&h->hit_scratch, b); rebase(&h->stage_sel, b);
  rebase(&h->stage_q, b); rebase(&h->stage_out, b);
  if (shared) {
    s.vbuf = s.kbuf;
    s.vstage = s.kstage;
  }

  // The side streams get the highest priority: when match ends, the CTAs of
  // the gather and the reservation are placed before those of the attention.
  int prio_low = 0, prio_high = 0;
  e = cudaDeviceGetStreamPriorityRange(&prio_low, &prio_high);
  if (e == cudaSuccess)
    e = cudaStreamCreateWithPriority(&h->side, cudaStreamNonBlocking, prio_high);
  if (e == cudaSuccess)
    e = cudaStreamCreateWithPriority(&h->side2, cudaStreamNonBlocking, prio_high);
  if (e == cudaSuccess)
    e = cudaStreamCreateWithPriority(&h->side3, cudaStreamNonBlocking, prio_low);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h->cap, cudaStreamNonBlocking);
  for (cudaEvent_t* ev : {&h->ev_fork, &h->ev_gather, &h->ev_reserve, &h->ev_commit, &h->ev_staged,
                          &h->ev_place, &h->ev_hits})
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
  if (e != cudaSuccess) {
    release(h);
    return AVSG_ERR_CUDA;
  }
  h->budget.assign((size_t)U, s.B);
  h->min_budget = s.B;
  rc = init_state(h, nullptr);
  if (rc == AVSG_OK) {  // the host store's translations, once, before the first step
    const size_t kb = (size_t)U * c.num_entries * ek, vb = shared ? 0 : (size_t)U * c.num_entries * ev;
    unsigned* sink = reinterpret_cast<unsigned*>(s.desc_count);  // zeroed again below
    e = launch_host_touch(s.host_k, kb, sink, h->num_sms, nullptr);
    if (e == cudaSuccess) e = launch_host_touch(s.host_v, vb, sink, h->num_sms, nullptr);
    if (e == cudaSuccess) e = cudaMemsetAsync(s.desc_count, 0, 2 * 4, nullptr);
    if (e != cudaSuccess) rc = AVSG_ERR_CUDA;
  }
  if (rc == AVSG_OK) {
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) rc = AVSG_ERR_CUDA;
  }
  if (rc != AVSG_OK) {
    release(h);
    return rc;
  }
  *out = h;
  return AVSG_OK;
}

extern "C" int avsg_destroy(avsg_handle h) {
  if (!h) return AVSG_OK;
  cudaError_t e = cudaDeviceSynchronize();
  release(h);
  return e == cudaSuccess ? AVSG_OK : AVSG_ERR_CUDA;
}

namespace {

cudaEvent_t take_event(avsg_handle h) {
  if (h->ev_used == h->ev_pool.size()) {
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    h->ev_pool.push_back(e);
  }
  return h->ev_pool[h->ev_used++];
}

// Per-kernel CUDA events (when profiling): begin(kernel, stream) before a
// launch, end() after it, on the stream the kernel runs on.
struct Prof {
  avsg_handle h;
  cudaEvent_t a = nullptr;
  int kernel = -1;
  void begin(int k, cudaStream_t st) {
    if (!h->prof) return;
    a = take_event(h);
    kernel = k;
    if (a) cudaEventRecord(a, st);
  }
  void end(cudaStream_t st) {
    if (!h->prof || !a) return;
    cudaEvent_t b = take_event(h);
    if (!b) return;
    cudaEventRecord(b, st);
    h->recs.push_back({kernel, a, b});
    a = nullptr;
  }
};

// NVTX range names of the launches (a profiler attached to the process shows
// each launch, or its capture into a step graph, under these).
const char* const kKernelNames[AVSG_NUM_KERNELS] = {
    "avsg_match", "avsg_victims", "avsg_gather", "avsg_attn", "avsg_attn_miss", "avsg_commit",
    "avsg_finish", "avsg_place"};

// Enqueues the kernels of one step on st (and the side streams, forked from
// and joined back into st); the step's pointers come in v.  With first !=
// null (capture), returns the graph node of the first kernel there.
int enqueue_dag(avsg_handle h, int32_t n_tok, int32_t k, const StepIO& v, cudaStream_t st,
                DeviceState* sc_out, cudaGraphNode_t* first) {
  const DeviceState& s = h->ds;
  cudaError_t e;
  AttnLaunch a{};
  a.n_tok = n_tok;
  a.k = k;
  a.splits = attn_splits(h, n_tok, k);
  a.identity_slots = h->no_reuse ? 1 : 0;
  a.scale_log2 = h->scale_log2;
  a.q = h->no_reuse ? nullptr : s.qbuf;  // match copies q (no-reuse: read through io)
  a.out = v.out;
  a.slot_map = v.slot_map;
  a.io = s.io;
  a.num_sms = h->num_sms;
  a.part_capacity = h->part_floats;
  a.count_capacity = (size_t)s.U * kMaxTokens * kCountsPerPair;
  Prof pf{h};
#define AVSG_RUN(kernel_index, stream, call)         \
  do {                                               \
    nvtxRangePushA(kKernelNames[kernel_index]);      \
    pf.begin(kernel_index, stream);                  \
    e = (call);                                      \
    nvtxRangePop();                                  \
    if (e != cudaSuccess) return fail_cuda(h, e);    \
    pf.end(stream);                                  \
  } while (0)
  // The graph node of the kernel just captured on st.
  auto take_first = [&]() -> cudaError_t {
    if (!first) return cudaSuccess;
    cudaStreamCaptureStatus cs;
    const cudaGraphNode_t* deps = nullptr;
    size_t nd = 0;
    cudaError_t ce = cudaStreamGetCaptureInfo(st, &cs, nullptr, nullptr, &deps, nullptr, &nd);
    if (ce == cudaSuccess && (cs != cudaStreamCaptureStatusActive || nd != 1))
      ce = cudaErrorStreamCaptureInvalidated;
    if (ce == cudaSuccess) *first = deps[0];
    return ce;
  };
  const DeviceState& sc = s;
  if (sc_out) *sc_out = sc;
  // With the per-kernel events on, every kernel runs on st in an order that
  // keeps the dependencies, so each is timed alone (as a serialised profiler
  // sees it) rather than beside the kernels of the other streams.
  cudaStream_t side = h->prof ? st : h->side, side2 = h->prof ? st : h->side2;
  cudaStream_t side3 = h->prof ? st : h->side3;
  if (h->no_reuse) {
    AVSG_RUN(AVSG_KERNEL_GATHER, st, launch_gather_all(sc, v, n_tok, k, h->gather_ctas, st));
    e = take_first();
    if (e != cudaSuccess) return fail_cuda(h, e);
    AVSG_RUN(AVSG_KERNEL_ATTENTION, st, launch_attention(sc, a, st));
    return AVSG_OK;
  }
  AVSG_RUN(AVSG_KERNEL_MATCH, st, launch_match(sc, v, n_tok, k, st));
  e = take_first();
  if (e != cudaSuccess) return fail_cuda(h, e);
  if (!h->overlap) {
    // The hash-table update is needed only by the next step's match: it runs
    // on side2 beside the gather and the attention.
    AVSG_RUN(AVSG_KERNEL_RESERVE, st, launch_victims(sc, n_tok, k, st));
    e = cudaEventRecord(h->ev_reserve, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(side2, h->ev_reserve, 0);
    if (e != cudaSuccess) return fail_cuda(h, e);
    AVSG_RUN(AVSG_KERNEL_COMMIT, side2, launch_commit(sc, n_tok, k, side2));
    e = cudaEventRecord(h->ev_commit, side2);
    if (e != cudaSuccess) return fail_cuda(h, e);
    AVSG_RUN(AVSG_KERNEL_GATHER, st, launch_gather(sc, h->gather_ctas, st));
    AVSG_RUN(AVSG_KERNEL_ATTENTION, st, launch_attention(sc, a, st));
    e = cudaStreamWaitEvent(st, h->ev_commit, 0);
    if (e != cudaSuccess) return fail_cuda(h, e);
    return AVSG_OK;
  }
  if (h->overlap_h16) {
    // 16-head shapes: after match, the staged gather and then the attention
    // on side (the attention reads hit rows from their slots while the
    // gather runs, missed rows from the staging area once it is done); the
    // reservation and then the move of the staged rows into their slots on
    // side2; the hash-table update on st once the reservation is done.
    a.staged_misses = 1;
    e = cudaEventRecord(h->ev_fork, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(side, h->ev_fork, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(side2, h->ev_fork, 0);
    if (e != cudaSuccess) return fail_cuda(h, e);
    AVSG_RUN(AVSG_KERNEL_GATHER, side, launch_gather_stage(sc, h->stage_ctas, h->by_request, side));
    e = cudaEventRecord(h->ev_staged, side);
    if (e != cudaSuccess) return fail_cuda(h, e);
    AVSG_RUN(AVSG_KERNEL_ATTENTION, side, launch_attention(sc, a, side));
    e = cudaEventRecord(h->ev_gather, side);
    if (e != cudaSuccess) return fail_cuda(h, e);
    AVSG_RUN(AVSG_KERNEL_RESERVE, side2, launch_victims(sc, n_tok, k, side2));
    e = cudaEventRecord(h->ev_reserve, side2);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(side2, h->ev_staged, 0);
    if (e != cudaSuccess) return fail_cuda(h, e);
    AVSG_RUN(AVSG_KERNEL_PLACE, side2, launch_place(sc, 0, h->num_sms, side2));
    e = cudaEventRecord(h->ev_commit, side2);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, h->ev_reserve, 0);
    if (e != cudaSuccess) return fail_cuda(h, e);
    AVSG_RUN(AVSG_KERNEL_COMMIT, st, launch_commit(sc, n_tok, k, st));
    e = cudaStreamWaitEvent(st, h->ev_gather, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, h->ev_commit, 0);
    if (e != cudaSuccess) return fail_cuda(h, e);
    return AVSG_OK;
  }
  // Two-pass pipeline (the tensor-core shapes).  After match, four
  // streams run side by side:
  //   side3:  (lowest priority) the rows the previous step staged, into the
  //           slots its reservation gave them: the deferred place, off the
  //           previous step's critical path, in the SMs this step's kernels
  //           leave free;
  //   st:     attention over the hit rows (a hit on a row the previous step
  //           loaded reads its staged copy: match points it there);
  //   side:   the missed rows, host -> this step's half of the staging area
  //           (host link), then the attention over them, which also merges
  //           both passes into the output (it waits for the hit pass);
  //   side2:  the reservation, then the hash-table update.
  // This step's staged rows reach their slots in the next step (or when an
  // entry point that reads the buffer flushes them).
  e = cudaEventRecord(h->ev_fork, st);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(side, h->ev_fork, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(side2, h->ev_fork, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(side3, h->ev_fork, 0);
  if (e != cudaSuccess) return fail_cuda(h, e);
  // Launched in this order, so the CTAs of the kernels the miss pass needs
  // are placed first: the gather's (on SMs of their own), the reservation's,
  // the hit pass's; then the hash update and the place.
  AVSG_RUN(AVSG_KERNEL_GATHER, side, launch_gather_stage(sc, h->stage_ctas, h->by_request, side));
  AVSG_RUN(AVSG_KERNEL_RESERVE, side2, launch_victims(sc, n_tok, k, side2));
  e = cudaEventRecord(h->ev_reserve, side2);
  if (e != cudaSuccess) return fail_cuda(h, e);
  AVSG_RUN(AVSG_KERNEL_ATTENTION, st, launch_attention_tc_pass(sc, a, 0, st));
  e = cudaEventRecord(h->ev_hits, st);
  if (e != cudaSuccess) return fail_cuda(h, e);
  AVSG_RUN(AVSG_KERNEL_COMMIT, side2, launch_commit(sc, n_tok, k, side2));
  e = cudaEventRecord(h->ev_commit, side2);
  if (e != cudaSuccess) return fail_cuda(h, e);
  AVSG_RUN(AVSG_KERNEL_PLACE, side3, launch_place(sc, 1, h->num_sms, side3));
  e = cudaEventRecord(h->ev_place, side3);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(side, h->ev_hits, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(side, h->ev_reserve, 0);
  if (e != cudaSuccess) return fail_cuda(h, e);
  AVSG_RUN(AVSG_KERNEL_ATTENTION_MISS, side, launch_attention_tc_pass(sc, a, 1, side));
  e = cudaEventRecord(h->ev_gather, side);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(st, h->ev_gather, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(st, h->ev_commit, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(st, h->ev_place, 0);
  if (e != cudaSuccess) return fail_cuda(h, e);
#undef AVSG_RUN
  return AVSG_OK;
}

constexpr size_t kMaxGraphs = 16;

// The captured step for (n_tok, k), captured now if it is not cached (the
// least recently used one is dropped beyond kMaxGraphs).
int step_graph(avsg_handle h, int32_t n_tok, int32_t k, const StepIO& v,
               avsg_handle_s::StepGraph** out) {
  h->graph_clock += 1;
  for (auto& g : h->graphs)
    if (g.n_tok == n_tok && g.k == k) {
      g.used = h->graph_clock;
      *out = &g;
      return AVSG_OK;
    }
  if (h->graphs.size() >= kMaxGraphs) {
    size_t lru = 0;
    for (size_t i = 1; i < h->graphs.size(); ++i)
      if (h->graphs[i].used < h->graphs[lru].used) lru = i;
    cudaGraphExecDestroy(h->graphs[lru].exec);
    cudaGraphDestroy(h->graphs[lru].graph);
    h->graphs.erase(h->graphs.begin() + (long)lru);
  }
  avsg_handle_s::StepGraph g;
  g.n_tok = n_tok;
  g.k = k;
  cudaError_t e = cudaStreamBeginCapture(h->cap, cudaStreamCaptureModeRelaxed);
  if (e != cudaSuccess) return fail_cuda(h, e);
  const int rc = enqueue_dag(h, n_tok, k, v, h->cap, &g.sc, &g.first);
  cudaGraph_t graph = nullptr;
  e = cudaStreamEndCapture(h->cap, &graph);
  if (rc != AVSG_OK) {
    if (graph) cudaGraphDestroy(graph);
    return rc;
  }
  if (e == cudaSuccess) e = cudaGraphKernelNodeGetParams(g.first, &g.kp);
  if (e == cudaSuccess)
    e = cudaGraphInstantiateWithFlags(&g.exec, graph, cudaGraphInstantiateFlagUseNodePriority);
  if (e != cudaSuccess) {
    if (graph) cudaGraphDestroy(graph);
    return fail_cuda(h, e);
  }
  g.graph = graph;
  g.kp.kernelParams = nullptr;
  g.kp.extra = nullptr;
  g.used = h->graph_clock;
  h->graphs.push_back(g);
  *out = &h->graphs.back();
  return AVSG_OK;
}

int enqueue_step(avsg_handle h, int32_t t, int32_t n_tok, int32_t k, const int32_t* d_sel,
                 const float* d_q, float* d_out, int32_t* d_slot_map, uint8_t* d_hit,
                 cudaStream_t st) {
  const DeviceState& s = h->ds;
  h->last_stream = st;
  h->has_t = true;
  h->last_t = t;
  h->steps += 1;
  h->selected += (uint64_t)s.U * n_tok * k;
  cudaError_t e;
  if (k == 0) {
    e = cudaMemsetAsync(d_out, 0, (size_t)s.U * n_tok * s.G * s.DV * sizeof(float), st);
    return e == cudaSuccess ? AVSG_OK : fail_cuda(h, e);
  }
  if (h->no_reuse) h->host_misses += (uint64_t)s.U * n_tok * k;
  StepIO v{};
  v.seq = (uint32_t)h->seq;
  v.parity = (int32_t)(h->seq & 1);
  h->seq += 1;
  // the two-pass pipeline leaves this step's staged rows to the next step
  h->pending_place = h->overlap && !h->overlap_h16;
  v.sel = d_sel;
  v.q = d_q;
  v.out = d_out;
  v.slot_map = d_slot_map ? d_slot_map : h->slot_scratch;
  v.hit = d_hit;
  v.t = t;
  v.live = (int32_t)h->live;
  if (h->prof || !graphs_enabled()) return enqueue_dag(h, n_tok, k, v, st, nullptr, nullptr);
  avsg_handle_s::StepGraph* g = nullptr;
  const int rc = step_graph(h, n_tok, k, v, &g);
  if (rc != AVSG_OK) return rc;
  DeviceState sc = g->sc;
  int32_t nt = n_tok, kk = k;
  void* args[] = {&sc, &v, &nt, &kk};  // (DeviceState, StepIO, n_tok, k): match or gather_all
  cudaKernelNodeParams kp = g->kp;
  kp.kernelParams = args;
  e = cudaGraphExecKernelNodeSetParams(g->exec, g->first, &kp);
  if (e == cudaSuccess) e = cudaGraphLaunch(g->exec, st);
  return e == cudaSuccess ? AVSG_OK : fail_cuda(h, e);
}

// Places the rows the last step staged, if the next step has not yet (for
// the entry points that read or change the buffer between steps).
// Synchronises.
int flush_place(avsg_handle h) {
  if (!h->pending_place) return AVSG_OK;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = launch_place(h->ds, 0, h->num_sms, nullptr);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return fail_cuda(h, e);
  h->pending_place = false;
  return AVSG_OK;
}

int check_step(avsg_handle h, int32_t t, int32_t n_tok, int32_t k) {
  if (!h) return AVSG_ERR_INVALID_ARG;
  if (h->latched) return AVSG_ERR_LATCHED;
  if (n_tok < 1 || n_tok > h->cfg.max_tokens_per_step || k < 0) return AVSG_ERR_INVALID_ARG;
  if (k > h->cfg.max_select) return AVSG_ERR_CAPACITY;
  if ((int64_t)n_tok * k > h->ds.max_union) return AVSG_ERR_CAPACITY;
  if (!h->no_reuse && (int64_t)n_tok * k > h->min_budget) return AVSG_ERR_CAPACITY;
  if (t < 0 || (h->has_t && t <= h->last_t)) return AVSG_ERR_BAD_STEP;
  return AVSG_OK;
}

}  // namespace

extern "C" int avsg_step(avsg_handle h, int32_t t, int32_t n_tok, int32_t k, const int32_t* d_sel,
                         const float* d_q, float* d_out, int32_t* d_slot_map, uint8_t* d_hit,
                         void* stream) {
  const int rc = check_step(h, t, n_tok, k);
  if (rc != AVSG_OK) return rc;
  if (!d_out || (k > 0 && (!d_sel || !d_q))) return AVSG_ERR_INVALID_ARG;
  nvtxRangePushA("avsg_step");
  const int r = enqueue_step(h, t, n_tok, k, d_sel, d_q, d_out, d_slot_map, d_hit,
                             static_cast<cudaStream_t>(stream));
  nvtxRangePop();
  return r;
}

extern "C" int avsg_step_host(avsg_handle h, int32_t t, int32_t n_tok, int32_t k,
                              const int32_t* h_sel, const float* h_q, float* h_out,
                              int32_t* h_slot_map, uint8_t* h_hit, void* stream) {
  int rc = check_step(h, t, n_tok, k);
  if (rc != AVSG_OK) return rc;
  if (!h_out || (k > 0 && (!h_sel || !h_q))) return AVSG_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const DeviceState& s = h->ds;
  const size_t n_sel = (size_t)s.U * n_tok * k;
  const size_t n_q = (size_t)s.U * n_tok * s.G * s.D;
  const size_t n_out = (size_t)s.U * n_tok * s.G * s.DV;
  cudaError_t e = cudaSuccess;
  if (k > 0) {
    e = cudaMemcpyAsync(h->stage_sel, h_sel, n_sel * 4, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(h->stage_q, h_q, n_q * 4, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return fail_cuda(h, e);
  }
  rc = enqueue_step(h, t, n_tok, k, h->stage_sel, h->stage_q, h->stage_out, h->slot_scratch,
                    h_hit ? h->hit_scratch : nullptr, st);
  if (rc != AVSG_OK) return rc;
  e = cudaMemcpyAsync(h_out, h->stage_out, n_out * 4, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess && h_slot_map && n_sel)
    e = cudaMemcpyAsync(h_slot_map, h->slot_scratch, n_sel * 4, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess && h_hit && n_sel)
    e = cudaMemcpyAsync(h_hit, h->hit_scratch, n_sel, cudaMemcpyDeviceToHost, st);
  return e == cudaSuccess ? AVSG_OK : fail_cuda(h, e);
}

extern "C" int avsg_append(avsg_handle h, const void* d_k, const void* d_v, void* stream) {
  if (!h || !d_k || (!h->cfg.kv_shared && !d_v)) return AVSG_ERR_INVALID_ARG;
  if (h->latched) return AVSG_ERR_LATCHED;
  if (h->live >= h->cfg.num_entries) return AVSG_ERR_CAPACITY;
  const DeviceState& s = h->ds;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // one entry per unit: unit u's new row goes to host row (u * L + live)
  const size_t ek = (size_t)s.ek, pitch = (size_t)h->cfg.num_entries * ek;
  cudaError_t e = cudaMemcpy2DAsync(static_cast<unsigned char*>(const_cast<void*>(h->host_k)) +
                                        (size_t)h->live * ek,
                                    pitch, d_k, ek, ek, (size_t)s.U, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess && !h->cfg.kv_shared) {
    const size_t ev = (size_t)s.ev, vpitch = (size_t)h->cfg.num_entries * ev;
    e = cudaMemcpy2DAsync(static_cast<unsigned char*>(const_cast<void*>(h->host_v)) +
                              (size_t)h->live * ev,
                          vpitch, d_v, ev, ev, (size_t)s.U, cudaMemcpyDeviceToHost, st);
  }
  if (e != cudaSuccess) return fail_cuda(h, e);
  h->live += 1;
  return AVSG_OK;
}

extern "C" int avsg_set_budget(avsg_handle h, const int32_t* slots_per_unit, void* stream) {
  if (!h || !slots_per_unit) return AVSG_ERR_INVALID_ARG;
  if (h->no_reuse) return AVSG_ERR_UNSUPPORTED;
  if (h->latched) return AVSG_ERR_LATCHED;
  const DeviceState& s = h->ds;
  int32_t lo = s.B;
  for (int u = 0; u < s.U; ++u) {
    if (slots_per_unit[u] < 1 || slots_per_unit[u] > s.B) return AVSG_ERR_INVALID_ARG;
    lo = slots_per_unit[u] < lo ? slots_per_unit[u] : lo;
  }
  const int rc = flush_place(h);
  if (rc != AVSG_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(h->budget_new, slots_per_unit, (size_t)s.U * sizeof(int32_t),
                                  cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = launch_budget(s, h->budget_new, st);
  if (e != cudaSuccess) return fail_cuda(h, e);
  h->budget.assign(slots_per_unit, slots_per_unit + s.U);
  h->min_budget = lo;
  return AVSG_OK;
}

extern "C" int avsg_plan_budget(int64_t total_slots, int32_t num_units, int32_t mandatory,
                                int32_t max_slots, const float* weights, int32_t* out) {
  if (num_units < 1 || mandatory < 1 || max_slots < mandatory || !out || total_slots < 0)
    return AVSG_ERR_INVALID_ARG;
  const int64_t extra = total_slots - (int64_t)num_units * mandatory;
  if (extra < 0) return AVSG_ERR_CAPACITY;
  double wsum = 0.0;
  if (weights)
    for (int u = 0; u < num_units; ++u) {
      if (!(weights[u] >= 0.f) || isinf(weights[u])) return AVSG_ERR_INVALID_ARG;
      wsum += weights[u];
    }
  for (int u = 0; u < num_units; ++u) {
    int64_t share;
    if (wsum > 0.0)
      share = (int64_t)floor((double)extra * (double)weights[u] / wsum);
    else
      share = extra / num_units + (u < extra % num_units ? 1 : 0);
    const int64_t b = (int64_t)mandatory + share;
    out[u] = (int32_t)(b < max_slots ? b : max_slots);
  }
  return AVSG_OK;
}

extern "C" int avsg_get_stats(avsg_handle h, avsg_stats* out) {
  if (!h || !out) return AVSG_ERR_INVALID_ARG;
  cudaError_t e = cudaDeviceSynchronize();
  std::vector<DevCounters> cu((size_t)h->ds.U);
  DevErr de{};
  if (e == cudaSuccess)
    e = cudaMemcpy(cu.data(), h->ds.counters, cu.size() * sizeof(DevCounters), cudaMemcpyDeviceToHost);
  DevCounters c{};
  for (const DevCounters& x : cu) {
    c.hits += x.hits;
    c.misses += x.misses;
  }
  if (e == cudaSuccess) e = cudaMemcpy(&de, h->ds.err, sizeof(de), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail_cuda(h, e);
  memset(out, 0, sizeof(*out));
  out->steps = h->steps;
  out->selected = h->selected;
  out->hits = h->no_reuse ? 0 : c.hits;
  out->misses = h->no_reuse ? h->host_misses : c.misses;
  out->unique_selected = out->hits + out->misses;
  out->miss_bytes = out->misses * (uint64_t)(h->ds.ek + h->ds.ev);
  out->device_error = de.code;
  out->error_unit = de.code ? de.unit : -1;
  out->error_position = de.code ? de.pos : -1;
  if (de.code) h->latched = true;
  return AVSG_OK;
}

extern "C" int avsg_get_info(avsg_handle h, avsg_info* out) {
  if (!h || !out) return AVSG_ERR_INVALID_ARG;
  memset(out, 0, sizeof(*out));
  out->device_bytes = h->dev_bytes;
  out->hash_capacity = h->no_reuse ? 0 : h->ds.HS;
  out->miss_set_capacity = h->no_reuse ? 0 : h->ds.MS;
  out->attn_splits = attn_splits(h, 1, h->cfg.max_select);
  out->gather_ctas = h->staged && overlap_enabled() && attention_tc_enabled() ? h->stage_ctas
                                                                            : h->gather_ctas;
  out->num_sms = h->num_sms;
  out->host_registered = (h->reg_k || h->reg_v) ? 1 : 0;
  return AVSG_OK;
}

extern "C" int avsg_read_state(avsg_handle h, int32_t unit, int32_t* tag, int32_t* last_step,
                               void* k_rows, void* v_rows) {
  if (!h || unit < 0 || unit >= h->ds.U) return AVSG_ERR_INVALID_ARG;
  if (h->no_reuse && (tag || last_step)) return AVSG_ERR_INVALID_ARG;
  const int rc = flush_place(h);
  if (rc != AVSG_OK) return rc;
  const DeviceState& s = h->ds;
  cudaError_t e = cudaDeviceSynchronize();
  const size_t ub = (size_t)unit * s.B;
  if (e == cudaSuccess && tag) e = cudaMemcpy(tag, s.tag + ub, (size_t)s.B * 4, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && last_step)
    e = cudaMemcpy(last_step, s.last + ub, (size_t)s.B * 4, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && k_rows)
    e = cudaMemcpy(k_rows, s.kbuf + ub * s.ek, (size_t)s.B * s.ek, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && v_rows && s.ev)
    e = cudaMemcpy(v_rows, s.vbuf + ub * s.ev, (size_t)s.B * s.ev, cudaMemcpyDeviceToHost);
  return e == cudaSuccess ? AVSG_OK : fail_cuda(h, e);
}

extern "C" int avsg_reset(avsg_handle h, void* stream) {
  if (!h) return AVSG_ERR_INVALID_ARG;
  return init_state(h, static_cast<cudaStream_t>(stream));
}

extern "C" int avsg_clear_error(avsg_handle h) {
  if (!h) return AVSG_ERR_INVALID_ARG;
  const int rc = flush_place(h);
  if (rc != AVSG_OK) return rc;
  const DeviceState& s = h->ds;
  cudaError_t e = cudaDeviceSynchronize();
  if (!h->no_reuse) {
    if (e == cudaSuccess) e = cudaMemset(s.hitbits, 0, (size_t)s.U * s.HT * s.HW * 4);
    if (e == cudaSuccess) e = cudaMemset(s.mset, 0xFF, (size_t)s.U * s.MS * 8);
  }
  if (e == cudaSuccess) e = cudaMemset(s.desc_count, 0, 2 * 4);
  if (e == cudaSuccess) e = cudaMemset(s.dcount, 0, 2 * (size_t)s.U * 4);
  if (e == cudaSuccess) e = cudaMemset(s.part_count, 0, (size_t)s.U * kMaxTokens * kCountsPerPair * 4);
  if (e == cudaSuccess) e = cudaMemset(s.err, 0, sizeof(DevErr));
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return fail_cuda(h, e);
  h->latched = false;
  return AVSG_OK;
}

extern "C" int avsg_profile(avsg_handle h, int32_t enable) {
  if (!h) return AVSG_ERR_INVALID_ARG;
  h->prof = enable != 0;
  if (h->prof) {
    for (int i = 0; i < AVSG_NUM_KERNELS; ++i) {
      h->prof_ms[i] = 0;
      h->prof_launches[i] = 0;
    }
    h->recs.clear();
    h->ev_used = 0;
  }
  return AVSG_OK;
}

extern "C" int avsg_profile_read(avsg_handle h, avsg_kernel_times* out) {
  if (!h || !out) return AVSG_ERR_INVALID_ARG;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return fail_cuda(h, e);
  for (const auto& r : h->recs) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, r.a, r.b) == cudaSuccess && r.kernel >= 0 &&
        r.kernel < AVSG_NUM_KERNELS) {
      h->prof_ms[r.kernel] += ms;
      h->prof_launches[r.kernel] += 1;
    }
  }
  h->recs.clear();
  h->ev_used = 0;
  for (int i = 0; i < AVSG_NUM_KERNELS; ++i) {
    out->ms[i] = h->prof_ms[i];
    out->launches[i] = h->prof_launches[i];
  }
  return AVSG_OK;
}

extern "C" int avsg_host_alloc(size_t bytes, void** out) {
  if (!out || bytes == 0) return AVSG_ERR_INVALID_ARG;
  *out = nullptr;
  cudaError_t e = cudaHostAlloc(out, bytes, cudaHostAllocMapped | cudaHostAllocPortable);
  return e == cudaSuccess ? AVSG_OK : AVSG_ERR_CUDA;
}

extern "C" int avsg_host_free(void* p) {
  if (!p) return AVSG_OK;
  return cudaFreeHost(p) == cudaSuccess ? AVSG_OK : AVSG_ERR_CUDA;
}

extern "C" const char* avsg_strerror(int code) {
  switch (code) {
    case AVSG_OK: return "ok";
    case AVSG_ERR_INVALID_ARG: return "invalid argument";
    case AVSG_ERR_CAPACITY: return "selection larger than the buffer or max_select";
    case AVSG_ERR_CUDA: return "CUDA runtime error";
    case AVSG_ERR_BAD_SELECTION: return "selected id out of range or repeated within a token";
    case AVSG_ERR_TIMEOUT: return "bounded device wait gave up";
    case AVSG_ERR_BAD_STEP: return "step index not strictly increasing";
    case AVSG_ERR_UNSUPPORTED: return "no compiled attention kernel for this shape";
    case AVSG_ERR_LATCHED: return "a device error is pending; call avsg_clear_error";
    case AVSG_ERR_INTERNAL: return "an index check of the bounds-checked build failed";
    default: return "unknown error";
  }
}

extern "C" int avsg_cuda_error(avsg_handle h) { return h ? (int)h->cuda_err : 0; }
