// avsg_match: match each selected id against its unit's resident ids.
//
// AVSG page (arxivdaily 2609.37538, English abstract): hash matching of the
// selected tokens against the entries retained in the HBM buffer identifies
// the reusable slots.
//
// A cluster of CL CTAs per unit, CL in {1, 2, 4, 8} sized to the step (about
// one selected id per thread, so a unit with few ids takes one CTA and a
// large step spreads its probes over 8 SMs); the unit's miss set (cells in
// contiguous blocks) and hit bitmaps (32-slot words dealt round-robin) are
// spread over the cluster's shared memories and updated with atomics on
// distributed shared memory.  A thread takes every (CL * 256)-th position of
// the unit's n_tok * k selected ids (at most kPer, 1 .. kMatchPerThread),
// loads all of them and then all of their first hash windows before it
// resolves any.
// Per id:
//   * range check (id in [0, live), the entries live this step), else BAD_SELECTION;
//   * lookup in the unit's open-addressed table (linear probing, Fibonacci
//     hash; a probe reads a 32-byte window of two 16-byte cells {key, slot,
//     seq, cell}, one DRAM sector);
//   * a hit writes its slot (slot map and the hit-slot list the attention
//     over hit rows reads: the staged copy when the cell's seq names the
//     previous step) and sets the slot's bit in the token's hit bitmap
//     (a bit already set means the id repeats within one token's list);
//   * a miss is entered in the step's miss set (one cell per distinct id,
//     claimed or extended with one compare-and-swap; token bits merged, so a
//     multi-token iteration reserves each id once); the slot map and the
//     hit-slot list get -2 - cell (the slot map until the reservation
//     kernel resolves it; the list keeps it for the attention that reads
//     missed rows from the staging area by cell).
// The unit's q is also copied to a fixed device buffer for the attention
// kernels.  The miss set and the hit bitmaps are then written out whole (coalesced),
// so neither needs clearing between steps.  Nothing in the buffer state
// (tags, last_step, hash table) changes here, so a BAD_SELECTION leaves the
// state as it was.
#include <cooperative_groups.h>

#include "avsg_internal.cuh"

namespace cg = cooperative_groups;

namespace avsg {
namespace {

constexpr int kThreads = kMatchThreads;

template <int kC, int kPer>
__global__ void __launch_bounds__(kThreads) match_kernel(DeviceState s, StepIO v, int n_tok,
                                                         int k) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int MSL = s.MS / kC;              // miss-set cells held by each CTA
  const int HWL = (s.HW + kC - 1) / kC;   // bitmap words per token held by each CTA
  unsigned long long* lset = reinterpret_cast<unsigned long long*>(smem);  // [MSL]
  uint32_t* lbits = reinterpret_cast<uint32_t*>(lset + MSL);               // [n_tok][HWL]
  __shared__ int s_stop;
  cg::cluster_group cl = cg::this_cluster();
  const int rank = (int)cl.block_rank();
  const int u = blockIdx.x / kC, tid = threadIdx.x;
  const int32_t* __restrict__ sel = v.sel;
  int32_t* __restrict__ slot_map = v.slot_map;
  uint8_t* __restrict__ hit = v.hit;
  const int n = n_tok * k;
  const int HW = s.HW;
  // shared memory is private: cleared before the wait on the previous kernel
  for (int i = tid; i < MSL; i += kThreads) lset[i] = kMissEmpty;
  for (int i = tid; i < n_tok * HWL; i += kThreads) lbits[i] = 0u;
  cl.sync();  // every CTA's part is cleared before any CTA updates it
  griddep_wait();
  griddep_launch();
  if (u == 0 && rank == 0 && tid == 0) {
    s.desc_count[v.parity] = 0;
    *s.gather_next = 0;
    *s.io = v;  // for the kernels after this one
  }
  // No descriptors of this step's parity until its reservation writes them
  // (a step that fails leaves none for the place that follows it).
  if (rank == 0 && tid == 0) s.dcount[(size_t)v.parity * s.U + u] = 0;
  if (tid == 0) s_stop = load_err(s.err);  // a latched error from an earlier step
  const size_t ubase = (size_t)u * n;
  const int first = rank * kThreads + tid;
  int32_t id[kPer];
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int pos = first + j * kC * kThreads;
    id[j] = pos < n ? __ldcg(sel + ubase + pos) : kEmpty;
  }
  __syncthreads();
  const bool stop = s_stop != 0;  // uniform over the cluster's work below

  // First windows of two 16-byte cells (one 32-byte sector), starting at the
  // even cell at or before the home cell.
  const int4* tab = s.htab + (size_t)u * s.HS;
  const uint32_t mask = (uint32_t)s.HS - 1u;
  int4 wa[kPer], wb[kPer];
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const bool valid = !stop && first + j * kC * kThreads < n && id[j] >= 0 && id[j] < v.live;
    wa[j] = wb[j] = make_int4(kEmpty, -1, -1, -1);
    if (valid) ldcg_cells2(tab + (fib_hash(id[j], s.hs_shift) & ~1u), wa[j], wb[j]);
  }
  {  // this unit's q, copied to a buffer the attention kernels read at a fixed
     // place (its loads in flight beside the windows)
    const int nq = n_tok * s.G * s.D;
    const float* src = v.q + (size_t)u * nq;
    float* dst = s.qbuf + (size_t)u * nq;
    for (int i = rank * kThreads + tid; i < nq; i += kC * kThreads) dst[i] = __ldcg(src + i);
  }
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int pos = first + j * kC * kThreads;
    if (stop || pos >= n) continue;
    const size_t off = ubase + pos;
    const int tok = pos / k;
    const int32_t x = id[j];
    if (x < 0 || x >= v.live) {
      raise_error(s.err, AVSG_ERR_BAD_SELECTION, u, pos);
      slot_map[off] = -1;
      s.hslot[off] = -1;
      if (hit) hit[off] = 0;
      continue;
    }
    // Windows of two cells: a cell before the home cell never holds this id,
    // and an empty one there does not end the probe.
    const uint32_t home = fib_hash(x, s.hs_shift);
    uint32_t cell = home & ~1u;
    bool skip_first = (home & 1u) != 0;
    int4 a = wa[j], b = wb[j];
    int4 found = make_int4(kEmpty, -1, -1, -1);
    for (int probes = 0; probes < s.HS; probes += 2) {
      if (probes) ldcg_cells2(tab + (cell & mask), a, b);  // cell is even: no wrap inside
      if (!skip_first) {
        if (a.x == x) { found = a; break; }
        if (a.x == kEmpty) break;
      }
      if (b.x == x) { found = b; break; }
      if (b.x == kEmpty) break;
      skip_first = false;
      cell += 2;
    }
    const int slot = found.x == x ? found.y : -1;
    if (slot >= 0 && !AVSG_IN_BOUNDS(slot < s.B, s.err, u, pos)) continue;
    if (slot >= 0) {
      const int word = slot >> 5;
      uint32_t* bits = cl.map_shared_rank(lbits, (unsigned)(word % kC));
      const uint32_t b = 1u << (slot & 31);
      const uint32_t old = atomicOr(&bits[tok * HWL + word / kC], b);
      if (old & b) raise_error(s.err, AVSG_ERR_BAD_SELECTION, u, pos);
      slot_map[off] = slot;
      s.hslot[off] = hit_row_slot(s, u, slot, found.z, found.w, v.seq);
      if (hit) hit[off] = 1;
    } else {
      const uint32_t mmask = (uint32_t)s.MS - 1u;
      const unsigned long long tokbit = 1ull << (32 + tok);
      uint32_t c = fib_hash(x, s.ms_shift);
      unsigned long long expect = kMissEmpty;  // first try: claim an empty cell
      int miss_cell = -1;
      // A failed compare-and-swap on the id's own cell means another token
      // added its bit, so retries are bounded by the token count.
      for (int iter = 0; iter < s.MS + 2 * kMaxTokens; ++iter) {
        const int mc = (int)(c & mmask);
        unsigned long long* cellp = cl.map_shared_rank(lset, (unsigned)(mc / MSL)) + (mc % MSL);
        const unsigned long long want =
            expect == kMissEmpty ? (tokbit | (uint32_t)x) : (expect | tokbit);
        const unsigned long long prev = atomicCAS(cellp, expect, want);
        if (prev == expect) {
          miss_cell = mc;
          break;
        }
        if ((uint32_t)prev == (uint32_t)x) {  // this id's cell, claimed by another token
          if (prev & tokbit) {
            raise_error(s.err, AVSG_ERR_BAD_SELECTION, u, pos);
            miss_cell = mc;
            break;
          }
          expect = prev;  // add this token's bit
          continue;
        }
        if (prev == kMissEmpty) {  // an empty cell after all: try it again
          expect = kMissEmpty;
          continue;
        }
        expect = kMissEmpty;  // another id's cell: probe on
        ++c;
      }
      if (miss_cell < 0) raise_error(s.err, AVSG_ERR_CAPACITY, u, pos);  // miss set full
      slot_map[off] = -2 - miss_cell;
      s.hslot[off] = miss_cell >= 0 ? -2 - miss_cell : -1;
      if (hit) hit[off] = 0;
    }
  }
  cl.sync();  // every update of this CTA's part is done (and no CTA exits early)
  if (stop) return;
  // This CTA's part of the step's miss set and hit bitmaps.
  unsigned long long* gset = s.mset + (size_t)u * s.MS + (size_t)rank * MSL;
  for (int i = tid; i < MSL; i += kThreads) gset[i] = lset[i];
  uint32_t* gbits = s.hitbits + (size_t)u * s.HT * HW;
  for (int i = tid; i < n_tok * HWL; i += kThreads) {
    const int t2 = i / HWL, wl = i - t2 * HWL, word = wl * kC + rank;
    if (word < HW) gbits[t2 * HW + word] = lbits[i];
  }
}

}  // namespace

size_t match_smem_bytes(int MS, int n_tok, int HW, int cl) {
  return (size_t)(MS / cl) * sizeof(unsigned long long) +
         (size_t)n_tok * ((HW + cl - 1) / cl) * sizeof(uint32_t);
}

int match_cluster_size(int MS, int n_tok, int HW, int n) {
  int cl = 1;
  while (cl < kMatchCluster && (int64_t)cl * kThreads < n) cl *= 2;  // about one id per thread
  while (cl < kMatchCluster && (match_smem_bytes(MS, n_tok, HW, cl) > kMatchSmemMax ||
                                (int64_t)cl * kThreads * kMatchPerThread < n || MS < 2 * cl))
    cl *= 2;
  return cl;
}

namespace {

template <int CL, int PER>
cudaError_t run_match(const DeviceState& s, const StepIO& v, int n_tok, int k, cudaStream_t st) {
  const size_t smem = match_smem_bytes(s.MS, n_tok, s.HW, CL);
  static int attr_done = 0;
  const cudaError_t e = ensure_smem((const void*)match_kernel<CL, PER>,
                                    match_smem_bytes(s.MS, s.HT, s.HW, CL), &attr_done);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(s.U * CL));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, match_kernel<CL, PER>, s, v, n_tok, k);
}

// ids per thread: 1, 2 or 4 (kMatchPerThread), the fewest that cover n
template <int CL>
cudaError_t run_match_per(const DeviceState& s, const StepIO& v, int n_tok, int k,
                          cudaStream_t st) {
  const int n = n_tok * k;
  if (n <= CL * kThreads) return run_match<CL, 1>(s, v, n_tok, k, st);
  if (n <= 2 * CL * kThreads) return run_match<CL, 2>(s, v, n_tok, k, st);
  return run_match<CL, kMatchPerThread>(s, v, n_tok, k, st);
}

}  // namespace

cudaError_t launch_match(const DeviceState& s, const StepIO& v, int n_tok, int k, cudaStream_t st) {
  const int n = n_tok * k;
  const int cl = match_cluster_size(s.MS, s.HT, s.HW, n);
  if ((int64_t)n > (int64_t)cl * kThreads * kMatchPerThread || s.MS < 2 * cl || n_tok > s.HT ||
      match_smem_bytes(s.MS, s.HT, s.HW, cl) > kMatchSmemMax)
    return cudaErrorInvalidValue;
  switch (cl) {
    case 1: return run_match_per<1>(s, v, n_tok, k, st);
    case 2: return run_match_per<2>(s, v, n_tok, k, st);
    case 4: return run_match_per<4>(s, v, n_tok, k, st);
    default: return run_match_per<8>(s, v, n_tok, k, st);
  }
}

}  // namespace avsg
