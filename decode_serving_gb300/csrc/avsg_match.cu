// avsg_match: match each selected id against its unit's resident ids.
//
// AVSG page (arxivdaily 2609.37538, English abstract): hash matching of the
// selected tokens against the entries retained in the HBM buffer identifies
// the reusable slots.  Here every lane of a warp probes one id, so a warp
// matches 32 ids at once; a probe reads a 16-byte window of two table cells.
//
// Grid (ceil(n_tok*k / 256), U), 256 threads.  Per id:
//   * range check (id in [0, L)), else BAD_SELECTION;
//   * lookup in the unit's open-addressed table (linear probing, Fibonacci
//     hash); a hit writes its slot (slot map and the internal hit-slot list
//     the attention over hit rows reads) and sets the token's bit in
//     seen[slot] (a bit already set means the id repeats within one token's
//     list);
//   * a miss is entered in the per-step miss set (one cell per distinct id,
//     claimed or extended with one compare-and-swap; token bits merged, so a
//     multi-token iteration reserves each id once); the slot map gets
//     -2 - cell until the reservation kernel resolves it.
// Nothing in the buffer state (tags, last_step, hash table) changes here, so a
// BAD_SELECTION leaves the state as it was.
#include "avsg_internal.cuh"

namespace avsg {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) match_kernel(DeviceState s, StepIO v, int n_tok,
                                                         int k) {
  const int32_t* __restrict__ sel = v.sel;
  int32_t* __restrict__ slot_map = v.slot_map;
  uint8_t* __restrict__ hit = v.hit;
  const int u = blockIdx.y;
  const int n = n_tok * k;
  const int pos = blockIdx.x * kThreads + threadIdx.x;
  griddep_wait();
  griddep_launch();
  if (blockIdx.x == 0 && u == 0 && threadIdx.x == 0) {
    *s.desc_count = 0;
    *s.io = v;  // for the kernels after this one
  }
  // The error word and the id are loaded together (no block barrier in
  // between); a latched error from an earlier step ends the thread.
  const int stop = load_err(s.err);
  int miss_cell = -1;
  if (pos < n) {
    const int tok = pos / k;
    const size_t off = (size_t)u * n + pos;
    const int32_t id = sel[off];
    if (stop) return;
    if (id < 0 || (int64_t)id >= s.L) {
      raise_error(s.err, AVSG_ERR_BAD_SELECTION, u, pos);
      slot_map[off] = -1;
      if (hit) hit[off] = 0;
    } else {
      // Hash lookup: 16-byte windows of two cells, starting at the even cell
      // at or before the home cell.  A cell before the home cell never holds
      // this id, and an empty one there does not end the probe.
      const int2* tab = s.htab + (size_t)u * s.HS;
      const uint32_t mask = (uint32_t)s.HS - 1u;
      const uint32_t home = fib_hash(id, s.hs_shift);
      uint32_t cell = home & ~1u;
      int slot = -1;
      bool skip_first = (home & 1u) != 0;
      for (int probes = 0; probes < s.HS; probes += 2) {
        const int4 w = __ldcg(reinterpret_cast<const int4*>(tab + (cell & mask)));
        if (!skip_first) {
          if (w.x == id) { slot = w.y; break; }
          if (w.x == kEmpty) break;
        }
        if (w.z == id) { slot = w.w; break; }
        if (w.z == kEmpty) break;
        skip_first = false;
        cell += 2;
      }
      const unsigned bit = 1u << tok;
      if (slot >= 0) {
        const int old = atomicOr(&s.seen[(size_t)u * s.B + slot], (int)bit);
        if (old & bit) raise_error(s.err, AVSG_ERR_BAD_SELECTION, u, pos);
        slot_map[off] = slot;
        s.hslot[off] = slot;
        if (hit) hit[off] = 1;
      } else {
        unsigned long long* ms = s.mset + (size_t)u * s.MS;
        const uint32_t mmask = (uint32_t)s.MS - 1u;
        const unsigned long long tokbit = (unsigned long long)bit << 32;
        uint32_t c = fib_hash(id, s.ms_shift);
        unsigned long long expect = kMissEmpty;  // first try: claim an empty cell
        // Each failed compare-and-swap on the id's own cell means another
        // token added its bit, so retries are bounded by the token count.
        for (int iter = 0; iter < s.MS + 2 * kMaxTokens; ++iter) {
          unsigned long long* p = ms + (c & mmask);
          const unsigned long long want = expect == kMissEmpty ? (tokbit | (uint32_t)id) : (expect | tokbit);
          const unsigned long long prev = atomicCAS(p, expect, want);
          if (prev == expect) {
            miss_cell = (int)(c & mmask);
            break;
          }
          if ((uint32_t)prev == (uint32_t)id) {  // this id's cell, claimed by another token
            if (prev & tokbit) {
              raise_error(s.err, AVSG_ERR_BAD_SELECTION, u, pos);
              miss_cell = (int)(c & mmask);
              break;
            }
            expect = prev;  // add this token's bit
            continue;
          }
          if (prev == kMissEmpty) {  // lost an empty cell to another id? it is now taken; retry it
            expect = kMissEmpty;
            continue;
          }
          expect = kMissEmpty;  // another id's cell: probe on
          ++c;
        }
        if (miss_cell < 0) raise_error(s.err, AVSG_ERR_CAPACITY, u, pos);  // miss set full
        slot_map[off] = -2 - miss_cell;
        s.hslot[off] = -1;
        if (hit) hit[off] = 0;
      }
    }
  }

}

}  // namespace

cudaError_t launch_match(const DeviceState& s, const StepIO& v, int n_tok, int k, cudaStream_t st) {
  const int n = n_tok * k;
  dim3 grid((unsigned)((n + kThreads - 1) / kThreads), (unsigned)s.U);
  static int attr_done = 0;
  const cudaError_t e = ensure_smem((const void*)match_kernel, 0, &attr_done);
  if (e != cudaSuccess) return e;
  return launch_pdl(match_kernel, grid, dim3(kThreads), 0, st, s, v, n_tok, k);
}

}  // namespace avsg
