// avsg_victims: reserve buffer slots for the step's missing ids.
//
// Retention policy: bucketed LRU (Spin page, "Unifying Sparse Attention with
// Hierarchical Memory for Scalable Long-Context LLM Serving", section 2B:
// recency buckets, about 64, no global sort, eviction decided in parallel on
// the GPU) combined with the AVSG page's slot reservation for entries that
// need a transfer (arxivdaily 2609.37538, English abstract).
//
// One CTA of 512 threads per unit.  Slots are put in 64 reservation orders:
//   order 0      : empty slot;
//   order 64 - b : occupied, not selected this step, bucket b = min(63, t - last);
//   excluded     : selected this step (a hit; its last_step becomes t).
// A slot's rank is the number of candidates in lower orders plus the number
// of lower-indexed slots in its own order: a per-warp order histogram (warp w
// owns a contiguous slot range), one exclusive scan over (order, warp), and,
// only for the orders that can hold one of the m victims, an in-order ballot
// count within each 32-slot chunk -- no sort of the slots.  The m distinct
// missing ids are ranked in ascending id order (a bit per entry of the unit
// and a prefix popcount when the unit has at most 2^17 entries, else by
// counting, or a bitonic sort for very many); the i-th takes the slot of
// rank i: its tag and last_step are set, a gather descriptor (with the
// evicted id and the tokens that selected it) is appended, and the slot map
// entries that pointed at its miss-set cell are resolved.
//
// The hash-table update of the step (commit_kernel below) runs separately:
// only the next step's match needs it.
#include "avsg_internal.cuh"

namespace avsg {
namespace {

constexpr int kThreads = 512;   // 2 per SM, or 1 beside a gather CTA
constexpr int kWarps = kThreads / 32;
static_assert(kOrders * kWarps == 2 * kThreads, "the (order, warp) scan takes 2 values per thread");

__device__ __forceinline__ int next_pow2(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

// Linear-probing erase of a key known to be present.  The cell becomes empty
// when the next cell is empty (then no probe path runs through it: a key
// stored further on would have stopped at that empty cell), otherwise a
// tombstone.  Concurrent erases stay valid: a cell only turns empty behind an
// empty cell.  Returns 1 when a cell was freed.
__device__ int hash_erase(int4* tab, uint32_t mask, int shift, int32_t key) {
  uint32_t c = fib_hash(key, shift);
  for (uint32_t i = 0; i <= mask; ++i, ++c) {
    int4* p = tab + (c & mask);
    const int32_t kk = *(volatile int32_t*)&p->x;
    if (kk == key) {
      const int32_t next = *(volatile int32_t*)&tab[(c + 1) & mask].x;
      if (next == kEmpty) {
        p->x = kEmpty;
        return 1;
      }
      p->x = kTomb;
      return 0;
    }
    if (kk == kEmpty) return 0;
  }
  return 0;
}

// Linear-probing insert of a key known to be absent; takes the first empty or
// erased cell on the probe path and stores {key, slot, mseq, mcell} there
// (mseq, mcell: the deferred-place marker, -1 when none).  Returns 1 if it
// consumed an empty cell.
__device__ int hash_insert(int4* tab, uint32_t mask, int shift, int32_t key, int32_t slot,
                           int32_t mseq, int32_t mcell, DevErr* err, int unit) {
  uint32_t c = fib_hash(key, shift);
  for (uint32_t i = 0; i <= 2 * mask + 2 * kThreads; ++i) {
    int4* p = tab + (c & mask);
    const int32_t kk = *(volatile int32_t*)&p->x;
    if (kk == kEmpty || kk == kTomb) {
      if (atomicCAS(&p->x, kk, key) == kk) {
        p->y = slot;
        p->z = mseq;
        p->w = mcell;
        return kk == kEmpty ? 1 : 0;
      }
      continue;  // another insert took this cell; look at it again
    }
    ++c;
  }
  raise_error(err, AVSG_ERR_CAPACITY, unit, -1);  // unreachable: live keys <= B < HS
  return 0;
}

__device__ __forceinline__ int warp_incl_scan(int v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

}  // namespace

namespace {

constexpr int kCountRankMax = 2048;  // above this many misses, sort instead of counting
constexpr int kCountRankCheap = 64;  // up to this many misses, counting is cheapest
constexpr int64_t kRankBitmapMax = 1 << 17;  // entries per unit a shared id bitmap covers

struct VictimsSmem {
  size_t keys, rank, victim, wstart, ord, bits, pre, total;
  int bitmap_words;  // 0: no id bitmap (more entries per unit than it covers)
};

__host__ __device__ inline VictimsSmem victims_layout(int max_union, int B, int64_t L) {
  int p = 1;
  while (p < max_union) p <<= 1;
  VictimsSmem l;
  const size_t mu = ((sizeof(int32_t) * (size_t)max_union + 15) & ~(size_t)15);
  l.bitmap_words = L <= kRankBitmapMax ? (int)((L + 31) / 32) : 0;
  l.keys = 0;
  l.rank = l.keys + sizeof(unsigned long long) * (size_t)p;
  l.victim = l.rank + mu;
  l.wstart = l.victim + mu;
  l.ord = l.wstart + sizeof(int32_t) * kOrders * kWarps;
  l.bits = l.ord + (((size_t)B + 15) & ~(size_t)15);
  l.pre = l.bits + sizeof(uint32_t) * (size_t)l.bitmap_words;
  l.total = l.pre + sizeof(int32_t) * (size_t)l.bitmap_words;
  return l;
}

// Exclusive prefix sum of v over the CTA (all threads call it); wsum: kWarps ints.
__device__ __forceinline__ int block_excl_scan(int v, int* wsum) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int incl = warp_incl_scan(v, lane);
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int x = lane < kWarps ? wsum[lane] : 0;
    const int y = warp_incl_scan(x, lane) - x;
    if (lane < kWarps) wsum[lane] = y;
  }
  __syncthreads();
  const int r = wsum[warp] + incl - v;
  __syncthreads();  // wsum is free again
  return r;
}

// A reservation key packs id << 32 | token bits << 24 | miss-set cell.
static_assert(kMaxTokens <= 8, "token bits fit the key's 8 bits");
static_assert(2LL * kMatchCluster * kMatchThreads * kMatchPerThread <= (1LL << 24),
              "a miss-set cell fits the key's 24 bits");

constexpr int kBatch = 8;  // 32-slot chunks whose state one warp loads before using it
static_assert(kBatch == 8, "the hit-word loads map lane & 7 to a chunk, lane >> 3 to a token");

__global__ void __launch_bounds__(kThreads, 2) victims_kernel(DeviceState s, int n_tok,
                                                              int k) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int s_stop, s_base, s_hits, s_omax, s_m;
  __shared__ int wsum[kWarps];
  const int u = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const VictimsSmem lay = victims_layout(s.max_union, s.B, s.L);
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(smem + lay.keys);
  int32_t* rank = reinterpret_cast<int32_t*>(smem + lay.rank);
  int32_t* victim = reinterpret_cast<int32_t*>(smem + lay.victim);
  int32_t* wstart = reinterpret_cast<int32_t*>(smem + lay.wstart);  // [order][warp]
  uint8_t* ord = smem + lay.ord;

  griddep_wait();
  const int B = s.B;
  const size_t ub = (size_t)u * B;
  unsigned long long* ms = s.mset + (size_t)u * s.MS;
  // Issued before anything waits: the step's record and the error word, this
  // unit's budget, the slot state of the first kBatch chunks and the first
  // round of the unit's miss-set cells.
  const StepIO io = load_io(s.io);
  const int budget = __ldcg(s.budget + u);  // this unit's usable slots (buffer elasticity)
  if (tid == 0) {
    s_stop = load_err(s.err);
    s_hits = 0;
    s_m = 0;
  }

  const int chunk = ((B + kWarps * 32 - 1) / (kWarps * 32)) * 32;  // slots per warp
  const int w_begin = warp * chunk, w_end = min(B, w_begin + chunk);
  int sn[kBatch], tg[kBatch], ls[kBatch];
  // Hit bitmap words of a batch: lane (b = lane & 7, t = lane >> 3) loads
  // chunk b's word of tokens t and t + 4 (chunks start at multiples of 32).
  uint32_t hw0 = 0u, hw1 = 0u;
  auto load_batch = [&](int base) {
    {
      const int b = lane & 7, t2 = lane >> 3;
      const int sl0 = base + b * 32;
      const bool inb = b < kBatch && sl0 < w_end && sl0 < w_begin + chunk;
      const uint32_t* hb = s.hitbits + (size_t)u * s.HT * s.HW + (sl0 >> 5);
      hw0 = (inb && t2 < n_tok) ? __ldcg(hb + (size_t)t2 * s.HW) : 0u;
      hw1 = (inb && t2 + 4 < n_tok) ? __ldcg(hb + (size_t)(t2 + 4) * s.HW) : 0u;
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int sl = base + b * 32 + lane;
      const bool in = sl < w_end && base + b * 32 < w_begin + chunk;
      tg[b] = in ? __ldcg(s.tag + ub + sl) : kEmpty;
      ls[b] = in ? __ldcg(s.last + ub + sl) : 0;
    }
  };
  // sn[b]: 1 if this lane's slot of chunk b is selected this step, 0 if not,
  // -1 past the warp's range (all lanes take part).
  auto batch_hits = [&](int base) {
    uint32_t x = hw0 | hw1;
    x |= __shfl_xor_sync(0xffffffffu, x, 8);
    x |= __shfl_xor_sync(0xffffffffu, x, 16);
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const uint32_t word = __shfl_sync(0xffffffffu, x, b);
      const int sl = base + b * 32 + lane;
      const bool in = sl < w_end && base + b * 32 < w_begin + chunk;
      sn[b] = in ? (int)((word >> lane) & 1u) : -1;
    }
  };
  load_batch(w_begin);
  constexpr int kCellsAhead = 8;  // miss-set cells a thread loads before compacting
  unsigned long long wv[kCellsAhead];
  auto load_cells = [&](int c0) {
#pragma unroll
    for (int e = 0; e < kCellsAhead; ++e) {
      const int cell = c0 + e * kThreads + tid;
      wv[e] = cell < s.MS ? __ldcg(ms + cell) : kMissEmpty;
    }
  };
  load_cells(0);
  __syncthreads();
  if (s_stop) {
    griddep_launch();
    return;
  }
  const int t = io.t;
  const StepBufs sb = step_bufs(s, io.parity);
  int32_t* __restrict__ slot_map = io.slot_map;

  // 1. Distinct missing ids: every claimed cell of the unit's miss set, as
  //    key = id << 32 | token bits << 24 | cell (one coalesced pass,
  //    compacted by ballots), and the rank of each in ascending id order:
  //    counted directly when there are few, otherwise by a bitonic sort.
  for (int c0 = 0; c0 < s.MS; c0 += kThreads * kCellsAhead) {
    if (c0) load_cells(c0);
#pragma unroll
    for (int e = 0; e < kCellsAhead; ++e) {
      if (c0 + e * kThreads >= s.MS) break;  // warp-uniform
      const int cell = c0 + e * kThreads + tid;
      const unsigned long long w = wv[e];
      const bool used = w != kMissEmpty;
      const unsigned bal = __ballot_sync(0xffffffffu, used);
      int wbase = 0;
      if (lane == 0 && bal) wbase = atomicAdd(&s_m, __popc(bal));
      wbase = __shfl_sync(0xffffffffu, wbase, 0);
      if (used)
        keys[wbase + __popc(bal & ((1u << lane) - 1u))] =
            ((unsigned long long)(uint32_t)w << 32) | (((w >> 32) & 0xFFull) << 24) |
            (uint32_t)cell;
    }
  }
  __syncthreads();
  const int m = s_m;
  // this unit's descriptor range, claimed now (its latency overlaps the ranking)
  int base_claim = 0;
  if (tid == 0 && m > 0) base_claim = atomicAdd(sb.desc_count, m);
  const bool counting = m <= kCountRankMax;
  const int P = counting ? m : next_pow2(m);
  for (int i = m + tid; i < P; i += kThreads) keys[i] = ~0ull;
  for (int i = tid; i < kOrders * kWarps; i += kThreads) wstart[i] = 0;
  __syncthreads();
  if (lay.bitmap_words > 0 && m > kCountRankCheap) {
    // The distinct missing ids as bits of a bitmap over the unit's entries;
    // the rank of an id is the number of bits below it (a prefix popcount).
    uint32_t* bits = reinterpret_cast<uint32_t*>(smem + lay.bits);
    int32_t* pre = reinterpret_cast<int32_t*>(smem + lay.pre);
    const int W = lay.bitmap_words;
    for (int i = tid; i < W; i += kThreads) bits[i] = 0u;
    __syncthreads();
    for (int i = tid; i < m; i += kThreads) {
      const uint32_t id = (uint32_t)(keys[i] >> 32);
      atomicOr(&bits[id >> 5], 1u << (id & 31));
    }
    __syncthreads();
    const int wpt = (W + kThreads - 1) / kThreads;  // words per thread, contiguous
    int cnt = 0;
    for (int w2 = tid * wpt; w2 < min(W, (tid + 1) * wpt); ++w2) cnt += __popc(bits[w2]);
    int run = block_excl_scan(cnt, wsum);
    for (int w2 = tid * wpt; w2 < min(W, (tid + 1) * wpt); ++w2) {
      pre[w2] = run;
      run += __popc(bits[w2]);
    }
    __syncthreads();
    for (int i = tid; i < m; i += kThreads) {
      const uint32_t id = (uint32_t)(keys[i] >> 32);
      rank[i] = pre[id >> 5] + __popc(bits[id >> 5] & ((1u << (id & 31)) - 1u));
    }
  } else if (counting) {
    // tpk threads per key, each counting smaller keys over a strided share.
    int tpk = 1;
    while (tpk < 32 && tpk * 2 * (m > 0 ? m : 1) <= kThreads) tpk <<= 1;
    const int per_round = kThreads / tpk;
    for (int base = 0; base < m; base += per_round) {
      const int i = base + tid / tpk, part = tid & (tpk - 1);
      const unsigned long long key = i < m ? keys[i] : ~0ull;
      int r = 0;
      if (i < m)
        for (int j = part; j < m; j += tpk) r += keys[j] < key ? 1 : 0;
      for (int o = tpk >> 1; o > 0; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
      if (i < m && part == 0) rank[i] = r;
    }
  } else {
    for (int kk = 2; kk <= P; kk <<= 1) {
      for (int j = kk >> 1; j > 0; j >>= 1) {
        for (int i = tid; i < P / 2; i += kThreads) {
          const int lo = 2 * i - (i & (j - 1));
          const int hi = lo + j;
          const bool up = (lo & kk) == 0;
          const unsigned long long a = keys[lo], b = keys[hi];
          if ((a > b) == up) {
            keys[lo] = b;
            keys[hi] = a;
          }
        }
        __syncthreads();
      }
    }
    for (int i = tid; i < m; i += kThreads) rank[i] = i;
  }

  // 2. Reservation order of every slot; per-warp histogram over orders (each
  //    warp owns a contiguous slot range and a private row of counters, so
  //    plain shared-memory atomics need no ordering).
  int hits = 0;
  for (int base = w_begin; base < w_begin + chunk; base += 32 * kBatch) {
    if (base != w_begin) load_batch(base);
    batch_hits(base);
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int sl = base + b * 32 + lane;
      if (sl >= w_end || base + b * 32 >= w_begin + chunk) continue;
      int o = kNotCandidate;
      if (sn[b] > 0) {
        s.last[ub + sl] = t;  // selected this step: refreshed, never a victim
        ++hits;
      } else if (sn[b] == 0 && sl < budget) {  // slots at or above the budget are not used
        if (tg[b] == kEmpty) {
          o = 0;
        } else {
          const int age = max(1, t - ls[b]);
          o = kOrders - min(kOrders - 1, age);
        }
        atomicAdd(&wstart[o * kWarps + warp], 1);
      }
      ord[sl] = (uint8_t)o;
    }
  }
  hits = __reduce_add_sync(0xffffffffu, hits);
  if (lane == 0 && hits) atomicAdd(&s_hits, hits);
  __syncthreads();

  // 3. Exclusive scan of wstart in (order, warp) order: 2 values per thread.
  //    The last order whose start is below m bounds the orders that can hold
  //    a victim (o_max).
  {
    const int a = wstart[2 * tid], b = wstart[2 * tid + 1];
    const int incl = warp_incl_scan(a + b, lane);
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      const int v = lane < kWarps ? wsum[lane] : 0;
      const int x = warp_incl_scan(v, lane) - v;
      if (lane < kWarps) wsum[lane] = x;
    }
    __syncthreads();
    const int excl = wsum[warp] + incl - (a + b);
    wstart[2 * tid] = excl;
    wstart[2 * tid + 1] = excl + a;
  }
  if (tid == 0) s_omax = -1;
  __syncthreads();
  if (tid < kOrders && wstart[tid * kWarps] < m) atomicMax(&s_omax, tid);
  __syncthreads();
  const int o_max = s_omax;

  // 4. Rank within order by slot index, only for orders <= o_max; the first
  //    m ranks are the victims.  Lanes of a chunk are grouped by order with a
  //    ballot per distinct order present (usually one or two).
  if (o_max >= 0) {
    for (int base = w_begin; base < w_begin + chunk; base += 32) {
      const int sl = base + lane;
      const int o = sl < w_end ? (int)ord[sl] : kNotCandidate;
      unsigned todo = __ballot_sync(0xffffffffu, o <= o_max);
      while (todo) {
        const int leader = __ffs(todo) - 1;
        const int ol = __shfl_sync(0xffffffffu, o, leader);
        const unsigned peers = __ballot_sync(0xffffffffu, o == ol && o <= o_max);
        const int start = wstart[ol * kWarps + warp];
        if (o == ol) {
          const int r = start + __popc(peers & ((1u << lane) - 1u));
          if (r < m) victim[r] = sl;
        }
        __syncwarp();
        if (lane == leader) wstart[ol * kWarps + warp] = start + __popc(peers);
        __syncwarp();
        todo &= ~peers;
      }
    }
  }
  if (tid == 0) s_base = base_claim;
  __syncthreads();

  // 5. Reserve: last_step, gather descriptors (with the tokens that selected
  //    the id), the cell -> slot map and the deferred-place marker; the new
  //    tags (and the evicted ids, for the hash-table update) here only when
  //    the update does not write them itself (late_commit = 0).
  for (int i = tid; i < m; i += kThreads) {
    const unsigned long long key = keys[i];
    const int32_t id = (int32_t)(key >> 32);
    const int cell = (int)(key & 0xFFFFFFu);
    const int32_t toks = (int32_t)((key >> 24) & 0xFFu);
    const int r = rank[i];
    if (!AVSG_IN_BOUNDS(r >= 0 && r < m, s.err, u, i)) continue;
    const int v = victim[r];
    if (!AVSG_IN_BOUNDS(v >= 0 && v < budget && cell >= 0 && cell < s.MS && id >= 0 &&
                            id < io.live && s_base + r < s.U * s.max_union,
                        s.err, u, i))
      continue;
    int32_t old = kEmpty;
    if (!s.late_commit) {
      old = s.tag[ub + v];
      s.tag[ub + v] = id;
    }
    s.last[ub + v] = t;
    s.mslot[(size_t)u * s.MS + cell] = v;
    if (s.deferred) s.pend[ub + v] = ((unsigned long long)io.seq << 32) | (uint32_t)cell;
    sb.desc[s_base + r] = GatherDesc{u, id, v, old, cell, toks, 0, 0};
  }
  __syncthreads();

  // 6. Resolve slot-map entries of misses (-2 - cell -> reserved slot),
  //    unless the hash-table update does (late_commit).  Thread t takes
  //    positions t, t + kThreads, ... (coalesced) and issues its loads
  //    before using them.
  const int n = s.late_commit ? 0 : n_tok * k;
  constexpr int kRun = 4;
  for (int c0 = 0; c0 < n; c0 += kThreads * kRun) {
    int sm[kRun];
#pragma unroll
    for (int e = 0; e < kRun; ++e) {
      const int p = c0 + e * kThreads + tid;
      sm[e] = p < n ? slot_map[(size_t)u * n + p] : 0;
    }
#pragma unroll
    for (int e = 0; e < kRun; ++e) {
      const int p = c0 + e * kThreads + tid;
      if (p < n && sm[e] <= -2 && AVSG_IN_BOUNDS(-2 - sm[e] < s.MS, s.err, u, p))
        slot_map[(size_t)u * n + p] = s.mslot[(size_t)u * s.MS + (-2 - sm[e])];
    }
  }

  // 7. Statistics and this step's descriptor range (for the table update).
  if (tid == 0) {
    sb.dbase[u] = s_base;
    sb.dcount[u] = m;
    s.counters[u].hits += (unsigned long long)s_hits;
    s.counters[u].misses += (unsigned long long)m;
  }
  griddep_launch();  // dependents launch as this kernel ends
}

// Hash-table update of one unit: erase the ids this step evicted, insert the
// ids it loaded, rebuild from the tags when erased cells pile up.  With
// late_commit, CTA (u, 0) also moves the reserved slots' tags and CTA (u, 1)
// resolves the unit's slot-map entries of misses.
constexpr int kCommitThreads = 256;  // small CTAs: they share SMs with the attention

__global__ void __launch_bounds__(kCommitThreads) commit_kernel(DeviceState s, int n_tok, int k) {
  __shared__ int s_stop, s_used, s_freed, s_rebuild, s_live;
  const int u = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31;
  griddep_wait();
  griddep_launch();
  if (tid == 0) {
    s_stop = load_err(s.err);
    s_used = 0;
    s_freed = 0;
    s_live = 0;
  }
  __syncthreads();
  if (s_stop) return;
  const StepIO io = load_io(s.io);
  const StepBufs sb = step_bufs(s, io.parity);
  const int m = sb.dcount[u], base = sb.dbase[u];
  const size_t ub = (size_t)u * s.B;
  int4* tab = s.htab + (size_t)u * s.HS;
  const uint32_t hmask = (uint32_t)s.HS - 1u;
  // the marker of an id this step loaded: its row stays staged until the
  // next step's place
  const int32_t mseq = s.deferred ? (int32_t)io.seq : -1;
  if (blockIdx.y == 1) {
    // (late_commit) the slot map's miss entries, -2 - cell -> the slot
    // reserved for the cell: a CTA of its own beside the hash update
    const int n = n_tok * k;
    int32_t* slot_map = io.slot_map + (size_t)u * n;
    for (int p = tid; p < n; p += kCommitThreads) {
      const int sm = slot_map[p];
      if (sm <= -2 && AVSG_IN_BOUNDS(-2 - sm < s.MS, s.err, u, p))
        slot_map[p] = s.mslot[(size_t)u * s.MS + (-2 - sm)];
    }
    return;
  }
  int freed = 0;
  for (int i = tid; i < m; i += kCommitThreads) {
    if (!AVSG_IN_BOUNDS(base + i < s.U * s.max_union, s.err, u, i)) continue;
    int32_t old;
    if (s.late_commit) {  // the reserved slot's evicted id, then its new one
      const GatherDesc d = sb.desc[base + i];
      if (!AVSG_IN_BOUNDS(d.slot >= 0 && d.slot < s.B, s.err, u, i)) continue;
      old = s.tag[ub + d.slot];
      s.tag[ub + d.slot] = d.id;
    } else {
      old = sb.desc[base + i].old_id;
    }
    if (old != kEmpty) freed += hash_erase(tab, hmask, s.hs_shift, old);
  }
  freed = __reduce_add_sync(0xffffffffu, freed);
  if (lane == 0 && freed) atomicAdd(&s_freed, freed);
  __syncthreads();
  int used = 0;
  for (int i = tid; i < m; i += kCommitThreads) {
    if (!AVSG_IN_BOUNDS(base + i < s.U * s.max_union, s.err, u, i)) continue;
    const GatherDesc d = sb.desc[base + i];
    if (!AVSG_IN_BOUNDS(d.slot >= 0 && d.slot < s.B && d.id >= 0 && d.id < s.L, s.err, u, i))
      continue;
    used += hash_insert(tab, hmask, s.hs_shift, d.id, d.slot, mseq, s.deferred ? d.cell : -1,
                        s.err, u);
  }
  used = __reduce_add_sync(0xffffffffu, used);
  if (lane == 0 && used) atomicAdd(&s_used, used);
  __syncthreads();
  if (tid == 0) {
    const int total = s.hused[u] + s_used - s_freed;  // cells not empty: live keys and tombstones
    s_rebuild = total > s.HS / 4;
    s.hused[u] = total;
  }
  __syncthreads();
  if (s_rebuild) {
    const int B = s.B;
    for (int i = tid; i < s.HS; i += kCommitThreads) tab[i] = make_int4(kEmpty, -1, -1, -1);
    __syncthreads();
    int live = 0;
    for (int sl = tid; sl < B; sl += kCommitThreads) {
      const int32_t tg = s.tag[ub + sl];
      if (tg != kEmpty) {
        int32_t ms = -1, mc = -1;  // this step's loads keep their marker (from pend)
        if (s.deferred) {
          const unsigned long long pm = s.pend[ub + sl];
          if (pm != ~0ull && (int32_t)(pm >> 32) == mseq) {
            ms = mseq;
            mc = (int32_t)(uint32_t)pm;
          }
        }
        hash_insert(tab, hmask, s.hs_shift, tg, sl, ms, mc, s.err, u);
        ++live;
      }
    }
    live = __reduce_add_sync(0xffffffffu, live);
    if (lane == 0 && live) atomicAdd(&s_live, live);
    __syncthreads();
    if (tid == 0) s.hused[u] = s_live;
  }
}

int g_victims_smem = 0;

}  // namespace

size_t victims_smem_bytes(const DeviceState& s) {
  return victims_layout(s.max_union, s.B, s.L).total;
}

namespace {

// Buffer elasticity (Spin page, section 2B): a unit's budget of usable slots
// changes between steps.  Entries held in slots at or above a lowered budget
// are dropped: erased from the hash table, the slot emptied.  Slots above a
// raised budget are already empty.  budget_new [U] takes effect here.
__global__ void __launch_bounds__(kCommitThreads) budget_kernel(DeviceState s,
                                                                 const int32_t* __restrict__ budget_new) {
  const int u = blockIdx.x;
  griddep_wait();
  griddep_launch();
  if (load_err(s.err) != 0) return;
  const int old_b = __ldcg(s.budget + u), new_b = budget_new[u];
  int4* tab = s.htab + (size_t)u * s.HS;
  const uint32_t hmask = (uint32_t)s.HS - 1u;
  const size_t ub = (size_t)u * s.B;
  int freed = 0;
  for (int sl = new_b + (int)threadIdx.x; sl < old_b; sl += kCommitThreads) {
    const int32_t tg = s.tag[ub + sl];
    if (tg != kEmpty) {
      freed += hash_erase(tab, hmask, s.hs_shift, tg);
      s.tag[ub + sl] = kEmpty;
      s.last[ub + sl] = -1;
    }
  }
  if (freed) atomicSub(&s.hused[u], freed);
  __syncthreads();
  if (threadIdx.x == 0) s.budget[u] = new_b;
}

}  // namespace

cudaError_t launch_budget(const DeviceState& s, const int32_t* budget_new, cudaStream_t st) {
  return launch_pdl(budget_kernel, dim3(s.U), dim3(kCommitThreads), 0, st, s, budget_new);
}

cudaError_t launch_victims(const DeviceState& s, int n_tok, int k, cudaStream_t st) {
  const size_t smem = victims_smem_bytes(s);
  cudaError_t e = ensure_smem((const void*)victims_kernel, smem, &g_victims_smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(victims_kernel, dim3(s.U), dim3(kThreads), smem, st, s, n_tok, k);
}

cudaError_t launch_commit(const DeviceState& s, int n_tok, int k, cudaStream_t st) {
  static int attr_done = 0;
  const cudaError_t e = ensure_smem((const void*)commit_kernel, 0, &attr_done);
  if (e != cudaSuccess) return e;
  return launch_pdl(commit_kernel, dim3(s.U, s.late_commit ? 2 : 1), dim3(kCommitThreads), 0, st, s,
                    n_tok, k);
}

}  // namespace avsg
