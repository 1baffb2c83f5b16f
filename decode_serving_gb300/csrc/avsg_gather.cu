// avsg_gather: copy the step's missing KV rows from host memory into their
// reserved buffer slots.
//
// AVSG page (arxivdaily 2609.37538, English abstract): only the misses cross
// the host link ("miss-only transfer"), and the transfers are split evenly
// across the accelerator's cores instead of by request.  Here the compacted
// descriptor list is cut into 16-byte chunks (K row chunks, then V row chunks
// of each miss) and every CTA takes an equal contiguous range of chunks, so a
// unit with many misses does not leave other SMs idle.  Host memory is mapped
// pinned memory read directly by the SMs (over NVLink-C2C on GB300) with
// 16-byte non-coherent loads, several in flight per thread; the buffer rows
// are written with 16-byte stores that bypass L1.
#include "avsg_internal.cuh"

namespace avsg {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 8;

__device__ __forceinline__ uint4 load_host16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// 16-byte load and store marked as the L2's first eviction candidates (the
// place: its rows are not read again this step, and the staged rows the miss
// pass is about to read should stay in the L2 instead).
__device__ __forceinline__ unsigned long long l2_evict_first() {
  unsigned long long p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint4 load16_evict_first(const uint4* p, unsigned long long pol) {
  uint4 v;
  asm volatile("ld.global.cg.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(pol));
  return v;
}
__device__ __forceinline__ void store16_evict_first(void* p, uint4 v, unsigned long long pol) {
  asm volatile("st.global.cg.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;" ::"l"(p), "r"(v.x),
               "r"(v.y), "r"(v.z), "r"(v.w), "l"(pol)
               : "memory");
}

__device__ __forceinline__ void store16(void* p, uint4 v) {
  asm volatile("st.global.cg.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// Copies chunks [begin, end) of the list: chunk c of descriptor d = c / cpe.
template <typename DescFn>
__device__ __forceinline__ void copy_chunks(const DeviceState& s, uint32_t begin, uint32_t end,
                                            DescFn desc_of) {
  const uint32_t cpk = (uint32_t)(s.ek >> 4), cpv = (uint32_t)(s.ev >> 4), cpe = cpk + cpv;
  for (uint32_t c0 = begin + threadIdx.x; c0 < end; c0 += kThreads * kUnroll) {
    uint4 v[kUnroll];
    unsigned char* dst[kUnroll];
#pragma unroll
    for (int r = 0; r < kUnroll; ++r) {
      const uint32_t c = c0 + (uint32_t)(r * kThreads);
      dst[r] = nullptr;
      if (c < end) {
        const uint32_t d = c / cpe, w = c - d * cpe;
        int unit, id, slot;
        if (desc_of(d, unit, id, slot)) {
          const unsigned char* src;
          if (w < cpk) {
            src = s.host_k + ((size_t)unit * s.L + id) * s.ek + ((size_t)w << 4);
            dst[r] = s.kbuf + ((size_t)unit * s.B + slot) * s.ek + ((size_t)w << 4);
          } else {
            src = s.host_v + ((size_t)unit * s.L + id) * s.ev + ((size_t)(w - cpk) << 4);
            dst[r] = s.vbuf + ((size_t)unit * s.B + slot) * s.ev + ((size_t)(w - cpk) << 4);
          }
          v[r] = load_host16(src);
        }
      }
    }
#pragma unroll
    for (int r = 0; r < kUnroll; ++r)
      if (dst[r]) store16(dst[r], v[r]);
  }
}

__global__ void __launch_bounds__(kThreads) gather_kernel(DeviceState s) {
  griddep_wait();
  griddep_launch();
  if (load_err(s.err) != 0) return;  // no barriers below: a per-thread exit is safe
  const StepBufs sb = step_bufs(s, load_io(s.io).parity);
  const uint32_t n = (uint32_t)*(volatile int32_t*)sb.desc_count;
  const uint32_t cpe = (uint32_t)((s.ek + s.ev) >> 4);
  const uint32_t total = n * cpe;
  const uint32_t per = (total + gridDim.x - 1) / gridDim.x;
  const uint32_t begin = blockIdx.x * per;
  const uint32_t end = min(total, begin + per);
  const GatherDesc* desc = sb.desc;
  copy_chunks(s, begin, end, [&](uint32_t d, int& unit, int& id, int& slot) {
    const int4 g = __ldcg(reinterpret_cast<const int4*>(desc + d));
    unit = g.x;
    id = g.y;
    slot = g.z;
    return AVSG_IN_BOUNDS(unit >= 0 && unit < s.U && id >= 0 && id < s.L && slot >= 0 &&
                              slot < s.B,
                          s.err, unit, (int)d);
  });
}

// Staged gather: runs right after match, before any slot is reserved.  Each
// CTA takes an equal contiguous range of all units' miss-set cells (with one
// CTA per request, exactly that request's units: the request-level
// assignment the AVSG page compares against) and walks it in rounds of
// kStageCells:
// the claimed cells of a round are compacted into a shared list, then the
// whole CTA copies the listed host rows into the staging area at their
// cells, consecutive threads on consecutive 16-byte chunks of a row and
// kUnroll chunks in flight per thread.  Few CTAs keep the host link busy, so
// the reservation kernel finds free SMs beside this one.
constexpr int kStageCells = 1024;
constexpr int kStageWarps = kThreads / 32;

__global__ void __launch_bounds__(kThreads) gather_stage_kernel(DeviceState s) {
  __shared__ uint32_t s_off[kStageCells];  // claimed cells of the round (offset in the round)
  __shared__ int32_t s_id[kStageCells];
  __shared__ int s_n;
  griddep_wait();
  // (dependents are released when the last round begins: the miss pass that
  // follows prepares its lists meanwhile, but must not take SMs any earlier)
  if (load_err(s.err) != 0) return;  // uniform over the CTA
  const StepBufs sb = step_bufs(s, load_io(s.io).parity);
  const int lane = threadIdx.x & 31;
  const long long ncell = (long long)s.U * s.MS;
  const long long c_begin = blockIdx.x * ncell / gridDim.x;
  const long long c_end = (blockIdx.x + 1) * ncell / gridDim.x;
  const uint32_t cpk = (uint32_t)(s.ek >> 4), cpv = (uint32_t)(s.ev >> 4), cpe = cpk + cpv;
  for (long long r0 = c_begin; r0 < c_end; r0 += kStageCells) {
    if (r0 + kStageCells >= c_end) griddep_launch();  // last round: the miss pass may start listing
    if (threadIdx.x == 0) s_n = 0;
    __syncthreads();
    const int span = (int)min((long long)kStageCells, c_end - r0);
    constexpr int kPer = kStageCells / kThreads;
    unsigned long long w[kPer];
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      const int off = e * kThreads + (int)threadIdx.x;
      w[e] = off < span ? __ldcg(s.mset + r0 + off) : kMissEmpty;
    }
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      const bool claimed = w[e] != kMissEmpty;
      const unsigned bal = __ballot_sync(0xffffffffu, claimed);
      if (bal == 0u) continue;  // uniform over the warp
      int base = 0;
      if (lane == 0) base = atomicAdd(&s_n, __popc(bal));
      base = __shfl_sync(0xffffffffu, base, 0);
      if (claimed) {
        const int r = base + __popc(bal & ((1u << lane) - 1u));
        s_off[r] = (uint32_t)(e * kThreads + (int)threadIdx.x);
        s_id[r] = (int32_t)(uint32_t)w[e];
      }
    }
    __syncthreads();
    const uint32_t items = (uint32_t)s_n * cpe;  // (row, 16-byte chunk) pairs
    for (uint32_t it0 = threadIdx.x; it0 < items; it0 += kThreads * kUnroll) {
      uint4 v[kUnroll];
      unsigned char* dst[kUnroll];
#pragma unroll
      for (int q = 0; q < kUnroll; ++q) {
        const uint32_t it = it0 + (uint32_t)(q * kThreads);
        dst[q] = nullptr;
        if (it < items) {
          const uint32_t r = it / cpe, j = it - r * cpe;
          const long long cg = r0 + s_off[r];
          const long long unit = cg / s.MS;
          if (!AVSG_IN_BOUNDS(cg < (long long)s.U * s.MS && s_id[r] >= 0 && s_id[r] < s.L, s.err,
                              (int)unit, (int)(cg - unit * s.MS)))
            continue;
          const long long hrow = unit * s.L + s_id[r];
          const unsigned char* src;
          if (j < cpk) {
            src = s.host_k + hrow * s.ek + ((size_t)j << 4);
            dst[q] = sb.kstage + cg * s.ek + ((size_t)j << 4);
          } else {
            src = s.host_v + hrow * s.ev + ((size_t)(j - cpk) << 4);
            dst[q] = sb.vstage + cg * s.ev + ((size_t)(j - cpk) << 4);
          }
          v[q] = load_host16(src);
        }
      }
#pragma unroll
      for (int q = 0; q < kUnroll; ++q)
        if (dst[q]) store16(dst[q], v[q]);
    }
    __syncthreads();  // the list is rewritten by the next round
  }
  griddep_launch();  // (no round at all)
}

// Copies the listed host rows of one chunk of miss-set cells into the
// staging area at their cells: consecutive threads on consecutive 16-byte
// chunks of a row, kUnroll chunks in flight per thread.  off[r]: cell of row
// r counted from c0; id[r]: its entry id.
__device__ __forceinline__ void copy_staged_rows(const DeviceState& s, const StepBufs& sb,
                                                 long long c0, const uint32_t* off,
                                                 const int32_t* id, int n) {
  const uint32_t cpk = (uint32_t)(s.ek >> 4), cpv = (uint32_t)(s.ev >> 4), cpe = cpk + cpv;
  const uint32_t items = (uint32_t)n * cpe;  // (row, 16-byte chunk) pairs
  for (uint32_t it0 = threadIdx.x; it0 < items; it0 += kThreads * kUnroll) {
    uint4 v[kUnroll];
    unsigned char* dst[kUnroll];
#pragma unroll
    for (int q = 0; q < kUnroll; ++q) {
      const uint32_t it = it0 + (uint32_t)(q * kThreads);
      dst[q] = nullptr;
      if (it < items) {
        const uint32_t r = it / cpe, j = it - r * cpe;
        const long long cg = c0 + off[r];
        const long long unit = cg / s.MS;
        if (!AVSG_IN_BOUNDS(cg < (long long)s.U * s.MS && id[r] >= 0 && id[r] < s.L, s.err,
                            (int)unit, (int)(cg - unit * s.MS)))
          continue;
        const long long hrow = unit * s.L + id[r];
        const unsigned char* src;
        if (j < cpk) {
          src = s.host_k + hrow * s.ek + ((size_t)j << 4);
          dst[q] = sb.kstage + cg * s.ek + ((size_t)j << 4);
        } else {
          src = s.host_v + hrow * s.ev + ((size_t)(j - cpk) << 4);
          dst[q] = sb.vstage + cg * s.ev + ((size_t)(j - cpk) << 4);
        }
        v[q] = load_host16(src);
      }
    }
#pragma unroll
    for (int q = 0; q < kUnroll; ++q)
      if (dst[q]) store16(dst[q], v[q]);
  }
}

// Staged gather, balanced: the same copy, with the cells of all units cut
// into chunks (a power of two of 128 .. kStageChunk cells, about two per CTA
// at least, so a small step still spreads over every CTA) that the CTAs take
// one at a time from a counter (match zeroes it): a CTA whose chunks held
// more misses simply takes fewer of them and the CTAs end together.  A chunk's cells are loaded, and
// the next chunk taken, while the previous chunk's rows are in flight, so
// the host link sees no gap between chunks.  Dependents (the miss pass) are
// released when a CTA finds no chunk left.
constexpr int kStageChunk = 512;

__global__ void __launch_bounds__(kThreads) gather_stage_dyn_kernel(DeviceState s) {
  __shared__ uint32_t s_off[2][kStageChunk];  // claimed cells of a chunk (offset in the chunk)
  __shared__ int32_t s_id[2][kStageChunk];
  __shared__ int s_n[2];
  __shared__ long long s_chunk[2];
  constexpr int kPer = kStageChunk / kThreads;
  constexpr int kMinChunk = 128;
  griddep_wait();
  if (load_err(s.err) != 0) {  // uniform over the CTA
    griddep_launch();
    return;
  }
  const StepBufs sb = step_bufs(s, load_io(s.io).parity);
  const int lane = threadIdx.x & 31;
  const long long ncell = (long long)s.U * s.MS;
  int chunk = kStageChunk;
  while (chunk > kMinChunk && ncell < 2LL * chunk * gridDim.x) chunk >>= 1;
  const long long nchunk = (ncell + chunk - 1) / chunk;
  unsigned long long w[kPer];
  // claimed cells of chunk c (held in w) -> list b
  auto compact = [&](long long c, int b) {
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      const bool claimed = w[e] != kMissEmpty;
      const unsigned bal = __ballot_sync(0xffffffffu, claimed);
      if (bal == 0u) continue;  // uniform over the warp
      int base = 0;
      if (lane == 0) base = atomicAdd(&s_n[b], __popc(bal));
      base = __shfl_sync(0xffffffffu, base, 0);
      if (claimed) {
        const int r = base + __popc(bal & ((1u << lane) - 1u));
        s_off[b][r] = (uint32_t)(e * kThreads + (int)threadIdx.x);
        s_id[b][r] = (int32_t)(uint32_t)w[e];
      }
    }
    (void)c;
  };
  auto load_cells = [&](long long c) {
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      const int off = e * kThreads + (int)threadIdx.x;
      const long long cell = c * chunk + off;
      w[e] = c < nchunk && off < chunk && cell < ncell ? __ldcg(s.mset + cell) : kMissEmpty;
    }
  };
  if (threadIdx.x == 0) {
    s_chunk[0] = atomicAdd(s.gather_next, 1);
    s_n[0] = 0;
  }
  __syncthreads();
  load_cells(s_chunk[0]);
  compact(s_chunk[0], 0);
  __syncthreads();
  for (int b = 0; s_chunk[b] < nchunk; b ^= 1) {
    if (threadIdx.x == 0) {
      s_chunk[b ^ 1] = atomicAdd(s.gather_next, 1);
      s_n[b ^ 1] = 0;
    }
    __syncthreads();
    const long long next = s_chunk[b ^ 1];
    if (next >= nchunk) griddep_launch();  // this CTA's last chunk
    load_cells(next);                      // in flight beside this chunk's copies
    copy_staged_rows(s, sb, s_chunk[b] * chunk, s_off[b], s_id[b], s_n[b]);
    compact(next, b ^ 1);
    __syncthreads();  // list b ^ 1 complete; list b is rewritten two chunks on
  }
  griddep_launch();  // (no chunk at all)
}

// Place: every miss's staged row (by miss-set cell) into its reserved slot
// (device to device), for the step of parity io.parity ^ which (see
// launch_place).  A persistent grid of one CTA per SM, each an equal
// contiguous share of all the step's (descriptor, 16-byte chunk) items,
// kPlaceRows items per thread in flight (the descriptors, then all the loads,
// then the stores); consecutive threads take consecutive chunks of a row, so
// 8 KiB page entries and 512-byte token rows both keep every thread busy.
// Few CTAs on the lowest-priority stream: it fills the SMs the other kernels
// of the step leave free.  It ignores the error word: a step whose
// reservation did not run has no descriptors (match zeroes the count).
constexpr int kPlaceRows = 8;

__global__ void __launch_bounds__(kThreads) place_kernel(DeviceState s, int which) {
  griddep_wait();
  griddep_launch();
  const StepBufs sb = step_bufs(s, load_io(s.io).parity ^ which);
  const uint32_t cpk = (uint32_t)(s.ek >> 4), cpe = cpk + (uint32_t)(s.ev >> 4);
  const long long total = (long long)__ldcg(sb.desc_count) * cpe;
  const unsigned long long pol = l2_evict_first();
  const long long begin = (long long)blockIdx.x * total / gridDim.x;
  const long long end = (long long)(blockIdx.x + 1) * total / gridDim.x;
  for (long long i0 = begin + threadIdx.x; i0 < end; i0 += (long long)kThreads * kPlaceRows) {
    uint4 v[kPlaceRows];
    void* dst[kPlaceRows];
    const uint4* src[kPlaceRows];
#pragma unroll
    for (int r = 0; r < kPlaceRows; ++r) {
      const long long item = i0 + (long long)r * kThreads;
      dst[r] = nullptr;
      src[r] = nullptr;
      if (item < end) {
        const long long d = item / cpe;
        const uint32_t c = (uint32_t)(item - d * cpe);
        const GatherDesc* g = sb.desc + d;
        const int u = __ldcg(&g->unit), cell = __ldcg(&g->cell), slot = __ldcg(&g->slot);
        if (!AVSG_IN_BOUNDS(u >= 0 && u < s.U && cell >= 0 && cell < s.MS && slot >= 0 &&
                                slot < s.B,
                            s.err, u, (int)d))
          continue;
        const size_t srow = (size_t)u * s.MS + cell;
        const size_t drow = (size_t)u * s.B + slot;
        if (c < cpk) {
          src[r] = reinterpret_cast<const uint4*>(sb.kstage + srow * s.ek) + c;
          dst[r] = reinterpret_cast<uint4*>(s.kbuf + drow * s.ek) + c;
        } else {
          src[r] = reinterpret_cast<const uint4*>(sb.vstage + srow * s.ev) + (c - cpk);
          dst[r] = reinterpret_cast<uint4*>(s.vbuf + drow * s.ev) + (c - cpk);
        }
      }
    }
#pragma unroll
    for (int r = 0; r < kPlaceRows; ++r)
      if (src[r]) v[r] = load16_evict_first(src[r], pol);
#pragma unroll
    for (int r = 0; r < kPlaceRows; ++r)
      if (dst[r]) store16_evict_first(dst[r], v[r], pol);
  }
}

// No-reuse comparison path: every selected row of every token is copied to
// staging slot tok * k + j of its unit; ids are range-checked.
__global__ void __launch_bounds__(kThreads) gather_all_kernel(DeviceState s, StepIO v, int n_tok,
                                                              int k) {
  const int32_t* __restrict__ sel = v.sel;
  int32_t* __restrict__ slot_map = v.slot_map;
  uint8_t* __restrict__ hit = v.hit;
  griddep_wait();
  griddep_launch();
  if (blockIdx.x == 0 && threadIdx.x == 0) *s.io = v;  // for the attention after this kernel
  if (load_err(s.err) != 0) return;
  const uint32_t per_unit = (uint32_t)(n_tok * k);
  const uint32_t n = (uint32_t)s.U * per_unit;
  // Slot map (identity) and hit flags, one entry per thread of the grid.
  for (uint32_t d = blockIdx.x * kThreads + threadIdx.x; d < n; d += gridDim.x * kThreads) {
    if (slot_map) slot_map[d] = (int32_t)(d % per_unit);
    if (hit) hit[d] = 0;
  }
  const uint32_t cpe = (uint32_t)((s.ek + s.ev) >> 4);
  const uint32_t total = n * cpe;
  const uint32_t per = (total + gridDim.x - 1) / gridDim.x;
  const uint32_t begin = blockIdx.x * per;
  const uint32_t end = min(total, begin + per);
  copy_chunks(s, begin, end, [&](uint32_t d, int& unit, int& id, int& slot) {
    unit = (int)(d / per_unit);
    slot = (int)(d - (uint32_t)unit * per_unit);
    id = __ldg(sel + d);
    if (id < 0 || id >= v.live) {
      raise_error(s.err, AVSG_ERR_BAD_SELECTION, unit, slot);
      return false;
    }
    return true;
  });
}

}  // namespace

cudaError_t launch_gather(const DeviceState& s, int ctas, cudaStream_t st) {
  static int attr_done = 0;
  const cudaError_t e = ensure_smem((const void*)gather_kernel, 0, &attr_done);
  if (e != cudaSuccess) return e;
  return launch_pdl(gather_kernel, dim3(ctas), dim3(kThreads), 0, st, s);
}

// Warms the device's path to a mapped host range before the first step: the
// whole range is read once (coalesced 16-byte loads, four in flight per
// thread).  The first device reads of host memory the host has just written
// pay for translations and for the state the host keeps about those lines,
// which later reads do not: on a 17 GB store the first tens of steps ran up
// to 3x slower, unevenly from run to run, when the store was only sampled
// here; read whole, the first steps run as fast as the later ones.  About
// 90 ms for 17 GB (once per handle).
__global__ void host_touch_kernel(const unsigned char* __restrict__ p, size_t bytes,
                                  unsigned* __restrict__ sink) {
  const uint4* q = reinterpret_cast<const uint4*>(p);
  const size_t n = bytes / 16;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  unsigned acc = 0;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += 4 * stride) {
    uint4 v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      v[j] = i + j * stride < n ? __ldcg(q + i + j * stride) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int j = 0; j < 4; ++j) acc += v[j].x ^ v[j].y ^ v[j].z ^ v[j].w;
  }
  if (acc == 0x9E3779B9u) *sink = acc;  // keeps the loads; practically never taken
}

cudaError_t launch_host_touch(const unsigned char* p, size_t bytes, unsigned* sink, int num_sms,
                              cudaStream_t st) {
  if (!p || bytes < 16 || ((uintptr_t)p & 15)) return cudaSuccess;
  host_touch_kernel<<<dim3((unsigned)(num_sms * 8)), dim3(256), 0, st>>>(p, bytes, sink);
  return cudaGetLastError();
}

cudaError_t launch_gather_stage(const DeviceState& s, int ctas, bool by_request, cudaStream_t st) {
  static int attr_done = 0, attr_dyn = 0;
  if (by_request) {
    const cudaError_t e = ensure_smem((const void*)gather_stage_kernel, 0, &attr_done);
    if (e != cudaSuccess) return e;
    return launch_pdl(gather_stage_kernel, dim3(ctas), dim3(kThreads), 0, st, s);
  }
  const cudaError_t e = ensure_smem((const void*)gather_stage_dyn_kernel, 0, &attr_dyn);
  if (e != cudaSuccess) return e;
  return launch_pdl(gather_stage_dyn_kernel, dim3(ctas), dim3(kThreads), 0, st, s);
}


static_assert(kStageCells % kThreads == 0, "a round is whole passes of the CTA");
static_assert(kStageChunk % kThreads == 0, "a chunk is whole passes of the CTA");

cudaError_t launch_place(const DeviceState& s, int which, int ctas, cudaStream_t st) {
  static int attr_done = 0;
  const cudaError_t e = ensure_smem((const void*)place_kernel, 0, &attr_done);
  if (e != cudaSuccess) return e;
  // Not launched early: resident early behind match, its CTAs would hold
  // registers on every SM that the hit pass needs when match ends.
  return launch_ex(false, place_kernel, dim3((unsigned)ctas), dim3(kThreads), 0, st, s, which);
}

cudaError_t launch_gather_all(const DeviceState& s, const StepIO& v, int n_tok, int k, int ctas,
                              cudaStream_t st) {
  return launch_pdl(gather_all_kernel, dim3(ctas), dim3(kThreads), 0, st, s, v, n_tok, k);
}

}  // namespace avsg
