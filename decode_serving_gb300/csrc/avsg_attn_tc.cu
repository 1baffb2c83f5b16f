// avsg_attn_tc: split-K decode attention on the tensor cores, for K rows of
// 64 or 128 values and up to 8 query heads per kv-head.
//
// Same operation as avsg_attn.cu (the Attention operation of the Spin page,
// "Unifying Sparse Attention with Hierarchical Memory for Scalable
// Long-Context LLM Serving", section 2A, over exactly the rows DSA selected,
// AVSG page arxivdaily 2609.37538, English abstract), built for GB300:
//
// * Rows are gathered into padded shared rows (so ldmatrix reads are free of
//   bank conflicts) with 16-byte cp.async: one warp instruction moves a whole
//   256-byte row (2 for 128-byte rows), slot ids are fetched a tile ahead, and
//   each warp runs its own 3-stage pipeline closed by cp.async.wait_group.
//   (Per-row TMA bulk copies were measured first: at ~40 cycles per 256-byte
//   request the TMA engine capped the kernel at ~1.9 TB/s.)
// * Scores and the V sum use mma.m16n8k16 (bf16 in, fp32 accumulate) with the
//   operands swapped: 16 selected rows form M, and the N = 8 columns hold the
//   G query heads twice -- the bf16 rounding of scale*log2(e)*q (hi) and the
//   bf16 rounding of what remains (lo).  hi + lo carries q to ~2^-16
//   relative, so the scores are fp32-accurate without wasting MMA rows on
//   padding.  P is split the same way for the V sum.
// * Single pass (attn_tc_kernel): a persistent grid of 2 CTAs per SM, each
//   taking an equal contiguous share of all 16-row tiles of all (unit, token)
//   pairs; a CTA writes one partial (max, sum, acc) per pair segment it
//   covers and the last CTA to finish a pair merges its segments.
// * Two passes: the hit pass (attn_tc_hits_kernel, persistent like the
//   single pass) covers the selected rows that were already resident (the
//   hit slots match wrote; misses are masked) and runs beside the gather and
//   the reservation; the miss pass (attn_tc_miss_kernel) covers the missed
//   rows, read from the staging area by miss-set cell from the reservation's
//   descriptors, with one CTA per (unit, token) -- or a cluster of two CTAs
//   per unit, over the union of a multi-token step's misses -- and merges
//   both passes into the output.
// No CTA waits for another kernel's CTAs; the union pass's cluster barriers
// are hardware barriers over co-scheduled CTAs.
#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <math.h>

#include <type_traits>

#include "avsg_internal.cuh"

namespace cg = cooperative_groups;

namespace avsg {
namespace {

constexpr int kWarpsTc = 4;
constexpr int kThreadsTc = kWarpsTc * 32;
constexpr int kTileRows = 16;
constexpr int kStages = 3;
constexpr int kAhead = 3;  // tiles whose slot ids are loaded beyond the staged ones
constexpr int kCtasPerSm = 2;

template <int D_, int G_, bool SHARED_>
struct TcShape {
  static constexpr int D = D_, G = G_;
  static constexpr bool SHARED = SHARED_;
  static constexpr int PITCH = 2 * D + 16;                    // bytes per staged row
  static constexpr int NCOL = 2 * G;                          // hi and lo columns
  static constexpr int NTN = (NCOL + 7) / 8;                  // n-tiles of 8 columns
  static constexpr int KS = D / 16;                           // k-steps of the score MMA
  static constexpr int MT = D / 16;                           // m-tiles of the V sum
  static constexpr int STAGE_BYTES = kTileRows * PITCH * (SHARED ? 1 : 2);
  static constexpr int PTILE_BYTES = NTN * kTileRows * 16;    // bf16 P tile per warp
  static constexpr int WARP_BYTES = kStages * STAGE_BYTES + PTILE_BYTES;
  static constexpr int MERGE_BYTES = kWarpsTc * G * (D + 2) * 4;
  static constexpr int SMEM = (kWarpsTc * WARP_BYTES > MERGE_BYTES ? kWarpsTc * WARP_BYTES
                                                                   : MERGE_BYTES) + 128;
  static_assert(D % 16 == 0 && (G == 1 || G == 2 || G == 4 || G == 8), "unsupported shape");
  static_assert(WARP_BYTES % 16 == 0, "alignment");
  // Most partials one merge takes: the four warps' outputs, the CTA's own
  // and 2 floats per partial and head must fit in the warps' staging.
  static constexpr int MAX_SEG = (kWarpsTc * WARP_BYTES / 4 - (kWarpsTc + 1) * G * D) / (2 * G);
  static_assert(MAX_SEG >= 16, "merge scratch");
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gmem_src)
               : "memory");
}
// The same with an L2 cache policy (from l2_evict_first_policy).
__device__ __forceinline__ void cp_async16_hint(void* smem_dst, const void* gmem_src,
                                                unsigned long long policy) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(
                   smem_u32(smem_dst)),
               "l"(gmem_src), "l"(policy)
               : "memory");
}
// Lines read under this policy are the first the L2 evicts.
__device__ __forceinline__ unsigned long long l2_evict_first_policy() {
  unsigned long long p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x2_t(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];"
               : "=r"(r0), "=r"(r1)
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float* c, uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// bf16 round-to-nearest of x (hi) and of the remainder x - hi (lo).
__device__ __forceinline__ void split_bf16(float x, uint16_t& hi, uint16_t& lo) {
  const __nv_bfloat16 h = __float2bfloat16_rn(x);
  hi = __bfloat16_as_ushort(h);
  lo = __bfloat16_as_ushort(__float2bfloat16_rn(x - __bfloat162float(h)));
}

__device__ __forceinline__ uint32_t pack2(uint16_t lo_k, uint16_t hi_k) {
  return (uint32_t)lo_k | ((uint32_t)hi_k << 16);
}

}  // namespace
}  // namespace avsg

namespace avsg {
namespace {

struct TcParams {
  int n_tok, k, ET;
  int identity;                 // slot of entry e of (unit, token) is token * k + e
  float scale_log2;
  const float* q;
  float* out;
  const int32_t* slots;         // [pairs][k] slot of each listed entry
  const StepIO* io;             // when set, q and out (and slots, single pass) come from here
  // persistent single pass
  int rows_per_pair, tiles_per_pair;
  long long tiles;              // all pairs
  int ctas, max_seg;
  // two passes: the hit pass is persistent (hit_ctas CTAs over all pairs'
  // tiles, like the single pass)
  int hit_ctas;
  // 1: rows are read as the L2's first eviction candidates.  The hit pass
  // streams every hit row once per step, beside the gather writing the
  // staging rows the miss pass reads next: read this way, the hit rows do
  // not push the staged rows out of the L2 before the miss pass gets them.
  int evict_first;
};

struct SegArgs {
  int pair, u, tok;
  int ent_base;                 // first listed entry of the range
  int rows;                     // rows of the range (entries * ET)
  int ta, tb;                   // this CTA's tiles [ta, tb) of the range
  const int32_t* list;          // when set: the slot of entry e is list[e] (shared memory)
  const float* qs;              // when set: the pair's q [G][D] in shared memory
};

// CTA c covers global tiles [c*T/C, (c+1)*T/C); the CTA holding tile x:
__device__ __forceinline__ int cta_of_tile(long long x, int C, long long T) {
  return (int)(((x + 1) * C - 1) / T);
}

// One segment: this CTA's tiles [ta, tb) of one (unit, token) row range.
// Every warp runs its own 3-stage pipeline over tiles ta + warp, ta + warp + 4,
// ...; the four warps are then merged and the CTA's result is left in shared
// memory: cm[h], cl[h] (max and sum of exp2 per head) and co[h * D + d]
// (unnormalised output).  All threads of the CTA call it.
template <class SH>
__device__ void tc_segment(const DeviceState& s, const TcParams& p, const SegArgs& a,
                           unsigned char* smem, float* cm, float* cl, float* co,
                           float (*s_m)[SH::G], float (*s_l)[SH::G]) {
  constexpr int D = SH::D, G = SH::G, NTN = SH::NTN, KS = SH::KS, MT = SH::MT;
  constexpr int PITCH = SH::PITCH;
  constexpr int NH = G == 1 ? 1 : 2;              // heads per thread
  constexpr int OWNERS = G >= 2 ? G / 2 : 1;      // lanes c < OWNERS own their heads
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int head_base = G == 1 ? 0 : 2 * (c % OWNERS);
  const bool owner = c < OWNERS;
  unsigned char* wbase = smem + warp * SH::WARP_BYTES;
  unsigned char* ptile = wbase + kStages * SH::STAGE_BYTES;
  const int pair = a.pair, u = a.u, tok = a.tok;

  // q of this lane's fragment columns: loaded now, turned into MMA B
  // fragments after the first row copies are issued (the two round trips
  // overlap).  Column n < G is hi(q_n), G <= n < 2G is lo(q_{n-G}).
  float qf[KS][NTN][4];
  {
    const float* qg = a.qs ? a.qs : p.q + (size_t)pair * G * D;
#pragma unroll
    for (int nt = 0; nt < NTN; ++nt) {
      const int col = g + 8 * nt;
      const int head = col < G ? col : col - G;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int d = 16 * ks + 2 * c + (i & 1) + 8 * (i >> 1);
          qf[ks][nt][i] = col >= 2 * G ? 0.f : a.qs ? qg[head * D + d] : __ldg(qg + head * D + d);
        }
    }
  }

  float m[NH], l[NH];
  float acc[MT][NTN][4];
#pragma unroll
  for (int j = 0; j < NH; ++j) {
    m[j] = -INFINITY;
    l[j] = 0.f;
  }
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int nt = 0; nt < NTN; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[mt][nt][i] = 0.f;

  const int n_my = a.tb - a.ta - warp > 0 ? (a.tb - a.ta - warp + kWarpsTc - 1) / kWarpsTc : 0;
  // Buffer row of row (lane & 15) of this warp's i-th tile, or -1.
  auto row_index = [&](int i) -> long long {
    const int row = (a.ta + warp + i * kWarpsTc) * kTileRows + (lane & 15);
    if (i >= n_my || row >= a.rows) return -1;
    const int ent = a.ent_base + (p.ET == 1 ? row : row / p.ET);
    const int sub = row - (ent - a.ent_base) * p.ET;
    const int slot = a.list ? a.list[ent]
                   : p.identity ? tok * p.k + ent
                                : __ldg(p.slots + (size_t)pair * p.k + ent);
    if (slot < 0) return -1;  // not a row of this pass (a miss in the pass over hit rows)
    // (a slot of B or more is a row still staged by the previous step)
    if (!AVSG_IN_BOUNDS(slot < s.B || (s.deferred && (long long)u * s.B + slot >= s.stage_entry0 &&
                                       (long long)u * s.B + slot < s.stage_entry0 + 2LL * s.U * s.MS),
                        s.err, u, ent))
      return -1;
    return ((long long)u * s.B + slot) * p.ET + sub;
  };
  constexpr int CPR = 2 * D / 16;  // 16-byte chunks per row
  constexpr int RPI = 32 / CPR;    // rows per warp instruction
  unsigned long long vmasks = 0;  // 16 bits per stage: which rows of the staged tile are real
  const unsigned long long policy = p.evict_first ? l2_evict_first_policy() : 0ull;
  auto issue = [&](long long myrow, int st) {
    const unsigned long long vm = __ballot_sync(0xffffffffu, myrow >= 0) & 0xFFFFu;
    vmasks = (vmasks & ~(0xFFFFull << (16 * st))) | (vm << (16 * st));
    unsigned char* kst = wbase + st * SH::STAGE_BYTES;
    unsigned char* vst = SH::SHARED ? kst : kst + kTileRows * PITCH;
    const int ch = lane % CPR, rsub = lane / CPR;
#pragma unroll
    for (int it = 0; it < kTileRows / RPI; ++it) {
      const int r = it * RPI + rsub;
      const long long srow = __shfl_sync(0xffffffffu, myrow, r);
      if (srow >= 0 && p.evict_first) {
        cp_async16_hint(kst + r * PITCH + ch * 16, s.kbuf + srow * (2 * D) + ch * 16, policy);
        if (!SH::SHARED)
          cp_async16_hint(vst + r * PITCH + ch * 16, s.vbuf + srow * (2 * D) + ch * 16, policy);
      } else if (srow >= 0) {
        cp_async16(kst + r * PITCH + ch * 16, s.kbuf + srow * (2 * D) + ch * 16);
        if (!SH::SHARED) cp_async16(vst + r * PITCH + ch * 16, s.vbuf + srow * (2 * D) + ch * 16);
      } else {  // no row: zeros (finite values, which P = 0 cancels)
        *reinterpret_cast<uint4*>(kst + r * PITCH + ch * 16) = make_uint4(0u, 0u, 0u, 0u);
        if (!SH::SHARED) *reinterpret_cast<uint4*>(vst + r * PITCH + ch * 16) = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    cp_async_commit();  // one group per tile (empty past the end) keeps the count uniform
  };

  // Rows of the tiles after the staged ones, kAhead tiles ahead (their slot
  // loads in flight while the staged tiles are computed).
  long long next_row[kAhead];
  {
    long long first_rows[kStages + kAhead];  // slot loads issued together, then the copies
#pragma unroll
    for (int i = 0; i < kStages + kAhead; ++i) first_rows[i] = row_index(i);
#pragma unroll
    for (int i = 0; i < kStages; ++i) issue(first_rows[i], i);
#pragma unroll
    for (int j = 0; j < kAhead; ++j) next_row[j] = first_rows[kStages + j];
  }
  uint32_t qb[KS][NTN][2];
#pragma unroll
  for (int nt = 0; nt < NTN; ++nt) {
    const int col = g + 8 * nt;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      uint16_t e[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint16_t hi = 0, lo = 0;
        if (col < 2 * G) split_bf16(qf[ks][nt][i] * p.scale_log2, hi, lo);
        e[i] = col < G ? hi : lo;
      }
      qb[ks][nt][0] = pack2(e[0], e[1]);
      qb[ks][nt][1] = pack2(e[2], e[3]);
    }
  }
  for (int i = 0; i < n_my; ++i) {
    const int st = i % kStages;
    cp_async_wait<kStages - 1>();
    __syncwarp();
    const unsigned vmask = (unsigned)(vmasks >> (16 * st)) & 0xFFFFu;
    const unsigned char* kst = wbase + st * SH::STAGE_BYTES;
    const unsigned char* vst = SH::SHARED ? kst : kst + kTileRows * PITCH;
    const uint32_t kaddr = smem_u32(kst), vaddr = smem_u32(vst);

    // scores^T (16 rows x 8 columns per n-tile), two chains: even and odd k-steps
    float sc[NTN][4], sc2[NTN][4];
#pragma unroll
    for (int nt = 0; nt < NTN; ++nt)
#pragma unroll
      for (int i2 = 0; i2 < 4; ++i2) sc[nt][i2] = sc2[nt][i2] = 0.f;
    {
      const int arow = (lane & 7) + ((lane >> 3) & 1) * 8;
      const int acol = (lane >> 4) * 8;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(kaddr + arow * PITCH + (16 * ks + acol) * 2, a0, a1, a2, a3);
#pragma unroll
        for (int nt = 0; nt < NTN; ++nt)
          mma_bf16((ks & 1) ? sc2[nt] : sc[nt], a0, a1, a2, a3, qb[ks][nt][0], qb[ks][nt][1]);
      }
#pragma unroll
      for (int nt = 0; nt < NTN; ++nt)
#pragma unroll
        for (int i2 = 0; i2 < 4; ++i2) sc[nt][i2] += sc2[nt][i2];
    }
    // hi + lo -> full scores sv[row half][head j] for rows g and g + 8
    float sv[2][2];
    if (G == 8) {
      sv[0][0] = sc[0][0] + sc[NTN - 1][0];
      sv[0][1] = sc[0][1] + sc[NTN - 1][1];
      sv[1][0] = sc[0][2] + sc[NTN - 1][2];
      sv[1][1] = sc[0][3] + sc[NTN - 1][3];
    } else if (G == 1) {
      sv[0][0] = sc[0][0] + sc[0][1];
      sv[1][0] = sc[0][2] + sc[0][3];
      sv[0][1] = sv[1][1] = -INFINITY;
    } else {
      const int xm = G / 2;  // lane distance from a hi column pair to its lo pair
      sv[0][0] = sc[0][0] + __shfl_xor_sync(0xffffffffu, sc[0][0], xm);
      sv[0][1] = sc[0][1] + __shfl_xor_sync(0xffffffffu, sc[0][1], xm);
      sv[1][0] = sc[0][2] + __shfl_xor_sync(0xffffffffu, sc[0][2], xm);
      sv[1][1] = sc[0][3] + __shfl_xor_sync(0xffffffffu, sc[0][3], xm);
    }
    if (!((vmask >> g) & 1u)) sv[0][0] = sv[0][1] = -INFINITY;
    if (!((vmask >> (g + 8)) & 1u)) sv[1][0] = sv[1][1] = -INFINITY;

    // online softmax per head over the 16 rows (lanes with equal c)
    float pv[2][2], alpha[2] = {1.f, 1.f};
#pragma unroll
    for (int j = 0; j < NH; ++j) {
      float mx = fmaxf(sv[0][j], sv[1][j]);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      const float m_new = fmaxf(m[j], mx);
      float p0 = 0.f, p1 = 0.f;
      if (m_new != -INFINITY) {
        alpha[j] = exp2f(m[j] - m_new);
        p0 = exp2f(sv[0][j] - m_new);
        p1 = exp2f(sv[1][j] - m_new);
      }
      float sum = p0 + p1;
      sum += __shfl_xor_sync(0xffffffffu, sum, 4);
      sum += __shfl_xor_sync(0xffffffffu, sum, 8);
      sum += __shfl_xor_sync(0xffffffffu, sum, 16);
      l[j] = l[j] * alpha[j] + sum;
      m[j] = m_new;
      pv[0][j] = p0;
      pv[1][j] = p1;
    }
    if (NH == 1) alpha[1] = alpha[0];
    if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int nt = 0; nt < NTN; ++nt) {
          acc[mt][nt][0] *= alpha[0];
          acc[mt][nt][1] *= alpha[1];
          acc[mt][nt][2] *= alpha[0];
          acc[mt][nt][3] *= alpha[1];
        }
    }

    // P^T tile in shared memory (rows x [hi columns | lo columns]) -> B fragments
    if (owner) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int rr = g + 8 * h;
        uint16_t hi0, lo0, hi1 = 0, lo1 = 0;
        split_bf16(pv[h][0], hi0, lo0);
        if (NH == 2) split_bf16(pv[h][1], hi1, lo1);
        if (G == 1) {
          *reinterpret_cast<uint32_t*>(ptile + rr * 16) = pack2(hi0, lo0);
        } else {
          const int chi = head_base, clo = G + head_base;
          *reinterpret_cast<uint32_t*>(ptile + (chi >> 3) * 256 + rr * 16 + (chi & 7) * 2) =
              pack2(hi0, hi1);
          *reinterpret_cast<uint32_t*>(ptile + (clo >> 3) * 256 + rr * 16 + (clo & 7) * 2) =
              pack2(lo0, lo1);
        }
      }
    }
    __syncwarp();
    uint32_t pb[NTN][2];
#pragma unroll
    for (int nt = 0; nt < NTN; ++nt)
      ldsm_x2_t(smem_u32(ptile + nt * 256 + (lane & 15) * 16), pb[nt][0], pb[nt][1]);

    // O^T += V^T P^T
    {
      const int vrow = (lane & 7) + ((lane >> 4) << 3);
      const int vcol = ((lane >> 3) & 1) * 8;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(vaddr + vrow * PITCH + (16 * mt + vcol) * 2, a0, a1, a2, a3);
#pragma unroll
        for (int nt = 0; nt < NTN; ++nt) mma_bf16(acc[mt][nt], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
      }
    }
    __syncwarp();  // every lane has read stage st
    issue(next_row[0], st);
#pragma unroll
    for (int j = 0; j + 1 < kAhead; ++j) next_row[j] = next_row[j + 1];
    next_row[kAhead - 1] = row_index(i + kStages + kAhead);
  }
  cp_async_wait<0>();

  // Per-warp result -> shared memory, then merge the 4 warps.
  __syncthreads();  // every warp is done with its staging (reused below)
  float* mo = reinterpret_cast<float*>(smem);  // [warp][G][D]
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int dv = 16 * mt + g + 8 * (i >> 1);
      float v;
      int head;
      if (G == 8) {
        v = acc[mt][0][i] + acc[mt][NTN - 1][i];
        head = 2 * c + (i & 1);
      } else if (G == 1) {
        v = (i & 1) ? 0.f : acc[mt][0][i] + acc[mt][0][i + 1];
        head = 0;
      } else {
        v = acc[mt][0][i] + __shfl_xor_sync(0xffffffffu, acc[mt][0][i], G / 2);
        head = head_base + (i & 1);
      }
      if (owner && (G != 1 || (i & 1) == 0)) mo[(warp * G + head) * D + dv] = v;
    }
  if (owner && g == 0) {
#pragma unroll
    for (int j = 0; j < NH; ++j) {
      s_m[warp][head_base + j] = m[j];
      s_l[warp][head_base + j] = l[j];
    }
  }
  __syncthreads();
  if (tid < G) {
    float M = -INFINITY, L = 0.f;
#pragma unroll
    for (int w = 0; w < kWarpsTc; ++w) M = fmaxf(M, s_m[w][tid]);
    if (M != -INFINITY)
#pragma unroll
      for (int w = 0; w < kWarpsTc; ++w) L = fmaf(s_l[w][tid], exp2f(s_m[w][tid] - M), L);
    cm[tid] = M;
    cl[tid] = L;
  }
  __syncthreads();
  for (int o = tid; o < G * D; o += kThreadsTc) {
    const int head = o / D;
    const float M = cm[head];
    float O = 0.f;
    if (M != -INFINITY)
#pragma unroll
      for (int w = 0; w < kWarpsTc; ++w) O = fmaf(mo[(w * G) * D + o], exp2f(s_m[w][head] - M), O);
    co[o] = O;
  }
  __syncthreads();
}

// The union of NT query tokens of a multi-token step: one pass over the rows
// the NT tokens selected together, every row staged once and attended by the
// query heads of each token that selected it (bit j of masks[e], the token
// bits of entry e; for the other tokens the row is masked).  Same tiles,
// pipeline and MMA layout as tc_segment, with NT sets of q fragments (q of
// token j at qs + j * G * D), softmax state and accumulators; the K and V
// fragments of a tile are loaded once for all tokens.  Per-warp shared
// memory: the stages, then NT P tiles.  Results, in shared memory: cm[j * G
// + h], cl[j * G + h], co[(j * G + h) * D + d].
template <class SH, int NT, int ST>
__device__ void tc_segment_union(const DeviceState& s, const TcParams& p, const SegArgs& a,
                                 const uint8_t* masks, unsigned char* smem, float* cm, float* cl,
                                 float* co, float (*s_m)[NT * SH::G],
                                 float (*s_l)[NT * SH::G]) {
  constexpr int D = SH::D, G = SH::G, NTN = SH::NTN, KS = SH::KS, MT = SH::MT;
  constexpr int PITCH = SH::PITCH;
  constexpr int NH = G == 1 ? 1 : 2;              // heads per thread
  constexpr int OWNERS = G >= 2 ? G / 2 : 1;      // lanes c < OWNERS own their heads
  constexpr int WB = ST * SH::STAGE_BYTES + NT * SH::PTILE_BYTES;
  static_assert(NT * 16 <= 64, "token row masks of a stage fit 64 bits");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int head_base = G == 1 ? 0 : 2 * (c % OWNERS);
  const bool owner = c < OWNERS;
  unsigned char* wbase = smem + warp * WB;
  unsigned char* ptile0 = wbase + ST * SH::STAGE_BYTES;
  const int u = a.u;

  float m[NT][NH], l[NT][NH];
  float acc[NT][MT][NTN][4];
#pragma unroll
  for (int j = 0; j < NT; ++j) {
#pragma unroll
    for (int h = 0; h < NH; ++h) {
      m[j][h] = -INFINITY;
      l[j][h] = 0.f;
    }
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int nt = 0; nt < NTN; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[j][mt][nt][i] = 0.f;
  }

  const int n_my = a.tb - a.ta - warp > 0 ? (a.tb - a.ta - warp + kWarpsTc - 1) / kWarpsTc : 0;
  // Buffer row of row (lane & 15) of this warp's i-th tile (or -1) and its token bits.
  auto row_index = [&](int i, uint32_t& tok_bits) -> long long {
    tok_bits = 0u;
    const int row = (a.ta + warp + i * kWarpsTc) * kTileRows + (lane & 15);
    if (i >= n_my || row >= a.rows) return -1;
    const int ent = a.ent_base + (p.ET == 1 ? row : row / p.ET);
    const int sub = row - (ent - a.ent_base) * p.ET;
    const int slot = a.list[ent];
    if (slot < 0 || !AVSG_IN_BOUNDS(slot < s.B, s.err, u, ent)) return -1;
    tok_bits = masks[ent];
    return ((long long)u * s.B + slot) * p.ET + sub;
  };
  constexpr int CPR = 2 * D / 16;  // 16-byte chunks per row
  constexpr int RPI = 32 / CPR;    // rows per warp instruction
  // Per stage: bits [16 j, 16 j + 16) mark the tile's rows token j selected.
  unsigned long long tm0 = 0, tm1 = 0, tm2 = 0;
  static_assert(ST == 2 || ST == 3, "two or three stage masks");
  auto issue = [&](long long myrow, uint32_t mybits, int st) {
    unsigned long long tm = 0;
#pragma unroll
    for (int j = 0; j < NT; ++j)
      tm |= (unsigned long long)(__ballot_sync(0xffffffffu, myrow >= 0 && ((mybits >> j) & 1u)) &
                                 0xFFFFu)
            << (16 * j);
    if (st == 0) tm0 = tm; else if (st == 1) tm1 = tm; else tm2 = tm;  // (tm2 unused at ST = 2)
    unsigned char* kst = wbase + st * SH::STAGE_BYTES;
    unsigned char* vst = SH::SHARED ? kst : kst + kTileRows * PITCH;
    const int ch = lane % CPR, rsub = lane / CPR;
#pragma unroll
    for (int it = 0; it < kTileRows / RPI; ++it) {
      const int r = it * RPI + rsub;
      const long long srow = __shfl_sync(0xffffffffu, myrow, r);
      if (srow >= 0) {
        cp_async16(kst + r * PITCH + ch * 16, s.kbuf + srow * (2 * D) + ch * 16);
        if (!SH::SHARED) cp_async16(vst + r * PITCH + ch * 16, s.vbuf + srow * (2 * D) + ch * 16);
      } else {
        *reinterpret_cast<uint4*>(kst + r * PITCH + ch * 16) = make_uint4(0u, 0u, 0u, 0u);
        if (!SH::SHARED) *reinterpret_cast<uint4*>(vst + r * PITCH + ch * 16) = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    cp_async_commit();
  };

  long long next_row;
  uint32_t next_bits;
  {
    long long first_rows[ST + 1];
    uint32_t first_bits[ST + 1];
#pragma unroll
    for (int i = 0; i <= ST; ++i) first_rows[i] = row_index(i, first_bits[i]);
#pragma unroll
    for (int i = 0; i < ST; ++i) issue(first_rows[i], first_bits[i], i);
    next_row = first_rows[ST];
    next_bits = first_bits[ST];
  }
  // q fragments of every token: column n < G is hi(q_n), G <= n < 2G is lo(q_{n-G})
  uint32_t qb[NT][KS][NTN][2];
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int nt = 0; nt < NTN; ++nt) {
      const int col = g + 8 * nt;
      const int head = col < G ? col : col - G;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        uint16_t e[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int d = 16 * ks + 2 * c + (i & 1) + 8 * (i >> 1);
          uint16_t hi = 0, lo = 0;
          if (col < 2 * G) split_bf16(a.qs[(j * G + head) * D + d] * p.scale_log2, hi, lo);
          e[i] = col < G ? hi : lo;
        }
        qb[j][ks][nt][0] = pack2(e[0], e[1]);
        qb[j][ks][nt][1] = pack2(e[2], e[3]);
      }
    }

  for (int i = 0; i < n_my; ++i) {
    const int st = i % ST;
    cp_async_wait<ST - 1>();
    __syncwarp();
    const unsigned long long tm = st == 0 ? tm0 : st == 1 ? tm1 : tm2;
    const unsigned char* kst = wbase + st * SH::STAGE_BYTES;
    const unsigned char* vst = SH::SHARED ? kst : kst + kTileRows * PITCH;
    const uint32_t kaddr = smem_u32(kst), vaddr = smem_u32(vst);

    // scores^T of every token; K fragments loaded once per k-step
    float sc[NT][NTN][4], sc2[NT][NTN][4];
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int nt = 0; nt < NTN; ++nt)
#pragma unroll
        for (int i2 = 0; i2 < 4; ++i2) sc[j][nt][i2] = sc2[j][nt][i2] = 0.f;
    {
      const int arow = (lane & 7) + ((lane >> 3) & 1) * 8;
      const int acol = (lane >> 4) * 8;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(kaddr + arow * PITCH + (16 * ks + acol) * 2, a0, a1, a2, a3);
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
          for (int nt = 0; nt < NTN; ++nt)
            mma_bf16((ks & 1) ? sc2[j][nt] : sc[j][nt], a0, a1, a2, a3, qb[j][ks][nt][0],
                     qb[j][ks][nt][1]);
      }
    }
#pragma unroll
    for (int j = 0; j < NT; ++j) {
#pragma unroll
      for (int nt = 0; nt < NTN; ++nt)
#pragma unroll
        for (int i2 = 0; i2 < 4; ++i2) sc[j][nt][i2] += sc2[j][nt][i2];
      float sv[2][2];
      if (G == 8) {
        sv[0][0] = sc[j][0][0] + sc[j][NTN - 1][0];
        sv[0][1] = sc[j][0][1] + sc[j][NTN - 1][1];
        sv[1][0] = sc[j][0][2] + sc[j][NTN - 1][2];
        sv[1][1] = sc[j][0][3] + sc[j][NTN - 1][3];
      } else if (G == 1) {
        sv[0][0] = sc[j][0][0] + sc[j][0][1];
        sv[1][0] = sc[j][0][2] + sc[j][0][3];
        sv[0][1] = sv[1][1] = -INFINITY;
      } else {
        const int xm = G / 2;
        sv[0][0] = sc[j][0][0] + __shfl_xor_sync(0xffffffffu, sc[j][0][0], xm);
        sv[0][1] = sc[j][0][1] + __shfl_xor_sync(0xffffffffu, sc[j][0][1], xm);
        sv[1][0] = sc[j][0][2] + __shfl_xor_sync(0xffffffffu, sc[j][0][2], xm);
        sv[1][1] = sc[j][0][3] + __shfl_xor_sync(0xffffffffu, sc[j][0][3], xm);
      }
      const unsigned vmask = (unsigned)(tm >> (16 * j)) & 0xFFFFu;  // rows token j selected
      if (!((vmask >> g) & 1u)) sv[0][0] = sv[0][1] = -INFINITY;
      if (!((vmask >> (g + 8)) & 1u)) sv[1][0] = sv[1][1] = -INFINITY;

      float pv[2][2], alpha[2] = {1.f, 1.f};
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        float mx = fmaxf(sv[0][h], sv[1][h]);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const float m_new = fmaxf(m[j][h], mx);
        float p0 = 0.f, p1 = 0.f;
        if (m_new != -INFINITY) {
          alpha[h] = exp2f(m[j][h] - m_new);
          p0 = exp2f(sv[0][h] - m_new);
          p1 = exp2f(sv[1][h] - m_new);
        }
        float sum = p0 + p1;
        sum += __shfl_xor_sync(0xffffffffu, sum, 4);
        sum += __shfl_xor_sync(0xffffffffu, sum, 8);
        sum += __shfl_xor_sync(0xffffffffu, sum, 16);
        l[j][h] = l[j][h] * alpha[h] + sum;
        m[j][h] = m_new;
        pv[0][h] = p0;
        pv[1][h] = p1;
      }
      if (NH == 1) alpha[1] = alpha[0];
      if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int nt = 0; nt < NTN; ++nt) {
            acc[j][mt][nt][0] *= alpha[0];
            acc[j][mt][nt][1] *= alpha[1];
            acc[j][mt][nt][2] *= alpha[0];
            acc[j][mt][nt][3] *= alpha[1];
          }
      }
      unsigned char* ptile = ptile0 + j * SH::PTILE_BYTES;
      if (owner) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int rr = g + 8 * h;
          uint16_t hi0, lo0, hi1 = 0, lo1 = 0;
          split_bf16(pv[h][0], hi0, lo0);
          if (NH == 2) split_bf16(pv[h][1], hi1, lo1);
          if (G == 1) {
            *reinterpret_cast<uint32_t*>(ptile + rr * 16) = pack2(hi0, lo0);
          } else {
            const int chi = head_base, clo = G + head_base;
            *reinterpret_cast<uint32_t*>(ptile + (chi >> 3) * 256 + rr * 16 + (chi & 7) * 2) =
                pack2(hi0, hi1);
            *reinterpret_cast<uint32_t*>(ptile + (clo >> 3) * 256 + rr * 16 + (clo & 7) * 2) =
                pack2(lo0, lo1);
          }
        }
      }
    }
    __syncwarp();
    uint32_t pb[NT][NTN][2];
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int nt = 0; nt < NTN; ++nt)
        ldsm_x2_t(smem_u32(ptile0 + j * SH::PTILE_BYTES + nt * 256 + (lane & 15) * 16), pb[j][nt][0],
                  pb[j][nt][1]);
    {
      const int vrow = (lane & 7) + ((lane >> 4) << 3);
      const int vcol = ((lane >> 3) & 1) * 8;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(vaddr + vrow * PITCH + (16 * mt + vcol) * 2, a0, a1, a2, a3);
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
          for (int nt = 0; nt < NTN; ++nt)
            mma_bf16(acc[j][mt][nt], a0, a1, a2, a3, pb[j][nt][0], pb[j][nt][1]);
      }
    }
    __syncwarp();  // every lane has read stage st and the P tiles
    issue(next_row, next_bits, st);
    next_row = row_index(i + ST + 1, next_bits);
  }
  cp_async_wait<0>();

  // Per-warp results -> shared memory [warp][token][head][D], then merge the 4 warps.
  __syncthreads();
  float* mo = reinterpret_cast<float*>(smem);
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int dv = 16 * mt + g + 8 * (i >> 1);
        float v;
        int head;
        if (G == 8) {
          v = acc[j][mt][0][i] + acc[j][mt][NTN - 1][i];
          head = 2 * c + (i & 1);
        } else if (G == 1) {
          v = (i & 1) ? 0.f : acc[j][mt][0][i] + acc[j][mt][0][i + 1];
          head = 0;
        } else {
          v = acc[j][mt][0][i] + __shfl_xor_sync(0xffffffffu, acc[j][mt][0][i], G / 2);
          head = head_base + (i & 1);
        }
        if (owner && (G != 1 || (i & 1) == 0)) mo[((warp * NT + j) * G + head) * D + dv] = v;
      }
  if (owner && g == 0) {
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        s_m[warp][j * G + head_base + h] = m[j][h];
        s_l[warp][j * G + head_base + h] = l[j][h];
      }
  }
  __syncthreads();
  if (tid < NT * G) {
    float M = -INFINITY, L = 0.f;
#pragma unroll
    for (int w = 0; w < kWarpsTc; ++w) M = fmaxf(M, s_m[w][tid]);
    if (M != -INFINITY)
#pragma unroll
      for (int w = 0; w < kWarpsTc; ++w) L = fmaf(s_l[w][tid], exp2f(s_m[w][tid] - M), L);
    cm[tid] = M;
    cl[tid] = L;
  }
  __syncthreads();
  for (int o = tid; o < NT * G * D; o += kThreadsTc) {
    const int jh = o / D;  // token * G + head
    const float M = cm[jh];
    float O = 0.f;
    if (M != -INFINITY)
#pragma unroll
      for (int w = 0; w < kWarpsTc; ++w)
        O = fmaf(mo[(w * NT * G + jh) * D + (o - jh * D)], exp2f(s_m[w][jh] - M), O);
    co[o] = O;
  }
  __syncthreads();
}

// Writes this CTA's segment result as partial `idx` of a pair.
template <int G, int D>
__device__ __forceinline__ void tc_write_partial(float* pp, const float* cm, const float* cl,
                                                 const float* co) {
  for (int o = threadIdx.x; o < G * D; o += kThreadsTc) pp[2 * G + o] = co[o];
  if (threadIdx.x < G) {
    pp[threadIdx.x] = cm[threadIdx.x];
    pp[G + threadIdx.x] = cl[threadIdx.x];
  }
}

// Merges nseg partials of a pair into its output (run by one CTA); value i
// of partial q2 (m of head h at i = h, l at G + h, output o at 2G + o) is
// part(q2, i).  Every partial's (m, l) and the first QB partials' output rows
// are loaded at once; later partials take one more round of loads per QB.
// wseg: 2 * nseg * G floats of shared memory.
template <int G, int D, class Part>
__device__ void tc_merge_partials(Part part, int nseg, float* out, float* wseg) {
  constexpr int R = (G * D + kThreadsTc - 1) / kThreadsTc;  // outputs per thread
  constexpr int QB = 8;                                     // partials per round of loads
  const int tid = threadIdx.x;
  float* wm = wseg;             // [nseg][G]: m, then the normalised weight
  float* wl = wseg + nseg * G;  // [nseg][G]: l
  for (int i = tid; i < nseg * G; i += kThreadsTc) {
    const int q2 = i / G, h = i - q2 * G;
    wm[i] = part(q2, h);
    wl[i] = part(q2, G + h);
  }
  float v[QB][R];
  auto load_round = [&](int q0) {
#pragma unroll
    for (int j = 0; j < QB; ++j)
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int o = tid + r * kThreadsTc;
        v[j][r] = (q0 + j < nseg && o < G * D) ? part(q0 + j, 2 * G + o) : 0.f;
      }
  };
  load_round(0);
  __syncthreads();
  if (tid < G) {
    float M = -INFINITY, L = 0.f;
    for (int q2 = 0; q2 < nseg; ++q2) M = fmaxf(M, wm[q2 * G + tid]);
    for (int q2 = 0; q2 < nseg; ++q2) {
      const float e = M == -INFINITY ? 0.f : exp2f(wm[q2 * G + tid] - M);
      wm[q2 * G + tid] = e;
      L = fmaf(wl[q2 * G + tid], e, L);
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    for (int q2 = 0; q2 < nseg; ++q2) wm[q2 * G + tid] *= inv;
  }
  __syncthreads();
  float O[R];
#pragma unroll
  for (int r = 0; r < R; ++r) O[r] = 0.f;
  for (int q0 = 0; q0 < nseg; q0 += QB) {
    if (q0) load_round(q0);
#pragma unroll
    for (int j = 0; j < QB; ++j)
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int o = tid + r * kThreadsTc;
        if (q0 + j < nseg && o < G * D) O[r] = fmaf(v[j][r], wm[(q0 + j) * G + o / D], O[r]);
      }
  }
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int o = tid + r * kThreadsTc;
    if (o < G * D) out[o] = O[r];
  }
}

// Single pass, persistent: 2 CTAs per SM, each an equal share of all tiles.
// A pair covered by several CTAs is merged from their partials.  A CTA's
// range cuts at most two pairs (its first and its last segment; the pairs in
// between it covers whole), so partials are stored by CTA: slot 2c for CTA
// c's first segment, 2c + 1 for its last one -- 2 * CTAs partials however
// many pairs there are.
template <class SH>
__global__ void __launch_bounds__(kThreadsTc) attn_tc_kernel(DeviceState s, TcParams p) {
  constexpr int D = SH::D, G = SH::G;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = (unsigned char*)(((uintptr_t)smem_raw + 127) & ~(uintptr_t)127);
  __shared__ float s_m[kWarpsTc][G], s_l[kWarpsTc][G], cm[G], cl[G];
  __shared__ int s_stop, s_last;
  const int tid = threadIdx.x;
  griddep_wait();
  griddep_launch();
  if (p.io) {  // this step's out and slot map (and q when it is not copied)
    const StepIO io = load_io(p.io);
    if (!p.q) p.q = io.q;
    p.out = io.out;
    p.slots = io.slot_map;
  }
  if (tid == 0) s_stop = load_err(s.err);
  __syncthreads();
  if (s_stop) return;
  float* co = reinterpret_cast<float*>(smem) + kWarpsTc * G * D;

  const long long T = p.tiles;
  const int C = p.ctas;
  const long long t_begin = (long long)blockIdx.x * T / C;
  const long long t_end = (long long)(blockIdx.x + 1) * T / C;
  const size_t stride = (size_t)G * (D + 2);
  for (long long t = t_begin; t < t_end;) {
    const int pair = (int)(t / p.tiles_per_pair);
    const long long pair_t0 = (long long)pair * p.tiles_per_pair;
    SegArgs a;
    a.pair = pair;
    a.u = pair / p.n_tok;
    a.tok = pair - a.u * p.n_tok;
    a.ent_base = 0;
    a.list = nullptr;
    a.qs = nullptr;
    a.rows = p.rows_per_pair;
    a.ta = (int)(t - pair_t0);
    a.tb = (int)(min(t_end, pair_t0 + p.tiles_per_pair) - pair_t0);
    const bool first_seg = t == t_begin;
    t = pair_t0 + a.tb;
    tc_segment<SH>(s, p, a, smem, cm, cl, co, s_m, s_l);

    const int first = cta_of_tile(pair_t0, C, T);
    const int last = cta_of_tile(pair_t0 + p.tiles_per_pair - 1, C, T);
    const int nseg = last - first + 1;
    float* out = p.out + (size_t)pair * G * D;
    if (nseg == 1) {
      for (int o = tid; o < G * D; o += kThreadsTc) {
        const float L = cl[o / D];
        out[o] = L > 0.f ? co[o] / L : 0.f;
      }
    } else {
      tc_write_partial<G, D>(s.part + (2 * (size_t)blockIdx.x + (first_seg ? 0 : 1)) * stride, cm,
                             cl, co);
      __threadfence();
      __syncthreads();
      if (tid == 0) s_last = atomicAdd(&s.part_count[a.u * kMaxTokens + a.tok], 1) == nseg - 1;
      __syncthreads();
      if (s_last) {
        __threadfence();
        // CTA `first` may have begun in an earlier pair (then this pair is its
        // last segment); every later CTA of the pair begins in it.
        const size_t slot0 = 2 * (size_t)first + ((long long)first * T / C == pair_t0 ? 0 : 1);
        const float* part = s.part;
        tc_merge_partials<G, D>(
            [&](int q2, int i) {
              return __ldcg(part + (q2 == 0 ? slot0 : 2 * (size_t)(first + q2)) * stride + i);
            },
            nseg, out, co + G * D);
        if (tid == 0) s.part_count[a.u * kMaxTokens + a.tok] = 0;
      }
    }
    __syncthreads();  // the merge area is staging again for the next segment
  }
}

// Hit-pass partials of the two-pass attention, G * (D + 2) floats each, in
// two groups: [pairs] the partial of a pair one CTA covered whole;
// [2 * hit_ctas] the partials of the pairs a CTA cut (its first and its last
// segment, as in the single pass).  The miss pass merges them with its own
// result, which never leaves its shared memory.
__device__ __forceinline__ int hit_segments(const TcParams& p, int pair, long long* slot0) {
  const long long T = p.tiles, t0 = (long long)pair * p.tiles_per_pair;
  const int C = p.hit_ctas;
  const int first = cta_of_tile(t0, C, T), last = cta_of_tile(t0 + p.tiles_per_pair - 1, C, T);
  const long long pairs = T / p.tiles_per_pair;
  *slot0 = first == last ? pair : pairs + 2LL * first + ((long long)first * T / C == t0 ? 0 : 1);
  return last - first + 1;
}
// Slot of a pair's hit-pass partial q2 (q2 < its hit_segments).
__device__ __forceinline__ long long two_pass_slot(const TcParams& p, int pair, int nseg_h,
                                                   long long slot0, int q2) {
  (void)nseg_h;
  const long long pairs = p.tiles / p.tiles_per_pair;
  if (q2 == 0) return slot0;
  const int first = (int)((slot0 - pairs) >> 1);
  return pairs + 2LL * (first + q2);
}

// Hit pass: every selected position of every (unit, token), with the hit
// slots that match wrote (a miss has slot -1 and is masked); runs while the
// missed rows are still crossing the host link.  Persistent: 2 CTAs per SM,
// each an equal contiguous share of all pairs' 16-row tiles, so every SM
// gets the same work whatever the pair count.  A CTA writes one partial per
// pair segment it covers (see hit_segments).
template <class SH>
__global__ void __launch_bounds__(kThreadsTc) attn_tc_hits_kernel(DeviceState s, TcParams p) {
  constexpr int D = SH::D, G = SH::G;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = (unsigned char*)(((uintptr_t)smem_raw + 127) & ~(uintptr_t)127);
  __shared__ float s_m[kWarpsTc][G], s_l[kWarpsTc][G], cm[G], cl[G];
  __shared__ __align__(16) float s_q[G * D];
  __shared__ int s_stop;
  const int tid = threadIdx.x;
  griddep_wait();
  if (tid == 0) s_stop = load_err(s.err);
  __syncthreads();
  if (s_stop) {
    griddep_launch();
    return;
  }
  float* co = reinterpret_cast<float*>(smem) + kWarpsTc * G * D;
  const long long T = p.tiles, pairs = T / p.tiles_per_pair;
  const int C = p.hit_ctas;
  const long long t_begin = (long long)blockIdx.x * T / C;
  const long long t_end = (long long)(blockIdx.x + 1) * T / C;
  const size_t stride = (size_t)G * (D + 2);
  for (long long t = t_begin; t < t_end;) {
    const int pair = (int)(t / p.tiles_per_pair);
    const long long pair_t0 = (long long)pair * p.tiles_per_pair;
    // this pair's q (the copy match made) -> shared memory
    for (int i = tid; i < G * D / 4; i += kThreadsTc)
      cp_async16(s_q + 4 * i, p.q + (size_t)pair * G * D + 4 * i);
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();
    SegArgs a;
    a.pair = pair;
    a.u = pair / p.n_tok;
    a.tok = pair - a.u * p.n_tok;
    a.ent_base = 0;
    a.list = nullptr;
    a.qs = s_q;
    a.rows = p.k * p.ET;
    a.ta = (int)(t - pair_t0);
    a.tb = (int)(min(t_end, pair_t0 + p.tiles_per_pair) - pair_t0);
    const bool first_seg = t == t_begin;
    const bool whole = a.ta == 0 && a.tb == p.tiles_per_pair;
    t = pair_t0 + a.tb;
    tc_segment<SH>(s, p, a, smem, cm, cl, co, s_m, s_l);
    const long long slot = whole ? pair : pairs + 2LL * blockIdx.x + (first_seg ? 0 : 1);
    tc_write_partial<G, D>(s.part + (size_t)slot * stride, cm, cl, co);
    __syncthreads();  // the staging (and s_q) is reused by the next segment
  }
  griddep_launch();  // dependents launch as this pass ends, not while it needs the SMs
}

// Miss pass: the rows this step copied from host into its half of the
// staging area, attended once the gather is done.  The list comes from the
// reservation's descriptors of the unit (each with the row's miss-set cell
// and the bits of the tokens that selected it), in chunks of kMissChunk
// entries whose results are merged as they come.  NT == 1: CTA = one (unit,
// token), over the unit's misses that token selected.  NT > 1 (a step of NT
// query tokens): a cluster of kUnionCluster CTAs per unit, CTA r on the r-th
// contiguous share of the unit's descriptors, over the union of its misses,
// each row attended by the tokens that selected it (tc_segment_union).  After
// a cluster barrier, CTA j merges token j's hit-pass partials with the
// cluster's miss results (read from the CTAs' shared memories) into the
// output; a second barrier keeps every CTA's shared memory alive until then.
// The grid-dependency wait covers the gather, and the launch follows the
// reservation and the hit pass.  `s` is the real state.
constexpr int kMissChunk = 512;

// Stages per warp of the union pass: two, so that two of its CTAs share an
// SM; and CTAs per unit (a cluster, merged through distributed shared memory).
constexpr int kUnionStages = 2;
constexpr int kUnionCluster = 2;

template <class SH, int NT>
struct MissSmem {
  static constexpr int ST = NT > 1 ? kUnionStages : kStages;               // stages per warp
  static constexpr int WB = ST * SH::STAGE_BYTES + NT * SH::PTILE_BYTES;  // per warp
  static constexpr int LIST = kWarpsTc * WB;                                  // [kMissChunk] cells
  static constexpr int MASKS = LIST + kMissChunk * 4;                         // [kMissChunk] bits
  static constexpr int RUN = MASKS + (NT > 1 ? kMissChunk : 0);                // [NT][G][D]
  static constexpr int BYTES = RUN + NT * SH::G * SH::D * 4 + 128;
  static_assert(kWarpsTc * NT * SH::G * SH::D * 4 + NT * SH::G * SH::D * 4 <= kWarpsTc * WB,
                "per-warp results and the segment result fit the staging");
  static_assert(MASKS % 16 == 0 && RUN % 16 == 0, "alignment");
};

template <class SH, int NT>
__global__ void __launch_bounds__(kThreadsTc) attn_tc_miss_kernel(DeviceState s, TcParams p) {
  constexpr int D = SH::D, G = SH::G;
  using L = MissSmem<SH, NT>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = (unsigned char*)(((uintptr_t)smem_raw + 127) & ~(uintptr_t)127);
  int32_t* list = reinterpret_cast<int32_t*>(smem + L::LIST);
  uint8_t* masks = smem + L::MASKS;
  float* run_o = reinterpret_cast<float*>(smem + L::RUN);
  __shared__ float s_m[kWarpsTc][NT * G], s_l[kWarpsTc][NT * G], cm[NT * G], cl[NT * G];
  __shared__ float run_m[NT * G], run_l[NT * G], wa[NT * G], wb[NT * G];
  __shared__ __align__(16) float s_q[NT * G * D];
  __shared__ int s_stop, s_wsum[kWarpsTc];
  cg::cluster_group clu = cg::this_cluster();
  const int cs = (int)clu.num_blocks(), crank = (int)clu.block_rank();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int u = NT == 1 ? (int)blockIdx.y / p.n_tok : (int)blockIdx.y;
  const int tok0 = NT == 1 ? (int)blockIdx.y - u * p.n_tok : 0;
  // q of the CTA's token(s): match wrote it before the gather began
  for (int i = tid; i < NT * G * D / 4; i += kThreadsTc)
    cp_async16(s_q + 4 * i, p.q + ((size_t)u * p.n_tok + tok0) * G * D + 4 * i);
  cp_async_commit();
  for (int i = tid; i < NT * G; i += kThreadsTc) {
    run_m[i] = -INFINITY;
    run_l[i] = 0.f;
  }
  for (int i = tid; i < NT * G * D; i += kThreadsTc) run_o[i] = 0.f;
  griddep_wait();  // the gather's rows are in the staging area
  griddep_launch();
  if (tid == 0) s_stop = load_err(s.err);
  // the step's record and this unit's descriptor range of both parities,
  // loaded together (the range of the step's parity is then picked)
  const StepIO io = load_io(s.io);
  const int m_p[2] = {__ldcg(s.dcount + u), __ldcg(s.dcount + s.U + u)};
  const int b_p[2] = {__ldcg(s.dbase + u), __ldcg(s.dbase + s.U + u)};
  cp_async_wait<0>();
  __syncthreads();
  // (a CTA that stops skips its work, not the cluster barriers)
  const bool stop = s_stop != 0;
  const StepBufs sb = step_bufs(s, io.parity);
  DeviceState sv = s;  // the staged view: rows by miss-set cell in this step's half
  sv.kbuf = sb.kstage;
  sv.vbuf = sb.vstage;
  sv.B = s.MS;
  const int m = stop ? 0 : io.parity ? m_p[1] : m_p[0], base = io.parity ? b_p[1] : b_p[0];
  const GatherDesc* desc = sb.desc + base;
  float* co = reinterpret_cast<float*>(smem) + kWarpsTc * NT * G * D;
  // this CTA's contiguous share of the unit's descriptors
  const int d0 = (int)((long long)crank * m / cs), d1 = (int)((long long)(crank + 1) * m / cs);

  for (int c0 = d0; c0 < d1; c0 += kMissChunk) {
    const int cn = min(kMissChunk, d1 - c0);
    int nlist = cn;
    if (NT == 1) {
      // the chunk's entries this token selected, in descriptor order
      const uint32_t tokbit = 1u << tok0;
      constexpr int kPer = kMissChunk / kThreadsTc;
      int2 e[kPer];
      int cnt = 0;
#pragma unroll
      for (int r = 0; r < kPer; ++r) {
        const int i = tid * kPer + r;
        e[r] = i < cn ? __ldcg(reinterpret_cast<const int2*>(&desc[c0 + i].cell)) : make_int2(-1, 0);
        cnt += ((uint32_t)e[r].y & tokbit) ? 1 : 0;
      }
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (lane == 31) s_wsum[warp] = incl;
      __syncthreads();
      int pos = incl - cnt;
      nlist = 0;
#pragma unroll
      for (int w2 = 0; w2 < kWarpsTc; ++w2) {
        pos += w2 < warp ? s_wsum[w2] : 0;
        nlist += s_wsum[w2];
      }
#pragma unroll
      for (int r = 0; r < kPer; ++r)
        if ((uint32_t)e[r].y & tokbit) list[pos++] = e[r].x;
    } else {
      for (int i = tid; i < cn; i += kThreadsTc) {
        const int2 e = __ldcg(reinterpret_cast<const int2*>(&desc[c0 + i].cell));
        list[i] = e.x;
        masks[i] = (uint8_t)e.y;
      }
    }
    __syncthreads();
    SegArgs a;
    a.pair = u * p.n_tok + tok0;
    a.u = u;
    a.tok = tok0;
    a.ent_base = 0;
    a.list = list;
    a.qs = s_q;
    a.rows = nlist * p.ET;
    a.ta = 0;
    a.tb = (a.rows + kTileRows - 1) / kTileRows;
    if constexpr (NT == 1)
      tc_segment<SH>(sv, p, a, smem, cm, cl, co, s_m, s_l);
    else
      tc_segment_union<SH, NT, L::ST>(sv, p, a, masks, smem, cm, cl, co, s_m, s_l);
    // fold the chunk's result into the running one
    if (tid < NT * G) {
      const float M = fmaxf(run_m[tid], cm[tid]);
      const float x = M == -INFINITY ? 0.f : exp2f(run_m[tid] - M);
      const float y = M == -INFINITY ? 0.f : exp2f(cm[tid] - M);
      run_l[tid] = run_l[tid] * x + cl[tid] * y;
      run_m[tid] = M;
      wa[tid] = x;
      wb[tid] = y;
    }
    __syncthreads();
    for (int o = tid; o < NT * G * D; o += kThreadsTc) run_o[o] = run_o[o] * wa[o / D] + co[o] * wb[o / D];
    __syncthreads();
  }

  clu.sync();  // every CTA's miss result is in its shared memory

  // each pair's hit-pass partials (global) merged with the cluster's miss
  // results (shared memory of its CTAs): CTA j of the cluster merges token j
  const size_t stride = (size_t)G * (D + 2);
  for (int j = crank; j < NT && !stop; j += cs) {
    const int pair = u * p.n_tok + tok0 + j;
    long long slot0 = 0;
    const int nseg_h = hit_segments(p, pair, &slot0);
    const float* part = s.part;
    tc_merge_partials<G, D>(
        [&](int q2, int i) -> float {
          if (q2 >= nseg_h) {
            const unsigned r = (unsigned)(q2 - nseg_h);
            if (i < G) return *clu.map_shared_rank(run_m + j * G + i, r);
            if (i < 2 * G) return *clu.map_shared_rank(run_l + j * G + i - G, r);
            return *clu.map_shared_rank(run_o + j * G * D + i - 2 * G, r);
          }
          return __ldcg(part + (size_t)two_pass_slot(p, pair, nseg_h, slot0, q2) * stride + i);
        },
        nseg_h + cs, io.out + (size_t)pair * G * D, co);
    __syncthreads();
  }
  clu.sync();  // no CTA leaves while another reads its shared memory
}

template <class SH>
TcParams tc_params(const DeviceState& s, const AttnLaunch& a) {
  TcParams p{};
  p.n_tok = a.n_tok;
  p.k = a.k;
  p.ET = s.ET;
  p.identity = a.identity_slots;
  p.scale_log2 = a.scale_log2;
  p.q = a.q;
  p.out = a.out;
  p.io = a.io;
  return p;
}

template <class SH>
cudaError_t run_tc(const DeviceState& s, const AttnLaunch& a, int num_sms, cudaStream_t st) {
  static int smem_done = 0;
  TcParams p = tc_params<SH>(s, a);
  p.slots = a.slot_map;
  p.rows_per_pair = a.k * s.ET;
  p.tiles_per_pair = (p.rows_per_pair + kTileRows - 1) / kTileRows;
  const long long pairs = (long long)s.U * a.n_tok;
  p.tiles = pairs * p.tiles_per_pair;
  long long C = (long long)num_sms * kCtasPerSm;
  if (C > (p.tiles + kWarpsTc - 1) / kWarpsTc) C = (p.tiles + kWarpsTc - 1) / kWarpsTc;  // a tile per warp
  if (C < 1) C = 1;
  const size_t stride = (size_t)SH::G * (SH::D + 2);
  for (;;) {
    const long long per = p.tiles / C;  // fewest tiles a CTA gets
    p.max_seg = (int)((p.tiles_per_pair + per - 1) / per + 1);  // most CTAs on one pair
    // partials: two per CTA (see attn_tc_kernel); the merge's weights fit
    // the staging while max_seg <= MAX_SEG
    if ((2 * (size_t)C * stride <= a.part_capacity && p.max_seg <= SH::MAX_SEG) || C == 1) break;
    C = C * 3 / 4 > 0 ? C * 3 / 4 : 1;
  }
  (void)pairs;
  p.ctas = (int)C;
  cudaError_t e = ensure_smem((const void*)attn_tc_kernel<SH>, SH::SMEM, &smem_done);
  if (e != cudaSuccess) return e;
  return launch_pdl(attn_tc_kernel<SH>, dim3(p.ctas), dim3(kThreadsTc), SH::SMEM, st, s, p);
}

// The persistent hit pass's shape for a step: tiles per pair, all tiles,
// CTAs, and the most hit-pass partials one pair has.
struct HitGrid {
  int tiles_per_pair, ctas, max_seg;
  long long tiles;
};
inline HitGrid hit_grid(int pairs, int k, int ET, int num_sms) {
  HitGrid g;
  g.tiles_per_pair = (k * ET + kTileRows - 1) / kTileRows;
  g.tiles = (long long)pairs * g.tiles_per_pair;
  // at least one tile per warp: fewer, fuller CTAs leave fewer partials
  long long C = (long long)num_sms * kCtasPerSm;
  if (C > (g.tiles + kWarpsTc - 1) / kWarpsTc) C = (g.tiles + kWarpsTc - 1) / kWarpsTc;
  g.ctas = (int)(C < 1 ? 1 : C);
  const long long per = g.tiles / g.ctas;  // fewest tiles a CTA gets
  g.max_seg = (int)((g.tiles_per_pair + per - 1) / per + 1);
  return g;
}

template <class SH>
TcParams two_pass_params(const DeviceState& s, const AttnLaunch& a) {
  TcParams p = tc_params<SH>(s, a);
  p.slots = s.hslot;
  p.identity = 0;
  const HitGrid g = hit_grid(s.U * a.n_tok, a.k, s.ET, a.num_sms);
  p.tiles_per_pair = g.tiles_per_pair;
  p.tiles = g.tiles;
  p.hit_ctas = g.ctas;
  return p;
}

template <class SH>
cudaError_t run_tc_pass(const DeviceState& s, const AttnLaunch& a, int pass, cudaStream_t st) {
  static int smem_hits = 0;
  TcParams p = two_pass_params<SH>(s, a);
  p.evict_first = pass == 0 ? 1 : 0;
  const HitGrid g = hit_grid(s.U * a.n_tok, a.k, s.ET, a.num_sms);
  const size_t parts = (size_t)s.U * a.n_tok * 2 + 2 * (size_t)g.ctas;
  if (parts * SH::G * (SH::D + 2) > a.part_capacity || g.max_seg + kUnionCluster > SH::MAX_SEG)
    return cudaErrorInvalidValue;
  if (pass == 0) {
    cudaError_t e = ensure_smem((const void*)attn_tc_hits_kernel<SH>, SH::SMEM, &smem_hits);
    if (e != cudaSuccess) return e;
    // Not launched early: its CTAs would take every SM while match runs,
    // ahead of the reservation and the gather on the other streams.
    return launch_ex(false, attn_tc_hits_kernel<SH>, dim3((unsigned)g.ctas), dim3(kThreadsTc),
                     SH::SMEM, st, s, p);
  }
  // Miss pass: one CTA per unit over the union of its tokens' misses (2 or 3
  // tokens), else one per (unit, token).
  auto launch_miss = [&](auto nt_tag) -> cudaError_t {
    constexpr int NT = decltype(nt_tag)::value;
    static int smem_miss = 0;
    using L = MissSmem<SH, NT>;
    cudaError_t e = ensure_smem((const void*)attn_tc_miss_kernel<SH, NT>, L::BYTES, &smem_miss);
    if (e != cudaSuccess) return e;
    // The union pass: a cluster of kUnionCluster CTAs per unit, each on a
    // share of the unit's rows (two of its CTAs fit an SM).
    const int cs = NT > 1 ? kUnionCluster : 1;
    dim3 grid((unsigned)cs, (unsigned)(NT == 1 ? s.U * a.n_tok : s.U));
    // Launched early behind the gather (its CTAs wait for it): the launch
    // also follows the hit pass and the reservation, which release their
    // dependents only as they end, so the early CTAs take no SM the hit
    // pass still needs.
    return launch_pdl_cluster(cs, attn_tc_miss_kernel<SH, NT>, grid, dim3(kThreadsTc), L::BYTES,
                              st, s, p);
  };
  // (the union keeps NT sets of accumulators in registers: shapes with one
  // n-tile of query columns only)
  if constexpr (SH::NTN == 1) {
    if (a.n_tok == 2) return launch_miss(std::integral_constant<int, 2>());
    if (a.n_tok == 3) return launch_miss(std::integral_constant<int, 3>());
  }
  return launch_miss(std::integral_constant<int, 1>());
}

}  // namespace

bool attention_tc_supported(int D, int DV, int G, int kv_shared) {
  (void)kv_shared;
  return D == DV && (D == 64 || D == 128) && (G == 1 || G == 2 || G == 4 || G == 8);
}

size_t attention_tc_two_pass_floats(int pairs, int k, int ET, int G, int DV, int num_sms) {
  const HitGrid g = hit_grid(pairs, k, ET, num_sms);
  return ((size_t)pairs * 2 + 2 * (size_t)g.ctas) * (size_t)G * (DV + 2);
}

size_t attention_tc_part_floats(int U, int max_tokens, int G, int DV, int num_sms) {
  // pairs * max_seg <= T / floor(T / C) + 2 * pairs <= 2 * C + 2 * pairs (see run_tc)
  const size_t pairs = (size_t)U * max_tokens;
  return (2 * (size_t)num_sms * kCtasPerSm + 2 * pairs) * (size_t)G * (DV + 2);
}

cudaError_t launch_attention_tc_pass(const DeviceState& s, const AttnLaunch& a, int pass,
                                     cudaStream_t st) {
#define X(d, g, sh)                                                         \
  if (s.D == d && s.G == g && (s.kv_shared != 0) == sh)                     \
    return run_tc_pass<TcShape<d, g, sh>>(s, a, pass, st);
  X(128, 1, false) X(128, 2, false) X(128, 4, false) X(128, 8, false)
  X(128, 1, true) X(128, 2, true) X(128, 4, true) X(128, 8, true)
  X(64, 1, false) X(64, 2, false) X(64, 4, false) X(64, 8, false)
  X(64, 1, true) X(64, 2, true) X(64, 4, true) X(64, 8, true)
#undef X
  return cudaErrorInvalidValue;
}

cudaError_t launch_attention_tc(const DeviceState& s, const AttnLaunch& a, int num_sms,
                                cudaStream_t st) {
#define X(d, g, sh)                                                         \
  if (s.D == d && s.G == g && (s.kv_shared != 0) == sh)                     \
    return run_tc<TcShape<d, g, sh>>(s, a, num_sms, st);
  X(128, 1, false) X(128, 2, false) X(128, 4, false) X(128, 8, false)
  X(128, 1, true) X(128, 2, true) X(128, 4, true) X(128, 8, true)
  X(64, 1, false) X(64, 2, false) X(64, 4, false) X(64, 8, false)
  X(64, 1, true) X(64, 2, true) X(64, 4, true) X(64, 8, true)
#undef X
  return cudaErrorInvalidValue;
}

}  // namespace avsg
