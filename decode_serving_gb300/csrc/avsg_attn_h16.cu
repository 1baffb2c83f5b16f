// avsg_attn_h16: split-K decode attention on the tensor cores for 16 query
// heads per kv-head over wide rows whose K and V are one array (the latent
// cache: K = V = the 576-wide latent row).
//
// Same operation as avsg_attn.cu (the Attention operation of the Spin page,
// "Unifying Sparse Attention with Hierarchical Memory for Scalable
// Long-Context LLM Serving", section 2A, over exactly the rows DSA selected,
// AVSG page arxivdaily 2609.37538, English abstract).  At 16 heads a staged
// row is worth 32 flop per byte, more than the fp32 pipes keep up with, and
// the 16 heads fill the M = 16 side of mma.m16n8k16 (bf16 in, fp32
// accumulate) exactly:
// * scores S = Q K^T: A = the 16 query rows, as scale*log2(e)*q rounded to
//   bf16 (hi) plus the bf16 rounding of the remainder (lo), two MMAs per
//   k-step, so the scores keep about 16 more bits than a bf16 q would.  The
//   8 warps split the row width: each holds the A fragments of its k-steps
//   in registers for the whole CTA and covers all 32 rows of a tile (four
//   n-tiles, B read by ldmatrix); the 8 partial score tiles are summed by
//   the softmax.
// * online softmax in the log2 domain: one warp per 2 heads, lane = row.
// * O += P V: A = P (16 heads x 32 rows, split hi/lo the same way), B = the
//   staged rows through ldmatrix.trans; each warp owns 72 of the 576 output
//   columns, so the accumulators need no cross-warp sum.
// Rows are staged by 16-byte cp.async into padded rows (the ldmatrix reads
// are free of bank conflicts), two tiles in flight; the rows past the range
// are zero-filled so that masked rows add exact zeros.
// The CTAs of a (unit, token) form clusters of 8 over consecutive row ranges.
// A cluster merges its 8 partial softmaxes in distributed shared memory:
// each CTA publishes (max, sum) per head and its accumulators, works out the
// 8 ranks' weights from the maxima, then sums one eighth of the output
// columns over the 8 CTAs with those weights.  One cluster per pair writes
// the output.  With several, rank r of each cluster writes its column slice
// with the cluster's (max, sum) and counts its arrival; the last to arrive
// for a slice merges the clusters' slices into the output.  (Without room
// for the counters, the clusters write (max, sum, acc) partials in the
// layout of avsg_attn.cu and its merge kernel combines them.)
#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <math.h>
#include <stdlib.h>

#include "avsg_internal.cuh"

namespace avsg {
namespace {

namespace cg = cooperative_groups;

constexpr int kH = 16;                 // query heads per kv-head (the MMA's M)
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kRows = 32;              // rows per tile
constexpr int kStagesH = 2;
constexpr int kSPitch = 40;            // floats per head row of a partial score tile
constexpr int kPPitch = kRows * 2 + 16;  // bytes per head row of the bf16 P tile
constexpr int kCl = 8;                 // CTAs per cluster (the in-cluster merge)
constexpr int kMaxFused = 32;          // most clusters per pair the last-arriver merge takes

template <int D_>
struct H16Shape {
  static constexpr int D = D_;
  static constexpr int PITCH = 2 * D + 16;              // bytes per staged row
  static constexpr int CH = D / 8;                      // 16-byte chunks per row
  static constexpr int CPL = (CH + 31) / 32;            // chunks per lane of a row copy
  static constexpr int KS = D / 16;                     // k-steps of the score MMA
  static constexpr int KSW = (KS + kWarps - 1) / kWarps;  // most k-steps one warp takes
  static constexpr int NCOL = D / kWarps;               // output columns per warp
  static constexpr int NTW = NCOL / 8;                  // n-tiles per warp in O += P V
  static constexpr int STAGE_BYTES = kRows * PITCH;
  static constexpr int SRED_BYTES = kWarps * kH * kSPitch * 4;
  static constexpr int P_BYTES = 2 * kH * kPPitch;
  static constexpr int FIXED = kStagesH * STAGE_BYTES + SRED_BYTES + P_BYTES;
  static constexpr int RPITCH = D + 8;                  // floats per head row of the merge buffer
  static constexpr int CCOL = D / kCl;                  // output columns each cluster rank sums
  static_assert(D % (8 * kWarps) == 0, "row width must split into 8-column tiles per warp");
  static_assert(CCOL % 4 == 0, "cluster ranks sum float4 columns");
  static_assert(kH * RPITCH * 4 <= kStagesH * STAGE_BYTES, "merge buffer reuses the staging");
  static_assert(NTW >= 1 && NTW <= 16, "bad per-warp column count");
  static_assert(FIXED % 16 == 0, "alignment");
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// 16-byte async copy; src_bytes 0 writes 16 zero bytes and reads nothing.
__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2_t(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];"
               : "=r"(r0), "=r"(r1)
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// bf16 pair (x in the low half: the lower column) of the rounding of x, y and
// of what that rounding leaves.
__device__ __forceinline__ void split_pair(float x, float y, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat16 hx = __float2bfloat16_rn(x), hy = __float2bfloat16_rn(y);
  const __nv_bfloat16 lx = __float2bfloat16_rn(x - __bfloat162float(hx));
  const __nv_bfloat16 ly = __float2bfloat16_rn(y - __bfloat162float(hy));
  hi = (uint32_t)__bfloat16_as_ushort(hx) | ((uint32_t)__bfloat16_as_ushort(hy) << 16);
  lo = (uint32_t)__bfloat16_as_ushort(lx) | ((uint32_t)__bfloat16_as_ushort(ly) << 16);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <class SH>
__global__ void __launch_bounds__(kThreads, 2) attn_h16_kernel(DeviceState s, AttnLaunch a) {
  constexpr int D = SH::D, PITCH = SH::PITCH, CH = SH::CH, KS = SH::KS, KSW = SH::KSW;
  constexpr int NTW = SH::NTW;
  extern __shared__ __align__(16) unsigned char smem[];
  unsigned char* stage = smem;                                              // [2][kRows][PITCH]
  float* sred = reinterpret_cast<float*>(smem + kStagesH * SH::STAGE_BYTES);  // [8][16][kSPitch]
  unsigned char* pt = smem + kStagesH * SH::STAGE_BYTES + SH::SRED_BYTES;     // [hi,lo][16][kPPitch]
  int32_t* slots = reinterpret_cast<int32_t*>(smem + SH::FIXED);
  __shared__ float alpha_s[kH], m_s[kH], l_s[kH], w_s[kCl * kH], mc_s[kH], lc_s[kH];
  __shared__ float wm_s[kMaxFused * kH];  // fused merge: weight of each cluster per head
  __shared__ int s_stop, s_last;
  cg::cluster_group cl = cg::this_cluster();
  const int crank = (int)cl.block_rank();

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;  // fragment row (head) and column pair
  const int sp = blockIdx.x, u = blockIdx.y, tok = blockIdx.z;
  griddep_launch();
  const int k = a.k, ET = s.ET, S = gridDim.x;
  const int eps = (k + S - 1) / S;
  const int e0 = sp * eps;
  const int ne = max(0, min(k, e0 + eps) - e0);
  const int rows = ne * ET;
  const size_t sel_base = ((size_t)u * a.n_tok + tok) * (size_t)k;
  const uint32_t stage_u = smem_u32(stage);
  const unsigned char* kb = s.kbuf;
  const unsigned char* kstg = s.kstage;  // this step's half of the staging area (set below)
  // slots[e]: >= 0 the slot of a row resident before this step (a hit);
  // -1 not known yet; <= -2 for a row this step's gather writes: its slot
  // (-2 - value), or with staged misses its miss-set cell.  which: 0 every
  // row, 1 the resident rows and the zero rows past the range, 2 the
  // gathered rows.  A slot or cell out of range (only after a latched
  // error) reads as a zero row.
  // Staged misses: the kernel this one waits for is the staged gather, and
  // both know a miss by its cell from match alone.
  const bool early = !a.identity_slots && a.io != nullptr;
  const bool staged = early && a.staged_misses != 0;
  // Warp w copies rows w, w + 8, ... of a tile (the row's slot and address
  // are worked out once per warp); lane l takes its 16-byte chunks l, l + 32
  // and l + 64.
  auto issue = [&](int tile, int buf, int which) {
    const int r0 = tile * kRows;
    for (int r = warp; r < kRows; r += kWarps) {
      const int row = r0 + r;
      const uint32_t dst = stage_u + (uint32_t)((buf * kRows + r) * PITCH) + lane * 16;
      const unsigned char* src = nullptr;  // a zero row
      if (row < rows) {
        const int ent = ET == 1 ? row : row / ET, sub = row - ent * ET;
        int sl = slots[ent];
        const bool late = sl <= -2;
        if ((which == 1 && sl < 0) || (which == 2 && !late)) continue;
        if (late) sl = -2 - sl;
        const bool stg = late && staged;  // a missed row, at its cell of the staging area
        const int nb = stg ? s.MS : s.B;
        if (sl >= 0 && sl < nb)
          src = (stg ? kstg : kb) + (((size_t)u * nb + sl) * ET + sub) * (size_t)(2 * D) + lane * 16;
      } else if (which == 2) {
        continue;
      }
      if (row < rows && !src) {
        const int ent = ET == 1 ? row : row / ET;
        const int sl = slots[ent] <= -2 ? -2 - slots[ent] : slots[ent];
        (void)AVSG_IN_BOUNDS(sl < 0 || sl < (slots[ent] <= -2 && staged ? s.MS : s.B), s.err, u, ent);
      }
#pragma unroll
      for (int j = 0; j < SH::CPL; ++j)
        if (lane + 32 * j < CH) cp_async16_zfill(dst + 512 * j, src ? src + 512 * j : kb, src ? 16 : 0);
    }
  };
  const int ntiles_all = (rows + kRows - 1) / kRows;

  // Reuse path: match (this step's first kernel) wrote the step's I/O, the
  // hit slots and the copy of q, and no kernel of the step writes a hit
  // row's slot, so those rows stream in while the gather (the kernel this
  // one waits for) runs.
  if (early) {
    const StepIO io = load_io(a.io);
    a.out = io.out;
    a.slot_map = io.slot_map;
    if (staged) kstg = step_bufs(s, io.parity).kstage;
    for (int i = tid; i < ne; i += kThreads) {
      const int sl = __ldcg(s.hslot + sel_base + e0 + i);
      slots[i] = sl >= 0 ? sl : !staged ? -1 : sl <= -2 ? sl : -2 - s.MS;
    }
    __syncthreads();
    issue(0, 0, 1);
    if (ntiles_all > 1) issue(1, 1, 1);
  }

  // A fragments of this warp's k-steps (q pre-scaled, hi and lo), for the
  // whole CTA: rows g and g + 8, columns 2c, 2c + 1 and 2c + 8, 2c + 9.
  const int ks0 = warp * KS / kWarps, ks1 = (warp + 1) * KS / kWarps;
  uint32_t qa[KSW][2][4];
  auto load_q = [&]() {
    const float* q0 = a.q + (((size_t)u * a.n_tok + tok) * kH + g) * D;
    const float* q1 = q0 + 8 * D;
    const float sc = a.scale_log2;
#pragma unroll
    for (int kk = 0; kk < KSW; ++kk) {
      const int ks = ks0 + kk;
      if (ks < ks1) {
        const int col = ks * 16 + 2 * c;
        const float2 x0 = __ldcg(reinterpret_cast<const float2*>(q0 + col));
        const float2 x1 = __ldcg(reinterpret_cast<const float2*>(q1 + col));
        const float2 x2 = __ldcg(reinterpret_cast<const float2*>(q0 + col + 8));
        const float2 x3 = __ldcg(reinterpret_cast<const float2*>(q1 + col + 8));
        split_pair(x0.x * sc, x0.y * sc, qa[kk][0][0], qa[kk][1][0]);
        split_pair(x1.x * sc, x1.y * sc, qa[kk][0][1], qa[kk][1][1]);
        split_pair(x2.x * sc, x2.y * sc, qa[kk][0][2], qa[kk][1][2]);
        split_pair(x3.x * sc, x3.y * sc, qa[kk][0][3], qa[kk][1][3]);
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) qa[kk][0][j] = qa[kk][1][j] = 0u;
      }
    }
  };
  const bool q_early = a.q != nullptr;  // match's copy; else the caller's q, known after the wait
  if (q_early) load_q();

  griddep_wait();
  if (a.io && !early) {
    const StepIO io = load_io(a.io);
    if (!a.q) a.q = io.q;
    a.out = io.out;
    a.slot_map = io.slot_map;
  }
  if (tid == 0) s_stop = load_err(s.err);
  __syncthreads();
  // A stopped CTA skips its rows but still takes part in every cluster
  // barrier below, so no CTA of the cluster waits for one that left.
  const bool run = s_stop == 0;
  if (!q_early) load_q();
  if (run) {
    if (staged) {
      issue(0, 0, 2);
      if (ntiles_all > 1) issue(1, 1, 2);
    } else if (early) {  // the gathered rows' slots, from the slot map
      for (int i = tid; i < ne; i += kThreads)
        if (slots[i] < 0) {
          const int sl = __ldcg(a.slot_map + sel_base + e0 + i);
          slots[i] = -2 - (sl >= 0 && sl < s.B ? sl : s.B);
        }
      __syncthreads();
      issue(0, 0, 2);
      if (ntiles_all > 1) issue(1, 1, 2);
    } else {
      for (int i = tid; i < ne; i += kThreads)
        slots[i] = a.identity_slots ? tok * k + e0 + i : __ldcg(a.slot_map + sel_base + e0 + i);
      __syncthreads();
      issue(0, 0, 0);
      if (ntiles_all > 1) issue(1, 1, 0);
    }
  }
  cp_async_commit();  // tiles 0 and 1 (both in this group)
  cp_async_commit();  // (empty: the loop expects one group per tile)
  const int ntiles = run ? ntiles_all : 0;

  float acc[NTW][4];
#pragma unroll
  for (int n = 0; n < NTW; ++n)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[n][j] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};  // heads 2*warp, 2*warp + 1

  const int lm = lane >> 3, lr = lane & 7;  // ldmatrix: matrix index and row of the address
  const uint32_t pt_u = smem_u32(pt);
  for (int tl = 0; tl < ntiles; ++tl) {
    const int buf = tl & 1;
    const int nvalid = min(kRows, rows - tl * kRows);
    const uint32_t tile_u = stage_u + (uint32_t)(buf * SH::STAGE_BYTES);
    cp_async_wait<1>();
    __syncthreads();
    {  // this warp's k-steps of S = Q K^T for the tile's 32 rows
      float sacc[4][4], slo[4][4];  // hi and lo products in separate chains, summed after
#pragma unroll
      for (int n = 0; n < 4; ++n)
#pragma unroll
        for (int j = 0; j < 4; ++j) sacc[n][j] = slo[n][j] = 0.f;
#pragma unroll
      for (int kk = 0; kk < KSW; ++kk) {
        const int ks = ks0 + kk;
        if (ks < ks1) {
          // matrix lm of each x4: n-tile (lm >> 1) (+2), columns ks*16 + (lm & 1)*8
          uint32_t b01[4], b23[4];
          const uint32_t off = (uint32_t)(((lm >> 1) * 8 + lr) * PITCH + (ks * 16 + (lm & 1) * 8) * 2);
          ldsm_x4(tile_u + off, b01);
          ldsm_x4(tile_u + off + 16 * PITCH, b23);
          mma_bf16(sacc[0], qa[kk][0], b01[0], b01[1]);
          mma_bf16(slo[0], qa[kk][1], b01[0], b01[1]);
          mma_bf16(sacc[1], qa[kk][0], b01[2], b01[3]);
          mma_bf16(slo[1], qa[kk][1], b01[2], b01[3]);
          mma_bf16(sacc[2], qa[kk][0], b23[0], b23[1]);
          mma_bf16(slo[2], qa[kk][1], b23[0], b23[1]);
          mma_bf16(sacc[3], qa[kk][0], b23[2], b23[3]);
          mma_bf16(slo[3], qa[kk][1], b23[2], b23[3]);
        }
      }
#pragma unroll
      for (int n = 0; n < 4; ++n)
#pragma unroll
        for (int j = 0; j < 4; ++j) sacc[n][j] += slo[n][j];
      float* sw = sred + warp * kH * kSPitch;
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        *reinterpret_cast<float2*>(sw + g * kSPitch + n * 8 + 2 * c) = make_float2(sacc[n][0], sacc[n][1]);
        *reinterpret_cast<float2*>(sw + (g + 8) * kSPitch + n * 8 + 2 * c) =
            make_float2(sacc[n][2], sacc[n][3]);
      }
    }
    __syncthreads();
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {  // online softmax, heads 2*warp and 2*warp + 1, lane = row
      const int h = 2 * warp + hh;
      float sv = 0.f;
#pragma unroll
      for (int w2 = 0; w2 < kWarps; ++w2) sv += sred[(w2 * kH + h) * kSPitch + lane];
      sv = lane < nvalid ? sv : -INFINITY;
      const float m_new = fmaxf(m_run[hh], warp_max(sv));
      float alpha = 1.f, p = 0.f;
      if (m_new != -INFINITY) {
        alpha = exp2f(m_run[hh] - m_new);
        p = exp2f(sv - m_new);
      }
      l_run[hh] = l_run[hh] * alpha + warp_sum(p);
      m_run[hh] = m_new;
      const __nv_bfloat16 ph = __float2bfloat16_rn(p);
      const __nv_bfloat16 pl = __float2bfloat16_rn(p - __bfloat162float(ph));
      reinterpret_cast<__nv_bfloat16*>(pt + h * kPPitch)[lane] = ph;
      reinterpret_cast<__nv_bfloat16*>(pt + (kH + h) * kPPitch)[lane] = pl;
      if (lane == 0) alpha_s[h] = alpha;
    }
    __syncthreads();
    {  // O += P V over this warp's columns
      const float al0 = alpha_s[g], al1 = alpha_s[g + 8];
#pragma unroll
      for (int n = 0; n < NTW; ++n) {
        acc[n][0] *= al0;
        acc[n][1] *= al0;
        acc[n][2] *= al1;
        acc[n][3] *= al1;
      }
      const int cbase = warp * SH::NCOL;
#pragma unroll
      for (int kq = 0; kq < kRows / 16; ++kq) {
        // A: matrix lm = heads (lm & 1)*8.., rows kq*16 + (lm >> 1)*8..
        uint32_t pa_hi[4], pa_lo[4];
        const uint32_t aoff = (uint32_t)(((lm & 1) * 8 + lr) * kPPitch + (kq * 16 + (lm >> 1) * 8) * 2);
        ldsm_x4(pt_u + aoff, pa_hi);
        ldsm_x4(pt_u + kH * kPPitch + aoff, pa_lo);
        // B: matrix lm = rows kq*16 + (lm & 1)*8.., columns of n-tile 2j + (lm >> 1)
        const uint32_t brow = tile_u + (uint32_t)((kq * 16 + (lm & 1) * 8 + lr) * PITCH);
#pragma unroll
        for (int j = 0; j < NTW / 2; ++j) {
          uint32_t b[4];
          ldsm_x4_t(brow + (uint32_t)((cbase + (2 * j + (lm >> 1)) * 8) * 2), b);
          mma_bf16(acc[2 * j], pa_hi, b[0], b[1]);
          mma_bf16(acc[2 * j], pa_lo, b[0], b[1]);
          mma_bf16(acc[2 * j + 1], pa_hi, b[2], b[3]);
          mma_bf16(acc[2 * j + 1], pa_lo, b[2], b[3]);
        }
        if (NTW & 1) {
          uint32_t b0, b1;
          ldsm_x2_t(brow + (uint32_t)((cbase + (NTW - 1) * 8) * 2), b0, b1);
          mma_bf16(acc[NTW - 1], pa_hi, b0, b1);
          mma_bf16(acc[NTW - 1], pa_lo, b0, b1);
        }
      }
    }
    __syncthreads();
    if (tl + 2 < ntiles) issue(tl + 2, buf, 0);
    cp_async_commit();
  }
  cp_async_wait<0>();
  __syncthreads();  // the staging is free: it takes this rank's accumulators
  if (lane == 0) {
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      m_s[2 * warp + hh] = m_run[hh];
      l_s[2 * warp + hh] = l_run[hh];
    }
  }
  float* red = reinterpret_cast<float*>(stage);  // [16][RPITCH], this rank's acc
  {
    const int cbase = warp * SH::NCOL;
#pragma unroll
    for (int n = 0; n < NTW; ++n) {
      const int col = cbase + n * 8 + 2 * c;
      *reinterpret_cast<float2*>(red + g * SH::RPITCH + col) = make_float2(acc[n][0], acc[n][1]);
      *reinterpret_cast<float2*>(red + (g + 8) * SH::RPITCH + col) = make_float2(acc[n][2], acc[n][3]);
    }
  }
  cl.sync();  // every rank's (max, sum) and accumulators are published

  // weight of rank r for head h: exp2(m_r - M) with M the cluster's max;
  // the cluster's sum L = sum over r of l_r times that weight
  if (tid < kCl * kH) {
    const int r = tid / kH, h = tid - r * kH;
    float mr[kCl];
#pragma unroll
    for (int q = 0; q < kCl; ++q) mr[q] = *cl.map_shared_rank(&m_s[h], q);
    float M = -INFINITY;
#pragma unroll
    for (int q = 0; q < kCl; ++q) M = fmaxf(M, mr[q]);
    float mine = 0.f;
#pragma unroll
    for (int q = 0; q < kCl; ++q)
      if (q == r) mine = mr[q] == -INFINITY ? 0.f : exp2f(mr[q] - M);
    w_s[r * kH + h] = mine;
    if (r == 0) {
      float L = 0.f;
#pragma unroll
      for (int q = 0; q < kCl; ++q)
        if (mr[q] != -INFINITY) L = fmaf(*cl.map_shared_rank(&l_s[h], q), exp2f(mr[q] - M), L);
      mc_s[h] = M;
      lc_s[h] = L;
    }
  }
  __syncthreads();

  // this rank's columns, summed over the cluster
  const int DV = D;
  const int nclu = S / kCl, clu = sp / kCl;
  const size_t pair = (size_t)u * a.n_tok + tok;
  constexpr int BS = 2 * kH + kH * SH::CCOL;  // a cluster's slice: (max, sum) per head, columns
  const bool fused = nclu > 1 && a.fused_merge;
  float* dst;       // where column col of head h goes: dst + h * hstride + col - cbias
  size_t hstride;
  int cbias = 0;
  if (nclu == 1) {
    dst = a.out + pair * (size_t)kH * DV;
    hstride = DV;
  } else if (fused) {
    float* blk = s.part + ((pair * kCl + crank) * nclu + clu) * (size_t)BS;
    if (tid < kH && run) {
      blk[tid] = mc_s[tid];
      blk[kH + tid] = lc_s[tid];
    }
    dst = blk + 2 * kH;
    hstride = SH::CCOL;
    cbias = crank * SH::CCOL;
  } else {
    float* pp = s.part + (pair * nclu + clu) * (size_t)kH * (DV + 2);
    if (crank == 0 && tid < kH && run) {
      pp[tid] = mc_s[tid];
      pp[kH + tid] = lc_s[tid];
    }
    dst = pp + 2 * kH;
    hstride = DV;
  }
  constexpr int C4 = SH::CCOL / 4;
  for (int i = tid; i < kH * C4; i += kThreads) {
    const int h = i / C4, col = crank * SH::CCOL + (i - h * C4) * 4;
    float4 x[kCl];
#pragma unroll
    for (int r = 0; r < kCl; ++r)
      x[r] = *reinterpret_cast<const float4*>(cl.map_shared_rank(red + h * SH::RPITCH + col, r));
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int r = 0; r < kCl; ++r) {
      const float wr = w_s[r * kH + h];
      v.x = fmaf(wr, x[r].x, v.x);
      v.y = fmaf(wr, x[r].y, v.y);
      v.z = fmaf(wr, x[r].z, v.z);
      v.w = fmaf(wr, x[r].w, v.w);
    }
    if (nclu == 1) {
      const float L = lc_s[h];
      const float inv = L > 0.f ? 1.f / L : 0.f;
      v.x *= inv;
      v.y *= inv;
      v.z *= inv;
      v.w *= inv;
    }
    if (run) *reinterpret_cast<float4*>(dst + (size_t)h * hstride + col - cbias) = v;
  }
  cl.sync();  // no rank leaves while another still reads its shared memory
  if (!fused || !run) return;

  // Arrival count per (pair, column slice): the last cluster to write its
  // slice merges the slices of all nclu clusters and writes the output
  // columns (the counter goes back to 0 for the next step).
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    int32_t* cnt = s.part_count + pair * kCl + crank;
    s_last = atomicAdd(cnt, 1) == nclu - 1;
    if (s_last) *cnt = 0;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const float* b0 = s.part + (pair * kCl + crank) * nclu * (size_t)BS;
  if (tid < kH) {
    float M = -INFINITY;
    for (int q = 0; q < nclu; ++q) M = fmaxf(M, __ldcg(b0 + (size_t)q * BS + tid));
    float L = 0.f;
    for (int q = 0; q < nclu; ++q) {
      const float mq = __ldcg(b0 + (size_t)q * BS + tid);
      const float wq = mq == -INFINITY ? 0.f : exp2f(mq - M);
      wm_s[q * kH + tid] = wq;
      L = fmaf(__ldcg(b0 + (size_t)q * BS + kH + tid), wq, L);
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    for (int q = 0; q < nclu; ++q) wm_s[q * kH + tid] *= inv;
  }
  __syncthreads();
  float* out = a.out + pair * (size_t)kH * DV;
  for (int i = tid; i < kH * C4; i += kThreads) {
    const int h = i / C4, c4 = (i - h * C4) * 4;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int q = 0; q < nclu; ++q) {
      const float4 x = __ldcg(reinterpret_cast<const float4*>(b0 + (size_t)q * BS + 2 * kH + h * SH::CCOL + c4));
      const float wq = wm_s[q * kH + h];
      v.x = fmaf(wq, x.x, v.x);
      v.y = fmaf(wq, x.y, v.y);
      v.z = fmaf(wq, x.z, v.z);
      v.w = fmaf(wq, x.w, v.w);
    }
    *reinterpret_cast<float4*>(out + (size_t)h * DV + crank * SH::CCOL + c4) = v;
  }
}

// a.splits (the caller's split count) rounded up to whole clusters: 8 CTAs
// per cluster, and one merged partial per cluster.
template <class SH>
cudaError_t run(const DeviceState& s, const AttnLaunch& a, cudaStream_t st) {
  static int smem_done = 0;
  static const int nclu_env = [] {
    const char* v = getenv("AVSG_H16_CLUSTERS");
    return (v && *v) ? atoi(v) : 0;
  }();
  // At most one CTA per SM in all, so that the grid, resident early and
  // waiting on the gather, leaves room for the reservation's kernels; a
  // larger grid (many pairs) is launched once the gather is done.
  const long long pairs = (long long)s.U * a.n_tok;
  int nclu = nclu_env > 0 ? nclu_env : (a.splits + kCl - 1) / kCl;
  if (nclu_env <= 0 && a.num_sms > 0) {
    const long long fit = a.num_sms / (kCl * pairs);
    if (fit >= 1 && nclu > fit) nclu = (int)fit;
  }
  const bool early = a.num_sms > 0 && (long long)nclu * kCl * pairs <= a.num_sms;
  const int ctas = nclu * kCl;
  static_assert(kCountsPerPair >= kCl, "one arrival counter per cluster rank");
  AttnLaunch b = a;
  b.fused_merge = nclu > 1 && nclu <= kMaxFused && (size_t)pairs * kCl <= a.count_capacity;
  const size_t part = b.fused_merge ? (size_t)pairs * kCl * nclu * (2 * kH + kH * SH::CCOL)
                                    : (size_t)pairs * nclu * kH * (s.DV + 2);
  if (nclu > 1 && part > a.part_capacity) return cudaErrorInvalidValue;
  const int eps = (a.k + ctas - 1) / ctas;
  const size_t smem = SH::FIXED + ((size_t)eps * 4 + 15) / 16 * 16;
  cudaError_t e = ensure_smem((const void*)attn_h16_kernel<SH>, smem, &smem_done);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ctas, (unsigned)s.U, (unsigned)a.n_tok);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = early && pdl_enabled() ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, attn_h16_kernel<SH>, s, b);
  if (e != cudaSuccess || nclu == 1 || b.fused_merge) return e;
  AttnLaunch m = a;
  m.splits = nclu;
  return launch_attention_merge(s, m, st);
}

// Compiled row widths (K = V, 16 heads).
#define AVSG_H16_WIDTHS(X) X(576)

}  // namespace

bool attention_h16_supported(int D, int DV, int G, int kv_shared) {
  if (G != kH || D != DV || !kv_shared) return false;
#define X(d) \
  if (D == d) return true;
  AVSG_H16_WIDTHS(X)
#undef X
  return false;
}

int attention_h16_rows_per_tile() { return kRows; }

cudaError_t launch_attention_h16(const DeviceState& s, const AttnLaunch& a, cudaStream_t st) {
#define X(d) \
  if (s.D == d) return run<H16Shape<d>>(s, a, st);
  AVSG_H16_WIDTHS(X)
#undef X
  return cudaErrorInvalidValue;
}

}  // namespace avsg
