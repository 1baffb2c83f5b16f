// avsg_attn: split-K decode attention over the selected buffer slots.
//
// The Attention operation of the Spin page ("Unifying Sparse Attention with
// Hierarchical Memory for Scalable Long-Context LLM Serving", section 2A) on
// exactly the rows DSA selected (AVSG page, arxivdaily 2609.37538, English
// abstract: the exact token selection is kept).  For unit u, query token j and
// query head g: o = softmax(scale * q_g . K_r) V_r over the rows r of the
// selected entries (an entry of T tokens is T rows).
//
// Grid (splits, U, n_tok).  Each CTA owns a contiguous range of the token's
// selected entries.  Rows are staged through shared memory in tiles of TR rows
// with 16-byte cp.async copies from the buffer slots named by the slot map
// (double-buffered: the next tile streams in while this one is computed).
// Per tile: scores (8 lanes per row, fp32 FMA, q held in registers when it
// fits), an online-softmax update per head in the log2 domain, then the
// probability-weighted V sum (each thread owns a slice of output dims for a
// group of heads and a subset of rows).  The CTA's partial (max, sum, acc) is
// written out, and a merge kernel spread over the output columns combines the
// splits of every (unit, token) (a CTA with the whole range writes the output
// itself).
#include <math.h>
#include <stdlib.h>

#include "avsg_internal.cuh"

namespace avsg {
namespace {

template <int D_, int DV_, int G_, bool SHARED_, int CW_, int HG_>
struct Shape {
  static constexpr int D = D_, DV = DV_, G = G_, CW = CW_, HG = HG_;
  static constexpr bool SHARED = SHARED_;
  static constexpr int NC = DV / CW;                      // output slices per head group
  static constexpr int NT_PV = NC * HG;
  static constexpr int RG = NT_PV >= 256 ? 1 : 256 / NT_PV;  // row groups in the V sum
  static constexpr int NT = NT_PV * RG;                   // threads per CTA
  static constexpr int NW = NT / 32;
  static constexpr int TR = NT / 8;                       // rows per tile: 8 lanes per row
  static constexpr int GH = G / HG;                       // heads per thread in the V sum
  static constexpr int KCH = D / 8;                       // 16-byte chunks per K row
  static constexpr int VCH = SHARED ? 0 : DV / 8;
  static constexpr int CPL = KCH / 8;                     // K chunks per lane
  static constexpr bool QREG = G * CPL * 8 <= 64;
  static constexpr size_t STAGE_BYTES = 2ull * TR * (D + (SHARED ? 0 : DV)) * 2;
  static constexpr size_t RED_BYTES = RG > 1 ? (size_t)RG * G * DV * 4 : (size_t)G * DV * 4;
  static constexpr size_t REGION0 = STAGE_BYTES > RED_BYTES ? STAGE_BYTES : RED_BYTES;
  static constexpr size_t QS_BYTES = QREG ? 0 : (size_t)G * D * 4;
  static_assert(D % 64 == 0, "K width must be a multiple of 64");
  static_assert(DV % CW == 0 && G % HG == 0, "bad split of the V sum");
  static_assert(NT % 32 == 0 && NT <= 1024 && TR <= 64, "bad CTA shape");
  static_assert(!SHARED || D == DV, "shared K/V needs equal widths");
};

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  const unsigned d = (unsigned)__cvta_generic_to_shared(smem_dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4 v, float* f) {
  f[0] = __uint_as_float(v.x << 16);
  f[1] = __uint_as_float(v.x & 0xFFFF0000u);
  f[2] = __uint_as_float(v.y << 16);
  f[3] = __uint_as_float(v.y & 0xFFFF0000u);
  f[4] = __uint_as_float(v.z << 16);
  f[5] = __uint_as_float(v.z & 0xFFFF0000u);
  f[6] = __uint_as_float(v.w << 16);
  f[7] = __uint_as_float(v.w & 0xFFFF0000u);
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
__global__ void __launch_bounds__(SH::NT) attn_kernel(DeviceState s, AttnLaunch a) {
  constexpr int D = SH::D, DV = SH::DV, G = SH::G, TR = SH::TR, NT = SH::NT;
  constexpr int CW = SH::CW, GH = SH::GH, NC = SH::NC, RG = SH::RG, NT_PV = SH::NT_PV;
  constexpr int KCH = SH::KCH, VCH = SH::VCH, CPL = SH::CPL, CH = KCH + VCH;
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ __align__(16) float Ss[TR * G];
  __shared__ __align__(16) float Ps[TR * G];
  __shared__ float alpha_s[G], mrun[G], lrun[G];
  __shared__ int s_stop;

  unsigned char* kt = smem;                                           // [2][TR][D] bf16
  unsigned char* vt = SH::SHARED ? smem : smem + 2ull * TR * D * 2;   // [2][TR][DV] bf16
  float* red = reinterpret_cast<float*>(smem);                        // reused after the loop
  float* qs = reinterpret_cast<float*>(smem + SH::REGION0);           // [G][D] when not in regs
  int32_t* slots = reinterpret_cast<int32_t*>(smem + SH::REGION0 + SH::QS_BYTES);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int sp = blockIdx.x, u = blockIdx.y, tok = blockIdx.z;
  griddep_wait();
  griddep_launch();
  if (a.io) {  // this step's out and slot map (and q when it is not copied)
    const StepIO io = load_io(a.io);
    if (!a.q) a.q = io.q;
    a.out = io.out;
    a.slot_map = io.slot_map;
  }
  if (tid == 0) s_stop = load_err(s.err);
  if (tid < G) {
    mrun[tid] = -INFINITY;
    lrun[tid] = 0.f;
  }
  __syncthreads();
  if (s_stop) return;

  const int k = a.k, ET = s.ET;
  const int eps = (k + a.splits - 1) / a.splits;
  const int e0 = sp * eps;
  const int ne = max(0, min(k, e0 + eps) - e0);
  const int rows = ne * ET;
  const int ntiles = (rows + TR - 1) / TR;
  const size_t sel_base = ((size_t)u * a.n_tok + tok) * (size_t)k;
  for (int i = tid; i < ne; i += NT)
    slots[i] = a.identity_slots ? tok * k + e0 + i : a.slot_map[sel_base + e0 + i];
  const float* qg = a.q + ((size_t)u * a.n_tok + tok) * (size_t)G * D;
  if (!SH::QREG)
    for (int i = tid; i < G * D; i += NT) qs[i] = qg[i];

  // Score-phase mapping: row rr of the tile, lane l8 of the row's 8 lanes,
  // which reads K chunks l8, l8 + 8, ... (consecutive lanes, consecutive chunks).
  const int rr = tid >> 3, l8 = tid & 7;
  float qr[SH::QREG ? G : 1][SH::QREG ? CPL * 8 : 1];
  if (SH::QREG) {
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int j = 0; j < CPL; ++j)
#pragma unroll
        for (int e = 0; e < 8; ++e) qr[g][j * 8 + e] = qg[g * D + (l8 + 8 * j) * 8 + e];
  }
  // V-sum mapping: row group rg, head group hg, output slice c of CW dims.
  const int rg = tid / NT_PV, rem = tid - rg * NT_PV, hg = rem / NC, c = rem - hg * NC;
  float acc[GH][CW];
#pragma unroll
  for (int gh = 0; gh < GH; ++gh)
#pragma unroll
    for (int e = 0; e < CW; ++e) acc[gh][e] = 0.f;
  __syncthreads();

  const size_t row_k = (size_t)D * 2, row_v = (size_t)DV * 2;
  auto issue = [&](int tile, int buf) {
    const int r0 = tile * TR;
    for (int i = tid; i < TR * CH; i += NT) {
      const int r = i / CH, w = i - r * CH;
      const int row = r0 + r;
      if (row < rows) {
        const int ent = row / ET, sub = row - ent * ET;
        if (!AVSG_IN_BOUNDS(slots[ent] >= 0 && slots[ent] < s.B, s.err, u, ent)) continue;
        const size_t srow = ((size_t)u * s.B + slots[ent]) * ET + sub;
        if (w < KCH)
          cp_async16(kt + ((size_t)(buf * TR + r) * D) * 2 + w * 16, s.kbuf + srow * row_k + w * 16);
        else
          cp_async16(vt + ((size_t)(buf * TR + r) * DV) * 2 + (w - KCH) * 16,
                     s.vbuf + srow * row_v + (w - KCH) * 16);
      }
    }
  };

  issue(0, 0);
  cp_async_commit();
  if (ntiles > 1) issue(1, 1);
  cp_async_commit();
  for (int tl = 0; tl < ntiles; ++tl) {
    const int buf = tl & 1;
    const int nvalid = min(TR, rows - tl * TR);
    cp_async_wait<1>();
    __syncthreads();
    {  // scores, log2 domain
      float part[G];
#pragma unroll
      for (int g = 0; g < G; ++g) part[g] = 0.f;
      const uint4* krow = reinterpret_cast<const uint4*>(kt + ((size_t)(buf * TR + rr) * D) * 2);
#pragma unroll
      for (int j = 0; j < CPL; ++j) {
        float kf[8];
        bf16x8_to_f32(krow[l8 + 8 * j], kf);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          if (SH::QREG) {
#pragma unroll
            for (int e = 0; e < 8; ++e) part[g] = fmaf(qr[g][j * 8 + e], kf[e], part[g]);
          } else {
            const float4* q4 = reinterpret_cast<const float4*>(qs + g * D + (l8 + 8 * j) * 8);
            const float4 qa = q4[0], qb = q4[1];
            part[g] = fmaf(qa.x, kf[0], part[g]);
            part[g] = fmaf(qa.y, kf[1], part[g]);
            part[g] = fmaf(qa.z, kf[2], part[g]);
            part[g] = fmaf(qa.w, kf[3], part[g]);
            part[g] = fmaf(qb.x, kf[4], part[g]);
            part[g] = fmaf(qb.y, kf[5], part[g]);
            part[g] = fmaf(qb.z, kf[6], part[g]);
            part[g] = fmaf(qb.w, kf[7], part[g]);
          }
        }
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        part[g] += __shfl_xor_sync(0xffffffffu, part[g], 1);
        part[g] += __shfl_xor_sync(0xffffffffu, part[g], 2);
        part[g] += __shfl_xor_sync(0xffffffffu, part[g], 4);
      }
      if (l8 == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g) Ss[rr * G + g] = rr < nvalid ? part[g] * a.scale_log2 : -INFINITY;
      }
    }
    __syncthreads();
    for (int g = warp; g < G; g += SH::NW) {  // online softmax, one warp per head
      const float s0 = lane < TR ? Ss[lane * G + g] : -INFINITY;
      const float s1 = lane + 32 < TR ? Ss[(lane + 32) * G + g] : -INFINITY;
      const float m_old = mrun[g];
      const float m_new = fmaxf(m_old, warp_max(fmaxf(s0, s1)));
      float alpha = 1.f, p0 = 0.f, p1 = 0.f;
      if (m_new != -INFINITY) {
        alpha = exp2f(m_old - m_new);
        p0 = exp2f(s0 - m_new);
        p1 = exp2f(s1 - m_new);
      }
      if (lane < TR) Ps[lane * G + g] = p0;
      if (lane + 32 < TR) Ps[(lane + 32) * G + g] = p1;
      const float sum = warp_sum(p0 + p1);
      if (lane == 0) {
        mrun[g] = m_new;
        lrun[g] = lrun[g] * alpha + sum;
        alpha_s[g] = alpha;
      }
    }
    __syncthreads();
    {  // probability-weighted V rows
#pragma unroll
      for (int gh = 0; gh < GH; ++gh) {
        const float al = alpha_s[hg * GH + gh];
#pragma unroll
        for (int e = 0; e < CW; ++e) acc[gh][e] *= al;
      }
      for (int r = rg; r < nvalid; r += RG) {
        const unsigned char* vrow = vt + ((size_t)(buf * TR + r) * DV) * 2 + (size_t)c * CW * 2;
        float vf[CW];
        if (CW == 8) {
          bf16x8_to_f32(*reinterpret_cast<const uint4*>(vrow), vf);
        } else {
          const uint2 v2 = *reinterpret_cast<const uint2*>(vrow);
          vf[0] = __uint_as_float(v2.x << 16);
          vf[1] = __uint_as_float(v2.x & 0xFFFF0000u);
          vf[2] = __uint_as_float(v2.y << 16);
          vf[3] = __uint_as_float(v2.y & 0xFFFF0000u);
        }
#pragma unroll
        for (int gh = 0; gh < GH; ++gh) {
          const float p = Ps[r * G + hg * GH + gh];
#pragma unroll
          for (int e = 0; e < CW; ++e) acc[gh][e] = fmaf(p, vf[e], acc[gh][e]);
        }
      }
    }
    __syncthreads();
    if (tl + 2 < ntiles) issue(tl + 2, buf);
    cp_async_commit();
  }
  cp_async_wait<0>();
  __syncthreads();

  // Sum the row groups: red[g][dv] = this CTA's unnormalised output.
#pragma unroll
  for (int gh = 0; gh < GH; ++gh)
#pragma unroll
    for (int e = 0; e < CW; ++e) red[((size_t)rg * G + hg * GH + gh) * DV + c * CW + e] = acc[gh][e];
  __syncthreads();
  if (RG > 1) {
    for (int o = tid; o < G * DV; o += NT) {
      float v = 0.f;
#pragma unroll 4
      for (int g2 = 0; g2 < RG; ++g2) v += red[(size_t)g2 * G * DV + o];
      red[o] = v;
    }
    __syncthreads();
  }

  float* out = a.out + ((size_t)u * a.n_tok + tok) * (size_t)G * DV;
  if (a.splits == 1) {
    for (int o = tid; o < G * DV; o += NT) {
      const float l = lrun[o / DV];
      out[o] = l > 0.f ? red[o] / l : 0.f;
    }
    return;
  }
  const size_t stride = (size_t)G * (DV + 2);
  float* pbase = s.part + ((size_t)u * a.n_tok + tok) * (size_t)a.splits * stride;
  float* pp = pbase + (size_t)sp * stride;
  for (int o = tid; o < G * DV; o += NT) pp[2 * G + o] = red[o];
  if (tid < G) {
    pp[tid] = mrun[tid];
    pp[G + tid] = lrun[tid];
  }
}

// Merge of the splits (launched after the attention when it has more than one
// split): CTA (pair, x) takes output columns [x * kMergeCols, ...) of the
// pair.  The (m, l) of every split for the CTA's heads are loaded at once into
// shared memory and turned into weights; each thread then sums its column
// over the splits, kMergeQB partials per round of loads.
constexpr int kMergeThreads = 256;
constexpr int kMergeCols = kMergeThreads;
constexpr int kMergeQB = 8;
constexpr int kMergeMaxW = 4096;  // (split, head) weights held in shared memory

__global__ void __launch_bounds__(kMergeThreads) merge_kernel(DeviceState s, AttnLaunch a) {
  __shared__ float s_w[kMergeMaxW];
  __shared__ float s_l[kMergeMaxW];
  __shared__ int s_stop;
  const int G = s.G, DV = s.DV;
  const int pair = blockIdx.x, tid = threadIdx.x;
  const int c0 = blockIdx.y * kMergeCols;
  const int h0 = c0 / DV, h1 = min(G - 1, (c0 + kMergeCols - 1) / DV), nh = h1 - h0 + 1;
  const int S = a.splits;
  griddep_wait();
  griddep_launch();
  if (a.io) {
    const StepIO io = load_io(a.io);
    a.out = io.out;
  }
  if (tid == 0) s_stop = load_err(s.err);
  const size_t stride = (size_t)G * (DV + 2);
  const float* pbase = s.part + (size_t)pair * S * stride;
  for (int i = tid; i < S * nh; i += kMergeThreads) {
    const int q = i / nh, h = h0 + (i - q * nh);
    s_w[i] = __ldcg(pbase + q * stride + h);
    s_l[i] = __ldcg(pbase + q * stride + G + h);
  }
  __syncthreads();
  if (s_stop) return;
  if (tid < nh) {  // per head: exp2(m_q - M) / L
    float M = -INFINITY;
    for (int q = 0; q < S; ++q) M = fmaxf(M, s_w[q * nh + tid]);
    float L = 0.f;
    for (int q = 0; q < S; ++q) {
      const float e = M == -INFINITY ? 0.f : exp2f(s_w[q * nh + tid] - M);
      s_w[q * nh + tid] = e;
      L = fmaf(s_l[q * nh + tid], e, L);
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    for (int q = 0; q < S; ++q) s_w[q * nh + tid] *= inv;
  }
  __syncthreads();
  const int o = c0 + tid;
  if (o >= G * DV) return;
  const int hh = o / DV - h0;
  float O = 0.f;
  for (int q0 = 0; q0 < S; q0 += kMergeQB) {
    float v[kMergeQB];
#pragma unroll
    for (int j = 0; j < kMergeQB; ++j)
      v[j] = q0 + j < S ? __ldcg(pbase + (q0 + j) * stride + 2 * G + o) : 0.f;
#pragma unroll
    for (int j = 0; j < kMergeQB; ++j)
      if (q0 + j < S) O = fmaf(v[j], s_w[(q0 + j) * nh + hh], O);
  }
  a.out[(size_t)pair * G * DV + o] = O;
}

template <class SH>
cudaError_t run(const DeviceState& s, const AttnLaunch& a, cudaStream_t st) {
  static int smem_done = 0;
  const int eps = (a.k + a.splits - 1) / a.splits;
  const size_t smem = SH::REGION0 + SH::QS_BYTES + ((size_t)eps * 4 + 15) / 16 * 16;
  cudaError_t e = ensure_smem((const void*)attn_kernel<SH>, smem, &smem_done);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)a.splits, (unsigned)s.U, (unsigned)a.n_tok);
  e = launch_pdl(attn_kernel<SH>, grid, dim3(SH::NT), smem, st, s, a);
  if (e != cudaSuccess || a.splits == 1) return e;
  return launch_attention_merge(s, a, st);
}

// Compiled shapes: (D, Dv, G, shared).
#define AVSG_ATTN_SHAPES(X)                \
  X(128, 128, 1, false, 8, 1)              \
  X(128, 128, 2, false, 8, 1)              \
  X(128, 128, 4, false, 8, 1)              \
  X(128, 128, 8, false, 8, 1)              \
  X(128, 128, 1, true, 8, 1)               \
  X(128, 128, 4, true, 8, 1)               \
  X(64, 64, 1, false, 8, 1)                \
  X(64, 64, 4, false, 8, 1)                \
  X(576, 576, 16, true, 4, 2)

}  // namespace

cudaError_t launch_attention_merge(const DeviceState& s, const AttnLaunch& a, cudaStream_t st) {
  if ((size_t)a.splits * ((kMergeCols + s.DV - 1) / s.DV + 1) > kMergeMaxW) return cudaErrorInvalidValue;
  dim3 mgrid((unsigned)(s.U * a.n_tok), (unsigned)((s.G * s.DV + kMergeCols - 1) / kMergeCols));
  return launch_pdl(merge_kernel, mgrid, dim3(kMergeThreads), 0, st, s, a);
}

bool attention_h16_enabled() {
  static const int on = [] {
    const char* v = getenv("AVSG_ATTN_H16");
    return (v && *v) ? atoi(v) : 1;
  }();
  return on != 0;
}

bool attention_supported(int D, int DV, int G, int kv_shared) {
#define X(d, dv, g, sh, cw, hgp) \
  if (D == d && DV == dv && G == g && (kv_shared != 0) == sh) return true;
  AVSG_ATTN_SHAPES(X)
#undef X
  return false;
}

int attention_rows_per_tile(int D, int DV, int G, int kv_shared) {
  if (attention_h16_enabled() && attention_h16_supported(D, DV, G, kv_shared))
    return attention_h16_rows_per_tile();
#define X(d, dv, g, sh, cw, hgp) \
  if (D == d && DV == dv && G == g && (kv_shared != 0) == sh) return Shape<d, dv, g, sh, cw, hgp>::TR;
  AVSG_ATTN_SHAPES(X)
#undef X
  return 0;
}

int attention_ctas_per_sm(int D, int DV, int G, int kv_shared) {
  // the 16-head kernel keeps 2 CTAs per SM resident, and each split adds a
  // 16 x (Dv + 2) partial for the merge: one CTA per SM in all
  if (attention_h16_enabled() && attention_h16_supported(D, DV, G, kv_shared)) return 1;
  return 4;
}

cudaError_t launch_attention(const DeviceState& s, const AttnLaunch& a, cudaStream_t st) {
  if (attention_tc_enabled() && attention_tc_supported(s.D, s.DV, s.G, s.kv_shared) &&
      a.num_sms > 0)
    return launch_attention_tc(s, a, a.num_sms, st);
  if (attention_h16_enabled() && attention_h16_supported(s.D, s.DV, s.G, s.kv_shared))
    return launch_attention_h16(s, a, st);
#define X(d, dv, g, sh, cw, hgp)                                      \
  if (s.D == d && s.DV == dv && s.G == g && (s.kv_shared != 0) == sh) \
    return run<Shape<d, dv, g, sh, cw, hgp>>(s, a, st);
  AVSG_ATTN_SHAPES(X)
#undef X
  return cudaErrorInvalidValue;
}

}  // namespace avsg
