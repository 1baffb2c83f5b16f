// avsg_attention_noalloc: decode attention over rows the caller already holds
// on the device, for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: code that runs inside another
// framework's memory pool or allocator budget, code that must not allocate
// once it is serving (a memory-capped inference process), or a plugin whose
// host forbids allocation.  This entry point allocates nothing.  The split-K
// scratch the attention kernel needs (one partial result per split, one
// arrival counter per (unit, token), one error word) lives in a file-scope
// device array of fixed size; every GPU that loads the library holds that
// array until the process exits.
//
// The first call on a device looks the array's device address up with
// cudaGetSymbolAddress (the array's name in host code is only a host-side
// stand-in); make that first call before any stream capture.  All calls share
// the one array, so calls that overlap on the GPU (other streams, other host
// threads) race; serialise them.  Each call clears the error word and the
// arrival counters before its kernels run.
#include <math.h>

#include <mutex>

#include "avsg_internal.cuh"

namespace avsg {
namespace {

constexpr size_t kScratchBytes = 8u << 20;   // 8 MiB per device
constexpr int kMaxUnits = 4096;              // arrival counters: units * kMaxTokens ints
constexpr size_t kErrBytes = 256;
constexpr size_t kCountBytes = (size_t)kMaxUnits * kMaxTokens * sizeof(int32_t);
constexpr size_t kPartOffset = kErrBytes + kCountBytes;  // a multiple of 256
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_attn_scratch[kScratchBytes];

std::mutex g_mu;
unsigned char* g_scratch_ptr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};

// Marks the call failed when an index is outside [0, rows).
__global__ void check_index_kernel(const int32_t* __restrict__ idx, size_t n, size_t per_unit,
                                   int32_t rows, DevErr* err) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    const int32_t v = idx[i];
    if (v < 0 || v >= rows)
      raise_error(err, AVSG_ERR_BAD_SELECTION, (int)(i / per_unit), (int)(i % per_unit));
  }
}

// After a failed check the attention kernel wrote nothing: fill NaN.
__global__ void fill_nan_on_error_kernel(const DevErr* err, float* out, size_t n) {
  if (load_err(err) == 0) return;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x)
    out[i] = __int_as_float(0x7fc00000);
}

int setup_device(int* dev_out, unsigned char** ptr, int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return AVSG_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return AVSG_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_attn_scratch) != cudaSuccess || !p) return AVSG_ERR_CUDA;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return AVSG_ERR_CUDA;
    g_sms[dev] = n;
    g_scratch_ptr[dev] = static_cast<unsigned char*>(p);
  }
  *dev_out = dev;
  *ptr = g_scratch_ptr[dev];
  *sms = g_sms[dev];
  return AVSG_OK;
}

}  // namespace
}  // namespace avsg

using namespace avsg;

extern "C" int avsg_attention_noalloc(int32_t num_units, int32_t rows_per_unit, int32_t q_per_kv,
                                      int32_t head_dim, int32_t v_dim, int32_t entry_tokens,
                                      int32_t kv_shared, int32_t n_tok, int32_t k,
                                      const void* d_k_rows, const void* d_v_rows,
                                      const int32_t* d_index, const float* d_q, float* d_out,
                                      float softmax_scale, void* stream) {
  if (num_units < 1 || rows_per_unit < 1 || n_tok < 1 || n_tok > kMaxTokens || k < 0 ||
      entry_tokens < 1 || entry_tokens > 64 || !d_out || !d_k_rows ||
      (!kv_shared && !d_v_rows) || (k > 0 && (!d_index || !d_q)) || !(softmax_scale >= 0.f) ||
      isinf(softmax_scale))
    return AVSG_ERR_INVALID_ARG;
  if (num_units > kMaxUnits || k > rows_per_unit) return AVSG_ERR_CAPACITY;
  if (!attention_supported(head_dim, v_dim, q_per_kv, kv_shared)) return AVSG_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t n_out = (size_t)num_units * n_tok * q_per_kv * v_dim;
  if (k == 0)
    return cudaMemsetAsync(d_out, 0, n_out * sizeof(float), st) == cudaSuccess ? AVSG_OK
                                                                               : AVSG_ERR_CUDA;
  int dev = 0, sms = 0;
  unsigned char* scratch = nullptr;
  int rc = setup_device(&dev, &scratch, &sms);
  if (rc != AVSG_OK) return rc;

  // Splits (read by the CUDA-core and 16-head launchers; the tensor-core
  // launcher sizes its own persistent grid against part_capacity): about 4
  // CTAs per SM in all, at least one tile of rows each, and no more partials
  // than the array holds.
  const int tr = attention_rows_per_tile(head_dim, v_dim, q_per_kv, kv_shared);
  const int64_t pairs = (int64_t)num_units * n_tok;
  int64_t splits = (4LL * sms + pairs - 1) / pairs;
  const int64_t by_rows = ((int64_t)k * entry_tokens + tr - 1) / tr;
  if (splits > by_rows) splits = by_rows;
  const size_t part_bytes_per_split = (size_t)pairs * q_per_kv * (v_dim + 2) * sizeof(float);
  const int64_t fit = (int64_t)((kScratchBytes - kPartOffset) / part_bytes_per_split);
  if (splits > fit) splits = fit;
  if (splits < 1) splits = 1;

  DeviceState s{};
  s.U = num_units;
  s.B = rows_per_unit;
  s.G = q_per_kv;
  s.D = head_dim;
  s.DV = v_dim;
  s.ET = entry_tokens;
  s.kv_shared = kv_shared ? 1 : 0;
  s.ek = (int64_t)entry_tokens * head_dim * 2;
  s.ev = kv_shared ? 0 : (int64_t)entry_tokens * v_dim * 2;
  s.kbuf = static_cast<unsigned char*>(const_cast<void*>(d_k_rows));
  s.vbuf = static_cast<unsigned char*>(const_cast<void*>(kv_shared ? d_k_rows : d_v_rows));
  s.err = reinterpret_cast<DevErr*>(scratch);
  s.part_count = reinterpret_cast<int32_t*>(scratch + kErrBytes);
  s.part = reinterpret_cast<float*>(scratch + kPartOffset);

  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf((float)head_dim);
  const size_t counts = (size_t)num_units * kMaxTokens * kCountsPerPair * 4;
  cudaError_t e = cudaMemsetAsync(scratch, 0, kErrBytes + (counts < kCountBytes ? counts : kCountBytes), st);
  const size_t n_idx = (size_t)num_units * n_tok * k;
  const int check_blocks = (int)((n_idx + 255) / 256 < (size_t)sms * 4 ? (n_idx + 255) / 256 : sms * 4);
  if (e == cudaSuccess) {
    check_index_kernel<<<check_blocks, 256, 0, st>>>(d_index, n_idx, (size_t)n_tok * k,
                                                     rows_per_unit, s.err);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) {
    AttnLaunch a{};
    a.n_tok = n_tok;
    a.k = k;
    a.splits = (int)splits;
    a.identity_slots = 0;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.q = d_q;
    a.out = d_out;
    a.slot_map = d_index;
    a.num_sms = sms;
    a.part_capacity = (kScratchBytes - kPartOffset) / sizeof(float);
    a.count_capacity = kCountBytes / sizeof(int32_t);
    e = launch_attention(s, a, st);
  }
  if (e == cudaSuccess) {
    const int fill_blocks = (int)((n_out + 255) / 256 < (size_t)sms * 4 ? (n_out + 255) / 256 : sms * 4);
    fill_nan_on_error_kernel<<<fill_blocks, 256, 0, st>>>(s.err, d_out, n_out);
    e = cudaGetLastError();
  }
  return e == cudaSuccess ? AVSG_OK : AVSG_ERR_CUDA;
}
