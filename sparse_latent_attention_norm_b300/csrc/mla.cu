// libmla: the C ABI (include/mla.h) over the three stages of the MLA sparse prefill.
// Host code here checks arguments, carves the workspace, encodes the TMA tensor maps and
// enqueues the kernels on the caller's stream; every step of the path runs in the kernels.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "mla.h"
#include "ptx.cuh"
#include "tmap.h"
#include "canon_select.cuh"
#include "kvnorm_wkvb.cuh"
#include "sparse_attn.cuh"
#include "prologue.cuh"

namespace mla {

// Diagnostic of the failure path: one thread waits, through the bounded wait every kernel uses,
// on an mbarrier nothing arrives on. The wait gives up at its limit, records the timeout in the
// status word and returns. result[0] = 1 if the wait completed, result[1] = milliseconds waited.
__global__ void selftest_wait_timeout_kernel(int32_t* result) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
    const uint64_t t0 = globaltimer_ns();
    const bool completed = mbar_wait(&bar, 0, nullptr);
    result[0] = completed ? 1 : 0;
    result[1] = static_cast<int32_t>((globaltimer_ns() - t0) / 1000000ull);
  }
}

}  // namespace mla

namespace {

constexpr int kLatent = 512, kQK = 192, kRope = 64, kKV = 256;
constexpr int kMaxT = 65536;
constexpr int kMaxH = 128;
constexpr int kMaxDevices = 64;

// Per-device launch set-up: kernel attributes and the SM count, done once per device.
struct DeviceInfo {
  bool ready = false;
  int num_sms = 0;
  int k1_ctas = 0;   // GEMM-stage CTAs resident at once (0: unknown)
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mutex;

mla_status device_setup(int* num_sms, int* k1_ctas) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MLA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MLA_ERR_CUDA;
    if (cudaFuncSetAttribute(mla::k1::kvnorm_wkvb_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             mla::k1::SMEM_BYTES) != cudaSuccess)
      return MLA_ERR_CUDA;
    if (cudaFuncSetAttribute(mla::k2::sparse_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             mla::k2::SMEM_BYTES) != cudaSuccess)
      return MLA_ERR_CUDA;
    {
      // the GEMM stage's grid is a fixed set of CTA pairs with fixed unit ranges: launch no more
      // pairs than can be resident together
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2, 1, 1);
      cfg.blockDim = dim3(mla::k1::THREADS, 1, 1);
      cfg.dynamicSmemBytes = mla::k1::SMEM_BYTES;
      int clusters = 0;
      if (cudaOccupancyMaxActiveClusters(&clusters, mla::k1::kvnorm_wkvb_kernel, &cfg) != cudaSuccess) {
        clusters = 0;
        (void)cudaGetLastError();   // the query's error is not the caller's
      }
      d.k1_ctas = 2 * clusters;
    }
    d.ready = true;
  }
  *num_sms = d.num_sms;
  if (k1_ctas) *k1_ctas = d.k1_ctas;
  return MLA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int bits_words(int T) { return (T + 127) / 128 * 4; }

mla_status check_dims(mla_dims d) {
  if (d.B < 1 || d.T < 1 || d.H < 1 || d.K < 1) return MLA_ERR_INVALID_ARG;
  if (d.T > kMaxT || d.H > kMaxH) return MLA_ERR_UNSUPPORTED;
  const int64_t BT = static_cast<int64_t>(d.B) * d.T;
  if (BT > INT32_MAX / 2) return MLA_ERR_UNSUPPORTED;
  const double work = static_cast<double>(BT) * d.H * d.K;
  if (work >= 1099511627776.0) return MLA_ERR_UNSUPPORTED;  // 2^40
  return MLA_OK;
}

size_t kv_bytes(mla_dims d) { return static_cast<size_t>(d.B) * d.H * d.T * kKV * 2; }
size_t klo_bytes(mla_dims d) { return static_cast<size_t>(d.B) * d.H * d.T * 128; }
size_t bits_bytes(mla_dims d) { return static_cast<size_t>(d.B) * d.T * bits_words(d.T) * 4; }
constexpr size_t kSchedBytes = 1024;   // the attention stage's tile counter (one word, padded)

cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

mla_status launch_canon(const int32_t* topk_idx, mla_dims d, uint32_t* sel_bits, int32_t* n_keys, unsigned flags,
                        uint32_t* sched, cudaStream_t st) {
  const int W = bits_words(d.T);
  const int rows_per_cta = mla::canon_rows_per_cta(W);
  const size_t smem = static_cast<size_t>(rows_per_cta) * W * 4;
  const int64_t rows = static_cast<int64_t>(d.B) * d.T;
  const unsigned grid = static_cast<unsigned>((rows + rows_per_cta - 1) / rows_per_cta);
  mla::canon_select_kernel<<<grid, 32 * rows_per_cta, smem, st>>>(topk_idx, rows, d.T, d.K, W, sel_bits, n_keys,
                                                                  (flags & MLA_FLAG_VALIDATE_INDICES) ? 1 : 0, sched);
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

mla_status launch_kvnorm_wkvb(const mla_bf16* c_kv, const float* gamma, const mla_bf16* wkv_b, mla_dims d,
                              uint16_t* kv, uint8_t* klo, int num_sms, int k1_max_ctas, cudaStream_t st,
                              bool fp8_latent = false, mla_bf16* kv_cache = nullptr, int cache_len = 0) {
  CUtensorMap tm_w;
  {
    const uint64_t dims[2] = {kLatent, static_cast<uint64_t>(d.H) * kKV};
    const uint64_t strides[1] = {kLatent * 2};
    const uint32_t box[2] = {64, mla::k1::BNH};
    if (!mla::make_tmap_bf16(&tm_w, wkv_b, 2, dims, strides, box)) return MLA_ERR_CUDA;
  }
  mla::k1::Params p;
  p.B = d.B;
  p.T = d.T;
  p.H = d.H;
  p.mt_per_b = (d.T + mla::k1::BM - 1) / mla::k1::BM;
  const int64_t n_mtiles = static_cast<int64_t>(d.B) * p.mt_per_b;
  const int64_t n_tpairs = (n_mtiles + 1) / 2;
  const int64_t units = n_tpairs * d.H;
  if (units > INT32_MAX / 2) return MLA_ERR_UNSUPPORTED;
  p.n_mtiles = static_cast<int>(n_mtiles);
  p.n_tpairs = static_cast<int>(n_tpairs);
  p.units = static_cast<int>(units);
  p.c_kv = c_kv;
  p.gamma = gamma;
  p.kv_out = kv;
  p.klo_out = klo;
  p.fp8_latent = fp8_latent ? 1 : 0;
  p.kv_cache = kv_cache;
  p.cache_len = cache_len;
  // CTA pairs (clusters of two), no more than can be resident at once (each pair's range of
  // units is fixed)
  int pairs = k1_max_ctas > 0 ? k1_max_ctas / 2 : num_sms / 2;
  if (pairs > p.units) pairs = p.units;
  if (pairs < 1) pairs = 1;
  const int grid = 2 * pairs;
  mla::k1::kvnorm_wkvb_kernel<<<grid, mla::k1::THREADS, mla::k1::SMEM_BYTES, st>>>(tm_w, p);
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

// `sched` must hold zero when the launch starts (the selection stage or a memset before it sets it).
mla_status launch_sparse_attn(const mla_bf16* q, const mla_bf16* k_pe, const uint16_t* kv, const uint8_t* klo,
                              const uint32_t* sel_bits, mla_bf16* out, float* lse, mla_dims d, uint32_t* sched,
                              int num_sms, cudaStream_t st, const float* rope_cs = nullptr) {
  CUtensorMap tm_q, tm_kv, tm_kpe, tm_klo;
  {
    const uint64_t dims[4] = {kQK, static_cast<uint64_t>(d.H), static_cast<uint64_t>(d.T), static_cast<uint64_t>(d.B)};
    const uint64_t strides[3] = {kQK * 2, static_cast<uint64_t>(d.H) * kQK * 2,
                                 static_cast<uint64_t>(d.T) * d.H * kQK * 2};
    const uint32_t box[4] = {64, 1, mla::k2::BQ, 1};
    if (!mla::make_tmap_bf16(&tm_q, q, 4, dims, strides, box)) return MLA_ERR_CUDA;
  }
  {
    const uint64_t dims[3] = {kKV, static_cast<uint64_t>(d.T), static_cast<uint64_t>(d.B) * d.H};
    const uint64_t strides[2] = {kKV * 2, static_cast<uint64_t>(d.T) * kKV * 2};
    const uint32_t box[3] = {64, mla::k2::BK, 1};
    if (!mla::make_tmap_f16(&tm_kv, kv, 3, dims, strides, box)) return MLA_ERR_CUDA;
  }
  {
    const uint64_t dims[3] = {kRope, static_cast<uint64_t>(d.T), static_cast<uint64_t>(d.B)};
    const uint64_t strides[2] = {kRope * 2, static_cast<uint64_t>(d.T) * kRope * 2};
    const uint32_t box[3] = {64, mla::k2::BK, 1};
    if (!mla::make_tmap_bf16(&tm_kpe, k_pe, 3, dims, strides, box)) return MLA_ERR_CUDA;
  }
  {
    const uint64_t dims[3] = {128, static_cast<uint64_t>(d.T), static_cast<uint64_t>(d.B) * d.H};
    const uint64_t strides[2] = {128, static_cast<uint64_t>(d.T) * 128};
    const uint32_t box[3] = {128, mla::k2::BK, 1};
    if (!mla::make_tmap_u8(&tm_klo, klo, 3, dims, strides, box)) return MLA_ERR_CUDA;
  }
  mla::k2::Params p;
  p.B = d.B;
  p.T = d.T;
  p.H = d.H;
  p.nqt = (d.T + mla::k2::BQ - 1) / mla::k2::BQ;
  const int64_t n_items = static_cast<int64_t>(d.B) * d.H * p.nqt;
  if (n_items > INT32_MAX / 2) return MLA_ERR_UNSUPPORTED;
  p.n_items = static_cast<int>(n_items);
  p.sched = sched;
  p.W = bits_words(d.T);
  p.scale_log2 = static_cast<float>(mla_softmax_scale() * 1.4426950408889634);
  p.q = q;
  p.sel_bits = sel_bits;
  p.out = out;
  p.lse = lse;
  p.rope_cs = reinterpret_cast<const float2*>(rope_cs);
  // persistent: one CTA per SM (the tiles fill its shared memory), tiles handed out dynamically
  const unsigned grid = static_cast<unsigned>(n_items < num_sms ? n_items : num_sms);
  mla::k2::sparse_attn_kernel<<<grid, mla::k2::THREADS, mla::k2::SMEM_BYTES, st>>>(tm_q, tm_kv, tm_kpe, tm_klo, p);
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

// YaRN frequencies of the 32 rotary pairs (ModelArgs: rope_theta 10000, rope_factor 40, beta_fast
// 32, beta_slow 1, original_seq_len 4096; max_seq_len 16384 > original, so the correction applies):
// RoPE's theta^(-2i/64), kept for pairs that turn more than beta_fast times over the original
// context, divided by rope_factor for pairs that turn fewer than beta_slow times, linear in i in
// between (YaRN, Peng et al. 2023).
void yarn_frequencies(double* f) {
  const double theta = 10000.0, factor = 40.0, fast = 32.0, slow = 1.0, L = 4096.0;
  const double pi = 3.14159265358979323846;
  // the pair index at which a pair turns n times over L: 64 ln(L / (2 pi n)) / (2 ln theta)
  auto pair_at = [&](double n) { return kRope * std::log(L / (2.0 * pi * n)) / (2.0 * std::log(theta)); };
  const double lo = std::fmax(std::floor(pair_at(fast)), 0.0);
  double hi = std::fmin(std::ceil(pair_at(slow)), static_cast<double>(kRope - 1));
  if (hi == lo) hi += 0.001;
  for (int i = 0; i < mla::kRopePairs; ++i) {
    const double base = std::pow(theta, -2.0 * i / kRope);
    const double w = std::fmin(1.0, std::fmax(0.0, (i - lo) / (hi - lo)));   // 0: keep, 1: divide
    f[i] = base * (1.0 - w) + base / factor * w;
  }
}

mla_status launch_rope_kpe(const mla_bf16* k_pe, mla_dims d, bool rotate, mla_bf16* k_pe_rot, float* rope_cs,
                           mla_bf16* pe_cache, int cache_len, cudaStream_t st) {
  mla::RopeFreqs f;
  yarn_frequencies(f.f);
  const int64_t threads = static_cast<int64_t>(d.B) * d.T * 32;
  const unsigned grid = static_cast<unsigned>((threads + 255) / 256);
  mla::rope_kpe_kernel<<<grid, 256, 0, st>>>(k_pe, d.B, d.T, rotate ? 1 : 0, f, k_pe_rot,
                                              reinterpret_cast<float2*>(rope_cs), pe_cache, cache_len);
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

mla_status launch_dequant(const uint8_t* w8, const float* scale, int rows, mla_bf16* w, cudaStream_t st) {
  const int64_t groups = static_cast<int64_t>(rows) * 32;
  mla::wkvb_dequant_kernel<<<static_cast<unsigned>((groups + 255) / 256), 256, 0, st>>>(w8, scale, rows, w);
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

// Tile counter of the staged attention entry point, which has no workspace: one word per device,
// zeroed on the caller's stream before each launch.
static __device__ uint32_t g_staged_sched;
void* g_staged_sched_ptr[kMaxDevices] = {};
std::mutex g_staged_sched_mutex;

mla_status staged_sched_counter(uint32_t** ptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MLA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_staged_sched_mutex);
  if (g_staged_sched_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_staged_sched) != cudaSuccess || p == nullptr) return MLA_ERR_CUDA;
    g_staged_sched_ptr[dev] = p;
  }
  *ptr = static_cast<uint32_t*>(g_staged_sched_ptr[dev]);
  return MLA_OK;
}

}  // namespace

extern "C" {

double mla_softmax_scale(void) {
  // MLA __init__: qk_head_dim ** -0.5, times mscale^2 (max_seq_len 16384 > original 4096),
  // mscale = 0.1 * 1 * ln(40) + 1.
  const double mscale = 0.1 * 1.0 * std::log(40.0) + 1.0;
  return std::pow(static_cast<double>(kQK), -0.5) * mscale * mscale;
}

const char* mla_status_string(mla_status s) {
  switch (s) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG: null, misaligned or out-of-range argument";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED: shape outside the supported range";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA: a CUDA call or launch failed";
    case MLA_ERR_INDEX: return "MLA_ERR_INDEX: top-k index outside [0, T)";
    case MLA_ERR_TIMEOUT: return "MLA_ERR_TIMEOUT: a device barrier wait ran out";
    case MLA_ERR_WORKSPACE: return "MLA_ERR_WORKSPACE: workspace too small or misaligned";
    case MLA_ERR_RANGE: return "MLA_ERR_RANGE: a value outside the range the kernels carry exactly";
    case MLA_ERR_BOUNDS: return "MLA_ERR_BOUNDS: a bounds check of the checked build failed";
  }
  return "unknown mla_status";
}

size_t mla_sparse_prefill_workspace_size(mla_dims d) {
  if (check_dims(d) != MLA_OK) return 0;
  return align_up(kv_bytes(d), 1024) + align_up(klo_bytes(d), 1024) + align_up(bits_bytes(d), 1024) + kSchedBytes;
}

mla_status mla_canon_select(const int32_t* topk_idx, mla_dims d, uint32_t* sel_bits, int32_t* n_keys,
                            unsigned flags, void* stream) {
  mla_status s = check_dims(d);
  if (s != MLA_OK) return s;
  if (!topk_idx || !sel_bits || !aligned16(topk_idx) || !aligned16(sel_bits)) return MLA_ERR_INVALID_ARG;
  if (n_keys && (reinterpret_cast<uintptr_t>(n_keys) & 3u)) return MLA_ERR_INVALID_ARG;
  int sms, k1_ctas;
  if ((s = device_setup(&sms, &k1_ctas)) != MLA_OK) return s;
  return launch_canon(topk_idx, d, sel_bits, n_keys, flags, nullptr, as_stream(stream));
}

mla_status mla_kvnorm_wkvb(const mla_bf16* c_kv, const float* gamma, const mla_bf16* wkv_b, mla_dims d,
                           uint16_t* kv, uint8_t* klo, void* stream) {
  return mla_kvnorm_wkvb_opt(c_kv, gamma, wkv_b, d, kv, klo, 0u, nullptr, 0, stream);
}

mla_status mla_sparse_attention(const mla_bf16* q, const mla_bf16* k_pe, const uint16_t* kv, const uint8_t* klo,
                                const uint32_t* sel_bits, mla_bf16* out, float* lse, mla_dims d, void* stream) {
  return mla_sparse_attention_opt(q, k_pe, kv, klo, sel_bits, out, lse, d, nullptr, stream);
}

namespace {

// Workspace layout of mla_sparse_prefill_opt: the base carve (kv, klo, bits, tile counter), then
// the dequantised wkv_b (FP8 weights), the RoPE table and the rotated k_pe (MLA_FLAG_ROPE).
struct Carve {
  uint16_t* kv;
  uint8_t* klo;
  uint32_t* bits;
  uint32_t* sched;
  mla_bf16* w_deq;
  float* rope_cs;
  mla_bf16* kpe_rot;
  size_t bytes;
};

Carve carve(void* base_ptr, mla_dims d, bool fp8_w, bool rope) {
  Carve c{};
  uint8_t* base = static_cast<uint8_t*>(base_ptr);
  size_t off = 0;
  auto take = [&](size_t n) { uint8_t* p = base ? base + off : nullptr; off += align_up(n, 1024); return p; };
  c.kv = reinterpret_cast<uint16_t*>(take(kv_bytes(d)));
  c.klo = take(klo_bytes(d));
  c.bits = reinterpret_cast<uint32_t*>(take(bits_bytes(d)));
  c.sched = reinterpret_cast<uint32_t*>(take(kSchedBytes));
  if (fp8_w) c.w_deq = reinterpret_cast<mla_bf16*>(take(static_cast<size_t>(d.H) * kKV * kLatent * 2));
  if (rope) {
    c.rope_cs = reinterpret_cast<float*>(take(static_cast<size_t>(d.T) * mla::kRopePairs * 8));
    c.kpe_rot = reinterpret_cast<mla_bf16*>(take(static_cast<size_t>(d.B) * d.T * kRope * 2));
  }
  c.bytes = off;
  return c;
}

constexpr unsigned kAllFlags = MLA_FLAG_VALIDATE_INDICES | MLA_FLAG_FP8_LATENT | MLA_FLAG_ROPE;

mla_status check_options(mla_dims d, const mla_prefill_options* opt) {
  if (opt == nullptr) return MLA_OK;
  if (opt->flags & ~kAllFlags) return MLA_ERR_INVALID_ARG;
  if (opt->n_keys && (reinterpret_cast<uintptr_t>(opt->n_keys) & 3u)) return MLA_ERR_INVALID_ARG;
  if (opt->wkv_b_scale && (reinterpret_cast<uintptr_t>(opt->wkv_b_scale) & 3u)) return MLA_ERR_INVALID_ARG;
  if (opt->kv_cache || opt->pe_cache) {
    if (opt->cache_len < d.T) return MLA_ERR_INVALID_ARG;
    if (opt->kv_cache && !aligned32(opt->kv_cache)) return MLA_ERR_INVALID_ARG;
    if (opt->pe_cache && (reinterpret_cast<uintptr_t>(opt->pe_cache) & 3u)) return MLA_ERR_INVALID_ARG;
  }
  return MLA_OK;
}

}  // namespace

size_t mla_sparse_prefill_opt_workspace_size(mla_dims d, const mla_prefill_options* opt) {
  if (check_dims(d) != MLA_OK || check_options(d, opt) != MLA_OK) return 0;
  const bool fp8_w = opt && opt->wkv_b_scale;
  const bool rope = opt && (opt->flags & MLA_FLAG_ROPE);
  return carve(nullptr, d, fp8_w, rope).bytes;
}

mla_status mla_sparse_prefill_opt(const mla_bf16* q, const mla_bf16* c_kv, const mla_bf16* k_pe, const float* gamma,
                                  const void* wkv_b, const int32_t* topk_idx, mla_bf16* out, float* lse, mla_dims d,
                                  void* workspace, size_t workspace_bytes, void* stream,
                                  const mla_prefill_options* opt) {
  mla_status s = check_dims(d);
  if (s != MLA_OK) return s;
  if ((s = check_options(d, opt)) != MLA_OK) return s;
  if (!q || !c_kv || !k_pe || !gamma || !wkv_b || !topk_idx || !out || !lse) return MLA_ERR_INVALID_ARG;
  if (!aligned32(q) || !aligned16(c_kv) || !aligned16(k_pe) || !aligned16(gamma) || !aligned16(wkv_b) ||
      !aligned16(topk_idx) || !aligned32(out) || (reinterpret_cast<uintptr_t>(lse) & 3u))
    return MLA_ERR_INVALID_ARG;
  const unsigned flags = opt ? opt->flags : 0u;
  const bool fp8_w = opt && opt->wkv_b_scale;
  const bool rope = (flags & MLA_FLAG_ROPE) != 0;
  const size_t need = carve(nullptr, d, fp8_w, rope).bytes;
  if (workspace != nullptr) {
    if ((reinterpret_cast<uintptr_t>(workspace) & 1023u) || workspace_bytes < need) return MLA_ERR_WORKSPACE;
  }
  int sms, k1_ctas;
  if ((s = device_setup(&sms, &k1_ctas)) != MLA_OK) return s;
  cudaStream_t st = as_stream(stream);
  void* ws = workspace;
  bool owned = false;
  if (ws == nullptr) {
    if (cudaMallocAsync(&ws, need, st) != cudaSuccess) return MLA_ERR_CUDA;
    owned = true;
  }
  const Carve c = carve(ws, d, fp8_w, rope);
  const mla_bf16* w_bf16 = static_cast<const mla_bf16*>(wkv_b);
  // the stages in order on the caller's stream: the optional prologue (FP8 weight, RoPE of k_pe
  // and the pe_cache copy), the selection, the GEMM stage, the attention stage
  if (fp8_w) {
    s = launch_dequant(static_cast<const uint8_t*>(wkv_b), opt->wkv_b_scale, d.H * kKV, c.w_deq, st);
    w_bf16 = c.w_deq;
  }
  const mla_bf16* k_pe_used = k_pe;
  if (s == MLA_OK && (rope || (opt && opt->pe_cache))) {
    s = launch_rope_kpe(k_pe, d, rope, c.kpe_rot, c.rope_cs, opt->pe_cache, opt->cache_len, st);
    if (rope) k_pe_used = c.kpe_rot;
  }
  if (s == MLA_OK) s = launch_canon(topk_idx, d, c.bits, opt ? opt->n_keys : nullptr, flags, c.sched, st);
  if (s == MLA_OK)
    s = launch_kvnorm_wkvb(c_kv, gamma, w_bf16, d, c.kv, c.klo, sms, k1_ctas, st, (flags & MLA_FLAG_FP8_LATENT) != 0,
                           opt ? opt->kv_cache : nullptr, opt ? opt->cache_len : 0);
  if (s == MLA_OK)
    s = launch_sparse_attn(q, k_pe_used, c.kv, c.klo, c.bits, out, lse, d, c.sched, sms, st, rope ? c.rope_cs : nullptr);
  if (owned && cudaFreeAsync(ws, st) != cudaSuccess && s == MLA_OK) s = MLA_ERR_CUDA;
  return s;
}

mla_status mla_sparse_prefill_ex(const mla_bf16* q, const mla_bf16* c_kv, const mla_bf16* k_pe, const float* gamma,
                                 const mla_bf16* wkv_b, const int32_t* topk_idx, mla_bf16* out, float* lse,
                                 mla_dims d, void* workspace, size_t workspace_bytes, void* stream,
                                 int32_t* n_keys, unsigned flags) {
  if (flags & ~MLA_FLAG_VALIDATE_INDICES) return MLA_ERR_INVALID_ARG;
  mla_prefill_options o{};
  o.flags = flags;
  o.n_keys = n_keys;
  return mla_sparse_prefill_opt(q, c_kv, k_pe, gamma, wkv_b, topk_idx, out, lse, d, workspace, workspace_bytes, stream,
                                &o);
}

mla_status mla_sparse_prefill(const mla_bf16* q, const mla_bf16* c_kv, const mla_bf16* k_pe, const float* gamma,
                              const mla_bf16* wkv_b, const int32_t* topk_idx, mla_bf16* out, float* lse,
                              mla_dims d, void* workspace, size_t workspace_bytes, void* stream) {
  return mla_sparse_prefill_opt(q, c_kv, k_pe, gamma, wkv_b, topk_idx, out, lse, d, workspace, workspace_bytes,
                                stream, nullptr);
}

mla_status mla_dequant_wkvb_fp8(const uint8_t* w8, const float* scale, int32_t rows, mla_bf16* w, void* stream) {
  if (!w8 || !scale || !w || rows < 128 || rows % 128 != 0 || rows > kMaxH * kKV) return MLA_ERR_INVALID_ARG;
  if (!aligned16(w8) || !aligned32(w) || (reinterpret_cast<uintptr_t>(scale) & 3u)) return MLA_ERR_INVALID_ARG;
  return launch_dequant(w8, scale, rows, w, as_stream(stream));
}

mla_status mla_kvnorm_wkvb_opt(const mla_bf16* c_kv, const float* gamma, const mla_bf16* wkv_b, mla_dims d,
                               uint16_t* kv, uint8_t* klo, unsigned flags, mla_bf16* kv_cache, int32_t cache_len,
                               void* stream) {
  mla_status s = check_dims(d);
  if (s != MLA_OK) return s;
  if (!c_kv || !gamma || !wkv_b || !kv || !klo) return MLA_ERR_INVALID_ARG;
  if (!aligned16(c_kv) || !aligned16(gamma) || !aligned16(wkv_b) || !aligned32(kv) || !aligned32(klo))
    return MLA_ERR_INVALID_ARG;
  if (flags & ~MLA_FLAG_FP8_LATENT) return MLA_ERR_INVALID_ARG;
  if (kv_cache && (!aligned32(kv_cache) || cache_len < d.T)) return MLA_ERR_INVALID_ARG;
  int sms, k1_ctas;
  if ((s = device_setup(&sms, &k1_ctas)) != MLA_OK) return s;
  return launch_kvnorm_wkvb(c_kv, gamma, wkv_b, d, kv, klo, sms, k1_ctas, as_stream(stream),
                            (flags & MLA_FLAG_FP8_LATENT) != 0, kv_cache, cache_len);
}

void mla_yarn_frequencies(double* f) {
  if (f) yarn_frequencies(f);
}

mla_status mla_rope_k_pe(const mla_bf16* k_pe, mla_dims d, mla_bf16* k_pe_rot, float* rope_cs, mla_bf16* pe_cache,
                         int32_t cache_len, void* stream) {
  mla_status s = check_dims(d);
  if (s != MLA_OK) return s;
  if (!k_pe || !k_pe_rot || !rope_cs) return MLA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(k_pe) & 3u) || (reinterpret_cast<uintptr_t>(k_pe_rot) & 3u) || !aligned32(rope_cs))
    return MLA_ERR_INVALID_ARG;
  if (pe_cache && ((reinterpret_cast<uintptr_t>(pe_cache) & 3u) || cache_len < d.T)) return MLA_ERR_INVALID_ARG;
  return launch_rope_kpe(k_pe, d, true, k_pe_rot, rope_cs, pe_cache, cache_len, as_stream(stream));
}

mla_status mla_sparse_attention_opt(const mla_bf16* q, const mla_bf16* k_pe, const uint16_t* kv, const uint8_t* klo,
                                    const uint32_t* sel_bits, mla_bf16* out, float* lse, mla_dims d,
                                    const float* rope_cs, void* stream) {
  mla_status s = check_dims(d);
  if (s != MLA_OK) return s;
  if (!q || !k_pe || !kv || !klo || !sel_bits || !out || !lse) return MLA_ERR_INVALID_ARG;
  if (!aligned32(q) || !aligned16(k_pe) || !aligned16(kv) || !aligned16(klo) || !aligned16(sel_bits) ||
      !aligned32(out) || (reinterpret_cast<uintptr_t>(lse) & 3u) || (rope_cs && !aligned32(rope_cs)))
    return MLA_ERR_INVALID_ARG;
  int sms, k1_ctas;
  if ((s = device_setup(&sms, &k1_ctas)) != MLA_OK) return s;
  uint32_t* sched = nullptr;
  if ((s = staged_sched_counter(&sched)) != MLA_OK) return s;
  if (cudaMemsetAsync(sched, 0, sizeof(uint32_t), as_stream(stream)) != cudaSuccess) return MLA_ERR_CUDA;
  return launch_sparse_attn(q, k_pe, kv, klo, sel_bits, out, lse, d, sched, sms, as_stream(stream), rope_cs);
}

// ---------------------------------------------------------------------------------------------
// Allocation-free variant of mla_sparse_prefill.
//
// Some callers cannot allocate device memory at the point where they run the prefill: code
// running inside a host-side allocator or memory-pool callback, engines that fix their whole
// device footprint up front, or plug-ins whose host framework forbids cudaMalloc during a step.
// They get a scratch region that the library owns: a file-scope device array, created when the
// library's module is loaded on a GPU and kept until the process exits, so every GPU that loads
// libmla holds these bytes whether or not this entry point is used.
//
// Host code cannot pass g_noalloc_scratch to a kernel directly: in host code that name is a
// host-side stand-in, not a device address. The device address is looked up once per device
// with cudaGetSymbolAddress (with that device current) on the first call made on that device.
// ---------------------------------------------------------------------------------------------
static __device__ __align__(256) uint8_t g_noalloc_scratch[MLA_NOALLOC_SCRATCH_BYTES];

namespace {
void* g_noalloc_ptr[kMaxDevices] = {};
std::mutex g_noalloc_mutex;

mla_status noalloc_scratch_address(void** ptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MLA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return MLA_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *ptr = g_noalloc_ptr[dev];
  return MLA_OK;
}
}  // namespace

mla_status mla_sparse_prefill_noalloc(const mla_bf16* q, const mla_bf16* c_kv, const mla_bf16* k_pe,
                                      const float* gamma, const mla_bf16* wkv_b, const int32_t* topk_idx,
                                      mla_bf16* out, float* lse, mla_dims d, void* stream) {
  mla_status s = check_dims(d);
  if (s != MLA_OK) return s;
  if (!q || !c_kv || !k_pe || !gamma || !wkv_b || !topk_idx || !out || !lse) return MLA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(c_kv) || !aligned16(k_pe) || !aligned16(gamma) || !aligned16(wkv_b) ||
      !aligned16(topk_idx) || !aligned16(out) || (reinterpret_cast<uintptr_t>(lse) & 3u))
    return MLA_ERR_INVALID_ARG;
  if (mla_sparse_prefill_workspace_size(d) > static_cast<size_t>(MLA_NOALLOC_SCRATCH_BYTES)) return MLA_ERR_WORKSPACE;
  int sms, k1_ctas;
  if ((s = device_setup(&sms, &k1_ctas)) != MLA_OK) return s;
  void* scratch = nullptr;
  if ((s = noalloc_scratch_address(&scratch)) != MLA_OK) return s;
  // Same carve as mla_sparse_prefill_ex. The only word that has to start at zero, the attention
  // stage's tile counter, is zeroed by the selection stage; every other word is written by the
  // launch before the one that reads it, so the previous call's leftovers are never used.
  cudaStream_t st = as_stream(stream);
  uint8_t* base = static_cast<uint8_t*>(scratch);
  uint16_t* kv = reinterpret_cast<uint16_t*>(base);
  uint8_t* klo = base + align_up(kv_bytes(d), 1024);
  uint32_t* bits = reinterpret_cast<uint32_t*>(klo + align_up(klo_bytes(d), 1024));
  uint32_t* sched = reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(bits) + align_up(bits_bytes(d), 1024));
  s = launch_canon(topk_idx, d, bits, nullptr, 0u, sched, st);
  if (s == MLA_OK) s = launch_kvnorm_wkvb(c_kv, gamma, wkv_b, d, kv, klo, sms, k1_ctas, st);
  if (s == MLA_OK) s = launch_sparse_attn(q, k_pe, kv, klo, bits, out, lse, d, sched, sms, st);
  return s;
}

mla_status mla_get_status(void) {
  if (cudaDeviceSynchronize() != cudaSuccess) return MLA_ERR_CUDA;
  unsigned word = 0;
  if (cudaMemcpyFromSymbol(&word, mla::g_status, sizeof word) != cudaSuccess) return MLA_ERR_CUDA;
  for (int code = 1; code < 32; ++code)
    if (word & (1u << code)) return static_cast<mla_status>(code);
  return MLA_OK;
}

mla_status mla_selftest_wait_timeout(int32_t* result, void* stream) {
  if (result == nullptr || (reinterpret_cast<uintptr_t>(result) & 3u) != 0) return MLA_ERR_INVALID_ARG;
  mla::selftest_wait_timeout_kernel<<<1, 32, 0, as_stream(stream)>>>(result);
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

mla_status mla_clear_status(void) {
  const unsigned zero = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return MLA_ERR_CUDA;
  if (cudaMemcpyToSymbol(mla::g_status, &zero, sizeof zero) != cudaSuccess) return MLA_ERR_CUDA;
  return MLA_OK;
}

}  // extern "C"
