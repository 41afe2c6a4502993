// Plain fp64 CPU statement of the DeepSeek-V3.2-Exp sparse latent attention (MLA) prefill:
// kv_norm -> wkv_b up-projection -> top-k and causal masked softmax attention.
//
// TEST INFRASTRUCTURE ONLY. This file is the oracle the CUDA library is checked against.
// Only the tests, the smoke check and the benchmark's CPU-baseline leg may load it. It shares
// no code, header, table or helper with the CUDA path, and the CUDA path never calls it.
//
// Sources (model atlas pages, DeepSeek-V3.2-Exp inference/model.py excerpts):
//   * "Key-value RMSNorm" page, RMSNorm class (model.py 281-293): x.float(), mean of squares
//     over the feature axis, x * rsqrt(var + eps), times the learned weight, eps default 1e-6.
//   * "Key-value down-projection" page, MLA __init__ (model.py 523-539): kv_norm =
//     RMSNorm(kv_lora_rank = 512) with the default eps; wkv_b = ColumnParallelLinear(512,
//     n_heads * (qk_nope_head_dim + v_head_dim)); softmax_scale = qk_head_dim ** -0.5, times
//     mscale^2 with mscale = 0.1 * args.mscale * ln(rope_factor) + 1 when max_seq_len >
//     original_seq_len. Linear weights are held [out, in] (same page, "Parameters").
//   * "Keys" page, MLA prefill (model.py 574-589) and ModelArgs (model.py 56-86): wkv_b output
//     viewed [B, T, H, 256] and split [128 | 128] into k_nope and v; k = cat(k_nope, k_pe
//     expanded over heads); scores = einsum(q, k) * softmax_scale; index mask = -inf
//     everywhere, scattered to 0 at the top-k indices, plus the causal mask; softmax over keys;
//     x = einsum(scores, v). max_seq_len 16384, original_seq_len 4096, rope_factor 40, mscale 1.
//   * "Scale scores" page: S' = S * m^2 / sqrt(192), m = 1 + 0.1 ln 40, m^2 ~ 1.874.
//
// Readings where the pages leave a step open (each also listed in the design notes):
//   * eps = 1e-6 (V3.2 builds RMSNorm(512) without eps; the 1e-20 printed on the V4.1 page
//     belongs to another model).
//   * The FP8 round trip of the latent shown in the KV-cache excerpt is an option of the path
//     (below), off in the MHA prefill excerpt's own form.
//   * Causal mask: key j is allowed for query t iff j <= t (prefill from position 0).
//   * The scatter makes the selection a set: duplicate indices count once, order is irrelevant;
//     indices outside [0, t] are masked.
//   * A row whose set is empty returns out = 0 and lse = -inf (the pages' softmax would be NaN).
//   * lse = natural log of sum_j exp(s_j) over the selected keys, with s already scaled.
//   * Precision: fp64 everywhere except where the pages fix it. The RMSNorm excerpt does: it
//     computes in fp32 (x.float()) and returns (weight * x).to(dtype), i.e. rounds the kv_norm
//     output to bf16, the latent's dtype. The oracle does that step in fp32 in a fixed order
//     (ascending features; IEEE sqrt and division) and rounds to bf16 (nearest, ties to even).
//     Nothing after it is rounded: the pages do not show the Linear forward, so wkv_b's output
//     precision is open and the oracle keeps it exact. Sums run in ascending index order.
//
// Options of the path beyond the MHA prefill excerpt, each off unless asked for (readings where
// the pages leave a step open are listed with each function below and in the design notes):
//   * FP8 round trip of the normalised latent ("Keys" page, KV-cache excerpt, model.py 541-573:
//     act_quant in blocks of block_size = 128 features, then fp8 * scale in fp32, cast to bf16).
//   * FP8 block-scaled wkv_b ("Key-value down-projection" page, Linear excerpt, model.py 15 and
//     179-193: a 1-byte weight carries one fp32 scale per 128 x 128 block).
//   * YaRN rotary embedding of k_pe and of q's rotary tail ("Key-value down-projection" page,
//     model.py 565-568: apply_rotary_emb(k_pe, freqs_cis); ModelArgs on the "Keys" page:
//     rope_theta 10000, rope_factor 40, beta_fast 32, beta_slow 1, original_seq_len 4096).
//
// Build: g++ -O3 -ffp-contract=off -std=c++17 -shared -fPIC -pthread mla_oracle.cpp -o libmla_oracle.so

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

namespace {

constexpr int kLatent = 512;   // kv_lora_rank
constexpr int kNope = 128;     // qk_nope_head_dim
constexpr int kRope = 64;      // qk_rope_head_dim
constexpr int kQK = 192;       // qk_head_dim = nope + rope
constexpr int kV = 128;        // v_head_dim
constexpr int kKV = kNope + kV; // wkv_b output features per head
constexpr double kRmsEps = 1e-6;

// bf16 bit pattern -> double, exactly (bf16 is the upper half of an IEEE binary32).
double bf16_bits_to_double(uint16_t bits) {
  uint32_t u = static_cast<uint32_t>(bits) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return static_cast<double>(f);
}

// MLA __init__: qk_head_dim ** -0.5, corrected by mscale^2 for the extended context.
double softmax_scale() {
  const int max_seq_len = 4096 * 4;      // ModelArgs.max_seq_len
  const int original_seq_len = 4096;     // ModelArgs.original_seq_len
  const double rope_factor = 40.0;       // ModelArgs.rope_factor
  const double mscale_arg = 1.0;         // ModelArgs.mscale
  double s = std::pow(static_cast<double>(kQK), -0.5);
  if (max_seq_len > original_seq_len) {
    double mscale = 0.1 * mscale_arg * std::log(rope_factor) + 1.0;
    s = s * mscale * mscale;
  }
  return s;
}

// Round a double to the nearest bfloat16 value (ties to even), returned as a double.
// bfloat16 keeps 8 significant bits and float's exponent range (normals down to 2^-126,
// subnormals in steps of 2^-133); magnitudes that round past the largest finite value give inf.
double round_to_bf16(double v) {
  if (v == 0.0 || !std::isfinite(v)) return v;
  int e;
  std::frexp(v, &e);                        // |v| = m * 2^e, m in [0.5, 1)
  const int lsb_exp = std::max(e - 8, -133);   // exponent of one unit in the last place
  const double q = std::nearbyint(std::ldexp(v, -lsb_exp));   // default mode: nearest, ties even
  const double r = std::ldexp(q, lsb_exp);
  return std::fabs(r) > 3.3895313892515355e38 ? std::copysign(INFINITY, v) : r;
}

// RMSNorm.forward on one 512-wide row, before its final cast. The excerpt fixes this step's
// precision: x = x.float() makes every operation fp32. So: the mean of squares in fp32 (summed in
// ascending feature order; each square of a bf16 value is exact in fp32), var + eps in fp32,
// rsqrt as 1 / sqrt with IEEE-rounded fp32 sqrt and division, then x * r and weight * x in fp32.
void kv_norm_row_precast(const uint16_t* x_bits, const float* gamma, float* y) {
  float x[kLatent];
  float sum_sq = 0.0f;
  for (int c = 0; c < kLatent; ++c) {
    x[c] = static_cast<float>(bf16_bits_to_double(x_bits[c]));
    sum_sq = sum_sq + x[c] * x[c];
  }
  const float var = sum_sq / static_cast<float>(kLatent);
  const float r = 1.0f / std::sqrt(var + static_cast<float>(kRmsEps));
  for (int c = 0; c < kLatent; ++c) y[c] = gamma[c] * (x[c] * r);
}

// The excerpt ends with `.to(dtype)`: the output goes back to the input's dtype, bf16 for the
// bf16 latent this path takes.
void kv_norm_row(const uint16_t* x_bits, const float* gamma, double* y) {
  float yf[kLatent];
  kv_norm_row_precast(x_bits, gamma, yf);
  for (int c = 0; c < kLatent; ++c) y[c] = round_to_bf16(static_cast<double>(yf[c]));
}

// Round a double to the nearest value of the FP8 format e4m3 (float8_e4m3fn: 4 exponent bits with
// bias 7, 3 mantissa bits, no infinities; largest finite 448, smallest normal 2^-6, subnormals in
// steps of 2^-9), ties to even. Magnitudes beyond 448 saturate to 448.
double round_to_e4m3(double v) {
  if (v == 0.0 || std::isnan(v)) return v;
  const double a = std::fabs(v);
  int e;
  std::frexp(a, &e);                           // a = m * 2^e, m in [0.5, 1): leading bit 2^(e-1)
  const int lsb_exp = std::max(e - 1 - 3, -9); // three bits below the leading one, or 2^-9
  double r = std::ldexp(std::nearbyint(std::ldexp(a, -lsb_exp)), lsb_exp);
  if (r > 448.0) r = 448.0;
  return std::copysign(r, v);
}

// The value of an e4m3 byte (NaN for the two NaN codes).
double e4m3_value(uint8_t b) {
  const int sign = b >> 7, e = (b >> 3) & 15, m = b & 7;
  double v;
  if (e == 15 && m == 7) return std::numeric_limits<double>::quiet_NaN();
  if (e == 0)
    v = std::ldexp(static_cast<double>(m), -9);               // m/8 * 2^-6
  else
    v = std::ldexp(1.0 + m / 8.0, e - 7);
  return sign ? -v : v;
}

// KV-cache excerpt: kv_fp8, kv_scale = act_quant(kv, block_size); kv = (kv_fp8 * kv_scale).to(bf16).
// act_quant's format and scale rule are not on the pages. Reading: FP8 e4m3 (the cache's format),
// one fp32 scale per block of 128 consecutive latent features, scale = max|x| / 448 over the
// block (1 for an all-zero block), x / scale in fp32 rounded to nearest e4m3; the dequantisation
// is e4m3 * scale in fp32 and the cast rounds to nearest bf16. Applied in place on one 512-wide
// row of bf16 values (held as doubles).
void fp8_latent_round_trip(double* y) {
  constexpr int kBlock = 128;
  for (int b0 = 0; b0 < kLatent; b0 += kBlock) {
    float amax = 0.0f;
    for (int c = b0; c < b0 + kBlock; ++c) amax = std::max(amax, static_cast<float>(std::fabs(y[c])));
    const float scale = amax > 0.0f ? amax / 448.0f : 1.0f;
    for (int c = b0; c < b0 + kBlock; ++c) {
      const float x = static_cast<float>(y[c]) / scale;
      const float qv = static_cast<float>(round_to_e4m3(static_cast<double>(x)));
      y[c] = round_to_bf16(static_cast<double>(qv * scale));
    }
  }
}

// Linear excerpt: a 1-byte weight [out, in] carries fp32 scales [ceil(out/128), ceil(in/128)],
// one per 128 x 128 block. The forward of such a layer is not on the pages. Reading: the layer
// uses the dequantised weight e4m3 * scale (fp32 product) in its compute dtype, bf16 (the dtype of
// every other Linear on the pages), i.e. rounded to nearest bf16.
double fp8_weight_value(const uint8_t* W8, const float* scale, int n, int c) {
  const float s = scale[(n / 128) * (kLatent / 128) + c / 128];
  const float w = static_cast<float>(e4m3_value(W8[static_cast<size_t>(n) * kLatent + c]));
  return round_to_bf16(static_cast<double>(w * s));
}

// YaRN rotary frequencies of the 64-wide rotary key (32 pairs). The construction of freqs_cis is
// not on the pages, only its parameters (ModelArgs). Reading: YaRN as published (Peng et al.,
// 2023) with those parameters: base frequencies theta^(-2i/64); pair i keeps its frequency when it
// turns more than beta_fast times over the original context, is divided by rope_factor when it
// turns fewer than beta_slow times, and is interpolated linearly in i between the two dims where
// those counts are reached (the rotation count n is reached at dim 64 ln(L / (2 pi n)) /
// (2 ln theta), L = original_seq_len; the lower dim rounded down, the upper up). Exact (fp64).
void yarn_inv_freq(double* f) {
  constexpr int dim = kRope;
  const double theta = 10000.0, factor = 40.0, beta_fast = 32.0, beta_slow = 1.0;
  const double orig = 4096.0;
  const int max_seq_len = 4096 * 4, original_seq_len = 4096;
  const double two_pi = 2.0 * 3.14159265358979323846;
  for (int i = 0; i < dim / 2; ++i) f[i] = std::pow(theta, -2.0 * i / dim);
  if (max_seq_len <= original_seq_len) return;
  auto corr_dim = [&](double n_rot) { return dim * std::log(orig / (n_rot * two_pi)) / (2.0 * std::log(theta)); };
  double lo = std::max(std::floor(corr_dim(beta_fast)), 0.0);
  double hi = std::min(std::ceil(corr_dim(beta_slow)), static_cast<double>(dim - 1));
  if (lo == hi) hi += 0.001;
  for (int i = 0; i < dim / 2; ++i) {
    const double ramp = std::min(1.0, std::max(0.0, (i - lo) / (hi - lo)));
    const double keep = 1.0 - ramp;   // 1: original frequency, 0: divided by the factor
    f[i] = f[i] / factor * (1.0 - keep) + f[i] * keep;
  }
}

// freqs_cis of position t as fp32 pairs (cos, sin) of the exact angle t * f_i: the rotation is
// applied in fp32, as the excerpt's `.float()` views of its inputs suggest.
void rope_cos_sin(int t, const double* f, float* cs) {
  for (int i = 0; i < kRope / 2; ++i) {
    const double a = static_cast<double>(t) * f[i];
    cs[2 * i] = static_cast<float>(std::cos(a));
    cs[2 * i + 1] = static_cast<float>(std::sin(a));
  }
}

// apply_rotary_emb on one 64-wide bf16 vector at position t. Its code is not on the pages.
// Reading: features (2i, 2i+1) form the complex number x_{2i} + i x_{2i+1} (the last dimension
// viewed as pairs), multiplied by (cos + i sin) in fp32 as (a c - b s, a s + b c), each product and
// sum rounded to fp32 (no fused multiply-add), and cast back to bf16 (nearest).
void rope_rotate(const uint16_t* x_bits, const float* cs, double* y) {
  for (int i = 0; i < kRope / 2; ++i) {
    const float a = static_cast<float>(bf16_bits_to_double(x_bits[2 * i]));
    const float b = static_cast<float>(bf16_bits_to_double(x_bits[2 * i + 1]));
    const float c = cs[2 * i], sn = cs[2 * i + 1];
    const float ac = a * c, bs = b * sn, as = a * sn, bc = b * c;
    y[2 * i] = round_to_bf16(static_cast<double>(ac - bs));
    y[2 * i + 1] = round_to_bf16(static_cast<double>(as + bc));
  }
}

// Canonical selection of query t: the set {j in topk row : 0 <= j <= t}, ascending.
// scatter_(-1, topk, 0) writes 0 once per distinct index; the causal mask removes j > t.
void canon_row(const int32_t* idx, int K, int t, std::vector<int32_t>& sel) {
  sel.clear();
  for (int i = 0; i < K; ++i) {
    const int32_t j = idx[i];
    if (j >= 0 && j <= t) sel.push_back(j);
  }
  std::sort(sel.begin(), sel.end());
  sel.erase(std::unique(sel.begin(), sel.end()), sel.end());
}

// Head h of wkv_b, transposed to [512][256] doubles: wt[c*256 + f] = W[h*256 + f][c].
// W is [H*256, 512] ([out, in]); rows h*256 + [0,128) give k_nope, h*256 + [128,256) give v
// (view(B, T, H, 256) then split([128, 128])).
// W is either bf16 bits (W8 == nullptr) or e4m3 bytes W8 with block scales `scale`.
void head_weight_t(const uint16_t* W, const uint8_t* W8, const float* scale, int h, std::vector<double>& wt) {
  wt.assign(static_cast<size_t>(kLatent) * kKV, 0.0);
  for (int f = 0; f < kKV; ++f) {
    const int n = h * kKV + f;
    for (int c = 0; c < kLatent; ++c)
      wt[static_cast<size_t>(c) * kKV + f] = W8 ? fp8_weight_value(W8, scale, n, c)
                                                : bf16_bits_to_double(W[static_cast<size_t>(n) * kLatent + c]);
  }
}

// One position of one head: kv[f] = sum_c W[h*256+f][c] * y[c], c ascending.
void up_proj_row(const double* y, const double* wt, double* kv) {
  for (int f = 0; f < kKV; ++f) kv[f] = 0.0;
  for (int c = 0; c < kLatent; ++c) {
    const double yc = y[c];
    const double* w = wt + static_cast<size_t>(c) * kKV;
    for (int f = 0; f < kKV; ++f) kv[f] += w[f] * yc;
  }
}

template <class F>
void parallel_for(int64_t n, int threads, F&& fn) {
  if (threads <= 0) threads = static_cast<int>(std::thread::hardware_concurrency());
  if (threads <= 0) threads = 1;
  if (threads > n) threads = static_cast<int>(std::max<int64_t>(n, 1));
  std::atomic<int64_t> next{0};
  auto worker = [&]() {
    for (;;) {
      const int64_t i = next.fetch_add(1);
      if (i >= n) break;
      fn(i);
    }
  };
  if (threads == 1) { worker(); return; }
  std::vector<std::thread> pool;
  for (int k = 0; k < threads; ++k) pool.emplace_back(worker);
  for (auto& th : pool) th.join();
}

}  // namespace

extern "C" {

// softmax_scale of MLA __init__ (about 0.13523378).
double oracle_softmax_scale(void) { return softmax_scale(); }

// kv_norm over N rows of 512: x bf16 bits [N, 512], gamma fp32 [512] -> y [N, 512] (the values
// of the bf16 output, as doubles).
void oracle_kv_norm(const uint16_t* x, const float* gamma, int64_t N, double* y) {
  for (int64_t r = 0; r < N; ++r) kv_norm_row(x + r * kLatent, gamma, y + r * kLatent);
}

// kv_norm before its final cast to bf16 (the fp32 values, as doubles).
void oracle_kv_norm_precast(const uint16_t* x, const float* gamma, int64_t N, double* y) {
  float yf[kLatent];
  for (int64_t r = 0; r < N; ++r) {
    kv_norm_row_precast(x + r * kLatent, gamma, yf);
    for (int c = 0; c < kLatent; ++c) y[r * kLatent + c] = yf[c];
  }
}

// The bf16 rounding the kv_norm output goes through, elementwise.
void oracle_round_to_bf16(const double* x, int64_t n, double* y) {
  for (int64_t i = 0; i < n; ++i) y[i] = round_to_bf16(x[i]);
}

// wkv_b up-projection of N normalized rows for all H heads:
// y fp64 [N, 512], W bf16 bits [H*256, 512] -> k_nope fp64 [N, H, 128], v fp64 [N, H, 128].
void oracle_up_proj(const double* y, const uint16_t* W, int H, int64_t N, double* k_nope, double* v) {
  std::vector<double> wt;
  double kv[kKV];
  for (int h = 0; h < H; ++h) {
    head_weight_t(W, nullptr, nullptr, h, wt);
    for (int64_t r = 0; r < N; ++r) {
      up_proj_row(y + r * kLatent, wt.data(), kv);
      for (int d = 0; d < kNope; ++d) k_nope[(r * H + h) * kNope + d] = kv[d];
      for (int d = 0; d < kV; ++d) v[(r * H + h) * kV + d] = kv[kNope + d];
    }
  }
}

// Canonical selection of one row; writes the ascending set to sel (capacity >= K), returns n.
int oracle_canon_row(const int32_t* idx, int K, int t, int32_t* sel) {
  std::vector<int32_t> s;
  canon_row(idx, K, t, s);
  std::copy(s.begin(), s.end(), sel);
  return static_cast<int>(s.size());
}

// The prefill path on selected query rows and heads.
//   q      bf16 bits [B, T, H, 192] (dims 0..127 pair with k_nope, 128..191 with k_pe)
//   c_kv   bf16 bits [B, T, 512]    (latent before kv_norm)
//   k_pe   bf16 bits [B, T, 64]     (rotary key shared by all heads)
//   gamma  fp32 [512]               (kv_norm weight)
//   W      bf16 bits [H*256, 512]   (wkv_b weight, [out, in]); unused when W8 is given
//   W8, W_scale  e4m3 bytes [H*256, 512] and fp32 scales [2H, 4] of an FP8 block-scaled wkv_b
//          (NULL: W is used)
//   topk   int32 [B, T, K]
//   rows   flat row ids b*T + t, n_rows of them; NULL means all B*T rows in order
//   heads  [h_begin, h_end)
//   opts   bit 0: rotate q[..., 128:192] at position t and k_pe at position j (YaRN RoPE, the
//          inputs then being unrotated); bit 1: FP8 round trip of the normalised latent;
//          bit 2: rounding emulation, a diagnostic of the pages' own bf16 arithmetic: wkv_b's
//          output, the scores before and after the scale, the softmax weights and out are
//          rounded to bf16 where the MHA prefill excerpt's bf16 tensors would hold them (lse is
//          taken from the rounded scores)
//   out    fp64 [n_rows, h_end - h_begin, 128];  lse fp64 [n_rows, h_end - h_begin];
//   n_keys int32 [n_rows] (may be NULL)
// Returns 0, or -1 on a bad argument.
int oracle_prefill_opt(int B, int T, int H, int K, const uint16_t* q, const uint16_t* c_kv,
                       const uint16_t* k_pe, const float* gamma, const uint16_t* W, const uint8_t* W8,
                       const float* W_scale, const int32_t* topk, int64_t n_rows, const int64_t* rows,
                       int h_begin, int h_end, int opts, double* out, double* lse, int32_t* n_keys,
                       int threads) {
  if (B < 1 || T < 1 || H < 1 || K < 1 || h_begin < 0 || h_end > H || h_begin >= h_end) return -1;
  if (W8 != nullptr && W_scale == nullptr) return -1;
  const bool rope = (opts & 1) != 0, fp8_latent = (opts & 2) != 0, emulate = (opts & 4) != 0;
  const int64_t BT = static_cast<int64_t>(B) * T;
  std::vector<int64_t> row_ids;
  if (rows == nullptr) {
    row_ids.resize(BT);
    for (int64_t r = 0; r < BT; ++r) row_ids[r] = r;
  } else {
    row_ids.assign(rows, rows + n_rows);
    for (int64_t r : row_ids)
      if (r < 0 || r >= BT) return -1;
  }
  const int64_t NR = static_cast<int64_t>(row_ids.size());
  const int HS = h_end - h_begin;
  const double scale = softmax_scale();

  // 1. Canonical selections of the requested rows.
  std::vector<std::vector<int32_t>> sel(NR);
  parallel_for(NR, threads, [&](int64_t i) {
    const int64_t r = row_ids[i];
    const int t = static_cast<int>(r % T);
    canon_row(topk + r * K, K, t, sel[i]);
  });
  if (n_keys)
    for (int64_t i = 0; i < NR; ++i) n_keys[i] = static_cast<int32_t>(sel[i].size());

  // 2. kv_norm (and the FP8 round trip) of every position any requested row can reach
  //    (j <= max t of its batch), and the rotary key of those positions.
  std::vector<int> tmax(B, -1);
  for (int64_t r : row_ids) tmax[r / T] = std::max(tmax[r / T], static_cast<int>(r % T));
  std::vector<double> y(static_cast<size_t>(BT) * kLatent, 0.0);
  std::vector<double> kpe(static_cast<size_t>(BT) * kRope, 0.0);
  double inv_freq[kRope / 2];
  yarn_inv_freq(inv_freq);
  parallel_for(BT, threads, [&](int64_t r) {
    if (static_cast<int>(r % T) > tmax[r / T]) return;
    kv_norm_row(c_kv + r * kLatent, gamma, y.data() + r * kLatent);
    if (fp8_latent) fp8_latent_round_trip(y.data() + r * kLatent);
    if (rope) {
      float cs[kRope];
      rope_cos_sin(static_cast<int>(r % T), inv_freq, cs);
      rope_rotate(k_pe + r * kRope, cs, kpe.data() + r * kRope);
    } else {
      for (int d = 0; d < kRope; ++d) kpe[r * kRope + d] = bf16_bits_to_double(k_pe[r * kRope + d]);
    }
  });

  // 3. Per (batch, head): up-project the reachable positions, then attend each requested row.
  std::vector<std::vector<int64_t>> rows_of_batch(B);
  for (int64_t i = 0; i < NR; ++i) rows_of_batch[row_ids[i] / T].push_back(i);
  const int64_t units = static_cast<int64_t>(B) * HS;
  parallel_for(units, threads, [&](int64_t u) {
    const int b = static_cast<int>(u / HS);
    const int h = h_begin + static_cast<int>(u % HS);
    if (rows_of_batch[b].empty()) return;
    std::vector<double> wt;
    head_weight_t(W, W8, W_scale, h, wt);
    const int npos = tmax[b] + 1;
    std::vector<double> kv(static_cast<size_t>(npos) * kKV);  // [j][k_nope 128 | v 128]
    for (int j = 0; j < npos; ++j) {
      double* kvj = kv.data() + static_cast<size_t>(j) * kKV;
      up_proj_row(y.data() + (static_cast<int64_t>(b) * T + j) * kLatent, wt.data(), kvj);
      if (emulate)   // kv = self.wkv_b(kv): a bf16 Linear's output
        for (int f = 0; f < kKV; ++f) kvj[f] = round_to_bf16(kvj[f]);
    }
    std::vector<double> s;
    for (int64_t i : rows_of_batch[b]) {
      const int64_t r = row_ids[i];
      double* o = out + (i * HS + (h - h_begin)) * kV;
      double* l = lse + i * HS + (h - h_begin);
      const std::vector<int32_t>& S = sel[i];
      if (S.empty()) {
        for (int d = 0; d < kV; ++d) o[d] = 0.0;
        *l = -std::numeric_limits<double>::infinity();
        continue;
      }
      // q row of this head (its rotary tail rotated at position t under RoPE), and
      // k = cat(k_nope, k_pe) for every selected key.
      double qh[kQK];
      const uint16_t* qrow = q + (r * H + h) * kQK;
      for (int d = 0; d < kNope; ++d) qh[d] = bf16_bits_to_double(qrow[d]);
      if (rope) {
        float cs[kRope];
        rope_cos_sin(static_cast<int>(r % T), inv_freq, cs);
        rope_rotate(qrow + kNope, cs, qh + kNope);
      } else {
        for (int d = 0; d < kRope; ++d) qh[kNope + d] = bf16_bits_to_double(qrow[kNope + d]);
      }
      s.resize(S.size());
      for (size_t a = 0; a < S.size(); ++a) {
        const int j = S[a];
        const double* kn = kv.data() + static_cast<size_t>(j) * kKV;
        const double* kp = kpe.data() + (static_cast<int64_t>(b) * T + j) * kRope;
        double dot = 0.0;
        for (int d = 0; d < kNope; ++d) dot += qh[d] * kn[d];
        for (int d = 0; d < kRope; ++d) dot += qh[kNope + d] * kp[d];
        // einsum(q, k) into a bf16 tensor, then .mul_(softmax_scale) in bf16 (emulation)
        s[a] = emulate ? round_to_bf16(round_to_bf16(dot) * scale) : dot * scale;
      }
      // softmax over the selected keys, then the value mix.
      double M = s[0];
      for (double x : s) M = std::max(M, x);
      double Z = 0.0;
      for (double& x : s) {
        x = std::exp(x - M);
        Z += x;
      }
      for (int d = 0; d < kV; ++d) o[d] = 0.0;
      if (emulate) {
        // scores.softmax(-1) into bf16 weights, einsum with v into a bf16 out
        for (size_t a = 0; a < S.size(); ++a) {
          const double* vj = kv.data() + static_cast<size_t>(S[a]) * kKV + kNope;
          const double p = round_to_bf16(s[a] / Z);
          for (int d = 0; d < kV; ++d) o[d] += p * vj[d];
        }
        for (int d = 0; d < kV; ++d) o[d] = round_to_bf16(o[d]);
      } else {
        for (size_t a = 0; a < S.size(); ++a) {
          const double* vj = kv.data() + static_cast<size_t>(S[a]) * kKV + kNope;
          const double p = s[a];
          for (int d = 0; d < kV; ++d) o[d] += p * vj[d];
        }
        for (int d = 0; d < kV; ++d) o[d] /= Z;
      }
      *l = M + std::log(Z);
    }
  });
  return 0;
}

// The MHA prefill excerpt alone (no RoPE, no FP8 step, bf16 wkv_b).
int oracle_prefill(int B, int T, int H, int K, const uint16_t* q, const uint16_t* c_kv,
                   const uint16_t* k_pe, const float* gamma, const uint16_t* W,
                   const int32_t* topk, int64_t n_rows, const int64_t* rows, int h_begin,
                   int h_end, double* out, double* lse, int32_t* n_keys, int threads) {
  return oracle_prefill_opt(B, T, H, K, q, c_kv, k_pe, gamma, W, nullptr, nullptr, topk, n_rows, rows, h_begin,
                            h_end, 0, out, lse, n_keys, threads);
}

// The normalised latent the path up-projects, per position: kv_norm, then (fp8_latent != 0) the
// FP8 round trip. c_kv bf16 bits [N, 512] -> y [N, 512] (bf16 values as doubles). This is what the
// KV-cache excerpt writes into kv_cache.
void oracle_latent(const uint16_t* c_kv, const float* gamma, int64_t N, int fp8_latent, double* y) {
  for (int64_t r = 0; r < N; ++r) {
    kv_norm_row(c_kv + r * kLatent, gamma, y + r * kLatent);
    if (fp8_latent) fp8_latent_round_trip(y + r * kLatent);
  }
}

// e4m3 rounding of n doubles (saturating at 448), and the value of each of the 256 e4m3 codes.
void oracle_round_to_e4m3(const double* x, int64_t n, double* y) {
  for (int64_t i = 0; i < n; ++i) y[i] = round_to_e4m3(x[i]);
}
void oracle_e4m3_values(double* v) {
  for (int b = 0; b < 256; ++b) v[b] = e4m3_value(static_cast<uint8_t>(b));
}

// The effective bf16 weight of an FP8 block-scaled wkv_b: W8 e4m3 [rows, 512], scales
// [ceil(rows/128), 4] -> w [rows, 512] (bf16 values as doubles).
void oracle_fp8_weight(const uint8_t* W8, const float* scale, int rows, double* w) {
  for (int n = 0; n < rows; ++n)
    for (int c = 0; c < kLatent; ++c) w[static_cast<size_t>(n) * kLatent + c] = fp8_weight_value(W8, scale, n, c);
}

// YaRN: the 32 rotary frequencies (radians per position), and rotary embedding of N 64-wide bf16
// vectors at positions pos[N] -> y [N, 64] (bf16 values as doubles).
void oracle_yarn_inv_freq(double* f) { yarn_inv_freq(f); }
void oracle_rope(const uint16_t* x, const int32_t* pos, int64_t N, double* y) {
  double f[kRope / 2];
  yarn_inv_freq(f);
  float cs[kRope];
  for (int64_t r = 0; r < N; ++r) {
    rope_cos_sin(pos[r], f, cs);
    rope_rotate(x + r * kRope, cs, y + r * kRope);
  }
}

}  // extern "C"
