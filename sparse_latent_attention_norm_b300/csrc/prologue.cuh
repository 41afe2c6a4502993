// Optional prologue stages of the prefill, each off unless the caller asks for it:
//
//   wkvb_dequant_kernel  FP8 block-scaled wkv_b -> the bf16 weight the GEMM stage reads.
//     "Key-value down-projection" page, Linear excerpt (model.py 15, 179-193): a 1-byte weight
//     [out, in] carries fp32 scales [ceil(out/128), ceil(in/128)], one per 128 x 128 block. The
//     layer's forward is not on the pages; the weight used is e4m3 * scale (fp32 product) in the
//     layer's compute dtype, bf16, rounded to nearest.
//
//   rope_kpe_kernel      YaRN rotary embedding of k_pe ("Key-value down-projection" page,
//     model.py 565-568: k_pe = apply_rotary_emb(k_pe, freqs_cis)) at positions 0..T-1, and the
//     table of (cos, sin) per position and pair that the attention stage uses to rotate q's
//     rotary tail the same way. Pair i of a 64-wide vector is features (2i, 2i+1), multiplied as
//     a complex number by e^{i t f_i} in fp32 (each product and sum rounded, no fused multiply-add)
//     and cast back to bf16. The angle t * f_i and its cos / sin are taken in fp64 and rounded to
//     fp32, so the table holds the fp32 values of the exact rotation. The frequencies f_i (YaRN,
//     from ModelArgs: rope_theta 10000, rope_factor 40, beta_fast 32, beta_slow 1,
//     original_seq_len 4096) come from the host in fp64. The same kernel copies k_pe (rotated or
//     as given) into the caller's pe_cache (KV-cache excerpt, model.py 541-573).
#pragma once

#include "ptx.cuh"

namespace mla {

constexpr int kRopePairs = 32;

struct RopeFreqs {
  double f[kRopePairs];   // radians per position of pair i
};

// One thread per 16 weight bytes: 16 e4m3 codes of one row -> 16 bf16 values (32 bytes).
__global__ void __launch_bounds__(256) wkvb_dequant_kernel(const uint8_t* __restrict__ w8,
                                                           const float* __restrict__ scale, int rows,
                                                           uint16_t* __restrict__ w) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;   // 16-byte group
  const int64_t groups = static_cast<int64_t>(rows) * (512 / 16);
  if (i >= groups) return;
  const int n = static_cast<int>(i / 32), c0 = static_cast<int>(i % 32) * 16;
  const float s = __ldg(scale + (n / 128) * 4 + c0 / 128);
  const uint4 v = __ldg(reinterpret_cast<const uint4*>(w8) + i);
  const uint32_t words[4] = {v.x, v.y, v.z, v.w};
  uint32_t o[8];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const uint16_t q2 = static_cast<uint16_t>(words[k] >> (16 * hh));
      uint32_t h2;
      asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(q2));   // exact
      const float lo = f16_bits_to_float(static_cast<uint16_t>(h2 & 0xFFFFu));
      const float hi = f16_bits_to_float(static_cast<uint16_t>(h2 >> 16));
      o[2 * k + hh] = pack_bf16x2(__fmul_rn(lo, s), __fmul_rn(hi, s));
    }
  }
  stg_v8(w + i * 16, o);
}

// One warp per position (b, t), lane i = pair i.
//   k_pe       [B, T, 64] bf16 input
//   k_pe_rot   [B, T, 64] bf16 output (rotated), or null
//   cs         [T, 32] float2 (cos, sin) output, written by the warps of batch 0, or null
//   pe_cache   [B, cache_len, 64] bf16 output, or null: k_pe rotated when `rotate`, as given otherwise
__global__ void __launch_bounds__(256) rope_kpe_kernel(const uint16_t* __restrict__ k_pe, int B, int T, int rotate,
                                                       const RopeFreqs freqs, uint16_t* __restrict__ k_pe_rot,
                                                       float2* __restrict__ cs, uint16_t* __restrict__ pe_cache,
                                                       int cache_len) {
  const int64_t pos = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int i = lane_id();
  if (pos >= static_cast<int64_t>(B) * T) return;
  const int b = static_cast<int>(pos / T), t = static_cast<int>(pos % T);
  const uint32_t x = __ldg(reinterpret_cast<const uint32_t*>(k_pe + pos * 64) + i);
  uint32_t y = x;
  if (rotate) {
    double sd, cd;
    sincos(static_cast<double>(t) * freqs.f[i], &sd, &cd);
    const float c = static_cast<float>(cd), sn = static_cast<float>(sd);
    if (b == 0 && cs != nullptr) cs[static_cast<int64_t>(t) * kRopePairs + i] = make_float2(c, sn);
    const float a = __uint_as_float(x << 16), bb = __uint_as_float(x & 0xFFFF0000u);
    y = pack_bf16x2(__fsub_rn(__fmul_rn(a, c), __fmul_rn(bb, sn)), __fadd_rn(__fmul_rn(a, sn), __fmul_rn(bb, c)));
    if (k_pe_rot != nullptr) reinterpret_cast<uint32_t*>(k_pe_rot + pos * 64)[i] = y;
  }
  if (pe_cache != nullptr)
    reinterpret_cast<uint32_t*>(pe_cache + (static_cast<int64_t>(b) * cache_len + t) * 64)[i] = y;
}

}  // namespace mla
