// Stages 2-3: kv_norm fused into the wkv_b up-projection (tcgen05 GEMM, TMA-fed, TMEM accumulators).
//
//   y[r, :]  = bf16( gamma * (c_kv[r, :] * (1 / sqrt(mean(c_kv[r, :]^2) + 1e-6))) )
//              (RMSNorm class, model.py 281-293: x.float(), mean of squares, x * rsqrt(var + eps),
//               weight * x, cast back to the input dtype; kv_norm = RMSNorm(512), MLA __init__).
//              Computed in fp32 as the excerpt does, in a fixed order: squares summed in
//              ascending feature order, IEEE-rounded sqrt and division, no fused multiply-adds.
//   kv[r, n] = sum_c y[r, c] * wkv_b[n, c]   (ColumnParallelLinear, weight [out, in])
// with r = b*T + t and n = h*256 + f ("Keys" page: kv.view(B, T, H, 256), split [128 | 128] into
// k_nope and v). Outputs, head-major so the attention stage reads each head's keys and values as
// contiguous blocks:
//   kv  [B, H, T, 256] fp16:  k_hi = fp16(k_nope) in features 0..127, fp16(v) in 128..255
//   klo [B, H, T, 128] e4m3:  (k_nope - k_hi) * 2^11, the part of k_nope fp16 drops
// k_hi + klo * 2^-11 carries k_nope to about 2^-14 relative, enough for lse to 1e-3 on rows
// whose softmax sits on one or two keys; fp16 alone (2^-11) is not.
//
// Tiling: one unit = 128 rows x one head (256 output features) x the whole latent (512). The A
// tile (128 x 512 bf16, 128 KB) stays in shared memory while a CTA walks the heads of its row
// tile; it is loaded by TMA, normalised in place (the norm's only input is that row), and then
// used by 32 UMMAs (M=128, N=256, K=16) per head. W streams through a 3-stage TMA ring of
// 256 x 64 slices. Accumulators are double-buffered in TMEM (2 x 256 columns) so the epilogue of
// one head overlaps the MMAs of the next.
//
// Warp roles (192 threads): warp 0 TMA producer, warp 1 TMEM owner + MMA issuer, warps 2-5
// normalise A and run the epilogue (warp w reads TMEM lanes 32*(w%4) .. +31).
#pragma once

#include "ptx.cuh"

namespace mla {
namespace k1 {

constexpr int BM = 128;
constexpr int BN = 256;                      // one head: 128 k_nope + 128 v features
constexpr int KDIM = 512;                    // kv_lora_rank
constexpr int KATOM = 64;                    // bf16 elements per 128-byte swizzle row
constexpr int NKATOM = KDIM / KATOM;         // 8
constexpr int A_ATOM_BYTES = BM * 128;       // 16 KB
constexpr int A_BYTES = NKATOM * A_ATOM_BYTES;  // 128 KB
constexpr int B_STAGE_BYTES = BN * 128;      // 32 KB
constexpr int NSTAGE = 3;
constexpr int THREADS = 192;
constexpr int SMEM_BYTES = A_BYTES + NSTAGE * B_STAGE_BYTES + 1024;  // + alignment slack
constexpr uint32_t TMEM_COLS = 512;
constexpr float RMS_EPS = 1e-6f;

struct Params {
  int M;          // B * T rows
  int T;          // positions per batch (row r -> b = r / T, t = r % T)
  int H;          // heads
  int units;      // ceil(M / 128) * H
  const float* gamma;
  uint16_t* kv;   // [B, H, T, 256] fp16 (k_hi | v)
  uint8_t* klo;   // [B, H, T, 128] e4m3 ((k_nope - k_hi) * 2^11)
};

constexpr float KLO_SCALE = 2048.0f;   // 2^11

__global__ void __launch_bounds__(THREADS, 1)
    kvnorm_wkvb_kernel(const __grid_constant__ CUtensorMap tm_ckv, const __grid_constant__ CUtensorMap tm_w,
                       const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + A_BYTES;

  __shared__ uint64_t a_full, a_ready, a_free, drain;
  __shared__ uint64_t b_full[NSTAGE], b_empty[NSTAGE];
  __shared__ uint64_t acc_full[2], acc_empty[2];
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  volatile int* abort_p = &abort_flag;

  const int warp = warp_id();
  const int lane = lane_id();

  // contiguous range of units for this CTA, m-major (u -> m = u / H, h = u % H)
  const int G = gridDim.x;
  const int u_begin = static_cast<int>((static_cast<int64_t>(p.units) * blockIdx.x) / G);
  const int u_end = static_cast<int>((static_cast<int64_t>(p.units) * (blockIdx.x + 1)) / G);

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&a_full, 1);
    mbar_init(&a_ready, 128);
    mbar_init(&a_free, 1);
    mbar_init(&drain, 1);
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(&b_full[s], 1);
      mbar_init(&b_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&acc_full[s], 1);
      mbar_init(&acc_empty[s], 128);
    }
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_ckv);
    tma_prefetch_desc(&tm_w);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      int cur_m = -1, seg = 0, stage = 0;
      uint32_t phase = 0;
      bool a_pending = false;
      uint32_t a_parity = 0;
      bool pending[NSTAGE] = {};
      uint32_t pend_parity[NSTAGE] = {};
      bool ok = true;
      for (int u = u_begin; u < u_end && ok; ++u) {
        const int m = u / p.H, h = u % p.H;
        if (m != cur_m) {
          if (seg > 0) {
            if (!mbar_wait(&a_free, (seg - 1) & 1, abort_p)) { ok = false; break; }
            a_pending = false;
          }
          mbar_arrive_expect_tx(&a_full, A_BYTES);
          for (int a = 0; a < NKATOM; ++a) tma_load_2d(sA + a * A_ATOM_BYTES, &tm_ckv, &a_full, a * KATOM, m * BM);
          a_pending = true;
          a_parity = seg & 1;
          cur_m = m;
          ++seg;
        }
        for (int ka = 0; ka < NKATOM; ++ka) {
          if (!mbar_wait(&b_empty[stage], phase ^ 1, abort_p)) { ok = false; break; }
          pending[stage] = false;
          mbar_arrive_expect_tx(&b_full[stage], B_STAGE_BYTES);
          tma_load_2d(sB + stage * B_STAGE_BYTES, &tm_w, &b_full[stage], ka * KATOM, h * BN);
          pending[stage] = true;
          pend_parity[stage] = phase;
          if (++stage == NSTAGE) { stage = 0; phase ^= 1; }
        }
      }
      if (!ok) {
        // unwinding: let the copies already issued land before the CTA's shared memory goes away
        for (int s = 0; s < NSTAGE; ++s)
          if (pending[s]) mbar_wait(&b_full[s], pend_parity[s], nullptr);
        if (a_pending) mbar_wait(&a_full, a_parity, nullptr);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(BM, BN, false, false);
      const uint32_t sa = smem_u32(sA), sb = smem_u32(sB);
      int cur_m = -1, seg = 0, stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool issued = false;
      for (int u = u_begin; u < u_end; ++u) {
        const int m = u / p.H;
        if (m != cur_m) {
          if (seg > 0) umma_commit(&a_free);
          if (!mbar_wait(&a_ready, seg & 1, abort_p)) break;
          tc_fence_after();
          cur_m = m;
          ++seg;
        }
        if (!mbar_wait(&acc_empty[acc], acc_phase ^ 1, abort_p)) break;
        tc_fence_after();
        const uint32_t d = tmem + static_cast<uint32_t>(acc * BN);
        bool ok = true;
        for (int ka = 0; ka < NKATOM; ++ka) {
          if (!mbar_wait(&b_full[stage], phase, abort_p)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const uint64_t ad = sdesc_sw128(sa + ka * A_ATOM_BYTES + k4 * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(sb + stage * B_STAGE_BYTES + k4 * 32, 16, 1024);
            umma_ss(d, ad, bd, idesc, (ka | k4) != 0 ? 1u : 0u);
          }
          issued = true;
          umma_commit(&b_empty[stage]);
          if (++stage == NSTAGE) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        umma_commit(&acc_full[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      if (issued) {
        // every MMA this thread issued has finished before TMEM is released
        umma_commit(&drain);
        mbar_wait(&drain, 0, nullptr);
      }
    }
  } else {
    // ------------------------------------------------ normalisation + epilogue (128 threads)
    const int q = warp & 3;
    const int r = q * 32 + lane;               // row within the tile == TMEM lane
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(q * 32) << 16);
    int cur_m = -1, seg = 0, acc = 0;
    uint32_t acc_phase = 0;
    for (int u = u_begin; u < u_end; ++u) {
      const int m = u / p.H, h = u % p.H;
      if (m != cur_m) {
        if (!mbar_wait(&a_full, seg & 1, abort_p)) break;
        // RMSNorm of row r, in place in the swizzled A tile: logical 16-byte chunk c of a 128-byte
        // row sits at chunk position c ^ (r & 7). Sum of squares in ascending feature order.
        uint8_t* row_base = sA + r * 128;
        float ss = 0.f;
#pragma unroll 1
        for (int a = 0; a < NKATOM; ++a) {
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 v = *reinterpret_cast<const uint4*>(row_base + a * A_ATOM_BYTES + ((c ^ (r & 7)) * 16));
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float lo = __uint_as_float(w[e] << 16);
              const float hi = __uint_as_float(w[e] & 0xFFFF0000u);
              ss = __fadd_rn(ss, __fmul_rn(lo, lo));
              ss = __fadd_rn(ss, __fmul_rn(hi, hi));
            }
          }
        }
        const float var = __fmul_rn(ss, 1.0f / KDIM);   // exact: division by a power of two
        const float rinv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(var, RMS_EPS)));
#pragma unroll 1
        for (int a = 0; a < NKATOM; ++a) {
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            uint4* ptr = reinterpret_cast<uint4*>(row_base + a * A_ATOM_BYTES + c * 16);
            const uint4 v = *ptr;
            const int col0 = a * KATOM + ((c ^ (r & 7)) * 8);
            const float4 g0 = __ldg(reinterpret_cast<const float4*>(p.gamma + col0));
            const float4 g1 = __ldg(reinterpret_cast<const float4*>(p.gamma + col0 + 4));
            const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            uint32_t o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float lo = __uint_as_float(w[e] << 16);
              const float hi = __uint_as_float(w[e] & 0xFFFF0000u);
              o[e] = pack_bf16x2(__fmul_rn(g[2 * e], __fmul_rn(lo, rinv)), __fmul_rn(g[2 * e + 1], __fmul_rn(hi, rinv)));
            }
            *ptr = make_uint4(o[0], o[1], o[2], o[3]);
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(&a_ready);
        cur_m = m;
        ++seg;
      }
      if (!mbar_wait(&acc_full[acc], acc_phase, abort_p)) break;
      tc_fence_after();
      const int row_g = m * BM + r;
      const bool valid = row_g < p.M;
      uint16_t* dst = nullptr;
      uint8_t* dlo = nullptr;
      if (valid) {
        const int b = row_g / p.T, t = row_g % p.T;
        const int64_t prow = (static_cast<int64_t>(b) * p.H + h) * p.T + t;
        dst = p.kv + prow * BN;
        dlo = p.klo + prow * 128;
      }
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 32) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(lane_addr + static_cast<uint32_t>(acc * BN + c0), v);
        tmem_ld_wait();
        if (valid) {
          uint32_t hw[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) hw[i] = pack_f16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
          uint4* d4 = reinterpret_cast<uint4*>(dst + c0);
#pragma unroll
          for (int i = 0; i < 4; ++i) d4[i] = make_uint4(hw[4 * i], hw[4 * i + 1], hw[4 * i + 2], hw[4 * i + 3]);
          if (c0 < 128) {
            // residual of k_nope after the fp16 rounding, scaled by 2^11, as e4m3
            uint32_t lw[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              float rr[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int k = 4 * i + e;
                const uint16_t hb = static_cast<uint16_t>((hw[k >> 1] >> ((k & 1) * 16)) & 0xFFFFu);
                rr[e] = __fmul_rn(__fsub_rn(__uint_as_float(v[k]), f16_bits_to_float(hb)), KLO_SCALE);
              }
              lw[i] = static_cast<uint32_t>(pack_e4m3x2(rr[0], rr[1])) | (static_cast<uint32_t>(pack_e4m3x2(rr[2], rr[3])) << 16);
            }
            uint4* l4 = reinterpret_cast<uint4*>(dlo + c0);
            l4[0] = make_uint4(lw[0], lw[1], lw[2], lw[3]);
            l4[1] = make_uint4(lw[4], lw[5], lw[6], lw[7]);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&acc_empty[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace k1
}  // namespace mla
