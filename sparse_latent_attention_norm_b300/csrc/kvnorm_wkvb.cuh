// Stages 2-3: kv_norm fused into the wkv_b up-projection (tcgen05 GEMM over SM pairs: A and W in
// shared memory, W in by TMA, accumulators in tensor memory).
//
//   y[r, :]  = bf16( gamma * (c_kv[r, :] * (1 / sqrt(mean(c_kv[r, :]^2) + 1e-6))) )
//              (RMSNorm class, model.py 281-293: x.float(), mean of squares, x * rsqrt(var + eps),
//               weight * x, cast back to the input dtype; kv_norm = RMSNorm(512), MLA __init__).
//              Computed in fp32 as the excerpt does, in a fixed order: squares summed in
//              ascending feature order, IEEE-rounded sqrt and division, no fused multiply-adds.
//   kv[r, n] = sum_c y[r, c] * wkv_b[n, c]   (ColumnParallelLinear, weight [out, in])
// with r = (b, t) and n = h*256 + f ("Keys" page: kv.view(B, T, H, 256), split [128 | 128] into
// k_nope and v). Outputs, head-major so the attention stage reads each head's keys and values as
// contiguous blocks:
//   kv  [B, H, T, 256] fp16:  k_hi = fp16(k_nope) in features 0..127, fp16(v) in 128..255
//   klo [B, H, T, 128] e4m3:  (k_nope - k_hi) * 2^11, the part of k_nope fp16 drops
// k_hi + klo * 2^-11 carries k_nope to about 2^-14 relative, enough for lse to 1e-3 on rows
// whose softmax sits on one or two keys; fp16 alone (2^-11) is not.
//
// Tiling: the kernel runs as CTA pairs (clusters of two, one per SM pair). A row tile is 128
// positions of one batch (the last tile of a batch may be partial); a pair takes row tiles 2i
// (rank 0) and 2i+1 (rank 1), and a unit is that row-tile pair x one head (W rows h*256 + [0,256))
// x the whole latent (512). Each CTA normalises its row tile into shared memory (128 x 512 bf16,
// K-major with the 128-byte swizzle) as its half of the A operand, and takes half of each W
// slice (rank 0 the head's k_nope rows, rank 1 its v rows) through a TMA ring whose copies
// complete on the leader's (rank 0's) barriers. The leader's MMA thread issues 32 UMMAs
// M=256 N=256 K=16 per unit (tcgen05 cta_group::2: each SM computes its 128 rows x all 256
// outputs, reading A from its own shared memory and both halves of B) into one of two
// accumulators of 256 TMEM columns in each SM, so a unit's epilogue overlaps the next unit's
// MMAs. Per unit each SM streams 128 KB of W for 4,096 tensor cycles, half of what one SM
// alone with M = 128 would. The epilogue converts the accumulator and stores each row straight
// from registers with 32-byte stores (kv: 256 bytes, klo: 128 bytes per row); staging the
// outputs in shared memory for TMA stores measured slower.
//
// Warp roles (320 threads): warp 0 TMA producer of this CTA's W half; warp 1 TMEM allocation
// (jointly for the pair) and, in the leader, the MMA issuer; in the other CTA, lane 0 of warp 1
// forwards that CTA's normalisation / epilogue hand-offs (arrivals at CTA scope, so the threads'
// outstanding output stores need not drain) to the leader's barriers; warps 2-9 normalise rows
// and run the epilogue, two per TMEM lane quadrant (warp w owns TMEM lanes 32*(w%4) .. +31, its
// column group (w-2)/4 takes half of the row's latent atoms and 64 of each 128 output columns).
#pragma once

#include "mla.h"
#include "ptx.cuh"

namespace mla {
namespace k1 {

constexpr int BM = 128;                         // positions per row tile (one CTA of the pair)
constexpr int BN = 256;                         // outputs per unit: one head (k_nope 128 | v 128)
constexpr int BNH = BN / 2;                     // W rows each CTA of the pair holds
constexpr int KDIM = 512;                       // kv_lora_rank
constexpr int KATOM = 64;                       // bf16 elements per 128-byte swizzle row
constexpr int NKATOM = KDIM / KATOM;            // 8
constexpr int A_ATOM_BYTES = BM * 128;          // 16 KB: 128 rows of y x 64 latent features
constexpr int A_BYTES = NKATOM * A_ATOM_BYTES;  // 128 KB: the CTA's row tile of y
constexpr int ATOM_BYTES = BNH * 128;           // 16 KB: 128 W rows x 64 latent features
constexpr int KPS = 2;                          // latent atoms (64 features) per W stage: 8 UMMAs
constexpr int STAGES_PER_UNIT = NKATOM / KPS;   // 4
constexpr int B_STAGE_BYTES = KPS * ATOM_BYTES; // 32 KB per CTA
constexpr int NSTAGE = 3;
constexpr int NEPI = 256;                       // normalisation / epilogue threads: two warps per TMEM lane quadrant
constexpr int THREADS = 64 + NEPI;
constexpr int TILE_BYTES = A_BYTES + NSTAGE * B_STAGE_BYTES;   // 224 KB
static_assert(NKATOM % KPS == 0, "stages split the latent evenly");

// Barriers after the tiles in the dynamic shared memory (no static shared memory: the dynamic
// region then starts 1024-byte aligned, as the 128-byte swizzle needs).
struct Ctrl {
  uint64_t a_free, a_ready, drain;
  uint64_t b_full[NSTAGE], b_empty[NSTAGE];
  uint64_t acc_full[2], acc_empty[2];
  uint32_t tmem_base;
  int abort_flag;
};
constexpr int SMEM_BYTES = TILE_BYTES + static_cast<int>(sizeof(Ctrl));
static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_ACC = 0;    // two accumulators of 256 columns: 0..255 and 256..511
constexpr float RMS_EPS = 1e-6f;
constexpr float KLO_SCALE = 2048.0f;   // 2^11
constexpr int EPI_BAR = 1;             // named barrier of the four epilogue warps
constexpr int NORM_LOADS = 16;         // 16-byte loads of a c_kv row in flight during the RMSNorm

struct Params {
  int B, T, H;
  int mt_per_b;            // row tiles per batch: ceil(T / 128)
  int n_mtiles;            // B * mt_per_b
  int n_tpairs;            // ceil(n_mtiles / 2): row tiles 2i and 2i+1 go to the two CTAs of a pair
  int units;               // n_tpairs * H
  const uint16_t* c_kv;    // [B, T, 512] bf16
  const float* gamma;      // [512]
  uint16_t* kv_out;        // [B, H, T, 256] fp16
  uint8_t* klo_out;        // [B, H, T, 128] e4m3
  int fp8_latent;          // 1: the normalised latent goes through the KV cache's FP8 round trip
  uint16_t* kv_cache;      // [B, cache_len, 512] bf16 or null: receives the latent the GEMM consumes
  int cache_len;
};

// One normalised latent value: gamma * (x * r) in fp32, rounded to bf16 (RMSNorm excerpt).
__device__ __forceinline__ float norm_value(float x, float r, float g) { return __fmul_rn(g, __fmul_rn(x, r)); }

// Two bf16 values (low, high half of w) -> two e4m3 codes of (value / scale), rounded to nearest
// (satfinite), -> the dequantised values e4m3 * scale in fp32, rounded to bf16: the KV cache's
// FP8 round trip of one pair ("Keys" page, KV-cache excerpt: act_quant in blocks of 128, then
// fp8 * scale cast back to bf16).
__device__ __forceinline__ uint32_t fp8_round_trip_bf16x2(uint32_t w, float scale) {
  const float lo = __uint_as_float(w << 16), hi = __uint_as_float(w & 0xFFFF0000u);
  const uint16_t q2 = pack_e4m3x2(__fdiv_rn(lo, scale), __fdiv_rn(hi, scale));
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(q2));   // exact: e4m3 values are fp16 values
  const float qlo = f16_bits_to_float(static_cast<uint16_t>(h2 & 0xFFFFu));
  const float qhi = f16_bits_to_float(static_cast<uint16_t>(h2 >> 16));
  return pack_bf16x2(__fmul_rn(qlo, scale), __fmul_rn(qhi, scale));
}

// Named barrier of the epilogue warps that also ANDs `pred` over their NEPI threads.
__device__ __forceinline__ bool epi_sync_and(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "n"(EPI_BAR), "n"(NEPI)
      : "memory");
  return r != 0;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    kvnorm_wkvb_kernel(const __grid_constant__ CUtensorMap tm_w, const Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) set_error(kErrUnsupportedLayout);
    return;
  }
  uint8_t* sA = smem_raw;
  uint8_t* sB = smem_raw + A_BYTES;
  Ctrl& ctl = *reinterpret_cast<Ctrl*>(smem_raw + TILE_BYTES);
  uint64_t& a_free = ctl.a_free;
  uint64_t& a_ready = ctl.a_ready;
  uint64_t& drain = ctl.drain;
  uint64_t* b_full = ctl.b_full;
  uint64_t* b_empty = ctl.b_empty;
  uint64_t* acc_full = ctl.acc_full;
  uint64_t* acc_empty = ctl.acc_empty;
  volatile int* abort_p = &ctl.abort_flag;

  const int warp = warp_id();
  const int lane = lane_id();
  const uint32_t rank = cluster_ctarank();   // 0: the pair's MMA issuer and barrier owner
  const bool leader = rank == 0;
  // shared::cluster address of a barrier in the CTA of rank `r`
  auto at = [](uint64_t* bar, uint32_t r) { return mapa_shared(smem_u32(bar), r); };

  // Contiguous range of units per pair: u -> row-tile pair u / H (this CTA's row tile
  // 2 * (u / H) + rank), head u % H.
  const int G = static_cast<int>(gridDim.x >> 1);
  const int pair = static_cast<int>(blockIdx.x >> 1);
  const int u_begin = static_cast<int>((static_cast<int64_t>(p.units) * pair) / G);
  const int u_end = static_cast<int>((static_cast<int64_t>(p.units) * (pair + 1)) / G);

  if (threadIdx.x == 0) {
    ctl.abort_flag = 0;
    mbar_init(&a_free, 1);
    // leader: its normalisation threads + the peer's forwarder; peer: its normalisation threads
    mbar_init(&a_ready, leader ? NEPI + 1 : NEPI);
    mbar_init(&drain, 1);
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(&b_full[s], 1);              // the leader's expect_tx (both CTAs' bytes)
      mbar_init(&b_empty[s], 1);             // the leader's MMA commit
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&acc_full[s], 1);
      mbar_init(&acc_empty[s], leader ? NEPI + 1 : NEPI);
    }
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(&ctl.tmem_base, TMEM_COLS);
    tmem_relinquish_pair();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_w);
    // the c_kv rows of this CTA's row tiles go to L2 now, so the RMSNorm's loads hit L2
    const int m0 = u_begin / p.H, m1 = (u_end - 1) / p.H;
    for (int mp = m0; mp <= m1; ++mp) {
      const int m = 2 * mp + static_cast<int>(rank);
      if (m >= p.n_mtiles) break;
      const int b = m / p.mt_per_b, t0 = (m % p.mt_per_b) * BM;
      const int rows = min(BM, p.T - t0);
      const uint16_t* src = p.c_kv + (static_cast<int64_t>(b) * p.T + t0) * KDIM;
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(static_cast<uint32_t>(rows * KDIM * 2))
                   : "memory");
    }
  }
  tc_fence_before();
  __syncthreads();
  // the peer's barriers are initialised before any arrival or copy targets them
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer: this CTA's half of W
    // A stage is refilled once the MMAs that read it have completed (b_empty); both CTAs'
    // halves complete on the leader's b_full.
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool pending[NSTAGE] = {};
      uint32_t pend_parity[NSTAGE] = {};
      bool ok = true;
      for (int u = u_begin; u < u_end && ok; ++u) {
        const int h = u % p.H;
        for (int sk = 0; sk < STAGES_PER_UNIT; ++sk) {
          if (!mbar_wait(&b_empty[stage], phase ^ 1, abort_p)) { ok = false; break; }
          const uint32_t full = at(&b_full[stage], 0);
          if (leader) mbar_arrive_expect_tx(&b_full[stage], 2 * B_STAGE_BYTES);
          for (int a = 0; a < KPS; ++a) {
            uint8_t* dst = sB + stage * B_STAGE_BYTES + a * ATOM_BYTES;
            const int x = (sk * KPS + a) * KATOM, y = h * 256 + static_cast<int>(rank) * BNH;
            if (in_bounds(x + KATOM <= KDIM && y + BNH <= p.H * 256))
              tma_load_2d_pair(dst, &tm_w, full, x, y);
            else
              mbar_complete_tx_cluster(full, ATOM_BYTES);
          }
          pending[stage] = true;
          pend_parity[stage] = phase;
          if (++stage == NSTAGE) { stage = 0; phase ^= 1; }
        }
      }
      if (!ok && leader) {
        // unwinding: let the copies already issued land before shared memory goes away (the
        // peer's copies are covered by the drain before the pair's final cluster barrier)
        for (int s = 0; s < NSTAGE; ++s)
          if (pending[s]) mbar_wait(&b_full[s], pend_parity[s], nullptr);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------------------------------------- MMA issuer for the pair (leader CTA)
      const uint32_t idesc = idesc_bf16_f32(2 * BM, BN, false, false);
      auto commit_both = [&](uint64_t* bar) {
        umma_pair_commit(at(bar, 0));
        umma_pair_commit(at(bar, 1));
      };
      // + atom (16 KB) and K-step (32 bytes) offsets, >> 4
      const uint64_t d_a0 = sdesc_sw128(smem_u32(sA), 16, 1024);
      const uint64_t d_b0 = sdesc_sw128(smem_u32(sB), 16, 1024);
      int cur_m = -1, seg = 0, stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool issued = false;
      for (int u = u_begin; u < u_end; ++u) {
        const int mp = u / p.H;
        if (mp != cur_m) {
          // a new row-tile pair: y in both CTAs' shared memory is rewritten once every MMA
          // issued so far has completed
          if (seg > 0) commit_both(&a_free);
          if (!mbar_wait_cl(&a_ready, seg & 1, abort_p)) break;
          tc_fence_after();
          cur_m = mp;
          ++seg;
        }
        if (!mbar_wait_cl(&acc_empty[acc], acc_phase ^ 1, abort_p)) break;
        tc_fence_after();
        const uint32_t d = tmem + TM_ACC + static_cast<uint32_t>(acc * BN);
        bool ok = true;
        for (int sk = 0; sk < STAGES_PER_UNIT; ++sk) {
          if (!mbar_wait(&b_full[stage], phase, abort_p)) { ok = false; break; }
          tc_fence_after();
          const uint64_t db = d_b0 + static_cast<uint64_t>(stage * (B_STAGE_BYTES >> 4));
#pragma unroll
          for (int a = 0; a < KPS; ++a)
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) {
              const int ka = sk * KPS + a;
              umma_pair_ss(d, d_a0 + static_cast<uint64_t>(ka * (A_ATOM_BYTES >> 4)) + k4 * 2,
                           db + a * (ATOM_BYTES >> 4) + k4 * 2, idesc, (ka | k4) != 0 ? 1u : 0u);
            }
          issued = true;
          commit_both(&b_empty[stage]);
          if (++stage == NSTAGE) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        commit_both(&acc_full[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      if (issued) {
        // every MMA this thread issued has finished before tensor memory is released
        umma_pair_commit(at(&drain, 0));
        mbar_wait(&drain, 0, nullptr);
      }
    } else if (lane == 0) {
      // ---------------------------------------------- the peer's forwarder
      // Its normalisation / epilogue threads arrive on this CTA's a_ready / acc_empty at CTA
      // scope (their outstanding output stores need not drain first); this thread passes each
      // completed phase on to the leader's barrier of the same name.
      const uint32_t a_ready_lead = at(&a_ready, 0);
      int cur_m = -1, seg = 0, acc = 0;
      uint32_t acc_phase = 0;
      for (int u = u_begin; u < u_end; ++u) {
        const int mp = u / p.H;
        if (mp != cur_m) {
          if (!mbar_wait(&a_ready, seg & 1, abort_p)) break;
          mbar_arrive_cluster(a_ready_lead);
          cur_m = mp;
          ++seg;
        }
        if (!mbar_wait(&acc_empty[acc], acc_phase, abort_p)) break;
        mbar_arrive_cluster(at(&acc_empty[acc], 0));
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
    }
  } else {
    // ------------------------------------------------ normalisation + epilogue (NEPI threads)
    // Two warps per TMEM lane quadrant: both normalise the same 32 rows (each computes the row's
    // sum of squares in the same fixed order) and write half of the row's latent atoms each;
    // in the epilogue each takes 64 of the 128 columns of k_nope and of v. tcgen05.ld is
    // warp-collective and the epilogue barriers take all eight warps: every branch below is
    // uniform over them (their exits agree through epi_sync_and).
    const int q = warp & 3;
    const int cg = (warp - 2) >> 2;            // column group: 0 or 1
    const int r = q * 32 + lane;               // row within the tile == TMEM lane
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(q * 32) << 16);
    // row r's 16-byte chunk c of latent atom cc, in the 128-byte swizzle (chunk c at c ^ (r & 7))
    auto a_chunk = [&](int cc, int c) -> uint4* {
      return reinterpret_cast<uint4*>(sA + cc * A_ATOM_BYTES + r * 128 + ((c ^ (r & 7)) * 16));
    };
    auto store_a = [&](int cc, const uint32_t (&o)[32]) {
#pragma unroll
      for (int c = 0; c < 8; ++c) *a_chunk(cc, c) = make_uint4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
    };
    int cur_m = -1, seg = 0, acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int u = u_begin; u < u_end; ++u) {
      const int mp = u / p.H, h = u % p.H;
      const int m = 2 * mp + static_cast<int>(rank);   // this CTA's row tile (past the end: rows of zeros)
      const bool tile_ok = m < p.n_mtiles;
      const int b = tile_ok ? m / p.mt_per_b : p.B, t0 = tile_ok ? (m % p.mt_per_b) * BM : p.T;
      if (mp != cur_m) {
        // RMSNorm of row (b, t0 + r) into shared memory once the previous tile's MMAs are done with y
        if (seg > 0) ok = __all_sync(0xffffffffu, mbar_wait(&a_free, (seg - 1) & 1, abort_p));
        ok = epi_sync_and(ok);
        if (!ok) break;
        const int t = t0 + r;
        const bool valid = tile_ok && t < p.T && in_bounds(b < p.B);
        const uint4* row = reinterpret_cast<const uint4*>(p.c_kv + (static_cast<int64_t>(b) * p.T + (valid ? t : 0)) * KDIM);
        // sum of squares in ascending feature order; the row's 16-byte loads go out 8 at a
        // time (the tile's rows usually come from DRAM: eight round trips instead of sixteen)
        float ss = 0.f;
#pragma unroll 1
        for (int a0 = 0; a0 < KDIM / 8; a0 += NORM_LOADS) {
          uint4 vv[NORM_LOADS];
#pragma unroll
          for (int j = 0; j < NORM_LOADS; ++j) vv[j] = valid ? __ldg(row + a0 + j) : make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int j = 0; j < NORM_LOADS; ++j) {
            const uint32_t w[4] = {vv[j].x, vv[j].y, vv[j].z, vv[j].w};
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
        // y of 64 features of the row (chunk cc) as 32 bf16 pairs
        auto norm_chunk = [&](int cc, uint32_t (&o)[32]) {
#pragma unroll
          for (int a = 0; a < 8; ++a) {
            const uint4 v = valid ? __ldg(row + cc * 8 + a) : make_uint4(0, 0, 0, 0);
            const float4 g0 = __ldg(reinterpret_cast<const float4*>(p.gamma + cc * 64 + a * 8));
            const float4 g1 = __ldg(reinterpret_cast<const float4*>(p.gamma + cc * 64 + a * 8 + 4));
            const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float lo = __uint_as_float(w[e] << 16);
              const float hi = __uint_as_float(w[e] & 0xFFFF0000u);
              o[a * 4 + e] = pack_bf16x2(norm_value(lo, rinv, g[2 * e]), norm_value(hi, rinv, g[2 * e + 1]));
            }
          }
        };
        uint16_t* cache_row = (p.kv_cache != nullptr && valid)
                                  ? p.kv_cache + (static_cast<int64_t>(b) * p.cache_len + t) * KDIM
                                  : nullptr;
        if (!p.fp8_latent) {
#pragma unroll 1
          for (int cc = cg * 4; cc < cg * 4 + 4; ++cc) {   // 64 features -> one 128-byte swizzled row of atom cc
            uint32_t o[32];
            norm_chunk(cc, o);
            store_a(cc, o);
            if (cache_row)
#pragma unroll
              for (int k = 0; k < 4; ++k) stg_v8(cache_row + cc * 64 + k * 16, *reinterpret_cast<const uint32_t(*)[8]>(&o[8 * k]));
          }
        } else {
          // per block of 128 features: the block's max |y| (first pass), then y again, its FP8
          // round trip with scale = max / 448 (1 for an all-zero block) into shared memory
#pragma unroll 1
          for (int blk = cg * 2; blk < cg * 2 + 2; ++blk) {
            float amax = 0.f;
#pragma unroll 1
            for (int hf = 0; hf < 2; ++hf) {
              uint32_t o[32];
              norm_chunk(blk * 2 + hf, o);
#pragma unroll
              for (int e = 0; e < 32; ++e)
                amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(o[e] << 16)), fabsf(__uint_as_float(o[e] & 0xFFFF0000u))));
            }
            const float scale = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
#pragma unroll 1
            for (int hf = 0; hf < 2; ++hf) {
              const int cc = blk * 2 + hf;
              uint32_t o[32];
              norm_chunk(cc, o);
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = fp8_round_trip_bf16x2(o[e], scale);
              store_a(cc, o);
              if (cache_row)
#pragma unroll
                for (int k = 0; k < 4; ++k) stg_v8(cache_row + cc * 64 + k * 16, *reinterpret_cast<const uint32_t(*)[8]>(&o[8 * k]));
            }
          }
        }
        // the tensor core (async proxy) reads what these generic-proxy stores wrote
        fence_proxy_async_smem();
        mbar_arrive(&a_ready);
        cur_m = mp;
        ++seg;
      }

      // accumulator -> registers in two halves of 128 columns (k_nope, then v); the
      // accumulator is free for the unit after next once the second half is in registers
      const bool got = __all_sync(0xffffffffu, mbar_wait(&acc_full[acc], acc_phase, abort_p));
      ok = epi_sync_and(got);
      if (!ok) break;
      tc_fence_after();
      const int t_row = t0 + r;
      const bool row_ok = tile_ok && t_row < p.T;
      const int64_t prow = (static_cast<int64_t>(b) * p.H + h) * p.T + t_row;
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        uint32_t v[64];
#pragma unroll
        for (int c = 0; c < 2; ++c)
          tmem_ld_32x32b_x32(lane_addr + TM_ACC + static_cast<uint32_t>(acc * BN + half * 128 + cg * 64 + c * 32),
                             *reinterpret_cast<uint32_t(*)[32]>(&v[c * 32]));
        tmem_ld_wait();
        if (half == 1) {
          tc_fence_before();
          mbar_arrive(&acc_empty[acc]);
        }
        if (row_ok) {
          // range of the values carried exactly: the e4m3 residual of k_nope saturates from 512
          // on, v is stored in fp16 (NaN counts as out of range)
          float am[4] = {0.f, 0.f, 0.f, 0.f};   // four independent chains
#pragma unroll
          for (int i = 0; i < 64; ++i) am[i & 3] = max_nan(am[i & 3], fabsf(__uint_as_float(v[i])));
          const float amax = max_nan(max_nan(am[0], am[1]), max_nan(am[2], am[3]));
          if (!(half == 0 ? amax < MLA_MAX_ABS_K_NOPE : amax <= MLA_MAX_ABS_V)) set_error(kErrRange);
        }
        if (row_ok && in_bounds(b < p.B && h < p.H)) {
          uint32_t hw[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) hw[i] = pack_f16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
          uint16_t* dst = p.kv_out + prow * 256 + half * 128 + cg * 64;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t o8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) o8[e] = hw[8 * c + e];
            stg_v8(dst + 16 * c, o8);
          }
          if (half == 0) {
            uint8_t* dlo = p.klo_out + prow * 128 + cg * 64;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              uint32_t lw[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                float rr[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const int k = c * 32 + i * 4 + e;
                  const uint16_t hb = static_cast<uint16_t>((hw[k >> 1] >> ((k & 1) * 16)) & 0xFFFFu);
                  // (k - k_hi) * 2^11 exactly: both products are exact and so is their difference
                  rr[e] = __fmaf_rn(__uint_as_float(v[k]), KLO_SCALE, -KLO_SCALE * f16_bits_to_float(hb));
                }
                lw[i] = static_cast<uint32_t>(pack_e4m3x2(rr[0], rr[1])) | (static_cast<uint32_t>(pack_e4m3x2(rr[2], rr[3])) << 16);
              }
              stg_v8(dlo + 32 * c, lw);
            }
          }
        }
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && (ctl.abort_flag || (*(volatile unsigned int*)&g_status & (1u << kErrTimeout)))) {
    // unwinding: the peer's W copies complete on the leader's barriers, which the peer cannot
    // wait on; give copies still in flight 200 us to land before either CTA's shared memory goes
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 200000ull) {
    }
  }
  __syncthreads();
  // the leader's MMAs (which write both CTAs' TMEM) have drained and both CTAs' epilogues have
  // read their accumulators before the pair frees its tensor memory
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, TMEM_COLS);
  }
}

}  // namespace k1
}  // namespace mla
