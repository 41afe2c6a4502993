// Stage 4: sparse causal MLA attention (prefill), tcgen05 + TMEM, flash-style online softmax.
//
// Per query t and head h ("Keys" / "Scale scores" pages, MHA prefill model.py 574-589):
//   k_j      = cat(k_nope[j, h], k_pe[j])                       (192 features)
//   s_j      = softmax_scale * <q[t, h], k_j>,  softmax_scale = 192^-0.5 * (1 + 0.1 ln 40)^2
//   out[t,h] = sum_{j in S(t)} exp(s_j - M) v[j, h] / sum_{j in S(t)} exp(s_j - M)
//   lse[t,h] = M + ln sum_{j in S(t)} exp(s_j - M)
// where S(t) is the canonical selection (top-k as a set, intersected with j <= t) produced by the
// selection stage as one bitset per query row. The [B, T, T] -inf mask is never built: each
// softmax thread reads its row's 128-bit slice of the bitset for the key block at hand.
//
// Work is cut into tiles of (batch, head, 128 queries); a tile's key blocks of 128 run from 0 to
// its diagonal block. Per block, the score tile S[128 x 128] (fp32, TMEM, double-buffered) is
//   q_nope . k_hi   8 UMMAs kind::f16, fp16: A = q_nope from TMEM, B = k_hi from shared memory
// + q_pe . k_pe     4 UMMAs kind::f16, bf16: both from shared memory (the inputs as given)
// + q8 . k_lo       4 UMMAs kind::f8f6f4: A = e5m2(q_nope * 2^-11), B = e4m3 residual * 2^11
// The third term restores the bits of k_nope that fp16 drops, so the scores carry k_nope to about
// 2^-14 relative (the up-projection stage writes k_hi and k_lo). Then:
//   softmax: four threads per query row (TMEM lane), 32 key columns each: apply the row's
//           selection bits, block max of the raw scores (combined across the four threads with
//           shared atomicMax), running max in the log2 domain with lazy rescaling (only when the
//           max grows by more than 8 log2 units; in between, a block above the running max is
//           shifted so that its largest key's exponent is exactly 0), p = 2^(s * scale * log2 e
//           - m) evaluated in fp16
//           (ex2.approx.f16x2) and written to TMEM (64 cols of fp16 pairs).
//   PV    : O[128 x 128] += P[128 x 128] . V[128 x 128], 8 UMMAs kind::f16 with P (fp16) read
//           from TMEM and V (fp16) from shared memory (MN-major), O in TMEM (128 cols).
// QK^T and PV are issued by two threads, each waiting only on its own barriers, so the scores of
// blocks i+1 and i+2 are computed while the softmax of block i runs and PV(i) is queued as soon
// as its probabilities are in TMEM.
//
// The kernel is persistent: one CTA per SM takes tiles from a global counter (head by head,
// longest tile of a head first) until none are left. All roles walk the CTA's tile sequence with
// continuous barrier phases, so the next tile's q_pe / K / V loads and its first QK^T blocks run
// while the current tile finishes; the next tile's queries are prepared before the current
// tile's epilogue, and its PV waits only for the epilogue to have read O.
//
// Warp roles (640 threads): warp 0 tile scheduler + TMA producer of q_pe and K blocks, warp 19
// TMA producer of V blocks, warp 1 TMEM owner + QK^T MMA issuer, warp 18 PV MMA issuer, warps
// 2-17 query preparation, softmax and epilogue (warp w owns TMEM lanes 32*(w%4) .. +31, i.e. 32
// rows, and key / value columns 32*((w-2)/4) .. +31).
#pragma once

#include "mla.h"
#include "ptx.cuh"

namespace mla {
namespace k2 {

constexpr int BQ = 128;                 // queries per tile
constexpr int BK = 128;                 // keys per block
constexpr int ATOM_BYTES = 128 * 128;   // 128 rows x 128 bytes, 128-byte swizzle
constexpr int QPE_BYTES = ATOM_BYTES;   // q[:, 128:192] bf16
constexpr int Q8_BYTES = ATOM_BYTES;    // e5m2(q[:, 0:128] * 2^-11)
constexpr int K_BYTES = 4 * ATOM_BYTES;   // k_hi 0-63, k_hi 64-127 (fp16), k_pe (bf16), k_lo (e4m3)
constexpr int V_BYTES = 2 * ATOM_BYTES;   // v 0-63, 64-127 (fp16)
constexpr int NK_STAGE = 2;
constexpr int NV_STAGE = 2;
constexpr int NPART = 4;                // softmax warps per TMEM lane quadrant (column parts)
constexpr int PCOLS = BK / NPART;       // key / value columns per softmax thread
constexpr int NSOFT = 128 * NPART;      // softmax / epilogue threads
constexpr int PV_WARP = 2 + NSOFT / 32; // warp 0 TMA (q_pe, K), warp 1 QK MMA, warps 2.. softmax, then PV MMA,
constexpr int VP_WARP = PV_WARP + 1;    // then TMA (V)
constexpr int THREADS = 32 * (VP_WARP + 1);
constexpr int NCONSUMER = 3 + NSOFT;    // threads that read each published tile index
constexpr int TILE_BYTES = QPE_BYTES + Q8_BYTES + NK_STAGE * K_BYTES + NV_STAGE * V_BYTES;

// Barriers and small shared state, placed after the tiles in the dynamic shared memory (the
// kernel declares no static shared memory, so the dynamic region starts 1024-byte aligned and
// needs no alignment slack: the tiles fill all but a few KB of the 227 KB a CTA may use).
struct Ctrl {
  int max_key[3][BQ];        // [block % 3][row]: block max of the row's selected raw scores, as an
                             // order-preserving integer key, reduced with shared atomicMax
  int4 item_pub[2];          // tiles published by the K producer: {index (-1: no more tiles), b, h, qt}
  uint64_t item_full[2], item_empty[2];
  uint64_t q_full, q_ready, q_free, o_free, drain, drain_pv;
  uint64_t k_full[NK_STAGE], k_empty[NK_STAGE];
  uint64_t v_full[NV_STAGE], v_empty[NV_STAGE];
  uint64_t s_full[2], s_free[2], p_full, pv_done[2];
  uint32_t tmem_base;
  int abort_flag;
};
constexpr int SMEM_BYTES = TILE_BYTES + static_cast<int>(sizeof(Ctrl));
static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_S = 0;            // S buffers at cols 0 and 128
constexpr uint32_t TM_O = 256;          // O at cols 256..383
constexpr uint32_t TM_QN = 384;         // q_nope as fp16 pairs, cols 384..447
constexpr uint32_t TM_P = 448;          // P as fp16 pairs, cols 448..511
// Online softmax in the log2 domain against a lagging reference max m. O and l are rescaled
// (a TMEM round trip of O) only when a block's max mb exceeds m by more than RESCALE_THRESHOLD
// log2 units. In between, a block whose max lies above m is shifted: with c = mb - m, each row
// exponentiates x - c = s * scale * log2 e - mb <= 0 in fp16, so the block's (and, once it is the
// row's, the row's) largest key gets p = 2^0 = 1 exactly. ex2.approx.f16x2 is not correctly
// rounded (up to one fp16 unit, ~1e-3 relative, measured over every fp16 input): a row that one
// key carries would take that error into lse if the key's exponent were anywhere but 0. The row
// sum adds the block's p in fp32 times 2^c in fp32 (lse keeps the exact weight of the largest
// key); P for the PV UMMA is p * fp16(2^c) in fp16 (two roundings of 2^-11, seen only in out).
constexpr float RESCALE_THRESHOLD = 8.0f;
constexpr float Q8_SCALE = 1.0f / 2048.0f; // 2^-11, undoes the 2^11 on k_lo

struct Params {
  int B, T, H;
  int nqt;                 // ceil(T / 128)
  int n_items;             // B * H * nqt tiles
  uint32_t* sched;         // tile counter, zero at launch; tiles are taken with atomicAdd
  int W;                   // bitset words per query row
  float scale_log2;        // softmax_scale * log2(e)
  const uint16_t* q;       // [B, T, H, 192] bf16
  const uint32_t* sel_bits;
  uint16_t* out;           // [B, T, H, 128] bf16
  float* lse;              // [B, T, H]
  const float2* rope_cs;   // null, or [T, 32] (cos, sin): q[..., 128:192] is unrotated and gets YaRN
                           // RoPE at position t here (pairs (2i, 2i+1), fp32, no fused multiply-add)
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 2^x for the two fp16 halves of `x` (low half first), fp16 results in the same places.
__device__ __forceinline__ uint32_t ex2_f16x2(uint32_t x) {
  uint32_t y;
  asm("ex2.approx.f16x2 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// a * b + c on two fp32 lanes at once (each lane an IEEE fma, as fmaf).
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

// x if bit `bit` (a one-bit constant) of `mask` is set, else -inf.
__device__ __forceinline__ float keep_if_bit(float x, uint32_t mask, uint32_t bit) {
  asm("{\n\t.reg .pred p;\n\t.reg .b32 t;\n\tand.b32 t, %1, %2;\n\tsetp.ne.u32 p, t, 0;\n\t"
      "selp.f32 %0, %0, 0fFF800000, p;\n\t}"
      : "+f"(x)
      : "r"(mask), "r"(bit));
  return x;
}

// Elementwise product of two fp16 pairs, rounded to nearest.
__device__ __forceinline__ uint32_t hmul2_bits(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// acc + lo(h) + hi(h): both fp16 halves of `h` added to an fp32 accumulator in fp32.
__device__ __forceinline__ float add_f16x2_to_f32(uint32_t h, float acc) {
  asm("{\n\t.reg .f16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\t"
      "add.rn.f32.f16 %0, lo, %0;\n\tadd.rn.f32.f16 %0, hi, %0;\n\t}"
      : "+f"(acc)
      : "r"(h));
  return acc;
}

__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Named barrier over the NPART softmax warps of a lane quadrant; returns the AND of `pred` over them.
__device__ __forceinline__ bool quad_sync_and(int id, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "n"(32 * NPART)
      : "memory");
  return r != 0;
}

// Order-preserving map from non-NaN floats to ints (a < b iff key(a) < key(b)) and its inverse.
__device__ __forceinline__ int float_order_key(float f) {
  const int i = __float_as_int(f);
  return i >= 0 ? i : (i ^ 0x7FFFFFFF);
}
__device__ __forceinline__ float float_from_order_key(int k) {
  return __int_as_float(k >= 0 ? k : (k ^ 0x7FFFFFFF));
}

// Tile index -> (batch, head, query tile). Tiles run head by head (so the CTAs at work at any
// time share a few heads' keys and values in L2) and, within a head, from the longest query tile
// (the most key blocks) down, so the dynamic hand-out ends with short tiles.
struct Tile {
  int b, h, qt, t0, nblk;
};
__device__ __forceinline__ Tile tile_of(int item, const Params& p) {
  Tile x;
  const int bh = item / p.nqt;
  x.qt = p.nqt - 1 - (item % p.nqt);
  x.b = bh / p.H;
  x.h = bh % p.H;
  x.t0 = x.qt * BQ;
  x.nblk = x.qt + 1;
  return x;
}


__global__ void __launch_bounds__(THREADS, 1)
    sparse_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kv,
                       const __grid_constant__ CUtensorMap tm_kpe, const __grid_constant__ CUtensorMap tm_klo,
                       const Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // The 128-byte swizzle of the tiles needs 1024-byte alignment; the region is only that aligned
  // when the kernel has no static shared memory, which is checked here once.
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) set_error(kErrUnsupportedLayout);
    return;
  }
  uint8_t* smem = smem_raw;
  uint8_t* sQpe = smem;
  uint8_t* sQ8 = sQpe + QPE_BYTES;
  uint8_t* sK = sQ8 + Q8_BYTES;
  uint8_t* sV = sK + NK_STAGE * K_BYTES;

  Ctrl& ctl = *reinterpret_cast<Ctrl*>(smem + TILE_BYTES);
  uint64_t* item_full = ctl.item_full;
  uint64_t* item_empty = ctl.item_empty;
  uint64_t& q_full = ctl.q_full;
  uint64_t& q_ready = ctl.q_ready;
  uint64_t& q_free = ctl.q_free;
  uint64_t& o_free = ctl.o_free;
  uint64_t& drain = ctl.drain;
  uint64_t& drain_pv = ctl.drain_pv;
  uint64_t* k_full = ctl.k_full;
  uint64_t* k_empty = ctl.k_empty;
  uint64_t* v_full = ctl.v_full;
  uint64_t* v_empty = ctl.v_empty;
  uint64_t* s_full = ctl.s_full;
  uint64_t* s_free = ctl.s_free;
  uint64_t& p_full = ctl.p_full;
  uint64_t* pv_done = ctl.pv_done;
  uint32_t& tmem_base = ctl.tmem_base;
  int& abort_flag = ctl.abort_flag;
  auto& max_key = ctl.max_key;
  volatile int* abort_p = &abort_flag;

  const int warp = warp_id();
  const int lane = lane_id();

  for (int i = threadIdx.x; i < 3 * BQ; i += THREADS) (&max_key[0][0])[i] = INT_MIN;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < 2; ++s) {
      mbar_init(&item_full[s], 1);
      mbar_init(&item_empty[s], NCONSUMER);
    }
    mbar_init(&q_full, 1);
    mbar_init(&q_ready, NSOFT);
    mbar_init(&q_free, 1);
    mbar_init(&o_free, NSOFT);
    mbar_init(&drain, 1);
    mbar_init(&drain_pv, 1);
    for (int s = 0; s < NK_STAGE; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < NV_STAGE; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&s_free[s], NSOFT);
      mbar_init(&pv_done[s], 1);
    }
    mbar_init(&p_full, NSOFT);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_kv);
    tma_prefetch_desc(&tm_kpe);
    tma_prefetch_desc(&tm_klo);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;

  // Every role walks the same tile sequence: tile number `it` of this CTA is published in slot
  // it & 1 of item_pub by the K producer, with its (batch, head, query tile) worked out once.
  // take_item returns the tile index (or -1 past the end) and the tile, and releases the slot;
  // false if the wait gave up.
  auto take_item = [&](int it, int& item, Tile& tl) -> bool {
    const int slot = it & 1;
    if (!mbar_wait(&item_full[slot], (it >> 1) & 1, abort_p)) return false;
    const int4 v = ctl.item_pub[slot];
    mbar_arrive(&item_empty[slot]);
    item = v.x;
    tl.b = v.y;
    tl.h = v.z;
    tl.qt = v.w;
    tl.t0 = v.w * BQ;
    tl.nblk = v.w + 1;
    return true;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ scheduler + TMA producer: q_pe, K
    // Takes the CTA's tiles from the global counter one tile ahead (the atomic's latency overlaps
    // the current tile's loads) and publishes them to the other roles.
    if (lane == 0) {
      bool ok = true;
      bool kpend[NK_STAGE] = {};
      uint32_t kpar[NK_STAGE] = {};
      bool qpend = false;
      uint32_t qpar = 0;
      int ks = 0;
      uint32_t kph = 0;
      int next = static_cast<int>(atomicAdd(p.sched, 1u));
      for (int it = 0; ok; ++it) {
        const int item = next < p.n_items ? next : -1;
        const int slot = it & 1;
        if (it >= 2 && !mbar_wait(&item_empty[slot], ((it - 2) >> 1) & 1, abort_p)) { ok = false; break; }
        Tile tl{};
        if (item >= 0) tl = tile_of(item, p);
        ctl.item_pub[slot] = make_int4(item, tl.b, tl.h, tl.qt);
        mbar_arrive(&item_full[slot]);
        if (item < 0) break;
        next = static_cast<int>(atomicAdd(p.sched, 1u));
        const int kv_plane = tl.b * p.H + tl.h;
        // q_pe of this tile replaces the previous tile's once its last QK^T has completed
        if (it >= 1 && !mbar_wait(&q_free, (it - 1) & 1, abort_p)) { ok = false; break; }
        qpend = false;
        if (p.rope_cs != nullptr) {
          // the query warps rotate q_pe into sQpe themselves (prepare_queries)
          mbar_arrive(&q_full);
        } else {
          mbar_arrive_expect_tx(&q_full, QPE_BYTES);
          if (in_bounds(tl.h < p.H && tl.t0 < p.T && tl.b < p.B))
            tma_load_4d(sQpe, &tm_q, &q_full, 128, tl.h, tl.t0, tl.b);
          else
            mbar_complete_tx(&q_full, QPE_BYTES);
        }
        qpend = true;
        qpar = it & 1;
        for (int i = 0; i < tl.nblk; ++i) {
          if (!mbar_wait(&k_empty[ks], kph ^ 1, abort_p)) { ok = false; break; }
          uint8_t* kdst = sK + ks * K_BYTES;
          const int j0 = i * BK;
          mbar_arrive_expect_tx(&k_full[ks], K_BYTES);
          if (in_bounds(j0 < p.T && kv_plane < p.B * p.H)) {
            tma_load_3d(kdst, &tm_kv, &k_full[ks], 0, j0, kv_plane);
            tma_load_3d(kdst + ATOM_BYTES, &tm_kv, &k_full[ks], 64, j0, kv_plane);
            tma_load_3d(kdst + 2 * ATOM_BYTES, &tm_kpe, &k_full[ks], 0, j0, tl.b);
            tma_load_3d(kdst + 3 * ATOM_BYTES, &tm_klo, &k_full[ks], 0, j0, kv_plane);
          } else {
            mbar_complete_tx(&k_full[ks], K_BYTES);
          }
          kpend[ks] = true;
          kpar[ks] = kph;
          if (++ks == NK_STAGE) { ks = 0; kph ^= 1; }
          if (i == tl.nblk - 1 && next < p.n_items) {
            // the next tile's q_nope rows, read with plain loads by the softmax warps when this
            // tile ends (about two blocks from now), go to L2: two 64-feature boxes of 128 rows.
            // Earlier, the key/value stream would evict them before use.
            const Tile nt = tile_of(next, p);
            tma_prefetch_l2_4d(&tm_q, 0, nt.h, nt.t0, nt.b);
            tma_prefetch_l2_4d(&tm_q, 64, nt.h, nt.t0, nt.b);
            if (p.rope_cs != nullptr) {
              // RoPE mode: the query warps also read the unrotated q_pe and the (cos, sin) rows
              tma_prefetch_l2_4d(&tm_q, 128, nt.h, nt.t0, nt.b);
              const int rows = min(BQ, p.T - nt.t0);
              asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.rope_cs + static_cast<int64_t>(nt.t0) * 32),
                           "r"(static_cast<uint32_t>(rows * 32 * 8))
                           : "memory");
            }
          }
        }
      }
      if (!ok) {
        // unwinding: let the copies already issued land before shared memory goes away
        if (qpend) mbar_wait(&q_full, qpar, nullptr);
        for (int s = 0; s < NK_STAGE; ++s)
          if (kpend[s]) mbar_wait(&k_full[s], kpar[s], nullptr);
      }
    }
  } else if (warp == VP_WARP) {
    // ------------------------------------------------------------ TMA producer: V
    // A thread of its own, so a K load never waits for a V stage to drain (and the reverse).
    if (lane == 0) {
      bool ok = true;
      bool vpend[NV_STAGE] = {};
      uint32_t vpar[NV_STAGE] = {};
      int vs = 0;
      uint32_t vph = 0;
      for (int it = 0; ok; ++it) {
        int item;
        Tile tl;
        if (!take_item(it, item, tl)) { ok = false; break; }
        if (item < 0) break;
        const int kv_plane = tl.b * p.H + tl.h;
        for (int i = 0; i < tl.nblk; ++i) {
          if (!mbar_wait(&v_empty[vs], vph ^ 1, abort_p)) { ok = false; break; }
          uint8_t* vdst = sV + vs * V_BYTES;
          const int j0 = i * BK;
          mbar_arrive_expect_tx(&v_full[vs], V_BYTES);
          if (in_bounds(j0 < p.T && kv_plane < p.B * p.H)) {
            tma_load_3d(vdst, &tm_kv, &v_full[vs], 128, j0, kv_plane);
            tma_load_3d(vdst + ATOM_BYTES, &tm_kv, &v_full[vs], 192, j0, kv_plane);
          } else {
            mbar_complete_tx(&v_full[vs], V_BYTES);
          }
          vpend[vs] = true;
          vpar[vs] = vph;
          if (++vs == NV_STAGE) { vs = 0; vph ^= 1; }
        }
      }
      if (!ok) {
        for (int s = 0; s < NV_STAGE; ++s)
          if (vpend[s]) mbar_wait(&v_full[s], vpar[s], nullptr);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ QK^T MMA issuer
    // Scores of global block g go to S buffer g & 1 once the softmax has read block g-2 out of it.
    if (lane == 0) {
      const uint32_t idesc_nope = idesc_f32acc(BQ, BK, kFmtF16, false, false);
      const uint32_t idesc_rope = idesc_f32acc(BQ, BK, kFmtBF16, false, false);
      const uint32_t idesc_lo = idesc_f8_f32acc(BQ, BK, kFmtE5M2, kFmtE4M3);
      // Descriptors of every operand tile, computed once: the start-address field is bits 0-13
      // (address >> 4) and no offset used below carries out of it (shared memory < 256 KB),
      // so the descriptor of (tile + offset) is the tile's descriptor + (offset >> 4).
      static_assert(NK_STAGE == 2 && NV_STAGE == 2, "stage descriptors below");
      const uint64_t d_k0 = sdesc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t d_k1 = sdesc_sw128(smem_u32(sK + K_BYTES), 16, 1024);
      const uint64_t d_qpe = sdesc_sw128(smem_u32(sQpe), 16, 1024);
      const uint64_t d_q8 = sdesc_sw128(smem_u32(sQ8), 16, 1024);
      bool issued = false;
      bool ok = true;
      int ks = 0;
      uint32_t kph = 0;
      int g = 0;   // global block counter of this CTA
      for (int it = 0; ok; ++it) {
        int item;
        Tile tl;
        if (!take_item(it, item, tl)) break;
        if (item < 0) break;
        if (!mbar_wait(&q_full, it & 1, abort_p) || !mbar_wait(&q_ready, it & 1, abort_p)) break;
        for (int i = 0; i < tl.nblk; ++i, ++g) {
          const int sb = g & 1;
          if (g >= 2 && !mbar_wait(&s_free[sb], ((g - 2) >> 1) & 1, abort_p)) { ok = false; break; }
          if (!mbar_wait(&k_full[ks], kph, abort_p)) { ok = false; break; }
          tc_fence_after();
          const uint32_t d = tmem + TM_S + static_cast<uint32_t>(sb * BK);
          const uint64_t dk = ks ? d_k1 : d_k0;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)   // q_nope (TMEM, fp16) . k_hi
            umma_ts(d, tmem + TM_QN + kk * 8, dk + (((kk >> 2) * ATOM_BYTES + (kk & 3) * 32) >> 4), idesc_nope,
                    kk > 0 ? 1u : 0u);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)   // q_pe . k_pe (bf16)
            umma_ss(d, d_qpe + kk * 2, dk + ((2 * ATOM_BYTES + kk * 32) >> 4), idesc_rope, 1u);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)   // e5m2(q_nope 2^-11) . e4m3(k_lo 2^11)
            umma_f8_ss(d, d_q8 + kk * 2, dk + ((3 * ATOM_BYTES + kk * 32) >> 4), idesc_lo, 1u);
          issued = true;
          umma_commit(&k_empty[ks]);
          umma_commit(&s_full[sb]);
          if (++ks == NK_STAGE) { ks = 0; kph ^= 1; }
        }
        // the tile's q_pe, q8 and q_nope are free once its last QK^T has completed
        if (ok) umma_commit(&q_free);
      }
      if (issued) {
        // every MMA this thread issued has finished before TMEM is released
        umma_commit(&drain);
        mbar_wait(&drain, 0, nullptr);
      }
    }
  } else if (warp == PV_WARP) {
    // ------------------------------------------------------------ PV MMA issuer
    // A second issuing thread, so that the tensor pipe is fed with the next block's QK^T while
    // this one waits for the softmax (and the reverse): one thread that waits on both sides
    // leaves the pipe idle for every wait.
    if (lane == 0) {
      const uint32_t idesc_pv = idesc_f32acc(BQ, 128, kFmtF16, false, true);
      const uint64_t d_v0 = sdesc_sw128(smem_u32(sV), ATOM_BYTES, 1024);
      const uint64_t d_v1 = sdesc_sw128(smem_u32(sV + V_BYTES), ATOM_BYTES, 1024);
      bool issued = false;
      bool ok = true;
      int vs = 0;
      uint32_t vph = 0;
      int g = 0;
      for (int it = 0; ok; ++it) {
        int item;
        Tile tl;
        if (!take_item(it, item, tl)) break;
        if (item < 0) break;
        // O is rewritten from the tile's first block on: the previous tile's epilogue must have read it
        if (it >= 1 && !mbar_wait(&o_free, (it - 1) & 1, abort_p)) break;
        for (int i = 0; i < tl.nblk; ++i, ++g) {
          // PV(g): P(g) from TMEM, V(g) from shared memory
          if (!mbar_wait(&p_full, g & 1, abort_p)) { ok = false; break; }
          if (!mbar_wait(&v_full[vs], vph, abort_p)) { ok = false; break; }
          tc_fence_after();
          const uint64_t dv = vs ? d_v1 : d_v0;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)   // 16 keys per UMMA: 16 rows of 128 bytes = 2048 bytes
            umma_ts(tmem + TM_O, tmem + TM_P + kk * 8, dv + ((kk * 2048) >> 4), idesc_pv, (i > 0 || kk > 0) ? 1u : 0u);
          issued = true;
          umma_commit(&v_empty[vs]);
          umma_commit(&pv_done[g & 1]);   // PV(g) is completion g >> 1 of pv_done[g & 1]
          if (++vs == NV_STAGE) { vs = 0; vph ^= 1; }
        }
      }
      if (issued) {
        umma_commit(&drain_pv);
        mbar_wait(&drain_pv, 0, nullptr);
      }
    }
  } else {
    // ------------------------------------------------------------ queries, softmax, epilogue
    // NPART warps per TMEM lane quadrant: warp w owns rows 32*(w%4) .. +31 and key / value
    // columns PCOLS*part .. +PCOLS-1 of every block, part = (w-2)/4. The quadrant's warps combine
    // their rows' block maxima with shared atomicMax on order-preserving integer keys and meet
    // once per block at a named barrier (id 1 + quadrant) that also ANDs their wait results, so
    // all of them take the same exit.
    // tcgen05.ld / tcgen05.st are warp-collective: every branch around them is warp-uniform.
    const int qw = warp & 3;
    const int part = (warp - 2) >> 2;
    const int r = qw * 32 + lane;           // query row in the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(qw * 32) << 16;
    const int quad_bar = 1 + qw;
    const float sl2 = p.scale_log2;

    // q_nope[32*part .. +31] of row r of tile `tl`: fp16 pairs into TMEM (exact for bf16 values
    // within fp16's range), and e5m2(q_nope * 2^-11) into the swizzled q8 tile (16-byte chunk c at
    // c ^ (r & 7)). Called once the previous tile's QK^T UMMAs have all completed.
    auto prepare_queries = [&](const Tile& tl) {
      const int t = tl.t0 + r;
      const bool row_valid = t < p.T;
      const uint4* qrow = reinterpret_cast<const uint4*>(
          p.q + ((static_cast<int64_t>(tl.b) * p.T + (row_valid ? t : 0)) * p.H + tl.h) * 192);
      uint32_t qn[16];
      uint32_t q8[8];
      uint32_t qw[2][8];   // this part's 32 q_nope features: two 32-byte loads
      float amax = 0.f;    // largest |q_nope| of the part (NaN propagates): fp16 must hold it
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        if (row_valid && in_bounds(tl.b < p.B && tl.h < p.H)) ldg_v8(qrow + part * 4 + 2 * c, qw[c]);
#pragma unroll
        for (int e = 0; e < 8; ++e)
          if (!row_valid) qw[c][e] = 0u;
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint32_t w[4] = {qw[c >> 1][(c & 1) * 4], qw[c >> 1][(c & 1) * 4 + 1], qw[c >> 1][(c & 1) * 4 + 2],
                               qw[c >> 1][(c & 1) * 4 + 3]};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float lo = __uint_as_float(w[e] << 16);
          const float hi = __uint_as_float(w[e] & 0xFFFF0000u);
          amax = max_nan(amax, max_nan(fabsf(lo), fabsf(hi)));
          qn[c * 4 + e] = pack_f16x2(lo, hi);
          const uint32_t b8 = pack_e5m2x2(lo * Q8_SCALE, hi * Q8_SCALE);
          if (e & 1)
            q8[c * 2 + (e >> 1)] |= b8 << 16;
          else
            q8[c * 2 + (e >> 1)] = b8;
        }
      }
      if (!(amax <= MLA_MAX_ABS_Q_NOPE)) set_error(kErrRange);
      tmem_st_32x32b_x16(tmem + lane_off + TM_QN + part * 16, qn);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int chunk = part * 2 + c;   // 16-byte chunk = 16 e5m2 values
        *reinterpret_cast<uint4*>(sQ8 + r * 128 + ((chunk ^ (r & 7)) * 16)) =
            make_uint4(q8[c * 4], q8[c * 4 + 1], q8[c * 4 + 2], q8[c * 4 + 3]);
      }
      if (p.rope_cs != nullptr) {
        // q_pe features 16*part .. +15 (pairs 8*part .. +7) rotated at position t into the
        // swizzled q_pe tile (16-byte chunk c of row r at c ^ (r & 7)), as the TMA copy would
        // have placed the rotated values
        uint32_t x[8], o[8];
        uint32_t csw[2][8];
        if (row_valid && in_bounds(tl.b < p.B && tl.h < p.H)) {
          ldg_v8(qrow + 16 + part * 2, x);
          const float2* crow = p.rope_cs + static_cast<int64_t>(t) * 32 + part * 8;
          ldg_v8(crow, csw[0]);
          ldg_v8(crow + 4, csw[1]);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float c = __uint_as_float(csw[e >> 2][(e & 3) * 2]), sn = __uint_as_float(csw[e >> 2][(e & 3) * 2 + 1]);
            const float a = __uint_as_float(x[e] << 16), bb = __uint_as_float(x[e] & 0xFFFF0000u);
            o[e] = pack_bf16x2(__fsub_rn(__fmul_rn(a, c), __fmul_rn(bb, sn)), __fadd_rn(__fmul_rn(a, sn), __fmul_rn(bb, c)));
          }
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) o[e] = 0u;
        }
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int chunk = part * 2 + c;
          *reinterpret_cast<uint4*>(sQpe + r * 128 + ((chunk ^ (r & 7)) * 16)) =
              make_uint4(o[c * 4], o[c * 4 + 1], o[c * 4 + 2], o[c * 4 + 3]);
        }
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&q_ready);
    };

    bool ok = true;
    int g = 0;        // global block counter of this CTA
    int slot3 = 0;    // g % 3: the max_key slot of block g
    int it = 0;
    int item = -1;
    Tile cur{};
    {
      const bool got = take_item(0, item, cur);
      ok = quad_sync_and(quad_bar, got);
    }
    uint32_t first_mask = 0u;   // selection word of the first block of the tile about to start
    if (ok && item >= 0) {
      const Tile& t0l = cur;
      const int tt = t0l.t0 + r;
      first_mask = (tt < p.T && in_bounds(t0l.b < p.B)) ? __ldg(p.sel_bits + (static_cast<int64_t>(t0l.b) * p.T + tt) * p.W + part) : 0u;
      prepare_queries(t0l);
    }
    while (ok && item >= 0) {
      const Tile tl = cur;
      const int t = tl.t0 + r;
      const bool row_valid = t < p.T;
      // this thread's selection word of block i: keys PCOLS*part .. +31 of the block
      const uint32_t* bits_row =
          p.sel_bits + (static_cast<int64_t>(tl.b) * p.T + (row_valid ? t : 0)) * p.W + part;
      float m_ref = -INFINITY;   // running reference max, log2 domain (identical in the quadrant's warps)
      float l = 0.f;             // running sum of this thread's columns' probabilities
      uint32_t mask_next = first_mask;
      for (int i = 0; i < tl.nblk; ++i, ++g) {
        const uint32_t mask = mask_next;
        if (i + 1 < tl.nblk)
          mask_next = (row_valid && in_bounds((i + 1) * 4 + part < p.W && tl.b < p.B)) ? __ldg(bits_row + (i + 1) * 4) : 0u;
        const int sb = g & 1;
        const int slot = slot3;
        bool got = __all_sync(0xffffffffu, mbar_wait(&s_full[sb], (g >> 1) & 1, abort_p));
        float s[PCOLS];
        if (got) {
          tc_fence_after();
          if (__any_sync(0xffffffffu, mask != 0u)) {
            tmem_ld_32x32b_x32(tmem + lane_off + TM_S + static_cast<uint32_t>(sb * BK + part * PCOLS),
                               *reinterpret_cast<uint32_t(*)[PCOLS]>(s));
            tmem_ld_wait();
            if (!__all_sync(0xffffffffu, mask == 0xFFFFFFFFu)) {   // some key of the part unselected
#pragma unroll
              for (int e = 0; e < PCOLS; ++e) s[e] = keep_if_bit(s[e], mask, 1u << e);
            }
          } else {
#pragma unroll
            for (int e = 0; e < PCOLS; ++e) s[e] = -INFINITY;
          }
          tc_fence_before();
          mbar_arrive(&s_free[sb]);
        } else {
#pragma unroll
          for (int e = 0; e < PCOLS; ++e) s[e] = -INFINITY;
        }
        // raw (unscaled) block max of the selected scores; the scale is positive, so scaling
        // the max gives the max of the scaled scores exactly
        float mx[4];   // four independent chains: mx[k] covers columns congruent to k mod 4
#pragma unroll
        for (int k = 0; k < 4; ++k) mx[k] = fmaxf(s[k], s[4 + k]);
#pragma unroll
        for (int e = 8; e < PCOLS; e += 8)
#pragma unroll
          for (int k = 0; k < 4; ++k) mx[k] = max3f(mx[k], s[e + k], s[e + 4 + k]);
        atomicMax(&max_key[slot][r], float_order_key(max3f(mx[0], mx[1], fmaxf(mx[2], mx[3]))));
        ok = quad_sync_and(quad_bar, ok && got);
        if (!ok) break;
        const float mb = float_from_order_key(max_key[slot][r]) * sl2;
        // the slot of block g-1 has been read by every warp of the quadrant (each read it before
        // arriving at this block's barrier); it is next written at block g+2, after the next barrier
        if (part == 0 && g > 0) max_key[slot3 == 0 ? 2 : slot3 - 1][r] = INT_MIN;
        slot3 = (slot3 == 2) ? 0 : slot3 + 1;
        const bool need = mb > m_ref + RESCALE_THRESHOLD;   // true on the first selected key
        const bool need_o = need && (m_ref != -INFINITY);   // O and l hold earlier blocks' mass
        const float alpha = need_o ? ex2(m_ref - mb) : 1.0f;
        if (need_o) l *= alpha;
        if (need) m_ref = mb;
        // shift of this row's exponents: 0 after a rescale, while no key is selected and when the
        // block's max lies below m; mb <= m_ref + RESCALE_THRESHOLD here, so 0 <= c <= 8
        const float c_shift = (mb == -INFINITY || m_ref == -INFINITY) ? 0.f : fmaxf(0.f, mb - m_ref);
        const float neg_m = (m_ref == -INFINITY) ? 0.f : -(m_ref + c_shift);   // no key yet: every p is 0
        // p = 2^x with x = s * scale * log2 e - m - c rounded to fp16 and exponentiated two at a
        // time in fp16 (P is consumed as fp16 by the PV UMMA); l sums the same fp16 values in
        // fp32 (times 2^c in fp32 when the block is shifted).
        uint32_t pk[PCOLS / 2];
        float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < PCOLS / 2; ++c) {
          const float2 xx = fma2(make_float2(s[2 * c], s[2 * c + 1]), make_float2(sl2, sl2), make_float2(neg_m, neg_m));
          pk[c] = ex2_f16x2(pack_f16x2(xx.x, xx.y));
        }
        if (__any_sync(0xffffffffu, c_shift > 0.f)) {
          // l += 2^c * sum p (fp32); P = p * 2^c in fp16 (p <= 1, so P <= 256)
          const float tc = ex2(c_shift);
          const uint32_t two_c = pack_f16x2(tc, tc);
#pragma unroll
          for (int c = 0; c < PCOLS / 2; ++c) ls[c & 3] = add_f16x2_to_f32(pk[c], ls[c & 3]);
          l += ((ls[0] + ls[1]) + (ls[2] + ls[3])) * tc;
#pragma unroll
          for (int c = 0; c < PCOLS / 2; ++c) pk[c] = hmul2_bits(pk[c], two_c);
        } else {
#pragma unroll
          for (int c = 0; c < PCOLS / 2; ++c) ls[c & 3] = add_f16x2_to_f32(pk[c], ls[c & 3]);
          l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
        }
        if (i > 0) {
          // P's TMEM columns and O are free once PV(g-1) has completed (for a tile's first block
          // the previous tile's epilogue waited for that). A failed wait here is carried into the
          // next quadrant barrier, so the quadrant's warps leave together; the writes below then
          // only touch this CTA's own TMEM.
          const bool pv_ok = __all_sync(0xffffffffu, mbar_wait(&pv_done[(g - 1) & 1], ((g - 1) >> 1) & 1, abort_p));
          ok = ok && pv_ok;
          tc_fence_after();
          if (pv_ok && __any_sync(0xffffffffu, need_o)) {
            uint32_t v[PCOLS];
            const uint32_t addr = tmem + lane_off + TM_O + static_cast<uint32_t>(part * PCOLS);
            tmem_ld_32x32b_x32(addr, v);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < PCOLS; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
            tmem_st_32x32b_x32(addr, v);
          }
        }
        tmem_st_32x32b_x16(tmem + lane_off + TM_P + part * (PCOLS / 2), pk);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&p_full);
      }
      if (!ok) break;

      // The next tile's queries go in now, so its first QK^T blocks overlap this tile's epilogue:
      // every QK^T of this tile has completed (its last scores were read above).
      int next_item = -1;
      Tile nt{};
      {
        const bool got = take_item(it + 1, next_item, nt);
        ok = quad_sync_and(quad_bar, got);
      }
      if (ok && next_item >= 0) {
        const int nt_t = nt.t0 + r;
        // the next tile's first selection word, loaded now so its latency passes during the
        // query preparation and this tile's epilogue
        first_mask = (nt_t < p.T && in_bounds(nt.b < p.B)) ? __ldg(p.sel_bits + (static_cast<int64_t>(nt.b) * p.T + nt_t) * p.W + part) : 0u;
        prepare_queries(nt);
      }

      // epilogue: out = O / l (bf16), lse = (m + log2 l) ln 2
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&pv_done[(g - 1) & 1], ((g - 1) >> 1) & 1, abort_p));
      // the row sum's four parts meet in TMEM: P's columns are idle until the next tile's first
      // block, which every part reaches only after the barrier below
      if (ok) {
        tc_fence_after();
        tmem_st_32x32b_x1(tmem + lane_off + TM_P + part, __float_as_uint(l));
        tmem_st_wait();
        tc_fence_before();
      }
      ok = quad_sync_and(quad_bar, ok);
      if (!ok) break;
      tc_fence_after();
      uint32_t lp[4];
      tmem_ld_32x32b_x4(tmem + lane_off + TM_P, lp);
      uint32_t v[PCOLS];
      tmem_ld_32x32b_x32(tmem + lane_off + TM_O + static_cast<uint32_t>(part * PCOLS), v);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&o_free);   // O is in registers: the next tile's PV may overwrite it
      const float lt = (__uint_as_float(lp[0]) + __uint_as_float(lp[1])) +
                       (__uint_as_float(lp[2]) + __uint_as_float(lp[3]));   // same order in every part
      const float inv_l = (lt > 0.f) ? 1.0f / lt : 0.f;
      if (row_valid && in_bounds(tl.b < p.B && tl.h < p.H)) {
        // this part's 32 output features = 64 bytes, as two 32-byte stores (each store instruction
        // of the warp touches one line per row, so fewer, wider stores take fewer L1 passes)
        uint16_t* orow = p.out + ((static_cast<int64_t>(tl.b) * p.T + t) * p.H + tl.h) * 128 + part * PCOLS;
#pragma unroll
        for (int k = 0; k < PCOLS / 16; ++k) {
          uint32_t o8[8];
#pragma unroll
          for (int e = 0; e < 8; ++e)
            o8[e] = pack_bf16x2(__uint_as_float(v[16 * k + 2 * e]) * inv_l, __uint_as_float(v[16 * k + 2 * e + 1]) * inv_l);
          stg_v8(orow + 16 * k, o8);
        }
        if (part == 0) {
          const float lse = (lt > 0.f) ? (m_ref + log2f(lt)) * 0.6931471805599453f : -INFINITY;
          p.lse[(static_cast<int64_t>(tl.b) * p.T + t) * p.H + tl.h] = lse;
        }
      }
      item = next_item;
      cur = nt;
      ++it;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace k2
}  // namespace mla
