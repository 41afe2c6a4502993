// Stage 1: canonical top-k selection.
//
// The MHA prefill excerpt (DeepSeek-V3.2-Exp model.py 574-589, "Keys" page) builds
// index_mask = full(-inf).scatter_(-1, topk_indices, 0) + mask: the scatter makes the selection a
// set (duplicates and order do not matter) and the causal mask removes keys after the query.
// This kernel produces that set directly as a bitset per query row, never the [B, T, T] float
// mask: bit j of row (b, t) is set iff j occurs in topk_idx[b, t, :] and 0 <= j <= t.
//
// Layout: sel_bits[(b*T + t) * W + w], W = ceil(T/128) * 4 words (128 keys per 4 words). Only the
// words the attention stage reads for query t are written: [0, (t/128 + 1) * 4).
// One warp per query row, several rows per CTA; each row's bitset is assembled in the warp's own
// slice of shared memory with atomicOr. A lane issues all its index loads of a batch (up to 8
// 16-byte loads, 4 KB per warp) before it touches the bitset, and every CTA of a typical launch is
// resident at once, so enough of the index array is in flight for the stage to run at the rate
// DRAM delivers it.
#pragma once

#include "ptx.cuh"

namespace mla {

constexpr int kCanonMaxRows = 8;     // query rows (warps) per CTA
constexpr int kCanonBatch = 8;       // index loads in flight per lane
constexpr unsigned kErrIndex = 4;

// Rows per CTA for bitsets of W words: as many as fit 48 KB of shared memory, at most 8.
inline int canon_rows_per_cta(int W) {
  const int fit = 49152 / (W * 4);
  return fit < 1 ? 1 : (fit > kCanonMaxRows ? kCanonMaxRows : fit);
}

__device__ __forceinline__ void canon_set(uint32_t* bits, int j, int t, int T, int words, bool& bad) {
  bad |= (j < 0) | (j >= T);
  if (j >= 0 && j <= t && in_bounds((j >> 5) < words)) atomicOr(&bits[j >> 5], 1u << (j & 31));
}

// `sched` (nullable): the attention stage's tile counter, set to zero here so that the attention
// launch that follows on the same stream starts handing out tiles from the first.
__global__ void __launch_bounds__(32 * kCanonMaxRows) canon_select_kernel(const int32_t* __restrict__ topk_idx,
                                                                          int64_t rows, int T, int K, int W,
                                                                          uint32_t* __restrict__ sel_bits,
                                                                          int32_t* __restrict__ n_keys, int validate,
                                                                          uint32_t* __restrict__ sched) {
  extern __shared__ uint32_t bits_all[];
  if (sched != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *sched = 0u;
  const int warp = static_cast<int>(threadIdx.x >> 5);
  const int lane = lane_id();
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + warp;
  if (row >= rows) return;   // the rest of the kernel is warp-level only
  uint32_t* bits = bits_all + static_cast<int64_t>(warp) * W;
  const int t = static_cast<int>(row % T);
  const int words = (t / 128 + 1) * 4;  // <= W
  if (!in_bounds(words <= W)) return;
  const int32_t* idx = topk_idx + row * K;
  bool bad = false;
  if ((K & 3) == 0) {
    const int4* idx4 = reinterpret_cast<const int4*>(idx);
    const int n4 = K >> 2;
    for (int base = 0; base < n4; base += 32 * kCanonBatch) {
      int4 v[kCanonBatch];
#pragma unroll
      for (int u = 0; u < kCanonBatch; ++u) {
        const int i = base + u * 32 + lane;
        if (i < n4) v[u] = __ldg(idx4 + i);
      }
      if (base == 0) {   // the first batch's loads are in flight while the bitset is cleared
        for (int w = lane; w < words; w += 32) bits[w] = 0u;
        __syncwarp();
      }
#pragma unroll
      for (int u = 0; u < kCanonBatch; ++u) {
        if (base + u * 32 + lane < n4) {
          canon_set(bits, v[u].x, t, T, words, bad);
          canon_set(bits, v[u].y, t, T, words, bad);
          canon_set(bits, v[u].z, t, T, words, bad);
          canon_set(bits, v[u].w, t, T, words, bad);
        }
      }
    }
  } else {
    for (int base = 0; base < K; base += 32 * kCanonBatch) {
      int v[kCanonBatch];
#pragma unroll
      for (int u = 0; u < kCanonBatch; ++u) {
        const int i = base + u * 32 + lane;
        if (i < K) v[u] = __ldg(idx + i);
      }
      if (base == 0) {
        for (int w = lane; w < words; w += 32) bits[w] = 0u;
        __syncwarp();
      }
#pragma unroll
      for (int u = 0; u < kCanonBatch; ++u)
        if (base + u * 32 + lane < K) canon_set(bits, v[u], t, T, words, bad);
    }
  }
  if (validate && bad) set_error(kErrIndex);
  __syncwarp();

  int count = 0;
  uint32_t* dst = sel_bits + row * static_cast<int64_t>(W);
  for (int w = lane; w < words; w += 32) {
    const uint32_t x = bits[w];
    dst[w] = x;
    count += __popc(x);
  }
  if (n_keys != nullptr) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) count += __shfl_xor_sync(0xffffffffu, count, o);
    if (lane == 0) n_keys[row] = count;
  }
}

}  // namespace mla
