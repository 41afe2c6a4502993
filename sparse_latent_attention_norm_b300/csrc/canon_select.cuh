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
// One CTA per query row; the row's bitset is assembled in shared memory with atomicOr.
#pragma once

#include "ptx.cuh"

namespace mla {

constexpr int kCanonThreads = 256;
constexpr unsigned kErrIndex = 4;

// `sched` (nullable): the attention stage's tile counter, set to zero here so that the attention
// launch that follows on the same stream starts handing out tiles from the first.
__global__ void __launch_bounds__(kCanonThreads) canon_select_kernel(const int32_t* __restrict__ topk_idx, int T,
                                                                     int K, int W, uint32_t* __restrict__ sel_bits,
                                                                     int32_t* __restrict__ n_keys, int validate,
                                                                     uint32_t* __restrict__ sched) {
  extern __shared__ uint32_t bits[];
  if (sched != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *sched = 0u;
  __shared__ int warp_counts[kCanonThreads / 32];
  const int64_t row = blockIdx.x;
  const int t = static_cast<int>(row % T);
  const int words = (t / 128 + 1) * 4;  // <= W
  if (!in_bounds(words <= W)) return;
  for (int w = threadIdx.x; w < words; w += kCanonThreads) bits[w] = 0u;
  __syncthreads();

  const int32_t* idx = topk_idx + row * K;
  bool bad = false;
  if ((K & 3) == 0) {
    const int4* idx4 = reinterpret_cast<const int4*>(idx);
    for (int i = threadIdx.x; i < (K >> 2); i += kCanonThreads) {
      const int4 v = __ldg(idx4 + i);
      const int js[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = js[e];
        bad |= (j < 0) | (j >= T);
        if (j >= 0 && j <= t && in_bounds((j >> 5) < words)) atomicOr(&bits[j >> 5], 1u << (j & 31));
      }
    }
  } else {
    for (int i = threadIdx.x; i < K; i += kCanonThreads) {
      const int j = __ldg(idx + i);
      bad |= (j < 0) | (j >= T);
      if (j >= 0 && j <= t && in_bounds((j >> 5) < words)) atomicOr(&bits[j >> 5], 1u << (j & 31));
    }
  }
  if (validate && bad) set_error(kErrIndex);
  __syncthreads();

  int count = 0;
  uint32_t* dst = sel_bits + row * static_cast<int64_t>(W);
  for (int w = threadIdx.x; w < words; w += kCanonThreads) {
    const uint32_t v = bits[w];
    dst[w] = v;
    count += __popc(v);
  }
  if (n_keys != nullptr) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) count += __shfl_xor_sync(0xffffffffu, count, o);
    if (lane_id() == 0) warp_counts[warp_id()] = count;
    __syncthreads();
    if (threadIdx.x == 0) {
      int total = 0;
#pragma unroll
      for (int w = 0; w < kCanonThreads / 32; ++w) total += warp_counts[w];
      n_keys[row] = total;
    }
  }
}

}  // namespace mla
