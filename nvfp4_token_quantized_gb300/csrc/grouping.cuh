// grouping.cuh - the expert grouping of a small batch (at most 64 tokens):
// per-expert offsets, the stable token-order permutation of the (token, slot)
// rows, the padded-row map and the GEMM tile list, from the top-k ids.  Run
// by one CTA of 256 threads, either at the end of the small-batch front
// kernel or by an extra CTA of the requantization kernel.
//
// The permutation is the expandInputRows step of "SM10X Command-A-Plus decode
// 2.3x faster, BCG capture memory -78%" (Motivation): rows grouped by expert,
// tokens in ascending order inside an expert.
#pragma once

#include "common.cuh"

namespace moe {

struct SmallGroupOut {
  int32_t* expert_offsets;  // [E+1]
  int32_t* src_of_row;      // [T*K]
  int32_t* row_of_src;      // [T*K]
  int32_t* pad_row_of_src;  // [T*K]: expert * 128 + token
  int4* tiles;              // one tile per expert with rows: {expert, expert*128, T, 0}
  int32_t* num_tiles;
};

// Exclusive scan of v over the CTA; returns this thread's prefix, total in *tot.
__device__ __forceinline__ int block_excl_scan(int v, int* red, int* tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  __syncthreads();
  if (lane == 31) red[warp] = incl;
  __syncthreads();
  int base = 0, all = 0;
  for (int w = 0; w < nw; ++w) {
    const int r = red[w];
    if (w < warp) base += r;
    all += r;
  }
  *tot = all;
  return base + incl - v;
}

// T <= 64: the tokens that chose expert e form one 64-bit mask, so counts and
// the stable (token-order) rank of every row are population counts.  All 256
// threads of the CTA must call it; tok_mask [256] and offs [256] are shared
// memory, red [8] shared scratch.  topk_ids is read through L2 (other CTAs or
// kernels wrote it).
__device__ __forceinline__ void small_grouping(const int32_t* __restrict__ topk_ids, int T, int K, int E,
                                               const SmallGroupOut& o, unsigned long long* tok_mask, int* offs,
                                               int* red) {
  const int n = T * K;
  const int e = threadIdx.x;  // E <= 256 = blockDim.x
  if (e < E) tok_mask[e] = 0ull;
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += blockDim.x) atomicOr(&tok_mask[__ldcg(topk_ids + i)], 1ull << (i / K));
  __syncthreads();
  const int cnt = e < E ? __popcll(tok_mask[e]) : 0;
  int total, touched;
  const int off = block_excl_scan(cnt, red, &total);
  const int tix = block_excl_scan(cnt > 0 ? 1 : 0, red, &touched);
  if (e < E) {
    offs[e] = off;
    o.expert_offsets[e] = off;
    if (e == E - 1) {
      o.expert_offsets[E] = off + cnt;
      o.num_tiles[0] = touched;
    }
    if (cnt > 0) o.tiles[tix] = make_int4(e, e * 128, T, 0);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int ei = __ldcg(topk_ids + i), t = i / K;
    const int r = offs[ei] + __popcll(tok_mask[ei] & ((1ull << t) - 1ull));
    o.src_of_row[r] = i;
    o.row_of_src[i] = r;
    o.pad_row_of_src[i] = ei * 128 + t;
  }
}

}  // namespace moe
