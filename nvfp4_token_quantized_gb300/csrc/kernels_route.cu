// kernels_route.cu - router logits, top-k selection and the expert
// permutation (expandInputRows) of the routed-MoE forward.
//
// Router arithmetic follows the canonical FP32 order the library documents
// (8-element chunks; partial p accumulates chunks p, p+32, ... with fused
// multiply-adds in ascending order; a pairwise tree over the 32 partials),
// so expert choices are reproducible bit for bit on any implementation of the
// same order.  The permutation groups rows by expert and keeps token order
// inside an expert, and pads each expert to whole 128-row tiles for the
// tensor-core GEMMs.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int ROUTER_WARPS = 8;

// Swizzle of the 16-byte units of one (k, partial) row of the staged router
// weight so that the 8 lanes of one shared-memory wavefront hit distinct banks.
template <int UNITS>
__device__ __forceinline__ int router_swz(int p) {
  if constexpr (UNITS == 4) return (p >> 1) & 3;
  else if constexpr (UNITS == 2) return (p >> 2) & 1;
  else return 0;
}

// grid: (ceil(T / (8*TB)), E / EB); block: 256 threads = 8 warps.
// Warp w handles tokens t0..t0+TB-1; lane p is partial p of every
// (token, expert) pair of the CTA's expert block.
template <int TB, int EB>
__global__ void __launch_bounds__(256) router_logits_kernel(const __nv_bfloat16* __restrict__ x,
                                                           const __nv_bfloat16* __restrict__ wg,
                                                           const float* __restrict__ bias,
                                                           float* __restrict__ logits, int T, int H, int E) {
  constexpr int UNITS = EB / 8;                 // 16-byte units (8 bf16) per staged row
  constexpr int NV = TB * EB;                   // partial sums per lane
  static_assert(NV % 32 == 0, "TB*EB must be a multiple of 32");
  __shared__ __align__(16) uint4 sw[2][8][32][UNITS];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e0 = blockIdx.y * EB;
  const int t0 = (blockIdx.x * ROUTER_WARPS + warp) * TB;
  const int rounds = H / 256;

  auto stage = [&](int j, int buf) {
    // thread i stages weight row h = 256 j + i: EB bf16 from wg[h][e0..]
    const int hr = threadIdx.x;
    const int h = j * 256 + hr;
    const int k = hr & 7, p = (hr >> 3) & 31;
    const char* src = reinterpret_cast<const char*>(wg + (size_t)h * E + e0);
#pragma unroll
    for (int u = 0; u < UNITS; ++u) {
      const uint32_t dst = smem_u32(&sw[buf][k][p][u ^ router_swz<UNITS>(p)]);
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src + 16 * u) : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };

  float acc[TB][EB];
#pragma unroll
  for (int t = 0; t < TB; ++t)
#pragma unroll
    for (int e = 0; e < EB; ++e) acc[t][e] = 0.0f;

  stage(0, 0);
  for (int j = 0; j < rounds; ++j) {
    const int buf = j & 1;
    if (j + 1 < rounds) {
      stage(j + 1, buf ^ 1);
      asm volatile("cp.async.wait_group 1;" ::: "memory");
    } else {
      asm volatile("cp.async.wait_group 0;" ::: "memory");
    }
    __syncthreads();
    const int c = j * 32 + lane;                // this lane's chunk
    uint4 xv[TB];
#pragma unroll
    for (int t = 0; t < TB; ++t) {
      const int tok = t0 + t;
      xv[t] = tok < T ? __ldg(reinterpret_cast<const uint4*>(x + (size_t)tok * H + 8 * c))
                      : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      float xf[TB];
#pragma unroll
      for (int t = 0; t < TB; ++t) {
        const uint32_t w32 = (k < 2) ? xv[t].x : (k < 4) ? xv[t].y : (k < 6) ? xv[t].z : xv[t].w;
        xf[t] = (k & 1) ? bf16_hi(w32) : bf16_lo(w32);
      }
#pragma unroll
      for (int u = 0; u < UNITS; ++u) {
        const uint4 wv = sw[buf][k][lane][u ^ router_swz<UNITS>(lane)];
        const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float w = (q & 1) ? bf16_hi(ww[q >> 1]) : bf16_lo(ww[q >> 1]);
#pragma unroll
          for (int t = 0; t < TB; ++t) acc[t][u * 8 + q] = __fmaf_rn(xf[t], w, acc[t][u * 8 + q]);
        }
      }
    }
    __syncthreads();
  }

  // Pairwise tree over the 32 partials (lanes), partial p with p^o for
  // o = 16..1.  Each level halves the values a lane keeps, so lane p ends
  // with the sums of values [p*M, p*M + M), M = NV / 32.
  float v[NV];
#pragma unroll
  for (int t = 0; t < TB; ++t)
#pragma unroll
    for (int e = 0; e < EB; ++e) v[t * EB + e] = acc[t][e];
#pragma unroll
  for (int lvl = 0; lvl < 5; ++lvl) {
    const int o = 16 >> lvl;
    const int half = NV >> (lvl + 1);
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = upper ? v[i] : v[half + i];
      const float keep = upper ? v[half + i] : v[i];
      const float recv = __shfl_xor_sync(0xffffffffu, send, o);
      v[i] = __fadd_rn(keep, recv);
    }
  }
  constexpr int M = NV / 32;
#pragma unroll
  for (int i = 0; i < M; ++i) {
    const int idx = lane * M + i;
    const int t = idx / EB, e = idx % EB;
    const int tok = t0 + t;
    if (tok < T) {
      float l = v[i];
      if (bias) l = __fadd_rn(l, bias[e0 + e]);
      logits[(size_t)tok * E + e0 + e] = l;
    }
  }
}

// One warp per token: top-k by (logit desc, expert asc), softmax weights of
// the chosen experts renormalised, and the per-expert row counts.
__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ logits, int T, int E, int K,
                                                  int32_t* __restrict__ topk_ids, float* __restrict__ topk_w,
                                                  int32_t* __restrict__ counts) {
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  constexpr int MAXE = 8;  // up to 256 experts
  float l[MAXE], cand[MAXE];
#pragma unroll
  for (int i = 0; i < MAXE; ++i) {
    const int e = lane + 32 * i;
    l[i] = e < E ? logits[(size_t)t * E + e] : -INFINITY;
    cand[i] = l[i];
  }
  float sel_l[16];
  int sel_e[16];
  for (int j = 0; j < K; ++j) {
    float bv = -INFINITY;
    int be = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < MAXE; ++i) {
      const int e = lane + 32 * i;
      if (e < E && (cand[i] > bv || (cand[i] == bv && e < be))) {
        bv = cand[i];
        be = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oe = __shfl_xor_sync(0xffffffffu, be, o);
      if (ov > bv || (ov == bv && oe < be)) {
        bv = ov;
        be = oe;
      }
    }
    sel_l[j] = bv;
    sel_e[j] = be;
#pragma unroll
    for (int i = 0; i < MAXE; ++i)
      if (lane + 32 * i == be) cand[i] = -INFINITY;
  }
  // softmax over all experts, then renormalise the chosen probabilities
  const float m = sel_l[0];
  float s = 0.0f;
#pragma unroll
  for (int i = 0; i < MAXE; ++i)
    if (lane + 32 * i < E) s += expf(l[i] - m);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  float p[16], psum = 0.0f;
  for (int j = 0; j < K; ++j) {
    p[j] = expf(sel_l[j] - m) / s;
    psum += p[j];
  }
  for (int j = 0; j < K; ++j) {
    if (lane == j) {
      topk_ids[(size_t)t * K + j] = sel_e[j];
      topk_w[(size_t)t * K + j] = p[j] / psum;
      atomicAdd(&counts[sel_e[j]], 1);
    }
  }
}

__device__ __forceinline__ int block_sum_int(int v, int* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  int tot = 0;
  for (int w = 0; w < nw; ++w) tot += red[w];
  return tot;
}

// Exclusive scan of v over the block; returns this thread's prefix, total in *tot.
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

constexpr int PERM_THREADS = 512;
constexpr int PERM_TPT = 8;  // tokens per thread per pass

// One CTA per expert: offsets from the counts, then a stable compaction of
// the (token, slot) pairs that chose this expert, in token order.
__global__ void __launch_bounds__(PERM_THREADS) permute_kernel(const int32_t* __restrict__ topk_ids,
                                                              const int32_t* __restrict__ counts, int T, int K,
                                                              int E, PermuteOut o) {
  __shared__ int red[PERM_THREADS / 32];
  const int e = blockIdx.x;
  int c_lt = 0, p_lt = 0, n_lt = 0;
  for (int i = threadIdx.x; i < e; i += blockDim.x) {
    const int c = counts[i];
    c_lt += c;
    p_lt += (c + 127) & ~127;
    n_lt += (c + 127) >> 7;
  }
  const int off = block_sum_int(c_lt, red);
  const int poff = block_sum_int(p_lt, red);
  const int tbase = block_sum_int(n_lt, red);
  const int cnt = counts[e];

  int carry = 0;
  for (int base = 0; base < T; base += PERM_THREADS * PERM_TPT) {
    const int tb = base + threadIdx.x * PERM_TPT;
    int slot[PERM_TPT];
    int n = 0;
#pragma unroll
    for (int i = 0; i < PERM_TPT; ++i) {
      slot[i] = -1;
      const int t = tb + i;
      if (t < T) {
        for (int j = 0; j < K; ++j)
          if (topk_ids[(size_t)t * K + j] == e) slot[i] = j;
      }
      n += slot[i] >= 0;
    }
    int tot;
    int pos = carry + block_excl_scan(n, red, &tot);
#pragma unroll
    for (int i = 0; i < PERM_TPT; ++i) {
      if (slot[i] >= 0) {
        const int src = (tb + i) * K + slot[i];
        const int r = off + pos;
        const int pr = poff + pos;
        o.src_of_row[r] = src;
        o.row_of_src[src] = r;
        o.pad_row_of_src[src] = pr;
        o.src_of_padrow[pr] = src;
        ++pos;
      }
    }
    carry += tot;
  }
  const int ntile = (cnt + 127) >> 7;
  for (int i = threadIdx.x; i < ntile; i += blockDim.x)
    o.tiles[tbase + i] = make_int4(e, poff + 128 * i, min(128, cnt - 128 * i), 0);
  if (threadIdx.x == 0) {
    o.expert_offsets[e] = off;
    if (e == E - 1) {
      o.expert_offsets[E] = off + cnt;
      o.num_tiles[0] = tbase + ntile;
    }
  }
}

template <int TB, int EB>
cudaError_t launch_router_t(const void* x, const void* gate_w, const float* bias, float* logits, int T, int H,
                            int E, cudaStream_t s) {
  dim3 grid((T + ROUTER_WARPS * TB - 1) / (ROUTER_WARPS * TB), E / EB);
  router_logits_kernel<TB, EB><<<grid, 256, 0, s>>>(reinterpret_cast<const __nv_bfloat16*>(x),
                                                    reinterpret_cast<const __nv_bfloat16*>(gate_w), bias, logits,
                                                    T, H, E);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_router_logits(const void* x, const void* gate_w, const float* bias, float* logits, int T,
                                 int H, int E, cudaStream_t s) {
  if (E % 32 == 0) return launch_router_t<4, 32>(x, gate_w, bias, logits, T, H, E, s);
  if (E % 16 == 0) return launch_router_t<4, 16>(x, gate_w, bias, logits, T, H, E, s);
  return launch_router_t<4, 8>(x, gate_w, bias, logits, T, H, E, s);
}

cudaError_t launch_topk(const float* logits, int T, int E, int K, int32_t* topk_ids, float* topk_w,
                        int32_t* counts, cudaStream_t s) {
  topk_kernel<<<(T + 7) / 8, 256, 0, s>>>(logits, T, E, K, topk_ids, topk_w, counts);
  return cudaGetLastError();
}

cudaError_t launch_permute(const int32_t* topk_ids, const int32_t* counts, int T, int K, int E,
                           const PermuteOut& o, cudaStream_t s) {
  permute_kernel<<<E, PERM_THREADS, 0, s>>>(topk_ids, counts, T, K, E, o);
  return cudaGetLastError();
}

}  // namespace moe
