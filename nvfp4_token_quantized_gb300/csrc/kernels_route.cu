// kernels_route.cu - router logits, top-k selection and the expert
// permutation (expandInputRows) of the routed-MoE forward.
//
// Router arithmetic follows the canonical FP32 order the library documents
// (8-element chunks; partial p accumulates chunks p, p+32, ... with fused
// multiply-adds in ascending order; a pairwise tree over the 32 partials),
// so expert choices are reproducible bit for bit on any implementation of the
// same order.  The permutation groups rows by expert and keeps token order
// inside an expert, and pads each GEMM tile of an expert to its own 128-row
// block for the tensor-core GEMMs.
#include <mutex>

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

// d = a * b + c on two FP32 lanes, each rounded once (the same result as two
// fmaf calls).
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(d)
      : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)),
        "l"(*reinterpret_cast<uint64_t*>(&c)));
  return *reinterpret_cast<float2*>(&d);
}

// grid: (ceil(T / (8*TB)), E / EB); block: 256 threads = 8 warps; dynamic
// shared memory H * EB * 2 bytes holding the CTA's whole router-weight slice,
// laid out [round j][k][partial p][EB] (row h = 256 j + 8 p + k).
// Warp w handles tokens t0..t0+TB-1; lane p is partial p of every
// (token, expert) pair of the CTA's expert block: it accumulates chunks
// c = p, p+32, ... in ascending order with one fused multiply-add per element,
// then the 32 partials are combined by the pairwise tree.
//
// XALL: every round's activations are loaded into registers up front (one
// memory round trip; H <= 2048), for small token counts where latency rules.
// The kernel also clears the per-expert row counters the top-k kernel fills.
template <int TB, int EB, bool XALL>
__global__ void __launch_bounds__(256) router_logits_kernel(const __nv_bfloat16* __restrict__ x,
                                                           const __nv_bfloat16* __restrict__ wg,
                                                           const float* __restrict__ bias,
                                                           float* __restrict__ logits, int T, int H, int E,
                                                           int32_t* __restrict__ counts) {
  constexpr int UNITS = EB / 8;                 // 16-byte units (8 bf16) per staged row
  constexpr int NV = TB * EB;                   // partial sums per lane
  static_assert(NV % 32 == 0, "TB*EB must be a multiple of 32");
  extern __shared__ uint4 sw[];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e0 = blockIdx.y * EB;
  const int t0 = (blockIdx.x * ROUTER_WARPS + warp) * TB;
  const int rounds = H / 256;
  pdl_trigger();
  if (blockIdx.x == 0 && blockIdx.y == 0)
    for (int e = threadIdx.x; e < E; e += blockDim.x) counts[e] = 0;

  for (int h = threadIdx.x; h < H; h += 256) {
    const int j = h >> 8, hr = h & 255, k = hr & 7, p = (hr >> 3) & 31;
    const char* src = reinterpret_cast<const char*>(wg + (size_t)h * E + e0);
#pragma unroll
    for (int u = 0; u < UNITS; ++u) {
      const uint32_t dst = smem_u32(&sw[((j * 8 + k) * 32 + p) * UNITS + (u ^ router_swz<UNITS>(p))]);
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src + 16 * u) : "memory");
    }
  }
  asm volatile("cp.async.commit_group;" ::: "memory");

  auto load_x = [&](int j, uint4 (&xv)[TB]) {
    const int c = j * 32 + lane;                // this lane's chunk in round j
#pragma unroll
    for (int t = 0; t < TB; ++t) {
      const int tok = t0 + t;
      xv[t] = tok < T ? __ldg(reinterpret_cast<const uint4*>(x + (size_t)tok * H + 8 * c)) : make_uint4(0, 0, 0, 0);
    }
  };
  constexpr int XR = XALL ? 8 : 2;              // rounds of activations held in registers
  uint4 xb[XR][TB];
  if constexpr (XALL) {
#pragma unroll
    for (int j = 0; j < XR; ++j)
      if (j < rounds) load_x(j, xb[j]);
  } else {
    load_x(0, xb[0]);
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  __syncthreads();

  float2 acc[TB][EB / 2];
#pragma unroll
  for (int t = 0; t < TB; ++t)
#pragma unroll
    for (int e = 0; e < EB / 2; ++e) acc[t][e] = make_float2(0.0f, 0.0f);

  auto round_fma = [&](int j, const uint4 (&xv)[TB]) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      float2 x2[TB];
#pragma unroll
      for (int t = 0; t < TB; ++t) {
        const uint32_t w32 = (k < 2) ? xv[t].x : (k < 4) ? xv[t].y : (k < 6) ? xv[t].z : xv[t].w;
        const float xf = (k & 1) ? bf16_hi(w32) : bf16_lo(w32);
        x2[t] = make_float2(xf, xf);
      }
#pragma unroll
      for (int u = 0; u < UNITS; ++u) {
        const uint4 wv = sw[((j * 8 + k) * 32 + lane) * UNITS + (u ^ router_swz<UNITS>(lane))];
        const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 w2 = make_float2(bf16_lo(ww[q]), bf16_hi(ww[q]));  // experts 8u+2q, 8u+2q+1
#pragma unroll
          for (int t = 0; t < TB; ++t) acc[t][u * 4 + q] = fma2(x2[t], w2, acc[t][u * 4 + q]);
        }
      }
    }
  };

  if constexpr (XALL) {
#pragma unroll
    for (int j = 0; j < XR; ++j)
      if (j < rounds) round_fma(j, xb[j]);
  } else {
    for (int j = 0; j < rounds; j += 2) {   // two register buffers, fixed indices
      if (j + 1 < rounds) load_x(j + 1, xb[1]);
      round_fma(j, xb[0]);
      if (j + 1 < rounds) {
        if (j + 2 < rounds) load_x(j + 2, xb[0]);
        round_fma(j + 1, xb[1]);
      }
    }
  }

  // Pairwise tree over the 32 partials (lanes), partial p with p^o for
  // o = 16..1.  Each level halves the values a lane keeps, so lane p ends
  // with the sums of values [p*M, p*M + M), M = NV / 32.
  float v[NV];
#pragma unroll
  for (int t = 0; t < TB; ++t)
#pragma unroll
    for (int e = 0; e < EB / 2; ++e) {
      v[t * EB + 2 * e] = acc[t][e].x;
      v[t * EB + 2 * e + 1] = acc[t][e].y;
    }
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
  pdl_trigger();
  pdl_wait();
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
// the (token, slot) pairs that chose this expert, in token order.  The
// expert's rows are cut into GEMM tiles of tile_rows (32 or 128) rows; each
// tile starts its own 128-row block of the padded operand layout, so a tile's
// rows always sit at the head of one block-scale atom.
__global__ void __launch_bounds__(PERM_THREADS) permute_kernel(const int32_t* __restrict__ topk_ids,
                                                              const int32_t* __restrict__ counts, int T, int K,
                                                              int E, int tile_shift, PermuteOut o) {
  __shared__ int red[PERM_THREADS / 32];
  const int e = blockIdx.x;
  const int tile_rows = 1 << tile_shift;   // 32 or 128 rows per GEMM tile
  pdl_trigger();
  pdl_wait();
  int c_lt = 0, p_lt = 0, n_lt = 0;
  for (int i = threadIdx.x; i < e; i += blockDim.x) {
    const int c = counts[i];
    const int nt = (c + tile_rows - 1) >> tile_shift;
    c_lt += c;
    p_lt += nt * 128;                      // every tile starts a 128-row block
    n_lt += nt;
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
        const int pr = poff + (pos >> tile_shift) * 128 + (pos & (tile_rows - 1));
        o.src_of_row[r] = src;
        o.row_of_src[src] = r;
        o.pad_row_of_src[src] = pr;
        o.src_of_padrow[pr] = src;
        ++pos;
      }
    }
    carry += tot;
  }
  const int ntile = (cnt + tile_rows - 1) >> tile_shift;
  for (int i = threadIdx.x; i < ntile; i += blockDim.x)
    o.tiles[tbase + i] = make_int4(e, poff + 128 * i, min(tile_rows, cnt - tile_rows * i), 0);
  if (threadIdx.x == 0) {
    o.expert_offsets[e] = off;
    if (e == E - 1) {
      o.expert_offsets[E] = off + cnt;
      o.num_tiles[0] = tbase + ntile;
    }
  }
}

template <int TB, int EB, bool XALL>
cudaError_t launch_router_t(const void* x, const void* gate_w, const float* bias, float* logits, int T, int H,
                            int E, int32_t* counts, cudaStream_t s) {
  dim3 grid((T + ROUTER_WARPS * TB - 1) / (ROUTER_WARPS * TB), E / EB);
  const size_t smem = (size_t)H * EB * 2;
  // first kernel of a forward: ordinary stream order (it may depend on the caller's work)
  return launch_k(router_logits_kernel<TB, EB, XALL>, grid, dim3(256), smem, s, false,
                  reinterpret_cast<const __nv_bfloat16*>(x), reinterpret_cast<const __nv_bfloat16*>(gate_w), bias,
                  logits, T, H, E, counts);
}

// Expert block: the widest of 32 / 16 / 8 experts that divides E and keeps
// the staged slice (H * EB * 2 bytes) within 96 KB, so two CTAs fit an SM.
int router_eb(int H, int E) {
  for (int eb : {32, 16, 8})
    if (E % eb == 0 && (size_t)H * eb * 2 <= 96 * 1024) return eb;
  return 8;
}

// Small batches: two tokens per warp with all activations prefetched.
bool router_small(int T, int H) { return T <= 512 && H <= 2048; }

// Raises (never lowers) the dynamic shared-memory cap of one router
// instantiation to `bytes`.  The cap belongs to the kernel, not to a handle,
// so a handle with a narrower hidden size must not shrink it under another.
template <int TB, int EB, bool XALL>
cudaError_t raise_router_attr(int bytes) {
  cudaFuncAttributes a{};
  cudaError_t e = cudaFuncGetAttributes(&a, router_logits_kernel<TB, EB, XALL>);
  if (e != cudaSuccess || a.maxDynamicSharedSizeBytes >= bytes) return e;
  return cudaFuncSetAttribute(router_logits_kernel<TB, EB, XALL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              bytes);
}

std::mutex router_attr_mutex;

}  // namespace

cudaError_t router_setup(int H, int E) {
  const int eb = router_eb(H, E);
  const int bytes = H * eb * 2;
  std::lock_guard<std::mutex> lock(router_attr_mutex);
  cudaError_t e;
  if (eb == 32) {
    if ((e = raise_router_attr<4, 32, false>(bytes)) != cudaSuccess) return e;
    return raise_router_attr<2, 32, true>(bytes);
  }
  if (eb == 16) {
    if ((e = raise_router_attr<4, 16, false>(bytes)) != cudaSuccess) return e;
    return raise_router_attr<2, 16, true>(bytes);
  }
  if ((e = raise_router_attr<4, 8, false>(bytes)) != cudaSuccess) return e;
  return raise_router_attr<4, 8, true>(bytes);
}

cudaError_t router_setup_max(int bytes) {
  std::lock_guard<std::mutex> lock(router_attr_mutex);
  cudaError_t e;
  if ((e = raise_router_attr<4, 32, false>(bytes)) != cudaSuccess) return e;
  if ((e = raise_router_attr<2, 32, true>(bytes)) != cudaSuccess) return e;
  if ((e = raise_router_attr<4, 16, false>(bytes)) != cudaSuccess) return e;
  if ((e = raise_router_attr<2, 16, true>(bytes)) != cudaSuccess) return e;
  if ((e = raise_router_attr<4, 8, false>(bytes)) != cudaSuccess) return e;
  return raise_router_attr<4, 8, true>(bytes);
}

int router_smem_bytes(int H, int E) { return H * router_eb(H, E) * 2; }

cudaError_t launch_router_logits(const void* x, const void* gate_w, const float* bias, float* logits, int T,
                                 int H, int E, int32_t* counts, cudaStream_t s) {
  const int eb = router_eb(H, E);
  const bool small = router_small(T, H);
  if (eb == 32) return small ? launch_router_t<2, 32, true>(x, gate_w, bias, logits, T, H, E, counts, s)
                             : launch_router_t<4, 32, false>(x, gate_w, bias, logits, T, H, E, counts, s);
  if (eb == 16) return small ? launch_router_t<2, 16, true>(x, gate_w, bias, logits, T, H, E, counts, s)
                             : launch_router_t<4, 16, false>(x, gate_w, bias, logits, T, H, E, counts, s);
  return small ? launch_router_t<4, 8, true>(x, gate_w, bias, logits, T, H, E, counts, s)
               : launch_router_t<4, 8, false>(x, gate_w, bias, logits, T, H, E, counts, s);
}

cudaError_t launch_topk(const float* logits, int T, int E, int K, int32_t* topk_ids, float* topk_w,
                        int32_t* counts, cudaStream_t s) {
  return launch_k(topk_kernel, dim3((T + 7) / 8), dim3(256), 0, s, true, logits, T, E, K, topk_ids, topk_w, counts);
}

cudaError_t launch_permute(const int32_t* topk_ids, const int32_t* counts, int T, int K, int E, int tile_rows,
                           const PermuteOut& o, cudaStream_t s) {
  const int shift = tile_rows == 32 ? 5 : 7;
  return launch_k(permute_kernel, dim3(E), dim3(PERM_THREADS), 0, s, true, topk_ids, counts, T, K, E, shift, o);
}

}  // namespace moe
