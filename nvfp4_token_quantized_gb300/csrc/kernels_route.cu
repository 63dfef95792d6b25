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
#include <type_traits>

#include "common.cuh"
#include "grouping.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int ROUTER_WARPS = 8;
// Large batches: each warp's activations stream through a shared-memory
// ring of ROUTER_XRING rounds, filled two rounds ahead by cp.async.
constexpr int ROUTER_XRING = 3;
// Bytes of a router instantiation's activation ring (0 for XALL).
__host__ __device__ constexpr int router_xring_bytes(int TB, bool XALL, int WARPS) {
  return XALL ? 0 : WARPS * ROUTER_XRING * TB * 512;
}

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

// Logits of one (token block, expert block) tile, for a CTA of a grid
// (ceil(T / (WARPS*TB)), E / EB) of WARPS warps; dynamic shared
// memory H * EB * 2 bytes holding the CTA's whole router-weight slice,
// laid out [round j][k][partial p][EB] (row h = 256 j + 8 p + k), then
// (without XALL) the warps' activation rings.
// Warp w handles tokens t0..t0+TB-1; lane p is partial p of every
// (token, expert) pair of the CTA's expert block: it accumulates chunks
// c = p, p+32, ... in ascending order with one fused multiply-add per element,
// then the 32 partials are combined by the pairwise tree.
//
// XALL: every round's activations are loaded into registers up front (one
// memory round trip; H <= 2048), for small token counts where latency rules.
// Otherwise round j's activations arrive in ring slot j % ROUTER_XRING,
// copied two rounds ahead.
// Ends with a __syncthreads-free store of the logits; the caller may reuse
// the shared memory only after its own barrier.
template <int TB, int EB, bool XALL, int WARPS>
__device__ __forceinline__ void router_tile(const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ wg,
                                            const float* __restrict__ bias, float* __restrict__ logits, int T,
                                            int H, int E) {
  constexpr int UNITS = EB / 8;                 // 16-byte units (8 bf16) per staged row
  constexpr int NV = TB * EB;                   // partial sums per lane
  static_assert(NV % 32 == 0 || NV == 8 || NV == 16, "TB*EB must be 8, 16 or a multiple of 32");
  extern __shared__ uint4 sw[];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e0 = blockIdx.y * EB;
  const int t0 = (blockIdx.x * WARPS + warp) * TB;
  const int rounds = H / 256;

  for (int h = threadIdx.x; h < H; h += 32 * WARPS) {
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
  // the activation ring: this warp's after the weight slice, slot r, token
  // t, lane p at [r][t][p]; each lane copies and later reads only its own
  // 16-byte pieces, so the ring needs no barrier (rows past T read as zeros)
  uint4* xs_w = sw + (size_t)H * EB * 2 / 16 + (size_t)warp * ROUTER_XRING * TB * 32;
  auto issue_x = [&](int j) {
    const int c = j * 32 + lane;
    uint4* slot = xs_w + (j % ROUTER_XRING) * TB * 32;
#pragma unroll
    for (int t = 0; t < TB; ++t) {
      const int tok = t0 + t;
      const __nv_bfloat16* src = x + (tok < T ? (size_t)tok * H + 8 * c : 0);
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(slot + t * 32 + lane)), "l"(src),
                   "r"(tok < T ? 16 : 0)
                   : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  constexpr int XR = XALL ? 8 : 1;              // rounds of activations held in registers
  uint4 xb[XR][TB];
  if constexpr (XALL) {
#pragma unroll
    for (int j = 0; j < XR; ++j)
      if (j < rounds) load_x(j, xb[j]);
    asm volatile("cp.async.wait_group 0;" ::: "memory");
  } else {
    issue_x(0);
    if (rounds > 1) issue_x(1);
    // the weight slice (the oldest group) has landed
    if (rounds > 1) asm volatile("cp.async.wait_group 2;" ::: "memory");
    else asm volatile("cp.async.wait_group 1;" ::: "memory");
  }
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
    for (int j = 0; j < rounds; ++j) {
      if (j + 2 < rounds) issue_x(j + 2);   // into the slot round j - 1 used
      // groups issued after round j's may stay in flight
      if (j + 2 < rounds) asm volatile("cp.async.wait_group 2;" ::: "memory");
      else if (j + 1 < rounds) asm volatile("cp.async.wait_group 1;" ::: "memory");
      else asm volatile("cp.async.wait_group 0;" ::: "memory");
      const uint4* slot = xs_w + (j % ROUTER_XRING) * TB * 32;
#pragma unroll
      for (int t = 0; t < TB; ++t) xb[0][t] = slot[t * 32 + lane];
      round_fma(j, xb[0]);
    }
  }

  // Pairwise tree over the 32 partials (lanes), partial p with p^o for
  // o = 16..1.  With NV >= 32 each level halves the values a lane keeps, so
  // lane p ends with the sums of values [p*M, p*M + M), M = NV / 32; with
  // fewer values every lane keeps all of them (a plain butterfly: the same
  // sums, since each level adds the same two partials) and lane i < NV
  // writes value i.
  float v[NV];
#pragma unroll
  for (int t = 0; t < TB; ++t)
#pragma unroll
    for (int e = 0; e < EB / 2; ++e) {
      v[t * EB + 2 * e] = acc[t][e].x;
      v[t * EB + 2 * e + 1] = acc[t][e].y;
    }
  if constexpr (NV < 32) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int i = 0; i < NV; ++i) v[i] = __fadd_rn(v[i], __shfl_xor_sync(0xffffffffu, v[i], o));
    float mine = v[0];
#pragma unroll
    for (int i = 1; i < NV; ++i)
      if (lane == i) mine = v[i];
    const int t = lane / EB, e = lane % EB;
    const int tok = t0 + t;
    if (lane < NV && tok < T) {
      if (bias) mine = __fadd_rn(mine, bias[e0 + e]);
      logits[(size_t)tok * E + e0 + e] = mine;
    }
    return;
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

// The router kernel: one (token block, expert block) tile per CTA.
template <int TB, int EB, bool XALL, int WARPS>
__global__ void __launch_bounds__(32 * WARPS) router_logits_kernel(const __nv_bfloat16* __restrict__ x,
                                                           const __nv_bfloat16* __restrict__ wg,
                                                           const float* __restrict__ bias,
                                                           float* __restrict__ logits, int T, int H, int E) {
  pdl_trigger();
  router_tile<TB, EB, XALL, WARPS>(x, wg, bias, logits, T, H, E);
}

// (value, expert) order of the top-k: larger logit first, ties to the lower
// expert id.  As one 64-bit key: the logit's bits mapped to an unsigned
// integer of the same order (-0 taken as +0, so that equal logits tie) in the
// high word, the complement of the expert id in the low word; the larger key
// comes first.
__device__ __forceinline__ uint64_t topk_key(float v, int e) {
  const uint32_t b = __float_as_uint(__fadd_rn(v, 0.0f));  // -0 -> +0
  const uint32_t o = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return ((uint64_t)o << 32) | (uint32_t)~e;
}
__device__ __forceinline__ float topk_key_value(uint32_t o) {
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}

// Compare-exchange of two keys: the larger ends up in a.
__device__ __forceinline__ void topk_cas(uint64_t& a, uint64_t& b) {
  const uint64_t hi = a > b ? a : b, lo = a > b ? b : a;
  a = hi;
  b = lo;
}

// Top-k of one token's logits by one warp.  Lane l holds the NE candidates
// l, l + 32, ... (E <= 32 NE) as keys sorted descending; each of the K rounds
// takes the largest lane head over the warp - two warp-wide unsigned maxima
// (redux.sync), of the high words, then of the low words among the lanes
// holding that high word - and the lane that held it moves on to its next
// candidate.  Softmax over all E experts (each lane sums its raw logits in
// ascending expert order, then the xor tree), chosen probabilities
// renormalised in slot order.  Lane j < K returns slot j: its expert in e_lane
// and its weight in w_lane.  Logits are read through L2 (another CTA of the
// same grid may have written them).  All 32 lanes must call it.
// SMEM: lrow is in shared memory (the CTA's own logits).
template <int NE, bool SMEM = false>
__device__ __forceinline__ void topk_warp_n(const float* __restrict__ lrow, int E, int K, int lane, int& e_lane,
                                            float& w_lane) {
  float raw[NE];
  uint64_t key[NE];
#pragma unroll
  for (int i = 0; i < NE; ++i) {
    const int e = lane + 32 * i;
    raw[i] = e < E ? (SMEM ? lrow[e] : __ldcg(lrow + e)) : -INFINITY;
    key[i] = e < E ? topk_key(raw[i], e) : 0ull;  // padding sorts last
  }
  // sorting network: 5 exchanges for 4 candidates, 19 for 8
  if constexpr (NE == 4) {
    topk_cas(key[0], key[1]);
    topk_cas(key[2], key[3]);
    topk_cas(key[0], key[2]);
    topk_cas(key[1], key[3]);
    topk_cas(key[1], key[2]);
  } else {
    static_assert(NE == 8, "4 or 8 candidates per lane");
    constexpr int net[19][2] = {{0, 2}, {1, 3}, {4, 6}, {5, 7}, {0, 4}, {1, 5}, {2, 6}, {3, 7}, {0, 1}, {2, 3},
                                {4, 5}, {6, 7}, {2, 4}, {3, 5}, {1, 4}, {3, 6}, {1, 2}, {3, 4}, {5, 6}};
#pragma unroll
    for (int c = 0; c < 19; ++c) topk_cas(key[net[c][0]], key[net[c][1]]);
  }
  uint32_t win_hi = 0, win_lo = 0, first_hi = 0;
#pragma unroll 1
  for (int j = 0; j < K; ++j) {
    const uint32_t hi = (uint32_t)(key[0] >> 32), lo = (uint32_t)key[0];
    const uint32_t mhi = __reduce_max_sync(0xffffffffu, hi);
    const uint32_t mlo = __reduce_max_sync(0xffffffffu, hi == mhi ? lo : 0u);
    if (j == 0) first_hi = mhi;
    if (lane == j) {
      win_hi = mhi;
      win_lo = mlo;
    }
    if (hi == mhi && lo == mlo) {  // this lane's head was taken
#pragma unroll
      for (int i = 0; i + 1 < NE; ++i) key[i] = key[i + 1];
      key[NE - 1] = 0ull;
    }
  }
  // the maximum logit: the softmax denominator over all experts
  const float m = topk_key_value(first_hi);
  float s = 0.0f;
#pragma unroll
  for (int i = 0; i < NE; ++i)
    if (lane + 32 * i < E) s += expf(raw[i] - m);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  e_lane = lane < K ? (int)~win_lo : 0;
  const float pj = lane < K ? expf(topk_key_value(win_hi) - m) / s : 0.0f;
  float psum = 0.0f;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float q = __shfl_sync(0xffffffffu, pj, j);
    if (j < K) psum += q;
  }
  w_lane = pj / psum;
}

template <bool SMEM = false>
__device__ __forceinline__ void topk_warp(const float* __restrict__ lrow, int E, int K, int lane, int& e_lane,
                                          float& w_lane) {
  if (E <= 128) topk_warp_n<4, SMEM>(lrow, E, K, lane, e_lane, w_lane);
  else topk_warp_n<8, SMEM>(lrow, E, K, lane, e_lane, w_lane);
}

// One warp per token: the top-k choice and weights.
__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ logits, int T, int E, int K,
                                                  int32_t* __restrict__ topk_ids, float* __restrict__ topk_w) {
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  pdl_trigger();
  pdl_wait();
  if (t >= T) return;
  int e;
  float w;
  topk_warp(logits + (size_t)t * E, E, K, lane, e, w);
  if (lane < K) {
    topk_ids[(size_t)t * K + lane] = e;
    topk_w[(size_t)t * K + lane] = w;
  }
}

constexpr int PERM_THREADS = 512;
constexpr int PERM_TPT = 8;  // tokens per thread per pass

// One CTA per expert: every expert's row count (a shared-memory histogram
// of all the top-k ids, which the CTA reads anyway), offsets from the
// counts, then a stable compaction of the (token, slot) pairs that chose this
// expert, in token order.  The expert's rows are cut into GEMM tiles of
// tile_rows (32 or 128) rows; each tile starts its own 128-row block of the
// padded operand layout, so a tile's rows always sit at the head of one
// block-scale atom.
__global__ void __launch_bounds__(PERM_THREADS) permute_kernel(const int32_t* __restrict__ topk_ids, int T, int K,
                                                              int E, int tile_shift, PermuteOut o) {
  __shared__ int red[PERM_THREADS / 32];
  __shared__ int hist[256];  // E <= 256
  // per-warp histograms (no contention between warps), summed into hist
  __shared__ int hist_w[PERM_THREADS / 32][256];
  const int e = blockIdx.x;
  const int tile_rows = 1 << tile_shift;   // 32 or 128 rows per GEMM tile
  pdl_trigger();
  for (int i = threadIdx.x; i < (PERM_THREADS / 32) * 256; i += blockDim.x) (&hist_w[0][0])[i] = 0;
  pdl_wait();
  // Tokens per thread per pass: up to PERM_TPT, fewer for small batches so
  // that every warp takes part.  Up to PERM_THREADS * PERM_TPT tokens the
  // histogram is filled by the compaction's own loads (one pass); above, by
  // a pass of its own first.
  const int tpt = min(PERM_TPT, (T + PERM_THREADS - 1) / PERM_THREADS);
  const bool one_pass = T <= PERM_THREADS * PERM_TPT;
  if (!one_pass) {
    __syncthreads();
    for (int i = threadIdx.x; i < T * K; i += blockDim.x) atomicAdd(&hist_w[threadIdx.x >> 5][__ldg(topk_ids + i)], 1);
  }
  int off = 0, poff = 0, tbase = 0, cnt = 0;
  // offsets of this expert's rows, padded rows and tiles: sums over the
  // experts below e by warp 0, broadcast through red[0..2] (all threads call)
  auto offsets = [&]() {
    __syncthreads();  // the warps' histograms are complete
    for (int i = threadIdx.x; i < E; i += blockDim.x) {
      int c = 0;
#pragma unroll
      for (int w = 0; w < PERM_THREADS / 32; ++w) c += hist_w[w][i];
      hist[i] = c;
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      int c_lt = 0, p_lt = 0, n_lt = 0;
      for (int i = threadIdx.x; i < e; i += 32) {
        const int c = hist[i];
        const int nt = (c + tile_rows - 1) >> tile_shift;
        c_lt += c;
        p_lt += nt * 128;                  // every tile starts a 128-row block
        n_lt += nt;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        c_lt += __shfl_xor_sync(0xffffffffu, c_lt, o);
        p_lt += __shfl_xor_sync(0xffffffffu, p_lt, o);
        n_lt += __shfl_xor_sync(0xffffffffu, n_lt, o);
      }
      if (threadIdx.x == 0) {
        red[0] = c_lt;
        red[1] = p_lt;
        red[2] = n_lt;
      }
    }
    __syncthreads();
    off = red[0];
    poff = red[1];
    tbase = red[2];
    cnt = hist[e];
  };
  if (!one_pass) offsets();

  // Pass over PERM_THREADS * tpt tokens: warp w takes the block's tokens
  // [w * 32 * tpt, +32 * tpt), lane l the tokens l, l + 32, ... of them, so
  // one load instruction covers 32 consecutive token rows.
  // A row's rank among the expert's rows (token order) is: the rows of the
  // earlier passes (carry), of the earlier warps (a scan over the warps'
  // counts), of the warp's earlier 32-token groups, and of the lower lanes
  // of its own group (ballots).
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned lanes_below = (1u << lane) - 1u;
  int carry = 0;
  for (int base = 0; base < T; base += PERM_THREADS * tpt) {
    const int wbase = base + warp * 32 * tpt;
    int slot[PERM_TPT];
    unsigned bal[PERM_TPT];
    int wcount = 0;
#pragma unroll
    for (int i = 0; i < PERM_TPT; ++i) {
      slot[i] = -1;
      const int t = wbase + 32 * i + lane;
      if (i < tpt && t < T) {
        // the token's K <= 16 ids into registers first (16- or 8-byte loads
        // when K allows), then the comparisons
        int id[16];
        const int32_t* row = topk_ids + (size_t)t * K;
        if ((K & 3) == 0) {
#pragma unroll
          for (int j = 0; j < 16; j += 4)
            if (j < K) {
              const int4 v = __ldg(reinterpret_cast<const int4*>(row + j));
              id[j] = v.x;
              id[j + 1] = v.y;
              id[j + 2] = v.z;
              id[j + 3] = v.w;
            }
        } else if ((K & 1) == 0) {
#pragma unroll
          for (int j = 0; j < 16; j += 2)
            if (j < K) {
              const int2 v = __ldg(reinterpret_cast<const int2*>(row + j));
              id[j] = v.x;
              id[j + 1] = v.y;
            }
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (j < K) id[j] = __ldg(row + j);
        }
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (j < K) {
            if (id[j] == e) slot[i] = j;
            if (one_pass) atomicAdd(&hist_w[threadIdx.x >> 5][id[j]], 1);
          }
      }
      bal[i] = __ballot_sync(0xffffffffu, slot[i] >= 0);
      wcount += __popc(bal[i]);
    }
    if (one_pass) offsets();
    // exclusive scan of the warps' counts
    __syncthreads();  // red[] is free again (previous pass or block sums)
    if (lane == 0) red[warp] = wcount;
    __syncthreads();
    int wpre = 0, tot = 0;
    for (int w = 0; w < PERM_THREADS / 32; ++w) {
      const int c = red[w];
      wpre += w < warp ? c : 0;
      tot += c;
    }
    int pos = carry + wpre;
#pragma unroll
    for (int i = 0; i < PERM_TPT; ++i) {
      if (slot[i] >= 0) {
        const int t = wbase + 32 * i + lane;
        const int src = t * K + slot[i];
        const int rank = pos + __popc(bal[i] & lanes_below);
        const int r = off + rank;
        const int pr = poff + (rank >> tile_shift) * 128 + (rank & (tile_rows - 1));
        o.src_of_row[r] = src;
        o.row_of_src[src] = r;
        o.pad_row_of_src[src] = pr;
        o.src_of_padrow[pr] = src;
      }
      pos += __popc(bal[i]);
    }
    carry += tot;
  }
  const int ntile = (cnt + tile_rows - 1) >> tile_shift;
  for (int i = threadIdx.x; i < ntile; i += blockDim.x)
    o.tiles[tbase + i] = make_int4(e, poff + 128 * i, min(tile_rows, cnt - tile_rows * i), poff + 128 * i);
  if (threadIdx.x == 0) {
    o.expert_offsets[e] = off;
    if (e == E - 1) {
      o.expert_offsets[E] = off + cnt;
      o.num_tiles[0] = tbase + ntile;
    }
  }
}

// Per-token NVFP4 quantization of token t into row t of the shared
// small-batch activation tile, by one warp: the row's global scale (or the
// calibrated per-tensor scale of the static contract), then each lane's
// 16-element blocks.
// xr: the token's H bf16 values (shared or global memory).
__device__ __forceinline__ void quantize_token_row(const uint4* xr, int t, int H,
                                                   const float* __restrict__ static_gs, uint8_t* __restrict__ a_codes,
                                                   float* __restrict__ gs_rows, int lane) {
  const int nblk = H / SF_VEC;
  float gs;
  if (static_gs) {
    gs = __ldg(static_gs);
  } else {
    float amax = 0.0f;
    for (int b = lane; b < nblk; b += 32) {
      float v[16];
      bf16x16_to_f32(xr[2 * b], xr[2 * b + 1], v);
#pragma unroll
      for (int q = 0; q < 16; ++q) amax = fmaxf(amax, fabsf(v[q]));
    }
    amax = warp_max(amax);
    gs = nvfp4_global_scale(amax);
  }
  for (int b0 = 0; b0 < nblk; b0 += 32) {  // nblk % 16 == 0: uniform bound
    const int b = b0 + lane;
    uint2 packed = make_uint2(0u, 0u);
    uint32_t sf = 0;
    if (b < nblk) {
      float v[16];
      bf16x16_to_f32(xr[2 * b], xr[2 * b + 1], v);
      sf = nvfp4_quant_block16(v, gs, packed);
    }
    // blocks 4m..4m+3 have consecutive scale bytes: one 32-bit store
    const uint32_t sf4 = sf | (__shfl_down_sync(0xffffffffu, sf, 1) << 8) | (__shfl_down_sync(0xffffffffu, sf, 2) << 16) |
                         (__shfl_down_sync(0xffffffffu, sf, 3) << 24);
    if (b < nblk) {
      *reinterpret_cast<uint2*>(a_codes + operand_offset(t, 8 * b, H / 2)) = packed;
      if ((lane & 3) == 0) *reinterpret_cast<uint32_t*>(a_codes + sf_atom_offset(t, b, nblk)) = sf4;
    }
  }
  if (lane == 0) gs_rows[t] = gs;
}

// Stages of the front kernel's router-weight ring: one round of the
// canonical order (256 rows of H, every expert) per stage, double-buffered
// while two stages fit; each row padded by 16 bytes.
__host__ __device__ constexpr int front_ring_buffers(int E) { return E <= 128 ? 2 : 1; }
__host__ __device__ constexpr int front_row_stride(int E) { return 2 * E + 16; }
__host__ __device__ constexpr int front_stage_bytes(int E) { return 32 * 9 * front_row_stride(E); }

// Small-batch front end (at most 64 tokens), one launch with no hand-off
// between CTAs on the path the expert GEMMs wait for.  CTA b takes tokens
// TPC*b .. TPC*b + TPC - 1 over all E experts:
//  1. router logits in the canonical order: the router weight streams
//     through a shared-memory ring, one round of the 32 partials (256 rows
//     of H) per stage; warp w holds the partials of expert units
//     [w*UPW, w*UPW + UPW) (8 experts each) for all the CTA's tokens, lane p
//     partial p; then the pairwise tree over the partials;
//  2. per-token NVFP4 quantization of its tokens into the shared activation
//     tile (row t = token t), and the clearing of their FP32 output rows for
//     the atomic finalize;
//  3. top-k of each of its tokens (one warp per token) from the logits in
//     shared memory, and every expert's padded-row source for its tokens:
//     src_of_padrow[e*128 + t] = t*K + slot, or -1;
//  4. unless the GEMMs run the all-experts schedule, the last CTA of the grid
//     to finish (an acquire-release counter, returned to zero) derives the
//     expert grouping from all top-k ids; with that schedule the grouping is
//     left to an extra CTA of the requantization kernel.
// A stage holds round j of the router weight: chunk p (Wg rows 256 j + 8 p
// .. + 7, all E experts) at p * 9 (2E + 16) bytes, row k of the chunk at
// k (2E + 16) bytes within it (the padding is never read).  Lane p reads
// chunk p, so the 8 lanes of one shared-memory wavefront hit distinct banks.
template <int TPC, int UPW>
__global__ void __launch_bounds__(256, 1) front_small_kernel(const __grid_constant__ FrontArgs p) {
  extern __shared__ __align__(128) uint8_t front_smem[];
  __shared__ int red[ROUTER_WARPS];
  __shared__ int last;
  __shared__ int chosen[TPC][16];
  __shared__ uint64_t ring_full[2];
  __shared__ uint64_t x_full;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = p.T, H = p.H, E = p.E, K = p.K;
  const int t0 = blockIdx.x * TPC;
  const int units = E / 8;
  const int rounds = H / 256;
  const int nbuf = front_ring_buffers(E);
  const int row_bytes = 2 * E, row_stride = front_row_stride(E);
  const int chunk_stride = 9 * row_stride;  // 8 rows of a chunk plus one padding row
  const int stage_bytes = front_stage_bytes(E);
  float* slog = reinterpret_cast<float*>(front_smem + (size_t)nbuf * stage_bytes);  // [TPC][E]
  // the CTA's activation rows [TPC][H] bf16, after the logits
  const uint4* sx = reinterpret_cast<const uint4*>(front_smem + (size_t)nbuf * stage_bytes + TPC * E * 4);
  const __nv_bfloat16* x = reinterpret_cast<const __nv_bfloat16*>(p.x);
  const char* wg = reinterpret_cast<const char*>(p.gate_w);
  // The w13 GEMM may launch now and stream weights; it reads this kernel's
  // outputs only after its dependency wait.
  pdl_trigger();
  const int ntok = min(TPC, T - t0);
  if (threadIdx.x == 0) {
    mbar_init(&ring_full[0], 1);
    mbar_init(&ring_full[1], 1);
    mbar_init(&x_full, 1);
    fence_mbarrier_init();
    // the CTA's token rows, whole, with one bulk copy each
    mbar_arrive_expect_tx(&x_full, ntok * H * 2);
    for (int t = 0; t < ntok; ++t)
      bulk_load(const_cast<uint4*>(sx) + (size_t)t * H / 8, x + (size_t)(t0 + t) * H, H * 2, &x_full);
  }
  __syncthreads();

  // Warp 0 fills stage buffer b with round j.  With the tensor map: one
  // tensor copy of the round's 32 chunks x 8 rows x E experts, whose box (one
  // row and 8 columns wider than the data) pads every row with 16 zero bytes
  // and every chunk with one zero row.  Without it: 256 bulk copies of one
  // row each into the same layout.
  const bool use_map = p.wg_map_ok != 0;
  auto stage = [&](int j, int b) {
    if (warp != 0) return;
    uint8_t* dst = front_smem + (size_t)b * stage_bytes;
    if (use_map) {
      if (lane == 0) {
        mbar_arrive_expect_tx(&ring_full[b], stage_bytes);
        asm volatile(
            "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
            " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
            "l"(reinterpret_cast<uint64_t>(&p.wg_map)), "r"(0), "r"(0), "r"(j * 32), "r"(smem_u32(&ring_full[b]))
            : "memory");
      }
      return;
    }
    if (lane == 0) mbar_arrive_expect_tx(&ring_full[b], 256 * row_bytes);
    __syncwarp();
    for (int hr = lane; hr < 256; hr += 32)
      bulk_load(dst + (hr >> 3) * chunk_stride + (hr & 7) * row_stride, wg + ((size_t)j * 256 + hr) * row_bytes,
                row_bytes, &ring_full[b]);
  };
  stage(0, 0);
  if (nbuf == 2 && rounds > 1) stage(1, 1);
  const int ubase = warp * UPW;
  float2 acc[TPC][UPW * 4];
#pragma unroll
  for (int t = 0; t < TPC; ++t)
#pragma unroll
    for (int i = 0; i < UPW * 4; ++i) acc[t][i] = make_float2(0.0f, 0.0f);
  bool ring_ok = true;
  if (!mbar_wait_bounded(&x_full, 0, nullptr)) {
    if (threadIdx.x == 0) report_device_error(p.status, DEV_ERR_TIMEOUT);
    ring_ok = false;
  }
  // per-token quantization first (warps 0 .. TPC-1, from the staged rows):
  // the w13 GEMM needs only the activations to start its MMAs
  if (warp < ntok) quantize_token_row(sx + (size_t)warp * H / 8, t0 + warp, H, p.static_gs, p.a_codes, p.gs_rows, lane);
  if (p.all_experts) {
    __syncthreads();
    if (threadIdx.x == 0) arrive_acq_rel_gpu(&p.sync[FRONT_SYNC_A_READY]);
  }
  for (int j = 0; j < rounds; ++j) {
    const int b = nbuf == 2 ? (j & 1) : 0;
    const uint32_t parity = (nbuf == 2 ? (j >> 1) : j) & 1;
    if (!mbar_wait_bounded(&ring_full[b], parity, nullptr)) {
      // the copy did not land in time: report it; the results are garbage
      // but every thread still leaves
      if (ring_ok && threadIdx.x == 0) report_device_error(p.status, DEV_ERR_TIMEOUT);
      ring_ok = false;
    }
    // this lane's 8-element chunk of round j (chunk j*32 + lane) of each token
    uint4 xc[TPC];
#pragma unroll
    for (int t = 0; t < TPC; ++t) xc[t] = t < ntok ? sx[(size_t)t * H / 8 + j * 32 + lane] : make_uint4(0, 0, 0, 0);
    // lane p reads chunk p: its rows k = 0..7 (the chunks are 9 (2E + 16)
    // bytes apart, so the 8 lanes of a wavefront hit distinct banks)
    const uint8_t* sb = front_smem + (size_t)b * stage_bytes + lane * chunk_stride + ubase * 16;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      float2 x2[TPC];
#pragma unroll
      for (int t = 0; t < TPC; ++t) {
        const uint32_t w32 = (k < 2) ? xc[t].x : (k < 4) ? xc[t].y : (k < 6) ? xc[t].z : xc[t].w;
        const float xf = (k & 1) ? bf16_hi(w32) : bf16_lo(w32);
        x2[t] = make_float2(xf, xf);
      }
#pragma unroll
      for (int i = 0; i < UPW; ++i) {
        if (ubase + i < units) {  // warp-uniform
          const uint4 wv = *reinterpret_cast<const uint4*>(sb + k * row_stride + i * 16);
          const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 w2 = make_float2(bf16_lo(ww[q]), bf16_hi(ww[q]));  // experts 8u+2q, 8u+2q+1
#pragma unroll
            for (int t = 0; t < TPC; ++t) acc[t][i * 4 + q] = fma2(x2[t], w2, acc[t][i * 4 + q]);
          }
        }
      }
    }
    __syncthreads();  // buffer b is free again
    if (warp == 0) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (nbuf == 2) {
      if (j + 2 < rounds) stage(j + 2, b);
    } else if (j + 1 < rounds) {
      stage(j + 1, 0);
    }
  }

  // Pairwise tree over the 32 partials; value index (t * UPW + i) * 8 + c is
  // token t0 + t, expert 8 (ubase + i) + c.
  constexpr int NV = TPC * UPW * 8;
  float v[NV];
#pragma unroll
  for (int t = 0; t < TPC; ++t)
#pragma unroll
    for (int i = 0; i < UPW * 4; ++i) {
      v[t * UPW * 8 + 2 * i] = acc[t][i].x;
      v[t * UPW * 8 + 2 * i + 1] = acc[t][i].y;
    }
  auto put_logit = [&](int idx, float l) {
    const int t = idx / (UPW * 8), rest = idx % (UPW * 8);
    const int u = ubase + rest / 8, e = 8 * u + rest % 8;
    if (u < units && t0 + t < T) {
      if (p.bias) l = __fadd_rn(l, p.bias[e]);
      slog[t * E + e] = l;
      p.logits[(size_t)(t0 + t) * E + e] = l;
    }
  };
  if constexpr (NV < 32) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int i = 0; i < NV; ++i) v[i] = __fadd_rn(v[i], __shfl_xor_sync(0xffffffffu, v[i], o));
    float mine = v[0];
#pragma unroll
    for (int i = 1; i < NV; ++i)
      if (lane == i) mine = v[i];
    if (lane < NV) put_logit(lane, mine);
  } else {
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
    for (int i = 0; i < M; ++i) put_logit(lane * M + i, v[i]);
  }
  __syncthreads();

  // top-k (warps 0 .. TPC-1) and the atomic finalize's row clearing (warps
  // 6, 7), in parallel
  if (warp < TPC) {
    const int t = t0 + warp;
    if (t < T) {
      int e_lane;
      float w;
      topk_warp<true>(slog + warp * E, E, K, lane, e_lane, w);
      if (lane < K) {
        p.topk_ids[(size_t)t * K + lane] = e_lane;
        p.topk_w[(size_t)t * K + lane] = w;
        chosen[warp][lane] = e_lane;
      }
    }
  } else if (warp >= 6 && p.out_acc) {
    for (int t = t0; t < min(t0 + TPC, T); ++t) {
      float4* o = reinterpret_cast<float4*>(p.out_acc + (size_t)t * H);
      for (int q = (warp - 6) * 32 + lane; q < H / 4; q += 64) o[q] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < TPC * E; i += blockDim.x) {
    const int t = i / E, e = i - t * E, tok = t0 + t;
    if (tok < T) {
      int src = -1;
      for (int j = 0; j < K; ++j)
        if (chosen[t][j] == e) src = tok * K + j;
      p.src_of_padrow[e * 128 + tok] = src;
    }
  }
  // Routing (and the row clearing) published.  With the all-experts
  // schedule the w13 GEMM completes only after every front CTA arrived on
  // the routed counter (the w2 GEMM returns it to zero); otherwise a counter
  // of its own (returned to zero below).  The last CTA to arrive derives the
  // expert grouping: on the all-experts path no GEMM waits for it.
  __syncthreads();
  uint32_t* ctr = p.all_experts ? &p.sync[FRONT_SYNC_ROUTED] : &p.sync[FRONT_SYNC_WORDS - 1];
  if (threadIdx.x == 0) last = arrive_acq_rel_gpu(ctr) == gridDim.x - 1;
  __syncthreads();
  if (!last) return;
  unsigned long long* tok_mask = reinterpret_cast<unsigned long long*>(front_smem);  // [256] (the ring is idle)
  int* offs = reinterpret_cast<int*>(tok_mask + 256);                                // [256]
  const SmallGroupOut go{p.expert_offsets, p.src_of_row, p.row_of_src, p.pad_row_of_src, p.tiles, p.num_tiles};
  small_grouping(p.topk_ids, T, K, E, go, tok_mask, offs, red);
  if (threadIdx.x == 0 && !p.all_experts) p.sync[FRONT_SYNC_WORDS - 1] = 0;
}

template <int TB, int EB, bool XALL, int WARPS = ROUTER_WARPS>
cudaError_t launch_router_t(const void* x, const void* gate_w, const float* bias, float* logits, int T, int H,
                            int E, cudaStream_t s) {
  dim3 grid((T + WARPS * TB - 1) / (WARPS * TB), E / EB);
  const size_t smem = (size_t)H * EB * 2 + router_xring_bytes(TB, XALL, WARPS);
  // first kernel of a forward: ordinary stream order (it may depend on the caller's work)
  return launch_k(router_logits_kernel<TB, EB, XALL, WARPS>, grid, dim3(32 * WARPS), smem, s, false,
                  reinterpret_cast<const __nv_bfloat16*>(x), reinterpret_cast<const __nv_bfloat16*>(gate_w), bias,
                  logits, T, H, E);
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
// `bytes` is the weight slice's size, to which the activation ring is added
// (with_ring), or the whole cap.
template <int TB, int EB, bool XALL, int WARPS = ROUTER_WARPS>
cudaError_t raise_router_attr(int bytes, bool with_ring = true) {
  if (with_ring) bytes += router_xring_bytes(TB, XALL, WARPS);
  cudaFuncAttributes a{};
  cudaError_t e = cudaFuncGetAttributes(&a, router_logits_kernel<TB, EB, XALL, WARPS>);
  if (e != cudaSuccess || a.maxDynamicSharedSizeBytes >= bytes) return e;
  return cudaFuncSetAttribute(router_logits_kernel<TB, EB, XALL, WARPS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
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
  if ((e = raise_router_attr<4, 32, false>(bytes, false)) != cudaSuccess) return e;
  if ((e = raise_router_attr<2, 32, true>(bytes, false)) != cudaSuccess) return e;
  if ((e = raise_router_attr<4, 16, false>(bytes, false)) != cudaSuccess) return e;
  if ((e = raise_router_attr<2, 16, true>(bytes, false)) != cudaSuccess) return e;
  if ((e = raise_router_attr<4, 8, false>(bytes, false)) != cudaSuccess) return e;
  return raise_router_attr<4, 8, true>(bytes, false);
}

int router_smem_bytes(int H, int E) { return H * router_eb(H, E) * 2 + router_xring_bytes(4, false, ROUTER_WARPS); }

namespace {


// Dynamic shared memory of the front kernel: the router-weight ring and the
// CTA's logits (at least the 3 KB the grouping reuses).
int front_smem_bytes(int H, int E, int tpc) {
  return std::max(front_ring_buffers(E) * front_stage_bytes(E) + tpc * E * 4 + tpc * H * 2, 3 * 1024);
}

template <int TPC, int UPW>
cudaError_t raise_front_attr(int H, int E) {
  const int bytes = front_smem_bytes(H, E, TPC);
  if (bytes > 227 * 1024) return cudaErrorInvalidValue;  // hidden sizes beyond 16384 at 128 experts
  cudaFuncAttributes a{};
  cudaError_t e = cudaFuncGetAttributes(&a, front_small_kernel<TPC, UPW>);
  if (e != cudaSuccess || a.maxDynamicSharedSizeBytes >= bytes) return e;
  return cudaFuncSetAttribute(front_small_kernel<TPC, UPW>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

// Tokens per CTA: one up to 32 tokens, two above (at most 32 CTAs at 64
// tokens, so that most SMs are free for the w13 GEMM launched behind the
// front kernel; the GEMM is persistent with one CTA per SM and cannot share
// an SM with a front CTA).  Expert units (8 experts) per warp: E/64 rounded
// up to 1, 2 or 4.  Calls f with (tokens per CTA, units per warp) as types.
int front_tpc(int T) { return T <= 32 ? 1 : 2; }

template <typename F>
cudaError_t with_front(int T, int E, F&& f) {
  using std::integral_constant;
  const int upw = (E / 8 + ROUTER_WARPS - 1) / ROUTER_WARPS;
  if (front_tpc(T) == 1) {
    if (upw <= 1) return f(integral_constant<int, 1>{}, integral_constant<int, 1>{});
    if (upw <= 2) return f(integral_constant<int, 1>{}, integral_constant<int, 2>{});
    return f(integral_constant<int, 1>{}, integral_constant<int, 4>{});
  }
  if (upw <= 1) return f(integral_constant<int, 2>{}, integral_constant<int, 1>{});
  if (upw <= 2) return f(integral_constant<int, 2>{}, integral_constant<int, 2>{});
  return f(integral_constant<int, 2>{}, integral_constant<int, 4>{});
}

template <int TPC, int UPW>
cudaError_t launch_front_t(const FrontArgs& a, cudaStream_t s) {
  // first kernel of a forward: ordinary stream order
  return launch_k(front_small_kernel<TPC, UPW>, dim3((a.T + TPC - 1) / TPC), dim3(256),
                  (size_t)front_smem_bytes(a.H, a.E, TPC), s, false, a);
}

}  // namespace


int front_ctas(int T, int E) {
  (void)E;
  const int tpc = front_tpc(T);
  return (T + tpc - 1) / tpc;
}

cudaError_t front_setup(int H, int E) {
  std::lock_guard<std::mutex> lock(router_attr_mutex);
  for (int T : {1, SMALL_BATCH_TOKENS}) {
    cudaError_t e = with_front(T, E, [&](auto tpc, auto upw) {
      return raise_front_attr<decltype(tpc)::value, decltype(upw)::value>(H, E);
    });
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once through the runtime (the
// library does not link against the driver library).
EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

// Router-weight map for the front kernel's ring: Wg [H][E] bf16 viewed as
// [H/8 chunks][8 rows][E], box of 32 chunks x 9 rows x (E + 8) columns: the
// row and the columns past the tensor are filled with zeros, which pads the
// staged rows and chunks (no swizzle).  False when E + 8 exceeds a box (256)
// or the encoder refuses.
bool encode_router_map(CUtensorMap* map, const void* gate_w, int H, int E) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn || E + 8 > 256 || H % 256) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)E, 8, (cuuint64_t)H / 8};
  const cuuint64_t strides[2] = {(cuuint64_t)E * 2, (cuuint64_t)E * 16};
  const cuuint32_t box[3] = {(cuuint32_t)(E + 8), 9, 32};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(gate_w), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_front_small(FrontArgs& a, cudaStream_t s) {
  if (a.T > SMALL_BATCH_TOKENS || a.E > 256 || a.K > 16 || a.H % 256) return cudaErrorInvalidValue;
  a.wg_map_ok = encode_router_map(&a.wg_map, a.gate_w, a.H, a.E) ? 1 : 0;
  return with_front(a.T, a.E, [&](auto tpc, auto upw) {
    return launch_front_t<decltype(tpc)::value, decltype(upw)::value>(a, s);
  });
}

cudaError_t launch_router_logits(const void* x, const void* gate_w, const float* bias, float* logits, int T,
                                 int H, int E, cudaStream_t s) {
  const int eb = router_eb(H, E);
  const bool small = router_small(T, H);
  if (eb == 32) return small ? launch_router_t<2, 32, true>(x, gate_w, bias, logits, T, H, E, s)
                             : launch_router_t<4, 32, false>(x, gate_w, bias, logits, T, H, E, s);
  if (eb == 16) return small ? launch_router_t<2, 16, true>(x, gate_w, bias, logits, T, H, E, s)
                             : launch_router_t<4, 16, false>(x, gate_w, bias, logits, T, H, E, s);
  return small ? launch_router_t<4, 8, true>(x, gate_w, bias, logits, T, H, E, s)
               : launch_router_t<4, 8, false>(x, gate_w, bias, logits, T, H, E, s);
}

cudaError_t launch_topk(const float* logits, int T, int E, int K, int32_t* topk_ids, float* topk_w,
                        cudaStream_t s) {
  return launch_k(topk_kernel, dim3((T + 7) / 8), dim3(256), 0, s, true, logits, T, E, K, topk_ids, topk_w);
}

cudaError_t launch_permute(const int32_t* topk_ids, int T, int K, int E, int tile_rows,
                           const PermuteOut& o, cudaStream_t s) {
  const int shift = tile_rows == 32 ? 5 : 7;
  if (E > 256) return cudaErrorInvalidValue;
  return launch_k(permute_kernel, dim3(E), dim3(PERM_THREADS), 0, s, true, topk_ids, T, K, E, shift, o);
}

}  // namespace moe
