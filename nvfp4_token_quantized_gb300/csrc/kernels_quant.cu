// kernels_quant.cu - per-token NVFP4 quantization of the activations (fused
// with the expert expansion), online NVFP4 conversion of the expert weights,
// the finalize kernels, and the parity exports.
//
// Quantization rules ("CuTe DSL backend gets per-token NVFP4 online
// quantization and reload", Implementation item 2; the stated reading):
// gs = 2688 / amax per token (or per expert for weights); per 16-element
// block sf = E4M3(amax_b * gs / 6); code = E2M1(x * (gs / sf)).
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

// Block pairs per lane whose codes the activation quantizer holds in
// registers across its dependency wait (rows of up to 32 * 4 * 32 = 4096
// elements).
constexpr int AQ_MAX_PAIRS = 4;

// One warp per token.  Lane L owns the 16-element blocks L, L+32, ...
// The token's codes, block scales and global scale are written to each of its
// K expanded rows (the rows of its K experts in the padded expert-grouped
// layout the w13 GEMM reads).  (Batches that reach this kernel take the
// ordered finalize, so no FP32 accumulator needs clearing.)
__global__ void __launch_bounds__(256, 4) act_quant_kernel(const __nv_bfloat16* __restrict__ x, int T, int H, int K,
                                                       const int32_t* __restrict__ pad_row_of_src,
                                                       uint8_t* __restrict__ a_codes, uint8_t* __restrict__ a_sf,
                                                       float* __restrict__ gs_rows,
                                                       const float* __restrict__ static_gs) {
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  pdl_trigger();
  if (t >= T) {
    pdl_wait();
    return;
  }
  const int nblk = H / SF_VEC;
  const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)t * H);

  // x is the caller's input: reading it and forming the row maximum may
  // overlap the permutation kernel; its outputs are read after pdl_wait().
  // per-token global scale from the row maximum, or the calibrated
  // per-tensor scale of the static contract
  float gs;
  if (static_gs) {
    gs = __ldg(static_gs);
  } else {
    float amax = 0.0f;
    for (int b = lane; b < nblk; b += 32) {
      float v[16];
      bf16x16_to_f32(__ldg(xr + 2 * b), __ldg(xr + 2 * b + 1), v);
#pragma unroll
      for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
    }
    amax = warp_max(amax);
    gs = nvfp4_global_scale(amax);
  }

  // Codes and block scales of the row, computed before the dependency wait
  // (they depend only on x) and held in registers: lane L owns the block
  // pairs L, L + 32, ... (blocks 2p and 2p + 1: one 16-byte unit of codes;
  // at most AQ_MAX_PAIRS pairs, longer rows take the loop below, which
  // quantizes after the wait).  nblk is a multiple of 16, so the loop bounds
  // are warp-uniform; blocks 4m..4m+3 (lanes 2k, 2k + 1) have consecutive
  // scale bytes, written as one 32-bit word by the even lane.
  const size_t row_bytes = (size_t)H / 2;
  const int npair = nblk / 2;
  const int np_lane = (npair + 31) / 32;
  if (np_lane <= AQ_MAX_PAIRS) {
    uint4 packed[AQ_MAX_PAIRS];
    uint32_t sf4[AQ_MAX_PAIRS];
#pragma unroll
    for (int i = 0; i < AQ_MAX_PAIRS; ++i) {
      if (i < np_lane) {
        const int pr = 32 * i + lane;
        uint32_t sf2 = 0;
        packed[i] = make_uint4(0u, 0u, 0u, 0u);
        if (pr < npair) {
          float v[16];
          uint2 c0, c1;
          bf16x16_to_f32(__ldg(xr + 4 * pr), __ldg(xr + 4 * pr + 1), v);
          const uint32_t s0 = nvfp4_quant_block16(v, gs, c0);
          bf16x16_to_f32(__ldg(xr + 4 * pr + 2), __ldg(xr + 4 * pr + 3), v);
          const uint32_t s1 = nvfp4_quant_block16(v, gs, c1);
          packed[i] = make_uint4(c0.x, c0.y, c1.x, c1.y);
          sf2 = s0 | (s1 << 8);
        }
        sf4[i] = sf2 | (__shfl_down_sync(0xffffffffu, sf2, 1) << 16);
      }
    }
    pdl_wait();
    // the K expanded rows, loaded at once (lane j holds row j)
    const int my_prow = lane < K ? pad_row_of_src[(size_t)t * K + lane] : 0;
    for (int j = 0; j < K; ++j) {
      const int prow = __shfl_sync(0xffffffffu, my_prow, j);
#pragma unroll
      for (int i = 0; i < AQ_MAX_PAIRS; ++i) {
        const int pr = 32 * i + lane;
        if (i < np_lane && pr < npair) {
          *reinterpret_cast<uint4*>(a_codes + operand_offset(prow, 16 * pr, (int)row_bytes)) = packed[i];
          if ((lane & 1) == 0) *reinterpret_cast<uint32_t*>(a_sf + sf_atom_offset(prow, 2 * pr, nblk)) = sf4[i];
        }
      }
      if (lane == 0) gs_rows[prow] = gs;
    }
    return;
  }

  pdl_wait();
  const int my_prow = lane < K ? pad_row_of_src[(size_t)t * K + lane] : 0;
  for (int b0 = 0; b0 < nblk; b0 += 32) {
    const int b = b0 + lane;
    const bool active = b < nblk;
    uint2 packed = make_uint2(0u, 0u);
    uint32_t sf = 0;
    if (active) {
      float v[16];
      bf16x16_to_f32(__ldg(xr + 2 * b), __ldg(xr + 2 * b + 1), v);
      sf = nvfp4_quant_block16(v, gs, packed);
    }
    const uint32_t sf4 = sf | (__shfl_down_sync(0xffffffffu, sf, 1) << 8) | (__shfl_down_sync(0xffffffffu, sf, 2) << 16) |
                         (__shfl_down_sync(0xffffffffu, sf, 3) << 24);
    for (int j = 0; j < K; ++j) {
      const int prow = __shfl_sync(0xffffffffu, my_prow, j);
      if (active) {
        *reinterpret_cast<uint2*>(a_codes + operand_offset(prow, 8 * b, (int)row_bytes)) = packed;
        if ((lane & 3) == 0) *reinterpret_cast<uint32_t*>(a_sf + sf_atom_offset(prow, b, nblk)) = sf4;
      }
    }
  }
  if (lane < K) gs_rows[my_prow] = gs;
}

// Requantization of the small-batch w13 output: one warp per expanded row
// (token * K + slot), at its padded row: topk_ids[row] * 128 + row / K in the
// small-batch layout, or row_map[row].  Row maximum -> global scale -> block
// scales and codes, the same arithmetic as the fused w13 epilogue; returns
// the row's maximum word to zero.
// do_all (the all-experts path): no dependency wait up front.  A warp waits
// (bounded, acquire) until the routing is published and its row's expert
// has all its column pairs done, so rows are requantized while the w13 GEMM
// still runs its last units; every CTA then waits for the GEMM (so that this
// kernel completes after it, as later kernels assume) and returns to zero the
// maxima of rows of tokens that did not route to an expert.
__global__ void __launch_bounds__(256) requant_rows_kernel(const float* __restrict__ hbuf,
                                                          float* __restrict__ row_amax,
                                                          const int32_t* __restrict__ row_map,
                                                          const int32_t* __restrict__ topk_ids, int K, int n_rows,
                                                          int I, int i_pad, uint8_t* __restrict__ h_codes,
                                                          float* __restrict__ h_gs, const RequantAllExperts all,
                                                          int do_all, int* __restrict__ status) {
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  pdl_trigger();
  if (!do_all) pdl_wait();
  if (row < n_rows) {
    bool ok = true;
    if (do_all) {
      if (lane == 0)
        ok = wait_counter_acquire(all.front_sync + FRONT_SYNC_ROUTED, (uint32_t)all.front_ctas, nullptr) &&
             wait_counter_acquire(all.expert_done + __ldcg(topk_ids + row), (uint32_t)all.pairs, nullptr);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok && lane == 0) report_device_error(status, DEV_ERR_TIMEOUT);
    }
    if (ok) {
      const int prow = topk_ids ? __ldcg(topk_ids + row) * 128 + row / K : row_map[row];
      const float gs = nvfp4_global_scale(__ldcg(row_amax + prow));
      requant_row_warp(hbuf + (size_t)prow * i_pad, I, i_pad, prow, gs, h_codes, lane);
      if (lane == 0) {
        h_gs[prow] = gs;
        row_amax[prow] = 0.0f;
      }
    }
  }
  if (do_all) {
    pdl_wait();
    const int T = n_rows / K;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < all.E * T; i += gridDim.x * blockDim.x) {
      const int prow = (i / T) * 128 + i % T;
      if (all.src_of_padrow[prow] < 0) row_amax[prow] = 0.0f;
    }
  }
}

// amax over each expert's whole matrix: grid (chunks, E).
__global__ void __launch_bounds__(256) weight_amax_kernel(const __nv_bfloat16* __restrict__ w, size_t per_expert,
                                                         uint32_t* __restrict__ amax_bits) {
  const int e = blockIdx.y;
  const uint4* src = reinterpret_cast<const uint4*>(w + (size_t)e * per_expert);
  const size_t n16 = per_expert / 8;
  float m = 0.0f;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += (size_t)gridDim.x * blockDim.x) {
    const uint4 q = __ldg(src + i);
    const uint32_t ww[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) m = fmaxf(m, fmaxf(fabsf(bf16_lo(ww[k])), fabsf(bf16_hi(ww[k]))));
  }
  m = warp_max(m);
  __shared__ float red[8];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float mm = 0.0f;
    for (int i = 0; i < 8; ++i) mm = fmaxf(mm, red[i]);
    atomicMax(&amax_bits[e], __float_as_uint(mm));  // non-negative floats order like their bits
  }
}

__device__ __forceinline__ int w13_internal_row(int n, int N) {
  // caller row n of [gate (I rows); up (I rows)] -> internal row where chunk f
  // of 128 rows is [gate rows 64f..64f+63, up rows 64f..64f+63], so one
  // 128-column MMA tile holds matching gate and up features
  const int I = N / 2;
  if (n < I) return (n >> 6) * 128 + (n & 63);
  const int u = n - I;
  return (u >> 6) * 128 + 64 + (u & 63);
}

// One warp per (expert, row): block scales and codes of the row with the
// expert's global scale, written into the weights' pair-tile layout.
__global__ void __launch_bounds__(256) weight_quant_kernel(const __nv_bfloat16* __restrict__ w, int E, int N,
                                                          int Kd, int Kpad, int interleave,
                                                          const uint32_t* __restrict__ amax_bits,
                                                          uint8_t* __restrict__ codes, uint8_t* __restrict__ sf,
                                                          float* __restrict__ gs_out) {
  const size_t gw = (size_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (gw >= (size_t)E * N) return;
  const int e = (int)(gw / N), n = (int)(gw % N);
  const float gs = nvfp4_global_scale(__uint_as_float(amax_bits[e]));
  const int irow = e * N + (interleave ? w13_internal_row(n, N) : n);
  const uint4* src = reinterpret_cast<const uint4*>(w + ((size_t)e * N + n) * Kd);
  const int nblk = Kd / SF_VEC;
  for (int b = lane; b < nblk; b += 32) {
    float v[16];
    bf16x16_to_f32(__ldg(src + 2 * b), __ldg(src + 2 * b + 1), v);
    uint2 packed;
    const uint32_t s = nvfp4_quant_block16(v, gs, packed);
    *reinterpret_cast<uint2*>(codes + wpair_offset(irow, 8 * b, Kpad / 2)) = packed;
    sf[wpair_sf_offset(irow, b, Kpad / SF_VEC)] = (uint8_t)s;
  }
  if (n == 0 && lane == 0) gs_out[e] = gs;
}

// Copy rows from an internal operand layout to canonical row-major arrays.
// mode 0: internal row = row_map[i * map_stride] (expanded activations /
//         intermediate);
// mode 1: internal row = i (weights in caller order);
// mode 2: internal row = w13 interleave of i within its expert (E_rows rows per expert).
// pair: the operand is in the weights' pair-tile layout.
__global__ void __launch_bounds__(256) export_rows_kernel(const uint8_t* __restrict__ codes,
                                                         const uint8_t* __restrict__ sf,
                                                         const float* __restrict__ gs_rows, int n_rows, int Kd,
                                                         int Kpad, const int32_t* __restrict__ row_map,
                                                         int map_stride, int mode, int E_rows, int pair,
                                                         uint8_t* __restrict__ out_codes,
                                                         uint8_t* __restrict__ out_sf, float* __restrict__ out_gs) {
  const int i = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (i >= n_rows) return;
  int r;
  if (mode == 0) r = row_map[(size_t)i * map_stride];
  else if (mode == 1) r = i;
  else r = (i / E_rows) * E_rows + w13_internal_row(i % E_rows, E_rows);
  if (out_codes)
    for (int b = lane; b < Kd / 2; b += 32)
      out_codes[(size_t)i * (Kd / 2) + b] = codes[pair ? wpair_offset(r, b, Kpad / 2) : operand_offset(r, b, Kpad / 2)];
  if (out_sf)
    for (int b = lane; b < Kd / SF_VEC; b += 32)
      out_sf[(size_t)i * (Kd / SF_VEC) + b] =
          sf[pair ? wpair_sf_offset(r, b, Kpad / SF_VEC) : sf_atom_offset(r, b, Kpad / SF_VEC)];
  if (out_gs && gs_rows && lane == 0) out_gs[i] = gs_rows[r];
}

__global__ void convert_kernel(const float* __restrict__ in, uint8_t* __restrict__ e2m1,
                               uint8_t* __restrict__ e4m3, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const float v = in[i];
    if (e2m1) e2m1[i] = (uint8_t)(cvt_e2m1x2(v, 0.0f) & 0xF);
    if (e4m3) e4m3[i] = (uint8_t)cvt_e4m3(v);
  }
}

// Row-major codes [rows, row_bytes] -> tiled operand layout (tests).
__global__ void codes_to_tiled_kernel(const uint8_t* __restrict__ codes, int rows, int row_bytes,
                                      uint8_t* __restrict__ tiled) {
  const int64_t n = (int64_t)rows * row_bytes;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    tiled[operand_offset(i / row_bytes, (int)(i % row_bytes), row_bytes)] = codes[i];
}

__global__ void sf_to_atoms_kernel(const uint8_t* __restrict__ sf, int rows, int k16, uint8_t* __restrict__ atoms) {
  const int64_t n = (int64_t)rows * k16;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int r = (int)(i / k16), b = (int)(i % k16);
    atoms[sf_atom_offset(r, b, k16)] = sf[i];
  }
}

// The shared expert's contribution to 8 consecutive outputs: the FP32 routed
// sums v[0..8) become fl32(fl32(v + shared) * scale) (scale 1: the sum; 0.5:
// the average), from the shared expert's bf16 output word `sh` (8 values).
__device__ __forceinline__ void add_shared8(float (&v)[8], const uint4& sh, float scale) {
  const uint32_t w[4] = {sh.x, sh.y, sh.z, sh.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    v[2 * q] = __fmul_rn(__fadd_rn(v[2 * q], bf16_lo(w[q])), scale);
    v[2 * q + 1] = __fmul_rn(__fadd_rn(v[2 * q + 1], bf16_hi(w[q])), scale);
  }
}

// out = bf16_rn(acc), 8 elements per thread; with a shared expert,
// bf16_rn(fl32(acc + shared) * scale).
__global__ void __launch_bounds__(256) finalize_atomic_kernel(const float* __restrict__ acc,
                                                             const uint16_t* __restrict__ shared, float shared_scale,
                                                             __nv_bfloat16* __restrict__ out, size_t n8) {
  pdl_trigger();
  pdl_wait();
  // FIN_ILP independent 8-float chunks per thread per pass (coalesced: chunk
  // q of a pass is blockDim.x apart), all loads issued before any store.
  constexpr int FIN_ILP = 4;
  const size_t step = (size_t)gridDim.x * blockDim.x * FIN_ILP;
  for (size_t base = (size_t)blockIdx.x * blockDim.x * FIN_ILP + threadIdx.x; base < n8; base += step) {
    float4 a[FIN_ILP], b[FIN_ILP];
#pragma unroll
    for (int q = 0; q < FIN_ILP; ++q) {
      const size_t i = base + (size_t)q * blockDim.x;
      if (i < n8) {
        a[q] = reinterpret_cast<const float4*>(acc)[2 * i];
        b[q] = reinterpret_cast<const float4*>(acc)[2 * i + 1];
      }
    }
#pragma unroll
    for (int q = 0; q < FIN_ILP; ++q) {
      const size_t i = base + (size_t)q * blockDim.x;
      if (i < n8) {
        float v[8] = {a[q].x, a[q].y, a[q].z, a[q].w, b[q].x, b[q].y, b[q].z, b[q].w};
        if (shared) add_shared8(v, reinterpret_cast<const uint4*>(shared)[i], shared_scale);
        reinterpret_cast<uint4*>(out)[i] = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                                                      pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
      }
    }
  }
}

// out[t][n] = bf16_rn(sum over j ascending of fl32(w[t][j] * y[t*K+j][n])),
// y the bf16 rows the w2 epilogue stored; FP32 partial sums, the first term
// taken as is.  One CTA per token row at a time, 8 columns per thread: the K
// rows' 16-byte words are all loaded before the sum starts.
constexpr int FIN_MAX_K = 16;
// KMAX bounds K at compile time: the K rows' words live in registers, so a
// small bound (top-k <= 8) leaves room for more resident CTAs.
// With a shared expert, its bf16 row t is added to the FP32 sum and the
// result scaled (add_shared8) before the rounding.
template <int KMAX>
__global__ void __launch_bounds__(256, KMAX <= 8 ? 4 : 2) finalize_ordered_kernel(const uint16_t* __restrict__ ybuf,
                                                                                  const float* __restrict__ topk_w,
                                                                                  const uint16_t* __restrict__ shared,
                                                                                  float shared_scale,
                                                                                  __nv_bfloat16* __restrict__ out, int T,
                                                                                  int H, int K) {
  pdl_trigger();
  pdl_wait();
  const int h8 = H / 8;
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    const uint4* yt = reinterpret_cast<const uint4*>(ybuf) + (size_t)t * K * h8;
    const float* wt = topk_w + (size_t)t * K;
    for (int c = threadIdx.x; c < h8; c += blockDim.x) {
      uint4 y[KMAX];
#pragma unroll
      for (int j = 0; j < KMAX; ++j)
        if (j < K) y[j] = __ldcs(yt + (size_t)j * h8 + c);  // read once: streaming
      float s[8];
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        if (j < K) {
          const float w = __ldg(wt + j);
          const uint32_t yw[4] = {y[j].x, y[j].y, y[j].z, y[j].w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float p0 = __fmul_rn(w, bf16_lo(yw[q])), p1 = __fmul_rn(w, bf16_hi(yw[q]));
            s[2 * q] = j == 0 ? p0 : __fadd_rn(s[2 * q], p0);
            s[2 * q + 1] = j == 0 ? p1 : __fadd_rn(s[2 * q + 1], p1);
          }
        }
      }
      if (shared) add_shared8(s, reinterpret_cast<const uint4*>(shared + (size_t)t * H)[c], shared_scale);
      reinterpret_cast<uint4*>(out + (size_t)t * H)[c] =
          make_uint4(pack_bf16x2(s[0], s[1]), pack_bf16x2(s[2], s[3]), pack_bf16x2(s[4], s[5]), pack_bf16x2(s[6], s[7]));
    }
  }
}

// The shared expert's tile list: rows 0..T-1 of expert 0 in 128-row tiles.
__global__ void shared_tiles_kernel(int T, int4* __restrict__ tiles, int32_t* __restrict__ num_tiles) {
  const int n = (T + 127) / 128;
  for (int i = threadIdx.x; i < n; i += blockDim.x) tiles[i] = make_int4(0, 128 * i, min(128, T - 128 * i), 128 * i);
  if (threadIdx.x == 0) *num_tiles = n;
}

int grid_for(size_t n, int per_block, int cap = 152 * 16) {
  size_t g = (n + per_block - 1) / per_block;
  if (g < 1) g = 1;
  if (g > (size_t)cap) g = cap;
  return (int)g;
}

}  // namespace

cudaError_t launch_act_quant(const void* x, int T, int H, int K, const int32_t* pad_row_of_src, uint8_t* a_codes,
                             uint8_t* a_sf, float* gs_rows, const float* static_gs, cudaStream_t s) {
  return launch_k(act_quant_kernel, dim3((T + 7) / 8), dim3(256), 0, s, true,
                  reinterpret_cast<const __nv_bfloat16*>(x), T, H, K, pad_row_of_src, a_codes, a_sf, gs_rows,
                  static_gs);
}

cudaError_t launch_weight_amax(const void* w, int E, int N, int Kd, uint32_t* amax_bits, cudaStream_t s) {
  const size_t per = (size_t)N * Kd;
  dim3 grid(grid_for(per / 8, 256 * 8, 64), E);
  weight_amax_kernel<<<grid, 256, 0, s>>>(reinterpret_cast<const __nv_bfloat16*>(w), per, amax_bits);
  return cudaGetLastError();
}

cudaError_t launch_weight_quant(const void* w, int E, int N, int Kd, int Kpad, int interleave,
                                const uint32_t* amax_bits, uint8_t* codes, uint8_t* sf, float* gs, cudaStream_t s) {
  const size_t warps = (size_t)E * N;
  weight_quant_kernel<<<(unsigned)((warps + 7) / 8), 256, 0, s>>>(reinterpret_cast<const __nv_bfloat16*>(w), E, N, Kd,
                                                                  Kpad, interleave, amax_bits, codes, sf, gs);
  return cudaGetLastError();
}

cudaError_t launch_export_rows(const uint8_t* codes, const uint8_t* sf, const float* gs_rows, int n_rows, int Kd,
                               int Kpad, const int32_t* row_map, int map_stride, int row_map_mode, int E_rows,
                               int pair, uint8_t* out_codes, uint8_t* out_sf, float* out_gs, cudaStream_t s) {
  if (n_rows <= 0) return cudaSuccess;
  export_rows_kernel<<<(n_rows + 7) / 8, 256, 0, s>>>(codes, sf, gs_rows, n_rows, Kd, Kpad, row_map, map_stride,
                                                      row_map_mode, E_rows, pair, out_codes, out_sf, out_gs);
  return cudaGetLastError();
}

cudaError_t launch_convert(const float* in, uint8_t* e2m1, uint8_t* e4m3, int64_t n, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  convert_kernel<<<grid_for((size_t)n, 256), 256, 0, s>>>(in, e2m1, e4m3, n);
  return cudaGetLastError();
}

cudaError_t launch_codes_to_tiled(const uint8_t* codes, int rows, int row_bytes, uint8_t* tiled, cudaStream_t s) {
  codes_to_tiled_kernel<<<grid_for((size_t)rows * row_bytes, 256), 256, 0, s>>>(codes, rows, row_bytes, tiled);
  return cudaGetLastError();
}

cudaError_t launch_sf_to_atoms(const uint8_t* sf, int rows, int k16, uint8_t* atoms, cudaStream_t s) {
  sf_to_atoms_kernel<<<grid_for((size_t)rows * k16, 256), 256, 0, s>>>(sf, rows, k16, atoms);
  return cudaGetLastError();
}

cudaError_t launch_requant_rows(const float* hbuf, float* row_amax, const int32_t* row_map,
                                const int32_t* topk_ids, int K, int n_rows, int I, int i_pad, uint8_t* h_codes,
                                float* h_gs, const RequantAllExperts* all, int* status, cudaStream_t s) {
  if (all && !topk_ids) return cudaErrorInvalidValue;
  const RequantAllExperts a = all ? *all : RequantAllExperts{};
  return launch_k(requant_rows_kernel, dim3((n_rows + 7) / 8), dim3(256), 0, s, true, hbuf, row_amax, row_map,
                  topk_ids, K, n_rows, I, i_pad, h_codes, h_gs, a, all ? 1 : 0, status);
}

cudaError_t launch_finalize_atomic(const float* out_acc, const uint16_t* shared, float shared_scale, void* out, int T,
                                   int H, cudaStream_t s) {
  const size_t n8 = (size_t)T * H / 8;
  // after the join of the shared expert's stream: plain stream order
  return launch_k(finalize_atomic_kernel, dim3(grid_for(n8, 256 * 4)), dim3(256), 0, s, !shared, out_acc, shared,
                  shared_scale, reinterpret_cast<__nv_bfloat16*>(out), n8);
}

cudaError_t launch_finalize_ordered(const uint16_t* ybuf, const float* topk_w, const uint16_t* shared,
                                    float shared_scale, void* out, int T, int H, int K, cudaStream_t s) {
  if (K > FIN_MAX_K || H % 8) return cudaErrorInvalidValue;
  // one token row per CTA and pass; plain stream order after a shared join
  if (K <= 8)
    return launch_k(finalize_ordered_kernel<8>, dim3(std::min(T, 152 * 8)), dim3(256), 0, s, !shared, ybuf, topk_w,
                    shared, shared_scale, reinterpret_cast<__nv_bfloat16*>(out), T, H, K);
  return launch_k(finalize_ordered_kernel<FIN_MAX_K>, dim3(std::min(T, 152 * 8)), dim3(256), 0, s, !shared, ybuf,
                  topk_w, shared, shared_scale, reinterpret_cast<__nv_bfloat16*>(out), T, H, K);
}

cudaError_t launch_shared_tiles(int T, int4* tiles, int32_t* num_tiles, cudaStream_t s) {
  if (T <= 0) return cudaErrorInvalidValue;
  // first kernel of the shared stream after the fork: ordinary stream order
  return launch_k(shared_tiles_kernel, dim3(1), dim3(128), 0, s, false, T, tiles, num_tiles);
}

}  // namespace moe
