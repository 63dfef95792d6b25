// kernels_gemm.cu - block-scaled FP4 grouped GEMMs of the routed-MoE forward
// on the sm_103a tensor cores (tcgen05.mma kind::mxf4nvf4, E2M1 operands with
// UE4M3 scales per 16 elements, FP32 accumulators in tensor memory).
//
// One CTA computes one 128-row x 256-column tile of one expert:
//   warp 0      TMA producer: A rows (only the tile's valid rows), B rows,
//               and both block-scale tiles into a 4-stage shared-memory ring;
//   warp 1      tensor-memory allocation and the single MMA-issuing thread:
//               block scales shared -> tensor memory (tcgen05.cp), then four
//               K=64 MMAs per 256-element stage;
//   warps 2-5   epilogue: one accumulator row (tensor-memory lane) per thread.
//
// Epilogues:
//   w13  the 256 columns are 128 gate and the matching 128 up features
//        (the weights are stored interleaved in chunks of 128), so each
//        thread forms SwiGLU for its row locally.  The row's absolute maximum
//        over all I features is combined across the I/128 CTAs of a thread
//        block cluster through distributed shared memory, and each CTA then
//        requantizes its 128 features with the row's global scale - the
//        per-row NVFP4 input of the w2 GEMM, written without a round trip of
//        the FP32 intermediate through global memory.
//   w2   y = acc / (gs_h * gs_w2), scaled by the token's top-k weight and
//        added into the FP32 output accumulator (atomic mode), or stored per
//        (token, slot) for the fixed-order finalize (ordered mode).
//   plain FP32 store (tests).
//
// The activation (routing, expandInputRows, activation, finalize) fusion
// around the expert GEMMs follows "SM10X Command-A-Plus decode 2.3x faster,
// BCG capture memory -78%" (Motivation); the per-token scales follow "CuTe
// DSL backend gets per-token NVFP4 online quantization and reload"
// (Implementation item 2).
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int STAGES = 4;
constexpr int A_STAGE = TILE_M * 128;        // 16 KB: 128 rows x 128 bytes
constexpr int B_STAGE = TILE_N * 128;        // 32 KB: 256 rows x 128 bytes
constexpr int SFA_STAGE = 4 * SF_ATOM_BYTES; // 2 KB: 128 rows x 16 scales
constexpr int SFB_STAGE = 8 * SF_ATOM_BYTES; // 4 KB: 256 rows x 16 scales
constexpr int A_BOX_ROWS = 32;
constexpr int TMEM_COLS = 512;
constexpr int TMEM_SF_BASE = 256;            // accumulator in columns [0, 256)
constexpr int TMEM_SF_STAGE = 48;            // 16 columns SFA + 32 columns SFB per stage
constexpr uint32_t IDESC = idesc_fp4(TILE_M, TILE_N);
constexpr int THREADS = 192;

enum Mode { MODE_W13 = 0, MODE_W2_ATOMIC = 1, MODE_W2_ORDERED = 2, MODE_PLAIN = 3 };

struct Smem {
  uint8_t a[STAGES][A_STAGE];
  uint8_t b[STAGES][B_STAGE];
  uint8_t sfa[STAGES][SFA_STAGE];
  uint8_t sfb[STAGES][SFB_STAGE];
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t acc_full;
  uint32_t tmem_base;
  int abort_flag;
  float part_amax[TILE_M];
};

constexpr int SMEM_BYTES = (int)sizeof(Smem) + 1024;  // + alignment slack

__device__ __forceinline__ float swiglu(float g_acc, float u_acc, float alpha) {
  const float g = __fmul_rn(g_acc, alpha);
  const float u = __fmul_rn(u_acc, alpha);
  return __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, expf(-g))), u);
}

__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

template <int MODE>
__global__ void __launch_bounds__(THREADS, 1) gemm_fp4_kernel(const __grid_constant__ CUtensorMap tmA,
                                                             const __grid_constant__ CUtensorMap tmB, GemmArgs p) {
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mt = blockIdx.y;
  int4 tile;
  if (MODE == MODE_PLAIN) {
    tile = make_int4(0, mt * TILE_M, TILE_M, 0);
  } else {
    if (mt >= *p.num_tiles) return;  // same decision for every CTA of a cluster
    tile = p.tiles[mt];
  }
  const int e = tile.x, row0 = tile.y, valid = tile.z;
  const int nb = blockIdx.x;  // w13: feature chunk (= cluster rank); w2 / plain: 256-column tile
  const int brow0 = (MODE == MODE_PLAIN) ? nb * TILE_N : e * p.b_rows_per_expert + nb * TILE_N;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    mbar_init(&sm.acc_full, 1);
    sm.abort_flag = 0;
    fence_mbarrier_init();
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const int KS = p.k_stages;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      const int a_boxes = (valid + A_BOX_ROWS - 1) / A_BOX_ROWS;
      const uint32_t bytes = a_boxes * A_BOX_ROWS * 128 + B_STAGE + SFA_STAGE + SFB_STAGE;
      const uint64_t pol = policy_evict_first();
      const uint64_t pol_a = policy_evict_last();
      const uint8_t* sfa_src = p.a_sf + ((size_t)(row0 >> 7) * p.kblocks) * SF_ATOM_BYTES;
      const uint8_t* sfb_src0 = p.b_sf + ((size_t)(brow0 >> 7) * p.kblocks) * SF_ATOM_BYTES;
      const uint8_t* sfb_src1 = sfb_src0 + (size_t)p.kblocks * SF_ATOM_BYTES;
      int issued = 0;
      for (int ks = 0; ks < KS; ++ks) {
        const int s = ks % STAGES;
        const uint32_t round = ks / STAGES;
        if (!mbar_wait_bounded(&sm.empty[s], (round & 1) ^ 1, &sm.abort_flag)) {
          sm.abort_flag = 1;
          report_device_error(p.status, DEV_ERR_TIMEOUT);
          break;
        }
        issued = ks + 1;
        mbar_arrive_expect_tx(&sm.full[s], bytes);
        for (int i = 0; i < a_boxes; ++i)
          tma_load_2d(&sm.a[s][i * A_BOX_ROWS * 128], &tmA, &sm.full[s], ks * 128, row0 + i * A_BOX_ROWS, pol_a);
        tma_load_2d(&sm.b[s][0], &tmB, &sm.full[s], ks * 128, brow0, pol);
        bulk_load(&sm.sfa[s][0], sfa_src + (size_t)ks * SFA_STAGE, SFA_STAGE, &sm.full[s]);
        bulk_load(&sm.sfb[s][0], sfb_src0 + (size_t)ks * SFA_STAGE, SFA_STAGE, &sm.full[s]);
        bulk_load(&sm.sfb[s][SFA_STAGE], sfb_src1 + (size_t)ks * SFA_STAGE, SFA_STAGE, &sm.full[s]);
      }
      if (sm.abort_flag) {
        // Unwinding: let the copies already issued land before the CTA's
        // shared memory is released (bounded, no early exit).
        for (int ks = issued - STAGES < 0 ? 0 : issued - STAGES; ks < issued; ++ks)
          mbar_wait_bounded(&sm.full[ks % STAGES], (ks / STAGES) & 1, nullptr, 1000000000ull);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      bool ok = true;
      for (int ks = 0; ks < KS; ++ks) {
        const int s = ks % STAGES;
        const uint32_t round = ks / STAGES;
        if (!mbar_wait_bounded(&sm.full[s], round & 1, &sm.abort_flag)) {
          sm.abort_flag = 1;
          report_device_error(p.status, DEV_ERR_TIMEOUT);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sfa_t = tmem + TMEM_SF_BASE + s * TMEM_SF_STAGE;
        const uint32_t sfb_t = sfa_t + 16;
#pragma unroll
        for (int kb = 0; kb < 4; ++kb) {
          tc_copy_sf(sfa_t + kb * 4, smem_desc_sf(smem_u32(&sm.sfa[s][kb * SF_ATOM_BYTES])));
          tc_copy_sf(sfb_t + kb * 8, smem_desc_sf(smem_u32(&sm.sfb[s][kb * SF_ATOM_BYTES])));
          tc_copy_sf(sfb_t + kb * 8 + 4, smem_desc_sf(smem_u32(&sm.sfb[s][SFA_STAGE + kb * SF_ATOM_BYTES])));
        }
        const uint32_t a_base = smem_u32(&sm.a[s][0]);
        const uint32_t b_base = smem_u32(&sm.b[s][0]);
#pragma unroll
        for (int kb = 0; kb < 4; ++kb) {
          tc_mma_fp4(tmem, smem_desc_sw128(a_base + kb * 32), smem_desc_sw128(b_base + kb * 32), IDESC,
                     sfa_t + kb * 4, sfb_t + kb * 8, (ks | kb) != 0);
        }
        tc_commit(&sm.empty[s]);
      }
      // Signal the epilogue even after an abort so that it does not wait for
      // the full timeout; it checks the abort flag.
      tc_commit(&sm.acc_full);
      (void)ok;
    }
    __syncwarp();
  }

  // ---------------- epilogue (warps 2..5) ----------------
  const bool epi = warp >= 2;
  const int quarter = warp & 3;                 // tensor-memory lanes [32q, 32q+32)
  const int m = quarter * 32 + lane;            // accumulator row of this thread
  const bool row_ok = m < valid;
  const int prow = row0 + m;
  const uint32_t trow = tmem + ((uint32_t)(quarter * 32) << 16);
  bool acc_ready = false;
  if (epi) {
    // No early exit here: the MMA thread always commits acc_full, and tensor
    // memory must not be released before the MMAs already issued are done.
    acc_ready = mbar_wait_bounded(&sm.acc_full, 0, nullptr);
    if (!acc_ready) report_device_error(p.status, DEV_ERR_TIMEOUT);
    acc_ready = acc_ready && !sm.abort_flag;
    tc_fence_after();
  }

  if constexpr (MODE == MODE_W13) {
    const float alpha = row_ok ? __fdiv_rn(1.0f, __fmul_rn(p.gs_rows[prow], p.gs_w[e])) : 0.0f;
    if (epi) {
      float amax = 0.0f;
      if (acc_ready) {
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          float g[16], u[16];
          tmem_ld16(trow + 16 * c, g);
          tmem_ld16(trow + 128 + 16 * c, u);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(swiglu(g[i], u[i], alpha)));
        }
      }
      sm.part_amax[m] = row_ok ? amax : 0.0f;
    }
    __syncwarp();
    cluster_sync_all();  // every CTA's partial row maxima are visible
    if (epi) {
      const uint32_t nranks = gridDim.x;
      float amax_row = 0.0f;
      for (uint32_t r = 0; r < nranks; ++r) amax_row = fmaxf(amax_row, ld_shared_cluster_f32(&sm.part_amax[m], r));
      const float gs_h = nvfp4_global_scale(amax_row);
      if (acc_ready) {
        const int k16_row = p.i_pad / SF_VEC;
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          float g[16], u[16], h[16];
          tmem_ld16(trow + 16 * c, g);
          tmem_ld16(trow + 128 + 16 * c, u);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) h[i] = swiglu(g[i], u[i], alpha);
          uint2 packed;
          const uint32_t sf = nvfp4_quant_block16(h, gs_h, packed);
          const int k = nb * 128 + 16 * c;  // feature index of this block
          if (row_ok) {
            *reinterpret_cast<uint2*>(p.h_codes + (size_t)prow * (p.i_pad / 2) + k / 2) = packed;
            p.h_sf[sf_atom_offset(prow, k / SF_VEC, k16_row)] = (uint8_t)sf;
          }
        }
      }
      if (row_ok && nb == 0) p.h_gs[prow] = gs_h;
    }
    __syncwarp();
    cluster_sync_all();  // peers are done reading this CTA's shared memory
  } else if constexpr (MODE == MODE_W2_ATOMIC || MODE == MODE_W2_ORDERED) {
    if (epi && acc_ready) {
      int src = 0;
      float alpha = 0.0f, wj = 0.0f;
      if (row_ok) {
        src = p.src_of_padrow[prow];
        alpha = __fdiv_rn(1.0f, __fmul_rn(p.gs_rows[prow], p.gs_w[e]));
        wj = p.topk_w[src];
      }
      const int t = src / p.top_k;
      const int n0 = nb * TILE_N;
#pragma unroll 1
      for (int c = 0; c < 16; ++c) {
        float a[16];
        tmem_ld16(trow + 16 * c, a);
        tmem_ld_wait();
        if (row_ok) {
          if constexpr (MODE == MODE_W2_ATOMIC) {
            float* dst = p.out_acc + (size_t)t * p.hidden + n0 + 16 * c;
#pragma unroll
            for (int i = 0; i < 16; i += 4)
              red_add_v4(dst + i, __fmul_rn(wj, __fmul_rn(a[i], alpha)), __fmul_rn(wj, __fmul_rn(a[i + 1], alpha)),
                         __fmul_rn(wj, __fmul_rn(a[i + 2], alpha)), __fmul_rn(wj, __fmul_rn(a[i + 3], alpha)));
          } else {
            float4* dst = reinterpret_cast<float4*>(p.ybuf + (size_t)src * p.hidden + n0 + 16 * c);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              dst[i] = make_float4(__fmul_rn(a[4 * i], alpha), __fmul_rn(a[4 * i + 1], alpha),
                                   __fmul_rn(a[4 * i + 2], alpha), __fmul_rn(a[4 * i + 3], alpha));
          }
        }
      }
    }
  } else {  // MODE_PLAIN
    if (epi && acc_ready) {
#pragma unroll 1
      for (int c = 0; c < 16; ++c) {
        float a[16];
        tmem_ld16(trow + 16 * c, a);
        tmem_ld_wait();
        float4* dst = reinterpret_cast<float4*>(p.d + (size_t)prow * p.ldd + nb * TILE_N + 16 * c);
#pragma unroll
        for (int i = 0; i < 4; ++i) dst[i] = make_float4(a[4 * i], a[4 * i + 1], a[4 * i + 2], a[4 * i + 3]);
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

template <int MODE>
cudaError_t set_attrs() {
  cudaError_t err = cudaFuncSetAttribute(gemm_fp4_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         SMEM_BYTES);
  if (err != cudaSuccess) return err;
  if (MODE == MODE_W13) {
    err = cudaFuncSetAttribute(gemm_fp4_kernel<MODE>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  }
  return err;
}

template <int MODE>
cudaError_t launch(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& a, dim3 grid, int cluster_x,
                   cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  if (cluster_x > 0) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster_x;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, gemm_fp4_kernel<MODE>, tmA, tmB, a);
}

}  // namespace

int gemm_smem_bytes() { return SMEM_BYTES; }

cudaError_t gemm_setup_attributes() {
  cudaError_t e;
  if ((e = set_attrs<MODE_W13>()) != cudaSuccess) return e;
  if ((e = set_attrs<MODE_W2_ATOMIC>()) != cudaSuccess) return e;
  if ((e = set_attrs<MODE_W2_ORDERED>()) != cudaSuccess) return e;
  return set_attrs<MODE_PLAIN>();
}

cudaError_t launch_gemm_w13(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& a, int n_chunks,
                            int tile_bound, cudaStream_t s) {
  return launch<MODE_W13>(tmA, tmB, a, dim3(n_chunks, tile_bound, 1), n_chunks, s);
}

cudaError_t launch_gemm_w2(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& a, int n_tiles,
                           int tile_bound, bool ordered, cudaStream_t s) {
  if (ordered) return launch<MODE_W2_ORDERED>(tmA, tmB, a, dim3(n_tiles, tile_bound, 1), 0, s);
  return launch<MODE_W2_ATOMIC>(tmA, tmB, a, dim3(n_tiles, tile_bound, 1), 0, s);
}

cudaError_t launch_gemm_plain(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& a, int n_tiles,
                              int m_tiles, cudaStream_t s) {
  return launch<MODE_PLAIN>(tmA, tmB, a, dim3(n_tiles, m_tiles, 1), 0, s);
}

}  // namespace moe
