// kernels_gemm.cu - block-scaled FP4 grouped GEMMs of the routed-MoE forward
// on the sm_103a tensor cores (tcgen05.mma kind::mxf4nvf4, E2M1 operands with
// UE4M3 scales per 16 elements, FP32 accumulators in tensor memory).
//
// Persistent kernels.  A work unit is one 128-row x 128-column tile of one
// expert; the expert GEMMs take units in pairs of adjacent 128-column tiles
// and compute a pair as one 128 x 256 tile.  Each CTA (w2, plain) or cluster
// (w13) walks a static list.
//   warp 0      producer: per 256-element K stage, bulk copies into a
//               STAGES-deep shared-memory ring - the activation tile's
//               scales plus its valid rows, and the weight tile(s) (a pair
//               is staged as [scales a | scales b | codes a | codes b] so its
//               256 rows of pre-swizzled codes are contiguous) - running
//               ahead across unit boundaries;
//   warp 1      tensor-memory allocation and the single MMA-issuing thread:
//               four K=64 MMAs per 256-element stage: N = 256 into the one
//               256-column accumulator (pairs), or N = 128 into one of two
//               128-column buffers (plain);
//   warps 2-9   epilogue, two warps per tensor-memory lane quadrant: warp w
//               reads lanes [32 (w % 4), +32) and takes column half
//               (w - 2) / 4 of every accumulator, one row per thread;
//   warp 10     per stage, the block scales shared -> tensor memory
//               (tcgen05.cp), committed to a barrier the MMA thread waits
//               on, so that the copies' issue runs ahead of the MMAs.
// With two accumulator buffers (plain) the epilogue drains unit u while the
// tensor cores compute unit u+1; with one 256-column accumulator (pairs) the
// tensor cores wait only for the epilogue's tensor-memory reads (each thread
// moves its 128 columns to registers and releases the accumulator before any
// arithmetic), while the ring keeps streaming weights.
//
// Epilogues:
//   w13  a unit's 128 columns are 64 gate features and the matching 64 up
//        features (weights stored interleaved in chunks of 64), so a thread
//        forms SwiGLU for its row locally.  A CTA owns 128 features (two
//        units) of an m-tile and keeps their SwiGLU values in registers.
//        The row's absolute maximum over all I features is combined across
//        the I/128 CTAs of a thread-block cluster: every CTA stores its partial
//        maximum (a non-negative float, so bit 31 is free) as one 32-bit word
//        into every peer's shared memory; successive m-tiles alternate
//        between two slot buffers, and bit 31 flips between successive uses
//        of a buffer, so each thread polls its own row's slots until every
//        tag matches - no barrier or fence on the path.
//        Each CTA then requantizes its 128 features with the row's global
//        scale: the per-row NVFP4 input of the w2 GEMM, written without a
//        round trip of the FP32 intermediate through HBM.
//   w2   y = acc / (gs_h * gs_w2) scaled by the token's top-k weight and
//        added into the FP32 output accumulator (atomic mode), or rounded to
//        bf16 and stored per (token, slot) for the fixed-order finalize
//        (ordered mode: half the bytes of an FP32 row, and plain stores where
//        the atomic mode's reductions at large batches saturate L2).
//   plain FP32 store (tests).
//
// The fusion of routing, expandInputRows, activation and finalize around the
// expert GEMMs follows "SM10X Command-A-Plus decode 2.3x faster, BCG capture
// memory -78%" (Motivation); the per-token scales follow "CuTe DSL backend
// gets per-token NVFP4 online quantization and reload" (Implementation
// item 2).
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int B_SLOT = OPERAND_TILE_BYTES;   // 18 KB: [scales | 128 rows x 128 bytes]
constexpr int MAX_STAGES = 8;
// Activation rows reserved per stage: 128, or 64 for small batches.  The MMA
// always reads 128 rows; with 64 reserved, rows 64..127 read the next stages'
// data (or the tail pad after the last stage) - in bounds, and their results
// are never used because such tiles have at most 64 valid rows.
constexpr int TMEM_COLS = 512;
constexpr int TMEM_SF_BASE = 2 * TILE_N;     // two accumulator buffers in columns [0, 256)
constexpr int TMEM_SF_STAGE = 32;            // 16 columns SFA + 16 columns SFB per stage
constexpr uint32_t IDESC = idesc_fp4(TILE_M, TILE_N);
// Column-pair kernels (w13): one 128 x 256 accumulator in columns [0, 256)
// fed by N = 256 MMAs over both 128-row weight tiles of a pair; the B scale
// factors of a K block take 8 columns (rows 128..255 after rows 0..127).
constexpr int TMEM_SF_STAGE_PAIR = 48;       // 16 columns SFA + 32 columns SFB per stage
constexpr uint32_t IDESC_PAIR = idesc_fp4(TILE_M, 2 * TILE_N);
constexpr int MAX_STAGES_PAIR = 5;
constexpr int EPI_WARPS = 8;
// warp 0 producer, warp 1 MMA issuer, warps 2..9 epilogue, warp 10 the block
// scales' copies to tensor memory
constexpr int SF_WARP = 2 + EPI_WARPS;
constexpr int THREADS = 64 + 32 * EPI_WARPS + 32;
constexpr int HALF_MAX_BYTES = 2 * 2 * TILE_M * 4;  // w13: per-half row maxima, two m-tile buffers
constexpr int CTRL_BYTES = 384;
// Ordered w2 epilogue: each epilogue warp stages its 32 rows, 64 columns
// (128 bytes of bf16) at a time, in shared memory with a 16-byte pad per row
// (conflict-free 16-byte writes of one row per lane, reads of one row per 8
// lanes), so that every store instruction writes four whole 128-byte row
// segments instead of 32 scattered 16-byte pieces.
constexpr int EPI_ROW_STRIDE = 144;
constexpr int EPI_STAGE_BYTES = 8 * 32 * EPI_ROW_STRIDE;
constexpr int MAX_SMEM = 232448;
static_assert(TMEM_SF_BASE + MAX_STAGES * TMEM_SF_STAGE <= TMEM_COLS, "tensor memory overflow");
static_assert(TMEM_SF_BASE + MAX_STAGES_PAIR * TMEM_SF_STAGE_PAIR <= TMEM_COLS, "tensor memory overflow");

// MODE_W13S: the small-batch w13 GEMM without clusters - its epilogue writes
// the FP32 SwiGLU rows and folds each row's absolute maximum into a global
// word; a separate kernel requantizes (the same arithmetic as MODE_W13's
// fused requantization).
enum Mode { MODE_W13 = 0, MODE_W2_ATOMIC = 1, MODE_W2_ORDERED = 2, MODE_PLAIN = 3, MODE_W13S = 4 };

// The expert GEMMs take their 128-column units in pairs (N = 256 MMAs); the
// plain GEMM (tests) does not.  The one definition the kernel's shared-memory
// layout and the host's launch size both use.
__host__ __device__ constexpr bool pair_mode(int mode) { return mode != MODE_PLAIN; }

constexpr int UNIT_QUEUE = 4;  // dynamic schedule: units published ahead by the producer

struct Ctrl {
  uint64_t full[MAX_STAGES];
  uint64_t empty[MAX_STAGES];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t a_full;  // resident activations loaded (resident-A kernels)
  // dynamic schedule: unit n of the CTA is q_unit[n % UNIT_QUEUE], published
  // by the producer (q_full) and released by the MMA thread and the 8
  // epilogue warps (q_empty)
  uint64_t q_full[UNIT_QUEUE];
  uint64_t q_empty[UNIT_QUEUE];
  // a stage's block scales are in tensor memory (committed by the scale warp)
  uint64_t sf_ready[MAX_STAGES];
  uint32_t tmem_base;
  int abort_flag;
  int q_unit[UNIT_QUEUE];
};
static_assert(sizeof(Ctrl) <= CTRL_BYTES, "control block too large");

// A slot: [2 KB scales | a_rows x 128 bytes of codes]
__host__ __device__ constexpr int a_slot_bytes(int a_rows) { return OPERAND_SF_BYTES + a_rows * 128; }
__host__ __device__ constexpr int a_tail_bytes(int a_rows) { return (TILE_M - a_rows) * 128; }
// B slot: one 18 KB weight tile, or for column pairs [scales a | scales b |
// codes a | codes b] (36 KB), so the pair's 256 rows of codes are contiguous.
__host__ __device__ constexpr int b_slot_bytes(bool pair) { return pair ? 2 * B_SLOT : B_SLOT; }
__host__ __device__ constexpr int stage_bytes(int a_rows, bool pair = false) {
  return a_slot_bytes(a_rows) + b_slot_bytes(pair);
}
__host__ __device__ constexpr int smem_bytes_for(int stages, int nch, int a_rows, bool pair = false,
                                                 bool stage_out = false) {
  return stages * stage_bytes(a_rows, pair) + a_tail_bytes(a_rows) + CTRL_BYTES + 2 * nch * TILE_M * 4 +
         HALF_MAX_BYTES + (stage_out ? EPI_STAGE_BYTES : 0) + 1024;
}
// Resident activations (the small-batch w13 GEMM, whose tiles all read the
// same shared activation tile): all K stages of A stay in shared memory for
// the whole kernel, loaded once; the ring carries only weight tiles.
constexpr int ARES_MAX_KS = 8;  // K <= 2048
__host__ __device__ constexpr int smem_bytes_res(int stages, int nch, int a_rows, bool pair = false) {
  return ARES_MAX_KS * a_slot_bytes(a_rows) + a_tail_bytes(a_rows) + stages * b_slot_bytes(pair) + CTRL_BYTES +
         2 * nch * TILE_M * 4 + HALF_MAX_BYTES + 1024;
}

// SwiGLU silu(g) * u.  Default sigmoid(g) = 1/2 + tanh(g/2)/2: one
// special-function operation per element (the hardware tanh, relative error
// about 2^-11, below the FP4 requantization that follows).  With
// `accurate`, sigmoid(g) = 1 / (1 + expf(-g)) with CUDA's expf and an IEEE
// division (a few ulp): fewer of the requantization's near-tie decisions
// differ from an FP64 evaluation.
__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float swiglu(float g_acc, float u_acc, float alpha, bool accurate) {
  const float g = __fmul_rn(g_acc, alpha);
  const float u = __fmul_rn(u_acc, alpha);
  const float sig = accurate ? __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-g))) : fmaf(0.5f, tanh_approx(0.5f * g), 0.5f);
  return __fmul_rn(__fmul_rn(g, u), sig);
}

__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

struct Unit {
  int e, row0, valid, col;  // expert, first padded row, valid rows, 128-column block of B
  int arow;                 // first row of the activation operand
};

template <int MODE, int A_ROWS, int STAGES, bool ARES>
__global__ void __launch_bounds__(THREADS, 1) gemm_fp4_kernel(const __grid_constant__ GemmArgs p) {
  constexpr int A_SLOT = a_slot_bytes(A_ROWS);
  constexpr int A_SLOTS = ARES ? ARES_MAX_KS : STAGES;  // resident: one slot per K stage
  constexpr bool PAIR = pair_mode(MODE);  // N = 256 over pairs of adjacent 128-column tiles
  constexpr int BS = b_slot_bytes(PAIR);
  constexpr int SF_STAGE = PAIR ? TMEM_SF_STAGE_PAIR : TMEM_SF_STAGE;
  static_assert(!PAIR || STAGES <= MAX_STAGES_PAIR, "tensor memory overflow");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = base;                                          // [A_SLOTS][A_SLOT] + tail
  uint8_t* sB = sA + A_SLOTS * A_SLOT + a_tail_bytes(A_ROWS);  // [STAGES][BS]
  Ctrl& c = *reinterpret_cast<Ctrl*>(sB + STAGES * BS);
  // [2][nch][128] words: partial row maximum bits (non-negative, so bit 31
  // is free) with bit 31 holding the m-tile tag
  uint32_t* part = reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(&c) + CTRL_BYTES);
  // [2][2][128] w13 row maxima of the two column halves of a CTA (m-tile
  // buffer i & 1, then half)
  float* half_max = reinterpret_cast<float*>(part + (MODE == MODE_W13 ? 2 * gridDim.x * TILE_M : 0));
  // ordered w2: the epilogue warps' output staging, [8 warps][32 rows][EPI_ROW_STRIDE]
  uint8_t* epi_stage = reinterpret_cast<uint8_t*>(half_max) + HALF_MAX_BYTES;
  {
    // The layout above must fit the launch's dynamic shared memory; if the
    // host sized it differently, report and leave before touching any of it
    // (the condition is the same in every CTA of the grid).
    uint32_t dyn;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
    const uint8_t* end = epi_stage + (MODE == MODE_W2_ORDERED ? EPI_STAGE_BYTES : 0);
    if (end > smem_raw + dyn) {
      if (threadIdx.x == 0) report_device_error(p.status, DEV_ERR_BAD_STATE);
      return;
    }
  }

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- static schedule, identical in every role ----
  // w13: cluster blockIdx.y takes m-tiles blockIdx.y, +gridDim.y, ...; CTA
  //      rank r of the cluster takes units (m-tile, B column blocks 2r, 2r+1).
  // w2: CTA b takes unit pairs b, b + gridDim.x, ... of (m-tile, n-tiles
  //      2c, 2c+1); plain: CTA b takes units b, b + gridDim.x, ...
  // w13s: CTA b takes unit pairs b, b + gridDim.x, ... of (m-tile, column
  //      pair r), pair index = m-tile * (I/128) + r.
  constexpr bool W13L = (MODE == MODE_W13 || MODE == MODE_W13S);  // units in column pairs
  const int nch = (MODE == MODE_W13) ? (int)gridDim.x : (MODE == MODE_W13S ? p.w13_pairs : 1);
  const uint32_t rank = (MODE == MODE_W13) ? blockIdx.x : 0;
  pdl_trigger();
  int first, stride;
  if constexpr (MODE == MODE_W13) {
    first = 2 * blockIdx.y;
    stride = 2 * gridDim.y;
  } else if constexpr (PAIR) {  // w13s, w2: unit pairs b, b + gridDim.x, ...
    first = 2 * blockIdx.x;
    stride = 2 * gridDim.x;
  } else {
    first = blockIdx.x;
    stride = gridDim.x;
  }
  // w13 units come in pairs (2 per m-tile); `next` skips to the next pair.
  auto next = [&](int u) -> int {
    if constexpr (PAIR) return (u & 1) ? u - 1 + stride : u + 1;
    else return u + stride;
  };
  auto unit_at = [&](int u) -> Unit {
    Unit r;
    if constexpr (MODE == MODE_W13) {
      const int4 ti = p.tiles[u >> 1];
      r.e = ti.x; r.row0 = ti.y; r.valid = ti.z; r.col = 2 * (int)rank + (u & 1); r.arow = ti.w;
    } else if constexpr (MODE == MODE_W13S) {
      const int pair = u >> 1;
      const int tile = pair / nch;
      r.col = 2 * (pair % nch) + (u & 1);
      if (p.all_experts) {  // tile i is expert i: padded rows i*128 + t, the shared activation tile
        r.e = tile; r.row0 = tile * TILE_M; r.valid = p.small_T; r.arow = 0;
      } else {
        const int4 ti = p.tiles[tile];
        r.e = ti.x; r.row0 = ti.y; r.valid = ti.z; r.arow = ti.w;
      }
    } else if constexpr (MODE == MODE_PLAIN) {
      r.e = 0; r.row0 = (u / p.n_tiles) * TILE_M; r.valid = TILE_M; r.col = u % p.n_tiles; r.arow = r.row0;
    } else {
      const int tile = u / p.n_tiles;
      r.col = u % p.n_tiles;
      if (p.all_experts) {
        r.e = tile; r.row0 = tile * TILE_M; r.valid = p.small_T;
      } else {
        const int4 ti = p.tiles[tile];
        r.e = ti.x; r.row0 = ti.y; r.valid = ti.z;
      }
      // the w2 GEMM's activations are the intermediate rows at the padded rows
      r.arow = r.row0;
    }
    return r;
  };
  // Work units of the launch.  With all_experts (small batches in which
  // nearly every expert has rows) the list is every expert in order and is
  // known before the previous kernels finish; otherwise it is the tile list
  // they write, read only after the dependency wait.
  auto count_units = [&]() -> int {
    if constexpr (MODE == MODE_W13) return 2 * (*p.num_tiles);
    else if constexpr (MODE == MODE_W13S) return 2 * nch * (p.all_experts ? p.num_experts : *p.num_tiles);
    else if constexpr (MODE == MODE_PLAIN) return p.m_tiles * p.n_tiles;
    else return (p.all_experts ? p.num_experts : *p.num_tiles) * p.n_tiles;
  };
  // Dynamic schedule (the small-batch w13 GEMM over all experts, launched
  // while the front kernel still runs): the CTAs take unit pairs from a
  // global counter, so that CTAs which start late - on the front kernel's
  // SMs - take fewer.  Instead of a dependency wait the kernel reads the
  // front kernel's counters: the producer waits until every front CTA has
  // quantized its tokens before it loads activations; the epilogue treats
  // every row as routed until every front CTA has routed its tokens; and no
  // CTA finishes before routing has finished (so later kernels, which wait
  // for this one, see it).
  const bool dyn = !ARES && MODE == MODE_W13S && p.all_experts && p.front_sync != nullptr;
  const uint32_t front_n = (uint32_t)p.front_ctas;
  auto static_unit = [&](int n) -> int {
    const int u = first + n * stride;
    return u < count_units() ? u : -1;
  };
  // consumer side of the queue: unit n, or -1 when the CTA is done (or gave up)
  auto queued_unit = [&](int n, bool single_thread) -> int {
    const int q = n % UNIT_QUEUE;
    bool ok = true;
    if (single_thread || lane == 0) ok = mbar_wait_bounded(&c.q_full[q], (n / UNIT_QUEUE) & 1, &c.abort_flag);
    if (!single_thread) ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    if (!ok) {
      if (single_thread || lane == 0) {
        c.abort_flag = 1;
        report_device_error(p.status, DEV_ERR_TIMEOUT);
      }
      return -1;
    }
    const int u = *reinterpret_cast<volatile int*>(&c.q_unit[q]);
    if (!single_thread) __syncwarp();
    if (single_thread || lane == 0) mbar_arrive(&c.q_empty[q]);
    return u;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&c.full[s], 1);
      mbar_init(&c.empty[s], 1);
      mbar_init(&c.sf_ready[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&c.acc_full[b], 1);
      mbar_init(&c.acc_empty[b], EPI_WARPS);
    }
    mbar_init(&c.a_full, 1);
    for (int q = 0; q < UNIT_QUEUE; ++q) {
      mbar_init(&c.q_full[q], 1);
      mbar_init(&c.q_empty[q], 2 + EPI_WARPS);  // the MMA thread, the scale warp, the epilogue warps
    }
    c.abort_flag = 0;
    if (MODE == MODE_W13)
      for (int i = 0; i < 2 * nch * TILE_M; ++i) part[i] = 0x80000000u;  // tag of no first use
    fence_mbarrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&c.tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (MODE == MODE_W13) cluster_sync_all();  // peers' exchange slots are cleared before any remote store
  tc_fence_after();
  const uint32_t tmem = c.tmem_base;
  const int KS = p.k_stages;
  // Stages of the ring whose weight tile the producer issued before the
  // dependency wait (their activation tiles follow after it).
  constexpr bool PRE_ISSUE = !ARES && (MODE == MODE_W13S || MODE == MODE_W2_ATOMIC || MODE == MODE_W2_ORDERED);
  uint32_t g_pre = 0;
  int u_first = -1;  // dynamic schedule: the producer's first unit
  // producer side of the queue: fetch the CTA's unit n from the global counter
  auto fetch_unit = [&](int n) -> int {
    const int q = n % UNIT_QUEUE;
    if (!mbar_wait_bounded(&c.q_empty[q], ((n / UNIT_QUEUE) & 1) ^ 1, &c.abort_flag)) {
      c.abort_flag = 1;
      report_device_error(p.status, DEV_ERR_TIMEOUT);
      return -1;
    }
    const int pair = (int)atomicAdd(p.front_sync + FRONT_SYNC_WORK, 1u);
    const int u = pair < count_units() / 2 ? 2 * pair : -1;
    c.q_unit[q] = u;
    mbar_arrive(&c.q_full[q]);
    return u;
  };
  if (MODE != MODE_PLAIN && warp == 0 && lane == 0) {
    if (p.prefetch_units > 0 && !dyn) {
      // Weights do not depend on the previous kernels: stream the expected
      // first units' weight tiles into L2 while those kernels still run.
      int u = first;
      for (int k = 0; k < p.prefetch_units; ++k, u = next(u)) {
        const int tile = (MODE == MODE_W13) ? (u >> 1) : (MODE == MODE_W13S ? (u >> 1) / nch : u / p.n_tiles);
        if (tile >= p.num_experts) break;
        const int col = (MODE == MODE_W13)    ? 2 * (int)rank + (u & 1)
                        : (MODE == MODE_W13S) ? 2 * ((u >> 1) % nch) + (u & 1)
                                              : u % p.n_tiles;
        if (u & 1) continue;  // the pair block of an even unit holds both tiles
        const int brow0 = tile * p.b_rows_per_expert + col * TILE_N;
        const uint8_t* b_src = p.b_codes + (size_t)(brow0 >> 8) * KS * WPAIR_BYTES;
        for (int ks = 0; ks < KS; ++ks) prefetch_l2_bulk(b_src + (size_t)ks * WPAIR_BYTES, WPAIR_BYTES);
      }
    }
    if (PRE_ISSUE && p.all_experts) {
      // The unit list does not depend on the previous kernels: fill the
      // ring's weight slots now.  Each slot's barrier first expects only the
      // weight bytes; the producer arrives (and adds the activation bytes)
      // when it issues the activation tile, once the activations are ready.
      if (dyn) u_first = fetch_unit(0);
      for (int n = 0; g_pre < (uint32_t)STAGES; ++n) {
        const int u = dyn ? (n == 0 ? u_first : -1) : static_unit(n);
        if (u < 0) break;
        const Unit un = unit_at(u);
        const int brow0 = un.e * p.b_rows_per_expert + un.col * TILE_N;
        for (int ks = 0; ks < KS && g_pre < (uint32_t)STAGES; ++ks, ++g_pre) {
          mbar_expect_tx(&c.full[g_pre], BS);
          bulk_load(sB + g_pre * BS, p.b_codes + ((size_t)(brow0 >> 8) * KS + ks) * WPAIR_BYTES, WPAIR_BYTES,
                    &c.full[g_pre]);
        }
      }
    }
  }
  // Everything above overlaps the previous kernel's tail; its outputs (the
  // tile list, operands, scales) are read only from here on.
  if (!dyn) pdl_wait();
  if (p.reset_sync && blockIdx.x == 0) {
    // the all-experts path's counters, no longer read by the earlier kernels
    if (threadIdx.x < FRONT_SYNC_RESET) p.reset_sync[threadIdx.x] = 0;
    for (int e = threadIdx.x; e < p.num_experts; e += blockDim.x) p.expert_done[e] = 0;
  }
  const int nunits = count_units();
  // block scales of one stage, shared memory -> tensor memory
  auto copy_stage_scales = [&](uint32_t sfa_t, uint32_t sfb_t, const uint8_t* slot_a, const uint8_t* slot_b) {
    constexpr int SFB_COLS = PAIR ? 8 : 4;  // B scale columns per K block
#pragma unroll
    for (int kb = 0; kb < 4; ++kb) {
      tc_copy_sf(sfa_t + kb * 4, smem_desc_sf(smem_u32(slot_a + kb * SF_ATOM_BYTES)));
      tc_copy_sf(sfb_t + kb * SFB_COLS, smem_desc_sf(smem_u32(slot_b + kb * SF_ATOM_BYTES)));
      if (PAIR)
        tc_copy_sf(sfb_t + kb * SFB_COLS + 4, smem_desc_sf(smem_u32(slot_b + OPERAND_SF_BYTES + kb * SF_ATOM_BYTES)));
    }
  };

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- producer ----------------
      uint32_t g = 0;  // stages issued so far (ring position)
      bool a_issued = false;
      if (ARES && first < nunits) {
        // every tile reads the same activation rows: load all K stages once
        const Unit un = unit_at(first);
        const uint32_t a_bytes = OPERAND_SF_BYTES + (uint32_t)((un.valid + 7) & ~7) * 128;
        const uint8_t* a_src = p.a_codes + (size_t)(un.arow >> 7) * KS * OPERAND_TILE_BYTES;
        mbar_arrive_expect_tx(&c.a_full, a_bytes * (uint32_t)KS);
        for (int ks = 0; ks < KS; ++ks)
          bulk_load(sA + ks * A_SLOT, a_src + (size_t)ks * OPERAND_TILE_BYTES, a_bytes, &c.a_full);
        a_issued = true;
      }
      if (dyn) {
        // the activations: every front CTA has quantized its tokens (bounded)
        bool ok = wait_counter_acquire(p.front_sync + FRONT_SYNC_A_READY, front_n, &c.abort_flag);
        if (!ok) {
          c.abort_flag = 1;
          report_device_error(p.status, DEV_ERR_TIMEOUT);
        }
        // they were written by another kernel's generic stores; the bulk
        // copies below read them through the async proxy
        asm volatile("fence.proxy.async.global;" ::: "memory");
      }
      int u = dyn ? u_first : static_unit(0);
      for (int n = 0; u >= 0 && !c.abort_flag;) {
        const Unit un = unit_at(u);
        const int brow0 = (MODE == MODE_PLAIN ? 0 : un.e * p.b_rows_per_expert) + un.col * TILE_N;
        // scales + valid rows, in whole 8-row swizzle groups
        const uint32_t a_bytes = OPERAND_SF_BYTES + (uint32_t)((un.valid + 7) & ~7) * 128;
        const uint32_t bytes = (ARES ? 0u : a_bytes) + BS;
        const uint8_t* a_src = p.a_codes + (size_t)(un.arow >> 7) * KS * OPERAND_TILE_BYTES;
        const uint8_t* b_src = p.b_codes + (size_t)(brow0 >> 7) * KS * OPERAND_TILE_BYTES;
        for (int ks = 0; ks < KS; ++ks, ++g) {
          const int s = g % STAGES;
          if (PRE_ISSUE && g < g_pre) {
            // the weight tile of this (first) use of the slot is in flight
            mbar_arrive_expect_tx(&c.full[s], a_bytes);
            bulk_load(sA + s * A_SLOT, a_src + (size_t)ks * OPERAND_TILE_BYTES, a_bytes, &c.full[s]);
            continue;
          }
          if (!mbar_wait_bounded(&c.empty[s], ((g / STAGES) & 1) ^ 1, &c.abort_flag)) {
            c.abort_flag = 1;
            report_device_error(p.status, DEV_ERR_TIMEOUT);
            break;
          }
          mbar_arrive_expect_tx(&c.full[s], bytes);
          if (!ARES) bulk_load(sA + s * A_SLOT, a_src + (size_t)ks * OPERAND_TILE_BYTES, a_bytes, &c.full[s]);
          uint8_t* slot_b = sB + s * BS;
          if constexpr (PAIR) {
            // weights are stored in pair tiles: the stage is one 36 KB block
            // [scales a | scales b | codes a | codes b]
            bulk_load(slot_b, p.b_codes + ((size_t)(brow0 >> 8) * KS + ks) * WPAIR_BYTES, WPAIR_BYTES, &c.full[s]);
          } else {
            bulk_load(slot_b, b_src + (size_t)ks * OPERAND_TILE_BYTES, B_SLOT, &c.full[s]);
          }
        }
        ++n;
        u = dyn ? fetch_unit(n) : static_unit(n);
      }
      if (PRE_ISSUE) {
        // After an abort the loop above may stop before it reached every
        // stage whose weight tile was issued before the dependency wait: arrive
        // on those barriers so that they complete once the weight bytes land,
        // and wait for them below.  (Without an abort g >= g_pre here.)
        for (; g < g_pre; ++g) mbar_arrive(&c.full[g]);
      }
      if (c.abort_flag) {
        // Unwinding: let the copies already issued land before the CTA's
        // shared memory is released (bounded, no early exit).
        for (uint32_t k = g > STAGES ? g - STAGES : 0; k < g; ++k)
          mbar_wait_bounded(&c.full[k % STAGES], (k / STAGES) & 1, nullptr, 1000000000ull);
        if (a_issued) mbar_wait_bounded(&c.a_full, 0, nullptr, 1000000000ull);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      uint32_t g = 0;
      int n = 0;  // units processed by this CTA
      if (ARES && first < nunits && !mbar_wait_bounded(&c.a_full, 0, &c.abort_flag)) {
        c.abort_flag = 1;
        report_device_error(p.status, DEV_ERR_TIMEOUT);
      }
      for (;; ++n) {
        const int u = dyn ? queued_unit(n, true) : static_unit(n);
        if (u < 0 || c.abort_flag) break;
        // column pairs: one accumulator (buffer 0), used by every pair
        const int buf = PAIR ? 0 : n & 1;
        const uint32_t acc_parity = PAIR ? ((n & 1) ^ 1) : (((n >> 1) & 1) ^ 1);
        if (!mbar_wait_bounded(&c.acc_empty[buf], acc_parity, &c.abort_flag)) {
          c.abort_flag = 1;
          report_device_error(p.status, DEV_ERR_TIMEOUT);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + buf * TILE_N;
        for (int ks = 0; ks < KS; ++ks, ++g) {
          const int s = g % STAGES;
          // the stage's operands landed, and the scale warp's copies of its
          // block scales completed
          if (!mbar_wait_bounded(&c.full[s], (g / STAGES) & 1, &c.abort_flag) ||
              !mbar_wait_bounded(&c.sf_ready[s], (g / STAGES) & 1, &c.abort_flag)) {
            c.abort_flag = 1;
            report_device_error(p.status, DEV_ERR_TIMEOUT);
            break;
          }
          tc_fence_after();
          const uint32_t sfa_t = tmem + TMEM_SF_BASE + s * SF_STAGE;
          const uint32_t sfb_t = sfa_t + 16;
          const uint8_t* slot_a = sA + (ARES ? ks : s) * A_SLOT;
          const uint8_t* slot_b = sB + s * BS;
          constexpr int SFB_COLS = PAIR ? 8 : 4;  // B scale columns per K block
          const uint32_t a_base = smem_u32(slot_a + OPERAND_SF_BYTES);
          const uint32_t b_base = smem_u32(slot_b + (PAIR ? 2 : 1) * OPERAND_SF_BYTES);
#pragma unroll
          for (int kb = 0; kb < 4; ++kb)
            tc_mma_fp4(d_tmem, smem_desc_sw128(a_base + kb * 32), smem_desc_sw128(b_base + kb * 32),
                       PAIR ? IDESC_PAIR : IDESC, sfa_t + kb * 4, sfb_t + kb * SFB_COLS, (ks | kb) != 0);
          tc_commit(&c.empty[s]);
        }
        // Always signal, even after an abort: the epilogue waits for the
        // MMAs already issued before it lets tensor memory go.
        tc_commit(&c.acc_full[buf]);
      }
    }
    __syncwarp();
  } else if (warp == SF_WARP) {
    if (lane == 0) {
      // ---------------- block-scale copies ----------------
      // Per stage, once its operands landed: the block scales into the
      // stage's tensor-memory slot, committed to sf_ready[s] for the MMA
      // thread.  (A slot's previous scales were read by the MMAs of the
      // stage STAGES earlier, which completed before the producer refilled
      // the ring slot whose landing this waits for.)
      bool ok = !ARES || first >= nunits || mbar_wait_bounded(&c.a_full, 0, &c.abort_flag);
      uint32_t g = 0;
      for (int n = 0; ok; ++n) {
        const int u = dyn ? queued_unit(n, true) : static_unit(n);
        if (u < 0 || c.abort_flag) break;
        for (int ks = 0; ks < KS; ++ks, ++g) {
          const int s = g % STAGES;
          if (!mbar_wait_bounded(&c.full[s], (g / STAGES) & 1, &c.abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sfa_t = tmem + TMEM_SF_BASE + s * SF_STAGE;
          copy_stage_scales(sfa_t, sfa_t + 16, sA + (ARES ? ks : s) * A_SLOT, sB + s * BS);
          tc_commit(&c.sf_ready[s]);
        }
      }
      if (!ok) {
        c.abort_flag = 1;
        report_device_error(p.status, DEV_ERR_TIMEOUT);
      }
    }
    __syncwarp();
  } else {
    // ---------------- epilogue (warps 2..9) ----------------
    const int quarter = warp & 3;          // tensor-memory lanes [32q, 32q+32)
    const int half = (warp - 2) >> 2;      // column half of every accumulator
    const int m = quarter * 32 + lane;     // accumulator row of this thread
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    int n = 0;  // units drained by this CTA

    // Wait for the accumulator of unit n; false if the device state is bad.
    auto wait_acc = [&](int buf, int nn) -> bool {
      bool ok = mbar_wait_bounded(&c.acc_full[buf], (nn >> 1) & 1, nullptr);
      if (!ok) {
        c.abort_flag = 1;
        report_device_error(p.status, DEV_ERR_TIMEOUT);
      }
      tc_fence_after();
      return ok && !c.abort_flag;
    };
    auto release_acc = [&](int buf) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&c.acc_empty[buf]);
    };

    if constexpr (W13L) {
      bool a_seen = !dyn;  // dynamic schedule: the activation scales acquired
      // i: m-tiles (w13s: unit pairs) processed
      for (int i = 0;; ++i) {
        const int u = dyn ? queued_unit(i, false) : static_unit(i);
        if (u < 0) break;
        if (!a_seen) {
          if (!wait_counter_acquire(p.front_sync + FRONT_SYNC_A_READY, front_n, &c.abort_flag)) {
            c.abort_flag = 1;
            report_device_error(p.status, DEV_ERR_TIMEOUT);
          }
          a_seen = true;
        }
        const Unit un = unit_at(u);
        const bool warp_rows = quarter * 32 < un.valid;  // warp-uniform
        const int prow = un.row0 + m;
        // rows of the shared small-batch tile whose token did not pick this
        // expert take no part (their amax counts as 0 in the exchange);
        // dynamic schedule: until the routing is known every row of the tile
        // is formed (the requantization reads only the routed ones)
        const bool routed =
            !dyn || ld_acquire_gpu_u32(p.front_sync + FRONT_SYNC_ROUTED) >= front_n;
        const bool row_ok = m < un.valid && (!routed || p.src_of_padrow[prow] >= 0);
        const float alpha = row_ok ? __fdiv_rn(1.0f, __fmul_rn(p.gs_rows[un.arow + m], p.gs_w[un.e])) : 0.0f;
        // this thread's tile of the pair's 128 x 256 accumulator: columns
        // [128 half, +64) are gate features, the next 64 the matching up
        // features; h takes the gate values, then the SwiGLU values
        float h[64], uv[64];
        float amax = 0.0f;
        bool ready = mbar_wait_bounded(&c.acc_full[0], i & 1, nullptr);
        if (!ready) {
          c.abort_flag = 1;
          report_device_error(p.status, DEV_ERR_TIMEOUT);
        }
        tc_fence_after();
        ready = ready && !c.abort_flag;
        if (ready && warp_rows) {
          const uint32_t t = lane_base + half * TILE_N;
          tmem_ld32(t, h);
          tmem_ld32(t + 32, h + 32);
          tmem_ld32(t + 64, uv);
          tmem_ld32(t + 96, uv + 32);
          tmem_ld_wait();
        }
        release_acc(0);  // everything is in registers: the tensor cores may refill the accumulator
        if (ready && warp_rows) {
          // (both loops fully unrolled: h and uv must stay in registers)
          if (p.accurate_sigmoid) {
#pragma unroll
            for (int q = 0; q < 64; ++q) {
              h[q] = swiglu(h[q], uv[q], alpha, true);
              amax = fmaxf(amax, fabsf(h[q]));
            }
          } else {
#pragma unroll
            for (int q = 0; q < 64; ++q) {
              h[q] = swiglu(h[q], uv[q], alpha, false);
              amax = fmaxf(amax, fabsf(h[q]));
            }
          }
        }
        if (!row_ok) amax = 0.0f;
        // this thread's 64 features of the row start at feature f0
        const int f0 = (MODE == MODE_W13 ? (int)rank : (u >> 1) % nch) * 128 + 64 * half;
        float gs_h;
        if (p.h_gs_static) {
          // static per-tensor contract: the expert's calibrated scale, no
          // row maximum needed (the same branch in every CTA of a cluster)
          gs_h = p.h_gs_static[un.e];
        } else {
          if constexpr (MODE == MODE_W13S) {
            // FP32 SwiGLU row to the scratch, its maximum folded into the
            // row's global word (non-negative floats order like their bits);
            // the requantization kernel finishes the row.
            if (ready && row_ok) {
              atomicMax(reinterpret_cast<unsigned int*>(p.row_amax) + prow, __float_as_uint(amax));
              float4* dst = reinterpret_cast<float4*>(p.hbuf + (size_t)prow * p.i_pad + f0);
#pragma unroll
              for (int q = 0; q < 16; ++q) dst[q] = make_float4(h[4 * q], h[4 * q + 1], h[4 * q + 2], h[4 * q + 3]);
            }
            if (dyn) {
              // the unit's column pair is done for its expert once every
              // epilogue warp stored its rows: the requantization kernel
              // starts on an expert as soon as all its column pairs are
              named_bar_sync(1, EPI_WARPS * 32);
              if (warp == 2 && lane == 0) {
                __threadfence();
                atomicAdd(p.expert_done + un.e, 1u);
              }
            }
            continue;
          }
          // The CTA's two halves first combine their maxima in shared memory
          // (buffer i & 1: a half can be at most one m-tile ahead, since it
          // passes the barrier of the next m-tile only with the other half).
          float* hm = half_max + (size_t)(i & 1) * 2 * TILE_M;
          hm[half * TILE_M + m] = amax;
          named_bar_sync(1, EPI_WARPS * 32);
          const float amax_cta = fmaxf(hm[m], hm[TILE_M + m]);
          // Exchange the row maxima across the cluster.  Slot buffer i & 1;
          // a peer can be at most one m-tile ahead (it needs this CTA's value
          // of its next m-tile first), so two buffers never overwrite a value
          // that has not been read, and the successive uses of a buffer
          // alternate the tag bit.  Half 0 stores; both halves read.
          const int b = i & 1;
          const uint32_t tag = ((uint32_t)(i >> 1) & 1u) << 31;
          const uint32_t* slots = part + (size_t)b * nch * TILE_M + m;
          if (half == 0)
            for (int r = 0; r < nch; ++r)
              st_shared_cluster_u32(slots + (size_t)rank * TILE_M, (uint32_t)r, tag | __float_as_uint(amax_cta));
          float amax_row = 0.0f;
          for (int r = 0; r < nch; ++r) {
            const uint32_t* slot = slots + (size_t)r * TILE_M;
            uint32_t v = ld_shared_relaxed_u32(slot);
            if ((v & 0x80000000u) != tag) {
              const uint64_t t0 = global_timer_ns();
              for (uint32_t it = 1; (v & 0x80000000u) != tag; ++it) {
                v = ld_shared_relaxed_u32(slot);
                if ((it & 255u) == 0 && global_timer_ns() - t0 > 2000000000ull) {
                  c.abort_flag = 1;
                  report_device_error(p.status, DEV_ERR_TIMEOUT);
                  ready = false;
                  break;
                }
              }
            }
            amax_row = fmaxf(amax_row, __uint_as_float(v & 0x7FFFFFFFu));
          }
          gs_h = nvfp4_global_scale(amax_row);
        }
        if (ready && row_ok) {
          const int k16_row = p.i_pad / SF_VEC;
          uint32_t sf4 = 0;  // the 4 blocks' scale bytes are consecutive in the row's atom
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            float v[16];
#pragma unroll
            for (int q = 0; q < 16; ++q) v[q] = h[16 * cc + q];
            uint2 packed;
            const uint32_t sf = nvfp4_quant_block16(v, gs_h, packed);
            const int k = f0 + 16 * cc;  // feature index of this block
            *reinterpret_cast<uint2*>(p.h_codes + operand_offset(prow, k / 2, p.i_pad / 2)) = packed;
            sf4 |= sf << (8 * cc);
          }
          *reinterpret_cast<uint32_t*>(p.h_sf + sf_atom_offset(prow, f0 / SF_VEC, k16_row)) = sf4;
          if (f0 == 0) p.h_gs[prow] = gs_h;
        }
      }
      if (dyn) {
        // No CTA finishes before the routing has: later kernels rely on it
        // through this kernel's completion.  Meanwhile the CTA's epilogue
        // warps, out of units, requantize the intermediate: each takes
        // expanded rows (token * K + slot) from a global counter and starts
        // one once its expert has all its column pairs done; then experts
        // from a second counter, whose rows of tokens that did not route
        // there get their maxima returned to zero (formed while the routing
        // was not known).  The w2 GEMM waits for this kernel as a whole.
        bool ok = true;
        if (lane == 0) ok = wait_counter_acquire(p.front_sync + FRONT_SYNC_ROUTED, front_n, nullptr);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok && lane == 0) report_device_error(p.status, DEV_ERR_TIMEOUT);
        const int T = p.small_T, K = p.top_k, n_rows = T * K;
        while (ok) {
          int r = 0;
          if (lane == 0) r = (int)atomicAdd(p.front_sync + FRONT_SYNC_RQ_ROW, 1u);
          r = __shfl_sync(0xffffffffu, r, 0);
          if (r >= n_rows) break;
          const int e = __ldcg(p.topk_ids_small + r);
          if (lane == 0) ok = wait_counter_acquire(p.expert_done + e, (uint32_t)nch, &c.abort_flag);
          ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
          if (!ok) {
            if (lane == 0) report_device_error(p.status, DEV_ERR_TIMEOUT);
            break;
          }
          const size_t prow = (size_t)e * TILE_M + r / K;
          const float gs_r = nvfp4_global_scale(__ldcg(p.row_amax + prow));
          requant_row_warp(p.hbuf + prow * p.i_pad, p.inter, p.i_pad, prow, gs_r, p.h_codes, lane);
          if (lane == 0) {
            p.h_gs[prow] = gs_r;
            p.row_amax[prow] = 0.0f;
          }
        }
        while (ok) {
          int e = 0;
          if (lane == 0) e = (int)atomicAdd(p.front_sync + FRONT_SYNC_RQ_EXPERT, 1u);
          e = __shfl_sync(0xffffffffu, e, 0);
          if (e >= p.num_experts) break;
          if (lane == 0) ok = wait_counter_acquire(p.expert_done + e, (uint32_t)nch, &c.abort_flag);
          ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
          if (!ok) {
            if (lane == 0) report_device_error(p.status, DEV_ERR_TIMEOUT);
            break;
          }
          for (int t = lane; t < T; t += 32) {
            const size_t prow = (size_t)e * TILE_M + t;
            if (__ldcg(p.src_of_padrow + prow) < 0) p.row_amax[prow] = 0.0f;
          }
        }
      }
    } else {
      // pairs: the thread's 128-column tile `half` of the 128 x 256
      // accumulator; plain: its 64-column half of the 128-column buffer
      constexpr int COLS = PAIR ? 128 : 64;
      for (int u = first; u < nunits; u = PAIR ? next(next(u)) : next(u), ++n) {
        const Unit un = unit_at(u);
        const bool warp_rows = quarter * 32 < un.valid;
        const int prow = un.row0 + m;
        int src = 0;
        bool row_ok = m < un.valid;
        if constexpr (MODE != MODE_PLAIN) {
          src = row_ok ? p.src_of_padrow[prow] : -1;
          row_ok = src >= 0;  // a token that did not pick this expert
        }
        // the row's scales and routing weight, loaded while the MMAs run
        float alpha = 1.0f, wj = 1.0f;
        if constexpr (MODE == MODE_W2_ATOMIC || MODE == MODE_W2_ORDERED) {
          if (warp_rows && row_ok) {
            alpha = __fdiv_rn(1.0f, __fmul_rn(p.gs_rows[prow], p.gs_w[un.e]));
            if constexpr (MODE == MODE_W2_ATOMIC) wj = p.topk_w[src];
          }
        }
        // pairs: one 128 x 256 accumulator (buffer 0) holding both tiles
        const int buf = PAIR ? 0 : n & 1;
        bool ready;
        if constexpr (PAIR) {
          ready = mbar_wait_bounded(&c.acc_full[0], n & 1, nullptr);
          if (!ready) {
            c.abort_flag = 1;
            report_device_error(p.status, DEV_ERR_TIMEOUT);
          }
          tc_fence_after();
          ready = ready && !c.abort_flag;
        } else {
          ready = wait_acc(buf, n);
        }
        float a[COLS];
        if (ready && warp_rows) {
          const uint32_t t = lane_base + (PAIR ? half * TILE_N : buf * TILE_N + 64 * half);
#pragma unroll
          for (int q = 0; q < COLS; q += 32) tmem_ld32(t + q, a + q);
          tmem_ld_wait();
        }
        release_acc(buf);  // everything is in registers now
        if (ready && warp_rows && row_ok) {
          const int col = PAIR ? (un.col + half) * TILE_N : un.col * TILE_N + 64 * half;
          if constexpr (MODE == MODE_W2_ATOMIC || MODE == MODE_W2_ORDERED) {
            if constexpr (MODE == MODE_W2_ATOMIC) {
              const int tok = src / (p.top_k > 0 ? p.top_k : 1);
              float* dst = p.out_acc + (size_t)tok * p.hidden + col;
#pragma unroll
              for (int q = 0; q < COLS; q += 4)
                red_add_v4(dst + q, __fmul_rn(wj, __fmul_rn(a[q], alpha)), __fmul_rn(wj, __fmul_rn(a[q + 1], alpha)),
                           __fmul_rn(wj, __fmul_rn(a[q + 2], alpha)), __fmul_rn(wj, __fmul_rn(a[q + 3], alpha)));
            }
          } else {
            float4* dst = reinterpret_cast<float4*>(p.d + (size_t)prow * p.ldd + col);
#pragma unroll
            for (int q = 0; q < COLS / 4; ++q) dst[q] = make_float4(a[4 * q], a[4 * q + 1], a[4 * q + 2], a[4 * q + 3]);
          }
        }
        if constexpr (MODE == MODE_W2_ORDERED) {
          // the (token, slot) rows of the expert output, rounded to bf16,
          // through the warp's staging rows (the warp's calls are uniform:
          // warp_rows is; rows without a routed token store nothing)
          if (warp_rows) {
            const int col = PAIR ? (un.col + half) * TILE_N : un.col * TILE_N + 64 * half;
            const int my_src = (ready && row_ok) ? src : -1;
            uint8_t* stg = epi_stage + (warp - 2) * (32 * EPI_ROW_STRIDE);
#pragma unroll
            for (int pass = 0; pass < COLS / 64; ++pass) {
              uint4* srow = reinterpret_cast<uint4*>(stg + lane * EPI_ROW_STRIDE);
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                const int c0 = pass * 64 + 8 * q;
                uint32_t w[4];
#pragma unroll
                for (int i = 0; i < 4; ++i)
                  w[i] = pack_bf16x2(__fmul_rn(a[c0 + 2 * i], alpha), __fmul_rn(a[c0 + 2 * i + 1], alpha));
                srow[q] = make_uint4(w[0], w[1], w[2], w[3]);
              }
              __syncwarp();
              // lanes 8j .. 8j + 7 store row 4i + j
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const int r = 4 * i + (lane >> 3);
                const int rsrc = __shfl_sync(0xffffffffu, my_src, r);
                const uint4 v = reinterpret_cast<const uint4*>(stg + r * EPI_ROW_STRIDE)[lane & 7];
                if (rsrc >= 0) reinterpret_cast<uint4*>(p.ybuf + (size_t)rsrc * p.hidden + col + pass * 64)[lane & 7] = v;
              }
              __syncwarp();
            }
          }
        }
      }
    }
  }

  __syncwarp();
  // No CTA of a cluster leaves while a peer may still write its shared memory.
  if constexpr (MODE == MODE_W13) cluster_sync_all();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

constexpr int stages_for(int nch, int a_rows, bool pair = false, bool stage_out = false) {
  for (int s = pair ? MAX_STAGES_PAIR : MAX_STAGES; s >= 3; --s)
    if (smem_bytes_for(s, nch, a_rows, pair, stage_out) <= MAX_SMEM) return s;
  return 0;
}
constexpr int stages_for_res(int nch, int a_rows, bool pair = false) {
  for (int s = pair ? MAX_STAGES_PAIR : MAX_STAGES; s >= 3; --s)
    if (smem_bytes_res(s, nch, a_rows, pair) <= MAX_SMEM) return s;
  return 0;
}

template <int MODE, int A_ROWS, int STAGES, bool ARES>
constexpr int kernel_smem(int nch) {
  constexpr bool pair = pair_mode(MODE);
  return ARES ? smem_bytes_res(STAGES, nch, A_ROWS, pair)
              : smem_bytes_for(STAGES, nch, A_ROWS, pair, MODE == MODE_W2_ORDERED);
}

// The shared-memory cap belongs to the kernel instantiation, which handles of
// different widths share: it is only ever raised.
template <int MODE, int A_ROWS, int STAGES, bool ARES = false>
cudaError_t set_attrs(int nch) {
  auto k = gemm_fp4_kernel<MODE, A_ROWS, STAGES, ARES>;
  const int bytes = kernel_smem<MODE, A_ROWS, STAGES, ARES>(nch);
  cudaFuncAttributes fa{};
  cudaError_t err = cudaFuncGetAttributes(&fa, k);
  if (err != cudaSuccess) return err;
  if (fa.maxDynamicSharedSizeBytes < bytes)
    err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (err != cudaSuccess) return err;
  if (MODE == MODE_W13) err = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return err;
}

template <int MODE, int A_ROWS, int STAGES, bool ARES = false>
cudaLaunchConfig_t make_cfg(dim3 grid, int nch, cudaStream_t s, cudaLaunchAttribute* attr, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = kernel_smem<MODE, A_ROWS, STAGES, ARES>(MODE == MODE_W13 ? nch : 0);
  cfg.stream = s;
  int n = 0;
  if (MODE == MODE_W13) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = nch;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = n ? attr : nullptr;
  cfg.numAttrs = n;
  return cfg;
}

template <int MODE, int A_ROWS, int STAGES, bool ARES = false>
cudaError_t launch(const GemmArgs& a, dim3 grid, int nch, cudaStream_t s) {
  cudaLaunchAttribute attr[2];
  // The expert GEMMs always follow another kernel of the same forward.
  cudaLaunchConfig_t cfg = make_cfg<MODE, A_ROWS, STAGES, ARES>(grid, nch, s, attr, MODE != MODE_PLAIN);
  return cudaLaunchKernelEx(&cfg, gemm_fp4_kernel<MODE, A_ROWS, STAGES, ARES>, a);
}

// Ring depths that occur: w2 / plain kernels (no exchange slots) and w13
// kernels with clusters of up to 6 CTAs get the deepest ring that fits; larger
// clusters one stage less.
constexpr int W2_STAGES_128 = stages_for(0, 128, true);
constexpr int W2_STAGES_64 = stages_for(0, 64, true);
// the ordered w2 epilogue's output staging takes a ring stage
constexpr int W2O_STAGES_128 = stages_for(0, 128, true, true);
constexpr int W2O_STAGES_64 = stages_for(0, 64, true, true);
constexpr int PLAIN_STAGES = stages_for(0, 128);
constexpr int W13_STAGES_128 = stages_for(6, 128, true);
constexpr int W13_STAGES_128_L = stages_for(16, 128, true);
constexpr int W13_STAGES_64 = stages_for(6, 64, true);
constexpr int W13_STAGES_64_L = stages_for(16, 64, true);
constexpr int W13S_STAGES_RES = stages_for_res(0, 64, true);
constexpr int W13S_STAGES = stages_for(0, 64, true);
static_assert(W2_STAGES_128 >= 4 && PLAIN_STAGES >= 4 && W13_STAGES_128_L >= 3 && W13_STAGES_64_L >= 3 && W13S_STAGES_RES >= 3,
              "ring too shallow");
static_assert(W13_STAGES_128 >= 4 && W13S_STAGES >= 4, "ring too shallow");
static_assert(W2O_STAGES_128 >= 3 && W2O_STAGES_64 >= 3, "ring too shallow");

template <typename F>
cudaError_t with_w13(int nch, int a_rows, F&& f) {
  using std::integral_constant;
  if (a_rows == 64) {
    if (nch <= 6) return f(integral_constant<int, 64>{}, integral_constant<int, W13_STAGES_64>{});
    return f(integral_constant<int, 64>{}, integral_constant<int, W13_STAGES_64_L>{});
  }
  if (nch <= 6) return f(integral_constant<int, 128>{}, integral_constant<int, W13_STAGES_128>{});
  return f(integral_constant<int, 128>{}, integral_constant<int, W13_STAGES_128_L>{});
}

}  // namespace

cudaError_t gemm_setup_attributes(int nch) {
  static std::mutex m;
  std::lock_guard<std::mutex> lock(m);
  cudaError_t e;
  for (int a_rows : {64, 128}) {
    e = with_w13(nch, a_rows, [&](auto ar, auto st) {
      return set_attrs<MODE_W13, decltype(ar)::value, decltype(st)::value>(nch);
    });
    if (e != cudaSuccess) return e;
  }
  if ((e = set_attrs<MODE_W13S, 64, W13S_STAGES_RES, true>(0)) != cudaSuccess) return e;
  if ((e = set_attrs<MODE_W13S, 64, W13S_STAGES, false>(0)) != cudaSuccess) return e;
  if ((e = set_attrs<MODE_W2_ATOMIC, 128, W2_STAGES_128>(0)) != cudaSuccess) return e;
  if ((e = set_attrs<MODE_W2_ATOMIC, 64, W2_STAGES_64>(0)) != cudaSuccess) return e;
  if ((e = set_attrs<MODE_W2_ORDERED, 128, W2O_STAGES_128>(0)) != cudaSuccess) return e;
  if ((e = set_attrs<MODE_W2_ORDERED, 64, W2O_STAGES_64>(0)) != cudaSuccess) return e;
  return set_attrs<MODE_PLAIN, 128, PLAIN_STAGES>(0);
}

int gemm_w13_max_clusters(int nch, int a_rows) {
  int n = 0;
  cudaError_t e = with_w13(nch, a_rows, [&](auto ar, auto st) {
    constexpr int AR = decltype(ar)::value, S = decltype(st)::value;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = make_cfg<MODE_W13, AR, S>(dim3(nch, 1, 1), nch, 0, attr, false);
    return cudaOccupancyMaxActiveClusters(&n, gemm_fp4_kernel<MODE_W13, AR, S, false>, &cfg);
  });
  if (e != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

cudaError_t launch_gemm_w13(const GemmArgs& a, int n_chunks, int n_clusters, int a_rows, cudaStream_t s) {
  const dim3 grid(n_chunks, n_clusters, 1);
  return with_w13(n_chunks, a_rows, [&](auto ar, auto st) {
    return launch<MODE_W13, decltype(ar)::value, decltype(st)::value>(a, grid, n_chunks, s);
  });
}

cudaError_t launch_gemm_w13s(const GemmArgs& a, int n_ctas, bool resident, cudaStream_t s) {
  if (resident && a.k_stages > ARES_MAX_KS) return cudaErrorInvalidValue;
  const dim3 grid(n_ctas, 1, 1);
  if (resident) return launch<MODE_W13S, 64, W13S_STAGES_RES, true>(a, grid, 0, s);
  return launch<MODE_W13S, 64, W13S_STAGES, false>(a, grid, 0, s);
}

cudaError_t launch_gemm_w2(const GemmArgs& a, int n_ctas, bool ordered, int a_rows, cudaStream_t s) {
  const dim3 grid(n_ctas, 1, 1);
  if (a_rows == 64) {
    if (ordered) return launch<MODE_W2_ORDERED, 64, W2O_STAGES_64>(a, grid, 0, s);
    return launch<MODE_W2_ATOMIC, 64, W2_STAGES_64>(a, grid, 0, s);
  }
  if (ordered) return launch<MODE_W2_ORDERED, 128, W2O_STAGES_128>(a, grid, 0, s);
  return launch<MODE_W2_ATOMIC, 128, W2_STAGES_128>(a, grid, 0, s);
}

cudaError_t launch_gemm_plain(const GemmArgs& a, int n_ctas, cudaStream_t s) {
  return launch<MODE_PLAIN, 128, PLAIN_STAGES>(a, dim3(n_ctas, 1, 1), 0, s);
}

}  // namespace moe
