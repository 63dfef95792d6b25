// common.cuh - device helpers shared by the sm_103a kernels of the routed-MoE
// forward: inline PTX for mbarrier / TMA / tcgen05, bounded waits, and the
// NVFP4 block quantizer.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace moe {

// ---------------------------------------------------------------------------
// Layout constants
// ---------------------------------------------------------------------------
constexpr int SF_VEC = 16;          // elements per E4M3 block scale
constexpr int MMA_K = 64;           // FP4 elements per tcgen05.mma (kind::mxf4nvf4)
constexpr int STAGE_K = 256;        // FP4 elements per pipeline stage (128 bytes per row)
constexpr int TILE_M = 128;         // rows per expert tile
constexpr int TILE_N = 128;         // output columns per MMA tile
constexpr int SF_ATOM_BYTES = 512;  // block scales of 128 rows x 64 K-elements

// Device status word bits (mapped host memory, read by the host without sync).
constexpr int DEV_ERR_TIMEOUT = 1;
constexpr int DEV_ERR_BAD_STATE = 2;

// Operand layout of every FP4 GEMM operand (activations, intermediate,
// weights): tiles of 128 rows x 256 elements of K, each one contiguous
// 18 KB block [2 KB block scales | 16 KB codes], ordered [row / 128][K / 256].
//  - the block scales of the tile are four "128x4 atoms" of 512 bytes (one
//    per 64 elements of K): the scale of row r, 16-element block j of the
//    atom at (r % 32) * 16 + (r / 32) * 4 + j - the layout the tensor cores
//    read after a 32x128b.warpx4 copy into tensor memory;
//  - the codes are 128 rows x 128 bytes (two E2M1 codes per byte, element
//    2i in the low nibble) already in the 128-byte-swizzled order the tensor
//    cores read from shared memory: 16-byte chunk c of row r at chunk
//    c ^ (r % 8).
// A pipeline stage then fetches a whole weight tile, scales included, with
// one linear bulk copy.  Codes and scales of an operand live in one buffer;
// both offsets below are relative to its base.
constexpr int OPERAND_SF_BYTES = 4 * 512;
constexpr int OPERAND_CODE_BYTES = 128 * 128;
constexpr int OPERAND_TILE_BYTES = OPERAND_SF_BYTES + OPERAND_CODE_BYTES;

// Bytes of an operand of `rows` rows (a multiple of 128) and row_bytes packed
// code bytes per row (a multiple of 128).
__host__ __device__ __forceinline__ size_t operand_bytes(size_t rows, int row_bytes) {
  return (rows >> 7) * (size_t)(row_bytes >> 7) * OPERAND_TILE_BYTES;
}

// Offset of packed code byte kb (elements 2kb, 2kb+1) of `row`.
__host__ __device__ __forceinline__ size_t operand_offset(size_t row, int kb, int row_bytes) {
  const int stages = row_bytes >> 7;
  const int r = (int)(row & 127), b = kb & 127;
  return ((row >> 7) * stages + (size_t)(kb >> 7)) * OPERAND_TILE_BYTES + OPERAND_SF_BYTES + (size_t)r * 128 +
         ((((b >> 4) ^ r) & 7) << 4) + (b & 15);
}

// Offset of the E4M3 block scale of (row, 16-element block k16) of an
// operand with k16_per_row blocks per row, in the layout above.
__host__ __device__ __forceinline__ size_t sf_atom_offset(size_t row, int k16, int k16_per_row) {
  const int stages = k16_per_row >> 4;
  return ((row >> 7) * stages + (size_t)(k16 >> 4)) * OPERAND_TILE_BYTES + (size_t)((k16 >> 2) & 3) * SF_ATOM_BYTES +
         (size_t)((row & 31) * 16 + ((row >> 5) & 3) * 4 + (k16 & 3));
}

// Weights are read by the expert GEMMs as pairs of 128-row tiles (N = 256
// MMAs), so they are stored as 256-row pair tiles: per (row / 256, K / 256)
// one contiguous 36 KB block [scales of rows 0..127 | scales of rows
// 128..255 | codes of rows 0..255], each part in the layout above (the codes'
// swizzle uses row % 8, the same in both halves).  A pipeline stage fetches a
// pair of weight tiles with one bulk copy.  Same total size as
// operand_bytes(); rows a multiple of 256.
constexpr int WPAIR_BYTES = 2 * OPERAND_TILE_BYTES;

__host__ __device__ __forceinline__ size_t wpair_offset(size_t row, int kb, int row_bytes) {
  const int stages = row_bytes >> 7;
  const int r = (int)(row & 255), b = kb & 127;
  return ((row >> 8) * stages + (size_t)(kb >> 7)) * WPAIR_BYTES + 2 * OPERAND_SF_BYTES + (size_t)r * 128 +
         ((((b >> 4) ^ r) & 7) << 4) + (b & 15);
}

__host__ __device__ __forceinline__ size_t wpair_sf_offset(size_t row, int k16, int k16_per_row) {
  const int stages = k16_per_row >> 4;
  const int r = (int)(row & 255);
  return ((row >> 8) * stages + (size_t)(k16 >> 4)) * WPAIR_BYTES + (size_t)(r >> 7) * OPERAND_SF_BYTES +
         (size_t)((k16 >> 2) & 3) * SF_ATOM_BYTES + (size_t)((r & 31) * 16 + ((r >> 5) & 3) * 4 + (k16 & 3));
}

// ---------------------------------------------------------------------------
// Generic helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void report_device_error(int* status_word, int bits) {
  if (status_word) atomicOr(status_word, bits);
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialisation may start while its predecessor in the stream is finishing;
// pdl_wait() blocks until the predecessor grid has completed and its memory
// is visible (a no-op for a normally serialised launch).  pdl_trigger() lets
// the successor launch early.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Launch with programmatic stream serialisation (pdl = true) or as a plain
// stream-ordered launch.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                            Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  if (pdl) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbarrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// Add `bytes` to the transaction count of the current phase without
// arriving.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n"
      ".reg .pred p;\n"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      "selp.u32 %0, 1, 0, p;\n"
      "}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase of `parity` to complete, for at most ~timeout_ns.  When
// `abort` is given, gives up early once another thread of the CTA raised it.
// Returns false on timeout or abort; the caller then records the error and
// unwinds.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, volatile int* abort,
                                                  uint64_t timeout_ns = 2000000000ull) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0) {
      if (abort != nullptr && *abort) return false;
      if (global_timer_ns() - t0 > timeout_ns) return false;
    }
  }
}

// ---------------------------------------------------------------------------
// TMA and bulk copies (global -> shared, completion on an mbarrier)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Hint: bring `bytes` (a multiple of 16, 16-byte aligned) of global memory
// into L2 without a destination or completion.
__device__ __forceinline__ void prefetch_l2_bulk(const void* gsrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(gsrc), "r"(bytes) : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05 (5th-generation tensor cores, accumulators in tensor memory)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_result, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_result)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrive on `bar` when every tcgen05 operation issued so far by this thread
// (MMAs and copies) has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// Copy 32 rows x 16 bytes of block scales from shared memory into tensor
// memory, replicated to the four 32-lane quarters (4 columns).
__device__ __forceinline__ void tc_copy_sf(uint32_t taddr, uint64_t src_desc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(src_desc) : "memory");
}

// D[tmem] (+)= A[smem] x B[smem]^T with E2M1 operands and UE4M3 scales per 16
// elements (scale_vec::4X), M=128, N from the instruction descriptor, K=64.
__device__ __forceinline__ void tc_mma_fp4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n"
      ".reg .pred p;\n"
      "setp.ne.b32 p, %6, 0;\n"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n"
      "}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// 32 consecutive FP32 columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor, K-major, 128-byte swizzle: rows of 128
// bytes, 8-row groups 1024 bytes apart.  The tile base must be 1024-byte
// aligned; a K offset inside the swizzle atom is added to the start address.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);          // start address
  d |= (uint64_t)(16u >> 4) << 16;                    // leading byte offset (unused here)
  d |= (uint64_t)(1024u >> 4) << 32;                  // stride byte offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;                             // descriptor version
  d |= (uint64_t)2 << 61;                             // 128-byte swizzle
  return d;
}

// Descriptor of a contiguous 32-row x 16-byte block-scale chunk (no swizzle,
// 8-row core matrices 128 bytes apart).
__device__ __forceinline__ uint64_t smem_desc_sf(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(128u >> 4) << 32;                   // stride byte offset
  d |= (uint64_t)1 << 46;
  return d;
}

// Instruction descriptor of tcgen05.mma kind::mxf4nvf4: E2M1 x E2M1, UE4M3
// block scales, both operands K-major, dense, M x N.
__host__ __device__ constexpr uint32_t idesc_fp4(int M, int N) {
  return (1u << 7)                         // A format: E2M1
         | (1u << 10)                      // B format: E2M1
         | ((uint32_t)(N >> 3) << 17)      // N / 8
         | (0u << 23)                      // scale format: UE4M3
         | ((uint32_t)(M >> 4) << 24);     // M / 16
}

// ---------------------------------------------------------------------------
// Cluster helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_map(const void* local_smem, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local_smem)), "r"(rank));
  return remote;
}

// Store a 32-bit word at the same shared-memory offset in CTA `rank` (one
// single-copy-atomic access).
__device__ __forceinline__ void st_shared_cluster_u32(const void* local_smem, uint32_t rank, uint32_t v) {
  asm volatile("st.relaxed.cluster.shared::cluster.u32 [%0], %1;" ::"r"(cluster_map(local_smem, rank)), "r"(v)
               : "memory");
}

__device__ __forceinline__ uint32_t ld_shared_relaxed_u32(const void* local_smem) {
  uint32_t v;
  asm volatile("ld.relaxed.cluster.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smem_u32(local_smem)) : "memory");
  return v;
}

// Arrival on a grid-wide completion counter: an atomic add with
// acquire-release semantics at GPU scope.  Called by one thread right after a
// CTA barrier, it publishes everything the CTA wrote before the barrier, and
// (followed by another barrier) makes everything earlier arrivals published
// visible to the whole CTA.  Returns the counter's previous value.
__device__ __forceinline__ uint32_t arrive_acq_rel_gpu(uint32_t* counter) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(counter) : "memory");
  return old;
}

__device__ __forceinline__ uint32_t ld_acquire_gpu_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Wait until *counter >= target (acquire, GPU scope), for at most
// ~timeout_ns; gives up early once `abort` is raised.  False if it gave up.
__device__ __forceinline__ bool wait_counter_acquire(const uint32_t* counter, uint32_t target, volatile int* abort,
                                                     uint64_t timeout_ns = 2000000000ull) {
  if (ld_acquire_gpu_u32(counter) >= target) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    __nanosleep(32);
    if (ld_acquire_gpu_u32(counter) >= target) return true;
    if ((it & 63u) == 0) {
      if (abort != nullptr && *abort) return false;
      if (global_timer_ns() - t0 > timeout_ns) return false;
    }
  }
}

// Barrier among `nthreads` threads (whole warps) on hardware barrier `id`.
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------------------
// NVFP4 conversions and the block quantizer
// ---------------------------------------------------------------------------

// E4M3 byte of v: round to nearest even, saturating at +-448.
__device__ __forceinline__ uint32_t cvt_e4m3(float v) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
  return (uint32_t)(r & 0xFFu);
}

// Two E2M1 codes packed in a byte: `lo` in bits 0-3, `hi` in bits 4-7; round
// to nearest even, saturating at +-6.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{\n"
      ".reg .b8 t;\n"
      "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n"
      "cvt.u32.u8 %0, t;\n"
      "}\n"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r & 0xFFu;
}

// Exact value of a non-negative E4M3 byte (sign ignored; NaN never produced).
__device__ __forceinline__ float e4m3_value(uint32_t b) {
  const uint32_t e = (b >> 3) & 0xFu, m = b & 7u;
  if (e == 0) return (float)m * 0.001953125f;                    // m * 2^-9
  return __uint_as_float(((e + 120u) << 23) | (m << 20));        // (1 + m/8) * 2^(e-7)
}

// Global scale 2688 / amax (amax >= 0): 1 for amax == 0, FLT_MAX when the
// quotient overflows.
__device__ __forceinline__ float nvfp4_global_scale(float amax) {
  if (!(amax > 0.0f)) return 1.0f;
  const float g = __fdiv_rn(2688.0f, amax);
  return isinf(g) ? 3.402823466e38f : g;
}

// Quantize one 16-element block given the global scale: returns the E4M3
// scale byte and writes 8 packed code bytes (element 2i low nibble).
__device__ __forceinline__ uint32_t nvfp4_quant_block16(const float (&v)[16], float gs, uint2& packed) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const float sf32 = __fdiv_rn(__fmul_rn(amax, gs), 6.0f);
  const uint32_t sf = cvt_e4m3(sf32);
  const float sfv = e4m3_value(sf);
  uint32_t w0 = 0, w1 = 0;
  if (sfv > 0.0f) {
    const float q = __fdiv_rn(gs, sfv);
#pragma unroll
    for (int i = 0; i < 4; ++i) w0 |= cvt_e2m1x2(__fmul_rn(v[2 * i], q), __fmul_rn(v[2 * i + 1], q)) << (8 * i);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      w1 |= cvt_e2m1x2(__fmul_rn(v[8 + 2 * i], q), __fmul_rn(v[8 + 2 * i + 1], q)) << (8 * i);
  }
  packed = make_uint2(w0, w1);
  return sf;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two floats rounded to bf16 (nearest even), lo in the low half of the word.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// 16 bf16 values (two 16-byte words) widened to float.
__device__ __forceinline__ void bf16x16_to_f32(const uint4& a, const uint4& b, float (&v)[16]) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v[2 * i] = bf16_lo(w[i]);
    v[2 * i + 1] = bf16_hi(w[i]);
  }
}

// One warp requantizes one FP32 row h [I] (I a multiple of 128) with the
// row's global scale gs into the operand layout at row `prow` of an operand
// whose rows hold i_pad elements: block scales and codes (codes and scales
// share the operand buffer).  All 32 lanes must call it.  L2 loads: the row
// may have been written by other CTAs.
__device__ __forceinline__ void requant_row_warp(const float* __restrict__ hr, int I, int i_pad, size_t prow, float gs,
                                                 uint8_t* __restrict__ h_codes, int lane) {
  const int nblk = I / SF_VEC, k16_row = i_pad / SF_VEC;
  for (int b0 = 0; b0 < nblk; b0 += 32) {  // nblk = I/16, a multiple of 8: uniform bound
    const int b = b0 + lane;
    uint2 packed = make_uint2(0u, 0u);
    uint32_t sf = 0;
    if (b < nblk) {
      float v[16];
      const float4* src = reinterpret_cast<const float4*>(hr + 16 * b);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 f = __ldcg(src + q);
        v[4 * q] = f.x;
        v[4 * q + 1] = f.y;
        v[4 * q + 2] = f.z;
        v[4 * q + 3] = f.w;
      }
      sf = nvfp4_quant_block16(v, gs, packed);
    }
    // blocks 4m..4m+3 have consecutive scale bytes: one 32-bit store
    const uint32_t sf4 = sf | (__shfl_down_sync(0xffffffffu, sf, 1) << 8) | (__shfl_down_sync(0xffffffffu, sf, 2) << 16) |
                         (__shfl_down_sync(0xffffffffu, sf, 3) << 24);
    if (b < nblk) {
      *reinterpret_cast<uint2*>(h_codes + operand_offset(prow, 8 * b, i_pad / 2)) = packed;
      if ((lane & 3) == 0) *reinterpret_cast<uint32_t*>(h_codes + sf_atom_offset(prow, b, k16_row)) = sf4;
    }
  }
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

}  // namespace moe
