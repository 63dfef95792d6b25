// kernels.h - host-side launchers of the sm_103a kernels (internal interface
// between the C ABI in moe_host.cu and the kernel translation units).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// ---- routing (kernels_route.cu) ----
// Raises the router kernel's dynamic shared-memory cap to what (H, E) needs;
// never lowers it (the cap is shared by every handle on the device).
cudaError_t router_setup(int H, int E);
// Raises the cap of every router instantiation to `bytes` (never lowers it).
cudaError_t router_setup_max(int bytes);
// Dynamic shared memory one router launch for (H, E) needs.
int router_smem_bytes(int H, int E);
cudaError_t launch_router_logits(const void* x, const void* gate_w, const float* bias, float* logits, int T,
                                 int H, int E, cudaStream_t s);
cudaError_t launch_topk(const float* logits, int T, int E, int K, int32_t* topk_ids, float* topk_w,
                        cudaStream_t s);
struct PermuteOut {
  int32_t* expert_offsets;  // [E+1]
  int32_t* src_of_row;      // [R]
  int32_t* row_of_src;      // [R]
  int32_t* pad_row_of_src;  // [R]
  int32_t* src_of_padrow;   // [Rpad]
  int4* tiles;              // [tile bound] {expert, first padded row, valid rows, first activation row}
  int32_t* num_tiles;       // [1]
};
// tile_rows: 128 rows per GEMM tile.
cudaError_t launch_permute(const int32_t* topk_ids, int T, int K, int E, int tile_rows, const PermuteOut& o,
                           cudaStream_t s);

// ---- quantization (kernels_quant.cu) ----
// static_gs: nullptr for per-token global scales, else the calibrated
// per-tensor scale (device scalar) every token uses.
cudaError_t launch_act_quant(const void* x, int T, int H, int K, const int32_t* pad_row_of_src,
                             uint8_t* a_codes, uint8_t* a_sf, float* gs_rows,
                             const float* static_gs, cudaStream_t s);
cudaError_t launch_weight_amax(const void* w, int E, int N, int Kd, uint32_t* amax_bits, cudaStream_t s);
// Weights go to the pair-tile layout (wpair_offset).  interleave: 0 = rows
// in caller order; 1 = w13 gate/up rows interleaved in chunks of 64 so that
// internal chunk f (128 rows) is [gate f, up f].
cudaError_t launch_weight_quant(const void* w, int E, int N, int Kd, int Kpad, int interleave,
                                const uint32_t* amax_bits, uint8_t* codes, uint8_t* sf, float* gs,
                                cudaStream_t s);
// pair: the operand is a weight buffer (pair-tile layout).
cudaError_t launch_export_rows(const uint8_t* codes, const uint8_t* sf, const float* gs_rows, int n_rows,
                               int Kd, int Kpad, const int32_t* row_map, int map_stride, int row_map_mode,
                               int E_rows, int pair, uint8_t* out_codes, uint8_t* out_sf, float* out_gs,
                               cudaStream_t s);
cudaError_t launch_convert(const float* in, uint8_t* e2m1, uint8_t* e4m3, int64_t n, cudaStream_t s);
cudaError_t launch_sf_to_atoms(const uint8_t* sf, int rows, int k16, uint8_t* atoms, cudaStream_t s);
cudaError_t launch_codes_to_tiled(const uint8_t* codes, int rows, int row_bytes, uint8_t* tiled, cudaStream_t s);

// ---- finalize (kernels_quant.cu) ----
// shared: nullptr, or bf16 rows [T][H] of a shared expert added to the
// routed sum in FP32 and the sum scaled by shared_scale before the bf16
// rounding.
cudaError_t launch_finalize_atomic(const float* out_acc, const uint16_t* shared, float shared_scale, void* out, int T,
                                   int H, cudaStream_t s);
// ybuf: bf16 rows [t * K + j][H] of the weighted-sum operands.
cudaError_t launch_finalize_ordered(const uint16_t* ybuf, const float* topk_w, const uint16_t* shared,
                                    float shared_scale, void* out, int T, int H, int K, cudaStream_t s);
// The shared expert's tile list: ceil(T/128) tiles of expert 0 over rows
// 0..T-1 ({0, 128 i, valid rows, 128 i}).
cudaError_t launch_shared_tiles(int T, int4* tiles, int32_t* num_tiles, cudaStream_t s);

// ---- block-scaled FP4 GEMMs (kernels_gemm.cu) ----
// Small batches (T <= SMALL_BATCH_TOKENS): router logits, per-token
// quantization, top-k and the expert grouping in one kernel.  Every token is
// quantized once into one shared activation tile (row t = token t), which
// every expert's w13 GEMM reads; the expanded row (token t, slot j) of expert
// e is padded row e*128 + t.
constexpr int SMALL_BATCH_TOKENS = 64;
struct FrontArgs {
  // tensor map of the router weight viewed as [H/8][8][E] bf16 whose box
  // reaches one row and 8 columns past the data (zeros): the staged rows and
  // 8-row chunks come out padded (see launch_front_small)
  CUtensorMap wg_map;
  int wg_map_ok;              // 0: stage rows with plain bulk copies instead
  const void* x;              // [T, H] bf16
  const void* gate_w;         // [H, E] bf16
  const float* bias;          // [E] or nullptr
  int T, H, E, K;
  float* logits;              // [T, E]
  int32_t* topk_ids;          // [T, K]
  float* topk_w;              // [T, K]
  uint8_t* a_codes;           // shared activation tile (operand layout, rows 0..T-1)
  float* gs_rows;             // [T] per-token global scales
  float* out_acc;             // [T, H] cleared here (atomic finalize), or nullptr
  int32_t* src_of_padrow;     // [E*128]
  int32_t* expert_offsets;    // [E+1]
  int32_t* src_of_row;        // [T*K]
  int32_t* row_of_src;        // [T*K]
  int32_t* pad_row_of_src;    // [T*K]
  int4* tiles;                // one tile per expert with rows
  int32_t* num_tiles;
  uint32_t* sync;             // FRONT_SYNC_WORDS counters, zero between launches
  const float* static_gs;     // calibrated per-tensor scale (static contract), or nullptr
  // The GEMMs run the all-experts schedule: they take the activations and
  // the routing from the sync counters and do not wait for the grouping
  // (expert_offsets, src_of_row, row_of_src, pad_row_of_src, tiles), which
  // the last front CTA to publish its routing derives off their path.
  int all_experts;
  int* status;                // device status word (a bounded wait that ran out)
};
constexpr int FRONT_SYNC_WORDS = 64;
// Words of the front kernel's sync block used by the all-experts small-batch
// path (returned to zero by the w2 GEMM): front CTAs that quantized their
// tokens, front CTAs that routed their tokens, the dynamic work counter of
// the w13 GEMM, and its requantization counters.
constexpr int FRONT_SYNC_A_READY = 0;
constexpr int FRONT_SYNC_ROUTED = 1;
constexpr int FRONT_SYNC_WORK = 2;
constexpr int FRONT_SYNC_RQ_ROW = 3;     // the w13 GEMM's requantization: next expanded row
constexpr int FRONT_SYNC_RQ_EXPERT = 4;  // and next expert whose unrouted rows' maxima return to zero
constexpr int FRONT_SYNC_RESET = 5;      // words the w2 GEMM returns to zero
// CTAs of the front kernel's grid for T tokens and E experts.
int front_ctas(int T, int E);
cudaError_t front_setup(int H, int E);
// Fills a.wg_map / a.wg_map_ok for a.gate_w, then launches.
cudaError_t launch_front_small(FrontArgs& a, cudaStream_t s);

struct GemmArgs {
  const uint8_t* a_codes;     // A operand (codes and block scales), operand layout
  const uint8_t* b_codes;     // B operand (codes and block scales), operand layout
  int k_stages;               // Kpad / 256
  // {expert, first padded row, valid rows, first activation row}.  The padded
  // row indexes the outputs (intermediate, scales, src_of_padrow); the w13
  // GEMM reads its activation rows from the fourth field, which equals the
  // second in the expanded layout and is 0 in the shared small-batch tile.
  const int4* tiles;
  const int32_t* num_tiles;   // device tile count
  int b_rows_per_expert;      // 2I (w13) or H (w2)
  const float* gs_rows;       // global scale per activation row
  const float* gs_w;          // global scale per expert
  // w13 epilogue: SwiGLU + requantization into the w2 operand (codes and
  // block scales share one operand buffer)
  uint8_t* h_codes;
  uint8_t* h_sf;
  float* h_gs;
  int i_pad;                  // K of the w2 GEMM (padded intermediate width)
  // padded row -> token * top_k + slot, or -1 for a row no token routed here
  // (both epilogues skip such rows)
  const int32_t* src_of_padrow;
  // w2 epilogue: top-k weighted reduction
  const float* topk_w;
  int top_k;
  float* out_acc;             // atomic mode
  uint16_t* ybuf;             // ordered mode: bf16 rows [token * top_k + slot][hidden]
  int hidden;
  // plain epilogue (tests)
  float* d;
  int ldd;
  int n_tiles;                // 128-column tiles per row tile (w2 / plain)
  int m_tiles;                // row tiles (plain)
  int* status;                // device status word
  // Before its dependency wait, each CTA may warm L2 with the weights of its
  // first prefetch_units work units, taking tile i to be expert i's (exact in
  // the small-batch layout when every expert has rows; only a hint).
  int prefetch_units;
  int num_experts;
  // small-batch w13 without clusters: column pairs per m-tile (I/128), the
  // FP32 SwiGLU rows [padded row][i_pad] and the per-row maxima (zero on
  // entry; the requantization kernel returns them to zero)
  int w13_pairs;
  float* hbuf;
  float* row_amax;
  // static per-tensor contract: the w2 input's calibrated global scale per
  // expert (the w13 epilogue requantizes with it directly), or nullptr
  const float* h_gs_static;
  // Small batches in which nearly every expert has rows (w13s and w2): the
  // units are every expert's tile in expert order (tile i = expert i, padded
  // rows i*128 .. i*128 + small_T - 1), independent of the tile list, so the
  // kernel streams weights into its ring before the dependency wait.
  int all_experts;
  int small_T;
  // all-experts small-batch w13 only: the front kernel's sync words and its
  // grid size (dynamic schedule, no dependency wait); nullptr otherwise
  uint32_t* front_sync;
  int front_ctas;
  // all-experts path: finished w13 column pairs per expert (the w13 GEMM
  // counts and waits on them to requantize, the w2 GEMM returns them to
  // zero); the w13 GEMM's requantization also needs the top-k ids [T, K],
  // top_k, and the intermediate width I
  uint32_t* expert_done;
  const int32_t* topk_ids_small;
  int inter;
  // w2 of the all-experts path: the front kernel's sync words and the
  // per-expert counts, returned to zero after the dependency wait
  uint32_t* reset_sync;
  // SwiGLU sigmoid: 0 = 1/2 + tanh.approx(g/2)/2, 1 = 1 / (1 + expf(-g))
  // with an IEEE division
  int accurate_sigmoid;
};

cudaError_t gemm_setup_attributes(int w13_chunks);
// Thread-block clusters of the w13 kernel (w13_chunks CTAs each) that fit on
// the device at once; 0 if none.
int gemm_w13_max_clusters(int w13_chunks, int a_rows);
// Persistent launches: the w13 kernel runs n_clusters clusters of n_chunks
// CTAs; the w2 / plain kernels run n_ctas CTAs.  Each walks a static tile list.
// a_rows: rows of the activation operand per tile (64 or 128; every tile of
// the list must have at most that many valid rows).
cudaError_t launch_gemm_w13(const GemmArgs& a, int n_chunks, int n_clusters, int a_rows, cudaStream_t s);
// Small batches (64-row tiles sharing one activation tile): the w13 GEMM
// without clusters over n_ctas CTAs, then the per-row requantization of its
// FP32 output into the w2 operand.  resident keeps the shared activation tile
// in shared memory for the whole kernel (K <= 2048).
cudaError_t launch_gemm_w13s(const GemmArgs& a, int n_ctas, bool resident, cudaStream_t s);
// The row of expanded row i (token * K + slot) is row_map[i], or with topk_ids
// given the small-batch padded row topk_ids[i] * 128 + i / K.
struct RequantAllExperts {
  const int32_t* src_of_padrow;  // routing of the padded rows
  const uint32_t* expert_done;   // finished w13 column pairs per expert
  const uint32_t* front_sync;    // the front kernel's counters
  int pairs;                     // column pairs per expert (I / 128)
  int front_ctas;
  int E;
};
// all: the all-experts path (nullptr otherwise).  The kernel does not wait
// for the w13 GEMM up front: each row starts once its expert's column pairs
// are all done (and the routing is), and every CTA waits for the GEMM only at
// its end - after which it returns to zero the maxima of the rows of tokens
// that did not route to an expert (the GEMM forms every row until the
// routing is known).
cudaError_t launch_requant_rows(const float* hbuf, float* row_amax, const int32_t* row_map,
                                const int32_t* topk_ids, int K, int n_rows, int I, int i_pad, uint8_t* h_codes,
                                float* h_gs, const RequantAllExperts* all, int* status, cudaStream_t s);
cudaError_t launch_gemm_w2(const GemmArgs& a, int n_ctas, bool ordered, int a_rows, cudaStream_t s);
cudaError_t launch_gemm_plain(const GemmArgs& a, int n_ctas, cudaStream_t s);

}  // namespace moe
