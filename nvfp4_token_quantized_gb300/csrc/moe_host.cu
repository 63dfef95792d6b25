// moe_host.cu - the C ABI (include/moe_nvfp4.h): handle lifetime, worst-case
// buffer planning, online weight conversion, in-place refresh, and the
// stream-ordered launch sequence of one forward.
//
// Buffers are sized once at moe_create from max_num_tokens ("size CuteDSL MoE
// allgather buffers for the worst-case forward", Implementation items 1-3);
// a larger forward is refused with MOE_ERR_TOO_MANY_TOKENS.  Weight reload
// rewrites the same buffers ("CuTe DSL backend gets per-token NVFP4 online
// quantization and reload", Implementation item 3 and the refresh snippet).
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "../../include/moe_nvfp4.h"
#include "common.cuh"
#include "kernels.h"

using namespace moe;

struct moe_handle {
  moe_config cfg{};
  int H = 0, I = 0, E = 0, K = 0, Tmax = 0;
  int Ipad = 0;         // intermediate width padded to a multiple of 256 (w2 GEMM K)
  int Rmax = 0;         // Tmax * K
  int Rpad = 0;         // padded expert-grouped rows, worst case
  int tile_cap = 0;     // worst-case number of GEMM tiles
  int num_sms = 0;      // persistent w2 grid
  int w13_clusters[2] = {0, 0};  // persistent w13 grid (clusters of I/128 CTAs), 64- / 128-row tiles
  bool deterministic = false;
  bool static_scales = false;   // MOE_FLAG_STATIC_ACT_SCALES
  bool static_set = false;      // moe_set_static_scales has been called
  bool loaded = false;
  moe_weight_desc w13_desc{}, w2_desc{};
  int last_T = -1;
  bool last_small = false;  // the last forward used the shared small-batch activation tile
  std::string err;
  size_t bytes = 0;
  std::vector<void*> allocs;

  // weights (internal operand layouts)
  uint8_t *w13_codes = nullptr, *w13_sf = nullptr, *w2_codes = nullptr, *w2_sf = nullptr;
  float *gs_w13 = nullptr, *gs_w2 = nullptr;
  uint32_t* amax_bits = nullptr;  // [2E]

  // routing workspace
  float* logits = nullptr;
  int32_t *topk_ids = nullptr, *expert_offsets = nullptr;
  float* topk_w = nullptr;
  int32_t *src_of_row = nullptr, *row_of_src = nullptr, *pad_row_of_src = nullptr, *src_of_padrow = nullptr;
  int4* tiles = nullptr;
  int32_t* num_tiles = nullptr;
  uint32_t* front_sync = nullptr;  // completion counters of the small-batch front kernel
  uint32_t* expert_done = nullptr; // all-experts path: finished w13 column pairs per expert [256]
  // Shared expert (Is > 0): its NVFP4 weights, the token-ordered activation
  // and intermediate operands (row t = token t, 128-row tiles), the
  // identity row map, its tile list, its bf16 output rows, and the second
  // stream with the fork / join events.
  int Is = 0, Ipad_s = 0, Tpad_s = 0;
  bool shared_loaded = false;
  uint8_t *sw13_codes = nullptr, *sw2_codes = nullptr, *s_a_codes = nullptr, *s_h_codes = nullptr;
  float *gs_sw13 = nullptr, *gs_sw2 = nullptr, *s_gs_rows = nullptr, *s_h_gs = nullptr;
  uint32_t* s_amax_bits = nullptr;
  int32_t *s_ident = nullptr, *s_num_tiles = nullptr;
  int4* s_tiles = nullptr;
  uint16_t* s_ybuf = nullptr;
  float *s_hbuf = nullptr, *s_row_amax = nullptr;  // small batches: FP32 SwiGLU rows [128][Ipad_s], row maxima
  int s_clusters[2] = {0, 0};
  cudaStream_t side = nullptr;
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
  float* static_x_gs = nullptr;    // static contract: the w13 input's calibrated scale [1]
  float* static_h_gs = nullptr;    // static contract: the w2 input's calibrated scale per expert [E]
  float* hbuf = nullptr;           // small batches: FP32 SwiGLU rows [E*128][Ipad]
  float* row_amax = nullptr;       // small batches: their row maxima [E*128], zero between forwards

  // operands of the two GEMMs
  uint8_t *a_codes = nullptr, *a_sf = nullptr, *h_codes = nullptr, *h_sf = nullptr;
  float *gs_rows = nullptr, *h_gs = nullptr;
  // atomic finalize (small batches): FP32 accumulator [min(Tmax, 64), H];
  // ordered finalize (deterministic mode, and every batch above 64 tokens):
  // bf16 rows [Tmax * K, H], one per (token, slot)
  float* out_acc = nullptr;
  uint16_t* ybuf = nullptr;

  // staging for moe_forward_host
  void *stage_x = nullptr, *stage_gate = nullptr, *stage_out = nullptr;
  float* stage_bias = nullptr;

  // host-visible device status word (mapped pinned memory)
  int* status_host = nullptr;
  int* status_dev = nullptr;


  // stage timing: events[0] before the first kernel, events[i+1] after stage i
  bool timing = false;
  cudaEvent_t events[MOE_NUM_STAGES + 1] = {};
};

namespace {

void set_err(moe_handle* h, const char* fmt, ...) {
  if (!h) return;
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  h->err = buf;
}

moe_status cuda_fail(moe_handle* h, cudaError_t e, const char* what) {
  set_err(h, "%s: %s", what, cudaGetErrorString(e));
  return MOE_ERR_CUDA;
}

#define CK(h, call)                                             \
  do {                                                          \
    cudaError_t e_ = (call);                                    \
    if (e_ != cudaSuccess) return cuda_fail((h), e_, #call);    \
  } while (0)

template <typename T>
moe_status dalloc(moe_handle* h, T** p, size_t bytes) {
  bytes = (bytes + 255) & ~size_t(255);
  if (bytes == 0) bytes = 256;
  void* q = nullptr;
  cudaError_t e = cudaMalloc(&q, bytes);
  if (e != cudaSuccess) return cuda_fail(h, e, "cudaMalloc");
  e = cudaMemset(q, 0, bytes);
  if (e != cudaSuccess) {
    cudaFree(q);
    return cuda_fail(h, e, "cudaMemset");
  }
  h->allocs.push_back(q);
  h->bytes += bytes;
  *p = reinterpret_cast<T*>(q);
  return MOE_OK;
}

#define TRY(x)                         \
  do {                                 \
    moe_status s_ = (x);               \
    if (s_ != MOE_OK) return s_;       \
  } while (0)

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

bool ranges_overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
  return a0 < b0 + nb && b0 < a0 + na;
}

int device_of(const void* p) {
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged) return -1;
  return at.device;
}

// Forwards of at most SMALL_BATCH_TOKENS tokens quantize every token once
// into one shared 64-row activation tile that all experts' w13 GEMMs read:
// their experts get a handful of rows each, no expanded copy of the
// activations is made, and reserving 64 instead of 128 activation rows per
// pipeline stage leaves room for a deeper weight-streaming ring.
int tile_rows_for(int T) { return T <= SMALL_BATCH_TOKENS ? 64 : 128; }

// Small batches: 128-column units whose weights each GEMM CTA streams into
// L2 before its dependency wait - its first 256-column pair.  Measured on the
// decode workload: one pair per CTA is as fast as two and faster than none;
// prefetching from the front kernel instead slowed the front kernel more
// than it saved.
constexpr int W13_PREFETCH_UNITS = 2;
constexpr int W2_PREFETCH_UNITS = 2;
// With the all-experts schedule the prefetched units are exactly the CTA's
// first ones: two column pairs.
constexpr int W13_PREFETCH_UNITS_ALL = 4;

// Worst-case number of GEMM tiles of tile_rows rows when T tokens each pick
// K of E experts (each tile is padded to its own 128-row block).
int tile_bound(int T, int K, int E, int tile_rows) {
  const long R = (long)T * K;
  const long busy = std::min<long>(E, R);
  const long a = (R + (tile_rows - 1L) * busy) / tile_rows;
  const long b = busy * ((T + tile_rows - 1L) / tile_rows);
  return (int)std::max<long>(1, std::min(a, b));
}

moe_status check_weight_desc(moe_handle* h, const moe_weight_desc* d, const void* ptr, int64_t d0, int64_t d1,
                             int64_t d2, const char* name) {
  if (!d || !ptr) {
    set_err(h, "%s: NULL pointer or descriptor", name);
    return MOE_ERR_INVALID_ARG;
  }
  if (d->dtype != MOE_DTYPE_BF16) {
    set_err(h, "%s: dtype must be MOE_DTYPE_BF16", name);
    return MOE_ERR_INVALID_ARG;
  }
  if (d->dims[0] != d0 || d->dims[1] != d1 || d->dims[2] != d2) {
    set_err(h, "%s: shape [%lld, %lld, %lld] does not match the configuration [%lld, %lld, %lld]", name,
            (long long)d->dims[0], (long long)d->dims[1], (long long)d->dims[2], (long long)d0, (long long)d1,
            (long long)d2);
    return MOE_ERR_INVALID_ARG;
  }
  if (d->device != h->cfg.device || device_of(ptr) != h->cfg.device) {
    set_err(h, "%s: data is not on device %d", name, h->cfg.device);
    return MOE_ERR_INVALID_ARG;
  }
  if (!aligned16(ptr)) {
    set_err(h, "%s: pointer must be 16-byte aligned", name);
    return MOE_ERR_INVALID_ARG;
  }
  return MOE_OK;
}

bool same_desc(const moe_weight_desc& a, const moe_weight_desc& b) {
  return a.dims[0] == b.dims[0] && a.dims[1] == b.dims[1] && a.dims[2] == b.dims[2] && a.dtype == b.dtype &&
         a.device == b.device;
}

moe_status quantize_weights(moe_handle* h, const void* w13, const void* w2, cudaStream_t s) {
  CK(h, cudaMemsetAsync(h->amax_bits, 0, sizeof(uint32_t) * 2 * h->E, s));
  CK(h, launch_weight_amax(w13, h->E, 2 * h->I, h->H, h->amax_bits, s));
  CK(h, launch_weight_amax(w2, h->E, h->H, h->I, h->amax_bits + h->E, s));
  CK(h, launch_weight_quant(w13, h->E, 2 * h->I, h->H, h->H, 1, h->amax_bits, h->w13_codes, h->w13_sf, h->gs_w13,
                            s));
  CK(h, launch_weight_quant(w2, h->E, h->H, h->I, h->Ipad, 0, h->amax_bits + h->E, h->w2_codes, h->w2_sf, h->gs_w2,
                            s));
  return MOE_OK;
}

struct DeviceGuard {
  int prev = -1;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (prev != dev) cudaSetDevice(dev);
  }
  ~DeviceGuard() {
    int cur;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

// Stage boundary i.  Inside a stream capture the record becomes an external
// event node (re-recorded on every replay); outside it is a plain record.
cudaError_t mark(moe_handle* h, int i, cudaStream_t s) {
  if (!h->timing) return cudaSuccess;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(s, &cs);
  if (e != cudaSuccess) return e;
  if (cs == cudaStreamCaptureStatusActive) return cudaEventRecordWithFlags(h->events[i], s, cudaEventRecordExternal);
  return cudaEventRecord(h->events[i], s);
}

// The shared expert on the handle's second stream, forked from `s`: x
// quantized per token into token-ordered rows (the same arithmetic as the
// routed experts' input), the w13 GEMM with the fused SwiGLU and
// requantization epilogue on clusters of Is/128 CTAs, the w2 GEMM storing
// bf16 rows; the join event is recorded at the end ("SM10X Command-A-Plus
// decode 2.3x faster, BCG capture memory -78%", key source listing: the
// shared experts on the 'alt' stream while gate, top-k and the routed
// experts stay on the main stream).
// CTAs of the shared expert's GEMMs up to 64 tokens: its w13 column pairs,
// or its w2 column-tile pairs, whichever is more.
int shared_gemm_ctas(const moe_handle* h) { return std::max(h->Is / 128, h->H / 256); }

moe_status shared_branch(moe_handle* h, const void* x, int T, cudaStream_t s) {
  const int H = h->H;
  const int ntiles = (T + 127) / 128;
  const int a_rows = T <= SMALL_BATCH_TOKENS ? 64 : 128;
  CK(h, cudaEventRecord(h->ev_fork, s));
  CK(h, cudaStreamWaitEvent(h->side, h->ev_fork, 0));
  CK(h, launch_shared_tiles(T, h->s_tiles, h->s_num_tiles, h->side));
  CK(h, launch_act_quant(x, T, H, 1, h->s_ident, h->s_a_codes, h->s_a_codes, h->s_gs_rows, nullptr, h->side));
  GemmArgs g{};
  g.status = h->status_dev;
  g.tiles = h->s_tiles;
  g.num_tiles = h->s_num_tiles;
  g.a_codes = h->s_a_codes;
  g.b_codes = h->sw13_codes;
  g.k_stages = H / STAGE_K;
  g.b_rows_per_expert = 2 * h->Is;
  g.gs_rows = h->s_gs_rows;
  g.gs_w = h->gs_sw13;
  g.h_codes = h->s_h_codes;
  g.h_sf = h->s_h_codes;
  g.h_gs = h->s_h_gs;
  g.i_pad = h->Ipad_s;
  g.src_of_padrow = h->s_ident;  // row t is token t
  g.num_experts = 1;
  g.accurate_sigmoid = (h->cfg.flags & MOE_FLAG_ACCURATE_SIGMOID) != 0;
  if (T <= SMALL_BATCH_TOKENS) {
    // one 64-row tile: column pairs spread over single CTAs (no cluster has
    // to find SMs of one GPC free next to the routed GEMMs), then the row
    // requantization
    g.w13_pairs = h->Is / 128;
    g.hbuf = h->s_hbuf;
    g.row_amax = h->s_row_amax;
    CK(h, launch_gemm_w13s(g, std::min(h->num_sms, g.w13_pairs), false, h->side));
    CK(h, launch_requant_rows(h->s_hbuf, h->s_row_amax, h->s_ident, nullptr, 1, T, h->Is, h->Ipad_s, h->s_h_codes,
                              h->s_h_gs, nullptr, h->status_dev, h->side));
  } else {
    CK(h, launch_gemm_w13(g, h->Is / 128, std::min(h->s_clusters[a_rows == 128], ntiles), a_rows, h->side));
  }
  GemmArgs g2{};
  g2.status = h->status_dev;
  g2.tiles = h->s_tiles;
  g2.num_tiles = h->s_num_tiles;
  g2.a_codes = h->s_h_codes;
  g2.b_codes = h->sw2_codes;
  g2.k_stages = h->Ipad_s / STAGE_K;
  g2.b_rows_per_expert = H;
  g2.gs_rows = h->s_h_gs;
  g2.gs_w = h->gs_sw2;
  g2.src_of_padrow = h->s_ident;
  g2.top_k = 1;
  g2.ybuf = h->s_ybuf;  // (ordered epilogue: row t of the shared output)
  g2.hidden = H;
  g2.n_tiles = H / TILE_N;
  g2.num_experts = 1;
  CK(h, launch_gemm_w2(g2, std::min(h->num_sms, ntiles * g2.n_tiles / 2), true, a_rows, h->side));
  CK(h, cudaEventRecord(h->ev_join, h->side));
  return MOE_OK;
}

moe_status forward_impl(moe_handle* h, const void* x, const void* gate_w, const float* bias, void* out, int T,
                        cudaStream_t s) {
  const int H = h->H, E = h->E, K = h->K;
  if (T > 0) {
    const int tile_rows = tile_rows_for(T);
    const bool small = T <= SMALL_BATCH_TOKENS;
    if (h->Is > 0) TRY(shared_branch(h, x, T, s));
    // Above the small-batch size the FP32 atomic reduction of R x H partial
    // rows saturates L2; the ordered finalize (bf16 rows, fixed slot order)
    // moves half the bytes with plain stores and is deterministic as well.
    const bool ordered = h->deterministic || !small;
    // Up to 64 tokens the routed GEMMs are persistent with one CTA per SM
    // and start early; with a shared expert they leave its GEMM CTAs SMs of
    // their own so that the two streams overlap instead of queueing.
    const int gemm_sms = (h->Is > 0 && small) ? std::max(h->num_sms / 2, h->num_sms - shared_gemm_ctas(h))
                                              : h->num_sms;
    // Small batches in which nearly every expert gets a row (T*K >= 4E: with
    // uniform routing at most e^-4 of the experts stay empty) run both GEMMs
    // over every expert in order: their weight streams need no routing
    // result and start before the front kernel finishes, and the expert
    // grouping moves off their path into the requantization kernel (the
    // static contract has no requantization kernel, so it keeps the tile
    // list).
    const bool all_experts = small && (long)T * K >= 4L * E && !h->static_scales;
    CK(h, mark(h, 0, s));
    if (small) {
      // one kernel for router, quantization, top-k and grouping; its time is
      // reported as the router stage, the next three stages as empty
      FrontArgs fa{};
      fa.x = x;
      fa.gate_w = gate_w;
      fa.bias = bias;
      fa.T = T;
      fa.H = H;
      fa.E = E;
      fa.K = K;
      fa.logits = h->logits;
      fa.topk_ids = h->topk_ids;
      fa.topk_w = h->topk_w;
      fa.a_codes = h->a_codes;
      fa.gs_rows = h->gs_rows;
      fa.out_acc = ordered ? nullptr : h->out_acc;
      fa.src_of_padrow = h->src_of_padrow;
      fa.expert_offsets = h->expert_offsets;
      fa.src_of_row = h->src_of_row;
      fa.row_of_src = h->row_of_src;
      fa.pad_row_of_src = h->pad_row_of_src;
      fa.tiles = h->tiles;
      fa.num_tiles = h->num_tiles;
      fa.sync = h->front_sync;
      fa.static_gs = h->static_scales ? h->static_x_gs : nullptr;
      fa.all_experts = all_experts;
      fa.status = h->status_dev;
      CK(h, launch_front_small(fa, s));
      for (int i = 1; i <= 4; ++i) CK(h, mark(h, i, s));
    } else {
      CK(h, launch_router_logits(x, gate_w, bias, h->logits, T, H, E, s));
      CK(h, mark(h, 1, s));
      CK(h, launch_topk(h->logits, T, E, K, h->topk_ids, h->topk_w, s));
      CK(h, mark(h, 2, s));
      PermuteOut po{h->expert_offsets, h->src_of_row, h->row_of_src, h->pad_row_of_src,
                    h->src_of_padrow,  h->tiles,      h->num_tiles};
      CK(h, launch_permute(h->topk_ids, T, K, E, tile_rows, po, s));
      CK(h, mark(h, 3, s));
      CK(h, launch_act_quant(x, T, H, K, h->pad_row_of_src, h->a_codes, h->a_sf, h->gs_rows,
                             h->static_scales ? h->static_x_gs : nullptr,
                             s));
      CK(h, mark(h, 4, s));
    }
    // bound on the tile count: one per expert with rows (small batches)
    const int tb = small ? std::min(E, T * K) : tile_bound(T, K, E, tile_rows);
    const int units_e = all_experts ? E : tb;
    GemmArgs g{};
    g.status = h->status_dev;
    g.tiles = h->tiles;
    g.num_tiles = h->num_tiles;
    // w13: A = expanded activations [Rpad, H], B = w13 [E*2I, H]
    g.a_codes = h->a_codes;
    g.b_codes = h->w13_codes;
    g.k_stages = H / STAGE_K;
    g.b_rows_per_expert = 2 * h->I;
    g.gs_rows = h->gs_rows;
    g.gs_w = h->gs_w13;
    g.h_codes = h->h_codes;
    g.h_sf = h->h_sf;
    g.h_gs = h->h_gs;
    g.i_pad = h->Ipad;
    g.src_of_padrow = h->src_of_padrow;
    g.num_experts = E;
    g.prefetch_units = small ? (all_experts ? W13_PREFETCH_UNITS_ALL : W13_PREFETCH_UNITS) : 0;
    g.all_experts = all_experts;
    g.small_T = T;
    if (all_experts) {  // dynamic schedule on the front kernel's counters
      g.front_sync = h->front_sync;
      g.front_ctas = front_ctas(T, E);
      g.expert_done = h->expert_done;
      g.topk_ids_small = h->topk_ids;
      g.top_k = K;
      g.inter = h->I;
    }
    g.h_gs_static = h->static_scales ? h->static_h_gs : nullptr;
    g.accurate_sigmoid = (h->cfg.flags & MOE_FLAG_ACCURATE_SIGMOID) != 0;
    if (small) {
      // every tile reads the one shared activation tile; no clusters: the
      // units spread over all SMs, and the requantization follows as its own
      // kernel.  The tile is streamed with the weights: keeping it resident
      // costs a ring stage, which measured slower.
      g.w13_pairs = h->I / 128;
      g.hbuf = h->hbuf;
      g.row_amax = h->row_amax;
      CK(h, launch_gemm_w13s(g, std::min(gemm_sms, units_e * g.w13_pairs), false, s));
      // (with static scales the w13 epilogue has already requantized; on the
      // all-experts path the w13 GEMM's CTAs requantize once out of units)
      if (!h->static_scales && !all_experts)
        CK(h, launch_requant_rows(h->hbuf, h->row_amax, nullptr, h->topk_ids, K, T * K, h->I, h->Ipad, h->h_codes,
                                  h->h_gs, nullptr, h->status_dev, s));
    } else {
      CK(h, launch_gemm_w13(g, h->I / 128, std::min(h->w13_clusters[tile_rows == 128], tb), tile_rows, s));
    }
    CK(h, mark(h, 5, s));
    // w2: A = requantized intermediate [Rpad, Ipad], B = w2 [E*H, Ipad]
    GemmArgs g2{};
    g2.status = h->status_dev;
    g2.tiles = h->tiles;
    g2.num_tiles = h->num_tiles;
    g2.a_codes = h->h_codes;
    g2.b_codes = h->w2_codes;
    g2.k_stages = h->Ipad / STAGE_K;
    g2.b_rows_per_expert = H;
    g2.gs_rows = h->h_gs;
    g2.gs_w = h->gs_w2;
    g2.src_of_padrow = h->src_of_padrow;
    g2.topk_w = h->topk_w;
    g2.top_k = K;
    g2.out_acc = h->out_acc;
    g2.ybuf = h->ybuf;
    g2.hidden = H;
    g2.n_tiles = H / TILE_N;
    g2.num_experts = E;
    g2.prefetch_units = small ? W2_PREFETCH_UNITS : 0;
    g2.all_experts = all_experts;
    g2.small_T = T;
    g2.reset_sync = all_experts ? h->front_sync : nullptr;
    g2.expert_done = h->expert_done;
    // units are pairs of 128-column tiles
    CK(h, launch_gemm_w2(g2, std::min(gemm_sms, units_e * g2.n_tiles / 2), ordered, tile_rows, s));
    CK(h, mark(h, 6, s));
    // the shared expert's rows join here (its stream's work is done)
    const uint16_t* shared = nullptr;
    float shared_scale = 1.0f;
    if (h->Is > 0) {
      CK(h, cudaStreamWaitEvent(s, h->ev_join, 0));
      shared = h->s_ybuf;
      shared_scale = (h->cfg.flags & MOE_FLAG_SHARED_AVERAGE) ? 0.5f : 1.0f;
    }
    if (ordered) CK(h, launch_finalize_ordered(h->ybuf, h->topk_w, shared, shared_scale, out, T, H, K, s));
    else CK(h, launch_finalize_atomic(h->out_acc, shared, shared_scale, out, T, H, s));
    CK(h, mark(h, 7, s));
  }
  h->last_T = T;
  h->last_small = T > 0 && T <= SMALL_BATCH_TOKENS;
  return MOE_OK;
}

}  // namespace

extern "C" {

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_TOO_MANY_TOKENS: return "MOE_ERR_TOO_MANY_TOKENS";
    case MOE_ERR_NOT_LOADED: return "MOE_ERR_NOT_LOADED";
    case MOE_ERR_METADATA_CHANGED: return "MOE_ERR_METADATA_CHANGED";
    case MOE_ERR_ALIAS: return "MOE_ERR_ALIAS";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_DEVICE_TIMEOUT: return "MOE_ERR_DEVICE_TIMEOUT";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
  }
  return "MOE_ERR_UNKNOWN";
}

moe_status moe_create(const moe_config* cfg, moe_handle** out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  if (!cfg) return MOE_ERR_INVALID_ARG;
  const int H = cfg->hidden, I = cfg->inter, E = cfg->num_experts, K = cfg->top_k, T = cfg->max_num_tokens;
  if (H <= 0 || I <= 0 || E <= 0 || K <= 0 || T <= 0) return MOE_ERR_INVALID_ARG;
  if (H % 256 || I % 128 || E % 8 || E > 256 || K > E || K > 16 || I / 128 > 16) return MOE_ERR_UNSUPPORTED;
  const int Is = cfg->shared_inter;
  if (Is < 0 || Is % 128 || Is / 128 > 16) return MOE_ERR_UNSUPPORTED;
  if (Is > 0 && (cfg->flags & MOE_FLAG_STATIC_ACT_SCALES)) return MOE_ERR_UNSUPPORTED;
  if ((long)T * K > (1L << 30)) return MOE_ERR_UNSUPPORTED;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || cfg->device < 0 || cfg->device >= ndev) {
    cudaGetLastError();
    return MOE_ERR_UNSUPPORTED;
  }
  cudaDeviceProp prop{};
  if (cudaGetDeviceProperties(&prop, cfg->device) != cudaSuccess || prop.major != 10 || prop.minor != 3) {
    cudaGetLastError();
    return MOE_ERR_UNSUPPORTED;
  }
  // the router's weight slice and activation rings share one CTA's memory
  if ((size_t)router_smem_bytes(H, E) > prop.sharedMemPerBlockOptin) return MOE_ERR_UNSUPPORTED;
  DeviceGuard dg(cfg->device);
  moe_handle* h = new moe_handle();
  h->cfg = *cfg;
  h->H = H;
  h->I = I;
  h->E = E;
  h->K = K;
  h->Tmax = T;
  h->Ipad = (I + 255) / 256 * 256;
  h->Rmax = T * K;
  // small batches: one tile (one 128-row block) per expert with rows
  h->tile_cap = std::max(tile_bound(T, K, E, 128), E);
  h->Rpad = h->tile_cap * 128;
  h->deterministic = (cfg->flags & MOE_FLAG_DETERMINISTIC) != 0;
  h->static_scales = (cfg->flags & MOE_FLAG_STATIC_ACT_SCALES) != 0;

  auto fail = [&](moe_status s) {
    moe_destroy(h);
    return s;
  };
#define A(ptr, bytes)                                \
  do {                                               \
    moe_status s_ = dalloc(h, &(ptr), (bytes));      \
    if (s_ != MOE_OK) return fail(s_);               \
  } while (0)
  const size_t Rp = h->Rpad;
  // FP4 operands: codes and block scales interleaved per tile in one buffer
  A(h->w13_codes, operand_bytes((size_t)E * 2 * I, H / 2));
  h->w13_sf = h->w13_codes;
  A(h->w2_codes, operand_bytes((size_t)E * H, h->Ipad / 2));
  h->w2_sf = h->w2_codes;
  A(h->gs_w13, sizeof(float) * E);
  A(h->gs_w2, sizeof(float) * E);
  if (h->static_scales) {
    A(h->static_x_gs, sizeof(float));
    A(h->static_h_gs, sizeof(float) * E);
  }
  A(h->amax_bits, sizeof(uint32_t) * 2 * E);
  A(h->logits, sizeof(float) * (size_t)T * E);
  A(h->topk_ids, sizeof(int32_t) * (size_t)T * K);
  A(h->topk_w, sizeof(float) * (size_t)T * K);
  A(h->expert_offsets, sizeof(int32_t) * (E + 1));
  A(h->src_of_row, sizeof(int32_t) * (size_t)h->Rmax);
  A(h->row_of_src, sizeof(int32_t) * (size_t)h->Rmax);
  A(h->pad_row_of_src, sizeof(int32_t) * (size_t)h->Rmax);
  A(h->src_of_padrow, sizeof(int32_t) * Rp);
  A(h->tiles, sizeof(int4) * (size_t)h->tile_cap);
  A(h->num_tiles, sizeof(int32_t) * 4);
  A(h->front_sync, sizeof(uint32_t) * FRONT_SYNC_WORDS);
  A(h->expert_done, sizeof(uint32_t) * 256);
  if (Is > 0) {
    h->Is = Is;
    h->Ipad_s = (Is + 255) / 256 * 256;
    h->Tpad_s = (T + 127) / 128 * 128;
    const size_t Ts = h->Tpad_s;
    A(h->sw13_codes, operand_bytes((size_t)2 * Is, H / 2));
    A(h->sw2_codes, operand_bytes((size_t)H, h->Ipad_s / 2));
    A(h->gs_sw13, sizeof(float));
    A(h->gs_sw2, sizeof(float));
    A(h->s_amax_bits, sizeof(uint32_t) * 2);
    A(h->s_a_codes, operand_bytes(Ts, H / 2));
    A(h->s_gs_rows, sizeof(float) * Ts);
    A(h->s_h_codes, operand_bytes(Ts, h->Ipad_s / 2));
    A(h->s_h_gs, sizeof(float) * Ts);
    A(h->s_ident, sizeof(int32_t) * Ts);
    A(h->s_tiles, sizeof(int4) * (Ts / 128));
    A(h->s_num_tiles, sizeof(int32_t));
    A(h->s_ybuf, sizeof(uint16_t) * (size_t)T * H);
    A(h->s_hbuf, sizeof(float) * 128 * (size_t)h->Ipad_s);
    A(h->s_row_amax, sizeof(float) * 128);
    std::vector<int32_t> ident(Ts);
    for (size_t i = 0; i < Ts; ++i) ident[i] = (int32_t)i;
    cudaError_t e = cudaMemcpy(h->s_ident, ident.data(), sizeof(int32_t) * Ts, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h->side, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->ev_fork, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->ev_join, cudaEventDisableTiming);
    if (e != cudaSuccess) return fail(cuda_fail(h, e, "shared-expert set-up"));
  }
  // small batches: FP32 SwiGLU rows and row maxima of the expert blocks
  A(h->hbuf, sizeof(float) * (size_t)E * 128 * h->Ipad);
  A(h->row_amax, sizeof(float) * (size_t)E * 128);
  A(h->a_codes, operand_bytes(Rp, H / 2));
  h->a_sf = h->a_codes;
  A(h->gs_rows, sizeof(float) * Rp);
  A(h->h_codes, operand_bytes(Rp, h->Ipad / 2));
  h->h_sf = h->h_codes;
  A(h->h_gs, sizeof(float) * Rp);
  if (h->deterministic || T > SMALL_BATCH_TOKENS) A(h->ybuf, sizeof(uint16_t) * (size_t)h->Rmax * H);
  if (!h->deterministic) A(h->out_acc, sizeof(float) * (size_t)std::min(T, SMALL_BATCH_TOKENS) * H);
  A(h->stage_x, sizeof(uint16_t) * (size_t)T * H);
  A(h->stage_gate, sizeof(uint16_t) * (size_t)H * E);
  A(h->stage_bias, sizeof(float) * E);
  A(h->stage_out, sizeof(uint16_t) * (size_t)T * H);
#undef A
  {
    cudaError_t e = cudaHostAlloc(reinterpret_cast<void**>(&h->status_host), sizeof(int), cudaHostAllocMapped);
    if (e != cudaSuccess) return fail(cuda_fail(h, e, "cudaHostAlloc"));
    *h->status_host = 0;
    e = cudaHostGetDevicePointer(reinterpret_cast<void**>(&h->status_dev), h->status_host, 0);
    if (e != cudaSuccess) return fail(cuda_fail(h, e, "cudaHostGetDevicePointer"));
  }
  {
    cudaError_t e = gemm_setup_attributes(I / 128);
    if (e != cudaSuccess) return fail(cuda_fail(h, e, "cudaFuncSetAttribute"));
    e = router_setup(H, E);
    if (e == cudaSuccess) e = front_setup(H, E);
    if (e != cudaSuccess) return fail(cuda_fail(h, e, "cudaFuncSetAttribute(router)"));
    h->num_sms = prop.multiProcessorCount;
    h->w13_clusters[0] = gemm_w13_max_clusters(I / 128, 64);
    h->w13_clusters[1] = gemm_w13_max_clusters(I / 128, 128);
    if (h->Is > 0) {
      e = gemm_setup_attributes(h->Is / 128);
      if (e != cudaSuccess) return fail(cuda_fail(h, e, "cudaFuncSetAttribute(shared)"));
      h->s_clusters[0] = gemm_w13_max_clusters(h->Is / 128, 64);
      h->s_clusters[1] = gemm_w13_max_clusters(h->Is / 128, 128);
      if (h->s_clusters[0] <= 0 || h->s_clusters[1] <= 0) {
        set_err(h, "no thread-block cluster of %d CTAs fits on the device", h->Is / 128);
        return fail(MOE_ERR_UNSUPPORTED);
      }
    }
    if (h->w13_clusters[0] <= 0 || h->w13_clusters[1] <= 0) {
      set_err(h, "no thread-block cluster of %d CTAs fits on the device", I / 128);
      return fail(MOE_ERR_UNSUPPORTED);
    }
  }
  *out = h;
  return MOE_OK;
}

moe_status moe_set_static_scales(moe_handle* h, const float* x_gs, const float* h_gs, void* stream) {
  if (!h) return MOE_ERR_INVALID_ARG;
  if (!h->static_scales) {
    set_err(h, "moe_set_static_scales: the handle was not created with MOE_FLAG_STATIC_ACT_SCALES");
    return MOE_ERR_INVALID_ARG;
  }
  if (!x_gs || !h_gs) {
    set_err(h, "moe_set_static_scales: NULL scale pointer");
    return MOE_ERR_INVALID_ARG;
  }
  DeviceGuard dg(h->cfg.device);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  CK(h, cudaMemcpyAsync(h->static_x_gs, x_gs, sizeof(float), cudaMemcpyDeviceToDevice, s));
  CK(h, cudaMemcpyAsync(h->static_h_gs, h_gs, sizeof(float) * h->E, cudaMemcpyDeviceToDevice, s));
  h->static_set = true;
  return MOE_OK;
}

moe_status moe_destroy(moe_handle* h) {
  if (!h) return MOE_OK;
  DeviceGuard dg(h->cfg.device);
  cudaDeviceSynchronize();
  for (void* p : h->allocs) cudaFree(p);
  if (h->status_host) cudaFreeHost(h->status_host);
  for (cudaEvent_t ev : h->events)
    if (ev) cudaEventDestroy(ev);
  if (h->ev_fork) cudaEventDestroy(h->ev_fork);
  if (h->ev_join) cudaEventDestroy(h->ev_join);
  if (h->side) cudaStreamDestroy(h->side);
  cudaGetLastError();
  delete h;
  return MOE_OK;
}

moe_status moe_load_shared_weights(moe_handle* h, const void* w13s, const moe_weight_desc* w13s_desc,
                                   const void* w2s, const moe_weight_desc* w2s_desc, void* stream) {
  if (!h) return MOE_ERR_INVALID_ARG;
  if (h->Is <= 0) {
    set_err(h, "the handle was created without a shared expert (shared_inter = 0)");
    return MOE_ERR_INVALID_ARG;
  }
  DeviceGuard dg(h->cfg.device);
  TRY(check_weight_desc(h, w13s_desc, w13s, 1, 2 * h->Is, h->H, "w13s"));
  TRY(check_weight_desc(h, w2s_desc, w2s, 1, h->H, h->Is, "w2s"));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // one expert: the routed experts' conversion (gate / up rows interleaved
  // in chunks of 64 for the w13 epilogue), into the same buffers every time
  CK(h, cudaMemsetAsync(h->s_amax_bits, 0, sizeof(uint32_t) * 2, s));
  CK(h, launch_weight_amax(w13s, 1, 2 * h->Is, h->H, h->s_amax_bits, s));
  CK(h, launch_weight_amax(w2s, 1, h->H, h->Is, h->s_amax_bits + 1, s));
  CK(h, launch_weight_quant(w13s, 1, 2 * h->Is, h->H, h->H, 1, h->s_amax_bits, h->sw13_codes, h->sw13_codes,
                            h->gs_sw13, s));
  CK(h, launch_weight_quant(w2s, 1, h->H, h->Is, h->Ipad_s, 0, h->s_amax_bits + 1, h->sw2_codes, h->sw2_codes,
                            h->gs_sw2, s));
  h->shared_loaded = true;
  h->err.clear();
  return MOE_OK;
}

moe_status moe_load_weights(moe_handle* h, const void* w13, const moe_weight_desc* w13_desc, const void* w2,
                            const moe_weight_desc* w2_desc, void* stream) {
  if (!h) return MOE_ERR_INVALID_ARG;
  DeviceGuard dg(h->cfg.device);
  TRY(check_weight_desc(h, w13_desc, w13, h->E, 2 * h->I, h->H, "w13"));
  TRY(check_weight_desc(h, w2_desc, w2, h->E, h->H, h->I, "w2"));
  TRY(quantize_weights(h, w13, w2, reinterpret_cast<cudaStream_t>(stream)));
  h->w13_desc = *w13_desc;
  h->w2_desc = *w2_desc;
  h->loaded = true;
  h->err.clear();
  return MOE_OK;
}

moe_status moe_refresh_scales_inplace(moe_handle* h, const void* w13, const moe_weight_desc* w13_desc,
                                      const void* w2, const moe_weight_desc* w2_desc, void* stream) {
  if (!h) return MOE_ERR_INVALID_ARG;
  DeviceGuard dg(h->cfg.device);
  if (!h->loaded) {
    set_err(h, "refresh before the first moe_load_weights");
    return MOE_ERR_NOT_LOADED;
  }
  if (!w13_desc || !w2_desc || !same_desc(*w13_desc, h->w13_desc) || !same_desc(*w2_desc, h->w2_desc)) {
    set_err(h, "weight metadata changed during reload; CUDA graph recapture is required");
    return MOE_ERR_METADATA_CHANGED;
  }
  TRY(check_weight_desc(h, w13_desc, w13, h->E, 2 * h->I, h->H, "w13"));
  TRY(check_weight_desc(h, w2_desc, w2, h->E, h->H, h->I, "w2"));
  TRY(quantize_weights(h, w13, w2, reinterpret_cast<cudaStream_t>(stream)));
  h->err.clear();
  return MOE_OK;
}

moe_status moe_forward_ex(moe_handle* h, const void* x, const void* gate_w, const float* gate_bias, void* out,
                          int num_tokens, void* stream) {
  if (!h) return MOE_ERR_INVALID_ARG;
  if (h->status_host && *(volatile int*)h->status_host) {
    set_err(h, "a kernel of this handle gave up a bounded wait (device status 0x%x)", *(volatile int*)h->status_host);
    return MOE_ERR_DEVICE_TIMEOUT;
  }
  if (!h->loaded) {
    set_err(h, "moe_forward before moe_load_weights");
    return MOE_ERR_NOT_LOADED;
  }
  if (h->static_scales && !h->static_set) {
    set_err(h, "static activation scales: moe_set_static_scales has not been called");
    return MOE_ERR_NOT_LOADED;
  }
  if (h->Is > 0 && !h->shared_loaded) {
    set_err(h, "shared expert: moe_load_shared_weights has not been called");
    return MOE_ERR_NOT_LOADED;
  }
  if (num_tokens < 0) {
    set_err(h, "num_tokens (%d) is negative", num_tokens);
    return MOE_ERR_INVALID_ARG;
  }
  if (num_tokens > h->Tmax) {
    set_err(h, "num_tokens (%d) exceeds max_num_tokens (%d)", num_tokens, h->Tmax);
    return MOE_ERR_TOO_MANY_TOKENS;
  }
  if (num_tokens == 0) {
    h->last_T = 0;
    return MOE_OK;
  }
  if (!x || !gate_w || !out) {
    set_err(h, "NULL x, gate_w or out");
    return MOE_ERR_INVALID_ARG;
  }
  if (!aligned16(x) || !aligned16(gate_w) || !aligned16(out) || (gate_bias && !aligned16(gate_bias))) {
    set_err(h, "x, gate_w, out and gate_bias must be 16-byte aligned");
    return MOE_ERR_INVALID_ARG;
  }
  const size_t act_bytes = (size_t)num_tokens * h->H * 2;
  if (ranges_overlap(x, act_bytes, out, act_bytes)) {
    set_err(h, "out must not overlap x (the routed output never aliases its input)");
    return MOE_ERR_ALIAS;
  }
  DeviceGuard dg(h->cfg.device);
  return forward_impl(h, x, gate_w, gate_bias, out, num_tokens, reinterpret_cast<cudaStream_t>(stream));
}

moe_status moe_forward(moe_handle* h, const void* x, const void* gate_w, void* out, int num_tokens, void* stream) {
  return moe_forward_ex(h, x, gate_w, nullptr, out, num_tokens, stream);
}

moe_status moe_forward_host(moe_handle* h, const void* x_host, const void* gate_w_host, const float* gate_bias_host,
                            void* out_host, int num_tokens, void* stream) {
  if (!h) return MOE_ERR_INVALID_ARG;
  if (num_tokens < 0 || num_tokens > h->Tmax) {
    set_err(h, "num_tokens (%d) outside [0, %d]", num_tokens, h->Tmax);
    return num_tokens < 0 ? MOE_ERR_INVALID_ARG : MOE_ERR_TOO_MANY_TOKENS;
  }
  if (num_tokens > 0 && (!x_host || !gate_w_host || !out_host)) {
    set_err(h, "NULL host pointer");
    return MOE_ERR_INVALID_ARG;
  }
  DeviceGuard dg(h->cfg.device);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (num_tokens == 0) return moe_forward_ex(h, nullptr, nullptr, nullptr, nullptr, 0, stream);
  const size_t xb = (size_t)num_tokens * h->H * 2;
  CK(h, cudaMemcpyAsync(h->stage_x, x_host, xb, cudaMemcpyHostToDevice, s));
  CK(h, cudaMemcpyAsync(h->stage_gate, gate_w_host, (size_t)h->H * h->E * 2, cudaMemcpyHostToDevice, s));
  if (gate_bias_host) CK(h, cudaMemcpyAsync(h->stage_bias, gate_bias_host, sizeof(float) * h->E, cudaMemcpyHostToDevice, s));
  TRY(moe_forward_ex(h, h->stage_x, h->stage_gate, gate_bias_host ? h->stage_bias : nullptr, h->stage_out,
                     num_tokens, stream));
  CK(h, cudaMemcpyAsync(out_host, h->stage_out, xb, cudaMemcpyDeviceToHost, s));
  CK(h, cudaStreamSynchronize(s));
  return moe_get_status(h);
}

moe_status moe_set_stage_timing(moe_handle* h, int enable) {
  if (!h) return MOE_ERR_INVALID_ARG;
  DeviceGuard dg(h->cfg.device);
  if (enable && !h->events[0]) {
    for (cudaEvent_t& ev : h->events) CK(h, cudaEventCreate(&ev));
  }
  h->timing = enable != 0;
  return MOE_OK;
}

moe_status moe_get_stage_times(const moe_handle* h, float* ms, int* n) {
  if (!h || !n || (*n > 0 && !ms)) return MOE_ERR_INVALID_ARG;
  if (!h->events[0]) return MOE_ERR_NOT_LOADED;
  DeviceGuard dg(h->cfg.device);
  const int m = std::min(*n, MOE_NUM_STAGES);
  for (int i = 0; i < m; ++i) {
    if (cudaEventElapsedTime(&ms[i], h->events[i], h->events[i + 1]) != cudaSuccess) {
      cudaGetLastError();
      return MOE_ERR_CUDA;
    }
  }
  *n = m;
  return MOE_OK;
}

const char* moe_stage_name(int i) {
  static const char* names[MOE_NUM_STAGES] = {"router", "topk", "permute", "quantize", "gemm_w13", "gemm_w2",
                                              "finalize"};
  return (i >= 0 && i < MOE_NUM_STAGES) ? names[i] : nullptr;
}

size_t moe_get_workspace_bytes(const moe_handle* h) { return h ? h->bytes : 0; }

const char* moe_get_last_error(const moe_handle* h) { return h ? h->err.c_str() : "NULL handle"; }

moe_status moe_get_status(const moe_handle* h) {
  if (!h) return MOE_ERR_INVALID_ARG;
  return (h->status_host && *(volatile int*)h->status_host) ? MOE_ERR_DEVICE_TIMEOUT : MOE_OK;
}

moe_status moe_debug_routing(moe_handle* h, int32_t* topk_ids, float* topk_w, int32_t* src_of_row,
                             int32_t* expert_offsets, void* stream) {
  if (!h) return MOE_ERR_INVALID_ARG;
  if (h->last_T < 0) {
    set_err(h, "no forward has run on this handle");
    return MOE_ERR_NOT_LOADED;
  }
  DeviceGuard dg(h->cfg.device);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t tk = (size_t)h->last_T * h->K;
  if (topk_ids && tk) CK(h, cudaMemcpyAsync(topk_ids, h->topk_ids, tk * 4, cudaMemcpyDeviceToDevice, s));
  if (topk_w && tk) CK(h, cudaMemcpyAsync(topk_w, h->topk_w, tk * 4, cudaMemcpyDeviceToDevice, s));
  if (src_of_row && tk) CK(h, cudaMemcpyAsync(src_of_row, h->src_of_row, tk * 4, cudaMemcpyDeviceToDevice, s));
  if (expert_offsets) {
    if (h->last_T == 0) CK(h, cudaMemsetAsync(expert_offsets, 0, sizeof(int32_t) * (h->E + 1), s));
    else CK(h, cudaMemcpyAsync(expert_offsets, h->expert_offsets, sizeof(int32_t) * (h->E + 1),
                               cudaMemcpyDeviceToDevice, s));
  }
  return MOE_OK;
}

moe_status moe_debug_logits(moe_handle* h, float* logits, void* stream) {
  if (!h || !logits) return MOE_ERR_INVALID_ARG;
  if (h->last_T < 0) return MOE_ERR_NOT_LOADED;
  DeviceGuard dg(h->cfg.device);
  if (h->last_T)
    CK(h, cudaMemcpyAsync(logits, h->logits, sizeof(float) * (size_t)h->last_T * h->E, cudaMemcpyDeviceToDevice,
                          reinterpret_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

moe_status moe_debug_act_quant(moe_handle* h, uint8_t* codes, uint8_t* sf, float* gs, void* stream) {
  if (!h) return MOE_ERR_INVALID_ARG;
  if (h->last_T < 0) return MOE_ERR_NOT_LOADED;
  DeviceGuard dg(h->cfg.device);
  // token t's quantization is the one written to its slot-0 expanded row,
  // pad_row_of_src[t*K].
  if (h->last_T == 0) return MOE_OK;
  // (small batches: row t of the shared activation tile)
  if (h->last_small)
    CK(h, launch_export_rows(h->a_codes, h->a_sf, h->gs_rows, h->last_T, h->H, h->H, nullptr, 0, 1, 0, 0, codes, sf,
                             gs, reinterpret_cast<cudaStream_t>(stream)));
  else
    CK(h, launch_export_rows(h->a_codes, h->a_sf, h->gs_rows, h->last_T, h->H, h->H, h->pad_row_of_src, h->K, 0,
                             0, 0, codes, sf, gs, reinterpret_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

moe_status moe_debug_weight_quant(moe_handle* h, int which, uint8_t* codes, uint8_t* sf, float* gs, void* stream) {
  if (!h || (which != 0 && which != 1)) return MOE_ERR_INVALID_ARG;
  if (!h->loaded) return MOE_ERR_NOT_LOADED;
  DeviceGuard dg(h->cfg.device);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (which == 0) {
    CK(h, launch_export_rows(h->w13_codes, h->w13_sf, nullptr, h->E * 2 * h->I, h->H, h->H, nullptr, 0, 2,
                             2 * h->I, 1, codes, sf, nullptr, s));
    if (gs) CK(h, cudaMemcpyAsync(gs, h->gs_w13, sizeof(float) * h->E, cudaMemcpyDeviceToDevice, s));
  } else {
    CK(h, launch_export_rows(h->w2_codes, h->w2_sf, nullptr, h->E * h->H, h->I, h->Ipad, nullptr, 0, 1, 0, 1, codes,
                             sf, nullptr, s));
    if (gs) CK(h, cudaMemcpyAsync(gs, h->gs_w2, sizeof(float) * h->E, cudaMemcpyDeviceToDevice, s));
  }
  return MOE_OK;
}

moe_status moe_debug_intermediate(moe_handle* h, uint8_t* h_codes, uint8_t* h_sf, float* h_gs, void* stream) {
  if (!h) return MOE_ERR_INVALID_ARG;
  if (h->last_T < 0) return MOE_ERR_NOT_LOADED;
  DeviceGuard dg(h->cfg.device);
  if (h->last_T == 0) return MOE_OK;
  CK(h, launch_export_rows(h->h_codes, h->h_sf, h->h_gs, h->last_T * h->K, h->I, h->Ipad, h->pad_row_of_src, 1, 0,
                           0, 0, h_codes, h_sf, h_gs, reinterpret_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

moe_status moe_debug_shared(moe_handle* h, uint16_t* rows, uint8_t* h_codes, uint8_t* h_sf, float* h_gs,
                            void* stream) {
  if (!h) return MOE_ERR_INVALID_ARG;
  if (h->Is <= 0) {
    set_err(h, "the handle was created without a shared expert (shared_inter = 0)");
    return MOE_ERR_INVALID_ARG;
  }
  if (h->last_T < 0) return MOE_ERR_NOT_LOADED;
  if (!h_codes != !h_sf || !h_codes != !h_gs) return MOE_ERR_INVALID_ARG;
  DeviceGuard dg(h->cfg.device);
  const int T = h->last_T;
  if (T == 0) return MOE_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (rows) CK(h, cudaMemcpyAsync(rows, h->s_ybuf, sizeof(uint16_t) * (size_t)T * h->H, cudaMemcpyDeviceToDevice, s));
  if (h_codes && h_sf && h_gs)
    CK(h, launch_export_rows(h->s_h_codes, h->s_h_codes, h->s_h_gs, T, h->Is, h->Ipad_s, h->s_ident, 1, 0, 0, 0,
                             h_codes, h_sf, h_gs, s));
  return MOE_OK;
}

moe_status moe_debug_shared_act_quant(moe_handle* h, uint8_t* codes, uint8_t* sf, float* gs, void* stream) {
  if (!h) return MOE_ERR_INVALID_ARG;
  if (h->Is <= 0) {
    set_err(h, "the handle was created without a shared expert (shared_inter = 0)");
    return MOE_ERR_INVALID_ARG;
  }
  if (h->last_T < 0) return MOE_ERR_NOT_LOADED;
  if (!codes || !sf || !gs) return MOE_ERR_INVALID_ARG;
  DeviceGuard dg(h->cfg.device);
  if (h->last_T == 0) return MOE_OK;
  // token t is row t of the shared expert's activation operand
  CK(h, launch_export_rows(h->s_a_codes, h->s_a_codes, h->s_gs_rows, h->last_T, h->H, h->H, h->s_ident, 1, 0, 0, 0,
                           codes, sf, gs, reinterpret_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

moe_status moe_debug_buffer_ptrs(const moe_handle* h, const void** ptrs, int* n) {
  if (!h || !n) return MOE_ERR_INVALID_ARG;
  const int have = (int)h->allocs.size();
  if (ptrs) {
    for (int i = 0; i < std::min(*n, have); ++i) ptrs[i] = h->allocs[i];
  }
  *n = have;
  return MOE_OK;
}

moe_status moe_debug_convert(const float* in, uint8_t* e2m1, uint8_t* e4m3, int64_t n, void* stream) {
  if (n < 0 || (n > 0 && !in)) return MOE_ERR_INVALID_ARG;
  cudaError_t e = launch_convert(in, e2m1, e4m3, n, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_debug_block_scaled_gemm(const uint8_t* a_codes, const uint8_t* a_sf, const uint8_t* b_codes,
                                       const uint8_t* b_sf, float* d, int M, int N, int K, void* stream) {
  if (!a_codes || !a_sf || !b_codes || !b_sf || !d) return MOE_ERR_INVALID_ARG;
  if (M <= 0 || N <= 0 || K <= 0 || M % 128 || N % 128 || K % 256) return MOE_ERR_UNSUPPORTED;
  if (!aligned16(a_codes) || !aligned16(b_codes) || !aligned16(d)) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // canonical codes / scales -> the interleaved operand layout
  uint8_t *opa = nullptr, *opb = nullptr;
  moe_status st = MOE_OK;
  if (cudaMalloc(&opa, operand_bytes(M, K / 2)) != cudaSuccess || cudaMalloc(&opb, operand_bytes(N, K / 2)) != cudaSuccess)
    st = MOE_ERR_CUDA;
  if (st == MOE_OK && (launch_sf_to_atoms(a_sf, M, K / 16, opa, s) != cudaSuccess ||
                       launch_sf_to_atoms(b_sf, N, K / 16, opb, s) != cudaSuccess ||
                       launch_codes_to_tiled(a_codes, M, K / 2, opa, s) != cudaSuccess ||
                       launch_codes_to_tiled(b_codes, N, K / 2, opb, s) != cudaSuccess))
    st = MOE_ERR_CUDA;
  if (st == MOE_OK && gemm_setup_attributes(1) != cudaSuccess) st = MOE_ERR_CUDA;
  int dev = 0, sms = 0;
  if (st == MOE_OK && (cudaGetDevice(&dev) != cudaSuccess ||
                       cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess))
    st = MOE_ERR_CUDA;
  if (st == MOE_OK) {
    GemmArgs g{};
    g.a_codes = opa;
    g.b_codes = opb;
    g.k_stages = K / STAGE_K;
    g.d = d;
    g.ldd = N;
    g.n_tiles = N / TILE_N;
    g.m_tiles = M / TILE_M;
    if (launch_gemm_plain(g, std::min(sms, g.n_tiles * g.m_tiles), s) != cudaSuccess) st = MOE_ERR_CUDA;
  }
  if (cudaStreamSynchronize(s) != cudaSuccess) st = MOE_ERR_CUDA;
  cudaFree(opa);
  cudaFree(opb);
  return st;
}

}  // extern "C"
