// The C ABI (include/moe.h): argument validation, workspace layout, and the order of the
// kernel groups of each call. No allocation, no synchronisation except in moe_get_status.
#include <math.h>
#include <string.h>

#include <atomic>
#include <climits>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {

static std::atomic<uint64_t> g_launches{0};
void note_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

int device_sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  if (dev >= 0 && dev < 64) cache[dev] = n;
  return n;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

bool encode_tmap_2d_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                         uint32_t box_inner, uint32_t box_outer) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || (reinterpret_cast<uintptr_t>(base) & 15) != 0 || (inner * 2) % 16 != 0) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tmap_mn_blocks_bf16(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows,
                                uint32_t box_rows, uint32_t blocks) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || (reinterpret_cast<uintptr_t>(base) & 15) != 0 || cols % 64 != 0) return false;
  const cuuint64_t dims[3] = {64, rows, cols / 64};
  const cuuint64_t strides[2] = {cols * 2, 128};
  const cuuint32_t box[3] = {64, box_rows, blocks};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tmap_3d_f32_sw128(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                              uint32_t box0, uint32_t box1) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || (reinterpret_cast<uintptr_t>(base) & 15) != 0 || (d0 * 4) % 16 != 0) return false;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {d0 * 4, d0 * d1 * 4};
  const cuuint32_t box[3] = {box0, box1, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

moe_status_t make_problem(const moe_config_t* c, Problem* p) {
  if (!c || !p) return MOE_ERR_INVALID_ARG;
  if (c->T < 0 || c->h < 1 || c->n_heads < 1 || c->h % c->n_heads != 0) return MOE_ERR_INVALID_ARG;
  if (c->E < 1 || c->K < 1 || c->K > c->E || c->d_ff < 1) return MOE_ERR_INVALID_ARG;
  if (c->n_groups < 1 || c->E % c->n_groups != 0 || c->topk_groups < 1 || c->topk_groups > c->n_groups)
    return MOE_ERR_INVALID_ARG;
  if ((int64_t)c->K > (int64_t)c->topk_groups * (c->E / c->n_groups)) return MOE_ERR_INVALID_ARG;
  if (c->score != MOE_SCORE_SOFTMAX && c->score != MOE_SCORE_SIGMOID) return MOE_ERR_INVALID_ARG;
  if (c->dtype != MOE_F32 && c->dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (!isfinite(c->aux_alpha) || isnan(c->capacity_factor)) return MOE_ERR_INVALID_ARG;
  if (c->E > kMaxExperts || c->K > kMaxTopK || c->n_groups > kMaxGroups) return MOE_ERR_UNSUPPORTED;
  const int64_t Tu = c->T * (int64_t)c->n_heads;
  const int hu = c->h / c->n_heads;
  if (Tu > (int64_t)INT_MAX / 8 || Tu * c->K > (int64_t)INT_MAX) return MOE_ERR_UNSUPPORTED;
  const bool bf16 = c->dtype == MOE_BF16;
  if (bf16 && (hu % 32 != 0 || c->d_ff % 32 != 0)) return MOE_ERR_UNSUPPORTED;
  if ((int64_t)c->E * (bf16 ? c->d_ff : 1) > (int64_t)INT_MAX || (int64_t)c->E * hu > (int64_t)INT_MAX)
    return MOE_ERR_UNSUPPORTED;
  p->cfg = *c;
  p->Tu = Tu;
  p->hu = hu;
  p->E = c->E;
  p->K = c->K;
  p->d_ff = c->d_ff;
  p->n_groups = c->n_groups;
  p->topk_groups = c->topk_groups;
  p->bf16 = bf16;
  p->sigmoid = c->score == MOE_SCORE_SIGMOID;
  const double cf = c->capacity_factor;
  if (!(cf > 0.0) || isinf(cf)) p->C = INT64_MAX;
  else p->C = (int64_t)ceil(cf * (double)c->K * (double)Tu / (double)c->E);
  p->rows = Tu * c->K;
  p->ntiles = (Tu + kTileUnits - 1) / kTileUnits;
  p->nchunks = (Tu + kChunk - 1) / kChunk;
  p->elt = bf16 ? 2 : 4;
  return MOE_OK;
}

WsLayout ws_layout(const Problem& p) {
  WsLayout L;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += (bytes + kWsAlign - 1) / kWsAlign * kWsAlign;
    return at;
  };
  const size_t E = (size_t)p.E, TK = (size_t)p.Tu * p.K, rows = (size_t)p.rows;
  L.status = take(kWsAlign);
  L.counts = take(E * 4);
  L.offsets = take((E + 1) * 4);
  L.chunk_hist = take((size_t)p.ntiles * E * 4);
  L.chunk_base = take((size_t)p.ntiles * E * 4);
  L.psum = take((size_t)p.ntiles * E * 4);
  L.aux_terms = take(E * 4);
  L.cap = take(E * 8);
  L.w_pad = take(p.bf16 ? (size_t)p.hu * ((E + 7) / 8 * 8) * 2 : 0);
  L.logits = take(p.bf16 ? 0 : (size_t)p.Tu * E * 4);
  L.rank = take(TK * 4);
  L.idx = take(TK * 4);
  L.gate = take(TK * 4);
  L.slot_of = take(TK * 4);
  L.row_token = take(rows * 4);
  L.x_packed = take(rows * (size_t)p.hu * p.elt);
  L.hidden = take(rows * (size_t)p.d_ff * p.elt);
  L.y_packed = take(rows * (size_t)p.hu * p.elt);
  L.arrivals = take(p.bf16 ? (size_t)p.Tu * (size_t)(p.hu / 32) * 4 : 0);
  L.total = off;
  return L;
}

// Backward scratch: the packed-row gradients and the router-gradient partials.
struct BwdLayout {
  size_t dy_packed;  // bf16 [T'K][h']
  size_t dgu;        // bf16 [T'K][2·d_ff]   dG | dU
  size_t dx_packed;  // bf16 [T'K][h']
  size_t dgate;      // fp32 [T'][K]
  size_t dl;         // fp32 [T'][E]
  size_t wg_part;    // fp32 [chunks][h'][E]
  size_t dy_t;       // bf16 [h'][padded cols]  dY_packed transposed, experts padded to 64 rows
  size_t x_t;        // bf16 [h'][padded cols]  X_packed transposed, likewise
  size_t wgt;        // bf16 [E][h']            W_g transposed (for dx += dl·W_gᵀ)
  size_t total;
};

static BwdLayout bwd_layout(const Problem& p) {
  BwdLayout L;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += (bytes + kWsAlign - 1) / kWsAlign * kWsAlign;
    return at;
  };
  const size_t rows = (size_t)p.rows, TK = (size_t)p.Tu * p.K;
  L.dy_packed = take(rows * p.hu * 2);
  L.dgu = take(rows * 2 * (size_t)p.d_ff * 2);
  L.dx_packed = take(rows * p.hu * 2);
  L.dgate = take(TK * 4);
  L.dl = take((size_t)p.Tu * p.E * 4);
  L.wg_part = take((size_t)backward_wg_chunks(p) * p.hu * p.E * 4);
  L.dy_t = take((size_t)p.hu * (size_t)backward_padded_cols(p) * 2);
  L.x_t = take((size_t)p.hu * (size_t)backward_padded_cols(p) * 2);
  L.wgt = take((size_t)p.E * p.hu * 2);
  L.total = off;
  return L;
}

static bool backward_supported(const Problem& p) { return p.bf16 && p.hu % 64 == 0 && p.d_ff % 64 == 0; }

}  // namespace moe

using namespace moe;

static bool aligned16(const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15) == 0; }
static bool ws_ok(const void* ws) { return ws && (reinterpret_cast<uintptr_t>(ws) & 255) == 0; }
static moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

extern "C" {

int32_t moe_abi_version(void) { return MOE_ABI_VERSION; }

moe_status_t moe_set_expert_gemm(int32_t pair_tiles, int32_t transposed_tails, int32_t fold_combine) {
  for (const int32_t v : {pair_tiles, transposed_tails, fold_combine})
    if (v < -1 || v > 1) return MOE_ERR_INVALID_ARG;
  set_expert_gemm(pair_tiles, transposed_tails, fold_combine);
  return MOE_OK;
}

uint64_t moe_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
    case MOE_ERR_WORKSPACE: return "workspace missing or misaligned";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE_STATUS: return "kernel found invalid data";
    case MOE_ERR_TIMEOUT: return "kernel wait timed out";
  }
  return "unknown status";
}

size_t moe_workspace_size(const moe_config_t* cfg) {
  Problem p;
  if (make_problem(cfg, &p) != MOE_OK) return 0;
  return ws_layout(p).total;
}

int64_t moe_capacity(const moe_config_t* cfg) {
  Problem p;
  if (make_problem(cfg, &p) != MOE_OK) return -2;
  return p.C == INT64_MAX ? -1 : p.C;
}

moe_status_t moe_workspace_init(const moe_config_t* cfg, void* ws, moe_stream_t stream) {
  Problem p;
  const moe_status_t st = make_problem(cfg, &p);
  if (st != MOE_OK) return st;
  if (!ws_ok(ws)) return MOE_ERR_WORKSPACE;
  return cuda_status(cudaMemsetAsync(ws, 0, kWsAlign, (cudaStream_t)stream));
}

}  // extern "C"

namespace moe {

// The routing kernel(s) of a call: bf16 → the fused tensor-core kernel; fp32 → the CUDA-core
// router into the workspace, then routing from those logits; given logits → routing from them.
// Leaves each tile's counts and Σp in the workspace and each pick's place in its tile in rank_out.
static cudaError_t route_stage(const Problem& p, const void* x, const void* w_router, const float* logits_in,
                               const float* logit_bias, const float* select_bias, int32_t* idx, float* gate,
                               float* logits_out, int32_t* rank_out, void* ws, cudaStream_t s) {
  if (p.Tu == 0) return cudaSuccess;
  const WsLayout L = ws_layout(p);
  SelectCtx sel;
  sel.select_bias = p.sigmoid ? select_bias : nullptr;
  sel.idx = idx;
  sel.gate = gate;
  sel.E = p.E;
  sel.K = p.K;
  sel.n_groups = p.n_groups;
  sel.topk_groups = p.topk_groups;
  int32_t* hist = ws_ptr<int32_t>(ws, L.chunk_hist);
  float* psum = ws_ptr<float>(ws, L.psum);
  if (logits_in)
    return launch_select_logits(p, logits_in, logit_bias, sel, nullptr, rank_out, hist, psum, s, false);
  if (p.bf16)
    return launch_route_tc(p, x, w_router, logit_bias, sel, logits_out, rank_out, hist, psum,
                           ws_ptr<void>(ws, L.w_pad), ws_ptr<uint32_t>(ws, L.status), s);
  float* lg = ws_ptr<float>(ws, L.logits);
  cudaError_t e = launch_router_simt_logits(p, x, w_router, lg, s);
  if (e != cudaSuccess) return e;
  return launch_select_logits(p, lg, logit_bias, sel, logits_out, rank_out, hist, psum, s, true);
}

// The per-expert scan over the routing tiles (counts, offsets, tile bases) and the aux loss.
static cudaError_t scan_stage(const Problem& p, void* ws, int32_t* counts_out, int32_t* offsets_out, float* aux_out,
                              cudaStream_t s, bool pdl = true) {
  const WsLayout L = ws_layout(p);
  return launch_scan(p, p.ntiles, ws_ptr<int32_t>(ws, L.chunk_hist), aux_out ? ws_ptr<float>(ws, L.psum) : nullptr,
                     ws_ptr<int32_t>(ws, L.chunk_base), ws_ptr<int32_t>(ws, L.counts), ws_ptr<int32_t>(ws, L.offsets),
                     counts_out, offsets_out, ws_ptr<float>(ws, L.aux_terms),
                     ws_ptr<unsigned int>(ws, L.status + 8), aux_out, s, pdl);
}

}  // namespace moe

extern "C" {

moe_status_t moe_route(const moe_config_t* cfg, const void* x, const void* w_router,
                       const float* logit_bias, const float* select_bias, int32_t* topk_idx,
                       float* topk_gate, float* logits_out, float* aux_out, void* ws,
                       moe_stream_t stream) {
  Problem p;
  const moe_status_t st = make_problem(cfg, &p);
  if (st != MOE_OK) return st;
  if (!ws_ok(ws)) return MOE_ERR_WORKSPACE;
  if (p.Tu > 0 && (!x || !w_router || !topk_idx || !topk_gate)) return MOE_ERR_INVALID_ARG;
  if (p.Tu > 0 && p.bf16 && !aligned16(x)) return MOE_ERR_INVALID_ARG;
  const cudaStream_t s = (cudaStream_t)stream;
  const WsLayout L = ws_layout(p);
  cudaError_t e = route_stage(p, x, w_router, nullptr, logit_bias, select_bias, topk_idx, topk_gate, logits_out,
                              ws_ptr<int32_t>(ws, L.rank), ws, s);
  if (e != cudaSuccess || !aux_out) return cuda_status(e);
  return cuda_status(scan_stage(p, ws, nullptr, nullptr, aux_out, s));
}

moe_status_t moe_route_logits(const moe_config_t* cfg, const float* logits, const float* logit_bias,
                              const float* select_bias, int32_t* topk_idx, float* topk_gate,
                              float* aux_out, void* ws, moe_stream_t stream) {
  Problem p;
  const moe_status_t st = make_problem(cfg, &p);
  if (st != MOE_OK) return st;
  if (!ws_ok(ws)) return MOE_ERR_WORKSPACE;
  if (p.Tu > 0 && (!logits || !topk_idx || !topk_gate)) return MOE_ERR_INVALID_ARG;
  const cudaStream_t s = (cudaStream_t)stream;
  const WsLayout L = ws_layout(p);
  cudaError_t e = route_stage(p, nullptr, nullptr, logits, logit_bias, select_bias, topk_idx, topk_gate, nullptr,
                              ws_ptr<int32_t>(ws, L.rank), ws, s);
  if (e != cudaSuccess || !aux_out) return cuda_status(e);
  return cuda_status(scan_stage(p, ws, nullptr, nullptr, aux_out, s));
}

moe_status_t moe_dispatch(const moe_config_t* cfg, const void* x, const int32_t* topk_idx,
                          int32_t* counts, int32_t* offsets, int32_t* slot_of, int32_t* row_token,
                          void* x_packed, void* ws, moe_stream_t stream) {
  Problem p;
  const moe_status_t st = make_problem(cfg, &p);
  if (st != MOE_OK) return st;
  if (!ws_ok(ws)) return MOE_ERR_WORKSPACE;
  if (!offsets) return MOE_ERR_INVALID_ARG;
  if (p.Tu > 0 && (!x || !topk_idx || !slot_of || !row_token || !x_packed)) return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(p);
  DispatchScratch sc;
  sc.chunk_hist = ws_ptr<int32_t>(ws, L.chunk_hist);
  sc.chunk_base = ws_ptr<int32_t>(ws, L.chunk_base);
  sc.counts = ws_ptr<int32_t>(ws, L.counts);
  sc.offsets = ws_ptr<int32_t>(ws, L.offsets);
  sc.ticket = ws_ptr<unsigned int>(ws, L.status + 8);
  sc.status = ws_ptr<uint32_t>(ws, L.status);
  return cuda_status(launch_dispatch_from_idx(p, x, topk_idx, counts, offsets, slot_of, row_token, x_packed, sc,
                                              (cudaStream_t)stream));
}

moe_status_t moe_dispatch_sharded(const moe_config_t* cfg, const void* x, const int32_t* topk_idx,
                                  const int32_t* queue_base, int64_t T_global, int32_t* counts, int32_t* offsets,
                                  int32_t* slot_of, int32_t* row_token, void* x_packed, void* ws, moe_stream_t stream) {
  Problem p;
  const moe_status_t st = make_problem(cfg, &p);
  if (st != MOE_OK) return st;
  if (!ws_ok(ws)) return MOE_ERR_WORKSPACE;
  if (!offsets || !queue_base || T_global < cfg->T) return MOE_ERR_INVALID_ARG;
  if (p.Tu > 0 && (!x || !topk_idx || !slot_of || !row_token || !x_packed)) return MOE_ERR_INVALID_ARG;
  // the capacity of the whole batch: C = ceil(CF·K·T'_global/E)
  moe_config_t g = *cfg;
  g.T = T_global;
  Problem pg;
  if (make_problem(&g, &pg) != MOE_OK) return MOE_ERR_UNSUPPORTED;
  p.C = pg.C;
  const WsLayout L = ws_layout(p);
  DispatchScratch sc;
  sc.chunk_hist = ws_ptr<int32_t>(ws, L.chunk_hist);
  sc.chunk_base = ws_ptr<int32_t>(ws, L.chunk_base);
  sc.counts = ws_ptr<int32_t>(ws, L.counts);
  sc.offsets = ws_ptr<int32_t>(ws, L.offsets);
  sc.ticket = ws_ptr<unsigned int>(ws, L.status + 8);
  sc.status = ws_ptr<uint32_t>(ws, L.status);
  sc.qbase = queue_base;
  sc.cap = ws_ptr<int64_t>(ws, L.cap);
  return cuda_status(launch_dispatch_from_idx(p, x, topk_idx, counts, offsets, slot_of, row_token, x_packed, sc,
                                              (cudaStream_t)stream));
}

moe_status_t moe_expert_ffn(const moe_config_t* cfg, const void* x_packed, const int32_t* offsets,
                            const void* w_gate, const void* w_up, const void* w_down,
                            void* y_packed, void* ws, moe_stream_t stream) {
  Problem p;
  const moe_status_t st = make_problem(cfg, &p);
  if (st != MOE_OK) return st;
  if (!ws_ok(ws)) return MOE_ERR_WORKSPACE;
  if (!offsets || !w_gate || !w_up || !w_down) return MOE_ERR_INVALID_ARG;
  if (p.rows > 0 && (!x_packed || !y_packed)) return MOE_ERR_INVALID_ARG;
  if (p.bf16 && !(aligned16(x_packed) && aligned16(w_gate) && aligned16(w_up) && aligned16(w_down) &&
                  aligned16(y_packed)))
    return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(p);
  return cuda_status(launch_expert_ffn(p, x_packed, offsets, w_gate, w_up, w_down,
                                       ws_ptr<void>(ws, L.hidden), y_packed,
                                       ws_ptr<uint32_t>(ws, L.status), (cudaStream_t)stream));
}

moe_status_t moe_combine(const moe_config_t* cfg, const void* y_packed, const int32_t* slot_of,
                         const float* topk_gate, void* y, void* ws, moe_stream_t stream) {
  Problem p;
  const moe_status_t st = make_problem(cfg, &p);
  if (st != MOE_OK) return st;
  if (!ws_ok(ws)) return MOE_ERR_WORKSPACE;
  if (p.Tu > 0 && (!y_packed || !slot_of || !topk_gate || !y)) return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(p);
  return cuda_status(launch_combine(p, y_packed, slot_of, topk_gate, y,
                                    ws_ptr<uint32_t>(ws, L.status), (cudaStream_t)stream));
}

// events: null, or kForwardEvents cudaEvent_t recorded on the stream before the routing, after it,
// after the scan, after the pack, after the expert GEMMs and after the combine (then the kernels of
// neighbouring stages are not overlapped by programmatic dependent launch).
static constexpr int kForwardEvents = 6;

// token_ids: null for the router, else the hash gate's token ids (K must be 1; no router weight).
static moe_status_t forward_impl(const moe_config_t* cfg, const void* x, const moe_weights_t* w, void* y,
                                 const moe_outputs_t* out, void* ws, moe_stream_t stream, void* gu,
                                 void* const* events = nullptr, const int32_t* token_ids = nullptr) {
  Problem p;
  const moe_status_t st = make_problem(cfg, &p);
  if (st != MOE_OK) return st;
  if (!ws_ok(ws)) return MOE_ERR_WORKSPACE;
  if (!w || (!token_ids && !w->w_router) || !w->w_gate || !w->w_up || !w->w_down) return MOE_ERR_INVALID_ARG;
  if (p.Tu > 0 && (!x || !y)) return MOE_ERR_INVALID_ARG;
  if (p.bf16 && !(aligned16(w->w_gate) && aligned16(w->w_up) && aligned16(w->w_down)))
    return MOE_ERR_INVALID_ARG;
  if (p.Tu > 0 && p.bf16 && !aligned16(x)) return MOE_ERR_INVALID_ARG;
  moe_outputs_t none;
  memset(&none, 0, sizeof(none));
  const moe_outputs_t& o = out ? *out : none;
  const WsLayout L = ws_layout(p);
  const cudaStream_t s = (cudaStream_t)stream;
  int32_t* idx = o.topk_idx ? o.topk_idx : ws_ptr<int32_t>(ws, L.idx);
  float* gate = o.topk_gate ? o.topk_gate : ws_ptr<float>(ws, L.gate);
  int32_t* slot_of = o.slot_of ? o.slot_of : ws_ptr<int32_t>(ws, L.slot_of);
  int32_t* row_token = ws_ptr<int32_t>(ws, L.row_token);
  int32_t* offsets_ws = ws_ptr<int32_t>(ws, L.offsets);
  void* x_packed = ws_ptr<void>(ws, L.x_packed);
  void* hidden = ws_ptr<void>(ws, L.hidden);
  void* y_packed = ws_ptr<void>(ws, L.y_packed);
  uint32_t* status = ws_ptr<uint32_t>(ws, L.status);

  auto mark = [&](int i) -> bool {
    return !events || cudaEventRecord(static_cast<cudaEvent_t>(events[i]), s) == cudaSuccess;
  };
  const bool pdl = events == nullptr;
  if (!mark(0)) return MOE_ERR_CUDA;
  // routing (each pick's place within its tile goes into slot_of, which the pack turns into slots)
  cudaError_t e = token_ids ? launch_hash_route(p, token_ids, idx, gate, slot_of, ws_ptr<int32_t>(ws, L.chunk_hist), s)
                            : route_stage(p, x, w->w_router, nullptr, w->logit_bias, w->select_bias, idx, gate,
                                          o.logits, slot_of, ws, s);
  if (e != cudaSuccess || !mark(1)) return MOE_ERR_CUDA;
  // counts, offsets (into the workspace; the caller's copies are optional) and the aux loss (the
  // hash gate has no routing probabilities, so no aux loss: 0)
  if (token_ids && o.aux && cudaMemsetAsync(o.aux, 0, sizeof(float), s) != cudaSuccess) return MOE_ERR_CUDA;
  e = scan_stage(p, ws, o.counts, o.offsets, token_ids ? nullptr : o.aux, s, pdl && !token_ids);
  if (e != cudaSuccess || !mark(2)) return MOE_ERR_CUDA;
  // the combine folded into the down GEMM (K == 1 unless set otherwise): the pack zeroes the
  // arrival counters and the y rows of units with no kept pick, and no combine launch follows
  const bool fold = p.bf16 && p.rows > 0 && aligned16(y) && fold_combine(p);
  uint32_t* arrivals = fold ? ws_ptr<uint32_t>(ws, L.arrivals) : nullptr;
  if (p.rows > 0) {
    e = launch_pack(p, x, idx, kTileShift, ws_ptr<int32_t>(ws, L.chunk_base), offsets_ws, slot_of, row_token, x_packed,
                    s, pdl, nullptr, fold ? y : nullptr, arrivals);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (!mark(3)) return MOE_ERR_CUDA;
  const FusedCombine fc = {y, row_token, slot_of, gate, arrivals, gu != nullptr};
  e = launch_expert_ffn(p, x_packed, offsets_ws, w->w_gate, w->w_up, w->w_down, hidden, y_packed,
                        status, s, gu, pdl, fold ? &fc : nullptr);
  if (e != cudaSuccess || !mark(4)) return MOE_ERR_CUDA;
  if (!fold) {
    e = launch_combine(p, y_packed, slot_of, gate, y, status, s, pdl);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (!mark(5)) return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status_t moe_forward(const moe_config_t* cfg, const void* x, const moe_weights_t* w, void* y,
                         const moe_outputs_t* out, void* ws, moe_stream_t stream) {
  return forward_impl(cfg, x, w, y, out, ws, stream, nullptr);
}

moe_status_t moe_forward_profiled(const moe_config_t* cfg, const void* x, const moe_weights_t* w, void* y,
                                  const moe_outputs_t* out, void* ws, void* const* events, moe_stream_t stream) {
  if (!events) return MOE_ERR_INVALID_ARG;
  for (int i = 0; i < kForwardEvents; ++i)
    if (!events[i]) return MOE_ERR_INVALID_ARG;
  return forward_impl(cfg, x, w, y, out, ws, stream, nullptr, events);
}

moe_status_t moe_route_hash(const moe_config_t* cfg, const int32_t* token_ids, int32_t* topk_idx, float* topk_gate,
                            void* ws, moe_stream_t stream) {
  Problem p;
  const moe_status_t st = make_problem(cfg, &p);
  if (st != MOE_OK) return st;
  if (p.K != 1) return MOE_ERR_UNSUPPORTED;
  if (!ws_ok(ws)) return MOE_ERR_WORKSPACE;
  if (p.Tu > 0 && (!token_ids || !topk_idx || !topk_gate)) return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(p);
  return cuda_status(launch_hash_route(p, token_ids, topk_idx, topk_gate, ws_ptr<int32_t>(ws, L.rank),
                                       ws_ptr<int32_t>(ws, L.chunk_hist), (cudaStream_t)stream));
}

moe_status_t moe_forward_hash(const moe_config_t* cfg, const void* x, const int32_t* token_ids, const moe_weights_t* w,
                              void* y, const moe_outputs_t* out, void* ws, moe_stream_t stream) {
  Problem p;
  const moe_status_t st = make_problem(cfg, &p);
  if (st != MOE_OK) return st;
  if (p.K != 1) return MOE_ERR_UNSUPPORTED;
  if (p.Tu > 0 && !token_ids) return MOE_ERR_INVALID_ARG;
  static const int32_t kNoUnits = 0;  // T' = 0: any non-null pointer selects the hash gate
  return forward_impl(cfg, x, w, y, out, ws, stream, nullptr, nullptr, token_ids ? token_ids : &kNoUnits);
}

size_t moe_saved_gu_size(const moe_config_t* cfg) {
  Problem p;
  if (make_problem(cfg, &p) != MOE_OK) return 0;
  return (size_t)p.rows * 2 * (size_t)p.d_ff * 2;
}

moe_status_t moe_forward_train(const moe_config_t* cfg, const void* x, const moe_weights_t* w, void* y,
                               const moe_outputs_t* out, void* gu, void* ws, moe_stream_t stream) {
  Problem p;
  const moe_status_t st = make_problem(cfg, &p);
  if (st != MOE_OK) return st;
  if (!backward_supported(p)) return MOE_ERR_UNSUPPORTED;
  // the per-unit outputs the backward reads (empty, possibly NULL, when there are no units)
  if (!out || (p.Tu > 0 && (!out->topk_idx || !out->topk_gate || !out->logits || !out->slot_of)))
    return MOE_ERR_INVALID_ARG;
  if (p.rows > 0 && (!gu || !aligned16(gu))) return MOE_ERR_INVALID_ARG;
  return forward_impl(cfg, x, w, y, out, ws, stream, gu);
}

size_t moe_backward_workspace_size(const moe_config_t* cfg) {
  Problem p;
  if (make_problem(cfg, &p) != MOE_OK || !backward_supported(p)) return 0;
  return bwd_layout(p).total;
}

moe_status_t moe_backward(const moe_config_t* cfg, const void* x, const moe_weights_t* w, const void* dy,
                          float d_aux, const moe_outputs_t* out, const void* gu, void* ws,
                          const moe_grads_t* grads, void* bws, moe_stream_t stream) {
  Problem p;
  const moe_status_t st = make_problem(cfg, &p);
  if (st != MOE_OK) return st;
  if (!backward_supported(p)) return MOE_ERR_UNSUPPORTED;
  if (!ws_ok(ws) || !ws_ok(bws)) return MOE_ERR_WORKSPACE;
  if (!w || !w->w_router || !w->w_gate || !w->w_up || !w->w_down) return MOE_ERR_INVALID_ARG;
  if (!out || (p.Tu > 0 && (!out->topk_idx || !out->topk_gate || !out->logits || !out->slot_of)))
    return MOE_ERR_INVALID_ARG;
  if (!grads || (p.Tu > 0 && !grads->dx) || !grads->dw_router || !grads->dw_gate || !grads->dw_up ||
      !grads->dw_down)
    return MOE_ERR_INVALID_ARG;
  if (!isfinite(d_aux)) return MOE_ERR_INVALID_ARG;
  if (p.Tu > 0 && (!x || !dy || !gu)) return MOE_ERR_INVALID_ARG;
  if (!(aligned16(w->w_gate) && aligned16(w->w_up) && aligned16(w->w_down) && aligned16(grads->dw_gate) &&
        aligned16(grads->dw_up) && aligned16(grads->dw_down) && aligned16(grads->dx) && aligned16(dy) &&
        aligned16(gu) && aligned16(x)))
    return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(p);
  const BwdLayout B = bwd_layout(p);
  const cudaStream_t s = (cudaStream_t)stream;
  uint32_t* status = ws_ptr<uint32_t>(ws, L.status);
  const int32_t* counts = ws_ptr<int32_t>(ws, L.counts);
  const int32_t* offsets = ws_ptr<int32_t>(ws, L.offsets);
  void* dy_packed = ws_ptr<void>(bws, B.dy_packed);
  void* dgu = ws_ptr<void>(bws, B.dgu);
  void* dx_packed = ws_ptr<void>(bws, B.dx_packed);
  float* dgate = grads->dgate ? grads->dgate : ws_ptr<float>(bws, B.dgate);
  float* dl = grads->dlogits ? grads->dlogits : ws_ptr<float>(bws, B.dl);

  cudaError_t e = launch_backward_misc_combine(p, dy, ws_ptr<void>(ws, L.y_packed), out->slot_of, out->topk_gate,
                                               dy_packed, dgate, status, s);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  e = launch_backward_logits(p, out->logits, out->topk_idx, out->topk_gate, dgate, counts, d_aux, dl, s);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  e = launch_expert_ffn_backward(p, offsets, ws_ptr<void>(ws, L.x_packed), ws_ptr<void>(ws, L.hidden), gu,
                                 dy_packed, w->w_gate, w->w_up, w->w_down, dgu, dx_packed, grads->dw_gate,
                                 grads->dw_up, grads->dw_down, ws_ptr<void>(bws, B.dy_t), ws_ptr<void>(bws, B.x_t),
                                 status, s);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  e = launch_backward_router(p, x, dl, backward_wg_chunks(p), ws_ptr<float>(bws, B.wg_part), grads->dw_router, s);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  e = launch_router_transpose(p, w->w_router, ws_ptr<void>(bws, B.wgt), s);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  e = launch_backward_dx(p, dx_packed, out->slot_of, dl, ws_ptr<void>(bws, B.wgt), grads->dx, s);
  return cuda_status(e);
}

moe_status_t moe_get_status(void* ws, moe_stream_t stream) {
  if (!ws_ok(ws)) return MOE_ERR_WORKSPACE;
  uint32_t word = 0;
  const cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemcpyAsync(&word, ws, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  if (word != 0) {
    if (cudaMemsetAsync(ws, 0, sizeof(word), s) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (word & kDevErrTimeout) return MOE_ERR_TIMEOUT;
  return word ? MOE_ERR_DEVICE_STATUS : MOE_OK;
}

}  // extern "C"
