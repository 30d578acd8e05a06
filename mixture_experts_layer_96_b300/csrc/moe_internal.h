// Host-side internals of the C ABI: validated problem description, workspace layout and the
// launchers of each kernel group. Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

constexpr int kMaxExperts = 256;
constexpr int kMaxTopK = 8;
constexpr int kMaxGroups = 32;
constexpr int kTileUnits = 128;      // units per routing tile (one router M tile); a dispatch chunk
constexpr int kTileShift = 7;
constexpr int kChunk = 256;          // units per chunk when the dispatch ranks given picks
constexpr int kChunkShift = 8;
constexpr size_t kWsAlign = 1024;

// A validated configuration with the derived sizes every launcher needs.
struct Problem {
  moe_config_t cfg;
  int64_t Tu;        // routed units T' = T·H
  int hu;            // unit width h' = h/H
  int E, K, d_ff;
  int n_groups, topk_groups;
  bool bf16;
  bool sigmoid;
  int64_t C;         // capacity, or INT64_MAX for no drop
  int64_t rows;      // packed-row capacity T'·K
  int64_t ntiles;    // ceil(T'/kTileUnits): routing tiles
  int64_t nchunks;   // ceil(T'/kChunk): chunks of the dispatch from given picks
  size_t elt;        // bytes per activation/weight element (2 or 4)
};

// Routing of one tile of units (select_tile.cuh): where the picks and gates go.
struct SelectCtx {
  const float* select_bias;  // [E] or null (sigmoid only)
  int32_t* idx;              // [T'][K]
  float* gate;               // [T'][K]
  int E, K, n_groups, topk_groups;
};

// Tensor-core router plan (route_tc.cu): MMA N = 64·nblk; a cluster of S CTAs per 128-unit tile,
// each over kbs of the nkb 64-wide k-blocks.
struct RouterPlan {
  int nblk, Np, m_tiles, nkb, S, kbs;
};
RouterPlan router_plan(const Problem& p, int sms);

// Offsets (bytes) of the workspace regions; every region starts 1024-byte aligned.
struct WsLayout {
  size_t status;       // uint32 status word at +0, uint32 scan ticket at +8
  size_t counts;       // int32 [E]
  size_t offsets;      // int32 [E+1]
  size_t chunk_hist;   // int32 [ntiles][E] picks per expert of each tile / chunk
  size_t chunk_base;   // int32 [ntiles][E] each tile's / chunk's base in the expert queues
  size_t psum;         // float [ntiles][E] Σ over the tile's units of p_{t,e}
  size_t aux_terms;    // float [E] per-expert aux terms
  size_t cap;          // int64 [E] capacity left per expert (dispatch of a shard)
  size_t w_pad;        // bf16 [h'][E rounded up to 8] router weight copy (bf16 layers, when needed)
  size_t logits;       // float [T'][E] router logits (fp32 layers)
  size_t rank;         // int32 [T'][K] pick places within their tile (routing calls alone)
  size_t idx;          // int32 [T'][K]
  size_t gate;         // float [T'][K]
  size_t slot_of;      // int32 [T'][K]
  size_t row_token;    // int32 [T'K]
  size_t x_packed;     // elt [T'K][h']
  size_t hidden;       // elt [T'K][d_ff]
  size_t y_packed;     // elt [T'K][h']
  size_t arrivals;     // uint32 [T'][h'/32] rows done per unit and 32-column chunk (bf16 layers)
  size_t total;
};

// Scratch of the dispatch from given picks (workspace regions, or the fixed array of the
// allocation-free call).
struct DispatchScratch {
  int32_t* chunk_hist;   // [nchunks][E]
  int32_t* chunk_base;   // [nchunks][E]
  int32_t* counts;       // [E]
  int32_t* offsets;      // [E+1]
  unsigned int* ticket;  // zero between calls
  uint32_t* status;      // or null
  const int32_t* qbase = nullptr;  // shard of a larger batch: picks per expert on earlier ranks [E]
  int64_t* cap = nullptr;          // then: capacity left per expert [E] (scratch)
};

moe_status_t make_problem(const moe_config_t* cfg, Problem* p);
WsLayout ws_layout(const Problem& p);

template <typename T>
inline T* ws_ptr(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

// Per-device facts (cached).
int device_sm_count();

// Counts every kernel this library enqueues.
void note_launch(int n = 1);

// Launch `kern` on `s` and return that launch's own error (no earlier error is picked up).
// cluster > 1: thread-block clusters of that many CTAs along x. pdl: programmatic dependent launch
// (the kernel may start before the previous kernel of the stream ends; it must call griddep_wait
// before reading anything that kernel writes, or writing anything it reads).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                          unsigned cluster, bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  unsigned n = 0;
  if (cluster > 1) {
    at[n].id = cudaLaunchAttributeClusterDimension;
    at[n].val.clusterDim.x = cluster;
    at[n].val.clusterDim.y = 1;
    at[n].val.clusterDim.z = 1;
    ++n;
  }
  if (pdl) {
    at[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = at;
  cfg.numAttrs = n;
  note_launch();
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// Tensor-map encoding through the driver entry point (no link-time libcuda dependency).
bool encode_tmap_2d_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                         uint32_t box_inner, uint32_t box_outer);

// A row-major bf16 matrix [rows][cols] (cols a multiple of 64) as the 3-D tensor
// {64 elements, rows, cols/64 column blocks}: a box of `box_rows` rows by `blocks` column blocks
// lands in shared memory as `blocks` MN-major 128-byte-swizzled tiles, box_rows·128 bytes apart.
bool encode_tmap_mn_blocks_bf16(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows,
                                uint32_t box_rows, uint32_t blocks);

// fp32 [d2][d1][d0] tensor (d0 contiguous) with a {box0, box1, 1} box and 128-byte swizzle
// (box0·4 must be 128 bytes or less): the target of tiled stores from swizzled shared memory.
bool encode_tmap_3d_f32_sw128(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                              uint32_t box0, uint32_t box1);

// ---- launchers (return cudaSuccess or the launch error) --------------------------------------
// pdl: the launch may overlap the previous kernel of the stream (see launch_kernel).

// bf16 layers: router GEMM + routing of each 128-unit tile in one kernel (plus a padded copy of W_g
// into w_pad first when E % 8 != 0 or W_g is not 16-byte aligned).
cudaError_t launch_route_tc(const Problem& p, const void* x, const void* w_router, const float* logit_bias,
                            const SelectCtx& sel, float* logits_out, int32_t* rank_out, int32_t* tile_hist,
                            float* tile_psum, void* w_pad, uint32_t* status, cudaStream_t s);
// fp32 layers: router logits [T'][E] on the CUDA cores.
cudaError_t launch_router_simt_logits(const Problem& p, const void* x, const void* w, float* logits, cudaStream_t s);
// Routing of each 128-unit tile from given fp32 logits (the logit bias added in fp32).
cudaError_t launch_select_logits(const Problem& p, const float* logits, const float* logit_bias, const SelectCtx& sel,
                                 float* logits_out, int32_t* rank_out, int32_t* tile_hist, float* tile_psum,
                                 cudaStream_t s, bool pdl);
// Hash gate (K = 1): expert fmix32(token id) mod E, gate 1, with the per-tile counts and places.
cudaError_t launch_hash_route(const Problem& p, const int32_t* token_ids, int32_t* idx, float* gate, int32_t* rank_out,
                              int32_t* tile_hist, cudaStream_t s);
// Per expert: chunk bases, pre-drop counts, offsets; the aux loss when psum and aux_out are given.
cudaError_t launch_scan(const Problem& p, int64_t nchunks, const int32_t* hist, const float* psum,
                        int32_t* chunk_base, int32_t* counts_ws, int32_t* offsets_ws, int32_t* counts_out,
                        int32_t* offsets_out, float* terms, unsigned int* ticket, float* aux_out, cudaStream_t s,
                        bool pdl, const int32_t* qbase = nullptr, int64_t* cap_out = nullptr);
// Slots of the picks (slot_of holds the places within chunks of 2^chunk_shift units on entry) and
// the packed rows.
cudaError_t launch_pack(const Problem& p, const void* x, const int32_t* idx, int chunk_shift, const int32_t* chunk_base,
                        const int32_t* offsets, int32_t* slot_of, int32_t* row_token, void* x_packed, cudaStream_t s,
                        bool pdl, const int64_t* cap_e = nullptr, void* y_zero = nullptr,
                        uint32_t* arrivals = nullptr);
// The whole dispatch from given picks: chunk ranks, scan, pack.
cudaError_t launch_dispatch_from_idx(const Problem& p, const void* x, const int32_t* idx, int32_t* counts_out,
                                     int32_t* offsets_out, int32_t* slot_of, int32_t* row_token, void* x_packed,
                                     const DispatchScratch& sc, cudaStream_t s);

// save_gu (bf16 layers): also write the SwiGLU inputs G | U as bf16 [rows][2·d_ff] for the backward.
// moe_set_expert_gemm: forced choices of the expert GEMMs (-1 automatic).
void set_expert_gemm(int pair_tiles, int transposed_tails, int fold_combine);
// Whether moe_forward folds the combine into the down GEMM (bf16 layers).
bool fold_combine(const Problem& p);

// The combine folded into the down GEMM (expert_tc.cu): the down launch also writes y.
struct FusedCombine {
  void* y;                   // [T'][h'] layer output
  const int32_t* row_token;  // [rows] packed row -> unit
  const int32_t* slot_of;    // [T'][K]
  const float* gate;         // [T'][K]
  uint32_t* arrivals;        // [T'][h'/32], zeroed by the pack of the same forward
  bool keep_packed;          // also leave every Y row in y_packed (the backward reads it)
};

cudaError_t launch_expert_ffn(const Problem& p, const void* x_packed, const int32_t* offsets,
                              const void* w_gate, const void* w_up, const void* w_down,
                              void* hidden, void* y_packed, uint32_t* status, cudaStream_t s,
                              void* save_gu = nullptr, bool pdl = false, const FusedCombine* fc = nullptr);

// ---- backward (bf16 layers, h' and d_ff multiples of 64) ---------------------------------------
cudaError_t launch_expert_ffn_backward(const Problem& p, const int32_t* offsets, const void* x_packed,
                                       const void* hidden, const void* gu, const void* dy_packed,
                                       const void* w_gate, const void* w_up, const void* w_down,
                                       void* dgu, void* dx_packed, float* dw_gate, float* dw_up,
                                       float* dw_down, void* dy_t, void* x_t, uint32_t* status, cudaStream_t s);
int64_t backward_padded_cols(const Problem& p);  // columns of the padded transposed copies
cudaError_t launch_backward_misc_combine(const Problem& p, const void* dy, const void* y_packed,
                                         const int32_t* slot_of, const float* gate, void* dy_packed,
                                         float* dgate, uint32_t* status, cudaStream_t s);
cudaError_t launch_backward_logits(const Problem& p, const float* logits, const int32_t* idx, const float* gate,
                                   const float* dgate, const int32_t* counts, float d_aux, float* dl,
                                   cudaStream_t s);
int backward_wg_chunks(const Problem& p);
cudaError_t launch_backward_router(const Problem& p, const void* x, const float* dl, int nchunks, float* part,
                                   float* dw_router, cudaStream_t s);
// W_gᵀ [E][h'] (bf16) for dx += dl·W_gᵀ.
cudaError_t launch_router_transpose(const Problem& p, const void* w_router, void* wt, cudaStream_t s);
cudaError_t launch_backward_dx(const Problem& p, const void* dx_packed, const int32_t* slot_of, const float* dl,
                               const void* w_router_t, void* dx, cudaStream_t s);

cudaError_t launch_combine(const Problem& p, const void* y_packed, const int32_t* slot_of,
                           const float* gate, void* y, uint32_t* status, cudaStream_t s, bool pdl = false);

}  // namespace moe
