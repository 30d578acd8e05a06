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
constexpr int kChunk = 256;          // units per dispatch chunk (one block, one thread per unit)
constexpr size_t kWsAlign = 1024;
constexpr int kRouterSplitTarget = 160;  // aim for about this many router CTAs (>= SMs of a B300)

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
  int64_t nchunks;   // ceil(T'/kChunk)
  int route_bt;      // units per router block
  int64_t route_blocks;
  size_t elt;        // bytes per activation/weight element (2 or 4)
};

// Tensor-core router GEMM plan: N = E rounded up to 16, K split into `splits` slices.
struct RouterPlan {
  int N, m_tiles, nkb, kb_per_split, splits;
};
RouterPlan router_plan(const Problem& p);

// Offsets (bytes) of the workspace regions; every region starts 1024-byte aligned.
struct WsLayout {
  size_t status;       // uint32 status word at +0, uint32 aux finalize ticket at +4
  size_t counts;       // int32 [E]
  size_t offsets;      // int32 [E+1]
  size_t chunk_hist;   // int32 [nchunks][E]
  size_t chunk_base;   // int32 [nchunks][E]
  size_t psum_part;    // float [route_blocks][E]
  size_t cnt_part;     // int32 [route_blocks][E]
  size_t aux_terms;    // double [E] per-expert aux terms
  size_t router_wt;    // bf16 [N][h'] transposed router weight (bf16 layers)
  size_t router_part;  // float [splits][T'][E] partial logits (bf16 layers)
  size_t idx;          // int32 [T'][K]
  size_t gate;         // float [T'][K]
  size_t slot_of;      // int32 [T'][K]
  size_t row_token;    // int32 [T'K]
  size_t x_packed;     // elt [T'K][h']
  size_t hidden;       // elt [T'K][d_ff]
  size_t y_packed;     // elt [T'K][h']
  size_t total;
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
cudaError_t launch_route(const Problem& p, const void* x, const void* w_router,
                         const float* logits_in, const float* logit_bias, const float* select_bias,
                         int32_t* idx, float* gate, float* logits_out, float* aux_out, void* ws,
                         cudaStream_t s);

cudaError_t launch_router_tc(const Problem& p, const void* x, const void* w_router, void* wt, float* part,
                             uint32_t* status, cudaStream_t s);

cudaError_t launch_dispatch(const Problem& p, const void* x, const int32_t* idx, int32_t* counts,
                            int32_t* offsets, int32_t* slot_of, int32_t* row_token, void* x_packed,
                            void* ws, cudaStream_t s);

// save_gu (bf16 layers): also write the SwiGLU inputs G | U as bf16 [rows][2·d_ff] for the backward.
cudaError_t launch_expert_ffn(const Problem& p, const void* x_packed, const int32_t* offsets,
                              const void* w_gate, const void* w_up, const void* w_down,
                              void* hidden, void* y_packed, uint32_t* status, cudaStream_t s,
                              void* save_gu = nullptr);

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
cudaError_t launch_backward_dx(const Problem& p, const void* dx_packed, const int32_t* slot_of, const float* dl,
                               const void* w_router_t, void* dx, cudaStream_t s);

cudaError_t launch_combine(const Problem& p, const void* y_packed, const int32_t* slot_of,
                           const float* gate, void* y, uint32_t* status, cudaStream_t s);

}  // namespace moe
