// Routing of a tile of units whose fp32 logits (logit bias included) sit in shared memory: scores,
// optional group limit, Top-K, gates, each unit's probabilities for the aux loss, and the
// per-expert pick counts and in-tile queue places that the dispatch needs.
//   [Lesson 10 "专家并行 EP", §1: s(x) = Softmax(TopK(x·W_g, K)) or sigmoid normalisation;
//    §4: L_aux = α·E·Σ f_i·P_i; §5: a unit's experts restricted to a few groups]
//
// Selection keys: softmax → the fp32 logit itself (TopK acts on x·W_g); sigmoid → σ(l) + b formed
// in fp64. Ties go to the lower expert index (and lower group index). Gates: softmax over the K
// picked logits, or σ_i/Σσ over the picks (unbiased).
//
// Used by the fused router kernel (route_tc.cu: logits reduced from the tensor-core partials) and by
// the kernel that routes given logits (route.cu). Two shapes, both block-level (every thread of the
// block calls them, with the same arguments):
//   E <= 64: one thread per unit scans its row in expert order keeping a sorted list of its K best
//            (key, index); an equal key never displaces a lower index.
//   E > 64:  one warp per unit, each lane E/32 experts; keys are compared as order-preserving
//            integers so shuffles and comparisons stay off the fp64 pipe.
// Each leaves the unit's picks in a shared [R][K] tile and overwrites the unit's logit row with its
// probabilities; column sums (fixed row order) then give the tile's Σ_t P_{t,i}, and the rank pass
// gives each pick's place among the tile's picks of the same expert (unit order) and the tile's
// pick count per expert.
#pragma once

#include <math.h>

#include <type_traits>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {

// Row stride of the shared [R][·] tiles of picks and places (the largest K).
constexpr int kPickStride = 8;

__device__ __forceinline__ double sigmoid64(float l) { return 1.0 / (1.0 + exp(-(double)l)); }

// Order-preserving map of a double to uint64 (−0 is folded into +0 first).
__device__ __forceinline__ uint64_t ord64(double d) {
  d = d + 0.0;
  const uint64_t u = (uint64_t)__double_as_longlong(d);
  return (u >> 63) ? ~u : (u | 0x8000000000000000ull);
}

// Order-preserving map of a float to uint32 (−0 folded into +0).
__device__ __forceinline__ uint32_t ord32(float f) {
  f = f + 0.0f;
  const uint32_t u = __float_as_uint(f);
  return (u >> 31) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float unord32(uint32_t u) {
  return __uint_as_float((u >> 31) ? (u & 0x7fffffffu) : ~u);
}

// Warp argmax on (ordered key desc, index asc) over candidates; returns the winner's index or
// 0x7fffffff (none) and its key.
__device__ __forceinline__ int warp_argmax32(uint32_t k, int idx, uint32_t& best_k) {
#pragma unroll
  for (int d = 16; d; d >>= 1) {
    const uint32_t ok = __shfl_xor_sync(0xffffffffu, k, d);
    const int oi = __shfl_xor_sync(0xffffffffu, idx, d);
    if (oi != 0x7fffffff && (idx == 0x7fffffff || ok > k || (ok == k && oi < idx))) { k = ok; idx = oi; }
  }
  best_k = k;
  return idx;
}

// ============================================================================ thread per unit
template <bool SIGMOID>
__device__ __forceinline__ typename std::conditional<SIGMOID, double, float>::type
sel_key(const SelectCtx& c, const float* row, int e) {
  if constexpr (SIGMOID) return sigmoid64(row[e]) + (c.select_bias ? (double)c.select_bias[e] : 0.0);
  else return row[e];
}

// Thread t < R routes unit u0 + t from row t of `lg` (row stride ld). picks: [R][kPickStride] in
// shared memory (entries past K are not written).
template <int KMAX, bool SIGMOID>
__device__ void select_rows_thread(const SelectCtx& c, float* lg, int ld, int R, int64_t u0, int* picks) {
  using KeyT = typename std::conditional<SIGMOID, double, float>::type;
  const int t = threadIdx.x;
  if (t >= R) return;
  const int E = c.E, K = c.K;
  float* row = lg + t * ld;

  // group limit: keep the topk_groups groups with the largest sum of their two best keys
  uint64_t eligible = ~0ull;
  if (c.n_groups > 1) {
    const int gs = E / c.n_groups;
    uint32_t chosen = 0;
    for (int q = 0; q < c.topk_groups; ++q) {
      int bg = -1;
      double bsc = 0.0;
      for (int g = 0; g < c.n_groups; ++g) {
        if ((chosen >> g) & 1u) continue;
        double t1 = -INFINITY, t2 = -INFINITY;
        for (int i = 0; i < gs; ++i) {
          const double k = (double)sel_key<SIGMOID>(c, row, g * gs + i);
          if (k > t1) { t2 = t1; t1 = k; }
          else if (k > t2) t2 = k;
        }
        const double sc = gs > 1 ? t1 + t2 : t1;
        if (bg < 0 || sc > bsc) { bg = g; bsc = sc; }
      }
      chosen |= 1u << bg;
    }
    eligible = 0;
    for (int e = 0; e < E; ++e)
      if ((chosen >> (e / gs)) & 1u) eligible |= 1ull << e;
  }

  // Top-K: experts in index order into bk[0..K) kept sorted by key, descending. A new key goes
  // below every kept key that is >= it (an equal key never displaces an earlier, lower index);
  // the entries it passes shift down one slot. be = -1 marks an empty slot.
  KeyT bk[KMAX];
  int be[KMAX];
#pragma unroll
  for (int j = 0; j < KMAX; ++j) { bk[j] = (KeyT)-INFINITY; be[j] = -1; }
  for (int e = 0; e < E; ++e) {
    if (!((eligible >> e) & 1ull)) continue;
    const KeyT ck = sel_key<SIGMOID>(c, row, e);
#pragma unroll
    for (int s = KMAX - 1; s >= 0; --s) {
      if (s < K) {
        const bool above = s > 0 && (be[s - 1] < 0 || ck > bk[s - 1]);
        const bool here = be[s] < 0 || ck > bk[s];
        if (above) { bk[s] = bk[s - 1]; be[s] = be[s - 1]; }
        else if (here) { bk[s] = ck; be[s] = e; }
      }
    }
  }

  // gates from the picked logits
  const int64_t u = u0 + t;
  float lv[KMAX];
#pragma unroll
  for (int j = 0; j < KMAX; ++j) lv[j] = (j < K && be[j] >= 0) ? row[be[j]] : 0.f;
  if (SIGMOID) {
    double sg[KMAX], z = 0.0;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) { sg[j] = (j < K) ? sigmoid64(lv[j]) : 0.0; z += sg[j]; }
#pragma unroll
    for (int j = 0; j < KMAX; ++j)
      if (j < K) { c.idx[u * K + j] = be[j]; c.gate[u * K + j] = (float)(sg[j] / z); }
  } else {
    float ev[KMAX], z = 0.f;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) { ev[j] = (j < K) ? expf(lv[j] - lv[0]) : 0.f; z += ev[j]; }
#pragma unroll
    for (int j = 0; j < KMAX; ++j)
      if (j < K) { c.idx[u * K + j] = be[j]; c.gate[u * K + j] = ev[j] / z; }
  }
#pragma unroll
  for (int j = 0; j < KMAX; ++j)
    if (j < K) picks[t * kPickStride + j] = be[j];

  // this unit's probabilities replace its logits
  float m = -INFINITY, z = 0.f;
  if (!SIGMOID)
    for (int e = 0; e < E; ++e) m = fmaxf(m, row[e]);
  for (int e = 0; e < E; ++e) {
    const float v = SIGMOID ? (float)sigmoid64(row[e]) : __expf(row[e] - m);
    z += v;
    row[e] = v;
  }
  const float iz = 1.f / z;
  for (int e = 0; e < E; ++e) row[e] = row[e] * iz;
}

// ============================================================================ warp per unit
// Warps take rows w, w + NW, ...; lanes hold EPL contiguous experts (E <= 32·EPL).
// gscratch: shared, 32 · EPL · 8 bytes per warp (the unit's keys, read per group by the group lanes).
template <int EPL, bool SIGMOID>
__device__ void select_rows_warp(const SelectCtx& c, float* lg, int ld, int R, int64_t u0, int* picks,
                                 unsigned char* gscratch) {
  constexpr int EP = 32 * EPL;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int E = c.E, K = c.K;
  const int gs = E / c.n_groups;
  double* kdbl_w = reinterpret_cast<double*>(gscratch) + (size_t)warp * EP;
  for (int r = warp; r < R; r += nw) {
    const int64_t u = u0 + r;
    float* row = lg + r * ld;
    float lv[EPL];
    bool valid[EPL];
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
      const int e = lane * EPL + j;
      valid[j] = e < E;
      lv[j] = valid[j] ? row[e] : -INFINITY;
    }
    // Sigmoid keys σ(l)+b are decided in fp64. First screen in fp32: |key32 − key64| <= 4.3e-7
    // (accurate expf, IEEE divide, one rounding of the add), so when every decision's fp32 margin
    // exceeds twice that bound (group scores: two keys and a rounded add each) the fp32 decisions
    // equal the fp64 ones; otherwise this unit takes the fp64 path below.
    int sel_e = -1;
    bool screened = false;
    uint32_t chosen = 0xffffffffu;
    if (SIGMOID) {
      constexpr float kDelta = 1e-6f;
      float k32[EPL];
      uint32_t o32[EPL];
#pragma unroll
      for (int j = 0; j < EPL; ++j) {
        const int e = lane * EPL + j;
        k32[j] = valid[j] ? (1.0f / (1.0f + expf(-lv[j]))) + (c.select_bias ? c.select_bias[e] : 0.0f) : -INFINITY;
        o32[j] = ord32(k32[j]);
      }
      bool safe = true;
      if (c.n_groups > 1) {
        float* gk = reinterpret_cast<float*>(kdbl_w);
#pragma unroll
        for (int j = 0; j < EPL; ++j) gk[lane * EPL + j] = k32[j];
        __syncwarp();
        uint32_t gord = 0;
        int gidx = 0x7fffffff;
        if (lane < c.n_groups) {
          float t1 = -INFINITY, t2 = -INFINITY;
          for (int i = 0; i < gs; ++i) {
            const float v = gk[lane * gs + i];
            if (v > t1) { t2 = t1; t1 = v; }
            else if (v > t2) t2 = v;
          }
          gord = ord32(gs > 1 ? t1 + t2 : t1);
          gidx = lane;
        }
        __syncwarp();
        chosen = 0;
        float last_sc = 0.f;
        for (int q = 0; q <= c.topk_groups && q < c.n_groups; ++q) {
          const bool cand = gidx != 0x7fffffff && !((chosen >> lane) & 1u);
          uint32_t bk;
          const int bg = warp_argmax32(cand ? gord : 0u, cand ? gidx : 0x7fffffff, bk);
          const float sc = unord32(bk);
          if (q < c.topk_groups) {
            chosen |= 1u << bg;
            last_sc = sc;
          } else if (!(last_sc - sc > 4.0f * kDelta + 4.0e-7f)) {
            safe = false;
          }
        }
      }
      bool taken[EPL];
#pragma unroll
      for (int j = 0; j < EPL; ++j) taken[j] = false;
      float prev = 0.f;
      for (int q = 0; q <= K; ++q) {
        uint32_t bk = 0;
        int be = 0x7fffffff;
#pragma unroll
        for (int j = 0; j < EPL; ++j) {
          const int e = lane * EPL + j;
          const bool elig = valid[j] && !taken[j] && ((chosen >> (e / gs)) & 1u);
          if (elig && (be == 0x7fffffff || o32[j] > bk)) { bk = o32[j]; be = e; }
        }
        uint32_t wk;
        be = warp_argmax32(bk, be, wk);
        if (be == 0x7fffffff) break;  // fewer than K+1 eligible experts: no further margin
        const float kv = unord32(wk);
        if (q > 0 && !(prev - kv > 2.0f * kDelta)) safe = false;
        prev = kv;
        if (q < K) {
#pragma unroll
          for (int j = 0; j < EPL; ++j)
            if (be == lane * EPL + j) taken[j] = true;
          if (lane == q) sel_e = be;
        }
      }
      screened = safe;
    }
    if (!screened) {
      // fp64 decision (all softmax units; sigmoid units whose fp32 screen was not conclusive)
      uint64_t ko[EPL];
      double kd[EPL];
#pragma unroll
      for (int j = 0; j < EPL; ++j) {
        const int e = lane * EPL + j;
        kd[j] = SIGMOID ? (valid[j] ? sigmoid64(lv[j]) + (c.select_bias ? (double)c.select_bias[e] : 0.0) : -INFINITY)
                        : (double)lv[j];
        ko[j] = ord64(kd[j]);
      }
      chosen = 0xffffffffu;
      if (c.n_groups > 1) {
        __syncwarp();
#pragma unroll
        for (int j = 0; j < EPL; ++j) kdbl_w[lane * EPL + j] = kd[j];
        __syncwarp();
        uint64_t gord = 0;
        bool gval = false;
        if (lane < c.n_groups) {
          double t1 = -INFINITY, t2 = -INFINITY;
          for (int i = 0; i < gs; ++i) {
            const double v = kdbl_w[lane * gs + i];
            if (v > t1) { t2 = t1; t1 = v; }
            else if (v > t2) t2 = v;
          }
          gord = ord64(gs > 1 ? t1 + t2 : t1);
          gval = true;
        }
        __syncwarp();
        chosen = 0;
        for (int q = 0; q < c.topk_groups; ++q) {
          const bool cand = gval && !((chosen >> lane) & 1u);
          uint64_t bk = cand ? gord : 0;
          int bg = cand ? lane : 0x7fffffff;
#pragma unroll
          for (int d = 16; d; d >>= 1) {
            const uint64_t ok = __shfl_xor_sync(0xffffffffu, bk, d);
            const int og = __shfl_xor_sync(0xffffffffu, bg, d);
            if (og != 0x7fffffff && (bg == 0x7fffffff || ok > bk || (ok == bk && og < bg))) { bk = ok; bg = og; }
          }
          if (bg != 0x7fffffff) chosen |= 1u << bg;
        }
      }
      // Top-K: K rounds of a warp argmax on (ordered key desc, index asc)
      bool taken[EPL];
#pragma unroll
      for (int j = 0; j < EPL; ++j) taken[j] = false;
      for (int q = 0; q < K; ++q) {
        uint64_t bk = 0;
        int be = 0x7fffffff;
#pragma unroll
        for (int j = 0; j < EPL; ++j) {
          const int e = lane * EPL + j;
          const bool elig = valid[j] && !taken[j] && ((chosen >> (e / gs)) & 1u);
          if (elig && (be == 0x7fffffff || ko[j] > bk)) { bk = ko[j]; be = e; }
        }
#pragma unroll
        for (int d = 16; d; d >>= 1) {
          const uint64_t ok = __shfl_xor_sync(0xffffffffu, bk, d);
          const int oe = __shfl_xor_sync(0xffffffffu, be, d);
          if (oe != 0x7fffffff && (be == 0x7fffffff || ok > bk || (ok == bk && oe < be))) { bk = ok; be = oe; }
        }
#pragma unroll
        for (int j = 0; j < EPL; ++j)
          if (be == lane * EPL + j) taken[j] = true;
        if (lane == q) sel_e = (be == 0x7fffffff) ? -1 : be;
      }
    }
    // gates from the picked logits (read before the row is overwritten below)
    const float l_sel = (lane < K && sel_e >= 0) ? row[sel_e] : 0.f;
    const float l_top = __shfl_sync(0xffffffffu, l_sel, 0);
    float g;
    if (SIGMOID) {
      const double s = (lane < K) ? sigmoid64(l_sel) : 0.0;
      double z = s;
#pragma unroll
      for (int d = 16; d; d >>= 1) z += __shfl_xor_sync(0xffffffffu, z, d);
      g = (float)(s / z);
    } else {
      const float ev = (lane < K) ? expf(l_sel - l_top) : 0.f;
      float z = ev;
#pragma unroll
      for (int d = 16; d; d >>= 1) z += __shfl_xor_sync(0xffffffffu, z, d);
      g = ev / z;
    }
    if (lane < K) {
      c.idx[u * K + lane] = sel_e;
      c.gate[u * K + lane] = g;
      picks[r * kPickStride + lane] = sel_e;
    }
    // P_i for the aux loss: the unit's probabilities replace its logits
    float pv[EPL], z = 0.f, m = -INFINITY;
    if (!SIGMOID) {
#pragma unroll
      for (int j = 0; j < EPL; ++j) m = fmaxf(m, lv[j]);
#pragma unroll
      for (int d = 16; d; d >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d));
    }
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
      pv[j] = !valid[j] ? 0.f : (SIGMOID ? 1.0f / (1.0f + expf(-lv[j])) : expf(lv[j] - m));
      z += pv[j];
    }
#pragma unroll
    for (int d = 16; d; d >>= 1) z += __shfl_xor_sync(0xffffffffu, z, d);
    __syncwarp();
#pragma unroll
    for (int j = 0; j < EPL; ++j)
      if (valid[j]) row[lane * EPL + j] = pv[j] / z;
    __syncwarp();
  }
}

// ============================================================================ tile reductions
// out[e] = Σ_{r<R} lg[r][e] for e < E, in a fixed order: P = blockDim/E threads per column each sum
// a contiguous block of rows, then the P partial sums of a column in order. scratch: blockDim floats.
// Requires E <= blockDim.x. Ends with a block barrier.
__device__ __forceinline__ void column_sums(const float* lg, int ld, int R, int E, float* out, float* scratch) {
  const int t = threadIdx.x, nt = blockDim.x;
  const int P = nt / E;
  const int e = t / P, part = t % P;
  const int rows_per = (R + P - 1) / P;
  float s = 0.f;
  if (e < E) {
    const int r0 = part * rows_per, r1 = min(R, r0 + rows_per);
    for (int r = r0; r < r1; ++r) s += lg[r * ld + e];
  }
  scratch[t] = s;
  __syncthreads();
  if (t < E) {
    float tot = 0.f;
    for (int q = 0; q < P; ++q) tot += scratch[t * P + q];
    out[t] = tot;
  }
  __syncthreads();
}

// Places of the picks within the tile: rank[r][k] = number of (r', k') with r' < r and the same
// expert (a unit's picks are distinct, so this is the unit-order queue of the expert within the
// tile); -1 for a pick of -1. hist[e] = picks of expert e in the tile. lanes_of / warp_pre: shared,
// blockDim/32 · E entries each. Ends with a block barrier.
__device__ __forceinline__ void rank_picks(const int* picks, int R, int K, int E, int* rank, int* hist,
                                           uint32_t* lanes_of, int* warp_pre) {
  constexpr int kstride = kPickStride;
  const int t = threadIdx.x, nt = blockDim.x, nw = nt >> 5, w = t >> 5, lane = t & 31;
  for (int i = t; i < nw * E; i += nt) lanes_of[i] = 0u;
  __syncthreads();
  if (t < R)
    for (int k = 0; k < K; ++k) {
      const int e = picks[t * kstride + k];
      if (e >= 0) atomicOr(&lanes_of[w * E + e], 1u << lane);
    }
  __syncthreads();
  for (int e = t; e < E; e += nt) {
    int run = 0;
    for (int q = 0; q < nw; ++q) {
      warp_pre[q * E + e] = run;
      run += __popc(lanes_of[q * E + e]);
    }
    hist[e] = run;
  }
  __syncthreads();
  if (t < R)
    for (int k = 0; k < K; ++k) {
      const int e = picks[t * kstride + k];
      rank[t * kstride + k] = e >= 0 ? warp_pre[w * E + e] + __popc(lanes_of[w * E + e] & lanemask_lt()) : -1;
    }
  __syncthreads();
}

}  // namespace moe
