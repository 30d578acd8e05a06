// Routing of a tile of units whose fp32 logits (logit bias included) sit in shared memory: scores,
// optional group limit, Top-K, gates, each unit's probabilities for the aux loss, and the
// per-expert pick counts and in-tile queue places that the dispatch needs.
//   [Lesson 10 "专家并行 EP", §1: s(x) = Softmax(TopK(x·W_g, K)) or sigmoid normalisation;
//    §4: L_aux = α·E·Σ f_i·P_i; §5: a unit's experts restricted to a few groups]
//
// Selection keys: softmax → the fp32 logit itself (TopK acts on x·W_g); sigmoid → σ(l) + b formed
// in fp64 (decided in fp32 first where the fp32 margins prove the same outcome). Ties go to the
// lower expert index (and lower group index). Gates, in fp32: softmax over the K picked logits, or
// σ_i/Σσ over the picks (unbiased).
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

// Warp argmax of 32-bit ordered keys over the lanes with `has` set: one reduction and one ballot.
// On equal keys the lowest such lane wins, so candidates must sit in lanes in index order. Returns
// the winning lane's idx (0x7fffffff if no lane has a candidate) and, in best, its key.
__device__ __forceinline__ int warp_argmax_redux(uint32_t key, bool has, int idx, uint32_t& best) {
  const uint32_t m = __reduce_max_sync(0xffffffffu, has ? key : 0u);
  const uint32_t w = __ballot_sync(0xffffffffu, has && key == m);
  best = m;
  if (!w) return 0x7fffffff;
  return __shfl_sync(0xffffffffu, idx, __ffs(w) - 1);
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
    for (int g = 0, e0 = 0; g < c.n_groups; ++g, e0 += gs)
      if ((chosen >> g) & 1u) eligible |= (gs >= 64 ? ~0ull : ((1ull << gs) - 1ull)) << e0;
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
    float sg[KMAX], z = 0.f;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) { sg[j] = (j < K) ? 1.0f / (1.0f + expf(-lv[j])) : 0.f; z += sg[j]; }
#pragma unroll
    for (int j = 0; j < KMAX; ++j)
      if (j < K) { c.idx[u * K + j] = be[j]; c.gate[u * K + j] = sg[j] / z; }
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
  // group of each of this lane's experts (integer division once, not in every argmax round)
  int grp[EPL];
#pragma unroll
  for (int j = 0; j < EPL; ++j) grp[j] = (lane * EPL + j) / gs;
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
    float sgm[EPL];  // σ(l) in fp32 (sigmoid scoring): the screen's keys and the unit's P_i
    if (SIGMOID) {
      constexpr float kDelta = 1e-6f;
      float k32[EPL];
      uint32_t o32[EPL];
#pragma unroll
      for (int j = 0; j < EPL; ++j) {
        const int e = lane * EPL + j;
        sgm[j] = valid[j] ? 1.0f / (1.0f + expf(-lv[j])) : 0.0f;
        k32[j] = valid[j] ? sgm[j] + (c.select_bias ? c.select_bias[e] : 0.0f) : -INFINITY;
        o32[j] = ord32(k32[j]);
      }
      bool safe = true;
      if (c.n_groups > 1) {
        // group scores: the sum of each group's two largest keys
        uint32_t gord = 0;
        bool gcand = false;
        int gidx = 0x7fffffff;
        const int lpg = gs / EPL;  // lanes per group when groups are whole lanes
        if (gs % EPL == 0 && (lpg & (lpg - 1)) == 0) {
          // a group is lpg adjacent lanes: local top-2, then a butterfly over the group's lanes
          float t1 = -INFINITY, t2 = -INFINITY;
#pragma unroll
          for (int j = 0; j < EPL; ++j) {
            const float v = k32[j];
            if (v > t1) { t2 = t1; t1 = v; }
            else if (v > t2) t2 = v;
          }
          for (int o = 1; o < lpg; o <<= 1) {
            const float b1 = __shfl_xor_sync(0xffffffffu, t1, o), b2 = __shfl_xor_sync(0xffffffffu, t2, o);
            const float n2 = fmaxf(fminf(t1, b1), fmaxf(t2, b2));
            t1 = fmaxf(t1, b1);
            t2 = n2;
          }
          gcand = (lane % lpg) == 0 && lane / lpg < c.n_groups;
          gord = ord32(gs > 1 ? t1 + t2 : t1);
          gidx = lane / lpg;
        } else {
          float* gk = reinterpret_cast<float*>(kdbl_w);
#pragma unroll
          for (int j = 0; j < EPL; ++j) gk[lane * EPL + j] = k32[j];
          __syncwarp();
          if (lane < c.n_groups) {
            float t1 = -INFINITY, t2 = -INFINITY;
            for (int i = 0; i < gs; ++i) {
              const float v = gk[lane * gs + i];
              if (v > t1) { t2 = t1; t1 = v; }
              else if (v > t2) t2 = v;
            }
            gord = ord32(gs > 1 ? t1 + t2 : t1);
            gidx = lane;
            gcand = true;
          }
          __syncwarp();
        }
        chosen = 0;
        float last_sc = 0.f;
        for (int q = 0; q <= c.topk_groups && q < c.n_groups; ++q) {
          const bool cand = gcand && !((chosen >> gidx) & 1u);
          uint32_t bk;
          const int bg = warp_argmax_redux(gord, cand, gidx, bk);
          const float sc = unord32(bk);
          if (q < c.topk_groups) {
            chosen |= 1u << bg;
            last_sc = sc;
          } else if (!(last_sc - sc > 4.0f * kDelta + 4.0e-7f)) {
            safe = false;
          }
        }
      }
      // Top-(K+1) over the eligible keys: each lane sorts its candidates once on (key desc, index
      // asc) — key in the high word, inverted index in the low word, 0 for none — then every round
      // compares the lanes' heads and the winning lane drops its head.
      uint64_t cand[EPL];
#pragma unroll
      for (int j = 0; j < EPL; ++j)
        cand[j] = (valid[j] && ((chosen >> grp[j]) & 1u))
                      ? ((uint64_t)o32[j] << 32) | (uint64_t)(~(uint32_t)(lane * EPL + j))
                      : 0ull;
#pragma unroll
      for (int ps = 0; ps < EPL; ++ps)
#pragma unroll
        for (int i = ps & 1; i + 1 < EPL; i += 2)
          if (cand[i] < cand[i + 1]) { const uint64_t t = cand[i]; cand[i] = cand[i + 1]; cand[i + 1] = t; }
      float prev = 0.f;
      for (int q = 0; q <= K; ++q) {
        const bool has = cand[0] != 0ull;
        uint32_t wk;
        const int be = warp_argmax_redux((uint32_t)(cand[0] >> 32), has, (int)(~(uint32_t)cand[0]), wk);
        if (be == 0x7fffffff) break;  // fewer than K+1 eligible experts: no further margin
        const float kv = unord32(wk);
        if (q > 0 && !(prev - kv > 2.0f * kDelta)) safe = false;
        prev = kv;
        if (has && (int)(~(uint32_t)cand[0]) == be) {
#pragma unroll
          for (int j = 0; j + 1 < EPL; ++j) cand[j] = cand[j + 1];
          cand[EPL - 1] = 0ull;
        }
        if (q < K && lane == q) sel_e = be;
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
          const bool elig = valid[j] && !taken[j] && ((chosen >> grp[j]) & 1u);
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
      const float s = (lane < K) ? 1.0f / (1.0f + expf(-l_sel)) : 0.0f;
      float z = s;
#pragma unroll
      for (int d = 16; d; d >>= 1) z += __shfl_xor_sync(0xffffffffu, z, d);
      g = s / z;
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
      pv[j] = !valid[j] ? 0.f : (SIGMOID ? sgm[j] : expf(lv[j] - m));
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

// ============================================================================ thread per unit, registers
// Softmax scoring without a group limit, E <= EMAX <= 64: the unit's fp32 logits (bias included) are
// in registers l[0..E). Top-K by K rounds of a pairwise tree argmax over (key desc, index asc) — at
// every level the left operand holds the lower indices, so an equal key keeps the lower index —
// with the experts already taken masked out. Gates: softmax over the picked logits (the root of each
// round carries its logit). p[e]: the unit's probabilities over all E experts (zero past E).
template <int EMAX, int KMAX>
__device__ __forceinline__ void route_unit_regs(const float (&l)[EMAX], int E, int K, int (&pk)[KMAX],
                                                float (&gv)[KMAX], float (&p)[EMAX]) {
  uint64_t taken = 0;
#pragma unroll
  for (int k = 0; k < KMAX; ++k) {
    pk[k] = -1;
    gv[k] = 0.f;
    if (k >= K) continue;
    float bv[EMAX];
    int bi[EMAX];
#pragma unroll
    for (int e = 0; e < EMAX; ++e) {
      const bool ok = e < E && !((taken >> e) & 1ull);
      bv[e] = ok ? l[e] : -INFINITY;
      bi[e] = ok ? e : 0x7fffffff;
    }
#pragma unroll
    for (int w = 1; w < EMAX; w <<= 1)
#pragma unroll
      for (int e = 0; e < EMAX; e += 2 * w) {
        // take the right operand only if it is valid and strictly better (or the left is invalid)
        const bool right = bi[e + w] != 0x7fffffff && (bi[e] == 0x7fffffff || bv[e + w] > bv[e]);
        if (right) { bv[e] = bv[e + w]; bi[e] = bi[e + w]; }
      }
    pk[k] = bi[0];
    gv[k] = bv[0];
    taken |= 1ull << bi[0];
  }
  // gates: softmax over the picked logits (pick 0 holds the largest)
  const float top = gv[0];
  float z = 0.f;
#pragma unroll
  for (int k = 0; k < KMAX; ++k)
    if (k < K) { gv[k] = expf(gv[k] - top); z += gv[k]; }
#pragma unroll
  for (int k = 0; k < KMAX; ++k)
    if (k < K) gv[k] = gv[k] / z;
  // probabilities over all experts
  float m = -INFINITY;
#pragma unroll
  for (int e = 0; e < EMAX; ++e)
    if (e < E) m = fmaxf(m, l[e]);
  float zs = 0.f;
#pragma unroll
  for (int e = 0; e < EMAX; ++e) {
    p[e] = e < E ? __expf(l[e] - m) : 0.f;
    zs += p[e];
  }
  const float iz = 1.f / zs;
#pragma unroll
  for (int e = 0; e < EMAX; ++e) p[e] *= iz;
}

// Sum of v[e] over the 32 lanes of the warp for every e < EMAX, by a butterfly reduce-scatter (fp32
// addition is commutative, so each result is one fixed function of the inputs). On return lane L
// holds, in v[0..max(1, EMAX/32)), the sums of experts [L·EMAX/32, (L+1)·EMAX/32) when EMAX >= 32,
// or, when EMAX < 32, the sum of expert L / (32/EMAX) (every lane of a group of 32/EMAX lanes holds
// it).
template <int LEN>
__device__ __forceinline__ void rs_step(float* v, int lane, int o) {
  const bool upper = (lane & o) != 0;
#pragma unroll
  for (int j = 0; j < LEN / 2; ++j) {
    const float send = upper ? v[j] : v[j + LEN / 2];
    const float keep = upper ? v[j + LEN / 2] : v[j];
    v[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
  }
}

template <int EMAX>
__device__ __forceinline__ void warp_reduce_scatter(float (&v)[EMAX], int lane) {
  static_assert(EMAX == 8 || EMAX == 16 || EMAX == 32 || EMAX == 64, "EMAX");
  // step i halves the live length (EMAX >> i) across lane offset 16 >> i
  rs_step<EMAX>(v, lane, 16);
  rs_step<EMAX / 2>(v, lane, 8);
  rs_step<EMAX / 4>(v, lane, 4);
  if constexpr (EMAX >= 16) rs_step<EMAX / 8>(v, lane, 2);
  if constexpr (EMAX >= 32) rs_step<EMAX / 16>(v, lane, 1);
  // below 32 experts, the lanes that hold the same expert (offsets under 32/EMAX) add their values
  if constexpr (EMAX < 32) {
#pragma unroll
    for (int o = (32 / EMAX) >> 1; o; o >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
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
// ceil(R/32) · E entries each (R <= blockDim). Ends with a block barrier.
__device__ __forceinline__ void rank_picks(const int* picks, int R, int K, int E, int* rank, int* hist,
                                           uint32_t* lanes_of, int* warp_pre) {
  constexpr int kstride = kPickStride;
  // only the warps that hold rows take part: ceil(R/32) of them
  const int t = threadIdx.x, nt = blockDim.x, nw = (R + 31) >> 5, w = t >> 5, lane = t & 31;
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
