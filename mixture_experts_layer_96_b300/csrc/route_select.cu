// Routing from fp32 logits: scores, optional group limit, Top-K, gates and the per-block
// statistics of the aux loss.
//   [Lesson 10 "专家并行 EP", §1: s(x) = Softmax(TopK(x·W_g, K)) or sigmoid normalisation;
//    §4: L_aux = α·E·Σ f_i·P_i; §5: a unit's experts restricted to a few groups]
//
// Input: the logits as `nparts` fp32 partial sums [part][T'][E] (K slices of the router GEMM, or
// one array of given logits); they are added in part order, then the logit bias (fp32).
// Selection keys: softmax → the fp32 logit itself (TopK acts on x·W_g); sigmoid → σ(l) + b
// formed in fp64. Ties go to the lower expert index (and lower group index). Gates: softmax
// over the K picked logits, or σ_i/Σσ over the picks (unbiased).
//
// Two shapes of kernel:
//   E <= 64: one thread per unit. A block stages its units' logits in shared memory; each
//            thread scans its row in expert order keeping a sorted list of its K best
//            (key, index) (an equal key never displaces a lower index), then overwrites its row
//            with its probabilities, and the block sums each column in row order.
//   E > 64:  one warp per unit, each lane E/32 experts; keys are compared as order-preserving
//            64-bit integers so shuffles and comparisons stay off the fp64 pipe.
// Both write per-block Σ_t P_{t,i} and pick counts; the aux kernel (route.cu) reduces them.
#include <math.h>

#include <type_traits>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {

constexpr int kSelThreads = 256;
constexpr int kSelWarpUnits = 8;  // units per block in the warp-per-unit kernel (one per warp)

struct SelectArgs {
  const float* logits;      // [nparts][Tu][E]
  int64_t part_stride;
  int nparts;
  const float* logit_bias;  // [E] or null
  const float* select_bias; // [E] or null (sigmoid only)
  int32_t* idx;             // [Tu][K]
  float* gate;              // [Tu][K]
  float* logits_out;        // [Tu][E] or null
  float* psum_part;         // [blocks][E]
  int32_t* cnt_part;        // [blocks][E]
  int64_t Tu;
  int E, K, n_groups, topk_groups;
};

__device__ __forceinline__ float load_logit(const SelectArgs& a, int64_t u, int e) {
  const int64_t o = u * a.E + e;
  float v = a.logits[o];
  for (int q = 1; q < a.nparts; ++q) v += a.logits[q * a.part_stride + o];
  if (a.logit_bias) v = v + a.logit_bias[e];
  return v;
}

__device__ __forceinline__ double sigmoid64(float l) { return 1.0 / (1.0 + exp(-(double)l)); }

// Order-preserving map of a double to uint64 (−0 is folded into +0 first).
__device__ __forceinline__ uint64_t ord64(double d) {
  d = d + 0.0;
  const uint64_t u = (uint64_t)__double_as_longlong(d);
  return (u >> 63) ? ~u : (u | 0x8000000000000000ull);
}

// Stage the logits of units [u0, u0+rows) into tile[r*LD + e] (partials added in order, then the
// logit bias), and copy them to logits_out if asked. Rows are loaded as float4 with several loads
// in flight per thread when E is a multiple of 4; otherwise one float at a time.
template <int NT, int LD>
__device__ __forceinline__ void stage_logits(const SelectArgs& a, int64_t u0, float* tile) {
  const int E = a.E, tid = threadIdx.x;
  const int64_t rows = (a.Tu - u0) < NT ? (a.Tu - u0) : NT;
  if ((E & 3) == 0) {
    const int per_row = E >> 2;
    const int n4 = (int)rows * per_row;
    constexpr int U = 8;
    for (int base = tid; base < n4; base += NT * U) {
      float4 v[U];
#pragma unroll
      for (int j = 0; j < U; ++j) {
        const int i = base + j * NT;
        v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (i < n4) v[j] = __ldg(reinterpret_cast<const float4*>(a.logits + u0 * E) + i);
      }
      for (int q = 1; q < a.nparts; ++q) {
#pragma unroll
        for (int j = 0; j < U; ++j) {
          const int i = base + j * NT;
          if (i < n4) {
            const float4 w = __ldg(reinterpret_cast<const float4*>(a.logits + q * a.part_stride + u0 * E) + i);
            v[j].x += w.x; v[j].y += w.y; v[j].z += w.z; v[j].w += w.w;
          }
        }
      }
#pragma unroll
      for (int j = 0; j < U; ++j) {
        const int i = base + j * NT;
        if (i >= n4) break;
        const int r = i / per_row, e = (i - r * per_row) * 4;
        float4 w = v[j];
        if (a.logit_bias) {
          w.x = w.x + a.logit_bias[e]; w.y = w.y + a.logit_bias[e + 1];
          w.z = w.z + a.logit_bias[e + 2]; w.w = w.w + a.logit_bias[e + 3];
        }
        tile[r * LD + e] = w.x; tile[r * LD + e + 1] = w.y; tile[r * LD + e + 2] = w.z; tile[r * LD + e + 3] = w.w;
        if (a.logits_out) reinterpret_cast<float4*>(a.logits_out + u0 * E)[i] = w;
      }
    }
  } else {
    for (int i = tid; i < rows * E; i += NT) {
      const int r = i / E, e = i % E;
      const float v = load_logit(a, u0 + r, e);
      tile[r * LD + e] = v;
      if (a.logits_out) a.logits_out[(u0 + r) * E + e] = v;
    }
  }
}

// Order-preserving map of a float to uint32 (−0 folded into +0).
__device__ __forceinline__ uint32_t ord32(float f) {
  f = f + 0.0f;
  const uint32_t u = __float_as_uint(f);
  return (u >> 31) ? ~u : (u | 0x80000000u);
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

__device__ __forceinline__ float unord32(uint32_t u) {
  return __uint_as_float((u >> 31) ? (u & 0x7fffffffu) : ~u);
}

// ============================================================================ thread per unit
// units (= threads) per block of the thread-per-unit kernel: the logit tile stays under 48 KB
template <int EMAX>
struct SelThreadCfg {
  static constexpr int T = EMAX <= 32 ? 256 : 128;
};

// Key of expert e of this thread's unit (the row `row` of the shared tile).
template <bool SIGMOID>
__device__ __forceinline__ typename std::conditional<SIGMOID, double, float>::type
sel_key(const SelectArgs& a, const float* row, int e) {
  if constexpr (SIGMOID) return sigmoid64(row[e]) + (a.select_bias ? (double)a.select_bias[e] : 0.0);
  else return row[e];
}

template <int EMAX, int KMAX, bool SIGMOID>
__global__ void __launch_bounds__(SelThreadCfg<EMAX>::T)
select_thread_kernel(SelectArgs a) {
  using KeyT = typename std::conditional<SIGMOID, double, float>::type;
  constexpr int kSelThreads = SelThreadCfg<EMAX>::T;
  constexpr int LD = EMAX + 1;
  __shared__ float tile[kSelThreads * LD];
  __shared__ int cnt_s[EMAX];
  const int tid = threadIdx.x;
  const int64_t u0 = (int64_t)blockIdx.x * kSelThreads;
  const int E = a.E, K = a.K;
  for (int e = tid; e < EMAX; e += kSelThreads) cnt_s[e] = 0;
  stage_logits<kSelThreads, LD>(a, u0, tile);
  __syncthreads();

  const int64_t u = u0 + tid;
  const bool valid = u < a.Tu;
  float* row = tile + tid * LD;

  // group limit: keep the topk_groups groups with the largest sum of their two best keys
  uint64_t eligible = ~0ull;
  if (a.n_groups > 1) {
    const int gs = E / a.n_groups;
    uint32_t chosen = 0;
    for (int q = 0; q < a.topk_groups; ++q) {
      int bg = -1;
      double bsc = 0.0;
      for (int g = 0; g < a.n_groups; ++g) {
        if ((chosen >> g) & 1u) continue;
        double t1 = -INFINITY, t2 = -INFINITY;
        for (int i = 0; i < gs; ++i) {
          const double k = (double)sel_key<SIGMOID>(a, row, g * gs + i);
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

  // Top-K: scan experts in index order keeping bk[0..K) sorted by key, descending. A new key is
  // placed below every kept key that is >= it (an equal key never displaces an earlier, lower
  // index), the entries it passes shift down one slot. Slots are filled in order; be = -1 marks
  // an empty slot.
  KeyT bk[KMAX];
  int be[KMAX];
#pragma unroll
  for (int j = 0; j < KMAX; ++j) { bk[j] = (KeyT)-INFINITY; be[j] = -1; }
  for (int e = 0; e < E; ++e) {
    if (!((eligible >> e) & 1ull)) continue;
    const KeyT ck = sel_key<SIGMOID>(a, row, e);
#pragma unroll
    for (int t = KMAX - 1; t >= 0; --t) {
      if (t < K) {
        const bool above = t > 0 && (be[t - 1] < 0 || ck > bk[t - 1]);
        const bool here = be[t] < 0 || ck > bk[t];
        if (above) { bk[t] = bk[t - 1]; be[t] = be[t - 1]; }
        else if (here) { bk[t] = ck; be[t] = e; }
      }
    }
  }

  // gates and picks
  if (valid) {
    float lv[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) lv[j] = (j < K && be[j] >= 0) ? row[be[j]] : 0.f;
    if (SIGMOID) {
      double sg[KMAX], z = 0.0;
#pragma unroll
      for (int j = 0; j < KMAX; ++j) { sg[j] = (j < K) ? sigmoid64(lv[j]) : 0.0; z += sg[j]; }
#pragma unroll
      for (int j = 0; j < KMAX; ++j)
        if (j < K) { a.idx[u * K + j] = be[j]; a.gate[u * K + j] = (float)(sg[j] / z); }
    } else {
      float ev[KMAX], z = 0.f;
#pragma unroll
      for (int j = 0; j < KMAX; ++j) { ev[j] = (j < K) ? expf(lv[j] - lv[0]) : 0.f; z += ev[j]; }
#pragma unroll
      for (int j = 0; j < KMAX; ++j)
        if (j < K) { a.idx[u * K + j] = be[j]; a.gate[u * K + j] = ev[j] / z; }
    }
#pragma unroll
    for (int j = 0; j < KMAX; ++j)
      if (j < K && be[j] >= 0) atomicAdd(&cnt_s[be[j]], 1);
  }

  // this unit's probabilities replace its logits in the tile; columns are then summed in row order
  {
    float m = -INFINITY, z = 0.f;
    if (!SIGMOID)
      for (int e = 0; e < E; ++e) m = fmaxf(m, row[e]);
    for (int e = 0; e < E; ++e) {
      const float v = SIGMOID ? (float)sigmoid64(row[e]) : __expf(row[e] - m);
      z += v;
      row[e] = v;
    }
    const float iz = valid ? 1.f / z : 0.f;
    for (int e = 0; e < E; ++e) row[e] = valid ? row[e] * iz : 0.f;
  }
  __syncthreads();
  // column sums: P threads per column, each over a contiguous block of rows, then the P partial
  // sums of a column in order (fixed order, so deterministic)
  __shared__ float colpart[kSelThreads];
  {
    const int P = kSelThreads / E;  // >= 2 for E <= 64
    const int e = tid / P, part = tid % P;
    const int rows_per = (kSelThreads + P - 1) / P;
    float s = 0.f;
    if (e < E) {
      const int r0 = part * rows_per, r1 = min(kSelThreads, r0 + rows_per);
      for (int r = r0; r < r1; ++r) s += tile[r * LD + e];
    }
    colpart[tid] = s;
    __syncthreads();
    if (tid < E) {
      float t = 0.f;
      for (int q = 0; q < P; ++q) t += colpart[tid * P + q];
      a.psum_part[(int64_t)blockIdx.x * E + tid] = t;
      a.cnt_part[(int64_t)blockIdx.x * E + tid] = cnt_s[tid];
    }
  }
}

// ============================================================================ warp per unit
template <int EPL, bool SIGMOID>
__global__ void __launch_bounds__(kSelThreads)
select_warp_kernel(SelectArgs a) {
  constexpr int EP = 32 * EPL;
  __shared__ float psum_w[kSelThreads / 32][EP];
  __shared__ int cnt_s[EP];
  __shared__ uint64_t kord_w[kSelThreads / 32][EP];   // ordered keys (group scores)
  __shared__ double kdbl_w[kSelThreads / 32][EP];     // keys (group sums)
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = a.E, K = a.K;
  for (int i = tid; i < (kSelThreads / 32) * EP; i += kSelThreads) (&psum_w[0][0])[i] = 0.f;
  for (int e = tid; e < EP; e += kSelThreads) cnt_s[e] = 0;
  __syncthreads();
  const int gs = E / a.n_groups;
  for (int r = warp; r < kSelWarpUnits; r += kSelThreads / 32) {
    const int64_t u = (int64_t)blockIdx.x * kSelWarpUnits + r;
    if (u >= a.Tu) break;
    float lv[EPL];
    uint64_t ko[EPL];
    double kd[EPL];
    bool valid[EPL];
    if ((E & 3) == 0 && (EPL & 3) == 0 && lane * EPL + EPL <= E) {
      // a lane's EPL experts are contiguous: float4 loads, every part's loads issued together
      const float4* src = reinterpret_cast<const float4*>(a.logits + u * E + lane * EPL);
      float4 v[EPL / 4];
#pragma unroll
      for (int j = 0; j < EPL / 4; ++j) v[j] = __ldg(src + j);
      for (int q = 1; q < a.nparts; ++q) {
        float4 w[EPL / 4];
#pragma unroll
        for (int j = 0; j < EPL / 4; ++j) w[j] = __ldg(src + (q * a.part_stride) / 4 + j);
#pragma unroll
        for (int j = 0; j < EPL / 4; ++j) { v[j].x += w[j].x; v[j].y += w[j].y; v[j].z += w[j].z; v[j].w += w[j].w; }
      }
#pragma unroll
      for (int j = 0; j < EPL / 4; ++j) {
        lv[4 * j] = v[j].x; lv[4 * j + 1] = v[j].y; lv[4 * j + 2] = v[j].z; lv[4 * j + 3] = v[j].w;
      }
#pragma unroll
      for (int j = 0; j < EPL; ++j) {
        const int e = lane * EPL + j;
        valid[j] = true;
        if (a.logit_bias) lv[j] = lv[j] + a.logit_bias[e];
        if (a.logits_out) a.logits_out[u * E + e] = lv[j];
      }
    } else {
#pragma unroll
      for (int j = 0; j < EPL; ++j) {
        const int e = lane * EPL + j;
        valid[j] = e < E;
        lv[j] = valid[j] ? load_logit(a, u, e) : -INFINITY;
        if (valid[j] && a.logits_out) a.logits_out[u * E + e] = lv[j];
      }
    }
    // Sigmoid keys σ(l)+b are decided in fp64. First screen in fp32: |key32 − key64| <= 4.3e-7
    // (accurate expf, IEEE divide, one rounding of the add), so when every decision's fp32 margin
    // exceeds twice the error bound (group scores: two keys and a rounded add each) the fp32
    // decisions equal the fp64 ones; otherwise this unit takes the fp64 path below.
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
        k32[j] = valid[j] ? (1.0f / (1.0f + expf(-lv[j]))) + (a.select_bias ? a.select_bias[e] : 0.0f) : -INFINITY;
        o32[j] = ord32(k32[j]);
      }
      bool safe = true;
      if (a.n_groups > 1) {
        float* gk = reinterpret_cast<float*>(&kdbl_w[warp][0]);
#pragma unroll
        for (int j = 0; j < EPL; ++j) gk[lane * EPL + j] = k32[j];
        __syncwarp();
        uint32_t gord = 0;
        int gidx = 0x7fffffff;
        if (lane < a.n_groups) {
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
        for (int q = 0; q <= a.topk_groups && q < a.n_groups; ++q) {
          const bool cand = gidx != 0x7fffffff && !((chosen >> lane) & 1u);
          uint32_t bk;
          const int bg = warp_argmax32(cand ? gord : 0u, cand ? gidx : 0x7fffffff, bk);
          const float sc = unord32(bk);
          if (q < a.topk_groups) {
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
      for (int q = 0; q <= a.K; ++q) {
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
        if (q < a.K) {
#pragma unroll
          for (int j = 0; j < EPL; ++j)
            if (be == lane * EPL + j) taken[j] = true;
          if (lane == q) sel_e = be;
        }
      }
      screened = safe;
    }
    if (!screened) {
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
      const int e = lane * EPL + j;
      kd[j] = SIGMOID ? (valid[j] ? sigmoid64(lv[j]) + (a.select_bias ? (double)a.select_bias[e] : 0.0) : -INFINITY)
                      : (double)lv[j];
      ko[j] = ord64(kd[j]);
    }
    }
    // P_i for the aux loss
    {
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
#pragma unroll
      for (int j = 0; j < EPL; ++j)
        if (valid[j]) psum_w[warp][lane * EPL + j] += pv[j] / z;
    }
    // fp64 decision (all softmax units; sigmoid units whose fp32 screen was not conclusive)
    if (!screened) {
    // group limit
    chosen = 0xffffffffu;
    if (a.n_groups > 1) {
#pragma unroll
      for (int j = 0; j < EPL; ++j) {
        kord_w[warp][lane * EPL + j] = ko[j];
        kdbl_w[warp][lane * EPL + j] = kd[j];
      }
      __syncwarp();
      uint64_t gord = 0;
      bool gval = false;
      if (lane < a.n_groups) {
        int i1 = -1, i2 = -1;
        uint64_t t1 = 0, t2 = 0;
        for (int i = 0; i < gs; ++i) {
          const uint64_t v = kord_w[warp][lane * gs + i];
          if (i1 < 0 || v > t1) { t2 = t1; i2 = i1; t1 = v; i1 = i; }
          else if (i2 < 0 || v > t2) { t2 = v; i2 = i; }
        }
        const double sc = kdbl_w[warp][lane * gs + i1] + (i2 >= 0 ? kdbl_w[warp][lane * gs + i2] : 0.0);
        gord = ord64(sc);
        gval = true;
      }
      __syncwarp();
      chosen = 0;
      for (int q = 0; q < a.topk_groups; ++q) {
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
    }  // fp64 decision
    for (int q = 0; q < K; ++q) {
      const int eq = __shfl_sync(0xffffffffu, sel_e, q);
      if (lane == 0 && eq >= 0) atomicAdd(&cnt_s[eq], 1);
    }
    // gates from the picked logits
    float l_sel = (lane < K && sel_e >= 0) ? load_logit(a, u, sel_e) : 0.f;
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
      a.idx[u * K + lane] = sel_e;
      a.gate[u * K + lane] = g;
    }
  }
  __syncthreads();
  for (int e = tid; e < E; e += kSelThreads) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kSelThreads / 32; ++w) s += psum_w[w][e];
    a.psum_part[(int64_t)blockIdx.x * E + e] = s;
    a.cnt_part[(int64_t)blockIdx.x * E + e] = cnt_s[e];
  }
}

int select_block_units(int E) {
  return E <= 32 ? SelThreadCfg<32>::T : (E <= 64 ? SelThreadCfg<64>::T : kSelWarpUnits);
}

template <int EMAX, int KMAX>
static void launch_thread_sel_k(const SelectArgs& a, int64_t blocks, bool sigmoid, cudaStream_t s) {
  constexpr int T = SelThreadCfg<EMAX>::T;
  if (sigmoid) select_thread_kernel<EMAX, KMAX, true><<<(unsigned)blocks, T, 0, s>>>(a);
  else select_thread_kernel<EMAX, KMAX, false><<<(unsigned)blocks, T, 0, s>>>(a);
}

template <int EMAX>
static void launch_thread_sel(const SelectArgs& a, int64_t blocks, bool sigmoid, cudaStream_t s) {
  if (a.K <= 2) launch_thread_sel_k<EMAX, 2>(a, blocks, sigmoid, s);
  else if (a.K <= 4) launch_thread_sel_k<EMAX, 4>(a, blocks, sigmoid, s);
  else launch_thread_sel_k<EMAX, 8>(a, blocks, sigmoid, s);
}

template <int EPL>
static void launch_warp_sel(const SelectArgs& a, int64_t blocks, bool sigmoid, cudaStream_t s) {
  if (sigmoid) select_warp_kernel<EPL, true><<<(unsigned)blocks, kSelThreads, 0, s>>>(a);
  else select_warp_kernel<EPL, false><<<(unsigned)blocks, kSelThreads, 0, s>>>(a);
}

cudaError_t launch_select(const Problem& p, const float* logits, int nparts, int64_t part_stride,
                          const float* logit_bias, const float* select_bias, int32_t* idx, float* gate,
                          float* logits_out, float* psum_part, int32_t* cnt_part, cudaStream_t s) {
  if (p.Tu == 0) return cudaSuccess;
  SelectArgs a;
  a.logits = logits;
  a.part_stride = part_stride;
  a.nparts = nparts;
  a.logit_bias = logit_bias;
  a.select_bias = p.sigmoid ? select_bias : nullptr;
  a.idx = idx;
  a.gate = gate;
  a.logits_out = logits_out;
  a.psum_part = psum_part;
  a.cnt_part = cnt_part;
  a.Tu = p.Tu;
  a.E = p.E;
  a.K = p.K;
  a.n_groups = p.n_groups;
  a.topk_groups = p.topk_groups;
  const int64_t blocks = p.route_blocks;
  if (p.E <= 8) launch_thread_sel<8>(a, blocks, p.sigmoid, s);
  else if (p.E <= 16) launch_thread_sel<16>(a, blocks, p.sigmoid, s);
  else if (p.E <= 32) launch_thread_sel<32>(a, blocks, p.sigmoid, s);
  else if (p.E <= 64) launch_thread_sel<64>(a, blocks, p.sigmoid, s);
  else if (p.E <= 128) launch_warp_sel<4>(a, blocks, p.sigmoid, s);
  else launch_warp_sel<8>(a, blocks, p.sigmoid, s);
  note_launch();
  return cudaGetLastError();
}

}  // namespace moe
