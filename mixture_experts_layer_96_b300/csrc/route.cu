// Router: logits l = x·W_g (+ logit bias), scoring, optional group limit, Top-K, gates and the
// per-block statistics of the aux loss, fused in one kernel per block of units.
//   [Lesson 10 "专家并行 EP", §1: s(x) = Softmax(TopK(x·W_g, K)) or sigmoid; §4: L_aux; §5: the
//    experts of a unit restricted to M groups]
//
// Block = 256 threads, BT units. Phase 1 computes the [BT][EP] logit tile (EP = E rounded up to
// a power of two >= 8) with fp32 FMAs; for small E the block splits the reduction dimension
// over warp groups. Phase 2 gives each warp whole units: each lane holds EP/32 experts (at least
// one), keys are formed in fp64 (the decision precision of the selection), Top-K is K rounds of a
// warp argmax on (key desc, index asc), and gates/statistics follow.
#include <math.h>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {

constexpr int kRouteThreads = 256;
constexpr int kRouteBK = 32;

template <int EP>
struct RouteTile {
  static constexpr int TN = 8;                                   // experts per thread
  static constexpr int BT = (EP <= 32) ? 32 : (EP == 64 ? 64 : 32);
  static constexpr int TM = (EP <= 32) ? 1 : (EP == 64 ? 2 : (EP == 128 ? 2 : 4));
  static constexpr int GT = BT * EP / (TM * TN);                  // threads per K-slice group
  static constexpr int KSPLIT = kRouteThreads / GT;
  static constexpr int ECOLS = EP / TN;
  static constexpr int TROWS = GT / ECOLS;
  static constexpr int KW = kRouteBK * KSPLIT;                   // columns staged per step
  static constexpr int XS = BT * (KW + 1);                       // floats
  static constexpr int WS = KW * EP;
  static constexpr int RED = (KSPLIT > 1) ? KSPLIT * BT * EP : 0;
  static constexpr int LS = BT * (EP + 1);
  static constexpr int GEMM_FLOATS = XS + WS + RED;
  static constexpr int MAIN_FLOATS = GEMM_FLOATS > LS ? GEMM_FLOATS : LS;
  static constexpr int EPL = EP >= 32 ? EP / 32 : 1;             // experts per lane (selection)
  static_assert(TROWS * TM == BT, "tile");
  static_assert(GT * KSPLIT == kRouteThreads, "split");
  // dynamic smem: [main | psum_w 8xEP f32 | cnt EP i32 | keys 8xEP f64]
  static constexpr size_t SMEM = (size_t)MAIN_FLOATS * 4 + 8 * EP * 4 + EP * 4 + 8 * EP * 8;
};

struct RouteArgs {
  const void* x;            // [Tu][hu] (TIn)
  const void* w;            // [hu][E] (TIn)
  const float* logits_in;   // [nparts][Tu][E] (summed in order) or null
  int64_t part_stride;      // elements between parts
  int nparts;
  const float* logit_bias;  // [E] or null
  const float* select_bias; // [E] or null
  int32_t* idx;             // [Tu][K]
  float* gate;              // [Tu][K]
  float* logits_out;        // [Tu][E] or null
  float* psum_part;         // [blocks][E]
  int32_t* cnt_part;        // [blocks][E]
  int64_t Tu;
  int hu, E, K, n_groups, topk_groups;
  int sigmoid;
};

// (key, index) order of the selection: larger key first, then lower index.
__device__ __forceinline__ bool better(double ka, int ea, double kb, int eb) {
  return ka > kb || (ka == kb && ea < eb);
}

template <typename TIn, int EP, bool FROM_LOGITS>
__global__ void __launch_bounds__(kRouteThreads)
route_kernel(RouteArgs a) {
  using Tl = RouteTile<EP>;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  float* main_f = reinterpret_cast<float*>(smem_raw);
  float* psum_w = main_f + Tl::MAIN_FLOATS;          // [8][EP]
  int* cnt_s = reinterpret_cast<int*>(psum_w + 8 * EP);
  double* keys_w = reinterpret_cast<double*>(cnt_s + EP);  // [8][EP] (8-byte aligned: offsets are multiples of 8 floats)

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int64_t u0 = (int64_t)blockIdx.x * Tl::BT;
  const int E = a.E;
  float* ls = main_f;  // [BT][EP+1] logits tile (aliases the GEMM staging after phase 1)

  for (int i = tid; i < 8 * EP; i += kRouteThreads) psum_w[i] = 0.f;
  for (int i = tid; i < EP; i += kRouteThreads) cnt_s[i] = 0;

  // ------------------------------------------------------------------ phase 1: logit tile
  if constexpr (FROM_LOGITS) {
    for (int i = tid; i < Tl::BT * EP; i += kRouteThreads) {
      const int r = i / EP, e = i % EP;
      const int64_t u = u0 + r;
      float v = 0.f;
      if (u < a.Tu && e < E) {
        v = a.logits_in[u * E + e];
        for (int q = 1; q < a.nparts; ++q) v += a.logits_in[q * a.part_stride + u * E + e];
        if (a.logit_bias) v = v + a.logit_bias[e];
      }
      ls[r * (EP + 1) + e] = v;
    }
  } else {
    float* xs = main_f;                 // [BT][KW+1]
    float* wsm = main_f + Tl::XS;       // [KW][EP]
    float* red = wsm + Tl::WS;          // [KSPLIT][BT][EP]
    const TIn* __restrict__ X = static_cast<const TIn*>(a.x);
    const TIn* __restrict__ W = static_cast<const TIn*>(a.w);
    const int g = tid / Tl::GT, lt = tid % Tl::GT;
    const int tr = lt / Tl::ECOLS, tc = lt % Tl::ECOLS;
    float acc[Tl::TM][Tl::TN];
#pragma unroll
    for (int i = 0; i < Tl::TM; ++i)
#pragma unroll
      for (int j = 0; j < Tl::TN; ++j) acc[i][j] = 0.f;

    constexpr int VEC = 16 / sizeof(TIn);
    const bool vec_ok = ((a.hu * (int)sizeof(TIn)) % 16 == 0) &&
                        ((reinterpret_cast<uintptr_t>(a.x) & 15) == 0);
    for (int k0 = 0; k0 < a.hu; k0 += Tl::KW) {
      __syncthreads();
      // x tile
      if (vec_ok) {
        constexpr int VPR = Tl::KW / VEC;  // vectors per row
        for (int i = tid; i < Tl::BT * VPR; i += kRouteThreads) {
          const int r = i / VPR, c = (i % VPR) * VEC;
          const int64_t u = u0 + r;
          float v[VEC];
          if (u < a.Tu && k0 + c < a.hu) {
            const uint4 q = __ldg(reinterpret_cast<const uint4*>(X + u * a.hu + k0 + c));
            const TIn* pv = reinterpret_cast<const TIn*>(&q);
#pragma unroll
            for (int j = 0; j < VEC; ++j) v[j] = to_f32<TIn>(pv[j]);
          } else {
#pragma unroll
            for (int j = 0; j < VEC; ++j) v[j] = 0.f;
          }
#pragma unroll
          for (int j = 0; j < VEC; ++j) xs[r * (Tl::KW + 1) + c + j] = v[j];
        }
      } else {
        for (int i = tid; i < Tl::BT * Tl::KW; i += kRouteThreads) {
          const int r = i / Tl::KW, c = i % Tl::KW;
          const int64_t u = u0 + r;
          xs[r * (Tl::KW + 1) + c] =
              (u < a.Tu && k0 + c < a.hu) ? to_f32<TIn>(X[u * a.hu + k0 + c]) : 0.f;
        }
      }
      // W_g tile
      for (int i = tid; i < Tl::KW * EP; i += kRouteThreads) {
        const int k = i / EP, e = i % EP;
        wsm[i] = (k0 + k < a.hu && e < E) ? to_f32<TIn>(W[(int64_t)(k0 + k) * E + e]) : 0.f;
      }
      __syncthreads();
      const float* xg = xs + g * kRouteBK;
      const float* wg = wsm + g * kRouteBK * EP;
#pragma unroll 4
      for (int kk = 0; kk < kRouteBK; ++kk) {
        float av[Tl::TM], bv[Tl::TN];
#pragma unroll
        for (int i = 0; i < Tl::TM; ++i) av[i] = xg[(tr + Tl::TROWS * i) * (Tl::KW + 1) + kk];
#pragma unroll
        for (int j = 0; j < Tl::TN; ++j) bv[j] = wg[kk * EP + tc + Tl::ECOLS * j];
#pragma unroll
        for (int i = 0; i < Tl::TM; ++i)
#pragma unroll
          for (int j = 0; j < Tl::TN; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
      }
    }
    __syncthreads();
    if constexpr (Tl::KSPLIT > 1) {
#pragma unroll
      for (int i = 0; i < Tl::TM; ++i)
#pragma unroll
        for (int j = 0; j < Tl::TN; ++j)
          red[(g * Tl::BT + tr + Tl::TROWS * i) * EP + tc + Tl::ECOLS * j] = acc[i][j];
      __syncthreads();
      // fixed-order sum over the K slices, then the logit bias, into the logit tile
      float tmp[(Tl::BT * EP + kRouteThreads - 1) / kRouteThreads];
      int n = 0;
      for (int i = tid; i < Tl::BT * EP; i += kRouteThreads, ++n) {
        float s = 0.f;
#pragma unroll
        for (int q = 0; q < Tl::KSPLIT; ++q) s += red[q * Tl::BT * EP + i];
        tmp[n] = s;
      }
      __syncthreads();
      n = 0;
      for (int i = tid; i < Tl::BT * EP; i += kRouteThreads, ++n) {
        const int r = i / EP, e = i % EP;
        float v = tmp[n];
        if (a.logit_bias && e < E) v = v + a.logit_bias[e];
        ls[r * (EP + 1) + e] = v;
      }
    } else {
#pragma unroll
      for (int i = 0; i < Tl::TM; ++i)
#pragma unroll
        for (int j = 0; j < Tl::TN; ++j) {
          const int e = tc + Tl::ECOLS * j;
          float v = acc[i][j];
          if (a.logit_bias && e < E) v = v + a.logit_bias[e];
          ls[(tr + Tl::TROWS * i) * (EP + 1) + e] = v;
        }
    }
  }
  __syncthreads();

  // ------------------------------------------------------------------ phase 2: selection
  constexpr int EPL = Tl::EPL;
  double* kw = keys_w + warp * EP;
  const int gs = E / a.n_groups;
  for (int r = warp; r < Tl::BT; r += 8) {
    const int64_t u = u0 + r;
    if (u >= a.Tu) break;
    float lv[EPL];
    double key[EPL], sg[EPL];
    bool valid[EPL], taken[EPL];
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
      const int e = lane * EPL + j;
      valid[j] = e < E;
      taken[j] = false;
      lv[j] = valid[j] ? ls[r * (EP + 1) + e] : -INFINITY;
      if (valid[j] && a.logits_out) a.logits_out[u * E + e] = lv[j];
      if (a.sigmoid) {
        sg[j] = valid[j] ? 1.0 / (1.0 + exp(-(double)lv[j])) : 0.0;
        key[j] = sg[j] + ((valid[j] && a.select_bias) ? (double)a.select_bias[e] : 0.0);
      } else {
        sg[j] = 0.0;
        key[j] = (double)lv[j];
      }
    }

    // aux statistics: this unit's probability of every expert [Lesson 10 §4: P_i]
    {
      float pv[EPL];
      if (a.sigmoid) {
        float z = 0.f;
#pragma unroll
        for (int j = 0; j < EPL; ++j) { pv[j] = valid[j] ? (float)sg[j] : 0.f; z += pv[j]; }
#pragma unroll
        for (int d = 16; d; d >>= 1) z += __shfl_xor_sync(0xffffffffu, z, d);
#pragma unroll
        for (int j = 0; j < EPL; ++j) pv[j] = pv[j] / z;
      } else {
        float m = -INFINITY;
#pragma unroll
        for (int j = 0; j < EPL; ++j) m = fmaxf(m, lv[j]);
#pragma unroll
        for (int d = 16; d; d >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d));
        float z = 0.f;
#pragma unroll
        for (int j = 0; j < EPL; ++j) { pv[j] = valid[j] ? expf(lv[j] - m) : 0.f; z += pv[j]; }
#pragma unroll
        for (int d = 16; d; d >>= 1) z += __shfl_xor_sync(0xffffffffu, z, d);
#pragma unroll
        for (int j = 0; j < EPL; ++j) pv[j] = pv[j] / z;
      }
#pragma unroll
      for (int j = 0; j < EPL; ++j)
        if (valid[j]) psum_w[warp * EP + lane * EPL + j] += pv[j];
    }

    // group limit [Lesson 10 §5]: keep the topk_groups groups with the largest top-2 key sums
    uint32_t chosen = 0xffffffffu;
    if (a.n_groups > 1) {
#pragma unroll
      for (int j = 0; j < EPL; ++j)
        if (valid[j]) kw[lane * EPL + j] = key[j];
      __syncwarp();
      double gscore = -INFINITY;
      if (lane < a.n_groups) {
        double t1 = -INFINITY, t2 = -INFINITY;
        for (int i = 0; i < gs; ++i) {
          const double v = kw[lane * gs + i];
          if (v > t1) { t2 = t1; t1 = v; }
          else if (v > t2) t2 = v;
        }
        gscore = (gs > 1) ? t1 + t2 : t1;
      }
      __syncwarp();
      chosen = 0;
      for (int q = 0; q < a.topk_groups; ++q) {
        const bool cand = lane < a.n_groups && !((chosen >> lane) & 1u);
        double bk = cand ? gscore : -INFINITY;
        int bg = cand ? lane : 0x7fffffff;
#pragma unroll
        for (int d = 16; d; d >>= 1) {
          const double ok = __shfl_xor_sync(0xffffffffu, bk, d);
          const int og = __shfl_xor_sync(0xffffffffu, bg, d);
          if (better(ok, og, bk, bg)) { bk = ok; bg = og; }
        }
        if (bg != 0x7fffffff) chosen |= 1u << bg;
      }
    }

    // Top-K [Lesson 10 §1]
    int sel_e = -1;
    float sel_l = 0.f;
    double sel_s = 0.0;
    for (int q = 0; q < a.K; ++q) {
      double bk = -INFINITY;
      int be = 0x7fffffff;
      float bl = 0.f;
      double bs = 0.0;
#pragma unroll
      for (int j = 0; j < EPL; ++j) {
        const int e = lane * EPL + j;
        const bool elig = valid[j] && !taken[j] && ((chosen >> (e / gs)) & 1u);
        if (elig && better(key[j], e, bk, be)) { bk = key[j]; be = e; bl = lv[j]; bs = sg[j]; }
      }
#pragma unroll
      for (int d = 16; d; d >>= 1) {
        const double ok = __shfl_xor_sync(0xffffffffu, bk, d);
        const int oe = __shfl_xor_sync(0xffffffffu, be, d);
        const float ol = __shfl_xor_sync(0xffffffffu, bl, d);
        const double os = __shfl_xor_sync(0xffffffffu, bs, d);
        if (better(ok, oe, bk, be)) { bk = ok; be = oe; bl = ol; bs = os; }
      }
#pragma unroll
      for (int j = 0; j < EPL; ++j)
        if (be == lane * EPL + j) taken[j] = true;
      if (lane == q) { sel_e = (be == 0x7fffffff) ? -1 : be; sel_l = bl; sel_s = bs; }
      if (lane == 0 && be != 0x7fffffff) atomicAdd(&cnt_s[be], 1);
    }

    // gates: softmax over the K picked logits, or σ/Σσ over the picks [Lesson 10 §1]
    const float l0 = __shfl_sync(0xffffffffu, sel_l, 0);
    float gnum;
    double snum = 0.0;
    if (a.sigmoid) {
      snum = (lane < a.K) ? sel_s : 0.0;
      double z = snum;
#pragma unroll
      for (int d = 16; d; d >>= 1) z += __shfl_xor_sync(0xffffffffu, z, d);
      gnum = (float)(snum / z);
    } else {
      float ev = (lane < a.K) ? expf(sel_l - l0) : 0.f;
      float z = ev;
#pragma unroll
      for (int d = 16; d; d >>= 1) z += __shfl_xor_sync(0xffffffffu, z, d);
      gnum = ev / z;
    }
    if (lane < a.K) {
      a.idx[u * a.K + lane] = sel_e;
      a.gate[u * a.K + lane] = gnum;
    }
  }
  __syncthreads();
  for (int e = tid; e < E; e += kRouteThreads) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) s += psum_w[w * EP + e];
    a.psum_part[(int64_t)blockIdx.x * E + e] = s;
    a.cnt_part[(int64_t)blockIdx.x * E + e] = cnt_s[e];
  }
}

// aux = α·E·Σ_i (count_i/(T'·K))·(ΣP_i/T')  [Lesson 10 §4]. One block per expert reduces that
// expert's per-block partials (fixed strided order, then a fixed tree, in fp64); the last block
// to finish (ticket counter) adds the E terms in expert order and resets the ticket.
__global__ void __launch_bounds__(256)
aux_finalize_kernel(const float* __restrict__ psum_part, const int32_t* __restrict__ cnt_part,
                    int64_t blocks, int E, int64_t Tu, int K, float alpha, double* terms,
                    unsigned int* ticket, float* aux_out) {
  __shared__ double sP[256];
  __shared__ long long sC[256];
  __shared__ bool last;
  const int tid = threadIdx.x, e = blockIdx.x;
  double P = 0.0;
  long long c = 0;
  for (int64_t b = tid; b < blocks; b += 256) {
    P += (double)psum_part[b * E + e];
    c += cnt_part[b * E + e];
  }
  sP[tid] = P;
  sC[tid] = c;
  __syncthreads();
  for (int s = 128; s; s >>= 1) {
    if (tid < s) {
      sP[tid] += sP[tid + s];
      sC[tid] += sC[tid + s];
    }
    __syncthreads();
  }
  if (tid == 0) {
    terms[e] = Tu > 0 ? ((double)sC[0] / ((double)Tu * K)) * (sP[0] / (double)Tu) : 0.0;
    __threadfence();
    last = atomicAdd(ticket, 1u) == (unsigned)(E - 1);
  }
  __syncthreads();
  if (last && tid == 0) {
    __threadfence();
    const volatile double* vt = terms;
    double acc = 0.0;
    for (int i = 0; i < E; ++i) acc += vt[i];
    *aux_out = (float)((double)alpha * E * acc);
    *ticket = 0u;
  }
}

template <typename TIn, int EP, bool FL>
static cudaError_t launch_route_t(const Problem& p, const RouteArgs& a, int64_t blocks, cudaStream_t s) {
  using Tl = RouteTile<EP>;
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(route_kernel<TIn, EP, FL>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Tl::SMEM);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  route_kernel<TIn, EP, FL><<<(unsigned)blocks, kRouteThreads, Tl::SMEM, s>>>(a);
  note_launch();
  return cudaGetLastError();
}

static int route_ep(int E) {
  int ep = 8;
  while (ep < E) ep <<= 1;
  return ep;
}

int route_block_units(int E) {
  switch (route_ep(E)) {
    case 8: return RouteTile<8>::BT;
    case 16: return RouteTile<16>::BT;
    case 32: return RouteTile<32>::BT;
    case 64: return RouteTile<64>::BT;
    case 128: return RouteTile<128>::BT;
    default: return RouteTile<256>::BT;
  }
}

template <typename TIn, bool FL>
static cudaError_t route_dispatch_ep(const Problem& p, const RouteArgs& a, int64_t blocks, cudaStream_t s) {
  switch (route_ep(p.E)) {
    case 8: return launch_route_t<TIn, 8, FL>(p, a, blocks, s);
    case 16: return launch_route_t<TIn, 16, FL>(p, a, blocks, s);
    case 32: return launch_route_t<TIn, 32, FL>(p, a, blocks, s);
    case 64: return launch_route_t<TIn, 64, FL>(p, a, blocks, s);
    case 128: return launch_route_t<TIn, 128, FL>(p, a, blocks, s);
    default: return launch_route_t<TIn, 256, FL>(p, a, blocks, s);
  }
}

cudaError_t launch_route(const Problem& p, const void* x, const void* w_router,
                         const float* logits_in, const float* logit_bias, const float* select_bias,
                         int32_t* idx, float* gate, float* logits_out, float* aux_out, void* ws,
                         cudaStream_t s) {
  const WsLayout L = ws_layout(p);
  RouteArgs a;
  a.x = x;
  a.w = w_router;
  a.logits_in = logits_in;
  a.logit_bias = logit_bias;
  a.select_bias = p.sigmoid ? select_bias : nullptr;
  a.idx = idx;
  a.gate = gate;
  a.logits_out = logits_out;
  a.psum_part = ws_ptr<float>(ws, L.psum_part);
  a.cnt_part = ws_ptr<int32_t>(ws, L.cnt_part);
  a.Tu = p.Tu;
  a.hu = p.hu;
  a.E = p.E;
  a.K = p.K;
  a.n_groups = p.n_groups;
  a.topk_groups = p.topk_groups;
  a.sigmoid = p.sigmoid ? 1 : 0;
  a.part_stride = 0;
  a.nparts = 1;
  const int64_t blocks = p.route_blocks;
  cudaError_t e = cudaSuccess;
  if (blocks > 0) {
    if (logits_in) {
      e = route_dispatch_ep<float, true>(p, a, blocks, s);
    } else if (p.bf16) {
      // logits on the tensor cores, then the selection from the (split) fp32 logits
      float* part = ws_ptr<float>(ws, L.router_part);
      e = launch_router_tc(p, x, w_router, ws_ptr<void>(ws, L.router_wt), part,
                           ws_ptr<uint32_t>(ws, L.status), s);
      if (e != cudaSuccess) return e;
      a.logits_in = part;
      a.part_stride = p.Tu * p.E;
      a.nparts = router_plan(p).splits;
      e = route_dispatch_ep<float, true>(p, a, blocks, s);
    } else {
      e = route_dispatch_ep<float, false>(p, a, blocks, s);
    }
    if (e != cudaSuccess) return e;
  }
  if (aux_out) {
    aux_finalize_kernel<<<p.E, 256, 0, s>>>(a.psum_part, a.cnt_part, blocks, p.E, p.Tu, p.K,
                                            p.cfg.aux_alpha, ws_ptr<double>(ws, L.aux_terms),
                                            ws_ptr<unsigned int>(ws, L.status + 4), aux_out);
    note_launch();
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace moe
