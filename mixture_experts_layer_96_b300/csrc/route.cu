// Router logits for fp32 layers on the CUDA cores: l = x·W_g, written as fp32 [T'][E] for the
// selection kernel (route_select.cu); bf16 layers use the tensor-core GEMM (route_tc.cu). Also
// the aux-loss reduction, and launch_route, which runs the router and the selection.
//   [Lesson 10 "专家并行 EP", §1: affinity scores x·W_g; §4: L_aux = α·E·Σ f_i·P_i]
//
// Block = 256 threads, BT units; the [BT][EP] logit tile (EP = E rounded up to a power of two
// >= 8) is accumulated with fp32 FMAs over 32-column steps of h' staged in shared memory; for
// small E the block splits the reduction dimension over warp groups and adds the slices in a
// fixed order.
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
  static_assert(TROWS * TM == BT, "tile");
  static_assert(GT * KSPLIT == kRouteThreads, "split");
  static constexpr size_t SMEM = (size_t)MAIN_FLOATS * 4;
};

struct RouteArgs {
  const void* x;            // [Tu][hu] (TIn)
  const void* w;            // [hu][E] (TIn)
  float* logits;            // [Tu][E] out
  int64_t Tu;
  int hu, E;
};

template <typename TIn, int EP>
__global__ void __launch_bounds__(kRouteThreads)
router_gemm_simt_kernel(RouteArgs a) {
  using Tl = RouteTile<EP>;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  float* main_f = reinterpret_cast<float*>(smem_raw);

  const int tid = threadIdx.x;
  const int64_t u0 = (int64_t)blockIdx.x * Tl::BT;
  const int E = a.E;
  float* ls = main_f;  // [BT][EP+1] logits tile (aliases the GEMM staging after phase 1)


  // ------------------------------------------------------------------ phase 1: logit tile
  {
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
        (void)e;
        ls[r * (EP + 1) + e] = tmp[n];
      }
    } else {
#pragma unroll
      for (int i = 0; i < Tl::TM; ++i)
#pragma unroll
        for (int j = 0; j < Tl::TN; ++j) {
          ls[(tr + Tl::TROWS * i) * (EP + 1) + tc + Tl::ECOLS * j] = acc[i][j];
        }
    }
  }
  __syncthreads();

  // the logit tile → global (valid units and experts only)
  for (int i = tid; i < Tl::BT * EP; i += kRouteThreads) {
    const int r = i / EP, e = i % EP;
    const int64_t u = u0 + r;
    if (u < a.Tu && e < E) a.logits[u * E + e] = ls[r * (EP + 1) + e];
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
  if (last) {
    __threadfence();
    const volatile double* vt = terms;
    for (int i = tid; i < E; i += 256) sP[i] = vt[i];  // all E terms, loaded in parallel
    __syncthreads();
    if (tid == 0) {
      double acc = 0.0;
      for (int i = 0; i < E; ++i) acc += sP[i];  // expert order
      *aux_out = (float)((double)alpha * E * acc);
      *ticket = 0u;
    }
  }
}

template <int EP>
static cudaError_t launch_router_simt_t(const RouteArgs& a, int64_t blocks, cudaStream_t s) {
  using Tl = RouteTile<EP>;
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(router_gemm_simt_kernel<float, EP>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Tl::SMEM);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  router_gemm_simt_kernel<float, EP><<<(unsigned)blocks, kRouteThreads, Tl::SMEM, s>>>(a);
  note_launch();
  return cudaGetLastError();
}

static cudaError_t launch_router_simt(const Problem& p, const void* x, const void* w, float* logits,
                                      cudaStream_t s) {
  int ep = 8;
  while (ep < p.E) ep <<= 1;
  RouteArgs a;
  a.x = x;
  a.w = w;
  a.logits = logits;
  a.Tu = p.Tu;
  a.hu = p.hu;
  a.E = p.E;
  auto blocks = [&](int bt) { return (p.Tu + bt - 1) / bt; };
  switch (ep) {
    case 8: return launch_router_simt_t<8>(a, blocks(RouteTile<8>::BT), s);
    case 16: return launch_router_simt_t<16>(a, blocks(RouteTile<16>::BT), s);
    case 32: return launch_router_simt_t<32>(a, blocks(RouteTile<32>::BT), s);
    case 64: return launch_router_simt_t<64>(a, blocks(RouteTile<64>::BT), s);
    case 128: return launch_router_simt_t<128>(a, blocks(RouteTile<128>::BT), s);
    default: return launch_router_simt_t<256>(a, blocks(RouteTile<256>::BT), s);
  }
}

int select_block_units(int E);  // route_select.cu
int route_block_units(int E) { return select_block_units(E); }

cudaError_t launch_select(const Problem& p, const float* logits, int nparts, int64_t part_stride,
                          const float* logit_bias, const float* select_bias, int32_t* idx, float* gate,
                          float* logits_out, float* psum_part, int32_t* cnt_part, cudaStream_t s);

cudaError_t launch_route(const Problem& p, const void* x, const void* w_router,
                         const float* logits_in, const float* logit_bias, const float* select_bias,
                         int32_t* idx, float* gate, float* logits_out, float* aux_out, void* ws,
                         cudaStream_t s) {
  const WsLayout L = ws_layout(p);
  float* psum_part = ws_ptr<float>(ws, L.psum_part);
  int32_t* cnt_part = ws_ptr<int32_t>(ws, L.cnt_part);
  cudaError_t e = cudaSuccess;
  if (p.Tu > 0) {
    const float* logits = logits_in;
    int nparts = 1;
    if (!logits_in) {
      float* part = ws_ptr<float>(ws, L.router_part);
      if (p.bf16) {
        // x·W_g on the tensor cores, as K-slice partial sums
        e = launch_router_tc(p, x, w_router, ws_ptr<void>(ws, L.router_wt), part,
                             ws_ptr<uint32_t>(ws, L.status), s);
        nparts = router_plan(p).splits;
      } else {
        e = launch_router_simt(p, x, w_router, part, s);
      }
      if (e != cudaSuccess) return e;
      logits = part;
    }
    e = launch_select(p, logits, nparts, p.Tu * p.E, logit_bias, select_bias, idx, gate, logits_out,
                      psum_part, cnt_part, s);
    if (e != cudaSuccess) return e;
  }
  if (aux_out) {
    aux_finalize_kernel<<<p.E, 256, 0, s>>>(psum_part, cnt_part, p.route_blocks, p.E, p.Tu, p.K,
                                            p.cfg.aux_alpha, ws_ptr<double>(ws, L.aux_terms),
                                            ws_ptr<unsigned int>(ws, L.status + 4), aux_out);
    note_launch();
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace moe
