// Routing of fp32 layers, and routing from given logits.
//   [Lesson 10 "专家并行 EP", §1: affinity scores x·W_g, s(x) = Softmax(TopK(x·W_g, K)) or sigmoid;
//    §4: L_aux = α·E·Σ f_i·P_i]
//
// fp32 layers: router_gemm_simt_kernel computes l = x·W_g on the CUDA cores into the workspace
// (bf16 layers use the tensor-core kernel of route_tc.cu, which routes in its epilogue). Block =
// 256 threads, BT units; the [BT][EP] logit tile (EP = E rounded up to a power of two >= 8) is
// accumulated with fp32 FMAs over 32-column steps of h' staged in shared memory; for small E the
// block splits the reduction dimension over warp groups and adds the slices in a fixed order.
//
// select_logits_kernel routes from fp32 logits [T'][E]: a block per 128 units stages the logits
// plus the logit bias (added in fp32) in shared memory and runs the same tile routing as the fused
// kernel (select_tile.cuh), so both leave the same per-tile counts, Σp and pick places for the
// dispatch and the aux loss.
#include <math.h>

#include "moe_device.cuh"
#include "moe_internal.h"
#include "select_tile.cuh"

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

namespace {

constexpr int kSelThreads = 256;

struct SelLogitsArgs {
  const float* logits;      // [T'][E]
  const float* logit_bias;  // [E] or null
  float* logits_out;        // [T'][E] or null (logits with the bias)
  SelectCtx sel;
  int32_t* rank_out;        // [T'][K]
  int32_t* tile_hist;       // [tiles][E]
  float* tile_psum;         // [tiles][E]
  int64_t Tu;
};

struct SelEpi {
  int ldl;
  size_t lg, picks, rank, lanes, wpre, gscr, psum, hist, scratch, total;
};

inline SelEpi sel_epi(int E, int epl) {
  SelEpi L;
  L.ldl = E + 1;
  size_t off = 0;
  auto take = [&](size_t bytes) { const size_t at = off; off = (off + bytes + 15) / 16 * 16; return at; };
  L.lg = take((size_t)kTileUnits * L.ldl * 4);
  L.picks = take((size_t)kTileUnits * kPickStride * 4);
  L.rank = take((size_t)kTileUnits * kPickStride * 4);
  L.lanes = take((size_t)(kSelThreads / 32) * E * 4);
  L.wpre = take((size_t)(kSelThreads / 32) * E * 4);
  L.gscr = take(epl > 0 ? (size_t)(kSelThreads / 32) * 32 * epl * 8 : 0);
  L.psum = take((size_t)E * 4);
  L.hist = take((size_t)E * 4);
  L.scratch = take((size_t)kSelThreads * 4);
  L.total = off;
  return L;
}

template <int EPL, int KMAX, bool SIGMOID>
__global__ void __launch_bounds__(kSelThreads)
select_logits_kernel(SelLogitsArgs a, SelEpi L) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  griddep_launch_dependents();
  griddep_wait();
  const int tid = threadIdx.x, E = a.sel.E, K = a.sel.K, ldl = L.ldl;
  const int64_t u0 = (int64_t)blockIdx.x * kTileUnits;
  const int R = (int)min((int64_t)kTileUnits, a.Tu - u0);
  float* lg = reinterpret_cast<float*>(smem_raw + L.lg);
  for (int i = tid; i < R * E; i += kSelThreads) {
    const int r = i / E, e = i - r * E;
    float v = a.logits[(u0 + r) * E + e];
    if (a.logit_bias) v = v + a.logit_bias[e];
    lg[r * ldl + e] = v;
    if (a.logits_out) a.logits_out[(u0 + r) * E + e] = v;
  }
  __syncthreads();
  int* picks = reinterpret_cast<int*>(smem_raw + L.picks);
  int* rank = reinterpret_cast<int*>(smem_raw + L.rank);
  float* psum_s = reinterpret_cast<float*>(smem_raw + L.psum);
  int* hist_s = reinterpret_cast<int*>(smem_raw + L.hist);
  if constexpr (EPL == 0)
    select_rows_thread<KMAX, SIGMOID>(a.sel, lg, ldl, R, u0, picks);
  else
    select_rows_warp<EPL, SIGMOID>(a.sel, lg, ldl, R, u0, picks, smem_raw + L.gscr);
  __syncthreads();
  column_sums(lg, ldl, R, E, psum_s, reinterpret_cast<float*>(smem_raw + L.scratch));
  rank_picks(picks, R, K, E, rank, hist_s, reinterpret_cast<uint32_t*>(smem_raw + L.lanes),
             reinterpret_cast<int*>(smem_raw + L.wpre));
  for (int e = tid; e < E; e += kSelThreads) {
    a.tile_hist[(int64_t)blockIdx.x * E + e] = hist_s[e];
    a.tile_psum[(int64_t)blockIdx.x * E + e] = psum_s[e];
  }
  for (int i = tid; i < R * K; i += kSelThreads) {
    const int t = i / K, k = i - t * K;
    a.rank_out[(u0 + t) * K + k] = rank[t * kPickStride + k];
  }
}

template <int EPL, int KMAX, bool SIGMOID>
cudaError_t launch_sel(const SelLogitsArgs& a, const SelEpi& L, unsigned grid, cudaStream_t s, bool pdl) {
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(select_logits_kernel<EPL, KMAX, SIGMOID>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  return launch_kernel(select_logits_kernel<EPL, KMAX, SIGMOID>, dim3(grid), dim3(kSelThreads), L.total, s, 1, pdl,
                       a, L);
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
  return launch_kernel(router_gemm_simt_kernel<float, EP>, dim3((unsigned)blocks), dim3(kRouteThreads), Tl::SMEM, s,
                       1, false, a);
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

// MurmurHash3's 32-bit finalizer (xor-shift 16, ·0x85ebca6b, xor-shift 13, ·0xc2b2ae35, xor-shift 16).
__device__ __forceinline__ uint32_t fmix32(uint32_t h) {
  h ^= h >> 16;
  h *= 0x85ebca6bu;
  h ^= h >> 13;
  h *= 0xc2b2ae35u;
  h ^= h >> 16;
  return h;
}

// Hash gate: unit u goes to expert fmix32(token_ids[u]) mod E with gate 1 (top-1). A block per
// 128-unit tile also leaves the tile's picks per expert and each pick's place among them, as the
// router kernels do, for the scan and pack.
__global__ void __launch_bounds__(kTileUnits)
hash_route_kernel(const int32_t* __restrict__ ids, int64_t Tu, int E, int32_t* __restrict__ idx,
                  float* __restrict__ gate, int32_t* __restrict__ rank_out, int32_t* __restrict__ tile_hist) {
  __shared__ int picks[kTileUnits * kPickStride];
  __shared__ int rank[kTileUnits * kPickStride];
  __shared__ uint32_t lanes_of[(kTileUnits / 32) * kMaxExperts];
  __shared__ int warp_pre[(kTileUnits / 32) * kMaxExperts];
  __shared__ int hist[kMaxExperts];
  griddep_launch_dependents();
  griddep_wait();
  const int t = threadIdx.x;
  const int64_t u0 = (int64_t)blockIdx.x * kTileUnits, u = u0 + t;
  const int R = (int)min((int64_t)kTileUnits, Tu - u0);
  if (t < R) {
    const int e = (int)(fmix32((uint32_t)ids[u]) % (uint32_t)E);
    idx[u] = e;
    gate[u] = 1.0f;
    picks[t * kPickStride] = e;
  }
  __syncthreads();
  rank_picks(picks, R, 1, E, rank, hist, lanes_of, warp_pre);
  if (t < R) rank_out[u] = rank[t * kPickStride];
  for (int e = t; e < E; e += kTileUnits) tile_hist[(int64_t)blockIdx.x * E + e] = hist[e];
}

}  // namespace

cudaError_t launch_hash_route(const Problem& p, const int32_t* token_ids, int32_t* idx, float* gate, int32_t* rank_out,
                              int32_t* tile_hist, cudaStream_t s) {
  if (p.Tu == 0) return cudaSuccess;
  return launch_kernel(hash_route_kernel, dim3((unsigned)p.ntiles), dim3(kTileUnits), 0, s, 1, false, token_ids, p.Tu,
                       p.E, idx, gate, rank_out, tile_hist);
}

cudaError_t launch_select_logits(const Problem& p, const float* logits, const float* logit_bias, const SelectCtx& sel,
                                 float* logits_out, int32_t* rank_out, int32_t* tile_hist, float* tile_psum,
                                 cudaStream_t s, bool pdl) {
  if (p.Tu == 0) return cudaSuccess;
  SelLogitsArgs a;
  a.logits = logits;
  a.logit_bias = logit_bias;
  a.logits_out = logits_out;
  a.sel = sel;
  a.rank_out = rank_out;
  a.tile_hist = tile_hist;
  a.tile_psum = tile_psum;
  a.Tu = p.Tu;
  const bool warp_sel = p.E > 64;
  const int epl = !warp_sel ? 0 : (p.E <= 128 ? 4 : 8);
  const SelEpi L = sel_epi(p.E, epl);
  const unsigned grid = (unsigned)p.ntiles;
  const int kb = p.K <= 2 ? 2 : (p.K <= 4 ? 4 : 8);
  if (warp_sel) {
    if (epl == 4) return p.sigmoid ? launch_sel<4, 8, true>(a, L, grid, s, pdl) : launch_sel<4, 8, false>(a, L, grid, s, pdl);
    return p.sigmoid ? launch_sel<8, 8, true>(a, L, grid, s, pdl) : launch_sel<8, 8, false>(a, L, grid, s, pdl);
  }
  if (p.sigmoid) {
    if (kb == 2) return launch_sel<0, 2, true>(a, L, grid, s, pdl);
    if (kb == 4) return launch_sel<0, 4, true>(a, L, grid, s, pdl);
    return launch_sel<0, 8, true>(a, L, grid, s, pdl);
  }
  if (kb == 2) return launch_sel<0, 2, false>(a, L, grid, s, pdl);
  if (kb == 4) return launch_sel<0, 4, false>(a, L, grid, s, pdl);
  return launch_sel<0, 8, false>(a, L, grid, s, pdl);
}

cudaError_t launch_router_simt_logits(const Problem& p, const void* x, const void* w, float* logits, cudaStream_t s) {
  return launch_router_simt(p, x, w, logits, s);
}

}  // namespace moe
