// Router logits on the tensor cores (bf16 layers): l = x·W_g as a dense GEMM
// [T'][h'] x [h'][E] → fp32, written as partial sums of K slices; the selection kernel
// (route.cu, logits path) adds the slices in a fixed order, adds the logit bias and routes.
//   [Lesson 10 "专家并行 EP", §1: affinity scores x·W_g]
//
// W_g is kept in the pages' [h'][E] orientation by the caller; a small kernel writes its
// transpose W_gᵀ [N][h'] (N = E rounded up to a multiple of 16, zero rows past E) into the
// workspace, the K-major B operand the MMA wants.
//
// One CTA per (128-unit tile, K slice); 128 threads: warp 0 lane 0 issues TMA loads (x tile
// 128 x 64 and W_gᵀ tile N x 64, 128-byte swizzle) into a ring of stages; warp 1 allocates TMEM
// and lane 0 issues tcgen05.mma (M = 128, N, K = 16); when the slice is done all four warps
// read their TMEM lane quarter (one unit per thread) and store the fp32 partial logits. When
// there are fewer 128-unit tiles than SMs, the reduction dimension is split so that the x stream
// is spread over about all SMs.
#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {

constexpr int kRtBM = 128, kRtBK = 64, kRtThreads = 128, kRtMaxStages = 8;
constexpr size_t kRtSmemBudget = 100 * 1024;  // two CTAs per SM

struct RouterTcParams {
  int64_t Tu;
  int E, N;
  int nkb;           // k-blocks in total
  int kb_per_split;  // k-blocks per slice
  float* part;       // [S][Tu][E]
  int64_t part_stride;
  int stages;
  uint32_t stage_bytes;
  uint32_t* status;
};

__global__ void __launch_bounds__(kRtThreads, 1)
router_gemm_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                      RouterTcParams p) {
  extern __shared__ unsigned char smem_dyn[];
  __shared__ __align__(8) uint64_t s_bar[2 * kRtMaxStages + 1];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = (smem_addr(smem_dyn) + 1023u) & ~1023u;
  const uint32_t bar0 = smem_addr(s_bar);
  const int S = p.stages;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
  const uint32_t done_bar = bar0 + 8u * (2 * S);
  const uint32_t tmem_cols = p.N <= 32 ? 32u : (p.N <= 64 ? 64u : (p.N <= 128 ? 128u : 256u));

  const int m0 = blockIdx.x * kRtBM;
  const int kb0 = blockIdx.y * p.kb_per_split;
  const int kb1 = min(p.nkb, kb0 + p.kb_per_split);
  const int nk = kb1 - kb0;

  if (warp == 0 && lane == 0) {
    s_abort = 0;
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(done_bar, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmW);
  } else if (warp == 1) {
    tmem_alloc(smem_addr(&s_tmem), tmem_cols);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  volatile int* abort_flag = &s_abort;
  const uint32_t idesc = idesc_bf16_f32(kRtBM, p.N);

  if (warp == 0) {
    if (lane == 0) {
      uint32_t filled = 0, last_parity = 0;
      for (int i = 0; i < nk; ++i) {
        const int st = i % S;
        const uint32_t ph = (uint32_t)(i / S) & 1u;
        if (!mbar_wait(empty_bar(st), ph ^ 1u, abort_flag)) {
          s_abort = 1;
          set_status(p.status, kDevErrTimeout);
          for (int s = 0; s < S; ++s)
            if ((filled >> s) & 1u) mbar_wait(full_bar(s), (last_parity >> s) & 1u, nullptr, 50000000ull);
          break;
        }
        const uint32_t sa = sbase + (uint32_t)st * p.stage_bytes;
        mbar_arrive_expect_tx(full_bar(st), p.stage_bytes);
        tma_load_2d(sa, &tmX, full_bar(st), (kb0 + i) * kRtBK, m0);
        tma_load_2d(sa + kRtBM * kRtBK * 2, &tmW, full_bar(st), (kb0 + i) * kRtBK, 0);
        filled |= 1u << st;
        last_parity = (last_parity & ~(1u << st)) | (ph << st);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      bool aborted = false;
      for (int i = 0; i < nk; ++i) {
        const int st = i % S;
        const uint32_t ph = (uint32_t)(i / S) & 1u;
        if (!mbar_wait(full_bar(st), ph, abort_flag)) {
          aborted = true;
          break;
        }
        tc_fence_after();
        const uint32_t sa = sbase + (uint32_t)st * p.stage_bytes;
        const uint64_t ad = sdesc_kmajor_sw128(sa), bd = sdesc_kmajor_sw128(sa + kRtBM * kRtBK * 2);
#pragma unroll
        for (int k = 0; k < kRtBK / 16; ++k)
          umma_bf16(tmem, ad + (uint64_t)(2 * k), bd + (uint64_t)(2 * k), idesc, (i > 0 || k > 0) ? 1u : 0u);
        umma_commit(empty_bar(st));
      }
      if (aborted) {
        s_abort = 1;
        set_status(p.status, kDevErrTimeout);
      }
      umma_commit(done_bar);  // also covers the no-work case: arrives once prior MMAs finish
    }
    __syncwarp();
  }

  // epilogue: every warp reads its 32 TMEM lanes = 32 units of the tile
  const bool ok = mbar_wait(done_bar, 0, abort_flag);
  if (!ok && lane == 0) {
    s_abort = 1;
    set_status(p.status, kDevErrTimeout);
  }
  tc_fence_after();
  const int64_t u = (int64_t)m0 + warp * 32 + lane;
  const bool row_ok = ok && nk > 0 && u < p.Tu;
  float* out = p.part + (int64_t)blockIdx.y * p.part_stride + u * p.E;
  const uint32_t t_row = tmem + ((uint32_t)(warp * 32) << 16);
  if (ok) {
    if (p.N == 16) {
      uint32_t v[16];
      tmem_ld_32x32b_x16(t_row, v);
      tmem_ld_wait();
      if (row_ok) {
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (j < p.E) out[j] = __uint_as_float(v[j]);
      }
    } else {
      for (int c = 0; c < p.N; c += 32) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(t_row + c, v);
        tmem_ld_wait();
        if (row_ok) {
          if ((p.E & 3) == 0 && c + 32 <= p.E) {
            float4* o4 = reinterpret_cast<float4*>(out + c);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              o4[j] = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                  __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (c + j < p.E) out[c + j] = __uint_as_float(v[j]);
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, tmem_cols);
  }
}

// W_gᵀ[n][k] = W_g[k][n] for n < E, 0 for E <= n < N.  (32 x 32 tiles through shared memory)
__global__ void __launch_bounds__(256)
router_transpose_kernel(const __nv_bfloat16* __restrict__ w, int hu, int E, int N,
                        __nv_bfloat16* __restrict__ wt) {
  __shared__ __nv_bfloat16 tile[32][33];
  const int k0 = blockIdx.x * 32, n0 = blockIdx.y * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  for (int r = ty; r < 32; r += 8) {
    const int k = k0 + r, n = n0 + tx;
    tile[r][tx] = (k < hu && n < E) ? w[(int64_t)k * E + n] : __float2bfloat16(0.f);
  }
  __syncthreads();
  for (int r = ty; r < 32; r += 8) {
    const int n = n0 + r, k = k0 + tx;
    if (n < N && k < hu) wt[(int64_t)n * hu + k] = tile[tx][r];
  }
}

RouterPlan router_plan(const Problem& p) {
  RouterPlan r;
  r.N = (p.E + 15) / 16 * 16;
  r.m_tiles = (int)((p.Tu + kRtBM - 1) / kRtBM);
  r.nkb = (p.hu + kRtBK - 1) / kRtBK;
  int S = r.m_tiles > 0 ? (int)(kRouterSplitTarget / r.m_tiles) : 1;
  if (S < 1) S = 1;
  if (S > 8) S = 8;
  if (S > r.nkb / 4) S = r.nkb / 4 > 0 ? r.nkb / 4 : 1;
  r.kb_per_split = (r.nkb + S - 1) / S;
  r.splits = (r.nkb + r.kb_per_split - 1) / r.kb_per_split;
  return r;
}

cudaError_t launch_router_tc(const Problem& p, const void* x, const void* w_router, void* wt, float* part,
                             uint32_t* status, cudaStream_t s) {
  const RouterPlan r = router_plan(p);
  if (p.Tu == 0) return cudaSuccess;
  dim3 tg((p.hu + 31) / 32, (r.N + 31) / 32);
  router_transpose_kernel<<<tg, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(w_router), p.hu, p.E, r.N,
                                             static_cast<__nv_bfloat16*>(wt));
  note_launch();
  CUtensorMap mX, mW;
  if (!encode_tmap_2d_bf16(&mX, x, (uint64_t)p.hu, (uint64_t)p.Tu, kRtBK, kRtBM) ||
      !encode_tmap_2d_bf16(&mW, wt, (uint64_t)p.hu, (uint64_t)r.N, kRtBK, (uint32_t)r.N))
    return cudaErrorInvalidValue;
  RouterTcParams g;
  g.Tu = p.Tu;
  g.E = p.E;
  g.N = r.N;
  g.nkb = r.nkb;
  g.kb_per_split = r.kb_per_split;
  g.part = part;
  g.part_stride = p.Tu * p.E;
  g.stage_bytes = (uint32_t)(kRtBM * kRtBK * 2 + r.N * kRtBK * 2);
  int stages = (int)(kRtSmemBudget / g.stage_bytes);
  if (stages < 3) stages = 3;
  g.stages = stages > kRtMaxStages ? kRtMaxStages : stages;
  g.status = status;
  const size_t smem = (size_t)g.stages * g.stage_bytes + 1024;
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(router_gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(3 * (kRtBM * kRtBK * 2 + 256 * kRtBK * 2) + 1024));
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  router_gemm_tc_kernel<<<dim3(r.m_tiles, r.splits), kRtThreads, smem, s>>>(mX, mW, g);
  note_launch();
  return cudaGetLastError();
}

}  // namespace moe
