// Expert FFN in fp32 on the CUDA cores (the fp32 layer; no TF32, no bf16 anywhere).
//   [Lesson 10 "专家并行 EP", §3 step 2: grouped GEMM over the units packed per expert]
// Same schedule as the tensor-core path (expert → n-tile → m-tile from device-side offsets),
// 64 x 64 tiles, 256 threads with 4 x 4 register tiles, K staged through shared memory by 16.
#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {

constexpr int kSB = 64, kSK = 16;

template <bool SWIGLU>
__global__ void __launch_bounds__(256)
expert_gemm_simt_kernel(const float* __restrict__ A, const float* __restrict__ B0,
                        const float* __restrict__ B1, const int32_t* __restrict__ offsets, int E,
                        int K, int w_rows, int n_tiles, int n_out, int64_t rows_cap,
                        float* __restrict__ out, uint32_t* status) {
  __shared__ int s_off[kMaxExperts + 1];
  __shared__ int s_pre[kMaxExperts + 1];
  __shared__ int s_ok;
  __shared__ float As[kSK][kSB + 4];
  __shared__ float Bs0[kSK][kSB + 4];
  __shared__ float Bs1[SWIGLU ? kSK : 1][kSB + 4];
  const int tid = threadIdx.x;
  griddep_launch_dependents();
  griddep_wait();
  if (tid < 32) {
    const bool ok = warp_tile_prefix(offsets, E, kSB, rows_cap, s_off, s_pre);
    if (tid == 0) {
      s_ok = ok;
      if (!ok && blockIdx.x == 0) set_status(status, kDevErrBadOffsets);
    }
  }
  __syncthreads();
  if (!s_ok) return;
  const int total = s_pre[E] * n_tiles;
  const int ty = tid / 16, tx = tid % 16;
  for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
    int e, mt, nt;
    decode_tile(tile, s_pre, E, n_tiles, e, mt, nt);
    const int rows_e = s_off[e + 1] - s_off[e];
    const int64_t r0 = (int64_t)s_off[e] + (int64_t)mt * kSB;
    const int n0 = nt * kSB;
    float acc0[4][4] = {}, acc1[4][4] = {};
    for (int k0 = 0; k0 < K; k0 += kSK) {
      __syncthreads();
      for (int i = tid; i < kSB * kSK; i += 256) {
        const int r = i / kSK, k = i % kSK;
        const bool kin = k0 + k < K;
        As[k][r] = (mt * kSB + r < rows_e && kin) ? A[(r0 + r) * K + k0 + k] : 0.f;
        const bool nin = n0 + r < w_rows && kin;
        Bs0[k][r] = nin ? B0[((int64_t)e * w_rows + n0 + r) * K + k0 + k] : 0.f;
        if (SWIGLU) Bs1[k][r] = nin ? B1[((int64_t)e * w_rows + n0 + r) * K + k0 + k] : 0.f;
      }
      __syncthreads();
#pragma unroll
      for (int k = 0; k < kSK; ++k) {
        float a[4], b0[4], b1[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] = As[k][ty + 16 * i];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          b0[j] = Bs0[k][tx + 16 * j];
          if (SWIGLU) b1[j] = Bs1[k][tx + 16 * j];
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            acc0[i][j] = fmaf(a[i], b0[j], acc0[i][j]);
            if (SWIGLU) acc1[i][j] = fmaf(a[i], b1[j], acc1[i][j]);
          }
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int rl = mt * kSB + ty + 16 * i;
      if (rl >= rows_e) continue;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c = n0 + tx + 16 * j;
        if (c >= n_out) continue;
        float v = acc0[i][j];
        if (SWIGLU) v = (v / (1.0f + expf(-v))) * acc1[i][j];
        out[((int64_t)s_off[e] + rl) * n_out + c] = v;
      }
    }
  }
}

cudaError_t launch_expert_ffn_simt(const Problem& p, const void* x_packed, const int32_t* offsets,
                                   const void* w_gate, const void* w_up, const void* w_down,
                                   void* hidden, void* y_packed, uint32_t* status, cudaStream_t s, bool pdl) {
  if (p.rows == 0) return cudaSuccess;
  const int64_t max_m = (p.rows + kSB - 1) / kSB + p.E;
  const int nt1 = (p.d_ff + kSB - 1) / kSB, nt2 = (p.hu + kSB - 1) / kSB;
  const int cap = device_sm_count() * 8;
  int g1 = (int)((max_m * nt1 < cap) ? max_m * nt1 : cap);
  int g2 = (int)((max_m * nt2 < cap) ? max_m * nt2 : cap);
  cudaError_t e = launch_kernel(expert_gemm_simt_kernel<true>, dim3(g1), dim3(256), 0, s, 1, pdl,
                                static_cast<const float*>(x_packed), static_cast<const float*>(w_gate),
                                static_cast<const float*>(w_up), offsets, p.E, p.hu, p.d_ff, nt1, p.d_ff, p.rows,
                                static_cast<float*>(hidden), status);
  if (e != cudaSuccess) return e;
  return launch_kernel(expert_gemm_simt_kernel<false>, dim3(g2), dim3(256), 0, s, 1, true,
                       static_cast<const float*>(hidden), static_cast<const float*>(w_down),
                       static_cast<const float*>(nullptr), offsets, p.E, p.d_ff, p.hu, nt2, p.hu, p.rows,
                       static_cast<float*>(y_packed), status);
}

}  // namespace moe
