// Combine: the gate-weighted sum of a unit's expert outputs, back in unit order.
//   [Lesson 10 "专家并行 EP", §1: y = Σ_{i∈TopK} s_i(x)·FFN_i(x); §3 steps 3-4: results return to
//    their source position and are summed with the gates kept from routing]
// One warp per unit; each lane owns 16-byte column slices; the K picks are summed in k order in
// fp32 (no atomics, so the result is deterministic); dropped picks (slot -1) add nothing.
#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {

// y viewed as one flat array of 16-byte vectors; each warp produces 64 consecutive vectors per
// step (vector wb + 32·j + lane, j = 0, 1), so loads and stores cover 512 contiguous bytes per
// instruction; each lane sums the K picks of its two vectors (2K independent loads in flight).
template <typename T, int KMAX>
__global__ void __launch_bounds__(256)
combine_kernel(const T* __restrict__ y_packed, const int32_t* __restrict__ slot_of,
               const float* __restrict__ gate, T* __restrict__ y, int64_t Tu, int K, int hu,
               int64_t rows, uint32_t* status) {
  constexpr int V = 16 / sizeof(T);
  const uint32_t nvec = (uint32_t)(hu / V);
  const uint64_t total = (uint64_t)Tu * nvec;
  const uint64_t nwarps = (uint64_t)gridDim.x * (blockDim.x >> 5);
  const uint32_t lane = threadIdx.x & 31u;
  const uint4* yp = reinterpret_cast<const uint4*>(y_packed);
  uint4* yo = reinterpret_cast<uint4*>(y);
  griddep_launch_dependents();
  griddep_wait();
  for (uint64_t wb = ((uint64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * 64u; wb < total;
       wb += nwarps * 64u) {
    uint4 raw[2][KMAX];
    float gw[2][KMAX];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const uint64_t i = wb + 32u * j + lane;
#pragma unroll
      for (int k = 0; k < KMAX; ++k) {
        gw[j][k] = 0.f;
        raw[j][k] = make_uint4(0u, 0u, 0u, 0u);
      }
      if (i >= total) continue;
      const uint64_t u = i / nvec, c = i - u * nvec;
#pragma unroll
      for (int k = 0; k < KMAX; ++k) {
        if (k < K) {
          int32_t sl = __ldg(slot_of + u * K + k);
          if (sl >= rows) {
            set_status(status, kDevErrBadIndex);
            sl = -1;
          }
          if (sl >= 0) {
            raw[j][k] = __ldg(yp + (int64_t)sl * nvec + c);
            gw[j][k] = __ldg(gate + u * K + k);
          }
        }
      }
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const uint64_t i = wb + 32u * j + lane;
      if (i >= total) continue;
      float acc[V];
#pragma unroll
      for (int q = 0; q < V; ++q) acc[q] = 0.f;
      // fixed k order, fp32 accumulation (a dropped pick adds 0·0)
#pragma unroll
      for (int k = 0; k < KMAX; ++k) {
        if (k >= K) break;
        const T* pv = reinterpret_cast<const T*>(&raw[j][k]);
#pragma unroll
        for (int q = 0; q < V; ++q) acc[q] = fmaf(gw[j][k], to_f32<T>(pv[q]), acc[q]);
      }
      uint4 o;
      if constexpr (sizeof(T) == 2) {
        uint32_t* po = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
        for (int q = 0; q < 4; ++q) po[q] = pack_bf16x2(acc[2 * q], acc[2 * q + 1]);
      } else {
        o = make_uint4(__float_as_uint(acc[0]), __float_as_uint(acc[1]), __float_as_uint(acc[2]),
                       __float_as_uint(acc[3]));
      }
      yo[i] = o;
    }
  }
}

// Any width: scalar columns.
template <typename T>
__global__ void __launch_bounds__(256)
combine_scalar_kernel(const T* __restrict__ y_packed, const int32_t* __restrict__ slot_of,
                      const float* __restrict__ gate, T* __restrict__ y, int64_t Tu, int K, int hu,
                      int64_t rows, uint32_t* status) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  griddep_launch_dependents();
  griddep_wait();
  for (int64_t u = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); u < Tu; u += warps) {
    for (int c = lane; c < hu; c += 32) {
      float acc = 0.f;
      for (int k = 0; k < K; ++k) {
        const int32_t s = slot_of[u * K + k];
        if (s >= rows) { set_status(status, kDevErrBadIndex); continue; }
        if (s >= 0) acc = fmaf(gate[u * K + k], to_f32<T>(y_packed[(int64_t)s * hu + c]), acc);
      }
      if constexpr (sizeof(T) == 2) y[u * hu + c] = __float2bfloat16_rn(acc);
      else y[u * hu + c] = acc;
    }
  }
}

cudaError_t launch_combine(const Problem& p, const void* y_packed, const int32_t* slot_of,
                           const float* gate, void* y, uint32_t* status, cudaStream_t s, bool pdl) {
  if (p.Tu == 0) return cudaSuccess;
  const int sms = device_sm_count();
  int64_t blocks = (p.Tu * ((int64_t)p.hu * (int64_t)p.elt / 16) + 511) / 512;
  if (blocks > (int64_t)sms * 8) blocks = (int64_t)sms * 8;
  if (blocks < 1) blocks = 1;
  const bool vec = ((int64_t)p.hu * (int64_t)p.elt) % 16 == 0 &&
                   (reinterpret_cast<uintptr_t>(y_packed) & 15) == 0 &&
                   (reinterpret_cast<uintptr_t>(y) & 15) == 0;
  const dim3 g((unsigned)blocks), b(256);
  const int kb = p.K <= 2 ? 2 : (p.K <= 4 ? 4 : 8);
  if (p.bf16) {
    auto yp = static_cast<const __nv_bfloat16*>(y_packed);
    auto yo = static_cast<__nv_bfloat16*>(y);
    if (!vec) return launch_kernel(combine_scalar_kernel<__nv_bfloat16>, g, b, 0, s, 1, pdl, yp, slot_of, gate, yo, p.Tu, p.K, p.hu, p.rows, status);
    if (kb == 2) return launch_kernel(combine_kernel<__nv_bfloat16, 2>, g, b, 0, s, 1, pdl, yp, slot_of, gate, yo, p.Tu, p.K, p.hu, p.rows, status);
    if (kb == 4) return launch_kernel(combine_kernel<__nv_bfloat16, 4>, g, b, 0, s, 1, pdl, yp, slot_of, gate, yo, p.Tu, p.K, p.hu, p.rows, status);
    return launch_kernel(combine_kernel<__nv_bfloat16, 8>, g, b, 0, s, 1, pdl, yp, slot_of, gate, yo, p.Tu, p.K, p.hu, p.rows, status);
  }
  auto yp = static_cast<const float*>(y_packed);
  auto yo = static_cast<float*>(y);
  if (!vec) return launch_kernel(combine_scalar_kernel<float>, g, b, 0, s, 1, pdl, yp, slot_of, gate, yo, p.Tu, p.K, p.hu, p.rows, status);
  if (kb == 2) return launch_kernel(combine_kernel<float, 2>, g, b, 0, s, 1, pdl, yp, slot_of, gate, yo, p.Tu, p.K, p.hu, p.rows, status);
  if (kb == 4) return launch_kernel(combine_kernel<float, 4>, g, b, 0, s, 1, pdl, yp, slot_of, gate, yo, p.Tu, p.K, p.hu, p.rows, status);
  return launch_kernel(combine_kernel<float, 8>, g, b, 0, s, 1, pdl, yp, slot_of, gate, yo, p.Tu, p.K, p.hu, p.rows, status);
}

}  // namespace moe
