// Combine: the gate-weighted sum of a unit's expert outputs, back in unit order.
//   [Lesson 10 "专家并行 EP", §1: y = Σ_{i∈TopK} s_i(x)·FFN_i(x); §3 steps 3-4: results return to
//    their source position and are summed with the gates kept from routing]
// One warp per unit; each lane owns 16-byte column slices; the K picks are summed in k order in
// fp32 (no atomics, so the result is deterministic); dropped picks (slot -1) add nothing.
#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {

template <typename T>
__global__ void __launch_bounds__(256)
combine_kernel(const T* __restrict__ y_packed, const int32_t* __restrict__ slot_of,
               const float* __restrict__ gate, T* __restrict__ y, int64_t Tu, int K, int hu,
               int64_t rows, uint32_t* status) {
  constexpr int V = 16 / sizeof(T);
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int nvec = hu / V;
  for (int64_t u = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); u < Tu; u += warps) {
    int32_t sl[kMaxTopK];
    float gw[kMaxTopK];
    bool bad = false;
#pragma unroll
    for (int k = 0; k < kMaxTopK; ++k) {
      sl[k] = (k < K) ? __ldg(slot_of + u * K + k) : -1;
      gw[k] = (k < K) ? __ldg(gate + u * K + k) : 0.f;
      if (sl[k] >= rows) { sl[k] = -1; bad = true; }
    }
    if (bad && lane == 0) set_status(status, kDevErrBadIndex);
    for (int v = lane; v < nvec; v += 32) {
      float acc[V];
#pragma unroll
      for (int j = 0; j < V; ++j) acc[j] = 0.f;
#pragma unroll
      for (int k = 0; k < kMaxTopK; ++k) {
        if (sl[k] < 0) continue;
        const uint4 q = __ldg(reinterpret_cast<const uint4*>(y_packed + (int64_t)sl[k] * hu) + v);
        const T* pv = reinterpret_cast<const T*>(&q);
#pragma unroll
        for (int j = 0; j < V; ++j) acc[j] = fmaf(gw[k], to_f32<T>(pv[j]), acc[j]);
      }
      uint4 o;
      if constexpr (sizeof(T) == 2) {
        uint32_t* po = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
        for (int j = 0; j < 4; ++j) po[j] = pack_bf16x2(acc[2 * j], acc[2 * j + 1]);
      } else {
        o = make_uint4(__float_as_uint(acc[0]), __float_as_uint(acc[1]), __float_as_uint(acc[2]),
                       __float_as_uint(acc[3]));
      }
      reinterpret_cast<uint4*>(y + u * hu)[v] = o;
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
                           const float* gate, void* y, uint32_t* status, cudaStream_t s) {
  if (p.Tu == 0) return cudaSuccess;
  const int sms = device_sm_count();
  int64_t blocks = (p.Tu + 7) / 8;
  if (blocks > (int64_t)sms * 16) blocks = (int64_t)sms * 16;
  const bool vec = ((int64_t)p.hu * (int64_t)p.elt) % 16 == 0 &&
                   (reinterpret_cast<uintptr_t>(y_packed) & 15) == 0 &&
                   (reinterpret_cast<uintptr_t>(y) & 15) == 0;
  if (p.bf16) {
    auto yp = static_cast<const __nv_bfloat16*>(y_packed);
    auto yo = static_cast<__nv_bfloat16*>(y);
    if (vec) combine_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, s>>>(yp, slot_of, gate, yo, p.Tu, p.K, p.hu, p.rows, status);
    else combine_scalar_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, s>>>(yp, slot_of, gate, yo, p.Tu, p.K, p.hu, p.rows, status);
  } else {
    auto yp = static_cast<const float*>(y_packed);
    auto yo = static_cast<float*>(y);
    if (vec) combine_kernel<float><<<(unsigned)blocks, 256, 0, s>>>(yp, slot_of, gate, yo, p.Tu, p.K, p.hu, p.rows, status);
    else combine_scalar_kernel<float><<<(unsigned)blocks, 256, 0, s>>>(yp, slot_of, gate, yo, p.Tu, p.K, p.hu, p.rows, status);
  }
  note_launch();
  return cudaGetLastError();
}

}  // namespace moe
