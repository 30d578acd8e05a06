// Backward of the layer outside the expert GEMMs (bf16 layers), with the routing held fixed:
//   combine   y[t] = Σ_k kept g[t,k]·Y_packed[slot]      →  dY_packed[slot] = g[t,k]·dy[t],
//                                                           dg[t,k] = <dy[t], Y_packed[slot]>
//             [Lesson 10 "专家并行 EP", §1 y = Σ s_i·FFN_i; §3 step 4]
//   gates     softmax over the picked logits, or σ(l_i)/Σ_picked σ(l_j)  →  dL/dl   [Lesson 10 §1]
//   aux loss  α·E·Σ_i f_i·P_i with f fixed, P_i = mean_t p[t,i]          →  dL/dl   [Lesson 10 §4]
//   router    l = x·W_g (+ bias)  →  dW_g = xᵀ·dl,  dx += dl·W_gᵀ                  [Lesson 10 §1]
//   dispatch  x_packed[slot] = x[t]  →  dx[t] += Σ_k kept dX_packed[slot]           [Lesson 10 §3 step 1]
// Every sum has a fixed order (warp butterflies, per-thread loops, chunk partials added in chunk
// order), so the gradients are deterministic.
#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

__device__ __forceinline__ void bf16x8_to_f32(const uint4 v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    f[2 * j] = __uint_as_float(w[j] << 16);
    f[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint4 f32x8_to_bf16(const float (&f)[8]) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                    pack_bf16x2(f[6], f[7]));
}

// One warp per unit: for each kept pick, dY_packed[slot] = g·dy[t] and dg = <dy[t], Y_packed[slot]>.
__global__ void bwd_combine_kernel(const uint4* __restrict__ dy, const uint4* __restrict__ y_packed,
                                   const int32_t* __restrict__ slot_of, const float* __restrict__ gate,
                                   int64_t Tu, int K, int vecs, int64_t rows, uint4* __restrict__ dy_packed,
                                   float* __restrict__ dgate, uint32_t* status) {
  const int lane = threadIdx.x & 31;
  const int64_t u = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (u >= Tu) return;
  const uint4* d = dy + u * vecs;
  for (int k = 0; k < K; ++k) {
    const int32_t slot = slot_of[u * K + k];
    float acc = 0.0f;
    if (slot >= 0 && slot < rows) {
      const float g = gate[u * K + k];
      const uint4* yp = y_packed + (int64_t)slot * vecs;
      uint4* o = dy_packed + (int64_t)slot * vecs;
      for (int v = lane; v < vecs; v += 32) {
        float a[8], b[8], c[8];
        bf16x8_to_f32(d[v], a);
        bf16x8_to_f32(yp[v], b);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          acc = fmaf(a[j], b[j], acc);
          c[j] = g * a[j];
        }
        o[v] = f32x8_to_bf16(c);
      }
    } else if (slot >= rows && lane == 0) {
      set_status(status, kDevErrBadIndex);
    }
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
    if (lane == 0) dgate[u * K + k] = acc;
  }
}

// One thread per unit: dL/dl[t][:] through the gates of its picks and through P_i of the aux loss.
template <bool SIGMOID>
__global__ void bwd_logits_kernel(const float* __restrict__ logits, const int32_t* __restrict__ idx,
                                  const float* __restrict__ gate, const float* __restrict__ dgate,
                                  const int32_t* __restrict__ counts, int64_t Tu, int E, int K, float aux_scale,
                                  float* __restrict__ dl) {
  const int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (u >= Tu) return;
  const float* l = logits + u * E;
  float* o = dl + u * E;
  // aux: dL/dp[t,i] = aux_scale·f_i with aux_scale = d_aux·α·E/T' and f_i = counts_i/(T'·K)
  const float f_scale = 1.0f / (float)((double)Tu * K);
  float mx = -INFINITY;
  if (!SIGMOID)
    for (int e = 0; e < E; ++e) mx = fmaxf(mx, l[e]);
  float z = 0.0f, inner = 0.0f;  // Σ_i q_i and Σ_i q_i·dp_i, q = exp(l − max) or σ(l)
  for (int e = 0; e < E; ++e) {
    const float q = SIGMOID ? 1.0f / (1.0f + __expf(-l[e])) : __expf(l[e] - mx);
    const float dp = aux_scale * (float)counts[e] * f_scale;
    z += q;
    inner = fmaf(q, dp, inner);
  }
  inner /= z;  // Σ_i p_i·dp_i
  for (int e = 0; e < E; ++e) {
    const float dp = aux_scale * (float)counts[e] * f_scale;
    if (SIGMOID) {
      const float s = 1.0f / (1.0f + __expf(-l[e]));
      o[e] = (dp - inner) / z * s * (1.0f - s);
    } else {
      o[e] = __expf(l[e] - mx) / z * (dp - inner);
    }
  }
  // gates: softmax over the picks (dl = g ⊙ (dg − Σ g·dg)) or s/Σs (ds = (dg − Σ g·dg)/Σs)
  float gin = 0.0f, ssum = 0.0f;
  for (int k = 0; k < K; ++k) {
    gin = fmaf(gate[u * K + k], dgate[u * K + k], gin);
    if (SIGMOID) ssum += 1.0f / (1.0f + __expf(-l[idx[u * K + k]]));
  }
  for (int k = 0; k < K; ++k) {
    const int e = idx[u * K + k];
    if (e < 0 || e >= E) continue;
    const float r = dgate[u * K + k] - gin;
    if (SIGMOID) {
      const float s = 1.0f / (1.0f + __expf(-l[e]));
      o[e] += r / ssum * s * (1.0f - s);
    } else {
      o[e] += gate[u * K + k] * r;
    }
  }
}

// dW_g partials: part[chunk][i][e] = Σ_{t in chunk} x[t][i]·dl[t][e]. A block covers 256 columns i
// (two per thread, one bf16x2 load per token) and EC experts (the thread's accumulators), its
// tokens' dl rows staged in shared memory; x is read once per expert chunk, coalesced.
constexpr int kWgCols = 256, kWgT = 64;
template <int EC>
__global__ void __launch_bounds__(128) bwd_wg_partial_kernel(const __nv_bfloat16* __restrict__ x,
                                                             const float* __restrict__ dl, int64_t Tu, int hu,
                                                             int E, int64_t chunk_len, float* __restrict__ part) {
  __shared__ float sd[kWgT][EC];
  const int i = blockIdx.x * kWgCols + 2 * threadIdx.x;
  const int e0 = blockIdx.y * EC;
  const int64_t t_begin = (int64_t)blockIdx.z * chunk_len;
  const int64_t t_end = t_begin + chunk_len < Tu ? t_begin + chunk_len : Tu;
  float a0[EC], a1[EC];
#pragma unroll
  for (int j = 0; j < EC; ++j) a0[j] = a1[j] = 0.0f;
  for (int64_t t0 = t_begin; t0 < t_end; t0 += kWgT) {
    __syncthreads();
    for (int j = threadIdx.x; j < kWgT * EC; j += 128) {
      const int r = j / EC, c = j % EC;
      const int64_t t = t0 + r;
      sd[r][c] = (t < t_end && e0 + c < E) ? dl[t * E + e0 + c] : 0.0f;
    }
    __syncthreads();
    const int n = (int)(t_end - t0 < kWgT ? t_end - t0 : kWgT);
    if (i < hu) {
#pragma unroll 2
      for (int r = 0; r < n; ++r) {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(x + (t0 + r) * hu + i);
        const float x0 = __uint_as_float(w << 16), x1 = __uint_as_float(w & 0xFFFF0000u);
#pragma unroll
        for (int j = 0; j < EC; ++j) {
          a0[j] = fmaf(x0, sd[r][j], a0[j]);
          a1[j] = fmaf(x1, sd[r][j], a1[j]);
        }
      }
    }
  }
  if (i < hu) {
    float* out = part + (int64_t)blockIdx.z * hu * E;
#pragma unroll
    for (int j = 0; j < EC; ++j) {
      if (e0 + j < E) {
        out[(int64_t)i * E + e0 + j] = a0[j];
        out[(int64_t)(i + 1) * E + e0 + j] = a1[j];
      }
    }
  }
}

__global__ void bwd_wg_reduce_kernel(const float* __restrict__ part, int nchunks, int64_t n, float* __restrict__ dwg) {
  const int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= n) return;
  float s = 0.0f;
  for (int c = 0; c < nchunks; ++c) s += part[(int64_t)c * n + j];
  dwg[j] = s;
}

// One warp per unit: dx[t] = Σ_k kept dX_packed[slot] + Σ_e dl[t][e]·W_gᵀ[e] (bf16 out).
__global__ void bwd_dx_kernel(const uint4* __restrict__ dx_packed, const int32_t* __restrict__ slot_of,
                              const float* __restrict__ dl, const uint4* __restrict__ wgt, int64_t Tu, int K,
                              int E, int vecs, int64_t rows, uint4* __restrict__ dx) {
  extern __shared__ float s_dl[];  // [warps][E]
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t u = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  float* my = s_dl + w * E;
  if (u < Tu)
    for (int e = lane; e < E; e += 32) my[e] = dl[u * E + e];
  __syncwarp();
  if (u >= Tu) return;
  int32_t slots[kMaxTopK];
#pragma unroll
  for (int k = 0; k < kMaxTopK; ++k) slots[k] = k < K ? slot_of[u * K + k] : -1;
  for (int v = lane; v < vecs; v += 32) {
    float acc[8] = {};
#pragma unroll
    for (int k = 0; k < kMaxTopK; ++k) {
      if (slots[k] >= 0 && slots[k] < rows) {
        float f[8];
        bf16x8_to_f32(dx_packed[(int64_t)slots[k] * vecs + v], f);
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] += f[j];
      }
    }
#pragma unroll 8
    for (int e = 0; e < E; ++e) {
      float f[8];
      bf16x8_to_f32(wgt[(int64_t)e * vecs + v], f);
      const float d = my[e];
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = fmaf(d, f[j], acc[j]);
    }
    dx[u * vecs + v] = f32x8_to_bf16(acc);
  }
}

// W_gᵀ[n][k] = W_g[k][n] (32 x 32 tiles through shared memory).
__global__ void __launch_bounds__(256)
router_transpose_kernel(const __nv_bfloat16* __restrict__ w, int hu, int E, __nv_bfloat16* __restrict__ wt) {
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
    if (n < E && k < hu) wt[(int64_t)n * hu + k] = tile[tx][r];
  }
}

}  // namespace

cudaError_t launch_router_transpose(const Problem& p, const void* w_router, void* wt, cudaStream_t s) {
  if (p.Tu == 0) return cudaSuccess;
  return launch_kernel(router_transpose_kernel, dim3((p.hu + 31) / 32, (p.E + 31) / 32), dim3(256), 0, s, 1, false,
                       static_cast<const __nv_bfloat16*>(w_router), p.hu, p.E, static_cast<__nv_bfloat16*>(wt));
}

cudaError_t launch_backward_misc_combine(const Problem& p, const void* dy, const void* y_packed,
                                         const int32_t* slot_of, const float* gate, void* dy_packed,
                                         float* dgate, uint32_t* status, cudaStream_t s) {
  if (p.Tu == 0) return cudaSuccess;
  const int vecs = p.hu / 8;
  const int64_t blocks = (p.Tu * 32 + 255) / 256;
  bwd_combine_kernel<<<(unsigned)blocks, 256, 0, s>>>(static_cast<const uint4*>(dy),
                                                       static_cast<const uint4*>(y_packed), slot_of, gate,
                                                       p.Tu, p.K, vecs, p.rows, static_cast<uint4*>(dy_packed),
                                                       dgate, status);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_backward_logits(const Problem& p, const float* logits, const int32_t* idx, const float* gate,
                                   const float* dgate, const int32_t* counts, float d_aux, float* dl,
                                   cudaStream_t s) {
  if (p.Tu == 0) return cudaSuccess;
  const float aux_scale = (float)((double)d_aux * p.cfg.aux_alpha * p.E / (double)p.Tu);
  const unsigned blocks = (unsigned)((p.Tu + 127) / 128);
  if (p.sigmoid)
    bwd_logits_kernel<true><<<blocks, 128, 0, s>>>(logits, idx, gate, dgate, counts, p.Tu, p.E, p.K, aux_scale, dl);
  else
    bwd_logits_kernel<false><<<blocks, 128, 0, s>>>(logits, idx, gate, dgate, counts, p.Tu, p.E, p.K, aux_scale, dl);
  note_launch();
  return cudaGetLastError();
}

// Chunks of the token range for the dW_g partials: about 600 blocks (four per SM on a B300),
// fixed by the config alone so that the backward workspace size needs no device query.
static int wg_expert_chunk(const Problem& p) { return p.E <= 8 ? 8 : 16; }
int backward_wg_chunks(const Problem& p) {
  const int64_t tiles = (int64_t)((p.hu + kWgCols - 1) / kWgCols) * ((p.E + wg_expert_chunk(p) - 1) / wg_expert_chunk(p));
  int64_t c = (600 + tiles - 1) / tiles;
  const int64_t max_c = (p.Tu + kWgT - 1) / kWgT;
  if (c > max_c) c = max_c;
  if (c < 1) c = 1;
  if (c > 1024) c = 1024;
  return (int)c;
}

cudaError_t launch_backward_router(const Problem& p, const void* x, const float* dl, int nchunks, float* part,
                                   float* dw_router, cudaStream_t s) {
  const int64_t n = (int64_t)p.hu * p.E;
  if (p.Tu == 0) return cudaMemsetAsync(dw_router, 0, (size_t)n * 4, s);
  int64_t chunk_len = (p.Tu + nchunks - 1) / nchunks;
  const int ec = wg_expert_chunk(p);
  const dim3 grid((p.hu + kWgCols - 1) / kWgCols, (p.E + ec - 1) / ec, (unsigned)nchunks);
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
  if (ec == 8) bwd_wg_partial_kernel<8><<<grid, 128, 0, s>>>(xb, dl, p.Tu, p.hu, p.E, chunk_len, part);
  else bwd_wg_partial_kernel<16><<<grid, 128, 0, s>>>(xb, dl, p.Tu, p.hu, p.E, chunk_len, part);
  note_launch();
  bwd_wg_reduce_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(part, nchunks, n, dw_router);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_backward_dx(const Problem& p, const void* dx_packed, const int32_t* slot_of, const float* dl,
                               const void* w_router_t, void* dx, cudaStream_t s) {
  if (p.Tu == 0) return cudaSuccess;
  const int vecs = p.hu / 8;
  const int64_t blocks = (p.Tu * 32 + 255) / 256;
  const size_t smem = (size_t)8 * p.E * sizeof(float);
  bwd_dx_kernel<<<(unsigned)blocks, 256, smem, s>>>(static_cast<const uint4*>(dx_packed), slot_of, dl,
                                                    static_cast<const uint4*>(w_router_t), p.Tu, p.K, p.E, vecs,
                                                    p.rows, static_cast<uint4*>(dx));
  note_launch();
  return cudaGetLastError();
}

}  // namespace moe
