// Dispatch: capacity drop and pack of the units per expert, plus the aux-loss reduction.
//   [Lesson 10 "专家并行 EP", §3 step 1: pack the token vectors per destination expert;
//    §4: capacity C = CF·K·T/E, picks past C dropped; L_aux = α·E·Σ f_i·P_i]
//
// The queue order inside an expert is unit order (a unit's K picks are distinct), so the place of
// pick (t,k) in expert e's queue is the number of earlier units that picked e: a stable counting
// sort over chunks of units. The routing kernels (route_tc.cu, route.cu) already leave, per chunk
// of 128 units, the picks per expert and each pick's place among the chunk's picks of its expert;
// from given picks, chunk_rank_kernel computes the same over chunks of 256 units. Then:
//   scan:  a block per expert: the exclusive scan of the expert's column of chunk counts gives
//          each chunk's base in the expert's queue and the pre-drop count; the same block reduces
//          the expert's Σp column for the aux loss. The last block to finish (ticket) scans the
//          kept rows n_e = min(count_e, C) into the offsets and adds the aux terms (fixed tree).
//   pack:  one warp per unit: place = chunk base + place in chunk; kept if place < C, at packed row
//          offsets[e] + place; the unit's x row is read once and written to each of its kept rows.
// Integer sums only (besides the fixed-order aux sums), no atomics whose order matters, no
// inter-block waits.
#include "moe_device.cuh"
#include "moe_internal.h"
#include "select_tile.cuh"

namespace moe {

namespace {

constexpr int kScanThreads = 256;
constexpr int kRankWarps = kChunk / 32;

// Places of given picks within chunks of kChunk units (bad units, with an index out of range or
// repeated, get place -1 for every pick and set the status bit).
__global__ void __launch_bounds__(kChunk)
chunk_rank_kernel(const int32_t* __restrict__ idx, int64_t Tu, int K, int E, int32_t* __restrict__ place,
                  int32_t* __restrict__ chunk_hist, uint32_t* status) {
  __shared__ int picks[kChunk * kPickStride];
  __shared__ int rank[kChunk * kPickStride];
  __shared__ uint32_t lanes_of[kRankWarps * kMaxExperts];
  __shared__ int warp_pre[kRankWarps * kMaxExperts];
  __shared__ int hist[kMaxExperts];
  griddep_launch_dependents();
  griddep_wait();
  const int t = threadIdx.x;
  const int64_t u0 = (int64_t)blockIdx.x * kChunk, u = u0 + t;
  const int R = (int)min((int64_t)kChunk, Tu - u0);
  if (t < R) {
    int pk[kMaxTopK];
    bool bad = false;
    for (int k = 0; k < K; ++k) {
      const int e = idx[u * K + k];
      pk[k] = e;
      if (e < 0 || e >= E) bad = true;
      for (int j = 0; j < k; ++j)
        if (pk[j] == e) bad = true;
    }
    if (bad) set_status(status, kDevErrBadIndex);
    for (int k = 0; k < K; ++k) picks[t * kPickStride + k] = bad ? -1 : pk[k];
  }
  __syncthreads();
  rank_picks(picks, R, K, E, rank, hist, lanes_of, warp_pre);
  if (t < R)
    for (int k = 0; k < K; ++k) place[u * K + k] = rank[t * kPickStride + k];
  for (int e = t; e < E; e += kChunk) chunk_hist[(int64_t)blockIdx.x * E + e] = hist[e];
}

// Σp in fixed point: a tile's Σ_t p_{t,e} (fp32, at most 128) times 2^40 is an exact integer for
// any value >= 2^-16, and integer sums do not depend on their order, so the per-expert totals are
// deterministic without a fixed summation tree (and without fp64, which is slow on this GPU).
constexpr float kPsumScale = 1099511627776.0f;  // 2^40

__device__ __forceinline__ long long warp_sum_ll(long long v) {
#pragma unroll
  for (int d = 16; d; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
  return v;
}

// One block per expert e:
//   chunk_base[c][e] = Σ_{c'<c} hist[c'][e]; count_e = Σ_c hist[c][e]   (one chunk per thread per
//   pass, a block scan per pass)
//   term_e = (count_e/(T'·K))·(Σ_c psum[c][e] / T')   when psum is given
// The last block (ticket): offsets = exclusive scan over experts of min(count_e, C); aux loss =
// α·E·Σ_e term_e (a fixed-order tree over the experts); the ticket is reset for the next call.
__global__ void __launch_bounds__(kScanThreads)
scan_kernel(const int32_t* __restrict__ hist, int64_t nchunks, int E, int64_t C, const float* __restrict__ psum,
            int64_t Tu, int K, float alpha, int32_t* __restrict__ chunk_base, int32_t* __restrict__ counts_ws,
            int32_t* __restrict__ offsets_ws, int32_t* counts_out, int32_t* offsets_out, float* terms,
            unsigned int* ticket, float* aux_out, const int32_t* __restrict__ qbase, int64_t* __restrict__ cap_out) {
  __shared__ int warp_tot[kScanThreads / 32];
  __shared__ long long warp_p[kScanThreads / 32];
  __shared__ int excl[kMaxExperts + 1];
  __shared__ float tv[kMaxExperts];
  __shared__ bool last;
  griddep_launch_dependents();
  griddep_wait();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int e = blockIdx.x;
  int carry = 0;
  long long pfx = 0;
  for (int64_t c0 = 0; c0 < nchunks; c0 += kScanThreads) {
    const int64_t c = c0 + tid;
    const int v = c < nchunks ? hist[c * E + e] : 0;
    if (psum && c < nchunks) pfx += __float2ll_rn(psum[c * E + e] * kPsumScale);
    int incl = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += t;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    int before = 0, pass_total = 0;
#pragma unroll
    for (int w = 0; w < kScanThreads / 32; ++w) {
      before += (w < warp) ? warp_tot[w] : 0;
      pass_total += warp_tot[w];
    }
    if (c < nchunks) chunk_base[c * E + e] = carry + before + incl - v;
    carry += pass_total;
    __syncthreads();
  }
  if (psum) {
    pfx = warp_sum_ll(pfx);
    if (lane == 0) warp_p[warp] = pfx;
    __syncthreads();
  }
  if (tid == 0) {
    counts_ws[e] = carry;
    if (counts_out) counts_out[e] = carry;
    // a shard of a larger batch: this expert's queue already holds qbase[e] picks of earlier ranks,
    // so the capacity left here is C - qbase[e]
    if (qbase) cap_out[e] = C == INT64_MAX ? C : C - (int64_t)qbase[e];
    if (psum) {
      long long P = 0;
      for (int w = 0; w < kScanThreads / 32; ++w) P += warp_p[w];
      const float Pe = __ll2float_rn(P) * (1.0f / kPsumScale);
      terms[e] = Tu > 0 ? ((float)carry / ((float)Tu * (float)K)) * (Pe / (float)Tu) : 0.0f;
    }
    __threadfence();
    last = atomicAdd(ticket, 1u) == (unsigned)(E - 1);
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  if (tid < 32) {  // warp scan of kept rows over E <= 256 experts (8 per lane)
    const volatile int32_t* cnt = counts_ws;
    int loc[8], sum = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int ee = lane * 8 + j;
      loc[j] = sum;
      if (ee < E) {
        const int64_t n = cnt[ee];
        int64_t cap = (qbase && C != INT64_MAX) ? C - (int64_t)qbase[ee] : C;
        if (cap < 0) cap = 0;
        sum += (int)(n < cap ? n : cap);
      }
    }
    int incl = sum;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += t;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int ee = lane * 8 + j;
      if (ee < E) excl[ee] = incl - sum + loc[j];
    }
    if (lane == 31) excl[E] = incl;
  }
  if (psum && aux_out) {
    const volatile float* vt = terms;
    for (int i = tid; i < kMaxExperts; i += kScanThreads) tv[i] = i < E ? vt[i] : 0.0f;
  }
  __syncthreads();
  for (int i = tid; i <= E; i += kScanThreads) {
    offsets_ws[i] = excl[i];
    if (offsets_out) offsets_out[i] = excl[i];
  }
  if (psum && aux_out) {  // pairwise tree over the 256 slots (fixed order), then the scale
    for (int s = kMaxExperts / 2; s; s >>= 1) {
      if (tid < s) tv[tid] += tv[tid + s];
      __syncthreads();
    }
    if (tid == 0) *aux_out = alpha * (float)E * tv[0];
  }
  if (tid == 0) *ticket = 0u;
}

// One warp per unit: slots of its picks, then its x row (row_vecs 16-byte vectors) copied to each
// kept slot. `slot_of` holds the picks' places within their chunk on entry and the packed rows (or
// -1) on exit; each entry is read and rewritten by the same lane. Rows past the kept total get
// row_token -1.
__global__ void __launch_bounds__(256)
pack_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ idx, const int32_t* __restrict__ chunk_base,
            const int32_t* __restrict__ offsets, int64_t Tu, int K, int E, int64_t C, const int64_t* __restrict__ cap_e,
            int chunk_shift, int row_vecs, int64_t rows, int32_t* __restrict__ slot_of, int32_t* __restrict__ row_token,
            uint4* __restrict__ x_packed, uint4* __restrict__ y_zero, uint32_t* __restrict__ arrivals,
            int arrivals_per_unit) {
  griddep_launch_dependents();
  griddep_wait();
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t u = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; u < Tu; u += nwarps) {
    int slot = -1;
    if (lane < K) {
      const int e = idx[u * K + lane];
      const int pl = slot_of[u * K + lane];
      if (pl >= 0 && e >= 0 && e < E) {
        const int64_t place = (int64_t)chunk_base[(u >> chunk_shift) * E + e] + pl;
        if (place < (cap_e ? cap_e[e] : C)) slot = offsets[e] + (int)place;
      }
      slot_of[u * K + lane] = slot;
      if (slot >= 0) row_token[slot] = (int32_t)u;
    }
    // combine folded into the down GEMM: its arrival counters start at zero, and a unit none of
    // whose picks was kept gets y = 0 here (no GEMM row writes it)
    if (arrivals != nullptr)
      for (int i = lane; i < arrivals_per_unit; i += 32) arrivals[u * arrivals_per_unit + i] = 0u;
    if (y_zero != nullptr && __ballot_sync(0xffffffffu, slot >= 0) == 0u)
      for (int v = lane; v < row_vecs; v += 32) y_zero[u * row_vecs + v] = make_uint4(0u, 0u, 0u, 0u);
    const uint4* src = x + u * row_vecs;
    for (int v0 = 0; v0 < row_vecs; v0 += 32 * 8) {
      uint4 buf[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int v = v0 + 32 * j + lane;
        if (v < row_vecs) buf[j] = __ldg(src + v);
      }
      for (int k = 0; k < K; ++k) {
        const int s = __shfl_sync(0xffffffffu, slot, k);
        if (s < 0) continue;
        uint4* dst = x_packed + (int64_t)s * row_vecs;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int v = v0 + 32 * j + lane;
          if (v < row_vecs) dst[v] = buf[j];
        }
      }
    }
  }
  const int64_t kept = offsets[E];
  const int64_t nthr = (int64_t)gridDim.x * blockDim.x;
  for (int64_t r = kept + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < rows; r += nthr) row_token[r] = -1;
}

// The same for rows whose byte length is not a multiple of 16 (or unaligned buffers): byte copies.
__global__ void __launch_bounds__(256)
pack_bytes_kernel(const unsigned char* __restrict__ x, const int32_t* __restrict__ idx,
                  const int32_t* __restrict__ chunk_base, const int32_t* __restrict__ offsets, int64_t Tu, int K,
                  int E, int64_t C, const int64_t* __restrict__ cap_e, int chunk_shift, int64_t row_bytes, int64_t rows,
                  int32_t* __restrict__ slot_of, int32_t* __restrict__ row_token, unsigned char* __restrict__ x_packed) {
  griddep_launch_dependents();
  griddep_wait();
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t u = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; u < Tu; u += nwarps) {
    int slot = -1;
    if (lane < K) {
      const int e = idx[u * K + lane];
      const int pl = slot_of[u * K + lane];
      if (pl >= 0 && e >= 0 && e < E) {
        const int64_t place = (int64_t)chunk_base[(u >> chunk_shift) * E + e] + pl;
        if (place < (cap_e ? cap_e[e] : C)) slot = offsets[e] + (int)place;
      }
      slot_of[u * K + lane] = slot;
      if (slot >= 0) row_token[slot] = (int32_t)u;
    }
    for (int k = 0; k < K; ++k) {
      const int s = __shfl_sync(0xffffffffu, slot, k);
      if (s < 0) continue;
      for (int64_t b = lane; b < row_bytes; b += 32) x_packed[(int64_t)s * row_bytes + b] = x[u * row_bytes + b];
    }
  }
  const int64_t kept = offsets[E];
  const int64_t nthr = (int64_t)gridDim.x * blockDim.x;
  for (int64_t r = kept + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < rows; r += nthr) row_token[r] = -1;
}

}  // namespace

cudaError_t launch_scan(const Problem& p, int64_t nchunks, const int32_t* hist, const float* psum,
                        int32_t* chunk_base, int32_t* counts_ws, int32_t* offsets_ws, int32_t* counts_out,
                        int32_t* offsets_out, float* terms, unsigned int* ticket, float* aux_out, cudaStream_t s,
                        bool pdl, const int32_t* qbase, int64_t* cap_out) {
  return launch_kernel(scan_kernel, dim3((unsigned)p.E), dim3(kScanThreads), 0, s, 1, pdl, hist, nchunks, p.E, p.C,
                       psum, p.Tu, p.K, p.cfg.aux_alpha, chunk_base, counts_ws, offsets_ws, counts_out, offsets_out,
                       terms, ticket, aux_out, qbase, cap_out);
}

cudaError_t launch_pack(const Problem& p, const void* x, const int32_t* idx, int chunk_shift, const int32_t* chunk_base,
                        const int32_t* offsets, int32_t* slot_of, int32_t* row_token, void* x_packed, cudaStream_t s,
                        bool pdl, const int64_t* cap_e, void* y_zero, uint32_t* arrivals) {
  const int64_t row_bytes = (int64_t)p.hu * (int64_t)p.elt;
  const int sms = device_sm_count();
  int64_t blocks = (p.Tu + 7) / 8;  // a warp per unit
  if (blocks > (int64_t)sms * 8) blocks = (int64_t)sms * 8;
  const int64_t tail_blocks = (p.rows + 255) / 256;
  if (blocks < 1) blocks = tail_blocks < 1 ? 1 : (tail_blocks < sms ? tail_blocks : sms);
  const bool vec = row_bytes % 16 == 0 && (reinterpret_cast<uintptr_t>(x) & 15) == 0 &&
                   (reinterpret_cast<uintptr_t>(x_packed) & 15) == 0;
  if (vec && (reinterpret_cast<uintptr_t>(y_zero) & 15) == 0)
    return launch_kernel(pack_kernel, dim3((unsigned)blocks), dim3(256), 0, s, 1, pdl, static_cast<const uint4*>(x),
                         idx, chunk_base, offsets, p.Tu, p.K, p.E, p.C, cap_e, chunk_shift, (int)(row_bytes / 16), p.rows,
                         slot_of, row_token, static_cast<uint4*>(x_packed), static_cast<uint4*>(y_zero), arrivals,
                         p.hu / 32);
  if (y_zero != nullptr || arrivals != nullptr) return cudaErrorInvalidValue;  // only the vector pack prepares the folded combine
  return launch_kernel(pack_bytes_kernel, dim3((unsigned)blocks), dim3(256), 0, s, 1, pdl,
                       static_cast<const unsigned char*>(x), idx, chunk_base, offsets, p.Tu, p.K, p.E, p.C, cap_e,
                       chunk_shift, row_bytes, p.rows, slot_of, row_token, static_cast<unsigned char*>(x_packed));
}

cudaError_t launch_dispatch_from_idx(const Problem& p, const void* x, const int32_t* idx, int32_t* counts_out,
                                     int32_t* offsets_out, int32_t* slot_of, int32_t* row_token, void* x_packed,
                                     const DispatchScratch& sc, cudaStream_t s) {
  const int64_t nch = p.nchunks;
  cudaError_t e = cudaSuccess;
  bool pdl = false;
  if (nch > 0) {
    e = launch_kernel(chunk_rank_kernel, dim3((unsigned)nch), dim3(kChunk), 0, s, 1, false, idx, p.Tu, p.K, p.E,
                      slot_of, sc.chunk_hist, sc.status);
    if (e != cudaSuccess) return e;
    pdl = true;
  }
  e = launch_scan(p, nch, sc.chunk_hist, nullptr, sc.chunk_base, sc.counts, sc.offsets, counts_out, offsets_out,
                  nullptr, sc.ticket, nullptr, s, pdl, sc.qbase, sc.cap);
  if (e != cudaSuccess) return e;
  if (p.rows == 0) return cudaSuccess;
  return launch_pack(p, x, idx, kChunkShift, sc.chunk_base, sc.offsets, slot_of, row_token, x_packed, s, true,
                     sc.qbase ? sc.cap : nullptr);
}

}  // namespace moe
