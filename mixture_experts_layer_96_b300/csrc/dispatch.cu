// Dispatch: capacity drop and pack of the units per expert.
//   [Lesson 10 "专家并行 EP", §3 step 1: pack the token vectors per destination expert;
//    §4: capacity C = CF·K·T/E, picks past C dropped]
//
// The queue order inside an expert is unit order (a unit's K picks are distinct), so the place of
// pick (t,k) in expert e's queue is the number of earlier units that picked e: a stable counting
// sort. Four kernels, no atomics whose order matters and no inter-block waits:
//   1. hist:   per chunk of 256 units, picks per expert (and index validation)
//   2. scan:   a block per expert: per-expert totals (pre-drop counts) and each chunk's base in
//              each queue; the last block scans the kept rows n_e = min(count, C) into offsets
//   3. rank:   per chunk, each pick's place = chunk base + earlier warps' picks + earlier lanes'
//              picks (a per-warp bitmask of the lanes that picked each expert); writes slot_of,
//              row_token and -1 into row_token past the kept rows
//   4. gather: x_packed[r] = x[row_token[r]] with 16-byte vector copies, one warp per row
#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {

constexpr int kWarps = kChunk / 32;

__global__ void __launch_bounds__(kChunk)
dispatch_hist_kernel(const int32_t* __restrict__ idx, int64_t Tu, int K, int E,
                     int32_t* __restrict__ chunk_hist, uint32_t* status) {
  __shared__ int cnt[kMaxExperts];
  const int tid = threadIdx.x;
  for (int e = tid; e < E; e += kChunk) cnt[e] = 0;
  __syncthreads();
  const int64_t u = (int64_t)blockIdx.x * kChunk + tid;
  if (u < Tu) {
    int picks[kMaxTopK];
    bool bad = false;
    for (int k = 0; k < K; ++k) {
      const int e = idx[u * K + k];
      picks[k] = e;
      if (e < 0 || e >= E) bad = true;
      for (int j = 0; j < k; ++j)
        if (picks[j] == e) bad = true;
    }
    if (bad) set_status(status, kDevErrBadIndex);
    else
      for (int k = 0; k < K; ++k) atomicAdd(&cnt[picks[k]], 1);
  }
  __syncthreads();
  for (int e = tid; e < E; e += kChunk) chunk_hist[(int64_t)blockIdx.x * E + e] = cnt[e];
}

// One block per expert: an exclusive scan of the expert's column of chunk counts (one chunk per
// thread per pass, a block scan per pass) gives each chunk's base in the expert's queue and the
// pre-drop count. The last block to finish (ticket) scans the kept rows n_e = min(count_e, C)
// over experts into the offsets and resets the ticket. Integer sums, so the result does not
// depend on which block finishes last.
constexpr int kScanThreads = 256;

__global__ void __launch_bounds__(kScanThreads)
dispatch_scan_kernel(const int32_t* __restrict__ chunk_hist, int64_t nchunks, int E, int64_t C,
                     int32_t* __restrict__ chunk_base, int32_t* __restrict__ counts_ws,
                     int32_t* __restrict__ offsets_ws, int32_t* counts_out, int32_t* offsets_out,
                     unsigned int* ticket) {
  __shared__ int warp_tot[kScanThreads / 32];
  __shared__ int excl[kMaxExperts + 1];
  __shared__ bool last;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int e = blockIdx.x;
  int carry = 0;
  for (int64_t c0 = 0; c0 < nchunks; c0 += kScanThreads) {
    const int64_t c = c0 + tid;
    const int v = c < nchunks ? chunk_hist[c * E + e] : 0;
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
  if (tid == 0) {
    counts_ws[e] = carry;
    if (counts_out) counts_out[e] = carry;
    __threadfence();
    last = atomicAdd(ticket, 1u) == (unsigned)(E - 1);
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  if (tid < 32) {  // warp scan of kept over E <= 256 (8 per lane)
    const volatile int32_t* cnt = counts_ws;
    int loc[8], sum = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int ee = lane * 8 + j;
      loc[j] = sum;
      if (ee < E) {
        const int64_t n = cnt[ee];
        sum += (int)(n < C ? n : C);
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
  __syncthreads();
  for (int i = tid; i <= E; i += kScanThreads) {
    offsets_ws[i] = excl[i];
    if (offsets_out) offsets_out[i] = excl[i];
  }
  if (tid == 0) *ticket = 0u;
}

__global__ void __launch_bounds__(kChunk)
dispatch_rank_kernel(const int32_t* __restrict__ idx, int64_t Tu, int K, int E, int64_t C,
                     const int32_t* __restrict__ chunk_base, const int32_t* __restrict__ offsets,
                     int32_t* __restrict__ slot_of, int32_t* __restrict__ row_token, int64_t rows) {
  __shared__ uint32_t lanes_of[kWarps][kMaxExperts];  // bit l: lane l of the warp picked e
  __shared__ int warp_pre[kWarps][kMaxExperts];       // picks of e by earlier warps of the chunk
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < kWarps * E; i += kChunk) lanes_of[i / E][i % E] = 0u;
  __syncthreads();
  const int64_t u = (int64_t)blockIdx.x * kChunk + tid;
  int picks[kMaxTopK];
  bool ok = u < Tu;
  if (ok) {
    for (int k = 0; k < K; ++k) {
      const int e = idx[u * K + k];
      picks[k] = e;
      if (e < 0 || e >= E) ok = false;
      for (int j = 0; j < k; ++j)
        if (picks[j] == e) ok = false;
    }
    if (ok)
      for (int k = 0; k < K; ++k) atomicOr(&lanes_of[warp][picks[k]], 1u << lane);
  }
  __syncthreads();
  for (int e = tid; e < E; e += kChunk) {
    int run = 0;
    for (int w = 0; w < kWarps; ++w) {
      warp_pre[w][e] = run;
      run += __popc(lanes_of[w][e]);
    }
  }
  __syncthreads();
  if (u < Tu) {
    for (int k = 0; k < K; ++k) {
      int32_t slot = -1;
      if (ok) {
        const int e = picks[k];
        const int64_t place = (int64_t)chunk_base[(int64_t)blockIdx.x * E + e] + warp_pre[warp][e] +
                              __popc(lanes_of[warp][e] & lanemask_lt());
        if (place < C) {
          slot = (int32_t)(offsets[e] + place);
          row_token[slot] = (int32_t)u;
        }
      }
      slot_of[u * K + k] = slot;
    }
  }
  // rows past the kept total carry no unit
  const int64_t kept = offsets[E];
  for (int64_t r = kept + (int64_t)blockIdx.x * kChunk + tid; r < rows; r += (int64_t)gridDim.x * kChunk)
    row_token[r] = -1;
}

// x_packed[r] = x[row_token[r]] for r < offsets[E]; rows are `row_vecs` 16-byte vectors. The
// packed rows are one flat array of vectors; each warp copies 128 consecutive vectors per step
// (vector wb + 32·j + lane, j = 0..3), so every load and store instruction covers 512 contiguous
// bytes, with four independent loads in flight per lane whatever the row length.
__global__ void __launch_bounds__(256)
dispatch_gather_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ row_token,
                       const int32_t* __restrict__ offsets, int E, int64_t row_vecs,
                       uint4* __restrict__ x_packed) {
  const uint32_t rv = (uint32_t)row_vecs;
  const uint64_t total = (uint64_t)offsets[E] * rv;
  const uint64_t nwarps = (uint64_t)gridDim.x * (blockDim.x >> 5);
  const uint32_t lane = threadIdx.x & 31u;
  for (uint64_t wb = ((uint64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * 128u; wb < total;
       wb += nwarps * 128u) {
    uint4 v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint64_t i = wb + 32u * j + lane;
      if (i < total) {
        const uint64_t r = i / rv;
        v[j] = __ldg(x + (int64_t)__ldg(row_token + r) * row_vecs + (i - r * rv));
      }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint64_t i = wb + 32u * j + lane;
      if (i < total) x_packed[i] = v[j];
    }
  }
}

// Scalar fallback for rows whose byte length is not a multiple of 16.
__global__ void __launch_bounds__(256)
dispatch_gather_scalar_kernel(const unsigned char* __restrict__ x, const int32_t* __restrict__ row_token,
                              const int32_t* __restrict__ offsets, int E, int64_t row_bytes,
                              unsigned char* __restrict__ x_packed) {
  const int64_t kept = offsets[E];
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < kept; r += warps) {
    const int64_t t = row_token[r];
    for (int64_t b = threadIdx.x & 31; b < row_bytes; b += 32) x_packed[r * row_bytes + b] = x[t * row_bytes + b];
  }
}

cudaError_t launch_dispatch(const Problem& p, const void* x, const int32_t* idx, int32_t* counts,
                            int32_t* offsets, int32_t* slot_of, int32_t* row_token, void* x_packed,
                            void* ws, cudaStream_t s) {
  const WsLayout L = ws_layout(p);
  int32_t* chunk_hist = ws_ptr<int32_t>(ws, L.chunk_hist);
  int32_t* chunk_base = ws_ptr<int32_t>(ws, L.chunk_base);
  int32_t* counts_ws = ws_ptr<int32_t>(ws, L.counts);
  int32_t* offsets_ws = ws_ptr<int32_t>(ws, L.offsets);
  uint32_t* status = ws_ptr<uint32_t>(ws, L.status);
  const unsigned nch = (unsigned)(p.nchunks > 0 ? p.nchunks : 0);
  if (nch > 0) {
    dispatch_hist_kernel<<<nch, kChunk, 0, s>>>(idx, p.Tu, p.K, p.E, chunk_hist, status);
    note_launch();
  }
  dispatch_scan_kernel<<<p.E, kScanThreads, 0, s>>>(chunk_hist, p.nchunks, p.E, p.C, chunk_base,
                                                    counts_ws, offsets_ws, counts, offsets,
                                                    ws_ptr<unsigned int>(ws, L.status + 8));
  note_launch();
  const int64_t rows = p.rows;
  const unsigned rank_blocks = nch > 0 ? nch : 1;
  dispatch_rank_kernel<<<rank_blocks, kChunk, 0, s>>>(idx, p.Tu, p.K, p.E, p.C, chunk_base,
                                                      offsets_ws, slot_of, row_token, rows);
  note_launch();
  if (rows > 0) {
    const int64_t row_bytes = (int64_t)p.hu * (int64_t)p.elt;
    const int sms = device_sm_count();
    int64_t blocks = (rows * (row_bytes / 16) + 1023) / 1024;
    const int64_t cap = (int64_t)sms * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    if (row_bytes % 16 == 0 && (reinterpret_cast<uintptr_t>(x) & 15) == 0 &&
        (reinterpret_cast<uintptr_t>(x_packed) & 15) == 0) {
      dispatch_gather_kernel<<<(unsigned)blocks, 256, 0, s>>>(
          static_cast<const uint4*>(x), row_token, offsets_ws, p.E, row_bytes / 16,
          static_cast<uint4*>(x_packed));
    } else {
      dispatch_gather_scalar_kernel<<<(unsigned)blocks, 256, 0, s>>>(
          static_cast<const unsigned char*>(x), row_token, offsets_ws, p.E, row_bytes,
          static_cast<unsigned char*>(x_packed));
    }
    note_launch();
  }
  return cudaGetLastError();
}

}  // namespace moe
