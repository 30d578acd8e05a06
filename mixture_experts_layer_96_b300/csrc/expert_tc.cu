// Expert FFN on the 5th-generation tensor cores (bf16 in, fp32 accumulate in TMEM).
//   [Lesson 10 "专家并行 EP", §3 step 2: the units gathered per local expert go through a grouped
//    GEMM; the expert is FFN_e(x) = W2_e·(silu(W1_e·x) ⊙ W3_e·x)]
//
// Two launches of one persistent, warp-specialised kernel:
//   gate/up:  H[r, n0:n0+128] = silu(X_e·W1_eᵀ) ⊙ (X_e·W3_eᵀ)   (tile N = 128 gate + 128 up columns)
//   down:     Y[r, n0:n0+256] = H_e·W2_eᵀ
// Tile 128 x 256 x 64, 4-stage TMA ring (48 KB/stage, 128-byte swizzle), two 256-column TMEM
// accumulators so the epilogue of one tile overlaps the main loop of the next.
//   warp 0     TMA producer (one lane)
//   warp 1     TMEM allocator + MMA issuer (one lane issues tcgen05.mma, commits to mbarriers)
//   warps 2-5  epilogue: tcgen05.ld → SwiGLU/convert → bf16 stores (rows masked to the expert)
// Tiles run expert by expert, n-tile by n-tile, with the m-tiles of an expert adjacent so the
// CTAs working at the same time share each weight tile through L2. The schedule comes from the
// device-side offsets: no host sync between dispatch and this kernel. Every wait is bounded.
#include <stdlib.h>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {

constexpr int kBM = 128, kBN = 256, kBK = 64, kStages = 4;
constexpr int kABytes = kBM * kBK * 2;           // 16 KB
constexpr int kBBytes = kBN * kBK * 2;           // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;   // 48 KB
constexpr int kTcThreads = 192;
constexpr int kTmemCols = 512;                   // two 256-column fp32 accumulators
constexpr size_t kTcSmem = (size_t)kStages * kStageBytes + 1024;
constexpr uint32_t kIdesc = idesc_bf16_f32(kBM, kBN);

enum { kEpiSwiGLU = 0, kEpiPlain = 1 };

struct TcParams {
  const int32_t* offsets;  // [E+1]
  int E;
  int K;                   // reduction length
  int w_rows;              // weight rows per expert (d_ff for gate/up, h' for down)
  int n_tiles;             // N tiles per expert
  int n_out;               // output row length
  int64_t rows_cap;        // packed-row capacity
  __nv_bfloat16* out;
  uint32_t* status;
};

template <int EPI>
__global__ void __launch_bounds__(kTcThreads, 1)
expert_gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                      const __grid_constant__ CUtensorMap tmB1, TcParams p) {
  extern __shared__ unsigned char smem_dyn[];
  __shared__ int s_off[kMaxExperts + 1];
  __shared__ int s_pre[kMaxExperts + 1];
  __shared__ __align__(8) uint64_t s_bar[2 * kStages + 5];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_ok;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = (smem_addr(smem_dyn) + 1023u) & ~1023u;
  const uint32_t bar0 = smem_addr(s_bar);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * kStages + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * kStages + 2 + a); };
  const uint32_t done_bar = bar0 + 8u * (2 * kStages + 4);

  if (warp == 0) {
    const bool ok = warp_tile_prefix(p.offsets, p.E, kBM, p.rows_cap, s_off, s_pre);
    if (lane == 0) {
      s_ok = ok ? 1 : 0;
      s_abort = 0;
      if (!ok && blockIdx.x == 0) set_status(p.status, kDevErrBadOffsets);
      for (int s = 0; s < kStages; ++s) {
        mbar_init(full_bar(s), 1);
        mbar_init(empty_bar(s), 1);
      }
      for (int a = 0; a < 2; ++a) {
        mbar_init(tfull_bar(a), 1);
        mbar_init(tempty_bar(a), 4);
      }
      mbar_init(done_bar, 1);
      fence_mbar_init();
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB0);
      if (EPI == kEpiSwiGLU) tma_prefetch_desc(&tmB1);
    }
    __syncwarp();
  } else if (warp == 1) {
    tmem_alloc(smem_addr(&s_tmem), kTmemCols);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = s_tmem;
  const bool valid = s_ok != 0;
  const int total = valid ? s_pre[p.E] * p.n_tiles : 0;
  const int nkb = (p.K + kBK - 1) / kBK;
  volatile int* abort_flag = &s_abort;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t filled = 0;  // bit s: stage s has been filled at least once
      uint32_t last_parity = 0;
      bool aborted = false;
      for (int tile = blockIdx.x; tile < total && !aborted; tile += gridDim.x) {
        int e, mt, nt;
        decode_tile(tile, s_pre, p.E, p.n_tiles, e, mt, nt);
        const int a_row = s_off[e] + mt * kBM;
        const int b_row = e * p.w_rows + nt * (EPI == kEpiSwiGLU ? kBN / 2 : kBN);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag)) { aborted = true; break; }
          const uint32_t sa = sbase + stage * kStageBytes, sb = sa + kABytes;
          mbar_arrive_expect_tx(full_bar(stage), kStageBytes);
          tma_load_2d(sa, &tmA, full_bar(stage), kb * kBK, a_row);
          if (EPI == kEpiSwiGLU) {
            tma_load_2d(sb, &tmB0, full_bar(stage), kb * kBK, b_row);
            tma_load_2d(sb + kBBytes / 2, &tmB1, full_bar(stage), kb * kBK, b_row);
          } else {
            tma_load_2d(sb, &tmB0, full_bar(stage), kb * kBK, b_row);
          }
          filled |= 1u << stage;
          last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
      }
      if (aborted) {
        s_abort = 1;
        set_status(p.status, kDevErrTimeout);
        // let copies already issued land before the CTA's shared memory goes away
        for (int s = 0; s < kStages; ++s)
          if ((filled >> s) & 1u) mbar_wait(full_bar(s), (last_parity >> s) & 1u, nullptr, 50000000ull);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool aborted = false;
      int it = 0;
      for (int tile = blockIdx.x; tile < total && !aborted; tile += gridDim.x, ++it) {
        const int acc = it & 1;
        const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
        if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag)) { aborted = true; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * kBN);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(full_bar(stage), phase, abort_flag)) { aborted = true; break; }
          tc_fence_after();
          const uint32_t sa = sbase + stage * kStageBytes, sb = sa + kABytes;
          const uint64_t ad = sdesc_kmajor_sw128(sa), bd = sdesc_kmajor_sw128(sb);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)  // 16 bf16 = 32 bytes per MMA along K
            umma_bf16(d_tmem, ad + (uint64_t)(2 * k), bd + (uint64_t)(2 * k), kIdesc,
                      (kb > 0 || k > 0) ? 1u : 0u);
          umma_commit(empty_bar(stage));
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
        if (aborted) break;
        umma_commit(tfull_bar(acc));
      }
      if (aborted) {
        s_abort = 1;
        set_status(p.status, kDevErrTimeout);
      }
      // every MMA this thread issued has completed before TMEM is released
      umma_commit(done_bar);
      mbar_wait(done_bar, 0, nullptr, 50000000ull);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..5)
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    int it = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++it) {
      int e, mt, nt;
      decode_tile(tile, s_pre, p.E, p.n_tiles, e, mt, nt);
      const int acc = it & 1;
      const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
      if (!mbar_wait(tfull_bar(acc), acc_phase, abort_flag)) {
        if (lane == 0) { s_abort = 1; set_status(p.status, kDevErrTimeout); }
        break;
      }
      tc_fence_after();
      const int rows_e = s_off[e + 1] - s_off[e];
      const int r_local = mt * kBM + q * 32 + lane;
      const bool row_ok = r_local < rows_e;
      __nv_bfloat16* orow = p.out + (int64_t)(s_off[e] + r_local) * p.n_out;
      const uint32_t t_row = tmem_base + (uint32_t)(acc * kBN) + ((uint32_t)(q * 32) << 16);
      if (EPI == kEpiSwiGLU) {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t g[32], u[32];
          tmem_ld_32x32b_x32(t_row + c * 32, g);
          tmem_ld_32x32b_x32(t_row + 128 + c * 32, u);
          tmem_ld_wait();
          const int col = nt * 128 + c * 32;
          if (row_ok && col < p.n_out) {
            uint32_t pk[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float h0 = silu_f32(__uint_as_float(g[2 * j])) * __uint_as_float(u[2 * j]);
              const float h1 = silu_f32(__uint_as_float(g[2 * j + 1])) * __uint_as_float(u[2 * j + 1]);
              pk[j] = pack_bf16x2(h0, h1);
            }
            uint4* dst = reinterpret_cast<uint4*>(orow + col);
#pragma unroll
            for (int j = 0; j < 4; ++j) dst[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
          }
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(t_row + c * 32, v);
          tmem_ld_wait();
          const int col = nt * kBN + c * 32;
          if (row_ok && col < p.n_out) {
            uint32_t pk[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) pk[j] = pack_bf16x2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
            uint4* dst = reinterpret_cast<uint4*>(orow + col);
#pragma unroll
            for (int j = 0; j < 4; ++j) dst[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar(acc));
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ------------------------------------------------------------------------------------------------
// CTA-pair variant (cta_group::2): a cluster of two CTAs computes a 256 x 256 tile. Each CTA loads
// its 128 rows of A and its 128 rows of B (gate/up: CTA 0 the W1 rows, CTA 1 the W3 rows; down:
// the two halves of the 256 output columns) into its own shared memory; one thread of CTA 0
// issues the pair MMA (M = 256, N = 256, K = 16), which leaves rows 0-127 of D in CTA 0's TMEM and
// rows 128-255 in CTA 1's. Per SM this halves the B bytes fetched and read from shared memory per
// FLOP compared with the single-CTA 128 x 256 tile.
//   barriers (same offsets in both CTAs):
//   full[s]   CTA 0 only: its producer arms it with both CTAs' bytes; both CTAs' TMA complete on it
//   empty[s]  both: the MMA commit multicasts to both CTAs when the stage's MMAs are done
//   tfull[a]  both: MMA commit multicast when accumulator a is complete
//   tempty[a] CTA 0 only: 4 epilogue warps of each CTA arrive (remote arrive from CTA 1)
constexpr int kPairBM = 256, kPairStages = 6;
constexpr int kPairHalf = 128 * kBK * 2;                 // 16 KB: 128 rows x 64 bf16
constexpr int kPairStageBytes = 2 * kPairHalf;           // A half + B half per CTA
constexpr size_t kPairSmem = (size_t)kPairStages * kPairStageBytes + 1024;
constexpr uint32_t kIdescPair = idesc_bf16_f32(kPairBM, kBN);

template <int EPI>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kTcThreads, 1)
expert_gemm_tc_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                           const __grid_constant__ CUtensorMap tmB1, TcParams p) {
  extern __shared__ unsigned char smem_dyn[];
  __shared__ int s_off[kMaxExperts + 1];
  __shared__ int s_pre[kMaxExperts + 1];
  __shared__ __align__(8) uint64_t s_bar[2 * kPairStages + 5];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_ok;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const uint32_t sbase = (smem_addr(smem_dyn) + 1023u) & ~1023u;
  const uint32_t bar0 = smem_addr(s_bar);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kPairStages + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * kPairStages + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * kPairStages + 2 + a); };
  const uint32_t done_bar = bar0 + 8u * (2 * kPairStages + 4);

  if (warp == 0) {
    const bool ok = warp_tile_prefix(p.offsets, p.E, kPairBM, p.rows_cap, s_off, s_pre);
    if (lane == 0) {
      s_ok = ok ? 1 : 0;
      s_abort = 0;
      if (!ok && blockIdx.x == 0) set_status(p.status, kDevErrBadOffsets);
      for (int s = 0; s < kPairStages; ++s) {
        mbar_init(full_bar(s), 1);
        mbar_init(empty_bar(s), 1);
      }
      for (int a = 0; a < 2; ++a) {
        mbar_init(tfull_bar(a), 1);
        mbar_init(tempty_bar(a), 8);
      }
      mbar_init(done_bar, 1);
      fence_mbar_init();
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB0);
      if (EPI == kEpiSwiGLU) tma_prefetch_desc(&tmB1);
    }
    __syncwarp();
  } else if (warp == 1) {
    tmem_alloc_pair(smem_addr(&s_tmem), kTmemCols);
    tmem_relinquish_pair();
    tc_fence_before();
  }
  __syncthreads();
  cluster_sync_all();  // the peer's barriers are initialised before any remote arrive or TMA
  tc_fence_after();
  const uint32_t tmem_base = s_tmem;
  const int total = s_ok ? s_pre[p.E] * p.n_tiles : 0;
  const int nkb = (p.K + kBK - 1) / kBK;
  const int cid = blockIdx.x >> 1, ncl = gridDim.x >> 1;
  volatile int* abort_flag = &s_abort;
  const uint32_t peer_abort = mapa_shared(smem_addr(&s_abort), rank ^ 1u);
  auto abort_both = [&]() {
    s_abort = 1;
    st_shared_cluster_u32(peer_abort, 1u);
    set_status(p.status, kDevErrTimeout);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      const uint32_t full0_leader = mapa_shared(full_bar(0), 0);
      const CUtensorMap* mb = (EPI == kEpiSwiGLU && !leader) ? &tmB1 : &tmB0;
      int stage = 0;
      uint32_t phase = 0, filled = 0, last_parity = 0;
      bool aborted = false;
      for (int tile = cid; tile < total && !aborted; tile += ncl) {
        int e, mt, nt;
        decode_tile(tile, s_pre, p.E, p.n_tiles, e, mt, nt);
        const int a_row = s_off[e] + mt * kPairBM + (int)rank * 128;
        const int b_row = (EPI == kEpiSwiGLU) ? e * p.w_rows + nt * (kBN / 2)
                                              : e * p.w_rows + nt * kBN + (int)rank * 128;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag)) { aborted = true; break; }
          const uint32_t sa = sbase + stage * kPairStageBytes;
          if (leader) mbar_arrive_expect_tx(full_bar(stage), 2 * kPairStageBytes);
          const uint32_t fb = full0_leader + 8u * stage;
          tma_load_2d_pair(sa, &tmA, fb, kb * kBK, a_row);
          tma_load_2d_pair(sa + kPairHalf, mb, fb, kb * kBK, b_row);
          filled |= 1u << stage;
          last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == kPairStages) { stage = 0; phase ^= 1u; }
        }
      }
      if (aborted) {
        abort_both();
        // let copies already issued land before shared memory goes away
        if (leader) {
          for (int s = 0; s < kPairStages; ++s)
            if ((filled >> s) & 1u) mbar_wait(full_bar(s), (last_parity >> s) & 1u, nullptr, 50000000ull);
        } else {
          const uint64_t t0 = globaltimer_ns();
          while (globaltimer_ns() - t0 < 200000ull) {
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ pair MMA issuer (CTA 0)
    if (leader && lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool aborted = false;
      int it = 0;
      for (int tile = cid; tile < total && !aborted; tile += ncl, ++it) {
        const int acc = it & 1;
        const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
        if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag)) { aborted = true; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * kBN);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(full_bar(stage), phase, abort_flag)) { aborted = true; break; }
          tc_fence_after();
          const uint32_t sa = sbase + stage * kPairStageBytes;
          const uint64_t ad = sdesc_kmajor_sw128(sa), bd = sdesc_kmajor_sw128(sa + kPairHalf);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            umma_bf16_pair(d_tmem, ad + (uint64_t)(2 * k), bd + (uint64_t)(2 * k), kIdescPair,
                           (kb > 0 || k > 0) ? 1u : 0u);
          umma_commit_pair_mc(empty_bar(stage), (uint16_t)0x3);
          if (++stage == kPairStages) { stage = 0; phase ^= 1u; }
        }
        if (aborted) break;
        umma_commit_pair_mc(tfull_bar(acc), (uint16_t)0x3);
      }
      if (aborted) abort_both();
      umma_commit_pair_mc(done_bar, (uint16_t)0x1);
      mbar_wait(done_bar, 0, nullptr, 50000000ull);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..5, both CTAs)
    const int q = warp & 3;
    const uint32_t tempty_leader0 = mapa_shared(tempty_bar(0), 0);
    int it = 0;
    for (int tile = cid; tile < total; tile += ncl, ++it) {
      int e, mt, nt;
      decode_tile(tile, s_pre, p.E, p.n_tiles, e, mt, nt);
      const int acc = it & 1;
      const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
      if (!mbar_wait(tfull_bar(acc), acc_phase, abort_flag)) {
        if (lane == 0) abort_both();
        break;
      }
      tc_fence_after();
      const int rows_e = s_off[e + 1] - s_off[e];
      const int r_local = mt * kPairBM + (int)rank * 128 + q * 32 + lane;
      const bool row_ok = r_local < rows_e;
      __nv_bfloat16* orow = p.out + (int64_t)(s_off[e] + r_local) * p.n_out;
      const uint32_t t_row = tmem_base + (uint32_t)(acc * kBN) + ((uint32_t)(q * 32) << 16);
      if (EPI == kEpiSwiGLU) {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t g[32], u[32];
          tmem_ld_32x32b_x32(t_row + c * 32, g);
          tmem_ld_32x32b_x32(t_row + 128 + c * 32, u);
          tmem_ld_wait();
          const int col = nt * 128 + c * 32;
          if (row_ok && col < p.n_out) {
            uint32_t pk[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float h0 = silu_f32(__uint_as_float(g[2 * j])) * __uint_as_float(u[2 * j]);
              const float h1 = silu_f32(__uint_as_float(g[2 * j + 1])) * __uint_as_float(u[2 * j + 1]);
              pk[j] = pack_bf16x2(h0, h1);
            }
            uint4* dst = reinterpret_cast<uint4*>(orow + col);
#pragma unroll
            for (int j = 0; j < 4; ++j) dst[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
          }
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(t_row + c * 32, v);
          tmem_ld_wait();
          const int col = nt * kBN + c * 32;
          if (row_ok && col < p.n_out) {
            uint32_t pk[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) pk[j] = pack_bf16x2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
            uint4* dst = reinterpret_cast<uint4*>(orow + col);
#pragma unroll
            for (int j = 0; j < 4; ++j) dst[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader) mbar_arrive(tempty_bar(acc));
        else mbar_arrive_remote(tempty_leader0 + 8u * acc);
      }
    }
  }

  __syncthreads();
  cluster_sync_all();  // neither CTA leaves while the other may still use its barriers or TMEM
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

template <int EPI>
static cudaError_t launch_tc_pair(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                                  const TcParams& p, int grid, cudaStream_t s) {
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(expert_gemm_tc_pair_kernel<EPI>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPairSmem);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  expert_gemm_tc_pair_kernel<EPI><<<grid, kTcThreads, kPairSmem, s>>>(a, b0, b1, p);
  note_launch();
  return cudaGetLastError();
}

// Pair tiles (256 rows) pay off when experts hold many rows; with few rows per expert (fine-grained
// layers) the single-CTA 128-row tile wastes less work on ragged tails. MOE_TC_PAIR=0/1 forces it.
static bool use_pair_tiles(const Problem& p) {
  const char* v = getenv("MOE_TC_PAIR");
  if (v && (v[0] == '0' || v[0] == '1') && v[1] == 0) return v[0] == '1';
  return p.rows / p.E >= kPairBM;
}

template <int EPI>
static cudaError_t launch_tc(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                             const TcParams& p, int grid, cudaStream_t s) {
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(expert_gemm_tc_kernel<EPI>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTcSmem);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  expert_gemm_tc_kernel<EPI><<<grid, kTcThreads, kTcSmem, s>>>(a, b0, b1, p);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_expert_ffn_simt(const Problem& p, const void* x_packed, const int32_t* offsets,
                                   const void* w_gate, const void* w_up, const void* w_down,
                                   void* hidden, void* y_packed, uint32_t* status, cudaStream_t s);

cudaError_t launch_expert_ffn(const Problem& p, const void* x_packed, const int32_t* offsets,
                              const void* w_gate, const void* w_up, const void* w_down,
                              void* hidden, void* y_packed, uint32_t* status, cudaStream_t s) {
  if (!p.bf16)
    return launch_expert_ffn_simt(p, x_packed, offsets, w_gate, w_up, w_down, hidden, y_packed, status, s);
  if (p.rows == 0) return cudaSuccess;
  CUtensorMap mA, mW1, mW3, mH, mW2;
  const uint64_t rows = (uint64_t)p.rows;
  if (!encode_tmap_2d_bf16(&mA, x_packed, (uint64_t)p.hu, rows, kBK, kBM) ||
      !encode_tmap_2d_bf16(&mW1, w_gate, (uint64_t)p.hu, (uint64_t)p.E * p.d_ff, kBK, kBN / 2) ||
      !encode_tmap_2d_bf16(&mW3, w_up, (uint64_t)p.hu, (uint64_t)p.E * p.d_ff, kBK, kBN / 2) ||
      !encode_tmap_2d_bf16(&mH, hidden, (uint64_t)p.d_ff, rows, kBK, kBM) ||
      !encode_tmap_2d_bf16(&mW2, w_down, (uint64_t)p.d_ff, (uint64_t)p.E * p.hu, kBK, kBN))
    return cudaErrorInvalidValue;
  const bool pair = use_pair_tiles(p);
  CUtensorMap mW2p;
  if (pair && !encode_tmap_2d_bf16(&mW2p, w_down, (uint64_t)p.d_ff, (uint64_t)p.E * p.hu, kBK, kBN / 2))
    return cudaErrorInvalidValue;
  const int sms = device_sm_count();
  const int grid = pair ? (sms / 2) * 2 : sms;
  TcParams g;
  g.offsets = offsets;
  g.E = p.E;
  g.rows_cap = p.rows;
  g.status = status;
  // gate/up + SwiGLU → hidden
  g.K = p.hu;
  g.w_rows = p.d_ff;
  g.n_tiles = (p.d_ff + kBN / 2 - 1) / (kBN / 2);
  g.n_out = p.d_ff;
  g.out = static_cast<__nv_bfloat16*>(hidden);
  cudaError_t e = pair ? launch_tc_pair<kEpiSwiGLU>(mA, mW1, mW3, g, grid, s)
                       : launch_tc<kEpiSwiGLU>(mA, mW1, mW3, g, grid, s);
  if (e != cudaSuccess) return e;
  // down → y_packed
  g.K = p.d_ff;
  g.w_rows = p.hu;
  g.n_tiles = (p.hu + kBN - 1) / kBN;
  g.n_out = p.hu;
  g.out = static_cast<__nv_bfloat16*>(y_packed);
  return pair ? launch_tc_pair<kEpiPlain>(mH, mW2p, mW2p, g, grid, s)
              : launch_tc<kEpiPlain>(mH, mW2, mW2, g, grid, s);
}

}  // namespace moe
