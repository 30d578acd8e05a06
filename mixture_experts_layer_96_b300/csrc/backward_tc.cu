// Backward of the expert FFN on the 5th-generation tensor cores (bf16 in, fp32 accumulate in TMEM).
// The forward is FFN_e(x) = W2_e·(silu(W1_e·x) ⊙ W3_e·x) on the packed rows of expert e
//   [Lesson 10 "专家并行 EP", §3 step 2]; its gradient, with the routing held fixed, is
//   dH  = dY·W2            → dG = dH ⊙ U ⊙ silu'(G),  dU = dH ⊙ silu(G)      (mode DH)
//   dX  = dG·W1 + dU·W3                                                     (mode DX)
//   dW2 = dYᵀ·H,  dW1 = dGᵀ·X,  dW3 = dUᵀ·X   (sums over the rows of e)     (mode DW)
// with G = X·W1ᵀ, U = X·W3ᵀ, H = silu(G) ⊙ U saved by the training forward.
//
// One persistent, warp-specialised kernel (192 threads, 128 x 256 x 64 tiles, 4-stage TMA ring,
// two 256-column TMEM accumulators) serves the three modes:
//   DH, DX  M-grouped like the forward: tiles over each expert's rows, reduction over features.
//           A (dY or dG|dU) is K-major; B (W2, or W1 then W3) is read in its stored layout,
//           which is MN-major for these products (the descriptors say so; no transposed copies).
//   DW      K-grouped: for every expert a dense [M][N] tile grid, the reduction running over the
//           expert's rows. A comes K-major from a transposed copy of packed rows in which every
//           expert's rows start at a multiple of 64 and are zero-padded to one (an MN-major A ran
//           at about half the tensor rate); B is packed rows read MN-major. B's last k-block
//           usually extends into the next expert's rows, which A's zero padding cancels exactly;
//           where it runs past the last packed row, the MMA warp's 32 lanes zero those K rows in
//           shared memory before the MMA (then a proxy fence), so no stale non-finite value can
//           meet the padding. An expert without rows gets a zero tile. dW1|dW3 come out
//           transposed (M = h', N = 2·d_ff) and are stored row by row of the weight.
//   warp 0     TMA producer (one lane)
//   warp 1     TMEM allocator + MMA issuer (lane 0 issues; all lanes zero K tails in DW)
//   warps 2-5  epilogue: tcgen05.ld → SwiGLU backward / bf16 / fp32 stores
// Every wait is bounded; a timeout sets the status word and the kernel drains and returns.
#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kBM = 128, kBN = 256, kBK = 64, kStages = 4;
constexpr int kABytes = kBM * kBK * 2;           // 16 KB
constexpr int kBBytes = kBN * kBK * 2;           // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;   // 48 KB
constexpr int kMnBox = 64 * kBK * 2;             // one MN-major box: 64 MN elements x 64 K rows, 8 KB
constexpr int kThreads = 192;
constexpr int kTmemCols = 512;
constexpr size_t kSmem = (size_t)kStages * kStageBytes + 1024;

enum { kModeDH = 0, kModeDX = 1, kModeDW = 2 };

struct BwdParams {
  const int32_t* offsets;        // [E+1] packed-row offsets of the forward
  int E;
  int64_t rows_cap;              // packed-row capacity
  int K;                         // DH/DX: reduction length (h' for DH, 2·d_ff for DX)
  int k_split;                   // DX: K index where B switches from W1 to W3 (d_ff)
  int w_rows;                    // DH/DX: B rows per expert in its map (h' for W2, d_ff for W1/W3)
  int n_out;                     // output columns (DH: d_ff, DX: h', DW: N extent)
  int n_tiles;                   // ceil(n_out / 256)
  int m_tiles;                   // DW: ceil(m_total / 128)
  int m_total;                   // DW: M extent (h' for dW2, 2·d_ff for dW1|dW3)
  int n_split;                   // DW transposed output: columns n >= n_split go to out_b (dW3)
  int transposed_out;            // DW: 0 → out_a[e][m][n]; 1 → out_{a|b}[e][n][m] (dW1|dW3)
  __nv_bfloat16* out_bf16;       // DH: dG|dU [rows][2·d_ff]; DX: dX_packed [rows][h']
  const __nv_bfloat16* gu;       // DH: G|U [rows][2·d_ff]
  float* out_a;                  // DW: dW2 [E][h'][d_ff], or dW1 [E][d_ff][h'] (transposed output)
  float* out_b;                  // DW: dW3 [E][d_ff][h'] (null for dW2)
  uint32_t* status;
};

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
expert_bwd_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                     const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmO0,
                     const __grid_constant__ CUtensorMap tmO1, BwdParams p) {
  extern __shared__ unsigned char smem_dyn[];
  __shared__ int s_off[kMaxExperts + 1];
  __shared__ int s_pre[kMaxExperts + 1];
  __shared__ __align__(8) uint64_t s_bar[2 * kStages + 5];
  // DW epilogue: per epilogue warp a 32 x 32 fp32 chunk, 16-byte pieces XOR-swizzled by row
  // DW: per epilogue warp a 32 x 32 fp32 tile in the 128-byte-swizzle layout of the store's map
  __shared__ __align__(1024) float s_epi[MODE == kModeDW ? 4 * 32 * 32 : 4];
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
    // M-grouped: m-tile prefix (128 rows); DW: 64-row block prefix = A's padded column offsets / 64
    const bool ok = warp_tile_prefix(p.offsets, p.E, MODE == kModeDW ? kBK : kBM, p.rows_cap, s_off, s_pre);
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
      if (MODE == kModeDX) tma_prefetch_desc(&tmB1);
      if (MODE == kModeDW) {
        tma_prefetch_desc(&tmO0);
        tma_prefetch_desc(&tmO1);
      }
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
  const int total = !s_ok ? 0 : (MODE == kModeDW ? p.E * p.m_tiles * p.n_tiles : s_pre[p.E] * p.n_tiles);
  volatile int* abort_flag = &s_abort;

  // (expert, m-tile, n-tile) of a linear tile index, and the k-blocks it runs
  auto tile_coords = [&](int tile, int& e, int& mt, int& nt, int& nkb) {
    if (MODE == kModeDW) {
      // m-tiles fastest: the tiles in flight share B's n-block (read from DRAM once) and cycle
      // through the expert's small transposed A (it stays in L2 while the fp32 output streams out)
      const int per_e = p.m_tiles * p.n_tiles;
      e = tile / per_e;
      const int r = tile - e * per_e;
      nt = r / p.m_tiles;
      mt = r - nt * p.m_tiles;
      nkb = (s_off[e + 1] - s_off[e] + kBK - 1) / kBK;
    } else {
      decode_tile(tile, s_pre, p.E, p.n_tiles, e, mt, nt);
      nkb = (p.K + kBK - 1) / kBK;
    }
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, filled = 0, last_parity = 0;
      bool aborted = false;
      for (int tile = blockIdx.x; tile < total && !aborted; tile += gridDim.x) {
        int e, mt, nt, nkb;
        tile_coords(tile, e, mt, nt, nkb);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag)) { aborted = true; break; }
          const uint32_t sa = sbase + stage * kStageBytes, sb = sa + kABytes;
          const uint32_t fb = full_bar(stage);
          mbar_arrive_expect_tx(fb, kStageBytes);
          // MN-major operands come through 3-D maps: one request per operand for all of its
          // 64-column blocks (A: 2, B: 4), each landing as an 8 KB swizzled tile
          if (MODE == kModeDW) {
            // A: K-major from the padded transposed copy (columns 64·s_pre[e] + ...); B: the same K
            // rows of the packed activations, MN-major
            tma_load_2d(sa, &tmA, fb, (s_pre[e] + kb) * kBK, mt * kBM);
            tma_load_3d(sb, &tmB0, fb, 0, s_off[e] + kb * kBK, nt * (kBN / 64));
          } else {
            tma_load_2d(sa, &tmA, fb, kb * kBK, s_off[e] + mt * kBM);
            const int kk = kb * kBK;
            const bool second = MODE == kModeDX && kk >= p.k_split;
            const CUtensorMap* mb = second ? &tmB1 : &tmB0;
            const int brow = e * p.w_rows + (second ? kk - p.k_split : kk);
            tma_load_3d(sb, mb, fb, 0, brow, nt * (kBN / 64));
          }
          filled |= 1u << stage;
          last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
      }
      if (aborted) {
        s_abort = 1;
        set_status(p.status, kDevErrTimeout);
        for (int s = 0; s < kStages; ++s)
          if ((filled >> s) & 1u) mbar_wait(full_bar(s), (last_parity >> s) & 1u, nullptr, 50000000ull);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (lane 0) + K-tail zeroing
    constexpr uint32_t idesc = idesc_bf16_f32(kBM, kBN) | kIdescBMajorMN;
    int stage = 0;
    uint32_t phase = 0;
    bool aborted = false;
    int it = 0;
    for (int tile = blockIdx.x; tile < total && !aborted; tile += gridDim.x, ++it) {
      int e, mt, nt, nkb;
      tile_coords(tile, e, mt, nt, nkb);
      const int acc = it & 1;
      const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
      if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag)) { aborted = true; break; }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + (uint32_t)(acc * kBN);
      for (int kb = 0; kb < nkb; ++kb) {
        if (!mbar_wait(full_bar(stage), phase, abort_flag)) { aborted = true; break; }
        const uint32_t sa = sbase + stage * kStageBytes, sb = sa + kABytes;
        if (MODE == kModeDW) {
          const int valid = s_off[e + 1] - s_off[e] - kb * kBK;
          // Rows past the expert meet A's zero padding, so they add exactly 0 while they hold
          // finite data: the next experts' rows do. Only a block that runs past the last packed
          // row (where the buffer holds whatever was there) gets those rows zeroed.
          if (valid < kBK && s_off[e] + (kb + 1) * kBK > s_off[p.E]) {
            // zero K rows valid..63 of the 4 B boxes (one 128-byte row each)
            const int nrow = (kBK - valid) * (kBN / 64);
            for (int i = lane; i < nrow * 8; i += 32) {
              const int row = i >> 3, chunk = i & 7;
              const int box = row / (kBK - valid), r = valid + row % (kBK - valid);
              asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(sb + box * kMnBox + r * 128 + chunk * 16),
                           "r"(0u)
                           : "memory");
            }
            fence_proxy_async_smem();
          }
          __syncwarp();
        }
        if (lane == 0) {
          tc_fence_after();
          uint64_t ad, bd;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            ad = sdesc_kmajor_sw128(sa) + (uint64_t)(2 * k);
            bd = sdesc_mnmajor_sw128(sb + k * 2048, kMnBox);
            umma_bf16(d_tmem, ad, bd, idesc, (kb > 0 || k > 0) ? 1u : 0u);
          }
          umma_commit(empty_bar(stage));
        }
        __syncwarp();
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
      }
      if (aborted) break;
      if (lane == 0) umma_commit(tfull_bar(acc));
      __syncwarp();
    }
    if (lane == 0) {
      if (aborted) { s_abort = 1; set_status(p.status, kDevErrTimeout); }
      umma_commit(done_bar);
      mbar_wait(done_bar, 0, nullptr, 50000000ull);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..5)
    const int q = warp & 3;  // TMEM lane quarter
    int it = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++it) {
      int e, mt, nt, nkb;
      tile_coords(tile, e, mt, nt, nkb);
      const int acc = it & 1;
      const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
      if (!mbar_wait(tfull_bar(acc), acc_phase, abort_flag)) {
        if (lane == 0) { s_abort = 1; set_status(p.status, kDevErrTimeout); }
        break;
      }
      tc_fence_after();
      const uint32_t t_row = tmem_base + (uint32_t)(acc * kBN) + ((uint32_t)(q * 32) << 16);
      if (MODE == kModeDW) {
        // A lane holds row m of the chunk's 32 x 32 fp32 block. It is staged in shared memory in
        // the 128-byte-swizzle layout (16-byte piece j of row r at piece j ^ (r & 7)) and one lane
        // writes it out with a TMA store: rows m of dW2[e], or, transposed, rows n of dW1 / dW3[e]
        // (the block staged with n as its row). Rows and columns past the tensor are not written.
        float* stg = s_epi + (warp - 2) * 32 * 32;
        const uint32_t stg_addr = smem_addr(stg);
        const int m0 = mt * kBM + q * 32;
#pragma unroll 1
        for (int c = 0; c < kBN / 32; ++c) {
          const int col = nt * kBN + c * 32;
          if (col >= p.n_out) break;  // n_out is a multiple of 64: chunks past it are whole
          uint32_t v[32];
          if (nkb > 0) {
            tmem_ld_32x32b_x32(t_row + c * 32, v);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = 0u;
          }
          if (lane == 0) bulk_wait_group_read0();  // the previous store has read the tile
          __syncwarp();
          if (!p.transposed_out) {
#pragma unroll
            for (int j = 0; j < 8; ++j)
              *reinterpret_cast<uint4*>(stg + lane * 32 + ((j ^ (lane & 7)) * 4)) =
                  make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)  // row n = j, column m = lane
              stg[j * 32 + ((((lane >> 2) ^ (j & 7)) << 2) | (lane & 3))] = __uint_as_float(v[j]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (!p.transposed_out) tma_store_3d(&tmO0, stg_addr, col, m0, e);
            else if (col < p.n_split) tma_store_3d(&tmO0, stg_addr, m0, col, e);
            else tma_store_3d(&tmO1, stg_addr, m0, col - p.n_split, e);
            bulk_commit_group();
          }
        }
      } else {
        const int rows_e = s_off[e + 1] - s_off[e];
        const int r_local = mt * kBM + q * 32 + lane;
        const bool row_ok = r_local < rows_e;
        const int64_t row = s_off[e] + r_local;
        if (MODE == kModeDH) {
          const int ld = 2 * p.n_out;  // G|U and dG|dU rows: [d_ff gate-side | d_ff up-side]
#pragma unroll 1
          for (int c = 0; c < kBN / 32; ++c) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(t_row + c * 32, v);
            tmem_ld_wait();
            const int col = nt * kBN + c * 32;
            if (row_ok && col < p.n_out) {
              const uint4* g4 = reinterpret_cast<const uint4*>(p.gu + row * ld + col);
              const uint4* u4 = reinterpret_cast<const uint4*>(p.gu + row * ld + p.n_out + col);
              uint32_t dg[16], du[16];
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const uint4 gq = g4[j], uq = u4[j];
                const uint32_t gw[4] = {gq.x, gq.y, gq.z, gq.w}, uw[4] = {uq.x, uq.y, uq.z, uq.w};
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                  float o_g[2], o_u[2];
#pragma unroll
                  for (int h = 0; h < 2; ++h) {
                    const float g = __uint_as_float((h ? gw[w] & 0xFFFF0000u : gw[w] << 16));
                    const float u = __uint_as_float((h ? uw[w] & 0xFFFF0000u : uw[w] << 16));
                    const float dh = __uint_as_float(v[8 * j + 2 * w + h]);
                    const float sg = __fdividef(1.0f, 1.0f + __expf(-g));  // σ(g)
                    const float sl = g * sg;                               // silu(g)
                    o_g[h] = dh * u * sg * (1.0f + g * (1.0f - sg));
                    o_u[h] = dh * sl;
                  }
                  dg[4 * j + w] = pack_bf16x2(o_g[0], o_g[1]);
                  du[4 * j + w] = pack_bf16x2(o_u[0], o_u[1]);
                }
              }
              uint4* dgo = reinterpret_cast<uint4*>(p.out_bf16 + row * ld + col);
              uint4* duo = reinterpret_cast<uint4*>(p.out_bf16 + row * ld + p.n_out + col);
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                dgo[j] = make_uint4(dg[4 * j], dg[4 * j + 1], dg[4 * j + 2], dg[4 * j + 3]);
                duo[j] = make_uint4(du[4 * j], du[4 * j + 1], du[4 * j + 2], du[4 * j + 3]);
              }
            }
          }
        } else {
          __nv_bfloat16* orow = p.out_bf16 + row * p.n_out;
#pragma unroll 1
          for (int c = 0; c < kBN / 32; ++c) {
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
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar(acc));
    }
    if (MODE == kModeDW && lane == 0) bulk_wait_group0();  // every output tile written
    __syncwarp();
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <int MODE>
cudaError_t launch_bwd(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1, const CUtensorMap& o0,
                       const CUtensorMap& o1, const BwdParams& p, int64_t max_tiles, cudaStream_t s) {
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(expert_bwd_tc_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmem);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  const int sms = device_sm_count();
  const int grid = (int)(max_tiles < sms ? (max_tiles > 0 ? max_tiles : 1) : sms);
  expert_bwd_tc_kernel<MODE><<<grid, kThreads, kSmem, s>>>(a, b0, b1, o0, o1, p);
  note_launch();
  return cudaGetLastError();
}

// Packed rows [rows][cols] (bf16; expert e's rows are offsets[e]..offsets[e+1]) → transposed
// [cols][pcols]: expert e's rows become columns 64·P_e .. 64·P_e + 64·ceil(n_e/64), with
// P_e = Σ_{e'<e} ceil(n_e'/64), zero past its n_e rows. One block per 64 x 64 tile.
__global__ void __launch_bounds__(256) transpose_pad_kernel(const __nv_bfloat16* __restrict__ in,
                                                            const int32_t* __restrict__ offsets, int E,
                                                            int64_t rows_cap, int cols, int64_t pcols,
                                                            __nv_bfloat16* __restrict__ out) {
  __shared__ int s_off[kMaxExperts + 1];
  __shared__ int s_pre[kMaxExperts + 1];
  __shared__ __align__(16) uint16_t tile[64][64 + 2];  // [row k][column i]; 33-word rows: few bank conflicts
  __shared__ int s_ok;
  if (threadIdx.x < 32) {
    const bool ok = warp_tile_prefix(offsets, E, 64, rows_cap, s_off, s_pre);
    if (threadIdx.x == 0) s_ok = ok ? 1 : 0;
  }
  __syncthreads();
  const int cb = blockIdx.y;
  if (!s_ok || cb >= s_pre[E]) return;
  int lo = 0, hi = E - 1;  // the expert whose blocks contain cb (largest e with s_pre[e] <= cb)
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_pre[mid] <= cb) lo = mid;
    else hi = mid - 1;
  }
  const int r0 = s_off[lo] + (cb - s_pre[lo]) * 64;
  const int valid = min(64, s_off[lo + 1] - r0);
  const int i0 = blockIdx.x * 64;
  for (int j = threadIdx.x; j < 64 * 8; j += 256) {
    const int k = j >> 3, v = j & 7;
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (k < valid && i0 + v * 8 < cols) val = *reinterpret_cast<const uint4*>(in + (int64_t)(r0 + k) * cols + i0 + v * 8);
    uint32_t* dst = reinterpret_cast<uint32_t*>(&tile[k][v * 8]);
    dst[0] = val.x;
    dst[1] = val.y;
    dst[2] = val.z;
    dst[3] = val.w;
  }
  __syncthreads();
  for (int j = threadIdx.x; j < 64 * 8; j += 256) {
    const int i = j >> 3, v = j & 7;
    if (i0 + i >= cols) continue;
    uint32_t w[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) w[t] = (uint32_t)tile[v * 8 + 2 * t][i] | ((uint32_t)tile[v * 8 + 2 * t + 1][i] << 16);
    *reinterpret_cast<uint4*>(out + (int64_t)(i0 + i) * pcols + (int64_t)cb * 64 + v * 8) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

cudaError_t launch_transpose_pad(const Problem& p, const void* in, const int32_t* offsets, int cols, int64_t pcols,
                                 void* out, cudaStream_t s) {
  const dim3 grid((unsigned)((cols + 63) / 64), (unsigned)(pcols / 64));
  transpose_pad_kernel<<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(in), offsets, p.E, p.rows, cols, pcols,
                                            static_cast<__nv_bfloat16*>(out));
  note_launch();
  return cudaGetLastError();
}

}  // namespace

// Columns of the padded transposed copies: every expert's rows rounded up to 64.
int64_t backward_padded_cols(const Problem& p) { return 64 * ((p.rows + 63) / 64 + p.E); }

// dY_packed, saved G|U, X_packed, H → dG|dU, dX_packed, dW1, dW3, dW2 (bf16 layers; h' and d_ff
// multiples of 64, checked by the caller).
cudaError_t launch_expert_ffn_backward(const Problem& p, const int32_t* offsets, const void* x_packed,
                                       const void* hidden, const void* gu, const void* dy_packed,
                                       const void* w_gate, const void* w_up, const void* w_down,
                                       void* dgu, void* dx_packed, float* dw_gate, float* dw_up,
                                       float* dw_down, void* dy_t, void* x_t, uint32_t* status, cudaStream_t s) {
  const uint64_t rows = (uint64_t)(p.rows > 0 ? p.rows : 1);
  const uint64_t E = (uint64_t)p.E, hu = (uint64_t)p.hu, dff = (uint64_t)p.d_ff;
  const int64_t pcols = backward_padded_cols(p);
  CUtensorMap mDYk, mDGUk, mW2, mW1, mW3, mDYt, mH, mDGUm, mXt;
  const uint32_t nbB = kBN / 64;  // 64-column blocks per MN-major B box
  if (!encode_tmap_2d_bf16(&mDYk, dy_packed, hu, rows, kBK, kBM) ||
      !encode_tmap_2d_bf16(&mDGUk, dgu, 2 * dff, rows, kBK, kBM) ||
      !encode_tmap_mn_blocks_bf16(&mW2, w_down, dff, E * hu, kBK, nbB) ||
      !encode_tmap_mn_blocks_bf16(&mW1, w_gate, hu, E * dff, kBK, nbB) ||
      !encode_tmap_mn_blocks_bf16(&mW3, w_up, hu, E * dff, kBK, nbB) ||
      !encode_tmap_2d_bf16(&mDYt, dy_t, (uint64_t)pcols, hu, kBK, kBM) ||
      !encode_tmap_mn_blocks_bf16(&mH, hidden, dff, rows, kBK, nbB) ||
      !encode_tmap_mn_blocks_bf16(&mDGUm, dgu, 2 * dff, rows, kBK, nbB) ||
      !encode_tmap_2d_bf16(&mXt, x_t, (uint64_t)pcols, hu, kBK, kBM))
    return cudaErrorInvalidValue;
  const int64_t m_tiles_rows = (p.rows + kBM - 1) / kBM + p.E;  // upper bound of the M-grouped m-tiles

  BwdParams b = {};
  b.offsets = offsets;
  b.E = p.E;
  b.rows_cap = p.rows;
  b.status = status;

  // DH: dH = dY·W2 → dG|dU
  b.K = p.hu;
  b.w_rows = p.hu;
  b.n_out = p.d_ff;
  b.n_tiles = (p.d_ff + kBN - 1) / kBN;
  b.out_bf16 = static_cast<__nv_bfloat16*>(dgu);
  b.gu = static_cast<const __nv_bfloat16*>(gu);
  cudaError_t e = launch_bwd<kModeDH>(mDYk, mW2, mW2, mW2, mW2, b, m_tiles_rows * b.n_tiles, s);
  if (e != cudaSuccess) return e;

  // DX: dX = dG·W1 + dU·W3
  b.K = 2 * p.d_ff;
  b.k_split = p.d_ff;
  b.w_rows = p.d_ff;
  b.n_out = p.hu;
  b.n_tiles = (p.hu + kBN - 1) / kBN;
  b.out_bf16 = static_cast<__nv_bfloat16*>(dx_packed);
  b.gu = nullptr;
  e = launch_bwd<kModeDX>(mDGUk, mW1, mW3, mW1, mW1, b, m_tiles_rows * b.n_tiles, s);
  if (e != cudaSuccess) return e;

  // DW: dW2 = dYᵀ·H ([E][h'][d_ff]): A = dY transposed (K-major), B = H (MN-major)
  e = launch_transpose_pad(p, dy_packed, offsets, p.hu, pcols, dy_t, s);
  if (e != cudaSuccess) return e;
  b.out_bf16 = nullptr;
  b.m_total = p.hu;
  b.m_tiles = (p.hu + kBM - 1) / kBM;
  b.n_out = p.d_ff;
  b.n_tiles = (p.d_ff + kBN - 1) / kBN;
  b.transposed_out = 0;
  b.out_a = dw_down;
  b.out_b = nullptr;
  CUtensorMap oW2, oW1, oW3;  // fp32 outputs, 32 x 32 boxes: dW2 [E][h'][d_ff]; dW1, dW3 [E][d_ff][h']
  if (!encode_tmap_3d_f32_sw128(&oW2, dw_down, dff, hu, E, 32, 32) ||
      !encode_tmap_3d_f32_sw128(&oW1, dw_gate, hu, dff, E, 32, 32) ||
      !encode_tmap_3d_f32_sw128(&oW3, dw_up, hu, dff, E, 32, 32))
    return cudaErrorInvalidValue;
  e = launch_bwd<kModeDW>(mDYt, mH, mH, oW2, oW2, b, (int64_t)p.E * b.m_tiles * b.n_tiles, s);
  if (e != cudaSuccess) return e;

  // DW: (dW1 | dW3)ᵀ = Xᵀ·(dG | dU) ([h'][2·d_ff] per expert, stored as dW1, dW3 [E][d_ff][h']):
  // A = X transposed (K-major), B = dG|dU (MN-major)
  e = launch_transpose_pad(p, x_packed, offsets, p.hu, pcols, x_t, s);
  if (e != cudaSuccess) return e;
  b.m_total = p.hu;
  b.m_tiles = (p.hu + kBM - 1) / kBM;
  b.n_out = 2 * p.d_ff;
  b.n_split = p.d_ff;
  b.n_tiles = (2 * p.d_ff + kBN - 1) / kBN;
  b.transposed_out = 1;
  b.out_a = dw_gate;
  b.out_b = dw_up;
  return launch_bwd<kModeDW>(mXt, mDGUm, mDGUm, oW1, oW3, b, (int64_t)p.E * b.m_tiles * b.n_tiles, s);
}

}  // namespace moe
