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
#include <atomic>

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
  int swap_max;            // pair tiles: last m-tiles of at most this many rows run transposed (0: none)
  __nv_bfloat16* save_gu;  // gate/up: G | U pre-activations [rows][2·n_out] (bf16) when not null
  // down GEMM with the combine folded in (kernels instantiated with FK > 0)
  __nv_bfloat16* y;            // [T'][n_out] layer output
  const int32_t* row_token;    // [rows] packed row -> unit
  const int32_t* slot_of;      // [T'][topk] packed row of each pick, -1: dropped
  const float* gate;           // [T'][topk]
  uint32_t* arrivals;          // [T'][n_out/32] rows of the unit done per 32-column chunk, zero on entry
  int64_t Tu;
  int topk;
  int keep_packed;             // write every Y row to out (the backward reads Y_packed)
};

// 32 fp32 values (as bits) → 32 bf16 at dst (64 bytes, 16-byte aligned).
__device__ __forceinline__ void store_bf16x32(__nv_bfloat16* dst, const uint32_t (&v)[32]) {
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int j = 0; j < 4; ++j)
    d4[j] = make_uint4(pack_bf16x2(__uint_as_float(v[8 * j]), __uint_as_float(v[8 * j + 1])),
                       pack_bf16x2(__uint_as_float(v[8 * j + 2]), __uint_as_float(v[8 * j + 3])),
                       pack_bf16x2(__uint_as_float(v[8 * j + 4]), __uint_as_float(v[8 * j + 5])),
                       pack_bf16x2(__uint_as_float(v[8 * j + 6]), __uint_as_float(v[8 * j + 7])));
}

// ------------------------------------------------------------------------------------------------
// Combine folded into the down GEMM's epilogue.
//   [Lesson 10 "专家并行 EP", §1: y = Σ_{i∈TopK} s_i(x)·FFN_i(x); §3 steps 3-4: each result goes
//    back to its unit and the unit's results are summed with the gates kept from routing]
// A unit with one kept pick is finished by that pick's row: the epilogue writes g·Y into y. A unit
// with k >= 2 kept picks is finished, per 32-column chunk, by whichever of its rows gets there last:
// every row writes its Y chunk to Y_packed, makes it visible (__threadfence) and adds one to the
// chunk's arrival counter; the row that reads k - 1 back loads the unit's k chunks (L2, bypassing
// L1) and writes y = Σ_k g_k·Y_k with the separate combine's arithmetic: the same fp32 fmaf chain in
// k order from +0, dropped picks adding 0·0. The result is therefore bit-identical to the two-launch
// path and independent of the order in which rows arrive. The pack zeroes the counters and the y
// rows of units whose picks were all dropped.

// What a lane knows about the unit of the packed row (or token) it owns.
template <int FK>
struct CombineRow {
  int t;           // unit, -1: this lane owns none
  int kept;        // kept picks of the unit
  int own;         // pick index of the owned row
  int32_t sl[FK];  // packed rows of the unit's picks (-1: dropped or k >= topk)
  float g[FK];     // their gates (0 where sl is -1)
};

template <int FK>
__device__ __forceinline__ void combine_row_clear(CombineRow<FK>& c) {
  c.t = -1;
  c.kept = 0;
  c.own = -1;
#pragma unroll
  for (int k = 0; k < FK; ++k) {
    c.sl[k] = -1;
    c.g[k] = 0.f;
  }
}

template <int FK>
__device__ __forceinline__ void combine_row_load(const TcParams& p, int64_t slot, CombineRow<FK>& c) {
  combine_row_clear(c);
  const int t = __ldg(p.row_token + slot);
  if (t < 0 || (int64_t)t >= p.Tu) {
    set_status(p.status, kDevErrBadIndex);
    return;
  }
  int own = -1, kept = 0;
#pragma unroll
  for (int k = 0; k < FK; ++k) {
    if (k < p.topk) {
      int s = __ldg(p.slot_of + (int64_t)t * p.topk + k);
      if ((int64_t)s >= p.rows_cap) {
        set_status(p.status, kDevErrBadIndex);
        s = -1;
      }
      if (s >= 0) {
        c.sl[k] = s;
        c.g[k] = __ldg(p.gate + (int64_t)t * p.topk + k);
        ++kept;
        if ((int64_t)s == slot) own = k;
      }
    }
  }
  if (own < 0) {  // the row is not among its unit's picks
    set_status(p.status, kDevErrBadIndex);
    combine_row_clear(c);
    return;
  }
  c.t = t;
  c.kept = kept;
  c.own = own;
}

__device__ __forceinline__ uint4 ld_global_cg_v4(const void* ptr) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(ptr));
  return v;
}

// Count the owned row into the arrival counters of its chunks (bit c of `chunks`: counter
// base[c]); returns the chunks this row completes. The caller's Y stores precede it.
template <int FK>
__device__ __forceinline__ uint32_t combine_arrive(const TcParams& p, const CombineRow<FK>& c, uint32_t* base,
                                                   uint32_t chunks) {
  if (c.t < 0) return 0u;
  if (c.kept == 1) return chunks;
  __threadfence();  // this row's Y chunks are visible before it is counted
  uint32_t last = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if ((chunks >> i) & 1u) {
      const uint32_t old = atomicAdd(base + i, 1u);
      if (old + 1u == (uint32_t)c.kept) last |= 1u << i;
      else if (old >= (uint32_t)c.kept) set_status(p.status, kDevErrBadIndex);
    }
  }
  if (last) __threadfence();  // the other rows' chunks are read after their counts were seen
  return last;
}

// y chunks of the units whose last rows are held by lanes with last != 0 (bit c: 32-column chunk c
// from col0). LPO lanes serve one owner, 16 bytes (8 columns) each: LPO = 32 covers 256 columns
// (a row of a 128 x 256 tile), LPO = 4 covers 32 (a transposed tile's warp). R batches of 32/LPO
// owners are loaded before any is summed. The whole warp calls this.
template <int FK, int LPO>
__device__ __forceinline__ void combine_owned(const TcParams& p, uint32_t last, const CombineRow<FK>& c, int col0) {
  constexpr int OPP = 32 / LPO;
  constexpr int R = FK <= 2 ? 8 : 2;
  const int lane = threadIdx.x & 31;
  const int sub = lane % LPO, pos = lane / LPO;
  const int col = col0 + sub * 8;
  uint32_t owners = __ballot_sync(0xffffffffu, last != 0u);
  while (owners != 0u) {
    uint4 raw[R][FK];
    float gw[R][FK];
    int64_t dst[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const uint32_t o = __fns(owners, 0, r * OPP + pos + 1);
      const int src = o < 32u ? (int)o : lane;
      const int t = __shfl_sync(0xffffffffu, c.t, src);
      const uint32_t m = __shfl_sync(0xffffffffu, last, src);
      const bool ok = o < 32u && ((m >> (sub >> 2)) & 1u) != 0u && col < p.n_out;
      dst[r] = ok ? (int64_t)t * p.n_out + col : -1;
#pragma unroll
      for (int k = 0; k < FK; ++k) {
        const int s = __shfl_sync(0xffffffffu, c.sl[k], src);
        gw[r][k] = __shfl_sync(0xffffffffu, c.g[k], src);
        raw[r][k] = make_uint4(0u, 0u, 0u, 0u);
        if (ok && s >= 0) raw[r][k] = ld_global_cg_v4(p.out + (int64_t)s * p.n_out + col);
      }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
      if (dst[r] < 0) continue;
      float acc[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] = 0.f;
#pragma unroll
      for (int k = 0; k < FK; ++k) {
        if (k < p.topk) {
          const __nv_bfloat16* pv = reinterpret_cast<const __nv_bfloat16*>(&raw[r][k]);
#pragma unroll
          for (int q = 0; q < 8; ++q) acc[q] = fmaf(gw[r][k], __bfloat162float(pv[q]), acc[q]);
        }
      }
      *reinterpret_cast<uint4*>(p.y + dst[r]) =
          make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                     pack_bf16x2(acc[6], acc[7]));
    }
#pragma unroll 1
    for (int i = 0; i < R * OPP && owners != 0u; ++i) owners &= owners - 1u;
  }
}

// g·Y of a unit with one kept pick (pick `own` of topk), 32 columns: the separate combine's chain
// (fp32 fmaf in k order from +0, dropped picks adding 0·0) with Y rounded to bf16 first.
template <int FK>
__device__ __forceinline__ void store_direct_x32(const TcParams& p, const CombineRow<FK>& c, __nv_bfloat16* dst,
                                                 const uint32_t (&pk)[16]) {
  uint32_t o[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const __nv_bfloat162 v2 = *reinterpret_cast<const __nv_bfloat162*>(&pk[j]);
    const float v0 = __low2float(v2), v1 = __high2float(v2);
    float a0 = 0.f, a1 = 0.f;
#pragma unroll
    for (int k = 0; k < FK; ++k) {
      if (k < p.topk) {
        const bool mine = k == c.own;
        a0 = fmaf(c.g[k], mine ? v0 : 0.f, a0);
        a1 = fmaf(c.g[k], mine ? v1 : 0.f, a1);
      }
    }
    o[j] = pack_bf16x2(a0, a1);
  }
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int j = 0; j < 4; ++j) d4[j] = make_uint4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
}

// Single-CTA tiles: an expert's last m-tile of at most kSwapMaxRowsSingle rows runs transposed,
// Dᵀ = W·Xᵀ, as two M = 128 MMAs over the tile's 256 weight rows with N = the tail's tokens rounded
// up to a multiple of 16 (both blocks fit one 256-column accumulator). Experts of about 128 rows
// (fine-grained layers) otherwise spend a mostly empty second 128-row tile.
constexpr int kSwapMaxRowsSingle = 112;
__device__ __forceinline__ int swap_tokens(int tail) { return (tail + 15) & ~15; }

template <int EPI, int FK>
__global__ void __launch_bounds__(kTcThreads, 1)
expert_gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                      const __grid_constant__ CUtensorMap tmB1, TcParams p) {
  extern __shared__ unsigned char smem_dyn[];
  // transposed tails: per epilogue warp, a [token][32 columns] bf16 chunk turned into row stores
  __shared__ __align__(16) __nv_bfloat16 s_stage[4 * 32 * 32];
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
    if (lane == 0) {
      s_abort = 0;
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
    griddep_wait();  // the offsets and packed rows come from the previous kernel of the stream
    const bool ok = warp_tile_prefix(p.offsets, p.E, kBM, p.rows_cap, s_off, s_pre);
    if (lane == 0) {
      s_ok = ok ? 1 : 0;
      if (!ok && blockIdx.x == 0) set_status(p.status, kDevErrBadOffsets);
    }
    __syncwarp();
  } else if (warp == 1) {
    tmem_alloc(smem_addr(&s_tmem), kTmemCols);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  griddep_wait();
  griddep_launch_dependents();
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
        int e, mt, nt;
        decode_tile(tile, s_pre, p.E, p.n_tiles, e, mt, nt);
        const int tail = s_off[e + 1] - s_off[e] - mt * kBM;
        const bool swap = tail <= p.swap_max;
        const int n_tok = swap_tokens(tail);
        const uint32_t idesc_t = idesc_bf16_f32(kBM, swap ? n_tok : 16);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(full_bar(stage), phase, abort_flag)) { aborted = true; break; }
          tc_fence_after();
          const uint32_t sa = sbase + stage * kStageBytes, sb = sa + kABytes;
          const uint64_t ad = sdesc_kmajor_sw128(sa), bd = sdesc_kmajor_sw128(sb);
          if (!swap) {
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k)  // 16 bf16 = 32 bytes per MMA along K
              umma_bf16(d_tmem, ad + (uint64_t)(2 * k), bd + (uint64_t)(2 * k), kIdesc,
                        (kb > 0 || k > 0) ? 1u : 0u);
          } else {
            // Dᵀ: weight rows 0-127 of the tile into columns [0, n_tok), rows 128-255 into
            // [n_tok, 2·n_tok); the tail's tokens (the first n_tok of the 128 loaded) are N
            const uint64_t bd1 = sdesc_kmajor_sw128(sb + kBBytes / 2);
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k) {
              umma_bf16(d_tmem, bd + (uint64_t)(2 * k), ad + (uint64_t)(2 * k), idesc_t, (kb > 0 || k > 0) ? 1u : 0u);
              umma_bf16(d_tmem + (uint32_t)n_tok, bd1 + (uint64_t)(2 * k), ad + (uint64_t)(2 * k), idesc_t,
                        (kb > 0 || k > 0) ? 1u : 0u);
            }
          }
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
      const int rows_e = s_off[e + 1] - s_off[e];
      const int r_local = mt * kBM + q * 32 + lane;
      const bool row_ok = r_local < rows_e;
      CombineRow<(FK > 0 ? FK : 1)> cr;
      if constexpr (FK > 0) {  // the row's unit, read while the MMAs run
        if (row_ok) combine_row_load(p, (int64_t)s_off[e] + r_local, cr);
        else combine_row_clear(cr);
      }
      if (!mbar_wait(tfull_bar(acc), acc_phase, abort_flag)) {
        if (lane == 0) { s_abort = 1; set_status(p.status, kDevErrTimeout); }
        break;
      }
      tc_fence_after();
      __nv_bfloat16* orow = p.out + (int64_t)(s_off[e] + r_local) * p.n_out;
      const uint32_t t_row = tmem_base + (uint32_t)(acc * kBN) + ((uint32_t)(q * 32) << 16);
      const int tail = rows_e - mt * kBM;
      if (tail <= p.swap_max) {
        // transposed tile: TMEM lane = output column (32 per warp), column = token of the tail;
        // block 0 (columns [0, n_tok)) holds weight rows 0-127 of the tile, block 1 rows 128-255:
        // for gate/up the gate and the up of the same output column, for down two column halves.
        // Each chunk of 32 tokens goes through the warp's staging area into 16-byte row pieces.
        const int n_tok = swap_tokens(tail);
        __nv_bfloat16* obase = p.out + (int64_t)(s_off[e] + mt * kBM) * p.n_out;
        __nv_bfloat16* stg = s_stage + (warp - 2) * 32 * 32;
#pragma unroll 1
        for (int c0 = 0; c0 < n_tok; c0 += 32) {
          uint32_t v0[32], v1[32];
          tmem_ld_32x32b_x32(t_row + c0, v0);
          tmem_ld_32x32b_x32(t_row + n_tok + c0, v1);
          tmem_ld_wait();
          // out: 0 = SwiGLU H (or down block 0), 1 = down block 1; then G and U for the backward
          const int nout = EPI == kEpiSwiGLU ? (p.save_gu != nullptr ? 3 : 1) : 2;
#pragma unroll 1
          for (int w = 0; w < nout; ++w) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float g = __uint_as_float(v0[i]), u = __uint_as_float(v1[i]);
              float val;
              if (EPI == kEpiSwiGLU) val = w == 0 ? silu_f32(g) * u : (w == 1 ? g : u);
              else val = w == 0 ? g : u;
              stg[i * 32 + lane] = __float2bfloat16_rn(val);
            }
            __syncwarp();
            __nv_bfloat16* dbase;
            int64_t ld;
            int col0;
            if (EPI == kEpiSwiGLU) {
              col0 = nt * 128 + q * 32;
              if (w == 0) { dbase = obase; ld = p.n_out; }
              else {
                dbase = p.save_gu + (int64_t)(s_off[e] + mt * kBM) * (2 * p.n_out) + (w == 2 ? p.n_out : 0);
                ld = 2 * (int64_t)p.n_out;
              }
            } else {
              col0 = nt * kBN + w * 128 + q * 32;
              dbase = obase;
              ld = p.n_out;
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int j = lane + 32 * k, t = j >> 2, part = j & 3;
              if (col0 < p.n_out && c0 + t < tail)
                *reinterpret_cast<uint4*>(dbase + (int64_t)(c0 + t) * ld + col0 + part * 8) =
                    *reinterpret_cast<const uint4*>(stg + t * 32 + part * 8);
            }
            __syncwarp();
          }
        }
      } else if (EPI == kEpiSwiGLU) {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t g[32], u[32];
          tmem_ld_32x32b_x32(t_row + c * 32, g);
          tmem_ld_32x32b_x32(t_row + 128 + c * 32, u);
          tmem_ld_wait();
          const int col = nt * 128 + c * 32;
          if (row_ok && col < p.n_out) {
            if (p.save_gu != nullptr) {
              __nv_bfloat16* sg = p.save_gu + (int64_t)(s_off[e] + r_local) * (2 * p.n_out) + col;
              store_bf16x32(sg, g);
              store_bf16x32(sg + p.n_out, u);
            }
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
            const bool direct = FK > 0 && cr.kept == 1;
            if (!direct || p.keep_packed) {
              uint4* dst = reinterpret_cast<uint4*>(orow + col);
#pragma unroll
              for (int j = 0; j < 4; ++j) dst[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
            }
            if constexpr (FK > 0) {
              if (direct) store_direct_x32(p, cr, p.y + (int64_t)cr.t * p.n_out + col, pk);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar(acc));
      if constexpr (FK > 0) {
        // the accumulator is free again; finish the units whose last row this was
        uint32_t chunks = 0;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          if (nt * kBN + c * 32 < p.n_out) chunks |= 1u << c;
        const uint32_t last =
            cr.kept >= 2 ? combine_arrive(p, cr, p.arrivals + (int64_t)cr.t * (p.n_out >> 5) + nt * (kBN / 32), chunks)
                         : 0u;
        combine_owned<FK, 32>(p, last, cr, nt * kBN);
      }
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
//
// Ragged tails. An expert's last m-tile usually holds fewer than 256 rows, and a 256-row tile
// spends its MMAs on the missing rows as well (about a tenth of the work of a layer with ~1000
// rows per expert). A tail of at most kSwapMaxRows rows is therefore computed transposed,
// Dᵀ = W·Xᵀ: the 256 weight rows of the tile are the M operand and the tail's tokens, rounded up
// to a multiple of 16, are the N operand (M = 256 allows any N that is a multiple of 16), so at
// most 15 padding rows are computed. Operands keep their shared-memory slots (slot 0 = M operand,
// slot 1 = N operand): in a swapped tile slot 0 holds weights and slot 1 holds token rows, CTA r
// the tokens [r·N/2, (r+1)·N/2) of the tail. TMEM lane = output column, TMEM column = token.
// For gate/up the 128 weight rows of CTA r are the W1 rows of output columns r·64 + [0,64) and
// then the W3 rows of the same columns (two 64-row TMA boxes), so TMEM lanes 0-63 hold gate and
// lanes 64-127 up. An epilogue warp reads only its own 32-lane quarter of TMEM, so the gate warp of
// 32 columns (quarter q < 2) and the up warp of the same columns (quarter q + 2) swap half of each
// 32-token chunk through shared memory, synchronised by an mbarrier per warp pair and buffer.
constexpr int kPairBM = 256, kPairStages = 6;
constexpr int kSwapMaxRows = 224;   // larger tails gain little and use the plain epilogue
// A transposed gate/up tile's epilogue (exchange between warps, more chunks) only hides behind the
// next tile's main loop when that is long enough; with fewer k-blocks the tails stay 256-row tiles.
constexpr int kSwapMinKBlocks = 16;
constexpr int kPairHalf = 128 * kBK * 2;                 // 16 KB: 128 rows x 64 bf16
constexpr int kPairStageBytes = 2 * kPairHalf;           // A half + B half per CTA
constexpr size_t kPairSmem = (size_t)kPairStages * kPairStageBytes + 1024;
constexpr uint32_t kIdescPair = idesc_bf16_f32(kPairBM, kBN);
constexpr int kSwapHalf = 64;       // W1 (then W3) rows per CTA in a swapped gate/up tile

// Tokens per CTA in a swapped tail tile of `tail` rows (N = twice this, a multiple of 16).
__device__ __forceinline__ int swap_half_n(int tail) { return ((tail + 15) & ~15) >> 1; }

template <int EPI, int FK>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kTcThreads, 1)
expert_gemm_tc_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                           const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmS0,
                           const __grid_constant__ CUtensorMap tmS1, TcParams p) {
  extern __shared__ unsigned char smem_dyn[];
  __shared__ int s_off[kMaxExperts + 1];
  __shared__ int s_pre[kMaxExperts + 1];
  __shared__ __align__(8) uint64_t s_bar[2 * kPairStages + 5 + 4];
  // gate/up ↔ exchange of swapped tiles: [buffer][warp pair][direction: 0 gate→up, 1 up→gate][token][lane]
  __shared__ __align__(16) float s_xch[EPI == kEpiSwiGLU ? 2 * 2 * 2 * 16 * 32 : 1];
  // swapped tiles: per epilogue warp, a [token][32 columns] bf16 chunk turned into row-vector stores
  __shared__ __align__(16) __nv_bfloat16 s_stage[4 * 32 * 32];
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
  auto xch_bar = [&](int pair, int buf) { return bar0 + 8u * (2 * kPairStages + 5 + 2 * pair + buf); };

  if (warp == 0) {
    if (lane == 0) {
      s_abort = 0;
      for (int s = 0; s < kPairStages; ++s) {
        mbar_init(full_bar(s), 1);
        mbar_init(empty_bar(s), 1);
      }
      for (int a = 0; a < 2; ++a) {
        mbar_init(tfull_bar(a), 1);
        mbar_init(tempty_bar(a), 8);
      }
      mbar_init(done_bar, 1);
      for (int b = 0; b < 4; ++b) mbar_init(xch_bar(b >> 1, b & 1), 64);  // both warps' lanes
      fence_mbar_init();
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB0);
      if (EPI == kEpiSwiGLU) {
        tma_prefetch_desc(&tmB1);
        tma_prefetch_desc(&tmS0);
        tma_prefetch_desc(&tmS1);
      }
    }
    __syncwarp();
    griddep_wait();  // the offsets and packed rows come from the previous kernel of the stream
    const bool ok = warp_tile_prefix(p.offsets, p.E, kPairBM, p.rows_cap, s_off, s_pre);
    if (lane == 0) {
      s_ok = ok ? 1 : 0;
      if (!ok && blockIdx.x == 0) set_status(p.status, kDevErrBadOffsets);
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
  griddep_wait();
  griddep_launch_dependents();
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
        const int tail = s_off[e + 1] - s_off[e] - mt * kPairBM;
        const bool swap = tail <= p.swap_max;
        const int a_row = s_off[e] + mt * kPairBM + (int)rank * (swap ? swap_half_n(tail) : 128);
        const int b_row = (EPI == kEpiSwiGLU) ? e * p.w_rows + nt * (kBN / 2)
                                              : e * p.w_rows + nt * kBN + (int)rank * 128;
        // swapped gate/up: first W1/W3 row of this CTA's 64 output columns
        const int s_row = e * p.w_rows + nt * (kBN / 2) + (int)rank * kSwapHalf;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag)) { aborted = true; break; }
          const uint32_t sa = sbase + stage * kPairStageBytes;
          if (leader) mbar_arrive_expect_tx(full_bar(stage), 2 * kPairStageBytes);
          const uint32_t fb = full0_leader + 8u * stage;
          if (!swap) {
            tma_load_2d_pair(sa, &tmA, fb, kb * kBK, a_row);
            tma_load_2d_pair(sa + kPairHalf, mb, fb, kb * kBK, b_row);
          } else {
            // token rows into slot 1 (the MMA reads the first N/2 of the 128 loaded)
            tma_load_2d_pair(sa + kPairHalf, &tmA, fb, kb * kBK, a_row);
            if (EPI == kEpiSwiGLU) {
              tma_load_2d_pair(sa, &tmS0, fb, kb * kBK, s_row);
              tma_load_2d_pair(sa + kSwapHalf * kBK * 2, &tmS1, fb, kb * kBK, s_row);
            } else {
              tma_load_2d_pair(sa, mb, fb, kb * kBK, b_row);
            }
          }
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
        int e, mt, nt;
        decode_tile(tile, s_pre, p.E, p.n_tiles, e, mt, nt);
        const int tail = s_off[e + 1] - s_off[e] - mt * kPairBM;
        const uint32_t idesc =
            tail <= p.swap_max ? idesc_bf16_f32(kPairBM, 2 * swap_half_n(tail)) : kIdescPair;
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * kBN);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(full_bar(stage), phase, abort_flag)) { aborted = true; break; }
          tc_fence_after();
          const uint32_t sa = sbase + stage * kPairStageBytes;
          const uint64_t ad = sdesc_kmajor_sw128(sa), bd = sdesc_kmajor_sw128(sa + kPairHalf);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            umma_bf16_pair(d_tmem, ad + (uint64_t)(2 * k), bd + (uint64_t)(2 * k), idesc,
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
    uint32_t xn = 0;     // exchange chunks done by this warp (its partner does the same sequence)
    bool failed = false;
    for (int tile = cid; tile < total && !failed; tile += ncl, ++it) {
      int e, mt, nt;
      decode_tile(tile, s_pre, p.E, p.n_tiles, e, mt, nt);
      const int acc = it & 1;
      const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
      const int rows_e = s_off[e + 1] - s_off[e];
      const int tail = rows_e - mt * kPairBM;
      const int r_local = mt * kPairBM + (int)rank * 128 + q * 32 + lane;
      const bool row_ok = r_local < rows_e;
      CombineRow<(FK > 0 ? FK : 1)> cr;
      if constexpr (FK > 0) {  // the row's unit (plain tiles), read while the MMAs run
        if (row_ok && tail > p.swap_max) combine_row_load(p, (int64_t)s_off[e] + r_local, cr);
        else combine_row_clear(cr);
      }
      if (!mbar_wait(tfull_bar(acc), acc_phase, abort_flag)) {
        if (lane == 0) abort_both();
        break;
      }
      tc_fence_after();
      __nv_bfloat16* orow = p.out + (int64_t)(s_off[e] + r_local) * p.n_out;
      const uint32_t t_row = tmem_base + (uint32_t)(acc * kBN) + ((uint32_t)(q * 32) << 16);
      if (tail <= p.swap_max) {
        // transposed tile: lane = output column, TMEM column = token of the tail. Each warp puts a
        // chunk of [tokens][its 32 columns] in bf16 into its staging area, then writes it out as
        // 16-byte pieces of output rows (four per token: 32 columns = 64 bytes).
        const int n_tok = 2 * swap_half_n(tail);
        __nv_bfloat16* obase = p.out + (int64_t)(s_off[e] + mt * kPairBM) * p.n_out;
        __nv_bfloat16* stg = s_stage + (warp - 2) * 32 * 32;
        if (EPI == kEpiSwiGLU) {
          // quarter q < 2: gate of columns 32q + lane; quarter q + 2: up of the same columns. The
          // gate warp finishes tokens c0..c0+15 of each chunk, the up warp c0+16..c0+31.
          const bool gate_warp = q < 2;
          const int wp = q & 1;
          const int col0 = nt * 128 + (int)rank * kSwapHalf + wp * 32;
          const bool cols_ok = col0 < p.n_out;  // n_out is a multiple of 32
#pragma unroll 1
          for (int c0 = 0; c0 < n_tok; c0 += 32, ++xn) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(t_row + c0, v);
            tmem_ld_wait();
            const int buf = (int)(xn & 1u);
            float* xb = s_xch + (size_t)((buf * 2 + wp) * 2) * 16 * 32;
            float* mine = xb + (gate_warp ? 0 : 16 * 32);       // what this warp hands over
            const float* theirs = xb + (gate_warp ? 16 * 32 : 0);
#pragma unroll
            for (int i = 0; i < 16; ++i) mine[i * 32 + lane] = __uint_as_float(gate_warp ? v[16 + i] : v[i]);
            mbar_arrive(xch_bar(wp, buf));
            if (!mbar_wait(xch_bar(wp, buf), (xn >> 1) & 1u, abort_flag)) {
              failed = true;
              break;
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float other = theirs[i * 32 + lane];
              const float g = gate_warp ? __uint_as_float(v[i]) : other;
              const float u = gate_warp ? other : __uint_as_float(v[16 + i]);
              stg[i * 32 + lane] = __float2bfloat16_rn(silu_f32(g) * u);
            }
            __syncwarp();
            const int t0 = c0 + (gate_warp ? 0 : 16);
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              const int j = lane + 32 * k, t = j >> 2, part = j & 3;
              if (cols_ok && t0 + t < tail)
                *reinterpret_cast<uint4*>(obase + (int64_t)(t0 + t) * p.n_out + col0 + part * 8) =
                    *reinterpret_cast<const uint4*>(stg + t * 32 + part * 8);
            }
            __syncwarp();
            if (p.save_gu != nullptr) {
              // G, then U, of the same 16 tokens x 32 columns, through the staging area
              __nv_bfloat16* sbase_gu = p.save_gu + (int64_t)(s_off[e] + mt * kPairBM) * (2 * p.n_out);
#pragma unroll 1
              for (int which = 0; which < 2; ++which) {
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                  const float other = theirs[i * 32 + lane];
                  const float g = gate_warp ? __uint_as_float(v[i]) : other;
                  const float u = gate_warp ? other : __uint_as_float(v[16 + i]);
                  stg[i * 32 + lane] = __float2bfloat16_rn(which == 0 ? g : u);
                }
                __syncwarp();
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                  const int j = lane + 32 * k, t = j >> 2, part = j & 3;
                  if (cols_ok && t0 + t < tail)
                    *reinterpret_cast<uint4*>(sbase_gu + (int64_t)(t0 + t) * (2 * p.n_out) + which * p.n_out +
                                              col0 + part * 8) = *reinterpret_cast<const uint4*>(stg + t * 32 + part * 8);
                }
                __syncwarp();
              }
            }
          }
          if (failed) {
            if (lane == 0) abort_both();
            break;
          }
        } else {
          const int col0 = nt * kBN + (int)rank * 128 + q * 32;
          const bool cols_ok = col0 < p.n_out;
#pragma unroll 1
          for (int c0 = 0; c0 < n_tok; c0 += 32) {
            if constexpr (FK > 0) {  // lane owns token c0 + lane of the tail
              if (cols_ok && c0 + lane < tail)
                combine_row_load(p, (int64_t)s_off[e] + mt * kPairBM + c0 + lane, cr);
              else
                combine_row_clear(cr);
            }
            uint32_t v[32];
            tmem_ld_32x32b_x32(t_row + c0, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) stg[i * 32 + lane] = __float2bfloat16_rn(__uint_as_float(v[i]));
            __syncwarp();
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int j = lane + 32 * k, t = j >> 2, part = j & 3;
              if constexpr (FK == 1) {
                // top-1: the token's row is its unit's output, g·Y straight into y (lane t owns it)
                const int tu = __shfl_sync(0xffffffffu, cr.t, t);
                const float g = __shfl_sync(0xffffffffu, cr.g[0], t);
                const uint4 v = *reinterpret_cast<const uint4*>(stg + t * 32 + part * 8);
                if (cols_ok && c0 + t < tail && tu >= 0) {
                  if (p.keep_packed)
                    *reinterpret_cast<uint4*>(obase + (int64_t)(c0 + t) * p.n_out + col0 + part * 8) = v;
                  const __nv_bfloat16* pv = reinterpret_cast<const __nv_bfloat16*>(&v);
                  uint32_t o[4];
#pragma unroll
                  for (int i = 0; i < 4; ++i)
                    o[i] = pack_bf16x2(fmaf(g, __bfloat162float(pv[2 * i]), 0.f),
                                       fmaf(g, __bfloat162float(pv[2 * i + 1]), 0.f));
                  *reinterpret_cast<uint4*>(p.y + (int64_t)tu * p.n_out + col0 + part * 8) =
                      make_uint4(o[0], o[1], o[2], o[3]);
                }
              } else {
                if (cols_ok && c0 + t < tail)
                  *reinterpret_cast<uint4*>(obase + (int64_t)(c0 + t) * p.n_out + col0 + part * 8) =
                      *reinterpret_cast<const uint4*>(stg + t * 32 + part * 8);
              }
            }
            __syncwarp();
            if constexpr (FK > 1) {
              // each token's chunk was stored by 4 lanes: all fence before the owners count it
              __threadfence();
              __syncwarp();
              const uint32_t last =
                  cr.t >= 0 ? combine_arrive(p, cr, p.arrivals + (int64_t)cr.t * (p.n_out >> 5) + (col0 >> 5), 1u)
                            : 0u;
              combine_owned<FK, 4>(p, last, cr, col0);
            }
          }
        }
      } else if (EPI == kEpiSwiGLU) {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t g[32], u[32];
          tmem_ld_32x32b_x32(t_row + c * 32, g);
          tmem_ld_32x32b_x32(t_row + 128 + c * 32, u);
          tmem_ld_wait();
          const int col = nt * 128 + c * 32;
          if (row_ok && col < p.n_out) {
            if (p.save_gu != nullptr) {
              __nv_bfloat16* sg = p.save_gu + (int64_t)(s_off[e] + r_local) * (2 * p.n_out) + col;
              store_bf16x32(sg, g);
              store_bf16x32(sg + p.n_out, u);
            }
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
            const bool direct = FK > 0 && cr.kept == 1;
            if (!direct || p.keep_packed) {
              uint4* dst = reinterpret_cast<uint4*>(orow + col);
#pragma unroll
              for (int j = 0; j < 4; ++j) dst[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
            }
            if constexpr (FK > 0) {
              if (direct) store_direct_x32(p, cr, p.y + (int64_t)cr.t * p.n_out + col, pk);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader) mbar_arrive(tempty_bar(acc));
        else mbar_arrive_remote(tempty_leader0 + 8u * acc);
      }
      if constexpr (FK > 0) {
        if (tail > p.swap_max) {  // plain tile: the accumulator is free again; finish the units
          uint32_t chunks = 0;
#pragma unroll
          for (int c = 0; c < 8; ++c)
            if (nt * kBN + c * 32 < p.n_out) chunks |= 1u << c;
          const uint32_t last =
              cr.kept >= 2
                  ? combine_arrive(p, cr, p.arrivals + (int64_t)cr.t * (p.n_out >> 5) + nt * (kBN / 32), chunks)
                  : 0u;
          combine_owned<FK, 32>(p, last, cr, nt * kBN);
        }
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

// The kernels are persistent: a cluster that could not be resident alongside the others would run
// its whole share of tiles after them. The grid is capped at the clusters the GPU holds at once
// (asked once per device).
template <typename Kern>
static int resident_cluster_grid(Kern kern, int cluster, size_t smem, int want) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)want);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = smem;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
    (void)cudaGetLastError();
    return want;
  }
  return n * cluster < want ? n * cluster : want;
}

template <int EPI, int FK>
static cudaError_t launch_tc_pair(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                                  const CUtensorMap& s0, const CUtensorMap& s1, const TcParams& p,
                                  int grid, cudaStream_t s, bool pdl) {
  static bool attr_done[64] = {false};
  static int grid_cap[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(expert_gemm_tc_pair_kernel<EPI, FK>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPairSmem);
    if (e != cudaSuccess) return e;
    grid_cap[dev] = resident_cluster_grid(expert_gemm_tc_pair_kernel<EPI, FK>, 2, kPairSmem, grid);
    attr_done[dev] = true;
  }
  if (dev < 64 && grid_cap[dev] > 0 && grid > grid_cap[dev]) grid = grid_cap[dev];
  // the 2-CTA cluster shape is compiled into the kernel
  return launch_kernel(expert_gemm_tc_pair_kernel<EPI, FK>, dim3(grid), dim3(kTcThreads), kPairSmem, s, 1, pdl, a, b0, b1,
                       s0, s1, p);
}

// Choices forced by moe_set_expert_gemm (-1: automatic).
static std::atomic<int> g_pair_tiles{-1}, g_transposed_tails{-1}, g_fold_combine{-1};

void set_expert_gemm(int pair_tiles, int transposed_tails, int fold) {
  g_pair_tiles.store(pair_tiles);
  g_transposed_tails.store(transposed_tails);
  g_fold_combine.store(fold);
}

// With K == 1 the fold only redirects each row's store (g·Y into y), so it saves the y_packed
// round trip and the combine launch. With K >= 2 each row also fences, counts itself in the arrival
// counters and, if last, loads its unit's other rows: a chain of dependent memory round trips per
// row that made the epilogue, not the MMA, set the tile rate on every layer measured.
bool fold_combine(const Problem& p) {
  const int forced = g_fold_combine.load(std::memory_order_relaxed);
  if (forced >= 0) return forced == 1;
  return p.K == 1;
}

// Pair tiles (256 rows) pay off when experts hold many rows; with few rows per expert (fine-grained
// layers) the single-CTA 128-row tile wastes less work on ragged tails.
static bool use_pair_tiles(const Problem& p) {
  const int forced = g_pair_tiles.load(std::memory_order_relaxed);
  if (forced >= 0) return forced == 1;
  return p.rows / p.E >= kPairBM;
}

// Largest tail (rows) that a GEMM with reduction length K runs transposed (pair or single tiles).
static int swap_max_rows(int K, bool pair) {
  const int most = pair ? kSwapMaxRows : kSwapMaxRowsSingle;
  const int forced = g_transposed_tails.load(std::memory_order_relaxed);
  if (forced >= 0) return forced == 1 ? most : 0;
  return (K + kBK - 1) / kBK >= kSwapMinKBlocks ? most : 0;
}

template <int EPI, int FK>
static cudaError_t launch_tc(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                             const TcParams& p, int grid, cudaStream_t s, bool pdl) {
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(expert_gemm_tc_kernel<EPI, FK>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTcSmem);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  return launch_kernel(expert_gemm_tc_kernel<EPI, FK>, dim3(grid), dim3(kTcThreads), kTcSmem, s, 1, pdl, a, b0, b1, p);
}

cudaError_t launch_expert_ffn_simt(const Problem& p, const void* x_packed, const int32_t* offsets,
                                   const void* w_gate, const void* w_up, const void* w_down,
                                   void* hidden, void* y_packed, uint32_t* status, cudaStream_t s, bool pdl);

cudaError_t launch_expert_ffn(const Problem& p, const void* x_packed, const int32_t* offsets,
                              const void* w_gate, const void* w_up, const void* w_down,
                              void* hidden, void* y_packed, uint32_t* status, cudaStream_t s,
                              void* save_gu, bool pdl, const FusedCombine* fc) {
  if (!p.bf16) {
    if (fc) return cudaErrorInvalidValue;  // the combine is folded only into the tensor-core GEMM
    return launch_expert_ffn_simt(p, x_packed, offsets, w_gate, w_up, w_down, hidden, y_packed, status, s, pdl);
  }
  if (p.rows == 0) return cudaSuccess;
  if (fc && (!fc->y || !fc->row_token || !fc->slot_of || !fc->gate || !fc->arrivals || p.K > kMaxTopK ||
             (reinterpret_cast<uintptr_t>(fc->y) & 15) != 0))
    return cudaErrorInvalidValue;
  CUtensorMap mA, mW1, mW3, mH, mW2;
  const uint64_t rows = (uint64_t)p.rows;
  if (!encode_tmap_2d_bf16(&mA, x_packed, (uint64_t)p.hu, rows, kBK, kBM) ||
      !encode_tmap_2d_bf16(&mW1, w_gate, (uint64_t)p.hu, (uint64_t)p.E * p.d_ff, kBK, kBN / 2) ||
      !encode_tmap_2d_bf16(&mW3, w_up, (uint64_t)p.hu, (uint64_t)p.E * p.d_ff, kBK, kBN / 2) ||
      !encode_tmap_2d_bf16(&mH, hidden, (uint64_t)p.d_ff, rows, kBK, kBM) ||
      !encode_tmap_2d_bf16(&mW2, w_down, (uint64_t)p.d_ff, (uint64_t)p.E * p.hu, kBK, kBN))
    return cudaErrorInvalidValue;
  const bool pair = use_pair_tiles(p);
  CUtensorMap mW2p, mW1s, mW3s;  // pair tiles: W2 in 128-row halves; W1/W3 in 64-row halves (tails)
  if (pair && (!encode_tmap_2d_bf16(&mW2p, w_down, (uint64_t)p.d_ff, (uint64_t)p.E * p.hu, kBK, kBN / 2) ||
               !encode_tmap_2d_bf16(&mW1s, w_gate, (uint64_t)p.hu, (uint64_t)p.E * p.d_ff, kBK, kSwapHalf) ||
               !encode_tmap_2d_bf16(&mW3s, w_up, (uint64_t)p.hu, (uint64_t)p.E * p.d_ff, kBK, kSwapHalf)))
    return cudaErrorInvalidValue;
  const int sms = device_sm_count();
  const int grid = pair ? (sms / 2) * 2 : sms;
  TcParams g = {};
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
  g.swap_max = swap_max_rows(g.K, pair);
  g.save_gu = static_cast<__nv_bfloat16*>(save_gu);
  cudaError_t e = pair ? launch_tc_pair<kEpiSwiGLU, 0>(mA, mW1, mW3, mW1s, mW3s, g, grid, s, pdl)
                       : launch_tc<kEpiSwiGLU, 0>(mA, mW1, mW3, g, grid, s, pdl);
  if (e != cudaSuccess) return e;
  // down → y_packed (and, folded in, y)
  g.K = p.d_ff;
  g.w_rows = p.hu;
  g.n_tiles = (p.hu + kBN - 1) / kBN;
  g.n_out = p.hu;
  g.out = static_cast<__nv_bfloat16*>(y_packed);
  g.swap_max = swap_max_rows(g.K, pair);
  g.save_gu = nullptr;
  if (!fc)
    return pair ? launch_tc_pair<kEpiPlain, 0>(mH, mW2p, mW2p, mW2p, mW2p, g, grid, s, true)
                : launch_tc<kEpiPlain, 0>(mH, mW2, mW2, g, grid, s, true);
  g.y = static_cast<__nv_bfloat16*>(fc->y);
  g.row_token = fc->row_token;
  g.slot_of = fc->slot_of;
  g.gate = fc->gate;
  g.arrivals = fc->arrivals;
  g.Tu = p.Tu;
  g.topk = p.K;
  g.keep_packed = fc->keep_packed ? 1 : 0;
  if (!pair) g.swap_max = 0;  // the single-CTA transposed epilogue does not fold the combine
  if (p.K == 1)
    return pair ? launch_tc_pair<kEpiPlain, 1>(mH, mW2p, mW2p, mW2p, mW2p, g, grid, s, true)
                : launch_tc<kEpiPlain, 1>(mH, mW2, mW2, g, grid, s, true);
  if (p.K == 2)
    return pair ? launch_tc_pair<kEpiPlain, 2>(mH, mW2p, mW2p, mW2p, mW2p, g, grid, s, true)
                : launch_tc<kEpiPlain, 2>(mH, mW2, mW2, g, grid, s, true);
  return pair ? launch_tc_pair<kEpiPlain, 8>(mH, mW2p, mW2p, mW2p, mW2p, g, grid, s, true)
              : launch_tc<kEpiPlain, 8>(mH, mW2, mW2, g, grid, s, true);
}

}  // namespace moe
