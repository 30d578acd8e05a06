// Routing of bf16 layers in one kernel: router logits on the tensor cores, then scores, group limit,
// Top-K, gates, the aux-loss statistics and the dispatch's per-tile counts in the epilogue.
//   [Lesson 10 "专家并行 EP", §1: affinity scores x·W_g, s(x) = Softmax(TopK(x·W_g, K)) or sigmoid;
//    §4: L_aux = α·E·Σ f_i·P_i; §5: node-limited (group-limited) routing]
//
// A cluster of S CTAs (S = 1, 2, 4 or 8) owns one tile of 128 units. CTA r of the cluster computes
// the partial logits of the tile over its slice of the reduction dimension h' with tcgen05.mma
// (M = 128 units, N = E rounded up to 64, K = 16): x comes K-major through TMA (128 x 64 boxes,
// 128-byte swizzle); W_g is read in the pages' own [h'][E] orientation, which is the MN-major
// layout of the B operand, through TMA boxes of 64 experts x 64 rows (experts past E read as
// zeros), so no transposed copy of W_g is made. Then, in column passes of 64 experts:
//   - every CTA copies its TMEM partial to shared memory;
//   - CTA r adds the S partials of its own 128/S units in cluster-rank order (reading the peers'
//     shared memory through the cluster window), adds the logit bias, and writes the logits;
// so the sum is deterministic and no partial logits go through HBM. Each CTA then routes its units
// (select_tile.cuh) and counts its picks per expert; the cluster adds the counts and the Σp of its
// CTAs in rank order into the tile's histogram and Σp row, and every pick gets its place among the
// tile's picks of the same expert (unit order), which the dispatch turns into a packed row.
//
// Threads: 256. Warp 0 lane 0 issues the TMA loads into a ring of stages, warp 1 owns TMEM and its
// lane 0 issues the MMAs; all eight warps read TMEM (warp w: lanes 32·(w%4), columns by w/4) and
// route. Every mbarrier wait is bounded; every CTA of a cluster passes the same cluster barriers
// whatever happens, so a timeout (status bit set) never leaves a peer waiting.
#include "moe_device.cuh"
#include "moe_internal.h"
#include "select_tile.cuh"

namespace moe {

namespace {

constexpr int kRtBM = 128, kRtBK = 64, kRtThreads = 256, kRtMaxStages = 4;
constexpr int kRtABytes = kRtBM * kRtBK * 2;       // 16 KB x tile
constexpr int kRtWBox = 64 * kRtBK * 2;            // 8 KB: 64 experts x 64 rows of W_g
constexpr int kRtStageBudget = 110 * 1024;         // ring or epilogue: two CTAs per SM
constexpr int kRtFastBudget = 110 * 1024;          // ring + fast epilogue, two CTAs per SM

struct RouteTcParams {
  int64_t Tu;
  int E, Np, nblk;       // experts; MMA N = 64·nblk
  int nkb, kbs;          // k-blocks in total; per cluster rank
  int S;                 // CTAs per cluster
  int stages;
  uint32_t stage_bytes;
  uint32_t epi_off;      // fast epilogue: its shared memory starts here (past the stage ring)
  const float* logit_bias;
  float* logits_out;     // [T'][E] or null
  SelectCtx sel;
  int32_t* rank_out;     // [T'][K] place of each pick among its tile's picks of the same expert
  int32_t* tile_hist;    // [tiles][E]
  float* tile_psum;      // [tiles][E]
  uint32_t* status;
};

// Shared-memory plan of the epilogue (byte offsets from the 1024-aligned base; the pipeline ring
// uses the same memory before it).
struct RtEpi {
  int R;          // units per CTA
  int ldl;        // row stride of the logit tile
  int cw, ldp;    // columns per reduction pass; row stride (floats) of the partial tile
  size_t lg, picks, rank, lanes, wpre, gscr, psum, hist, scratch, prefix, total;
};

__host__ __device__ inline size_t rt_align(size_t n) { return (n + 15) / 16 * 16; }

// Reduction passes of 128 columns when a cluster adds partials of at least 128 experts (half the
// cluster barriers of 64-column passes), else 64.
__host__ __device__ inline RtEpi rt_epi(int S, int E, int epl) {
  RtEpi L;
  L.R = kRtBM / S;
  L.ldl = E + 1;
  L.cw = (S > 1 && E > 64) ? 128 : 64;
  L.ldp = L.cw + 4;
  size_t off = rt_align((size_t)kRtBM * L.ldp * 4);  // the partial tile P first
  auto take = [&](size_t bytes) { const size_t at = off; off = rt_align(off + bytes); return at; };
  const int rw = (L.R + 31) / 32;  // warps holding rows
  L.lg = take((size_t)L.R * L.ldl * 4);
  L.picks = take((size_t)L.R * kPickStride * 4);
  L.rank = take((size_t)L.R * kPickStride * 4);
  L.lanes = take((size_t)rw * E * 4);
  L.wpre = take((size_t)rw * E * 4);
  L.gscr = take(epl > 0 ? (size_t)(kRtThreads / 32) * 32 * epl * 8 : 0);
  L.psum = take((size_t)E * 4);
  L.hist = take((size_t)E * 4);
  L.scratch = take((size_t)kRtThreads * 4);
  L.prefix = take((size_t)E * 4);
  L.total = off;
  return L;
}

// Shared memory of the fast epilogue (softmax, no group limit, E <= 64), placed past the stage ring:
// peers push into recv_* while this CTA may still be in its main loop.
struct RtFast {
  int R, ec;      // units per CTA; E rounded up to 4
  int ldr;        // row stride (floats) of the receive buffer: ec + 4, so a warp's 16-byte row
                  // writes and reads spread over all banks
  size_t recv_l, recv_h, recv_p, picks, rank, lanes, wpre, wpsum, psum, hist, total;
};

__host__ __device__ inline RtFast rt_fast(int S, int E) {
  RtFast L;
  L.R = kRtBM / S;
  L.ec = (E + 3) / 4 * 4;
  L.ldr = L.ec + 4;
  size_t off = 0;
  auto take = [&](size_t bytes) { const size_t at = off; off = rt_align(off + bytes); return at; };
  const bool cl = S > 1;
  L.recv_l = take(cl ? (size_t)S * L.R * L.ldr * 4 : 0);
  L.recv_h = take(cl ? (size_t)S * E * 4 : 0);
  L.recv_p = take(cl ? (size_t)S * E * 4 : 0);
  L.picks = take((size_t)L.R * kPickStride * 4);
  L.rank = take((size_t)L.R * kPickStride * 4);
  L.lanes = take((size_t)(kRtThreads / 32) * E * 4);
  L.wpre = take((size_t)(kRtThreads / 32) * E * 4);
  L.wpsum = take((size_t)4 * E * 4);
  L.psum = take((size_t)E * 4);
  L.hist = take((size_t)E * 4);
  L.total = off;
  return L;
}

// One TMEM row (this thread's lane) of EM fp32 columns into registers.
template <int EM>
__device__ __forceinline__ void tmem_row(uint32_t taddr, float (&v)[EM]) {
  if constexpr (EM <= 16) {
    uint32_t r[16];
    tmem_ld_32x32b_x16(taddr, r);
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < EM; ++j) v[j] = __uint_as_float(r[j]);
  } else {
#pragma unroll
    for (int c = 0; c < EM; c += 32) {
      uint32_t r[32];
      tmem_ld_32x32b_x32(taddr + (uint32_t)c, r);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 32; ++j) v[c + j] = __uint_as_float(r[j]);
    }
  }
}

// Threads per CTA: the fast epilogue routes one unit per thread of warps 0-3, so it runs 128.
__host__ __device__ constexpr int rt_threads(int fem) { return fem > 0 ? 128 : kRtThreads; }

template <int EPL, int KMAX, bool SIGMOID, int FEM>
__global__ void __launch_bounds__(rt_threads(FEM), 1)
route_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW, RouteTcParams p) {
  extern __shared__ unsigned char smem_dyn[];
  __shared__ __align__(8) uint64_t s_bar[2 * kRtMaxStages + 1];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  const uint32_t sbase = (smem_addr(smem_dyn) + 1023u) & ~1023u;
  unsigned char* gbase = smem_dyn + (sbase - smem_addr(smem_dyn));
  const uint32_t bar0 = smem_addr(s_bar);
  const int S = p.S, NS = p.stages;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (NS + s); };
  const uint32_t done_bar = bar0 + 8u * (2 * NS);
  const uint32_t tmem_cols = p.Np <= 64 ? 64u : (p.Np <= 128 ? 128u : 256u);

  const int r = S > 1 ? (int)cluster_ctarank() : 0;
  const int tile = blockIdx.x / S;
  const int kb0 = r * p.kbs;
  const int nk = max(0, min(p.nkb, kb0 + p.kbs) - kb0);

  if (warp == 0 && lane == 0) {
    s_abort = 0;
    for (int s = 0; s < NS; ++s) {
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
  // fast epilogue: peers write into this CTA's shared memory, which is only valid once every CTA of
  // the cluster runs; the matching wait comes before the first such write
  if constexpr (FEM > 0)
    if (S > 1) cluster_arrive_relaxed();
  griddep_launch_dependents();
  griddep_wait();  // x and W_g may come from the previous kernel of the stream
  const uint32_t tmem = s_tmem;
  volatile int* abort_flag = &s_abort;
  const uint32_t idesc = idesc_bf16_f32(kRtBM, p.Np) | kIdescBMajorMN;

  if (warp == 0) {
    if (lane == 0) {
      uint32_t filled = 0, last_parity = 0;
      for (int i = 0; i < nk; ++i) {
        const int st = i % NS;
        const uint32_t ph = (uint32_t)(i / NS) & 1u;
        if (!mbar_wait(empty_bar(st), ph ^ 1u, abort_flag)) {
          s_abort = 1;
          set_status(p.status, kDevErrTimeout);
          for (int s = 0; s < NS; ++s)
            if ((filled >> s) & 1u) mbar_wait(full_bar(s), (last_parity >> s) & 1u, nullptr, 50000000ull);
          break;
        }
        const uint32_t sa = sbase + (uint32_t)st * p.stage_bytes;
        const int k = (kb0 + i) * kRtBK;
        mbar_arrive_expect_tx(full_bar(st), p.stage_bytes);
        tma_load_2d(sa, &tmX, full_bar(st), k, tile * kRtBM);
        for (int j = 0; j < p.nblk; ++j) tma_load_2d(sa + kRtABytes + j * kRtWBox, &tmW, full_bar(st), 64 * j, k);
        filled |= 1u << st;
        last_parity = (last_parity & ~(1u << st)) | (ph << st);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      bool aborted = false;
      for (int i = 0; i < nk; ++i) {
        const int st = i % NS;
        const uint32_t ph = (uint32_t)(i / NS) & 1u;
        if (!mbar_wait(full_bar(st), ph, abort_flag)) {
          aborted = true;
          break;
        }
        tc_fence_after();
        const uint32_t sa = sbase + (uint32_t)st * p.stage_bytes;
        const uint64_t ad = sdesc_kmajor_sw128(sa);
#pragma unroll
        for (int k = 0; k < kRtBK / 16; ++k)
          umma_bf16(tmem, ad + (uint64_t)(2 * k), sdesc_mnmajor_sw128(sa + kRtABytes + k * 2048, kRtWBox), idesc,
                    (i > 0 || k > 0) ? 1u : 0u);
        umma_commit(empty_bar(st));
      }
      if (aborted) {
        s_abort = 1;
        set_status(p.status, kDevErrTimeout);
      }
      umma_commit(done_bar);  // also covers nk == 0: arrives once the earlier MMAs (none) complete
    }
    __syncwarp();
  }

  const bool ok = mbar_wait(done_bar, 0, abort_flag);
  if (!ok && tid == 0) set_status(p.status, kDevErrTimeout);
  tc_fence_after();

  if constexpr (FEM > 0) {
    constexpr int NT = rt_threads(FEM);
    // ---------------------------------------------------------- fast epilogue (registers)
    const RtFast F = rt_fast(S, p.E);
    unsigned char* fb = gbase + p.epi_off;
    const uint32_t fb_sh = sbase + p.epi_off;
    const int R = F.R, E = p.E, K = p.sel.K;
    const int row0 = r * R;
    const int64_t u0 = (int64_t)tile * kRtBM + row0;
    const int Rv = (int)max((int64_t)0, min((int64_t)R, p.Tu - u0));
    float l[FEM];
    if (S > 1) cluster_wait();  // every CTA of the cluster has started
    // 1. this CTA's partial logits of TMEM row `row` (warps 0-3: one row per thread)
    if (warp < 4) {
      const int row = 32 * warp + lane;
      if (ok && nk > 0) tmem_row<FEM>(tmem + ((uint32_t)(32 * warp) << 16), l);
      else {
#pragma unroll
        for (int e = 0; e < FEM; ++e) l[e] = 0.f;
      }
      if (S > 1) {
        // push the row to the CTA that routes it: slice r of its receive buffer
        const int q = row / R, rr = row - q * R;
        const uint32_t dst = mapa_shared(fb_sh + (uint32_t)(F.recv_l + ((size_t)(r * R + rr) * F.ldr) * 4), (uint32_t)q);
#pragma unroll
        for (int e = 0; e < FEM; e += 4)
          if (e < F.ec) st_shared_cluster_v4f32(dst + 4u * e, l[e], l[e + 1], l[e + 2], l[e + 3]);
      }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc(tmem, tmem_cols);
    }
    if (S > 1) {
      cluster_sync_all();  // every slice of my units is in my receive buffer
      if (tid < R) {
        const float* rl = reinterpret_cast<const float*>(fb + F.recv_l);
#pragma unroll
        for (int e = 0; e < FEM; e += 4) {
          if (e >= F.ec) break;
          const float4 a = *reinterpret_cast<const float4*>(rl + (size_t)tid * F.ldr + e);
          l[e] = a.x; l[e + 1] = a.y; l[e + 2] = a.z; l[e + 3] = a.w;
        }
        for (int q = 1; q < S; ++q)
#pragma unroll
          for (int e = 0; e < FEM; e += 4) {
            if (e >= F.ec) break;
            const float4 a = *reinterpret_cast<const float4*>(rl + ((size_t)q * R + tid) * F.ldr + e);
            l[e] += a.x; l[e + 1] += a.y; l[e + 2] += a.z; l[e + 3] += a.w;
          }
      }
    }
    // 2. route my units: thread t < Rv routes unit u0 + t
    uint32_t* wcount = reinterpret_cast<uint32_t*>(fb + F.lanes);  // [4 warps][E] picks per expert
    float* wpsum = reinterpret_cast<float*>(fb + F.wpsum);
    float* psum_s = reinterpret_cast<float*>(fb + F.psum);
    int* hist_s = reinterpret_cast<int*>(fb + F.hist);
    float pr[FEM];
    int pk[KMAX], rk[KMAX];
#pragma unroll
    for (int e = 0; e < FEM; ++e) pr[e] = 0.f;
#pragma unroll
    for (int k = 0; k < KMAX; ++k) { pk[k] = -1; rk[k] = 0; }
    if (tid < Rv) {
#pragma unroll
      for (int e = 0; e < FEM; ++e)
        if (e < E && p.logit_bias) l[e] = l[e] + p.logit_bias[e];
      const int64_t u = u0 + tid;
      if (p.logits_out) {
#pragma unroll
        for (int e = 0; e < FEM; ++e)
          if (e < E) p.logits_out[u * E + e] = l[e];
      }
      float gv[KMAX];
      route_unit_regs<FEM, KMAX>(l, E, K, pk, gv, pr);
#pragma unroll
      for (int k = 0; k < KMAX; ++k)
        if (k < K) {
          p.sel.idx[u * K + k] = pk[k];
          p.sel.gate[u * K + k] = gv[k];
        }
    }
    // 3. Σ_t p[t][e] over my units (warp reduce-scatter, then the warps in order), and the picks per
    // expert of each warp with each pick's place among them (a ballot per expert)
    const uint32_t lt = lanemask_lt();
    if (warp < 4) {
      warp_reduce_scatter<FEM>(pr, lane);
      if constexpr (FEM >= 32) {
#pragma unroll
        for (int j = 0; j < FEM / 32; ++j) {
          const int e = lane * (FEM / 32) + j;
          if (e < E) wpsum[warp * E + e] = pr[j];
        }
      } else {
        const int g = 32 / FEM;
        if ((lane % g) == 0 && lane / g < E) wpsum[warp * E + lane / g] = pr[0];
      }
      for (int e = 0; e < E; ++e) {
        bool mine = false;
#pragma unroll
        for (int k = 0; k < KMAX; ++k) mine |= pk[k] == e;
        const uint32_t m = __ballot_sync(0xffffffffu, mine);
#pragma unroll
        for (int k = 0; k < KMAX; ++k)
          if (pk[k] == e) rk[k] = __popc(m & lt);
        if (lane == 0) wcount[warp * E + e] = (uint32_t)__popc(m);
      }
    }
    __syncthreads();
    for (int e = tid; e < E; e += NT) {
      psum_s[e] = ((wpsum[e] + wpsum[E + e]) + wpsum[2 * E + e]) + wpsum[3 * E + e];
      hist_s[e] = (int)(wcount[e] + wcount[E + e] + wcount[2 * E + e] + wcount[3 * E + e]);
    }
#pragma unroll
    for (int k = 0; k < KMAX; ++k)
      if (pk[k] >= 0)
        for (int w = 0; w < warp; ++w) rk[k] += (int)wcount[w * E + pk[k]];
    __syncthreads();
    // 4. the tile's counts and Σp; each pick's place in the tile
    if (S == 1) {
      for (int e = tid; e < E; e += NT) {
        p.tile_hist[(int64_t)tile * E + e] = hist_s[e];
        p.tile_psum[(int64_t)tile * E + e] = psum_s[e];
      }
      if (tid < Rv)
#pragma unroll
        for (int k = 0; k < KMAX; ++k)
          if (k < K) p.rank_out[(u0 + tid) * K + k] = rk[k];
    } else {
      // push my counts to every CTA (prefixes) and my Σp to rank 0 (tile totals)
      for (int i = tid; i < S * E; i += NT) {
        const int q = i / E, e = i - q * E;
        st_shared_cluster_u32(mapa_shared(fb_sh + (uint32_t)(F.recv_h + ((size_t)r * E + e) * 4), (uint32_t)q),
                              (uint32_t)hist_s[e]);
        if (q == 0)
          st_shared_cluster_f32(mapa_shared(fb_sh + (uint32_t)(F.recv_p + ((size_t)r * E + e) * 4), 0u), psum_s[e]);
      }
      cluster_sync_all();  // every CTA's counts (and Σp at rank 0) have arrived; no remote access follows
      const int* rh = reinterpret_cast<const int*>(fb + F.recv_h);
      const float* rp = reinterpret_cast<const float*>(fb + F.recv_p);
      int* prefix = reinterpret_cast<int*>(fb + F.wpre);
      for (int e = tid; e < E; e += NT) {
        int pre = 0, tot = 0;
        float ps = 0.f;
        for (int q = 0; q < S; ++q) {
          const int h = rh[q * E + e];
          if (q < r) pre += h;
          tot += h;
          if (r == 0) ps += rp[q * E + e];
        }
        prefix[e] = pre;
        if (r == 0) {
          p.tile_hist[(int64_t)tile * E + e] = tot;
          p.tile_psum[(int64_t)tile * E + e] = ps;
        }
      }
      __syncthreads();
      if (tid < Rv)
#pragma unroll
        for (int k = 0; k < KMAX; ++k)
          if (k < K) p.rank_out[(u0 + tid) * K + k] = rk[k] + prefix[pk[k]];
    }
    return;
  }

  // ------------------------------------------------------------ logits: partials → my units
  const RtEpi L = rt_epi(S, p.E, EPL);
  float* P = reinterpret_cast<float*>(gbase);
  float* lg = reinterpret_cast<float*>(gbase + L.lg);
  const int R = L.R, ldl = L.ldl, E = p.E;
  const int row0 = r * R;
  const int64_t u0 = (int64_t)tile * kRtBM + row0;
  const int Rv = (int)max((int64_t)0, min((int64_t)R, p.Tu - u0));
  const uint32_t p_sh = smem_addr(P);
  const int cw = L.cw, ldp = L.ldp;
  const int npass = p.Np / cw;
  for (int pass = 0; pass < npass; ++pass) {
    {
      // warp w: TMEM lanes 32·(w%4) (its rows), columns cw/2·(w/4) .. of the pass
      const int q4 = warp & 3, half = warp >> 2;
      const int row = 32 * q4 + lane;
      for (int c0 = 0; c0 < cw / 2; c0 += 32) {
        uint32_t v[32];
        if (ok && nk > 0) {
          tmem_ld_32x32b_x32(tmem + ((uint32_t)(32 * q4) << 16) + (uint32_t)(cw * pass + (cw / 2) * half + c0), v);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = 0u;
        }
        float4* dst = reinterpret_cast<float4*>(P + row * ldp + (cw / 2) * half + c0);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          dst[j] = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]), __uint_as_float(v[4 * j + 2]),
                               __uint_as_float(v[4 * j + 3]));
      }
    }
    tc_fence_before();
    __syncthreads();
    if (S > 1) cluster_sync_all();  // every peer's partial is in its shared memory
    // 4 columns per thread: all S partial loads are issued before the first add (the adds run in
    // rank order)
    const int c4n = cw / 4;
    for (int i = tid; i < R * c4n; i += kRtThreads) {
      const int rr = i / c4n, c4 = (i - rr * c4n) * 4, e0 = cw * pass + c4;
      if (e0 >= E) continue;
      const int prow = row0 + rr;
      const uint32_t off = (uint32_t)((prow * ldp + c4) * 4);
      float4 part[8];
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (q < S)
          part[q] = (q == r) ? *reinterpret_cast<const float4*>(P + prow * ldp + c4)
                             : ld_shared_cluster_v4f32(mapa_shared(p_sh + off, (uint32_t)q));
      float v[4] = {part[0].x, part[0].y, part[0].z, part[0].w};
#pragma unroll
      for (int q = 1; q < 8; ++q)
        if (q < S) {
          v[0] += part[q].x; v[1] += part[q].y; v[2] += part[q].z; v[3] += part[q].w;
        }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int e = e0 + j;
        if (e >= E) break;
        float w = v[j];
        if (p.logit_bias) w = w + p.logit_bias[e];
        lg[rr * ldl + e] = w;
        if (p.logits_out && rr < Rv) p.logits_out[(u0 + rr) * E + e] = w;
      }
    }
    if (S > 1) cluster_sync_all();  // peers are done reading this pass's partial
    else __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, tmem_cols);
  }

  // ------------------------------------------------------------ routing of my units
  int* picks = reinterpret_cast<int*>(gbase + L.picks);
  int* rank = reinterpret_cast<int*>(gbase + L.rank);
  float* psum_s = reinterpret_cast<float*>(gbase + L.psum);
  int* hist_s = reinterpret_cast<int*>(gbase + L.hist);
  int* prefix = reinterpret_cast<int*>(gbase + L.prefix);
  if constexpr (EPL == 0)
    select_rows_thread<KMAX, SIGMOID>(p.sel, lg, ldl, Rv, u0, picks);
  else
    select_rows_warp<EPL, SIGMOID>(p.sel, lg, ldl, Rv, u0, picks, gbase + L.gscr);
  __syncthreads();
  column_sums(lg, ldl, Rv, E, psum_s, reinterpret_cast<float*>(gbase + L.scratch));
  rank_picks(picks, Rv, p.sel.K, E, rank, hist_s, reinterpret_cast<uint32_t*>(gbase + L.lanes),
             reinterpret_cast<int*>(gbase + L.wpre));

  // ------------------------------------------------------------ the tile's counts and Σp
  if (S > 1) cluster_sync_all();  // every CTA's counts and Σp are in its shared memory
  const uint32_t hist_sh = smem_addr(hist_s), psum_sh = smem_addr(psum_s);
  for (int e = tid; e < E; e += kRtThreads) {
    int h[8];
    float ps[8];
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (q < S) {
        h[q] = (q == r) ? hist_s[e] : ld_shared_cluster_s32(mapa_shared(hist_sh + 4u * e, (uint32_t)q));
        if (r == 0) ps[q] = (q == 0) ? psum_s[e] : ld_shared_cluster_f32(mapa_shared(psum_sh + 4u * e, (uint32_t)q));
      }
    int pre = 0, tot = 0;
    float psum = 0.f;
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (q < S) {
        if (q < r) pre += h[q];
        tot += h[q];
        if (r == 0) psum += ps[q];
      }
    prefix[e] = pre;
    if (r == 0) {
      p.tile_hist[(int64_t)tile * E + e] = tot;
      p.tile_psum[(int64_t)tile * E + e] = psum;
    }
  }
  __syncthreads();
  const int K = p.sel.K;
  for (int i = tid; i < Rv * K; i += kRtThreads) {
    const int t = i / K, k = i - t * K;
    const int e = picks[t * kPickStride + k];
    p.rank_out[(u0 + t) * K + k] = rank[t * kPickStride + k] + prefix[e];
  }
  if (S > 1) cluster_sync_all();  // no CTA leaves while a peer may still read its shared memory
}

// Copy of W_g [h'][E] with its rows padded to Ep columns (zeros past E), for E not a multiple of 8
// or an unaligned W_g: TMA needs 16-byte row strides.
__global__ void __launch_bounds__(256)
router_pad_kernel(const __nv_bfloat16* __restrict__ w, int64_t hu, int E, int Ep, __nv_bfloat16* __restrict__ wp) {
  const int64_t n = hu * Ep;
  for (int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x; i < n; i += (int64_t)gridDim.x * 256) {
    const int64_t k = i / Ep;
    const int e = (int)(i - k * Ep);
    wp[i] = e < E ? w[k * E + e] : __float2bfloat16(0.f);
  }
}

template <int EPL, int KMAX, bool SIGMOID, int FEM>
cudaError_t launch_rt(const CUtensorMap& mX, const CUtensorMap& mW, const RouteTcParams& g, unsigned grid,
                      size_t smem, cudaStream_t s, bool pdl) {
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(route_tc_kernel<EPL, KMAX, SIGMOID, FEM>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)((kRtFastBudget > kRtStageBudget ? kRtFastBudget : kRtStageBudget) + 1024));
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  return launch_kernel(route_tc_kernel<EPL, KMAX, SIGMOID, FEM>, dim3(grid), dim3(rt_threads(FEM)), smem, s,
                       (unsigned)g.S, pdl, mX, mW, g);
}

template <int FEM>
cudaError_t launch_rt_fast(const CUtensorMap& mX, const CUtensorMap& mW, const RouteTcParams& g, int K, unsigned grid,
                           size_t smem, cudaStream_t s, bool pdl) {
  if (K <= 2) return launch_rt<0, 2, false, FEM>(mX, mW, g, grid, smem, s, pdl);
  if (K <= 4) return launch_rt<0, 4, false, FEM>(mX, mW, g, grid, smem, s, pdl);
  return launch_rt<0, 8, false, FEM>(mX, mW, g, grid, smem, s, pdl);
}

}  // namespace

RouterPlan router_plan(const Problem& p, int sms) {
  RouterPlan r;
  r.nblk = (p.E + 63) / 64;
  r.Np = 64 * r.nblk;
  r.m_tiles = (int)((p.Tu + kRtBM - 1) / kRtBM);
  r.nkb = (p.hu + kRtBK - 1) / kRtBK;
  // K slices per tile: about two CTAs per SM stream x, each slice at least one k-block; then as
  // many more as the epilogue's shared memory needs (its logit tile shrinks with 128/S units)
  const int epl = p.E <= 64 ? 0 : (p.E <= 128 ? 4 : 8);
  int S = 1;
  while (S < 8 && (int64_t)r.m_tiles * S * 2 <= 2LL * sms && S * 2 <= r.nkb) S *= 2;
  while (S < 8 && rt_epi(S, p.E, epl).total > (size_t)kRtStageBudget) S *= 2;
  r.S = S;
  r.kbs = (r.nkb + S - 1) / S;
  return r;
}

static bool router_needs_pad(const Problem& p, const void* w_router) {
  return p.E % 8 != 0 || (reinterpret_cast<uintptr_t>(w_router) & 15) != 0;
}

cudaError_t launch_route_tc(const Problem& p, const void* x, const void* w_router, const float* logit_bias,
                            const SelectCtx& sel, float* logits_out, int32_t* rank_out, int32_t* tile_hist,
                            float* tile_psum, void* w_pad, uint32_t* status, cudaStream_t s) {
  if (p.Tu == 0) return cudaSuccess;
  const RouterPlan r = router_plan(p, device_sm_count());
  const void* wsrc = w_router;
  int Ew = p.E;
  bool pdl = false;
  if (router_needs_pad(p, w_router)) {
    Ew = (p.E + 7) / 8 * 8;
    const int64_t n = (int64_t)p.hu * Ew;
    int64_t blocks = (n + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    cudaError_t e = launch_kernel(router_pad_kernel, dim3((unsigned)blocks), dim3(256), 0, s, 1, false,
                                  static_cast<const __nv_bfloat16*>(w_router), (int64_t)p.hu, p.E, Ew,
                                  static_cast<__nv_bfloat16*>(w_pad));
    if (e != cudaSuccess) return e;
    wsrc = w_pad;
    pdl = true;
  }
  CUtensorMap mX, mW;
  if (!encode_tmap_2d_bf16(&mX, x, (uint64_t)p.hu, (uint64_t)p.Tu, kRtBK, kRtBM) ||
      !encode_tmap_2d_bf16(&mW, wsrc, (uint64_t)Ew, (uint64_t)p.hu, 64, kRtBK))
    return cudaErrorInvalidValue;
  RouteTcParams g = {};
  g.Tu = p.Tu;
  g.E = p.E;
  g.Np = r.Np;
  g.nblk = r.nblk;
  g.nkb = r.nkb;
  g.kbs = r.kbs;
  g.S = r.S;
  g.stage_bytes = (uint32_t)(kRtABytes + r.nblk * kRtWBox);
  int stages = (int)(kRtStageBudget / g.stage_bytes);
  g.stages = stages < 2 ? 2 : (stages > kRtMaxStages ? kRtMaxStages : stages);
  g.logit_bias = logit_bias;
  g.logits_out = logits_out;
  g.sel = sel;
  g.rank_out = rank_out;
  g.tile_hist = tile_hist;
  g.tile_psum = tile_psum;
  g.status = status;
  const bool warp_sel = p.E > 64;
  const int epl = !warp_sel ? 0 : (p.E <= 128 ? 4 : 8);
  const unsigned grid = (unsigned)(r.m_tiles * r.S);
  const int kb = p.K <= 2 ? 2 : (p.K <= 4 ? 4 : 8);
  if (!p.sigmoid && p.n_groups == 1 && p.E <= 64) {
    // softmax without a group limit, E <= 64: units routed in registers
    const RtFast F = rt_fast(r.S, p.E);
    int st = (int)((kRtFastBudget - F.total) / g.stage_bytes);
    g.stages = st < 2 ? 2 : (st > kRtMaxStages ? kRtMaxStages : st);
    g.epi_off = (uint32_t)((size_t)g.stages * g.stage_bytes);
    const size_t smem = (size_t)g.epi_off + F.total + 1024;
    if (smem > (size_t)kRtFastBudget + 1024) return cudaErrorInvalidConfiguration;
    if (p.E <= 8) return launch_rt_fast<8>(mX, mW, g, p.K, grid, smem, s, pdl);
    if (p.E <= 16) return launch_rt_fast<16>(mX, mW, g, p.K, grid, smem, s, pdl);
    if (p.E <= 32) return launch_rt_fast<32>(mX, mW, g, p.K, grid, smem, s, pdl);
    return launch_rt_fast<64>(mX, mW, g, p.K, grid, smem, s, pdl);
  }
  g.epi_off = 0;
  const RtEpi L = rt_epi(r.S, p.E, epl);
  size_t smem = (size_t)g.stages * g.stage_bytes;
  if (L.total > smem) smem = L.total;
  smem += 1024;
  if (smem > (size_t)kRtStageBudget + 1024) return cudaErrorInvalidConfiguration;
  if (warp_sel) {
    if (epl == 4) return p.sigmoid ? launch_rt<4, 8, true, 0>(mX, mW, g, grid, smem, s, pdl)
                                   : launch_rt<4, 8, false, 0>(mX, mW, g, grid, smem, s, pdl);
    return p.sigmoid ? launch_rt<8, 8, true, 0>(mX, mW, g, grid, smem, s, pdl)
                     : launch_rt<8, 8, false, 0>(mX, mW, g, grid, smem, s, pdl);
  }
  if (p.sigmoid) {
    if (kb == 2) return launch_rt<0, 2, true, 0>(mX, mW, g, grid, smem, s, pdl);
    if (kb == 4) return launch_rt<0, 4, true, 0>(mX, mW, g, grid, smem, s, pdl);
    return launch_rt<0, 8, true, 0>(mX, mW, g, grid, smem, s, pdl);
  }
  if (kb == 2) return launch_rt<0, 2, false, 0>(mX, mW, g, grid, smem, s, pdl);
  if (kb == 4) return launch_rt<0, 4, false, 0>(mX, mW, g, grid, smem, s, pdl);
  return launch_rt<0, 8, false, 0>(mX, mW, g, grid, smem, s, pdl);
}

}  // namespace moe
