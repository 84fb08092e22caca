// fa_bwd.cu — fused attention backward for sm_103a.
//
// Three launches:
//   bwd_pre   D_i = sum_c dO_ic O_ic, LSE2_i = LSE_i log2(e) (rows padded to a
//             multiple of 128 with LSE2 = +inf, D = 0), dQ accumulator zeroed;
//   bwd_main  one CTA per (batch, kv head, 128-row key/value tile j): K_j, V_j
//             stay in shared memory while every (query head of the group, query
//             tile i) streams past; the P_ij are recomputed from LSE and never
//             leave the SM;
//   bwd_post  dQ = bf16(scale * dQ accumulator).
//
// Per streamed query tile the tensor core runs, accumulating in TMEM:
//   S^T  = K_j Q_i^T            (lanes = key rows)       -> P^T = 2^(S^T c - LSE2)
//   dP^T = V_j dO_i^T                                     -> dS^T = P^T (dP^T - D)
//   dV  += P^T dO_i             (P^T read from TMEM)
//   dK  += dS^T Q_i             (dS^T from shared memory)
//   dQ_i = dS K_j               (same shared-memory dS, read as MN-major)
// and dQ_i is added into the fp32 accumulator with vector reductions.  The
// pages place the backward's bottleneck in shared-memory traffic and its atomic
// dQ updates (FlashAttention-4 article, "Por que el enfoque estandar ya no
// funciona"; FA4 paper summary, section 2.C); this kernel is the one-CTA form
// (the 2-CTA pairing of section 2.C is not used here).
//
// TMEM (512 columns): S^T/P^T at 0, dP^T at 128 (dQ_i reuses these columns once
// dS^T has been formed), dV at 256, dK at 256 + d.  dQ_i sits in the dP^T
// columns so that S^T_{i+1} can start while the drain warps still read dQ_i.
//
// Warp roles: warps 0-3 P/dS (one thread per key row), warps 4-7 dQ drain and
// dK epilogue, warp 8 MMA issue, warp 9 TMA producer.
#include <cuda_bf16.h>

#include "exp2_poly.cuh"
#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

// Opt-in event trace (build with -DFA_TRACE): SM clock at fixed points of the
// first 64 iterations of one CTA, read back with fa_debug_trace().  Off by
// default; the macro then expands to nothing.
#ifdef FA_TRACE
#ifndef FA_TRACE_CTA
#define FA_TRACE_CTA 7
#endif
__device__ unsigned long long g_trace[64][16];
#define FA_TRACE_EV(it, ev)                                                                      \
  do {                                                                                           \
    if (blockIdx.x == FA_TRACE_CTA && blockIdx.y == 0 && blockIdx.z == 0 && (it) < 64)           \
      g_trace[(it)][(ev)] = clock64();                                                           \
  } while (0)
#else
#define FA_TRACE_EV(it, ev) \
  do {                      \
  } while (0)
#endif

// ------------------------------------------------------------------ pre / post
template <int E> struct BfVec;  // E bf16 values loaded at once
template <> struct BfVec<2> { using T = uint32_t; };
template <> struct BfVec<4> { using T = uint2; };
template <> struct BfVec<8> { using T = uint4; };

// One warp per row (b, n, h) of the padded range n < Npad; lane l holds
// elements [l E, l E + E) of the row.
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const __nv_bfloat16 *__restrict__ o,
                                                      const __nv_bfloat16 *__restrict__ dO,
                                                      const float *__restrict__ lse, float *__restrict__ lse2,
                                                      float *__restrict__ delta, float *__restrict__ dq_acc, int B,
                                                      int H, int N, int Npad) {
  constexpr int E = D / 32;
  using V = typename BfVec<E>::T;
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= (long long)B * Npad * H) return;
  const int h = (int)(row % H);
  const long long bn = row / H;
  const int n = (int)(bn % Npad);
  const int b = (int)(bn / Npad);
  const size_t rw = ((size_t)b * H + h) * Npad + n;
  if (n >= N) {
    if (lane == 0) {
      lse2[rw] = INFINITY;  // padded query rows: P = 2^(s - inf) = 0
      delta[rw] = 0.f;
    }
    return;
  }
  const size_t off = (((size_t)b * N + n) * H + h) * D + lane * E;
  const V va = *reinterpret_cast<const V *>(o + off);
  const V vg = *reinterpret_cast<const V *>(dO + off);
  const __nv_bfloat162 *a2 = reinterpret_cast<const __nv_bfloat162 *>(&va);
  const __nv_bfloat162 *g2 = reinterpret_cast<const __nv_bfloat162 *>(&vg);
  float acc = 0.f;
#pragma unroll
  for (int w = 0; w < E / 2; ++w) {
    acc = fmaf(__low2float(a2[w]), __low2float(g2[w]), acc);
    acc = fmaf(__high2float(a2[w]), __high2float(g2[w]), acc);
  }
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
  float *acc_row = dq_acc + (((size_t)b * N + n) * H + h) * D;
#pragma unroll
  for (int c = lane * 4; c < D; c += 128) *reinterpret_cast<float4 *>(acc_row + c) = make_float4(0.f, 0.f, 0.f, 0.f);
  if (lane == 0) {
    lse2[rw] = lse[((size_t)b * H + h) * N + n] * kLog2e;
    delta[rw] = acc;
  }
}

// dq = bf16(scale * acc), 8 elements per thread.
__global__ void __launch_bounds__(256) bwd_post_kernel(const float *__restrict__ acc, __nv_bfloat16 *__restrict__ dq,
                                                       long long n8, float scale) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n8) return;
  const float4 a = reinterpret_cast<const float4 *>(acc)[2 * i];
  const float4 c = reinterpret_cast<const float4 *>(acc)[2 * i + 1];
  uint4 w;
  w.x = pack_bf16x2(a.x * scale, a.y * scale);
  w.y = pack_bf16x2(a.z * scale, a.w * scale);
  w.z = pack_bf16x2(c.x * scale, c.y * scale);
  w.w = pack_bf16x2(c.z * scale, c.w * scale);
  reinterpret_cast<uint4 *>(dq)[i] = w;
}

// ------------------------------------------------------------------ main kernel
template <int D>
struct BwdCfg {
  static constexpr int kTile = 128 * D * 2;  // one 128-row bf16 tile
  static constexpr int kStages = 2;          // (Q_i, dO_i, LSE2_i, D_i) ring depth
  static constexpr int kThreads = 448;
  static constexpr int kDrainWarp0 = 8, kMmaWarp = 12, kLoadWarp = 13;
  static constexpr int kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D;
  static constexpr int kTmemCols = 512;
  static_assert(kColDK + D <= kTmemCols, "TMEM budget");
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kTile;
  static constexpr int kOffStage = 2 * kTile;  // stage s: Q at +2s*kTile, dO at +(2s+1)*kTile
  static constexpr int kOffDS = kOffStage + 2 * kStages * kTile;  // dS^T 128 x 128 bf16; also dQ staging
  static constexpr int kOffRows = kOffDS + 128 * 128 * 2;          // stage s: LSE2 at +1024s, D at +1024s+512
  enum { kBarKV, kBarFull0, kBarEmpty0 = kBarFull0 + kStages, kBarS = kBarEmpty0 + kStages, kBarDP, kBarP, kBarDS,
         kBarDQFull, kBarDQEmpty, kBarStageFree, kBarFinal, kBarDrain, kNumBars };
  static constexpr int kOffBar = kOffRows + 1024 * kStages;
  static constexpr int kOffMisc = kOffBar + 8 * kNumBars;
  static constexpr int kSmemBytes = kOffMisc + 16;  // base must be 1024-aligned (checked in the kernel)
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

enum BwdSite : int {
  kBSiteKV = 11, kBSiteFull = 12, kBSiteEmpty = 13, kBSiteS = 14, kBSiteDP = 15, kBSiteP = 16, kBSiteDS = 17,
  kBSiteStageFree = 18, kBSiteDQFull = 19, kBSiteDQEmpty = 20, kBSiteFinal = 21, kBSiteDrain = 22, kBSiteAlign = 23
};

// Writes 16 packed bf16 pairs (32 columns starting at col0) of row r into a
// 128B-swizzled bf16 tile made of 64-column boxes of 128 rows (16 KB each).
__device__ __forceinline__ void st_swizzled_32cols(uint8_t *tile, int r, int col0, const uint32_t (&w)[16]) {
  const int box = col0 >> 6;
  const int chunk0 = (col0 & 63) >> 3;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int chunk = (chunk0 + k) ^ (r & 7);
    *reinterpret_cast<uint4 *>(tile + box * 16384 + r * 128 + chunk * 16) =
        make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
  }
}

// Writes 32 fp32 of row r into one 128B-swizzled fp32 box (32 columns x 128 rows, 16 KB).
__device__ __forceinline__ void st_swizzled_f32_box(uint8_t *box, int r, const uint32_t (&v)[32]) {
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int chunk = k ^ (r & 7);
    *reinterpret_cast<uint4 *>(box + r * 128 + chunk * 16) = make_uint4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
  }
}

__device__ __forceinline__ void tma_reduce_add_4d(const void *map, uint32_t src, int c0, int c1, int c2, int c3) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.4d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(map),
      "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(448, 1) bwd_main_kernel(const __grid_constant__ BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::kOffBar;
  auto bar = [&](int i) { return bar0 + 8u * i; };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 4);
  const WaitCtx wctx{abort_flag, p.status};
  if ((sbase & 1023u) != 0) {  // swizzled tiles need 1024-byte alignment
    if (threadIdx.x == 0) {
      atomicOr(p.status, 1u);
      atomicCAS(p.status + 1, 0u, (unsigned)kBSiteAlign);
    }
    return;
  }

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int jt = blockIdx.x;  // key/value tile
  const int kh = blockIdx.y, b = blockIdx.z;
  const int g = p.H / p.Hkv;
  const int n_q = (p.N + 127) / 128;
  const int Npad = n_q * 128;
  const int i_start = CAUSAL ? jt : 0;
  const int per_head = n_q - i_start;
  const int n_iter = g * per_head;  // (head, query tile) pairs, head-major
  const int kv0 = jt * 128;
  // Each key tile walks the query tiles from a different starting point, so
  // that the CTAs of one head, which run together, reduce into different dQ
  // rows at any moment instead of all into the same ones.
  const int rot = (int)(((unsigned)jt * 2654435761u) % (unsigned)per_head);
  auto q_tile = [&](int it) { return i_start + (it % per_head + rot) % per_head; };

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kNumBars; ++i) {
      uint32_t count = 1;
      if (i == C::kBarP || i == C::kBarDS) count = 256;  // both P/dS warpgroups
      if (i == C::kBarDQEmpty) count = 128;              // the drain warpgroup
      mbar_init(bar(i), count);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == C::kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  if (warp == C::kLoadWarp && lane == 0) {
    prefetch_tmap(&p.tm_q);
    prefetch_tmap(&p.tm_k);
    prefetch_tmap(&p.tm_v);
    prefetch_tmap(&p.tm_do);
    prefetch_tmap(&p.tm_dqacc);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 8) {
    // ===================================================== P^T and dS^T, one warpgroup per 64 query columns
    const int wg = warp >> 2;         // query columns [64 wg, 64 wg + 64)
    const int r = threadIdx.x & 127;  // key row within the tile == TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t s_tm = tmem + lane_off + C::kColS + 64 * wg;   // this warpgroup's S^T columns
    const uint32_t p_tm = s_tm;                                   // P^T (bf16) over their first 32
    const uint32_t dp_tm = tmem + lane_off + C::kColDP + 64 * wg;
    const int kv_row = kv0 + r;
    const bool row_valid = kv_row < p.N;
    uint8_t *ds_tile = smem + C::kOffDS;
    bool ok = true;
    for (int it = 0; it < n_iter && ok; ++it) {
      const int st = it % C::kStages;
      const int i = q_tile(it);
      const float *lse2_s = reinterpret_cast<const float *>(smem + C::kOffRows + 1024 * st) + 64 * wg;
      const float *dlt_s = lse2_s + 128;
      // ---- P^T = 2^(S^T c - LSE2), masked; bf16 into TMEM over S^T
      ok = mbar_wait_warp(bar(C::kBarS), it & 1, wctx, kBSiteS);
      if (!ok) break;
      if (threadIdx.x == 0) FA_TRACE_EV(it, 0);
      tc_fence_after();
      const bool diag = CAUSAL && (i == jt);
      uint32_t sv[2][32];
      tmem_ld_32x32b_x32(s_tm, sv[0]);
      tmem_ld_32x32b_x32(s_tm + 32, sv[1]);
      tmem_wait_ld(sv[0]);
      reg_tie(sv[1]);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t w[16];
#pragma unroll
        for (int k = 0; k < 32; k += 4) {
          const float4 l4 = *reinterpret_cast<const float4 *>(lse2_s + 32 * c + k);
          float pe[4];
          pe[0] = ex2_mufu(fmaf(__uint_as_float(sv[c][k]), p.scale_log2, -l4.x));
          pe[1] = ex2_mufu(fmaf(__uint_as_float(sv[c][k + 1]), p.scale_log2, -l4.y));
          pe[2] = ex2_mufu(fmaf(__uint_as_float(sv[c][k + 2]), p.scale_log2, -l4.z));
          pe[3] = ex2_mufu(fmaf(__uint_as_float(sv[c][k + 3]), p.scale_log2, -l4.w));
          const int qc = 64 * wg + 32 * c + k;  // query column within tile i
#pragma unroll
          for (int u = 0; u < 4; ++u)
            if (!row_valid || (diag && qc + u < r)) pe[u] = 0.f;
          w[k >> 1] = pack_bf16x2(pe[0], pe[1]);
          w[(k >> 1) + 1] = pack_bf16x2(pe[2], pe[3]);
        }
        tmem_st_32x32b_x16(p_tm + 16 * c, w);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(C::kBarP));
      if (threadIdx.x == 0) FA_TRACE_EV(it, 1);
      // ---- dS^T = P^T (dP^T - D) -> shared memory (bf16, 128B swizzle, box = wg)
      ok = mbar_wait_warp(bar(C::kBarDP), it & 1, wctx, kBSiteDP);
      if (threadIdx.x == 0) FA_TRACE_EV(it, 2);
      if (ok && it > 0) ok = mbar_wait_warp(bar(C::kBarStageFree), (it - 1) & 1, wctx, kBSiteStageFree);
      if (!ok) break;
      if (threadIdx.x == 0) FA_TRACE_EV(it, 3);
      tc_fence_after();
      uint32_t dpv[2][32], pv[32];
      tmem_ld_32x32b_x32(dp_tm, dpv[0]);
      tmem_ld_32x32b_x32(dp_tm + 32, dpv[1]);
      tmem_ld_32x32b_x32(p_tm, pv);
      tmem_wait_ld(dpv[0]);
      reg_tie(dpv[1]);
      reg_tie(pv);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t w[16];
#pragma unroll
        for (int k = 0; k < 32; k += 4) {
          const float4 d4 = *reinterpret_cast<const float4 *>(dlt_s + 32 * c + k);
          const __nv_bfloat162 p01 = *reinterpret_cast<const __nv_bfloat162 *>(&pv[16 * c + (k >> 1)]);
          const __nv_bfloat162 p23 = *reinterpret_cast<const __nv_bfloat162 *>(&pv[16 * c + (k >> 1) + 1]);
          const float ds0 = __low2float(p01) * (__uint_as_float(dpv[c][k]) - d4.x);
          const float ds1 = __high2float(p01) * (__uint_as_float(dpv[c][k + 1]) - d4.y);
          const float ds2 = __low2float(p23) * (__uint_as_float(dpv[c][k + 2]) - d4.z);
          const float ds3 = __high2float(p23) * (__uint_as_float(dpv[c][k + 3]) - d4.w);
          w[k >> 1] = pack_bf16x2(ds0, ds1);
          w[(k >> 1) + 1] = pack_bf16x2(ds2, ds3);
        }
        st_swizzled_32cols(ds_tile, r, 64 * wg + 32 * c, w);
      }
      fence_proxy_async_smem();  // generic-proxy writes -> visible to the MMA (async proxy)
      tc_fence_before();
      mbar_arrive(bar(C::kBarDS));
      if (threadIdx.x == 0) FA_TRACE_EV(it, 4);
    }
    // ---- epilogue: warpgroup 0 stores dV, warpgroup 1 stores dK * scale (via stage 0's Q / dO slots)
    if (ok) ok = mbar_wait_warp(bar(C::kBarFinal), 0, wctx, kBSiteFinal);
    tc_fence_after();
    uint8_t *stage = smem + C::kOffStage + wg * C::kTile;
    const uint32_t acc_tm = tmem + lane_off + (wg == 0 ? C::kColDV : C::kColDK);
    const float mul = wg == 0 ? 1.0f : p.scale;
    if (ok) {
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(acc_tm + 32 * c, v);
        tmem_wait_ld(v);
        uint32_t w[16];
#pragma unroll
        for (int k = 0; k < 16; ++k)
          w[k] = pack_bf16x2(__uint_as_float(v[2 * k]) * mul, __uint_as_float(v[2 * k + 1]) * mul);
        st_swizzled_32cols(stage, r, 32 * c, w);
      }
    }
    fence_proxy_async_smem();
    if (wg == 0) named_bar_sync(1, 128);
    else named_bar_sync(2, 128);
    if (r == 0 && ok) {
      const CUtensorMap *map = wg == 0 ? &p.tm_dv : &p.tm_dk;
      for (int bx = 0; bx < D / 64; ++bx) tma_store_4d(map, smem_u32(stage) + bx * 16384, bx * 64, kh, kv0, b);
      bulk_commit();
      bulk_wait_read_all();
    }
  } else if (warp < C::kMmaWarp) {
    // ===================================================== dQ drain: TMEM -> staging (dS tile) -> TMA reduce-add
    const int r = threadIdx.x - 256;  // query row within tile i == TMEM lane
    const uint32_t lane_off = (uint32_t)((warp - C::kDrainWarp0) * 32) << 16;
    const uint32_t dq_tm = tmem + lane_off + C::kColDP;
    uint8_t *staging = smem + C::kOffDS;  // free from dQ_i's completion until dS_{i+1} is written
    // Every thread of this warpgroup runs every iteration (and every named
    // barrier in it), also after an abort, so the barriers always match; waits
    // return at once once the abort flag is set.
    bool ok = true;
    for (int it = 0; it < n_iter; ++it) {
      const int hh = kh * g + it / per_head;
      const int i = q_tile(it);
      if (ok) ok = mbar_wait_warp(bar(C::kBarDQFull), it & 1, wctx, kBSiteDQFull);
      if (r == 0) FA_TRACE_EV(it, 5);
      tc_fence_after();
#pragma unroll
      for (int half = 0; half < D / 64; ++half) {
        uint32_t v[2][32];
        if (ok) {
          tmem_ld_32x32b_x32(dq_tm + 64 * half, v[0]);
          tmem_ld_32x32b_x32(dq_tm + 64 * half + 32, v[1]);
          tmem_wait_ld(v[0]);
          reg_tie(v[1]);
          if (half == D / 64 - 1) {  // every TMEM read of dQ_i done: dP^T_{i+1} may overwrite it
            tc_fence_before();
            mbar_arrive(bar(C::kBarDQEmpty));
          }
          st_swizzled_f32_box(staging, r, v[0]);
          st_swizzled_f32_box(staging + 16384, r, v[1]);
        }
        fence_proxy_async_smem();
        named_bar_sync(3, 128);
        if (r == 0 && !*abort_flag) {
          const uint32_t src = smem_u32(staging);
          tma_reduce_add_4d(&p.tm_dqacc, src, 64 * half, hh, i * 128, b);
          tma_reduce_add_4d(&p.tm_dqacc, src + 16384, 64 * half + 32, hh, i * 128, b);
          bulk_commit();
          bulk_wait_read_all();  // staging may be overwritten once the copies have read it
          FA_TRACE_EV(it, 12 + half);
        }
        named_bar_sync(3, 128);
      }
      if (r == 0) mbar_arrive(bar(C::kBarStageFree));
      if (r == 0) FA_TRACE_EV(it, 6);
    }
    if (threadIdx.x == 256) bulk_wait_all();  // reductions complete before the CTA exits
  } else if (warp == C::kMmaWarp) {
    // ===================================================== MMA issue
    if (lane == 0) {
      constexpr uint32_t id_kk = make_idesc_bf16(128, 128, false, false);  // S^T, dP^T
      constexpr uint32_t id_dv = make_idesc_bf16(128, D, false, true);     // dV (A in TMEM), dK
      constexpr uint32_t id_dq = make_idesc_bf16(128, D, true, true);      // dQ: A = dS MN-major
      const uint32_t k_s = sbase + C::kOffK, v_s = sbase + C::kOffV, ds_s = sbase + C::kOffDS;
      bool ok = mbar_wait(bar(C::kBarKV), 0, wctx, kBSiteKV);
      for (int it = 0; it < n_iter && ok; ++it) {
        const int st = it % C::kStages;
        const uint32_t q_s = sbase + C::kOffStage + 2 * st * C::kTile, do_s = q_s + C::kTile;
        ok = mbar_wait(bar(C::kBarFull0 + st), (it / C::kStages) & 1, wctx, kBSiteFull);
        if (!ok) break;
        FA_TRACE_EV(it, 7);
        tc_fence_after();
        // S^T = K Q^T   (both K-major, K dim = d)
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_ss(tmem + C::kColS, make_sdesc_sw128(k_s + off, 0, 1024), make_sdesc_sw128(q_s + off, 0, 1024), id_kk,
                 kk > 0);
        }
        tc_commit(bar(C::kBarS));
        // dP^T = V dO^T  (into the dP columns: dQ_{i-1} must have been read out)
        if (it > 0) ok = mbar_wait(bar(C::kBarDQEmpty), (it - 1) & 1, wctx, kBSiteDQEmpty);
        if (!ok) break;
        FA_TRACE_EV(it, 8);
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_ss(tmem + C::kColDP, make_sdesc_sw128(v_s + off, 0, 1024), make_sdesc_sw128(do_s + off, 0, 1024),
                 id_kk, kk > 0);
        }
        tc_commit(bar(C::kBarDP));
        // dV += P^T dO   (A = P^T in TMEM: query columns 64w..64w+63 at column 64w, two bf16 per column)
        ok = mbar_wait(bar(C::kBarP), it & 1, wctx, kBSiteP);
        if (!ok) break;
        FA_TRACE_EV(it, 9);
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts(tmem + C::kColDV, tmem + C::kColS + 64u * (kk >> 2) + 8u * (kk & 3),
                 make_sdesc_sw128(do_s + kk * 2048, 16384, 1024), id_dv, (it > 0 || kk > 0));
        // dK += dS^T Q  (A = dS^T K-major [key][query]; B = Q MN-major)
        ok = mbar_wait(bar(C::kBarDS), it & 1, wctx, kBSiteDS);
        if (!ok) break;
        FA_TRACE_EV(it, 10);
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_ss(tmem + C::kColDK, make_sdesc_sw128(ds_s + off, 0, 1024),
                 make_sdesc_sw128(q_s + kk * 2048, 16384, 1024), id_dv, (it > 0 || kk > 0));
        }
        // dQ_i = dS K   (A = the same dS^T tile read MN-major; B = K MN-major)
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ss(tmem + C::kColDP, make_sdesc_sw128(ds_s + kk * 2048, 16384, 1024),
                 make_sdesc_sw128(k_s + kk * 2048, 16384, 1024), id_dq, kk > 0);
        tc_commit(bar(C::kBarDQFull));
        tc_commit(bar(C::kBarEmpty0 + st));
        FA_TRACE_EV(it, 11);
      }
      tc_commit(bar(C::kBarFinal));
      tc_commit(bar(C::kBarDrain));
      if (!mbar_wait(bar(C::kBarDrain), 0, wctx, kBSiteDrain) && *abort_flag) {
        const uint64_t t0 = global_timer_ns();
        while (!mbar_test(bar(C::kBarDrain), 0) && global_timer_ns() - t0 < kWaitLimitNs) {}
      }
    }
  } else {
    // ===================================================== TMA producer
    if (lane == 0) {
      const uint64_t keep = policy_evict_last();   // Q, dO, LSE2, D are re-read by every key tile
      mbar_arrive_expect_tx(bar(C::kBarKV), 2 * C::kTile);
      for (int bx = 0; bx < D / 64; ++bx) {
        tma_load_4d(sbase + C::kOffK + bx * 16384, &p.tm_k, bar(C::kBarKV), bx * 64, kh, kv0, b);
        tma_load_4d(sbase + C::kOffV + bx * 16384, &p.tm_v, bar(C::kBarKV), bx * 64, kh, kv0, b);
      }
      bool ok = true;
      int it = 0;
      for (; it < n_iter && ok; ++it) {
        const int st = it % C::kStages;
        const int hh = kh * g + it / per_head;
        const int i = q_tile(it);
        ok = mbar_wait(bar(C::kBarEmpty0 + st), ((it / C::kStages) & 1) ^ 1, wctx, kBSiteEmpty);
        if (!ok) break;
        const uint32_t fb = bar(C::kBarFull0 + st);
        mbar_arrive_expect_tx(fb, 2 * C::kTile + 1024);
        const uint32_t q_s = sbase + C::kOffStage + 2 * st * C::kTile;
        for (int bx = 0; bx < D / 64; ++bx) {
          tma_load_4d_hint(q_s + bx * 16384, &p.tm_q, fb, bx * 64, hh, i * 128, b, keep);
          tma_load_4d_hint(q_s + C::kTile + bx * 16384, &p.tm_do, fb, bx * 64, hh, i * 128, b, keep);
        }
        const size_t roff = ((size_t)b * p.H + hh) * Npad + (size_t)i * 128;
        bulk_load(sbase + C::kOffRows + 1024 * st, p.lse2 + roff, 512, fb);
        bulk_load(sbase + C::kOffRows + 1024 * st + 512, p.delta + roff, 512, fb);
      }
      const uint64_t t0 = global_timer_ns();
      for (int f = max(0, it - C::kStages); f < it; ++f)
        while (!mbar_test(bar(C::kBarFull0 + f % C::kStages), (f / C::kStages) & 1) &&
               global_timer_ns() - t0 < kWaitLimitNs) {}
      while (!mbar_test(bar(C::kBarKV), 0) && global_timer_ns() - t0 < kWaitLimitNs) {}
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D, bool CAUSAL>
int launch_main(const BwdParams &p, cudaStream_t stream) {
  using C = BwdCfg<D>;
  auto kern = bwd_main_kernel<D, CAUSAL>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) != cudaSuccess)
    return FA_ERR_CUDA;
  dim3 grid((p.N + 127) / 128, p.Hkv, p.B);
  kern<<<grid, C::kThreads, C::kSmemBytes, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

template <int D>
int launch_pre_t(const BwdParams &p, const void *o, const void *dO, const float *lse, cudaStream_t stream) {
  const int Npad = (p.N + 127) / 128 * 128;
  const long long rows = (long long)p.B * Npad * p.H;
  bwd_pre_kernel<D><<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(
      static_cast<const __nv_bfloat16 *>(o), static_cast<const __nv_bfloat16 *>(dO), lse, p.lse2,
      const_cast<float *>(p.delta), p.dq_acc, p.B, p.H, p.N, Npad);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

int launch_bwd_pre(const BwdParams &p, int d, const void *o, const void *dO, const float *lse, cudaStream_t stream) {
  switch (d) {
    case 64: return launch_pre_t<64>(p, o, dO, lse, stream);
    case 128: return launch_pre_t<128>(p, o, dO, lse, stream);
    default: return FA_ERR_UNSUPPORTED;
  }
}

int launch_bwd_main(const BwdParams &p, int d, bool causal, cudaStream_t stream) {
  switch (d) {
    case 64: return causal ? launch_main<64, true>(p, stream) : launch_main<64, false>(p, stream);
    case 128: return causal ? launch_main<128, true>(p, stream) : launch_main<128, false>(p, stream);
    default: return FA_ERR_UNSUPPORTED;
  }
}

int launch_bwd_post(const BwdParams &p, int d, void *dq, cudaStream_t stream) {
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  const long long n8 = (long long)p.B * p.N * p.H * d / 8;
  bwd_post_kernel<<<(unsigned)((n8 + 255) / 256), 256, 0, stream>>>(p.dq_acc, static_cast<__nv_bfloat16 *>(dq), n8,
                                                                     p.scale);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace fa

#ifdef FA_TRACE
extern "C" int fa_debug_trace(unsigned long long *host_out) {
  return cudaMemcpyFromSymbol(host_out, fa::g_trace, sizeof(fa::g_trace)) == cudaSuccess ? 0 : -5;
}
#endif
