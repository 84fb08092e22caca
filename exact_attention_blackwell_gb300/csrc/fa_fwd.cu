// fa_fwd.cu — fused attention forward for sm_103a.
//
// One CTA owns QT query tiles of 128 rows of one (batch, head) and streams the
// key/value blocks of 128 rows past them:
//   S_t = Q_t K_j^T      tcgen05 MMA, accumulated in TMEM          (FA4 paper
//   P_t = 2^(S_t - m)    softmax warps, online row max / row sum    summary,
//   O_t += P_t V_j       tcgen05 MMA, P read from TMEM             section 2.A)
// so the N x N scores never leave the SM (FlashAttention-3 page, "FlashAttention
// y FlashAttention-2": tiling plus fusion).
//
// Warp roles (FA4 paper summary, section 2.A: producers, softmax consumers,
// specialised warps; FlashAttention-3 page, section 1: producer/consumer warps):
//   warps 0..4*QT-1 : softmax, one warpgroup per query tile, one thread per row;
//                     also the conditional O rescale and the epilogue
//   warp  4*QT      : MMA issue (one thread) and TMEM allocation
//   warp  4*QT+1    : TMA producer (one thread): Q once, then K_j, V_j into a
//                     STAGES-deep shared-memory ring
//
// MMA order per key block j (two query tiles):  PV_0,j  S_0,j+1  PV_1,j  S_1,j+1
// so that each softmax warpgroup works while the tensor core runs the other
// tile's two MMAs (the ping-pong idea of the FlashAttention-3 page, section 1,
// carried over to asynchronous tcgen05 MMAs).  P_t is written over the first 64
// columns of S_t in TMEM; the tensor pipe executes one thread's MMAs in order, so
// S_t,j+1 never overwrites P_t,j before PV_t,j has read it.
//
// Softmax (FA4 paper summary, section 2.B): 2^x on MUFU.EX2 for most columns and
// on the FMA pipe (exp2_poly) for FA_FWD_POLY_PER16 of every 16; the running
// maximum m_ref is only moved (with an O rescale) when a new block's maximum
// exceeds it by more than kRescaleTau.  The result is exact either way: O and l
// share the same stale m_ref, and O / l and m_ref + log2 l are what is stored.
#include <cuda_bf16.h>

#include "exp2_poly.cuh"
#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

// Opt-in event trace (build with -DFA_TRACE): SM clock at fixed points of the
// first 64 key blocks of one CTA, read back with fa_debug_trace_fwd().
#ifdef FA_TRACE
#ifndef FA_TRACE_CTA
#define FA_TRACE_CTA 7
#endif
__device__ unsigned long long g_trace_fwd[64][16];
// Lifecycle of CTA FA_TRACE_CTA (SM clock), and for every CTA its SM and the
// global timer at entry and exit.
__device__ unsigned long long g_life_fwd[16];
__device__ unsigned long long g_cta_fwd[65536][3];
#define FA_LIFE(ev)                                                   \
  do {                                                                \
    if (blockIdx.x == FA_TRACE_CTA) g_life_fwd[(ev)] = clock64();     \
  } while (0)
#define FA_CTA_MARK(slot)                                                       \
  do {                                                                          \
    if (threadIdx.x == 0 && blockIdx.x < 65536) {                               \
      unsigned sm_;                                                             \
      asm volatile("mov.u32 %0, %%smid;" : "=r"(sm_));                          \
      g_cta_fwd[blockIdx.x][0] = sm_;                                           \
      g_cta_fwd[blockIdx.x][(slot)] = global_timer_ns();                        \
    }                                                                           \
  } while (0)
#define FA_TRACE_EV(j, ev)                                                                       \
  do {                                                                                           \
    if (blockIdx.x == FA_TRACE_CTA && (j) < 64)                                                 \
      g_trace_fwd[(j)][(ev)] = clock64();                                                        \
  } while (0)
#else
#define FA_TRACE_EV(j, ev) \
  do {                     \
  } while (0)
#define FA_LIFE(ev) \
  do {              \
  } while (0)
#define FA_CTA_MARK(slot) \
  do {                    \
  } while (0)
#endif

template <int D, int QT_ = (D <= 128) ? 2 : 1>
struct FwdCfg {
  static constexpr int kQT = QT_;  // query tiles per CTA
  // Short form (head dim <= 128, one query tile): half the TMEM and under half
  // the shared memory, so two CTAs share an SM and one's set-up and epilogue
  // overlap the other's main loop; the launcher takes it for short sequences
  // at head dim 64.
  static constexpr bool kShort = D <= 128 && QT_ == 1;
  static constexpr int kMinBlocks = kShort ? 2 : 1;
  static constexpr int kStages = kShort ? (D == 64 ? 5 : 2) : (D == 64) ? 6 : (D == 128 ? 4 : 2);
  static constexpr int kTileBytes = 128 * D * 2;  // one 128-row tile of Q, K, V or O
  static constexpr int kBoxes = D / 64;           // 64-column TMA boxes per tile (16 KB each)
  static constexpr int kThreads = 128 * kQT + 64;
  static constexpr int kMmaWarp = 4 * kQT;
  static constexpr int kLoadWarp = 4 * kQT + 1;
  static constexpr int kOCol = 128 * kQT;  // TMEM column of O_0 (S_t at 128 t)
  static constexpr int kTmemCols = kShort ? 256 : 512;
  static_assert(kOCol + kQT * D <= kTmemCols, "TMEM budget");
  // shared memory (offsets from a 1024-aligned base)
  static constexpr int kOffQ = 0;
  static constexpr int kOffRing = kQT * kTileBytes;
  static constexpr int kOffBar = kOffRing + kStages * kTileBytes;
  // barriers: full[S], empty[S], q_full, s_full[QT], p_full[QT], o_full[QT], drain
  static constexpr int kNumBars = 2 * kStages + 2 + 3 * kQT;
  static constexpr int kOffMisc = kOffBar + 8 * kNumBars;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + alignment slack
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
  static_assert(kMinBlocks == 1 || kMinBlocks * (kSmemBytes + 1024) <= 228 * 1024, "two CTAs per SM");
};

FA_STALL_FLAG_DECL

enum WaitSite : int {
  kSiteQ = 1, kSiteKFull = 2, kSiteVFull = 3, kSitePFull = 4, kSiteEmpty = 5,
  kSiteSFull = 6, kSiteOFull = 7, kSiteDrain = 8
};

template <int D, bool CAUSAL, int POLY16, bool VARLEN, int QT_>
__global__ void __launch_bounds__(FwdCfg<D, QT_>::kThreads, FwdCfg<D, QT_>::kMinBlocks)
    fa_fwd_kernel(const __grid_constant__ FwdParams p) {
  using C = FwdCfg<D, QT_>;
  constexpr int QT = C::kQT;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::kOffBar;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (C::kStages + s); };
  const uint32_t q_bar = bar0 + 8u * (2 * C::kStages);
  auto s_bar = [&](int t) { return bar0 + 8u * (2 * C::kStages + 1 + t); };
  auto p_bar = [&](int t) { return bar0 + 8u * (2 * C::kStages + 1 + QT + t); };
  auto o_bar = [&](int t) { return bar0 + 8u * (2 * C::kStages + 1 + 2 * QT + t); };
  const uint32_t drain_bar = bar0 + 8u * (2 * C::kStages + 1 + 3 * QT);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 4);
  const WaitCtx wctx{abort_flag, p.status};
  FA_CTA_MARK(1);
  if (threadIdx.x == 0) FA_LIFE(0);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_groups = (p.N + 128 * QT - 1) / (128 * QT);
  int rank, head;
  work_order((int)blockIdx.x, n_groups, p.B * p.H, p.sched_chunk, rank, head);
  const int group = CAUSAL ? n_groups - 1 - rank : rank;  // causal: the longest query rows first
  const int h = head % p.H, b = head / p.H;
  const int kh = h / (p.H / p.Hkv);
  const SeqSpan sq = VARLEN ? seq_span(p.cu_seqlens, b, p.N, p.total) : SeqSpan{0, p.N, b};
  const int L = sq.len;  // rows of this sequence (queries and keys)
  const int n_kv_all = (L + 127) / 128;

  int q0[QT], nb[QT];
  int nb_max = 0;
#pragma unroll
  for (int t = 0; t < QT; ++t) {
    q0[t] = (group * QT + t) * 128;
    if (q0[t] >= L) nb[t] = 0;
    else nb[t] = CAUSAL ? (min(q0[t] + 127, L - 1) / 128 + 1) : n_kv_all;
    nb_max = max(nb_max, nb[t]);
  }

  if (threadIdx.x == 0) {
    // p_full[t] collects one arrival per softmax warp; every other barrier one.
    for (int i = 0; i < C::kNumBars; ++i) {
      const uint32_t bar = bar0 + 8u * i;
      const bool is_p = bar >= p_bar(0) && bar < p_bar(0) + 8u * QT;
      mbar_init(bar, is_p ? 4u : 1u);
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
    prefetch_tmap(&p.tm_o);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (threadIdx.x == 0) FA_LIFE(1);

  if (warp < 4 * QT) {
    // ===================================================== softmax warpgroups
    const int t = warp >> 2;
    const int r = threadIdx.x & 127;  // row within the tile == TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t s_tm = tmem + lane_off + 128u * t;
    const uint32_t o_tm = tmem + lane_off + C::kOCol + (uint32_t)(D * t);
    const int q_row = q0[t] + r;
    const float c2 = p.scale_log2;
    float m_ref = -INFINITY;  // running maximum, scaled log2 units
    float l_sum = 0.f;        // running row sum relative to m_ref
    bool ok = true;
    unsigned rescales = 0;

    for (int j = 0; j < nb[t] && ok; ++j) {
      ok = mbar_wait_warp(s_bar(t), j & 1, wctx, kSiteSFull);
      if (!ok) break;
      if (r == 0) FA_TRACE_EV(j, 0 + 4 * t);
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld_32x32b_x32(s_tm + 32 * c, sr[c]);
      tmem_wait_ld(sr[0]);
      reg_tie(sr[1]);
      reg_tie(sr[2]);
      reg_tie(sr[3]);
      float s[128];
#pragma unroll
      for (int c = 0; c < 128; ++c) s[c] = __uint_as_float(sr[c >> 5][c & 31]);
      if (r == 0) FA_TRACE_EV(j, 1 + 4 * t);

      const int kv0 = j * 128;
      const bool need_mask = (kv0 + 128 > L) || (CAUSAL && kv0 + 127 > q0[t]);
      if (need_mask) {
        const int lim = CAUSAL ? min(L - 1, q_row) - kv0 : L - 1 - kv0;  // last visible column
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c > lim) s[c] = -INFINITY;
      }
      // row maximum: four independent chains of 3-input max
      float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
      for (int c = 4; c < 124; c += 8) {
        mx0 = fmax3(mx0, s[c], s[c + 1]);
        mx1 = fmax3(mx1, s[c + 2], s[c + 3]);
        mx2 = fmax3(mx2, s[c + 4], s[c + 5]);
        mx3 = fmax3(mx3, s[c + 6], s[c + 7]);
      }
      mx0 = fmax3(mx0, s[124], s[125]);
      mx1 = fmax3(mx1, s[126], s[127]);
      const float m_blk = fmax3(mx0, mx1, fmaxf(mx2, mx3)) * c2;
      if (j == 0) {
        m_ref = m_blk;
      } else {
        const bool need = (m_blk - m_ref) > kRescaleTau;
        if (__any_sync(0xffffffffu, need)) {
          // Whole warp rescales (tcgen05.ld/st are warp-collective); rows whose
          // maximum did not move use alpha = 1.  PV_t,j-1 is complete: its
          // commit preceded S_t,j's.  32 columns per TMEM round trip.  (Scaling
          // O after P is stored instead, when the scores' registers are free,
          // measured 5 % faster on inputs with outliers and 5 % slower on the
          // headline shape: the extra live state through the exponential loop
          // costs registers at this kernel's 168-register cap.)
          const float m_new = fmaxf(m_ref, m_blk);
          const float alpha = ex2_mufu(m_ref - m_new);
          m_ref = m_new;
          l_sum *= alpha;
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld_32x32b_x32(o_tm + 32 * c, o);
            tmem_wait_ld(o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st_32x32b_x32(o_tm + 32 * c, o);
          }
          rescales += (lane == 0);
        }
      }
      if (r == 0) FA_TRACE_EV(j, 2 + 4 * t);
      const float neg_m = -m_ref;
      // p = 2^(s c - m): scale-shift two columns per packed FMA; row sum in
      // two packed accumulators
      float l0 = 0.f, l1 = 0.f, l2 = 0.f, l3 = 0.f;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 64; c += 4) {
          float x[4], e[4];
          ffma2(x[0], x[1], s[64 * half + c], s[64 * half + c + 1], c2, c2, neg_m, neg_m);
          ffma2(x[2], x[3], s[64 * half + c + 2], s[64 * half + c + 3], c2, c2, neg_m, neg_m);
#pragma unroll
          for (int u = 0; u < 4; ++u) e[u] = ((c + u) % 16 < POLY16) ? exp2_poly(x[u]) : ex2_mufu(x[u]);
          fadd2(l0, l1, l0, l1, e[0], e[1]);
          fadd2(l2, l3, l2, l3, e[2], e[3]);
          pk[c >> 1] = pack_bf16x2(e[0], e[1]);
          pk[(c >> 1) + 1] = pack_bf16x2(e[2], e[3]);
        }
        tmem_st_32x32b_x32(s_tm + 32 * half, pk);
      }
      l_sum += (l0 + l1) + (l2 + l3);
      tmem_wait_st();
      tc_fence_before();
      if (!(FA_STALL(1) && j == 0 && t == 0)) mbar_arrive_warp(p_bar(t));
      if (r == 0) FA_TRACE_EV(j, 3 + 4 * t);
    }

    // ----------------------------------------------------- epilogue
    if (nb[t] > 0) {
      if (ok) ok = mbar_wait_warp(o_bar(t), 0, wctx, kSiteOFull);
      if (threadIdx.x == 0) FA_LIFE(4);
      tc_fence_after();
      uint8_t *stage = smem + C::kOffQ + t * C::kTileBytes;  // Q_t is dead once O_t is final
      // A varlen tile that runs past its sequence is written row by row (the
      // rows after it belong to the next sequence); every other tile goes
      // through shared memory and one TMA store per 64-column box.
      const bool direct = VARLEN && q0[t] + 128 > L;
      if (ok) {
        const float inv_l = 1.0f / l_sum;
        uint4 *orow = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.o) +
                                                ((size_t)(sq.start + q_row) * p.H + h) * D);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld_32x32b_x32(o_tm + 32 * c, o);
          tmem_wait_ld(o);
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            w[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
          if (direct) {
            if (q_row < L) {
#pragma unroll
              for (int k4 = 0; k4 < 4; ++k4)
                orow[4 * c + k4] = make_uint4(w[4 * k4], w[4 * k4 + 1], w[4 * k4 + 2], w[4 * k4 + 3]);
            }
          } else {
            const int box = c >> 1;
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) {
              const int chunk = ((c & 1) * 4 + k4) ^ (r & 7);
              uint4 *dst = reinterpret_cast<uint4 *>(stage + box * 16384 + r * 128 + chunk * 16);
              *dst = make_uint4(w[4 * k4], w[4 * k4 + 1], w[4 * k4 + 2], w[4 * k4 + 3]);
            }
          }
        }
        if (p.lse != nullptr && q_row < L) {
          const size_t li = VARLEN ? (size_t)h * p.total + sq.start + q_row : ((size_t)b * p.H + h) * p.N + q_row;
          p.lse[li] = (m_ref + __log2f(l_sum)) * 0.69314718055994531f;
        }
      }
      fence_proxy_async_smem();
      if (t == 0) named_bar_sync(1, 128);
      else named_bar_sync(2, 128);
      if (r == 0 && ok && !direct) {
#pragma unroll
        for (int bx = 0; bx < C::kBoxes; ++bx)
          tma_store_4d(&p.tm_o, smem_u32(stage) + bx * 16384, bx * 64, h, sq.start + q0[t], sq.bc);
        bulk_commit();
        bulk_wait_read_all();
        if (threadIdx.x == 0) FA_LIFE(5);
      }
    }
    if (rescales) atomicAdd(p.status + 2, rescales);
  } else if (warp == C::kMmaWarp) {
    // ===================================================== MMA issue
    // The whole warp runs the loop and waits; the elected lane issues.
    {
      constexpr uint32_t idesc_s = make_idesc_bf16(128, 128, false, false);
      constexpr uint32_t idesc_pv = make_idesc_bf16(128, D, false, true);
      const uint32_t q_smem = sbase + C::kOffQ;
      const uint32_t ring = sbase + C::kOffRing;
      auto slot_of = [&](int fill) { return fill % C::kStages; };
      auto par_of = [&](int fill) { return (uint32_t)((fill / C::kStages) & 1); };
      // Descriptors are built once; a K step only moves the start-address
      // field (bits 0-13, address >> 4), which never carries out for
      // addresses inside the 228 KB shared-memory window.
      uint64_t q_desc[QT];
#pragma unroll
      for (int t = 0; t < QT; ++t) q_desc[t] = make_sdesc_sw128(q_smem + t * C::kTileBytes, 0, 1024);
      const uint64_t ring_desc_k = make_sdesc_sw128(ring, 0, 1024);
      const uint64_t ring_desc_v = make_sdesc_sw128(ring, 16384, 1024);
      auto issue_s = [&](int t, int slot) {
        const uint64_t kd = ring_desc_k + (uint64_t)((slot * C::kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
          mma_ss(tmem + 128u * t, q_desc[t] + off, kd + off, idesc_s, kk > 0);
        }
      };
      auto issue_pv = [&](int t, int slot, bool acc) {
        const uint64_t vd = ring_desc_v + (uint64_t)((slot * C::kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts(tmem + C::kOCol + (uint32_t)(D * t), tmem + 128u * t + 8u * kk, vd + (uint64_t)(kk * 128), idesc_pv,
                 (acc || kk > 0));
      };
      bool ok = nb_max > 0;
      if (ok) ok = mbar_wait_warp(q_bar, 0, wctx, kSiteQ);
      if (ok) ok = mbar_wait_warp(full_bar(slot_of(0)), par_of(0), wctx, kSiteKFull);
      if (ok) {
        tc_fence_after();
        if (elect_one()) {
          for (int t = 0; t < QT; ++t)
            if (nb[t] > 0) {
              issue_s(t, slot_of(0));
              tc_commit(s_bar(t));
            }
          tc_commit(empty_bar(slot_of(0)));
        }
        __syncwarp();
        if (lane == 0) FA_LIFE(3);
      }
      for (int j = 0; j < nb_max && ok; ++j) {
        const int fv = 2 * j + 1, fk = 2 * j + 2;
        ok = mbar_wait_warp(full_bar(slot_of(fv)), par_of(fv), wctx, kSiteVFull);
        if (!ok) break;
        tc_fence_after();
        bool k_next = false;
        for (int t = 0; t < QT && ok; ++t) {
          if (j >= nb[t]) continue;
          ok = mbar_wait_warp(p_bar(t), j & 1, wctx, kSitePFull);
          if (!ok) break;
          FA_TRACE_EV(j, 8 + 2 * t);
          tc_fence_after();
          if (elect_one()) issue_pv(t, slot_of(fv), j > 0);
          __syncwarp();
          if (j + 1 < nb[t]) {
            if (!k_next) {
              ok = mbar_wait_warp(full_bar(slot_of(fk)), par_of(fk), wctx, kSiteKFull);
              if (!ok) break;
              tc_fence_after();
              k_next = true;
            }
            if (elect_one()) {
              issue_s(t, slot_of(fk));
              tc_commit(s_bar(t));
            }
            __syncwarp();
            FA_TRACE_EV(j, 9 + 2 * t);
          } else {
            if (elect_one()) tc_commit(o_bar(t));
            __syncwarp();
          }
        }
        if (elect_one()) {
          tc_commit(empty_bar(slot_of(fv)));
          if (k_next) tc_commit(empty_bar(slot_of(fk)));
        }
        __syncwarp();
      }
      // Drain: every MMA this thread issued completes before TMEM is released.
      if (elect_one()) tc_commit(drain_bar);
      __syncwarp();
      WaitCtx drain_ctx{abort_flag, p.status};
      if (!mbar_wait_warp(drain_bar, 0, drain_ctx, kSiteDrain) && *abort_flag) {
        const uint64_t t0 = global_timer_ns();  // aborted: still give in-flight MMAs time to land
        while (!mbar_test(drain_bar, 0) && global_timer_ns() - t0 < kWaitLimitNs) {}
      }
    }
  } else {
    // ===================================================== TMA producer
    if (lane == 0 && nb_max > 0) {
      const uint32_t q_smem = sbase + C::kOffQ;
      const uint32_t ring = sbase + C::kOffRing;
      const uint64_t keep = policy_evict_last();   // K/V are re-read by the other query tiles
      const uint64_t once = policy_evict_first();  // Q is read once
      int nq = 0;
      for (int t = 0; t < QT; ++t) nq += (nb[t] > 0);
      mbar_arrive_expect_tx(q_bar, nq * C::kTileBytes);
      for (int t = 0; t < QT; ++t)
        if (nb[t] > 0)
          for (int bx = 0; bx < C::kBoxes; ++bx)
            tma_load_4d_hint(q_smem + t * C::kTileBytes + bx * 16384, &p.tm_q, q_bar, bx * 64, h, sq.start + q0[t],
                             sq.bc, once);
      bool ok = true;
      int fill = 0;
      for (int j = 0; j < nb_max && ok; ++j) {
        for (int kv = 0; kv < 2 && ok; ++kv, ++fill) {
          const int s = fill % C::kStages;
          ok = mbar_wait(empty_bar(s), ((fill / C::kStages) & 1) ^ 1, wctx, kSiteEmpty);
          if (!ok) break;
          mbar_arrive_expect_tx(full_bar(s), C::kTileBytes);
          const CUtensorMap *map = kv ? &p.tm_v : &p.tm_k;
          for (int bx = 0; bx < C::kBoxes; ++bx)
            tma_load_4d_hint(ring + s * C::kTileBytes + bx * 16384, map, full_bar(s), bx * 64, kh, sq.start + j * 128,
                             sq.bc, keep);
        }
      }
      // Every copy issued lands before the CTA exits (normally they already have).
      const uint64_t t0 = global_timer_ns();
      for (int f = max(0, fill - C::kStages); f < fill; ++f)
        while (!mbar_test(full_bar(f % C::kStages), (f / C::kStages) & 1) && global_timer_ns() - t0 < kWaitLimitNs) {}
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  FA_CTA_MARK(2);
  if (threadIdx.x == 0) FA_LIFE(6);
}

// ================================================================== CTA pairs (head dim 256)
// At head dim 256 one query tile per CTA is all TMEM holds (S 128 + O 256
// columns), so the kernel above serialises S_j -> softmax_j -> PV_j, and each
// key block brings 128 KB of K and V into one SM.  Here two CTAs of a cluster
// share 256 query rows (128 each) and the rank-0 CTA issues M = 256
// `cta_group::2` MMAs (FA4 paper summary, section 2.C: each SM holds its own
// rows of A and half of B):
//   S_j  = Q K_j^T   N = 128 keys: CTA c loads key rows 64c..64c+63 (32 KB)
//   O   += P_j V_j   N = 256 = d: CTA c loads head-dim columns 128c..128c+127
//                    of all 128 keys (32 KB); P_j read from TMEM
// TMEM per CTA: S in two buffers (columns 0 and 128) and O (256 columns), so
// S_{j+1} runs on the tensor core while the softmax works on S_j.  MMA order:
// S_0 S_1 | PV_0 S_2 | PV_1 S_3 | ...  With S_{j+1} already issued when the
// softmax meets block j, a rescale of O first waits for PV_{j-1}.
template <int D>
struct FwdPairCfg {
  static constexpr int kTileBytes = 128 * D * 2;  // the CTA's Q tile: D / 64 boxes of 128 rows
  // K half: 64 rows x D (D / 64 boxes of 8 KB); V half: 128 rows x D / 2 (D / 128 boxes of 16 KB)
  static constexpr int kHalf = 64 * D * 2;
  static constexpr int kStages = (232448 - kTileBytes - 256) / kHalf;  // 5 at D = 256, 12 at D = 128
  static constexpr int kThreads = 192;  // 4 softmax warps, MMA warp, TMA warp
  static constexpr int kMmaWarp = 4, kLoadWarp = 5;
  static constexpr int kColO = 256, kTmemCols = 512;  // S_j in columns 128 (j % 2)
  static constexpr int kOffQ = 0, kOffRing = kTileBytes;
  enum { kBarFull0, kBarEmpty0 = kBarFull0 + kStages, kBarQ = kBarEmpty0 + kStages, kBarS0, kBarP0 = kBarS0 + 2,
         kBarPV = kBarP0 + 2, kBarO, kBarDrain, kBarQFree, kNumBars };
  static constexpr int kOffBar = kOffRing + kStages * kHalf;
  static constexpr int kOffMisc = kOffBar + 8 * kNumBars;
  static constexpr int kSmemBytes = kOffMisc + 16;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// One work unit of the CTA-pair forward: query rows 256 pg .. 256 pg + 255 of one
// (batch, head), the cluster's CTA c taking rows 128 c .. 128 c + 127 of them.
struct FwdPairUnit {
  SeqSpan sq;
  int b, h, kh, qp0, nb;
  bool skip;  // packed batch: the pair's rows lie past its sequence
};

template <bool CAUSAL, bool VARLEN>
__device__ __forceinline__ FwdPairUnit fwd_pair_unit(const FwdParams &p, int u) {
  FwdPairUnit w;
  const int n_q = (p.N + 127) / 128;
  const int n_pairs = (n_q + 1) / 2;
  int rank, head;
  work_order(u, n_pairs, p.B * p.H, p.sched_chunk, rank, head);
  const int pg = CAUSAL ? n_pairs - 1 - rank : rank;  // causal: the longest query rows first
  w.h = head % p.H;
  w.b = head / p.H;
  w.kh = w.h / (p.H / p.Hkv);
  w.sq = VARLEN ? seq_span(p.cu_seqlens, w.b, p.N, p.total) : SeqSpan{0, p.N, w.b};
  const int L = w.sq.len;
  w.qp0 = 256 * pg;  // the pair's first query row
  w.skip = VARLEN && w.qp0 >= L;
  // key blocks: the pair computes every block its later tile needs; the earlier
  // tile's rows mask the last one whole under the causal mask
  w.nb = CAUSAL ? min(w.qp0 + 255, L - 1) / 128 + 1 : (L + 127) / 128;
  return w;
}

// PERSIST: at most one cluster per SM pair, cluster c running units c, c + gridDim.x / 2, ...;
// both CTAs walk the same units.  The K/V ring, the S buffers and every barrier
// phase count over the units (S, P, PV per key block; Q, O per unit).  The MMA
// warp commits q_free (to both CTAs) right after a unit's last S, up to two key
// blocks before the unit ends, and each CTA's producer then loads its next Q
// tile; the epilogue writes O rows straight from TMEM (the Q region is no
// longer free to stage them), while the next unit's first S run.
template <int D, bool CAUSAL, bool VARLEN, bool PERSIST>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(192, 1)
    fa_fwd_pair_kernel(const __grid_constant__ FwdParams p) {
  using C = FwdPairCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) {  // same layout in both CTAs: both return before any cluster work
    if (threadIdx.x == 0) {
      atomicOr(p.status, 1u);
      atomicCAS(p.status + 1, 0u, (unsigned)kSiteQ);
    }
    return;
  }
  const uint32_t bar0 = sbase + C::kOffBar;
  auto bar = [&](int i) { return bar0 + 8u * i; };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 4);
  const WaitCtx wctx{abort_flag, p.status};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int crank = (int)cluster_ctarank();
  const int n_units = ((p.N + 127) / 128 + 1) / 2 * p.B * p.H;
  const int cid = (int)(blockIdx.x >> 1), n_clusters = (int)(gridDim.x >> 1);

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kNumBars; ++i)  // P collects one arrival per softmax warp of both CTAs
      mbar_init(bar(i), (i == C::kBarP0 || i == C::kBarP0 + 1) ? 8u : 1u);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == C::kMmaWarp) {
    tmem_alloc_pair(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish_pair();
  }
  if (warp == C::kLoadWarp && lane == 0) {
    prefetch_tmap(&p.tm_q);
    prefetch_tmap(&p.tm_k64);
    prefetch_tmap(&p.tm_v);
    prefetch_tmap(&p.tm_o);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // barriers of both CTAs initialised, TMEM of both allocated
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
    // ===================================================== softmax (one thread per query row of this CTA)
    const int r = threadIdx.x;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const uint32_t o_tm = tmem + lane_off + C::kColO;
    const float c2 = p.scale_log2;
    bool ok = true;
    unsigned rescales = 0;
    int G = 0, uc = 0;  // key blocks and units before this one
    for (int u = cid; u < n_units && ok; u += n_clusters) {
      int nb, L, q_row;
      {
        const FwdPairUnit w = fwd_pair_unit<CAUSAL, VARLEN>(p, u);
        if (w.skip) continue;
        nb = w.nb;
        L = w.sq.len;
        q_row = w.qp0 + 128 * crank + r;
      }
      float m_ref = -INFINITY, l_sum = 0.f;
      for (int j = 0; j < nb && ok; ++j) {
        const unsigned gb = (unsigned)(G + j);
        const unsigned sb = gb & 1u;
        const uint32_t s_tm = tmem + lane_off + 128u * sb;
        ok = mbar_wait_warp_cl(bar(C::kBarS0 + sb), (gb >> 1) & 1u, wctx, kSiteSFull);
        if (!ok) break;
        tc_fence_after();
        uint32_t sr[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld_32x32b_x32(s_tm + 32 * c, sr[c]);
        tmem_wait_ld(sr[0]);
        reg_tie(sr[1]);
        reg_tie(sr[2]);
        reg_tie(sr[3]);
        float s[128];
#pragma unroll
        for (int c = 0; c < 128; ++c) s[c] = __uint_as_float(sr[c >> 5][c & 31]);
        const int kv0 = j * 128;
        const int lim = (CAUSAL ? min(L - 1, q_row) : L - 1) - kv0;  // last visible column
        if (__any_sync(0xffffffffu, lim < 127)) {
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c > lim) s[c] = -INFINITY;
        }
        float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
        for (int c = 4; c < 124; c += 8) {
          mx0 = fmax3(mx0, s[c], s[c + 1]);
          mx1 = fmax3(mx1, s[c + 2], s[c + 3]);
          mx2 = fmax3(mx2, s[c + 4], s[c + 5]);
          mx3 = fmax3(mx3, s[c + 6], s[c + 7]);
        }
        mx0 = fmax3(mx0, s[124], s[125]);
        mx1 = fmax3(mx1, s[126], s[127]);
        const float m_blk = fmax3(mx0, mx1, fmaxf(mx2, mx3)) * c2;
        float alpha = 1.f;
        bool rescale = false;  // uniform across the warp; O is scaled once P is stored
        if (j == 0) {
          m_ref = m_blk;
        } else {
          const bool need = (m_blk - m_ref) > kRescaleTau;
          if (__any_sync(0xffffffffu, need)) {
            const float m_new = fmaxf(m_ref, m_blk);
            alpha = ex2_mufu(m_ref - m_new);
            m_ref = m_new;
            l_sum *= alpha;
            rescale = true;
          }
        }
        const float neg_m = -m_ref;
        float l0 = 0.f, l1 = 0.f, l2 = 0.f, l3 = 0.f;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 64; c += 4) {
            float x[4], e[4];
            ffma2(x[0], x[1], s[64 * half + c], s[64 * half + c + 1], c2, c2, neg_m, neg_m);
            ffma2(x[2], x[3], s[64 * half + c + 2], s[64 * half + c + 3], c2, c2, neg_m, neg_m);
#pragma unroll
            for (int u4 = 0; u4 < 4; ++u4)
              e[u4] = ((c + u4) % 16 < FA_FWD_POLY_PER16) ? exp2_poly(x[u4]) : ex2_mufu(x[u4]);
            fadd2(l0, l1, l0, l1, e[0], e[1]);
            fadd2(l2, l3, l2, l3, e[2], e[3]);
            pk[c >> 1] = pack_bf16x2(e[0], e[1]);
            pk[(c >> 1) + 1] = pack_bf16x2(e[2], e[3]);
          }
          tmem_st_32x32b_x32(s_tm + 32 * half, pk);
        }
        l_sum += (l0 + l1) + (l2 + l3);
        if (rescale) {
          // PV of the previous key block must have landed in O before it is
          // scaled (S_j was issued before it); PV_j waits for the P signal below
          ok = mbar_wait_warp_cl(bar(C::kBarPV), (gb - 1u) & 1u, wctx, kSiteOFull);
          if (!ok) break;
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < D / 64; ++c) {
            uint32_t o0[32], o1[32];
            tmem_ld_32x32b_x32(o_tm + 64 * c, o0);
            tmem_ld_32x32b_x32(o_tm + 64 * c + 32, o1);
            tmem_wait_ld(o0);
            reg_tie(o1);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              o0[i] = __float_as_uint(__uint_as_float(o0[i]) * alpha);
              o1[i] = __float_as_uint(__uint_as_float(o1[i]) * alpha);
            }
            tmem_st_32x32b_x32(o_tm + 64 * c, o0);
            tmem_st_32x32b_x32(o_tm + 64 * c + 32, o1);
          }
          rescales += (lane == 0);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive_warp_cluster(mapa_shared(bar(C::kBarP0 + sb), 0));
      }
      G += nb;
      // ----------------------------------------------------- epilogue (this CTA's 128 rows)
      if (ok) ok = mbar_wait_warp_cl(bar(C::kBarO), (unsigned)uc & 1u, wctx, kSiteOFull);
      ++uc;
      tc_fence_after();
      {
        // the unit's coordinates again, from a copy of u the compiler cannot
        // match to the first: only u stays live across the key blocks
        const FwdPairUnit w = fwd_pair_unit<CAUSAL, VARLEN>(p, PERSIST ? __shfl_sync(0xffffffffu, u, 0) : u);
        const int q0 = w.qp0 + 128 * crank;
        uint8_t *stage = smem + C::kOffQ;  // Q is dead once O is final
        const bool has_rows = q0 < L;
        // row by row: persistent CTAs (the Q region holds the next unit's Q), or
        // a varlen tile that runs past its sequence (the next sequence's rows follow)
        const bool direct = PERSIST || (VARLEN && q0 + 128 > L);
        const size_t row0 = VARLEN ? (size_t)w.sq.start : (size_t)w.b * p.N;  // the sequence's first row
        if (ok && has_rows) {
          const float inv_l = 1.0f / l_sum;
          uint4 *orow = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.o) + ((row0 + q_row) * p.H + w.h) * D);
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld_32x32b_x32(o_tm + 32 * c, o);
            tmem_wait_ld(o);
            uint32_t wv[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              wv[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
            if (direct) {
              if (q_row < L) {
#pragma unroll
                for (int k4 = 0; k4 < 4; ++k4)
                  orow[4 * c + k4] = make_uint4(wv[4 * k4], wv[4 * k4 + 1], wv[4 * k4 + 2], wv[4 * k4 + 3]);
              }
            } else {
#pragma unroll
              for (int k4 = 0; k4 < 4; ++k4) {
                const int chunk = ((c & 1) * 4 + k4) ^ (r & 7);
                *reinterpret_cast<uint4 *>(stage + (c >> 1) * 16384 + r * 128 + chunk * 16) =
                    make_uint4(wv[4 * k4], wv[4 * k4 + 1], wv[4 * k4 + 2], wv[4 * k4 + 3]);
              }
            }
          }
          if (p.lse != nullptr && q_row < L) {
            const size_t li = VARLEN ? (size_t)w.h * p.total + w.sq.start + q_row : ((size_t)w.b * p.H + w.h) * p.N + q_row;
            p.lse[li] = (m_ref + __log2f(l_sum)) * 0.69314718055994531f;
          }
        }
        tc_fence_before();  // the O reads precede the next unit's first PV
        if (!PERSIST) {
          fence_proxy_async_smem();
          named_bar_sync(1, 128);
          if (r == 0 && ok && has_rows && !direct) {
            for (int bx = 0; bx < D / 64; ++bx)
              tma_store_4d(&p.tm_o, smem_u32(stage) + bx * 16384, bx * 64, w.h, w.sq.start + q0, w.sq.bc);
            bulk_commit();
            bulk_wait_read_all();
          }
        }
      }
      if (!PERSIST) break;  // one unit per cluster
    }
    if (rescales) atomicAdd(p.status + 2, rescales);
  } else if (warp == C::kMmaWarp) {
    // ===================================================== MMA issue (rank-0 CTA, for both)
    if (crank == 0) {
      constexpr uint32_t id_s = make_idesc_bf16(256, 128, false, false);
      constexpr uint32_t id_pv = make_idesc_bf16(256, D, false, true);
      const uint64_t q_d = make_sdesc_sw128(sbase + C::kOffQ, 0, 1024);
      const uint64_t k_d = make_sdesc_sw128(sbase + C::kOffRing, 0, 1024);
      const uint64_t v_mn = make_sdesc_sw128(sbase + C::kOffRing, 16384, 1024);
      auto slot_of = [](int fill) { return (int)((unsigned)fill % C::kStages); };
      auto full_ok = [&](int fill) {
        return mbar_wait_warp_cl(bar(C::kBarFull0 + slot_of(fill)), ((unsigned)fill / C::kStages) & 1u, wctx,
                                 (fill & 1) ? kSiteVFull : kSiteKFull);
      };
      // S of key block gb (over the CTA's units) into buffer gb % 2; K from ring fill fk
      auto issue_s = [&](unsigned gb, int fk, bool last) {
        const uint64_t kd = k_d + (uint64_t)((slot_of(fk) * C::kHalf) >> 4);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss_pair(tmem + 128u * (gb & 1u), q_d + (uint64_t)(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4),
                        kd + (uint64_t)(((kk >> 2) * 8192 + (kk & 3) * 32) >> 4), id_s, kk > 0);
          tc_commit_pair(bar(C::kBarS0 + (gb & 1u)));
          tc_commit_pair(bar(C::kBarEmpty0 + slot_of(fk)));
          if (PERSIST && last) tc_commit_pair(bar(C::kBarQFree));  // the unit's last MMA reading Q
        }
        __syncwarp();
      };
      bool ok = true;
      int G = 0, F = 0, uc = 0;  // key blocks, ring fills and units before this one
      for (int u = cid; u < n_units && ok; u += n_clusters) {
        const FwdPairUnit w = fwd_pair_unit<CAUSAL, VARLEN>(p, u);
        if (w.skip) continue;
        const int nb = w.nb;  // K_j is fill F + 2 j, V_j fill F + 2 j + 1
        ok = mbar_wait_warp_cl(bar(C::kBarQ), (unsigned)uc & 1u, wctx, kSiteQ);
        for (int j = 0; j < 2 && j < nb && ok; ++j) {
          ok = full_ok(F + 2 * j);
          if (!ok) break;
          tc_fence_after();
          issue_s((unsigned)(G + j), F + 2 * j, j + 1 == nb);
        }
        for (int j = 0; j < nb && ok; ++j) {
          const unsigned gb = (unsigned)(G + j);
          ok = full_ok(F + 2 * j + 1);
          if (ok) ok = mbar_wait_warp_cl(bar(C::kBarP0 + (gb & 1u)), (gb >> 1) & 1u, wctx, kSitePFull);
          if (!ok) break;
          tc_fence_after();
          if (elect_one()) {  // O += P_j V_j
            const uint64_t vd = v_mn + (uint64_t)((slot_of(F + 2 * j + 1) * C::kHalf) >> 4);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ts_pair(tmem + C::kColO, tmem + 128u * (gb & 1u) + 8u * kk, vd + (uint64_t)(kk * 128), id_pv,
                          (j > 0 || kk > 0));
            tc_commit_pair(bar(C::kBarPV));
            tc_commit_pair(bar(C::kBarEmpty0 + slot_of(F + 2 * j + 1)));
            if (j + 1 == nb) tc_commit_pair(bar(C::kBarO));
          }
          __syncwarp();
          if (j + 2 < nb) {  // S_{j+2} over P_j (its PV was issued first)
            ok = full_ok(F + 2 * j + 4);
            if (!ok) break;
            tc_fence_after();
            issue_s(gb + 2u, F + 2 * j + 4, j + 3 == nb);
          }
        }
        G += nb;
        F += 2 * nb;
        ++uc;
        if (!PERSIST) break;
      }
      if (elect_one()) tc_commit_pair(bar(C::kBarDrain));
      __syncwarp();
      if (!mbar_wait_warp_cl(bar(C::kBarDrain), 0, wctx, kSiteDrain) && *abort_flag) {
        const uint64_t t0 = global_timer_ns();
        while (!mbar_test_cl(bar(C::kBarDrain), 0) && global_timer_ns() - t0 < kWaitLimitNs) {}
      }
    }
  } else {
    // ===================================================== TMA producer (both CTAs; bytes counted by rank 0)
    if (lane == 0) {
      const uint64_t keep = policy_evict_last();
      const uint64_t once = policy_evict_first();
      const uint32_t qb = mapa_shared(bar(C::kBarQ), 0);
      bool ok = true;
      int fill = 0, uc = 0;
      for (int u = cid; u < n_units && ok; u += n_clusters) {
        const FwdPairUnit w = fwd_pair_unit<CAUSAL, VARLEN>(p, u);
        if (w.skip) continue;
        // this CTA's Q tile, once the MMAs that read the previous unit's have completed
        if (PERSIST && uc > 0) ok = mbar_wait_cl(bar(C::kBarQFree), (unsigned)(uc - 1) & 1u, wctx, kSiteEmpty);
        if (!ok) break;
        if (crank == 0) mbar_arrive_expect_tx(bar(C::kBarQ), 2 * C::kTileBytes);
        for (int bx = 0; bx < D / 64; ++bx)
          tma_load_4d_pair(sbase + C::kOffQ + bx * 16384, &p.tm_q, qb, bx * 64, w.h, w.sq.start + w.qp0 + 128 * crank,
                           w.sq.bc, once);
        ++uc;
        for (int f = 0; f < 2 * w.nb && ok; ++f, ++fill) {
          const int j = f >> 1, s = (int)((unsigned)fill % C::kStages);
          ok = mbar_wait_cl(bar(C::kBarEmpty0 + s), (((unsigned)fill / C::kStages) & 1u) ^ 1u, wctx, kSiteEmpty);
          if (!ok) break;
          if (crank == 0) mbar_arrive_expect_tx(bar(C::kBarFull0 + s), 2 * C::kHalf);
          const uint32_t fb = mapa_shared(bar(C::kBarFull0 + s), 0);
          const uint32_t dst = sbase + C::kOffRing + s * C::kHalf;
          if ((f & 1) == 0) {  // K_j: this CTA's 64 key rows, all D columns
            for (int bx = 0; bx < D / 64; ++bx)
              tma_load_4d_pair(dst + bx * 8192, &p.tm_k64, fb, bx * 64, w.kh, w.sq.start + 128 * j + 64 * crank,
                               w.sq.bc, keep);
          } else {  // V_j: all 128 key rows, this CTA's head-dim half
            for (int bx = 0; bx < D / 128; ++bx)
              tma_load_4d_pair(dst + bx * 16384, &p.tm_v, fb, (D / 2) * crank + 64 * bx, w.kh, w.sq.start + 128 * j,
                               w.sq.bc, keep);
          }
        }
        if (!PERSIST) break;
      }
      // drain: rank 0's barriers count both CTAs' copies
      if (crank == 0) {
        const uint64_t t0 = global_timer_ns();
        for (int f = max(0, fill - C::kStages); f < fill; ++f)
          while (!mbar_test_cl(bar(C::kBarFull0 + f % C::kStages), (f / C::kStages) & 1) &&
                 global_timer_ns() - t0 < kWaitLimitNs) {}
        if (uc > 0)
          while (!mbar_test_cl(bar(C::kBarQ), (unsigned)(uc - 1) & 1u) && global_timer_ns() - t0 < kWaitLimitNs) {}
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the rank-0 CTA's MMAs and both CTAs' copies are done with both CTAs' memory
  if (warp == C::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, C::kTmemCols);
  }
}

template <int D, bool CAUSAL, bool VARLEN, bool PERSIST>
int launch_fwd_pair(const FwdParams &p_in, cudaStream_t stream) {
  using C = FwdPairCfg<D>;
  auto kern = fa_fwd_pair_kernel<D, CAUSAL, VARLEN, PERSIST>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) != cudaSuccess)
    return FA_ERR_CUDA;
  const long long n_pairs = ((p_in.N + 127) / 128 + 1) / 2;
  const long long n_ctas = 2 * n_pairs * p_in.H * p_in.B;
  if (n_ctas > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  FwdParams p = p_in;
  const int g = p.H / p.Hkv;
  p.sched_chunk = CAUSAL ? g * sched_chunk_for(true, (size_t)2 * p.N * D * 2, p.B * p.Hkv) : 1;
  long long grid = n_ctas;
  if (PERSIST) {  // at most one cluster per SM pair, each running a strided share of the units
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return FA_ERR_CUDA;
    if (grid > 2LL * (sms / 2)) grid = 2LL * (sms / 2);
  }
  if (grid > 0) kern<<<(unsigned)grid, C::kThreads, C::kSmemBytes, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// CTA-pair forward: persistent clusters for sequences up to these lengths.
// Measured at head dim 256 (interleaved medians): N = 1024 -15 %, causal -22 %;
// N = 4096 -7 %, causal -9 %; N = 16384 -3 %, but causal +3.5 %: there the
// strided static share of units of 1 to N / 256 key-block pairs loses to the
// hardware's greedy cluster placement.
#ifndef FA_FWD_PAIR_PERSIST_MAX_N
#define FA_FWD_PAIR_PERSIST_MAX_N (1 << 30)
#endif
#ifndef FA_FWD_PAIR_PERSIST_MAX_N_CAUSAL
#define FA_FWD_PAIR_PERSIST_MAX_N_CAUSAL 8192
#endif

template <int D, bool CAUSAL, bool VARLEN>
int launch_fwd_pair_any(const FwdParams &p, cudaStream_t stream) {
  if (p.N <= (CAUSAL ? FA_FWD_PAIR_PERSIST_MAX_N_CAUSAL : FA_FWD_PAIR_PERSIST_MAX_N))
    return launch_fwd_pair<D, CAUSAL, VARLEN, true>(p, stream);
  return launch_fwd_pair<D, CAUSAL, VARLEN, false>(p, stream);
}

template <int D, bool CAUSAL, bool VARLEN, int QT>
int launch_fwd_q(const FwdParams &p_in, cudaStream_t stream) {
  using C = FwdCfg<D, QT>;
  auto kern = fa_fwd_kernel<D, CAUSAL, FA_FWD_POLY_PER16, VARLEN, QT>;
  // set on every launch: the attribute belongs to the function on the current
  // device, and a process may drive several devices from several threads
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) != cudaSuccess)
    return FA_ERR_CUDA;
  const int rows_per_cta = 128 * C::kQT;
  const long long n_groups = (p_in.N + rows_per_cta - 1) / rows_per_cta;
  const long long n_ctas = n_groups * p_in.H * p_in.B;
  if (n_ctas > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  FwdParams p = p_in;
  // K and V of one kv head are re-read by every query tile of its query heads
  const int g = p.H / p.Hkv;
  p.sched_chunk = CAUSAL ? g * sched_chunk_for(true, (size_t)2 * p.N * D * 2, p.B * p.Hkv) : 1;
  kern<<<(unsigned)n_ctas, C::kThreads, C::kSmemBytes, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// Head dim 64, sequences of at most FA_FWD_SHORT_MAX_N_D64 rows (the longest
// one, for packed batches): the short form, two CTAs per SM.  Measured on
// GB300 at B*N = 32768, H = 16: +10-17 % at N = 512, +8-14 % at 1024, +5 % at
// 2048, +1-4 % at 4096 over the two-tile form.  At head dim 128 its two-stage
// ring is too shallow for the load latency (2-11 % slower), so it is not used.
#ifndef FA_FWD_SHORT_MAX_N_D64
#define FA_FWD_SHORT_MAX_N_D64 4096
#endif

// Head dim 256 on CTA pairs (1, the default) or one query tile per CTA (0).
#ifndef FA_FWD256_PAIR
#define FA_FWD256_PAIR 1
#endif
// Head dim 128 on CTA pairs (1) or two query tiles per CTA (0, the default).
// The pair form passes the forward tests but measured 5-45 % slower on GB300
// (headline 1.34 against 1.28 ms, causal B8 N4096 0.48 against 0.40 ms,
// N = 1024 0.32 against 0.24 ms): at this head dim one softmax warpgroup per
// 128 rows cannot keep up with MMAs half as long as at 256, and the two-tile
// CTA overlaps one tile's softmax with the other's MMAs.
#ifndef FA_FWD128_PAIR
#define FA_FWD128_PAIR 0
#endif

template <int D, bool CAUSAL, bool VARLEN>
int launch_fwd_v(const FwdParams &p, cudaStream_t stream) {
  if constexpr (D == 64) {
    if (p.N <= FA_FWD_SHORT_MAX_N_D64) return launch_fwd_q<D, CAUSAL, VARLEN, 1>(p, stream);
  }
  if constexpr (D == 256 && FA_FWD256_PAIR) return launch_fwd_pair_any<256, CAUSAL, VARLEN>(p, stream);
  if constexpr (D == 128 && FA_FWD128_PAIR) return launch_fwd_pair_any<128, CAUSAL, VARLEN>(p, stream);
  return launch_fwd_q<D, CAUSAL, VARLEN, FwdCfg<D>::kQT>(p, stream);
}

template <int D, bool CAUSAL>
int launch_fwd_t(const FwdParams &p, cudaStream_t stream) {
  return p.cu_seqlens ? launch_fwd_v<D, CAUSAL, true>(p, stream) : launch_fwd_v<D, CAUSAL, false>(p, stream);
}

}  // namespace

int launch_fwd(const FwdParams &p, int d, bool causal, cudaStream_t stream) {
  switch (d) {
    case 64: return causal ? launch_fwd_t<64, true>(p, stream) : launch_fwd_t<64, false>(p, stream);
    case 128: return causal ? launch_fwd_t<128, true>(p, stream) : launch_fwd_t<128, false>(p, stream);
    case 256: return causal ? launch_fwd_t<256, true>(p, stream) : launch_fwd_t<256, false>(p, stream);
    default: return FA_ERR_UNSUPPORTED;
  }
}

#ifdef FA_TEST_STALL
int set_test_stall_fwd(int mode) {
  return cudaMemcpyToSymbol(g_test_stall, &mode, sizeof(int)) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}
#endif

}  // namespace fa

#ifdef FA_TRACE
extern "C" int fa_debug_trace_fwd(unsigned long long *host_out) {
  return cudaMemcpyFromSymbol(host_out, fa::g_trace_fwd, sizeof(fa::g_trace_fwd)) == cudaSuccess ? 0 : -5;
}
// life: 16 SM-clock stamps; ctas: 65536 x {smid, entry ns, exit ns}
extern "C" int fa_debug_trace_ctas_fwd(unsigned long long *life, unsigned long long *ctas) {
  if (cudaMemcpyFromSymbol(life, fa::g_life_fwd, sizeof(fa::g_life_fwd)) != cudaSuccess) return -5;
  return cudaMemcpyFromSymbol(ctas, fa::g_cta_fwd, sizeof(fa::g_cta_fwd)) == cudaSuccess ? 0 : -5;
}
#endif
