// fa_bwd.cu — fused attention backward for sm_103a.
//
// Three launches, none of which uses atomics:
//   bwd_pre   D_i = sum_c dO_ic O_ic and LSE2_i = LSE_i log2(e), per query row,
//             rows padded to a multiple of 128 (LSE2 = +inf, D = 0);
//   bwd_dkdv  one CTA per (batch, kv head, 128-row key tile j).  K_j, V_j stay
//             in shared memory while every (query head of the group, query
//             tile i) streams past:
//                 S^T  = K_j Q_i^T  -> P^T = 2^(S^T c - LSE2)   (P never leaves the SM)
//                 dP^T = V_j dO_i^T -> dS^T = P^T (dP^T - D)
//                 dV  += P^T dO_i,  dK += dS^T Q_i             (accumulated in TMEM)
//   bwd_dq    one CTA per (batch, query head, 128-row query tile i), streaming
//             the key tiles j:
//                 S = Q_i K_j^T, dP = dO_i V_j^T -> dS = P (dP - D)  (dS kept in TMEM)
//                 dQ += dS K_j                                       (accumulated in TMEM)
//
// The pages place the backward's bottleneck in shared-memory traffic and in its
// atomic dQ updates (FlashAttention-4 article, "Por que el enfoque estandar ya
// no funciona"; FA4 paper summary, section 2.C).  Measured on GB300, one fp32
// reduction of dQ per (key tile, query tile) pair costs more time than the
// pair's five MMAs; recomputing S and dP in a query-stationary pass costs two
// extra MMAs and no reductions, and makes the backward deterministic.
//
// Warp roles (both main kernels): warps 0-7 elementwise, two warpgroups split
// by columns (64 each), one thread per TMEM lane; warp 8 MMA issue; warp 9 TMA.
#include <cuda_bf16.h>

#include "exp2_poly.cuh"
#include "fa_internal.h"
#include "ptx.cuh"

// Share of the dK/dV kernel's exponentials taken on the FMA pipe (exp2_poly2):
// columns with (column % 16) < FA_BWD_POLY_PER16; even, 0 = all on MUFU.EX2.
#ifndef FA_BWD_POLY_PER16
#define FA_BWD_POLY_PER16 0
#endif

// dK/dV at head dim 128 on CTA pairs (1, the default) or on single CTAs (0).
#ifndef FA_DKDV_PAIR
#define FA_DKDV_PAIR 1
#endif
// Sequence lengths (the longest one for packed batches) up to which the one-CTA
// dK/dV kernel runs at head dim 128 even with pairs enabled.  Measured on GB300
// (back-to-back launches, H = 16, B*N = 32768 unless noted): one CTA faster by
// 0-7 % non-causal at N <= 2048 and by 3-15 % causal at N <= 4096 (the pair's
// second key tile spends one iteration on a query tile it masks whole); pairs
// faster by 2-3 % non-causal at N = 4096, 3-4 % at the B4 N8192 headline shape,
// 0.5-6 % causal at N = 8192, 2-4 % at N = 16384 and 6 % on B1 H32/8 N32768.
#ifndef FA_DKDV_PAIR_MIN_N
#define FA_DKDV_PAIR_MIN_N 2048
#endif
#ifndef FA_DKDV_PAIR_MIN_N_CAUSAL
#define FA_DKDV_PAIR_MIN_N_CAUSAL 4096
#endif
// Head-dim-64 dK/dV: persistent CTAs (one per SM, each running a strided
// share of the work units) for sequences up to this many rows; longer ones get
// one CTA per unit, scheduled by the hardware.  Causal: the persistent kernel
// carries a few spilled registers, which cost more than the set-up it saves
// once a unit runs tens of iterations.
#ifndef FA_DKDV_PERSIST_MAX_N
#define FA_DKDV_PERSIST_MAX_N (1 << 30)
#endif
#ifndef FA_DKDV_PERSIST_MAX_N_CAUSAL
#define FA_DKDV_PERSIST_MAX_N_CAUSAL 8192
#endif
// Persistent dQ CTAs stage their epilogue through shared memory (1) or write
// dQ rows straight from TMEM (0).
#ifndef FA_DQ_PERSIST_STAGE
#define FA_DQ_PERSIST_STAGE 1
#endif
// dQ (one CTA per query tile, head dims 64 and 128): persistent CTAs for
// sequences up to these lengths.  Causal units range from 1 to N / 128 key
// tiles; past 8192 rows at head dim 128 the strided static share of them
// measured 1.5-2 % slower than the hardware's dynamic CTA scheduling.
#ifndef FA_DQ_PERSIST_MAX_N
#define FA_DQ_PERSIST_MAX_N (1 << 30)
#endif
#ifndef FA_DQ_PERSIST_MAX_N_CAUSAL
#define FA_DQ_PERSIST_MAX_N_CAUSAL (1 << 30)
#endif
#ifndef FA_DQ128_PERSIST_MAX_N
#define FA_DQ128_PERSIST_MAX_N (1 << 30)
#endif
#ifndef FA_DQ128_PERSIST_MAX_N_CAUSAL
#define FA_DQ128_PERSIST_MAX_N_CAUSAL 8192
#endif
// The same at head dim 128, where the one-CTA kernel runs up to FA_DKDV_PAIR_MIN_N
// (_CAUSAL) rows; at causal 4096 rows the two forms measured the same.
#ifndef FA_DKDV128_PERSIST_MAX_N
#define FA_DKDV128_PERSIST_MAX_N (1 << 30)
#endif
#ifndef FA_DKDV128_PERSIST_MAX_N_CAUSAL
#define FA_DKDV128_PERSIST_MAX_N_CAUSAL 2048
#endif
// dQ at head dim 128 on CTA pairs (1) or on single CTAs (0, the default).
#ifndef FA_DQ_PAIR
#define FA_DQ_PAIR 0
#endif
// dK/dV at head dim 256 on CTA pairs of 64 keys each (1, the default) or on
// one CTA per (key tile, head-dim half) (0).
#ifndef FA_DKDV256_PAIR
#define FA_DKDV256_PAIR 1
#endif
// dQ at head dim 256 on CTA pairs of 64 query rows each (1, the default) or on
// one CTA per query tile (0).
#ifndef FA_DQ256_PAIR
#define FA_DQ256_PAIR 1
#endif

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

// Opt-in event trace (build with -DFA_TRACE): SM clock at fixed points of the
// first 64 iterations of one CTA of each main kernel, read back with
// fa_debug_trace().  Off by default; the macro then expands to nothing.
#ifdef FA_TRACE
#ifndef FA_TRACE_CTA
#define FA_TRACE_CTA 7
#endif
__device__ unsigned long long g_trace[2][64][16];
// Lifecycle of CTA FA_TRACE_CTA (SM clock), and for every CTA its SM and the
// global timer at entry and exit; kernel 0 = dK/dV, 1 = dQ (head dim <= 128).
__device__ unsigned long long g_life[2][16];
__device__ unsigned long long g_cta[2][65536][3];
#define FA_LIFE(k, ev)                                      \
  do {                                                      \
    if (blockIdx.x == FA_TRACE_CTA) g_life[(k)][(ev)] = clock64(); \
  } while (0)
#define FA_CTA_MARK(k, slot)                                                    \
  do {                                                                          \
    if (threadIdx.x == 0 && blockIdx.x < 65536) {                               \
      unsigned sm_;                                                             \
      asm volatile("mov.u32 %0, %%smid;" : "=r"(sm_));                          \
      g_cta[(k)][blockIdx.x][0] = sm_;                                          \
      g_cta[(k)][blockIdx.x][(slot)] = global_timer_ns();                       \
    }                                                                           \
  } while (0)
#define FA_TRACE_EV(k, it, ev)                                                                   \
  do {                                                                                           \
    if (blockIdx.x == FA_TRACE_CTA && (it) < 64)                                                \
      g_trace[(k)][(it)][(ev)] = clock64();                                                      \
  } while (0)
#else
#define FA_TRACE_EV(k, it, ev) \
  do {                         \
  } while (0)
#define FA_LIFE(k, ev) \
  do {                 \
  } while (0)
#define FA_CTA_MARK(k, slot) \
  do {                       \
  } while (0)
#endif

// ------------------------------------------------------------------ pre
// Rows (b, n, h) of the padded range n < Npad.  A row of D bf16 is read as
// D / 8 16-byte chunks by D / 8 consecutive lanes, so a warp covers 32 / (D / 8)
// rows at a time; each warp takes kPreIters such groups and issues all of its
// loads before it reduces.  One group per warp (more warps in flight) measured
// fastest on GB300: 61.6 us per headline launch against 69.6 with two groups
// and 73.9 with four.  With a varlen table (cu != nullptr) the rows of sequence
// b are packed at its offset and lse is [H, total].
constexpr int kPreIters = 1;

template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const __nv_bfloat16 *__restrict__ o,
                                                      const __nv_bfloat16 *__restrict__ dO,
                                                      const float *__restrict__ lse, float *__restrict__ lse2,
                                                      float *__restrict__ delta, int B, int H, int N, int Npad,
                                                      const int *__restrict__ cu, int total,
                                                      float *__restrict__ dqacc) {
  constexpr int L = D / 8;      // lanes per row
  constexpr int RPW = 32 / L;   // rows per warp per iteration
  const int lane = threadIdx.x & 31;
  const int sub = lane / L, part = lane % L;
  const long long rows = (long long)B * Npad * H;
  const long long base = ((long long)blockIdx.x * 8 + (threadIdx.x >> 5)) * (RPW * kPreIters);
  uint4 va[kPreIters], vg[kPreIters];
  long long rw_[kPreIters];
  bool live[kPreIters];
  size_t lse_i[kPreIters];
#pragma unroll
  for (int it = 0; it < kPreIters; ++it) {
    const long long row = base + it * RPW + sub;
    live[it] = false;
    rw_[it] = -1;
    va[it] = vg[it] = make_uint4(0u, 0u, 0u, 0u);
    if (row >= rows) continue;
    const int h = (int)(row % H);
    const long long bn = row / H;
    const int n = (int)(bn % Npad);
    const int b = (int)(bn / Npad);
    rw_[it] = ((long long)b * H + h) * Npad + n;
    const SeqSpan sq = seq_span(cu, b, N, total);
    if (n >= sq.len) continue;  // padded query row
    live[it] = true;
    const size_t grow = cu ? (size_t)sq.start + n : (size_t)b * N + n;  // row in the [rows, H, D] tensors
    lse_i[it] = cu ? (size_t)h * total + sq.start + n : ((size_t)b * H + h) * N + n;
    const size_t off = (grow * H + h) * D + part * 8;
    va[it] = *reinterpret_cast<const uint4 *>(o + off);
    vg[it] = *reinterpret_cast<const uint4 *>(dO + off);
    if (dqacc != nullptr) {  // the fused backward accumulates dQ here: start from zero
      float4 *z = reinterpret_cast<float4 *>(dqacc + off);
      z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
      z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
#pragma unroll
  for (int it = 0; it < kPreIters; ++it) {
    const __nv_bfloat162 *a2 = reinterpret_cast<const __nv_bfloat162 *>(&va[it]);
    const __nv_bfloat162 *g2 = reinterpret_cast<const __nv_bfloat162 *>(&vg[it]);
    float acc = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      acc = fmaf(__low2float(a2[w]), __low2float(g2[w]), acc);
      acc = fmaf(__high2float(a2[w]), __high2float(g2[w]), acc);
    }
#pragma unroll
    for (int s = L / 2; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
    if (part == 0 && rw_[it] >= 0) {
      // padded query rows: LSE2 = +inf gives P = 2^(s - inf) = 0, and D = 0
      lse2[rw_[it]] = live[it] ? lse[lse_i[it]] * kLog2e : INFINITY;
      delta[rw_[it]] = live[it] ? acc : 0.f;
    }
  }
}

// ------------------------------------------------------------------ shared pieces
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

// TMEM epilogue of one 128 x D fp32 accumulator: this thread's row, columns
// [c0, c0 + NCOLS), times `mul`, to bf16 in a swizzled staging tile.
template <int NCOLS>
__device__ __forceinline__ void acc_to_smem(uint32_t tm_row, uint8_t *stage, int r, int c0, float mul) {
#pragma unroll
  for (int c = 0; c < NCOLS / 32; ++c) {
    uint32_t v[32];
    tmem_ld_32x32b_x32(tm_row + c0 + 32 * c, v);
    tmem_wait_ld(v);
    uint32_t w[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) w[k] = pack_bf16x2(__uint_as_float(v[2 * k]) * mul, __uint_as_float(v[2 * k + 1]) * mul);
    st_swizzled_32cols(stage, r, c0 + 32 * c, w);
  }
}

// The same epilogue for one row straight to global memory (bf16 row `dst`,
// columns [c0, c0 + NCOLS)): used for the rows of a varlen tile that belong to
// its sequence when the tile runs past the sequence's end, and by the
// persistent head-dim-128 dK/dV kernel, which has no room for a stage.
template <int NCOLS>
__device__ __forceinline__ void acc_to_global(uint32_t tm_row, __nv_bfloat16 *dst, int c0, float mul, bool write) {
#pragma unroll
  for (int c = 0; c < NCOLS / 32; ++c) {
    uint32_t v[32];
    tmem_ld_32x32b_x32(tm_row + c0 + 32 * c, v);
    tmem_wait_ld(v);
    uint32_t w[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) w[k] = pack_bf16x2(__uint_as_float(v[2 * k]) * mul, __uint_as_float(v[2 * k + 1]) * mul);
    if (write) {
      uint4 *d4 = reinterpret_cast<uint4 *>(dst + c0 + 32 * c);
#pragma unroll
      for (int k4 = 0; k4 < 4; ++k4) d4[k4] = make_uint4(w[4 * k4], w[4 * k4 + 1], w[4 * k4 + 2], w[4 * k4 + 3]);
    }
  }
}

FA_STALL_FLAG_DECL

enum BwdSite : int {
  kBSiteKV = 11, kBSiteFull = 12, kBSiteEmpty = 13, kBSiteS = 14, kBSiteDP = 15, kBSiteP = 16, kBSiteDS = 17,
  kBSiteDSFree = 18, kBSiteFinal = 19, kBSiteDrain = 20, kBSiteAlign = 21, kBSiteQ = 22, kBSiteDQ = 23,
  kBSiteSL = 24, kBSiteDQF = 25
};

__device__ __forceinline__ bool check_align(uint32_t sbase, unsigned *status) {
  if ((sbase & 1023u) == 0) return true;  // swizzled tiles need 1024-byte alignment
  if (threadIdx.x == 0) {
    atomicOr(status, 1u);
    atomicCAS(status + 1, 0u, (unsigned)kBSiteAlign);
  }
  return false;
}

// P^T = 2^(S^T c - LSE2) for one key row and 64 query columns, kept in pe
// (fp32) and stored to TMEM as bf16 for the dV MMA.  MASK is a template
// argument so that unmasked tiles run a branch-free body; the caller picks it
// uniformly per warp (tcgen05.st is warp-collective), and the masked body zeroes
// key rows past the sequence and, under the causal mask (diag: the query tile
// does not lie wholly after the key tile), keys after the query: key row r is
// hidden from query column qc when qc + qoff < r, qoff = 128 (query tile - key
// tile), which is 0 on the diagonal tile and -128 on the tile before it (all
// hidden; a CTA pair's second key tile meets it).
template <bool MASK, int QW = 64, int POLY16 = FA_BWD_POLY_PER16>
__device__ __forceinline__ void dkdv_p(const uint32_t (&sv)[QW / 32][32], float (&pe)[QW], const float *lse2_s,
                                       float scale_log2, int wg, int r, bool row_valid, bool diag, int qoff,
                                       uint32_t p_tm) {
#pragma unroll
  for (int c = 0; c < QW / 32; ++c) {
    uint32_t w[16];
#pragma unroll
    for (int k = 0; k < 32; k += 4) {
      const float4 l4 = *reinterpret_cast<const float4 *>(lse2_s + 32 * c + k);
      float x[4];
      ffma2(x[0], x[1], __uint_as_float(sv[c][k]), __uint_as_float(sv[c][k + 1]), scale_log2, scale_log2, -l4.x,
            -l4.y);
      ffma2(x[2], x[3], __uint_as_float(sv[c][k + 2]), __uint_as_float(sv[c][k + 3]), scale_log2, scale_log2, -l4.z,
            -l4.w);
      static_assert(POLY16 % 2 == 0, "pairs of columns share one packed evaluation");
#pragma unroll
      for (int u = 0; u < 4; u += 2) {
        if ((32 * c + k + u) % 16 < POLY16) {
          exp2_poly2(x[u], x[u + 1], pe[32 * c + k + u], pe[32 * c + k + u + 1]);
        } else {
          pe[32 * c + k + u] = ex2_mufu(x[u]);
          pe[32 * c + k + u + 1] = ex2_mufu(x[u + 1]);
        }
      }
      if (MASK) {
        const int qc = QW * wg + 32 * c + k + qoff;  // query column within tile i, relative to the key tile
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (!row_valid || (diag && qc + u < r)) pe[32 * c + k + u] = 0.f;
      }
      w[k >> 1] = pack_bf16x2(pe[32 * c + k], pe[32 * c + k + 1]);
      w[(k >> 1) + 1] = pack_bf16x2(pe[32 * c + k + 2], pe[32 * c + k + 3]);
    }
    tmem_st_32x32b_x16(p_tm + 16 * c, w);
  }
}

// Key-row elementwise work of the dK/dV kernels over all iterations: one thread
// per key row (TMEM lane), warpgroup wg owns query columns [64 wg, 64 wg + 64).
//   P^T  = 2^(S^T c - LSE2), masked -> registers (fp32) and TMEM over S^T (bf16, dV's A operand)
//   dS^T = P^T (dP^T - D)            -> TMEM over dP^T (bf16, dK's A operand)
// C names the barriers, the row ring and the TMEM columns.  PAIR: the kernel
// runs as a CTA pair whose rank-0 CTA issues the MMAs; the P and dS signals go
// to that CTA's barriers and every wait has cluster scope.  Returns false if a
// wait ran out.
// git0: iterations the CTA ran before this work unit (rings and barrier phases
// count across units).
template <class C, bool CAUSAL, bool PAIR = false>
__device__ __forceinline__ bool dkdv_rows(const BwdParams &p, const uint8_t *smem, uint32_t bar0, uint32_t tmem,
                                          const WaitCtx &wctx, int warp, int n_iter, int i_start, int per_head,
                                          int jt, int kv0, int L, int git0 = 0) {
  auto bar = [&](int i) { return bar0 + 8u * i; };
  auto wait_warp = [&](uint32_t b, uint32_t parity, int site) {
    return PAIR ? mbar_wait_warp_cl(b, parity, wctx, site) : mbar_wait_warp(b, parity, wctx, site);
  };
  auto signal_mma = [&](int i) {  // the MMA-issuing CTA's barrier i
    if (PAIR) mbar_arrive_warp_cluster(mapa_shared(bar(i), 0));
    else mbar_arrive_warp(bar(i));
  };
  constexpr int QW = 128 / C::kNumWG;  // query columns per warpgroup
  constexpr int NC = QW / 32;          // 32-column chunks per thread
  const int wg = warp >> 2;            // query columns [QW wg, QW wg + QW)
  const int r = threadIdx.x & 127;     // key row within the tile == TMEM lane
  const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
  const uint32_t s_tm0 = tmem + lane_off + C::kColS + QW * wg;  // S^T columns of this warpgroup (buffer 0)
  const uint32_t dp_tm = tmem + lane_off + C::kColDP + QW * wg;
  const uint32_t ds_tm = dp_tm;                                // dS^T (bf16) over the first QW / 2 dP^T columns
  const bool row_valid = kv0 + r < L;  // key rows past the sequence: P = 0
  const bool warp_has_invalid = __any_sync(0xffffffffu, !row_valid);
  bool ok = true;
  for (int it = 0; it < n_iter && ok; ++it) {
    const unsigned gi = (unsigned)(git0 + it);  // iteration count over the CTA's units
    const int rs = gi % C::kRowStages;
    const int i = i_start + it % per_head;
    const float *lse2_s = reinterpret_cast<const float *>(smem + C::kOffRows + 1024 * rs) + QW * wg;
    const float *dlt_s = lse2_s + 128;
    // ---- P^T = 2^(S^T c - LSE2), masked; bf16 into TMEM over S^T
    const int sb = gi % C::kSBufs;  // S^T buffer of this iteration
    const uint32_t s_tm = s_tm0 + 128u * sb;
    const uint32_t p_tm = s_tm;  // P^T (bf16) over the first QW / 2 of the S^T columns
    ok = wait_warp(bar(C::kBarS + sb), (gi / C::kSBufs) & 1, kBSiteS);
    if (ok) ok = mbar_wait_warp(bar(C::kBarRowFull0 + rs), (gi / C::kRowStages) & 1, wctx, kBSiteFull);
    if (!ok) break;
    if (threadIdx.x == 0) FA_TRACE_EV(0, it, 0);
    tc_fence_after();
    const bool diag = CAUSAL && i <= jt;
    const int qoff = 128 * (i - jt);
    const bool need_mask = warp_has_invalid || diag;  // uniform across the warp
    uint32_t sv[NC][32];
#pragma unroll
    for (int c = 0; c < NC; ++c) tmem_ld_32x32b_x32(s_tm + 32 * c, sv[c]);
    tmem_wait_ld(sv[0]);
#pragma unroll
    for (int c = 1; c < NC; ++c) reg_tie(sv[c]);
    float pe[QW];
    if (need_mask)
      dkdv_p<true, QW>(sv, pe, lse2_s, p.scale_log2, wg, r, row_valid, diag, qoff, p_tm);
    else
      dkdv_p<false, QW>(sv, pe, lse2_s, p.scale_log2, wg, r, row_valid, diag, qoff, p_tm);
    tmem_wait_st();
    tc_fence_before();
    if (!(FA_STALL(2) && gi == 0)) signal_mma(C::kBarP + sb);
    if (threadIdx.x == 0) FA_TRACE_EV(0, it, 1);
    // ---- dS^T = P^T (dP^T - D) -> TMEM (bf16) over the dP^T columns just read
    ok = wait_warp(bar(C::kBarDP), gi & 1, kBSiteDP);
    if (!ok) break;
    if (threadIdx.x == 0) FA_TRACE_EV(0, it, 2);
    tc_fence_after();
    uint32_t dpv[NC][32];
#pragma unroll
    for (int c = 0; c < NC; ++c) tmem_ld_32x32b_x32(dp_tm + 32 * c, dpv[c]);
    tmem_wait_ld(dpv[0]);
#pragma unroll
    for (int c = 1; c < NC; ++c) reg_tie(dpv[c]);
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      uint32_t w[16];
#pragma unroll
      for (int k = 0; k < 32; k += 4) {
        const float4 d4 = *reinterpret_cast<const float4 *>(dlt_s + 32 * c + k);
        float t[4], ds[4];
        fadd2(t[0], t[1], __uint_as_float(dpv[c][k]), __uint_as_float(dpv[c][k + 1]), -d4.x, -d4.y);
        fadd2(t[2], t[3], __uint_as_float(dpv[c][k + 2]), __uint_as_float(dpv[c][k + 3]), -d4.z, -d4.w);
        fmul2(ds[0], ds[1], pe[32 * c + k], pe[32 * c + k + 1], t[0], t[1]);
        fmul2(ds[2], ds[3], pe[32 * c + k + 2], pe[32 * c + k + 3], t[2], t[3]);
        w[k >> 1] = pack_bf16x2(ds[0], ds[1]);
        w[(k >> 1) + 1] = pack_bf16x2(ds[2], ds[3]);
      }
      tmem_st_32x32b_x16(ds_tm + 16 * c, w);
    }
    tmem_wait_st();
    tc_fence_before();
    signal_mma(C::kBarDS);
    mbar_arrive_warp(bar(C::kBarRowEmpty0 + rs));  // LSE2 / D rows of this stage no longer read
    if (threadIdx.x == 0) FA_TRACE_EV(0, it, 3);
  }
  return ok;
}

// ================================================================== dK, dV
template <int D, bool PERSIST = false>
struct DkdvCfg {
  static constexpr int kTile = 128 * D * 2;  // one 128-row bf16 tile
  // Q_i and dO_i stream through a ring of single-tile slots (Q_i = fill 2i,
  // dO_i = fill 2i + 1), so loads run more than two iterations ahead; the
  // per-iteration LSE2 / D rows go through their own small ring.
  static constexpr int kSlots = (D == 64) ? 10 : 5;
  // Q and dO have rings of their own: a Q slot is released when dK_i completes,
  // a dO slot when dV_i does (earlier), so each load gets more than a load
  // latency of lead.  (One shared round-robin ring tied every dO load to the dK
  // of two iterations back and left it short of its latency.)
  static constexpr int kQSlots = (3 * kSlots + 4) / 5;  // 5 -> 3, 10 -> 6
  static constexpr int kDoSlots = kSlots - kQSlots;
  // fill 2 i = Q_i, fill 2 i + 1 = dO_i (fills count up from 0: unsigned
  // arithmetic, no sign fix-ups on the MMA warp's handoff path)
  __device__ static int slot(int fill) {
    const unsigned i = (unsigned)fill >> 1;
    return (int)((fill & 1) ? kQSlots + i % kDoSlots : i % kQSlots);
  }
  __device__ static uint32_t phase(int fill) {
    const unsigned i = (unsigned)fill >> 1;
    return ((fill & 1) ? i / kDoSlots : i / kQSlots) & 1u;
  }
  static constexpr int kRowStages = 2;  // own full/empty barriers, released after each dS
  // Elementwise warpgroups (thread = key row, a warpgroup per 128 / kNumWG query
  // columns).  Four at head dim 64 (576 threads, 95 registers) halve each
  // thread's share of the exponentials and dS, but measured 1-4 % slower on
  // GB300 than two: the iteration is bound by the chain of handoffs between the
  // MMA and elementwise warps, not by their throughput.
  static constexpr int kNumWG = 2;
  static constexpr int kThreads = 32 * (4 * kNumWG + 2);
  static constexpr int kMmaWarp = 4 * kNumWG, kLoadWarp = 4 * kNumWG + 1;
  // S^T buffers: at head dim 64 TMEM holds two, so S^T_{i+2} is computed while
  // the elementwise warps work on iteration i and they never wait for S^T; at
  // 128 the accumulators leave room for one.
  static constexpr int kSBufs = (D == 64) ? 2 : 1;
  static constexpr int kColS = 0, kColDP = 128 * kSBufs, kColDV = kColDP + 128, kColDK = kColDV + D;
  static constexpr int kTmemCols = 512;
  static_assert(kColDK + D <= kTmemCols, "TMEM budget");
  // PERSIST: the grid is at most one CTA per SM and each CTA runs work units
  // blockIdx.x, blockIdx.x + gridDim.x, ...; the ring then already holds the
  // next unit's Q and dO when the dK/dV epilogue runs, so at head dim 64 the
  // epilogue stages through a region of its own and at 128 (no room for one)
  // each thread writes its key row to global memory directly.  With one unit
  // per CTA the staging reuses ring slots 0 and 1, drained once every MMA has
  // completed.
  static constexpr bool kPersist = PERSIST;
  static constexpr bool kOwnStage = PERSIST && D == 64, kDirectStore = PERSIST && D == 128;
  static_assert(!PERSIST || D <= 128, "persistent dK/dV CTAs: head dim 64 or 128");
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kTile;
  static constexpr int kOffRing = 2 * kTile;
  static constexpr int kOffRows = kOffRing + kSlots * kTile;  // row stage r: LSE2 at +1024r, D at +1024r+512
  static constexpr int kOffStage = kOwnStage ? kOffRows + 1024 * kRowStages : kOffRing;  // dV, then dK at +kTile
  enum { kBarKV, kBarFull0, kBarEmpty0 = kBarFull0 + kSlots, kBarRowFull0 = kBarEmpty0 + kSlots,
         kBarRowEmpty0 = kBarRowFull0 + kRowStages, kBarS = kBarRowEmpty0 + kRowStages,  // S, P: one per S^T buffer
         kBarDP = kBarS + kSBufs, kBarP, kBarDS = kBarP + kSBufs, kBarFinal, kBarDrain,
         kBarKVFree,  // the unit's last S^T and dP^T have read K and V
         kNumBars };
  static constexpr int kOffBar = kOwnStage ? kOffStage + 2 * kTile : kOffRows + 1024 * kRowStages;
  static constexpr int kOffMisc = kOffBar + 8 * kNumBars;
  static constexpr int kSmemBytes = kOffMisc + 16;  // base must be 1024-aligned (checked in the kernel)
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// One work unit of the one-CTA dK/dV kernel: key tile jt of one (batch, kv head).
struct DkdvUnit {
  SeqSpan sq;
  int b, jt, kh, kv0, n_iter, i_start, per_head;
  bool skip;  // packed batch: the tile lies past its sequence, no rows to produce
};

template <bool CAUSAL, bool VARLEN>
__device__ __forceinline__ DkdvUnit dkdv_unit(const BwdParams &p, int u) {
  DkdvUnit w;
  int rank, head;
  work_order(u, (p.N + 127) / 128, p.B * p.Hkv, p.sched_chunk, rank, head);
  w.jt = rank;  // causal: tile 0 sees the most query tiles
  w.kh = head % p.Hkv;
  w.b = head / p.Hkv;
  w.sq = VARLEN ? seq_span(p.cu_seqlens, w.b, p.N, p.total) : SeqSpan{0, p.N, w.b};
  w.kv0 = w.jt * 128;
  w.skip = VARLEN && w.kv0 >= w.sq.len;
  const int n_q = (w.sq.len + 127) / 128;
  w.i_start = CAUSAL ? w.jt : 0;
  w.per_head = n_q - w.i_start;
  w.n_iter = (p.H / p.Hkv) * w.per_head;  // (head, query tile) pairs, head-major; >= 1 unless skip
  return w;
}

// The CTA runs work units blockIdx.x, blockIdx.x + gridDim.x, ... (one per CTA
// at head dim 128, where the grid covers every unit).  The roles go from one
// unit into the next without a block-wide barrier: every ring, S^T buffer and
// barrier phase counts iterations over the CTA's units, the producer loads the
// next unit's K and V once the last MMA reading this unit's has completed
// (kBarKVFree), and the next unit's first S^T and dP^T overlap this unit's
// last elementwise step and epilogue.
template <int D, bool CAUSAL, bool VARLEN, bool PERSIST>
__global__ void __launch_bounds__(DkdvCfg<D, PERSIST>::kThreads, 1) bwd_dkdv_kernel(const __grid_constant__ BwdParams p) {
  using C = DkdvCfg<D, PERSIST>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  if (!check_align(sbase, p.status)) return;
  const uint32_t bar0 = sbase + C::kOffBar;
  auto bar = [&](int i) { return bar0 + 8u * i; };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 4);
  const WaitCtx wctx{abort_flag, p.status};
  FA_CTA_MARK(0, 1);
  if (threadIdx.x == 0) FA_LIFE(0, 0);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = p.H / p.Hkv;
  const int Npad = (p.N + 127) / 128 * 128;  // row-term arrays are [B, H, Npad]
  const int n_units = (p.N + 127) / 128 * p.B * p.Hkv;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kNumBars; ++i) {
      const bool all = (i >= C::kBarP && i < C::kBarP + C::kSBufs) || i == C::kBarDS ||
                       (i >= C::kBarRowEmpty0 && i < C::kBarRowEmpty0 + C::kRowStages);
      mbar_init(bar(i), all ? (uint32_t)(4 * C::kNumWG) : 1u);  // one arrival per elementwise warp
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == C::kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  if (warp == C::kLoadWarp && lane == 0) {
    prefetch_tmap(&p.tm_k);
    prefetch_tmap(&p.tm_v);
    prefetch_tmap(&p.tm_q);
    prefetch_tmap(&p.tm_do);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (threadIdx.x == 0) FA_LIFE(0, 1);

  if (warp < 4 * C::kNumWG) {
    // ===================================================== P^T and dS^T, one warpgroup per 128 / kNumWG query columns
    // P stays in registers (fp32) from its computation to dS; P^T (bf16) goes
    // to TMEM over the S^T columns for the dV MMA, dS^T (bf16) over the dP^T
    // columns once they have been read, for the dK MMA.  After a wait has run
    // out these warps still step through every unit (doing nothing but the
    // epilogue's named barrier), so both warpgroups' barriers stay matched.
    const int wg = warp >> 2;
    const int r = threadIdx.x & 127;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    bool ok = true;
    int git = 0, uc = 0;  // iterations and units this CTA has run
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
      const DkdvUnit w = dkdv_unit<CAUSAL, VARLEN>(p, u);
      if (w.skip) continue;
      if (ok)
        ok = dkdv_rows<C, CAUSAL>(p, smem, bar0, tmem, wctx, warp, w.n_iter, w.i_start, w.per_head, w.jt, w.kv0,
                                  w.sq.len, git);
      git += w.n_iter;
      // ---- epilogue: warpgroup 0 stores dV, warpgroup 1 stores dK * scale; any further warpgroups are done.
      if (wg < 2) {
        // the unit's coordinates again, from a copy of u the compiler cannot
        // match to the first: only u stays live across the iterations
        const DkdvUnit w = dkdv_unit<CAUSAL, VARLEN>(p, C::kPersist ? __shfl_sync(0xffffffffu, u, 0) : u);
        if (ok) ok = mbar_wait_warp(bar(C::kBarFinal), uc & 1, wctx, kBSiteFinal);
        if (threadIdx.x == 0) FA_LIFE(0, 4);
        tc_fence_after();
        uint8_t *stage = smem + C::kOffStage + wg * C::kTile;
        const uint32_t acc_tm = tmem + lane_off + (wg == 0 ? C::kColDV : C::kColDK);
        const float mul = wg == 0 ? 1.0f : p.scale;
        // row by row: no stage (persistent, head dim 128), or the next sequence's rows follow
        const bool direct = C::kDirectStore || (VARLEN && w.kv0 + 128 > w.sq.len);
        if (C::kOwnStage) {
          // every thread of the warpgroup, whatever ok: the previous unit's TMA
          // store has read the stage (its wait is deferred to here, off the
          // unit boundary; measured 1-6 % faster at short sequences)
          if (r == 0) bulk_wait_read_all();
          if (wg == 0) named_bar_sync(1, 128);
          else named_bar_sync(2, 128);
        }
        if (ok && direct) {
          __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(wg == 0 ? p.dv : p.dk);
          // first row of the sequence: packed batches start at sq.start, fixed-length ones at b N
          const size_t row0 = VARLEN ? (size_t)w.sq.start : (size_t)w.b * p.N;
          acc_to_global<D>(acc_tm, out + ((row0 + w.kv0 + r) * p.Hkv + w.kh) * D, 0, mul, w.kv0 + r < w.sq.len);
        } else if (ok) {
          acc_to_smem<D>(acc_tm, stage, r, 0, mul);
        }
        tc_fence_before();  // the accumulator reads precede the next unit's first dV / dK MMA
        fence_proxy_async_smem();
        if (wg == 0) named_bar_sync(1, 128);
        else named_bar_sync(2, 128);
        if (r == 0 && ok && !direct) {
          const CUtensorMap *map = wg == 0 ? &p.tm_dv : &p.tm_dk;
          for (int bx = 0; bx < D / 64; ++bx)
            tma_store_4d(map, smem_u32(stage) + bx * 16384, bx * 64, w.kh, w.sq.start + w.kv0, w.sq.bc);
          bulk_commit();
          if (!C::kOwnStage) bulk_wait_read_all();
          if (threadIdx.x == 0) FA_LIFE(0, 5);
        }
      }
      ++uc;
      if (!C::kPersist) break;  // one unit per CTA
    }
    if (C::kOwnStage && r == 0 && wg < 2) bulk_wait_read_all();  // the last unit's store
  } else if (warp == C::kMmaWarp) {
    // ===================================================== MMA issue
    // Order (one S^T buffer): S_0 dP_0 | [P_0] dV_0 S_1 [dS_0] dK_0 dP_1 | [P_1] dV_1 S_2 [dS_1] dK_1 dP_2 | ...
    // P^T_i (S^T columns) is read by dV_i, which precedes S_{i+1}; dS^T_i (dP^T
    // columns) is read by dK_i, which precedes dP_{i+1}: the tensor pipe runs
    // one thread's MMAs in order.  The elementwise warps have loaded S^T_i and
    // dP^T_i into registers before they signal P_i and dS_i.  With two S^T
    // buffers S runs one iteration further ahead: S_0 S_1 dP_0 | [P_0] dV_0 S_2
    // [dS_0] dK_0 dP_1 | ..., S_{i+2} overwriting buffer i % 2 after dV_i.
    // Indices count over the CTA's units; a unit's first S and dP wait for its
    // K and V, and its first dV and dK (which overwrite the accumulators) follow
    // its first P and dS, signalled after the previous epilogue read them.
    // The whole warp runs the loop and waits; the elected lane issues.
    {
      constexpr uint32_t id_kk = make_idesc_bf16(128, 128, false, false);  // S^T, dP^T
      constexpr uint32_t id_dv = make_idesc_bf16(128, D, false, true);     // dV, dK (A in TMEM, B MN-major)
      const uint64_t k_d = make_sdesc_sw128(sbase + C::kOffK, 0, 1024);
      const uint64_t v_d = make_sdesc_sw128(sbase + C::kOffV, 0, 1024);
      const uint64_t ring_d = make_sdesc_sw128(sbase + C::kOffRing, 0, 1024);        // K-major view
      const uint64_t ring_mn = make_sdesc_sw128(sbase + C::kOffRing, 16384, 1024);   // MN-major view
      auto kmaj = [](int kk) { return (uint64_t)((((kk >> 2) * 16384 + (kk & 3) * 32)) >> 4); };
      auto slot_of = [](int fill) { return C::slot(fill); };
      auto soff = [&](int fill) { return (uint64_t)((slot_of(fill) * C::kTile) >> 4); };
      auto full_ok = [&](int fill) {
        return mbar_wait_warp(bar(C::kBarFull0 + slot_of(fill)), C::phase(fill), wctx, kBSiteFull);
      };
      auto issue_s = [&](unsigned gi) {  // S^T = K Q^T   (Q_gi is fill 2 gi) into buffer gi % kSBufs
        const unsigned sb = gi % C::kSBufs;
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss(tmem + C::kColS + 128u * sb, k_d + kmaj(kk), ring_d + soff(2 * gi) + kmaj(kk), id_kk, kk > 0);
          tc_commit(bar(C::kBarS + sb));
        }
        __syncwarp();
      };
      auto issue_dp = [&](unsigned gi, bool last) {  // dP^T = V dO^T   (dO_gi is fill 2 gi + 1)
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss(tmem + C::kColDP, v_d + kmaj(kk), ring_d + soff(2 * gi + 1) + kmaj(kk), id_kk, kk > 0);
          tc_commit(bar(C::kBarDP));
          if (C::kPersist && last) tc_commit(bar(C::kBarKVFree));  // the unit's last MMA reading K or V
        }
        __syncwarp();
      };
      // A operand in TMEM: the QW query columns of warpgroup w start at column
      // QW w of the region, in bf16 pairs; 16 query rows per K step = 8 columns.
      constexpr int QW = 128 / C::kNumWG, KPW = QW / 16;  // query columns and 16-row K steps per warpgroup
      auto a_col = [](int kk) { return (uint32_t)(QW * (kk / KPW) + 8 * (kk % KPW)); };
      bool ok = true;
      int git = 0, uc = 0;
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
        const DkdvUnit w = dkdv_unit<CAUSAL, VARLEN>(p, u);
        if (w.skip) continue;
        const int n_iter = w.n_iter, G = git;
        ok = mbar_wait_warp(bar(C::kBarKV), uc & 1, wctx, kBSiteKV);
        if (ok) ok = full_ok(2 * G);
        if (ok) {
          tc_fence_after();
          issue_s(G);
          if (uc == 0 && lane == 0) FA_LIFE(0, 3);
          if (C::kSBufs == 2 && n_iter > 1) {
            ok = full_ok(2 * (G + 1));
            if (ok) {
              tc_fence_after();
              issue_s(G + 1);
            }
          }
          if (ok) ok = full_ok(2 * G + 1);
        }
        if (ok) {
          tc_fence_after();
          issue_dp(G, n_iter == 1);
        }
        for (int it = 0; it < n_iter && ok; ++it) {
          const unsigned gi = (unsigned)(G + it);
          const bool more = it + 1 < n_iter;
          const unsigned sb = gi % C::kSBufs;
          FA_TRACE_EV(0, it, 8);
          ok = mbar_wait_warp(bar(C::kBarP + sb), (gi / C::kSBufs) & 1, wctx, kBSiteP);
          if (!ok) break;
          FA_TRACE_EV(0, it, 9);
          tc_fence_after();
          // dV += P^T dO_gi
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ts(tmem + C::kColDV, tmem + C::kColS + 128u * sb + a_col(kk),
                     ring_mn + soff(2 * gi + 1) + (uint64_t)(kk * 128), id_dv, (it > 0 || kk > 0));
            tc_commit(bar(C::kBarEmpty0 + slot_of(2 * gi + 1)));  // dO_gi consumed (dP_gi, dV_gi)
          }
          __syncwarp();
          if (it + C::kSBufs < n_iter) {  // S^T of iteration gi + kSBufs, over P^T_gi's buffer
            FA_TRACE_EV(0, it, 12);
            ok = full_ok(2 * (gi + C::kSBufs));
            if (!ok) break;
            FA_TRACE_EV(0, it, 13);
            tc_fence_after();
            issue_s(gi + C::kSBufs);
          }
          ok = mbar_wait_warp(bar(C::kBarDS), gi & 1, wctx, kBSiteDS);
          if (!ok) break;
          FA_TRACE_EV(0, it, 10);
          tc_fence_after();
          // dK += dS^T Q_gi
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ts(tmem + C::kColDK, tmem + C::kColDP + a_col(kk), ring_mn + soff(2 * gi) + (uint64_t)(kk * 128),
                     id_dv, (it > 0 || kk > 0));
            tc_commit(bar(C::kBarEmpty0 + slot_of(2 * gi)));  // Q_gi consumed (S_gi, dK_gi)
          }
          __syncwarp();
          if (more) {
            ok = full_ok(2 * gi + 3);
            if (!ok) break;
            tc_fence_after();
            issue_dp(gi + 1, it + 2 == n_iter);
          }
          FA_TRACE_EV(0, it, 11);
        }
        if (elect_one()) tc_commit(bar(C::kBarFinal));  // the unit's accumulators are complete
        __syncwarp();
        git += n_iter;
        ++uc;
        if (!C::kPersist) break;
      }
      if (elect_one()) tc_commit(bar(C::kBarDrain));
      __syncwarp();
      if (!mbar_wait_warp(bar(C::kBarDrain), 0, wctx, kBSiteDrain) && *abort_flag) {
        const uint64_t t0 = global_timer_ns();
        while (!mbar_test(bar(C::kBarDrain), 0) && global_timer_ns() - t0 < kWaitLimitNs) {}
      }
    }
  } else {
    // ===================================================== TMA producer
    if (lane == 0) {
      const uint64_t keep = policy_evict_last();  // Q, dO, LSE2, D are re-read by every key tile
      bool ok = true;
      int fill = 0, rows_issued = 0, git = 0, uc = 0;
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
        const DkdvUnit w = dkdv_unit<CAUSAL, VARLEN>(p, u);
        if (w.skip) continue;
        // K and V of this unit, once the previous unit's last S^T and dP^T have read theirs
        if (uc > 0) ok = mbar_wait(bar(C::kBarKVFree), (uc - 1) & 1, wctx, kBSiteEmpty);
        if (!ok) break;
        mbar_arrive_expect_tx(bar(C::kBarKV), 2 * C::kTile);
        for (int bx = 0; bx < D / 64; ++bx) {
          tma_load_4d(sbase + C::kOffK + bx * 16384, &p.tm_k, bar(C::kBarKV), bx * 64, w.kh, w.sq.start + w.kv0,
                      w.sq.bc);
          tma_load_4d(sbase + C::kOffV + bx * 16384, &p.tm_v, bar(C::kBarKV), bx * 64, w.kh, w.sq.start + w.kv0,
                      w.sq.bc);
        }
        // LSE2 / D rows of the unit's iteration it2 into row stage (git + it2) % kRowStages,
        // once the elementwise warps are done with the iteration kRowStages before it
        int next_row = 0;  // the unit's first iteration whose rows are not issued yet
        auto row_stage_free = [&](int it2) {
          const unsigned g2 = (unsigned)(git + it2);
          return mbar_test(bar(C::kBarRowEmpty0 + g2 % C::kRowStages), ((g2 / C::kRowStages) & 1u) ^ 1u);
        };
        auto issue_rows = [&](int it2, bool wait) {
          const unsigned g2 = (unsigned)(git + it2);
          const unsigned rs = g2 % C::kRowStages;
          if (wait && !mbar_wait(bar(C::kBarRowEmpty0 + rs), ((g2 / C::kRowStages) & 1u) ^ 1u, wctx, kBSiteEmpty))
            return false;
          const int hh2 = w.kh * g + it2 / w.per_head;
          const int i2 = w.i_start + it2 % w.per_head;
          const uint32_t rb = bar(C::kBarRowFull0 + rs);
          mbar_arrive_expect_tx(rb, 1024);
          const size_t roff = ((size_t)w.b * p.H + hh2) * Npad + (size_t)i2 * 128;
          const uint32_t rdst = sbase + C::kOffRows + 1024 * rs;
          bulk_load(rdst, p.lse2 + roff, 512, rb);
          bulk_load(rdst + 512, p.delta + roff, 512, rb);
          FA_TRACE_EV(0, it2, 6);
          ++rows_issued;
          return true;
        };
        for (int it = 0; it < w.n_iter && ok; ++it) {
          const int hh = w.kh * g + it / w.per_head;
          const int i = w.i_start + it % w.per_head;
          for (int t = 0; t < 2 && ok; ++t, ++fill) {  // t = 0: Q_gi, t = 1: dO_gi
            const int s = C::slot(fill);
            ok = mbar_wait(bar(C::kBarEmpty0 + s), C::phase(fill) ^ 1, wctx, kBSiteEmpty);
            if (!ok) break;
            const uint32_t fb = bar(C::kBarFull0 + s);
            mbar_arrive_expect_tx(fb, C::kTile);
            const uint32_t dst = sbase + C::kOffRing + s * C::kTile;
            for (int bx = 0; bx < D / 64; ++bx)
              tma_load_4d_hint(dst + bx * 16384, t == 0 ? &p.tm_q : &p.tm_do, fb, bx * 64, hh, w.sq.start + i * 128,
                               w.sq.bc, keep);
            FA_TRACE_EV(0, it, 4 + t);
          }
          if (!ok) break;
          if (D == 64) {
            // Head dim 64: a blocking wait for this iteration's row stage would hold
            // back the next Q and dO fills (two row stages let the producer run only
            // two iterations ahead).  Issue the previous iteration's rows if still
            // pending (blocking: they lag by at most one), then this iteration's only
            // if its stage is already free.  (Measured 1.5-3.5 % faster at d = 64,
            // no gain at 128.)
            while (ok && next_row < it) ok = issue_rows(next_row++, true);
            if (ok && row_stage_free(it)) ok = issue_rows(next_row++, false);
          } else {
            ok = issue_rows(next_row++, true);
          }
        }
        while (ok && next_row < w.n_iter) ok = issue_rows(next_row++, true);  // the unit's last rows
        git += w.n_iter;
        ++uc;
        if (!C::kPersist) break;
      }
      const uint64_t t0 = global_timer_ns();
      // the last issued fill of each slot: Q_i for the last kQSlots i issued, dO_i for the last kDoSlots
      const int nq = (fill + 1) / 2, nd = fill / 2;
      for (int i = max(0, nq - C::kQSlots); i < nq; ++i)
        while (!mbar_test(bar(C::kBarFull0 + C::slot(2 * i)), C::phase(2 * i)) &&
               global_timer_ns() - t0 < kWaitLimitNs) {}
      for (int i = max(0, nd - C::kDoSlots); i < nd; ++i)
        while (!mbar_test(bar(C::kBarFull0 + C::slot(2 * i + 1)), C::phase(2 * i + 1)) &&
               global_timer_ns() - t0 < kWaitLimitNs) {}
      for (int f = max(0, rows_issued - C::kRowStages); f < rows_issued; ++f)
        while (!mbar_test(bar(C::kBarRowFull0 + f % C::kRowStages), (f / C::kRowStages) & 1) &&
               global_timer_ns() - t0 < kWaitLimitNs) {}
      // the last K / V load issued (unit uc - 1; a load is issued for every unit counted)
      if (uc > 0)
        while (!mbar_test(bar(C::kBarKV), (uc - 1) & 1) && global_timer_ns() - t0 < kWaitLimitNs) {}
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  FA_CTA_MARK(0, 2);
  if (threadIdx.x == 0) FA_LIFE(0, 6);
}

// ================================================================== dK, dV on CTA pairs (head dim 128)
// The pages put the backward's bottleneck in shared-memory bandwidth and name
// the tensor cores' CTA-pair mode as its remedy (FA4 paper summary, section
// 2.C; FA4 article, "Capacidades de Blackwell que lo hicieron posible"): one
// MMA of M = 256 rows runs on the two SMs of a cluster pair, each holding its
// own 128 rows of A and half of B, so each SM reads half of every B operand.
//
// A cluster of two CTAs shares one 256-row key tile: CTA c (cluster rank c)
// owns key rows 128c..128c+127 of it (K, V resident, dK, dV, S^T, dP^T in its
// own TMEM, its own elementwise warps), and the pair walks the query tiles
// together.  The rank-0 CTA issues every MMA for both:
//   S^T  = K Q^T,  dP^T = V dO^T   M = 256 keys, N = 128 queries: CTA c
//                                  supplies query rows 64c..64c+63 (all d)
//   dV += P^T dO,  dK += dS^T Q     M = 256 keys, N = 128 = d: CTA c supplies
//                                  head-dim columns 64c..64c+63 (all queries)
// Each ring slot of Q (or dO) therefore holds, at the same offsets in both CTAs,
// the CTA's head-dim half for all 128 rows (16 KB, read MN-major by dK/dV) and
// its 64 query rows in both halves (2 x 8 KB, read K-major by S^T/dP^T).  The
// MMAs read 2/3 of the shared-memory bytes of the one-CTA kernel per SM.
// Both CTAs' loads complete on the rank-0 CTA's barriers; its commits arrive
// on the barriers of both CTAs; the elementwise warps of both signal the rank-0
// CTA.  Every wait is bounded, and every thread reaches the final cluster
// barrier, so neither CTA leaves while the other may still use its memory.
struct DkdvPairCfg : DkdvCfg<128> {
  static constexpr int kHalfBytes = 64 * 128;    // 64 rows x 64 columns of bf16 (8 KB)
  static constexpr int kOffRowHalves = 16384;    // in a slot: the MN-major half first, then the row halves
};

template <bool CAUSAL, bool VARLEN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(320, 1) bwd_dkdv_pair_kernel(const __grid_constant__ BwdParams p) {
  using C = DkdvPairCfg;
  constexpr int D = 128;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  if (!check_align(sbase, p.status)) return;  // same layout in both CTAs: both return
  const uint32_t bar0 = sbase + C::kOffBar;
  auto bar = [&](int i) { return bar0 + 8u * i; };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 4);
  const WaitCtx wctx{abort_flag, p.status};
  FA_CTA_MARK(0, 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t crank = cluster_ctarank();
  const int n_kv = (p.N + 127) / 128;
  const int n_pairs = (n_kv + 1) / 2;
  int rank, head;
  work_order((int)(blockIdx.x >> 1), n_pairs, p.B * p.Hkv, p.sched_chunk, rank, head);
  const int jt = 2 * rank + (int)crank;  // this CTA's key tile; causal: pair 0 sees the most query tiles
  const int kh = head % p.Hkv, b = head / p.Hkv;
  const int g = p.H / p.Hkv;
  const SeqSpan sq = VARLEN ? seq_span(p.cu_seqlens, b, p.N, p.total) : SeqSpan{0, p.N, b};
  const int L = sq.len;
  const int Npad = (p.N + 127) / 128 * 128;
  const int kv0 = jt * 128;
  if (VARLEN && 256 * rank >= L) return;  // the pair's tile lies past its sequence (both CTAs return)
  const int n_q = (L + 127) / 128;
  const int i_start = CAUSAL ? 2 * rank : 0;  // the pair's first key tile decides; the second masks it whole
  const int per_head = n_q - i_start;
  const int n_iter = g * per_head;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kNumBars; ++i) {
      // P and dS collect one arrival per elementwise warp of both CTAs; the row
      // ring is local (8 warps); the rest take one arrival (a producer or a commit)
      const bool pair_warps = i == C::kBarP || i == C::kBarDS;
      const bool local_warps = i >= C::kBarRowEmpty0 && i < C::kBarRowEmpty0 + C::kRowStages;
      mbar_init(bar(i), pair_warps ? 16u : local_warps ? 8u : 1u);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == C::kMmaWarp) {
    tmem_alloc_pair(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish_pair();
  }
  if (warp == C::kLoadWarp && lane == 0) {
    prefetch_tmap(&p.tm_q);
    prefetch_tmap(&p.tm_q64);
    prefetch_tmap(&p.tm_k);
    prefetch_tmap(&p.tm_v);
    prefetch_tmap(&p.tm_do);
    prefetch_tmap(&p.tm_do64);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // barriers of both CTAs initialised, TMEM of both allocated
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 8) {
    // ===================================================== P^T and dS^T (this CTA's key rows)
    const int wg = warp >> 2;
    const int r = threadIdx.x & 127;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    bool ok = dkdv_rows<C, CAUSAL, true>(p, smem, bar0, tmem, wctx, warp, n_iter, i_start, per_head, jt, kv0, L);
    if (ok) ok = mbar_wait_warp_cl(bar(C::kBarFinal), 0, wctx, kBSiteFinal);
    tc_fence_after();
    uint8_t *stage = smem + C::kOffRing + wg * C::kTile;
    const uint32_t acc_tm = tmem + lane_off + (wg == 0 ? C::kColDV : C::kColDK);
    const float mul = wg == 0 ? 1.0f : p.scale;
    const bool has_rows = kv0 < L;                    // the pair's second tile may lie past the end
    const bool direct = VARLEN && kv0 + 128 > L;      // the next sequence's rows follow: write row by row
    if (ok && has_rows && direct) {
      __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(wg == 0 ? p.dv : p.dk);
      acc_to_global<D>(acc_tm, out + ((size_t)(sq.start + kv0 + r) * p.Hkv + kh) * D, 0, mul, kv0 + r < L);
    } else if (ok && has_rows) {
      acc_to_smem<D>(acc_tm, stage, r, 0, mul);
    }
    fence_proxy_async_smem();
    if (wg == 0) named_bar_sync(1, 128);
    else named_bar_sync(2, 128);
    if (r == 0 && ok && has_rows && !direct) {
      const CUtensorMap *map = wg == 0 ? &p.tm_dv : &p.tm_dk;
      for (int bx = 0; bx < D / 64; ++bx)
        tma_store_4d(map, smem_u32(stage) + bx * 16384, bx * 64, kh, sq.start + kv0, sq.bc);
      bulk_commit();
      bulk_wait_read_all();
    }
  } else if (warp == C::kMmaWarp) {
    // ===================================================== MMA issue (rank-0 CTA, for both)
    // Same order as the one-CTA kernel: S_0 dP_0 | [P_0] dV_0 S_1 [dS_0] dK_0 dP_1 | ...
    if (crank == 0) {
      constexpr uint32_t id_kk = make_idesc_bf16(256, 128, false, false);  // S^T, dP^T
      constexpr uint32_t id_dv = make_idesc_bf16(256, D, false, true);     // dV, dK (A in TMEM, B MN-major)
      const uint64_t k_d = make_sdesc_sw128(sbase + C::kOffK, 0, 1024);
      const uint64_t v_d = make_sdesc_sw128(sbase + C::kOffV, 0, 1024);
      const uint64_t ring_d = make_sdesc_sw128(sbase + C::kOffRing + C::kOffRowHalves, 0, 1024);  // row halves
      const uint64_t ring_mn = make_sdesc_sw128(sbase + C::kOffRing, 16384, 1024);                 // column half
      auto kmaj = [](int kk) { return (uint64_t)((((kk >> 2) * 16384 + (kk & 3) * 32)) >> 4); };
      auto kmaj_half = [](int kk) { return (uint64_t)(((kk >> 2) * C::kHalfBytes + (kk & 3) * 32) >> 4); };
      auto soff = [&](int fill) { return (uint64_t)((C::slot(fill) * C::kTile) >> 4); };
      auto full_ok = [&](int fill) {
        return mbar_wait_warp_cl(bar(C::kBarFull0 + C::slot(fill)), C::phase(fill), wctx, kBSiteFull);
      };
      auto issue_s = [&](int it) {  // S^T = K Q^T   (Q_it is fill 2 it)
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss_pair(tmem + C::kColS, k_d + kmaj(kk), ring_d + soff(2 * it) + kmaj_half(kk), id_kk, kk > 0);
          tc_commit_pair(bar(C::kBarS));
        }
        __syncwarp();
      };
      auto issue_dp = [&](int it) {  // dP^T = V dO^T   (dO_it is fill 2 it + 1)
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss_pair(tmem + C::kColDP, v_d + kmaj(kk), ring_d + soff(2 * it + 1) + kmaj_half(kk), id_kk, kk > 0);
          tc_commit_pair(bar(C::kBarDP));
        }
        __syncwarp();
      };
      auto a_col = [](int kk) { return (uint32_t)(64 * (kk >> 2) + 8 * (kk & 3)); };
      bool ok = mbar_wait_warp_cl(bar(C::kBarKV), 0, wctx, kBSiteKV);
      if (ok) ok = full_ok(0);
      if (ok) {
        tc_fence_after();
        issue_s(0);
        ok = full_ok(1);
      }
      if (ok) {
        tc_fence_after();
        issue_dp(0);
      }
      for (int it = 0; it < n_iter && ok; ++it) {
        const bool more = it + 1 < n_iter;
        FA_TRACE_EV(0, it, 8);
        ok = mbar_wait_warp_cl(bar(C::kBarP), it & 1, wctx, kBSiteP);
        if (!ok) break;
        FA_TRACE_EV(0, it, 9);
        tc_fence_after();
        if (elect_one()) {  // dV += P^T dO_it
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts_pair(tmem + C::kColDV, tmem + C::kColS + a_col(kk), ring_mn + soff(2 * it + 1) + (uint64_t)(kk * 128),
                        id_dv, (it > 0 || kk > 0));
          tc_commit_pair(bar(C::kBarEmpty0 + C::slot(2 * it + 1)));  // dO_it consumed (dP_it, dV_it)
        }
        __syncwarp();
        if (more) {
          FA_TRACE_EV(0, it, 12);
          ok = full_ok(2 * it + 2);
          if (!ok) break;
          FA_TRACE_EV(0, it, 13);
          tc_fence_after();
          issue_s(it + 1);
        }
        ok = mbar_wait_warp_cl(bar(C::kBarDS), it & 1, wctx, kBSiteDS);
        if (!ok) break;
        FA_TRACE_EV(0, it, 10);
        tc_fence_after();
        if (elect_one()) {  // dK += dS^T Q_it
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts_pair(tmem + C::kColDK, tmem + C::kColDP + a_col(kk), ring_mn + soff(2 * it) + (uint64_t)(kk * 128),
                        id_dv, (it > 0 || kk > 0));
          tc_commit_pair(bar(C::kBarEmpty0 + C::slot(2 * it)));  // Q_it consumed (S_it, dK_it)
        }
        __syncwarp();
        if (more) {
          ok = full_ok(2 * it + 3);
          if (!ok) break;
          tc_fence_after();
          issue_dp(it + 1);
        }
        FA_TRACE_EV(0, it, 11);
      }
      if (elect_one()) {
        tc_commit_pair(bar(C::kBarFinal));
        tc_commit_pair(bar(C::kBarDrain));
      }
      __syncwarp();
      if (!mbar_wait_warp_cl(bar(C::kBarDrain), 0, wctx, kBSiteDrain) && *abort_flag) {
        const uint64_t t0 = global_timer_ns();
        while (!mbar_test_cl(bar(C::kBarDrain), 0) && global_timer_ns() - t0 < kWaitLimitNs) {}
      }
    }
  } else {
    // ===================================================== TMA producer (both CTAs; bytes counted by rank 0)
    if (lane == 0) {
      const uint64_t keep = policy_evict_last();
      const uint32_t kv_bar = mapa_shared(bar(C::kBarKV), 0);
      if (crank == 0) mbar_arrive_expect_tx(bar(C::kBarKV), 2 * 2 * C::kTile);  // K and V of both CTAs
      for (int bx = 0; bx < D / 64; ++bx) {
        tma_load_4d_pair(sbase + C::kOffK + bx * 16384, &p.tm_k, kv_bar, bx * 64, kh, sq.start + kv0, sq.bc, keep);
        tma_load_4d_pair(sbase + C::kOffV + bx * 16384, &p.tm_v, kv_bar, bx * 64, kh, sq.start + kv0, sq.bc, keep);
      }
      bool ok = true;
      int fill = 0, rows_issued = 0;
      for (int it = 0; it < n_iter && ok; ++it) {
        const int hh = kh * g + it / per_head;
        const int i = i_start + it % per_head;
        const int row0 = sq.start + i * 128;
        for (int t = 0; t < 2 && ok; ++t, ++fill) {  // t = 0: Q_it, t = 1: dO_it
          const int s = C::slot(fill);
          ok = mbar_wait_cl(bar(C::kBarEmpty0 + s), C::phase(fill) ^ 1, wctx, kBSiteEmpty);
          if (!ok) break;
          if (crank == 0) mbar_arrive_expect_tx(bar(C::kBarFull0 + s), 2 * C::kTile);  // both CTAs' 32 KB
          const uint32_t fb = mapa_shared(bar(C::kBarFull0 + s), 0);
          const uint32_t dst = sbase + C::kOffRing + s * C::kTile;
          const CUtensorMap *m128 = t == 0 ? &p.tm_q : &p.tm_do;
          const CUtensorMap *m64 = t == 0 ? &p.tm_q64 : &p.tm_do64;
          // this CTA's head-dim half, all 128 rows (MN-major operand of dK / dV)
          tma_load_4d_pair(dst, m128, fb, 64 * (int)crank, hh, row0, sq.bc, keep);
          // this CTA's 64 query rows, both halves (K-major operand of S^T / dP^T)
          for (int bx = 0; bx < 2; ++bx)
            tma_load_4d_pair(dst + C::kOffRowHalves + bx * C::kHalfBytes, m64, fb, bx * 64, hh,
                             row0 + 64 * (int)crank, sq.bc, keep);
        }
        if (!ok) break;
        const int rs = it % C::kRowStages;
        ok = mbar_wait(bar(C::kBarRowEmpty0 + rs), ((it / C::kRowStages) & 1) ^ 1, wctx, kBSiteEmpty);
        if (!ok) break;
        const uint32_t rb = bar(C::kBarRowFull0 + rs);
        mbar_arrive_expect_tx(rb, 1024);
        const size_t roff = ((size_t)b * p.H + hh) * Npad + (size_t)i * 128;
        const uint32_t rdst = sbase + C::kOffRows + 1024 * rs;
        bulk_load(rdst, p.lse2 + roff, 512, rb);
        bulk_load(rdst + 512, p.delta + roff, 512, rb);
        ++rows_issued;
      }
      // drain: rank 0's full barriers count both CTAs' copies; the row ring is local
      const uint64_t t0 = global_timer_ns();
      if (crank == 0) {
        const int nq = (fill + 1) / 2, nd = fill / 2;
        for (int i = max(0, nq - C::kQSlots); i < nq; ++i)
          while (!mbar_test_cl(bar(C::kBarFull0 + C::slot(2 * i)), C::phase(2 * i)) &&
                 global_timer_ns() - t0 < kWaitLimitNs) {}
        for (int i = max(0, nd - C::kDoSlots); i < nd; ++i)
          while (!mbar_test_cl(bar(C::kBarFull0 + C::slot(2 * i + 1)), C::phase(2 * i + 1)) &&
                 global_timer_ns() - t0 < kWaitLimitNs) {}
        while (!mbar_test_cl(bar(C::kBarKV), 0) && global_timer_ns() - t0 < kWaitLimitNs) {}
      }
      for (int f = max(0, rows_issued - C::kRowStages); f < rows_issued; ++f)
        while (!mbar_test(bar(C::kBarRowFull0 + f % C::kRowStages), (f / C::kRowStages) & 1) &&
               global_timer_ns() - t0 < kWaitLimitNs) {}
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the rank-0 CTA's MMAs and both CTAs' copies are done with both CTAs' memory
  if (warp == C::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, C::kTmemCols);
  }
  FA_CTA_MARK(0, 2);
}

// ================================================================== fused backward on CTA pairs (head dim 128)
// The pages' backward (FA4 paper summary, section 2.C): one KV-stationary pass
// computes dK, dV and dQ; the two CTAs of a pair exchange their halves of dS
// through distributed shared memory, so that each adds dQ for half of the query
// rows, summed over the pair's 256 keys, and the fp32 reductions into global
// memory are halved against a one-CTA kernel.
//
// A cluster of two CTAs shares one 256-row key tile as in bwd_dkdv_pair_kernel
// (same S^T, dP^T, dV, dK MMAs and ring layout), plus per query tile i
//   dQ_i[64c..64c+63, :] += dS[64c..64c+63, 256 keys] K[256 keys, :]
// as one M = 128 CTA-pair MMA: CTA c supplies the 64 dS rows of its query half
// (MN-major: one 128-byte line per key holds its 64 queries) and head-dim
// columns 64c..64c+63 of all 256 K rows; TMEM receives the 64 rows in 64
// columns, lanes 0-63 holding head-dim columns 0-63 and lanes 64-127 the rest.
// Elementwise warpgroup w of either CTA computes dS for query half w of its own
// key rows and writes those lines into CTA w's dS buffer (its own or the
// peer's).  The warps then move the dQ partial from TMEM to the fp32
// accumulator with vector reductions, which makes the result depend on the
// order of the additions (not bitwise reproducible).
//
// TMEM: S^T in columns 0-127 (P^T in bf16 packed into 0-63 once S^T is in
// registers), the dQ partial in 64-127 once the next S^T is in registers; dP^T
// in 128-255 (dS^T over it), dV 256-383, dK 384-511.  Shared memory: K, V, the
// dQ operand K (32 KB each), the dS buffer (32 KB), a three-slot Q/dO ring
// (two Q slots, one dO slot) and the row terms.
struct FusedCfg {
  static constexpr int kTile = 128 * 128 * 2;
  static constexpr int kHalfBytes = 64 * 128;
  static constexpr int kOffRowHalves = 16384;
  static constexpr int kQSlots = 2, kDoSlots = 1, kSlots = kQSlots + kDoSlots;
  __device__ static int slot(int fill) {  // fill 2 i = Q_i, fill 2 i + 1 = dO_i
    const int i = fill >> 1;
    return (fill & 1) ? kQSlots + i % kDoSlots : i % kQSlots;
  }
  __device__ static uint32_t phase(int fill) {
    const int i = fill >> 1;
    return (uint32_t)(((fill & 1) ? i / kDoSlots : i / kQSlots) & 1);
  }
  static constexpr int kRowStages = 2;
  static constexpr int kThreads = 320;
  static constexpr int kMmaWarp = 8, kLoadWarp = 9;
  static constexpr int kColS = 0, kColDQ = 64, kColDP = 128, kColDV = 256, kColDK = 384, kTmemCols = 512;
  static constexpr int kOffK = 0, kOffV = kTile, kOffKB = 2 * kTile, kOffDS = 3 * kTile, kOffRing = 4 * kTile;
  static constexpr int kOffRows = kOffRing + kSlots * kTile;
  enum { kBarKV, kBarFull0, kBarEmpty0 = kBarFull0 + kSlots, kBarRowFull0 = kBarEmpty0 + kSlots,
         kBarRowEmpty0 = kBarRowFull0 + kRowStages, kBarS = kBarRowEmpty0 + kRowStages, kBarDP, kBarDQ, kBarSL,
         kBarP, kBarDS, kBarDQF, kBarFinal, kBarDrain, kBarWG0, kNumBars = kBarWG0 + 4 };
  static constexpr int kOffBar = kOffRows + 1024 * kRowStages;
  static constexpr int kOffMisc = kOffBar + 8 * kNumBars;
  static constexpr int kSmemBytes = kOffMisc + 16;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// dQ partial of query tile t: TMEM -> fp32 reductions into dqacc.  The thread
// of TMEM lane r holds query row 64 crank + (r % 64) of the tile and head-dim
// columns 64 (r / 64) + 32 wg .. + 31.
__device__ __forceinline__ bool fused_dq_out(const BwdParams &p, uint32_t bar0, uint32_t dq_tm, const WaitCtx &wctx,
                                             int t, int row0, int hh, int b, int wg, int r, int L, bool signal_free) {
  using C = FusedCfg;
  auto bar = [&](int i) { return bar0 + 8u * i; };
  if (!mbar_wait_warp(bar(C::kBarDQ), t & 1, wctx, kBSiteDQ)) return false;
  tc_fence_after();
  uint32_t v[2][16];
  tmem_ld_32x32b_x16(dq_tm, v[0]);
  tmem_ld_32x32b_x16(dq_tm + 16, v[1]);
  tmem_wait_ld(v[0]);
  tmem_wait_ld(v[1]);
  tc_fence_before();
  if (signal_free) mbar_arrive_warp_cluster(mapa_shared(bar(C::kBarDQF), 0));  // columns 64-127 may take the next S
  const int q = row0 + (r & 63);
  if (q < L) {
    float *dst = p.dqacc + (((size_t)b * p.N + q) * p.H + hh) * 128 + (r >> 6) * 64 + 32 * wg;
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
      for (int k = 0; k < 16; k += 4)
        red_add_v4(dst + 16 * c + k, __uint_as_float(v[c][k]), __uint_as_float(v[c][k + 1]),
                   __uint_as_float(v[c][k + 2]), __uint_as_float(v[c][k + 3]));
  }
  return true;
}

template <bool CAUSAL>
__device__ __forceinline__ bool fused_rows(const BwdParams &p, const uint8_t *smem, uint32_t sbase, uint32_t bar0,
                                           uint32_t tmem, const WaitCtx &wctx, int warp, uint32_t crank, int n_iter,
                                           int i_start, int per_head, int jt, int kv0, int L, int b, int kh, int g) {
  using C = FusedCfg;
  auto bar = [&](int i) { return bar0 + 8u * i; };
  auto signal_mma = [&](int i) { mbar_arrive_warp_cluster(mapa_shared(bar(i), 0)); };
  const int wg = warp >> 2;         // query columns [64 wg, 64 wg + 64)
  const int r = threadIdx.x & 127;  // key row == TMEM lane
  const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
  const uint32_t s_tm = tmem + lane_off + C::kColS + 64 * wg;
  const uint32_t p_tm = tmem + lane_off + C::kColS + 32 * wg;  // P^T packed: wg 0 in 0-31, wg 1 in 32-63
  const uint32_t dq_tm = tmem + lane_off + C::kColDQ + 32 * wg;
  const uint32_t dp_tm = tmem + lane_off + C::kColDP + 64 * wg;
  const uint32_t ds_tm = dp_tm;
  const bool row_valid = kv0 + r < L;
  const bool warp_has_invalid = __any_sync(0xffffffffu, !row_valid);
  // this key's dS line (64 queries of half wg) in CTA wg's dS buffer
  const int kline = 128 * (int)crank + r;
  const uint32_t ds_line = sbase + C::kOffDS + (uint32_t)kline * 128u;
  const bool ds_local = wg == (int)crank;
  const uint32_t ds_remote = mapa_shared(ds_line, (uint32_t)wg);
  bool ok = true;
  for (int it = 0; it < n_iter && ok; ++it) {
    const int rs = it % C::kRowStages;
    const int i = i_start + it % per_head;
    const float *lse2_s = reinterpret_cast<const float *>(smem + C::kOffRows + 1024 * rs) + 64 * wg;
    const float *dlt_s = lse2_s + 128;
    // ---- S^T -> registers; P^T (bf16) packed into columns 0-63
    ok = mbar_wait_warp(bar(C::kBarS), it & 1, wctx, kBSiteS);
    if (ok) ok = mbar_wait_warp(bar(C::kBarRowFull0 + rs), (it / C::kRowStages) & 1, wctx, kBSiteFull);
    if (!ok) break;
    if (threadIdx.x == 0) FA_TRACE_EV(0, it, 0);
    tc_fence_after();
    uint32_t sv[2][32];
    tmem_ld_32x32b_x32(s_tm, sv[0]);
    tmem_ld_32x32b_x32(s_tm + 32, sv[1]);
    tmem_wait_ld(sv[0]);
    reg_tie(sv[1]);
    tc_fence_before();
    signal_mma(C::kBarSL);  // columns 64-127 may take the previous tile's dQ
    // warps w and w+4 (the same TMEM lanes) both hold their S^T before P^T of
    // warpgroup 1 overwrites columns 32-63 (a bounded wait, unlike bar.sync)
    mbar_arrive_warp(bar(C::kBarWG0 + (warp & 3)));
    ok = mbar_wait_warp(bar(C::kBarWG0 + (warp & 3)), it & 1, wctx, kBSiteS);
    if (!ok) break;
    const bool diag = CAUSAL && i <= jt;
    const int qoff = 128 * (i - jt);
    float pe[64];
    if (warp_has_invalid || diag)
      dkdv_p<true>(sv, pe, lse2_s, p.scale_log2, wg, r, row_valid, diag, qoff, p_tm);
    else
      dkdv_p<false>(sv, pe, lse2_s, p.scale_log2, wg, r, row_valid, diag, qoff, p_tm);
    tmem_wait_st();
    tc_fence_before();
    signal_mma(C::kBarP);
    if (threadIdx.x == 0) FA_TRACE_EV(0, it, 1);
    // ---- the previous tile's dQ partial -> fp32 reductions
    if (it > 0) {
      const int t = it - 1;
      ok = fused_dq_out(p, bar0, dq_tm, wctx, t, (i_start + t % per_head) * 128 + 64 * (int)crank,
                        kh * g + t / per_head, b, wg, r, L, true);
      if (!ok) break;
    }
    if (threadIdx.x == 0) FA_TRACE_EV(0, it, 2);
    // ---- dS^T = P^T (dP^T - D): bf16 into TMEM (dK's A) and as a line of dQ's A
    ok = mbar_wait_warp(bar(C::kBarDP), it & 1, wctx, kBSiteDP);
    if (!ok) break;
    if (threadIdx.x == 0) FA_TRACE_EV(0, it, 3);
    tc_fence_after();
    uint32_t dpv[2][32];
    tmem_ld_32x32b_x32(dp_tm, dpv[0]);
    tmem_ld_32x32b_x32(dp_tm + 32, dpv[1]);
    tmem_wait_ld(dpv[0]);
    reg_tie(dpv[1]);
    uint32_t dsw[32];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
#pragma unroll
      for (int k = 0; k < 32; k += 4) {
        const float4 d4 = *reinterpret_cast<const float4 *>(dlt_s + 32 * c + k);
        float t4[4], ds[4];
        fadd2(t4[0], t4[1], __uint_as_float(dpv[c][k]), __uint_as_float(dpv[c][k + 1]), -d4.x, -d4.y);
        fadd2(t4[2], t4[3], __uint_as_float(dpv[c][k + 2]), __uint_as_float(dpv[c][k + 3]), -d4.z, -d4.w);
        fmul2(ds[0], ds[1], pe[32 * c + k], pe[32 * c + k + 1], t4[0], t4[1]);
        fmul2(ds[2], ds[3], pe[32 * c + k + 2], pe[32 * c + k + 3], t4[2], t4[3]);
        dsw[16 * c + (k >> 1)] = pack_bf16x2(ds[0], ds[1]);
        dsw[16 * c + (k >> 1) + 1] = pack_bf16x2(ds[2], ds[3]);
      }
    }
    tmem_st_32x32b_x16(ds_tm, *reinterpret_cast<const uint32_t(*)[16]>(&dsw[0]));
    tmem_st_32x32b_x16(ds_tm + 16, *reinterpret_cast<const uint32_t(*)[16]>(&dsw[16]));
    // 128B-swizzled line: 16-byte chunk j (queries 8j..8j+7) at chunk j ^ (line % 8)
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t off = (uint32_t)((j ^ (kline & 7)) * 16);
      if (ds_local)
        st_shared_v4(ds_line + off, dsw[4 * j], dsw[4 * j + 1], dsw[4 * j + 2], dsw[4 * j + 3]);
      else
        st_cluster_v4(ds_remote + off, dsw[4 * j], dsw[4 * j + 1], dsw[4 * j + 2], dsw[4 * j + 3]);
    }
    tmem_wait_st();
    fence_proxy_async_cluster();  // the lines reach the tensor core's reads of either CTA
    tc_fence_before();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive_release_cluster(mapa_shared(bar(C::kBarDS), 0));
    mbar_arrive_warp(bar(C::kBarRowEmpty0 + rs));
    if (threadIdx.x == 0) FA_TRACE_EV(0, it, 4);
  }
  if (ok && n_iter > 0) {  // the last tile's dQ
    const int t = n_iter - 1;
    ok = fused_dq_out(p, bar0, dq_tm, wctx, t, (i_start + t % per_head) * 128 + 64 * (int)crank,
                      kh * g + t / per_head, b, wg, r, L, false);
  }
  return ok;
}

template <bool CAUSAL>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(320, 1) bwd_fused_pair_kernel(const __grid_constant__ BwdParams p) {
  using C = FusedCfg;
  constexpr int D = 128;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  if (!check_align(sbase, p.status)) return;  // same layout in both CTAs: both return
  const uint32_t bar0 = sbase + C::kOffBar;
  auto bar = [&](int i) { return bar0 + 8u * i; };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 4);
  const WaitCtx wctx{abort_flag, p.status};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t crank = cluster_ctarank();
  const int n_kv = (p.N + 127) / 128;
  const int n_pairs = (n_kv + 1) / 2;
  int rank, head;
  work_order((int)(blockIdx.x >> 1), n_pairs, p.B * p.Hkv, p.sched_chunk, rank, head);
  const int jt = 2 * rank + (int)crank;
  const int kh = head % p.Hkv, b = head / p.Hkv;
  const int g = p.H / p.Hkv;
  const int L = p.N;
  const int Npad = (p.N + 127) / 128 * 128;
  const int kv0 = jt * 128;
  const int n_q = (L + 127) / 128;
  const int i_start = CAUSAL ? 2 * rank : 0;
  const int per_head = n_q - i_start;
  const int n_iter = g * per_head;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kNumBars; ++i) {
      const bool pair_warps = i == C::kBarP || i == C::kBarDS || i == C::kBarSL || i == C::kBarDQF;
      const bool local_warps = i >= C::kBarRowEmpty0 && i < C::kBarRowEmpty0 + C::kRowStages;
      const bool two_warps = i >= C::kBarWG0;
      mbar_init(bar(i), pair_warps ? 16u : local_warps ? 8u : two_warps ? 2u : 1u);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == C::kMmaWarp) {
    tmem_alloc_pair(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish_pair();
  }
  if (warp == C::kLoadWarp && lane == 0) {
    prefetch_tmap(&p.tm_q);
    prefetch_tmap(&p.tm_q64);
    prefetch_tmap(&p.tm_k);
    prefetch_tmap(&p.tm_v);
    prefetch_tmap(&p.tm_do);
    prefetch_tmap(&p.tm_do64);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 8) {
    // ===================================================== P^T, dS^T, dS lines, dQ reductions
    const int wg = warp >> 2;
    const int r = threadIdx.x & 127;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    bool ok = fused_rows<CAUSAL>(p, smem, sbase, bar0, tmem, wctx, warp, crank, n_iter, i_start, per_head, jt, kv0, L,
                                 b, kh, g);
    if (ok) ok = mbar_wait_warp(bar(C::kBarFinal), 0, wctx, kBSiteFinal);
    tc_fence_after();
    uint8_t *stage = smem + C::kOffRing + wg * C::kTile;
    const uint32_t acc_tm = tmem + lane_off + (wg == 0 ? C::kColDV : C::kColDK);
    const float mul = wg == 0 ? 1.0f : p.scale;
    const bool has_rows = kv0 < L;
    if (ok && has_rows) acc_to_smem<D>(acc_tm, stage, r, 0, mul);
    fence_proxy_async_smem();
    if (wg == 0) named_bar_sync(1, 128);
    else named_bar_sync(2, 128);
    if (r == 0 && ok && has_rows) {
      const CUtensorMap *map = wg == 0 ? &p.tm_dv : &p.tm_dk;
      for (int bx = 0; bx < D / 64; ++bx) tma_store_4d(map, smem_u32(stage) + bx * 16384, bx * 64, kh, kv0, b);
      bulk_commit();
      bulk_wait_read_all();
    }
  } else if (warp == C::kMmaWarp) {
    // ===================================================== MMA issue (rank-0 CTA, for both)
    // S_0 dP_0 | [P_0] dV_0 [DQF_-1] S_1 [dS_0] dK_0 [SL_1] dQ_0 dP_1 | [P_1] dV_1 [DQF_0] S_2 ...
    if (crank == 0) {
      constexpr uint32_t id_kk = make_idesc_bf16(256, 128, false, false);  // S^T, dP^T
      constexpr uint32_t id_dv = make_idesc_bf16(256, D, false, true);     // dV, dK
      constexpr uint32_t id_dq = make_idesc_bf16(128, D, true, true);      // dQ: A (dS) and B (K) MN-major
      const uint64_t k_d = make_sdesc_sw128(sbase + C::kOffK, 0, 1024);
      const uint64_t v_d = make_sdesc_sw128(sbase + C::kOffV, 0, 1024);
      const uint64_t kb_d = make_sdesc_sw128(sbase + C::kOffKB, 16384, 1024);
      const uint64_t ds_d = make_sdesc_sw128(sbase + C::kOffDS, 16384, 1024);
      const uint64_t ring_d = make_sdesc_sw128(sbase + C::kOffRing + C::kOffRowHalves, 0, 1024);
      const uint64_t ring_mn = make_sdesc_sw128(sbase + C::kOffRing, 16384, 1024);
      auto kmaj = [](int kk) { return (uint64_t)((((kk >> 2) * 16384 + (kk & 3) * 32)) >> 4); };
      auto kmaj_half = [](int kk) { return (uint64_t)(((kk >> 2) * C::kHalfBytes + (kk & 3) * 32) >> 4); };
      auto soff = [&](int fill) { return (uint64_t)((C::slot(fill) * C::kTile) >> 4); };
      auto full_ok = [&](int fill) {
        return mbar_wait_warp(bar(C::kBarFull0 + C::slot(fill)), C::phase(fill), wctx, kBSiteFull);
      };
      auto issue_s = [&](int it) {
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss_pair(tmem + C::kColS, k_d + kmaj(kk), ring_d + soff(2 * it) + kmaj_half(kk), id_kk, kk > 0);
          tc_commit_pair(bar(C::kBarS));
        }
        __syncwarp();
      };
      auto issue_dp = [&](int it) {
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss_pair(tmem + C::kColDP, v_d + kmaj(kk), ring_d + soff(2 * it + 1) + kmaj_half(kk), id_kk, kk > 0);
          tc_commit_pair(bar(C::kBarDP));
        }
        __syncwarp();
      };
      auto a_col_ds = [](int kk) { return (uint32_t)(64 * (kk >> 2) + 8 * (kk & 3)); };
      bool ok = mbar_wait_warp(bar(C::kBarKV), 0, wctx, kBSiteKV);
      if (ok) ok = full_ok(0);
      if (ok) {
        tc_fence_after();
        issue_s(0);
        ok = full_ok(1);
      }
      if (ok) {
        tc_fence_after();
        issue_dp(0);
      }
      for (int it = 0; it < n_iter && ok; ++it) {
        const bool more = it + 1 < n_iter;
        FA_TRACE_EV(0, it, 8);
        ok = mbar_wait_warp(bar(C::kBarP), it & 1, wctx, kBSiteP);
        if (!ok) break;
        FA_TRACE_EV(0, it, 9);
        tc_fence_after();
        if (elect_one()) {  // dV += P^T dO_it   (P^T packed in columns 0-63)
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts_pair(tmem + C::kColDV, tmem + C::kColS + 8 * kk, ring_mn + soff(2 * it + 1) + (uint64_t)(kk * 128),
                        id_dv, (it > 0 || kk > 0));
          tc_commit_pair(bar(C::kBarEmpty0 + C::slot(2 * it + 1)));
        }
        __syncwarp();
        if (more) {
          if (it > 0) ok = mbar_wait_warp(bar(C::kBarDQF), (it - 1) & 1, wctx, kBSiteDQF);  // dQ_{it-1} read out
          if (ok) ok = full_ok(2 * it + 2);
          if (!ok) break;
          FA_TRACE_EV(0, it, 12);
          tc_fence_after();
          issue_s(it + 1);
        }
        ok = mbar_wait_warp_acq_cluster(bar(C::kBarDS), it & 1, wctx, kBSiteDS);
        if (!ok) break;
        FA_TRACE_EV(0, it, 10);
        tc_fence_after();
        if (elect_one()) {  // dK += dS^T Q_it
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts_pair(tmem + C::kColDK, tmem + C::kColDP + a_col_ds(kk), ring_mn + soff(2 * it) + (uint64_t)(kk * 128),
                        id_dv, (it > 0 || kk > 0));
          tc_commit_pair(bar(C::kBarEmpty0 + C::slot(2 * it)));
        }
        __syncwarp();
        if (more) {  // the next S^T is in registers: its columns 64-127 may take dQ_it
          ok = mbar_wait_warp(bar(C::kBarSL), (it + 1) & 1, wctx, kBSiteSL);
        } else if (it > 0) {  // no S^T follows (else waited before it): dQ_{it-1} must have been read out
          ok = mbar_wait_warp(bar(C::kBarDQF), (it - 1) & 1, wctx, kBSiteDQF);
        }
        if (!ok) break;
        FA_TRACE_EV(0, it, 11);
        tc_fence_after();
        if (elect_one()) {  // dQ_it = dS K over the pair's 256 keys (16 steps of 16 keys)
#pragma unroll
          for (int kk = 0; kk < 16; ++kk)
            mma_ss_pair(tmem + C::kColDQ, ds_d + (uint64_t)(kk * 128), kb_d + (uint64_t)(kk * 128), id_dq, kk > 0);
          tc_commit_pair(bar(C::kBarDQ));
        }
        __syncwarp();
        if (more) {
          ok = full_ok(2 * it + 3);
          if (!ok) break;
          FA_TRACE_EV(0, it, 13);
          tc_fence_after();
          issue_dp(it + 1);
        }
        FA_TRACE_EV(0, it, 14);
      }
      if (elect_one()) {
        tc_commit_pair(bar(C::kBarFinal));
        tc_commit_pair(bar(C::kBarDrain));
      }
      __syncwarp();
      if (!mbar_wait_warp(bar(C::kBarDrain), 0, wctx, kBSiteDrain) && *abort_flag) {
        const uint64_t t0 = global_timer_ns();
        while (!mbar_test(bar(C::kBarDrain), 0) && global_timer_ns() - t0 < kWaitLimitNs) {}
      }
    }
  } else {
    // ===================================================== TMA producer (both CTAs; bytes counted by rank 0)
    if (lane == 0) {
      const uint64_t keep = policy_evict_last();
      const uint32_t kv_bar = mapa_shared(bar(C::kBarKV), 0);
      if (crank == 0) mbar_arrive_expect_tx(bar(C::kBarKV), 2 * 3 * C::kTile);  // K, V, dQ's K operand, both CTAs
      for (int bx = 0; bx < D / 64; ++bx) {
        tma_load_4d_pair(sbase + C::kOffK + bx * 16384, &p.tm_k, kv_bar, bx * 64, kh, kv0, b, keep);
        tma_load_4d_pair(sbase + C::kOffV + bx * 16384, &p.tm_v, kv_bar, bx * 64, kh, kv0, b, keep);
      }
      // dQ's B operand: head-dim half crank of both key tiles of the pair
      for (int t = 0; t < 2; ++t)
        tma_load_4d_pair(sbase + C::kOffKB + t * 16384, &p.tm_k, kv_bar, 64 * (int)crank, kh, 256 * rank + 128 * t, b,
                         keep);
      bool ok = true;
      int fill = 0, rows_issued = 0;
      for (int it = 0; it < n_iter && ok; ++it) {
        const int hh = kh * g + it / per_head;
        const int i = i_start + it % per_head;
        const int row0 = i * 128;
        for (int t = 0; t < 2 && ok; ++t, ++fill) {
          const int s = C::slot(fill);
          ok = mbar_wait(bar(C::kBarEmpty0 + s), C::phase(fill) ^ 1, wctx, kBSiteEmpty);
          if (!ok) break;
          if (crank == 0) mbar_arrive_expect_tx(bar(C::kBarFull0 + s), 2 * C::kTile);
          const uint32_t fb = mapa_shared(bar(C::kBarFull0 + s), 0);
          const uint32_t dst = sbase + C::kOffRing + s * C::kTile;
          const CUtensorMap *m128 = t == 0 ? &p.tm_q : &p.tm_do;
          const CUtensorMap *m64 = t == 0 ? &p.tm_q64 : &p.tm_do64;
          tma_load_4d_pair(dst, m128, fb, 64 * (int)crank, hh, row0, b, keep);
          for (int bx = 0; bx < 2; ++bx)
            tma_load_4d_pair(dst + C::kOffRowHalves + bx * C::kHalfBytes, m64, fb, bx * 64, hh, row0 + 64 * (int)crank,
                             b, keep);
        }
        if (!ok) break;
        const int rs = it % C::kRowStages;
        ok = mbar_wait(bar(C::kBarRowEmpty0 + rs), ((it / C::kRowStages) & 1) ^ 1, wctx, kBSiteEmpty);
        if (!ok) break;
        const uint32_t rb = bar(C::kBarRowFull0 + rs);
        mbar_arrive_expect_tx(rb, 1024);
        const size_t roff = ((size_t)b * p.H + hh) * Npad + (size_t)i * 128;
        const uint32_t rdst = sbase + C::kOffRows + 1024 * rs;
        bulk_load(rdst, p.lse2 + roff, 512, rb);
        bulk_load(rdst + 512, p.delta + roff, 512, rb);
        ++rows_issued;
      }
      const uint64_t t0 = global_timer_ns();
      if (crank == 0) {
        const int nq = (fill + 1) / 2, nd = fill / 2;
        for (int i = max(0, nq - C::kQSlots); i < nq; ++i)
          while (!mbar_test(bar(C::kBarFull0 + C::slot(2 * i)), C::phase(2 * i)) &&
                 global_timer_ns() - t0 < kWaitLimitNs) {}
        for (int i = max(0, nd - C::kDoSlots); i < nd; ++i)
          while (!mbar_test(bar(C::kBarFull0 + C::slot(2 * i + 1)), C::phase(2 * i + 1)) &&
                 global_timer_ns() - t0 < kWaitLimitNs) {}
        while (!mbar_test(bar(C::kBarKV), 0) && global_timer_ns() - t0 < kWaitLimitNs) {}
      }
      for (int f = max(0, rows_issued - C::kRowStages); f < rows_issued; ++f)
        while (!mbar_test(bar(C::kBarRowFull0 + f % C::kRowStages), (f / C::kRowStages) & 1) &&
               global_timer_ns() - t0 < kWaitLimitNs) {}
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == C::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, C::kTmemCols);
  }
}

// dQ = bf16(scale * dQacc), 8 elements per thread.
__global__ void __launch_bounds__(256) bwd_post_kernel(const float *__restrict__ acc, __nv_bfloat16 *__restrict__ dq,
                                                       long long n8, float scale) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += stride) {
    const float4 a = reinterpret_cast<const float4 *>(acc)[2 * i];
    const float4 c = reinterpret_cast<const float4 *>(acc)[2 * i + 1];
    reinterpret_cast<uint4 *>(dq)[i] = make_uint4(pack_bf16x2(a.x * scale, a.y * scale), pack_bf16x2(a.z * scale, a.w * scale),
                                                  pack_bf16x2(c.x * scale, c.y * scale), pack_bf16x2(c.z * scale, c.w * scale));
  }
}

// Query-row elementwise work of the dQ kernels over all key tiles: one thread
// per query row (TMEM lane), warpgroup wg owns key columns [64 wg, 64 wg + 64).
//   P  = 2^(S c - LSE2), masked -> registers (fp32)
//   dS = P (dP - D)             -> TMEM over dP (bf16, dQ's A operand)
// PAIR: the kernel runs as a CTA pair whose rank-0 CTA issues the MMAs; the S
// and dS signals go to that CTA's barriers.
// gj0: iterations the CTA ran before this work unit (barrier phases and dP
// buffers count across units).
template <class C, bool CAUSAL, bool PAIR = false>
__device__ __forceinline__ bool dq_rows(const BwdParams &p, uint32_t bar0, uint32_t tmem, const WaitCtx &wctx,
                                        int warp, int nb, int q_row, float lse2, float dlt, int L, int gj0 = 0) {
  auto bar = [&](int i) { return bar0 + 8u * i; };
  auto signal_mma = [&](int i) {  // the MMA-issuing CTA's barrier i
    if (PAIR) mbar_arrive_warp_cluster(mapa_shared(bar(i), 0));
    else mbar_arrive_warp(bar(i));
  };
  constexpr int KW = 128 / C::kNumWG;  // key columns per warpgroup
  constexpr int NC = KW / 32;
  const int wg = warp >> 2;
  const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
  const uint32_t s_tm = tmem + lane_off + C::kColS + KW * wg;
  const uint32_t dp_tm0 = tmem + lane_off + C::kColDP + KW * wg;  // dP columns of this warpgroup (buffer 0)
  bool ok = true;
  for (int j = 0; j < nb && ok; ++j) {
    const unsigned gj = (unsigned)(gj0 + j);  // iteration count over the CTA's units
    const unsigned db = gj % C::kDPBufs;      // dP buffer of this key tile
    const uint32_t dp_tm = dp_tm0 + 128u * db;
    const uint32_t ds_tm = dp_tm;  // dS (bf16) over the first KW / 2 of this warpgroup's dP columns
    ok = mbar_wait_warp(bar(C::kBarS), gj & 1u, wctx, kBSiteS);
    if (!ok) break;
    if (threadIdx.x == 0) FA_TRACE_EV(1, j, 0);
    tc_fence_after();
    uint32_t sv[NC][32];
#pragma unroll
    for (int c = 0; c < NC; ++c) tmem_ld_32x32b_x32(s_tm + 32 * c, sv[c]);
    tmem_wait_ld(sv[0]);
#pragma unroll
    for (int c = 1; c < NC; ++c) reg_tie(sv[c]);
    tc_fence_before();
    signal_mma(C::kBarSFree);  // S is in registers: S_{j+1} may overwrite it
    const int kvc0 = j * 128 + KW * wg;                           // first key column of this warpgroup
    const int lim = (CAUSAL ? min(q_row, L - 1) : L - 1) - kvc0;  // last visible column offset
    float pe[KW];
#pragma unroll
    for (int c = 0; c < KW; c += 2) {
      float x0, x1;
      ffma2(x0, x1, __uint_as_float(sv[c >> 5][c & 31]), __uint_as_float(sv[c >> 5][(c & 31) + 1]), p.scale_log2,
            p.scale_log2, -lse2, -lse2);
      pe[c] = ex2_mufu(x0);
      pe[c + 1] = ex2_mufu(x1);
    }
    if (lim < KW - 1) {
#pragma unroll
      for (int c = 0; c < KW; ++c)
        if (c > lim) pe[c] = 0.f;
    }
    ok = mbar_wait_warp(bar(C::kBarDP + db), (gj / C::kDPBufs) & 1u, wctx, kBSiteDP);
    if (!ok) break;
    if (threadIdx.x == 0) FA_TRACE_EV(1, j, 1);
    tc_fence_after();
    uint32_t dpv[NC][32];
#pragma unroll
    for (int c = 0; c < NC; ++c) tmem_ld_32x32b_x32(dp_tm + 32 * c, dpv[c]);
    tmem_wait_ld(dpv[0]);
#pragma unroll
    for (int c = 1; c < NC; ++c) reg_tie(dpv[c]);
    uint32_t w[KW / 2];
#pragma unroll
    for (int c = 0; c < KW; c += 2) {
      float t0, t1, d0, d1;
      fadd2(t0, t1, __uint_as_float(dpv[c >> 5][c & 31]), __uint_as_float(dpv[c >> 5][(c & 31) + 1]), -dlt, -dlt);
      fmul2(d0, d1, pe[c], pe[c + 1], t0, t1);
      w[c >> 1] = pack_bf16x2(d0, d1);
    }
    if constexpr (KW == 64)
      tmem_st_32x32b_x32(ds_tm, *reinterpret_cast<const uint32_t(*)[32]>(&w[0]));
    else
      tmem_st_32x32b_x16(ds_tm, *reinterpret_cast<const uint32_t(*)[16]>(&w[0]));
    tmem_wait_st();
    tc_fence_before();
    if (!(FA_STALL(3) && gj == 0)) signal_mma(C::kBarDS + db);
    if (threadIdx.x == 0) FA_TRACE_EV(1, j, 2);
  }
  return ok;
}

// ================================================================== dQ
template <int D, bool PERSIST = false>
struct DqCfg {
  static constexpr int kTile = 128 * D * 2;
  // Persistent CTAs with a stage of their own for the dQ epilogue (the ring
  // already holds the next unit's tiles) give up one ring slot for it.
  static constexpr bool kOwnStage = PERSIST && FA_DQ_PERSIST_STAGE;
  static constexpr int kStages = ((D == 64) ? 14 : 7) - (kOwnStage ? 1 : 0);  // ring slots of one tile
  // K and V have rings of their own (Q is the K ring's first item, dO the V
  // ring's): a K slot is released when dQ_j completes, a V slot when dP_j does,
  // so neither load waits on the other's late release.
  static constexpr int kKSlots = (4 * kStages + 6) / 7;  // 7 -> 4, 14 -> 8, 6 -> 4, 13 -> 8
  static constexpr int kVSlots = kStages - kKSlots;
  // a unit's fills: 0 = Q, 1 = dO, 2 + 2 j = K_j, 3 + 2 j = V_j (counted on over
  // the CTA's units, from 0: unsigned arithmetic)
  __device__ static int slot(int fill) {
    const unsigned m = (unsigned)fill >> 1;
    return (int)((fill & 1) ? kKSlots + m % kVSlots : m % kKSlots);
  }
  __device__ static uint32_t phase(int fill) {
    const unsigned m = (unsigned)fill >> 1;
    return ((fill & 1) ? m / kVSlots : m / kKSlots) & 1u;
  }
  // PERSIST: at most one CTA per SM, each running work units blockIdx.x,
  // blockIdx.x + gridDim.x, ...; the epilogue then writes dQ rows straight to
  // global memory (the ring already holds the next unit's tiles).
  static constexpr bool kPersist = PERSIST;
  // Elementwise warpgroups: thread = query row, a warpgroup per 128 / kNumWG
  // key columns (four at head dim 64 measured 3-4 % slower than two, as for
  // the dK/dV kernel).
  static constexpr int kNumWG = 2;
  static constexpr int kThreads = 32 * (4 * kNumWG + 2);
  static constexpr int kMmaWarp = 4 * kNumWG, kLoadWarp = 4 * kNumWG + 1;
  // TMEM: S (fp32), dP (fp32; dS bf16 over it once read), dQ (fp32), and the
  // CTA's Q and dO tiles (bf16, two per column) as A operands of the S and dP MMAs.
  // At head dim 64 dP has two buffers, so dP_{j+1} can be issued before dS_j
  // is ready (it overwrites dS_{j-1}, which dQ_{j-1} read earlier in issue order).
  static constexpr int kDPBufs = (D == 64) ? 2 : 1;
  static constexpr int kColS = 0, kColDP = 128, kColDQ = 128 + 128 * kDPBufs, kColQ = kColDQ + D, kColDO = kColQ + D / 2;
  static constexpr int kTmemCols = 512;
  static_assert(kColDO + D / 2 <= kTmemCols, "TMEM budget");
  static constexpr int kOffRing = 0;
  // dQ epilogue staging: a region of its own (kOwnStage), else ring slot 0, drained by then
  static constexpr int kOffStage = kOwnStage ? kOffRing + kStages * kTile : 0;
  static constexpr int kOffBar = kOffRing + (kStages + (kOwnStage ? 1 : 0)) * kTile;
  enum { kBarQdo, kBarFull0, kBarEmpty0 = kBarFull0 + kStages, kBarS = kBarEmpty0 + kStages, kBarSFree, kBarDP,
         kBarDS = kBarDP + kDPBufs, kBarFinal = kBarDS + kDPBufs, kBarDrain, kNumBars };  // DP, DS: one per dP buffer
  static constexpr int kOffMisc = kOffBar + 8 * kNumBars;
  static constexpr int kSmemBytes = kOffMisc + 16;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// One work unit of the one-CTA dQ kernel: query tile it_q of one (batch, head).
struct DqUnit {
  SeqSpan sq;
  int b, h, kh, q0, nb;
  bool skip;  // packed batch: the tile lies past its sequence, no rows to produce
};

template <bool CAUSAL, bool VARLEN>
__device__ __forceinline__ DqUnit dq_unit(const BwdParams &p, int u) {
  DqUnit w;
  const int n_q = (p.N + 127) / 128;
  int rank, head;
  work_order(u, n_q, p.B * p.H, p.sched_chunk, rank, head);
  const int it_q = CAUSAL ? n_q - 1 - rank : rank;  // causal: the longest query rows first
  w.h = head % p.H;
  w.b = head / p.H;
  w.kh = w.h / (p.H / p.Hkv);
  w.q0 = it_q * 128;
  w.sq = VARLEN ? seq_span(p.cu_seqlens, w.b, p.N, p.total) : SeqSpan{0, p.N, w.b};
  w.skip = VARLEN && w.q0 >= w.sq.len;
  w.nb = CAUSAL ? it_q + 1 : (w.sq.len + 127) / 128;  // key tiles this query tile sees
  return w;
}

// The CTA runs work units blockIdx.x, blockIdx.x + gridDim.x, ... (PERSIST: at
// most one CTA per SM; else one unit per CTA).  A unit's ring fills are Q, dO,
// then K_j, V_j for its key tiles: the producer issues the next unit's Q and
// dO right after this unit's last K and V.  The elementwise warps copy them
// into TMEM after this unit's epilogue has waited for its last MMA, so the S
// and dP MMAs that read the previous Q and dO are done.  Every ring, dP buffer
// and barrier phase counts over the CTA's units.
template <int D, bool CAUSAL, bool VARLEN, bool PERSIST>
__global__ void __launch_bounds__(DqCfg<D, PERSIST>::kThreads, 1) bwd_dq_kernel(const __grid_constant__ BwdParams p) {
  using C = DqCfg<D, PERSIST>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  if (!check_align(sbase, p.status)) return;
  const uint32_t bar0 = sbase + C::kOffBar;
  auto bar = [&](int i) { return bar0 + 8u * i; };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 4);
  const WaitCtx wctx{abort_flag, p.status};
  FA_CTA_MARK(1, 1);
  if (threadIdx.x == 0) FA_LIFE(1, 0);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_q = (p.N + 127) / 128;
  const int Npad = n_q * 128;  // row-term arrays are [B, H, Npad]
  const int n_units = n_q * p.B * p.H;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kNumBars; ++i)
      // per elementwise warp: Q and dO come from the first two warpgroups only
      mbar_init(bar(i), i == C::kBarQdo ? 8u
                        : (i == C::kBarSFree || (i >= C::kBarDS && i < C::kBarDS + C::kDPBufs)) ? (uint32_t)(4 * C::kNumWG)
                                                                                                  : 1u);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == C::kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  if (warp == C::kLoadWarp && lane == 0) {
    prefetch_tmap(&p.tm_q);
    prefetch_tmap(&p.tm_do);
    prefetch_tmap(&p.tm_k);
    prefetch_tmap(&p.tm_v);
    prefetch_tmap(&p.tm_dq);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (threadIdx.x == 0) FA_LIFE(1, 1);

  if (warp < 4 * C::kNumWG) {
    // ===================================================== dS = P (dP - D), one warpgroup per 128 / kNumWG key columns
    // After a wait has run out these warps still step through every unit,
    // skipping the work but not the epilogue's named barriers, so the two
    // warpgroups' barriers stay matched (every wait gives up at once then).
    const int wg = warp >> 2;
    const int r = threadIdx.x & 127;  // query row within the tile == TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    bool ok = true;
    int gj = 0, uc = 0;  // iterations and units this CTA has run
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
      const DqUnit w = dq_unit<CAUSAL, VARLEN>(p, u);
      if (w.skip) continue;
      const int q_row = w.q0 + r;
      if (wg < 2 && ok) {
        // Q (warpgroup 0) or dO (warpgroup 1): this unit's ring fill 0 / 1
        // (TMA, zero rows past N); this thread's row, bf16 pairs in memory
        // order, into TMEM as the A operand of the S / dP MMAs.
        const int fill = 2 * uc + 2 * gj + wg;
        uint32_t row[D / 2];
        const bool got = mbar_wait_warp(bar(C::kBarFull0 + C::slot(fill)), C::phase(fill), wctx, kBSiteQ);
        const uint8_t *tile = smem + C::kOffRing + C::slot(fill) * C::kTile;
#pragma unroll
        for (int v = 0; v < D / 8; ++v) {
          uint4 x = make_uint4(0u, 0u, 0u, 0u);
          if (got) x = *reinterpret_cast<const uint4 *>(tile + (v >> 3) * 16384 + r * 128 + (((v & 7) ^ (r & 7)) << 4));
          row[4 * v] = x.x;
          row[4 * v + 1] = x.y;
          row[4 * v + 2] = x.z;
          row[4 * v + 3] = x.w;
        }
        const uint32_t dst = tmem + lane_off + (wg == 0 ? C::kColQ : C::kColDO);
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          uint32_t (&part)[32] = *reinterpret_cast<uint32_t(*)[32]>(&row[32 * c]);
          tmem_st_32x32b_x32(dst + 32 * c, part);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive_warp(bar(C::kBarQdo));
        if (threadIdx.x == 0) FA_LIFE(1, 2);
      }
      const size_t rw = ((size_t)w.b * p.H + w.h) * Npad + q_row;
      const float lse2 = p.lse2[rw];  // +inf on padded rows: P = 0
      const float dlt = p.delta[rw];
      if (ok) ok = dq_rows<C, CAUSAL>(p, bar0, tmem, wctx, warp, w.nb, q_row, lse2, dlt, w.sq.len, gj);
      gj += w.nb;
      // ---- epilogue (warpgroups 0 and 1, half the head dim each): dQ * scale -> bf16 -> global memory
      if (wg < 2) {
        if (ok) ok = mbar_wait_warp(bar(C::kBarFinal), uc & 1, wctx, kBSiteFinal);
        if (threadIdx.x == 0) FA_LIFE(1, 4);
        tc_fence_after();
        // straight from TMEM, a query row per thread: persistent CTAs without a
        // stage (the ring already holds the next unit's tiles), or the next
        // sequence's rows follow
        const bool direct = (C::kPersist && !C::kOwnStage) || (VARLEN && w.q0 + 128 > w.sq.len);
        const size_t row0 = VARLEN ? (size_t)w.sq.start : (size_t)w.b * p.N;  // the sequence's first row
        if (C::kOwnStage) {  // every thread of both warpgroups, whatever ok: the previous store has read the stage
          if (threadIdx.x == 0) bulk_wait_read_all();
          named_bar_sync(1, 256);
        }
        if (ok && direct)
          acc_to_global<D / 2>(tmem + lane_off + C::kColDQ,
                               static_cast<__nv_bfloat16 *>(p.dq) + ((row0 + q_row) * p.H + w.h) * D, wg * (D / 2),
                               p.scale, q_row < w.sq.len);
        if (!C::kPersist || C::kOwnStage) {
          uint8_t *stage = smem + C::kOffStage;
          if (ok && !direct) acc_to_smem<D / 2>(tmem + lane_off + C::kColDQ, stage, r, wg * (D / 2), p.scale);
          fence_proxy_async_smem();
        }
        tc_fence_before();  // the accumulator reads precede the next unit's first dQ MMA
        if (!C::kPersist || C::kOwnStage) {
          named_bar_sync(1, 256);
          if (threadIdx.x == 0 && ok && !direct) {
            for (int bx = 0; bx < D / 64; ++bx)
              tma_store_4d(&p.tm_dq, sbase + C::kOffStage + bx * 16384, bx * 64, w.h, w.sq.start + w.q0, w.sq.bc);
            bulk_commit();
            if (!C::kOwnStage) bulk_wait_read_all();  // persistent: deferred to the next epilogue
            if (threadIdx.x == 0) FA_LIFE(1, 5);
          }
        }
      }
      ++uc;
      if (!C::kPersist) break;  // one unit per CTA
    }
    if (C::kOwnStage && threadIdx.x == 0) bulk_wait_read_all();  // the last unit's store
  } else if (warp == C::kMmaWarp) {
    // ===================================================== MMA issue
    // Order: S_0 dP_0 | [S read] S_{j+1} [dS_j] dQ_j dP_{j+1} | ...
    // S_{j+1} overwrites S_j once the elementwise warps hold it in registers;
    // dS_j (bf16, over the dP columns) is read by dQ_j, which precedes dP_{j+1}
    // (the tensor pipe runs one thread's MMAs in order).  With two dP buffers
    // the order is S_{j+1} dP_{j+1} [dS_j] dQ_j: dP_{j+1} goes to the buffer of
    // dS_{j-1}, whose dQ_{j-1} was issued before it.  Iterations count over
    // the CTA's units; a unit's first S and dP follow its Q and dO in TMEM,
    // copied after the previous unit's epilogue read its dQ.  The whole warp
    // runs the loop and waits; the elected lane issues.
    {
      constexpr uint32_t id_s = make_idesc_bf16(128, 128, false, false);  // S, dP (A in TMEM, B K-major)
      constexpr uint32_t id_dq = make_idesc_bf16(128, D, false, true);    // dQ (A = dS in TMEM, B = K MN-major)
      const uint64_t ring_d = make_sdesc_sw128(sbase + C::kOffRing, 0, 1024);
      const uint64_t ring_mn = make_sdesc_sw128(sbase + C::kOffRing, 16384, 1024);
      auto kmaj = [](int kk) { return (uint64_t)((((kk >> 2) * 16384 + (kk & 3) * 32)) >> 4); };
      auto slot_off = [](int fill) { return (uint64_t)((C::slot(fill) * C::kTile) >> 4); };
      auto par = [](int fill) { return C::phase(fill); };
      // dS of warpgroup w (its KW key columns, bf16 pairs) starts at column KW w
      constexpr int KW = 128 / C::kNumWG, KPW = KW / 16;
      auto a_col = [](int kk) { return (uint32_t)(KW * (kk / KPW) + 8 * (kk % KPW)); };
      auto issue_s = [&](int fk_) {  // S = Q K^T   (K from ring fill fk_)
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ts(tmem + C::kColS, tmem + C::kColQ + 8u * kk, ring_d + slot_off(fk_) + kmaj(kk), id_s, kk > 0);
          tc_commit(bar(C::kBarS));
        }
        __syncwarp();
      };
      auto issue_dp = [&](unsigned gjj, int fv_) {  // dP = dO V^T into buffer gjj % kDPBufs   (V from fill fv_)
        const unsigned db = gjj % C::kDPBufs;
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ts(tmem + C::kColDP + 128u * db, tmem + C::kColDO + 8u * kk, ring_d + slot_off(fv_) + kmaj(kk),
                   id_s, kk > 0);
          tc_commit(bar(C::kBarDP + db));
          tc_commit(bar(C::kBarEmpty0 + C::slot(fv_)));  // V consumed
        }
        __syncwarp();
      };
      bool ok = true;
      int gj = 0, uc = 0;
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
        const DqUnit w = dq_unit<CAUSAL, VARLEN>(p, u);
        if (w.skip) continue;
        const int nb = w.nb;
        const int fb = 2 * uc + 2 * gj;  // this unit's first ring fill (Q; dO at fb + 1)
        // K_j is fill fb + 2 + 2 j, V_j fill fb + 3 + 2 j
        auto fk = [&](int j) { return fb + 2 + 2 * j; };
        auto fv = [&](int j) { return fb + 3 + 2 * j; };
        ok = mbar_wait_warp(bar(C::kBarQdo), uc & 1, wctx, kBSiteQ);
        // Q and dO are in TMEM: their ring slots may take later fills
        if (ok && elect_one()) {
          mbar_arrive(bar(C::kBarEmpty0 + C::slot(fb)));
          mbar_arrive(bar(C::kBarEmpty0 + C::slot(fb + 1)));
        }
        __syncwarp();
        if (ok) ok = mbar_wait_warp(bar(C::kBarFull0 + C::slot(fk(0))), par(fk(0)), wctx, kBSiteFull);
        if (ok) {
          tc_fence_after();
          issue_s(fk(0));
          if (uc == 0 && lane == 0) FA_LIFE(1, 3);
          ok = mbar_wait_warp(bar(C::kBarFull0 + C::slot(fv(0))), par(fv(0)), wctx, kBSiteFull);
        }
        if (ok) {
          tc_fence_after();
          issue_dp((unsigned)gj, fv(0));
        }
        for (int j = 0; j < nb && ok; ++j) {
          const unsigned gjj = (unsigned)(gj + j);
          FA_TRACE_EV(1, j, 8);
          const bool more = j + 1 < nb;
          if (more) {
            ok = mbar_wait_warp(bar(C::kBarSFree), gjj & 1u, wctx, kBSiteS);
            FA_TRACE_EV(1, j, 12);
            if (ok) ok = mbar_wait_warp(bar(C::kBarFull0 + C::slot(fk(j + 1))), par(fk(j + 1)), wctx, kBSiteFull);
            if (!ok) break;
            FA_TRACE_EV(1, j, 13);
            tc_fence_after();
            issue_s(fk(j + 1));
            if (C::kDPBufs == 2) {
              ok = mbar_wait_warp(bar(C::kBarFull0 + C::slot(fv(j + 1))), par(fv(j + 1)), wctx, kBSiteFull);
              if (!ok) break;
              tc_fence_after();
              issue_dp(gjj + 1, fv(j + 1));
            }
          }
          const unsigned db = gjj % C::kDPBufs;
          ok = mbar_wait_warp(bar(C::kBarDS + db), (gjj / C::kDPBufs) & 1u, wctx, kBSiteDS);
          if (!ok) break;
          FA_TRACE_EV(1, j, 9);
          tc_fence_after();
          // dQ += dS_j K_j
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ts(tmem + C::kColDQ, tmem + C::kColDP + 128u * db + a_col(kk),
                     ring_mn + slot_off(fk(j)) + (uint64_t)(kk * 128), id_dq, (j > 0 || kk > 0));
            tc_commit(bar(C::kBarEmpty0 + C::slot(fk(j))));  // K_j consumed
          }
          __syncwarp();
          if (C::kDPBufs == 1 && more) {
            ok = mbar_wait_warp(bar(C::kBarFull0 + C::slot(fv(j + 1))), par(fv(j + 1)), wctx, kBSiteFull);
            if (!ok) break;
            tc_fence_after();
            issue_dp(gjj + 1, fv(j + 1));
          }
          FA_TRACE_EV(1, j, 10);
        }
        if (elect_one()) tc_commit(bar(C::kBarFinal));  // the unit's dQ is complete
        __syncwarp();
        gj += nb;
        ++uc;
        if (!C::kPersist) break;
      }
      if (elect_one()) tc_commit(bar(C::kBarDrain));
      __syncwarp();
      if (!mbar_wait_warp(bar(C::kBarDrain), 0, wctx, kBSiteDrain) && *abort_flag) {
        const uint64_t t0 = global_timer_ns();
        while (!mbar_test(bar(C::kBarDrain), 0) && global_timer_ns() - t0 < kWaitLimitNs) {}
      }
    }
  } else {
    // ===================================================== TMA producer: per unit Q, dO, then K_j and V_j in turn, each into its own ring
    if (lane == 0) {
      const uint64_t keep = policy_evict_last();  // K, V are re-read by every query tile
      const uint64_t once = policy_evict_first();  // this CTA's Q and dO rows are read once
      bool ok = true;
      int fill = 0;
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
        const DqUnit w = dq_unit<CAUSAL, VARLEN>(p, u);
        if (w.skip) continue;
        // Q and dO of this unit (the MMA warp releases their slots once the
        // elementwise warps have copied them into TMEM), then K_j, V_j
        for (int t = 0; t < 2 + 2 * w.nb && ok; ++t, ++fill) {
          const int s = C::slot(fill);
          ok = mbar_wait(bar(C::kBarEmpty0 + s), C::phase(fill) ^ 1, wctx, kBSiteEmpty);
          if (!ok) break;
          mbar_arrive_expect_tx(bar(C::kBarFull0 + s), C::kTile);
          const uint32_t dst = sbase + C::kOffRing + s * C::kTile;
          if (t < 2) {
            for (int bx = 0; bx < D / 64; ++bx)
              tma_load_4d_hint(dst + bx * 16384, t ? &p.tm_do : &p.tm_q, bar(C::kBarFull0 + s), bx * 64, w.h,
                               w.sq.start + w.q0, w.sq.bc, once);
          } else {
            const int j = (t - 2) >> 1;
            const CUtensorMap *map = (t & 1) ? &p.tm_v : &p.tm_k;
            for (int bx = 0; bx < D / 64; ++bx)
              tma_load_4d_hint(dst + bx * 16384, map, bar(C::kBarFull0 + s), bx * 64, w.kh, w.sq.start + j * 128,
                               w.sq.bc, keep);
          }
        }
        if (!C::kPersist) break;
      }
      const uint64_t t0 = global_timer_ns();
      // the last issued fill of each slot: the last kKSlots even fills, the last kVSlots odd ones
      const int ne = (fill + 1) / 2, no = fill / 2;
      for (int m = max(0, ne - C::kKSlots); m < ne; ++m)
        while (!mbar_test(bar(C::kBarFull0 + C::slot(2 * m)), C::phase(2 * m)) && global_timer_ns() - t0 < kWaitLimitNs) {}
      for (int m = max(0, no - C::kVSlots); m < no; ++m)
        while (!mbar_test(bar(C::kBarFull0 + C::slot(2 * m + 1)), C::phase(2 * m + 1)) &&
               global_timer_ns() - t0 < kWaitLimitNs) {}
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  FA_CTA_MARK(1, 2);
  if (threadIdx.x == 0) FA_LIFE(1, 6);
}

// ================================================================== dQ on CTA pairs (head dim 128)
// The query-stationary counterpart of bwd_dkdv_pair_kernel: a cluster of two
// CTAs shares one 256-row query tile, CTA c owning query rows 128c..128c+127
// (its Q and dO in its own TMEM as the A operands, its S, dP and dQ), and the
// pair walks the key tiles together.  The rank-0 CTA issues every MMA for both:
//   S = Q K_j^T, dP = dO V_j^T   M = 256 queries, N = 128 keys: CTA c supplies
//                                key rows 64c..64c+63 of K_j (V_j), all head-dim columns
//   dQ += dS K_j                 M = 256 queries, N = 128 = d: CTA c supplies
//                                head-dim columns 64c..64c+63 of all 128 rows of K_j
// so each SM's MMAs read half of every B operand and each CTA loads 48 KB per
// key tile instead of 64.  Q and dO arrive by TMA into the first slot of each
// ring (local barriers), the elementwise warps copy them into TMEM and signal
// the rank-0 CTA, which then frees those slots in both CTAs.
struct DqPairCfg : DqCfg<128> {
  static constexpr int kHalfBytes = 64 * 128;  // 64 rows x 64 columns of bf16
  static constexpr int kOffRowHalves = 16384;  // in a slot: K's head-dim half, then the 64-row halves
};

template <bool CAUSAL, bool VARLEN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(320, 1) bwd_dq_pair_kernel(const __grid_constant__ BwdParams p) {
  using C = DqPairCfg;
  constexpr int D = 128;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  if (!check_align(sbase, p.status)) return;  // same layout in both CTAs: both return
  const uint32_t bar0 = sbase + C::kOffBar;
  auto bar = [&](int i) { return bar0 + 8u * i; };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 4);
  const WaitCtx wctx{abort_flag, p.status};
  FA_CTA_MARK(1, 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t crank = cluster_ctarank();
  const int n_q = (p.N + 127) / 128;
  const int n_pairs = (n_q + 1) / 2;
  int rank, head;
  work_order((int)(blockIdx.x >> 1), n_pairs, p.B * p.H, p.sched_chunk, rank, head);
  const int pq = CAUSAL ? n_pairs - 1 - rank : rank;  // causal: the longest query rows first
  const int it_q = 2 * pq + (int)crank;               // this CTA's query tile
  const int h = head % p.H, b = head / p.H;
  const int kh = h / (p.H / p.Hkv);
  const int Npad = n_q * 128;  // row-term arrays are [B, H, Npad]
  const int q0 = it_q * 128;
  const SeqSpan sq = VARLEN ? seq_span(p.cu_seqlens, b, p.N, p.total) : SeqSpan{0, p.N, b};
  const int L = sq.len;
  if (VARLEN && 256 * pq >= L) return;  // the pair's tile lies past its sequence (both CTAs return)
  const int n_kv = (L + 127) / 128;
  const int nb = CAUSAL ? min(2 * pq + 2, n_kv) : n_kv;  // key tiles the pair's second query tile sees

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kNumBars; ++i)
      mbar_init(bar(i), (i == C::kBarQdo || i == C::kBarSFree || i == C::kBarDS) ? 16u : 1u);  // warps of both
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == C::kMmaWarp) {
    tmem_alloc_pair(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish_pair();
  }
  if (warp == C::kLoadWarp && lane == 0) {
    prefetch_tmap(&p.tm_q);
    prefetch_tmap(&p.tm_do);
    prefetch_tmap(&p.tm_k);
    prefetch_tmap(&p.tm_k64);
    prefetch_tmap(&p.tm_v64);
    prefetch_tmap(&p.tm_dq);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 8) {
    // ===================================================== dS = P (dP - D) for this CTA's query rows
    const int wg = warp >> 2;
    const int r = threadIdx.x & 127;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const int q_row = q0 + r;
    {
      // Q (warpgroup 0) or dO (warpgroup 1) of this CTA into its TMEM (A operands of S and dP)
      uint32_t row[D / 2];
      const bool got = mbar_wait_warp(bar(C::kBarFull0 + C::slot(wg)), 0, wctx, kBSiteQ);
      const uint8_t *tile = smem + C::kOffRing + C::slot(wg) * C::kTile;
#pragma unroll
      for (int v = 0; v < D / 8; ++v) {
        uint4 x = make_uint4(0u, 0u, 0u, 0u);
        if (got) x = *reinterpret_cast<const uint4 *>(tile + (v >> 3) * 16384 + r * 128 + (((v & 7) ^ (r & 7)) << 4));
        row[4 * v] = x.x;
        row[4 * v + 1] = x.y;
        row[4 * v + 2] = x.z;
        row[4 * v + 3] = x.w;
      }
      const uint32_t dst = tmem + lane_off + (wg == 0 ? C::kColQ : C::kColDO);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        uint32_t (&part)[32] = *reinterpret_cast<uint32_t(*)[32]>(&row[32 * c]);
        tmem_st_32x32b_x32(dst + 32 * c, part);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive_warp_cluster(mapa_shared(bar(C::kBarQdo), 0));
    }
    // rows past the row-term arrays (the pair's second tile past the last one): P = 0
    const bool in_rows = q_row < Npad;
    const size_t rw = ((size_t)b * p.H + h) * Npad + (in_rows ? q_row : 0);
    const float lse2 = in_rows ? p.lse2[rw] : INFINITY;
    const float dlt = in_rows ? p.delta[rw] : 0.f;
    bool ok = dq_rows<C, CAUSAL, true>(p, bar0, tmem, wctx, warp, nb, q_row, lse2, dlt, L);
    // ---- epilogue: dQ * scale -> bf16 -> shared staging -> TMA store
    if (ok) ok = mbar_wait_warp(bar(C::kBarFinal), 0, wctx, kBSiteFinal);
    tc_fence_after();
    uint8_t *stage = smem + C::kOffStage;
    const bool has_rows = q0 < L;
    const bool direct = VARLEN && q0 + 128 > L;
    if (ok && has_rows && direct)
      acc_to_global<D / 2>(tmem + lane_off + C::kColDQ,
                           static_cast<__nv_bfloat16 *>(p.dq) + ((size_t)(sq.start + q_row) * p.H + h) * D, wg * (D / 2),
                           p.scale, q_row < L);
    else if (ok && has_rows)
      acc_to_smem<D / 2>(tmem + lane_off + C::kColDQ, stage, r, wg * (D / 2), p.scale);
    fence_proxy_async_smem();
    named_bar_sync(1, 256);
    if (threadIdx.x == 0 && ok && has_rows && !direct) {
      for (int bx = 0; bx < D / 64; ++bx)
        tma_store_4d(&p.tm_dq, sbase + C::kOffStage + bx * 16384, bx * 64, h, sq.start + q0, sq.bc);
      bulk_commit();
      bulk_wait_read_all();
    }
  } else if (warp == C::kMmaWarp) {
    // ===================================================== MMA issue (rank-0 CTA, for both)
    // Order: S_0 dP_0 | [S read] S_{j+1} [dS_j] dQ_j dP_{j+1} | ...   (as in bwd_dq_kernel)
    if (crank == 0) {
      constexpr uint32_t id_s = make_idesc_bf16(256, 128, false, false);  // S, dP (A in TMEM, B K-major)
      constexpr uint32_t id_dq = make_idesc_bf16(256, D, false, true);    // dQ (A = dS in TMEM, B = K MN-major)
      const uint64_t ring_d = make_sdesc_sw128(sbase + C::kOffRing + C::kOffRowHalves, 0, 1024);  // row halves
      const uint64_t ring_mn = make_sdesc_sw128(sbase + C::kOffRing, 16384, 1024);                 // head-dim half
      auto kmaj_half = [](int kk) { return (uint64_t)(((kk >> 2) * C::kHalfBytes + (kk & 3) * 32) >> 4); };
      auto slot_off = [](int fill) { return (uint64_t)((C::slot(fill) * C::kTile) >> 4); };
      auto par = [](int fill) { return C::phase(fill); };
      constexpr int KW = 128 / C::kNumWG, KPW = KW / 16;
      auto a_col = [](int kk) { return (uint32_t)(KW * (kk / KPW) + 8 * (kk % KPW)); };
      auto fk = [](int j) { return 2 + 2 * j; };
      auto fv = [](int j) { return 3 + 2 * j; };
      auto issue_s = [&](int j) {  // S_j = Q K_j^T
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ts_pair(tmem + C::kColS, tmem + C::kColQ + 8u * kk, ring_d + slot_off(fk(j)) + kmaj_half(kk), id_s,
                        kk > 0);
          tc_commit_pair(bar(C::kBarS));
        }
        __syncwarp();
      };
      auto issue_dp = [&](int j) {  // dP_j = dO V_j^T
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ts_pair(tmem + C::kColDP, tmem + C::kColDO + 8u * kk, ring_d + slot_off(fv(j)) + kmaj_half(kk), id_s,
                        kk > 0);
          tc_commit_pair(bar(C::kBarDP));
          tc_commit_pair(bar(C::kBarEmpty0 + C::slot(fv(j))));  // V_j consumed
        }
        __syncwarp();
      };
      bool ok = mbar_wait_warp(bar(C::kBarQdo), 0, wctx, kBSiteQ);
      // Q and dO of both CTAs are in TMEM: the first slot of each ring may take K/V fills in both
      if (ok && elect_one()) {
        for (int t = 0; t < 2; ++t) {
          mbar_arrive(bar(C::kBarEmpty0 + C::slot(t)));
          mbar_arrive_cluster(mapa_shared(bar(C::kBarEmpty0 + C::slot(t)), 1));
        }
      }
      __syncwarp();
      if (ok) ok = mbar_wait_warp(bar(C::kBarFull0 + C::slot(fk(0))), par(fk(0)), wctx, kBSiteFull);
      if (ok) {
        tc_fence_after();
        issue_s(0);
        ok = mbar_wait_warp(bar(C::kBarFull0 + C::slot(fv(0))), par(fv(0)), wctx, kBSiteFull);
      }
      if (ok) {
        tc_fence_after();
        issue_dp(0);
      }
      for (int j = 0; j < nb && ok; ++j) {
        const bool more = j + 1 < nb;
        if (more) {
          ok = mbar_wait_warp(bar(C::kBarSFree), j & 1, wctx, kBSiteS);
          if (ok) ok = mbar_wait_warp(bar(C::kBarFull0 + C::slot(fk(j + 1))), par(fk(j + 1)), wctx, kBSiteFull);
          if (!ok) break;
          tc_fence_after();
          issue_s(j + 1);
        }
        ok = mbar_wait_warp(bar(C::kBarDS), j & 1, wctx, kBSiteDS);
        if (!ok) break;
        tc_fence_after();
        if (elect_one()) {  // dQ += dS_j K_j
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts_pair(tmem + C::kColDQ, tmem + C::kColDP + a_col(kk), ring_mn + slot_off(fk(j)) + (uint64_t)(kk * 128),
                        id_dq, (j > 0 || kk > 0));
          tc_commit_pair(bar(C::kBarEmpty0 + C::slot(fk(j))));  // K_j consumed
        }
        __syncwarp();
        if (more) {
          ok = mbar_wait_warp(bar(C::kBarFull0 + C::slot(fv(j + 1))), par(fv(j + 1)), wctx, kBSiteFull);
          if (!ok) break;
          tc_fence_after();
          issue_dp(j + 1);
        }
      }
      if (elect_one()) {
        tc_commit_pair(bar(C::kBarFinal));
        tc_commit_pair(bar(C::kBarDrain));
      }
      __syncwarp();
      if (!mbar_wait_warp(bar(C::kBarDrain), 0, wctx, kBSiteDrain) && *abort_flag) {
        const uint64_t t0 = global_timer_ns();
        while (!mbar_test(bar(C::kBarDrain), 0) && global_timer_ns() - t0 < kWaitLimitNs) {}
      }
    }
  } else {
    // ===================================================== TMA producer: this CTA's Q and dO (local), then its halves of K_j, V_j
    if (lane == 0) {
      const uint64_t keep = policy_evict_last();
      const uint64_t once = policy_evict_first();
      for (int t = 0; t < 2; ++t) {  // fills 0, 1: Q and dO, completed on this CTA's own barriers
        const int st = C::slot(t);
        mbar_arrive_expect_tx(bar(C::kBarFull0 + st), C::kTile);
        for (int bx = 0; bx < D / 64; ++bx)
          tma_load_4d_hint(sbase + C::kOffRing + st * C::kTile + bx * 16384, t ? &p.tm_do : &p.tm_q,
                           bar(C::kBarFull0 + st), bx * 64, h, sq.start + q0, sq.bc, once);
      }
      bool ok = true;
      int fill = 2;
      for (int j = 0; j < nb && ok; ++j) {
        const int row0 = sq.start + j * 128;
        for (int kv = 0; kv < 2 && ok; ++kv, ++fill) {  // kv = 0: K_j (both parts), kv = 1: V_j (row halves)
          const int s = C::slot(fill);
          ok = mbar_wait(bar(C::kBarEmpty0 + s), C::phase(fill) ^ 1, wctx, kBSiteEmpty);
          if (!ok) break;
          if (crank == 0) mbar_arrive_expect_tx(bar(C::kBarFull0 + s), kv ? 2 * C::kHalfBytes * 2 : 2 * C::kTile);
          const uint32_t fb = mapa_shared(bar(C::kBarFull0 + s), 0);
          const uint32_t dst = sbase + C::kOffRing + s * C::kTile;
          if (kv == 0)  // K's head-dim half crank, all 128 rows (MN-major operand of dQ)
            tma_load_4d_pair(dst, &p.tm_k, fb, 64 * (int)crank, kh, row0, sq.bc, keep);
          for (int bx = 0; bx < 2; ++bx)  // this CTA's 64 key rows, both halves (K-major operand of S / dP)
            tma_load_4d_pair(dst + C::kOffRowHalves + bx * C::kHalfBytes, kv ? &p.tm_v64 : &p.tm_k64, fb, bx * 64, kh,
                             row0 + 64 * (int)crank, sq.bc, keep);
        }
      }
      const uint64_t t0 = global_timer_ns();
      if (crank == 0) {  // rank 0's full barriers count both CTAs' copies
        const int nk = (fill + 1) / 2, nv = fill / 2;  // fills issued per ring, Q and dO included
        for (int m = max(0, nk - C::kKSlots); m < nk; ++m)
          while (!mbar_test(bar(C::kBarFull0 + C::slot(2 * m)), C::phase(2 * m)) &&
                 global_timer_ns() - t0 < kWaitLimitNs) {}
        for (int m = max(0, nv - C::kVSlots); m < nv; ++m)
          while (!mbar_test(bar(C::kBarFull0 + C::slot(2 * m + 1)), C::phase(2 * m + 1)) &&
                 global_timer_ns() - t0 < kWaitLimitNs) {}
      } else {  // this CTA's own Q and dO copies
        for (int t = 0; t < 2; ++t)
          while (!mbar_test(bar(C::kBarFull0 + C::slot(t)), 0) && global_timer_ns() - t0 < kWaitLimitNs) {}
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == C::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, C::kTmemCols);
  }
  FA_CTA_MARK(1, 2);
}

// ================================================================== head dim 256
// At d = 256, dV and dK alone would fill the 512 TMEM columns and a K, V, Q, dO
// tile set would not fit in shared memory.  So:
//  * bwd_dkdv256: one CTA per (key tile, half e of the head dim); it produces
//    columns [128 e, 128 e + 128) of dV and dK, recomputing S^T and dP^T in
//    full (TMEM: S^T 128 | dP^T 128 | dV_e 128 | dK_e 128).  K_j and V_j stay in
//    shared memory; Q_i and dO_i stream as 128-column halves through three
//    32 KB slots, the half that is only needed for S^T / dP^T first.
//  * bwd_dq256: one CTA per query tile (TMEM: S 128 | dP 128 | dQ 256); Q_i and
//    dO_i stay in shared memory; V_j then K_j stream as halves through three
//    slots, dP_j issued before S_j so that V_j's slots free early.
template <bool CAUSAL>
struct Dkdv256Cfg {
  static constexpr int D = 256;
  static constexpr int kTile = 128 * D * 2;  // 64 KB
  static constexpr int kHalf = kTile / 2;    // 32 KB: 128 rows x 128 columns
  static constexpr int kSlots = 3;
  static constexpr int kRowStages = 2;
  static constexpr int kNumWG = 2;
  static constexpr int kThreads = 320;
  static constexpr int kMmaWarp = 8;  // warp 9: TMA producer
  static constexpr int kSBufs = 1;  // one S^T buffer (the elementwise rows are shared with the other kernels)
  static constexpr int kColS = 0, kColDP = 128, kColDV = 256, kColDK = 384;
  static constexpr int kTmemCols = 512;
  static constexpr int kOffK = 0, kOffV = kTile, kOffRing = 2 * kTile;
  static constexpr int kOffRows = kOffRing + kSlots * kHalf;
  enum { kBarKV, kBarFull0, kBarEmpty0 = kBarFull0 + kSlots, kBarRowFull0 = kBarEmpty0 + kSlots,
         kBarRowEmpty0 = kBarRowFull0 + kRowStages, kBarS = kBarRowEmpty0 + kRowStages, kBarDP, kBarP, kBarDS,
         kBarFinal, kBarDrain, kNumBars };
  static constexpr int kOffBar = kOffRows + 1024 * kRowStages;
  static constexpr int kOffMisc = kOffBar + 8 * kNumBars;
  static constexpr int kSmemBytes = kOffMisc + 16;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

template <bool CAUSAL, bool VARLEN>
__global__ void __launch_bounds__(320, 1) bwd_dkdv256_kernel(const __grid_constant__ BwdParams p) {
  using C = Dkdv256Cfg<CAUSAL>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  if (!check_align(sbase, p.status)) return;
  const uint32_t bar0 = sbase + C::kOffBar;
  auto bar = [&](int i) { return bar0 + 8u * i; };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 4);
  const WaitCtx wctx{abort_flag, p.status};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  int rank, head;
  work_order((int)blockIdx.x, 2 * ((p.N + 127) / 128), p.B * p.Hkv, p.sched_chunk, rank, head);
  const int jt = rank >> 1;  // key/value tile
  const int e = rank & 1;    // half of the head dim this CTA produces
  const int kh = head % p.Hkv, b = head / p.Hkv;
  const int g = p.H / p.Hkv;
  const SeqSpan sq = VARLEN ? seq_span(p.cu_seqlens, b, p.N, p.total) : SeqSpan{0, p.N, b};
  const int L = sq.len;                      // rows of this sequence
  const int Npad = (p.N + 127) / 128 * 128;  // row-term arrays are [B, H, Npad]
  const int kv0 = jt * 128;
  if (VARLEN && kv0 >= L) return;  // the tile lies past its sequence: no rows to produce
  const int n_q = (L + 127) / 128;
  const int i_start = CAUSAL ? jt : 0;
  const int per_head = n_q - i_start;
  const int n_iter = g * per_head;
  // per iteration four fills: Q half (1-e), Q half e, dO half (1-e), dO half e
  auto fill_of = [&](int it, bool is_do, int half) { return 4 * it + (is_do ? 2 : 0) + (half == e ? 1 : 0); };
  auto slot_of = [](int fill) { return fill % C::kSlots; };

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kNumBars; ++i) {
      const bool all = i == C::kBarP || i == C::kBarDS || (i >= C::kBarRowEmpty0 && i < C::kBarRowEmpty0 + C::kRowStages);
      mbar_init(bar(i), all ? 8u : 1u);  // one arrival per elementwise warp
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == C::kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 8) {
    const int wg = warp >> 2;
    const int r = threadIdx.x & 127;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    bool ok = dkdv_rows<C, CAUSAL>(p, smem, bar0, tmem, wctx, warp, n_iter, i_start, per_head, jt, kv0, L);
    // ---- epilogue: warpgroup 0 stores dV[:, half e], warpgroup 1 dK[:, half e] * scale (ring slots 0, 1)
    if (ok) ok = mbar_wait_warp(bar(C::kBarFinal), 0, wctx, kBSiteFinal);
    tc_fence_after();
    uint8_t *stage = smem + C::kOffRing + wg * C::kHalf;
    const uint32_t acc_tm = tmem + lane_off + (wg == 0 ? C::kColDV : C::kColDK);
    const float mul = wg == 0 ? 1.0f : p.scale;
    const bool direct = VARLEN && kv0 + 128 > L;  // the next sequence's rows follow: write row by row
    if (ok && direct) {
      __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(wg == 0 ? p.dv : p.dk);
      acc_to_global<128>(acc_tm, out + ((size_t)(sq.start + kv0 + r) * p.Hkv + kh) * 256 + 128 * e, 0, mul,
                         kv0 + r < L);
    } else if (ok) {
      acc_to_smem<128>(acc_tm, stage, r, 0, mul);
    }
    fence_proxy_async_smem();
    if (wg == 0) named_bar_sync(1, 128);
    else named_bar_sync(2, 128);
    if (r == 0 && ok && !direct) {
      const CUtensorMap *map = wg == 0 ? &p.tm_dv : &p.tm_dk;
      for (int bx = 0; bx < 2; ++bx)
        tma_store_4d(map, smem_u32(stage) + bx * 16384, 128 * e + bx * 64, kh, sq.start + kv0, sq.bc);
      bulk_commit();
      bulk_wait_read_all();
    }
  } else if (warp == C::kMmaWarp) {
    // ===================================================== MMA issue: S^T, dP^T, [P] dV_e, [dS] dK_e per iteration
    // The whole warp runs the loop and waits; the elected lane issues.
    {
      constexpr uint32_t id_kk = make_idesc_bf16(128, 128, false, false);
      constexpr uint32_t id_out = make_idesc_bf16(128, 128, false, true);  // A in TMEM, B MN-major half tile
      const uint64_t k_d = make_sdesc_sw128(sbase + C::kOffK, 0, 1024);
      const uint64_t v_d = make_sdesc_sw128(sbase + C::kOffV, 0, 1024);
      const uint64_t ring_d = make_sdesc_sw128(sbase + C::kOffRing, 0, 1024);
      const uint64_t ring_mn = make_sdesc_sw128(sbase + C::kOffRing, 16384, 1024);
      auto kmaj = [](int kk) { return (uint64_t)((((kk >> 2) * 16384 + (kk & 3) * 32)) >> 4); };
      auto soff = [&](int fill) { return (uint64_t)((slot_of(fill) * C::kHalf) >> 4); };
      auto full_ok = [&](int fill) {
        return mbar_wait_warp(bar(C::kBarFull0 + slot_of(fill)), (uint32_t)((fill / C::kSlots) & 1), wctx,
                              kBSiteFull);
      };
      auto release = [&](int fill) { tc_commit(bar(C::kBarEmpty0 + slot_of(fill))); };
      auto a_col = [](int kk) { return (uint32_t)(64 * (kk >> 2) + 8 * (kk & 3)); };
      bool ok = mbar_wait_warp(bar(C::kBarKV), 0, wctx, kBSiteKV);
      for (int it = 0; it < n_iter && ok; ++it) {
        // S^T = K Q^T over the full head dim: K steps 0-7 read Q half 0, 8-15 Q half 1
        ok = full_ok(fill_of(it, false, 0)) && full_ok(fill_of(it, false, 1));
        if (!ok) break;
        tc_fence_after();
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < 16; ++kk)
            mma_ss(tmem + C::kColS, k_d + kmaj(kk), ring_d + soff(fill_of(it, false, kk >> 3)) + kmaj(kk & 7), id_kk,
                   kk > 0);
          tc_commit(bar(C::kBarS));
          release(fill_of(it, false, 1 - e));
        }
        __syncwarp();
        // dP^T = V dO^T
        ok = full_ok(fill_of(it, true, 0)) && full_ok(fill_of(it, true, 1));
        if (!ok) break;
        tc_fence_after();
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < 16; ++kk)
            mma_ss(tmem + C::kColDP, v_d + kmaj(kk), ring_d + soff(fill_of(it, true, kk >> 3)) + kmaj(kk & 7), id_kk,
                   kk > 0);
          tc_commit(bar(C::kBarDP));
          release(fill_of(it, true, 1 - e));
        }
        __syncwarp();
        // dV_e += P^T dO[:, half e]
        ok = mbar_wait_warp(bar(C::kBarP), it & 1, wctx, kBSiteP);
        if (!ok) break;
        tc_fence_after();
        const uint64_t do_mn = ring_mn + soff(fill_of(it, true, e));
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts(tmem + C::kColDV, tmem + C::kColS + a_col(kk), do_mn + (uint64_t)(kk * 128), id_out,
                   (it > 0 || kk > 0));
          release(fill_of(it, true, e));
        }
        __syncwarp();
        // dK_e += dS^T Q[:, half e]
        ok = mbar_wait_warp(bar(C::kBarDS), it & 1, wctx, kBSiteDS);
        if (!ok) break;
        tc_fence_after();
        const uint64_t q_mn = ring_mn + soff(fill_of(it, false, e));
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts(tmem + C::kColDK, tmem + C::kColDP + a_col(kk), q_mn + (uint64_t)(kk * 128), id_out,
                   (it > 0 || kk > 0));
          release(fill_of(it, false, e));
        }
        __syncwarp();
      }
      if (elect_one()) {
        tc_commit(bar(C::kBarFinal));
        tc_commit(bar(C::kBarDrain));
      }
      __syncwarp();
      if (!mbar_wait_warp(bar(C::kBarDrain), 0, wctx, kBSiteDrain) && *abort_flag) {
        const uint64_t t0 = global_timer_ns();
        while (!mbar_test(bar(C::kBarDrain), 0) && global_timer_ns() - t0 < kWaitLimitNs) {}
      }
    }
  } else {
    // ===================================================== TMA producer
    if (lane == 0) {
      const uint64_t keep = policy_evict_last();
      mbar_arrive_expect_tx(bar(C::kBarKV), 2 * C::kTile);
      for (int bx = 0; bx < 4; ++bx) {
        tma_load_4d(sbase + C::kOffK + bx * 16384, &p.tm_k, bar(C::kBarKV), bx * 64, kh, sq.start + kv0, sq.bc);
        tma_load_4d(sbase + C::kOffV + bx * 16384, &p.tm_v, bar(C::kBarKV), bx * 64, kh, sq.start + kv0, sq.bc);
      }
      bool ok = true;
      int fill = 0, rows_issued = 0;
      for (int it = 0; it < n_iter && ok; ++it) {
        const int hh = kh * g + it / per_head;
        const int i = i_start + it % per_head;
        for (int t = 0; t < 4 && ok; ++t, ++fill) {  // Q(1-e), Q(e), dO(1-e), dO(e)
          const int half = (t & 1) ? e : 1 - e;
          const int s = slot_of(fill);
          ok = mbar_wait(bar(C::kBarEmpty0 + s), ((fill / C::kSlots) & 1) ^ 1, wctx, kBSiteEmpty);
          if (!ok) break;
          const uint32_t fb = bar(C::kBarFull0 + s);
          mbar_arrive_expect_tx(fb, C::kHalf);
          for (int bx = 0; bx < 2; ++bx)
            tma_load_4d_hint(sbase + C::kOffRing + s * C::kHalf + bx * 16384, t < 2 ? &p.tm_q : &p.tm_do, fb,
                             128 * half + bx * 64, hh, sq.start + i * 128, sq.bc, keep);
        }
        if (!ok) break;
        const int rs = it % C::kRowStages;
        ok = mbar_wait(bar(C::kBarRowEmpty0 + rs), ((it / C::kRowStages) & 1) ^ 1, wctx, kBSiteEmpty);
        if (!ok) break;
        const uint32_t rb = bar(C::kBarRowFull0 + rs);
        mbar_arrive_expect_tx(rb, 1024);
        const size_t roff = ((size_t)b * p.H + hh) * Npad + (size_t)i * 128;
        const uint32_t rdst = sbase + C::kOffRows + 1024 * rs;
        bulk_load(rdst, p.lse2 + roff, 512, rb);
        bulk_load(rdst + 512, p.delta + roff, 512, rb);
        ++rows_issued;
      }
      const uint64_t t0 = global_timer_ns();
      for (int f = max(0, fill - C::kSlots); f < fill; ++f)
        while (!mbar_test(bar(C::kBarFull0 + f % C::kSlots), (f / C::kSlots) & 1) &&
               global_timer_ns() - t0 < kWaitLimitNs) {}
      for (int f = max(0, rows_issued - C::kRowStages); f < rows_issued; ++f)
        while (!mbar_test(bar(C::kBarRowFull0 + f % C::kRowStages), (f / C::kRowStages) & 1) &&
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

// ================================================================== dK, dV at head dim 256 on CTA pairs
// Two CTAs of a cluster share one 128-row key tile, 64 keys each, and the
// rank-0 CTA issues every MMA as an M = 128 `cta_group::2` MMA.  With 64 keys
// per CTA the accumulators dV, dK (64 x 256 fp32 each) take 128 TMEM columns
// apiece, so S^T and dP^T are computed once over the whole head dim: no
// recomputation, unlike the one-CTA kernel above (which splits the head dim).
//
// In an M = 128 pair MMA, CTA c supplies rows 0-63 of A and half of B's N, and
// receives its 64 rows of D with N columns [0, N/2) in TMEM lanes 0-63 and
// [N/2, N) in lanes 64-127; an A operand in TMEM is read twice, from lanes 0-63
// for the first half of N and from lanes 64-127 for the second (both measured
// with a probe on GB300).  So:
//   S^T  = K Q^T    N = 128 queries: CTA c supplies query rows 64c..64c+63 (all
//                   of d); A = K from TMEM, copied there once and duplicated in
//                   both lane halves (128 columns)
//   dP^T = V dO^T   the same with V from shared memory
//   dV  += P^T dO   N = 256 = d: CTA c supplies head-dim columns 128c..128c+127
//   dK  += dS^T Q   (all queries); A = P^T, dS^T from shared memory, written by
//                   the elementwise warps (lane m holds key m with queries 0-63,
//                   lane 64+m the same key with queries 64-127)
// A CTA therefore needs three of the four 64 x 128 quarters of Q_i (and of dO_i):
// its query half in both head-dim halves, then the other query half in its
// head-dim half.  The MMAs address both CTAs' shared memory at one offset, and
// no fixed placement serves both uses, so each stage holds two quarter slots:
// S^T (dP^T) reads them as loaded, then the slot holding the quarter that only
// S^T needed is reloaded in place with the quarter that only dK (dV) needs.
// MMA order per iteration: S_i, dP_i, dV_{i-1}, dK_i, which gives every load and
// reload about two MMAs of lead with two Q stages and three dO stages; dS^T is
// computed while dV_{i-1} runs, and P^T is written once dV_{i-1} has read the
// previous one.
struct Dkdv256PairCfg {
  static constexpr int D = 256;
  static constexpr int kBox = 64 * 128;       // 64 rows x 64 columns of bf16 (one 128B-swizzled TMA box)
  static constexpr int kQuarter = 2 * kBox;   // 64 rows x 128 columns
  static constexpr int kStage = 2 * kQuarter;  // two quarter slots
  static constexpr int kQStages = 2, kDoStages = 3, kRowStages = 2;
  static constexpr int kThreads = 320;
  static constexpr int kMmaWarp = 8, kLoadWarp = 9;  // warps 0-7: elementwise (two warpgroups of 32 query columns)
  static constexpr int kColK = 0, kColS = 128, kColDP = 192, kColDV = 256, kColDK = 384, kTmemCols = 512;
  static constexpr int kOffV = 0;                                 // 64 keys x 256: 4 boxes
  static constexpr int kOffP = 4 * kBox;                          // P^T: 64 keys x 128 queries, 2 boxes
  static constexpr int kOffDS = kOffP + 2 * kBox;                 // dS^T
  static constexpr int kOffQ = kOffDS + 2 * kBox;                 // Q stages
  static constexpr int kOffDO = kOffQ + kQStages * kStage;        // dO stages
  static constexpr int kOffKTmp = kOffDO + 2 * kStage;            // K before its copy into TMEM: dO stage 2
  static constexpr int kOffRows = kOffDO + kDoStages * kStage;    // LSE2 / D per row stage
  enum { kBarKV, kBarK, kBarKT, kBarKCopied, kBarFullQ0, kBarEmptyQ0 = kBarFullQ0 + kQStages,
         kBarReQ0 = kBarEmptyQ0 + kQStages, kBarFullD0 = kBarReQ0 + kQStages, kBarEmptyD0 = kBarFullD0 + kDoStages,
         kBarReD0 = kBarEmptyD0 + kDoStages, kBarRowFull0 = kBarReD0 + kDoStages,
         kBarRowEmpty0 = kBarRowFull0 + kRowStages, kBarS = kBarRowEmpty0 + kRowStages, kBarDP, kBarP, kBarDS,
         kBarVdone, kBarFinal, kBarDrain, kNumBars };
  static constexpr int kOffBar = kOffRows + 1024 * kRowStages;
  static constexpr int kOffMisc = kOffBar + 8 * kNumBars;
  static constexpr int kSmemBytes = kOffMisc + 16;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// P^T = 2^(S^T c - LSE2) for one key row and 32 query columns (fp32 in pe,
// packed bf16 pairs in w).  Key row kr (within the pair's 128-key tile) is
// hidden from query column qc when qc + qoff < kr under the causal mask (diag),
// qoff = 128 (query tile - key tile); rows past the sequence give 0.
template <bool MASK>
__device__ __forceinline__ void dkdv256_p(const uint32_t (&sv)[32], float (&pe)[32], uint32_t (&w)[16],
                                          const float *lse2_s, float scale_log2, int qc0, int kr, bool row_valid,
                                          bool diag, int qoff) {
#pragma unroll
  for (int k = 0; k < 32; k += 4) {
    const float4 l4 = *reinterpret_cast<const float4 *>(lse2_s + k);
    float x[4];
    ffma2(x[0], x[1], __uint_as_float(sv[k]), __uint_as_float(sv[k + 1]), scale_log2, scale_log2, -l4.x, -l4.y);
    ffma2(x[2], x[3], __uint_as_float(sv[k + 2]), __uint_as_float(sv[k + 3]), scale_log2, scale_log2, -l4.z, -l4.w);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      pe[k + u] = ex2_mufu(x[u]);
      if (MASK && (!row_valid || (diag && qc0 + k + u + qoff < kr))) pe[k + u] = 0.f;
    }
    w[k >> 1] = pack_bf16x2(pe[k], pe[k + 1]);
    w[(k >> 1) + 1] = pack_bf16x2(pe[k + 2], pe[k + 3]);
  }
}

// 16 packed words (32 columns from col0) of row r into a K-major operand tile
// of 64-row, 64-column boxes (8 KB each, 128-byte swizzle).
__device__ __forceinline__ void st_swizzled_32cols_r64(uint32_t tile, int r, int col0, const uint32_t (&w)[16]) {
  const uint32_t row = tile + (uint32_t)(col0 >> 6) * 8192u + (uint32_t)r * 128u;
  const int chunk0 = (col0 & 63) >> 3;
#pragma unroll
  for (int k = 0; k < 4; ++k)
    st_shared_v4(row + (uint32_t)(((chunk0 + k) ^ (r & 7)) * 16), w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
}

template <bool CAUSAL, bool VARLEN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(320, 1)
    bwd_dkdv256_pair_kernel(const __grid_constant__ BwdParams p) {
  using C = Dkdv256PairCfg;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  if (!check_align(sbase, p.status)) return;  // same layout in both CTAs: both return
  const uint32_t bar0 = sbase + C::kOffBar;
  auto bar = [&](int i) { return bar0 + 8u * i; };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 4);
  const WaitCtx wctx{abort_flag, p.status};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int crank = (int)cluster_ctarank();
  const int n_kv = (p.N + 127) / 128;
  int rank, head;
  work_order((int)(blockIdx.x >> 1), n_kv, p.B * p.Hkv, p.sched_chunk, rank, head);
  const int jt = rank;  // the pair's key tile; causal: rank 0 sees the most query tiles
  const int kh = head % p.Hkv, b = head / p.Hkv;
  const int g = p.H / p.Hkv;
  const SeqSpan sq = VARLEN ? seq_span(p.cu_seqlens, b, p.N, p.total) : SeqSpan{0, p.N, b};
  const int L = sq.len;
  const int Npad = (p.N + 127) / 128 * 128;
  const int kv0 = jt * 128;
  if (VARLEN && kv0 >= L) return;  // the tile lies past its sequence (both CTAs return)
  const int n_q = (L + 127) / 128;
  const int i_start = CAUSAL ? jt : 0;
  const int per_head = n_q - i_start;
  const int n_iter = g * per_head;
  const int key0 = kv0 + 64 * crank;  // this CTA's first key row

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kNumBars; ++i) {
      // P, dS and K-in-TMEM collect one arrival per elementwise warp of both CTAs;
      // the row ring and the K copy are local (8 warps); the rest take one arrival
      const bool pair_warps = i == C::kBarP || i == C::kBarDS || i == C::kBarKT;
      const bool local_warps = i == C::kBarKCopied || (i >= C::kBarRowEmpty0 && i < C::kBarRowEmpty0 + C::kRowStages);
      mbar_init(bar(i), pair_warps ? 16u : local_warps ? 8u : 1u);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == C::kMmaWarp) {
    tmem_alloc_pair(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish_pair();
  }
  if (warp == C::kLoadWarp && lane == 0) {
    prefetch_tmap(&p.tm_q64);
    prefetch_tmap(&p.tm_do64);
    prefetch_tmap(&p.tm_k64);
    prefetch_tmap(&p.tm_v64);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // barriers of both CTAs initialised, TMEM of both allocated
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 8) {
    const int wg = warp >> 2;
    const int r = threadIdx.x & 127;  // TMEM lane
    const int m = r & 63, h = r >> 6;  // key row of this CTA, query half of the S^T / dP^T columns
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    bool ok = true;
    // ---- K -> TMEM (A of S^T): row m in lanes m and 64 + m, head-dim columns 2x, 2x+1 in column x
    ok = mbar_wait_warp(bar(C::kBarK), 0, wctx, kBSiteKV);
    if (ok) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int bx = 2 * wg + half;  // 64-column box of K
        uint32_t kw[32];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint4 v = *reinterpret_cast<const uint4 *>(smem + C::kOffKTmp + bx * C::kBox + m * 128 +
                                                           ((j ^ (m & 7)) * 16));
          kw[4 * j] = v.x;
          kw[4 * j + 1] = v.y;
          kw[4 * j + 2] = v.z;
          kw[4 * j + 3] = v.w;
        }
        tmem_st_32x32b_x32(tmem + lane_off + C::kColK + 32 * bx, kw);
      }
      tmem_wait_st();
    }
    fence_proxy_async_smem();  // the region is refilled by TMA (dO stage 2) after this
    tc_fence_before();
    mbar_arrive_warp_cluster(mapa_shared(bar(C::kBarKT), 0));
    mbar_arrive_warp(bar(C::kBarKCopied));

    // ---- P^T and dS^T of this CTA's 64 keys, 32 query columns per thread
    const uint32_t s_tm = tmem + lane_off + C::kColS + 32 * wg;
    const uint32_t dp_tm = tmem + lane_off + C::kColDP + 32 * wg;
    const int kr = 64 * crank + m;  // key row within the pair's tile
    const bool row_valid = kv0 + kr < L;
    const bool warp_has_invalid = __any_sync(0xffffffffu, !row_valid);
    const int qc0 = 64 * h + 32 * wg;  // this thread's first query column
    for (int it = 0; it < n_iter && ok; ++it) {
      const int rs = it % C::kRowStages;
      const int i = i_start + it % per_head;
      const float *lse2_s = reinterpret_cast<const float *>(smem + C::kOffRows + 1024 * rs) + qc0;
      const float *dlt_s = lse2_s + 128;
      ok = mbar_wait_warp_cl(bar(C::kBarS), it & 1, wctx, kBSiteS);
      if (ok) ok = mbar_wait_warp(bar(C::kBarRowFull0 + rs), (it / C::kRowStages) & 1, wctx, kBSiteFull);
      if (!ok) break;
      tc_fence_after();
      uint32_t sv[32];
      tmem_ld_32x32b_x32(s_tm, sv);
      tmem_wait_ld(sv);
      const bool diag = CAUSAL && i <= jt;
      const int qoff = 128 * (i - jt);
      float pe[32];
      uint32_t wp[16];
      if (warp_has_invalid || diag)
        dkdv256_p<true>(sv, pe, wp, lse2_s, p.scale_log2, qc0, kr, row_valid, diag, qoff);
      else
        dkdv256_p<false>(sv, pe, wp, lse2_s, p.scale_log2, qc0, kr, row_valid, diag, qoff);
      // dS^T = P^T (dP^T - D) first: dK_i waits for it while dV_{i-1} runs
      ok = mbar_wait_warp_cl(bar(C::kBarDP), it & 1, wctx, kBSiteDP);
      if (!ok) break;
      tc_fence_after();
      uint32_t dpv[32];
      tmem_ld_32x32b_x32(dp_tm, dpv);
      tmem_wait_ld(dpv);
      uint32_t wd[16];
#pragma unroll
      for (int k = 0; k < 32; k += 4) {
        const float4 d4 = *reinterpret_cast<const float4 *>(dlt_s + k);
        float t[4], ds[4];
        fadd2(t[0], t[1], __uint_as_float(dpv[k]), __uint_as_float(dpv[k + 1]), -d4.x, -d4.y);
        fadd2(t[2], t[3], __uint_as_float(dpv[k + 2]), __uint_as_float(dpv[k + 3]), -d4.z, -d4.w);
        fmul2(ds[0], ds[1], pe[k], pe[k + 1], t[0], t[1]);
        fmul2(ds[2], ds[3], pe[k + 2], pe[k + 3], t[2], t[3]);
        wd[k >> 1] = pack_bf16x2(ds[0], ds[1]);
        wd[(k >> 1) + 1] = pack_bf16x2(ds[2], ds[3]);
      }
      // the dS^T buffer is free: dK_{i-1} was issued before dP_i, whose completion was just seen
      st_swizzled_32cols_r64(sbase + C::kOffDS, m, qc0, wd);
      fence_proxy_async_smem();
      tc_fence_before();  // S^T and dP^T have been read: the next S, dP may overwrite them
      mbar_arrive_warp_cluster(mapa_shared(bar(C::kBarDS), 0));
      mbar_arrive_warp(bar(C::kBarRowEmpty0 + rs));  // LSE2 / D rows of this stage no longer read
      // P^T once dV_{i-1} has read the previous one
      if (it > 0) {
        ok = mbar_wait_warp_cl(bar(C::kBarVdone), (it - 1) & 1, wctx, kBSiteP);
        if (!ok) break;
      }
      st_swizzled_32cols_r64(sbase + C::kOffP, m, qc0, wp);
      fence_proxy_async_smem();
      mbar_arrive_warp_cluster(mapa_shared(bar(C::kBarP), 0));
    }
    // ---- epilogue: warpgroup 0 stores dV, warpgroup 1 dK * scale (staged in the Q ring)
    if (ok) ok = mbar_wait_warp_cl(bar(C::kBarFinal), 0, wctx, kBSiteFinal);
    tc_fence_after();
    const uint32_t stage = sbase + C::kOffQ + wg * 4 * C::kBox;
    const uint32_t acc_tm = tmem + lane_off + (wg == 0 ? C::kColDV : C::kColDK);
    const float mul = wg == 0 ? 1.0f : p.scale;
    const bool has_rows = key0 < L;
    const bool direct = VARLEN && key0 + 64 > L;  // the next sequence's rows follow: write row by row
    if (ok && has_rows && direct) {
      __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(wg == 0 ? p.dv : p.dk);
      acc_to_global<128>(acc_tm, out + ((size_t)(sq.start + key0 + m) * p.Hkv + kh) * 256 + 128 * h, 0, mul,
                         key0 + m < L);
    } else if (ok && has_rows) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(acc_tm + 32 * j, v);
        tmem_wait_ld(v);
        uint32_t w[16];
#pragma unroll
        for (int k = 0; k < 16; ++k)
          w[k] = pack_bf16x2(__uint_as_float(v[2 * k]) * mul, __uint_as_float(v[2 * k + 1]) * mul);
        st_swizzled_32cols_r64(stage, m, 128 * h + 32 * j, w);
      }
    }
    fence_proxy_async_smem();
    named_bar_sync(1 + wg, 128);
    if (r == 0 && ok && has_rows && !direct) {
      const CUtensorMap *map = wg == 0 ? &p.tm_dv64 : &p.tm_dk64;
      for (int bx = 0; bx < 4; ++bx) tma_store_4d(map, stage + bx * C::kBox, bx * 64, kh, sq.start + key0, sq.bc);
      bulk_commit();
      bulk_wait_read_all();
    }
  } else if (warp == C::kMmaWarp) {
    // ===================================================== MMA issue (rank-0 CTA, for both)
    if (crank == 0) {
      constexpr uint32_t id_s = make_idesc_bf16(128, 128, false, false);  // S^T (A in TMEM), dP^T
      constexpr uint32_t id_o = make_idesc_bf16(128, 256, false, true);   // dV, dK (B MN-major)
      const uint64_t v_d = make_sdesc_sw128(sbase + C::kOffV, 0, 1024);
      const uint64_t p_d = make_sdesc_sw128(sbase + C::kOffP, 0, 1024);
      const uint64_t ds_d = make_sdesc_sw128(sbase + C::kOffDS, 0, 1024);
      const uint64_t q_d = make_sdesc_sw128(sbase + C::kOffQ, 0, 1024);
      const uint64_t q_mn = make_sdesc_sw128(sbase + C::kOffQ, C::kBox, 1024);
      const uint64_t do_d = make_sdesc_sw128(sbase + C::kOffDO, 0, 1024);
      const uint64_t do_mn = make_sdesc_sw128(sbase + C::kOffDO, C::kBox, 1024);
      auto kmaj = [](int kk) { return (uint64_t)(((kk >> 2) * C::kBox + (kk & 3) * 32) >> 4); };
      auto off = [](int bytes) { return (uint64_t)(bytes >> 4); };
      bool ok = mbar_wait_warp_cl(bar(C::kBarKV), 0, wctx, kBSiteKV);
      if (ok) ok = mbar_wait_warp_cl(bar(C::kBarKT), 0, wctx, kBSiteKV);
      for (int it = 0; it <= n_iter && ok; ++it) {
        if (it < n_iter) {
          const int s = it % C::kQStages, sd = it % C::kDoStages;
          ok = mbar_wait_warp_cl(bar(C::kBarFullQ0 + s), (it / C::kQStages) & 1, wctx, kBSiteFull);
          if (!ok) break;
          tc_fence_after();
          if (elect_one()) {  // S^T = K Q^T: head-dim half kk / 8 of this CTA's query rows
#pragma unroll
            for (int kk = 0; kk < 16; ++kk)
              mma_ts_pair(tmem + C::kColS, tmem + C::kColK + 8 * kk,
                          q_d + off(s * C::kStage + (kk >> 3) * C::kQuarter) + kmaj(kk & 7), id_s, kk > 0);
            tc_commit_pair(bar(C::kBarS));
          }
          __syncwarp();
          ok = mbar_wait_warp_cl(bar(C::kBarFullD0 + sd), (it / C::kDoStages) & 1, wctx, kBSiteFull);
          if (!ok) break;
          tc_fence_after();
          if (elect_one()) {  // dP^T = V dO^T
#pragma unroll
            for (int kk = 0; kk < 16; ++kk)
              mma_ss_pair(tmem + C::kColDP, v_d + kmaj(kk),
                          do_d + off(sd * C::kStage + (kk >> 3) * C::kQuarter) + kmaj(kk & 7), id_s, kk > 0);
            tc_commit_pair(bar(C::kBarDP));
          }
          __syncwarp();
        }
        if (it > 0) {  // dV += P^T dO of the previous iteration (its second dO quarter reloaded)
          const int j = it - 1, sd = j % C::kDoStages;
          ok = mbar_wait_warp_cl(bar(C::kBarP), j & 1, wctx, kBSiteP);
          if (ok) ok = mbar_wait_warp_cl(bar(C::kBarReD0 + sd), (j / C::kDoStages) & 1, wctx, kBSiteFull);
          if (!ok) break;
          tc_fence_after();
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ss_pair(tmem + C::kColDV, p_d + kmaj(kk),
                          do_mn + off(sd * C::kStage + (kk >> 2) * C::kQuarter + (kk & 3) * 2048), id_o,
                          (j > 0 || kk > 0));
            tc_commit_pair(bar(C::kBarVdone));
            tc_commit_pair(bar(C::kBarEmptyD0 + sd));
          }
          __syncwarp();
        }
        if (it < n_iter) {  // dK += dS^T Q (the second Q quarter reloaded)
          const int s = it % C::kQStages;
          ok = mbar_wait_warp_cl(bar(C::kBarDS), it & 1, wctx, kBSiteDS);
          if (ok) ok = mbar_wait_warp_cl(bar(C::kBarReQ0 + s), (it / C::kQStages) & 1, wctx, kBSiteFull);
          if (!ok) break;
          tc_fence_after();
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ss_pair(tmem + C::kColDK, ds_d + kmaj(kk),
                          q_mn + off(s * C::kStage + (kk >> 2) * C::kQuarter + (kk & 3) * 2048), id_o,
                          (it > 0 || kk > 0));
            tc_commit_pair(bar(C::kBarEmptyQ0 + s));
          }
          __syncwarp();
        }
      }
      if (elect_one()) {
        tc_commit_pair(bar(C::kBarFinal));
        tc_commit_pair(bar(C::kBarDrain));
      }
      __syncwarp();
      if (!mbar_wait_warp_cl(bar(C::kBarDrain), 0, wctx, kBSiteDrain) && *abort_flag) {
        const uint64_t t0 = global_timer_ns();
        while (!mbar_test_cl(bar(C::kBarDrain), 0) && global_timer_ns() - t0 < kWaitLimitNs) {}
      }
    }
  } else {
    // ===================================================== TMA producer (both CTAs; stage bytes counted by rank 0)
    if (lane == 0) {
      const uint64_t keep = policy_evict_last();
      auto head_of = [&](int it) { return kh * g + it / per_head; };
      auto row0_of = [&](int it) { return sq.start + (i_start + it % per_head) * 128; };
      // V on the rank-0 CTA's barrier (both CTAs' MMAs read it); K on this CTA's own (copied into TMEM here)
      if (crank == 0) mbar_arrive_expect_tx(bar(C::kBarKV), 2 * 4 * C::kBox);
      mbar_arrive_expect_tx(bar(C::kBarK), 4 * C::kBox);
      const uint32_t kv_bar = mapa_shared(bar(C::kBarKV), 0);
      for (int bx = 0; bx < 4; ++bx) {
        tma_load_4d_pair(sbase + C::kOffV + bx * C::kBox, &p.tm_v64, kv_bar, bx * 64, kh, sq.start + key0, sq.bc,
                         keep);
        tma_load_4d(sbase + C::kOffKTmp + bx * C::kBox, &p.tm_k64, bar(C::kBarK), bx * 64, kh, sq.start + key0,
                    sq.bc);
      }
      bool ok = true;
      int nfq = 0, nrq = 0, nfd = 0, nrd = 0, rows_issued = 0;
      for (int it = 0; it <= n_iter && ok; ++it) {
        if (it < n_iter) {  // Q_it: this CTA's query half, both head-dim halves
          const int s = it % C::kQStages;
          ok = mbar_wait_cl(bar(C::kBarEmptyQ0 + s), ((it / C::kQStages) & 1) ^ 1, wctx, kBSiteEmpty);
          if (!ok) break;
          if (crank == 0) mbar_arrive_expect_tx(bar(C::kBarFullQ0 + s), 2 * C::kStage);
          const uint32_t fb = mapa_shared(bar(C::kBarFullQ0 + s), 0);
          for (int dh = 0; dh < 2; ++dh)
            for (int bx = 0; bx < 2; ++bx)
              tma_load_4d_pair(sbase + C::kOffQ + s * C::kStage + dh * C::kQuarter + bx * C::kBox, &p.tm_q64, fb,
                               128 * dh + 64 * bx, head_of(it), row0_of(it) + 64 * crank, sq.bc, keep);
          ++nfq;
        }
        if (it > 0) {  // reloads for the previous iteration: the other query half, this CTA's head-dim half
          const int j = it - 1;
          ok = mbar_wait_cl(bar(C::kBarS), j & 1, wctx, kBSiteS);  // S^T_j has read the slot
          if (!ok) break;
          const int s = j % C::kQStages;
          if (crank == 0) mbar_arrive_expect_tx(bar(C::kBarReQ0 + s), 2 * C::kQuarter);
          const uint32_t rq = mapa_shared(bar(C::kBarReQ0 + s), 0);
          for (int bx = 0; bx < 2; ++bx)
            tma_load_4d_pair(sbase + C::kOffQ + s * C::kStage + (1 - crank) * C::kQuarter + bx * C::kBox, &p.tm_q64,
                             rq, 128 * crank + 64 * bx, head_of(j), row0_of(j) + 64 * (1 - crank), sq.bc, keep);
          ++nrq;
          ok = mbar_wait_cl(bar(C::kBarDP), j & 1, wctx, kBSiteDP);  // dP^T_j has read the slot
          if (!ok) break;
          const int sd = j % C::kDoStages;
          if (crank == 0) mbar_arrive_expect_tx(bar(C::kBarReD0 + sd), 2 * C::kQuarter);
          const uint32_t rd = mapa_shared(bar(C::kBarReD0 + sd), 0);
          for (int bx = 0; bx < 2; ++bx)
            tma_load_4d_pair(sbase + C::kOffDO + sd * C::kStage + (1 - crank) * C::kQuarter + bx * C::kBox,
                             &p.tm_do64, rd, 128 * crank + 64 * bx, head_of(j), row0_of(j) + 64 * (1 - crank), sq.bc,
                             keep);
          ++nrd;
        }
        if (it < n_iter) {  // dO_it, then the row terms
          const int sd = it % C::kDoStages;
          if (it == 2) {  // dO stage 2 held the K tile
            ok = mbar_wait(bar(C::kBarKCopied), 0, wctx, kBSiteKV);
            if (!ok) break;
          }
          ok = mbar_wait_cl(bar(C::kBarEmptyD0 + sd), ((it / C::kDoStages) & 1) ^ 1, wctx, kBSiteEmpty);
          if (!ok) break;
          if (crank == 0) mbar_arrive_expect_tx(bar(C::kBarFullD0 + sd), 2 * C::kStage);
          const uint32_t fb = mapa_shared(bar(C::kBarFullD0 + sd), 0);
          for (int dh = 0; dh < 2; ++dh)
            for (int bx = 0; bx < 2; ++bx)
              tma_load_4d_pair(sbase + C::kOffDO + sd * C::kStage + dh * C::kQuarter + bx * C::kBox, &p.tm_do64, fb,
                               128 * dh + 64 * bx, head_of(it), row0_of(it) + 64 * crank, sq.bc, keep);
          ++nfd;
          const int rs = it % C::kRowStages;
          ok = mbar_wait(bar(C::kBarRowEmpty0 + rs), ((it / C::kRowStages) & 1) ^ 1, wctx, kBSiteEmpty);
          if (!ok) break;
          const uint32_t rb = bar(C::kBarRowFull0 + rs);
          mbar_arrive_expect_tx(rb, 1024);
          const size_t roff = ((size_t)b * p.H + head_of(it)) * Npad + (size_t)(i_start + it % per_head) * 128;
          const uint32_t rdst = sbase + C::kOffRows + 1024 * rs;
          bulk_load(rdst, p.lse2 + roff, 512, rb);
          bulk_load(rdst + 512, p.delta + roff, 512, rb);
          ++rows_issued;
        }
      }
      // drain: the stage barriers of rank 0 count both CTAs' copies; K and the row ring are local
      const uint64_t t0 = global_timer_ns();
      auto drain = [&](int base, int stages, int n) {
        for (int u = max(0, n - stages); u < n; ++u)
          while (!mbar_test_cl(bar(base + u % stages), (u / stages) & 1) && global_timer_ns() - t0 < kWaitLimitNs) {}
      };
      if (crank == 0) {
        drain(C::kBarFullQ0, C::kQStages, nfq);
        drain(C::kBarReQ0, C::kQStages, nrq);
        drain(C::kBarFullD0, C::kDoStages, nfd);
        drain(C::kBarReD0, C::kDoStages, nrd);
        while (!mbar_test_cl(bar(C::kBarKV), 0) && global_timer_ns() - t0 < kWaitLimitNs) {}
      }
      while (!mbar_test(bar(C::kBarK), 0) && global_timer_ns() - t0 < kWaitLimitNs) {}
      for (int f = max(0, rows_issued - C::kRowStages); f < rows_issued; ++f)
        while (!mbar_test(bar(C::kBarRowFull0 + f % C::kRowStages), (f / C::kRowStages) & 1) &&
               global_timer_ns() - t0 < kWaitLimitNs) {}
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

struct Dq256Cfg {
  static constexpr int D = 256;
  static constexpr int kTile = 128 * D * 2;
  static constexpr int kHalf = kTile / 2;
  static constexpr int kSlots = 3;
  static constexpr int kNumWG = 2;
  static constexpr int kThreads = 320;
  static constexpr int kMmaWarp = 8;  // warp 9: TMA producer
  static constexpr int kDPBufs = 1;
  static constexpr int kColS = 0, kColDP = 128, kColDQ = 256;
  static constexpr int kTmemCols = 512;
  static constexpr int kOffQ = 0, kOffDO = kTile, kOffRing = 2 * kTile;
  enum { kBarQdo, kBarFull0, kBarEmpty0 = kBarFull0 + kSlots, kBarS = kBarEmpty0 + kSlots, kBarSFree, kBarDP,
         kBarDS, kBarFinal, kBarDrain, kNumBars };
  static constexpr int kOffBar = kOffRing + kSlots * kHalf;
  static constexpr int kOffMisc = kOffBar + 8 * kNumBars;
  static constexpr int kSmemBytes = kOffMisc + 16;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

template <bool CAUSAL, bool VARLEN>
__global__ void __launch_bounds__(320, 1) bwd_dq256_kernel(const __grid_constant__ BwdParams p) {
  using C = Dq256Cfg;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  if (!check_align(sbase, p.status)) return;
  const uint32_t bar0 = sbase + C::kOffBar;
  auto bar = [&](int i) { return bar0 + 8u * i; };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 4);
  const WaitCtx wctx{abort_flag, p.status};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_q = (p.N + 127) / 128;
  int rank, head;
  work_order((int)blockIdx.x, n_q, p.B * p.H, p.sched_chunk, rank, head);
  const int it_q = CAUSAL ? n_q - 1 - rank : rank;
  const int h = head % p.H, b = head / p.H;
  const int kh = h / (p.H / p.Hkv);
  const int Npad = n_q * 128;  // row-term arrays are [B, H, Npad]
  const int q0 = it_q * 128;
  const SeqSpan sq = VARLEN ? seq_span(p.cu_seqlens, b, p.N, p.total) : SeqSpan{0, p.N, b};
  const int L = sq.len;  // rows of this sequence
  if (VARLEN && q0 >= L) return;  // the tile lies past its sequence: no rows to produce
  const int nb = CAUSAL ? it_q + 1 : (L + 127) / 128;
  // per key tile four fills: V half 0, V half 1, K half 0, K half 1
  auto fill_of = [](int j, bool is_k, int half) { return 4 * j + (is_k ? 2 : 0) + half; };
  auto slot_of = [](int fill) { return fill % C::kSlots; };

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kNumBars; ++i)  // per elementwise warp
      mbar_init(bar(i), (i == C::kBarSFree || i == C::kBarDS) ? 8u : 1u);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == C::kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 8) {
    const int wg = warp >> 2;
    const int r = threadIdx.x & 127;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const int q_row = q0 + r;
    const size_t rw = ((size_t)b * p.H + h) * Npad + q_row;
    const float lse2 = p.lse2[rw];
    const float dlt = p.delta[rw];
    bool ok = dq_rows<C, CAUSAL>(p, bar0, tmem, wctx, warp, nb, q_row, lse2, dlt, L);
    // ---- epilogue: dQ * scale -> bf16 -> shared (the Q tile, free once every S MMA is done) -> TMA store
    if (ok) ok = mbar_wait_warp(bar(C::kBarFinal), 0, wctx, kBSiteFinal);
    tc_fence_after();
    uint8_t *stage = smem + C::kOffQ;
    const bool direct = VARLEN && q0 + 128 > L;  // the next sequence's rows follow: write row by row
    if (ok && direct)
      acc_to_global<128>(tmem + lane_off + C::kColDQ,
                         static_cast<__nv_bfloat16 *>(p.dq) + ((size_t)(sq.start + q_row) * p.H + h) * 256, wg * 128,
                         p.scale, q_row < L);
    else if (ok)
      acc_to_smem<128>(tmem + lane_off + C::kColDQ, stage, r, wg * 128, p.scale);
    fence_proxy_async_smem();
    named_bar_sync(1, 256);
    if (threadIdx.x == 0 && ok && !direct) {
      for (int bx = 0; bx < 4; ++bx)
        tma_store_4d(&p.tm_dq, sbase + C::kOffQ + bx * 16384, bx * 64, h, sq.start + q0, sq.bc);
      bulk_commit();
      bulk_wait_read_all();
    }
  } else if (warp == C::kMmaWarp) {
    // ===================================================== MMA issue: dP_j, S_j, [dS_j] dQ_j per key tile
    // The whole warp runs the loop and waits; the elected lane issues.
    {
      constexpr uint32_t id_s = make_idesc_bf16(128, 128, false, false);
      constexpr uint32_t id_dq = make_idesc_bf16(128, 128, false, true);  // A = dS in TMEM, B = K half MN-major
      const uint64_t q_d = make_sdesc_sw128(sbase + C::kOffQ, 0, 1024);
      const uint64_t do_d = make_sdesc_sw128(sbase + C::kOffDO, 0, 1024);
      const uint64_t ring_d = make_sdesc_sw128(sbase + C::kOffRing, 0, 1024);
      const uint64_t ring_mn = make_sdesc_sw128(sbase + C::kOffRing, 16384, 1024);
      auto kmaj = [](int kk) { return (uint64_t)((((kk >> 2) * 16384 + (kk & 3) * 32)) >> 4); };
      auto soff = [&](int fill) { return (uint64_t)((slot_of(fill) * C::kHalf) >> 4); };
      auto full_ok = [&](int fill) {
        return mbar_wait_warp(bar(C::kBarFull0 + slot_of(fill)), (uint32_t)((fill / C::kSlots) & 1), wctx,
                              kBSiteFull);
      };
      auto release = [&](int fill) { tc_commit(bar(C::kBarEmpty0 + slot_of(fill))); };
      auto a_col = [](int kk) { return (uint32_t)(64 * (kk >> 2) + 8 * (kk & 3)); };
      bool ok = mbar_wait_warp(bar(C::kBarQdo), 0, wctx, kBSiteQ);
      for (int j = 0; j < nb && ok; ++j) {
        // dP_j = dO V_j^T (the dP columns are free: dQ_{j-1} has read dS_{j-1} from them)
        ok = full_ok(fill_of(j, false, 0)) && full_ok(fill_of(j, false, 1));
        if (!ok) break;
        tc_fence_after();
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < 16; ++kk)
            mma_ss(tmem + C::kColDP, do_d + kmaj(kk), ring_d + soff(fill_of(j, false, kk >> 3)) + kmaj(kk & 7), id_s,
                   kk > 0);
          tc_commit(bar(C::kBarDP));
          release(fill_of(j, false, 0));
          release(fill_of(j, false, 1));
        }
        __syncwarp();
        // S_j = Q K_j^T (the S columns are free: S_{j-1} was read before dS_{j-1})
        ok = full_ok(fill_of(j, true, 0)) && full_ok(fill_of(j, true, 1));
        if (!ok) break;
        tc_fence_after();
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < 16; ++kk)
            mma_ss(tmem + C::kColS, q_d + kmaj(kk), ring_d + soff(fill_of(j, true, kk >> 3)) + kmaj(kk & 7), id_s,
                   kk > 0);
          tc_commit(bar(C::kBarS));
        }
        __syncwarp();
        // dQ[:, half] += dS_j K_j[:, half]
        ok = mbar_wait_warp(bar(C::kBarDS), j & 1, wctx, kBSiteDS);
        if (!ok) break;
        tc_fence_after();
        if (elect_one()) {
#pragma unroll
          for (int half = 0; half < 2; ++half)
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ts(tmem + C::kColDQ + 128u * half, tmem + C::kColDP + a_col(kk),
                     ring_mn + soff(fill_of(j, true, half)) + (uint64_t)(kk * 128), id_dq, (j > 0 || kk > 0));
          release(fill_of(j, true, 0));
          release(fill_of(j, true, 1));
        }
        __syncwarp();
      }
      if (elect_one()) {
        tc_commit(bar(C::kBarFinal));
        tc_commit(bar(C::kBarDrain));
      }
      __syncwarp();
      if (!mbar_wait_warp(bar(C::kBarDrain), 0, wctx, kBSiteDrain) && *abort_flag) {
        const uint64_t t0 = global_timer_ns();
        while (!mbar_test(bar(C::kBarDrain), 0) && global_timer_ns() - t0 < kWaitLimitNs) {}
      }
    }
  } else {
    // ===================================================== TMA producer
    if (lane == 0) {
      const uint64_t keep = policy_evict_last();
      const uint64_t once = policy_evict_first();
      mbar_arrive_expect_tx(bar(C::kBarQdo), 2 * C::kTile);
      for (int bx = 0; bx < 4; ++bx) {
        tma_load_4d_hint(sbase + C::kOffQ + bx * 16384, &p.tm_q, bar(C::kBarQdo), bx * 64, h, sq.start + q0, sq.bc,
                         once);
        tma_load_4d_hint(sbase + C::kOffDO + bx * 16384, &p.tm_do, bar(C::kBarQdo), bx * 64, h, sq.start + q0, sq.bc,
                         once);
      }
      bool ok = true;
      int fill = 0;
      for (int j = 0; j < nb && ok; ++j) {
        for (int t = 0; t < 4 && ok; ++t, ++fill) {  // V0, V1, K0, K1
          const int s = slot_of(fill);
          ok = mbar_wait(bar(C::kBarEmpty0 + s), ((fill / C::kSlots) & 1) ^ 1, wctx, kBSiteEmpty);
          if (!ok) break;
          const uint32_t fb = bar(C::kBarFull0 + s);
          mbar_arrive_expect_tx(fb, C::kHalf);
          for (int bx = 0; bx < 2; ++bx)
            tma_load_4d_hint(sbase + C::kOffRing + s * C::kHalf + bx * 16384, t < 2 ? &p.tm_v : &p.tm_k, fb,
                             128 * (t & 1) + bx * 64, kh, sq.start + j * 128, sq.bc, keep);
        }
      }
      const uint64_t t0 = global_timer_ns();
      for (int f = max(0, fill - C::kSlots); f < fill; ++f)
        while (!mbar_test(bar(C::kBarFull0 + f % C::kSlots), (f / C::kSlots) & 1) &&
               global_timer_ns() - t0 < kWaitLimitNs) {}
      while (!mbar_test(bar(C::kBarQdo), 0) && global_timer_ns() - t0 < kWaitLimitNs) {}
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ================================================================== dQ at head dim 256 on CTA pairs
// Two CTAs of a cluster share one 128-row query tile, 64 query rows each, with
// M = 128 `cta_group::2` MMAs issued by the rank-0 CTA (the TMEM and operand
// layouts of the head-dim-256 dK/dV pair kernel above):
//   S  = Q K_j^T    N = 128 keys: CTA c supplies key rows 64c..64c+63 (all d);
//   dP = dO V_j^T   A = Q, dO from TMEM (copied once, both lane halves)
//   dQ += dS K_j    N = 256 = d: CTA c supplies head-dim columns 128c..128c+127
//                   of all keys; A = dS from shared memory (two buffers)
// K_j streams as two quarter slots per stage, the one only S needed reloaded
// in place for dQ; V_j only feeds dP.  TMEM: Q 128 | dO 128 | S 64 | dP 64 |
// dQ 128 columns.  MMA order per key tile: S_j, dP_j, dQ_{j-1}; S and dP are
// single-buffered, so the elementwise warps signal as soon as they have read them.
struct Dq256PairCfg {
  static constexpr int kBox = 64 * 128;        // 64 rows x 64 columns of bf16
  static constexpr int kQuarter = 2 * kBox;    // 64 rows x 128 columns
  static constexpr int kStage = 2 * kQuarter;  // two quarter slots
  static constexpr int kKStages = 3, kVStages = 3, kDsBufs = 2;
  static constexpr int kThreads = 320;
  static constexpr int kMmaWarp = 8, kLoadWarp = 9;
  static constexpr int kColQ = 0, kColDO = 128, kColS = 256, kColDP = 320, kColDQ = 384, kTmemCols = 512;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kKStages * kStage;
  static constexpr int kOffDS = kOffV + kVStages * kStage;     // dS buffers: 64 queries x 128 keys, 2 boxes each
  static constexpr int kOffQTmp = kOffV + 2 * kStage;          // Q before its copy into TMEM: V stage 2
  static constexpr int kOffDOTmp = kOffK + 2 * kStage;         // dO before its copy: K stage 2
  enum { kBarQdo, kBarQT, kBarCopied, kBarFullK0, kBarEmptyK0 = kBarFullK0 + kKStages,
         kBarReK0 = kBarEmptyK0 + kKStages, kBarSK0 = kBarReK0 + kKStages, kBarFullV0 = kBarSK0 + kKStages,
         kBarEmptyV0 = kBarFullV0 + kVStages, kBarS = kBarEmptyV0 + kVStages, kBarDP, kBarSFree, kBarDPFree,
         kBarDSFull0, kBarDSFree0 = kBarDSFull0 + kDsBufs, kBarFinal = kBarDSFree0 + kDsBufs, kBarDrain, kNumBars };
  static constexpr int kOffBar = kOffDS + kDsBufs * 2 * kBox;
  static constexpr int kOffMisc = kOffBar + 8 * kNumBars;
  static constexpr int kSmemBytes = kOffMisc + 16;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// Copies this thread's row m of a 64 x 256 bf16 tile (four 64-row boxes, 128-byte
// swizzle) into TMEM as an A operand: boxes 2 wg, 2 wg + 1 to columns 32 bx.
__device__ __forceinline__ void tile256_row_to_tmem(const uint8_t *tile, int m, int wg, uint32_t t_row) {
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int bx = 2 * wg + half;
    uint32_t w[32];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint4 v = *reinterpret_cast<const uint4 *>(tile + bx * 8192 + m * 128 + ((j ^ (m & 7)) * 16));
      w[4 * j] = v.x;
      w[4 * j + 1] = v.y;
      w[4 * j + 2] = v.z;
      w[4 * j + 3] = v.w;
    }
    tmem_st_32x32b_x32(t_row + 32 * bx, w);
  }
}

template <bool CAUSAL, bool VARLEN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(320, 1)
    bwd_dq256_pair_kernel(const __grid_constant__ BwdParams p) {
  using C = Dq256PairCfg;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  if (!check_align(sbase, p.status)) return;  // same layout in both CTAs: both return
  const uint32_t bar0 = sbase + C::kOffBar;
  auto bar = [&](int i) { return bar0 + 8u * i; };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 4);
  const WaitCtx wctx{abort_flag, p.status};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int crank = (int)cluster_ctarank();
  const int n_q = (p.N + 127) / 128;
  int rank, head;
  work_order((int)(blockIdx.x >> 1), n_q, p.B * p.H, p.sched_chunk, rank, head);
  const int it_q = CAUSAL ? n_q - 1 - rank : rank;  // causal: the longest tiles first
  const int h = head % p.H, b = head / p.H;
  const int kh = h / (p.H / p.Hkv);
  const int Npad = n_q * 128;  // row-term arrays are [B, H, Npad]
  const int q0 = it_q * 128;
  const SeqSpan sq = VARLEN ? seq_span(p.cu_seqlens, b, p.N, p.total) : SeqSpan{0, p.N, b};
  const int L = sq.len;
  if (VARLEN && q0 >= L) return;  // the tile lies past its sequence (both CTAs return)
  const int nb = CAUSAL ? it_q + 1 : (L + 127) / 128;
  const int qrow0 = q0 + 64 * crank;  // this CTA's first query row

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kNumBars; ++i) {
      const bool pair_warps = i == C::kBarQT || i == C::kBarSFree || i == C::kBarDPFree ||
                              (i >= C::kBarDSFull0 && i < C::kBarDSFull0 + C::kDsBufs);
      mbar_init(bar(i), pair_warps ? 16u : i == C::kBarCopied ? 8u : 1u);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == C::kMmaWarp) {
    tmem_alloc_pair(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish_pair();
  }
  if (warp == C::kLoadWarp && lane == 0) {
    prefetch_tmap(&p.tm_q64);
    prefetch_tmap(&p.tm_do64);
    prefetch_tmap(&p.tm_k64);
    prefetch_tmap(&p.tm_v64);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // barriers of both CTAs initialised, TMEM of both allocated
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 8) {
    const int wg = warp >> 2;
    const int r = threadIdx.x & 127;
    const int m = r & 63, hk = r >> 6;  // query row of this CTA; key half of the S / dP columns
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const int q_row = qrow0 + m;
    const size_t rw = ((size_t)b * p.H + h) * Npad + q_row;
    const float lse2 = p.lse2[rw];
    const float dlt = p.delta[rw];
    // ---- Q, dO -> TMEM (A of S, dP), row m in lanes m and 64 + m
    bool ok = mbar_wait_warp(bar(C::kBarQdo), 0, wctx, kBSiteQ);
    if (ok) {
      tile256_row_to_tmem(smem + C::kOffQTmp, m, wg, tmem + lane_off + C::kColQ);
      tile256_row_to_tmem(smem + C::kOffDOTmp, m, wg, tmem + lane_off + C::kColDO);
      tmem_wait_st();
    }
    fence_proxy_async_smem();  // both regions are refilled by TMA after this
    tc_fence_before();
    mbar_arrive_warp_cluster(mapa_shared(bar(C::kBarQT), 0));
    mbar_arrive_warp(bar(C::kBarCopied));

    const uint32_t s_tm = tmem + lane_off + C::kColS + 32 * wg;
    const uint32_t dp_tm = tmem + lane_off + C::kColDP + 32 * wg;
    const int kc0 = 64 * hk + 32 * wg;  // this thread's first key column within a key tile
    const int last_key = CAUSAL ? min(q_row, L - 1) : L - 1;
    for (int j = 0; j < nb && ok; ++j) {
      ok = mbar_wait_warp_cl(bar(C::kBarS), j & 1, wctx, kBSiteS);
      if (!ok) break;
      tc_fence_after();
      uint32_t sv[32];
      tmem_ld_32x32b_x32(s_tm, sv);
      tmem_wait_ld(sv);
      tc_fence_before();
      mbar_arrive_warp_cluster(mapa_shared(bar(C::kBarSFree), 0));  // S is in registers: S_{j+1} may overwrite it
      const int lim = last_key - (j * 128 + kc0);                   // last visible column offset
      float pe[32];
#pragma unroll
      for (int c = 0; c < 32; c += 2) {
        float x0, x1;
        ffma2(x0, x1, __uint_as_float(sv[c]), __uint_as_float(sv[c + 1]), p.scale_log2, p.scale_log2, -lse2, -lse2);
        pe[c] = ex2_mufu(x0);
        pe[c + 1] = ex2_mufu(x1);
      }
      if (lim < 31) {
#pragma unroll
        for (int c = 0; c < 32; ++c)
          if (c > lim) pe[c] = 0.f;
      }
      ok = mbar_wait_warp_cl(bar(C::kBarDP), j & 1, wctx, kBSiteDP);
      if (!ok) break;
      tc_fence_after();
      uint32_t dpv[32];
      tmem_ld_32x32b_x32(dp_tm, dpv);
      tmem_wait_ld(dpv);
      tc_fence_before();
      mbar_arrive_warp_cluster(mapa_shared(bar(C::kBarDPFree), 0));
      uint32_t wd[16];
#pragma unroll
      for (int c = 0; c < 32; c += 2) {
        float t0, t1, d0, d1;
        fadd2(t0, t1, __uint_as_float(dpv[c]), __uint_as_float(dpv[c + 1]), -dlt, -dlt);
        fmul2(d0, d1, pe[c], pe[c + 1], t0, t1);
        wd[c >> 1] = pack_bf16x2(d0, d1);
      }
      const int db = j % C::kDsBufs;
      if (j >= C::kDsBufs) {  // dQ_{j-2} has read this buffer
        ok = mbar_wait_warp_cl(bar(C::kBarDSFree0 + db), ((j / C::kDsBufs) - 1) & 1, wctx, kBSiteDSFree);
        if (!ok) break;
      }
      st_swizzled_32cols_r64(sbase + C::kOffDS + db * 2 * C::kBox, m, kc0, wd);
      fence_proxy_async_smem();
      mbar_arrive_warp_cluster(mapa_shared(bar(C::kBarDSFull0 + db), 0));
    }
    // ---- epilogue: dQ * scale -> bf16 -> shared (the K ring) -> TMA store; warpgroup wg takes 64 of its 128 columns
    if (ok) ok = mbar_wait_warp_cl(bar(C::kBarFinal), 0, wctx, kBSiteFinal);
    tc_fence_after();
    const uint32_t acc_tm = tmem + lane_off + C::kColDQ;
    const bool has_rows = qrow0 < L;
    const bool direct = VARLEN && qrow0 + 64 > L;  // the next sequence's rows follow: write row by row
    if (ok && has_rows && direct) {
      acc_to_global<64>(acc_tm, static_cast<__nv_bfloat16 *>(p.dq) + ((size_t)(sq.start + q_row) * p.H + h) * 256 +
                                    128 * hk,
                        64 * wg, p.scale, q_row < L);
    } else if (ok && has_rows) {
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(acc_tm + 64 * wg + 32 * c, v);
        tmem_wait_ld(v);
        uint32_t w[16];
#pragma unroll
        for (int k = 0; k < 16; ++k)
          w[k] = pack_bf16x2(__uint_as_float(v[2 * k]) * p.scale, __uint_as_float(v[2 * k + 1]) * p.scale);
        st_swizzled_32cols_r64(sbase + C::kOffK, m, 128 * hk + 64 * wg + 32 * c, w);
      }
    }
    fence_proxy_async_smem();
    named_bar_sync(1, 256);
    if (threadIdx.x == 0 && ok && has_rows && !direct) {
      for (int bx = 0; bx < 4; ++bx)
        tma_store_4d(&p.tm_dq64, sbase + C::kOffK + bx * C::kBox, bx * 64, h, sq.start + qrow0, sq.bc);
      bulk_commit();
      bulk_wait_read_all();
    }
  } else if (warp == C::kMmaWarp) {
    // ===================================================== MMA issue (rank-0 CTA, for both)
    if (crank == 0) {
      constexpr uint32_t id_s = make_idesc_bf16(128, 128, false, false);  // S, dP (A in TMEM)
      constexpr uint32_t id_o = make_idesc_bf16(128, 256, false, true);   // dQ (B MN-major)
      const uint64_t k_d = make_sdesc_sw128(sbase + C::kOffK, 0, 1024);
      const uint64_t k_mn = make_sdesc_sw128(sbase + C::kOffK, C::kBox, 1024);
      const uint64_t v_d = make_sdesc_sw128(sbase + C::kOffV, 0, 1024);
      const uint64_t ds_d = make_sdesc_sw128(sbase + C::kOffDS, 0, 1024);
      auto kmaj = [](int kk) { return (uint64_t)(((kk >> 2) * C::kBox + (kk & 3) * 32) >> 4); };
      auto off = [](int bytes) { return (uint64_t)(bytes >> 4); };
      bool ok = mbar_wait_warp_cl(bar(C::kBarQT), 0, wctx, kBSiteQ);
      for (int jj = 0; jj <= nb && ok; ++jj) {
        if (jj < nb) {
          const int sk = jj % C::kKStages, sv = jj % C::kVStages;
          ok = mbar_wait_warp_cl(bar(C::kBarFullK0 + sk), (jj / C::kKStages) & 1, wctx, kBSiteFull);
          if (ok && jj > 0) ok = mbar_wait_warp_cl(bar(C::kBarSFree), (jj - 1) & 1, wctx, kBSiteSL);
          if (!ok) break;
          tc_fence_after();
          if (elect_one()) {  // S = Q K^T: head-dim half kk / 8 of this CTA's key rows
#pragma unroll
            for (int kk = 0; kk < 16; ++kk)
              mma_ts_pair(tmem + C::kColS, tmem + C::kColQ + 8 * kk,
                          k_d + off(sk * C::kStage + (kk >> 3) * C::kQuarter) + kmaj(kk & 7), id_s, kk > 0);
            tc_commit_pair(bar(C::kBarS));
            tc_commit_pair(bar(C::kBarSK0 + sk));
          }
          __syncwarp();
          ok = mbar_wait_warp_cl(bar(C::kBarFullV0 + sv), (jj / C::kVStages) & 1, wctx, kBSiteFull);
          if (ok && jj > 0) ok = mbar_wait_warp_cl(bar(C::kBarDPFree), (jj - 1) & 1, wctx, kBSiteSL);
          if (!ok) break;
          tc_fence_after();
          if (elect_one()) {  // dP = dO V^T
#pragma unroll
            for (int kk = 0; kk < 16; ++kk)
              mma_ts_pair(tmem + C::kColDP, tmem + C::kColDO + 8 * kk,
                          v_d + off(sv * C::kStage + (kk >> 3) * C::kQuarter) + kmaj(kk & 7), id_s, kk > 0);
            tc_commit_pair(bar(C::kBarDP));
            tc_commit_pair(bar(C::kBarEmptyV0 + sv));
          }
          __syncwarp();
        }
        if (jj > 0) {  // dQ += dS K of the previous key tile (its second K quarter reloaded)
          const int j = jj - 1, sk = j % C::kKStages, db = j % C::kDsBufs;
          ok = mbar_wait_warp_cl(bar(C::kBarDSFull0 + db), (j / C::kDsBufs) & 1, wctx, kBSiteDS);
          if (ok) ok = mbar_wait_warp_cl(bar(C::kBarReK0 + sk), (j / C::kKStages) & 1, wctx, kBSiteFull);
          if (!ok) break;
          tc_fence_after();
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ss_pair(tmem + C::kColDQ, ds_d + off(db * 2 * C::kBox) + kmaj(kk),
                          k_mn + off(sk * C::kStage + (kk >> 2) * C::kQuarter + (kk & 3) * 2048), id_o,
                          (j > 0 || kk > 0));
            tc_commit_pair(bar(C::kBarDSFree0 + db));
            tc_commit_pair(bar(C::kBarEmptyK0 + sk));
          }
          __syncwarp();
        }
      }
      if (elect_one()) {
        tc_commit_pair(bar(C::kBarFinal));
        tc_commit_pair(bar(C::kBarDrain));
      }
      __syncwarp();
      if (!mbar_wait_warp_cl(bar(C::kBarDrain), 0, wctx, kBSiteDrain) && *abort_flag) {
        const uint64_t t0 = global_timer_ns();
        while (!mbar_test_cl(bar(C::kBarDrain), 0) && global_timer_ns() - t0 < kWaitLimitNs) {}
      }
    }
  } else {
    // ===================================================== TMA producer (both CTAs; stage bytes counted by rank 0)
    if (lane == 0) {
      const uint64_t keep = policy_evict_last();
      const uint64_t once = policy_evict_first();
      mbar_arrive_expect_tx(bar(C::kBarQdo), 8 * C::kBox);
      for (int bx = 0; bx < 4; ++bx) {
        tma_load_4d_hint(sbase + C::kOffQTmp + bx * C::kBox, &p.tm_q64, bar(C::kBarQdo), bx * 64, h, sq.start + qrow0,
                         sq.bc, once);
        tma_load_4d_hint(sbase + C::kOffDOTmp + bx * C::kBox, &p.tm_do64, bar(C::kBarQdo), bx * 64, h,
                         sq.start + qrow0, sq.bc, once);
      }
      bool ok = true;
      int nfk = 0, nrk = 0, nfv = 0;
      for (int j = 0; j <= nb && ok; ++j) {
        const int kv_row = sq.start + j * 128;
        if (j < nb) {  // K_j: this CTA's key half, both head-dim halves
          const int sk = j % C::kKStages;
          if (j == 2) {  // K stage 2 and V stage 2 held dO and Q
            ok = mbar_wait(bar(C::kBarCopied), 0, wctx, kBSiteQ);
            if (!ok) break;
          }
          ok = mbar_wait_cl(bar(C::kBarEmptyK0 + sk), ((j / C::kKStages) & 1) ^ 1, wctx, kBSiteEmpty);
          if (!ok) break;
          if (crank == 0) mbar_arrive_expect_tx(bar(C::kBarFullK0 + sk), 2 * C::kStage);
          const uint32_t fb = mapa_shared(bar(C::kBarFullK0 + sk), 0);
          for (int dh = 0; dh < 2; ++dh)
            for (int bx = 0; bx < 2; ++bx)
              tma_load_4d_pair(sbase + C::kOffK + sk * C::kStage + dh * C::kQuarter + bx * C::kBox, &p.tm_k64, fb,
                               128 * dh + 64 * bx, kh, kv_row + 64 * crank, sq.bc, keep);
          ++nfk;
        }
        if (j > 0) {  // reload for the previous tile: the other key half, this CTA's head-dim half
          const int jp = j - 1, sk = jp % C::kKStages;
          ok = mbar_wait_cl(bar(C::kBarSK0 + sk), (jp / C::kKStages) & 1, wctx, kBSiteS);  // S_jp has read the slot
          if (!ok) break;
          if (crank == 0) mbar_arrive_expect_tx(bar(C::kBarReK0 + sk), 2 * C::kQuarter);
          const uint32_t rk = mapa_shared(bar(C::kBarReK0 + sk), 0);
          for (int bx = 0; bx < 2; ++bx)
            tma_load_4d_pair(sbase + C::kOffK + sk * C::kStage + (1 - crank) * C::kQuarter + bx * C::kBox, &p.tm_k64,
                             rk, 128 * crank + 64 * bx, kh, sq.start + jp * 128 + 64 * (1 - crank), sq.bc, keep);
          ++nrk;
        }
        if (j < nb) {  // V_j: this CTA's key half, both head-dim halves
          const int sv = j % C::kVStages;
          ok = mbar_wait_cl(bar(C::kBarEmptyV0 + sv), ((j / C::kVStages) & 1) ^ 1, wctx, kBSiteEmpty);
          if (!ok) break;
          if (crank == 0) mbar_arrive_expect_tx(bar(C::kBarFullV0 + sv), 2 * C::kStage);
          const uint32_t fb = mapa_shared(bar(C::kBarFullV0 + sv), 0);
          for (int dh = 0; dh < 2; ++dh)
            for (int bx = 0; bx < 2; ++bx)
              tma_load_4d_pair(sbase + C::kOffV + sv * C::kStage + dh * C::kQuarter + bx * C::kBox, &p.tm_v64, fb,
                               128 * dh + 64 * bx, kh, kv_row + 64 * crank, sq.bc, keep);
          ++nfv;
        }
      }
      // drain: the stage barriers of rank 0 count both CTAs' copies; Q / dO are local
      const uint64_t t0 = global_timer_ns();
      auto drain = [&](int base, int stages, int n) {
        for (int u = max(0, n - stages); u < n; ++u)
          while (!mbar_test_cl(bar(base + u % stages), (u / stages) & 1) && global_timer_ns() - t0 < kWaitLimitNs) {}
      };
      if (crank == 0) {
        drain(C::kBarFullK0, C::kKStages, nfk);
        drain(C::kBarReK0, C::kKStages, nrk);
        drain(C::kBarFullV0, C::kVStages, nfv);
      }
      while (!mbar_test(bar(C::kBarQdo), 0) && global_timer_ns() - t0 < kWaitLimitNs) {}
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

// ------------------------------------------------------------------ launches
template <typename Kern>
int launch_kernel(Kern kern, dim3 grid, int threads, int smem, const BwdParams &p, cudaStream_t stream) {
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return FA_ERR_CUDA;
  kern<<<grid, threads, smem, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

template <int D>
int launch_pre_t(const BwdParams &p, const void *o, const void *dO, const float *lse, cudaStream_t stream) {
  const int Npad = (p.N + 127) / 128 * 128;
  const long long rows = (long long)p.B * Npad * p.H;
  const long long rows_per_block = 8LL * (32 / (D / 8)) * kPreIters;  // 8 warps
  bwd_pre_kernel<D><<<(unsigned)((rows + rows_per_block - 1) / rows_per_block), 256, 0, stream>>>(
      static_cast<const __nv_bfloat16 *>(o), static_cast<const __nv_bfloat16 *>(dO), lse, p.lse2,
      const_cast<float *>(p.delta), p.B, p.H, p.N, Npad, p.cu_seqlens, p.total, p.dqacc);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// Scheduling chunk of the key/value-stationary kernels: Q and dO of every
// query head of a kv group are re-read by each key tile of the group.
BwdParams with_kv_order(const BwdParams &p_in, bool causal, int d) {
  BwdParams p = p_in;
  const int g = p.H / p.Hkv;
  p.sched_chunk = sched_chunk_for(causal, (size_t)g * 2 * p.N * d * 2, p.B * p.Hkv);
  return p;
}

// Scheduling chunk of the query-stationary kernels: K and V of a kv head are
// re-read by each query tile of its query heads (kept together in a chunk).
BwdParams with_q_order(const BwdParams &p_in, bool causal, int d) {
  BwdParams p = p_in;
  const int g = p.H / p.Hkv;
  p.sched_chunk = causal ? g * sched_chunk_for(true, (size_t)2 * p.N * d * 2, p.B * p.Hkv) : 1;
  return p;
}

unsigned grid_1d(long long n_tiles, long long n_heads) {
  const long long n = n_tiles * n_heads;
  return n > 0x7fffffffLL ? 0u : (unsigned)n;  // 0: too many CTAs for a 1-D grid
}

int sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  return sms;
}

template <int D, bool CAUSAL>
int launch_dkdv_t(const BwdParams &p_in, cudaStream_t stream) {
  const BwdParams p = with_kv_order(p_in, CAUSAL, D);
  unsigned grid = grid_1d((p.N + 127) / 128, (long long)p.B * p.Hkv);
  if (!grid) return FA_ERR_UNSUPPORTED;
  if constexpr (D == 64 || D == 128) {
    const int max_n = D == 64 ? (CAUSAL ? FA_DKDV_PERSIST_MAX_N_CAUSAL : FA_DKDV_PERSIST_MAX_N)
                              : (CAUSAL ? FA_DKDV128_PERSIST_MAX_N_CAUSAL : FA_DKDV128_PERSIST_MAX_N);
    if (p.N <= max_n) {  // at most one CTA per SM
      using PC = DkdvCfg<D, true>;
      const int sms = sm_count();
      if (sms > 0 && grid > (unsigned)sms) grid = (unsigned)sms;
      return p.cu_seqlens ? launch_kernel(bwd_dkdv_kernel<D, CAUSAL, true, true>, dim3(grid), PC::kThreads,
                                          PC::kSmemBytes, p, stream)
                          : launch_kernel(bwd_dkdv_kernel<D, CAUSAL, false, true>, dim3(grid), PC::kThreads,
                                          PC::kSmemBytes, p, stream);
    }
  }
  return p.cu_seqlens
             ? launch_kernel(bwd_dkdv_kernel<D, CAUSAL, true, false>, dim3(grid), DkdvCfg<D>::kThreads,
                             DkdvCfg<D>::kSmemBytes, p, stream)
             : launch_kernel(bwd_dkdv_kernel<D, CAUSAL, false, false>, dim3(grid), DkdvCfg<D>::kThreads,
                             DkdvCfg<D>::kSmemBytes, p, stream);
}

// Head dim 128: CTA pairs, one per 256-row key tile (a final odd tile pairs
// with an empty one).
template <bool CAUSAL>
int launch_dkdv_pair_t(const BwdParams &p_in, cudaStream_t stream) {
  const BwdParams p = with_kv_order(p_in, CAUSAL, 128);
  const long long n_pairs = ((p.N + 127) / 128 + 1) / 2;
  const unsigned grid = grid_1d(2 * n_pairs, (long long)p.B * p.Hkv);
  if (!grid) return FA_ERR_UNSUPPORTED;
  return p.cu_seqlens ? launch_kernel(bwd_dkdv_pair_kernel<CAUSAL, true>, dim3(grid), DkdvPairCfg::kThreads,
                                      DkdvPairCfg::kSmemBytes, p, stream)
                      : launch_kernel(bwd_dkdv_pair_kernel<CAUSAL, false>, dim3(grid), DkdvPairCfg::kThreads,
                                      DkdvPairCfg::kSmemBytes, p, stream);
}

template <bool CAUSAL>
int launch_fused_t(const BwdParams &p_in, cudaStream_t stream) {
  const BwdParams p = with_kv_order(p_in, CAUSAL, 128);
  const long long n_pairs = ((p.N + 127) / 128 + 1) / 2;
  const unsigned grid = grid_1d(2 * n_pairs, (long long)p.B * p.Hkv);
  if (!grid) return FA_ERR_UNSUPPORTED;
  return launch_kernel(bwd_fused_pair_kernel<CAUSAL>, dim3(grid), FusedCfg::kThreads, FusedCfg::kSmemBytes, p, stream);
}

// Head dim 128: CTA pairs, one per 256-row query tile (a final odd tile pairs
// with an empty one).
template <bool CAUSAL>
int launch_dq_pair_t(const BwdParams &p_in, cudaStream_t stream) {
  const BwdParams p = with_q_order(p_in, CAUSAL, 128);
  const long long n_pairs = ((p.N + 127) / 128 + 1) / 2;
  const unsigned grid = grid_1d(2 * n_pairs, (long long)p.B * p.H);
  if (!grid) return FA_ERR_UNSUPPORTED;
  return p.cu_seqlens ? launch_kernel(bwd_dq_pair_kernel<CAUSAL, true>, dim3(grid), DqPairCfg::kThreads,
                                      DqPairCfg::kSmemBytes, p, stream)
                      : launch_kernel(bwd_dq_pair_kernel<CAUSAL, false>, dim3(grid), DqPairCfg::kThreads,
                                      DqPairCfg::kSmemBytes, p, stream);
}

template <int D, bool CAUSAL>
int launch_dq_t(const BwdParams &p_in, cudaStream_t stream) {
  const BwdParams p = with_q_order(p_in, CAUSAL, D);
  unsigned grid = grid_1d((p.N + 127) / 128, (long long)p.B * p.H);
  if (!grid) return FA_ERR_UNSUPPORTED;
  const int max_n = CAUSAL ? (D == 64 ? FA_DQ_PERSIST_MAX_N_CAUSAL : FA_DQ128_PERSIST_MAX_N_CAUSAL)
                           : (D == 64 ? FA_DQ_PERSIST_MAX_N : FA_DQ128_PERSIST_MAX_N);
  if (p.N <= max_n) {  // persistent CTAs: at most one per SM
    using PC = DqCfg<D, true>;
    const int sms = sm_count();
    if (sms > 0 && grid > (unsigned)sms) grid = (unsigned)sms;
    return p.cu_seqlens
               ? launch_kernel(bwd_dq_kernel<D, CAUSAL, true, true>, dim3(grid), PC::kThreads, PC::kSmemBytes, p, stream)
               : launch_kernel(bwd_dq_kernel<D, CAUSAL, false, true>, dim3(grid), PC::kThreads, PC::kSmemBytes, p,
                               stream);
  }
  return p.cu_seqlens
             ? launch_kernel(bwd_dq_kernel<D, CAUSAL, true, false>, dim3(grid), DqCfg<D>::kThreads, DqCfg<D>::kSmemBytes,
                             p, stream)
             : launch_kernel(bwd_dq_kernel<D, CAUSAL, false, false>, dim3(grid), DqCfg<D>::kThreads,
                             DqCfg<D>::kSmemBytes, p, stream);
}

}  // namespace

int launch_bwd_pre(const BwdParams &p, int d, const void *o, const void *dO, const float *lse, cudaStream_t stream) {
  switch (d) {
    case 64: return launch_pre_t<64>(p, o, dO, lse, stream);
    case 128: return launch_pre_t<128>(p, o, dO, lse, stream);
    case 256: return launch_pre_t<256>(p, o, dO, lse, stream);
    default: return FA_ERR_UNSUPPORTED;
  }
}

int launch_bwd_dkdv(const BwdParams &p, int d, bool causal, cudaStream_t stream) {
  switch (d) {
    case 64: return causal ? launch_dkdv_t<64, true>(p, stream) : launch_dkdv_t<64, false>(p, stream);
    case 128:
      if (FA_DKDV_PAIR && p.N > (causal ? FA_DKDV_PAIR_MIN_N_CAUSAL : FA_DKDV_PAIR_MIN_N))
        return causal ? launch_dkdv_pair_t<true>(p, stream) : launch_dkdv_pair_t<false>(p, stream);
      return causal ? launch_dkdv_t<128, true>(p, stream) : launch_dkdv_t<128, false>(p, stream);
    case 256: {
      const BwdParams q = with_kv_order(p, causal, 256);
      // pairs: (key tile, CTA of the pair); else (key tile, head-dim half)
      const unsigned n = grid_1d(2 * ((p.N + 127) / 128), (long long)p.B * p.Hkv);
      if (!n) return FA_ERR_UNSUPPORTED;
      const dim3 grid(n);
      if (FA_DKDV256_PAIR) {
        using PC = Dkdv256PairCfg;
        if (causal)
          return q.cu_seqlens ? launch_kernel(bwd_dkdv256_pair_kernel<true, true>, grid, PC::kThreads, PC::kSmemBytes,
                                              q, stream)
                              : launch_kernel(bwd_dkdv256_pair_kernel<true, false>, grid, PC::kThreads,
                                              PC::kSmemBytes, q, stream);
        return q.cu_seqlens ? launch_kernel(bwd_dkdv256_pair_kernel<false, true>, grid, PC::kThreads, PC::kSmemBytes,
                                            q, stream)
                            : launch_kernel(bwd_dkdv256_pair_kernel<false, false>, grid, PC::kThreads, PC::kSmemBytes,
                                            q, stream);
      }
      if (causal)
        return q.cu_seqlens ? launch_kernel(bwd_dkdv256_kernel<true, true>, grid, Dkdv256Cfg<true>::kThreads,
                                            Dkdv256Cfg<true>::kSmemBytes, q, stream)
                            : launch_kernel(bwd_dkdv256_kernel<true, false>, grid, Dkdv256Cfg<true>::kThreads,
                                            Dkdv256Cfg<true>::kSmemBytes, q, stream);
      return q.cu_seqlens ? launch_kernel(bwd_dkdv256_kernel<false, true>, grid, Dkdv256Cfg<false>::kThreads,
                                          Dkdv256Cfg<false>::kSmemBytes, q, stream)
                          : launch_kernel(bwd_dkdv256_kernel<false, false>, grid, Dkdv256Cfg<false>::kThreads,
                                          Dkdv256Cfg<false>::kSmemBytes, q, stream);
    }
    default: return FA_ERR_UNSUPPORTED;
  }
}

int launch_bwd_fused(const BwdParams &p, bool causal, cudaStream_t stream) {
  if (p.dqacc == nullptr || p.cu_seqlens != nullptr) return FA_ERR_UNSUPPORTED;
  return causal ? launch_fused_t<true>(p, stream) : launch_fused_t<false>(p, stream);
}

int launch_bwd_post(const BwdParams &p, int d, cudaStream_t stream) {
  const long long n8 = (long long)p.B * p.N * p.H * d / 8;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return FA_ERR_CUDA;
  const long long want = (n8 + 255) / 256;
  const int blocks = (int)(want < (long long)sms * 8 ? want : (long long)sms * 8);
  if (blocks > 0)
    bwd_post_kernel<<<blocks, 256, 0, stream>>>(p.dqacc, static_cast<__nv_bfloat16 *>(p.dq), n8, p.scale);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int launch_bwd_dq(const BwdParams &p, int d, bool causal, cudaStream_t stream) {
  switch (d) {
    case 64: return causal ? launch_dq_t<64, true>(p, stream) : launch_dq_t<64, false>(p, stream);
    case 128:
      if (FA_DQ_PAIR) return causal ? launch_dq_pair_t<true>(p, stream) : launch_dq_pair_t<false>(p, stream);
      return causal ? launch_dq_t<128, true>(p, stream) : launch_dq_t<128, false>(p, stream);
    case 256: {
      const BwdParams q = with_q_order(p, causal, 256);
      const unsigned n = grid_1d((p.N + 127) / 128, (long long)p.B * p.H);
      if (!n) return FA_ERR_UNSUPPORTED;
      if (FA_DQ256_PAIR) {
        using PC = Dq256PairCfg;
        const unsigned n2 = grid_1d(2 * ((p.N + 127) / 128), (long long)p.B * p.H);  // (query tile, CTA of the pair)
        if (!n2) return FA_ERR_UNSUPPORTED;
        if (causal)
          return q.cu_seqlens ? launch_kernel(bwd_dq256_pair_kernel<true, true>, dim3(n2), PC::kThreads,
                                              PC::kSmemBytes, q, stream)
                              : launch_kernel(bwd_dq256_pair_kernel<true, false>, dim3(n2), PC::kThreads,
                                              PC::kSmemBytes, q, stream);
        return q.cu_seqlens ? launch_kernel(bwd_dq256_pair_kernel<false, true>, dim3(n2), PC::kThreads, PC::kSmemBytes,
                                            q, stream)
                            : launch_kernel(bwd_dq256_pair_kernel<false, false>, dim3(n2), PC::kThreads,
                                            PC::kSmemBytes, q, stream);
      }
      const dim3 grid(n);
      if (causal)
        return q.cu_seqlens ? launch_kernel(bwd_dq256_kernel<true, true>, grid, Dq256Cfg::kThreads, Dq256Cfg::kSmemBytes,
                                            q, stream)
                            : launch_kernel(bwd_dq256_kernel<true, false>, grid, Dq256Cfg::kThreads,
                                            Dq256Cfg::kSmemBytes, q, stream);
      return q.cu_seqlens ? launch_kernel(bwd_dq256_kernel<false, true>, grid, Dq256Cfg::kThreads,
                                          Dq256Cfg::kSmemBytes, q, stream)
                          : launch_kernel(bwd_dq256_kernel<false, false>, grid, Dq256Cfg::kThreads,
                                          Dq256Cfg::kSmemBytes, q, stream);
    }
    default: return FA_ERR_UNSUPPORTED;
  }
}

#ifdef FA_TEST_STALL
int set_test_stall_bwd(int mode) {
  return cudaMemcpyToSymbol(g_test_stall, &mode, sizeof(int)) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}
#endif

}  // namespace fa

#ifdef FA_TRACE
extern "C" int fa_debug_trace(unsigned long long *host_out) {
  return cudaMemcpyFromSymbol(host_out, fa::g_trace, sizeof(fa::g_trace)) == cudaSuccess ? 0 : -5;
}
// life: 2 x 16 SM-clock stamps; ctas: 2 x 65536 x {smid, entry ns, exit ns}
extern "C" int fa_debug_trace_ctas(unsigned long long *life, unsigned long long *ctas) {
  if (cudaMemcpyFromSymbol(life, fa::g_life, sizeof(fa::g_life)) != cudaSuccess) return -5;
  return cudaMemcpyFromSymbol(ctas, fa::g_cta, sizeof(fa::g_cta)) == cudaSuccess ? 0 : -5;
}
#endif
