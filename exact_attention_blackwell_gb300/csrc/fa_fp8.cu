// fa_fp8.cu — FP8 (e4m3) attention forward with incoherent processing, sm_103a.
//
// The FlashAttention-3 page, section 3 ("Baja precision (FP8) con reduccion del
// error de cuantizacion"), gives the method: multiply the query and key
// feature vectors by a random orthogonal matrix (a Hadamard matrix, for
// example) so that outlier coordinates spread over all coordinates, then
// quantize to FP8; the orthogonal factor cancels in Q K^T.  Here:
//   * M = diag(signs) H_128 / sqrt(128) (signs: a +-1 vector from the caller,
//     or no rotation at all), applied to every row of Q and K by an in-register
//     fast Walsh-Hadamard transform;
//   * e4m3 with one fp32 scale per 128-row block of one (batch, head) for Q and
//     K, and one per (batch, kv head) for V (not rotated), the block's largest
//     magnitude mapped to 448 (round to nearest even, saturating);
//   * V is stored transposed (keys contiguous) so that both products read
//     K-major operands;
//   * the forward kernel multiplies e4m3 operands on the tensor core
//     (tcgen05 kind::f8f6f4, fp32 accumulation in TMEM), folds the scales into
//     the softmax's scale-shift, rounds P to e4m3 in shared memory for the P V
//     product, keeps the row sum in fp32 from the unrounded P, and writes O
//     (bf16) and LSE (natural log) like the bf16 forward.
// Three launches: fp8_prep_qk_kernel (Q, K blocks and the V block maxima),
// fp8_prep_v_kernel (V per kv head, transposed), fa_fwd_fp8_kernel.
#include <cuda_bf16.h>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

// P of the P V product: in TMEM over S's columns (1, the default; the MMA reads
// its A operand from TMEM) or in a shared-memory tile (0).
#ifndef FA_FP8_P_TMEM
#define FA_FP8_P_TMEM 1
#endif

constexpr int kD = 128;           // head dim of the FP8 path
constexpr float kE4m3Max = 448.f;

// Two floats to packed e4m3 (lo in the low byte), round to nearest even, saturating.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  return e4m3x2(a, b) | (e4m3x2(c, d) << 16);
}

// In-register fast Walsh-Hadamard transform of 128 values (natural order):
// 7 stages of 64 butterflies; stage s pairs index i with i + 2^s, where i runs
// over the indices whose bit s is clear.
__device__ __forceinline__ void fwht128(float (&x)[kD]) {
#pragma unroll
  for (int s = 0; s < 7; ++s) {
#pragma unroll
    for (int j = 0; j < kD / 2; ++j) {
      const int i = ((j >> s) << (s + 1)) | (j & ((1 << s) - 1));
      const float a = x[i], b = x[i + (1 << s)];
      x[i] = a + b;
      x[i + (1 << s)] = a - b;
    }
  }
}

__device__ __forceinline__ float block_max128(float v, float *red) {
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, s));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  const float m = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
  __syncthreads();
  return m;
}

__device__ __forceinline__ void load_row_bf16(const __nv_bfloat16 *src, bool valid, float (&x)[kD]) {
#pragma unroll
  for (int v = 0; v < kD / 8; ++v) {
    uint4 u = valid ? reinterpret_cast<const uint4 *>(src)[v] : make_uint4(0u, 0u, 0u, 0u);
    const __nv_bfloat162 *p2 = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      x[8 * v + 2 * w] = __low2float(p2[w]);
      x[8 * v + 2 * w + 1] = __high2float(p2[w]);
    }
  }
}

// ------------------------------------------------------------------ prepare: Q, K blocks; V block maxima
// One CTA (128 threads, one per row) per 128-row block of one (batch, head) of
// Q, then of K, then of V.
__global__ void __launch_bounds__(128) fp8_prep_qk_kernel(const Fp8PrepParams p) {
  __shared__ float sgn[kD];
  __shared__ float red[4];
  const int r = threadIdx.x;
  long long L = blockIdx.x;
  const long long nq = (long long)p.B * p.H * p.nt, nk = (long long)p.B * p.Hkv * p.nt;
  int kind = 0;  // 0: Q, 1: K, 2: V
  if (L >= nq) {
    L -= nq;
    kind = 1;
    if (L >= nk) {
      L -= nk;
      kind = 2;
    }
  }
  const int Hx = kind == 0 ? p.H : p.Hkv;
  const int t = (int)(L % p.nt);
  const int head = (int)((L / p.nt) % Hx);
  const int b = (int)(L / ((long long)p.nt * Hx));
  const bool rot = p.signs != nullptr && kind < 2;
  if (rot) sgn[r] = p.signs[r];
  __syncthreads();
  const int n = t * 128 + r;
  const bool valid = n < p.N;
  const __nv_bfloat16 *src = (kind == 0 ? p.q : kind == 1 ? p.k : p.v) + (((size_t)b * p.N + n) * Hx + head) * kD;
  float x[kD];
  load_row_bf16(src, valid, x);
  if (rot) {
#pragma unroll
    for (int i = 0; i < kD; ++i) x[i] *= sgn[i];
    fwht128(x);
    const float norm = 0.088388347648318440f;  // 1 / sqrt(128)
#pragma unroll
    for (int i = 0; i < kD; ++i) x[i] *= norm;
  }
  float am = 0.f;
#pragma unroll
  for (int i = 0; i < kD; ++i) am = fmaxf(am, fabsf(x[i]));
  const float amax = block_max128(am, red);
  const size_t si = ((size_t)b * Hx + head) * p.nt + t;
  if (kind == 2) {
    if (r == 0) p.vblk[si] = amax;
    return;
  }
  const float inv = amax > 0.f ? kE4m3Max / amax : 1.f;
  if (r == 0) (kind == 0 ? p.sq : p.sk)[si] = amax > 0.f ? amax / kE4m3Max : 1.f;
  if (valid) {
    uint4 *dst = reinterpret_cast<uint4 *>((kind == 0 ? p.q8 : p.k8) + (((size_t)b * p.N + n) * Hx + head) * kD);
#pragma unroll
    for (int c = 0; c < kD / 16; ++c) {
      const float *y = x + 16 * c;
      dst[c] = make_uint4(e4m3x4(y[0] * inv, y[1] * inv, y[2] * inv, y[3] * inv),
                          e4m3x4(y[4] * inv, y[5] * inv, y[6] * inv, y[7] * inv),
                          e4m3x4(y[8] * inv, y[9] * inv, y[10] * inv, y[11] * inv),
                          e4m3x4(y[12] * inv, y[13] * inv, y[14] * inv, y[15] * inv));
    }
  }
}

// ------------------------------------------------------------------ prepare: V per kv head, transposed
// One CTA per 128-row block of one (batch, kv head): the head's scale from the
// block maxima, the block quantized into shared memory, then written out as
// 128 rows of V^T (one per head-dim column, keys contiguous; keys >= N zero).
__global__ void __launch_bounds__(128) fp8_prep_v_kernel(const Fp8PrepParams p) {
  __shared__ __align__(16) uint8_t tile[128][kD + 16];
  __shared__ float red[4];
  const int r = threadIdx.x;
  const int t = (int)(blockIdx.x % p.nt);
  const int kh = (int)((blockIdx.x / p.nt) % p.Hkv);
  const int b = (int)(blockIdx.x / ((long long)p.nt * p.Hkv));
  const size_t hb = (size_t)b * p.Hkv + kh;
  float am = 0.f;
  for (int i = r; i < p.nt; i += 128) am = fmaxf(am, p.vblk[hb * p.nt + i]);
  const float amax = block_max128(am, red);
  const float inv = amax > 0.f ? kE4m3Max / amax : 1.f;
  if (t == 0 && r == 0) p.sv[hb] = amax > 0.f ? amax / kE4m3Max : 1.f;
  const int n = t * 128 + r;
  float x[kD];
  load_row_bf16(p.v + (((size_t)b * p.N + n) * p.Hkv + kh) * kD, n < p.N, x);
#pragma unroll
  for (int c = 0; c < kD / 16; ++c) {
    const float *y = x + 16 * c;
    *reinterpret_cast<uint4 *>(&tile[r][16 * c]) =
        make_uint4(e4m3x4(y[0] * inv, y[1] * inv, y[2] * inv, y[3] * inv),
                   e4m3x4(y[4] * inv, y[5] * inv, y[6] * inv, y[7] * inv),
                   e4m3x4(y[8] * inv, y[9] * inv, y[10] * inv, y[11] * inv),
                   e4m3x4(y[12] * inv, y[13] * inv, y[14] * inv, y[15] * inv));
  }
  __syncthreads();
  // thread r now writes head-dim column r: keys 128 t .. 128 t + 127
  uint32_t w[32];
#pragma unroll
  for (int i = 0; i < 32; ++i)
    w[i] = (uint32_t)tile[4 * i][r] | ((uint32_t)tile[4 * i + 1][r] << 8) | ((uint32_t)tile[4 * i + 2][r] << 16) |
           ((uint32_t)tile[4 * i + 3][r] << 24);
  uint4 *dst = reinterpret_cast<uint4 *>(p.vt8 + (hb * kD + r) * (size_t)p.Npad + (size_t)t * 128);
#pragma unroll
  for (int c = 0; c < 8; ++c) dst[c] = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
}

// ------------------------------------------------------------------ forward
struct Fp8Cfg {
  static constexpr int kQT = 2;           // query tiles per CTA
  static constexpr int kStages = 8;       // K / V^T ring slots (16 KB e4m3 tiles)
  static constexpr int kTile = 128 * kD;  // bytes of one 128 x 128 e4m3 tile
  static constexpr int kThreads = 320;
  static constexpr int kMmaWarp = 8, kLoadWarp = 9;
  static constexpr int kOCol = 256;  // TMEM: S_t at 128 t, O_t at 256 + 128 t
  static constexpr int kTmemCols = 512;
  static constexpr int kOffQ = 0;
  static constexpr int kOffP = kQT * kTile;
  static constexpr int kOffRing = 2 * kQT * kTile;
  static constexpr int kOffBar = kOffRing + kStages * kTile;
  static constexpr int kNumBars = 2 * kStages + 2 + 3 * kQT;  // full, empty, q, s[QT], p[QT], o[QT], drain
  static constexpr int kOffMisc = kOffBar + 8 * kNumBars;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + alignment slack
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

enum Fp8Site : int { kF8Q = 31, kF8K = 32, kF8V = 33, kF8P = 34, kF8Empty = 35, kF8S = 36, kF8O = 37, kF8Drain = 38 };

// A from TMEM (M rows = lanes, four e4m3 per 32-bit column), B from shared memory.
__device__ __forceinline__ void mma_f8_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                          uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(acc)
      : "memory");
}

template <bool CAUSAL>
__global__ void __launch_bounds__(Fp8Cfg::kThreads, 1) fa_fwd_fp8_kernel(const __grid_constant__ Fp8Params p) {
  using C = Fp8Cfg;
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

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_groups = (p.N + 128 * QT - 1) / (128 * QT);
  int rank, head;
  work_order((int)blockIdx.x, n_groups, p.B * p.H, p.sched_chunk, rank, head);
  const int group = CAUSAL ? n_groups - 1 - rank : rank;  // causal: the longest query rows first
  const int h = head % p.H, b = head / p.H;
  const int kh = h / (p.H / p.Hkv);
  const int n_kv_all = (p.N + 127) / 128;
  int q0[QT], nb[QT];
  int nb_max = 0;
#pragma unroll
  for (int t = 0; t < QT; ++t) {
    q0[t] = (group * QT + t) * 128;
    if (q0[t] >= p.N) nb[t] = 0;
    else nb[t] = CAUSAL ? (min(q0[t] + 127, p.N - 1) / 128 + 1) : n_kv_all;
    nb_max = max(nb_max, nb[t]);
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kNumBars; ++i) {
      const uint32_t bar = bar0 + 8u * i;
      const bool is_p = bar >= p_bar(0) && bar < p_bar(0) + 8u * QT;
      mbar_init(bar, is_p ? 128u : 1u);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == C::kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  if (warp == C::kLoadWarp && lane == 0) {
    prefetch_tmap(&p.tm_q8);
    prefetch_tmap(&p.tm_k8);
    prefetch_tmap(&p.tm_vt8);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4 * QT) {
    // ===================================================== softmax warpgroups (one thread per query row)
    const int t = warp >> 2;
    const int r = threadIdx.x & 127;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t s_tm = tmem + lane_off + 128u * t;
    const uint32_t o_tm = tmem + lane_off + C::kOCol + 128u * t;
#if !FA_FP8_P_TMEM
    uint8_t *prow = smem + C::kOffP + t * C::kTile + r * 128;  // this row of P_t (128 keys, e4m3, swizzled)
#endif
    const int q_row = q0[t] + r;
    const size_t kblk = ((size_t)b * p.Hkv + kh) * p.nt;
    // S = (Q8 K8^T) sq sk: the block scales join the softmax scale in one coefficient
    const float c2q = nb[t] > 0 ? p.scale_log2 * p.sq[((size_t)b * p.H + h) * p.nt + q0[t] / 128] : 0.f;
    float m_ref = -INFINITY, l_sum = 0.f;
    bool ok = true;
    unsigned rescales = 0;
    for (int j = 0; j < nb[t] && ok; ++j) {
      const float coef = c2q * p.sk[kblk + j];
      ok = mbar_wait_warp(s_bar(t), j & 1, wctx, kF8S);
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
      if ((kv0 + 128 > p.N) || (CAUSAL && kv0 + 127 > q0[t])) {
        const int lim = CAUSAL ? min(p.N - 1, q_row) - kv0 : p.N - 1 - kv0;
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
      const float m_blk = fmax3(mx0, mx1, fmaxf(mx2, mx3)) * coef;
      if (j == 0) {
        m_ref = m_blk;
      } else {
        const bool need = (m_blk - m_ref) > kRescaleTau;
        if (__any_sync(0xffffffffu, need)) {
          const float m_new = fmaxf(m_ref, m_blk);
          const float alpha = ex2_mufu(m_ref - m_new);
          m_ref = m_new;
          l_sum *= alpha;
#pragma unroll 1
          for (int c = 0; c < kD / 16; ++c) {
            uint32_t o[16];
            tmem_ld_32x32b_x16(o_tm + 16 * c, o);
            tmem_wait_ld(o);
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st_32x32b_x16(o_tm + 16 * c, o);
          }
          tmem_wait_st();
          rescales += (lane == 0);
        }
      }
      const float neg_m = -m_ref;
      float l0 = 0.f, l1 = 0.f, l2 = 0.f, l3 = 0.f;
      // p = 2^(s coef - m) <= 2^tau, rounded to e4m3 for the P V product; the row
      // sum takes the unrounded p
      uint32_t pw[32];  // 128 keys, four e4m3 per word, key order
#pragma unroll
      for (int chunk = 0; chunk < 8; ++chunk) {  // 16 keys per 16-byte chunk
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int c = 16 * chunk + 4 * q4;
          float x[4], e[4];
          ffma2(x[0], x[1], s[c], s[c + 1], coef, coef, neg_m, neg_m);
          ffma2(x[2], x[3], s[c + 2], s[c + 3], coef, coef, neg_m, neg_m);
#pragma unroll
          for (int u = 0; u < 4; ++u) e[u] = ex2_mufu(x[u]);
          fadd2(l0, l1, l0, l1, e[0], e[1]);
          fadd2(l2, l3, l2, l3, e[2], e[3]);
          pw[4 * chunk + q4] = e4m3x4(e[0], e[1], e[2], e[3]);
        }
#if !FA_FP8_P_TMEM
        *reinterpret_cast<uint4 *>(prow + ((chunk ^ (r & 7)) << 4)) =
            make_uint4(pw[4 * chunk], pw[4 * chunk + 1], pw[4 * chunk + 2], pw[4 * chunk + 3]);
#endif
      }
      l_sum += (l0 + l1) + (l2 + l3);
#if FA_FP8_P_TMEM
      // P_t over the first 32 of S_t's columns (read already): the A operand of
      // PV_t,j; S_t,j+1 overwrites them only after PV_t,j (the tensor pipe runs
      // one thread's MMAs in order)
      tmem_st_32x32b_x32(s_tm, pw);
      tmem_wait_st();
#else
      fence_proxy_async_smem();  // P_t (generic stores) becomes visible to the tensor core
#endif
      tc_fence_before();  // and so do the O rescale's TMEM stores
      mbar_arrive(p_bar(t));
    }
    // ----------------------------------------------------- epilogue: O sv / l -> bf16, row by row
    if (nb[t] > 0) {
      if (ok) ok = mbar_wait_warp(o_bar(t), 0, wctx, kF8O);
      tc_fence_after();
      if (ok) {
        const float mul = p.sv[(size_t)b * p.Hkv + kh] / l_sum;
        uint4 *orow = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.o) +
                                                (((size_t)b * p.N + q_row) * p.H + h) * kD);
#pragma unroll
        for (int c = 0; c < kD / 32; ++c) {
          uint32_t o[32];
          tmem_ld_32x32b_x32(o_tm + 32 * c, o);
          tmem_wait_ld(o);
          uint32_t wv[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) wv[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * mul, __uint_as_float(o[2 * i + 1]) * mul);
          if (q_row < p.N) {
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) orow[4 * c + k4] = make_uint4(wv[4 * k4], wv[4 * k4 + 1], wv[4 * k4 + 2], wv[4 * k4 + 3]);
          }
        }
        if (p.lse != nullptr && q_row < p.N)
          p.lse[((size_t)b * p.H + h) * p.N + q_row] = (m_ref + __log2f(l_sum)) * 0.69314718055994531f;
      }
    }
    if (rescales) atomicAdd(p.status + 2, rescales);
  } else if (warp == C::kMmaWarp) {
    // ===================================================== MMA issue (warp-wide, elected lane issues)
    // Per key block j: PV_0,j S_0,j+1 PV_1,j S_1,j+1; both products read K-major
    // e4m3 tiles (Q, K: rows x head dim; P: query rows x keys; V^T: head dim x keys).
    constexpr uint32_t idesc = (1u << 4) | ((128u >> 3) << 17) | ((128u >> 4) << 24);  // f32 D, e4m3 A and B
    const uint64_t q_desc0 = make_sdesc_sw128(sbase + C::kOffQ, 0, 1024);
    const uint64_t p_desc0 = make_sdesc_sw128(sbase + C::kOffP, 0, 1024);
    const uint64_t ring_desc = make_sdesc_sw128(sbase + C::kOffRing, 0, 1024);
    constexpr uint64_t kTileStep = (uint64_t)(C::kTile >> 4);
    auto slot_of = [&](int fill) { return fill % C::kStages; };
    auto par_of = [&](int fill) { return (uint32_t)((fill / C::kStages) & 1); };
    auto issue_s = [&](int t, int slot) {
      const uint64_t kd = ring_desc + (uint64_t)slot * kTileStep;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) mma_f8(tmem + 128u * t, q_desc0 + t * kTileStep + 2 * kk, kd + 2 * kk, idesc, kk > 0);
    };
    auto issue_pv = [&](int t, int slot, bool acc) {
      const uint64_t vd = ring_desc + (uint64_t)slot * kTileStep;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
#if FA_FP8_P_TMEM
        mma_f8_ts(tmem + C::kOCol + 128u * t, tmem + 128u * t + 8u * kk, vd + 2 * kk, idesc, (acc || kk > 0));
#else
        mma_f8(tmem + C::kOCol + 128u * t, p_desc0 + t * kTileStep + 2 * kk, vd + 2 * kk, idesc, (acc || kk > 0));
#endif
    };
    bool ok = nb_max > 0;
    if (ok) ok = mbar_wait_warp(q_bar, 0, wctx, kF8Q);
    if (ok) ok = mbar_wait_warp(full_bar(slot_of(0)), par_of(0), wctx, kF8K);
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
    }
    for (int j = 0; j < nb_max && ok; ++j) {
      const int fv = 2 * j + 1, fk = 2 * j + 2;
      ok = mbar_wait_warp(full_bar(slot_of(fv)), par_of(fv), wctx, kF8V);
      if (!ok) break;
      tc_fence_after();
      bool k_next = false;
      for (int t = 0; t < QT && ok; ++t) {
        if (j >= nb[t]) continue;
        ok = mbar_wait_warp(p_bar(t), j & 1, wctx, kF8P);
        if (!ok) break;
        tc_fence_after();
        if (elect_one()) issue_pv(t, slot_of(fv), j > 0);
        __syncwarp();
        if (j + 1 < nb[t]) {
          if (!k_next) {
            ok = mbar_wait_warp(full_bar(slot_of(fk)), par_of(fk), wctx, kF8K);
            if (!ok) break;
            tc_fence_after();
            k_next = true;
          }
          if (elect_one()) {
            issue_s(t, slot_of(fk));
            tc_commit(s_bar(t));
          }
          __syncwarp();
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
    if (elect_one()) tc_commit(drain_bar);
    __syncwarp();
    if (!mbar_wait_warp(drain_bar, 0, wctx, kF8Drain) && *abort_flag) {
      const uint64_t t0 = global_timer_ns();
      while (!mbar_test(drain_bar, 0) && global_timer_ns() - t0 < kWaitLimitNs) {}
    }
  } else {
    // ===================================================== TMA producer: Q tiles, then K_j, V^T_j through the ring
    if (lane == 0 && nb_max > 0) {
      const uint64_t keep = policy_evict_last();
      const uint64_t once = policy_evict_first();
      int nq = 0;
      for (int t = 0; t < QT; ++t) nq += (nb[t] > 0);
      mbar_arrive_expect_tx(q_bar, nq * C::kTile);
      for (int t = 0; t < QT; ++t)
        if (nb[t] > 0) tma_load_4d_hint(sbase + C::kOffQ + t * C::kTile, &p.tm_q8, q_bar, 0, h, q0[t], b, once);
      bool ok = true;
      int fill = 0;
      for (int j = 0; j < nb_max && ok; ++j) {
        for (int kv = 0; kv < 2 && ok; ++kv, ++fill) {
          const int s = fill % C::kStages;
          ok = mbar_wait(empty_bar(s), ((fill / C::kStages) & 1) ^ 1, wctx, kF8Empty);
          if (!ok) break;
          mbar_arrive_expect_tx(full_bar(s), C::kTile);
          const uint32_t dst = sbase + C::kOffRing + s * C::kTile;
          if (kv == 0) tma_load_4d_hint(dst, &p.tm_k8, full_bar(s), 0, kh, j * 128, b, keep);
          else tma_load_4d_hint(dst, &p.tm_vt8, full_bar(s), j * 128, 0, kh, b, keep);
        }
      }
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
}

template <bool CAUSAL>
int launch_fwd_fp8_t(const Fp8Params &p_in, cudaStream_t stream) {
  using C = Fp8Cfg;
  auto kern = fa_fwd_fp8_kernel<CAUSAL>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) != cudaSuccess)
    return FA_ERR_CUDA;
  const long long n_groups = (p_in.N + 128 * C::kQT - 1) / (128 * C::kQT);
  const long long n_ctas = n_groups * p_in.H * p_in.B;
  if (n_ctas > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  Fp8Params p = p_in;
  const int g = p.H / p.Hkv;
  p.sched_chunk = CAUSAL ? g * sched_chunk_for(true, (size_t)2 * p.N * kD, p.B * p.Hkv) : 1;
  kern<<<(unsigned)n_ctas, C::kThreads, C::kSmemBytes, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

int launch_fp8_prepare(const Fp8PrepParams &p, cudaStream_t stream) {
  const long long blocks = (long long)p.B * p.nt * (p.H + 2LL * p.Hkv);
  const long long vblocks = (long long)p.B * p.nt * p.Hkv;
  if (blocks > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  fp8_prep_qk_kernel<<<(unsigned)blocks, 128, 0, stream>>>(p);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
  fp8_prep_v_kernel<<<(unsigned)vblocks, 128, 0, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int launch_fwd_fp8(const Fp8Params &p, bool causal, cudaStream_t stream) {
  return causal ? launch_fwd_fp8_t<true>(p, stream) : launch_fwd_fp8_t<false>(p, stream);
}

}  // namespace fa
