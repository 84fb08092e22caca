// fa_internal.h — declarations shared by the translation units of the library
// (not part of the public C ABI in include/fa.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include <cuda_bf16.h>

#include "../../include/fa.h"

namespace fa {

// Software-exp2 share: of every 16 score columns, this many are exponentiated
// with the FMA-pipe polynomial and the rest with MUFU.EX2.
#ifndef FA_FWD_POLY_PER16
#define FA_FWD_POLY_PER16 0
#endif

// Conditional-rescale threshold tau, log2 units (FlashAttention-4 paper
// summary, section 2.B: rescale only when the running maximum moves by more
// than a threshold; the pages give no value).  A build-time define so that a
// tau = 0 build (rescale whenever the maximum moves) can be checked against the
// default; the result is the same up to rounding for every tau.
#ifndef FA_RESCALE_TAU
#define FA_RESCALE_TAU 8.0f
#endif
constexpr float kRescaleTau = FA_RESCALE_TAU;

struct FwdParams {
  CUtensorMap tm_q;  // [B, N, H, d] bf16, box 128 rows x 64 cols, 128B swizzle
  CUtensorMap tm_k;  // [B, N, Hkv, d]
  CUtensorMap tm_v;  // [B, N, Hkv, d]
  CUtensorMap tm_o;  // [B, N, H, d] (store)
  CUtensorMap tm_k64;  // K in boxes of 64 rows (CTA-pair kernels)
  float *lse;        // [B, H, N] or nullptr
  unsigned *status;  // device status word: [0] error bits, [1] failing site, [2] rescale count
  int B, H, Hkv, N;
  float scale_log2;  // scale * log2(e)
  int sched_chunk;   // heads per scheduling chunk (see work_order)
  // Packed variable-length batch (nullptr: B sequences of N rows each).  With a
  // table, N is the longest sequence, tensors are [total, Hx, d] (the tensor
  // maps see them as one batch of `total` rows) and lse is [H, total].
  const int *cu_seqlens;
  int total;
  void *o;  // output rows of partial varlen tiles are written directly
};

struct BwdParams {
  CUtensorMap tm_q, tm_k, tm_v, tm_do;  // loads
  CUtensorMap tm_q64, tm_do64;          // the same tensors in boxes of 64 rows (CTA-pair kernels)
  CUtensorMap tm_k64, tm_v64;           // K, V in boxes of 64 rows (CTA-pair kernels)
  CUtensorMap tm_dk, tm_dv;             // stores [B, N, Hkv, d]
  CUtensorMap tm_dk64, tm_dv64;         // the same in boxes of 64 rows (head-dim-256 CTA-pair dK/dV kernel)
  CUtensorMap tm_dq;                    // store [B, N, H, d]
  CUtensorMap tm_dq64;                  // the same in boxes of 64 rows (head-dim-256 CTA-pair dQ kernel)
  float *lse2;                          // [B, H, Npad] LSE * log2(e) (workspace)
  const float *delta;                   // [B, H, Npad] D = rowsum(dO * O) (workspace)
  unsigned *status;
  int B, H, Hkv, N;
  float scale;       // softmax scale
  float scale_log2;  // scale * log2(e)
  int sched_chunk;   // heads per scheduling chunk (see work_order)
  const int *cu_seqlens;  // as in FwdParams
  int total;
  void *dq, *dk, *dv;  // rows of partial varlen tiles are written directly
  float *dqacc;        // [B, N, H, d] fp32 dQ accumulator of the fused backward (workspace), else nullptr
};

// Rows of sequence b: the first one's index in the tensor's row dimension, the
// length, and the batch coordinate of the tensor maps.  A table entry outside
// its contract is clamped to [0, N] rows inside [0, total), so it can give
// wrong numbers but never an out-of-bounds access.
struct SeqSpan {
  int start, len, bc;
};

// CTA order of the main kernels.  Each launch is a 1-D grid of n_heads x
// n_tiles CTAs; the hardware starts them roughly in index order.  Heads are
// taken in chunks of `chunk`; inside a chunk the tile rank is the slow index,
// so the chunk's heads run side by side.  Rank 0 is each kernel's heaviest
// tile under the causal mask, so the short tiles fill the tail of the launch.
// The chunk is sized so that the tensors every tile of a head re-reads (K and
// V, or Q and dO) stay in L2 while the chunk runs; chunk = 1 gives plain
// head-major order with tiles in rank order (used without the causal mask,
// where all tiles cost the same).
constexpr size_t kSchedL2Budget = 32ull << 20;

inline int sched_chunk_for(bool causal, size_t reused_bytes_per_head, int n_heads) {
  if (!causal || n_heads <= 1) return 1;
  size_t c = kSchedL2Budget / (reused_bytes_per_head ? reused_bytes_per_head : 1);
  if (c < 1) c = 1;
  if (c > (size_t)n_heads) c = (size_t)n_heads;
  return (int)c;
}

#ifdef __CUDACC__
__device__ __forceinline__ SeqSpan seq_span(const int *cu, int b, int N, int total) {
  if (cu == nullptr) return SeqSpan{0, N, b};
  int s0 = cu[b], s1 = cu[b + 1];
  s0 = max(0, min(s0, total));
  const int len = max(0, min(s1 - s0, min(N, total - s0)));
  return SeqSpan{s0, len, 0};
}

__device__ __forceinline__ void work_order(int L, int n_tiles, int n_heads, int chunk, int &rank, int &head) {
  const int per_chunk = chunk * n_tiles;
  const int c = L / per_chunk;
  const int r = L - c * per_chunk;
  const int hc = min(chunk, n_heads - c * chunk);  // the last chunk may be short
  rank = r / hc;
  head = c * chunk + (r - rank * hc);
}
#endif

// FP8 forward (head dim 128).  Prepare: Q, K rotated and quantized to e4m3 per
// 128-row block of one (batch, head); V quantized per (batch, kv head) and
// stored transposed.  Layouts (bytes / fp32 arrays, all in the caller's workspace):
//   q8 [B, N, H, 128], k8 [B, N, Hkv, 128], vt8 [B, Hkv, 128, Npad] (keys contiguous, zero past N),
//   sq [B, H, nt], sk [B, Hkv, nt], vblk [B, Hkv, nt] (V block maxima), sv [B, Hkv];  nt = Npad / 128.
struct Fp8PrepParams {
  const __nv_bfloat16 *q, *k, *v;
  const float *signs;  // [128] of +-1, or nullptr: no rotation
  uint8_t *q8, *k8, *vt8;
  float *sq, *sk, *vblk, *sv;
  int B, H, Hkv, N, nt, Npad;
};

struct Fp8Params {
  CUtensorMap tm_q8, tm_k8, tm_vt8;  // e4m3 tiles of 128 x 128 bytes, 128B swizzle
  void *o;                            // [B, N, H, 128] bf16
  float *lse;                         // [B, H, N] or nullptr
  const float *sq, *sk, *sv;
  unsigned *status;
  int B, H, Hkv, N, nt;
  float scale_log2;
  int sched_chunk;
};

int launch_fp8_prepare(const Fp8PrepParams &p, cudaStream_t stream);
int launch_fwd_fp8(const Fp8Params &p, bool causal, cudaStream_t stream);

// Encodes a 4-D tensor map over bytes (e4m3): dims[0] innermost, strides in
// bytes for dims 1..3, box extents per dim (box[0] <= 128 bytes), 128-byte swizzle.
int encode_u8_tile_map(CUtensorMap *map, const void *base, const uint64_t dims[4], const uint64_t strides[3],
                       const uint32_t box[4]);

// Device status word of the current device (a small static device array).
unsigned *device_status_ptr();

// Encodes a 4-D tensor map over a bf16 [B, N, Hx, d] tensor, box = 64 columns x
// `box_rows` rows of one head, 128-byte swizzle.  Returns 0 on success.
int encode_bf16_tile_map(CUtensorMap *map, const void *base, int B, int N, int Hx, int d, int box_rows);

// Test builds only (-DFA_TEST_STALL): block 0 of the chosen kernel skips one
// barrier arrival (1: the forward's first P, 2: the dK/dV kernels' first P,
// 3: the dQ kernels' first dS), so that a bounded wait runs out and the kernel
// unwinds through its abort path.  Each translation unit keeps its own flag.
#ifdef FA_TEST_STALL
int set_test_stall_fwd(int mode);
int set_test_stall_bwd(int mode);
#define FA_STALL_FLAG_DECL static __device__ int g_test_stall;
#define FA_STALL(k) (g_test_stall == (k) && blockIdx.x == 0)
#else
#define FA_STALL_FLAG_DECL
#define FA_STALL(k) false
#endif

int launch_fwd(const FwdParams &p, int d, bool causal, cudaStream_t stream);
// The three launches of the backward pass (fa_bwd runs them in this order).
int launch_bwd_pre(const BwdParams &p, int d, const void *o, const void *dO, const float *lse, cudaStream_t stream);
int launch_bwd_dkdv(const BwdParams &p, int d, bool causal, cudaStream_t stream);
int launch_bwd_dq(const BwdParams &p, int d, bool causal, cudaStream_t stream);
// The fused backward on CTA pairs (head dim 128): dK, dV and dQ partials in one
// kernel, dQ accumulated in p.dqacc (zeroed by launch_bwd_pre when p.dqacc is
// set), then scaled and rounded to bf16 by launch_bwd_post.
int launch_bwd_fused(const BwdParams &p, bool causal, cudaStream_t stream);
int launch_bwd_post(const BwdParams &p, int d, cudaStream_t stream);

}  // namespace fa
