// fa_api.cu — the C ABI (include/fa.h): argument checks, tensor-map encoding,
// launches, the device status word and the standalone software-exp2 kernel.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "exp2_poly.cuh"
#include "fa_internal.h"

namespace fa {

// [0] error bits (1 = a bounded wait ran out), [1] id of the first wait site
// that ran out, [2] number of warp-level O rescales (forward), [3] spare.
static __device__ unsigned g_status[4];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned *g_status_ptr[kMaxDevices] = {};
int g_dev_ok[kMaxDevices] = {};  // 0 unknown, 1 GB300, -1 other
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int current_device(int *dev) {
  if (cudaGetDevice(dev) != cudaSuccess || *dev < 0 || *dev >= kMaxDevices) return FA_ERR_CUDA;
  return FA_OK;
}

// Once per device: compute capability must be 10.3 (GB300, sm_103a).
int check_device() {
  int dev;
  if (current_device(&dev) != FA_OK) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_dev_ok[dev] == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return FA_ERR_CUDA;
    g_dev_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
  }
  return g_dev_ok[dev] == 1 ? FA_OK : FA_ERR_UNSUPPORTED;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_common(int B, int H, int Hkv, int N, int d, float scale) {
  if (B <= 0 || H <= 0 || Hkv <= 0 || N <= 0 || d <= 0) return FA_ERR_INVALID_ARG;
  if (H % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
  if (H > 65535 || B > 65535) return FA_ERR_UNSUPPORTED;
  // fewer than 2^40 elements: offsets are 64-bit, and this keeps them far from overflow
  if ((long long)B * N * H * d >= (1ll << 40)) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

// Varlen arguments: the table must be a 4-byte aligned device array of B + 1
// entries (its contents are not read on the host); total rows >= 0.
int check_varlen(const int *cu_seqlens, int total, int H, int d) {
  if (cu_seqlens == nullptr || (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u)) return FA_ERR_INVALID_ARG;
  if (total < 0) return FA_ERR_INVALID_ARG;
  if ((long long)total * H * d >= (1ll << 40)) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

}  // namespace

unsigned *device_status_ptr() {
  int dev;
  if (current_device(&dev) != FA_OK) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_status_ptr[dev] == nullptr) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_status) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<unsigned *>(ptr);
  }
  return g_status_ptr[dev];
}

namespace {
int get_encoder() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_encode == nullptr) {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
      return FA_ERR_CUDA;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return FA_OK;
}
}  // namespace

int encode_bf16_tile_map(CUtensorMap *map, const void *base, int B, int N, int Hx, int d, int box_rows) {
  if (get_encoder() != FA_OK) return FA_ERR_CUDA;
  const cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)Hx, (cuuint64_t)N, (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)Hx * d * 2, (cuuint64_t)N * Hx * d * 2};
  const cuuint32_t box[4] = {64, 1, (cuuint32_t)box_rows, 1};
  const cuuint32_t estride[4] = {1, 1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box,
                        estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

int encode_u8_tile_map(CUtensorMap *map, const void *base, const uint64_t dims[4], const uint64_t strides[3],
                       const uint32_t box_dims[4]) {
  if (get_encoder() != FA_OK) return FA_ERR_CUDA;
  const cuuint64_t d[4] = {dims[0], dims[1], dims[2], dims[3]};
  const cuuint64_t st[3] = {strides[0], strides[1], strides[2]};
  const cuuint32_t box[4] = {box_dims[0], box_dims[1], box_dims[2], box_dims[3]};
  const cuuint32_t estride[4] = {1, 1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void *>(base), d, st, box, estride,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

// Workspace of the FP8 forward: the arrays of Fp8PrepParams, each on a 256-byte boundary.
struct Fp8Layout {
  size_t q8, k8, vt8, sq, sk, vblk, sv, total;
};
Fp8Layout fp8_layout(int B, int H, int Hkv, int N) {
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  const size_t nt = ((size_t)N + 127) / 128, Npad = nt * 128;
  Fp8Layout l;
  l.q8 = 0;
  l.k8 = l.q8 + up((size_t)B * N * H * 128);
  l.vt8 = l.k8 + up((size_t)B * N * Hkv * 128);
  l.sq = l.vt8 + up((size_t)B * Hkv * 128 * Npad);
  l.sk = l.sq + up((size_t)B * H * nt * 4);
  l.vblk = l.sk + up((size_t)B * Hkv * nt * 4);
  l.sv = l.vblk + up((size_t)B * Hkv * nt * 4);
  l.total = l.sv + up((size_t)B * Hkv * 4);
  return l;
}

namespace {

// Elements in pairs through the packed form (exp2_poly2, as in the dK/dV
// kernel); the scalar form (forward kernel) is evaluated as well and any bitwise
// difference between the two is returned as NaN, which the accuracy checks catch.
__global__ void exp2_poly_kernel(const float *__restrict__ x, float *__restrict__ y, long long n) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  const long long pairs = (n + 1) / 2;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < pairs; i += stride) {
    const long long a = 2 * i, b = a + 1;
    const float x0 = x[a], x1 = b < n ? x[b] : 0.0f;
    float y0, y1;
    exp2_poly2(x0, x1, y0, y1);
    const float s0 = exp2_poly(x0), s1 = exp2_poly(x1);
    y[a] = __float_as_uint(y0) == __float_as_uint(s0) ? y0 : __uint_as_float(0x7fc00000u);
    if (b < n) y[b] = __float_as_uint(y1) == __float_as_uint(s1) ? y1 : __uint_as_float(0x7fc00000u);
  }
}

}  // namespace
}  // namespace fa

using namespace fa;

extern "C" {

int fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H, int Hkv, int N, int d,
           float scale, int causal, void *stream) {
  if (!q || !k || !v || !o) return FA_ERR_INVALID_ARG;
  int rc = check_common(B, H, Hkv, N, d, scale);
  if (rc != FA_OK) return rc;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
      (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return FA_ERR_ALIGNMENT;
  if ((rc = check_device()) != FA_OK) return rc;
  FwdParams p;
  std::memset(&p, 0, sizeof(p));
  if (encode_bf16_tile_map(&p.tm_q, q, B, N, H, d, 128) || encode_bf16_tile_map(&p.tm_k, k, B, N, Hkv, d, 128) ||
      encode_bf16_tile_map(&p.tm_v, v, B, N, Hkv, d, 128) || encode_bf16_tile_map(&p.tm_o, o, B, N, H, d, 128) ||
      (d >= 128 && encode_bf16_tile_map(&p.tm_k64, k, B, N, Hkv, d, 64)))
    return FA_ERR_CUDA;
  p.o = o;
  p.lse = lse;
  p.status = device_status_ptr();
  if (!p.status) return FA_ERR_CUDA;
  p.B = B;
  p.H = H;
  p.Hkv = Hkv;
  p.N = N;
  p.scale_log2 = scale * 1.4426950408889634f;
  return launch_fwd(p, d, causal != 0, static_cast<cudaStream_t>(stream));
}

int fa_fwd_varlen(const void *q, const void *k, const void *v, void *o, float *lse, const int *cu_seqlens, int B,
                  int max_seqlen, int total, int H, int Hkv, int d, float scale, int causal, void *stream) {
  if (!q || !k || !v || !o) return FA_ERR_INVALID_ARG;
  int rc = check_common(B, H, Hkv, max_seqlen, d, scale);
  if (rc != FA_OK) return rc;
  if ((rc = check_varlen(cu_seqlens, total, H, d)) != FA_OK) return rc;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
      (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return FA_ERR_ALIGNMENT;
  if ((rc = check_device()) != FA_OK) return rc;
  if (total == 0) return FA_OK;
  FwdParams p;
  std::memset(&p, 0, sizeof(p));
  // the packed tensors as one batch of `total` rows
  if (encode_bf16_tile_map(&p.tm_q, q, 1, total, H, d, 128) || encode_bf16_tile_map(&p.tm_k, k, 1, total, Hkv, d, 128) ||
      encode_bf16_tile_map(&p.tm_v, v, 1, total, Hkv, d, 128) || encode_bf16_tile_map(&p.tm_o, o, 1, total, H, d, 128) ||
      (d >= 128 && encode_bf16_tile_map(&p.tm_k64, k, 1, total, Hkv, d, 64)))
    return FA_ERR_CUDA;
  p.o = o;
  p.lse = lse;
  p.cu_seqlens = cu_seqlens;
  p.total = total;
  p.status = device_status_ptr();
  if (!p.status) return FA_ERR_CUDA;
  p.B = B;
  p.H = H;
  p.Hkv = Hkv;
  p.N = max_seqlen;
  p.scale_log2 = scale * 1.4426950408889634f;
  return launch_fwd(p, d, causal != 0, static_cast<cudaStream_t>(stream));
}

size_t fa_fwd_fp8_workspace_bytes(int B, int H, int Hkv, int N, int d) {
  if (check_common(B, H, Hkv, N, d, 1.0f) != FA_OK || d != 128) return 0;
  return fp8_layout(B, H, Hkv, N).total;
}

int fa_fwd_fp8(const void *q, const void *k, const void *v, const float *rot_signs, void *o, float *lse, int B,
               int H, int Hkv, int N, int d, float scale, int causal, void *workspace, size_t workspace_bytes,
               void *stream) {
  if (!q || !k || !v || !o) return FA_ERR_INVALID_ARG;
  int rc = check_common(B, H, Hkv, N, d, scale);
  if (rc != FA_OK) return rc;
  if (d != 128) return FA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
      (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) || (rot_signs && (reinterpret_cast<uintptr_t>(rot_signs) & 3u)))
    return FA_ERR_ALIGNMENT;
  const Fp8Layout l = fp8_layout(B, H, Hkv, N);
  if (!workspace || workspace_bytes < l.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return FA_ERR_WORKSPACE;
  if ((rc = check_device()) != FA_OK) return rc;
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  const int nt = (N + 127) / 128, Npad = nt * 128;
  Fp8PrepParams pp;
  std::memset(&pp, 0, sizeof(pp));
  pp.q = static_cast<const __nv_bfloat16 *>(q);
  pp.k = static_cast<const __nv_bfloat16 *>(k);
  pp.v = static_cast<const __nv_bfloat16 *>(v);
  pp.signs = rot_signs;
  pp.q8 = ws + l.q8;
  pp.k8 = ws + l.k8;
  pp.vt8 = ws + l.vt8;
  pp.sq = reinterpret_cast<float *>(ws + l.sq);
  pp.sk = reinterpret_cast<float *>(ws + l.sk);
  pp.vblk = reinterpret_cast<float *>(ws + l.vblk);
  pp.sv = reinterpret_cast<float *>(ws + l.sv);
  pp.B = B;
  pp.H = H;
  pp.Hkv = Hkv;
  pp.N = N;
  pp.nt = nt;
  pp.Npad = Npad;
  Fp8Params p;
  std::memset(&p, 0, sizeof(p));
  const uint64_t dq[4] = {128, (uint64_t)H, (uint64_t)N, (uint64_t)B};
  const uint64_t sq_[3] = {128, (uint64_t)H * 128, (uint64_t)N * H * 128};
  const uint64_t dk[4] = {128, (uint64_t)Hkv, (uint64_t)N, (uint64_t)B};
  const uint64_t sk_[3] = {128, (uint64_t)Hkv * 128, (uint64_t)N * Hkv * 128};
  const uint64_t dv[4] = {(uint64_t)Npad, 128, (uint64_t)Hkv, (uint64_t)B};
  const uint64_t sv_[3] = {(uint64_t)Npad, (uint64_t)Npad * 128, (uint64_t)Npad * 128 * Hkv};
  // boxes: 128 rows of one head (128 bytes each) for q8 / k8; 128 head-dim rows x 128 keys for vt8
  const uint32_t box_rows[4] = {128, 1, 128, 1}, box_vt[4] = {128, 128, 1, 1};
  if (encode_u8_tile_map(&p.tm_q8, pp.q8, dq, sq_, box_rows) || encode_u8_tile_map(&p.tm_k8, pp.k8, dk, sk_, box_rows) ||
      encode_u8_tile_map(&p.tm_vt8, pp.vt8, dv, sv_, box_vt))
    return FA_ERR_CUDA;
  p.o = o;
  p.lse = lse;
  p.sq = pp.sq;
  p.sk = pp.sk;
  p.sv = pp.sv;
  p.status = device_status_ptr();
  if (!p.status) return FA_ERR_CUDA;
  p.B = B;
  p.H = H;
  p.Hkv = Hkv;
  p.N = N;
  p.nt = nt;
  p.scale_log2 = scale * 1.4426950408889634f;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if ((rc = launch_fp8_prepare(pp, st)) != FA_OK) return rc;
  return launch_fwd_fp8(p, causal != 0, st);
}

size_t fa_bwd_workspace_bytes(int B, int H, int Hkv, int N, int d) {
  if (check_common(B, H, Hkv, N, d, 1.0f) != FA_OK) return 0;
  const size_t Npad = ((size_t)N + 127) / 128 * 128;
  const size_t rows = (size_t)B * H * Npad * sizeof(float);
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  return 2 * up(rows);
}

size_t fa_bwd_fused_workspace_bytes(int B, int H, int Hkv, int N, int d) {
  if (d != 128) return 0;
  const size_t rows = fa_bwd_workspace_bytes(B, H, Hkv, N, d);
  if (rows == 0) return 0;
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  return rows + up((size_t)B * N * H * d * sizeof(float));
}

}  // extern "C"

namespace {

// Validation and parameter set-up shared by fa_bwd and its three stages.
// Pointers passed as nullptr are not needed by the stage and are not checked.
// With a varlen table (cu != nullptr) N is the longest sequence and the tensors
// are packed [total, Hx, d]; the row-term workspace keeps its [B, H, Npad] layout.
int setup_bwd(BwdParams *p, const void *q, const void *k, const void *v, const void *dO, const void *dq,
              const void *dk, const void *dv, int B, int H, int Hkv, int N, int d, float scale, void *workspace,
              size_t workspace_bytes, const int *cu = nullptr, int total = 0) {
  int rc = check_common(B, H, Hkv, N, d, scale);
  if (rc != FA_OK) return rc;
  if (cu && (rc = check_varlen(cu, total, H, d)) != FA_OK) return rc;
  for (const void *x : {q, k, v, dO, dq, dk, dv})
    if (x && !aligned16(x)) return FA_ERR_ALIGNMENT;
  const size_t need = fa_bwd_workspace_bytes(B, H, Hkv, N, d);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return FA_ERR_WORKSPACE;
  if ((rc = check_device()) != FA_OK) return rc;
  std::memset(p, 0, sizeof(*p));
  // tensor maps of the tensors this stage touches (nullptr: not used by it);
  // packed varlen tensors are one batch of `total` rows
  const int mb = cu ? 1 : B, mn = cu ? total : N;
  if ((q && encode_bf16_tile_map(&p->tm_q, q, mb, mn, H, d, 128)) ||
      (k && encode_bf16_tile_map(&p->tm_k, k, mb, mn, Hkv, d, 128)) ||
      (v && encode_bf16_tile_map(&p->tm_v, v, mb, mn, Hkv, d, 128)) ||
      (dO && encode_bf16_tile_map(&p->tm_do, dO, mb, mn, H, d, 128)) ||
      // 64-row boxes: only the CTA-pair kernels (head dims 128 and 256) use them
      (q && d >= 128 && encode_bf16_tile_map(&p->tm_q64, q, mb, mn, H, d, 64)) ||
      (dO && d >= 128 && encode_bf16_tile_map(&p->tm_do64, dO, mb, mn, H, d, 64)) ||
      (k && d >= 128 && encode_bf16_tile_map(&p->tm_k64, k, mb, mn, Hkv, d, 64)) ||
      (v && d >= 128 && encode_bf16_tile_map(&p->tm_v64, v, mb, mn, Hkv, d, 64)) ||
      (dk && d == 256 && encode_bf16_tile_map(&p->tm_dk64, dk, mb, mn, Hkv, d, 64)) ||
      (dv && d == 256 && encode_bf16_tile_map(&p->tm_dv64, dv, mb, mn, Hkv, d, 64)) ||
      (dq && d == 256 && encode_bf16_tile_map(&p->tm_dq64, dq, mb, mn, H, d, 64)) ||
      (dq && encode_bf16_tile_map(&p->tm_dq, dq, mb, mn, H, d, 128)) ||
      (dk && encode_bf16_tile_map(&p->tm_dk, dk, mb, mn, Hkv, d, 128)) ||
      (dv && encode_bf16_tile_map(&p->tm_dv, dv, mb, mn, Hkv, d, 128)))
    return FA_ERR_CUDA;
  p->cu_seqlens = cu;
  p->total = total;
  p->dq = const_cast<void *>(dq);
  p->dk = const_cast<void *>(dk);
  p->dv = const_cast<void *>(dv);
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  const size_t Npad = ((size_t)N + 127) / 128 * 128;
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  p->lse2 = reinterpret_cast<float *>(ws);
  p->delta = reinterpret_cast<const float *>(ws + up((size_t)B * H * Npad * sizeof(float)));
  p->status = device_status_ptr();
  if (!p->status) return FA_ERR_CUDA;
  p->B = B;
  p->H = H;
  p->Hkv = Hkv;
  p->N = N;
  p->scale = scale;
  p->scale_log2 = scale * 1.4426950408889634f;
  return FA_OK;
}

bool misaligned4(const void *x) { return (reinterpret_cast<uintptr_t>(x) & 3u) != 0; }

}  // namespace

extern "C" {

int fa_bwd_prepare(const void *o, const float *lse, const void *dO, int B, int H, int Hkv, int N, int d,
                   void *workspace, size_t workspace_bytes, void *stream) {
  if (!o || !lse || !dO) return FA_ERR_INVALID_ARG;
  if (!aligned16(o) || misaligned4(lse)) return FA_ERR_ALIGNMENT;
  BwdParams p;
  int rc = setup_bwd(&p, nullptr, nullptr, nullptr, dO, nullptr, nullptr, nullptr, B, H, Hkv, N, d, 1.0f, workspace,
                     workspace_bytes);
  if (rc != FA_OK) return rc;
  return launch_bwd_pre(p, d, o, dO, lse, static_cast<cudaStream_t>(stream));
}

int fa_bwd_dkdv(const void *q, const void *k, const void *v, const void *dO, void *dk, void *dv, int B, int H,
                int Hkv, int N, int d, float scale, int causal, void *workspace, size_t workspace_bytes,
                void *stream) {
  if (!q || !k || !v || !dO || !dk || !dv) return FA_ERR_INVALID_ARG;
  BwdParams p;
  int rc = setup_bwd(&p, q, k, v, dO, nullptr, dk, dv, B, H, Hkv, N, d, scale, workspace, workspace_bytes);
  if (rc != FA_OK) return rc;
  return launch_bwd_dkdv(p, d, causal != 0, static_cast<cudaStream_t>(stream));
}

int fa_bwd_dq(const void *q, const void *k, const void *v, const void *dO, void *dq, int B, int H, int Hkv, int N,
              int d, float scale, int causal, void *workspace, size_t workspace_bytes, void *stream) {
  if (!q || !k || !v || !dO || !dq) return FA_ERR_INVALID_ARG;
  BwdParams p;
  int rc = setup_bwd(&p, q, k, v, dO, dq, nullptr, nullptr, B, H, Hkv, N, d, scale, workspace, workspace_bytes);
  if (rc != FA_OK) return rc;
  return launch_bwd_dq(p, d, causal != 0, static_cast<cudaStream_t>(stream));
}

int fa_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse, const void *dO, void *dq,
           void *dk, void *dv, int B, int H, int Hkv, int N, int d, float scale, int causal, void *workspace,
           size_t workspace_bytes, void *stream) {
  if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  int rc = check_common(B, H, Hkv, N, d, scale);
  if (rc != FA_OK) return rc;
  if (!aligned16(o) || misaligned4(lse)) return FA_ERR_ALIGNMENT;
  BwdParams p;
  if ((rc = setup_bwd(&p, q, k, v, dO, dq, dk, dv, B, H, Hkv, N, d, scale, workspace, workspace_bytes)) != FA_OK)
    return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if ((rc = launch_bwd_pre(p, d, o, dO, lse, s)) != FA_OK) return rc;
  if ((rc = launch_bwd_dkdv(p, d, causal != 0, s)) != FA_OK) return rc;
  return launch_bwd_dq(p, d, causal != 0, s);
}

int fa_bwd_fused(const void *q, const void *k, const void *v, const void *o, const float *lse, const void *dO,
                 void *dq, void *dk, void *dv, int B, int H, int Hkv, int N, int d, float scale, int causal,
                 void *workspace, size_t workspace_bytes, void *stream) {
  if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  int rc = check_common(B, H, Hkv, N, d, scale);
  if (rc != FA_OK) return rc;
  if (d != 128) return FA_ERR_UNSUPPORTED;
  if (!aligned16(o) || misaligned4(lse)) return FA_ERR_ALIGNMENT;
  if (workspace_bytes < fa_bwd_fused_workspace_bytes(B, H, Hkv, N, d)) return FA_ERR_WORKSPACE;
  BwdParams p;
  if ((rc = setup_bwd(&p, q, k, v, dO, dq, dk, dv, B, H, Hkv, N, d, scale, workspace, workspace_bytes)) != FA_OK)
    return rc;
  p.dqacc = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + fa_bwd_workspace_bytes(B, H, Hkv, N, d));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if ((rc = launch_bwd_pre(p, d, o, dO, lse, s)) != FA_OK) return rc;  // also zeroes the dQ accumulator
  if ((rc = launch_bwd_fused(p, causal != 0, s)) != FA_OK) return rc;
  return launch_bwd_post(p, d, s);
}

int fa_bwd_varlen(const void *q, const void *k, const void *v, const void *o, const float *lse, const void *dO,
                  void *dq, void *dk, void *dv, const int *cu_seqlens, int B, int max_seqlen, int total, int H,
                  int Hkv, int d, float scale, int causal, void *workspace, size_t workspace_bytes, void *stream) {
  if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  if (!aligned16(o) || misaligned4(lse)) return FA_ERR_ALIGNMENT;
  if (!cu_seqlens) return FA_ERR_INVALID_ARG;
  BwdParams p;
  int rc = setup_bwd(&p, q, k, v, dO, dq, dk, dv, B, H, Hkv, max_seqlen, d, scale, workspace, workspace_bytes,
                     cu_seqlens, total);
  if (rc != FA_OK) return rc;
  if (total == 0) return FA_OK;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if ((rc = launch_bwd_pre(p, d, o, dO, lse, s)) != FA_OK) return rc;
  if ((rc = launch_bwd_dkdv(p, d, causal != 0, s)) != FA_OK) return rc;
  return launch_bwd_dq(p, d, causal != 0, s);
}

}  // extern "C"

// ------------------------------------------------------------------ allocation-free backward
// Some callers cannot allocate device memory when they run the backward pass:
// plug-ins living inside a host framework that owns every device allocation
// through its own pool, and serving or training loops that forbid cudaMalloc
// after start-up because it synchronises the device and fragments memory.
// fa_bwd_noalloc serves them: its scratch (the per-row D and log2-LSE terms
// that fa_bwd keeps in the caller's workspace) is this file-scope device array
// instead.  Every GPU that loads the library holds
// it until the process exits.
namespace fa {
namespace {

constexpr size_t kNoAllocScratchBytes = FA_BWD_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_bwd_scratch[kNoAllocScratchBytes];
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of g_bwd_scratch on the current device.  In host code the
// array's name only stands for it; the address is looked up once per device,
// with that device current, and cached.
int scratch_address(void **out) {
  int dev;
  if (current_device(&dev) != FA_OK) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_bwd_scratch) != cudaSuccess || ptr == nullptr) return FA_ERR_CUDA;
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return FA_OK;
}

}  // namespace
}  // namespace fa

extern "C" {

int fa_bwd_noalloc(const void *q, const void *k, const void *v, const void *o, const float *lse, const void *dO,
                   void *dq, void *dk, void *dv, int B, int H, int Hkv, int N, int d, float scale, int causal,
                   void *stream) {
  if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  int rc = check_common(B, H, Hkv, N, d, scale);
  if (rc != FA_OK) return rc;
  if (!aligned16(o) || !aligned16(dq) || misaligned4(lse)) return FA_ERR_ALIGNMENT;
  const size_t need = fa_bwd_workspace_bytes(B, H, Hkv, N, d);
  if (need > kNoAllocScratchBytes) return FA_ERR_WORKSPACE;  // problem too large for the built-in scratch
  // the device check first: on a GPU other than sm_103 the library's kernels
  // cannot load, and the call must fail as fa_bwd does (FA_ERR_UNSUPPORTED)
  if ((rc = check_device()) != FA_OK) return rc;
  void *ws = nullptr;
  if ((rc = scratch_address(&ws)) != FA_OK) return rc;
  BwdParams p;
  if ((rc = setup_bwd(&p, q, k, v, dO, dq, dk, dv, B, H, Hkv, N, d, scale, ws, kNoAllocScratchBytes)) != FA_OK)
    return rc;
  // bwd_pre writes every part of the scratch that the other launches read
  // (D and log2-LSE of every padded row), so stale contents left by an earlier
  // call do not matter.
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if ((rc = launch_bwd_pre(p, d, o, dO, lse, s)) != FA_OK) return rc;
  if ((rc = launch_bwd_dkdv(p, d, causal != 0, s)) != FA_OK) return rc;
  return launch_bwd_dq(p, d, causal != 0, s);
}

size_t fa_bwd_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

int fa_exp2_poly(const float *x, float *y, long long n, void *stream) {
  if (n < 0 || (n > 0 && (!x || !y))) return FA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) & 3u) || (reinterpret_cast<uintptr_t>(y) & 3u)) return FA_ERR_ALIGNMENT;
  if (n == 0) return FA_OK;
  int rc = check_device();
  if (rc != FA_OK) return rc;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return FA_ERR_CUDA;
  const long long want = (n + 255) / 256;
  const int blocks = (int)(want < (long long)sms * 8 ? want : (long long)sms * 8);
  exp2_poly_kernel<<<blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(x, y, n);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_last_device_status_site(void *stream, int *site) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
  unsigned *st = device_status_ptr();
  if (!st) return FA_ERR_CUDA;
  unsigned h[2] = {0, 0};
  if (cudaMemcpy(h, st, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return FA_ERR_CUDA;
  if (site) *site = h[0] != 0 ? (int)h[1] : 0;
  if (h[0] != 0) {
    const unsigned zero[2] = {0, 0};
    if (cudaMemcpy(st, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return FA_ERR_CUDA;
    return FA_ERR_TIMEOUT;
  }
  return FA_OK;
}

int fa_last_device_status(void *stream) { return fa_last_device_status_site(stream, nullptr); }

int fa_debug_stall(int mode) {
#ifdef FA_TEST_STALL
  if (mode < 0 || mode > 3) return FA_ERR_INVALID_ARG;
  int rc = check_device();
  if (rc != FA_OK) return rc;
  if ((rc = set_test_stall_fwd(mode)) != FA_OK) return rc;
  return set_test_stall_bwd(mode);
#else
  (void)mode;
  return FA_ERR_UNSUPPORTED;
#endif
}

int fa_rescale_count(void *stream, unsigned *count) {
  if (!count) return FA_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
  unsigned *st = device_status_ptr();
  if (!st) return FA_ERR_CUDA;
  unsigned h = 0;
  if (cudaMemcpy(&h, st + 2, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return FA_ERR_CUDA;
  const unsigned zero = 0;
  if (cudaMemcpy(st + 2, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return FA_ERR_CUDA;
  *count = h;
  return FA_OK;
}

const char *fa_status_string(int status) {
  switch (status) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_ALIGNMENT: return "FA_ERR_ALIGNMENT";
    case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE";
    case FA_ERR_CUDA: return "FA_ERR_CUDA";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
    default: return "FA_ERR_UNKNOWN";
  }
}

}  // extern "C"
