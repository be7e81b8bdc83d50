// C-ABI entry points of libfp8attn.so: argument validation, TMA descriptor
// encoding and kernel launches.  No device memory is allocated here.
#include <algorithm>
#include <climits>
#include <cmath>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "../../include/fp8attn.h"
#include "kernels.cuh"

using namespace fp8attn;

namespace {

constexpr int kAbiVersion = 7;   // 2: fp8attn_prepped.v_offset, fp8attn_prep_smooth; 3: fp8attn_v_cluster;
                                 // 4: fp8attn_fwd_split; 5: NVFP4 V (fp8attn_prep_ex, prepped.v4,
                                 //    fp8attn_fwd_ex); 6: fp8attn_selftest_wait_timeout;
                                 // 7: FP8ATTN_ERR_BAD_PERMUTATION
constexpr size_t kStatusBytes = 256;          // status word lives in the first bytes of a workspace
constexpr unsigned long long kWaitLimitNs = 1000ull * 1000ull * 1000ull;   // 1 s per wait

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Device capability cache: 1 = sm_103, 0 = other, -1 = unknown.
int g_dev_ok[64];
std::once_flag g_dev_once;

fp8attn_status check_device() {
  std::call_once(g_dev_once, [] { for (int& v : g_dev_ok) v = -1; });
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FP8ATTN_ERR_CUDA;
  if (dev < 0 || dev >= 64) return FP8ATTN_ERR_UNSUPPORTED_DEVICE;
  if (g_dev_ok[dev] < 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return FP8ATTN_ERR_CUDA;
    g_dev_ok[dev] = (major == 10 && minor == 3) ? 1 : 0;
  }
  return g_dev_ok[dev] == 1 ? FP8ATTN_OK : FP8ATTN_ERR_UNSUPPORTED_DEVICE;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}

bool shape_ok(int B, int T, int H, int D) {
  if (B < 1 || T < 1 || H < 1 || D != kHeadDim) return false;
  if (H > 65535 || B > 32767) return false;
  const long long elems = static_cast<long long>(B) * T * H;
  return elems <= 0x7FFFFFFFll;
}

size_t round16(size_t x) { return (x + 15) & ~static_cast<size_t>(15); }

constexpr int kMaxSplits = 16;

// Clustering workspace: status word | amax u32 [BH][128] | dims, dim_exp i32 [BH][16]
// | centroids i32 [BH][64][16] | sums i64 [BH][64][16] | counts i32 [BH][64]
// | hist i32 [BH][nchunks][64] | labels u8 [BH][T] | codes i16 [BH][T][stride]
struct ClusterLayout {
  size_t amax, dims, dim_exp, cent, sums, counts, hist, labels8, codes, total;
};

ClusterLayout cluster_layout(int B, int T, int H, int r) {
  const size_t BH = static_cast<size_t>(B) * H;
  const size_t nchunks = (static_cast<size_t>(T) + 1023) / 1024;
  ClusterLayout L;
  size_t o = kStatusBytes;
  L.amax = o;    o = round16(o + BH * kHeadDim * 4);
  L.dims = o;    o = round16(o + BH * kClusterMaxDims * 4);
  L.dim_exp = o; o = round16(o + BH * kClusterMaxDims * 4);
  L.cent = o;    o = round16(o + BH * kClusterMaxK * kClusterMaxDims * 4);
  L.sums = o;    o = round16(o + BH * kClusterMaxK * kClusterMaxDims * 8);
  L.counts = o;  o = round16(o + BH * kClusterMaxK * 4);
  L.hist = o;    o = round16(o + BH * nchunks * kClusterMaxK * 4);
  L.labels8 = o; o = round16(o + BH * static_cast<size_t>(T));
  L.codes = o;   o = round16(o + BH * static_cast<size_t>(T) * cluster_code_stride(r) * 2);
  L.total = o;
  return L;
}

// Last-wave split plan.  With C = B H nQt query tiles on num_sms SMs the
// last wave holds C mod num_sms of them; when that is at most half the SMs,
// each of them is cut into P = min(4, num_sms / n_tail) parts of its nV key
// tiles.  Part p first takes max-only steps over the part_lo[p] positions
// before its range, about half the cost of a full step, so the parts are
// balanced by part_lo[p] = nV (1 - 2^-p) / (1 - 2^-P), rounded to a multiple
// of 4 (the kernel needs that).  Returns P, or 1 when the last wave is kept
// whole (then n_tail is 0 and part_lo is not written).
int tail_plan(int B, int T, int H, int num_sms, int* n_tail, int* part_lo) {
  *n_tail = 0;
  if (!shape_ok(B, T, H, kHeadDim) || num_sms < 2) return 1;
  const int nQt = (T + kTile - 1) / kTile;
  const int nV = (T + kVBlock - 1) / kVBlock;
  const long long total = static_cast<long long>(B) * H * nQt;
  if (total <= num_sms) return 1;                  // one wave: that is what split-KV is for
  const int tail = static_cast<int>(total % num_sms);
  if (tail == 0 || 2 * tail > num_sms) return 1;
  for (int P = std::min(kMaxTailParts, num_sms / tail); P >= 2; --P) {
    int lo[kMaxTailParts + 1];
    lo[0] = 0;
    lo[P] = nV;
    bool ok = true;
    for (int k = 1; k < P; ++k) {
      const double f = (1.0 - std::ldexp(1.0, -k)) / (1.0 - std::ldexp(1.0, -P));
      lo[k] = 4 * static_cast<int>(std::lround(nV * f / 4.0));
      if (lo[k] <= lo[k - 1] || lo[k] >= nV) ok = false;
    }
    if (!ok) continue;
    *n_tail = tail;
    for (int k = 0; k <= P; ++k) part_lo[k] = lo[k];
    return P;
  }
  return 1;
}

}  // namespace

extern "C" {

size_t fp8attn_cluster_workspace_bytes(int B, int T, int H, int n_dims) {
  if (B < 1 || T < 1 || H < 1 || n_dims < 1 || n_dims > kClusterMaxDims) return 0;
  return cluster_layout(B, T, H, n_dims).total;
}

fp8attn_status fp8attn_v_cluster(const void* v, int B, int T, int H, int D, int n_clusters,
                                 int n_dims, int iters, int32_t* perm, int32_t* labels,
                                 void* workspace, size_t workspace_bytes, void* stream) {
  if (!shape_ok(B, T, H, D) || !v || !perm) return FP8ATTN_ERR_INVALID_ARG;
  if (n_clusters < 1 || n_clusters > kClusterMaxK || n_dims < 1 || n_dims > kClusterMaxDims ||
      iters < 0 || iters > 64)
    return FP8ATTN_ERR_INVALID_ARG;
  if (!aligned16(v) || (reinterpret_cast<uintptr_t>(perm) & 3u) ||
      (labels && (reinterpret_cast<uintptr_t>(labels) & 3u)))
    return FP8ATTN_ERR_INVALID_ARG;
  const ClusterLayout L = cluster_layout(B, T, H, n_dims);
  if (!workspace || !aligned16(workspace) || workspace_bytes < L.total) return FP8ATTN_ERR_WORKSPACE;
  fp8attn_status st = check_device();
  if (st != FP8ATTN_OK) return st;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  ClusterParams p;
  p.v = static_cast<const __nv_bfloat16*>(v);
  p.B = B;
  p.T = T;
  p.H = H;
  p.K = n_clusters;
  p.r = n_dims;
  p.iters = iters;
  p.nchunks = (T + 1023) / 1024;
  p.amax = reinterpret_cast<uint32_t*>(ws + L.amax);
  p.dims = reinterpret_cast<int*>(ws + L.dims);
  p.dim_exp = reinterpret_cast<int*>(ws + L.dim_exp);
  p.cent = reinterpret_cast<int*>(ws + L.cent);
  p.sums = reinterpret_cast<long long*>(ws + L.sums);
  p.counts = reinterpret_cast<int*>(ws + L.counts);
  p.hist = reinterpret_cast<int*>(ws + L.hist);
  p.labels8 = ws + L.labels8;
  p.codes = reinterpret_cast<int16_t*>(ws + L.codes);
  p.perm = perm;
  p.labels = labels;
  return launch_cluster(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FP8ATTN_OK
                                                                             : FP8ATTN_ERR_CUDA;
}

// Prep workspace: status word | v_amax u32 [BH*128] | sequence statistics:
// chan_sum u64 [2][BH*128] | chan_max u32 [2][BH*128] | chan_low f32 [2][BH*128]
// | chan_mean f32 [2][BH*128] | vbias_acc f32 [BH*128]
size_t fp8attn_prep_workspace_bytes(int B, int T, int H) {
  (void)T;
  if (B < 1 || H < 1) return 0;
  const size_t n = static_cast<size_t>(B) * H * kHeadDim;
  return kStatusBytes + n * (4 + 2 * 8 + 2 * 4 + 2 * 4 + 2 * 4 + 4);
}

size_t fp8attn_workspace_size(int B, int T, int H, int D) {
  if (D != kHeadDim) return 0;
  return std::max(fp8attn_prep_workspace_bytes(B, T, H), fp8attn_fwd_workspace_bytes(B, T, H));
}

size_t fp8attn_fwd_workspace_bytes(int B, int T, int H) {
  (void)B;
  (void)T;
  (void)H;
  return kStatusBytes;
}

size_t fp8attn_v_padded_T(int T) {
  if (T < 1) return 0;
  return static_cast<size_t>((T + kVBlock - 1) / kVBlock) * kVBlock;
}

int fp8attn_abi_version(void) { return kAbiVersion; }

const char* fp8attn_status_string(fp8attn_status s) {
  switch (s) {
    case FP8ATTN_OK: return "ok";
    case FP8ATTN_ERR_INVALID_ARG: return "invalid argument";
    case FP8ATTN_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs sm_103)";
    case FP8ATTN_ERR_CUDA: return "CUDA error";
    case FP8ATTN_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case FP8ATTN_ERR_WORKSPACE: return "workspace missing or too small";
    case FP8ATTN_ERR_BAD_TILE_LIST: return "sparse tile index out of range";
    case FP8ATTN_ERR_BAD_PERMUTATION: return "permutation entry out of range";
  }
  return "unknown status";
}

fp8attn_status fp8attn_prep_smooth(const void* q, const void* k, const void* v, int B, int T,
                                   int H, int D, const int32_t* perm, int vsmooth, int smooth,
                                   int v_bias, const fp8attn_prepped* out, void* workspace,
                                   size_t workspace_bytes, void* stream) {
  return fp8attn_prep_ex(q, k, v, B, T, H, D, perm, vsmooth, smooth, v_bias, 0, out, workspace,
                         workspace_bytes, stream);
}

fp8attn_status fp8attn_prep_ex(const void* q, const void* k, const void* v, int B, int T, int H,
                               int D, const int32_t* perm, int vsmooth, int smooth, int v_bias,
                               int v_format, const fp8attn_prepped* out, void* workspace,
                               size_t workspace_bytes, void* stream) {
  if (!shape_ok(B, T, H, D) || !q || !k || !v || !out) return FP8ATTN_ERR_INVALID_ARG;
  if (smooth < 0 || smooth > 2 || v_bias < 0 || v_bias > 1) return FP8ATTN_ERR_INVALID_ARG;
  if (v_format < 0 || v_format > 1 || (v_format == 1 && v_bias)) return FP8ATTN_ERR_INVALID_ARG;
  if (!out->q8 || !out->k8 || !out->q_scale || !out->k_scale || !out->v_scale || !out->v_mean)
    return FP8ATTN_ERR_INVALID_ARG;
  if (v_format == 0 ? !out->v8 : (!out->v4 || !out->v4_sf || !aligned16(out->v4) || !aligned16(out->v4_sf)))
    return FP8ATTN_ERR_INVALID_ARG;
  if ((smooth == 2 || v_bias) && !out->v_offset) return FP8ATTN_ERR_INVALID_ARG;
  if (out->v_offset && !aligned16(out->v_offset)) return FP8ATTN_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, out->q8, out->k8, v_format == 0 ? out->v8 : out->v4, out->q_scale,
                        out->k_scale, out->v_scale, out->v_mean};
  for (const void* ptr : ptrs)
    if (!aligned16(ptr)) return FP8ATTN_ERR_INVALID_ARG;
  if (perm && (reinterpret_cast<uintptr_t>(perm) & 3u)) return FP8ATTN_ERR_INVALID_ARG;
  if (!workspace || !aligned16(workspace) || workspace_bytes < fp8attn_prep_workspace_bytes(B, T, H))
    return FP8ATTN_ERR_WORKSPACE;
  fp8attn_status st = check_device();
  if (st != FP8ATTN_OK) return st;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t n = static_cast<size_t>(B) * H * kHeadDim;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  PrepParams p;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k = static_cast<const __nv_bfloat16*>(k);
  p.v = static_cast<const __nv_bfloat16*>(v);
  p.perm = perm;
  p.q8 = static_cast<uint8_t*>(out->q8);
  p.k8 = static_cast<uint8_t*>(out->k8);
  p.v8 = static_cast<uint8_t*>(out->v8);
  p.q_scale = out->q_scale;
  p.k_scale = out->k_scale;
  p.v_scale = out->v_scale;
  p.v_mean = static_cast<__nv_bfloat16*>(out->v_mean);
  p.status = reinterpret_cast<int*>(ws);
  p.v_amax = reinterpret_cast<uint32_t*>(ws + kStatusBytes);
  p.chan_sum = reinterpret_cast<unsigned long long*>(ws + kStatusBytes + n * 4);   // 8-byte aligned
  p.chan_max = reinterpret_cast<uint32_t*>(ws + kStatusBytes + n * 4 + n * 16);
  p.chan_low = reinterpret_cast<float*>(ws + kStatusBytes + n * 4 + n * 16 + n * 8);
  p.chan_mean = reinterpret_cast<float*>(ws + kStatusBytes + n * 4 + n * 16 + n * 16);
  p.vbias_acc = reinterpret_cast<float*>(ws + kStatusBytes + n * 4 + n * 16 + n * 24);
  p.v_offset = out->v_offset;
  p.smooth = smooth;
  p.v_bias = v_bias;
  p.v_fp4 = v_format;
  p.v4 = static_cast<uint8_t*>(out->v4);
  p.v4_sf = static_cast<uint8_t*>(out->v4_sf);
  int lg = 0;
  while ((1ll << lg) < T) ++lg;
  p.sum_window = std::min(37, 62 - 8 - lg);   // T * 2^(W + 8) <= 2^62, 2^(W + 8) <= 2^45
  p.B = B;
  p.T = T;
  p.H = H;
  p.nQK = (T + kQKBlock - 1) / kQKBlock;
  p.nV = (T + kVBlock - 1) / kVBlock;
  p.Tpad = p.nV * kVBlock;
  p.vsmooth = vsmooth ? 1 : 0;
  if (cudaMemsetAsync(workspace, 0, fp8attn_prep_workspace_bytes(B, T, H), s) != cudaSuccess)
    return FP8ATTN_ERR_CUDA;
  return launch_prep(p, s) == cudaSuccess ? FP8ATTN_OK : FP8ATTN_ERR_CUDA;
}

fp8attn_status fp8attn_prep(const void* q, const void* k, const void* v, int B, int T, int H,
                            int D, const int32_t* perm, int vsmooth, const fp8attn_prepped* out,
                            void* workspace, size_t workspace_bytes, void* stream) {
  return fp8attn_prep_smooth(q, k, v, B, T, H, D, perm, vsmooth, 0, 0, out, workspace,
                             workspace_bytes, stream);
}

// Split-KV workspace: status word | (m, l) fp32 pairs [S][BH][T] | partial outputs fp32 [S][BH][T][128]
size_t fp8attn_fwd_split_workspace_bytes(int B, int T, int H, int n_splits) {
  if (B < 1 || T < 1 || H < 1 || n_splits < 1 || n_splits > kMaxSplits) return 0;
  if (n_splits == 1) return kStatusBytes;
  const size_t rows = static_cast<size_t>(n_splits) * B * H * T;
  return round16(kStatusBytes + rows * 8) + rows * kHeadDim * 4;
}

int fp8attn_fwd_auto_splits(int B, int T, int H, int num_sms) {
  if (B < 1 || T < 1 || H < 1 || num_sms < 1) return 1;
  const int n_tiles = (T + kTile - 1) / kTile;
  const long long ctas = static_cast<long long>(B) * H * n_tiles;
  // the parts of all query tiles must fit in one wave (a second wave costs
  // more than the split saves), and every part keeps at least 8 key tiles (the
  // CTA's fixed cost and the merge outweigh shorter parts); measured on GB300
  long long s = num_sms / ctas;
  s = std::min<long long>(s, n_tiles / 8);
  s = std::min<long long>(s, kMaxSplits);
  if (static_cast<long long>(B) * s > 65535) s = 65535LL / B;
  return static_cast<int>(std::max(1LL, s));
}

fp8attn_status fp8attn_fwd(const fp8attn_prepped* in, int B, int T, int H, int D,
                           const int32_t* tile_row_ptr, const int32_t* tile_col, int reverse_kv,
                           int pcast, float p_scale, float expcast_beta, float softmax_scale,
                           int vsmooth, void* out, void* workspace, size_t workspace_bytes,
                           void* stream) {
  return fp8attn_fwd_split(in, B, T, H, D, tile_row_ptr, tile_col, reverse_kv, pcast, p_scale,
                           expcast_beta, softmax_scale, vsmooth, 1, out, workspace, workspace_bytes,
                           stream);
}

fp8attn_status fp8attn_fwd_split(const fp8attn_prepped* in, int B, int T, int H, int D,
                                 const int32_t* tile_row_ptr, const int32_t* tile_col,
                                 int reverse_kv, int pcast, float p_scale, float expcast_beta,
                                 float softmax_scale, int vsmooth, int n_splits, void* out,
                                 void* workspace, size_t workspace_bytes, void* stream) {
  return fp8attn_fwd_ex(in, B, T, H, D, tile_row_ptr, tile_col, reverse_kv, pcast, p_scale,
                        expcast_beta, softmax_scale, vsmooth, n_splits, 0, out, workspace,
                        workspace_bytes, stream);
}

}  // extern "C"

namespace {

// fp8attn_fwd_ex, and with tail_sms > 0 fp8attn_fwd_tail_split (dense, 8-bit
// PV, n_splits 1): the last wave's query tiles of a tail_sms-SM device go to a
// second, split launch (tail_plan).
fp8attn_status fwd_impl(const fp8attn_prepped* in, int B, int T, int H, int D,
                        const int32_t* tile_row_ptr, const int32_t* tile_col, int reverse_kv,
                        int pcast, float p_scale, float expcast_beta, float softmax_scale,
                        int vsmooth, int n_splits, int pv_format, void* out, void* workspace,
                        size_t workspace_bytes, void* stream, int tail_sms) {
  if (!shape_ok(B, T, H, D) || !in || !out) return FP8ATTN_ERR_INVALID_ARG;
  if (pv_format < 0 || pv_format > 1) return FP8ATTN_ERR_INVALID_ARG;
  const bool fp4 = pv_format == 1;
  if (fp4 && (pcast != FP8ATTN_PCAST_EXP2_CVT || !in->v4 || !in->v4_sf || !aligned16(in->v4) ||
              !aligned16(in->v4_sf)))
    return FP8ATTN_ERR_INVALID_ARG;
  if (n_splits < 1 || n_splits > kMaxSplits || static_cast<long long>(B) * n_splits > 65535)
    return FP8ATTN_ERR_INVALID_ARG;
  if (tail_sms < 0 || (tail_sms > 0 && (tile_row_ptr || tile_col || fp4 || n_splits != 1)))
    return FP8ATTN_ERR_INVALID_ARG;
  if (!in->q8 || !in->k8 || (!fp4 && !in->v8) || !in->q_scale || !in->k_scale || !in->v_scale)
    return FP8ATTN_ERR_INVALID_ARG;
  if (vsmooth && !in->v_mean) return FP8ATTN_ERR_INVALID_ARG;
  if ((tile_row_ptr == nullptr) != (tile_col == nullptr)) return FP8ATTN_ERR_INVALID_ARG;
  if (pcast != FP8ATTN_PCAST_EXP2_CVT && pcast != FP8ATTN_PCAST_EXPCAST)
    return FP8ATTN_ERR_INVALID_ARG;
  if (!(p_scale >= 1.f && p_scale <= 448.f)) return FP8ATTN_ERR_INVALID_ARG;
  if (!(std::fabs(expcast_beta) < 0.5f)) return FP8ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(softmax_scale)) return FP8ATTN_ERR_INVALID_ARG;
  const void* ptrs[] = {in->q8, in->k8, fp4 ? in->v4 : in->v8, in->q_scale, in->k_scale, in->v_scale, out};
  for (const void* ptr : ptrs)
    if (!aligned16(ptr)) return FP8ATTN_ERR_INVALID_ARG;
  if (vsmooth && !aligned16(in->v_mean)) return FP8ATTN_ERR_INVALID_ARG;
  if (in->v_offset && !aligned16(in->v_offset)) return FP8ATTN_ERR_INVALID_ARG;
  const size_t ws_need = tail_sms > 0 ? fp8attn_fwd_tail_workspace_bytes(B, T, H, tail_sms)
                                      : fp8attn_fwd_split_workspace_bytes(B, T, H, n_splits);
  if (!workspace || !aligned16(workspace) || workspace_bytes < ws_need) return FP8ATTN_ERR_WORKSPACE;
  fp8attn_status st = check_device();
  if (st != FP8ATTN_OK) return st;
  PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
  if (!enc) return FP8ATTN_ERR_CUDA;

  const int nQK = (T + kQKBlock - 1) / kQKBlock;
  const int nV = (T + kVBlock - 1) / kVBlock;
  const int Tpad = nV * kVBlock;
  AttnParams p;
  std::memset(&p, 0, sizeof(p));
  {
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(H),
                                static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(B)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(kHeadDim),
                                   static_cast<cuuint64_t>(H) * kHeadDim,
                                   static_cast<cuuint64_t>(T) * H * kHeadDim};
    const cuuint32_t box[4] = {128, 1, 128, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    if (enc(&p.tm_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, in->q8, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return FP8ATTN_ERR_CUDA;
    if (enc(&p.tm_k, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, in->k8, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return FP8ATTN_ERR_CUDA;
  }
  {
    // E4M3 V: rows of Tpad bytes, 128x128 boxes, 128-byte swizzle; packed E2M1 V:
    // rows of Tpad/2 bytes, 64-byte x 128-row boxes, 64-byte swizzle
    const cuuint64_t row = fp4 ? static_cast<cuuint64_t>(Tpad / 2) : static_cast<cuuint64_t>(Tpad);
    const cuuint64_t dims[3] = {row, static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(B) * H};
    const cuuint64_t strides[2] = {row, row * kHeadDim};
    const cuuint32_t box[3] = {fp4 ? 64u : 128u, 128, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (enc(&p.tm_v, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, fp4 ? in->v4 : in->v8, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, fp4 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return FP8ATTN_ERR_CUDA;
  }
  p.q_scale = in->q_scale;
  p.k_scale = in->k_scale;
  p.v_scale = in->v_scale;
  p.v_mean = static_cast<const __nv_bfloat16*>(in->v_mean);
  p.v_offset = in->v_offset;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.row_ptr = tile_row_ptr;
  p.col = tile_col;
  p.status = static_cast<int*>(workspace);
  p.B = B;
  p.T = T;
  p.H = H;
  p.nQK = nQK;
  p.nV = nV;
  p.nQt = (T + kTile - 1) / kTile;
  p.reverse = reverse_kv ? 1 : 0;
  // ExpCast: the code of p = 1 is rne(8 log2 S + 56 + beta); only when that can
  // round past 126 (S above ~430) does the kernel need its top clamp (kernel
  // variant 2).  A small margin covers the kernel's fp32 evaluation.
  p.pcast = pcast;
  if (pcast == FP8ATTN_PCAST_EXPCAST && 8.0 * std::log2(static_cast<double>(p_scale)) + 56.0 + expcast_beta >= 126.5 - 1e-3)
    p.pcast = 2;
  p.vsmooth = vsmooth ? 1 : 0;
  p.log2_pscale = std::log2(p_scale);
  p.beta = expcast_beta;
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / std::sqrt(static_cast<float>(kHeadDim));
  p.sm_scale_log2 = scale * 1.4426950408889634f;
  p.timeout_ns = kWaitLimitNs;
  p.n_splits = n_splits;
  p.fp4 = fp4 ? 1 : 0;
  p.v4_sf = static_cast<const uint8_t*>(in->v4_sf);
  p.cta_limit = INT_MAX;
  p.tail_cta0 = -1;
  if (n_splits > 1) {
    const size_t rows = static_cast<size_t>(n_splits) * B * H * T;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    p.part_ml = reinterpret_cast<float2*>(ws + kStatusBytes);
    p.part_o = reinterpret_cast<float*>(ws + round16(kStatusBytes + rows * 8));
  }

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(workspace, 0, 16 * sizeof(int), s) != cudaSuccess) return FP8ATTN_ERR_CUDA;
  int n_tail = 0, lo[kMaxTailParts + 1];
  const int parts = tail_sms > 0 ? tail_plan(B, T, H, tail_sms, &n_tail, lo) : 1;
  if (parts < 2) return launch_attn(p, s) == cudaSuccess ? FP8ATTN_OK : FP8ATTN_ERR_CUDA;
  // the whole waves, then the last wave's query tiles in parts, merged by log-sum-exp
  const int total = B * H * p.nQt;
  p.cta_limit = total - n_tail;
  if (launch_attn(p, s) != cudaSuccess) return FP8ATTN_ERR_CUDA;
  AttnParams q = p;
  q.n_splits = parts;
  q.tail_cta0 = total - n_tail;
  q.n_tail = n_tail;
  for (int k = 0; k <= parts; ++k) q.part_lo[k] = lo[k];
  const size_t rows = static_cast<size_t>(parts) * n_tail * kTile;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  q.part_ml = reinterpret_cast<float2*>(ws + kStatusBytes);
  q.part_o = reinterpret_cast<float*>(ws + round16(kStatusBytes + rows * 8));
  return launch_attn(q, s) == cudaSuccess ? FP8ATTN_OK : FP8ATTN_ERR_CUDA;
}

}  // namespace

extern "C" {

fp8attn_status fp8attn_fwd_ex(const fp8attn_prepped* in, int B, int T, int H, int D,
                              const int32_t* tile_row_ptr, const int32_t* tile_col, int reverse_kv,
                              int pcast, float p_scale, float expcast_beta, float softmax_scale,
                              int vsmooth, int n_splits, int pv_format, void* out, void* workspace,
                              size_t workspace_bytes, void* stream) {
  return fwd_impl(in, B, T, H, D, tile_row_ptr, tile_col, reverse_kv, pcast, p_scale, expcast_beta,
                  softmax_scale, vsmooth, n_splits, pv_format, out, workspace, workspace_bytes, stream, 0);
}

fp8attn_status fp8attn_fwd_tail_split(const fp8attn_prepped* in, int B, int T, int H, int D,
                                      int reverse_kv, int pcast, float p_scale, float expcast_beta,
                                      float softmax_scale, int vsmooth, int num_sms, void* out,
                                      void* workspace, size_t workspace_bytes, void* stream) {
  if (num_sms < 1) return FP8ATTN_ERR_INVALID_ARG;
  return fwd_impl(in, B, T, H, D, nullptr, nullptr, reverse_kv, pcast, p_scale, expcast_beta,
                  softmax_scale, vsmooth, 1, 0, out, workspace, workspace_bytes, stream, num_sms);
}

// Last-wave split workspace: status word | (m, l) fp32 pairs [P][n_tail][128] |
// partial outputs fp32 [P][n_tail][128][128]
size_t fp8attn_fwd_tail_workspace_bytes(int B, int T, int H, int num_sms) {
  if (!shape_ok(B, T, H, kHeadDim) || num_sms < 1) return 0;
  int n_tail = 0, lo[kMaxTailParts + 1];
  const int parts = tail_plan(B, T, H, num_sms, &n_tail, lo);
  if (parts < 2) return kStatusBytes;
  const size_t rows = static_cast<size_t>(parts) * n_tail * kTile;
  return round16(kStatusBytes + rows * 8) + rows * kHeadDim * 4;
}

int fp8attn_fwd_tail_plan(int B, int T, int H, int num_sms, int* n_tail, int* part_lo) {
  int nt = 0, lo[kMaxTailParts + 1];
  const int parts = tail_plan(B, T, H, num_sms, &nt, lo);
  if (n_tail) *n_tail = nt;
  if (part_lo && parts >= 2)
    for (int k = 0; k <= parts; ++k) part_lo[k] = lo[k];
  return parts;
}

fp8attn_status fp8attn_e2m1_encode(const float* x, uint8_t* codes, size_t n, void* stream) {
  if (n == 0) return FP8ATTN_OK;
  if (!x || !codes || (reinterpret_cast<uintptr_t>(x) & 3u)) return FP8ATTN_ERR_INVALID_ARG;
  fp8attn_status st = check_device();
  if (st != FP8ATTN_OK) return st;
  return launch_e2m1_encode(x, codes, n, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? FP8ATTN_OK : FP8ATTN_ERR_CUDA;
}

fp8attn_status fp8attn_e4m3_encode(const float* x, uint8_t* codes, size_t n, void* stream) {
  if (n == 0) return FP8ATTN_OK;
  if (!x || !codes || (reinterpret_cast<uintptr_t>(x) & 3u)) return FP8ATTN_ERR_INVALID_ARG;
  fp8attn_status st = check_device();
  if (st != FP8ATTN_OK) return st;
  return launch_e4m3_encode(x, codes, n, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? FP8ATTN_OK : FP8ATTN_ERR_CUDA;
}

fp8attn_status fp8attn_selftest_wait_timeout(void* workspace, unsigned long long limit_ns, void* stream) {
  if (!workspace || !aligned16(workspace)) return FP8ATTN_ERR_WORKSPACE;
  if (limit_ns < 100000ull || limit_ns > kWaitLimitNs) return FP8ATTN_ERR_INVALID_ARG;
  fp8attn_status st = check_device();
  if (st != FP8ATTN_OK) return st;
  return launch_selftest_wait(static_cast<int*>(workspace), limit_ns, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? FP8ATTN_OK
             : FP8ATTN_ERR_CUDA;
}

fp8attn_status fp8attn_check_status(void* workspace, void* stream) {
  if (!workspace) return FP8ATTN_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int word = 0;
  if (cudaMemcpyAsync(&word, workspace, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return FP8ATTN_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return FP8ATTN_ERR_CUDA;
  if (word == 0) return FP8ATTN_OK;
  if (cudaMemsetAsync(workspace, 0, sizeof(int), s) != cudaSuccess) return FP8ATTN_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return FP8ATTN_ERR_CUDA;
  if (word == kStatusBadTile) return FP8ATTN_ERR_BAD_TILE_LIST;
  if (word == kStatusBadPerm) return FP8ATTN_ERR_BAD_PERMUTATION;
  return FP8ATTN_ERR_DEVICE_TIMEOUT;
}

}  // extern "C"
