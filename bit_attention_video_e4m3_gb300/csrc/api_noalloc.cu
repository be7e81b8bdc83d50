// fp8attn_prep_noalloc: the stage-1 prep for callers that cannot allocate
// device memory.  fp8attn_prep needs a caller-provided device workspace for the
// per-(batch, head, channel) residual maxima of the V prep.  Some callers have
// no way to provide one: code that runs where allocation is forbidden after
// start-up (a serving loop with a fixed memory budget, a plugin inside a host
// framework that owns every device allocation), or C code that has no
// allocator of its own at hand.  This entry point keeps that scratch in a
// fixed array compiled into the library instead, so the caller passes only
// inputs and outputs.
//
// Limits and sharing:
//   - the array holds FP8ATTN_NOALLOC_MAX_BH (batch, head) pairs of 128 fp32
//     maxima (1 MiB); every GPU that loads the library holds one copy of it
//     until the process exits;
//   - every call on a device uses the same array, so calls whose work overlaps
//     on the GPU (different streams, or different host threads) race; order
//     them on one stream or synchronise between them;
//   - the first call on each device looks up the array's device address
//     (cudaGetSymbolAddress) with that device current; make that first call
//     before any stream capture starts;
//   - there is no status word (that lives in a workspace), so a permutation
//     entry outside [0, T) is handled on the device as in fp8attn_prep but
//     not reported to the caller.
#include <mutex>

#include "../../include/fp8attn.h"
#include "kernels.cuh"

using namespace fp8attn;

namespace {

static __device__ __align__(256) uint32_t g_prep_scratch[FP8ATTN_NOALLOC_MAX_BH * kHeadDim];

std::mutex g_scratch_mu;
uint32_t* g_scratch_addr[64] = {};   // device address of g_prep_scratch per device ordinal

fp8attn_status scratch_for_current_device(uint32_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FP8ATTN_ERR_CUDA;
  if (dev < 0 || dev >= 64) return FP8ATTN_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_prep_scratch) != cudaSuccess) return FP8ATTN_ERR_CUDA;
    g_scratch_addr[dev] = static_cast<uint32_t*>(addr);
  }
  *out = g_scratch_addr[dev];
  return FP8ATTN_OK;
}

fp8attn_status device_is_sm103() {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return FP8ATTN_ERR_CUDA;
  return (major == 10 && minor == 3) ? FP8ATTN_OK : FP8ATTN_ERR_UNSUPPORTED_DEVICE;
}

bool is_aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" fp8attn_status fp8attn_prep_noalloc(const void* q, const void* k, const void* v, int B,
                                               int T, int H, int D, const int32_t* perm,
                                               int vsmooth, const fp8attn_prepped* out,
                                               void* stream) {
  if (B < 1 || T < 1 || H < 1 || D != kHeadDim || H > 65535 || B > 32767)
    return FP8ATTN_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * T * H > 0x7FFFFFFFll) return FP8ATTN_ERR_INVALID_ARG;
  if (!q || !k || !v || !out || !out->q8 || !out->k8 || !out->v8 || !out->q_scale ||
      !out->k_scale || !out->v_scale || !out->v_mean)
    return FP8ATTN_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, out->q8, out->k8, out->v8, out->q_scale, out->k_scale,
                        out->v_scale, out->v_mean};
  for (const void* ptr : ptrs)
    if (!is_aligned16(ptr)) return FP8ATTN_ERR_INVALID_ARG;
  if (out->v_offset && !is_aligned16(out->v_offset)) return FP8ATTN_ERR_INVALID_ARG;
  if (perm && (reinterpret_cast<uintptr_t>(perm) & 3u)) return FP8ATTN_ERR_INVALID_ARG;
  // the fixed scratch covers FP8ATTN_NOALLOC_MAX_BH (batch, head) pairs
  if (static_cast<long long>(B) * H > FP8ATTN_NOALLOC_MAX_BH) return FP8ATTN_ERR_WORKSPACE;
  fp8attn_status st = device_is_sm103();
  if (st != FP8ATTN_OK) return st;
  uint32_t* amax = nullptr;
  st = scratch_for_current_device(&amax);
  if (st != FP8ATTN_OK) return st;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
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
  p.v_amax = amax;
  p.status = nullptr;                         // no workspace to report into (see the header)
  p.chan_max = nullptr;                       // no sequence-mean smoothing here
  p.chan_sum = nullptr;
  p.chan_low = nullptr;
  p.chan_mean = nullptr;
  p.vbias_acc = nullptr;
  p.v_offset = out->v_offset;                 // written with zeros when set
  p.smooth = 0;
  p.v_bias = 0;
  p.v_fp4 = 0;
  p.v4 = nullptr;
  p.v4_sf = nullptr;
  p.sum_window = 0;
  p.B = B;
  p.T = T;
  p.H = H;
  p.nQK = (T + kQKBlock - 1) / kQKBlock;
  p.nV = (T + kVBlock - 1) / kVBlock;
  p.Tpad = p.nV * kVBlock;
  p.vsmooth = vsmooth ? 1 : 0;
  // the maxima accumulate with atomicMax, so the part this call uses starts at zero;
  // the array keeps whatever the previous call left in it
  if (cudaMemsetAsync(amax, 0, static_cast<size_t>(B) * H * kHeadDim * sizeof(uint32_t), s) !=
      cudaSuccess)
    return FP8ATTN_ERR_CUDA;
  return launch_prep(p, s) == cudaSuccess ? FP8ATTN_OK : FP8ATTN_ERR_CUDA;
}
