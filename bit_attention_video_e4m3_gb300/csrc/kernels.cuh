// Internal interface between the C-ABI layer (api.cu) and the kernels.
#pragma once
#include <atomic>
#include <cstdint>
#include <mutex>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace fp8attn {

constexpr int kHeadDim = 128;
constexpr int kQKBlock = 64;    // tokens per Q/K scale block
constexpr int kVBlock = 128;    // rows per V-Smooth block
constexpr int kMaxTailParts = 4; // parts of a last-wave query tile
constexpr int kTile = 128;      // query rows per CTA and keys per KV tile

// Device status word values (written into the caller's workspace).
constexpr int kStatusOk = 0;
constexpr int kStatusTimeout = 1;
constexpr int kStatusBadTile = 2;
constexpr int kStatusBadPerm = 3;

// One-time set-up per device (kernel attributes such as the dynamic
// shared-memory limit apply to the current device only).  Safe when several
// host threads make their first call at once; later calls cost one atomic load.
class PerDeviceOnce {
 public:
  template <class F>
  cudaError_t run(F&& setup) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    const uint64_t bit = 1ull << dev;
    if (done_.load(std::memory_order_acquire) & bit) return cudaSuccess;
    std::lock_guard<std::mutex> lock(mu_);
    if (done_.load(std::memory_order_relaxed) & bit) return cudaSuccess;
    e = setup();
    if (e == cudaSuccess) done_.fetch_or(bit, std::memory_order_release);
    return e;
  }

 private:
  std::mutex mu_;
  std::atomic<uint64_t> done_{0};
};

struct PrepParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const int32_t* perm;        // [B,H,T] or null
  uint8_t* q8;
  uint8_t* k8;
  uint8_t* v8;                // [B,H,128,Tpad]
  float* q_scale;             // [B,H,nQK]
  float* k_scale;
  float* v_scale;             // [B,H,128]
  __nv_bfloat16* v_mean;      // [B,H,nV,128]
  uint32_t* v_amax;           // workspace [B,H,128], fp32 bits of the channel max |R|
  int* status;                // workspace status word, or null (no report)
  // sequence-mean smoothing (workspace arrays of [2][B*H*128]: index 0 = K, 1 = V)
  uint32_t* chan_max;         // fp32 bits of max|x| over T
  unsigned long long* chan_sum;  // fixed-point sums (two's complement)
  float* chan_low;            // values below the fixed-point window
  float* chan_mean;           // exact means rounded to fp32
  float* vbias_acc;           // [B*H*128] sum over tokens of (dequantised V' - V')
  float* v_offset;            // output [B,H,128] or null
  int smooth, v_bias, sum_window;
  int v_fp4;                  // 1: V residual as NVFP4 (v4, v4_sf) instead of E4M3 (v8)
  uint8_t* v4;                // [B,H,128,Tpad/2] packed E2M1, token-contiguous (even token in the low nibble)
  uint8_t* v4_sf;             // [B,H,nV][2][32][16] UE4M3 block scales in tcgen05.cp 32x128b.warpx4 order
  int B, T, H, nQK, nV, Tpad, vsmooth;
};

struct AttnParams {
  CUtensorMap tm_q;           // uint8 {128, H, T, B}, box {128,1,128,1}, 128B swizzle
  CUtensorMap tm_k;           // same layout as tm_q
  CUtensorMap tm_v;           // uint8 {Tpad, 128, B*H}, box {128,128,1}, 128B swizzle
  const float* q_scale;
  const float* k_scale;
  const float* v_scale;
  const __nv_bfloat16* v_mean;
  const float* v_offset;      // [B,H,128] added to every output row, or null
  __nv_bfloat16* out;
  const int32_t* row_ptr;     // null = dense
  const int32_t* col;
  int* status;
  int B, T, H, nQK, nV, nQt;
  int reverse, pcast, vsmooth;
  float log2_pscale;          // log2(S)
  float beta;                 // ExpCast beta
  float sm_scale_log2;        // softmax_scale * log2(e)
  unsigned long long timeout_ns;
  int n_splits;               // split-KV parts per query tile (1: no split)
  float* part_o;              // [n_splits][B*H][T][128] fp32 partial outputs (n_splits > 1)
  float2* part_ml;            // [n_splits][B*H][T] (running max, row sum) of each part
  int fp4;                    // 1: 4-bit PV product (tm_v maps the packed E2M1 V, v4_sf its scales)
  const uint8_t* v4_sf;       // [B,H,nV][1024] UE4M3 block scales of the E2M1 V
  // Last-wave split (dense 8-bit PV only).  CTA c = qt + nQt (h + H b) is the
  // linear index of a query tile.  The plain launch leaves the CTAs from
  // cta_limit on to a split launch (tail_cta0 = cta_limit, grid {n_tail, 1,
  // n_splits}) whose part s covers key-tile positions [part_lo[s],
  // part_lo[s + 1]) after max-only steps over positions [0, part_lo[s]).
  int cta_limit;              // plain launch: CTAs with c >= cta_limit return at once
  int tail_cta0;              // split launch of the last wave: its first c; -1 otherwise
  int n_tail;                 // query tiles of that launch
  int part_lo[kMaxTailParts + 1];
};

// Online V clustering (the V-Smooth permutation).
constexpr int kClusterMaxK = 64;      // clusters
constexpr int kClusterMaxDims = 16;   // representative dimensions

struct ClusterParams {
  const __nv_bfloat16* v;     // [B,T,H,128]
  int B, T, H;
  int K, r, iters;
  int nchunks;                // ceil(T / 1024)
  uint32_t* amax;             // [BH][128] fp32 bits of max |v|
  int* dims;                  // [BH][16] representative channels, ascending
  int* dim_exp;               // [BH][16] exponent of each channel's max
  int16_t* codes;             // [BH][T][stride] fixed-point codes
  int* cent;                  // [BH][64][16] centroids
  long long* sums;            // [BH][64][16] member code sums
  int* counts;                // [BH][64] member counts
  int* hist;                  // [BH][nchunks][64] label counts per chunk, then scatter bases
  uint8_t* labels8;           // [BH][T]
  int32_t* perm;              // [B,H,T]
  int32_t* labels;            // [B,H,T] or null
};

int cluster_code_stride(int r);
cudaError_t launch_cluster(const ClusterParams& p, cudaStream_t stream);

cudaError_t launch_prep(const PrepParams& p, cudaStream_t stream);
size_t prep_v_smem_bytes();
cudaError_t launch_e2m1_encode(const float* x, uint8_t* codes, size_t n, cudaStream_t stream);
cudaError_t launch_e4m3_encode(const float* x, uint8_t* codes, size_t n, cudaStream_t stream);
cudaError_t launch_attn(const AttnParams& p, cudaStream_t stream);
cudaError_t launch_selftest_wait(int* status, unsigned long long limit_ns, cudaStream_t stream);
size_t attn_smem_bytes();

}  // namespace fp8attn
