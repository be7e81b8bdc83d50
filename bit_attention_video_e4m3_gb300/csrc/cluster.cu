// Online V clustering that produces the V-Smooth token permutation
// (VC-Attention news article, section 2, first step of V-Smooth: value tokens
// of one head are clustered on a few representative dimensions, and the
// tokens of a cluster are laid out contiguously so that the 128-row blocks of
// the prep hold similar rows; clusters need not be balanced).
//
// Per (batch, head):
//   1. amax_c = max_t |v[t,c]| over the head's tokens;
//   2. the r channels of largest amax (ties: lower channel) are the
//      representative dimensions; channel d with 2^E_d <= amax_d < 2^(E_d+1)
//      gives 12-bit codes rne(v * 2^(11 - E_d)) (exact scaling, |code| <= 4096);
//   3. Lloyd's k-means on the codes: seeds are tokens floor(k T / K); a token
//      joins the nearest centroid (squared Euclidean distance, ties to the
//      lower cluster); a centroid moves to the floor of its members' mean,
//      an empty cluster keeps its centroid; `iters` rounds of move + assign;
//   4. perm = stable sort of the tokens by cluster id.
// Everything after the code conversion is integer arithmetic, so the result
// does not depend on the order of any sum.
#include <climits>

#include "kernels.cuh"

namespace fp8attn {
namespace {

constexpr int kChunk = 1024;          // tokens per CTA in the assign and scatter kernels
constexpr int kNoScale = -100000;     // exponent marker of a channel of zeros
constexpr uint8_t kNoLabel = 255;

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// E with 2^E <= a < 2^(E+1) for a finite a > 0 (subnormals included).
__device__ __forceinline__ int exponent_of(float a) {
  const uint32_t b = __float_as_uint(a);
  const int e = static_cast<int>((b >> 23) & 0xFFu);
  if (e) return e - 127;
  return (31 - __clz(static_cast<int>(b & 0x7FFFFFu))) - 149;
}

// The fixed-point code of x in a channel of exponent E: x * 2^(11 - E) is
// exact (|x| < 2^(E+1), so the result is below 2^12; a result that would be
// subnormal is below 1/2 and rounds to 0 in any case), rounded to nearest even.
__device__ __forceinline__ int code_of(float x, int E) {
  if (E == kNoScale) return 0;
  return __float2int_rn(ldexpf(x, 11 - E));
}

__device__ __forceinline__ size_t v_index(const ClusterParams& p, int b, int t, int h) {
  return ((static_cast<size_t>(b) * p.T + t) * p.H + h) * kHeadDim;
}

// grid (ceil(T/128), H, B), 256 threads: per-channel max |v|.
__global__ void __launch_bounds__(256) cluster_amax_kernel(const ClusterParams p) {
  __shared__ float s_red[8][kHeadDim];
  const int j = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  const int t0 = j * 128;
  const int n = min(128, p.T - t0);
  float am[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
  for (int r = w; r < n; r += 8) {
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(p.v + v_index(p, b, t0 + r, h)) + l);
    am[0] = fmaxf(am[0], fabsf(bf16_lo(u.x)));
    am[1] = fmaxf(am[1], fabsf(bf16_hi(u.x)));
    am[2] = fmaxf(am[2], fabsf(bf16_lo(u.y)));
    am[3] = fmaxf(am[3], fabsf(bf16_hi(u.y)));
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) s_red[w][4 * l + k] = am[k];
  __syncthreads();
  if (threadIdx.x < kHeadDim) {
    float m = s_red[0][threadIdx.x];
#pragma unroll
    for (int ww = 1; ww < 8; ++ww) m = fmaxf(m, s_red[ww][threadIdx.x]);
    atomicMax(p.amax + (static_cast<size_t>(b) * p.H + h) * kHeadDim + threadIdx.x, __float_as_uint(m));
  }
}

// grid (B*H), 128 threads: representative dimensions, seed centroids, zeroed sums.
__global__ void __launch_bounds__(128) cluster_setup_kernel(const ClusterParams p) {
  __shared__ float s_am[kHeadDim];
  __shared__ int s_sel[kHeadDim];
  __shared__ int s_dims[kClusterMaxDims], s_exp[kClusterMaxDims];
  const int bh = blockIdx.x, b = bh / p.H, h = bh % p.H;
  const int c = threadIdx.x;
  const float a = __uint_as_float(p.amax[static_cast<size_t>(bh) * kHeadDim + c]);
  s_am[c] = a;
  __syncthreads();
  int rank = 0;
  for (int c2 = 0; c2 < kHeadDim; ++c2) {
    const float a2 = s_am[c2];
    rank += (a2 > a) || (a2 == a && c2 < c);
  }
  const bool sel = rank < p.r;
  s_sel[c] = sel;
  __syncthreads();
  if (sel) {
    int pos = 0;
    for (int c2 = 0; c2 < c; ++c2) pos += s_sel[c2];
    s_dims[pos] = c;
    s_exp[pos] = a > 0.f ? exponent_of(a) : kNoScale;
  }
  __syncthreads();
  if (c < kClusterMaxDims) {
    p.dims[bh * kClusterMaxDims + c] = c < p.r ? s_dims[c] : 0;
    p.dim_exp[bh * kClusterMaxDims + c] = c < p.r ? s_exp[c] : kNoScale;
  }
  const size_t cbase = static_cast<size_t>(bh) * kClusterMaxK * kClusterMaxDims;
  for (int idx = c; idx < kClusterMaxK * kClusterMaxDims; idx += blockDim.x) {
    const int k = idx / kClusterMaxDims, d = idx % kClusterMaxDims;
    int val = 0;
    if (k < p.K && d < p.r) {
      const int t = static_cast<int>((static_cast<long long>(k) * p.T) / p.K);
      const uint16_t raw = reinterpret_cast<const uint16_t*>(p.v)[v_index(p, b, t, h) + s_dims[d]];
      val = code_of(__uint_as_float(static_cast<uint32_t>(raw) << 16), s_exp[d]);
    }
    p.cent[cbase + idx] = val;
    p.sums[cbase + idx] = 0;
  }
  if (c < kClusterMaxK) p.counts[bh * kClusterMaxK + c] = 0;
}

// grid (nchunks, B*H), 256 threads, 4 tokens per thread.  FROM_V: convert the
// tokens' representative values to codes (and store them); else read codes.
// RS: code row stride (8 or 16 int16).  Assigns labels and accumulates the
// members' code sums and counts; writes the chunk's label histogram.
// The nearest centroid minimises |c|^2 - 2 x.c, which differs from |x - c|^2
// by the token's own |x|^2: the same integer order, the same ties.
template <bool FROM_V, int RS>
__global__ void __launch_bounds__(256) cluster_assign_kernel(const ClusterParams p) {
  constexpr int kTok = kChunk / 256;
  __shared__ __align__(16) int s_cent[kClusterMaxK][RS];
  __shared__ int s_cn[kClusterMaxK];
  __shared__ int s_sum[kClusterMaxK][RS];
  __shared__ int s_cnt[kClusterMaxK];
  __shared__ int s_dims[kClusterMaxDims], s_exp[kClusterMaxDims];
  const int chunk = blockIdx.x, bh = blockIdx.y, b = bh / p.H, h = bh % p.H;
  const size_t cbase = static_cast<size_t>(bh) * kClusterMaxK * kClusterMaxDims;
  for (int idx = threadIdx.x; idx < kClusterMaxK * RS; idx += blockDim.x) {
    const int k = idx / RS, d = idx % RS;
    s_cent[k][d] = p.cent[cbase + k * kClusterMaxDims + d];
    s_sum[k][d] = 0;
  }
  if (threadIdx.x < kClusterMaxDims) {
    s_dims[threadIdx.x] = p.dims[bh * kClusterMaxDims + threadIdx.x];
    s_exp[threadIdx.x] = p.dim_exp[bh * kClusterMaxDims + threadIdx.x];
  }
  __syncthreads();
  if (threadIdx.x < kClusterMaxK) {
    int n2 = 0;                                   // |c|^2 <= 16 * 4096^2 = 2^28
#pragma unroll
    for (int d = 0; d < RS; ++d) n2 += s_cent[threadIdx.x][d] * s_cent[threadIdx.x][d];
    s_cn[threadIdx.x] = n2;
    s_cnt[threadIdx.x] = 0;
  }

  int c[kTok][RS];
  bool valid[kTok];
#pragma unroll
  for (int i = 0; i < kTok; ++i) {
    const int t = chunk * kChunk + i * 256 + threadIdx.x;
    valid[i] = t < p.T;
    const int tt = valid[i] ? t : 0;
    int16_t* row = p.codes + (static_cast<size_t>(bh) * p.T + tt) * RS;
    if (FROM_V) {
      const uint16_t* vrow = reinterpret_cast<const uint16_t*>(p.v) + v_index(p, b, tt, h);
#pragma unroll
      for (int d = 0; d < RS; ++d)
        c[i][d] = (valid[i] && d < p.r)
                      ? code_of(__uint_as_float(static_cast<uint32_t>(__ldg(vrow + s_dims[d])) << 16), s_exp[d])
                      : 0;
      if (valid[i]) {
        uint32_t packed[RS / 2];
#pragma unroll
        for (int d = 0; d < RS / 2; ++d)
          packed[d] = (static_cast<uint32_t>(c[i][2 * d]) & 0xFFFFu) | (static_cast<uint32_t>(c[i][2 * d + 1]) << 16);
#pragma unroll
        for (int q = 0; q < RS / 8; ++q)
          reinterpret_cast<uint4*>(row)[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2],
                                                        packed[4 * q + 3]);
      }
    } else {
#pragma unroll
      for (int q = 0; q < RS / 8; ++q) {
        const uint4 u = valid[i] ? reinterpret_cast<const uint4*>(row)[q] : make_uint4(0, 0, 0, 0);
        const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          c[i][8 * q + 2 * e] = static_cast<int16_t>(w4[e] & 0xFFFFu);
          c[i][8 * q + 2 * e + 1] = static_cast<int16_t>(w4[e] >> 16);
        }
      }
    }
  }
  __syncthreads();                                // s_cn, s_cnt ready

  int best[kTok], lab[kTok];
#pragma unroll
  for (int i = 0; i < kTok; ++i) {
    best[i] = INT_MAX;
    lab[i] = 0;
  }
  for (int k = 0; k < p.K; ++k) {
    int cc[RS];
#pragma unroll
    for (int q = 0; q < RS / 4; ++q) {
      const int4 v4 = reinterpret_cast<const int4*>(&s_cent[k][0])[q];
      cc[4 * q] = v4.x;
      cc[4 * q + 1] = v4.y;
      cc[4 * q + 2] = v4.z;
      cc[4 * q + 3] = v4.w;
    }
    const int cn = s_cn[k];
#pragma unroll
    for (int i = 0; i < kTok; ++i) {
      int dot = 0;                                // |x.c| <= 2^28
#pragma unroll
      for (int d = 0; d < RS; ++d) dot += c[i][d] * cc[d];
      const int sc = cn - 2 * dot;
      if (sc < best[i]) {
        best[i] = sc;
        lab[i] = k;
      }
    }
  }
#pragma unroll
  for (int i = 0; i < kTok; ++i) {
    if (!valid[i]) continue;
    const int t = chunk * kChunk + i * 256 + threadIdx.x;
    p.labels8[static_cast<size_t>(bh) * p.T + t] = static_cast<uint8_t>(lab[i]);
#pragma unroll
    for (int d = 0; d < RS; ++d)
      if (d < p.r) atomicAdd(&s_sum[lab[i]][d], c[i][d]);      // <= 1024 * 4096 per chunk
    atomicAdd(&s_cnt[lab[i]], 1);
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < p.K * RS; idx += blockDim.x) {
    const int k = idx / RS, d = idx % RS;
    const int sv = s_sum[k][d];
    if (d < p.r && sv != 0)
      atomicAdd(reinterpret_cast<unsigned long long*>(p.sums + cbase + k * kClusterMaxDims + d),
                static_cast<unsigned long long>(static_cast<long long>(sv)));
  }
  if (threadIdx.x < p.K) {
    const int n = s_cnt[threadIdx.x];
    p.hist[(static_cast<size_t>(bh) * p.nchunks + chunk) * kClusterMaxK + threadIdx.x] = n;
    if (n) atomicAdd(p.counts + bh * kClusterMaxK + threadIdx.x, n);
  }
}

// grid (B*H), K*16 threads: centroid = floor(sum / count); sums and counts reset.
__global__ void cluster_move_kernel(const ClusterParams p) {
  const int bh = blockIdx.x;
  const int k = threadIdx.x / kClusterMaxDims, d = threadIdx.x % kClusterMaxDims;
  const size_t i = static_cast<size_t>(bh) * kClusterMaxK * kClusterMaxDims + threadIdx.x;
  const int n = p.counts[bh * kClusterMaxK + k];
  if (d < p.r && n > 0) {
    const long long S = p.sums[i];
    long long q = S / n;
    if (S % n != 0 && S < 0) --q;                  // floor, not truncation
    p.cent[i] = static_cast<int>(q);
  }
  p.sums[i] = 0;
  __syncthreads();
  if (d == 0) p.counts[bh * kClusterMaxK + k] = 0;
}

// grid (B*H), 64 threads: chunk histograms -> the first output position of
// each (chunk, cluster) (clusters in index order, chunks in token order).
__global__ void __launch_bounds__(64) cluster_scan_kernel(const ClusterParams p) {
  __shared__ int s_tot[kClusterMaxK];
  const int bh = blockIdx.x, k = threadIdx.x;
  int* hist = p.hist + static_cast<size_t>(bh) * p.nchunks * kClusterMaxK;
  int tot = 0;
  if (k < p.K)
    for (int c = 0; c < p.nchunks; ++c) tot += hist[c * kClusterMaxK + k];
  s_tot[k] = tot;
  __syncthreads();
  int run = 0;
  for (int k2 = 0; k2 < k; ++k2) run += s_tot[k2];
  if (k < p.K)
    for (int c = 0; c < p.nchunks; ++c) {
      const int n = hist[c * kClusterMaxK + k];
      hist[c * kClusterMaxK + k] = run;
      run += n;
    }
}

// grid (nchunks, B*H), 256 threads: stable scatter.  Warp w owns tokens
// [w*128, w*128+128) of the chunk and walks them 32 at a time in order; lanes
// with the same label are ranked by lane index.
__global__ void __launch_bounds__(256) cluster_scatter_kernel(const ClusterParams p) {
  __shared__ int s_wc[8][kClusterMaxK];
  const int chunk = blockIdx.x, bh = blockIdx.y;
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  for (int idx = threadIdx.x; idx < 8 * kClusterMaxK; idx += blockDim.x) (&s_wc[0][0])[idx] = 0;
  __syncthreads();
  const int tw = chunk * kChunk + w * 128;
  const uint8_t* lab8 = p.labels8 + static_cast<size_t>(bh) * p.T;
  for (int rnd = 0; rnd < 4; ++rnd) {
    const int t = tw + rnd * 32 + l;
    const int lab = t < p.T ? lab8[t] : kNoLabel;
    const unsigned peers = __match_any_sync(0xFFFFFFFFu, lab);
    if (lab != kNoLabel && l == __ffs(peers) - 1) s_wc[w][lab] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  if (threadIdx.x < p.K) {
    int run = p.hist[(static_cast<size_t>(bh) * p.nchunks + chunk) * kClusterMaxK + threadIdx.x];
    for (int ww = 0; ww < 8; ++ww) {
      const int n = s_wc[ww][threadIdx.x];
      s_wc[ww][threadIdx.x] = run;
      run += n;
    }
  }
  __syncthreads();
  int32_t* perm = p.perm + static_cast<size_t>(bh) * p.T;
  for (int rnd = 0; rnd < 4; ++rnd) {
    const int t = tw + rnd * 32 + l;
    const int lab = t < p.T ? lab8[t] : kNoLabel;
    const unsigned peers = __match_any_sync(0xFFFFFFFFu, lab);
    if (lab != kNoLabel) {
      const int pos = s_wc[w][lab] + __popc(peers & ((1u << l) - 1u));
      perm[pos] = t;
      if (p.labels) p.labels[static_cast<size_t>(bh) * p.T + t] = lab;
    }
    __syncwarp();
    if (lab != kNoLabel && l == __ffs(peers) - 1) s_wc[w][lab] += __popc(peers);
    __syncwarp();
  }
}

template <int RS>
cudaError_t run_lloyd(const ClusterParams& p, cudaStream_t s) {
  const int BH = p.B * p.H;
  const dim3 g(p.nchunks, BH);
  cluster_assign_kernel<true, RS><<<g, 256, 0, s>>>(p);
  for (int it = 0; it < p.iters; ++it) {
    cluster_move_kernel<<<BH, kClusterMaxK * kClusterMaxDims, 0, s>>>(p);
    cluster_assign_kernel<false, RS><<<g, 256, 0, s>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace

int cluster_code_stride(int r) { return r <= 8 ? 8 : 16; }

cudaError_t launch_cluster(const ClusterParams& p, cudaStream_t s) {
  const int BH = p.B * p.H;
  cudaError_t e = cudaMemsetAsync(p.amax, 0, static_cast<size_t>(BH) * kHeadDim * sizeof(uint32_t), s);
  if (e != cudaSuccess) return e;
  cluster_amax_kernel<<<dim3((p.T + 127) / 128, p.H, p.B), 256, 0, s>>>(p);
  cluster_setup_kernel<<<BH, kHeadDim, 0, s>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = cluster_code_stride(p.r) == 8 ? run_lloyd<8>(p, s) : run_lloyd<16>(p, s);
  if (e != cudaSuccess) return e;
  cluster_scan_kernel<<<BH, kClusterMaxK, 0, s>>>(p);
  cluster_scatter_kernel<<<dim3(p.nchunks, BH), 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace fp8attn
