/*
 * fp8attn — block-scaled FP8 (E4M3) attention forward for long video-DiT
 * sequences at head dim 128, on sm_103a (GB300).
 *
 * Two stages, each one call:
 *   fp8attn_prep  bf16 Q/K/V  ->  E4M3 codes + fp32 scales (+ bf16 V block means)
 *   fp8attn_fwd   prepared operands  ->  bf16 attention output
 *
 * Conventions shared by every call
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library
 *     never allocates device memory and keeps no state between calls (except
 *     fp8attn_prep_noalloc, whose scratch is a fixed array inside the library).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls are stream-ordered and asynchronous: argument errors are
 *     reported synchronously by the return value; errors found by a kernel
 *     while it runs (a bounded wait that expired, a tile index or permutation
 *     entry out of range) are written to a status word inside the caller's
 *     workspace and read back with fp8attn_check_status.
 *   - Shapes follow the pages: Q, K, V and the output are [B, T, H, D] with
 *     D = 128 (row-major, D contiguous).  nQK = ceil(T/64), nV = ceil(T/128),
 *     Tpad = 128 * nV.
 *   - Pointers must be 16-byte aligned.  T, H, B must be >= 1 (T >= 1), and
 *     B * H * T must fit in 31 bits.
 *   - The device must be compute capability 10.3 (sm_103); other devices get
 *     FP8ATTN_ERR_UNSUPPORTED_DEVICE.
 */
#ifndef FP8ATTN_H_
#define FP8ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FP8ATTN_OK = 0,
  FP8ATTN_ERR_INVALID_ARG = 1,        /* bad shape, null or misaligned pointer, bad scale */
  FP8ATTN_ERR_UNSUPPORTED_DEVICE = 2, /* current device is not sm_103 */
  FP8ATTN_ERR_CUDA = 3,               /* a CUDA runtime/driver call or a launch failed */
  FP8ATTN_ERR_DEVICE_TIMEOUT = 4,     /* a kernel's bounded wait expired (see check_status) */
  FP8ATTN_ERR_WORKSPACE = 5,          /* workspace null or smaller than *_workspace_bytes */
  FP8ATTN_ERR_BAD_TILE_LIST = 6,      /* a sparse tile index was outside [0, nV) */
  FP8ATTN_ERR_BAD_PERMUTATION = 7     /* a permutation entry was outside [0, T) */
} fp8attn_status;

typedef enum {
  FP8ATTN_PCAST_EXP2_CVT = 0, /* P code = E4M3_RNE_satfinite(S * exp(x - m)) */
  FP8ATTN_PCAST_EXPCAST = 1   /* P code = clamp(rne(8 z + 56 + beta), 0, 126), z = log2(S p) */
} fp8attn_pcast;

/* Outputs of fp8attn_prep / inputs of fp8attn_fwd (all device pointers). */
typedef struct {
  void* q8;        /* E4M3 [B, T, H, 128], queries in original token order               */
  void* k8;        /* E4M3 [B, T, H, 128], keys in permuted order (perm applied)           */
  void* v8;        /* E4M3 [B, H, 128, Tpad] residual codes, token-contiguous, permuted,
                      pad tokens = 0                                                       */
  float* q_scale;  /* [B, H, nQK]   amax(64-token block) / 448                              */
  float* k_scale;  /* [B, H, nQK]   same, over permuted key blocks                          */
  float* v_scale;  /* [B, H, 128]   amax over all tokens of the residual channel / 448       */
  void* v_mean;    /* bf16 [B, H, nV, 128] V-Smooth block means (zeros when vsmooth == 0)   */
  float* v_offset; /* [B, H, 128] added to every output row (sequence-mean smoothing of V
                      and the V bias correction), or NULL: nothing is added.  Written by
                      fp8attn_prep_smooth; the plain preps write zeros when it is set.  */
  void* v4;        /* NVFP4 V (fp8attn_prep_ex with v_format 1; NULL otherwise): packed E2M1
                      [B, H, 128, Tpad/2], token-contiguous, even token in the low nibble;
                      v_scale then holds amax / 2688 per channel                            */
  void* v4_sf;     /* UE4M3 block scales of v4, one per (channel, 16 tokens), 1024 bytes per
                      (batch, head, 128-token tile): [2 k-steps][32 rows][4 words][4 bytes],
                      word j of row l = channel 32 j + l, byte b = token block 4 k + b     */
} fp8attn_prepped;

/* One workspace size that serves fp8attn_prep, fp8attn_prep_smooth, fp8attn_prep_ex and
 * fp8attn_fwd (the larger of the two sizes below; split-KV needs
 * fp8attn_fwd_split_workspace_bytes).  0 for D != 128.  Host only. */
size_t fp8attn_workspace_size(int B, int T, int H, int D);

/* Bytes of device workspace fp8attn_prep and fp8attn_prep_smooth need (status word,
 * channel maxima, sequence statistics). */
size_t fp8attn_prep_workspace_bytes(int B, int T, int H);

/* Bytes of device workspace fp8attn_fwd needs (status word). */
size_t fp8attn_fwd_workspace_bytes(int B, int T, int H);

/* 128 * ceil(T / 128): the token extent of the v8 layout. */
size_t fp8attn_v_padded_T(int T);

/*
 * Stage 1: FP8 preparation of post-RoPE bf16 Q, K, V.
 *
 * TeleFuser "FP8 Sol-Attn" blog, section "FP8 Preparation for attention"
 * (per-(batch, head, 64-token block) Q/K scale = max|block| / 448; per-channel
 * V scale over all tokens; V stored token-contiguous for the PV product), and
 * the VC-Attention news article, section 2 "V-Smooth" (rows gathered by a token
 * permutation, 128-row block mean removed and kept as a 16-bit vector, only
 * the residual quantised).
 *
 *   q, k, v   bf16 [B, T, H, 128] device pointers (read only)
 *   perm      int32 [B, H, T] token permutation or NULL (identity).  It
 *             reorders K and V rows together; Q keeps its order.  Entries
 *             must be a permutation of 0..T-1.  An entry outside [0, T) is
 *             read as token 0 (no access leaves the tensors) and makes
 *             fp8attn_check_status return FP8ATTN_ERR_BAD_PERMUTATION; a
 *             repeated entry is not detected (the rows are then simply
 *             those tokens).
 *   vsmooth   1: subtract the bf16 mean of every 128-row block of permuted V
 *             (the mean is written to out->v_mean); 0: no mean (v_mean is
 *             written with zeros and may be used or ignored).
 *   out       where to write; every pointer in it must be set.
 *   workspace device scratch of at least fp8attn_prep_workspace_bytes bytes,
 *             reused freely between calls on the same stream.
 * Scale arithmetic is IEEE fp32: s = amax / 448, code = E4M3_RNE_satfinite(
 * x * (448 / amax)); a block or channel with amax == 0 gets s = 0 and codes 0.
 * Block means are the exact mean rounded once to bf16 (nearest even) whenever
 * every nonzero value of a channel block lies within 2^37 of the block's
 * largest magnitude (otherwise the values below that window are added in fp32
 * and the mean is close but not guaranteed correctly rounded).
 * Errors: FP8ATTN_ERR_INVALID_ARG / _WORKSPACE / _UNSUPPORTED_DEVICE / _CUDA
 * are returned before any work is queued.  The prep kernels never wait on the
 * device; the only error they find while running is a permutation entry out of
 * range, left in the workspace's status word for fp8attn_check_status.
 */
fp8attn_status fp8attn_prep(const void* q, const void* k, const void* v, int B, int T, int H,
                            int D, const int32_t* perm, int vsmooth,
                            const fp8attn_prepped* out, void* workspace, size_t workspace_bytes,
                            void* stream);

/*
 * Stage 1 with sequence-mean smoothing (TeleFuser blog, section "Diffusion
 * precision guards": per head K' = K - mean_T(K), V' = V - mean_T(V), fp32
 * statistics fused into the E4M3 preparation, and the V mean bias measured
 * after the E4M3 rounding compensated).  Same arguments as fp8attn_prep, plus
 *   smooth   0: none (exactly fp8attn_prep), 1: centre K, 2: centre K and V
 *   v_bias   1: measure b_c = mean_t(dequantised V' - V') per channel and
 *            subtract it from the output; 0: no correction
 *   out->v_offset  fp32 [B, H, 128]: required (non-NULL, 16-byte aligned) when
 *            smooth == 2 or v_bias == 1; receives (smooth == 2 ? mean_T(V) : 0)
 *            - (v_bias ? b : 0), which fp8attn_fwd adds to every output row.
 * mean_T is the exact mean over the T tokens of one (batch, head, channel)
 * rounded once to fp32 (whenever the channel's nonzero values lie within
 * 2^W of its largest magnitude, W = min(37, 54 - ceil(log2 T)); values further below
 * are added in fp32); K' = fl32(K - mean), V' = fl32(V - mean).  Centring K
 * leaves the softmax unchanged (every logit of a row moves by the same
 * constant) and only improves the E4M3 quantisation of K.
 * Errors: as fp8attn_prep; FP8ATTN_ERR_INVALID_ARG also for smooth outside
 * 0..2, v_bias outside 0..1, or a missing out->v_offset.
 */
fp8attn_status fp8attn_prep_smooth(const void* q, const void* k, const void* v, int B, int T,
                                   int H, int D, const int32_t* perm, int vsmooth, int smooth,
                                   int v_bias, const fp8attn_prepped* out, void* workspace,
                                   size_t workspace_bytes, void* stream);

/*
 * Stage 1 with a choice of V residual format: v_format 0 is exactly
 * fp8attn_prep_smooth (E4M3 residual in out->v8); v_format 1 writes the
 * residual as NVFP4 for the 4-bit PV product (VC-Attention news article,
 * 4-bit V-Smooth configuration: 4-bit values with a scale per 16 elements):
 * per channel s_c = amax_c / 2688 (2688 = 6 x 448) into out->v_scale and
 * G_c = 2688 / amax_c; per (channel, 16-token block) the UE4M3 scale
 * sf = UE4M3(fl32(a G_c) * fl32(1/6)) (a = the block's largest |R|) into
 * out->v4_sf, and E2M1(R * fl32(G_c / sf)) codes into out->v4 (all fp32
 * arithmetic round to nearest, E2M1 and UE4M3 round to nearest even,
 * saturating).  Q and K are E4M3 as always.  out->v8 is not touched.
 * Errors: as fp8attn_prep_smooth; FP8ATTN_ERR_INVALID_ARG also for v_format
 * outside 0..1, v_format 1 with v_bias 1 (not offered for the 4-bit residual),
 * or a NULL / unaligned out->v4 or out->v4_sf with v_format 1.
 */
fp8attn_status fp8attn_prep_ex(const void* q, const void* k, const void* v, int B, int T, int H,
                               int D, const int32_t* perm, int vsmooth, int smooth, int v_bias,
                               int v_format, const fp8attn_prepped* out, void* workspace,
                               size_t workspace_bytes, void* stream);

/* E2M1 codes (one per byte, low nibble) of n fp32 values: the prep kernels'
 * conversion alone, round to nearest even, saturating at 6, sign kept.  Same
 * argument rules and errors as fp8attn_e4m3_encode. */
fp8attn_status fp8attn_e2m1_encode(const float* x, uint8_t* codes, size_t n, void* stream);

/*
 * Stage 2: FP8 attention mainloop.
 *
 * TeleFuser "FP8 Sol-Attn" blog, section "SM90 CuTe mainloop" (E4M3 QK and PV
 * with fp32 accumulation, scales applied before the online softmax, P cast to
 * E4M3, V channel scale applied after all PV products, bf16 output); VC-Attention
 * news article sections 2 and 3 (rank-one mean restore r_ij mu_j^T from the
 * block's row sum; ExpCast code c = round(8 z + 56 + beta)); P-Cast Precision
 * review, sections 3-5 (static P scale S, forward or reverse KV order);
 * FPSAttention article, section 2.2 (sliding-tile key lists).
 *
 *   in            prepared operands (fp8attn_prep output)
 *   tile_row_ptr  int32 [ceil(T/128) + 1] CSR row pointers over 128-row query
 *   tile_col      tiles and int32 [nnz] key-tile indices in [0, nV), device
 *                 pointers; both NULL = dense (every key tile).  Key tiles are
 *                 in permuted key order.  An empty list gives a zero output row.
 *   reverse_kv    0: visit the list (or 0..nV-1) in order; 1: backwards.
 *   pcast         fp8attn_pcast.
 *   p_scale       static P scale S, 1 <= S <= 448 (S = 256 recommended).
 *   expcast_beta  beta of the ExpCast map (page value -0.35), |beta| < 0.5.
 *   softmax_scale logit scale; <= 0 selects 1/sqrt(128).
 *   vsmooth       1: add the rank-one block-mean term from in->v_mean; 0: ignore it.
 *   out           bf16 [B, T, H, 128] device pointer (written).
 *   workspace     device scratch of at least fp8attn_fwd_workspace_bytes bytes.
 * The row max is updated exactly at every 128-key tile, so P * S <= S.
 */
fp8attn_status fp8attn_fwd(const fp8attn_prepped* in, int B, int T, int H, int D,
                           const int32_t* tile_row_ptr, const int32_t* tile_col, int reverse_kv,
                           int pcast, float p_scale, float expcast_beta, float softmax_scale,
                           int vsmooth, void* out, void* workspace, size_t workspace_bytes,
                           void* stream);

/*
 * Stage 2 with split-KV (TeleFuser "FP8 Sol-Attn" blog, mainloop feature list:
 * long-sequence split-KV, partial results merged by a log-sum-exp
 * reduction).  The visiting order of every query tile (dense, reversed or
 * the CSR list) is cut into n_splits contiguous parts, part s holding
 * positions [s*n/n_splits, (s+1)*n/n_splits); each part runs its own online
 * softmax (its own running max, so its P codes are cast against that max) in
 * its own CTA, writing O_s = acc_s * s_v / l_s, m_s and l_s to the workspace;
 * a merge kernel then forms O = sum_s w_s O_s / sum_s w_s with
 * w_s = l_s 2^(m_s - max m) over the parts that saw a key, adds
 * in->v_offset, and rounds to bf16.  n_splits == 1 is exactly fp8attn_fwd.
 * Splitting pays when B*H*ceil(T/128) query-tile CTAs leave SMs idle;
 * fp8attn_fwd_auto_splits gives this library's choice.
 *   n_splits   1..16, and B * n_splits <= 65535
 *   workspace  fp8attn_fwd_split_workspace_bytes(B, T, H, n_splits) bytes
 *              (n_splits * B * H * T * (8 + 512) bytes + 256 for n_splits > 1)
 * Other arguments and errors as fp8attn_fwd.
 */
fp8attn_status fp8attn_fwd_split(const fp8attn_prepped* in, int B, int T, int H, int D,
                                 const int32_t* tile_row_ptr, const int32_t* tile_col,
                                 int reverse_kv, int pcast, float p_scale, float expcast_beta,
                                 float softmax_scale, int vsmooth, int n_splits, void* out,
                                 void* workspace, size_t workspace_bytes, void* stream);
size_t fp8attn_fwd_split_workspace_bytes(int B, int T, int H, int n_splits);

/*
 * Stage 2 with a choice of PV precision: pv_format 0 is exactly
 * fp8attn_fwd_split; pv_format 1 runs the 4-bit PV product on the NVFP4 V of
 * fp8attn_prep_ex (v_format 1): P = 2688 * 2^(x - m) (p_scale is not used) is
 * cast to E2M1 with one UE4M3 scale per 16 keys of the tile (scale =
 * UE4M3(max * fl32(1/6)), code = E2M1(p * fl32(1/scale))), O += P V on the
 * block-scaled FP4 tensor-core MMA, the row sum is the sum of the decoded P,
 * and the output is O * v_scale / l (+ v_offset).  QK stays E4M3.  The pages'
 * 4-bit configuration does not use the ExpCast cast, so pcast must be
 * FP8ATTN_PCAST_EXP2_CVT with pv_format 1.
 * Errors: as fp8attn_fwd_split; FP8ATTN_ERR_INVALID_ARG also for pv_format
 * outside 0..1, or pv_format 1 with ExpCast or without in->v4 / in->v4_sf.
 */
fp8attn_status fp8attn_fwd_ex(const fp8attn_prepped* in, int B, int T, int H, int D,
                              const int32_t* tile_row_ptr, const int32_t* tile_col, int reverse_kv,
                              int pcast, float p_scale, float expcast_beta, float softmax_scale,
                              int vsmooth, int n_splits, int pv_format, void* out, void* workspace,
                              size_t workspace_bytes, void* stream);

/*
 * Host-only rule (no GPU call): the largest S with S * B*H*ceil(T/128) <=
 * num_sms (all parts in one wave), S <= ceil(T/128) / 8 (at least 8 key tiles
 * per part) and S <= 16; at least 1.  On GB300 this picks, for one head,
 * S = 4 at T = 4096 (31.1 -> 22.6 us) and S = 2 at T = 8192 (51.5 -> 38.4 us),
 * and no split from B*H*ceil(T/128) >= 76 query tiles on.
 */
int fp8attn_fwd_auto_splits(int B, int T, int H, int num_sms);

/*
 * Stage 2 with the last wave split (dense attention, 8-bit PV).  The
 * B*H*ceil(T/128) query tiles run num_sms at a time; when the last wave holds
 * n_tail <= num_sms / 2 of them, those query tiles are each cut into
 * P = min(4, num_sms / n_tail) parts of the visiting order (the key-tile
 * positions fp8attn_fwd_tail_plan gives) and run in a second launch, the
 * parts merged as in fp8attn_fwd_split.  Unlike fp8attn_fwd_split, a part
 * first takes the row maxima of the key tiles before its range (their QK
 * products only), so it enters its range with the running max of the unsplit
 * order and casts exactly the P codes of fp8attn_fwd (the method's P cast is
 * framed by that running max: TeleFuser "FP8 Sol-Attn" blog, SM90 CuTe
 * mainloop, and the VC-Attention news article, ExpCast-FP8); the result
 * differs from fp8attn_fwd only in fp32 rounding order (the log-sum-exp
 * merge), which can move an output by one bf16 step.  Without a split plan
 * (a single wave, whole waves only, or a last wave above num_sms / 2) this is
 * exactly fp8attn_fwd.
 *   num_sms    SMs of the device the call runs on (>= 1; any value is correct,
 *              the device's own count makes the split pay)
 *   workspace  fp8attn_fwd_tail_workspace_bytes(B, T, H, num_sms) bytes
 *              (P * n_tail * 128 * (8 + 512) bytes + 256 with a split plan)
 * Other arguments as fp8attn_fwd (no key-tile list, n_splits 1, pv_format 0).
 * Errors: as fp8attn_fwd; FP8ATTN_ERR_INVALID_ARG also for num_sms < 1 or an
 * NVFP4 V (in->v8 null).
 */
fp8attn_status fp8attn_fwd_tail_split(const fp8attn_prepped* in, int B, int T, int H, int D,
                                      int reverse_kv, int pcast, float p_scale, float expcast_beta,
                                      float softmax_scale, int vsmooth, int num_sms, void* out,
                                      void* workspace, size_t workspace_bytes, void* stream);
/* 0 for an invalid shape or num_sms < 1. */
size_t fp8attn_fwd_tail_workspace_bytes(int B, int T, int H, int num_sms);

/*
 * Host-only plan of fp8attn_fwd_tail_split: returns P (2..4), writes the
 * number of last-wave query tiles to *n_tail and the P + 1 key-tile position
 * bounds of the parts to part_lo (0 = part_lo[0] < ... < part_lo[P] =
 * ceil(T/128), inner bounds multiples of 4, balanced for a max-only step
 * costing half a full one: part_lo[p] ~ nV (1 - 2^-p) / (1 - 2^-P)).
 * Returns 1 (n_tail 0, part_lo untouched) when the last wave is kept whole.
 * Null pointers are skipped.
 */
int fp8attn_fwd_tail_plan(int B, int T, int H, int num_sms, int* n_tail, int* part_lo);

/*
 * Stage 1 without a workspace, for callers that cannot allocate device memory.
 * The pages have no counterpart of this call: it exists for integrations where
 * the caller cannot hand the library a device buffer (allocation forbidden
 * after start-up, a host framework that owns all device memory, plain C code
 * without an allocator).
 *
 * Same arguments and results as fp8attn_prep, minus the workspace.  The
 * per-channel scratch lives in a fixed device array inside the library that
 * holds FP8ATTN_NOALLOC_MAX_BH (batch, head) pairs; larger problems get
 * FP8ATTN_ERR_WORKSPACE without any work being queued.  With no workspace
 * there is no status word either, so errors a kernel finds while it runs are
 * not reported by this call: a permutation entry outside [0, T) is still read
 * as token 0 (no access leaves the tensors) but goes unreported.  Callers that
 * need that report use fp8attn_prep with a workspace.  Every GPU that loads
 * the library keeps that array (1 MiB) until the process exits.  All calls on
 * a device share it, so calls whose GPU work overlaps (other streams, other
 * host threads) race: order them on one stream.  The first call on each device
 * looks up the array's device address with that device current; make that
 * first call before any stream capture begins.  Allocates nothing.
 */
#define FP8ATTN_NOALLOC_MAX_BH 2048
fp8attn_status fp8attn_prep_noalloc(const void* q, const void* k, const void* v, int B, int T,
                                    int H, int D, const int32_t* perm, int vsmooth,
                                    const fp8attn_prepped* out, void* stream);

/*
 * Synchronises `stream`, then reads and clears the status word a previous
 * fp8attn_prep or fp8attn_fwd call left in `workspace`.  Returns FP8ATTN_OK,
 * FP8ATTN_ERR_DEVICE_TIMEOUT, FP8ATTN_ERR_BAD_TILE_LIST,
 * FP8ATTN_ERR_BAD_PERMUTATION or FP8ATTN_ERR_CUDA.
 */
fp8attn_status fp8attn_check_status(void* workspace, void* stream);

/*
 * The library's fp32 -> E4M3 conversion on its own: the round-to-nearest-even,
 * satfinite E4M3 encoding the prep and the P-cast use (P-Cast Precision review,
 * section 3: 3 mantissa bits, largest magnitude 448, values below 2^-10 round to
 * zero; TeleFuser blog, section "FP8 Preparation for attention").  Exposed so
 * the codec can be checked value by value against a reference encoder.
 *   x      n fp32 values (device, 4-byte aligned, read only)
 *   codes  n E4M3 codes (device, written); NaN inputs give a NaN code
 *   n      number of values (0 is a no-op)
 * Errors: FP8ATTN_ERR_INVALID_ARG (null pointer with n > 0, misaligned x),
 * FP8ATTN_ERR_UNSUPPORTED_DEVICE, FP8ATTN_ERR_CUDA; asynchronous on `stream`.
 */
fp8attn_status fp8attn_e4m3_encode(const float* x, uint8_t* codes, size_t n, void* stream);

/*
 * Online V clustering that produces the V-Smooth permutation (VC-Attention
 * news article, section 2, first step: the value tokens of a head are grouped
 * by a light clustering on a few representative dimensions and each cluster
 * is laid out as one contiguous run, so that the 128-row blocks of the prep
 * hold similar rows; the clusters need not be balanced).  Per (batch, head):
 *   - the n_dims channels with the largest max_t |v| (ties: lower channel);
 *   - 12-bit codes rne(v * 2^(11 - E_d)), 2^E_d <= max |v_d| < 2^(E_d + 1)
 *     (a channel of zeros gives codes 0);
 *   - Lloyd's k-means on the codes: seeds are tokens floor(k T / n_clusters);
 *     squared Euclidean distance, ties to the lower cluster; centroids move to
 *     the floor of the members' mean code, an empty cluster keeps its
 *     centroid; `iters` rounds of (move, assign) after the first assignment;
 *   - perm = the stable sort of the tokens by cluster id.
 * All steps after the code conversion are integer arithmetic, so the result
 * is deterministic.  The permutation is the `perm` argument of
 * fp8attn_prep / fp8attn_prep_smooth (V'[j] = V[perm[j]]); it can be reused
 * across calls while V keeps its structure.
 *   v          bf16 [B, T, H, 128] device, 16-byte aligned, finite values
 *   n_clusters 1..64;  n_dims 1..16;  iters 0..64
 *   perm       int32 [B, H, T] device output (4-byte aligned)
 *   labels     int32 [B, H, T] device output of the final cluster ids, or NULL
 *   workspace  device scratch of fp8attn_cluster_workspace_bytes(B, T, H,
 *              n_dims) bytes, 16-byte aligned
 * Errors: FP8ATTN_ERR_INVALID_ARG (shape, range, NULL or misaligned pointer),
 * FP8ATTN_ERR_WORKSPACE, FP8ATTN_ERR_UNSUPPORTED_DEVICE, FP8ATTN_ERR_CUDA,
 * all returned before any work is queued; asynchronous on `stream`.
 */
size_t fp8attn_cluster_workspace_bytes(int B, int T, int H, int n_dims);
fp8attn_status fp8attn_v_cluster(const void* v, int B, int T, int H, int D, int n_clusters,
                                 int n_dims, int iters, int32_t* perm, int32_t* labels,
                                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * Failure-detection self test: one CTA waits, through the kernels' own bounded
 * mbarrier wait, on a barrier that nothing arrives on.  After limit_ns
 * (100 us .. 1 s) the wait gives up, the status word in `workspace` (any
 * workspace of this library, 16-byte aligned) records FP8ATTN_ERR_DEVICE_TIMEOUT
 * for fp8attn_check_status, and the CUDA context stays usable.  No fault, trap
 * or endless loop is involved.  Errors: FP8ATTN_ERR_WORKSPACE,
 * FP8ATTN_ERR_INVALID_ARG (limit out of range), FP8ATTN_ERR_UNSUPPORTED_DEVICE,
 * FP8ATTN_ERR_CUDA.
 */
fp8attn_status fp8attn_selftest_wait_timeout(void* workspace, unsigned long long limit_ns, void* stream);

/* Static, human-readable name of a status code. */
const char* fp8attn_status_string(fp8attn_status s);

/* Library ABI version (increments on any signature change). */
int fp8attn_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FP8ATTN_H_ */
