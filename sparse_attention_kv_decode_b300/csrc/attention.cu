// Sparse MQA over gathered FP4 entries (csa2_sparse_decode) and the
// sliding-window branch with its log-sum-exp merge (csa2_swa_merge).
//
// Ref: "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression":
// the blog repost (sparse attention over the whole context combined with a
// sliding-window branch), the picx.dev summary (Methodology / 2. CSA2: the
// global KV and its top-K indices; 5. FP4 Main KV Cache), and the wesearch.press
// card (head-count reduction: one latent KV shared by every query head).
//
// One CTA handles one query token and a split of its key set: a tile of 64
// keys is staged (cp.async gather of FP4 codes + scales, or bf16 window rows),
// converted to fp16 in shared memory (FP4 -> fp16 is exact), and attended by 8
// warps with m16n8k16 fp16 MMAs and an online softmax in the exp2 domain.
// Partials (unnormalised O, running max, running sum) of every split are then
// merged by a combine kernel, which also folds in an external branch for the
// SWA merge.
#include "csa2_internal.cuh"

namespace csa2 {

constexpr int kTE = 64;            // keys per tile
constexpr int kRowBytes = 1152;    // 576 fp16
constexpr int kChunks = 72;        // 16-byte chunks per row
constexpr int kDV = 512;
static_assert(kPartStride == kDV + 2, "partial layout");
constexpr int kSxStride = 68;      // floats per S-exchange row (64 + pad)
constexpr int kAttnThreads = 256;

__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return (uint32_t)(row * kRowBytes + ((chunk ^ (row & 7)) << 4));
}

struct AttnSmem {
  static constexpr int kQ = 0;
  static constexpr int kC = kQ + 64 * kRowBytes;
  static constexpr int kS = kC + kTE * kRowBytes;
  static constexpr int kStage = kS + 64 * kSxStride * 4;
  static constexpr int kStageCodes = kTE * CSA2_CODE_BYTES;    // 18432
  static constexpr int kStageScales = kTE * CSA2_SCALE_BYTES;  // 2304
  static constexpr int kStageBytes = kStageCodes + kStageScales;
  static constexpr int kValid = kStage + 2 * kStageBytes;
  static constexpr int kTotalFp4 = kValid + 2 * kTE * 4;
  static constexpr int kValidSwa = kStage;
  static constexpr int kTotalSwa = kValidSwa + kTE * 4;
};

// Source of keys for one query: FP4 entries named by an index list, or a
// contiguous window of raw bf16 rows.
struct Fp4Source {
  const uint8_t* codes;   // [B][n_stride][288]
  const uint8_t* scales;  // [B][n_stride][36]
  int64_t n_stride;
  const int32_t* idx;     // [Q][K]
  int K;
};
struct SwaSource {
  const uint16_t* rows;   // [B][s_stride][576]
  int64_t s_stride;
  const int32_t* win_start;
  const int32_t* win_len;
  int n_win;
};

// Stage Q (bf16 [H][576]) into fp16 rows of the swizzled Q buffer; rows >= H are zero.
// Loads are issued in batches of 6 per thread before any conversion, so their
// latencies overlap instead of forming a chain.
__device__ __forceinline__ void stage_q(uint8_t* smem, const uint16_t* q, int H) {
  constexpr int kPer = 64 * kChunks / kAttnThreads;  // 18
  constexpr int kBatch = 6;
#pragma unroll
  for (int b0 = 0; b0 < kPer; b0 += kBatch) {
    uint4 v[kBatch];
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int i = threadIdx.x + (b0 + k) * kAttnThreads;
      const int row = i / kChunks, ch = i % kChunks;
      v[k] = row < H ? *reinterpret_cast<const uint4*>(q + (int64_t)row * CSA2_D_KV + ch * 8)
                     : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int i = threadIdx.x + (b0 + k) * kAttnThreads;
      const int row = i / kChunks, ch = i % kChunks;
      uint4 o;
      o.x = bf16x2_to_h2(v[k].x); o.y = bf16x2_to_h2(v[k].y);
      o.z = bf16x2_to_h2(v[k].z); o.w = bf16x2_to_h2(v[k].w);
      *reinterpret_cast<uint4*>(smem + AttnSmem::kQ + swz(row, ch)) = o;
    }
  }
}

// Issue the cp.async gather of one FP4 tile (entries [p0, p0+64) of the index list).
__device__ __forceinline__ void fp4_prefetch(uint8_t* smem, int buf, const Fp4Source& src, int b,
                                             const int32_t* idx_row, int p0, int p_end,
                                             uint32_t* status) {
  uint8_t* stage = smem + AttnSmem::kStage + buf * AttnSmem::kStageBytes;
  int* valid = reinterpret_cast<int*>(smem + AttnSmem::kValid) + buf * kTE;
  const uint8_t* cbase = src.codes + (int64_t)b * src.n_stride * CSA2_CODE_BYTES;
  const uint8_t* sbase = src.scales + (int64_t)b * src.n_stride * CSA2_SCALE_BYTES;
  if (threadIdx.x < kTE) {
    const int p = p0 + threadIdx.x;
    int e = p < p_end ? idx_row[p] : -1;
    if (e < -1 || e >= src.n_stride) {
      atomicOr(status, CSA2_DEV_BAD_INDEX);
      e = -1;
    }
    valid[threadIdx.x] = e;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < kTE * 18; i += kAttnThreads) {
    const int e = i / 18, c = i % 18;
    const int ent = valid[e];
    const uint8_t* g = cbase + (int64_t)(ent < 0 ? 0 : ent) * CSA2_CODE_BYTES + c * 16;
    cp_async16(smem_u32(stage + e * CSA2_CODE_BYTES + c * 16), g, ent >= 0);
  }
  for (int i = threadIdx.x; i < kTE * 9; i += kAttnThreads) {
    const int e = i / 9, w = i % 9;
    const int ent = valid[e];
    const uint8_t* g = sbase + (int64_t)(ent < 0 ? 0 : ent) * CSA2_SCALE_BYTES + w * 4;
    cp_async4(smem_u32(stage + AttnSmem::kStageCodes + e * CSA2_SCALE_BYTES + w * 4), g, ent >= 0);
  }
}

// FP4 stage -> fp16 C tile (exact: e2m1 * e4m3 fits fp16).
__device__ __forceinline__ void fp4_dequant(uint8_t* smem, int buf) {
  const uint8_t* stage = smem + AttnSmem::kStage + buf * AttnSmem::kStageBytes;
  for (int i = threadIdx.x; i < kTE * 36; i += kAttnThreads) {
    const int e = i / 36, bk = i % 36;
    const uint2 cw = *reinterpret_cast<const uint2*>(stage + e * CSA2_CODE_BYTES + bk * 8);
    const uint32_t s2 = e4m3_to_h2(stage[AttnSmem::kStageCodes + e * CSA2_SCALE_BYTES + bk]);
    uint32_t h[8];
    e2m1x4_to_h2x2(cw.x & 0xFFFFu, h[0], h[1]);
    e2m1x4_to_h2x2(cw.x >> 16, h[2], h[3]);
    e2m1x4_to_h2x2(cw.y & 0xFFFFu, h[4], h[5]);
    e2m1x4_to_h2x2(cw.y >> 16, h[6], h[7]);
#pragma unroll
    for (int k = 0; k < 8; ++k) h[k] = hmul2_u32(h[k], s2);
    *reinterpret_cast<uint4*>(smem + AttnSmem::kC + swz(e, 2 * bk)) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(smem + AttnSmem::kC + swz(e, 2 * bk + 1)) = make_uint4(h[4], h[5], h[6], h[7]);
  }
}

// Raw bf16 window rows [r0, r0+64) (clipped to r_end) -> fp16 C tile (batched loads).
__device__ __forceinline__ void swa_load(uint8_t* smem, const uint16_t* rows, int r0, int r_end) {
  int* valid = reinterpret_cast<int*>(smem + AttnSmem::kValidSwa);
  if (threadIdx.x < kTE) valid[threadIdx.x] = (r0 + (int)threadIdx.x < r_end) ? 1 : -1;
  constexpr int kPer = kTE * kChunks / kAttnThreads;  // 18
  constexpr int kBatch = 6;
#pragma unroll
  for (int b0 = 0; b0 < kPer; b0 += kBatch) {
    uint4 v[kBatch];
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int i = threadIdx.x + (b0 + k) * kAttnThreads;
      const int e = i / kChunks, ch = i % kChunks;
      v[k] = (r0 + e < r_end) ? *reinterpret_cast<const uint4*>(rows + (int64_t)(r0 + e) * CSA2_D_KV + ch * 8)
                              : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int i = threadIdx.x + (b0 + k) * kAttnThreads;
      const int e = i / kChunks, ch = i % kChunks;
      uint4 o;
      o.x = bf16x2_to_h2(v[k].x); o.y = bf16x2_to_h2(v[k].y);
      o.z = bf16x2_to_h2(v[k].z); o.w = bf16x2_to_h2(v[k].w);
      *reinterpret_cast<uint4*>(smem + AttnSmem::kC + swz(e, ch)) = o;
    }
  }
}

// Per-warp running state of the online softmax for 16 heads x 256 value dims.
struct WarpAcc {
  float o[32][4];
  float m0, m1;   // running max (log2 domain) of rows g, g+8
  float l0, l1;   // running (thread-partial) sums
};

// Phase A: S = (Q . C^T) * scale_log2 for heads 16hg.. and keys 32eh.. -> S exchange.
__device__ __forceinline__ void phase_qk(uint8_t* smem, const int* valid, float scale_log2) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hg = warp & 3, eh = warp >> 2;
  const int g = lane >> 2, tig = lane & 3;
  const uint32_t qb = smem_u32(smem + AttnSmem::kQ);
  const uint32_t cb = smem_u32(smem + AttnSmem::kC);
  float acc[4][4];
#pragma unroll
  for (int n = 0; n < 4; ++n)
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[n][k] = 0.f;
  const int arow = hg * 16 + (lane & 15);
  const int brow0 = eh * 32 + (lane & 7) + ((lane >> 4) << 3);
#pragma unroll 4
  for (int j = 0; j < 36; ++j) {
    uint32_t a0, a1, a2, a3;
    ldsm_x4(qb + swz(arow, 2 * j + (lane >> 4)), a0, a1, a2, a3);
#pragma unroll
    for (int np = 0; np < 2; ++np) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4(cb + swz(brow0 + np * 16, 2 * j + ((lane >> 3) & 1)), b0, b1, b2, b3);
      mma_f16(acc[2 * np], a0, a1, a2, a3, b0, b1);
      mma_f16(acc[2 * np + 1], a0, a1, a2, a3, b2, b3);
    }
  }
  float* Sx = reinterpret_cast<float*>(smem + AttnSmem::kS);
#pragma unroll
  for (int n = 0; n < 4; ++n) {
    const int e = eh * 32 + n * 8 + 2 * tig;
    const bool v0 = valid[e] >= 0, v1 = valid[e + 1] >= 0;
    float2 r0 = make_float2(v0 ? acc[n][0] * scale_log2 : -INFINITY, v1 ? acc[n][1] * scale_log2 : -INFINITY);
    float2 r1 = make_float2(v0 ? acc[n][2] * scale_log2 : -INFINITY, v1 ? acc[n][3] * scale_log2 : -INFINITY);
    *reinterpret_cast<float2*>(Sx + (hg * 16 + g) * kSxStride + e) = r0;
    *reinterpret_cast<float2*>(Sx + (hg * 16 + g + 8) * kSxStride + e) = r1;
  }
}

// Phases B and C: online softmax of the tile's scores and O += P . V.
__device__ __forceinline__ void phase_softmax_pv(uint8_t* smem, WarpAcc& A) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hg = warp & 3, dh = warp >> 2;
  const int g = lane >> 2, tig = lane & 3;
  const float* Sx = reinterpret_cast<const float*>(smem + AttnSmem::kS);
  float s[8][4];
#pragma unroll
  for (int n = 0; n < 8; ++n) {
    float2 r0 = *reinterpret_cast<const float2*>(Sx + (hg * 16 + g) * kSxStride + n * 8 + 2 * tig);
    float2 r1 = *reinterpret_cast<const float2*>(Sx + (hg * 16 + g + 8) * kSxStride + n * 8 + 2 * tig);
    s[n][0] = r0.x; s[n][1] = r0.y; s[n][2] = r1.x; s[n][3] = r1.y;
  }
  float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
  for (int n = 0; n < 8; ++n) {
    mx0 = fmaxf(mx0, fmaxf(s[n][0], s[n][1]));
    mx1 = fmaxf(mx1, fmaxf(s[n][2], s[n][3]));
  }
  mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
  mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
  mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
  mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
  const float mn0 = fmaxf(A.m0, mx0), mn1 = fmaxf(A.m1, mx1);
  const float mu0 = mn0 == -INFINITY ? 0.f : mn0;
  const float mu1 = mn1 == -INFINITY ? 0.f : mn1;
  const float al0 = exp2f(A.m0 - mu0), al1 = exp2f(A.m1 - mu1);
  A.m0 = mn0;
  A.m1 = mn1;
  float ps0 = 0.f, ps1 = 0.f;
  uint32_t pa[4][4];
#pragma unroll
  for (int n = 0; n < 8; ++n) {
    const float p0 = exp2f(s[n][0] - mu0), p1 = exp2f(s[n][1] - mu0);
    const float p2 = exp2f(s[n][2] - mu1), p3 = exp2f(s[n][3] - mu1);
    ps0 += p0 + p1;
    ps1 += p2 + p3;
    pa[n >> 1][(n & 1) * 2 + 0] = pack_h2(p0, p1);
    pa[n >> 1][(n & 1) * 2 + 1] = pack_h2(p2, p3);
  }
  A.l0 = A.l0 * al0 + ps0;
  A.l1 = A.l1 * al1 + ps1;
#pragma unroll
  for (int n = 0; n < 32; ++n) {
    A.o[n][0] *= al0; A.o[n][1] *= al0;
    A.o[n][2] *= al1; A.o[n][3] *= al1;
  }
  const uint32_t cb = smem_u32(smem + AttnSmem::kC);
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    const int erow = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
    for (int cc = 0; cc < 16; ++cc) {
      const int ch = dh * 32 + 2 * cc + (lane >> 4);
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(cb + swz(erow, ch), b0, b1, b2, b3);
      // pa[kk] = {rows g k0-7 (n=2kk), rows g+8 k0-7, rows g k8-15 (n=2kk+1), rows g+8 k8-15}
      mma_f16(A.o[2 * cc], pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], b0, b1);
      mma_f16(A.o[2 * cc + 1], pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], b2, b3);
    }
  }
}

// Write this CTA's partial (unnormalised O, max, sum) for its 16 heads x 256 dims.
__device__ __forceinline__ void write_partial(float* part, int H, WarpAcc& A) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hg = warp & 3, dh = warp >> 2;
  const int g = lane >> 2, tig = lane & 3;
  float l0 = A.l0, l1 = A.l1;
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  const int h0 = hg * 16 + g, h1 = h0 + 8;
  constexpr int kPS = kDV + 2;
#pragma unroll
  for (int n = 0; n < 32; ++n) {
    const int d = dh * 256 + n * 8 + 2 * tig;
    if (h0 < H) *reinterpret_cast<float2*>(part + h0 * kPS + d) = make_float2(A.o[n][0], A.o[n][1]);
    if (h1 < H) *reinterpret_cast<float2*>(part + h1 * kPS + d) = make_float2(A.o[n][2], A.o[n][3]);
  }
  if (dh == 0 && tig == 0) {
    if (h0 < H) { part[h0 * kPS + kDV] = A.m0; part[h0 * kPS + kDV + 1] = l0; }
    if (h1 < H) { part[h1 * kPS + kDV] = A.m1; part[h1 * kPS + kDV + 1] = l1; }
  }
}

__device__ __forceinline__ void init_acc(WarpAcc& A) {
#pragma unroll
  for (int n = 0; n < 32; ++n) A.o[n][0] = A.o[n][1] = A.o[n][2] = A.o[n][3] = 0.f;
  A.m0 = A.m1 = -INFINITY;
  A.l0 = A.l1 = 0.f;
}

// grid: (nsplit, Q). Partials: [Q][nsplit][H][514].
__global__ void __launch_bounds__(kAttnThreads, 1) sparse_attn_partial_kernel(
    const uint16_t* __restrict__ q, Fp4Source src, int T, int H, float scale_log2, int nsplit,
    int split_len, float* __restrict__ partials, uint32_t* __restrict__ status) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int sp = blockIdx.x, qi = blockIdx.y, b = qi / T;
  stage_q(smem, q + (int64_t)qi * H * CSA2_D_KV, H);
  const int p_begin = sp * split_len;
  const int p_end = min(p_begin + split_len, src.K);
  const int ntiles = p_end > p_begin ? (p_end - p_begin + kTE - 1) / kTE : 0;
  const int32_t* idx_row = src.idx + (int64_t)qi * src.K;
  WarpAcc A;
  init_acc(A);
  if (ntiles > 0) {
    fp4_prefetch(smem, 0, src, b, idx_row, p_begin, p_end, status);
    cp_async_commit();
  }
  for (int it = 0; it < ntiles; ++it) {
    const int buf = it & 1;
    if (it + 1 < ntiles) {
      fp4_prefetch(smem, buf ^ 1, src, b, idx_row, p_begin + (it + 1) * kTE, p_end, status);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    fp4_dequant(smem, buf);
    __syncthreads();
    phase_qk(smem, reinterpret_cast<const int*>(smem + AttnSmem::kValid) + buf * kTE, scale_log2);
    __syncthreads();
    phase_softmax_pv(smem, A);
  }
  write_partial(partials + ((int64_t)qi * nsplit + sp) * H * (kDV + 2), H, A);
}

// grid: (nsplit, Q); split sp covers window rows [sp*64, sp*64+64).
__global__ void __launch_bounds__(kAttnThreads, 1) swa_attn_partial_kernel(
    const uint16_t* __restrict__ q, SwaSource src, int T, int H, float scale_log2, int nsplit,
    float* __restrict__ partials, uint32_t* __restrict__ status) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int sp = blockIdx.x, qi = blockIdx.y, b = qi / T;
  int ws = src.win_start[qi], wl = src.win_len[qi];
  if (wl > src.n_win) wl = src.n_win;
  if (ws < 0 || wl < 0 || (int64_t)ws + wl > src.s_stride) {
    if (sp == 0 && threadIdx.x == 0) atomicOr(status, CSA2_DEV_BAD_WINDOW);
    if (wl < 0) wl = 0;
    if (ws < 0) { wl += ws; ws = 0; if (wl < 0) wl = 0; }
    if ((int64_t)ws + wl > src.s_stride) wl = (int)(src.s_stride > ws ? src.s_stride - ws : 0);
  }
  WarpAcc A;
  init_acc(A);
  const int r0 = sp * kTE;
  if (r0 < wl) {
    stage_q(smem, q + (int64_t)qi * H * CSA2_D_KV, H);
    swa_load(smem, src.rows + ((int64_t)b * src.s_stride + ws) * CSA2_D_KV, r0, wl);
    __syncthreads();
    phase_qk(smem, reinterpret_cast<const int*>(smem + AttnSmem::kValidSwa), scale_log2);
    __syncthreads();
    phase_softmax_pv(smem, A);
  }
  write_partial(partials + ((int64_t)qi * nsplit + sp) * H * (kDV + 2), H, A);
}

// Merge nsplit partials (and optionally an external normalised branch with
// natural-log LSE) into normalised O and natural-log LSE. One warp per (query,
// head): the split maxima and sums are loaded in parallel by the lanes, then
// every lane combines 16 value dims. grid: (ceil(H/8), Q), 256 threads.
__global__ void __launch_bounds__(256) attn_combine_kernel(
    const float* __restrict__ partials, int nsplit, int H, const float* __restrict__ o_ext,
    const float* __restrict__ lse_ext, float* __restrict__ o_out, float* __restrict__ lse_out) {
  constexpr float kLn2 = 0.69314718055994530942f, kLog2e = 1.4426950408889634074f;
  constexpr int kPS = kDV + 2;
  const int qi = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x * 8 + warp;
  if (h >= H) return;
  // lane s < nsplit holds split s; lane 31 holds the external branch
  float m = -INFINITY, l = 0.f;
  if (lane < nsplit) {
    const float* p = partials + ((int64_t)(qi * nsplit + lane) * H + h) * kPS;
    m = p[kDV];
    l = p[kDV + 1];
  } else if (lane == 31 && o_ext) {
    m = lse_ext[(int64_t)qi * H + h] * kLog2e;  // a normalised branch: sum 1 at max lse
    l = m == -INFINITY ? 0.f : 1.f;
  }
  float M = m;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  const float Mu = M == -INFINITY ? 0.f : M;
  const float w = l > 0.f ? exp2f(m - Mu) : 0.f;   // weight of this lane's branch
  float L = l * w;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
  const float inv = L > 0.f ? 1.f / L : 0.f;
  float4 acc[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s = 0; s < nsplit; ++s) {
    const float ws = __shfl_sync(0xffffffffu, w, s);
    if (ws == 0.f) continue;
    const float* p = partials + ((int64_t)(qi * nsplit + s) * H + h) * kPS;
    float2 x[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      x[2 * j] = *reinterpret_cast<const float2*>(p + j * 128 + lane * 4);
      x[2 * j + 1] = *reinterpret_cast<const float2*>(p + j * 128 + lane * 4 + 2);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      acc[j].x += ws * x[2 * j].x; acc[j].y += ws * x[2 * j].y;
      acc[j].z += ws * x[2 * j + 1].x; acc[j].w += ws * x[2 * j + 1].y;
    }
  }
  const float we = __shfl_sync(0xffffffffu, w, 31);
  if (o_ext && we > 0.f) {
    const float* e = o_ext + ((int64_t)qi * H + h) * kDV;
    float4 x[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) x[j] = *reinterpret_cast<const float4*>(e + j * 128 + lane * 4);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      acc[j].x += we * x[j].x; acc[j].y += we * x[j].y;
      acc[j].z += we * x[j].z; acc[j].w += we * x[j].w;
    }
  }
  __syncwarp();
  float* out = o_out + ((int64_t)qi * H + h) * kDV;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float4 r = acc[j];
    r.x *= inv; r.y *= inv; r.z *= inv; r.w *= inv;
    *reinterpret_cast<float4*>(out + j * 128 + lane * 4) = r;
  }
  if (lane == 0 && lse_out) lse_out[(int64_t)qi * H + h] = L > 0.f ? (Mu + log2f(L)) * kLn2 : -INFINITY;
}

static cudaError_t set_smem(int slot, const void* fn, int bytes) {
  return set_attr_once(slot, fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

cudaError_t launch_sparse_attn(int B, int T, int H, const void* q, const uint8_t* codes,
                               const uint8_t* scales, int64_t n_stride, const int32_t* idx, int K,
                               float scale_log2, float* o_g, float* lse_g, float* partials,
                               int nsplit, uint32_t* status, cudaStream_t st) {
  const int Q = B * T;
  if (Q == 0) return cudaSuccess;
  cudaError_t e = set_smem(2, (const void*)sparse_attn_partial_kernel, AttnSmem::kTotalFp4);
  if (e != cudaSuccess) return e;
  int split_len = (K + nsplit - 1) / nsplit;
  split_len = (split_len + kTE - 1) / kTE * kTE;
  Fp4Source src{codes, scales, n_stride, idx, K};
  sparse_attn_partial_kernel<<<dim3(nsplit, Q), kAttnThreads, AttnSmem::kTotalFp4, st>>>(
      static_cast<const uint16_t*>(q), src, T, H, scale_log2, nsplit, split_len, partials, status);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  attn_combine_kernel<<<dim3((H + 7) / 8, Q), 256, 0, st>>>(partials, nsplit, H, nullptr,
                                                              nullptr, o_g, lse_g);
  return cudaGetLastError();
}

cudaError_t launch_swa_merge(int B, int T, int H, const void* q, const void* swa,
                             int64_t s_stride, const int32_t* win_start, const int32_t* win_len,
                             int n_win, float scale_log2, const float* o_g, const float* lse_g,
                             float* o_out, float* lse_out, float* partials, uint32_t* status,
                             cudaStream_t st) {
  const int Q = B * T;
  if (Q == 0) return cudaSuccess;
  cudaError_t e = set_smem(3, (const void*)swa_attn_partial_kernel, AttnSmem::kTotalSwa);
  if (e != cudaSuccess) return e;
  const int nsplit = swa_splits(n_win);
  SwaSource src{static_cast<const uint16_t*>(swa), s_stride, win_start, win_len, n_win};
  swa_attn_partial_kernel<<<dim3(nsplit, Q), kAttnThreads, AttnSmem::kTotalSwa, st>>>(
      static_cast<const uint16_t*>(q), src, T, H, scale_log2, nsplit, partials, status);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  attn_combine_kernel<<<dim3((H + 7) / 8, Q), 256, 0, st>>>(partials, nsplit, H, o_g, lse_g,
                                                              o_out, lse_out);
  return cudaGetLastError();
}

}  // namespace csa2
