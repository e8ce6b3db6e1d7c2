// Sparse MQA over gathered FP4 entries (csa2_sparse_decode) and the
// sliding-window branch with its log-sum-exp merge (csa2_swa_merge).
//
// Ref: "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression":
// the blog repost (sparse attention over the whole context combined with a
// sliding-window branch), the picx.dev summary (Methodology / 2. CSA2: the
// global KV and its top-K indices; 5. FP4 Main KV Cache), and the wesearch.press
// card (head-count reduction: one latent KV shared by every query head).
//
// One CTA attends one query token over a split of its keys, 128 keys per tile,
// on the 5th-generation tensor cores with the scores transposed so that the
// 128 keys fill the MMA's M dimension (64 heads are N):
//   S^T[key, head]  = C[key, 0:576] . Q[head, 0:576]^T     (K-major A and B)
//   O^T[dim, head] += V^T[dim, key] . P^T[key, head]        (MN-major A and B)
// C is the tile's key rows in fp16 (FP4 entries dequantise exactly to fp16;
// bf16 window rows are converted), V = C[:, 0:512], and both products read the
// same 128-byte-swizzled shared-memory tile. S^T (two buffers) and the four
// 128x64 O^T accumulators live in TMEM.
// Warp roles (288 threads):
//   warps 0-3  loaders: stage Q; per tile, gather + dequantise one key row per
//              thread (FP4) or convert TMA-loaded window rows (bf16)
//   warps 4-7  softmax: one key row (TMEM lane) per thread; running max per head
//              kept lazily (rescale only when a score exceeds it by 2^8), P^T
//              written over the rope chunk of C once the S^T product has read it
//   warp 8     TMEM allocation and the single-thread MMA issuer
// Partials (unnormalised O, max, sum per head) of every split are merged by the
// combine kernel, which also folds in the global branch for the SWA merge.
#include <cstddef>

#include "csa2_internal.cuh"

namespace csa2 {

constexpr int kDV = 512;
static_assert(kPartStride == kDV + 2, "partial layout");

namespace {

constexpr int kTK = 128;                 // keys per tile
constexpr int kQChunk = 64 * 128;        // 64 heads x 64 dims fp16
constexpr int kCChunk = kTK * 128;       // 128 keys x 64 dims fp16
constexpr int kQBytes = 9 * kQChunk;
constexpr int kCBytes = 9 * kCChunk;
constexpr int kThreadsTC = 288;
constexpr int kTmemCols = 512;
constexpr int kColS = 0;                 // S^T buffers at columns [0, 64) and [64, 128)
constexpr int kColO = 128;               // O^T M-tile i at columns [128 + 64 i, +64)
constexpr float kRescale = 8.0f;         // lazy-max slack, log2 units (factor 256)
constexpr int kMiscBytes = 4096;
constexpr int kSmemTC = 1024 + kQBytes + kCBytes + kMiscBytes;

// mbarrier slots (8 bytes each) in the misc area
enum Bar { kQReady = 0, kChunkFull = 1, kGroupFree = 6, kSFull = 11, kPFull = 13, kTmaFull = 14,
           kDrain = 15, kQTma = 16, kNumBars = 17 };

struct Misc {
  uint64_t bars[kNumBars];
  alignas(16) uint32_t tmem_base;
  int abort_flag;
  int vote[2];
  int valid[2][kTK];
  float mrun[64];
  float mnew[64];
  float alpha[64];
  float red[4][64];
};
static_assert(sizeof(Misc) <= kMiscBytes, "misc area");
static_assert(offsetof(Misc, tmem_base) % 16 == 0, "TMEM address slot alignment");

struct Fp4Src {
  const uint8_t* codes;   // [B][n_stride][288]
  const uint8_t* scales;  // [B][n_stride][36]
  int64_t n_stride;
  const int32_t* idx;     // [Q][K]
  int K;
};
struct RowSrc {
  int64_t s_stride;
  const int32_t* win_start;
  const int32_t* win_len;
  int n_win;
};

// AND of a predicate over the `n` threads of named barrier `id` (all get the result).
__device__ __forceinline__ bool named_and(int id, int n, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ uint32_t cswz(int c, int row, int j) {
  // byte offset of 16-byte piece j of row `row` in 128-byte-swizzled chunk c
  return (uint32_t)(c * kCChunk + row * 128 + ((j ^ (row & 7)) << 4));
}

// Reduce 32 per-thread values (heads h0..h0+31) over the 128 softmax threads
// (4 warps), max or sum, into out[h0 .. h0+31]. Reduce-scatter inside each warp
// (31 shuffles: lane ends with one head), then across the warps in shared
// memory. All 128 threads must call it (named barrier 1).
template <bool kMax>
__device__ __forceinline__ float red_op(float a, float b) { return kMax ? fmaxf(a, b) : a + b; }

template <bool kMax>
__device__ __forceinline__ void reduce32(const float (&v)[32], Misc& ms, float* out, int h0, int lane,
                                         int w) {
  float a[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const bool hi = lane & 16;
    const float got = __shfl_xor_sync(0xffffffffu, hi ? v[i] : v[16 + i], 16);
    a[i] = red_op<kMax>(hi ? v[16 + i] : v[i], got);
  }
  float b[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const bool hi = lane & 8;
    const float got = __shfl_xor_sync(0xffffffffu, hi ? a[i] : a[8 + i], 8);
    b[i] = red_op<kMax>(hi ? a[8 + i] : a[i], got);
  }
  float c[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const bool hi = lane & 4;
    const float got = __shfl_xor_sync(0xffffffffu, hi ? b[i] : b[4 + i], 4);
    c[i] = red_op<kMax>(hi ? b[4 + i] : b[i], got);
  }
  float d[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const bool hi = lane & 2;
    const float got = __shfl_xor_sync(0xffffffffu, hi ? c[i] : c[2 + i], 2);
    d[i] = red_op<kMax>(hi ? c[2 + i] : c[i], got);
  }
  const bool hi = lane & 1;
  const float got = __shfl_xor_sync(0xffffffffu, hi ? d[0] : d[1], 1);
  const float e = red_op<kMax>(hi ? d[1] : d[0], got);
  // lane holds head index 16*b4 + 8*b3 + 4*b2 + 2*b1 + b0 of the 32
  const int idx = ((lane >> 4) & 1) * 16 + ((lane >> 3) & 1) * 8 + ((lane >> 2) & 1) * 4 +
                  ((lane >> 1) & 1) * 2 + (lane & 1);
  ms.red[w][h0 + idx] = e;
  asm volatile("bar.sync 1, 128;" ::: "memory");
  const int t = w * 32 + lane;
  if (t < 32) {
    float r = ms.red[0][h0 + t];
#pragma unroll
    for (int k = 1; k < 4; ++k) r = red_op<kMax>(r, ms.red[k][h0 + t]);
    out[h0 + t] = r;
  }
  asm volatile("bar.sync 1, 128;" ::: "memory");
}

// Scaled, masked scores of this thread's key row for heads h0..h0+31 (from S^T in TMEM).
__device__ __forceinline__ void load_scores32(uint32_t taddr, bool valid, float scale_log2, float (&s)[32]) {
  uint32_t r[32];
  tmem_ld32(taddr, r);
  tmem_wait_ld();
#pragma unroll
  for (int h = 0; h < 32; ++h) s[h] = valid ? __uint_as_float(r[h]) * scale_log2 : -INFINITY;
}

template <bool kFp4>
__global__ void __launch_bounds__(kThreadsTC, 1) attn_tc_kernel(
    const __grid_constant__ CUtensorMap tm_q, Fp4Src fsrc, RowSrc rsrc,
    const __grid_constant__ CUtensorMap tm_rows, int T, int H, float scale_log2, int nsplit,
    int split_len, float* __restrict__ partials, uint32_t* __restrict__ status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sC = smem + kQBytes;
  Misc& ms = *reinterpret_cast<Misc*>(smem + kQBytes + kCBytes);
  const uint32_t uQ = smem_u32(sQ), uC = smem_u32(sC);
  const uint32_t uP = uC + 8 * kCChunk;
  auto bar = [&](int i) { return smem_u32(&ms.bars[i]); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sp = blockIdx.x, qi = blockIdx.y, b = qi / T;

  // key range of this CTA
  int p_begin, p_end;
  int row_base = 0;  // window rows: first store row of this split (SWA)
  if (kFp4) {
    p_begin = sp * split_len;
    p_end = min(p_begin + split_len, fsrc.K);
  } else {
    int ws = rsrc.win_start[qi], wl = rsrc.win_len[qi];
    if (wl > rsrc.n_win) wl = rsrc.n_win;
    if (ws < 0 || wl < 0 || (int64_t)ws + wl > rsrc.s_stride) {
      if (sp == 0 && threadIdx.x == 0) atomicOr(status, CSA2_DEV_BAD_WINDOW);
      if (wl < 0) wl = 0;
      if (ws < 0) { wl += ws; ws = 0; if (wl < 0) wl = 0; }
      if ((int64_t)ws + wl > rsrc.s_stride) wl = (int)(rsrc.s_stride > ws ? rsrc.s_stride - ws : 0);
    }
    p_begin = sp * split_len;
    p_end = min(p_begin + split_len, wl);
    row_base = (int)((int64_t)b * rsrc.s_stride + ws);
  }
  const int ntiles = p_end > p_begin ? (p_end - p_begin + kTK - 1) / kTK : 0;
  float* part = partials + ((int64_t)qi * nsplit + sp) * H * kPartStride;

  if (threadIdx.x == 0) {
    mbar_init(bar(kQReady), 128);
    for (int g = 0; g < 5; ++g) {
      mbar_init(bar(kChunkFull + g), 128);
      mbar_init(bar(kGroupFree + g), 1);
    }
    mbar_init(bar(kSFull), 1);
    mbar_init(bar(kSFull + 1), 1);
    mbar_init(bar(kPFull), 128);
    mbar_init(bar(kTmaFull), 1);
    mbar_init(bar(kDrain), 1);
    mbar_init(bar(kQTma), 1);
    ms.abort_flag = 0;
    ms.vote[0] = ms.vote[1] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 8) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&ms.tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ms.tmem_base;
  volatile int* abort_flag = &ms.abort_flag;
  auto fail = [&]() {
    atomicOr(status, CSA2_DEV_PIPELINE_TIMEOUT);
    *abort_flag = 1;
  };

  if (warp < 4) {
    // ======================= loaders =======================
    const int e = threadIdx.x;  // key row within a tile / staging thread
    // Q (bf16 rows qi*H .. qi*H+63) arrives by TMA in nine 64x64 swizzled boxes and is
    // converted to fp16 in place; rows past H belong to other queries (or are zero) and
    // only feed heads that are never written out.
    if (e == 0) {
      mbar_arrive_expect_tx(bar(kQTma), 9 * kQChunk);
      for (int c = 0; c < 9; ++c) tma_load_2d(uQ + c * kQChunk, &tm_q, 64 * c, qi * H, bar(kQTma));
    }
    bool q_ok = true;
    auto convert_q = [&]() {
      q_ok = mbar_wait(bar(kQTma), 0);
      if (!q_ok) { fail(); return; }
      // 64 rows x 72 pieces: thread e converts rows e/2 (half e&1 of the pieces)
      const int h = e >> 1;
#pragma unroll 4
      for (int k = 0; k < 36; ++k) {
        const int pc = (e & 1) * 36 + k;
        uint4* pp = reinterpret_cast<uint4*>(sQ + (pc >> 3) * kQChunk + h * 128 + (((pc & 7) ^ (h & 7)) << 4));
        uint4 v = *pp;
        v.x = bf16x2_to_h2(v.x); v.y = bf16x2_to_h2(v.y);
        v.z = bf16x2_to_h2(v.z); v.w = bf16x2_to_h2(v.w);
        *pp = v;
      }
      fence_proxy_async_smem();
      mbar_arrive(bar(kQReady));
    };
    if (kFp4) {
      const uint8_t* cbase = fsrc.codes + (int64_t)b * fsrc.n_stride * CSA2_CODE_BYTES;
      const uint8_t* sbase = fsrc.scales + (int64_t)b * fsrc.n_stride * CSA2_SCALE_BYTES;
      const int32_t* idx_row = fsrc.idx + (int64_t)qi * fsrc.K;
      uint4 cw[18];
      uint32_t sw[9];
      int ent = -1;
      auto load_tile = [&](int t) {
        const int p = p_begin + t * kTK + e;
        ent = p < p_end ? idx_row[p] : -1;
        if (ent < -1 || ent >= fsrc.n_stride) {
          atomicOr(status, CSA2_DEV_BAD_INDEX);
          ent = -1;
        }
        if (ent >= 0) {
          const uint4* cp = reinterpret_cast<const uint4*>(cbase + (int64_t)ent * CSA2_CODE_BYTES);
          const uint32_t* spt = reinterpret_cast<const uint32_t*>(sbase + (int64_t)ent * CSA2_SCALE_BYTES);
#pragma unroll
          for (int k = 0; k < 18; ++k) cw[k] = __ldg(cp + k);
#pragma unroll
          for (int k = 0; k < 9; ++k) sw[k] = __ldg(spt + k);
        } else {
#pragma unroll
          for (int k = 0; k < 18; ++k) cw[k] = make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int k = 0; k < 9; ++k) sw[k] = 0u;
        }
      };
      if (ntiles > 0) load_tile(0);
      convert_q();
      bool lok = q_ok;
      for (int t = 0; t < ntiles && lok; ++t) {
        if (*abort_flag) break;
#pragma unroll
        for (int g = 0; g < 5; ++g) {
          if (lok && t > 0 && !mbar_wait(bar(kGroupFree + g), (t - 1) & 1)) { fail(); lok = false; }
          if (lok) {
            if (g == 0) ms.valid[t & 1][e] = ent;
            const int blk0 = g < 4 ? 8 * g : 32, nblk = g < 4 ? 8 : 4;
#pragma unroll
            for (int kb = 0; kb < nblk; ++kb) {
              const int blk = blk0 + kb;
              // 16 codes of block blk: bytes [8 blk, 8 blk + 8) of the row
              const uint4 w4 = cw[blk >> 1];
              const uint32_t lo = (blk & 1) ? w4.z : w4.x, hi = (blk & 1) ? w4.w : w4.y;
              const uint32_t s2 = e4m3_to_h2((sw[blk >> 2] >> (8 * (blk & 3))) & 0xFFu);
              uint32_t hv[8];
              e2m1x4_to_h2x2(lo & 0xFFFFu, hv[0], hv[1]);
              e2m1x4_to_h2x2(lo >> 16, hv[2], hv[3]);
              e2m1x4_to_h2x2(hi & 0xFFFFu, hv[4], hv[5]);
              e2m1x4_to_h2x2(hi >> 16, hv[6], hv[7]);
#pragma unroll
              for (int k = 0; k < 8; ++k) hv[k] = hmul2_u32(hv[k], s2);
              const int c = blk >> 2, j = (blk & 3) * 2;
              *reinterpret_cast<uint4*>(sC + cswz(c, e, j)) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
              *reinterpret_cast<uint4*>(sC + cswz(c, e, j + 1)) = make_uint4(hv[4], hv[5], hv[6], hv[7]);
            }
            fence_proxy_async_smem();
            mbar_arrive(bar(kChunkFull + g));
          }
        }
        if (lok && t + 1 < ntiles) load_tile(t + 1);
      }
    } else {
      int issued_t = -1, waited_t = -1;
      convert_q();
      for (int t = 0; t < ntiles && q_ok; ++t) {
        if (*abort_flag) break;
        if (t > 0 && !mbar_wait(bar(kGroupFree + 4), (t - 1) & 1)) { fail(); break; }
        if (e == 0) {
          mbar_arrive_expect_tx(bar(kTmaFull), 9 * kCChunk);
          for (int c = 0; c < 9; ++c)
            tma_load_2d(uC + c * kCChunk, &tm_rows, 64 * c, row_base + p_begin + t * kTK, bar(kTmaFull));
          issued_t = t;
        }
        const int key = p_begin + t * kTK + e;
        ms.valid[t & 1][e] = key < p_end ? 1 : -1;
        if (!mbar_wait(bar(kTmaFull), t & 1)) { fail(); break; }
        waited_t = t;
        // bf16 -> fp16 in place, one row per thread
        for (int g = 0; g < 5; ++g) {
          const int c0 = g < 4 ? 2 * g : 8, nc = g < 4 ? 2 : 1;
          for (int cc = 0; cc < nc; ++cc) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              uint4* pp = reinterpret_cast<uint4*>(sC + cswz(c0 + cc, e, j));
              uint4 v = *pp;
              v.x = bf16x2_to_h2(v.x); v.y = bf16x2_to_h2(v.y);
              v.z = bf16x2_to_h2(v.z); v.w = bf16x2_to_h2(v.w);
              *pp = v;
            }
          }
          fence_proxy_async_smem();
          mbar_arrive(bar(kChunkFull + g));
        }
      }
      // copies in flight must land before the CTA exits
      if (e == 0 && issued_t > waited_t) mbar_wait(bar(kTmaFull), issued_t & 1);
    }
    if (e == 0 && !q_ok) mbar_wait(bar(kQTma), 0);
  } else if (warp < 8) {
    // ======================= softmax =======================
    const int w = warp - 4;          // TMEM lane quarter
    const int ts = w * 32 + lane;    // key row (S^T lane) / value dim row (O^T lane)
    const uint32_t lane_off = (uint32_t)(w * 32) << 16;
    float l[64];                     // running sums of this key row's p, per head
#pragma unroll
    for (int h = 0; h < 64; ++h) l[h] = 0.f;
    bool ok = true;
    for (int t = 0; t < ntiles; ++t) {
      const int sb = t & 1;
      bool got = !*abort_flag && mbar_wait(bar(kSFull + sb), (t >> 1) & 1) &&
                 mbar_wait(bar(kChunkFull + 4), t & 1);
      if (!named_and(1, 128, got)) { if (ts == 0) fail(); ok = false; break; }
      tc_fence_after();
      const bool vld = ms.valid[sb][ts] >= 0;
      const uint32_t ts_addr = tmem + lane_off + kColS + 64 * sb;
      if (t == 0) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float s[32];
          load_scores32(ts_addr + 32 * hh, vld, scale_log2, s);
          reduce32<true>(s, ms, ms.mrun, 32 * hh, lane, w);
        }
      } else {
        bool need = false;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float s[32];
          load_scores32(ts_addr + 32 * hh, vld, scale_log2, s);
#pragma unroll
          for (int h = 0; h < 32; ++h) need |= s[h] > ms.mrun[32 * hh + h] + kRescale;
        }
        if (__any_sync(0xffffffffu, need) && lane == 0) atomicOr(&ms.vote[sb], 1);
        asm volatile("bar.sync 1, 128;" ::: "memory");
        const bool rescale = ms.vote[sb] != 0;
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (ts == 0) ms.vote[sb] = 0;
        if (rescale) {
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            float s[32];
            load_scores32(ts_addr + 32 * hh, vld, scale_log2, s);
            reduce32<true>(s, ms, ms.mnew, 32 * hh, lane, w);
          }
          // O^T must be final for tile t-1 before it is rescaled
          if (!named_and(1, 128, mbar_wait(bar(kGroupFree + 4), (t - 1) & 1))) {
            if (ts == 0) fail();
            ok = false;
            break;
          }
          tc_fence_after();
          if (ts < 64) {
            const float mo = ms.mrun[ts], mn = fmaxf(mo, ms.mnew[ts]);
            ms.alpha[ts] = mo == mn ? 1.f : exp2f(mo - mn);
          }
          asm volatile("bar.sync 1, 128;" ::: "memory");
#pragma unroll
          for (int h = 0; h < 64; ++h) l[h] *= ms.alpha[h];
          for (int i = 0; i < 8; ++i) {
            uint32_t r[32];
            const uint32_t ta = tmem + lane_off + kColO + 32 * i;
            tmem_ld32(ta, r);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k)
              r[k] = __float_as_uint(__uint_as_float(r[k]) * ms.alpha[(32 * i + k) & 63]);
            tmem_st32(ta, r);
          }
          tmem_wait_st();
          asm volatile("bar.sync 1, 128;" ::: "memory");
          if (ts < 64) ms.mrun[ts] = fmaxf(ms.mrun[ts], ms.mnew[ts]);
          asm volatile("bar.sync 1, 128;" ::: "memory");
        }
      }
      // P^T row of this key: exp2(s - m) in fp16, written over the rope chunk (the S^T
      // product of this tile has consumed it)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float s[32];
        load_scores32(ts_addr + 32 * hh, vld, scale_log2, s);
        uint32_t pk[16];
#pragma unroll
        for (int h = 0; h < 32; h += 2) {
          const float m0 = ms.mrun[32 * hh + h], m1 = ms.mrun[32 * hh + h + 1];
          const float p0 = exp2f(s[h] - (m0 == -INFINITY ? 0.f : m0));
          const float p1 = exp2f(s[h + 1] - (m1 == -INFINITY ? 0.f : m1));
          l[32 * hh + h] += p0;
          l[32 * hh + h + 1] += p1;
          pk[h >> 1] = pack_h2(p0, p1);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
          *reinterpret_cast<uint4*>(sC + cswz(8, ts, 4 * hh + j)) =
              make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(kPFull));
    }
    // ---- epilogue: partial O (unnormalised), max and sum per head
    if (ok && ntiles > 0) {
      ok = named_and(1, 128, mbar_wait(bar(kGroupFree + 4), (ntiles - 1) & 1));
      if (!ok && ts == 0) fail();
    }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      float v[32];
#pragma unroll
      for (int h = 0; h < 32; ++h) v[h] = l[32 * hh + h];
      reduce32<false>(v, ms, ms.mnew, 32 * hh, lane, w);
    }
    if (ok && ntiles > 0) {
      tc_fence_after();
      for (int i = 0; i < 8; ++i) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + kColO + 32 * i, r);
        tmem_wait_ld();
        const int d = 128 * (i >> 1) + ts, h0 = 32 * (i & 1);
#pragma unroll
        for (int k = 0; k < 32; ++k)
          if (h0 + k < H) part[(h0 + k) * kPartStride + d] = __uint_as_float(r[k]);
      }
    } else {
      for (int i = 0; i < 4; ++i)
        for (int h = 0; h < H; ++h) part[h * kPartStride + 128 * i + ts] = 0.f;
    }
    if (ts < H) {
      const bool has = ok && ntiles > 0;
      part[ts * kPartStride + kDV] = has ? ms.mrun[ts] : -INFINITY;
      part[ts * kPartStride + kDV + 1] = has ? ms.mnew[ts] : 0.f;
    }
  } else {
    // ======================= MMA issuer =======================
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_f16(kTK, 64, 0, 0, 0, 0);
      constexpr uint32_t idesc_pv = idesc_f16(kTK, 64, 0, 0, 1, 1);
      bool issued = false;
      bool ok = mbar_wait(bar(kQReady), 0);
      if (!ok) fail();
      for (int t = 0; t < ntiles && ok; ++t) {
        if (*abort_flag) break;
        const int sb = t & 1;
        const uint32_t d_s = tmem + kColS + 64 * sb;
        for (int g = 0; g < 5 && ok; ++g) {
          if (!mbar_wait(bar(kChunkFull + g), t & 1)) { fail(); ok = false; break; }
          tc_fence_after();
          const int c0 = g < 4 ? 2 * g : 8, nc = g < 4 ? 2 : 1;
          for (int cc = 0; cc < nc; ++cc) {
            const int c = c0 + cc;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t a = umma_desc_sw128(uC + c * kCChunk + 32 * k);
              const uint64_t bq = umma_desc_sw128(uQ + c * kQChunk + 32 * k);
              umma_f16(d_s, a, bq, idesc_qk, (c | k) != 0);
              issued = true;
            }
          }
        }
        if (!ok) break;
        umma_commit(bar(kSFull + sb));
        if (!mbar_wait(bar(kPFull), t & 1)) { fail(); ok = false; break; }
        tc_fence_after();
        for (int i = 0; i < 4; ++i) {
#pragma unroll
          for (int kk = 0; kk < kTK / 16; ++kk) {
            const uint64_t a = umma_desc_sw128_mn(uC + 2 * i * kCChunk + kk * 2048, kCChunk, 1024);
            const uint64_t bp = umma_desc_sw128_mn(uP + kk * 2048, kCChunk, 1024);
            umma_f16(tmem + kColO + 64 * i, a, bp, idesc_pv, (t > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(bar(kGroupFree + i));
        }
        umma_commit(bar(kGroupFree + 4));
      }
      if (issued) {
        umma_commit(bar(kDrain));
        mbar_wait(bar(kDrain), 0);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                 : "memory");
  }
}

}  // namespace

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
  // splits in groups of 4 with all loads of a group issued before the FMAs
  for (int s0 = 0; s0 < nsplit; s0 += 4) {
    float4 x[4][4];
    float ws[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int s = s0 + u;
      ws[u] = __shfl_sync(0xffffffffu, w, s < nsplit ? s : 0);
      if (s >= nsplit) ws[u] = 0.f;
      const float* p = partials + ((int64_t)(qi * nsplit + (s < nsplit ? s : 0)) * H + h) * kPS;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 a = *reinterpret_cast<const float2*>(p + j * 128 + lane * 4);
        const float2 b = *reinterpret_cast<const float2*>(p + j * 128 + lane * 4 + 2);
        x[u][j] = make_float4(a.x, a.y, b.x, b.y);
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        acc[j].x += ws[u] * x[u][j].x; acc[j].y += ws[u] * x[u][j].y;
        acc[j].z += ws[u] * x[u][j].z; acc[j].w += ws[u] * x[u][j].w;
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


static cudaError_t launch_combine(const float* partials, int nsplit, int Q, int H, const float* o_ext,
                                  const float* lse_ext, float* o_out, float* lse_out, cudaStream_t st) {
  attn_combine_kernel<<<dim3((H + 7) / 8, Q), 256, 0, st>>>(partials, nsplit, H, o_ext, lse_ext, o_out,
                                                            lse_out);
  return cudaGetLastError();
}

cudaError_t launch_sparse_attn(int B, int T, int H, const void* q, const uint8_t* codes,
                               const uint8_t* scales, int64_t n_stride, const int32_t* idx, int K,
                               float scale_log2, float* o_g, float* lse_g, float* partials,
                               int nsplit, uint32_t* status, cudaStream_t st) {
  const int Q = B * T;
  if (Q == 0) return cudaSuccess;
  cudaError_t e = set_attr_once(2, (const void*)attn_tc_kernel<true>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemTC);
  if (e != cudaSuccess) return e;
  int split_len = (K + nsplit - 1) / nsplit;
  split_len = (split_len + kTK - 1) / kTK * kTK;
  Fp4Src f{codes, scales, n_stride, idx, K};
  RowSrc r{0, nullptr, nullptr, 0};
  CUtensorMap tq, dummy;
  memset(&dummy, 0, sizeof(dummy));
  if (!encode_tensor_map_2d_bf16(&tq, q, CSA2_D_KV, (uint64_t)Q * H, 64, 64)) return cudaErrorInvalidValue;
  attn_tc_kernel<true><<<dim3(nsplit, Q), kThreadsTC, kSmemTC, st>>>(
      tq, f, r, dummy, T, H, scale_log2, nsplit, split_len, partials, status);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_combine(partials, nsplit, Q, H, nullptr, nullptr, o_g, lse_g, st);
}

cudaError_t launch_swa_merge(int B, int T, int H, const void* q, const void* swa,
                             int64_t s_stride, const int32_t* win_start, const int32_t* win_len,
                             int n_win, float scale_log2, const float* o_g, const float* lse_g,
                             float* o_out, float* lse_out, float* partials, uint32_t* status,
                             cudaStream_t st) {
  const int Q = B * T;
  if (Q == 0) return cudaSuccess;
  const int nsplit = swa_splits(n_win);
  if (n_win > 0 && s_stride > 0) {
    cudaError_t e = set_attr_once(3, (const void*)attn_tc_kernel<false>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemTC);
    if (e != cudaSuccess) return e;
    CUtensorMap tm, tq;
    if (!encode_tensor_map_2d_bf16(&tm, swa, CSA2_D_KV, (uint64_t)B * s_stride, 64, kTK) ||
        !encode_tensor_map_2d_bf16(&tq, q, CSA2_D_KV, (uint64_t)Q * H, 64, 64))
      return cudaErrorInvalidValue;
    Fp4Src f{nullptr, nullptr, 0, nullptr, 0};
    RowSrc r{s_stride, win_start, win_len, n_win};
    attn_tc_kernel<false><<<dim3(nsplit, Q), kThreadsTC, kSmemTC, st>>>(
        tq, f, r, tm, T, H, scale_log2, nsplit, kTK, partials, status);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_combine(partials, nsplit, Q, H, o_g, lse_g, o_out, lse_out, st);
  }
  // empty window: the merge is the global branch itself
  return launch_combine(partials, 0, Q, H, o_g, lse_g, o_out, lse_out, st);
}

}  // namespace csa2
