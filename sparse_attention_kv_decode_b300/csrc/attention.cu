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
//
// Warp roles (320 threads):
//   warps 0-7  workers. Warp w stages key rows 16w .. 16w+15 of each tile: the
//              FP4 gather (prefetched one tile ahead in registers) is laid out
//              so that one warp load reads 8 rows x 64 contiguous bytes, and
//              each lane dequantises the pieces it loaded; bf16 window rows
//              are landed by TMA and converted in place. For the softmax,
//              thread (warp w, lane) owns key row / TMEM lane 32*(w%4)+lane
//              and head half w/4, and runs the softmax for 32 heads of it:
//              a lazy running max per head (rescale only when a score exceeds
//              it by 2^8), p written as fp16 P^T over the rope chunk of C once
//              the S^T product has read it.
//   warp 8     TMEM allocation and the single-thread MMA issuer.
//   warp 9     requests every entry the split gathers after its first tile into
//              L2 at the start (the register prefetch runs only one tile ahead).
// The splits of one query form a thread-block cluster. After the last P.V each
// CTA pushes its (max, sum) per head and its unnormalised O^T rows to the CTA
// that owns those value dims (distributed shared memory stores into the freed
// tile buffer); each CTA then merges every split's contribution for its dims
// (and, for the SWA merge, the global branch) and writes normalised O and LSE.
#include <cstddef>

#include "csa2_internal.cuh"

namespace csa2 {

constexpr int kDV = 512;

namespace {

constexpr int kTK = 128;                 // keys per tile
constexpr int kQChunk = 64 * 128;        // 64 heads x 64 dims fp16
constexpr int kCChunk = kTK * 128;       // 128 keys x 64 dims fp16
constexpr int kQBytes = 9 * kQChunk;
constexpr int kCBytes = 9 * kCChunk;
constexpr int kWorkers = 256;
constexpr int kThreadsTC = kWorkers + 64;   // + MMA warp + L2 prefetch warp
constexpr int kTmemCols = 512;
constexpr int kColS = 0;                 // S^T buffers at columns [0, 64) and [64, 128)
constexpr int kColO = 128;               // O^T M-tile i at columns [128 + 64 i, +64)
constexpr float kRescale = 8.0f;         // lazy-max slack, log2 units (factor 256)
constexpr int kMiscBytes = 6144;
constexpr int kSmemTC = 1024 + kQBytes + kCBytes + kMiscBytes;
constexpr int kMaxSplitsTC = 16;
// merge buffers inside the (finished) tile buffer
constexpr int kRecvStride = 68;          // floats per received O^T row (64 heads + pad), > 4 splits
constexpr int kRecvBytes = kDV * kRecvStride * 4;                    // 139,264
constexpr int kMlOffset = kRecvBytes;                                // [split][2][64] floats
static_assert(kRecvBytes + kMaxSplitsTC * 2 * 64 * 4 <= kCBytes, "merge buffers fit the tile");

// mbarrier slots (8 bytes each); kChunkFull: chunks 0-5 of the tile staged,
// kChunkFull + 1: chunks 6-8
enum Bar { kQReady = 0, kChunkFull = 1, kGroupFree = 6, kSFull = 11, kPFull = 13, kTmaFull = 14,
           kDrain = 15, kQTma = 16, kRecv = 17, kNumBars = 18 };

struct Misc {
  uint64_t bars[kNumBars];
  alignas(16) uint32_t tmem_base;
  int abort_flag;
  int valid[2][kTK];       // key validity of the tile, by tile parity
  // per-head arrays, read as 16-byte vectors
  alignas(16) float mrun[64];   // running max per head (log2 domain)
  alignas(16) float mnew[64];
  alignas(16) float alpha[64];
  alignas(16) float lsum[64];
  alignas(16) float red[4][64];
  alignas(16) float ml_in[4][2][64];   // (max, sum) per head pushed by each split (merge of <= 4 splits)
};
static_assert(sizeof(Misc) <= kMiscBytes, "misc area");
static_assert(offsetof(Misc, tmem_base) % 16 == 0, "TMEM address slot alignment");
static_assert(offsetof(Misc, mrun) % 16 == 0 && offsetof(Misc, ml_in) % 16 == 0 &&
                  offsetof(Misc, alpha) % 16 == 0 && offsetof(Misc, mnew) % 16 == 0,
              "vector reads of the per-head arrays");
static_assert((kQBytes + kCBytes) % 16 == 0, "Misc placement");

struct Fp4Src {
  const uint8_t* codes;   // entry rows [B][n_stride], CSA2_ENTRY_BYTES apart
  const uint8_t* scales;  // (same row stride)
  bool record;            // scales == codes + 288: one row holds both
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
struct OutArgs {
  float* o;               // [Q][H][512]
  float* lse;             // [Q][H] (nullable)
  const float* o_ext;     // external normalised branch (SWA merge), nullable
  const float* lse_ext;
  float* xchg;            // split exchange through L2: [Q][owner][source][64][512 / nsplit], nullable
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
// OR of a predicate over the `n` threads of named barrier `id` (all get the result).
__device__ __forceinline__ bool named_or(int id, int n, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}
// 2^x with the SFU's approximation (relative error ~2^-22; 2^-inf = 0): p is
// stored as fp16, whose rounding (2^-11) dominates.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ void named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// 2-D TMA load delivered to the same shared-memory offset (data and mbarrier
// transaction bytes) of every CTA of the cluster in `mask`.
__device__ __forceinline__ void tma_load_2d_mc(uint32_t dst, const CUtensorMap* map, int x, int y,
                                               uint32_t mbar, uint16_t mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(mbar), "h"(mask)
      : "memory");
}
__device__ __forceinline__ uint32_t map_rank(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster_v4(uint32_t addr, float a, float b, float c, float d) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b),
               "f"(c), "f"(d)
               : "memory");
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float a) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(a) : "memory");
}

__device__ __forceinline__ uint32_t cswz(int c, int row, int j) {
  // byte offset of 16-byte piece j of row `row` in 128-byte-swizzled chunk c
  return (uint32_t)(c * kCChunk + row * 128 + ((j ^ (row & 7)) << 4));
}

template <bool kMax>
__device__ __forceinline__ float red_op(float a, float b) { return kMax ? fmaxf(a, b) : a + b; }

// Reduce-scatter of 32 per-thread values (heads h0 .. h0+31) inside one warp, max or
// sum: lane l returns the warp's result for head h0 + l (31 shuffles).
template <bool kMax>
__device__ __forceinline__ float warp_reduce32(const float (&v)[32], int lane) {
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
  // each step kept the half selected by one lane bit, so lane l ends with head l
  return red_op<kMax>(hi ? d[1] : d[0], got);
}

// Reduce 32 per-thread values (heads h0..h0+31) over the 128 threads of one head
// half (4 warps, lane quarters 0..3), max or sum, into out[h0 .. h0+31] (or added
// to it with kAcc): reduce-scatter inside each warp, then across the 4 warps in
// shared memory under named barrier `bid`.
template <bool kMax, bool kAcc = false>
__device__ __forceinline__ void reduce32(const float (&v)[32], Misc& ms, float* out, int h0, int lane,
                                         int quarter, int bid) {
  ms.red[quarter][h0 + lane] = warp_reduce32<kMax>(v, lane);
  named_sync(bid, 128);
  if (quarter == 0) {
    float r = ms.red[0][h0 + lane];
#pragma unroll
    for (int k = 1; k < 4; ++k) r = red_op<kMax>(r, ms.red[k][h0 + lane]);
    out[h0 + lane] = kAcc ? out[h0 + lane] + r : r;
  }
  named_sync(bid, 128);
}

// Scaled, masked scores of one key row for 32 heads (from S^T in TMEM).
__device__ __forceinline__ void load_scores32(uint32_t taddr, bool valid, float scale_log2, float (&s)[32]) {
  uint32_t r[32];
  tmem_ld32(taddr, r);
  tmem_wait_ld();
#pragma unroll
  for (int h = 0; h < 32; ++h) s[h] = valid ? __uint_as_float(r[h]) * scale_log2 : -INFINITY;
}

// Dequantise one 16-byte piece of FP4 codes (elements 32 pc .. 32 pc + 31 of key
// row `row`, two 16-element blocks) into C: w holds the code bytes, s2 the two
// scale bytes (block 2 pc in the low byte). The piece fills 16-byte slots
// 4 (pc & 1) .. +3 of the row in chunk pc / 2.
__device__ __forceinline__ void dequant_piece(uint8_t* sC, int row, int pc, const uint4& w, uint32_t s2) {
  uint32_t sh;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(sh) : "h"((uint16_t)s2));
  const uint32_t sa = __byte_perm(sh, 0, 0x1010), sb = __byte_perm(sh, 0, 0x3232);
  uint32_t hv[16];
  e2m1x4_to_h2x2(w.x & 0xFFFFu, hv[0], hv[1]);
  e2m1x4_to_h2x2(w.x >> 16, hv[2], hv[3]);
  e2m1x4_to_h2x2(w.y & 0xFFFFu, hv[4], hv[5]);
  e2m1x4_to_h2x2(w.y >> 16, hv[6], hv[7]);
  e2m1x4_to_h2x2(w.z & 0xFFFFu, hv[8], hv[9]);
  e2m1x4_to_h2x2(w.z >> 16, hv[10], hv[11]);
  e2m1x4_to_h2x2(w.w & 0xFFFFu, hv[12], hv[13]);
  e2m1x4_to_h2x2(w.w >> 16, hv[14], hv[15]);
#pragma unroll
  for (int k = 0; k < 8; ++k) hv[k] = hmul2_u32(hv[k], sa);
#pragma unroll
  for (int k = 8; k < 16; ++k) hv[k] = hmul2_u32(hv[k], sb);
  const int c = pc >> 1, j = (pc & 1) * 4;
#pragma unroll
  for (int s = 0; s < 4; ++s)
    *reinterpret_cast<uint4*>(sC + cswz(c, row, j + s)) =
        make_uint4(hv[4 * s], hv[4 * s + 1], hv[4 * s + 2], hv[4 * s + 3]);
}

// One code piece and its two scale bytes of entry `ent` (zeros for ent < 0).
__device__ __forceinline__ void load_piece(const uint8_t* cbase, const uint8_t* sbase, int ent, int pc,
                                           uint4& w, uint32_t& s2) {
  if (ent >= 0) {
    w = __ldg(reinterpret_cast<const uint4*>(cbase + (int64_t)ent * CSA2_ENTRY_BYTES) + pc);
    s2 = __ldg(reinterpret_cast<const unsigned short*>(sbase + (int64_t)ent * CSA2_ENTRY_BYTES) + pc);
  } else {
    w = make_uint4(0, 0, 0, 0);
    s2 = 0u;
  }
}

__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void allow_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Kernel kinds: FP4 entries only (global branch), window rows only (the window
// branch, merged with an external global branch by log-sum-exp), or both key sets
// in one softmax (the window rows are the first tiles of the last split).
enum Kind { kSparse = 0, kWindow = 1, kFused = 2 };

template <int kKind>
__global__ void __launch_bounds__(kThreadsTC, 1) attn_tc_kernel(
    const __grid_constant__ CUtensorMap tm_q, Fp4Src fsrc, RowSrc rsrc,
    const __grid_constant__ CUtensorMap tm_rows, int T, int H, float scale_log2, int split_len,
    OutArgs out, uint32_t* __restrict__ status) {
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
  uint32_t nsplit;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(nsplit));

  if (threadIdx.x == 0) {
    mbar_init(bar(kQReady), kWorkers);
    mbar_init(bar(kChunkFull), kWorkers);
    mbar_init(bar(kChunkFull + 1), kWorkers);
    for (int g = 0; g < 5; ++g) mbar_init(bar(kGroupFree + g), 1);
    mbar_init(bar(kSFull), 1);
    mbar_init(bar(kSFull + 1), 1);
    mbar_init(bar(kPFull), kWorkers);
    mbar_init(bar(kTmaFull), 1);
    mbar_init(bar(kDrain), 1);
    mbar_init(bar(kQTma), 1);
    mbar_init(bar(kRecv), 1);
    ms.abort_flag = 0;
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
  // the splits of a query share one Q load (multicast): every CTA's barriers must be
  // initialised before a peer's copy lands, so the cluster meets once before it
  if (nsplit > 1) cluster_arrive();
  const uint32_t tmem = ms.tmem_base;
  volatile int* abort_flag = &ms.abort_flag;
  auto fail = [&]() {
    atomicOr(status, CSA2_DEV_PIPELINE_TIMEOUT);
    *abort_flag = 1;
  };
  // Inputs may be written by the preceding kernel in the stream: nothing below
  // reads global memory before it has completed.
  grid_dependency_wait();
  if (nsplit > 1) cluster_wait();

  constexpr bool kFp4 = kKind != kWindow;   // FP4 entry tiles
  constexpr bool kRows = kKind != kSparse;  // bf16 window row tiles
  // key ranges of this CTA: window rows [r_begin, r_end) (tiles 0 .. nt_r-1), then
  // FP4 entries [p_begin, p_end) of the index list (tiles nt_r ..)
  int p_begin = 0, p_end = 0, r_begin = 0, r_end = 0, row_base = 0;
  if (kFp4) {
    p_begin = sp * split_len;
    p_end = min(p_begin + split_len, fsrc.K);
  }
  if (kRows) {
    int ws = rsrc.win_start[qi], wl = rsrc.win_len[qi];
    if (wl > rsrc.n_win) wl = rsrc.n_win;
    if (ws < 0 || wl < 0 || (int64_t)ws + wl > rsrc.s_stride) {
      if (sp == 0 && threadIdx.x == 0) atomicOr(status, CSA2_DEV_BAD_WINDOW);
      if (wl < 0) wl = 0;
      if (ws < 0) { wl += ws; ws = 0; if (wl < 0) wl = 0; }
      if ((int64_t)ws + wl > rsrc.s_stride) wl = (int)(rsrc.s_stride > ws ? rsrc.s_stride - ws : 0);
    }
    if (kKind == kWindow) {
      r_begin = sp * split_len;
      r_end = min(r_begin + split_len, wl);
    } else if (sp == (int)nsplit - 1) {
      r_end = wl;
    }
    row_base = (int)((int64_t)b * rsrc.s_stride + ws);
  }
  const int nt_r = r_end > r_begin ? (r_end - r_begin + kTK - 1) / kTK : 0;
  const int nt_f = p_end > p_begin ? (p_end - p_begin + kTK - 1) / kTK : 0;
  const int ntiles = nt_r + nt_f;

  if (warp < 8) {
    // ======================= workers: loads / dequant + softmax =======================
    const int quarter = warp & 3, half = warp >> 2;
    const int e = quarter * 32 + lane;        // key row of a tile; TMEM lane
    const int wt = threadIdx.x;               // 0..255
    const int bid = 1 + half;                 // named barrier of this head half
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    bool wok = true;                          // pipeline state (uniform within a head half)
    // Q: nine 64x64 swizzled TMA boxes (rows qi*H ..), converted to fp16 in place;
    // rows past H belong to other queries (or are zero) and feed unused heads.
    int issued_t = -1, waited_t = -1;  // window tiles loaded by TMA (wt == 0)
    if (wt == 0) {
      mbar_arrive_expect_tx(bar(kQTma), 9 * kQChunk);
      if (nsplit > 1) {
        // split sp loads chunks sp, sp + nsplit, .. for every CTA of the cluster
        for (int c = sp; c < 9; c += (int)nsplit)
          tma_load_2d_mc(uQ + c * kQChunk, &tm_q, 64 * c, qi * H, bar(kQTma), (uint16_t)((1u << nsplit) - 1u));
      } else {
        for (int c = 0; c < 9; ++c) tma_load_2d(uQ + c * kQChunk, &tm_q, 64 * c, qi * H, bar(kQTma));
      }
      // the first window tile goes to the still empty tile buffer right away
      if (kRows && nt_r > 0) {
        mbar_arrive_expect_tx(bar(kTmaFull), 9 * kCChunk);
        for (int c = 0; c < 9; ++c)
          tma_load_2d(uC + c * kCChunk, &tm_rows, 64 * c, row_base + r_begin, bar(kTmaFull));
        issued_t = 0;
      }
    }
    // the FP4 gather of tile 0 is issued before the Q conversion so the two overlap
    const uint8_t* cbase = nullptr;
    const uint8_t* sbase = nullptr;
    const int32_t* idx_row = nullptr;
    // gather layout of warp w (rows 16w .. 16w+15 of a tile): for chunk group g < 4
    // (code pieces 4g .. 4g+3) lane l takes piece 4g + (l & 3) of rows ra and rb;
    // for group 4 (pieces 16, 17) piece 16 + (l & 1) of row rc
    const int ra = 16 * warp + (lane >> 2), rb = ra + 8, rc = 16 * warp + (lane >> 1);
    uint4 cw[9];       // pieces [2g + k] (g < 4, k: row ra / rb) and [8] (group 4)
    uint32_t sw[5];    // their scale byte pairs: [g] = row ra | row rb << 16, [4] group 4
    int ent16 = -1, ent16_next = -1;  // entry of row 16w + lane (lanes < 16), this / next tile
    // the index word of row 16w + lane of FP4 tile tf (checked when fetch uses it, so the
    // load is not waited for here)
    auto read_idx = [&](int tf) -> int {
      const int p = p_begin + tf * kTK + 16 * warp + lane;
      return (lane < 16 && tf < nt_f && p < p_end) ? idx_row[p] : -1;
    };
    auto fetch = [&](int e16) {
      if (e16 < -1 || e16 >= fsrc.n_stride) {
        atomicOr(status, CSA2_DEV_BAD_INDEX);
        e16 = -1;
      }
      ent16 = e16;
      const int ea = __shfl_sync(0xffffffffu, e16, lane >> 2);
      const int eb = __shfl_sync(0xffffffffu, e16, 8 + (lane >> 2));
      const int ec = __shfl_sync(0xffffffffu, e16, lane >> 1);
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        uint32_t s0, s1;
        load_piece(cbase, sbase, ea, 4 * g + (lane & 3), cw[2 * g], s0);
        load_piece(cbase, sbase, eb, 4 * g + (lane & 3), cw[2 * g + 1], s1);
        sw[g] = s0 | (s1 << 16);
      }
      load_piece(cbase, sbase, ec, 16 + (lane & 1), cw[8], sw[4]);
    };
    if (kFp4) {
      cbase = fsrc.codes + (int64_t)b * fsrc.n_stride * CSA2_ENTRY_BYTES;
      sbase = fsrc.scales + (int64_t)b * fsrc.n_stride * CSA2_ENTRY_BYTES;
      idx_row = fsrc.idx + (int64_t)qi * fsrc.K;
      if (nt_f > 0) fetch(read_idx(0));
    }
    wok = mbar_wait(bar(kQTma), 0);
    if (!wok) fail();
    else {
      const int h = wt >> 2;  // 64 rows x 72 pieces: 4 threads per row, 18 pieces each
      uint32_t mag = 0u;      // largest bf16 magnitude (bits) of each half-word seen
#pragma unroll 6
      for (int k = 0; k < 18; ++k) {
        const int pc = (wt & 3) * 18 + k;
        uint4* pp = reinterpret_cast<uint4*>(sQ + (pc >> 3) * kQChunk + h * 128 + (((pc & 7) ^ (h & 7)) << 4));
        uint4 v = *pp;
        mag = __vmaxu2(mag, __vmaxu2(__vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu),
                                     __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu)));
        v.x = bf16x2_to_h2(v.x); v.y = bf16x2_to_h2(v.y);
        v.z = bf16x2_to_h2(v.z); v.w = bf16x2_to_h2(v.w);
        *pp = v;
      }
      // a query value outside the fp16 range (rows past H are not this query's)
      if (bf16_mag_beyond_fp16(mag) && h < H) atomicOr(status, CSA2_DEV_RANGE);
      fence_proxy_async_smem();
    }
    mbar_arrive(bar(kQReady));
    // the index words of tile 1 (the gather of tile 0 is in flight)
    if (kFp4) ent16_next = read_idx(1);

    // running sum of p: this warp's share for head 32 * half + lane (its key rows), across
    // tiles; the four warps of a head half are added once, after the last tile
    float wsum = 0.f;

    for (int t = 0; t < ntiles; ++t) {
      const int sb = t & 1;
      // ---- stage the tile into C (group by group, as P.V of tile t-1 releases it)
      const bool row_tile = kRows && t < nt_r;
      if (kFp4 && !row_tile) {
        const int tf = t - nt_r;
        bool ok = wok && !*abort_flag;
#pragma unroll
        for (int g = 0; g < 5; ++g) {
          if (ok && t > 0 && !mbar_wait(bar(kGroupFree + g), (t - 1) & 1)) { fail(); ok = false; }
          if (ok) {
            if (g == 0 && lane < 16) ms.valid[sb][16 * warp + lane] = ent16;
            if (g < 4) {
              dequant_piece(sC, ra, 4 * g + (lane & 3), cw[2 * g], sw[g] & 0xFFFFu);
              dequant_piece(sC, rb, 4 * g + (lane & 3), cw[2 * g + 1], sw[g] >> 16);
            } else {
              dequant_piece(sC, rc, 16 + (lane & 1), cw[8], sw[4]);
            }
          }
          // chunks 0-5 are released as soon as they are staged: the S^T product of
          // this tile starts on them while the last two groups wait for the end of the
          // previous P.V
          if (g == 2) {
            fence_proxy_async_smem();
            if (ok) mbar_arrive(bar(kChunkFull));
          }
        }
        fence_proxy_async_smem();
        if (ok) mbar_arrive(bar(kChunkFull + 1));
        wok = ok;
        if (wok && tf + 1 < nt_f) {
          fetch(ent16_next);
          ent16_next = read_idx(tf + 2);
        }
      } else if (kRows) {
        bool ok = wok && !*abort_flag;
        if (ok && t > 0 && !mbar_wait(bar(kGroupFree + 4), (t - 1) & 1)) { fail(); ok = false; }
        if (ok && wt == 0 && issued_t < t) {
          mbar_arrive_expect_tx(bar(kTmaFull), 9 * kCChunk);
          for (int c = 0; c < 9; ++c)
            tma_load_2d(uC + c * kCChunk, &tm_rows, 64 * c, row_base + r_begin + t * kTK, bar(kTmaFull));
          issued_t = t;
        }
        if (ok && half == 0) ms.valid[sb][e] = (r_begin + t * kTK + e < r_end) ? 1 : -1;
        if (ok && !mbar_wait(bar(kTmaFull), t & 1)) { fail(); ok = false; }
        if (ok && wt == 0) waited_t = t;
        if (ok) {
          const bool row_ok = r_begin + t * kTK + e < r_end;
          uint32_t mag = 0u;
          // bf16 -> fp16 in place; half 0 converts the first 36 pieces of row e, half 1 the rest
#pragma unroll 6
          for (int k = 0; k < 36; ++k) {
            const int pc = 36 * half + k;
            uint4* pp = reinterpret_cast<uint4*>(sC + cswz(pc >> 3, e, pc & 7));
            uint4 v = *pp;
            mag = __vmaxu2(mag, __vmaxu2(__vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu),
                                         __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu)));
            v.x = bf16x2_to_h2(v.x); v.y = bf16x2_to_h2(v.y);
            v.z = bf16x2_to_h2(v.z); v.w = bf16x2_to_h2(v.w);
            // rows past the window are zeroed: their p is 0, and 0 * NaN would not be
            if (!row_ok) v = make_uint4(0, 0, 0, 0);
            *pp = v;
          }
          // a window value outside the fp16 range
          if (bf16_mag_beyond_fp16(mag) && row_ok) atomicOr(status, CSA2_DEV_RANGE);
          fence_proxy_async_smem();
          mbar_arrive(bar(kChunkFull));
          mbar_arrive(bar(kChunkFull + 1));
        }
        wok = ok;
      }

      // ---- softmax of this tile for heads [32*half, 32*half+32)
      bool got = wok && !*abort_flag && mbar_wait(bar(kSFull + sb), (t >> 1) & 1);
      if (!named_and(bid, 128, got)) { if (e == 0) fail(); wok = false; break; }
      tc_fence_after();
      const bool vld = ms.valid[sb][e] >= 0;
      const uint32_t s_addr = tmem + lane_off + kColS + 64 * sb + 32 * half;
      const int h0 = 32 * half;
      float s[32];
      load_scores32(s_addr, vld, scale_log2, s);
      if (t == 0) reduce32<true>(s, ms, ms.mrun, h0, lane, quarter, bid);
      // P^T row of this key for the 32 heads: 2^(s - m) in fp16, over the rope chunk
      uint32_t pk[16];
      bool need = false;
#pragma unroll
      for (int h = 0; h < 32; h += 4) {
        const float4 m4 = *reinterpret_cast<const float4*>(&ms.mrun[h0 + h]);
        const float m[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) need |= s[h + k] > m[k] + kRescale;
        pk[h >> 1] = pack_h2(ex2_approx(s[h] - (m[0] == -INFINITY ? 0.f : m[0])),
                             ex2_approx(s[h + 1] - (m[1] == -INFINITY ? 0.f : m[1])));
        pk[(h >> 1) + 1] = pack_h2(ex2_approx(s[h + 2] - (m[2] == -INFINITY ? 0.f : m[2])),
                                   ex2_approx(s[h + 3] - (m[3] == -INFINITY ? 0.f : m[3])));
      }
      if (t > 0) {
        // one barrier: does any key of this head half exceed its running max by 2^8?
        const bool rescale = named_or(bid, 128, need);
        if (rescale) {
          reduce32<true>(s, ms, ms.mnew, h0, lane, quarter, bid);
          // O^T must be final for tile t-1 before it is rescaled
          if (!named_and(bid, 128, mbar_wait(bar(kGroupFree + 4), (t - 1) & 1))) {
            if (e == 0) fail();
            wok = false;
            break;
          }
          tc_fence_after();
          if (quarter == 0) {
            const float mo = ms.mrun[h0 + lane], mn = fmaxf(mo, ms.mnew[h0 + lane]);
            ms.alpha[h0 + lane] = mo == mn ? 1.f : exp2f(mo - mn);
          }
          named_sync(bid, 128);
          wsum *= ms.alpha[h0 + lane];
          for (int i = 0; i < 8; ++i) {
            uint32_t r[16];
            const uint32_t ta = tmem + lane_off + kColO + 64 * (i >> 1) + 32 * half + 16 * (i & 1);
            tmem_ld16(ta, r);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 16; ++k)
              r[k] = __float_as_uint(__uint_as_float(r[k]) * ms.alpha[h0 + 16 * (i & 1) + k]);
            tmem_st16(ta, r);
          }
          tmem_wait_st();
          named_sync(bid, 128);
          if (quarter == 0) ms.mrun[h0 + lane] = fmaxf(ms.mrun[h0 + lane], ms.mnew[h0 + lane]);
          named_sync(bid, 128);
          // the scores again (S^T of this tile is intact until the QK of tile t+2)
          load_scores32(s_addr, vld, scale_log2, s);
#pragma unroll
          for (int h = 0; h < 32; h += 2) {
            const float m0 = ms.mrun[h0 + h], m1 = ms.mrun[h0 + h + 1];
            pk[h >> 1] = pack_h2(ex2_approx(s[h] - (m0 == -INFINITY ? 0.f : m0)),
                                 ex2_approx(s[h + 1] - (m1 == -INFINITY ? 0.f : m1)));
          }
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j)
        *reinterpret_cast<uint4*>(sC + cswz(8, e, 4 * half + j)) =
            make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(kPFull));
      // the sums use the fp16 p that P.V consumes (while P.V runs)
      {
        float pf[32];
#pragma unroll
        for (int h = 0; h < 32; h += 2) {
          const float2 f2 = __half22float2(*reinterpret_cast<const __half2*>(&pk[h >> 1]));
          pf[h] = f2.x;
          pf[h + 1] = f2.y;
        }
        wsum += warp_reduce32<false>(pf, lane);
      }
    }
    // the sums per head: the four warps of each head half
    ms.red[quarter][32 * half + lane] = wsum;
    named_sync(bid, 128);
    if (quarter == 0)
      ms.lsum[32 * half + lane] = (ms.red[0][32 * half + lane] + ms.red[1][32 * half + lane]) +
                                  (ms.red[2][32 * half + lane] + ms.red[3][32 * half + lane]);
    if (kRows && wt == 0 && issued_t > waited_t) mbar_wait(bar(kTmaFull), issued_t & 1);

    // ---- wait for the last P.V, then the sums per head
    if (wok && ntiles > 0) {
      wok = named_and(bid, 128, mbar_wait(bar(kGroupFree + 4), (ntiles - 1) & 1));
      if (!wok && e == 0) fail();
    }
  } else if (warp == 8) {
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
        // two waits (chunks 0-5, then 6-8), each followed by its MMAs back to back: a
        // barrier poll costs the tensor pipe a few hundred cycles, so there is no
        // finer release
        if (!mbar_wait(bar(kChunkFull), t & 1)) { fail(); ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 6; ++c) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint64_t a = umma_desc_sw128(uC + c * kCChunk + 32 * k);
            const uint64_t bq = umma_desc_sw128(uQ + c * kQChunk + 32 * k);
            umma_f16(d_s, a, bq, idesc_qk, (c | k) != 0);
          }
        }
        issued = true;
        if (!mbar_wait(bar(kChunkFull + 1), t & 1)) { fail(); ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int c = 6; c < 9; ++c) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint64_t a = umma_desc_sw128(uC + c * kCChunk + 32 * k);
            const uint64_t bq = umma_desc_sw128(uQ + c * kQChunk + 32 * k);
            umma_f16(d_s, a, bq, idesc_qk, 1u);
          }
        }
        issued = true;
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
    __syncwarp();
  } else if (kFp4) {
    // ======================= L2 prefetch of the gathered entries =======================
    // Each tile's FP4 gather is issued one tile ahead into registers; from a cold L2 its
    // latency is longer than the tile's S^T product, so every entry this split gathers
    // after its first tile is requested into L2 once, up front.
    const uint8_t* cb = fsrc.codes + (int64_t)b * fsrc.n_stride * CSA2_ENTRY_BYTES;
    const uint8_t* sb = fsrc.scales + (int64_t)b * fsrc.n_stride * CSA2_ENTRY_BYTES;
    const int32_t* ir = fsrc.idx + (int64_t)qi * fsrc.K;
    // eight index loads in flight per lane before their requests go out
    constexpr int kBatch = 8;
    for (int p0 = p_begin + kTK; p0 < p_end; p0 += 32 * kBatch) {
      int ent[kBatch];
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int p = p0 + 32 * k + lane;
        ent[k] = p < p_end ? ir[p] : -1;
      }
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        if (ent[k] >= 0 && ent[k] < fsrc.n_stride) {
          if (fsrc.record) {
            // codes and scales in one row: one request for the whole row
            prefetch_l2_bulk(cb + (int64_t)ent[k] * CSA2_ENTRY_BYTES, CSA2_ENTRY_BYTES);
          } else {
            prefetch_l2_bulk(cb + (int64_t)ent[k] * CSA2_ENTRY_BYTES, CSA2_CODE_BYTES);
            const uint8_t* s0 = sb + (int64_t)ent[k] * CSA2_ENTRY_BYTES;
            prefetch_l2(s0);
            prefetch_l2(s0 + CSA2_SCALE_BYTES - 1);
          }
        }
      }
    }
  }

  // ======================= merge the splits of this query =======================
  allow_dependents();
  __syncthreads();
  const bool has = ntiles > 0 && !*abort_flag;
  if (nsplit > 1 && nsplit <= 4 && out.xchg != nullptr) {
    // CTA o owns value dims [o*Dn, (o+1)*Dn). Each split writes its unnormalised O^T
    // rows of the peers' dims to the exchange buffer in global memory (L2) as soon as
    // its last P.V is done, pushes its (max, sum) per head to every peer, and meets the
    // cluster once; each owner then weights every split's rows by exp2(m_s - M) / L,
    // adds them to its own rows (TMEM) and drops the exchange lines from L2 unwritten.
    constexpr float kLn2 = 0.69314718055994530942f, kLog2e = 1.4426950408889634074f;
    const int Dn = kDV / (int)nsplit, tiles_own = Dn / 128;
    const int tid = threadIdx.x;
    const int quarter = warp & 3, half = warp >> 2;
    const int e = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    // [owner o][source s][head][Dn dims] of this query
    float* xq = out.xchg + (size_t)qi * nsplit * kDV * 64;
    auto part = [&](int o, int s) { return xq + ((size_t)o * nsplit + s) * Dn * 64; };
    if (tid < 64) {
      const float m = has ? ms.mrun[tid] : -INFINITY;
      const float sm = has ? ms.lsum[tid] : 0.f;
      for (uint32_t p = 0; p < nsplit; ++p) {
        st_cluster_f32(map_rank(smem_u32(&ms.ml_in[sp][0][tid]), p), m);
        st_cluster_f32(map_rank(smem_u32(&ms.ml_in[sp][1][tid]), p), sm);
      }
    }
    if (warp < 8) {
      // consecutive lanes hold consecutive dims: every store of a warp is one 128-byte line
      for (int i = 0; i < 4; ++i) {
        const int o = i / tiles_own;
        if (o == sp) continue;
        uint32_t r[32];
        if (has) {
          tmem_ld32(tmem + lane_off + kColO + 64 * i + 32 * half, r);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) r[k] = 0u;
        }
        float* dst = part(o, sp) + (128 * i + e - o * Dn);
#pragma unroll
        for (int k = 0; k < 32; ++k) __stcg(dst + (size_t)(32 * half + k) * Dn, __uint_as_float(r[k]));
      }
    }
    // release / acquire at cluster scope: every split's rows and (max, sum) are visible
    tc_fence_before();
    cluster_sync_all();
    tc_fence_after();
    // weights per (split, head) overwrite the pushed maxima
    if (tid >= 32 && tid < 96) {
      const int h = tid - 32;
      float M = -INFINITY;
      for (uint32_t s2 = 0; s2 < nsplit; ++s2) M = fmaxf(M, ms.ml_in[s2][0][h]);
      const float Mu = M == -INFINITY ? 0.f : M;
      float L = 0.f;
      for (uint32_t s2 = 0; s2 < nsplit; ++s2) {
        const float ls = ms.ml_in[s2][1][h];
        L += ls > 0.f ? ls * exp2f(ms.ml_in[s2][0][h] - Mu) : 0.f;
      }
      const float inv = L > 0.f ? 1.f / L : 0.f;
      for (uint32_t s2 = 0; s2 < nsplit; ++s2) {
        const float ls = ms.ml_in[s2][1][h];
        ms.ml_in[s2][0][h] = ls > 0.f ? exp2f(ms.ml_in[s2][0][h] - Mu) * inv : 0.f;
      }
      if (sp == 0 && out.lse && h < H)
        out.lse[(int64_t)qi * H + h] = L > 0.f ? (Mu + log2f(L)) * kLn2 : -INFINITY;
      (void)kLog2e;
    }
    __syncthreads();
    if (warp < 8) {
      float* o = out.o + (int64_t)qi * H * kDV;
      for (int j = 0; j < tiles_own; ++j) {
        const int i = sp * tiles_own + j;
        const int dl = 128 * j + e, d = 128 * i + e;
        uint32_t r[32];
        if (has) {
          tmem_ld32(tmem + lane_off + kColO + 64 * i + 32 * half, r);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) r[k] = 0u;
        }
        float acc[32];
#pragma unroll
        for (int k = 0; k < 32; k += 4) {
          const float4 w = *reinterpret_cast<const float4*>(&ms.ml_in[sp][0][32 * half + k]);
          acc[k] = __uint_as_float(r[k]) * w.x;
          acc[k + 1] = __uint_as_float(r[k + 1]) * w.y;
          acc[k + 2] = __uint_as_float(r[k + 2]) * w.z;
          acc[k + 3] = __uint_as_float(r[k + 3]) * w.w;
        }
        for (int s2 = 0; s2 < (int)nsplit; ++s2) {
          if (s2 == sp) continue;
          const float* src = part(sp, s2) + dl;
          float v[32];
#pragma unroll
          for (int k = 0; k < 32; ++k) v[k] = __ldcg(src + (size_t)(32 * half + k) * Dn);
#pragma unroll
          for (int k = 0; k < 32; k += 4) {
            const float4 w = *reinterpret_cast<const float4*>(&ms.ml_in[s2][0][32 * half + k]);
            acc[k] += w.x * v[k]; acc[k + 1] += w.y * v[k + 1];
            acc[k + 2] += w.z * v[k + 2]; acc[k + 3] += w.w * v[k + 3];
          }
          // every lane has its values: lane l drops the line of head 32 half + l that this
          // warp read (the next call writes it again before reading it)
          __syncwarp();
          const float* line = part(sp, s2) + (size_t)(32 * half + lane) * Dn + 128 * j + 32 * quarter;
          asm volatile("discard.global.L2 [%0], 128;" ::"l"(line) : "memory");
        }
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const int h = 32 * half + k;
          if (h < H) o[(int64_t)h * kDV + d] = acc[k];
        }
      }
    }
    // (nothing of this CTA's shared memory is read or written by a peer after the barrier)
  } else if (nsplit <= 4) {
    // CTA o owns value dims [o*Dn, (o+1)*Dn) (whole 128-dim M-tiles). Each split
    // stages its raw O^T rows of the peers' M-tiles (rows of 64 heads, 16-byte pieces
    // swizzled by row) while the slower splits finish, and ships each peer's slice
    // with one bulk shared-to-shared copy; the owner weights every split's rows by
    // exp2(m_s - M) / L and adds them to its own M-tiles read from TMEM.
    constexpr float kLn2 = 0.69314718055994530942f, kLog2e = 1.4426950408889634074f;
    const int Dn = kDV / (int)nsplit, tiles_own = Dn / 128;
    const uint32_t slice_bytes = (uint32_t)Dn * 64 * 4;
    auto recv_slot = [&](int j) { return reinterpret_cast<float*>(sC + (size_t)j * slice_bytes); };
    auto staging = [&](int k) {
      return reinterpret_cast<float*>(k < 2 ? sQ + (size_t)k * slice_bytes : sC + (size_t)3 * slice_bytes);
    };
    // float offset of 16-byte piece j (0..15) of row r in a slice
    auto piece = [](int r, int j) { return r * 64 + ((j ^ (r & 7)) << 2); };
    const int tid = threadIdx.x;
    const int quarter = warp & 3, half = warp >> 2;
    const int e = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    if (tid < 64) {
      const float m = has ? ms.mrun[tid] : -INFINITY;
      const float s = has ? ms.lsum[tid] : 0.f;
      for (uint32_t p = 0; p < nsplit; ++p) {
        st_cluster_f32(map_rank(smem_u32(&ms.ml_in[sp][0][tid]), p), m);
        st_cluster_f32(map_rank(smem_u32(&ms.ml_in[sp][1][tid]), p), s);
      }
    }
    if (tid == 0 && nsplit > 1) mbar_arrive_expect_tx(bar(kRecv), (nsplit - 1) * slice_bytes);
    // this CTA is past its last P.V: its own Q and tile buffers are free for staging
    if (warp < 8 && nsplit > 1) {
      for (int i = 0; i < 4; ++i) {
        const int o = i / tiles_own;
        if (o == sp) continue;
        uint32_t r[32];
        if (has) {
          tmem_ld32(tmem + lane_off + kColO + 64 * i + 32 * half, r);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) r[k] = 0u;
        }
        const int k_st = (o - sp - 1 + (int)nsplit) % (int)nsplit;
        float* dst = staging(k_st);
        const int row = 128 * i + e - o * Dn;
#pragma unroll
        for (int k = 0; k < 8; ++k)
          *reinterpret_cast<uint4*>(dst + piece(row, 8 * half + k)) =
              make_uint4(r[4 * k], r[4 * k + 1], r[4 * k + 2], r[4 * k + 3]);
      }
      fence_proxy_async_smem();
    }
    // (max, sum) of every split visible; every CTA past its last P.V, so the tile
    // buffers of all of them may be written
    tc_fence_before();
    cluster_sync_all();
    tc_fence_after();
    // split sp sends to sp+1, sp+2, .. (each owner gets one of its slices first)
    if (tid == 0)
      for (int k = 1; k < (int)nsplit; ++k) {
        const int o = (sp + k) % (int)nsplit;
        const int k_st = (o - sp - 1 + (int)nsplit) % (int)nsplit;  // slot of this split at the owner
        asm volatile(
            "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                map_rank(smem_u32(recv_slot(k_st)), (uint32_t)o)),
            "r"(smem_u32(staging(k_st))), "r"(slice_bytes), "r"(map_rank(bar(kRecv), (uint32_t)o))
            : "memory");
      }
    // weights per (split, head) overwrite the pushed maxima; the external branch's in alpha
    if (tid >= 32 && tid < 96) {
      const int h = tid - 32;
      float M = -INFINITY;
      for (uint32_t s = 0; s < nsplit; ++s) M = fmaxf(M, ms.ml_in[s][0][h]);
      float mext = -INFINITY;
      if (out.o_ext) {
        mext = out.lse_ext[(int64_t)qi * H + (h < H ? h : 0)] * kLog2e;
        M = fmaxf(M, mext);
      }
      const float Mu = M == -INFINITY ? 0.f : M;
      float L = 0.f;
      for (uint32_t s = 0; s < nsplit; ++s) {
        const float ls = ms.ml_in[s][1][h];
        L += ls > 0.f ? ls * exp2f(ms.ml_in[s][0][h] - Mu) : 0.f;
      }
      const float wext = (out.o_ext && mext != -INFINITY) ? exp2f(mext - Mu) : 0.f;
      L += wext;
      const float inv = L > 0.f ? 1.f / L : 0.f;
      for (uint32_t s = 0; s < nsplit; ++s) {
        const float ls = ms.ml_in[s][1][h];
        ms.ml_in[s][0][h] = ls > 0.f ? exp2f(ms.ml_in[s][0][h] - Mu) * inv : 0.f;
      }
      ms.alpha[h] = wext * inv;
      if (sp == 0 && out.lse && h < H)
        out.lse[(int64_t)qi * H + h] = L > 0.f ? (Mu + log2f(L)) * kLn2 : -INFINITY;
    }
    __syncthreads();
    bool got = true;
    if (nsplit > 1) got = mbar_wait(bar(kRecv), 0);
    if (!__syncthreads_and(got)) {
      if (tid == 0) atomicOr(status, CSA2_DEV_PIPELINE_TIMEOUT);
    } else if (warp < 8) {
      // own M-tiles: every split's rows times its weight, plus the external branch;
      // each head's output row is written by consecutive lanes
      float* o = out.o + (int64_t)qi * H * kDV;
      const float* oe = out.o_ext ? out.o_ext + (int64_t)qi * H * kDV : nullptr;
      for (int j = 0; j < tiles_own; ++j) {
        const int i = sp * tiles_own + j;
        const int dl = 128 * j + e, d = 128 * i + e;
        uint32_t r[32];
        if (has) {
          tmem_ld32(tmem + lane_off + kColO + 64 * i + 32 * half, r);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) r[k] = 0u;
        }
        float acc[32];
#pragma unroll
        for (int k = 0; k < 32; k += 4) {
          const float4 w = *reinterpret_cast<const float4*>(&ms.ml_in[sp][0][32 * half + k]);
          acc[k] = __uint_as_float(r[k]) * w.x;
          acc[k + 1] = __uint_as_float(r[k + 1]) * w.y;
          acc[k + 2] = __uint_as_float(r[k + 2]) * w.z;
          acc[k + 3] = __uint_as_float(r[k + 3]) * w.w;
        }
        for (int s = 0; s + 1 < (int)nsplit; ++s) {
          const int src_sp = (sp - s - 1 + (int)nsplit) % (int)nsplit;  // sender of slot s
          const float* src = recv_slot(s);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float4 v = *reinterpret_cast<const float4*>(src + piece(dl, 8 * half + k));
            const float4 w = *reinterpret_cast<const float4*>(&ms.ml_in[src_sp][0][32 * half + 4 * k]);
            acc[4 * k] += w.x * v.x; acc[4 * k + 1] += w.y * v.y;
            acc[4 * k + 2] += w.z * v.z; acc[4 * k + 3] += w.w * v.w;
          }
        }
        if (kKind == kWindow && oe) {
          // all 32 loads issued before the first use
          float ev[32];
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            const int h = 32 * half + k;
            ev[k] = h < H ? __ldcs(oe + (int64_t)h * kDV + d) : 0.f;
          }
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            const float w = ms.alpha[32 * half + k];
            if (w > 0.f) acc[k] += w * ev[k];
          }
        }
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const int h = 32 * half + k;
          if (h < H) o[(int64_t)h * kDV + d] = acc[k];
        }
      }
    }
    // no CTA leaves while a peer may still copy out of (or into) it
    tc_fence_before();
    cluster_sync_all();
  } else {
  const int Dn = kDV / (int)nsplit;  // value dims owned by each CTA
  float* recv = reinterpret_cast<float*>(sC);                     // [src][dl][kRecvStride]
  float* ml = reinterpret_cast<float*>(sC + kMlOffset);           // [src][2][64]
  // every CTA of the cluster is past its last P.V: tile buffers may be overwritten
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  if (warp < 8) {
    const int quarter = warp & 3, half = warp >> 2;
    const int e = quarter * 32 + lane;
    const int wt = threadIdx.x;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    // (max, sum) per head of this split -> ml[sp] of every CTA
    if (wt < 64) {
      const float m = has ? ms.mrun[wt] : -INFINITY;
      const float s = has ? ms.lsum[wt] : 0.f;
      for (uint32_t p = 0; p < nsplit; ++p) {
        st_cluster_f32(map_rank(smem_u32(&ml[(sp * 2 + 0) * 64 + wt]), p), m);
        st_cluster_f32(map_rank(smem_u32(&ml[(sp * 2 + 1) * 64 + wt]), p), s);
      }
    }
    // unnormalised O^T rows (value dim 128 i + e, heads of this half) -> owner of the dim;
    // the M-tile order is rotated by split rank so the CTAs of a cluster push to
    // different owners at each step
    for (int ii = 0; ii < 4; ++ii) {
      const int i = (ii + sp) & 3;
      const int d = 128 * i + e;
      const uint32_t owner = (uint32_t)(d / Dn);
      const int dl = d - (int)owner * Dn;
      uint32_t r[32];
      if (has) {
        tmem_ld32(tmem + lane_off + kColO + 64 * i + 32 * half, r);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) r[k] = 0u;
      }
      const uint32_t dst =
          map_rank(smem_u32(&recv[((size_t)sp * Dn + dl) * kRecvStride + 32 * half]), owner);
#pragma unroll
      for (int k = 0; k < 8; ++k)
        st_cluster_v4(dst + 16 * k, __uint_as_float(r[4 * k]), __uint_as_float(r[4 * k + 1]),
                      __uint_as_float(r[4 * k + 2]), __uint_as_float(r[4 * k + 3]));
    }
  }
  tc_fence_before();
  cluster_sync_all();
  // weights per (split, head), the external branch, and normalised O for the owned dims
  if (warp < 8) {
    const int wt = threadIdx.x;
    constexpr float kLn2 = 0.69314718055994530942f, kLog2e = 1.4426950408889634074f;
    if (wt < 64) {
      float M = -INFINITY;
      for (uint32_t s = 0; s < nsplit; ++s) M = fmaxf(M, ml[(s * 2 + 0) * 64 + wt]);
      float mext = -INFINITY;
      if (out.o_ext) {
        mext = out.lse_ext[(int64_t)qi * H + (wt < H ? wt : 0)] * kLog2e;
        M = fmaxf(M, mext);
      }
      const float Mu = M == -INFINITY ? 0.f : M;
      float L = 0.f;
      for (uint32_t s = 0; s < nsplit; ++s) {
        const float ls = ml[(s * 2 + 1) * 64 + wt];
        L += ls > 0.f ? ls * exp2f(ml[(s * 2 + 0) * 64 + wt] - Mu) : 0.f;
      }
      const float wext = (out.o_ext && mext != -INFINITY) ? exp2f(mext - Mu) : 0.f;
      L += wext;
      const float inv = L > 0.f ? 1.f / L : 0.f;
      // overwrite the pushed maxima with the per-split weights
      for (uint32_t s = 0; s < nsplit; ++s) {
        const float ls = ml[(s * 2 + 1) * 64 + wt];
        ml[(s * 2 + 0) * 64 + wt] = ls > 0.f ? exp2f(ml[(s * 2 + 0) * 64 + wt] - Mu) * inv : 0.f;
      }
      ms.alpha[wt] = wext * inv;
      if (sp == 0 && out.lse && wt < H)
        out.lse[(int64_t)qi * H + wt] = L > 0.f ? (Mu + log2f(L)) * kLn2 : -INFINITY;
    }
    named_sync(1, kWorkers);
    float* o = out.o + (int64_t)qi * H * kDV;
    const float* oe = out.o_ext ? out.o_ext + (int64_t)qi * H * kDV : nullptr;
    const int base = sp * Dn;
    // item = (value dim dl, head quad hq) with dl fastest: the received rows are read
    // as conflict-free 16-byte vectors, and each head's output row is written by
    // consecutive threads (coalesced)
    const int items = Dn * 16;
    constexpr int kBatch = 4;
    for (int j0 = 0; j0 < items; j0 += kWorkers * kBatch) {
      float ext[kBatch][4];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int j = j0 + u * kWorkers + wt;
        const int dl = j % Dn, hq = j / Dn;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int h = 4 * hq + k;
          ext[u][k] = (oe && j < items && h < H && ms.alpha[h] > 0.f) ? oe[(int64_t)h * kDV + base + dl] : 0.f;
        }
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int j = j0 + u * kWorkers + wt;
        if (j >= items) continue;
        const int dl = j % Dn, hq = j / Dn;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (uint32_t s = 0; s < nsplit; ++s) {
          const float4 v = *reinterpret_cast<const float4*>(&recv[((size_t)s * Dn + dl) * kRecvStride + 4 * hq]);
          const float4 w = *reinterpret_cast<const float4*>(&ml[(s * 2 + 0) * 64 + 4 * hq]);
          acc.x += w.x * v.x; acc.y += w.y * v.y; acc.z += w.z * v.z; acc.w += w.w * v.w;
        }
        const float r4[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int h = 4 * hq + k;
          if (h < H) o[(int64_t)h * kDV + base + dl] = r4[k] + ms.alpha[h] * ext[u][k];
        }
      }
    }
  }
  }  // nsplit > 4

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

// Launch the (split, query) grid as clusters of nsplit CTAs (a power of two <= 16),
// allowing programmatic dependent launch after the preceding kernel.
template <int kKind>
static cudaError_t launch_tc(const CUtensorMap& tq, const Fp4Src& f, const RowSrc& r,
                             const CUtensorMap& trows, int Q, int T, int H, float scale_log2,
                             int nsplit, int split_len, const OutArgs& out, uint32_t* status,
                             cudaStream_t st) {
  constexpr int kSlotSmem = kKind == kSparse ? 2 : (kKind == kWindow ? 3 : 9);
  constexpr int kSlotCluster = kKind == kSparse ? 7 : (kKind == kWindow ? 8 : 10);
  cudaError_t e = set_attr_once(kSlotSmem, (const void*)attn_tc_kernel<kKind>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemTC);
  if (e != cudaSuccess) return e;
  e = set_attr_once(kSlotCluster, (const void*)attn_tc_kernel<kKind>,
                    cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)nsplit, (unsigned)Q);
  cfg.blockDim = dim3(kThreadsTC);
  cfg.dynamicSmemBytes = kSmemTC;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)nsplit;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, attn_tc_kernel<kKind>, tq, f, r, trows, T, H, scale_log2, split_len,
                            out, status);
}

cudaError_t launch_sparse_attn(int B, int T, int H, const void* q, const uint8_t* codes,
                               const uint8_t* scales, int64_t n_stride, const int32_t* idx, int K,
                               float scale_log2, float* o_g, float* lse_g, int nsplit,
                               float* xchg, uint32_t* status, cudaStream_t st) {
  const int Q = B * T;
  if (Q == 0) return cudaSuccess;
  if (nsplit < 1 || nsplit > kMaxSplitsTC || (nsplit & (nsplit - 1))) return cudaErrorInvalidValue;
  int split_len = (K + nsplit - 1) / nsplit;
  split_len = (split_len + kTK - 1) / kTK * kTK;
  Fp4Src f{codes, scales, codes != nullptr && scales == codes + CSA2_CODE_BYTES, n_stride, idx, K};
  RowSrc r{0, nullptr, nullptr, 0};
  CUtensorMap tq, dummy;
  memset(&dummy, 0, sizeof(dummy));
  if (!encode_tensor_map_2d_bf16(&tq, q, CSA2_D_KV, (uint64_t)Q * H, 64, 64)) return cudaErrorInvalidValue;
  OutArgs out{o_g, lse_g, nullptr, nullptr, xchg};
  return launch_tc<kSparse>(tq, f, r, dummy, Q, T, H, scale_log2, nsplit, split_len, out, status, st);
}

cudaError_t launch_swa_merge(int B, int T, int H, const void* q, const void* swa,
                             int64_t s_stride, const int32_t* win_start, const int32_t* win_len,
                             int n_win, float scale_log2, const float* o_g, const float* lse_g,
                             float* o_out, float* lse_out, uint32_t* status, cudaStream_t st) {
  const int Q = B * T;
  if (Q == 0) return cudaSuccess;
  int nsplit = 1;
  while (nsplit * kTK < n_win) nsplit <<= 1;   // power of two covering the window
  if (nsplit > kMaxSplitsTC) return cudaErrorInvalidValue;
  CUtensorMap tm, tq;
  memset(&tm, 0, sizeof(tm));
  if (!encode_tensor_map_2d_bf16(&tq, q, CSA2_D_KV, (uint64_t)Q * H, 64, 64)) return cudaErrorInvalidValue;
  if (s_stride > 0 && !encode_tensor_map_2d_bf16(&tm, swa, CSA2_D_KV, (uint64_t)B * s_stride, 64, kTK))
    return cudaErrorInvalidValue;
  Fp4Src f{nullptr, nullptr, false, 0, nullptr, 0};
  RowSrc r{s_stride, win_start, win_len, n_win};
  OutArgs out{o_out, lse_out, o_g, lse_g, nullptr};
  return launch_tc<kWindow>(tq, f, r, tm, Q, T, H, scale_log2, nsplit, kTK, out, status, st);
}

cudaError_t launch_decode_attn(int B, int T, int H, const void* q, const uint8_t* codes,
                               const uint8_t* scales, int64_t n_stride, const int32_t* idx, int K,
                               const void* swa, int64_t s_stride, const int32_t* win_start,
                               const int32_t* win_len, int n_win, float scale_log2, float* o,
                               float* lse, int nsplit, float* xchg, uint32_t* status, cudaStream_t st) {
  const int Q = B * T;
  if (Q == 0) return cudaSuccess;
  if (nsplit < 1 || nsplit > kMaxSplitsTC || (nsplit & (nsplit - 1))) return cudaErrorInvalidValue;
  int split_len = (K + nsplit - 1) / nsplit;
  split_len = (split_len + kTK - 1) / kTK * kTK;
  Fp4Src f{codes, scales, codes != nullptr && scales == codes + CSA2_CODE_BYTES, n_stride, idx, K};
  RowSrc r{s_stride, win_start, win_len, n_win};
  CUtensorMap tq, tm;
  memset(&tm, 0, sizeof(tm));
  if (!encode_tensor_map_2d_bf16(&tq, q, CSA2_D_KV, (uint64_t)Q * H, 64, 64)) return cudaErrorInvalidValue;
  if (s_stride > 0 && !encode_tensor_map_2d_bf16(&tm, swa, CSA2_D_KV, (uint64_t)B * s_stride, 64, kTK))
    return cudaErrorInvalidValue;
  OutArgs out{o, lse, nullptr, nullptr, xchg};
  return launch_tc<kFused>(tq, f, r, tm, Q, T, H, scale_log2, nsplit, split_len, out, status, st);
}

}  // namespace csa2
