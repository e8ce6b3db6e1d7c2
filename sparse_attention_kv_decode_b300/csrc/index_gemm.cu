// Indexer scoring of many query tokens of one sequence on the tensor cores.
//
// Ref: "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression", picx.dev
// summary, Methodology / 2. CSA2 (the indexer ranks every compressed entry for every
// query token before the top-K) and / 3 (indexer cost grows with the context). The
// pages give no indexer formula; this library scores
//   I[t, n] = sum_h w[t, h] * max(0, q[t, h] . z[n])   (h < H_I).
//
// With T query tokens of one sequence (a prefill chunk) the dot products form a GEMM:
// S[n, (t, h)] = z[n] . q[t, h], keys as M (128 per tile), a tile of T_tile = 256 / H_I
// tokens x H_I heads as N = 256, and the 64 channels as K (four K = 16 steps). The keys
// are then read once per token tile instead of once per token.
//   warp 0      TMA producer: the token tile's q rows (32 KB, once per work item) and
//               one 128-key z box per key tile into a ring of stages (128-byte swizzle)
//   warp 1      TMEM allocation and the MMA issuer: tcgen05.mma kind::f16, M=128,
//               N=256, K=16, fp32 accumulators in TMEM, double-buffered (2 x 256
//               columns) so the epilogue of one key tile overlaps the MMAs of the next
//   warps 2..17 epilogue: thread = key row (TMEM lane); each of the four warpgroups
//               takes a quarter of the columns, applies max(0, .), weights the heads
//               by w[t, h] (fp32), sums them, and stores one fp32 score per (token, key) below the
//               token's causal limit, plus the token's running min / max score (the
//               range words the selection starts from).
// A work item is (sequence, token tile, chunk of key tiles); the key tiles past the
// token tile's largest visible count are skipped. Every mbarrier wait is bounded.
#include <climits>
#include <cuda.h>

#include "csa2_internal.cuh"

namespace csa2 {
namespace {

constexpr int kGM = 128;                         // keys per tile
constexpr int kGN = 256;                         // (token, head) columns per tile
constexpr int kGStages = 6;
constexpr int kGZBytes = kGM * CSA2_D_IDX * 2;   // 16 KB
constexpr int kGQBytes = kGN * CSA2_D_IDX * 2;   // 32 KB
constexpr int kGEpiWarps = 16;                   // four warpgroups, a quarter of the columns each
constexpr int kGThreads = 64 + 32 * kGEpiWarps;
constexpr int kGTmemCols = 512;
constexpr int kGMaxTT = 64;                      // tokens per tile for H_I = 4
constexpr size_t kGSmem = 1024 + kGQBytes + kGStages * kGZBytes + 4096;

struct GemmShape {
  int B, T, ntt, nchunks, kpc;
  int64_t n_stride;
  __device__ __forceinline__ int total() const { return B * ntt * nchunks; }
};

template <int HI>
__device__ __forceinline__ void item_coords(const GemmShape& g, const int32_t* n_visible, int it, int& b,
                                            int& t0, int& nt, int& kt0, int& kt1) {
  constexpr int TT = kGN / HI;
  const int c = it % g.nchunks;
  const int j = (it / g.nchunks) % g.ntt;
  b = it / (g.nchunks * g.ntt);
  t0 = j * TT;
  nt = min(TT, g.T - t0);
  int maxnv = 0;
  for (int t = 0; t < nt; ++t) {
    int v = n_visible[(int64_t)b * g.T + t0 + t];
    v = v < 0 ? 0 : (v > g.n_stride ? (int)g.n_stride : v);
    maxnv = max(maxnv, v);
  }
  const int nkt = (maxnv + kGM - 1) / kGM;
  kt0 = c * g.kpc;
  kt1 = min(kt0 + g.kpc, nkt);
}

__device__ __forceinline__ void named_bar(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
// OR of a predicate over the n threads of named barrier id (all of them get the result).
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

template <int HI>
__global__ void __launch_bounds__(kGThreads, 1) index_gemm_kernel(
    const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_q,
    const float* __restrict__ w_idx, const int32_t* __restrict__ n_visible, GemmShape g,
    float* __restrict__ scores, int64_t score_stride, uint32_t* __restrict__ range,
    uint32_t* __restrict__ status) {
  constexpr int TT = kGN / HI;
  static_assert(TT <= kGMaxTT && kGN % HI == 0 && 32 % HI == 0 && HI % 4 == 0, "token tile");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sq = smem_u32(smem);
  const uint32_t sz = sq + kGQBytes;
  uint8_t* misc = smem + kGQBytes + kGStages * kGZBytes;
  const uint32_t bar_full = smem_u32(misc);
  const uint32_t bar_empty = bar_full + 8 * kGStages;
  const uint32_t bar_tfull = bar_empty + 8 * kGStages;
  const uint32_t bar_tempty = bar_tfull + 16;
  const uint32_t bar_qfull = bar_tempty + 16;
  const uint32_t bar_qempty = bar_qfull + 8;
  const uint32_t bar_drain = bar_qempty + 8;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(misc + 256);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 260);
  float* w_s = reinterpret_cast<float*>(misc + 512);                  // [TT * HI]
  int* nv_s = reinterpret_cast<int*>(misc + 512 + kGN * 4);           // [TT]
  uint32_t* rng_s = reinterpret_cast<uint32_t*>(misc + 512 + kGN * 4 + kGMaxTT * 4);  // [TT][2]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kGStages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar_tfull + 8 * a, 1);
      mbar_init(bar_tempty + 8 * a, kGEpiWarps);
    }
    mbar_init(bar_qfull, 1);
    mbar_init(bar_qempty, 1);
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_holder)),
                 "r"(kGTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  // inputs may be written by the preceding kernel in the stream
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int total = g.total();

  if (warp == 0) {
    // ---------------- TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, qphase = 0;
      bool armed[kGStages];
      uint32_t armed_phase[kGStages];
      for (int s = 0; s < kGStages; ++s) armed[s] = false, armed_phase[s] = 0;
      bool q_armed = false;
      uint32_t q_armed_phase = 0;
      for (int it = blockIdx.x; it < total && !*abort_flag; it += gridDim.x) {
        int b, t0, nt, kt0, kt1;
        item_coords<HI>(g, n_visible, it, b, t0, nt, kt0, kt1);
        if (kt0 >= kt1) continue;
        // the q tile of the previous item is released by its last MMAs
        if (!mbar_wait(bar_qempty, qphase ^ 1)) {
          atomicOr(status, CSA2_DEV_PIPELINE_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(bar_qfull, kGQBytes);
        q_armed = true;
        q_armed_phase = qphase;
        tma_load_2d(sq, &tm_q, 0, (b * g.T + t0) * HI, bar_qfull);
        qphase ^= 1;
        for (int kt = kt0; kt < kt1; ++kt) {
          if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1)) {
            atomicOr(status, CSA2_DEV_PIPELINE_TIMEOUT);
            *abort_flag = 1;
            break;
          }
          const uint32_t fb = bar_full + 8 * stage;
          mbar_arrive_expect_tx(fb, kGZBytes);
          armed[stage] = true;
          armed_phase[stage] = phase;
          // rows past this sequence's cache belong to the next one (or read as zeros): their
          // keys are past every token's visible count, so their scores are never stored
          tma_load_2d(sz + stage * kGZBytes, &tm_z, 0, (int)((int64_t)b * g.n_stride + (int64_t)kt * kGM), fb);
          if (++stage == kGStages) stage = 0, phase ^= 1;
        }
      }
      // drain: every armed copy has landed before the CTA may exit
      for (int s = 0; s < kGStages; ++s)
        if (armed[s]) mbar_wait(bar_full + 8 * s, armed_phase[s]);
      if (q_armed) mbar_wait(bar_qfull, q_armed_phase);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kGM, kGN);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0, qphase = 0;
      bool issued = false;
      for (int it = blockIdx.x; it < total && !*abort_flag; it += gridDim.x) {
        int b, t0, nt, kt0, kt1;
        item_coords<HI>(g, n_visible, it, b, t0, nt, kt0, kt1);
        if (kt0 >= kt1) continue;
        if (!mbar_wait(bar_qfull, qphase)) {
          atomicOr(status, CSA2_DEV_PIPELINE_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        qphase ^= 1;
        tc_fence_after();
        const uint64_t bd = umma_desc_sw128(sq);
        bool ok = true;
        for (int kt = kt0; kt < kt1; ++kt) {
          if (!mbar_wait(bar_tempty + 8 * acc, acc_phase ^ 1) || !mbar_wait(bar_full + 8 * stage, phase)) {
            atomicOr(status, CSA2_DEV_PIPELINE_TIMEOUT);
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = umma_desc_sw128(sz + stage * kGZBytes);
          const uint32_t d_tmem = tmem + acc * kGN;
#pragma unroll
          for (int k = 0; k < CSA2_D_IDX / 16; ++k)
            umma_bf16(d_tmem, ad + (uint64_t)(k * 2), bd + (uint64_t)(k * 2), idesc, k != 0);
          umma_commit(bar_empty + 8 * stage);
          umma_commit(bar_tfull + 8 * acc);
          issued = true;
          if (++stage == kGStages) stage = 0, phase ^= 1;
          if (++acc == 2) acc = 0, acc_phase ^= 1;
        }
        umma_commit(bar_qempty);
        if (!ok) break;
      }
      if (issued) {
        umma_commit(bar_drain);
        mbar_wait(bar_drain, 0);
      }
    }
  } else {
    // ---------------- epilogue: thread = key row, warpgroup = a quarter of the columns
    constexpr int kCols = kGN / (kGEpiWarps / 4);   // 64 columns per warpgroup
    const int ew = warp - 2;                 // 0..15
    const int quarter = warp & 3;            // TMEM lanes 32 * quarter ..
    const int grp = ew >> 2;                 // columns [kCols grp, kCols grp + kCols)
    const int et = threadIdx.x - 64;         // 0..511
    const int key = quarter * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    // The epilogue warps meet at named barrier 1 only at item boundaries, and every one of
    // them reaches each of those meetings (a warp whose wait gave up skips its remaining
    // tiles, not the meetings), so the abort decision taken there is the same for all.
    for (int it = blockIdx.x; it < total; it += gridDim.x) {
      int b, t0, nt, kt0, kt1;
      item_coords<HI>(g, n_visible, it, b, t0, nt, kt0, kt1);
      if (kt0 >= kt1) continue;
      // also: the previous item's readers of w_s / nv_s / rng_s are done
      if (named_or(1, 32 * kGEpiWarps, *abort_flag != 0)) break;
      if (et < kGN) {
        const int tl = et / HI;
        w_s[et] = tl < nt ? w_idx[((int64_t)b * g.T + t0) * HI + et] : 0.f;
        if (et < TT) {
          int v = et < nt ? n_visible[(int64_t)b * g.T + t0 + et] : 0;
          nv_s[et] = v < 0 ? 0 : (v > g.n_stride ? (int)g.n_stride : v);
          rng_s[2 * et] = 0u;
          rng_s[2 * et + 1] = 0u;
        }
      }
      named_bar(1, 32 * kGEpiWarps);
      // this thread's tokens are tl0 .. tl0 + kTh - 1 (its warpgroup's columns); running
      // min / max of their visible scores over the item's key tiles
      constexpr int kTh = kCols / HI;
      const int tl0 = kCols * grp / HI;
      float mn[kTh], mx[kTh];
#pragma unroll
      for (int i = 0; i < kTh; ++i) mn[i] = INFINITY, mx[i] = -INFINITY;
      int min_nv = INT_MAX;
#pragma unroll
      for (int i = 0; i < kTh; ++i)
        if (tl0 + i < nt) min_nv = min(min_nv, nv_s[tl0 + i]);
      for (int kt = kt0; kt < kt1; ++kt) {
        const bool got = __all_sync(0xffffffffu, mbar_wait(bar_tfull + 8 * acc, acc_phase));
        if (!got) {
          if (lane == 0) atomicOr(status, CSA2_DEV_PIPELINE_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const int n = kt * kGM + key;
        // every token of these columns sees every key of the tile (the common case)
        const bool full = (kt + 1) * kGM <= min_nv;
        const uint32_t tbase = tmem + acc * kGN + ((uint32_t)(quarter * 32) << 16) + kCols * grp;
#pragma unroll
        for (int c4 = 0; c4 < kCols / 32; ++c4) {
          uint32_t r[32];
          tmem_ld32(tbase + 32 * c4, r);
          tmem_wait_ld();
#pragma unroll
          for (int tk = 0; tk < 32 / HI; ++tk) {
            const int ti = c4 * (32 / HI) + tk;   // token of these columns
            const int tl = tl0 + ti;
            // the token's head weights as 16-byte shared-memory loads
            float wt[HI];
#pragma unroll
            for (int h = 0; h < HI; h += 4) {
              const float4 w4 = *reinterpret_cast<const float4*>(w_s + tl * HI + h);
              wt[h] = w4.x; wt[h + 1] = w4.y; wt[h + 2] = w4.z; wt[h + 3] = w4.w;
            }
            // two independent partial sums (even / odd heads)
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int h = 0; h < HI; h += 2) {
              s0 = fmaf(wt[h], fmaxf(__uint_as_float(r[tk * HI + h]), 0.f), s0);
              s1 = fmaf(wt[h + 1], fmaxf(__uint_as_float(r[tk * HI + h + 1]), 0.f), s1);
            }
            const float sc = s0 + s1;
            const bool valid = tl < nt && (full || n < nv_s[tl]);
            if (valid) {
              scores[((int64_t)b * g.T + t0 + tl) * score_stride + n] = sc;
              mn[ti] = fminf(mn[ti], sc);
              mx[ti] = fmaxf(mx[ti], sc);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_tempty + 8 * acc);
        if (++acc == 2) acc = 0, acc_phase ^= 1;
      }
      // this warp's share of each token's range, then the CTA's into the range words
#pragma unroll
      for (int i = 0; i < kTh; ++i) {
        const bool any = mx[i] >= mn[i];
        const uint32_t kmax = __reduce_max_sync(0xffffffffu, any ? f2key(mx[i]) : 0u);
        const uint32_t kinv = __reduce_max_sync(0xffffffffu, any ? ~f2key(mn[i]) : 0u);
        if (lane == 0 && kmax != 0u) {
          atomicMax(&rng_s[2 * (tl0 + i)], kinv);
          atomicMax(&rng_s[2 * (tl0 + i) + 1], kmax);
        }
      }
      // the item's score range per token into the range words
      named_bar(1, 32 * kGEpiWarps);
      if (et < nt && rng_s[2 * et + 1] != 0u) {
        atomicMax(range + 2 * ((int64_t)b * g.T + t0 + et), rng_s[2 * et]);
        atomicMax(range + 2 * ((int64_t)b * g.T + t0 + et) + 1, rng_s[2 * et + 1]);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kGTmemCols)
                 : "memory");
  }
}


// ---------------------------------------------------------------------------
// Few query tokens per sequence (decode): the same contraction with N = 16, i.e. the
// indexer heads of 16 / H_I tokens, so that every key is read once per 16 / H_I tokens
// and the tensor cores do the dot products while the key stream runs at HBM speed.
//   warp 0      TMA producer: one 128-key z box (16 KB) per stage into a ring of
//               kSStages stages, and the q rows (2 KB) of each (sequence, token tile)
//               into one of two q buffers
//   warp 1      TMEM allocation and the MMA issuer: M = 128, N = 16, K = 16 x 4,
//               accumulators in kSAcc TMEM buffers of 16 columns
//   warps 2..9  epilogue, two warpgroups taking alternate key tiles: thread = key row,
//               one 16-column TMEM load, max(0, .) and the head weights per token, one
//               fp32 score per (token, key) below the token's visible count, and the
//               token's running min / max score (the range words)
// The key tiles each (sequence, token tile) needs (its largest visible count, in
// 128-key tiles) are counted on the device and the whole list is split evenly over
// the CTAs, so ragged batches keep every SM equally busy.
constexpr int kSN = 16;
constexpr int kSStages = 8;
constexpr int kSAcc = 4;
constexpr int kSQBytes = kSN * CSA2_D_IDX * 2;   // 2 KB
constexpr int kSEpiWarps = 8;
constexpr int kSThreads = 64 + 32 * kSEpiWarps;
constexpr int kSTmemCols = 64;
constexpr int kSMaxBj = 2048;                   // (sequence, token tile) pairs
constexpr size_t kSSmem = 1024 + kSStages * kGZBytes + 2 * kSQBytes + 1024 + 4 * (kSMaxBj + 1);

struct StreamShape {
  int B, T, ntt, nbj;
  int64_t n_stride;
};

// The first (sequence, token tile) whose tiles reach past tile t: pre[bj + 1] > t.
__device__ __forceinline__ int first_bj(const int* pre, int nbj, int t) {
  int lo = 0, hi = nbj - 1;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (pre[mid + 1] > t) hi = mid;
    else lo = mid + 1;
  }
  return lo;
}

template <int HI>
__global__ void __launch_bounds__(kSThreads, 1) index_stream_kernel(
    const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_q,
    const float* __restrict__ w_idx, const int32_t* __restrict__ n_visible, StreamShape g,
    float* __restrict__ scores, int64_t score_stride, uint32_t* __restrict__ range,
    uint32_t* __restrict__ status) {
  constexpr int TT = kSN / HI;
  static_assert(kSN % HI == 0, "token tile");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sz = smem_u32(smem);
  const uint32_t sq = sz + kSStages * kGZBytes;
  uint8_t* misc = smem + kSStages * kGZBytes + 2 * kSQBytes;
  const uint32_t bar_full = smem_u32(misc);
  const uint32_t bar_empty = bar_full + 8 * kSStages;
  const uint32_t bar_tfull = bar_empty + 8 * kSStages;
  const uint32_t bar_tempty = bar_tfull + 8 * kSAcc;
  const uint32_t bar_qfull = bar_tempty + 8 * kSAcc;
  const uint32_t bar_qempty = bar_qfull + 16;
  const uint32_t bar_drain = bar_qempty + 16;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(misc + 512);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 516);
  int* pre = reinterpret_cast<int*>(misc + 1024);   // [nbj + 1] key tiles before each pair

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kSStages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int a = 0; a < kSAcc; ++a) {
      mbar_init(bar_tfull + 8 * a, 1);
      mbar_init(bar_tempty + 8 * a, 4);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar_qfull + 8 * a, 1);
      mbar_init(bar_qempty + 8 * a, 1);
    }
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_holder)),
                 "r"(kSTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // inputs (and the visible counts) may be written by the preceding kernel in the stream
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // key tiles per (sequence, token tile), then their running sum
  for (int bj = threadIdx.x; bj < g.nbj; bj += kSThreads) {
    const int b = bj / g.ntt, t0 = (bj % g.ntt) * TT, nt = min(TT, g.T - t0);
    int mx = 0;
    for (int t = 0; t < nt; ++t) {
      int v = n_visible[(int64_t)b * g.T + t0 + t];
      v = v < 0 ? 0 : (v > g.n_stride ? (int)g.n_stride : v);
      mx = max(mx, v);
    }
    pre[bj + 1] = (mx + kGM - 1) / kGM;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) {
    int carry = 0;
    for (int base = 0; base < g.nbj; base += 32) {
      const int j = base + lane;
      int v = j < g.nbj ? pre[j + 1] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += y;
      }
      if (j < g.nbj) pre[j + 1] = v + carry;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
    if (lane == 0) pre[0] = 0;
  }
  __syncthreads();
  const uint32_t tmem = *tmem_holder;
  const int total = g.nbj > 0 ? pre[g.nbj] : 0;
  const int t_begin = (int)((int64_t)total * blockIdx.x / gridDim.x);
  const int t_end = (int)((int64_t)total * (blockIdx.x + 1) / gridDim.x);

  if (warp == 0) {
    // ---------------- TMA producer
    if (lane == 0 && t_begin < t_end) {
      // bit s: stage s (q buffer s) holds a copy; its phase bit: the parity of that copy
      uint32_t armed = 0u, armed_phase = 0u, q_armed = 0u, q_armed_phase = 0u;
      int bj = first_bj(pre, g.nbj, t_begin), prev_bj = -1, qn = -1;
      for (int t = t_begin, i = 0; t < t_end && !*abort_flag; ++t, ++i) {
        while (t >= pre[bj + 1]) ++bj;
        const int b = bj / g.ntt, t0 = (bj % g.ntt) * TT;
        if (bj != prev_bj) {
          ++qn;
          const int qb = qn & 1;
          const uint32_t qph = (uint32_t)(qn >> 1) & 1u;
          if (!mbar_wait(bar_qempty + 8 * qb, qph ^ 1u)) {
            atomicOr(status, CSA2_DEV_PIPELINE_TIMEOUT);
            *abort_flag = 1;
            break;
          }
          mbar_arrive_expect_tx(bar_qfull + 8 * qb, kSQBytes);
          q_armed |= 1u << qb;
          q_armed_phase = (q_armed_phase & ~(1u << qb)) | (qph << qb);
          // rows past the last token of the tile (another sequence's, or zeros past the
          // end) only feed columns whose scores are never stored
          tma_load_2d(sq + qb * kSQBytes, &tm_q, 0, (b * g.T + t0) * HI, bar_qfull + 8 * qb);
          prev_bj = bj;
        }
        const int stage = i % kSStages;
        const uint32_t ph = (uint32_t)(i / kSStages) & 1u;
        if (!mbar_wait(bar_empty + 8 * stage, ph ^ 1u)) {
          atomicOr(status, CSA2_DEV_PIPELINE_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(bar_full + 8 * stage, kGZBytes);
        armed |= 1u << stage;
        armed_phase = (armed_phase & ~(1u << stage)) | (ph << stage);
        const int kt = t - pre[bj];
        tma_load_2d(sz + stage * kGZBytes, &tm_z, 0, (int)((int64_t)b * g.n_stride + (int64_t)kt * kGM),
                    bar_full + 8 * stage);
      }
      // drain: every armed copy has landed before the CTA may exit
      for (int s = 0; s < kSStages; ++s)
        if ((armed >> s) & 1u) mbar_wait(bar_full + 8 * s, (armed_phase >> s) & 1u);
      for (int a = 0; a < 2; ++a)
        if ((q_armed >> a) & 1u) mbar_wait(bar_qfull + 8 * a, (q_armed_phase >> a) & 1u);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0 && t_begin < t_end) {
      constexpr uint32_t idesc = idesc_bf16_f32(kGM, kSN);
      bool issued = false;
      int bj = first_bj(pre, g.nbj, t_begin), prev_bj = -1, qn = -1;
      for (int t = t_begin, i = 0; t < t_end && !*abort_flag; ++t, ++i) {
        while (t >= pre[bj + 1]) ++bj;
        if (bj != prev_bj) {
          // the previous q buffer is free once the MMAs issued so far are done
          if (qn >= 0) umma_commit(bar_qempty + 8 * (qn & 1));
          ++qn;
          if (!mbar_wait(bar_qfull + 8 * (qn & 1), (uint32_t)(qn >> 1) & 1u)) {
            atomicOr(status, CSA2_DEV_PIPELINE_TIMEOUT);
            *abort_flag = 1;
            break;
          }
          prev_bj = bj;
        }
        const int stage = i % kSStages, acc = i % kSAcc;
        const uint32_t ph = (uint32_t)(i / kSStages) & 1u, aph = (uint32_t)(i / kSAcc) & 1u;
        if (!mbar_wait(bar_tempty + 8 * acc, aph ^ 1u) || !mbar_wait(bar_full + 8 * stage, ph)) {
          atomicOr(status, CSA2_DEV_PIPELINE_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint64_t ad = umma_desc_sw128(sz + stage * kGZBytes);
        const uint64_t bd = umma_desc_sw128(sq + (qn & 1) * kSQBytes);
#pragma unroll
        for (int k = 0; k < CSA2_D_IDX / 16; ++k)
          umma_bf16(tmem + acc * kSN, ad + (uint64_t)(k * 2), bd + (uint64_t)(k * 2), idesc, k != 0);
        umma_commit(bar_empty + 8 * stage);
        umma_commit(bar_tfull + 8 * acc);
        issued = true;
      }
      if (issued) {
        umma_commit(bar_drain);
        mbar_wait(bar_drain, 0);
      }
    }
  } else {
    // ---------------- epilogue: warpgroup wg takes the CTA's key tiles i with i % 2 == wg
    const int wg = (warp - 2) >> 2;
    const int quarter = warp & 3;   // TMEM lanes 32 * quarter ..
    const uint32_t tlane = (uint32_t)(quarter * 32) << 16;
    float wv[TT][HI];
    int nv[TT];
    float mn[TT], mx[TT];
    int q0 = 0, nt = 0, cur_bj = -1;
    auto flush = [&]() {
#pragma unroll
      for (int tl = 0; tl < TT; ++tl) {
        const bool any = tl < nt && mx[tl] >= mn[tl];
        const uint32_t kmax = __reduce_max_sync(0xffffffffu, any ? f2key(mx[tl]) : 0u);
        const uint32_t kinv = __reduce_max_sync(0xffffffffu, any ? ~f2key(mn[tl]) : 0u);
        if (lane == 0 && kmax != 0u) {
          atomicMax(range + 2 * (int64_t)(q0 + tl), kinv);
          atomicMax(range + 2 * (int64_t)(q0 + tl) + 1, kmax);
        }
      }
    };
    if (t_begin < t_end) {
      int bj = first_bj(pre, g.nbj, t_begin);
      for (int t = t_begin, i = 0; t < t_end; ++t, ++i) {
        while (t >= pre[bj + 1]) ++bj;
        if ((i & 1) != wg) continue;
        if (bj != cur_bj) {
          if (cur_bj >= 0) flush();
          const int b = bj / g.ntt, t0 = (bj % g.ntt) * TT;
          q0 = b * g.T + t0;
          nt = min(TT, g.T - t0);
#pragma unroll
          for (int tl = 0; tl < TT; ++tl) {
            int v = tl < nt ? n_visible[q0 + tl] : 0;
            nv[tl] = v < 0 ? 0 : (v > g.n_stride ? (int)g.n_stride : v);
            mn[tl] = INFINITY;
            mx[tl] = -INFINITY;
#pragma unroll
            for (int h = 0; h < HI; ++h) wv[tl][h] = tl < nt ? w_idx[(int64_t)(q0 + tl) * HI + h] : 0.f;
          }
          cur_bj = bj;
        }
        const int acc = i % kSAcc;
        const bool got = __all_sync(0xffffffffu, mbar_wait(bar_tfull + 8 * acc, (uint32_t)(i / kSAcc) & 1u));
        if (!got) {
          if (lane == 0) atomicOr(status, CSA2_DEV_PIPELINE_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        uint32_t r[kSN];
        tmem_ld16(tmem + acc * kSN + tlane, r);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_tempty + 8 * acc);
        const int n = (t - pre[bj]) * kGM + quarter * 32 + lane;
#pragma unroll
        for (int tl = 0; tl < TT; ++tl) {
          // two independent partial sums (even / odd heads)
          float s0 = 0.f, s1 = 0.f;
#pragma unroll
          for (int h = 0; h < HI; h += 2) {
            s0 = fmaf(wv[tl][h], fmaxf(__uint_as_float(r[tl * HI + h]), 0.f), s0);
            s1 = fmaf(wv[tl][h + 1], fmaxf(__uint_as_float(r[tl * HI + h + 1]), 0.f), s1);
          }
          const float sc = s0 + s1;
          if (tl < nt && n < nv[tl]) {
            scores[(int64_t)(q0 + tl) * score_stride + n] = sc;
            mn[tl] = fminf(mn[tl], sc);
            mx[tl] = fmaxf(mx[tl], sc);
          }
        }
      }
      if (cur_bj >= 0) flush();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kSTmemCols)
                 : "memory");
  }
}

}  // namespace

bool index_gemm_applies(int T, int H_I) {
  return (H_I == 4 || H_I == 8 || H_I == 16) && T >= kGN / H_I;
}

cudaError_t launch_index_gemm(const void* q_idx, const float* w_idx, const void* z, int64_t n_stride,
                              const int32_t* n_visible, int B, int T, int H_I, float* scores,
                              int64_t score_stride, uint32_t* range, uint32_t* status, cudaStream_t st) {
  if (B == 0 || T == 0 || n_stride == 0) return cudaSuccess;
  if (!index_gemm_applies(T, H_I)) return cudaErrorInvalidValue;
  if ((int64_t)B * n_stride > ((int64_t)1 << 31) - kGM || (int64_t)B * T * H_I > ((int64_t)1 << 31) - kGN)
    return cudaErrorInvalidValue;
  CUtensorMap tz, tq;
  if (!encode_tensor_map_2d_bf16(&tz, z, CSA2_D_IDX, (uint64_t)B * n_stride, CSA2_D_IDX, kGM) ||
      !encode_tensor_map_2d_bf16(&tq, q_idx, CSA2_D_IDX, (uint64_t)B * T * H_I, CSA2_D_IDX, kGN))
    return cudaErrorInvalidValue;
  GemmShape g;
  g.B = B;
  g.T = T;
  g.n_stride = n_stride;
  const int TT = kGN / H_I;
  g.ntt = (T + TT - 1) / TT;
  const int nkt = (int)((n_stride + kGM - 1) / kGM);
  const int n_sm = device_sm_count();
  const int64_t base = (int64_t)B * g.ntt;
  int64_t nch = (4 * (int64_t)n_sm + base - 1) / base;   // about four items per SM
  if (nch > nkt) nch = nkt;
  if (nch < 1) nch = 1;
  g.kpc = (int)((nkt + nch - 1) / nch);
  g.nchunks = (nkt + g.kpc - 1) / g.kpc;
  const int64_t total = base * g.nchunks;
  if (total > ((int64_t)1 << 31) - 1) return cudaErrorInvalidValue;
  const int grid = (int)(total < n_sm ? total : n_sm);
  const void* fn = H_I == 4 ? (const void*)index_gemm_kernel<4>
                   : (H_I == 8 ? (const void*)index_gemm_kernel<8> : (const void*)index_gemm_kernel<16>);
  const int slot = H_I == 4 ? 11 : (H_I == 8 ? 12 : 13);
  cudaError_t e = set_attr_once(slot, fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kGThreads);
  cfg.dynamicSmemBytes = kGSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (H_I == 4)
    return cudaLaunchKernelEx(&cfg, index_gemm_kernel<4>, tz, tq, w_idx, n_visible, g, scores, score_stride, range,
                              status);
  if (H_I == 8)
    return cudaLaunchKernelEx(&cfg, index_gemm_kernel<8>, tz, tq, w_idx, n_visible, g, scores, score_stride, range,
                              status);
  return cudaLaunchKernelEx(&cfg, index_gemm_kernel<16>, tz, tq, w_idx, n_visible, g, scores, score_stride, range,
                            status);
}


// Worth it when a key tile serves more than one token (T >= 2 with H_I = 4 or 8): the
// tile's TMA copies stream at a little under the HBM rate on this part, so with one token
// per tile the direct-load scoring kernel (which keeps more bytes in flight) is faster.
bool index_stream_applies(int B, int T, int H_I) {
  if (!(H_I == 4 || H_I == 8) || B <= 0 || T < 2) return false;
  const int tt = kSN / H_I;
  return (int64_t)B * ((T + tt - 1) / tt) <= kSMaxBj;
}

cudaError_t launch_index_stream(const void* q_idx, const float* w_idx, const void* z, int64_t n_stride,
                                const int32_t* n_visible, int B, int T, int H_I, float* scores,
                                int64_t score_stride, uint32_t* range, uint32_t* status, cudaStream_t st) {
  if (B == 0 || T == 0 || n_stride == 0) return cudaSuccess;
  if (!index_stream_applies(B, T, H_I)) return cudaErrorInvalidValue;
  if ((int64_t)B * n_stride > ((int64_t)1 << 31) - kGM || (int64_t)B * T * H_I > ((int64_t)1 << 31) - kSN)
    return cudaErrorInvalidValue;
  CUtensorMap tz, tq;
  if (!encode_tensor_map_2d_bf16(&tz, z, CSA2_D_IDX, (uint64_t)B * n_stride, CSA2_D_IDX, kGM) ||
      !encode_tensor_map_2d_bf16(&tq, q_idx, CSA2_D_IDX, (uint64_t)B * T * H_I, CSA2_D_IDX, kSN))
    return cudaErrorInvalidValue;
  StreamShape g;
  g.B = B;
  g.T = T;
  g.n_stride = n_stride;
  const int tt = kSN / H_I;
  g.ntt = (T + tt - 1) / tt;
  g.nbj = B * g.ntt;
  const int64_t nkt = (n_stride + kGM - 1) / kGM;
  const int n_sm = device_sm_count();
  const int64_t most = (int64_t)g.nbj * nkt;   // key tiles with every position visible
  const int grid = (int)(most < n_sm ? most : n_sm);
  const void* fn = H_I == 4 ? (const void*)index_stream_kernel<4> : (const void*)index_stream_kernel<8>;
  const int slot = H_I == 4 ? 14 : 15;
  cudaError_t e = set_attr_once(slot, fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kSThreads);
  cfg.dynamicSmemBytes = kSSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (H_I == 4)
    return cudaLaunchKernelEx(&cfg, index_stream_kernel<4>, tz, tq, w_idx, n_visible, g, scores, score_stride,
                              range, status);
  return cudaLaunchKernelEx(&cfg, index_stream_kernel<8>, tz, tq, w_idx, n_visible, g, scores, score_stride,
                            range, status);
}

}  // namespace csa2
