// Indexer scoring and per-query top-K selection (csa2_index_topk).
//
// CSA2 layer modes: "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache
// Compression", picx.dev summary, Methodology / 2. Compressed Sparse Attention
// 2: FULL and REINDEX layers compute fresh top-K indices from their indexer,
// REUSE layers take the preceding layer's. The pages give no indexer formula;
// this library scores I[n] = sum_h w[h] * max(0, q[h] . z[n]).
//
// Scoring (HBM-bound: 128 B of keys per entry, ~8 FLOP per key byte) runs on
// the tensor cores through m16n8k16 bf16 MMAs with 16 keys as M and 8 indexer
// heads as N, fed by plain 16-byte loads. Selection runs in one thread-block cluster
// per query: every CTA keeps its slice of scores in shared memory and the
// cluster agrees on the K-th score through a few histogram rounds exchanged
// over distributed shared memory (no global atomics, no spin waits).
#include "csa2_internal.cuh"

namespace csa2 {

// ---------------------------------------------------------------------------
// Scoring
// ---------------------------------------------------------------------------
// The scoring is a pure stream over the keys (4 MiB per query at 128K context),
// so it is written for memory-level parallelism with nothing to synchronise:
// every warp owns a contiguous, balanced run of 16-key groups (a query at a
// time) and loads each group's MMA fragments straight from global memory into
// registers, kScoreUnroll groups (8 x 16-byte loads per thread) in flight. A
// group is scored with four m16n8k16 bf16 MMAs per 8 indexer heads: thread
// (g = lane/4, tig = lane%4) holds, for key rows g and g+8, the 16-byte pieces
// at byte offsets 16*tig and 64+16*tig; the MMA's k-slots are assigned to
// channels so that these words are exactly the A fragment, and the B fragment
// (the indexer query of head g) is read from the same offsets: the contraction
// order is a permutation of the 64 channels, which leaves each dot product
// unchanged.
constexpr int kScoreThreads = 512;
constexpr int kScoreCtasPerSm = 2;
constexpr int kScoreUnroll = 2;
constexpr int kGroupKeys = 16;

template <int NT>
__device__ __forceinline__ void load_q_frag(const uint16_t* q_idx, const float* w_idx, int qi,
                                            int H_I, int g, int tig, uint32_t (&qa)[NT][8],
                                            float (&wv)[NT][2]) {
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int head = nt * 8 + g;
    if (head < H_I) {
      const uint16_t* qrow = q_idx + ((int64_t)qi * H_I + head) * CSA2_D_IDX;
      uint4 c0 = *reinterpret_cast<const uint4*>(qrow + 8 * tig);
      uint4 c1 = *reinterpret_cast<const uint4*>(qrow + 32 + 8 * tig);
      qa[nt][0] = c0.x; qa[nt][1] = c0.y; qa[nt][2] = c0.z; qa[nt][3] = c0.w;
      qa[nt][4] = c1.x; qa[nt][5] = c1.y; qa[nt][6] = c1.z; qa[nt][7] = c1.w;
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) qa[nt][k] = 0u;
    }
    const int h0 = nt * 8 + 2 * tig;
    wv[nt][0] = h0 < H_I ? w_idx[(int64_t)qi * H_I + h0] : 0.f;
    wv[nt][1] = h0 + 1 < H_I ? w_idx[(int64_t)qi * H_I + h0 + 1] : 0.f;
  }
}

__device__ __forceinline__ int clamp_nvis(const int32_t* n_visible, int qi, int64_t n_stride) {
  int v = n_visible[qi];
  return v < 0 ? 0 : (v > n_stride ? (int)n_stride : v);
}

// With a candidate pool (pool != nullptr: per query the ascending block ids [pool_stride]
// of the pool and, in pool_nv, its number of visible positions) a query's positions are
// the pool's, 8 per block: group j covers pool blocks 2j and 2j+1, i.e. key rows g of the
// MMA from the first block and rows g+8 from the second, and its scores land at pool
// positions 16j .. 16j+15.
template <int NT>
__global__ void __launch_bounds__(kScoreThreads, kScoreCtasPerSm) index_score_kernel(
    const uint16_t* __restrict__ q_idx, const float* __restrict__ w_idx,
    const uint16_t* __restrict__ z, int64_t n_stride, const int32_t* __restrict__ n_visible, int T,
    int H_I, int Q, float* __restrict__ scores, int64_t score_stride, uint32_t* __restrict__ range,
    const int32_t* __restrict__ pool, const int32_t* __restrict__ pool_nv, int pool_stride) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, tig = lane & 3;
  const bool pooled = pool != nullptr;
  const int64_t npos = pooled ? 8 * (int64_t)pool_stride : n_stride;   // positions per query
  const int gpq = (int)((npos + kGroupKeys - 1) / kGroupKeys);           // groups per query
  const int64_t total = (int64_t)Q * gpq;
  const int64_t nwarps = (int64_t)gridDim.x * (kScoreThreads / 32);
  const int64_t wid = (int64_t)blockIdx.x * (kScoreThreads / 32) + (threadIdx.x >> 5);
  const int64_t w_begin = total * wid / nwarps, w_end = total * (wid + 1) / nwarps;

  uint32_t qa[NT][8];
  float wv[NT][2];
  int cur_q = -1, nv = 0;
  uint32_t rmax = 0u, rmin_inv = 0u;  // score range of the current query seen by this warp
  for (int64_t g0 = w_begin; g0 < w_end;) {
    // fragments of up to kScoreUnroll groups (all loads issued before any use); a batch
    // ends at a query boundary, since the indexer rows in registers are one query's
    const int64_t q_end = (g0 / gpq + 1) * gpq;
    const int nb = (int)min((int64_t)kScoreUnroll, min(w_end, q_end) - g0);
    uint4 v[kScoreUnroll][4];
    int qg[kScoreUnroll], key0g[kScoreUnroll], okg[kScoreUnroll];
#pragma unroll
    for (int u = 0; u < kScoreUnroll; ++u) {
      const int64_t gi = g0 + u;
      const int qi = (int)(gi / gpq);
      const int key0 = (int)(gi - (int64_t)qi * gpq) * kGroupKeys;
      qg[u] = u < nb ? qi : -1;
      key0g[u] = key0;
      if (u == 0 && qi != cur_q) {
        // a new query: flush the range of the previous one, load its indexer rows
        if (cur_q >= 0 && lane == 0 && rmax != 0u) {
          atomicMax(range + 2 * cur_q, rmin_inv);
          atomicMax(range + 2 * cur_q + 1, rmax);
        }
        rmax = 0u;
        rmin_inv = 0u;
        load_q_frag<NT>(q_idx, w_idx, qi, H_I, g, tig, qa, wv);
        nv = pooled ? min(max(pool_nv[qi], 0), 8 * pool_stride) : clamp_nvis(n_visible, qi, n_stride);
        cur_q = qi;
      }
      const int b = qi / T;
      // positions key0 + g and key0 + 8 + g; their key rows (pool: the blocks' entries)
      bool oka = u < nb && key0 + g < nv, okb = u < nb && key0 + 8 + g < nv;
      int64_t ra = key0 + g, rb = ra + 8;
      if (pooled) {
        const int32_t* blk = pool + (int64_t)qi * pool_stride + (key0 >> 3);
        ra = oka ? (int64_t)blk[0] * 8 + g : 0;
        rb = okb ? (int64_t)blk[1] * 8 + g : 0;
        oka = oka && ra >= 0 && ra < n_stride;
        okb = okb && rb >= 0 && rb < n_stride;
      }
      okg[u] = (oka ? 1 : 0) | (okb ? 2 : 0);
      const uint16_t* zb = z + (int64_t)b * n_stride * CSA2_D_IDX;
      const uint4* pa = reinterpret_cast<const uint4*>(zb + (int64_t)ra * CSA2_D_IDX);
      const uint4* pb = reinterpret_cast<const uint4*>(zb + (int64_t)rb * CSA2_D_IDX);
      v[u][0] = oka ? pa[tig] : make_uint4(0, 0, 0, 0);
      v[u][1] = oka ? pa[4 + tig] : make_uint4(0, 0, 0, 0);
      v[u][2] = okb ? pb[tig] : make_uint4(0, 0, 0, 0);
      v[u][3] = okb ? pb[4 + tig] : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kScoreUnroll; ++u) {
      if (qg[u] < 0) continue;
      const int qi = qg[u], key0 = key0g[u];
      if (key0 >= nv) continue;   // past the visible keys (qi is the current query)
      const uint32_t ra_[16] = {v[u][0].x, v[u][0].y, v[u][0].z, v[u][0].w, v[u][1].x, v[u][1].y,
                                v[u][1].z, v[u][1].w, v[u][2].x, v[u][2].y, v[u][2].z, v[u][2].w,
                                v[u][3].x, v[u][3].y, v[u][3].z, v[u][3].w};
      float pg = 0.f, pg8 = 0.f;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < 4; ++j)
          mma_bf16(acc, ra_[2 * j], ra_[8 + 2 * j], ra_[2 * j + 1], ra_[8 + 2 * j + 1], qa[nt][2 * j],
                   qa[nt][2 * j + 1]);
        pg += wv[nt][0] * fmaxf(acc[0], 0.f) + wv[nt][1] * fmaxf(acc[1], 0.f);
        pg8 += wv[nt][0] * fmaxf(acc[2], 0.f) + wv[nt][1] * fmaxf(acc[3], 0.f);
      }
      pg += __shfl_xor_sync(0xffffffffu, pg, 1);
      pg += __shfl_xor_sync(0xffffffffu, pg, 2);
      pg8 += __shfl_xor_sync(0xffffffffu, pg8, 1);
      pg8 += __shfl_xor_sync(0xffffffffu, pg8, 2);
      float* srow = scores + (int64_t)qi * score_stride + key0;
      const bool ok0 = tig == 0 && (okg[u] & 1), ok1 = tig == 1 && (okg[u] & 2);
      if (ok0) srow[g] = pg;
      if (ok1) srow[g + 8] = pg8;
      const uint32_t kk = ok0 ? f2key(pg) : (ok1 ? f2key(pg8) : 0u);
      rmax = max(rmax, __reduce_max_sync(0xffffffffu, kk));
      rmin_inv = max(rmin_inv, __reduce_max_sync(0xffffffffu, (ok0 || ok1) ? ~kk : 0u));
    }
    g0 += nb;
  }
  if (cur_q >= 0 && lane == 0 && rmax != 0u) {
    atomicMax(range + 2 * cur_q, rmin_inv);
    atomicMax(range + 2 * cur_q + 1, rmax);
  }
}

cudaError_t launch_index_score(const void* q_idx, const float* w_idx, const void* z,
                               int64_t n_stride, const int32_t* n_visible, int B, int T, int H_I,
                               float* scores, int64_t score_stride, uint32_t* range,
                               uint32_t* status, cudaStream_t st, const int32_t* pool,
                               const int32_t* pool_nv, int pool_stride) {
  (void)status;
  const int Q = B * T;
  if (n_stride == 0 || Q == 0) return cudaSuccess;
  const int64_t npos = pool ? 8 * (int64_t)pool_stride : n_stride;
  const int64_t total = (int64_t)Q * ((npos + kGroupKeys - 1) / kGroupKeys);
  const int64_t warps = (int64_t)device_sm_count() * kScoreCtasPerSm * (kScoreThreads / 32);
  int64_t grid = (int64_t)device_sm_count() * kScoreCtasPerSm;
  if (total < warps) grid = (total + kScoreThreads / 32 - 1) / (kScoreThreads / 32);
  auto qp = static_cast<const uint16_t*>(q_idx);
  auto zp = static_cast<const uint16_t*>(z);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kScoreThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (H_I <= 8)
    return cudaLaunchKernelEx(&cfg, index_score_kernel<1>, qp, w_idx, zp, n_stride, n_visible, T, H_I, Q, scores,
                              score_stride, range, pool, pool_nv, pool_stride);
  return cudaLaunchKernelEx(&cfg, index_score_kernel<2>, qp, w_idx, zp, n_stride, n_visible, T, H_I, Q, scores,
                            score_stride, range, pool, pool_nv, pool_stride);
}

// ---------------------------------------------------------------------------
// Top-K selection: one cluster of C CTAs per query
// ---------------------------------------------------------------------------
// CTA r of the cluster owns the visible entries [r*slice, (r+1)*slice) (slice a
// multiple of 4) and lands their scores in shared memory with one bulk copy.
// Every exchange is a push: before a cluster barrier each CTA writes its record
// into slot r of every peer's receive buffer (distributed shared memory stores,
// no remote loads), so after the barrier all reads are local and no CTA touches
// a peer once it has passed the last barrier.
//
// Fast path (two barriers). The scoring kernel left the query's score range
// [lo, hi] in the workspace; each CTA bins its scores into kNB monotone bins of
// that range and pushes the 16-bit histogram. After the barrier every CTA knows
// all histograms, hence the bin b* holding the K-th score, how many entries each
// CTA has above it, and how many candidates (bin b*) each CTA holds. If they are
// at most kCandCap, each CTA pushes its candidates; after the second barrier
// every CTA ranks all candidates by (score desc, index asc), so it knows how
// many each CTA contributes, i.e. its own output offset, with no further
// exchange.
// General path (range missing, or too many candidates in b*): rounds of
//   round 0  min / max / count of the surviving candidates (+ the candidate
//            list itself when small enough) -> every CTA knows the range
//   round 1  histogram of the candidates over kNB monotone bins of that range
//            -> the bin b* holding the K-th score: higher bins are selected,
//            lower ones dropped; repeat from round 0 on the bin-b* survivors
//   exact    when at most kCandCap candidates survive, each CTA ranks its own
//            candidates against all of them by (score desc, index asc);
//            when they all tie, the lowest indices win
//   output   selected counts are pushed, each CTA writes its selected indices
//            at its prefix offset (ascending by construction).
// The bin map floor((s - lo) * kNB / (hi - lo)) (clamped) is monotone in s, so
// bins never reorder scores; equal scores always share a bin.
constexpr int kSelThreads = 1024;
constexpr int kNBMax = 2048;        // histogram bins per refinement round (small clusters)
constexpr int kNBMin = 1024;        // (clusters of more than 4 CTAs)
constexpr int kCandCap = 512;       // candidates resolved exactly by ranking
constexpr int kMaxLevels = 12;
constexpr int kMaxCluster = 16;
constexpr size_t kSelSmemMax = 200 * 1024;

struct SelRec {
  float lo, hi;
  int cnt, pad;
};

struct SelShared {
  SelRec rec_in[kMaxCluster];           // pushed candidate statistics
  int sel_in[kMaxCluster];              // pushed selected counts
  int above_r[kMaxCluster];             // entries above b* per CTA (fast path, pushed)
  int cand_sel[kMaxCluster];            // selected candidates per CTA (fast path)
  uint32_t hist_local[kNBMax];
  int scan[kSelThreads / 32];
  float red_f[2][kSelThreads / 32];
  int red_i[kSelThreads / 32];
  int bstar, above, cand_n, my_above;
  uint64_t bar_load;
  float cand_s[kCandCap];               // own candidates (compacted)
  int cand_i[kCandCap];
};
// Regions after the header start at a 128-byte boundary (the histogram pushes
// are 16-byte vector stores).
constexpr size_t kSelHdr = (sizeof(SelShared) + 127) & ~size_t(127);
// followed in dynamic shared memory by: uint16_t hist_in[C][NB] (pushed histograms),
// float cand_in_s[C][kCandCap], int cand_in_i[C][kCandCap], float sc[slice_cap],
// uint8_t state[slice_cap]

__device__ __forceinline__ int bin_of(float s, float lo, float scl, int nb) {
  float t = (s - lo) * scl;
  int bi = (int)t;
  return bi < 0 ? 0 : (bi > nb - 1 ? nb - 1 : bi);
}

// Block-wide exclusive scan of one int per thread; returns the prefix, writes the total.
__device__ __forceinline__ int block_excl_scan(int v, int* scan, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scan[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int s = lane < kSelThreads / 32 ? scan[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < kSelThreads / 32) scan[lane] = s;
  }
  __syncthreads();
  total = scan[kSelThreads / 32 - 1];
  int pre = (warp > 0 ? scan[warp - 1] : 0) + x - v;
  __syncthreads();
  return pre;
}

// ---------------------------------------------------------------------------
// Candidate pool of the Hierarchical Sparse Indexer ("DeepSeek-V4.1-Flash", picx.dev
// summary, Methodology / 3): the aligned 8-position blocks that hold an entry of the
// first FULL layer's selection bound the search of the REINDEX layers after it.
// ---------------------------------------------------------------------------
// One CTA per query over its (ascending, -1 padded) selection sel [K]: a new block
// starts wherever an entry's block differs from the previous entry's; the block ids are
// compacted in order into blocks [K] and pool_nv gets the number of pool positions below
// n_visible. A selection that is not ascending or holds an index outside [-1, n_stride)
// sets CSA2_DEV_BAD_INDEX.
constexpr int kPoolPerThread = (kMaxK + kSelThreads - 1) / kSelThreads;

__global__ void __launch_bounds__(kSelThreads) pool_build_kernel(
    const int32_t* __restrict__ sel, int K, const int32_t* __restrict__ n_visible, int64_t n_stride,
    int32_t* __restrict__ blocks, int32_t* __restrict__ pool_nv, uint32_t* __restrict__ status) {
  __shared__ int scan[kSelThreads / 32];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int qi = blockIdx.x, tid = threadIdx.x;
  const int32_t* s = sel + (int64_t)qi * K;
  const int per = (K + kSelThreads - 1) / kSelThreads;
  const int i0 = tid * per;
  const int nvis = clamp_nvis(n_visible, qi, n_stride);
  int prev = (i0 > 0 && i0 - 1 < K) ? s[i0 - 1] : -1;
  if (prev < -1 || prev >= n_stride) prev = -1;
  int mine[kPoolPerThread];
  int cnt = 0, vis = 0;
  bool bad = false;
#pragma unroll
  for (int k = 0; k < kPoolPerThread; ++k) {
    if (k >= per) break;
    const int i = i0 + k;
    int v = i < K ? s[i] : -1;
    if (v < -1 || v >= n_stride) { bad = true; v = -1; }
    if (v >= 0) {
      if (prev >= 0 && v < prev) bad = true;
      if (prev < 0 || (v >> 3) != (prev >> 3)) {
        mine[cnt++] = v >> 3;
        vis += min(max(nvis - 8 * (v >> 3), 0), 8);
      }
      prev = v;
    }
  }
  int total;
  const int off = block_excl_scan(cnt, scan, total);
#pragma unroll
  for (int k = 0; k < kPoolPerThread; ++k)
    if (k < cnt) blocks[(int64_t)qi * K + off + k] = mine[k];
  int vis_total;
  block_excl_scan(vis, scan, vis_total);
  if (tid == 0) pool_nv[qi] = vis_total;
  if (bad) atomicOr(status, CSA2_DEV_BAD_INDEX);
}

cudaError_t launch_pool_build(const int32_t* sel, int Q, int K, const int32_t* n_visible, int64_t n_stride,
                              int32_t* blocks, int32_t* pool_nv, uint32_t* status, cudaStream_t st) {
  if (Q == 0) return cudaSuccess;
  if (K > kMaxK) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)Q);
  cfg.blockDim = dim3(kSelThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, pool_build_kernel, sel, K, n_visible, n_stride, blocks, pool_nv, status);
}


__device__ __forceinline__ void st_remote_u32(uint32_t* local_addr, int rank, uint32_t v) {
  uint32_t la = smem_u32(local_addr), ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(la), "r"(rank));
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(ra), "r"(v) : "memory");
}
__device__ __forceinline__ void st_remote_v4(void* local_addr, int rank, uint4 v) {
  uint32_t la = smem_u32(local_addr), ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(la), "r"(rank));
  asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(ra), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void cluster_barrier() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// Histogram of this CTA's surviving candidates over [lo, hi] into sh.hist_local,
// pushed as 16-bit counts into slot r of every peer's hist_in.
__device__ __forceinline__ void build_push_hist(SelShared& sh, uint16_t* hist_in, const float* sc,
                                                const uint8_t* state, int my_len, float lo, float scl,
                                                int NB, uint32_t C, uint32_t r) {
  const int tid = threadIdx.x;
  for (int i = tid; i < NB; i += kSelThreads) sh.hist_local[i] = 0u;
  __syncthreads();
  // loads first, 8 per thread in flight, then the atomics
  for (int e0 = tid; e0 < my_len; e0 += 8 * kSelThreads) {
    float v[8];
    uint8_t s[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int e = e0 + k * kSelThreads;
      v[k] = e < my_len ? sc[e] : 0.f;
      s[k] = e < my_len ? state[e] : 1;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k)
      if (s[k] == 0) atomicAdd(&sh.hist_local[bin_of(v[k], lo, scl, NB)], 1u);
  }
  __syncthreads();
  for (int j = tid; j < (int)C * (NB / 8); j += kSelThreads) {
    const int peer = j / (NB / 8), o8 = j % (NB / 8);
    const uint32_t* h = &sh.hist_local[8 * o8];
    const uint4 v = make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16),
                               h[6] | (h[7] << 16));
    st_remote_v4(&hist_in[r * NB + 8 * o8], peer, v);
  }
}

// Suffix counts of the summed histograms: the bin b* with above < remaining <=
// above + count(b*) goes to sh.bstar / sh.above (thread t owns bins from the top).
__device__ __forceinline__ void find_bstar(SelShared& sh, const uint16_t* hist_in, int NB, uint32_t C,
                                           int remaining) {
  const int tid = threadIdx.x;
  const int per = NB / kSelThreads;
  const int btop = NB - 1 - per * tid;
  uint32_t hs[kNBMax / kSelThreads];
  int mine = 0;
#pragma unroll
  for (int k = 0; k < kNBMax / kSelThreads; ++k) {
    uint32_t h = 0;
    if (k < per)
      for (int rr = 0; rr < (int)C; ++rr) h += hist_in[rr * NB + btop - k];
    hs[k] = h;
    mine += (int)h;
  }
  int total;
  int above = block_excl_scan(mine, sh.scan, total);
#pragma unroll
  for (int k = 0; k < kNBMax / kSelThreads; ++k) {
    if (k < per) {
      const int h = (int)hs[k];
      if (above < remaining && remaining <= above + h) {
        sh.bstar = btop - k;
        sh.above = above;
      }
      above += h;
    }
  }
  __syncthreads();
}

// One round of the general path: min / max / count of this CTA's surviving
// candidates (and the candidates themselves when few) pushed to every peer,
// then a cluster barrier. Returns the cluster-wide range and count, and the
// number of survivors in lower-ranked CTAs.
__device__ __noinline__ void stats_round(SelShared& sh, float* cand_in_s, int* cand_in_i, const float* sc,
                                         const uint8_t* state, int my0, int my_len, uint32_t C, uint32_t r,
                                         float& glo, float& ghi, int& gcnt, int& pre_cnt, int& mine_cnt) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float lo = INFINITY, hi = -INFINITY;
  int cnt = 0;
  for (int e = tid; e < my_len; e += kSelThreads)
    if (state[e] == 0) {
      const float v = sc[e];
      lo = fminf(lo, v);
      hi = fmaxf(hi, v);
      ++cnt;
    }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
  }
  if (lane == 0) {
    sh.red_f[0][warp] = lo;
    sh.red_f[1][warp] = hi;
    sh.red_i[warp] = cnt;
  }
  if (tid == 0) sh.cand_n = 0;
  __syncthreads();
  lo = INFINITY; hi = -INFINITY; cnt = 0;
#pragma unroll 1
  for (int w = 0; w < kSelThreads / 32; ++w) {
    lo = fminf(lo, sh.red_f[0][w]);
    hi = fmaxf(hi, sh.red_f[1][w]);
    cnt += sh.red_i[w];
  }
  mine_cnt = cnt;
  if (cnt <= kCandCap) {
    for (int e = tid; e < my_len; e += kSelThreads)
      if (state[e] == 0) {
        const int p = atomicAdd(&sh.cand_n, 1);
        sh.cand_s[p] = sc[e];
        sh.cand_i[p] = my0 + e;
      }
  }
  __syncthreads();
  if (tid < (int)C)
    st_remote_v4(&sh.rec_in[r], tid, make_uint4(__float_as_uint(lo), __float_as_uint(hi), (uint32_t)cnt, 0u));
  if (cnt <= kCandCap) {
    for (int j = tid; j < (int)C * cnt; j += kSelThreads) {
      const int peer = j / cnt, k = j % cnt;
      st_remote_u32(reinterpret_cast<uint32_t*>(&cand_in_s[r * kCandCap + k]), peer, __float_as_uint(sh.cand_s[k]));
      st_remote_u32(reinterpret_cast<uint32_t*>(&cand_in_i[r * kCandCap + k]), peer, (uint32_t)sh.cand_i[k]);
    }
  }
  cluster_barrier();
  glo = INFINITY; ghi = -INFINITY; gcnt = 0; pre_cnt = 0;
#pragma unroll 1
  for (int rr = 0; rr < (int)C; ++rr) {
    const SelRec v = sh.rec_in[rr];
    if (v.cnt > 0) {
      glo = fminf(glo, v.lo);
      ghi = fmaxf(ghi, v.hi);
    }
    if (rr < (int)r) pre_cnt += v.cnt;
    gcnt += v.cnt;
  }
}

__global__ void __launch_bounds__(kSelThreads) topk_select_kernel(
    const float* __restrict__ scores, int64_t score_stride, const int32_t* __restrict__ n_visible,
    int64_t n_stride, int K, int slice_cap, uint32_t* __restrict__ range, int32_t* __restrict__ out_idx,
    float* __restrict__ out_scores, uint32_t* __restrict__ status, const uint8_t* __restrict__ pf_codes,
    const uint8_t* __restrict__ pf_scales, int T, int64_t kv_stride, const int32_t* __restrict__ pool,
    int pool_stride) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  SelShared& sh = *reinterpret_cast<SelShared*>(smem_raw);
  uint32_t C, r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(C));
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  const int NB = C <= 4 ? kNBMax : kNBMin;
  uint16_t* hist_in = reinterpret_cast<uint16_t*>(smem_raw + kSelHdr);
  float* cand_in_s = reinterpret_cast<float*>(hist_in + C * NB);
  int* cand_in_i = reinterpret_cast<int*>(cand_in_s + C * kCandCap);
  float* sc = reinterpret_cast<float*>(cand_in_i + C * kCandCap);
  uint8_t* state = reinterpret_cast<uint8_t*>(sc + slice_cap);

  const int tid = threadIdx.x, lane = tid & 31;
  const int qi = blockIdx.y;
  if (tid == 0) {
    mbar_init(smem_u32(&sh.bar_load), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  asm volatile("griddepcontrol.wait;" ::: "memory");
  int nvis = n_visible[qi];
  nvis = nvis < 0 ? 0 : (nvis > n_stride ? (int)n_stride : nvis);
  const int slice = (((nvis + (int)C - 1) / (int)C) + 3) & ~3;
  const int my0 = (int)r * slice;
  int my_len = nvis - my0;
  my_len = my_len < 0 ? 0 : (my_len > slice ? slice : my_len);
  const int need = nvis < K ? nvis : K;
  int32_t* out = out_idx + (int64_t)qi * K;
  float* outs = out_scores ? out_scores + (int64_t)qi * K : nullptr;

  // this CTA's scores: one bulk copy (16-byte aligned start, length rounded up to 16 bytes)
  bool loaded = true;
  if (my_len > 0) {
    const uint32_t bytes = (uint32_t)(((my_len + 3) & ~3) * 4);
    if (tid == 0) {
      mbar_arrive_expect_tx(smem_u32(&sh.bar_load), bytes);
      bulk_g2s(smem_u32(sc), scores + (int64_t)qi * score_stride + my0, bytes, smem_u32(&sh.bar_load));
    }
    loaded = mbar_wait(smem_u32(&sh.bar_load), 0);
  }
  // the score range left by the scoring kernel (read by every CTA before the first barrier)
  const uint32_t kminv = range[2 * qi], kmax = range[2 * qi + 1];
  const float rlo = key2f(~kminv), rhi = key2f(kmax);
  const bool have_range = kmax != 0u && rlo < rhi && isfinite(rlo) && isfinite(rhi);
  if (!__syncthreads_and(loaded)) {
    if (tid == 0) atomicOr(status, CSA2_DEV_PIPELINE_TIMEOUT);
    my_len = 0;  // score nothing; the selection below still completes
  }
  const uint8_t init = nvis <= K ? 1 : 0;
  for (int e = tid; e < my_len; e += kSelThreads) state[e] = init;
  if (tid < kMaxCluster) {
    sh.above_r[tid] = 0;
    sh.cand_sel[tid] = 0;
  }
  if (tid == 0) sh.my_above = 0;
  __syncthreads();

  bool settled = false;     // output offsets known without the final exchange
  int off_fast = 0, total_fast = 0;
  if (nvis <= K) {
    // everything visible is selected: CTA r's offset is the visible entries before its slice
    settled = true;
    off_fast = my0 < nvis ? my0 : nvis;
    total_fast = nvis;
    if (r == 0 && tid == 0) {
      range[2 * qi] = 0u;
      range[2 * qi + 1] = 0u;
    }
  } else {
    int rem = need;
    int level = 0;
    bool done = false;
    if (have_range) {
      // ---- fast path: histogram of the known range, then the b* candidates
      const float scl = (float)NB / (rhi - rlo);
      build_push_hist(sh, hist_in, sc, state, my_len, rlo, scl, NB, C, r);
      cluster_barrier();
      if (r == 0 && tid == 0) {
        range[2 * qi] = 0u;
        range[2 * qi + 1] = 0u;
      }
      find_bstar(sh, hist_in, NB, C, rem);
      const int bstar = sh.bstar;
      rem -= sh.above;
      level = 1;
      int cand_tot = 0;
#pragma unroll 1
      for (int rr = 0; rr < (int)C; ++rr) cand_tot += hist_in[rr * NB + bstar];
      if (tid == 0) sh.cand_n = 0;
      __syncthreads();
      // classify (all entries are candidates at this point), count the ones above b*
      // and collect the b* ones
      int n_above = 0;
      for (int e0 = tid; e0 < my_len; e0 += 8 * kSelThreads) {
        float v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int e = e0 + k * kSelThreads;
          v[k] = e < my_len ? sc[e] : 0.f;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int e = e0 + k * kSelThreads;
          if (e < my_len) {
            const int bi = bin_of(v[k], rlo, scl, NB);
            state[e] = bi > bstar ? 1 : (bi < bstar ? 2 : 0);
            n_above += bi > bstar;
            if (bi == bstar && cand_tot <= kCandCap) {
              const int p = atomicAdd(&sh.cand_n, 1);
              sh.cand_s[p] = v[k];
              sh.cand_i[p] = my0 + e;
            }
          }
        }
      }
      n_above = __reduce_add_sync(0xffffffffu, n_above);
      if (lane == 0 && n_above) atomicAdd(&sh.my_above, n_above);
      __syncthreads();
      if (cand_tot <= kCandCap) {
        // push own candidates (their number, hist_in[r][b*], is known to every peer)
        // and own count above b*
        if (tid < (int)C) st_remote_u32(reinterpret_cast<uint32_t*>(&sh.above_r[r]), tid, (uint32_t)sh.my_above);
        const int mine = sh.cand_n;
        for (int j = tid; j < (int)C * mine; j += kSelThreads) {
          const int peer = j / mine, k = j % mine;
          st_remote_u32(reinterpret_cast<uint32_t*>(&cand_in_s[r * kCandCap + k]), peer,
                        __float_as_uint(sh.cand_s[k]));
          st_remote_u32(reinterpret_cast<uint32_t*>(&cand_in_i[r * kCandCap + k]), peer, (uint32_t)sh.cand_i[k]);
        }
        cluster_barrier();
        // rank every candidate of every CTA (one warp per candidate, the lanes split
        // the comparisons): own ones set the state, all of them the per-CTA counts
        {
          int cnt_r[kMaxCluster];
          int tot = 0;
#pragma unroll 1
          for (int rr = 0; rr < (int)C; ++rr) {
            cnt_r[rr] = hist_in[rr * NB + bstar];
            tot += cnt_r[rr];
          }
          const int warp = tid >> 5;
          for (int j = warp; j < tot; j += kSelThreads / 32) {
            int rr = 0, k = j;
            while (k >= cnt_r[rr]) { k -= cnt_r[rr]; ++rr; }
            const float s = cand_in_s[rr * kCandCap + k];
            const int i = cand_in_i[rr * kCandCap + k];
            int rank = 0;
            for (int c = lane; c < tot; c += 32) {
              int r2 = 0, k2 = c;
              while (k2 >= cnt_r[r2]) { k2 -= cnt_r[r2]; ++r2; }
              const float t = cand_in_s[r2 * kCandCap + k2];
              const int ti = cand_in_i[r2 * kCandCap + k2];
              rank += (t > s) || (t == s && ti < i);
            }
            rank = __reduce_add_sync(0xffffffffu, rank);
            if (lane == 0) {
              const bool take = rank < rem;
              if (take) atomicAdd(&sh.cand_sel[rr], 1);
              if (rr == (int)r) state[i - my0] = take ? 1 : 2;
            }
          }
        }
        __syncthreads();
#pragma unroll 1
        for (int rr = 0; rr < (int)C; ++rr) {
          const int v = sh.above_r[rr] + sh.cand_sel[rr];
          if (rr < (int)r) off_fast += v;
          total_fast += v;
        }
        settled = true;
        done = true;
      }
    }
    // ---- general path (no usable range, or too many candidates in b*)
    while (!done) {
      float glo, ghi;
      int gcnt, pre_cnt, mine_cnt;
      stats_round(sh, cand_in_s, cand_in_i, sc, state, my0, my_len, C, r, glo, ghi, gcnt, pre_cnt, mine_cnt);
      if (level == 0 && r == 0 && tid == 0) {
        range[2 * qi] = 0u;
        range[2 * qi + 1] = 0u;
      }
      if (rem >= gcnt) {
        for (int e = tid; e < my_len; e += kSelThreads)
          if (state[e] == 0) state[e] = 1;
        break;
      }
      if (gcnt <= kCandCap) {
        for (int j = tid; j < mine_cnt; j += kSelThreads) {
          const float s = sh.cand_s[j];
          const int i = sh.cand_i[j];
          int rank = 0;
#pragma unroll 1
          for (int rr = 0; rr < (int)C; ++rr) {
            const int n = sh.rec_in[rr].cnt;
            const float* cs = cand_in_s + rr * kCandCap;
            const int* ci = cand_in_i + rr * kCandCap;
            for (int c = 0; c < n; ++c) {
              const float t = cs[c];
              rank += (t > s) || (t == s && ci[c] < i);
            }
          }
          state[i - my0] = rank < rem ? 1 : 2;
        }
        break;
      }
      if (glo == ghi || level == kMaxLevels - 1) {
        // all candidates tie (or refinement did not settle): lowest indices first
        if (glo != ghi && tid == 0) atomicOr(status, CSA2_DEV_TOPK_LEVELS);
        const int chunk = (my_len + kSelThreads - 1) / kSelThreads;
        const int e0 = tid * chunk, e1 = min(e0 + chunk, my_len);
        int c = 0;
        for (int e = e0; e < e1; ++e) c += state[e] == 0;
        int total;
        int ord = block_excl_scan(c, sh.scan, total) + pre_cnt;
        for (int e = e0; e < e1; ++e)
          if (state[e] == 0) {
            state[e] = ord < rem ? 1 : 2;
            ++ord;
          }
        break;
      }
      const float scl2 = (float)NB / (ghi - glo);
      build_push_hist(sh, hist_in, sc, state, my_len, glo, scl2, NB, C, r);
      cluster_barrier();
      find_bstar(sh, hist_in, NB, C, rem);
      const int bs = sh.bstar;
      rem -= sh.above;
      for (int e = tid; e < my_len; e += kSelThreads)
        if (state[e] == 0) {
          const int bi = bin_of(sc[e], glo, scl2, NB);
          state[e] = bi > bs ? 1 : (bi < bs ? 2 : 0);
        }
      __syncthreads();
      ++level;
    }
    __syncthreads();
  }

  // ---- ordered output: warp w owns a contiguous run of entries, compacted 32 at a time
  // with ballots (a count pass, one scan of the 32 warp counts, a write pass)
  const int warp = tid >> 5;
  constexpr int kWarps = kSelThreads / 32;
  const int per_warp = ((my_len + kWarps - 1) / kWarps + 31) & ~31;
  const int wb = warp * per_warp, we = min(wb + per_warp, my_len);
  int wc = 0;
  for (int e0 = wb; e0 < we; e0 += 32) {
    const int e = e0 + lane;
    wc += __popc(__ballot_sync(0xffffffffu, e < we && state[e] == 1));
  }
  __syncthreads();   // sh.scan is free (any earlier use is complete)
  if (lane == 0) sh.scan[warp] = wc;
  __syncthreads();
  const int wcnt = sh.scan[lane];
  int incl = wcnt;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += t;
  }
  const int my_sel = __shfl_sync(0xffffffffu, incl, 31);
  int pos = __shfl_sync(0xffffffffu, incl - wcnt, warp);
  int offset = off_fast, total_sel = total_fast;
  if (!settled) {
    if (tid < (int)C) st_remote_u32(reinterpret_cast<uint32_t*>(&sh.sel_in[r]), tid, (uint32_t)my_sel);
    cluster_barrier();
    offset = 0;
    total_sel = 0;
#pragma unroll 1
    for (int rr = 0; rr < (int)C; ++rr) {
      const int v = sh.sel_in[rr];
      if (rr < (int)r) offset += v;
      total_sel += v;
    }
  }
  pos += offset;
  // the FP4 rows of the selected entries are requested into L2 for the attention that
  // gathers them next
  const uint8_t* pfc = pf_codes ? pf_codes + (int64_t)(qi / T) * kv_stride * CSA2_CODE_BYTES : nullptr;
  const uint8_t* pfs = pf_codes ? pf_scales + (int64_t)(qi / T) * kv_stride * CSA2_SCALE_BYTES : nullptr;
  // with a candidate pool the positions are the pool's: position j is entry
  // block[j / 8] * 8 + j % 8
  const int32_t* pblk = pool ? pool + (int64_t)qi * pool_stride : nullptr;
  for (int e0 = wb; e0 < we; e0 += 32) {
    const int e = e0 + lane;
    const bool take = e < we && state[e] == 1;
    const uint32_t bal = __ballot_sync(0xffffffffu, take);
    const int p = pos + __popc(bal & ((1u << lane) - 1u));
    if (take && p < K) {
      const int ent = pblk ? pblk[(my0 + e) >> 3] * 8 + ((my0 + e) & 7) : my0 + e;
      out[p] = ent;
      if (outs) outs[p] = sc[e];
      if (pfc && ent >= 0 && ent < kv_stride) {
        prefetch_l2_bulk(pfc + (int64_t)ent * CSA2_CODE_BYTES, CSA2_CODE_BYTES);
        prefetch_l2(pfs + (int64_t)ent * CSA2_SCALE_BYTES);
        prefetch_l2(pfs + (int64_t)ent * CSA2_SCALE_BYTES + CSA2_SCALE_BYTES - 1);
      }
    }
    pos += __popc(bal);
  }
  if (r == C - 1)
    for (int p = total_sel + tid; p < K; p += kSelThreads) {
      out[p] = -1;
      if (outs) outs[p] = __int_as_float(0x7fc00000);
    }
}

// ---------------------------------------------------------------------------
// Top-K selection, one CTA per query (up to kRowMaxN visible positions)
// ---------------------------------------------------------------------------
// The query's scores land in shared memory (a few bulk copies). Selection state is two
// bitmaps over the positions, one bit per position (word w holds positions 32w ..
// 32w+31): selected, and still in play.
//   round 0  thread t visits positions k * kRowThreads + t (conflict-free reads): a
//            histogram of all scores over kRowBins monotone bins of [lo, hi] (the range
//            the scoring kernel left, else the scores' min / max); one block scan from
//            the top gives the bin b* holding the K-th score; a second pass marks the
//            higher bins selected and b*'s scores in play (one ballot per 32 positions
//            gives a bitmap word);
//   round i  the scores in play (few) are binned again over their own min / max;
//   exact    when at most kRowRankCap scores remain in play, they are listed in shared
//            memory and each is ranked against all of them by (score desc, position
//            asc);
//   ties     when they all tie (min == max), the lowest positions win.
// The bin map ((s - lo) * (NB-1) / (hi - lo), rounded to an integer by adding 2^23) is
// monotone in s, so bins never reorder scores and equal scores share a bin. Thread t then
// owns bitmap word t: one block scan of the per-word counts orders both the tie rule and
// the output (ascending by position).
constexpr int kRowThreads = 1024;
constexpr int kRowBins = 2048;
constexpr int kRowRankCap = 128;
constexpr int kRowMaxN = 32 * kRowThreads;
constexpr int kRowCopies = 8;    // bulk copies that land the scores

struct RowShared {
  uint32_t hist[kRowBins];
  uint32_t selw[kRowThreads];    // selected bitmap
  uint32_t candw[kRowThreads];   // in-play bitmap
  int scan[kRowThreads / 32];
  float red[2][kRowThreads / 32];
  int bstar, above, cand_n;
  uint32_t rng[2];
  uint64_t bar_load;
  float cand_s[kRowRankCap];
  int cand_i[kRowRankCap];
};

// Bin of s in [0, kRowBins) for s in [lo, hi], scl = (NB-1) / (hi - lo): (s - lo) * scl
// is at most NB-1 up to rounding, and adding 2^23 rounds it to an integer held in the
// low mantissa bits. Each step is monotone in s.
__device__ __forceinline__ uint32_t row_bin(float s, float lo, float scl) {
  return __float_as_uint(fmaf(s - lo, scl, 8388608.f)) & (uint32_t)(kRowBins - 1);
}

// Block-wide min of a and max of b (all threads get them).
__device__ __forceinline__ void row_minmax(float& a, float& b, RowShared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a = fminf(a, __shfl_xor_sync(0xffffffffu, a, o));
    b = fmaxf(b, __shfl_xor_sync(0xffffffffu, b, o));
  }
  __syncthreads();   // sh.red may still be read by a previous call
  if (lane == 0) {
    sh.red[0][warp] = a;
    sh.red[1][warp] = b;
  }
  __syncthreads();
  a = sh.red[0][lane];
  b = sh.red[1][lane];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a = fminf(a, __shfl_xor_sync(0xffffffffu, a, o));
    b = fmaxf(b, __shfl_xor_sync(0xffffffffu, b, o));
  }
}

// b* of a histogram in sh.hist for the rem-th largest: sets sh.bstar / sh.above.
__device__ __forceinline__ void row_find_bstar(RowShared& sh, int rem) {
  const int tid = threadIdx.x;
  const int b1 = kRowBins - 1 - 2 * tid, b0 = b1 - 1;
  const int h1 = (int)sh.hist[b1], h0 = (int)sh.hist[b0];
  int total;
  const int above = block_excl_scan(h1 + h0, sh.scan, total);
  if (above < rem && rem <= above + h1) {
    sh.bstar = b1;
    sh.above = above;
  } else if (above + h1 < rem && rem <= above + h1 + h0) {
    sh.bstar = b0;
    sh.above = above + h1;
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kRowThreads, 1) topk_row_kernel(
    const float* __restrict__ scores, int64_t score_stride, const int32_t* __restrict__ n_visible,
    int64_t n_stride, int K, uint32_t* __restrict__ range, int32_t* __restrict__ out_idx,
    float* __restrict__ out_scores, uint32_t* __restrict__ status, const uint8_t* __restrict__ pf_codes,
    const uint8_t* __restrict__ pf_scales, int T, int64_t kv_stride, const int32_t* __restrict__ pool,
    int pool_stride) {
  extern __shared__ __align__(128) float sv[];   // the query's scores, position order
  __shared__ RowShared sh;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int qi = blockIdx.x;
  if (tid == 0) {
    mbar_init(smem_u32(&sh.bar_load), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  sh.selw[tid] = 0u;
  sh.candw[tid] = 0u;
  __syncthreads();
  asm volatile("griddepcontrol.wait;" ::: "memory");
  int nvis = clamp_nvis(n_visible, qi, n_stride);
  // 16-byte pieces of the row (a score row is score_stride >= roundup4(nvis) floats)
  const int n16 = (nvis + 3) >> 2;
  if (tid == 0) {
    if (nvis > 0) mbar_arrive_expect_tx(smem_u32(&sh.bar_load), (uint32_t)n16 * 16);
    // the score range the scoring kernel left (consumed: set back to zero)
    sh.rng[0] = range[2 * qi];
    sh.rng[1] = range[2 * qi + 1];
    range[2 * qi] = 0u;
    range[2 * qi + 1] = 0u;
  }
  __syncthreads();   // expect_tx precedes every copy's completion
  if (tid < kRowCopies && nvis > 0) {
    const int per = (n16 + kRowCopies - 1) / kRowCopies;
    const int a = tid * per, b = min(a + per, n16);
    if (b > a)
      bulk_g2s(smem_u32(sv + 4 * a), scores + (int64_t)qi * score_stride + 4 * a, (uint32_t)(b - a) * 16,
               smem_u32(&sh.bar_load));
  }
  // one warp waits for the copies, the others at the barrier
  const bool loaded = nvis == 0 || tid >= 32 || mbar_wait(smem_u32(&sh.bar_load), 0);
  if (!__syncthreads_and(loaded)) {
    if (tid == 0) atomicOr(status, CSA2_DEV_PIPELINE_TIMEOUT);
    nvis = 0;   // select nothing; the output below still completes
  }
  const int nk = (nvis + kRowThreads - 1) / kRowThreads;
  if (nvis <= K) {
    // everything visible is selected: bitmap words of the first nvis positions
    const int p0 = 32 * tid;
    const int nmine = min(max(nvis - p0, 0), 32);
    sh.selw[tid] = nmine >= 32 ? 0xffffffffu : ((1u << nmine) - 1u);
  } else {
    int rem = K;
    float lo = key2f(~sh.rng[0]), hi = key2f(sh.rng[1]);
    if (!(sh.rng[1] != 0u && lo < hi && isfinite(lo) && isfinite(hi))) {
      float a = INFINITY, b = -INFINITY;
      for (int k = 0; k < nk; ++k) {
        const int p = k * kRowThreads + tid;
        if (p < nvis) {
          a = fminf(a, sv[p]);
          b = fmaxf(b, sv[p]);
        }
      }
      row_minmax(a, b, sh);
      lo = a;
      hi = b;
    }
    bool done = false;
    int nplay = nvis;   // positions in play
    const float scl0 = (float)(kRowBins - 1) / (hi - lo);
    const bool round0 = lo < hi && scl0 <= 1e30f;
    if (round0) {
      // ---- round 0 over every visible position
      for (int i = tid; i < kRowBins; i += kRowThreads) sh.hist[i] = 0u;
      __syncthreads();
#pragma unroll 8
      for (int k = 0; k < nk; ++k) {
        const int p = k * kRowThreads + tid;
        if (p < nvis) atomicAdd(&sh.hist[row_bin(sv[p], lo, scl0)], 1u);
      }
      __syncthreads();
      row_find_bstar(sh, rem);
      const uint32_t bstar = (uint32_t)sh.bstar;
      nplay = (int)sh.hist[bstar];
      rem -= sh.above;
      // lane k of each warp collects bitmap word k * 32 + warp (positions k * 1024 + 32 warp ..)
      uint32_t my_sel = 0u, my_cand = 0u;
#pragma unroll 8
      for (int k = 0; k < nk; ++k) {
        const int p = k * kRowThreads + tid;
        const bool ok = p < nvis;
        const uint32_t bi = ok ? row_bin(sv[p], lo, scl0) : 0u;
        const uint32_t bs = __ballot_sync(0xffffffffu, ok && bi > bstar);
        const uint32_t bc = __ballot_sync(0xffffffffu, ok && bi == bstar);
        if (lane == k) {
          my_sel = bs;
          my_cand = bc;
        }
      }
      if (lane < nk) {
        sh.selw[lane * 32 + warp] = my_sel;
        sh.candw[lane * 32 + warp] = my_cand;
      }
      __syncthreads();
      if (nplay == rem) {   // every score of b* is taken
        sh.selw[tid] |= sh.candw[tid];
        done = true;
      }
    }
    // ---- later rounds over the positions still in play (thread t: bitmap word t), binned
    // by their order-preserving integer keys relative to the smallest: each round
    // divides the key span by 2^11, so single keys are reached in at most three rounds
    uint32_t cw = sh.candw[tid];
    if (!round0) {
      const int nmine = min(max(nvis - 32 * tid, 0), 32);
      cw = nmine >= 32 ? 0xffffffffu : ((1u << nmine) - 1u);
    }
#pragma unroll 1
    for (int level = 1; !done; ++level) {
      // invariant: rem >= 1, nplay > rem positions in play, every higher score selected
      if (nplay <= kRowRankCap) {
        // exact: list the scores in play, rank each by (score desc, position asc)
        if (tid == 0) sh.cand_n = 0;
        __syncthreads();
        for (uint32_t m = cw; m; m &= m - 1u) {
          const int p = 32 * tid + __ffs(m) - 1;
          const int slot = atomicAdd(&sh.cand_n, 1);
          sh.cand_s[slot] = sv[p];
          sh.cand_i[slot] = p;
        }
        __syncthreads();
        if (tid < nplay) {
          const float sc = sh.cand_s[tid];
          const int i = sh.cand_i[tid];
          int rank = 0;
          for (int j = 0; j < nplay; ++j) {
            const float t = sh.cand_s[j];
            rank += (t > sc) || (t == sc && sh.cand_i[j] < i);
          }
          if (rank < rem) atomicOr(&sh.selw[i >> 5], 1u << (i & 31));
        }
        break;
      }
      // key range of the scores in play
      uint32_t ka = 0xffffffffu, kb = 0u;
      for (uint32_t m = cw; m; m &= m - 1u) {
        const uint32_t x = f2key(sv[32 * tid + __ffs(m) - 1]);
        ka = min(ka, x);
        kb = max(kb, x);
      }
      {
        ka = __reduce_min_sync(0xffffffffu, ka);
        kb = __reduce_max_sync(0xffffffffu, kb);
        __syncthreads();   // sh.red may still be read by a previous use
        if (lane == 0) {
          sh.red[0][warp] = __uint_as_float(ka);
          sh.red[1][warp] = __uint_as_float(kb);
        }
        __syncthreads();
        ka = __reduce_min_sync(0xffffffffu, __float_as_uint(sh.red[0][lane]));
        kb = __reduce_max_sync(0xffffffffu, __float_as_uint(sh.red[1][lane]));
      }
      const uint32_t span = kb - ka;
      if (span == 0u || level >= kMaxLevels) {
        // all tie (or the search did not settle): lowest positions first
        if (span != 0u && tid == 0) atomicOr(status, CSA2_DEV_TOPK_LEVELS);
        const int c = __popc(cw);
        int total;
        const int pre = block_excl_scan(c, sh.scan, total);
        int take = min(max(rem - pre, 0), c);
        uint32_t t = 0u;
        for (uint32_t m = cw; take > 0; --take) {
          t |= m & (~m + 1u);
          m &= m - 1u;
        }
        sh.selw[tid] |= t;
        break;
      }
      const int shift = span < (uint32_t)kRowBins ? 0 : 32 - __clz((int)span) - 11;
      for (int i = tid; i < kRowBins; i += kRowThreads) sh.hist[i] = 0u;
      __syncthreads();
      for (uint32_t m = cw; m; m &= m - 1u)
        atomicAdd(&sh.hist[(f2key(sv[32 * tid + __ffs(m) - 1]) - ka) >> shift], 1u);
      __syncthreads();
      row_find_bstar(sh, rem);
      const uint32_t bstar = (uint32_t)sh.bstar;
      nplay = (int)sh.hist[bstar];
      rem -= sh.above;
      uint32_t ns = 0u, nc = 0u;
      for (uint32_t m = cw; m; m &= m - 1u) {
        const int j = __ffs(m) - 1;
        const uint32_t bi = (f2key(sv[32 * tid + j]) - ka) >> shift;
        ns |= (uint32_t)(bi > bstar) << j;
        nc |= (uint32_t)(bi == bstar) << j;
      }
      cw = nc;
      if (nplay == rem) ns |= nc;
      sh.selw[tid] |= ns;
      if (nplay == rem) break;
      __syncthreads();   // every thread has read sh.hist[b*] and sh.above
    }
  }
  __syncthreads();

  // ---- ordered output: thread t writes the selected positions of bitmap word t
  const uint32_t sel = sh.selw[tid];
  int total;
  int r = block_excl_scan(__popc(sel), sh.scan, total);
  int32_t* out = out_idx + (int64_t)qi * K;
  float* outs = out_scores ? out_scores + (int64_t)qi * K : nullptr;
  const uint8_t* pfc = pf_codes ? pf_codes + (int64_t)(qi / T) * kv_stride * CSA2_CODE_BYTES : nullptr;
  const uint8_t* pfs = pf_codes ? pf_scales + (int64_t)(qi / T) * kv_stride * CSA2_SCALE_BYTES : nullptr;
  const int32_t* pblk = pool ? pool + (int64_t)qi * pool_stride : nullptr;
  for (uint32_t m = sel; m && r < K; m &= m - 1u, ++r) {
    const int pos = 32 * tid + __ffs(m) - 1;
    const int ent = pblk ? pblk[pos >> 3] * 8 + (pos & 7) : pos;
    out[r] = ent;
    if (outs) outs[r] = sv[pos];
    if (pfc && ent >= 0 && ent < kv_stride) {
      prefetch_l2_bulk(pfc + (int64_t)ent * CSA2_CODE_BYTES, CSA2_CODE_BYTES);
      prefetch_l2(pfs + (int64_t)ent * CSA2_SCALE_BYTES);
      prefetch_l2(pfs + (int64_t)ent * CSA2_SCALE_BYTES + CSA2_SCALE_BYTES - 1);
    }
  }
  for (int q = total + tid; q < K; q += kRowThreads) {
    out[q] = -1;
    if (outs) outs[q] = __int_as_float(0x7fc00000);
  }
}

// CTAs per query: enough for at most 8192 scores each; while the grid stays within one
// CTA per SM, more (slices of at least 2048), since the selection's phases scale with
// the slice, not with the cluster.
static int select_cluster_size(int64_t n_stride, int Q) {
  int64_t per = (n_stride + 8191) / 8192;
  int c = 1;
  while (c < per && c < kMaxCluster) c <<= 1;
  while (c < kMaxCluster && (int64_t)Q * 2 * c <= device_sm_count() && n_stride >= (int64_t)4096 * c) c <<= 1;
  return c;
}

cudaError_t launch_topk_select(const float* scores, int64_t score_stride, const int32_t* n_visible,
                               int Q, int64_t n_stride, int K, uint32_t* range, int32_t* out_idx,
                               float* out_scores, uint32_t* status, cudaStream_t st,
                               const uint8_t* pf_codes, const uint8_t* pf_scales, int T,
                               int64_t kv_stride, const int32_t* pool, int pool_stride) {
  static_assert(kNBMax % kSelThreads == 0 && kNBMin % kSelThreads == 0, "bins per thread");
  static_assert(kRowBins == 2 * kRowThreads, "two bins per thread in the row kernel's scan");
  if (Q == 0) return cudaSuccess;
  if (n_stride <= kRowMaxN && (int64_t)Q * select_cluster_size(n_stride, Q) > device_sm_count()) {
    // many queries: one CTA per query, the scores in shared memory (with few queries the
    // clusters below spread each query over several SMs and finish sooner)
    const size_t smem = (size_t)((n_stride + 3) & ~3) * 4;
    cudaError_t e = set_attr_once(5, (const void*)topk_row_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  kRowMaxN * 4);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)Q);
    cfg.blockDim = dim3(kRowThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int tt = T < 1 ? 1 : T;
    const int64_t kvs = kv_stride < 0 ? n_stride : kv_stride;
    return cudaLaunchKernelEx(&cfg, topk_row_kernel, scores, score_stride, n_visible, n_stride, K, range, out_idx,
                              out_scores, status, pf_codes, pf_scales, tt, kvs, pool, pool_stride);
  }
  const int C = select_cluster_size(n_stride, Q);
  const int NB = C <= 4 ? kNBMax : kNBMin;
  int slice_cap = (int)((n_stride + C - 1) / C);
  slice_cap = (slice_cap + 15) & ~15;
  const size_t smem = kSelHdr + (size_t)C * NB * 2 + (size_t)C * kCandCap * 8 +
                      (size_t)slice_cap * 5;
  if (smem > kSelSmemMax) return cudaErrorInvalidValue;
  cudaError_t e = set_attr_once(0, (const void*)topk_select_kernel,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSelSmemMax);
  if (e != cudaSuccess) return e;
  e = set_attr_once(1, (const void*)topk_select_kernel,
                    cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)C, (unsigned)Q);
  cfg.blockDim = dim3(kSelThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, topk_select_kernel, scores, score_stride, n_visible, n_stride, K,
                            slice_cap, range, out_idx, out_scores, status, pf_codes, pf_scales,
                            T < 1 ? 1 : T, kv_stride < 0 ? n_stride : kv_stride, pool, pool_stride);
}

__global__ void copy_idx_kernel(const int32_t* __restrict__ src, int32_t* __restrict__ dst,
                                int64_t n) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    dst[i] = src[i];
}

cudaError_t launch_copy_idx(const int32_t* src, int32_t* dst, int64_t n, cudaStream_t st) {
  if (n == 0 || src == dst) return cudaSuccess;
  int64_t want = (n + 255) / 256;
  int grid = (int)(want < 1024 ? want : 1024);
  copy_idx_kernel<<<grid, 256, 0, st>>>(src, dst, n);
  return cudaGetLastError();
}

}  // namespace csa2
