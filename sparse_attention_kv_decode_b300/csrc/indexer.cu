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
// so it is written for memory-level parallelism with almost nothing to
// synchronise: every CTA owns a contiguous, balanced run of chunks of
// kScoreUnroll 16-key groups of one query, its warps take the chunks one at a
// time from a shared counter, and a warp loads each group's MMA fragments
// straight from global memory into registers (8 x 16-byte loads per thread in
// flight). A
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

// Read-only 16-byte load that asks L2 for the whole 256-byte block (the keys are a
// contiguous stream, so the neighbouring lines are the next requests).
__device__ __forceinline__ uint4 ldg_key(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

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
  // Work comes in chunks of up to kScoreUnroll groups of one query (cpq per query). The
  // CTAs split the chunks evenly; inside a CTA the warps take them one at a time from a
  // shared counter, so that warps whose loads return sooner take more of them.
  const int cpq = (gpq + kScoreUnroll - 1) / kScoreUnroll;
  const int64_t total = (int64_t)Q * cpq;
  const int k0 = (int)(total * blockIdx.x / gridDim.x), k1 = (int)(total * (blockIdx.x + 1) / gridDim.x);
  __shared__ int s_next;
  if (threadIdx.x == 0) s_next = 0;
  __syncthreads();
  auto grab = [&]() {
    int v = 0;
    if (lane == 0) v = atomicAdd(&s_next, 1);
    return v;
  };
  int k = k0 + __shfl_sync(0xffffffffu, grab(), 0);

  int qi = -1;
  uint32_t qa[NT][8];
  float wv[NT][2];
  int nv = 0;
  const uint16_t* zb = nullptr;
  const int32_t* blk_row = nullptr;
  // running range of the scores this thread stored for query qi
  float smax = -INFINITY, smin = INFINITY;
  auto start_query = [&]() {
    load_q_frag<NT>(q_idx, w_idx, qi, H_I, g, tig, qa, wv);
    nv = pooled ? min(max(pool_nv[qi], 0), 8 * pool_stride) : clamp_nvis(n_visible, qi, n_stride);
    zb = z + (int64_t)(qi / T) * n_stride * CSA2_D_IDX;
    if (pooled) blk_row = pool + (int64_t)qi * pool_stride;
  };
  auto flush_range = [&]() {
    const bool any = smax >= smin;
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, any ? f2key(smax) : 0u);
    const uint32_t kinv = __reduce_max_sync(0xffffffffu, any ? ~f2key(smin) : 0u);
    if (lane == 0 && kmax != 0u) {
      atomicMax(range + 2 * qi, kinv);
      atomicMax(range + 2 * qi + 1, kmax);
    }
    smax = -INFINITY;
    smin = INFINITY;
  };
  while (k < k1) {
    // the next chunk is taken now; its index is needed only after this chunk
    const int nx = grab();
    // a warp's chunks increase, so its queries do too
    const int cq = k / cpq;
    if (cq != qi) {
      if (qi >= 0) flush_range();
      qi = cq;
      start_query();
    }
    const int grp = (k - cq * cpq) * kScoreUnroll;
    const int nb = min(kScoreUnroll, gpq - grp);
    // fragments of up to kScoreUnroll groups of the current query, all loads issued
    // before any use
    uint4 v[kScoreUnroll][4];
    int okm[kScoreUnroll];
#pragma unroll
    for (int u = 0; u < kScoreUnroll; ++u) {
      const int key0 = (grp + u) * kGroupKeys;
      // positions key0 + g and key0 + 8 + g; their key rows (pool: the blocks' entries)
      bool oka = u < nb && key0 + g < nv, okb = u < nb && key0 + 8 + g < nv;
      int64_t ra = key0 + g, rb = ra + 8;
      if (pooled) {
        const int32_t* blk = blk_row + (key0 >> 3);
        ra = oka ? (int64_t)blk[0] * 8 + g : 0;
        rb = okb ? (int64_t)blk[1] * 8 + g : 0;
        oka = oka && ra >= 0 && ra < n_stride;
        okb = okb && rb >= 0 && rb < n_stride;
      }
      okm[u] = (oka ? 1 : 0) | (okb ? 2 : 0);
      const uint4* pa = reinterpret_cast<const uint4*>(zb + ra * CSA2_D_IDX);
      const uint4* pb = reinterpret_cast<const uint4*>(zb + rb * CSA2_D_IDX);
      v[u][0] = oka ? ldg_key(pa + tig) : make_uint4(0, 0, 0, 0);
      v[u][1] = oka ? ldg_key(pa + 4 + tig) : make_uint4(0, 0, 0, 0);
      v[u][2] = okb ? ldg_key(pb + tig) : make_uint4(0, 0, 0, 0);
      v[u][3] = okb ? ldg_key(pb + 4 + tig) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kScoreUnroll; ++u) {
      const int key0 = (grp + u) * kGroupKeys;
      if (u >= nb || key0 >= nv) continue;   // (uniform over the warp)
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
      // thread tig 0 stores row g, tig 1 row g + 8
      const float sc = tig == 0 ? pg : pg8;
      const bool ok = (tig == 0 && (okm[u] & 1)) || (tig == 1 && (okm[u] & 2));
      if (ok) {
        scores[(int64_t)qi * score_stride + key0 + g + 8 * tig] = sc;
        smax = fmaxf(smax, sc);
        smin = fminf(smin, sc);
      }
    }
    k = k0 + __shfl_sync(0xffffffffu, nx, 0);
  }
  if (qi >= 0) flush_range();
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
  const int64_t gpq = (npos + kGroupKeys - 1) / kGroupKeys;
  const int64_t total = (int64_t)Q * ((gpq + kScoreUnroll - 1) / kScoreUnroll);   // chunks
  if (total >= ((int64_t)1 << 31)) return cudaErrorInvalidValue;
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
// Top-K selection: shared pieces
// ---------------------------------------------------------------------------
// Every selection kernel bins scores into monotone bins (equal scores share a bin,
// bins never reorder scores), finds the bin b* holding the K-th score from the top,
// takes the higher bins and refines b* until at most a rank-able handful remains;
// the output lists the selected positions in ascending order.
constexpr int kSelThreads = 1024;
constexpr int kMaxLevels = 12;
constexpr int kMaxCluster = 16;
constexpr size_t kSelSmemMax = 200 * 1024;

// Exclusive prefix sum of v over the block (1024 threads); total = the sum.
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

// The same over 64-bit words (fields that never carry into each other: several
// independent sums in one scan).
__device__ __forceinline__ uint64_t block_excl_scan64(uint64_t v, unsigned long long* scan) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scan[warp] = x;
  __syncthreads();
  if (warp == 0) {
    unsigned long long s = lane < kSelThreads / 32 ? scan[lane] : 0ull;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < kSelThreads / 32) scan[lane] = s;
  }
  __syncthreads();
  const uint64_t pre = (warp > 0 ? scan[warp - 1] : 0ull) + x - v;
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
  const uint8_t* pfc = pf_codes ? pf_codes + (int64_t)(qi / T) * kv_stride * CSA2_ENTRY_BYTES : nullptr;
  const uint8_t* pfs = pf_codes ? pf_scales + (int64_t)(qi / T) * kv_stride * CSA2_ENTRY_BYTES : nullptr;
  const bool pf_record = pf_codes != nullptr && pf_scales == pf_codes + CSA2_CODE_BYTES;
  const int32_t* pblk = pool ? pool + (int64_t)qi * pool_stride : nullptr;
  for (uint32_t m = sel; m && r < K; m &= m - 1u, ++r) {
    const int pos = 32 * tid + __ffs(m) - 1;
    const int ent = pblk ? pblk[pos >> 3] * 8 + (pos & 7) : pos;
    out[r] = ent;
    if (outs) outs[r] = sv[pos];
    if (pfc && ent >= 0 && ent < kv_stride) {
      if (pf_record) {
        prefetch_l2_bulk(pfc + (int64_t)ent * CSA2_ENTRY_BYTES, CSA2_ENTRY_BYTES);
      } else {
        prefetch_l2_bulk(pfc + (int64_t)ent * CSA2_ENTRY_BYTES, CSA2_CODE_BYTES);
        prefetch_l2(pfs + (int64_t)ent * CSA2_ENTRY_BYTES);
        prefetch_l2(pfs + (int64_t)ent * CSA2_ENTRY_BYTES + CSA2_SCALE_BYTES - 1);
      }
    }
  }
  for (int q = total + tid; q < K; q += kRowThreads) {
    out[q] = -1;
    if (outs) outs[q] = __int_as_float(0x7fc00000);
  }
}

// ---------------------------------------------------------------------------
// Top-K selection, one cluster of C CTAs per query (few queries, long score rows)
// ---------------------------------------------------------------------------
// CTA r owns the positions [r*slice, (r+1)*slice) of the scored row, the visible ones
// among them in play (slice = ceil(row / C) rounded up to a multiple of 32, so the CTAs'
// bitmap words do not overlap), lands their scores in shared memory with a few bulk
// copies, and visits local positions k * kRowThreads + t. Every exchange is a push into
// the peers' receive buffers followed by one cluster barrier, and every decision after it
// is taken from the same pushed data, so all CTAs follow the same path:
//   round 0  local histogram over the range the scoring kernel left (kRowBins monotone
//            bins, row_bin), pushed as 16-bit counts; after the barrier every CTA sums
//            them: b* (the K-th score's bin), the scores above it and every CTA's share
//            of them and of b* follow; local positions above b* are selected, b*'s stay
//            in play (bitmap words built with ballots);
//   exact    when at most kRowRankCap scores remain in play, each CTA pushes its
//            (score, position) pairs into one list of all of them (CTA r's after those
//            of the CTAs before it); after the barrier every CTA ranks the whole list by
//            (score desc, position asc), so it knows every CTA's selected count;
//   refine   otherwise the scores in play are binned by their integer keys over the
//            cluster-wide key range (one barrier for the range, one for the histogram);
//            when they all tie, the lowest positions win.
// A CTA's output offset is the number selected in the CTAs before it.
struct ClusterShared {
  uint32_t hist[kRowBins];
  uint32_t selw[kRowThreads / 2];    // selected bitmap (slices of at most 16384)
  uint32_t candw[kRowThreads / 2];   // in-play bitmap
  int scan[kRowThreads / 32];
  unsigned long long scan64[kRowThreads / 32];
  float red[2][kRowThreads / 32];
  uint4 rec_in[kMaxCluster];         // pushed (min, max, count) of each CTA
  int cta_sel[kMaxCluster];          // selected positions of each CTA so far
  int cta_play[kMaxCluster];         // positions in play of each CTA
  int cta_taken[kMaxCluster];        // ranked and taken in the exact round
  int cta_warp[kMaxCluster][kRowThreads / 32];   // per-warp counts above b*, per CTA
  int bstar, above;
  uint64_t bar_chunk[kRowThreads / 64];   // one per 1024-score chunk of the slice (<= 16384)
};

// Block-wide min of a and max of b (all threads get them).
__device__ __forceinline__ void block_minmax(float& a, float& b, float (&red)[2][kRowThreads / 32]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a = fminf(a, __shfl_xor_sync(0xffffffffu, a, o));
    b = fmaxf(b, __shfl_xor_sync(0xffffffffu, b, o));
  }
  __syncthreads();   // red may still be read by a previous call
  if (lane == 0) {
    red[0][warp] = a;
    red[1][warp] = b;
  }
  __syncthreads();
  a = red[0][lane];
  b = red[1][lane];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a = fminf(a, __shfl_xor_sync(0xffffffffu, a, o));
    b = fmaxf(b, __shfl_xor_sync(0xffffffffu, b, o));
  }
}

// Push this CTA's histogram (sh.hist, as 16-bit counts) into slot r of every peer's hist_in.
__device__ __forceinline__ void push_hist(ClusterShared& sh, uint16_t* hist_in, uint32_t C, uint32_t r) {
  for (int j = threadIdx.x; j < (int)C * (kRowBins / 8); j += kRowThreads) {
    const int peer = j / (kRowBins / 8), o8 = j % (kRowBins / 8);
    const uint32_t* h = &sh.hist[8 * o8];
    st_remote_v4(&hist_in[r * kRowBins + 8 * o8], peer,
                 make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16), h[6] | (h[7] << 16)));
  }
}

// From the C pushed histograms: b* and the count above it for the rem-th largest
// (sh.bstar, sh.above), and for every CTA its count above b* (added to sh.cta_sel) and in
// b* (sh.cta_play). Returns the total in b*.
__device__ __forceinline__ int cluster_bstar(ClusterShared& sh, const uint16_t* hist_in, uint32_t C, int rem) {
  const int tid = threadIdx.x, lane = tid & 31;
  const int b1 = kRowBins - 1 - 2 * tid, b0 = b1 - 1;
  if (C <= 4) {
    // every CTA's counts in one scan: CTA rr's in bits [16 rr, 16 rr + 16) (a slice holds
    // at most 16384 positions, so no field carries)
    uint64_t v1 = 0u, v0 = 0u;
    for (uint32_t rr = 0; rr < C; ++rr) {
      v1 |= (uint64_t)hist_in[rr * kRowBins + b1] << (16 * rr);
      v0 |= (uint64_t)hist_in[rr * kRowBins + b0] << (16 * rr);
    }
    const uint64_t pre = block_excl_scan64(v1 + v0, sh.scan64);
    auto fsum = [](uint64_t x) {
      return (int)((x & 0xFFFFu) + ((x >> 16) & 0xFFFFu) + ((x >> 32) & 0xFFFFu) + (x >> 48));
    };
    const int above = fsum(pre), h1 = fsum(v1), h0 = fsum(v0);
    uint64_t at = 0u, in = 0u;
    bool mine = false;
    if (above < rem && rem <= above + h1) {
      sh.bstar = b1;
      sh.above = above;
      at = pre;
      in = v1;
      mine = true;
    } else if (above + h1 < rem && rem <= above + h1 + h0) {
      sh.bstar = b0;
      sh.above = above + h1;
      at = pre + v1;
      in = v0;
      mine = true;
    }
    if (mine)
      for (uint32_t rr = 0; rr < C; ++rr) {
        sh.cta_sel[rr] += (int)((at >> (16 * rr)) & 0xFFFFu);
        sh.cta_play[rr] = (int)((in >> (16 * rr)) & 0xFFFFu);
      }
    __syncthreads();
    int n = 0;
    for (uint32_t rr = 0; rr < C; ++rr) n += sh.cta_play[rr];
    return n;
  }
  int h1 = 0, h0 = 0;
  for (uint32_t rr = 0; rr < C; ++rr) {
    h1 += hist_in[rr * kRowBins + b1];
    h0 += hist_in[rr * kRowBins + b0];
  }
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
  const int bstar = sh.bstar, warp = tid >> 5;
  // every CTA's count above b*: per-warp sums, then one warp per CTA adds its 32 of them
  for (uint32_t rr = 0; rr < C; ++rr) {
    const int a = (b1 > bstar ? (int)hist_in[rr * kRowBins + b1] : 0) +
                  (b0 > bstar ? (int)hist_in[rr * kRowBins + b0] : 0);
    const int s = __reduce_add_sync(0xffffffffu, a);
    if (lane == 0) sh.cta_warp[rr][warp] = s;
  }
  if (tid < (int)C) sh.cta_play[tid] = hist_in[tid * kRowBins + bstar];
  __syncthreads();
  if (warp < (int)C) {
    const int s = __reduce_add_sync(0xffffffffu, sh.cta_warp[warp][lane]);
    if (lane == 0) sh.cta_sel[warp] += s;
  }
  int n = 0;
  for (uint32_t rr = 0; rr < C; ++rr) n += sh.cta_play[rr];
  return n;
}

__global__ void __launch_bounds__(kRowThreads, 1) topk_cluster_kernel(
    const float* __restrict__ scores, int64_t score_stride, const int32_t* __restrict__ n_visible,
    int64_t n_stride, int K, uint32_t* __restrict__ range, int32_t* __restrict__ out_idx,
    float* __restrict__ out_scores, uint32_t* __restrict__ status, const uint8_t* __restrict__ pf_codes,
    const uint8_t* __restrict__ pf_scales, int T, int64_t kv_stride, const int32_t* __restrict__ pool,
    int pool_stride, int slice_cap) {
  extern __shared__ __align__(128) uint8_t cl_raw[];
  __shared__ ClusterShared sh;
  uint32_t C, r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(C));
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  float* sv = reinterpret_cast<float*>(cl_raw);                                     // [slice_cap]
  uint16_t* hist_in = reinterpret_cast<uint16_t*>(cl_raw + (size_t)slice_cap * 4);  // [C][kRowBins]
  float* cand_s = reinterpret_cast<float*>(hist_in + (size_t)C * kRowBins);          // [kRowRankCap]
  int* cand_i = reinterpret_cast<int*>(cand_s + kRowRankCap);                        // [kRowRankCap]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int qi = blockIdx.y;
  if (tid < kRowThreads / 64) {
    // the thread that initialises chunk tid's barrier also arms it and issues its copy
    mbar_init(smem_u32(&sh.bar_chunk[tid]), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (tid < kRowThreads / 2) {
    sh.selw[tid] = 0u;
    sh.candw[tid] = 0u;
  }
  if (tid < kMaxCluster) {
    sh.cta_sel[tid] = 0;
    sh.cta_taken[tid] = 0;
  }
  __syncthreads();
  // no CTA writes into a peer's shared memory before every CTA of the cluster runs: the
  // matching wait comes after the score load
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // CTA r's slice is positions [r * slice_cap, ..) of the scored row (n_stride long), so
  // its copies go out before the visible count is known. Chunk k (scores k * 1024 ..)
  // lands with its own bulk copy and mbarrier, so that the first pass over it starts as
  // soon as it is there (a score row is score_stride >= roundup4(n_stride) floats).
  const int slice = slice_cap;
  const int my0 = (int)r * slice;
  const int my_cap = min(max((int)n_stride - my0, 0), slice);
  const int nk_all = (my_cap + kRowThreads - 1) / kRowThreads;
  if (tid < nk_all) {
    const uint32_t bytes = (uint32_t)((min(my_cap - tid * kRowThreads, kRowThreads) + 3) >> 2) * 16;
    mbar_arrive_expect_tx(smem_u32(&sh.bar_chunk[tid]), bytes);
    bulk_g2s(smem_u32(sv + tid * kRowThreads), scores + (int64_t)qi * score_stride + my0 + tid * kRowThreads, bytes,
             smem_u32(&sh.bar_chunk[tid]));
  }
  // every thread reads the range words and the visible count itself (one request per
  // warp), so that nothing waits for them before the first score chunk is needed
  const uint32_t rng0 = range[2 * qi], rng1 = range[2 * qi + 1];
  const int nvis = clamp_nvis(n_visible, qi, n_stride);
  auto len_of = [&](int rr) { return min(max(nvis - rr * slice, 0), slice); };
  int my_len = len_of((int)r);
  const int nk = (my_len + kRowThreads - 1) / kRowThreads;   // chunks holding visible scores
  // (a copy that did not land leaves stale scores: the selection still completes, flagged)
  bool load_ok = true;
  auto wait_chunk = [&](int k) {
    if (!mbar_wait(smem_u32(&sh.bar_chunk[k]), 0)) load_ok = false;
  };
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
  const int nwords = (my_len + 31) >> 5;
  const uint32_t my_valid = [&] {
    const int n = min(max(my_len - 32 * tid, 0), 32);
    return n >= 32 ? 0xffffffffu : ((1u << n) - 1u);
  }();
  int off = 0, total = 0;
  // the range words are set back to zero by CTA 0 once every CTA has read them, i.e. after
  // the first cluster barrier (with nvis <= K no CTA uses them)
  bool range_clear = false;
  auto barrier = [&]() {
    cluster_barrier();
    if (!range_clear) {
      if (r == 0 && tid == 0) {
        range[2 * qi] = 0u;
        range[2 * qi + 1] = 0u;
      }
      range_clear = true;
    }
  };
  if (nvis <= K) {
    // everything visible is selected: position order is the output order
    for (int k = 0; k < nk; ++k) wait_chunk(k);
    if (tid < nwords) sh.selw[tid] = my_valid;
    off = my0 < nvis ? my0 : nvis;
    total = nvis;
    if (r == 0 && tid == 0) {
      range[2 * qi] = 0u;
      range[2 * qi + 1] = 0u;
    }
    __syncthreads();
  } else {
    int rem = K;
    float lo = key2f(~rng0), hi = key2f(rng1);
    if (!(rng1 != 0u && lo < hi && isfinite(lo) && isfinite(hi))) {
      // no range left by the scoring kernel: the cluster-wide min / max
      float a = INFINITY, b = -INFINITY;
      for (int k = 0; k < nk; ++k) {
        wait_chunk(k);
        const int p = k * kRowThreads + tid;
        if (p < my_len) {
          a = fminf(a, sv[p]);
          b = fmaxf(b, sv[p]);
        }
      }
      block_minmax(a, b, sh.red);
      if (tid < (int)C) st_remote_v4(&sh.rec_in[r], tid, make_uint4(__float_as_uint(a), __float_as_uint(b), 0u, 0u));
      barrier();
      lo = INFINITY;
      hi = -INFINITY;
      for (uint32_t rr = 0; rr < C; ++rr) {
        lo = fminf(lo, __uint_as_float(sh.rec_in[rr].x));
        hi = fmaxf(hi, __uint_as_float(sh.rec_in[rr].y));
      }
    }
    int nplay = nvis;
    bool done = false;
    const float scl0 = (float)(kRowBins - 1) / (hi - lo);
    if (lo < hi && scl0 <= 1e30f) {
      // ---- round 0 over every visible position
      for (int i = tid; i < kRowBins; i += kRowThreads) sh.hist[i] = 0u;
      __syncthreads();
      for (int k = 0; k < nk; ++k) {
        wait_chunk(k);
        const int p = k * kRowThreads + tid;
        if (p < my_len) atomicAdd(&sh.hist[row_bin(sv[p], lo, scl0)], 1u);
      }
      __syncthreads();
      push_hist(sh, hist_in, C, r);
      barrier();
      nplay = cluster_bstar(sh, hist_in, C, rem);
      const uint32_t bstar = (uint32_t)sh.bstar;
      rem -= sh.above;
      // lane k of each warp collects bitmap word k * 32 + warp (local positions k * 1024 + 32 warp ..)
      uint32_t my_sel = 0u, my_cand = 0u;
      for (int k = 0; k < nk; ++k) {
        const int p = k * kRowThreads + tid;
        const bool ok = p < my_len;
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
        if (tid < nwords) sh.selw[tid] |= sh.candw[tid];
        if (tid < (int)C) sh.cta_sel[tid] += sh.cta_play[tid];
        done = true;
      }
    } else {
      // all visible scores tie (or their range is degenerate): all in play
      for (int k = 0; k < nk; ++k) wait_chunk(k);
      if (tid < nwords) sh.candw[tid] = my_valid;
      if (tid < (int)C) sh.cta_play[tid] = len_of(tid);
    }
    __syncthreads();
    // ---- later rounds over the positions in play (thread t: bitmap word t)
#pragma unroll 1
    for (int level = 1; !done; ++level) {
      const uint32_t cw = tid < nwords ? sh.candw[tid] : 0u;
      if (nplay <= kRowRankCap) {
        // exact: push this CTA's (score, position) list to every peer
        // one list of all nplay candidates, CTA r's at offset sum(cta_play[< r])
        int tot;
        int pre = block_excl_scan(__popc(cw), sh.scan, tot);
        for (uint32_t rr = 0; rr < r; ++rr) pre += sh.cta_play[rr];
        for (uint32_t m = cw; m; m &= m - 1u, ++pre) {
          const int lp = 32 * tid + __ffs(m) - 1;
          for (uint32_t pr = 0; pr < C; ++pr) {
            st_remote_u32(reinterpret_cast<uint32_t*>(&cand_s[pre]), pr, __float_as_uint(sv[lp]));
            st_remote_u32(reinterpret_cast<uint32_t*>(&cand_i[pre]), pr, (uint32_t)(my0 + lp));
          }
        }
        barrier();
        // rank every candidate: eight threads per candidate, each comparing it with every
        // eighth of the others
        static_assert(kRowRankCap * 8 <= kRowThreads, "eight rankers per candidate");
        const int c = tid >> 3, sub = tid & 7;
        int rank = 0, i = 0;
        if (c < nplay) {
          const float sc = cand_s[c];
          i = cand_i[c];
#pragma unroll 4
          for (int k2 = sub; k2 < nplay; k2 += 8) {
            const float t2 = cand_s[k2];
            rank += (t2 > sc) || (t2 == sc && cand_i[k2] < i);
          }
        }
        rank += __shfl_xor_sync(0xffffffffu, rank, 1);
        rank += __shfl_xor_sync(0xffffffffu, rank, 2);
        rank += __shfl_xor_sync(0xffffffffu, rank, 4);
        if (c < nplay && sub == 0 && rank < rem) {
          const int rr = i / slice;   // the CTA that holds candidate c
          atomicAdd(&sh.cta_taken[rr], 1);
          if (rr == (int)r) atomicOr(&sh.selw[(i - my0) >> 5], 1u << ((i - my0) & 31));
        }
        __syncthreads();
        if (tid < (int)C) sh.cta_sel[tid] += sh.cta_taken[tid];
        break;
      }
      // the cluster-wide key range of the scores in play
      uint32_t ka = 0xffffffffu, kb = 0u;
      for (uint32_t m = cw; m; m &= m - 1u) {
        const uint32_t x = f2key(sv[32 * tid + __ffs(m) - 1]);
        ka = min(ka, x);
        kb = max(kb, x);
      }
      {
        ka = __reduce_min_sync(0xffffffffu, ka);
        kb = __reduce_max_sync(0xffffffffu, kb);
        __syncthreads();
        if (lane == 0) {
          sh.red[0][warp] = __uint_as_float(ka);
          sh.red[1][warp] = __uint_as_float(kb);
        }
        __syncthreads();
        ka = __reduce_min_sync(0xffffffffu, __float_as_uint(sh.red[0][lane]));
        kb = __reduce_max_sync(0xffffffffu, __float_as_uint(sh.red[1][lane]));
      }
      if (tid < (int)C) st_remote_v4(&sh.rec_in[r], tid, make_uint4(ka, kb, 0u, 0u));
      barrier();
      ka = 0xffffffffu;
      kb = 0u;
      for (uint32_t rr = 0; rr < C; ++rr)
        if (sh.cta_play[rr] > 0) {
          ka = min(ka, sh.rec_in[rr].x);
          kb = max(kb, sh.rec_in[rr].y);
        }
      const uint32_t span = kb - ka;
      if (span == 0u || level >= kMaxLevels) {
        // all tie (or the search did not settle): lowest positions first
        if (span != 0u && r == 0 && tid == 0) atomicOr(status, CSA2_DEV_TOPK_LEVELS);
        int pre_cta = 0;
        for (uint32_t rr = 0; rr < r; ++rr) pre_cta += sh.cta_play[rr];
        int tot;
        const int pre = block_excl_scan(__popc(cw), sh.scan, tot);
        int take = min(max(rem - pre_cta - pre, 0), __popc(cw));
        uint32_t tk = 0u;
        for (uint32_t m = cw; take > 0; --take) {
          tk |= m & (~m + 1u);
          m &= m - 1u;
        }
        if (tid < nwords) sh.selw[tid] |= tk;
        __syncthreads();
        if (tid == 0) {
          int acc = 0;
          for (uint32_t rr = 0; rr < C; ++rr) {
            sh.cta_sel[rr] += min(max(rem - acc, 0), sh.cta_play[rr]);
            acc += sh.cta_play[rr];
          }
        }
        break;
      }
      const int shift = span < (uint32_t)kRowBins ? 0 : 32 - __clz((int)span) - 11;
      for (int i = tid; i < kRowBins; i += kRowThreads) sh.hist[i] = 0u;
      __syncthreads();
      for (uint32_t m = cw; m; m &= m - 1u)
        atomicAdd(&sh.hist[(f2key(sv[32 * tid + __ffs(m) - 1]) - ka) >> shift], 1u);
      __syncthreads();
      push_hist(sh, hist_in, C, r);
      barrier();
      nplay = cluster_bstar(sh, hist_in, C, rem);
      const uint32_t bstar = (uint32_t)sh.bstar;
      rem -= sh.above;
      uint32_t ns = 0u, nc = 0u;
      for (uint32_t m = cw; m; m &= m - 1u) {
        const int j = __ffs(m) - 1;
        const uint32_t bi = (f2key(sv[32 * tid + j]) - ka) >> shift;
        ns |= (uint32_t)(bi > bstar) << j;
        nc |= (uint32_t)(bi == bstar) << j;
      }
      if (tid < nwords) {
        sh.selw[tid] |= ns | (nplay == rem ? nc : 0u);
        sh.candw[tid] = nc;
      }
      __syncthreads();
      if (nplay == rem) {
        if (tid < (int)C) sh.cta_sel[tid] += sh.cta_play[tid];
        break;
      }
    }
    __syncthreads();
    for (uint32_t rr = 0; rr < C; ++rr) {
      if (rr < r) off += sh.cta_sel[rr];
      total += sh.cta_sel[rr];
    }
  }

  // copies of chunks past the visible scores land before the CTA exits
  for (int k = nk; k < nk_all; ++k) wait_chunk(k);
  if (!load_ok) atomicOr(status, CSA2_DEV_PIPELINE_TIMEOUT);
  // ---- ordered output: thread t writes the selected positions of bits [t b, t b + b)
  // of the bitmap, b = 8 (slices of at most 8192) or 16, so that every warp has a share
  const int obits = nwords <= kRowThreads / 4 ? 8 : 16;
  const int obit0 = tid * obits;
  const uint32_t sel = (obit0 >> 5) < nwords
                           ? (sh.selw[obit0 >> 5] >> (obit0 & 31)) & ((1u << obits) - 1u)
                           : 0u;
  int cnt;
  int p = off + block_excl_scan(__popc(sel), sh.scan, cnt);
  int32_t* out = out_idx + (int64_t)qi * K;
  float* outs = out_scores ? out_scores + (int64_t)qi * K : nullptr;
  const uint8_t* pfc = pf_codes ? pf_codes + (int64_t)(qi / T) * kv_stride * CSA2_ENTRY_BYTES : nullptr;
  const uint8_t* pfs = pf_codes ? pf_scales + (int64_t)(qi / T) * kv_stride * CSA2_ENTRY_BYTES : nullptr;
  const bool pf_record = pf_codes != nullptr && pf_scales == pf_codes + CSA2_CODE_BYTES;
  const int32_t* pblk = pool ? pool + (int64_t)qi * pool_stride : nullptr;
  for (uint32_t m = sel; m && p < K; m &= m - 1u, ++p) {
    const int lp = obit0 + __ffs(m) - 1;
    const int pos = my0 + lp;
    const int ent = pblk ? pblk[pos >> 3] * 8 + (pos & 7) : pos;
    out[p] = ent;
    if (outs) outs[p] = sv[lp];
    if (pfc && ent >= 0 && ent < kv_stride) {
      if (pf_record) {
        prefetch_l2_bulk(pfc + (int64_t)ent * CSA2_ENTRY_BYTES, CSA2_ENTRY_BYTES);
      } else {
        prefetch_l2_bulk(pfc + (int64_t)ent * CSA2_ENTRY_BYTES, CSA2_CODE_BYTES);
        prefetch_l2(pfs + (int64_t)ent * CSA2_ENTRY_BYTES);
        prefetch_l2(pfs + (int64_t)ent * CSA2_ENTRY_BYTES + CSA2_SCALE_BYTES - 1);
      }
    }
  }
  if (r == C - 1)
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
  const int slice_cap = (int)(((n_stride + C - 1) / C + 31) & ~31);
  if (slice_cap > kRowThreads * 16 || C > kMaxCluster) return cudaErrorInvalidValue;
  const size_t smem = (size_t)slice_cap * 4 + (size_t)C * kRowBins * 2 + (size_t)kRowRankCap * 8;
  if (smem > kSelSmemMax) return cudaErrorInvalidValue;
  cudaError_t e = set_attr_once(0, (const void*)topk_cluster_kernel,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSelSmemMax);
  if (e != cudaSuccess) return e;
  e = set_attr_once(1, (const void*)topk_cluster_kernel,
                    cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)C, (unsigned)Q);
  cfg.blockDim = dim3(kRowThreads);
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
  return cudaLaunchKernelEx(&cfg, topk_cluster_kernel, scores, score_stride, n_visible, n_stride, K, range,
                            out_idx, out_scores, status, pf_codes, pf_scales, T < 1 ? 1 : T,
                            kv_stride < 0 ? n_stride : kv_stride, pool, pool_stride, slice_cap);
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
