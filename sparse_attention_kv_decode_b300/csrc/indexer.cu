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
// heads as N; each thread streams two 16-byte pieces of a key row, so a warp
// reads 2 KB contiguous per tile. Selection runs in one thread-block cluster
// per query: every CTA keeps its slice of scores in shared memory and the
// cluster agrees on the K-th score through a few histogram rounds exchanged
// over distributed shared memory (no global atomics, no spin waits).
#include <cooperative_groups.h>

#include "csa2_internal.cuh"

namespace cg = cooperative_groups;

namespace csa2 {

// ---------------------------------------------------------------------------
// Scoring
// ---------------------------------------------------------------------------
// Each thread (g = lane/4, tig = lane%4) loads, for key rows g and g+8 of a
// 16-key tile, the 16-byte pieces at byte offsets 16*tig and 64+16*tig. The
// MMA's k-slots are assigned to channels so that the A fragment registers are
// exactly those loaded words, and the B fragment (indexer query of head g) is
// read from the same offsets: the contraction order is a permutation of the
// 64 channels, which leaves the dot products unchanged.
template <int NT>
__global__ void __launch_bounds__(256) index_score_kernel(
    const uint16_t* __restrict__ q_idx, const float* __restrict__ w_idx,
    const uint16_t* __restrict__ z, int64_t n_stride, const int32_t* __restrict__ n_visible, int T,
    int H_I, float* __restrict__ scores, int64_t score_stride) {
  const int qi = blockIdx.y;
  const int b = qi / T;
  int nvis = n_visible[qi];
  nvis = nvis < 0 ? 0 : (nvis > n_stride ? (int)n_stride : nvis);
  const int64_t base = (int64_t)blockIdx.x * kScoreTile;
  if (base >= nvis) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tig = lane & 3;

  uint32_t qa[NT][8];
  float wv[NT][2];
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

  const uint16_t* zb = z + (int64_t)b * n_stride * CSA2_D_IDX;
  float* srow = scores + (int64_t)qi * score_stride;
  constexpr int kTilesPerWarp = kScoreTile / 16 / 8;  // 8
  constexpr int kU = 4;
#pragma unroll 1
  for (int t0 = 0; t0 < kTilesPerWarp; t0 += kU) {
    uint32_t ra[kU][16];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int64_t kg = base + (int64_t)(warp * kTilesPerWarp + t0 + u) * 16 + g;
      const int64_t kg8 = kg + 8;
      uint4 v0 = make_uint4(0, 0, 0, 0), v1 = v0, v2 = v0, v3 = v0;
      if (kg < nvis) {
        const uint16_t* p = zb + kg * CSA2_D_IDX;
        v0 = ldg_stream(p + 8 * tig);
        v1 = ldg_stream(p + 32 + 8 * tig);
      }
      if (kg8 < nvis) {
        const uint16_t* p = zb + kg8 * CSA2_D_IDX;
        v2 = ldg_stream(p + 8 * tig);
        v3 = ldg_stream(p + 32 + 8 * tig);
      }
      ra[u][0] = v0.x; ra[u][1] = v0.y; ra[u][2] = v0.z; ra[u][3] = v0.w;
      ra[u][4] = v1.x; ra[u][5] = v1.y; ra[u][6] = v1.z; ra[u][7] = v1.w;
      ra[u][8] = v2.x; ra[u][9] = v2.y; ra[u][10] = v2.z; ra[u][11] = v2.w;
      ra[u][12] = v3.x; ra[u][13] = v3.y; ra[u][14] = v3.z; ra[u][15] = v3.w;
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      float pg = 0.f, pg8 = 0.f;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          // k-step j uses words 2j, 2j+1 of the row-g / row-g+8 register sets
          mma_bf16(acc, ra[u][2 * j], ra[u][8 + 2 * j], ra[u][2 * j + 1], ra[u][8 + 2 * j + 1],
                   qa[nt][2 * j], qa[nt][2 * j + 1]);
        }
        pg += wv[nt][0] * fmaxf(acc[0], 0.f) + wv[nt][1] * fmaxf(acc[1], 0.f);
        pg8 += wv[nt][0] * fmaxf(acc[2], 0.f) + wv[nt][1] * fmaxf(acc[3], 0.f);
      }
      pg += __shfl_xor_sync(0xffffffffu, pg, 1);
      pg += __shfl_xor_sync(0xffffffffu, pg, 2);
      pg8 += __shfl_xor_sync(0xffffffffu, pg8, 1);
      pg8 += __shfl_xor_sync(0xffffffffu, pg8, 2);
      const int64_t kg = base + (int64_t)(warp * kTilesPerWarp + t0 + u) * 16 + g;
      if (tig == 0 && kg < nvis) srow[kg] = pg;
      if (tig == 1 && kg + 8 < nvis) srow[kg + 8] = pg8;
    }
  }
}

cudaError_t launch_index_score(const void* q_idx, const float* w_idx, const void* z,
                               int64_t n_stride, const int32_t* n_visible, int B, int T, int H_I,
                               float* scores, int64_t score_stride, cudaStream_t st) {
  const int Q = B * T;
  dim3 grid((unsigned)((n_stride + kScoreTile - 1) / kScoreTile), (unsigned)Q);
  if (grid.x == 0 || Q == 0) return cudaSuccess;
  auto qp = static_cast<const uint16_t*>(q_idx);
  auto zp = static_cast<const uint16_t*>(z);
  if (H_I <= 8)
    index_score_kernel<1><<<grid, 256, 0, st>>>(qp, w_idx, zp, n_stride, n_visible, T, H_I, scores,
                                                score_stride);
  else
    index_score_kernel<2><<<grid, 256, 0, st>>>(qp, w_idx, zp, n_stride, n_visible, T, H_I, scores,
                                                score_stride);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Top-K selection: one cluster of C CTAs per query
// ---------------------------------------------------------------------------
constexpr int kSelThreads = 512;
constexpr int kNB = 1024;          // histogram bins per refinement round
constexpr int kCandCap = 1024;     // candidates resolved exactly by ranking
constexpr int kMaxLevels = 12;
constexpr size_t kSelSmemMax = 220 * 1024;

struct SelRec {
  float lo, hi;
  int cnt, pad;
};

struct SelShared {
  uint32_t hist[kNB];
  uint32_t ghist[kNB];
  SelRec rec[kMaxLevels + 1];
  int sel_cnt;
  int bstar;
  int scan[kSelThreads / 32];
  float red_f[2][kSelThreads / 32];
  int red_i[kSelThreads / 32];
  int cand_n;
  float cand_s[kCandCap];
  int cand_i[kCandCap];
  float all_s[kCandCap];
  int all_i[kCandCap];
};

__device__ __forceinline__ int bin_of(float s, float lo, float scl) {
  float t = (s - lo) * scl;
  int bi = (int)t;
  return bi < 0 ? 0 : (bi > kNB - 1 ? kNB - 1 : bi);
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

__global__ void __launch_bounds__(kSelThreads) topk_select_kernel(
    const float* __restrict__ scores, int64_t score_stride, const int32_t* __restrict__ n_visible,
    int64_t n_stride, int K, int slice_cap, int32_t* __restrict__ out_idx,
    float* __restrict__ out_scores, uint32_t* __restrict__ status) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  SelShared& sh = *reinterpret_cast<SelShared*>(smem_raw);
  float* sc = reinterpret_cast<float*>(smem_raw + sizeof(SelShared));
  uint8_t* state = reinterpret_cast<uint8_t*>(sc + slice_cap);

  cg::cluster_group cluster = cg::this_cluster();
  const int C = (int)cluster.num_blocks();
  const int r = (int)cluster.block_rank();
  const int tid = threadIdx.x;
  const int qi = blockIdx.y;
  int nvis = n_visible[qi];
  nvis = nvis < 0 ? 0 : (nvis > n_stride ? (int)n_stride : nvis);
  const int slice = (nvis + C - 1) / C;
  const int my0 = r * slice;
  int my_len = nvis - my0;
  my_len = my_len < 0 ? 0 : (my_len > slice ? slice : my_len);
  const int need = nvis < K ? nvis : K;
  int32_t* out = out_idx + (int64_t)qi * K;
  float* outs = out_scores ? out_scores + (int64_t)qi * K : nullptr;
  const float* srow = scores + (int64_t)qi * score_stride + my0;

  for (int e = tid; e < my_len; e += kSelThreads) {
    sc[e] = srow[e];
    state[e] = (nvis <= K) ? 1 : 0;
  }
  __syncthreads();

  if (nvis > K) {
    int remaining = need;
    int level = 0;
    for (;; ++level) {
      // ---- local statistics of the surviving candidates
      float lo = INFINITY, hi = -INFINITY;
      int cnt = 0;
      for (int e = tid; e < my_len; e += kSelThreads)
        if (state[e] == 0) {
          float s = sc[e];
          lo = fminf(lo, s);
          hi = fmaxf(hi, s);
          ++cnt;
        }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
        hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
        cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
      }
      if ((tid & 31) == 0) {
        sh.red_f[0][tid >> 5] = lo;
        sh.red_f[1][tid >> 5] = hi;
        sh.red_i[tid >> 5] = cnt;
      }
      if (tid == 0) sh.cand_n = 0;
      __syncthreads();
      if (tid == 0) {
        float l = INFINITY, h = -INFINITY;
        int c = 0;
        for (int w = 0; w < kSelThreads / 32; ++w) {
          l = fminf(l, sh.red_f[0][w]);
          h = fmaxf(h, sh.red_f[1][w]);
          c += sh.red_i[w];
        }
        sh.rec[level].lo = l;
        sh.rec[level].hi = h;
        sh.rec[level].cnt = c;
      }
      __syncthreads();
      const int my_cnt = sh.rec[level].cnt;
      if (my_cnt <= kCandCap) {
        for (int e = tid; e < my_len; e += kSelThreads)
          if (state[e] == 0) {
            int p = atomicAdd(&sh.cand_n, 1);
            sh.cand_s[p] = sc[e];
            sh.cand_i[p] = my0 + e;
          }
      }
      cluster.sync();  // publish rec[level] and the candidate list

      float glo = INFINITY, ghi = -INFINITY;
      int gcnt = 0, pre_cnt = 0;
      for (int rr = 0; rr < C; ++rr) {
        const SelRec* rec = cluster.map_shared_rank(&sh.rec[level], rr);
        SelRec v = *rec;
        if (v.cnt > 0) {
          glo = fminf(glo, v.lo);
          ghi = fmaxf(ghi, v.hi);
        }
        if (rr < r) pre_cnt += v.cnt;
        gcnt += v.cnt;
      }

      if (remaining >= gcnt) {
        // every surviving candidate is needed
        for (int e = tid; e < my_len; e += kSelThreads)
          if (state[e] == 0) state[e] = 1;
        __syncthreads();
        break;
      }
      if (gcnt <= kCandCap) {
        // exact resolution: rank own candidates among all, by (score desc, index asc)
        int off = 0;
        for (int rr = 0; rr < C; ++rr) {
          const SelRec* rec = cluster.map_shared_rank(&sh.rec[level], rr);
          const int n = rec->cnt;
          const float* rs = cluster.map_shared_rank(sh.cand_s, rr);
          const int* ri = cluster.map_shared_rank(sh.cand_i, rr);
          for (int j = tid; j < n; j += kSelThreads) {
            sh.all_s[off + j] = rs[j];
            sh.all_i[off + j] = ri[j];
          }
          off += n;
        }
        __syncthreads();
        for (int j = tid; j < my_cnt; j += kSelThreads) {
          const float s = sh.cand_s[j];
          const int i = sh.cand_i[j];
          int rank = 0;
          for (int c = 0; c < gcnt; ++c) {
            const float t = sh.all_s[c];
            rank += (t > s) || (t == s && sh.all_i[c] < i);
          }
          state[i - my0] = rank < remaining ? 1 : 2;
        }
        __syncthreads();
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
            state[e] = ord < remaining ? 1 : 2;
            ++ord;
          }
        __syncthreads();
        break;
      }
      // ---- histogram refinement round
      const float scl = (float)kNB / (ghi - glo);
      for (int i = tid; i < kNB; i += kSelThreads) sh.hist[i] = 0u;
      __syncthreads();
      for (int e = tid; e < my_len; e += kSelThreads)
        if (state[e] == 0) atomicAdd(&sh.hist[bin_of(sc[e], glo, scl)], 1u);
      cluster.sync();  // publish hist
      for (int i = tid; i < kNB; i += kSelThreads) {
        uint32_t s = 0;
        for (int rr = 0; rr < C; ++rr) s += *cluster.map_shared_rank(&sh.hist[i], rr);
        sh.ghist[i] = s;
      }
      __syncthreads();
      // suffix sums from the top bin: find b* with above(b*) < remaining <= above(b*) + h(b*)
      {
        constexpr int kPer = kNB / kSelThreads;  // 2 bins per thread, thread 0 owns the top
        const int bhi = kNB - 1 - tid * kPer;
        int mine = 0;
#pragma unroll
        for (int k = 0; k < kPer; ++k) mine += (int)sh.ghist[bhi - k];
        int total;
        int above = block_excl_scan(mine, sh.scan, total);
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
          const int bb = bhi - k;
          const int h = (int)sh.ghist[bb];
          if (above < remaining && remaining <= above + h) {
            sh.bstar = bb;
            sh.red_i[0] = above;
          }
          above += h;
        }
      }
      __syncthreads();
      const int bstar = sh.bstar;
      remaining -= sh.red_i[0];
      for (int e = tid; e < my_len; e += kSelThreads)
        if (state[e] == 0) {
          const int bi = bin_of(sc[e], glo, scl);
          state[e] = bi > bstar ? 1 : (bi < bstar ? 2 : 0);
        }
      __syncthreads();
    }
  }

  // ---- ordered output
  const int chunk = (my_len + kSelThreads - 1) / kSelThreads;
  const int e0 = tid * chunk, e1 = min(e0 + chunk, my_len);
  int c = 0;
  for (int e = e0; e < e1; ++e) c += state[e] == 1;
  int my_sel;
  int pos = block_excl_scan(c, sh.scan, my_sel);
  if (tid == 0) sh.sel_cnt = my_sel;
  cluster.sync();  // publish sel_cnt
  int offset = 0, total_sel = 0;
  for (int rr = 0; rr < C; ++rr) {
    const int v = *cluster.map_shared_rank(&sh.sel_cnt, rr);
    if (rr < r) offset += v;
    total_sel += v;
  }
  pos += offset;
  for (int e = e0; e < e1; ++e)
    if (state[e] == 1) {
      if (pos < K) {
        out[pos] = my0 + e;
        if (outs) outs[pos] = sc[e];
      }
      ++pos;
    }
  if (r == C - 1)
    for (int p = total_sel + tid; p < K; p += kSelThreads) {
      out[p] = -1;
      if (outs) outs[p] = __int_as_float(0x7fc00000);
    }
  cluster.sync();  // keep shared memory alive until every remote read is done
}

static int select_cluster_size(int64_t n_stride) {
  int64_t per = (n_stride + 4095) / 4096;
  int c = 1;
  while (c < per && c < 16) c <<= 1;
  return c;
}

cudaError_t launch_topk_select(const float* scores, int64_t score_stride, const int32_t* n_visible,
                               int Q, int64_t n_stride, int K, int32_t* out_idx, float* out_scores,
                               uint32_t* status, cudaStream_t st) {
  if (Q == 0) return cudaSuccess;
  const int C = select_cluster_size(n_stride);
  int slice_cap = (int)((n_stride + C - 1) / C);
  slice_cap = (slice_cap + 15) & ~15;
  const size_t smem = sizeof(SelShared) + (size_t)slice_cap * 5;
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
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, topk_select_kernel, scores, score_stride, n_visible, n_stride, K,
                            slice_cap, out_idx, out_scores, status);
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
