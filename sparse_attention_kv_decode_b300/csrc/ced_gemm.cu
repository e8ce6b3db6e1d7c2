// CED prefill KV projection fused with the FP4 cache write.
//
// Ref: "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression",
// picx.dev summary, Methodology / 1. Causal Encoder-Decoder (CED), Eq. (1):
// C_l = H_{L/2} W_l^KV and Z_l = H_{L/2} W_l^Z for every decoder layer l. C_l is
// stored in the FP4 main-KV format (Methodology / 5. FP4 Main KV Cache), Z_l in
// bf16.
//
// One persistent, warp-specialised tcgen05 GEMM over the concatenated output
// columns of every layer ([576 kv | 64 z] per layer, 640 per layer). The CTAs run
// in pairs (clusters of 2) on the row tiles 2i and 2i+1 of the same column tile:
// each loads half of the weight boxes and multicasts them to both, so the weight
// lines that many SMs read at the same moment leave L2 once per pair (those
// shared reads, not the H tiles, were what held the tensor pipe back):
//   warp 0      TMA producer: own H tile 128x64 and two of the four 64-row weight
//               boxes per k-block (multicast to the pair) into a 4-stage
//               shared-memory ring (128-byte swizzle); a stage is refilled once
//               the MMAs of both CTAs have released it
//   warp 1      TMEM allocation and the MMA issuer: tcgen05.mma kind::f16,
//               M=128, N=256, K=16, fp32 accumulators in TMEM, double-buffered
//               (2 x 256 columns) so the epilogue of one tile overlaps the
//               MMAs of the next
//   warps 2..5  epilogue: tcgen05.ld of one accumulator row per thread, FP4
//               quantisation of each 16-channel block (same codec as the
//               quantise-only path) or bf16 rounding of Z, and the stores.
// Every mbarrier wait is bounded; a wait that gives up sets a status bit, the
// CTA stops issuing work, drains what it started and frees its TMEM.
#include <cuda.h>
#include "csa2_internal.cuh"

namespace csa2 {
namespace {

constexpr int kBM = 128, kBN = 256, kBK = 64;
constexpr int kStages = 4;
constexpr int kABytes = kBM * kBK * 2;          // 16 KB
constexpr int kSegBytes = 64 * kBK * 2;         // 8 KB: one 64-row weight box
constexpr int kBBytes = kBN * kBK * 2;          // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;  // 48 KB
constexpr int kSegPerLayer = 10;                // 9 kv segments (576) + 1 z segment (64)
constexpr int kThreads = 192;
constexpr int kTmemCols = 512;
constexpr int kGroupM = 8;                      // m-tile pairs per raster group
constexpr size_t kSmemBytes = kStages * kStageBytes + 1024 + 256;

// Work item t of a pair: m-tile pair mp (row tiles 2mp, 2mp+1) x column tile n,
// m-pairs fastest inside groups of kGroupM pairs.
struct TileMap {
  int m_pairs, n_tiles, total;
  __device__ __forceinline__ void coords(int t, int rank, int& m, int& n) const {
    const int per_group = kGroupM * n_tiles;
    const int grp = t / per_group;
    const int in = t - grp * per_group;
    const int gm = min(kGroupM, m_pairs - grp * kGroupM);
    n = in / gm;
    m = 2 * (grp * kGroupM + in % gm) + rank;
  }
};

__device__ __forceinline__ void cluster_sync_pair() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
// arrive on the same mbarrier of both CTAs of the pair once the MMAs issued so far complete
__device__ __forceinline__ void umma_commit_pair(uint32_t mbar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          mbar),
      "h"((uint16_t)3)
      : "memory");
}
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, int x, int y,
                                                 uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(mbar), "h"((uint16_t)3)
      : "memory");
}

__global__ void __launch_bounds__(kThreads, 1) ced_proj_kernel(
    const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmWkv,
    const __grid_constant__ CUtensorMap tmWz, int rows, int d_model, int n_layers,
    uint8_t* __restrict__ codes, uint8_t* __restrict__ scales, uint16_t* __restrict__ z_out,
    uint32_t* __restrict__ status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + kStages * kStageBytes;
  const uint32_t bar_empty = bar_full + kStages * 8;
  const uint32_t bar_tfull = bar_empty + kStages * 8;
  const uint32_t bar_tempty = bar_tfull + 2 * 8;
  const uint32_t bar_drain = bar_tempty + 2 * 8;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + kStages * kStageBytes + 128);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_segs = n_layers * kSegPerLayer;
  uint32_t rank;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
  const int pair = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;
  TileMap tm;
  tm.m_pairs = ((rows + kBM - 1) / kBM + 1) / 2;
  tm.n_tiles = (n_segs + 3) / 4;
  tm.total = tm.m_pairs * tm.n_tiles;
  const int kblocks = d_model / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 2);   // released by the MMAs of both CTAs
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar_tfull + 8 * a, 1);
      mbar_init(bar_tempty + 8 * a, 128);
    }
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_holder)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // both CTAs' barriers exist before the pair's first multicast or remote arrive
  cluster_sync_pair();
  const uint32_t tmem = *tmem_holder;

  if (warp == 0) {
    // ---------------- TMA producer
    uint32_t armed_phase[kStages];
    bool armed[kStages];
    for (int s = 0; s < kStages; ++s) armed[s] = false, armed_phase[s] = 0;
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int t = pair; t < tm.total && !*abort_flag; t += n_pairs) {
        int m, n;
        tm.coords(t, (int)rank, m, n);
        int nseg = n_segs - 4 * n;
        nseg = nseg > 4 ? 4 : nseg;
        const uint32_t bytes = kABytes + nseg * kSegBytes;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1)) {
            atomicOr(status, CSA2_DEV_PIPELINE_TIMEOUT);
            *abort_flag = 1;
            break;
          }
          const uint32_t fb = bar_full + 8 * stage;
          mbar_arrive_expect_tx(fb, bytes);
          armed[stage] = true;
          armed_phase[stage] = phase;
          const uint32_t sa = sbase + stage * kStageBytes;
          // rows past the matrix (an odd last pair) read as zeros
          tma_load_2d(sa, &tmA, kb * kBK, m * kBM, fb);
          // weight boxes s of this CTA's parity, into the same stage of both CTAs
          for (int s = (int)rank; s < nseg; s += 2) {
            const int g = 4 * n + s, l = g / kSegPerLayer, sl = g % kSegPerLayer;
            const uint32_t sb = sa + kABytes + s * kSegBytes;
            if (sl < 9)
              tma_load_2d_pair(sb, &tmWkv, kb * kBK, l * CSA2_D_KV + sl * 64, fb);
            else
              tma_load_2d_pair(sb, &tmWz, kb * kBK, l * CSA2_D_IDX, fb);
          }
          if (++stage == kStages) stage = 0, phase ^= 1;
        }
      }
      // drain: every armed stage's copies have landed before the CTA may exit
      for (int s = 0; s < kStages; ++s)
        if (armed[s]) mbar_wait(bar_full + 8 * s, armed_phase[s]);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kBM, kBN);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool issued = false;
      for (int t = pair; t < tm.total && !*abort_flag; t += n_pairs) {
        if (!mbar_wait(bar_tempty + 8 * acc, acc_phase ^ 1)) {
          atomicOr(status, CSA2_DEV_PIPELINE_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + acc * kBN;
        bool ok = true;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(bar_full + 8 * stage, phase)) {
            atomicOr(status, CSA2_DEV_PIPELINE_TIMEOUT);
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = sbase + stage * kStageBytes;
          const uint64_t ad = umma_desc_sw128(sa), bd = umma_desc_sw128(sa + kABytes);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            umma_bf16(d_tmem, ad + (uint64_t)(k * 2), bd + (uint64_t)(k * 2), idesc,
                      (kb | k) != 0);
          umma_commit_pair(bar_empty + 8 * stage);
          issued = true;
          if (++stage == kStages) stage = 0, phase ^= 1;
        }
        if (!ok) break;
        umma_commit(bar_tfull + 8 * acc);
        if (++acc == 2) acc = 0, acc_phase ^= 1;
      }
      if (issued) {
        umma_commit(bar_drain);
        mbar_wait(bar_drain, 0);
      }
    }
  } else {
    // ---------------- epilogue: one accumulator row per thread
    const int quarter = warp & 3;
    const int r_in = quarter * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = pair; t < tm.total; t += n_pairs) {
      if (*abort_flag) break;
      int m, n;
      tm.coords(t, (int)rank, m, n);
      bool ok = mbar_wait(bar_tfull + 8 * acc, acc_phase);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        if (lane == 0) atomicOr(status, CSA2_DEV_PIPELINE_TIMEOUT);
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const int row = m * kBM + r_in;
      const uint32_t tbase = tmem + acc * kBN + ((uint32_t)(quarter * 32) << 16);
      for (int s = 0; s < 4; ++s) {
        const int g = 4 * n + s;
        if (g >= n_segs) break;  // uniform across the CTA
        uint32_t r[64];
        tmem_ld32(tbase + s * 64, r);
        tmem_ld32(tbase + s * 64 + 32, r + 32);
        tmem_wait_ld();
        if (row >= rows) continue;
        const int l = g / kSegPerLayer, sl = g % kSegPerLayer;
        const int64_t orow = (int64_t)l * rows + row;
        if (sl < 9) {
          uint32_t cw[8], sc4 = 0;
#pragma unroll
          for (int bk = 0; bk < 4; ++bk) {
            float v[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[16 * bk + i]);
            uint32_t lo, hi, sc;
            quant_block16(v, lo, hi, sc);
            cw[2 * bk] = lo;
            cw[2 * bk + 1] = hi;
            sc4 |= sc << (8 * bk);
          }
          uint8_t* cdst = codes + orow * CSA2_ENTRY_BYTES + sl * 32;
          *reinterpret_cast<uint4*>(cdst) = make_uint4(cw[0], cw[1], cw[2], cw[3]);
          *reinterpret_cast<uint4*>(cdst + 16) = make_uint4(cw[4], cw[5], cw[6], cw[7]);
          *reinterpret_cast<uint32_t*>(scales + orow * CSA2_ENTRY_BYTES + sl * 4) = sc4;
        } else {
          uint32_t pk[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(r[2 * i]),
                                                      __uint_as_float(r[2 * i + 1]));
            pk[i] = *reinterpret_cast<uint32_t*>(&h2);
          }
          uint4* zdst = reinterpret_cast<uint4*>(z_out + orow * CSA2_D_IDX);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            zdst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
      }
      tc_fence_before();
      mbar_arrive(bar_tempty + 8 * acc);
      if (++acc == 2) acc = 0, acc_phase ^= 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
  // the peer's multicasts into this CTA and its releases of this CTA's stages have
  // landed before either CTA exits
  cluster_sync_pair();
}

}  // namespace

cudaError_t launch_ced_project(const void* h, int64_t rows, int d_model, const void* w_kv,
                               const void* w_z, int n_layers, uint8_t* codes, uint8_t* scales,
                               void* z_out, uint32_t* status, cudaStream_t st) {
  if (rows <= 0 || n_layers <= 0) return cudaSuccess;
  if (rows > (int64_t)1 << 30) return cudaErrorInvalidValue;
  CUtensorMap ta, tkv, tz;
  if (!encode_tensor_map_2d_bf16(&ta, h, (uint64_t)d_model, (uint64_t)rows, kBK, kBM) ||
      !encode_tensor_map_2d_bf16(&tkv, w_kv, (uint64_t)d_model, (uint64_t)n_layers * CSA2_D_KV, kBK, 64) ||
      !encode_tensor_map_2d_bf16(&tz, w_z, (uint64_t)d_model, (uint64_t)n_layers * CSA2_D_IDX, kBK, 64))
    return cudaErrorInvalidValue;
  cudaError_t e = set_attr_once(4, (const void*)ced_proj_kernel,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  const int64_t m_pairs = ((rows + kBM - 1) / kBM + 1) / 2;
  const int64_t n_tiles = ((int64_t)n_layers * kSegPerLayer + 3) / 4;
  const int64_t total = m_pairs * n_tiles;
  const int n_pairs_max = device_sm_count() / 2;
  const int grid = 2 * (int)(total < n_pairs_max ? total : n_pairs_max);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, ced_proj_kernel, ta, tkv, tz, (int)rows, d_model, n_layers, codes,
                            scales, static_cast<uint16_t*>(z_out), status);
}

}  // namespace csa2
