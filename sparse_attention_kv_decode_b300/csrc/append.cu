// Decode-time cache append (csa2_cache_append): one new token per sequence.
//
// "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression": the sliding
// window covers the most recent n_win tokens (blog repost), the cache holds one
// compressed entry per four tokens (wesearch.press card), stored in FP4 with one E4M3
// scale per 16 channels (picx.dev summary, Methodology / 5).
//
// Window rows live in a mirrored ring of R = n_win slots stored twice: token p goes to
// rows p % R and p % R + R, so the last min(p+1, R) tokens are always the contiguous
// rows [(p+1-len) % R, +len), which the attention kernels read as one 2-D box. Token p
// completes entry e = (p+1)/ratio - 1 when (p+1) % ratio == 0; the caller supplies that
// entry's latent row and indexer key (the token-to-entry compressor is not part of the
// library), and the entry is quantised with the cache codec.
//
// One CTA of 128 threads per sequence: threads 0-71 copy the 1152-byte window row to
// both ring rows (16 bytes each), threads 0-35 quantise one 16-channel block of the
// entry each, threads 0-7 copy the 128-byte indexer key. A few KB per sequence: the
// call is launch-bound.
#include "csa2_internal.cuh"

namespace csa2 {

constexpr int kAppendThreads = 128;

__global__ void __launch_bounds__(kAppendThreads) cache_append_kernel(
    int32_t* __restrict__ n_tokens, int advance, int ratio, const uint16_t* __restrict__ swa_row,
    uint16_t* __restrict__ swa_kv, int64_t s_stride, int n_win, const void* __restrict__ entry_kv,
    int entry_bf16, const uint16_t* __restrict__ entry_z, uint8_t* __restrict__ codes,
    uint8_t* __restrict__ scales, uint16_t* __restrict__ z, int64_t n_stride,
    int32_t* __restrict__ n_visible, int32_t* __restrict__ win_start, int32_t* __restrict__ win_len,
    uint32_t* __restrict__ status) {
  // the previous step's attention may still read the ring row this token replaces
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int b = blockIdx.x, t = threadIdx.x;
  // the inputs' addresses do not depend on the token position: issue every load at once
  const int p = n_tokens[b];
  uint4 wrow = make_uint4(0, 0, 0, 0), zrow = make_uint4(0, 0, 0, 0);
  if (swa_row != nullptr && t < CSA2_D_KV / 8)
    wrow = reinterpret_cast<const uint4*>(swa_row + (int64_t)b * CSA2_D_KV)[t];
  if (entry_z != nullptr && t < CSA2_D_IDX / 8)
    zrow = reinterpret_cast<const uint4*>(entry_z + (int64_t)b * CSA2_D_IDX)[t];
  float v[16];
  if (entry_kv != nullptr && t < CSA2_D_KV / 16) {
    if (entry_bf16) {
      const uint4* src =
          reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(entry_kv) + (int64_t)b * CSA2_D_KV) + 2 * t;
      const uint4 a = src[0], c = src[1];
      const uint32_t w[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        v[2 * k] = bf16_lo(w[k]);
        v[2 * k + 1] = bf16_hi(w[k]);
      }
    } else {
      const float4* src =
          reinterpret_cast<const float4*>(static_cast<const float*>(entry_kv) + (int64_t)b * CSA2_D_KV) + 4 * t;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float4 f = src[k];
        v[4 * k] = f.x; v[4 * k + 1] = f.y; v[4 * k + 2] = f.z; v[4 * k + 3] = f.w;
      }
    }
  }
  if (p < 0) return;  // idle sequence (the same value for the whole CTA)
  const int64_t p1 = (int64_t)p + 1;

  if (swa_row != nullptr && t < CSA2_D_KV / 8) {
    const int64_t slot = p % n_win;
    uint16_t* base = swa_kv + (int64_t)b * s_stride * CSA2_D_KV;
    reinterpret_cast<uint4*>(base + slot * CSA2_D_KV)[t] = wrow;
    reinterpret_cast<uint4*>(base + (slot + n_win) * CSA2_D_KV)[t] = wrow;
  }
  if (p1 % ratio == 0) {
    const int64_t e = p1 / ratio - 1;
    if (e >= n_stride) {
      if (t == 0 && (entry_kv != nullptr || entry_z != nullptr)) atomicOr(status, CSA2_DEV_BAD_INDEX);
    } else {
      const int64_t row = (int64_t)b * n_stride + e;
      if (entry_kv != nullptr && t < CSA2_D_KV / 16) {
        uint32_t lo, hi, sc;
        quant_block16(v, lo, hi, sc);
        *reinterpret_cast<uint2*>(codes + row * CSA2_ENTRY_BYTES + 8 * t) = make_uint2(lo, hi);
        scales[row * CSA2_ENTRY_BYTES + t] = (uint8_t)sc;
      }
      if (entry_z != nullptr && t < CSA2_D_IDX / 8) reinterpret_cast<uint4*>(z + row * CSA2_D_IDX)[t] = zrow;
    }
  }
  if (t == 0) {
    if (n_visible != nullptr) n_visible[b] = (int32_t)(p1 / ratio);
    if (win_start != nullptr) {
      const int64_t len = p1 < n_win ? p1 : n_win;
      win_start[b] = (int32_t)((p1 - len) % n_win);
      win_len[b] = (int32_t)len;
    }
  }
  __syncthreads();  // every thread has read n_tokens[b]
  if (advance && t == 0) {
    if (p1 <= INT32_MAX) n_tokens[b] = (int32_t)p1;
    else atomicOr(status, CSA2_DEV_BAD_INDEX);
  }
}

cudaError_t launch_cache_append(int B, int32_t* n_tokens, int advance, int ratio, const void* swa_row,
                                void* swa_kv, int64_t s_stride, int n_win, const void* entry_kv,
                                int entry_dtype, const void* entry_z, uint8_t* codes, uint8_t* scales,
                                void* z, int64_t n_stride, int32_t* n_visible, int32_t* win_start,
                                int32_t* win_len, uint32_t* status, cudaStream_t st) {
  if (B == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)B);
  cfg.blockDim = dim3(kAppendThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, cache_append_kernel, n_tokens, advance, ratio,
                            static_cast<const uint16_t*>(swa_row), static_cast<uint16_t*>(swa_kv), s_stride,
                            n_win < 1 ? 1 : n_win, entry_kv, entry_dtype == CSA2_BF16 ? 1 : 0,
                            static_cast<const uint16_t*>(entry_z), codes, scales, static_cast<uint16_t*>(z),
                            n_stride, n_visible, win_start, win_len, status);
}

}  // namespace csa2
