// FP4 main-KV quantiser (quantise-only path of csa2_encode_kv).
//
// Format: "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression",
// picx.dev summary, Methodology / 5. FP4 Main KV Cache: E2M1 elements with one
// E4M3 scale per 16 channels. Per block: s = E4M3(fl32(amax/6)), code_i =
// E2M1(fl32(x_i/s)), both round-to-nearest-even with saturation; a zero scale
// gives zero codes. The kernel is HBM-bound: one thread per 16-channel block,
// 64-byte (fp32) or 32-byte (bf16) coalesced reads, 8-byte code stores into the
// entry's CSA2_ENTRY_BYTES row.
#include "csa2_internal.cuh"

namespace csa2 {

template <bool kBf16>
__global__ void __launch_bounds__(256) encode_quant_kernel(const void* __restrict__ h,
                                                           int64_t nblk,
                                                           uint8_t* __restrict__ codes,
                                                           uint8_t* __restrict__ scales) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < nblk;
       i += (int64_t)gridDim.x * blockDim.x) {
    float v[16];
    if (kBf16) {
      const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(h) + i * 16);
      uint4 a = __ldcs(src), b = __ldcs(src + 1);
      uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        v[2 * k] = bf16_lo(w[k]);
        v[2 * k + 1] = bf16_hi(w[k]);
      }
    } else {
      const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(h) + i * 16);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float4 f = __ldcs(src + k);
        v[4 * k] = f.x; v[4 * k + 1] = f.y; v[4 * k + 2] = f.z; v[4 * k + 3] = f.w;
      }
    }
    uint32_t lo, hi, sc;
    quant_block16(v, lo, hi, sc);
    // block j = i % 36 of entry row i / 36 (rows of CSA2_ENTRY_BYTES)
    const int64_t row = i / (CSA2_D_KV / 16), j = i - row * (CSA2_D_KV / 16);
    *reinterpret_cast<uint2*>(codes + row * CSA2_ENTRY_BYTES + j * 8) = make_uint2(lo, hi);
    scales[row * CSA2_ENTRY_BYTES + j] = (uint8_t)sc;
  }
}

cudaError_t launch_encode_quant(const void* h, int h_dtype, int64_t rows, uint8_t* codes,
                                uint8_t* scales, cudaStream_t st) {
  int64_t nblk = rows * (CSA2_D_KV / 16);
  if (nblk == 0) return cudaSuccess;
  int n_sm = device_sm_count();
  int64_t want = (nblk + 255) / 256;
  int grid = (int)(want < (int64_t)n_sm * 8 ? want : (int64_t)n_sm * 8);
  if (h_dtype == CSA2_BF16)
    encode_quant_kernel<true><<<grid, 256, 0, st>>>(h, nblk, codes, scales);
  else
    encode_quant_kernel<false><<<grid, 256, 0, st>>>(h, nblk, codes, scales);
  return cudaGetLastError();
}

}  // namespace csa2
